// K4, channels-last: backward of the offset convolution, for the problems the
// channels-last sampling backward handles (bf16, one offset group).
//
// The offset convolution is a plain convolution of x ("Following a deformable
// layer through DefT", Step 1 of 5, on the explainer page "DefT: Boosting
// Scalability of Deformable Convolution Operations on GPUs"): its output has
// M = 2K channels per pixel.  With goff, the gradient of that output (summed
// over all channels by the sampling backward),
//
//   input part   grad_x[c][q]  += sum_(k,m) w_off[m][c][k] * goff[m][px(q,k)]
//                px(q,k) = the output pixel whose tap k reads position q
//   weight part  gw_off[m][c][k] = sum_(n,px) goff[m][px] * x[c][pos(px,k)]
//   bias         gb_off[m]      = sum_(n,px) goff[m][px]
//
// Input part (k4cl_input): one CTA per (tile of 8 x 16 input positions,
// slice of up to 128 channels, image).  It stages the goff pixels whose taps
// read its positions, builds their im2col A[q][(k,m)] (bf16) in shared memory,
// copies w_off as B[c][(k,m)] (bf16, laid out once per call by the weight
// part, which runs first), multiplies them on the tensor cores (mma.sync
// m16n8k16, fp32 accumulate), adds the sampling backward's contribution from
// its NHWC float32 buffer and writes grad_x (NCHW) once: no atomics, no
// separate transpose.  When x is a ReLU's output (in_relu), that store is the
// ReLU's backward: bf16, zero where x is not above zero.
//
// Weight part (k4cl_weight): the reduction runs over every pixel of the batch,
// so the CTAs split the pixels into chunks and the channels into slices of
// 64; two warps own each tap and keep D[c][m] = sum_px x[pos(px,k)][c] *
// goff[m][px] for 32 channels each in registers (mma.sync, A = x^T from the staged
// NHWC window by ldmatrix.trans, B = goff).  Each CTA writes its partial sums
// once; a small kernel adds the chunks (and the bias partials) in a fixed
// order.
#include <string.h>

#include "dc_band.cuh"
#include "dc_tma.cuh"

namespace dc {

// Raised by this file's bounded waits (read by dc_device_error).
__device__ unsigned int g_k4cl_error;

namespace {

// ------------------------------------------------------------------ input part
constexpr int kTY = 8, kTX = 16, kQ = kTY * kTX;  // positions per CTA
constexpr int kInThreads = 256;
static_assert(kInThreads % kQ == 0, "each input-part thread keeps one position");
constexpr int kMaxKMp = 192;  // (tap, offset channel) pairs, padded to 16
constexpr int kMaxK = 9;      // taps (the offset channels are M = 2K)
constexpr int kPermCh = 128;  // input channels per block of the grad_w permutation

__host__ __device__ inline int km_padded(const Geom& g) { return (g.K * g.M + 15) / 16 * 16; }
__host__ __device__ inline int in_pitch(const Geom& g) { return km_padded(g) + 8; }  // bf16 elements

// goff rows / columns read by a tile of positions
__host__ __device__ inline int in_gy(const Geom& g) { return (kTY - 1 + (g.kh - 1) * g.dh) / g.sh + 2; }
__host__ __device__ inline int in_gx(const Geom& g) { return (kTX - 1 + (g.kw - 1) * g.dw) / g.sw + 2; }
// The goff tile arrives by one TMA box when goff's rows are 16-byte aligned
// (Wo a multiple of 4): the box starts at the column rounded down to a
// multiple of 4 and is as many columns wider, a multiple of 4 in all.
__host__ __device__ inline bool in_goff_tma(const Geom& g) { return g.wo % 4 == 0; }
__host__ __device__ inline int in_gxp(const Geom& g) {
  return in_goff_tma(g) ? (in_gx(g) + 3 + 3) / 4 * 4 : in_gx(g);
}
__host__ __device__ inline int floor_div(int a, int b) { return a >= 0 ? a / b : -((-a + b - 1) / b); }
// shared memory: A [kQ][pitch] and B [cpc][pitch] (bf16), then the goff tile
// (float); the transposed result later lies over A and B
// (offsets from the dynamic array advanced to a 128-byte boundary; the goff
// tile is a TMA destination, its mbarrier follows it)
__host__ __device__ inline size_t in_g_off(const Geom& g, int cpc) {
  const size_t ab = (size_t)(kQ + cpc) * in_pitch(g) * 2;
  const size_t t = (size_t)cpc * (kQ + 4) * 4;
  return ((ab > t ? ab : t) + 127) / 128 * 128;
}
__host__ __device__ inline size_t in_bar_off(const Geom& g, int cpc) {
  return in_g_off(g, cpc) + ((size_t)g.M * in_gy(g) * in_gxp(g) * 4 + 7) / 8 * 8;
}
__host__ inline size_t input_smem(const Geom& g, int cpc) { return in_bar_off(g, cpc) + 8 + 128; }

__device__ __forceinline__ void mma16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ unsigned short bf16_bits_rn(float v) {
  const __nv_bfloat16 b = __float2bfloat16_rn(v);
  return *reinterpret_cast<const unsigned short*>(&b);
}

struct K4InArgs {
  Geom g;
  const float* goff;                // [n][M][Ho][Wo]
  const unsigned short* bt;         // [C][KMp] bf16 bits: w_off as B (written by k4cl_weight)
  const float* gx_nhwc;             // sampling backward's grad_x, [n][H][W][C]
  const unsigned short* x;          // [n][C][H][W] bf16 bits, the ReLU mask (g.in_relu)
  void* grad_x;                     // [n][C][H][W] float32, or bf16 masked by x > 0 (g.in_relu)
  int tiles_x, cpc;
};

// The ReLU backward fused into the grad_x store: v where the activation x is
// above zero, else 0, rounded to bf16 (nearest even) -- the same value the
// stand-alone ReLU backward kernel writes for v.
__device__ __forceinline__ unsigned int relu_grad2(float v0, float v1, unsigned int x2) {
  const float a0 = __uint_as_float(x2 << 16), a1 = __uint_as_float(x2 & 0xffff0000u);
  const __nv_bfloat162 b = __floats2bfloat162_rn(a0 > 0.f ? v0 : 0.f, a1 > 0.f ? v1 : 0.f);
  return *reinterpret_cast<const unsigned int*>(&b);
}

// CPC channels per CTA (64 or 128).  Warps: 8 m-tiles of 16 positions x
// CPC/8 n-tiles of 8 channels; a warp holds MTW m-tiles x 8 n-tiles.
// gmap: goff [n][M][Ho][Wo] fp32, box {GXP, GY, M, 1}, used when in_goff_tma.
template <int CPC>
__global__ void __launch_bounds__(kInThreads, 2)
    k4cl_input(const __grid_constant__ CUtensorMap gmap, K4InArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const uint32_t raw = px::smem_u32(smem_raw);
  unsigned char* smem = smem_raw + (((raw + 127u) & ~127u) - raw);
  constexpr int MTW = CPC / 64;  // m-tiles per warp (2 or 1)
  const Geom g = a.g;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ty = blockIdx.x / a.tiles_x, tx = blockIdx.x - ty * a.tiles_x;
  const int y0 = ty * kTY, x0 = tx * kTX;
  const int cbeg = blockIdx.y * CPC;
  const int n = blockIdx.z;
  const int M = g.M, K = g.K, C = g.c_in;
  const int KM = K * M, KMp = km_padded(g), P = in_pitch(g);
  unsigned short* A = reinterpret_cast<unsigned short*>(smem);  // [kQ][P]
  unsigned short* B = A + (size_t)kQ * P;                          // [CPC][P]

  // zero padding of the (tap, offset channel) columns of A
  for (int e = tid; e < kQ * (KMp - KM) / 2; e += kInThreads) {
    const int r = e / ((KMp - KM) / 2), j = e - r * ((KMp - KM) / 2);
    reinterpret_cast<uint32_t*>(A + (size_t)r * P + KM)[j] = 0u;
  }
  // the pixels whose taps read this tile's positions: rows hlo .. hlo + GY - 1,
  // columns wlo .. wlo + GX - 1 of goff
  const int GY = in_gy(g), GX = in_gx(g);  // GX <= 32 (k4cl_supported)
  const int hlo = floor_div(y0 + g.ph - (g.kh - 1) * g.dh, g.sh);
  const int wlo = floor_div(x0 + g.pw - (g.kw - 1) * g.dw, g.sw);
  const bool tma = in_goff_tma(g);
  const int GXP = in_gxp(g), wlo0 = tma ? (wlo & ~3) : wlo;  // the tile's first column and pitch
  float* G = reinterpret_cast<float*>(smem + in_g_off(g, CPC));  // [M][GY][GXP]
  uint64_t* gbar = reinterpret_cast<uint64_t*>(smem + in_bar_off(g, CPC));
  if (tma) {
    if (tid == 0) {
      px::mbar_init(gbar, 1);
      px::fence_mbar_init();
    }
    __syncthreads();
  }
  pdl_wait();  // goff and gx_nhwc from the sampling backward, Bt from the weight part
  // goff tile: one TMA box (zero outside goff), or else a warp per (m, row),
  // lanes over the columns (GX <= 32), all rows in flight as 4-byte
  // asynchronous copies (zero-filled outside goff)
  if (tma) {
    if (tid == 0) {
      px::mbar_expect_tx(gbar, (uint32_t)(M * GY * GXP * 4));
      px::tma_load_4d(G, &gmap, gbar, wlo0, hlo, 0, n);
    }
  } else {
    const float* gimg = a.goff + (size_t)n * M * g.howo;
    const int wo = wlo + lane;
    const bool colok = lane < GX && wo >= 0 && wo < g.wo;
    if (lane < GX) {
      for (int r = warp; r < M * GY; r += kInThreads / 32) {
        const int m = r / GY, ho = hlo + (r - m * GY);
        const bool ok = colok && ho >= 0 && ho < g.ho;
        const float* src = ok ? gimg + (size_t)m * g.howo + (size_t)ho * g.wo + wo : gimg;
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(px::smem_u32(G + r * GX + lane)),
                     "l"(src), "r"(ok ? 4 : 0)
                     : "memory");
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  // B rows: Bt[cbeg + c][0 .. KMp) by 16-byte asynchronous copies
  {
    // a warp per row, lanes over its 16-byte pieces (KMp / 8 <= 24)
    const unsigned short* src = a.bt + (size_t)cbeg * KMp;
    for (int c = warp; c < CPC; c += kInThreads / 32)
      if (lane < KMp / 8)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                         px::smem_u32(B + (size_t)c * P + lane * 8)),
                     "l"(src + (size_t)c * KMp + lane * 8)
                     : "memory");
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  if (tma) {
    // the goff tile (B may still be in flight); on a wait that gave up, the
    // copy this CTA issued is waited for once more (bounded) before leaving
    const bool ok = px::mbar_wait(gbar, 0, &g_k4cl_error);
    if (!__syncthreads_and(ok)) {
      if (tid == 0 && !ok) px::mbar_wait(gbar, 0, &g_k4cl_error);
      asm volatile("cp.async.wait_group 0;" ::: "memory");
      pdl_release();
      return;
    }
  } else {
    asm volatile("cp.async.wait_group 1;" ::: "memory");  // the goff tile (B may still be in flight)
    __syncthreads();
  }
  // A[q][k*M + m] = goff[m][pixel whose tap k reads position q], 0 if none:
  // a thread per (q, k), m pairs written as one word (M is even)
  // (kInThreads is a multiple of kQ: each thread keeps its position q)
  const int q = tid % kQ;
  const int yq = y0 + q / kTX + g.ph, xq = x0 + q % kTX + g.pw;
  int ki = 0, kj = tid / kQ;  // this thread's first tap, then every (kInThreads / kQ)-th
  while (kj >= g.kw) {
    kj -= g.kw;
    ++ki;
  }
  for (int k = tid / kQ; k < K; k += kInThreads / kQ) {
    const int ty_ = yq - ki * g.dh, tx_ = xq - kj * g.dw;
    kj += kInThreads / kQ;
    while (kj >= g.kw) {
      kj -= g.kw;
      ++ki;
    }
    int gi = -1;
    if (ty_ >= 0 && tx_ >= 0 && (g.sh == 1 || ty_ % g.sh == 0) && (g.sw == 1 || tx_ % g.sw == 0)) {
      const int ho = ty_ / g.sh, wo = tx_ / g.sw;
      if (ho < g.ho && wo < g.wo) gi = (ho - hlo) * GXP + (wo - wlo0);
    }
    uint32_t* row = reinterpret_cast<uint32_t*>(A + (size_t)q * P + k * M);
    const int plane = GY * GXP;
    const float* gq = G + (gi >= 0 ? gi : 0);
#pragma unroll
    for (int m = 0; m < 2 * kMaxK; m += 2) {
      if (m >= M) break;
      uint32_t w = 0u;
      if (gi >= 0)
        w = (uint32_t)bf16_bits_rn(gq[m * plane]) | ((uint32_t)bf16_bits_rn(gq[(m + 1) * plane]) << 16);
      row[m >> 1] = w;
    }
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  __syncthreads();

  // ---------------------------------------------------------------- MMA
  const int mw = warp % (8 / MTW), nw = warp / (8 / MTW);  // m-tile group, n-tile group
  float acc[MTW][8][4];
#pragma unroll
  for (int i = 0; i < MTW; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[i][j][r] = 0.f;
  const uint32_t abase = px::smem_u32(A), bbase = px::smem_u32(B);
  // ldmatrix row addresses: A x4 = rows 0-15 of the m-tile at k 0-7 / 8-15;
  // B x4 = n rows 0-7 / 8-15 at k 0-7 / 8-15
  const int lr = lane & 15, lk = (lane >> 4) * 8;
  const int br = (lane & 7) + ((lane >> 4) << 3), bk = ((lane >> 3) & 1) * 8;
  for (int k0 = 0; k0 < KMp; k0 += 16) {
    uint32_t af[MTW][4];
#pragma unroll
    for (int i = 0; i < MTW; ++i)
      ldsm_x4(abase + (uint32_t)((((mw * MTW + i) * 16 + lr) * P + k0 + lk) * 2), af[i]);
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      uint32_t bf[4];
      ldsm_x4(bbase + (uint32_t)((((nw * 8 + jj * 2) * 8 + br) * P + k0 + bk) * 2), bf);
#pragma unroll
      for (int i = 0; i < MTW; ++i) {
        mma16816(acc[i][2 * jj], af[i], bf[0], bf[1]);
        mma16816(acc[i][2 * jj + 1], af[i], bf[2], bf[3]);
      }
    }
  }
  __syncthreads();  // A and B are free: the result goes over them

  // ---------------------------------------------------------------- epilogue
  // add the sampling backward's part (NHWC) and transpose through shared
  // memory: T[c][q], pitch kQ + 4
  float* T = reinterpret_cast<float*>(smem);
  constexpr int TP = kQ + 4;
  const int gid = lane >> 2, tig = lane & 3;
#pragma unroll
  for (int i = 0; i < MTW; ++i) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int q = (mw * MTW + i) * 16 + gid + 8 * h;
      const int y = y0 + q / kTX, x = x0 + q % kTX;
      const bool in = y < g.h && x < g.w;
      const float* src = a.gx_nhwc + (((size_t)n * g.h + y) * g.w + x) * C + cbeg;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int c = (nw * 8 + j) * 8 + 2 * tig;
        float2 s = make_float2(0.f, 0.f);
        if (in) s = __ldg(reinterpret_cast<const float2*>(src + c));
        T[(size_t)c * TP + q] = acc[i][j][2 * h] + s.x;
        T[(size_t)(c + 1) * TP + q] = acc[i][j][2 * h + 1] + s.y;
      }
    }
  }
  __syncthreads();
  // grad_x rows: a warp per channel at a time, lanes over four positions
  // each (one 16-byte store when the row length keeps them aligned), else
  // over 32 positions (two rows of the tile)
  const size_t plane0 = ((size_t)n * C + cbeg) * g.hw;
  if (g.in_relu) {
    // the ReLU backward of the layer before: bf16, masked by x > 0 (x read
    // at the same positions, four per lane in one 8-byte load when aligned)
    unsigned short* dst = static_cast<unsigned short*>(a.grad_x) + plane0;
    const unsigned short* act = a.x + plane0;
    if (g.w % 4 == 0) {
      const int q = lane * 4;
      const int y = y0 + q / kTX, x = x0 + q % kTX;
      if (y < g.h && x < g.w) {
        // every load of x in flight before the first store
        constexpr int kIt = CPC / (kInThreads / 32);
        const size_t pos = (size_t)y * g.w + x;
        uint2 xa[kIt];
#pragma unroll
        for (int i = 0; i < kIt; ++i)
          xa[i] = __ldg(reinterpret_cast<const uint2*>(act + (size_t)(warp + i * (kInThreads / 32)) * g.hw + pos));
#pragma unroll
        for (int i = 0; i < kIt; ++i) {
          const int c = warp + i * (kInThreads / 32);
          const float4 v = *reinterpret_cast<const float4*>(T + (size_t)c * TP + q);
          *reinterpret_cast<uint2*>(dst + (size_t)c * g.hw + pos) =
              make_uint2(relu_grad2(v.x, v.y, xa[i].x), relu_grad2(v.z, v.w, xa[i].y));
        }
      }
    } else {
      for (int e = warp; e < CPC * (kQ / 32); e += kInThreads / 32) {
        const int c = e / (kQ / 32), q = (e - c * (kQ / 32)) * 32 + lane;
        const int y = y0 + q / kTX, x = x0 + q % kTX;
        if (y < g.h && x < g.w) {
          const size_t at = (size_t)c * g.hw + (size_t)y * g.w + x;
          dst[at] = (unsigned short)relu_grad2(T[(size_t)c * TP + q], 0.f, act[at]);
        }
      }
    }
    pdl_release();
    return;
  }
  float* dst = static_cast<float*>(a.grad_x) + plane0;
  if (g.w % 4 == 0) {
    static_assert(kTX % 4 == 0 && kQ == 4 * 32 && TP % 4 == 0, "four positions per lane");
    const int q = lane * 4;
    const int y = y0 + q / kTX, x = x0 + q % kTX;
    if (y < g.h && x < g.w) {
      for (int c = warp; c < CPC; c += kInThreads / 32)
        *reinterpret_cast<float4*>(dst + (size_t)c * g.hw + (size_t)y * g.w + x) =
            *reinterpret_cast<const float4*>(T + (size_t)c * TP + q);
    }
  } else {
    for (int e = warp; e < CPC * (kQ / 32); e += kInThreads / 32) {
      const int c = e / (kQ / 32), q = (e - c * (kQ / 32)) * 32 + lane;
      const int y = y0 + q / kTX, x = x0 + q % kTX;
      if (y < g.h && x < g.w) dst[(size_t)c * g.hw + (size_t)y * g.w + x] = T[(size_t)c * TP + q];
    }
  }
  pdl_release();
}

// ------------------------------------------------------------------ weight part
constexpr int kWY = 8, kWX = 16, kWP = kWY * kWX;  // output pixels per tile
constexpr int kWCh = 64;                           // channels per CTA
constexpr int kGbPitch = kWP + 8;                  // bf16 elements per goff row in shared memory
constexpr int kWStages = 3;                        // tiles in flight (two ahead of the one computed)

struct K4WArgs {
  Geom g;
  const float* goff;  // [n][M][Ho][Wo]
  const unsigned short* w_off;  // [M][C][K] bf16 bits
  unsigned short* bt;           // out: [C][KMp], w_off as the input part's B operand
  float* part;        // [chunk][M][C][K]
  float* bpart;       // [chunk][M] (written by the CTAs of channel slice 0)
  int tiles_x, tiles_y, tiles, nchunks;
  int rows, cols;     // the staged x window of a tile
  uint32_t win_pitch; // bytes per window buffer (1024-aligned)
};

__host__ inline size_t weight_smem(uint32_t win_pitch) {
  return 1024 + kWStages * ((size_t)win_pitch + 24 * kGbPitch * 2) + 64;
}

// Two warps per tap (2K warps), M = 2K offset channels: warp w takes tap
// k = w % K for channels 32 hh .. 32 hh + 31 of the slice (hh = w / K) and
// loads goff row k + hh K of each tile (lane l: pixels 4l .. 4l + 3).
__global__ void __launch_bounds__(576, 1)
    k4cl_weight(const __grid_constant__ CUtensorMap xmap, K4WArgs a) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = px::align1024(smem_raw);
  const Geom g = a.g;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int K = g.K, M = g.M, C = g.c_in;
  const int slice = blockIdx.x, chunk = blockIdx.y;
  const int cbeg = slice * kWCh;
  const int tb = (int)((long long)a.tiles * chunk / a.nchunks);
  const int te = (int)((long long)a.tiles * (chunk + 1) / a.nchunks);
  unsigned char* win = smem;  // [kWStages][win_pitch]
  unsigned short* gb =
      reinterpret_cast<unsigned short*>(smem + kWStages * (size_t)a.win_pitch);  // [kWStages][24][pitch]
  uint64_t* wfull = reinterpret_cast<uint64_t*>(gb + kWStages * 24 * kGbPitch);
  const int per_img = a.tiles_x * a.tiles_y;
  const int k = warp % K, hh = warp / K;  // this warp's tap and channel half
  const int ki = k / g.kw, kj = k - ki * g.kw;

  if (tid == 0) {
    for (int q = 0; q < kWStages; ++q) px::mbar_init(&wfull[q], 1);
    px::fence_mbar_init();
  }
  // rows M .. 23 of the goff buffers stay zero
  for (int e = tid; e < kWStages * 24 * kGbPitch; e += blockDim.x) {
    const int r = (e / kGbPitch) % 24;
    if (r >= M) gb[e] = 0;
  }
  __syncthreads();

  auto tile_at = [&](int t, int& n, int& ho0, int& wo0) {
    n = t / per_img;
    const int r = t - n * per_img;
    const int ty = r / a.tiles_x;
    ho0 = ty * kWY;
    wo0 = (r - ty * a.tiles_x) * kWX;
  };
  auto issue = [&](int t, int s) {
    int n, ho0, wo0;
    tile_at(t, n, ho0, wo0);
    px::mbar_expect_tx(&wfull[s], (uint32_t)a.rows * a.cols * 128u);
    px::tma_load_4d(win + (size_t)s * a.win_pitch, &xmap, &wfull[s], cbeg, wo0 * g.sw - g.pw,
                    ho0 * g.sh - g.ph, n);
  };
  // goff row k + hh K of a tile, pixels 4l .. 4l + 3 of lane l
  const int mrow = k + hh * K;
  auto load_goff = [&](int t, float4& v) {
    int n, ho0, wo0;
    tile_at(t, n, ho0, wo0);
    const int ho = ho0 + (lane >> 2), wo = wo0 + (lane & 3) * 4;
    v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (ho < g.ho && wo < g.wo) {
      const float* src = a.goff + ((size_t)n * M + mrow) * g.howo + (size_t)ho * g.wo + wo;
      if (wo + 3 < g.wo && (reinterpret_cast<uintptr_t>(src) & 15) == 0) {
        v = __ldg(reinterpret_cast<const float4*>(src));
      } else {
        v.x = __ldg(src);
        if (wo + 1 < g.wo) v.y = __ldg(src + 1);
        if (wo + 2 < g.wo) v.z = __ldg(src + 2);
        if (wo + 3 < g.wo) v.w = __ldg(src + 3);
      }
    }
  };
  float bsum = 0.f;
  auto store_goff = [&](int s, const float4& v) {
    bsum += (v.x + v.y) + (v.z + v.w);
    uint2 w;
    w.x = (uint32_t)bf16_bits_rn(v.x) | ((uint32_t)bf16_bits_rn(v.y) << 16);
    w.y = (uint32_t)bf16_bits_rn(v.z) | ((uint32_t)bf16_bits_rn(v.w) << 16);
    reinterpret_cast<uint2*>(gb + ((size_t)s * 24 + mrow) * kGbPitch)[lane] = w;
  };

  // D[c][m] for this warp's 32 channels (two 16-channel tiles) and tap
  float acc[2][3][4];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 3; ++j)
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[i][j][r] = 0.f;

  // side job before the wait (w_off only): Bt[c][k*M + m] = w_off[m][c][k],
  // zero in the padding columns, for the input part that runs next
  {
    const int KM = K * M, KMp = km_padded(g);
    const int nthreads = gridDim.x * gridDim.y * blockDim.x;
    const int gtid = (blockIdx.y * gridDim.x + blockIdx.x) * blockDim.x + tid;
    for (int e = gtid; e < C * K; e += nthreads) {
      const int c = e / K, kk = e - c * K;
      const unsigned short* src = a.w_off + (size_t)c * K + kk;
      uint32_t* row = reinterpret_cast<uint32_t*>(a.bt + (size_t)c * KMp + kk * M);
      for (int m = 0; m < M; m += 2)
        row[m >> 1] = (uint32_t)__ldg(src + (size_t)m * C * K) | ((uint32_t)__ldg(src + (size_t)(m + 1) * C * K) << 16);
      if (kk == 0)
        for (int j = KM; j < KMp; j += 2) reinterpret_cast<uint32_t*>(a.bt + (size_t)c * KMp + j)[0] = 0u;
    }
  }
  pdl_wait();  // goff comes from the sampling backward
  float4 g1, g2;  // goff of the next two tiles
  if (tb < te) {
    if (tid == 0) {
      issue(tb, 0);
      if (tb + 1 < te) issue(tb + 1, 1);
    }
    load_goff(tb, g1);
    store_goff(0, g1);
    if (tb + 1 < te) load_goff(tb + 1, g1);
  }
  // ldmatrix lanes: matrix mi = lane >> 3, row lane & 7
  const int mi = lane >> 3, lrow = lane & 7;
  const int a_px = (mi >> 1) * 8 + lrow;  // A (x^T): pixel column of this lane's row
  const int a_half = mi & 1;              //          channel half of the 16-channel tile
  const int b_m = (mi >> 1) * 8 + lrow;   // B (goff): offset channel of this lane's row
  const int b_k = (mi & 1) * 8;           //           pixel half
  for (int t = tb, i = 0; t < te; ++t, ++i) {
    const int s = i % kWStages;
    __syncthreads();  // goff of tile t stored; tile t - 1's buffers are free
    if (tid == 0 && t + 2 < te) issue(t + 2, (i + 2) % kWStages);
    if (t + 2 < te) load_goff(t + 2, g2);
    // every copy is waited for (bounded), so none is in flight at exit
    if (px::mbar_wait(&wfull[s], (uint32_t)(i / kWStages) & 1u, &g_k4cl_error)) {
      const uint32_t wb = px::smem_u32(win + (size_t)s * a.win_pitch);
      const uint32_t gbb = px::smem_u32(gb + (size_t)s * 24 * kGbPitch);
#pragma unroll 2
      for (int pr = 0; pr < kWY; ++pr) {
        // window position of this lane's A row: pixel (pr, a_px), tap k
        const uint32_t pos = (uint32_t)((pr * g.sh + ki * g.dh) * a.cols + a_px * g.sw + kj * g.dw);
        uint32_t bf[6];
        ldsm_x4(gbb + (uint32_t)((b_m * kGbPitch + pr * kWX + b_k) * 2), bf);
        // n-tile 2 (offset channels 16-23): two matrices, addresses from lanes 0-15
        ldsm_x2(gbb + (uint32_t)(((16 + (lane & 7)) * kGbPitch + pr * kWX + ((lane >> 3) & 1) * 8) * 2),
                bf + 4);
#pragma unroll
        for (int ct = 0; ct < 2; ++ct) {
          uint32_t af[4];
          const uint32_t piece = (uint32_t)((2 * hh + ct) * 2 + a_half);
          ldsm_x4_t(wb + pos * 128u + ((piece ^ (pos & 7u)) << 4), af);
          mma16816(acc[ct][0], af, bf[0], bf[1]);
          mma16816(acc[ct][1], af, bf[2], bf[3]);
          mma16816(acc[ct][2], af, bf[4], bf[5]);
        }
      }
    }
    if (t + 1 < te) store_goff((i + 1) % kWStages, g1);
    g1 = g2;
  }
  // this CTA's partial sums: D[c][m] of tap k -> part[chunk][m][c][k]
  float* dst = a.part + (size_t)chunk * M * C * K;
  const int gid = lane >> 2, tig = lane & 3;
#pragma unroll
  for (int ct = 0; ct < 2; ++ct)
#pragma unroll
    for (int nt = 0; nt < 3; ++nt)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int c = cbeg + (2 * hh + ct) * 16 + gid + 8 * (r >> 1);
        const int m = nt * 8 + 2 * tig + (r & 1);
        if (m < M) dst[((size_t)m * C + c) * K + k] = acc[ct][nt][r];
      }
  if (slice == 0) {
    float v = bsum;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) a.bpart[(size_t)chunk * M + mrow] = v;
  }
  pdl_release();
}

// grad_w_off = sum over chunks of the partials; grad_b_off likewise.  A
// block of 32 outputs x 8 chunk groups: thread (x, y) sums the chunks
// y, y + 8, ..., then thread row 0 adds the eight group sums (fixed order).
__global__ void __launch_bounds__(256) k4cl_reduce(const float* __restrict__ part,
                                                   const float* __restrict__ bpart, float* gw_off,
                                                   float* gb_off, int count, int M, int nchunks,
                                                   const float* __restrict__ gw_perm, float* grad_w,
                                                   int wcount, int C, int K) {
  __shared__ float tr[kPermCh * kMaxK];
  pdl_wait();
  const int nred = (count + 255) / 256;
  if ((int)blockIdx.x >= nred) {
    // grad_w[o][c][k] = gw_perm[o][k][c] (the main weight gradient, added in
    // w' order by the GEMM): one block per (o, kPermCh channels), the slice
    // [K][kPermCh] read by rows (every load of the block in flight at once)
    // and written as one run of kPermCh * K floats
    const int b = (int)blockIdx.x - nred;
    const int cch = (C + kPermCh - 1) / kPermCh;
    const int o = b / cch, c0 = (b - o * cch) * kPermCh;
    const int nc = min(kPermCh, C - c0);
    const float* src = gw_perm + (size_t)o * C * K;
    constexpr int kPer = (kPermCh * kMaxK + 255) / 256;  // elements per thread
    float v[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int e = (int)threadIdx.x + 256 * u, k = e / nc;
      if (k < K) v[u] = src[(size_t)k * C + c0 + (e - k * nc)];
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int e = (int)threadIdx.x + 256 * u, k = e / nc;
      if (k < K) tr[(e - k * nc) * K + k] = v[u];
    }
    __syncthreads();
    float* dst = grad_w + ((size_t)o * C + c0) * K;
    for (int e = threadIdx.x; e < nc * K; e += blockDim.x) dst[e] = tr[e];
    pdl_release();
    return;
  }
  // one output per thread: the chunks' partials added in chunk order, sixteen
  // loads in flight; the last sum block's first M threads also add the bias
  const int i = blockIdx.x * 256 + threadIdx.x;
  if (i < count) {
    float v = 0.f;
    int c = 0;
    for (; c + 16 <= nchunks; c += 16) {
      float t[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) t[u] = part[(size_t)(c + u) * count + i];
#pragma unroll
      for (int u = 0; u < 16; ++u) v += t[u];
    }
    for (; c < nchunks; ++c) v += part[(size_t)c * count + i];
    gw_off[i] = v;
  }
  if (gb_off != nullptr && (int)blockIdx.x == nred - 1 && (int)threadIdx.x < M) {
    float v = 0.f;
    for (int c = 0; c < nchunks; ++c) v += bpart[(size_t)c * M + threadIdx.x];
    gb_off[threadIdx.x] = v;
  }
  pdl_release();
}

int sm_count4() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return sms;
}

cudaError_t launch_pdl4(const void* func, dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                        void** args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelExC(&cfg, func, args);
  note_launches(1);
  return e;
}

struct WeightShape {
  int tiles_x, tiles_y, tiles, rows, cols, slices, nchunks;
  uint32_t win_pitch;
};

WeightShape weight_shape(const Geom& g, int sms) {
  WeightShape w{};
  w.tiles_x = (int)ceil_div_ll(g.wo, kWX);
  w.tiles_y = (int)ceil_div_ll(g.ho, kWY);
  w.tiles = g.n * w.tiles_x * w.tiles_y;
  w.rows = (kWY - 1) * g.sh + (g.kh - 1) * g.dh + 1;
  w.cols = (kWX - 1) * g.sw + (g.kw - 1) * g.dw + 1;
  w.win_pitch = ((uint32_t)w.rows * w.cols * 128u + 1023u) / 1024u * 1024u;
  w.slices = g.c_in / kWCh;
  w.nchunks = sms / w.slices > 0 ? sms / w.slices : 1;
  return w;
}

}  // namespace

bool k4cl_supported(const Geom& g) {
  if (g.groups != 1 || g.M != 2 * g.K || g.K > kMaxK || km_padded(g) > kMaxKMp) return false;
  if (g.c_in % 64 != 0 || g.c_in > 256) return false;
  const int sms = sm_count4();
  if (sms <= 0) return false;
  const WeightShape w = weight_shape(g, sms);
  if (w.rows > 256 || w.cols > 256 || weight_smem(w.win_pitch) > 225 * 1024) return false;
  const int cpc = g.c_in >= 128 ? 128 : 64;
  return in_gx(g) <= 32 && input_smem(g, cpc) <= 113 * 1024;
}

// The workspace region: chunk partials [nchunks][M][C][K], bias partials
// [nchunks][M] (floats), then Bt [C][KMp] (bf16) at a 16-byte boundary.
size_t bt_offset_bytes(const Geom& g, int nchunks) {
  return (((size_t)nchunks * g.M * g.c_in * g.K + (size_t)nchunks * g.M) * sizeof(float) + 15) / 16 * 16;
}

size_t k4cl_part_bytes(const Geom& g) {
  const int sms = sm_count4();
  const WeightShape w = weight_shape(g, sms > 0 ? sms : 152);
  return bt_offset_bytes(g, w.nchunks) + (size_t)g.c_in * km_padded(g) * 2;
}

cudaError_t launch_k4cl_input(const K4ClArgs& in, cudaStream_t s) {
  const Geom& g = in.g;
  const int cpc = g.c_in >= 128 ? 128 : 64;
  K4InArgs a{};
  a.g = g;
  a.goff = in.goff;
  const int sms = sm_count4();
  if (sms <= 0) return cudaErrorInvalidDevice;
  a.bt = reinterpret_cast<const unsigned short*>(reinterpret_cast<const char*>(in.part) +
                                                 bt_offset_bytes(g, weight_shape(g, sms).nchunks));
  a.gx_nhwc = in.gx_nhwc;
  a.x = static_cast<const unsigned short*>(in.x);
  a.grad_x = in.grad_x;
  a.tiles_x = (int)ceil_div_ll(g.w, kTX);
  a.cpc = cpc;
  const int tiles_y = (int)ceil_div_ll(g.h, kTY);
  const size_t smem = input_smem(g, cpc);
  CUtensorMap gmap;
  memset(&gmap, 0, sizeof(gmap));
  if (in_goff_tma(g)) {
    const unsigned long long dims[4] = {(unsigned long long)g.wo, (unsigned long long)g.ho,
                                        (unsigned long long)g.M, (unsigned long long)g.n};
    const unsigned long long strides[3] = {(unsigned long long)g.wo * 4, (unsigned long long)g.howo * 4,
                                           (unsigned long long)g.M * g.howo * 4};
    const unsigned int box[4] = {(unsigned)in_gxp(g), (unsigned)in_gy(g), (unsigned)g.M, 1u};
    if (!make_tmap_f32(&gmap, in.goff, 4, dims, strides, box)) return cudaErrorInvalidValue;
  }
  const void* func = cpc == 128 ? (const void*)k4cl_input<128> : (const void*)k4cl_input<64>;
  cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  void* args[] = {&gmap, &a};
  return launch_pdl4(func, dim3((unsigned)(a.tiles_x * tiles_y), (unsigned)(g.c_in / cpc), (unsigned)g.n),
                     dim3(kInThreads), smem, s, args);
}

cudaError_t launch_k4cl_weight(const K4ClArgs& in, cudaStream_t s) {
  const Geom& g = in.g;
  const int sms = sm_count4();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const WeightShape w = weight_shape(g, sms);
  CUtensorMap xmap;
  const unsigned long long dims[4] = {(unsigned long long)g.c_in, (unsigned long long)g.w,
                                      (unsigned long long)g.h, (unsigned long long)g.n};
  const unsigned long long strides[3] = {(unsigned long long)g.c_in * 2,
                                         (unsigned long long)g.w * g.c_in * 2,
                                         (unsigned long long)g.hw * g.c_in * 2};
  const unsigned int box[4] = {64u, (unsigned)w.cols, (unsigned)w.rows, 1u};
  if (!make_tmap_bf16(&xmap, in.xc, 4, dims, strides, box, true)) return cudaErrorInvalidValue;
  K4WArgs a{};
  a.g = g;
  a.goff = in.goff;
  a.part = in.part;
  a.bpart = in.part + (size_t)w.nchunks * g.M * g.c_in * g.K;
  a.w_off = static_cast<const unsigned short*>(in.w_off);
  a.bt = reinterpret_cast<unsigned short*>(reinterpret_cast<char*>(in.part) + bt_offset_bytes(g, w.nchunks));
  a.tiles_x = w.tiles_x;
  a.tiles_y = w.tiles_y;
  a.tiles = w.tiles;
  a.nchunks = w.nchunks;
  a.rows = w.rows;
  a.cols = w.cols;
  a.win_pitch = w.win_pitch;
  const size_t smem = weight_smem(w.win_pitch);
  cudaError_t e = cudaFuncSetAttribute((const void*)k4cl_weight,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  void* args[] = {&xmap, &a};
  return launch_pdl4((const void*)k4cl_weight, dim3((unsigned)w.slices, (unsigned)w.nchunks),
                     dim3((unsigned)(64 * g.K)), smem, s, args);
}

cudaError_t launch_k4cl_reduce(const K4ClArgs& in, cudaStream_t s) {
  const Geom& g = in.g;
  const int sms = sm_count4();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const WeightShape w = weight_shape(g, sms);
  const float* part = in.part;
  const float* bpart = in.part + (size_t)w.nchunks * g.M * g.c_in * g.K;
  float* gw = in.grad_w_off;
  float* gb = in.grad_b_off;
  int count = g.M * g.c_in * g.K, M = g.M, nch = w.nchunks;
  const float* gwp = in.gw_perm;
  float* gwd = in.grad_w;
  int wcount = in.c_out * g.c_in * g.K, C = g.c_in, K = g.K;
  void* args[] = {&part, &bpart, &gw, &gb, &count, &M, &nch, &gwp, &gwd, &wcount, &C, &K};
  // blocks [0, count / 256): the chunk sums; then, with gw_perm, one block per
  // (output channel, kPermCh input channels) for the permutation
  const long long nperm = gwp ? (long long)in.c_out * ceil_div_ll(g.c_in, kPermCh) : 0;
  return launch_pdl4((const void*)k4cl_reduce, dim3((unsigned)(ceil_div_ll(count, 256) + nperm)), dim3(256), 0,
                     s, args);
}

// This file's share of dc_device_error.
unsigned int k4cl_read_error(int clear) {
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_k4cl_error, sizeof(v)) != cudaSuccess) return 2u;
  if (clear && v) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_k4cl_error, &zero, sizeof(zero)) != cudaSuccess) return 2u;
  }
  return v;
}

}  // namespace dc
