// Main-convolution GEMMs of float32 problems on the 5th-generation tensor
// cores, by the three-product TF32 split.
//
// Explainer page "DefT: Boosting Scalability of Deformable Convolution
// Operations on GPUs", "The argument in one glance / This paper's idea": the
// main convolution over the deformed map is a dense GEMM.  For float32
// problems it is computed here as
//   a * b  ~=  a_hi * b_hi + a_hi * b_lo + a_lo * b_hi,
// with a_hi = a with its low 13 mantissa bits cleared (a TF32 number) and
// a_lo = a - a_hi (exact in float32) with its low 13 bits cleared as well,
// the split of the "3xTF32" error-compensated tensor-core method.  Each of
// the three products is exact in the tensor core's float32 accumulation up to
// its own rounding; the dropped a_lo * b_lo term and the truncation of the lo
// parts are below 2^-21 relative to |a b|, so the result carries about the
// accuracy of a float32 dot product.
//
// With the plane-major column layout col[kdim][image][pixel]:
//   FWD   y[b][o][q]    = sum_r   w[o][r]  * col[r][b][q]     A = w   (K-major in memory)
//                                                              B = col (MN-major in memory)
//   GCOL  gcol[r][b][q] = sum_o   w[o][r]  * gy[b][o][q]      A = w^T (MN-major)
//                                                              B = gy  (MN-major)
//   GW    gw[o][r]     += sum_b,q gy[b][o][q] * col[r][b][q]  A = gy  (K-major)
//                                                              B = col (K-major)
// TMA brings each k-block of 32 float32 values per row into a "raw" ring of
// shared-memory stages in the tensor's own orientation.  Four converter warps
// split every raw tile into hi and lo tiles, always K-major with the 128-byte
// swizzle (transposing the MN-major ones on the way), in a second ring that
// the MMA thread reads: 12 tcgen05.mma.kind::tf32 per k-block (4 k-steps of
// 8, three products each) into one of two tensor-memory accumulators.
// Warp roles: 0-3 epilogue (one TMEM lane quarter each), 4 TMA producer,
// 5 MMA issuer, 6-9 converters.  The launch is persistent: one CTA per SM,
// each taking output tiles blockIdx.x, + gridDim.x, ...  Every mbarrier wait
// is bounded; on expiry the kernel raises this file's device error flag,
// drains what it issued, frees its tensor memory and returns.
#include <cuda.h>

#include "dc_common.cuh"
#include "dc_tma.cuh"

namespace dc {
namespace {

__device__ unsigned int g_tf32_error;

constexpr int kBM = 128;            // output rows per tile (tensor-memory lanes)
constexpr int kBK = 32;             // k per block: one 128-byte row of float32
constexpr int kThreads = 320;       // ten warps
constexpr int kConvWarp0 = 6;       // first converter warp
constexpr uint32_t kTf32Mask = 0xffffe000u;  // sign, exponent and 10 mantissa bits

enum Kind { FWD = 0, GCOL = 1, GW = 2 };

struct Tf32Args {
  int c_out, kdim, howo, nimg;
  int kb_total;       // k-blocks of the whole reduction
  int kb_per_split;   // GW: k-blocks per tile along the split index
  int qblocks;        // GW: k-blocks per image (ceil(howo / 32))
  float* out;
  long long out_row, out_img;  // GCOL: gcol pitches (elements)
  ZeroArgs zero;               // GCOL: buffers the rest of the backward accumulates into
  int vgx, vgy, vgz;           // tile grid: x column tiles, y row tiles, z images or splits
  int relu;                    // FWD: y = max(y, 0) in the epilogue (NaN kept)
};

template <int KIND, int BN>
struct Cfg {
  static constexpr int kARaw = kBM * 128;  // 128 rows x 32 float32
  static constexpr int kBRaw = BN * 128;
  static constexpr int kRaw = kARaw + kBRaw;
  static constexpr int kSplit = 2 * kRaw;  // A hi, A lo, B hi, B lo
  static constexpr int kR = BN == 64 ? 3 : 2;  // raw stages
  static constexpr int kS = 2;                 // split stages
  static constexpr int kTmemCols = 2 * BN;     // two accumulators
  static constexpr size_t kSmem = 1024 + (size_t)kR * kRaw + (size_t)kS * kSplit + 256;
  static constexpr bool kAMn = KIND == GCOL;  // raw A tile is MN-major
  static constexpr bool kBMn = KIND != GW;    // raw B tile is MN-major
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return px::smem_u32(p); }

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity) {
  return px::mbar_wait(bar, parity, &g_tf32_error);
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void tma_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0,
                                       int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ void tma_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0,
                                       int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory descriptor of a K-major operand with the 128-byte swizzle:
// 8-row atoms of 1024 bytes (stride 1024), the leading offset unused.
__device__ __forceinline__ uint64_t kdesc(uint32_t addr) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::tf32: TF32 A and B (both K-major), fp32 D,
// M = 128, N = bn.
__host__ __device__ constexpr uint32_t idesc_tf32(int bn) {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(bn >> 3) << 17) |
         ((uint32_t)(kBM >> 4) << 24);
}

__device__ __forceinline__ void umma_tf32(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// hi = x with the low 13 mantissa bits cleared; lo = (x - hi), likewise
// truncated.  x - hi is exact: both share x's exponent range.
__device__ __forceinline__ void split_tf32(uint32_t x, uint32_t& hi, uint32_t& lo) {
  hi = x & kTf32Mask;
  lo = __float_as_uint(__uint_as_float(x) - __uint_as_float(hi)) & kTf32Mask;
}

// A raw tile already K-major (rows of 32 k, 128-byte swizzle): the hi and lo
// tiles keep every element at its byte offset.  ct = converter thread 0..127.
__device__ __forceinline__ void split_same(const unsigned char* src, unsigned char* hi,
                                           unsigned char* lo, int bytes, int ct) {
  for (int v = ct; v < bytes / 16; v += 128) {
    const uint4 x = *reinterpret_cast<const uint4*>(src + v * 16);
    uint4 h, l;
    split_tf32(x.x, h.x, l.x);
    split_tf32(x.y, h.y, l.y);
    split_tf32(x.z, h.z, l.z);
    split_tf32(x.w, h.w, l.w);
    *reinterpret_cast<uint4*>(hi + v * 16) = h;
    *reinterpret_cast<uint4*>(lo + v * 16) = l;
  }
}

// A raw tile MN-major: chunks of 32 MN values x 32 k-rows (4096 bytes, one
// 128-byte swizzled row per k).  Element (mn, k) goes to row mn, column k of
// the K-major hi and lo tiles.  Work unit u = (chunk u / 2, pieces 4 (u & 1)
// .. + 3 of every row); lane = k.  For a fixed piece and element the 32 lanes
// write the 32 words of one 128-byte row: no bank conflicts.
__device__ __forceinline__ void split_transpose(const unsigned char* src, unsigned char* hi,
                                                unsigned char* lo, int nchunks, int cw, int lane) {
  const int k = lane;
  for (int u = cw; u < 2 * nchunks; u += 4) {
    const int c = u >> 1;
    const unsigned char* row = src + c * 4096 + k * 128;
#pragma unroll
    for (int pp = 0; pp < 4; ++pp) {
      const int p = (u & 1) * 4 + pp;
      const uint4 x = *reinterpret_cast<const uint4*>(row + ((p ^ (k & 7)) << 4));
      const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int n = c * 32 + p * 4 + e;
        const int off = n * 128 + (((k >> 2) ^ (n & 7)) << 4) + (k & 3) * 4;
        uint32_t h, l;
        split_tf32(xs[e], h, l);
        *reinterpret_cast<uint32_t*>(hi + off) = h;
        *reinterpret_cast<uint32_t*>(lo + off) = l;
      }
    }
  }
}

// Row of 32 fp32 results at dst (columns n_first ..), clipped at `limit`.
__device__ __forceinline__ void store_row(float* dst, const uint32_t* r, int n_first, int limit) {
  if (n_first + 32 <= limit) {
#pragma unroll
    for (int v = 0; v < 8; ++v)
      *reinterpret_cast<float4*>(dst + v * 4) =
          make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                      __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (n_first + j < limit) dst[j] = __uint_as_float(r[j]);
  }
}

template <int KIND, int BN>
__global__ void __launch_bounds__(kThreads, 1)
    tf32_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
              Tf32Args a) {
  using C = Cfg<KIND, BN>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = px::align1024(smem_raw);
  unsigned char* raw0 = smem;                      // raw ring (TMA -> converters)
  unsigned char* spl0 = smem + C::kR * C::kRaw;    // split ring (converters -> MMA)
  uint64_t* rfull = reinterpret_cast<uint64_t*>(spl0 + C::kS * C::kSplit);
  uint64_t* rempty = rfull + C::kR;
  uint64_t* sfull = rempty + C::kR;
  uint64_t* sempty = sfull + C::kS;
  uint64_t* tfull = sempty + C::kS;  // accumulator b complete (MMA -> epilogue)
  uint64_t* tempty = tfull + 2;      // accumulator b drained (epilogue -> MMA)
  uint64_t* drain = tempty + 2;      // MMA completion on the way out
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntiles = (a.vgx * a.vgy * a.vgz - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
  struct Tile {
    int m0, n0, z, kb_begin, nkb;
  };
  auto tile = [&](int j) {
    Tile T;
    const int t = (int)blockIdx.x + j * (int)gridDim.x;
    const int bx = t % a.vgx;
    const int r = t / a.vgx;
    T.m0 = (r % a.vgy) * kBM;
    T.z = r / a.vgy;
    T.n0 = bx * BN;
    int kb_begin = 0, kb_end = a.kb_total;
    if (KIND == GW) {
      kb_begin = T.z * a.kb_per_split;
      kb_end = min(a.kb_total, kb_begin + a.kb_per_split);
    }
    T.kb_begin = kb_begin;
    T.nkb = kb_end > kb_begin ? kb_end - kb_begin : 0;
    return T;
  };
  bool ok = true;

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_holder)),
                 "r"((uint32_t)C::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (threadIdx.x == 32) {
    for (int s = 0; s < C::kR; ++s) {
      px::mbar_init(&rfull[s], 1);
      px::mbar_init(&rempty[s], 4);  // one arrival per converter warp
    }
    for (int s = 0; s < C::kS; ++s) {
      px::mbar_init(&sfull[s], 4);
      px::mbar_init(&sempty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      px::mbar_init(&tfull[b], 1);
      px::mbar_init(&tempty[b], 4);  // one arrival per epilogue warp
    }
    px::mbar_init(drain, 1);
    px::fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  pdl_wait();  // the operands (and GCOL's zeroed buffers) belong to earlier launches

  if (warp == 4) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      int it = 0;  // k-blocks issued so far, over all tiles
      for (int j = 0; j < ntiles && ok; ++j) {
        const Tile T = tile(j);
        for (int i = 0; i < T.nkb; ++i, ++it) {
          const int s = it % C::kR;
          if (it >= C::kR && !wait_bar(&rempty[s], ((it / C::kR) - 1) & 1)) {
            ok = false;
            break;
          }
          unsigned char* ra = raw0 + s * C::kRaw;
          unsigned char* rb = ra + C::kARaw;
          px::mbar_expect_tx(&rfull[s], C::kRaw);
          const int kb = T.kb_begin + i;
          if (KIND == FWD) {
            // A: w {kdim, c_out}, box {32, 128}; B: col {pixel, image, row}, boxes {32, 1, 32}
            tma_2d(ra, &tmA, &rfull[s], kb * kBK, T.m0);
#pragma unroll
            for (int h = 0; h < BN / 32; ++h) tma_3d(rb + h * 4096, &tmB, &rfull[s], T.n0 + 32 * h, T.z, kb * kBK);
          } else if (KIND == GCOL) {
            // A: w {kdim, c_out}, boxes {32, 32}; B: gy {pixel, channel, image}, boxes {32, 32, 1}
#pragma unroll
            for (int h = 0; h < kBM / 32; ++h) tma_2d(ra + h * 4096, &tmA, &rfull[s], T.m0 + 32 * h, kb * kBK);
#pragma unroll
            for (int h = 0; h < BN / 32; ++h) tma_3d(rb + h * 4096, &tmB, &rfull[s], T.n0 + 32 * h, kb * kBK, T.z);
          } else {
            // A: gy {pixel, channel, image}, box {32, 128, 1}; B: col {pixel, image, row}, box {32, 1, BN}
            const int img = kb / a.qblocks, q0 = (kb - img * a.qblocks) * kBK;
            tma_3d(ra, &tmA, &rfull[s], q0, T.m0, img);
            tma_3d(rb, &tmB, &rfull[s], q0, img, T.n0);
          }
        }
      }
      // on the way out: the last loads issued have landed (bounded; on the
      // normal path they were consumed long ago)
      for (int d = 1; d <= C::kR && d <= it; ++d) {
        const int i2 = it - d;
        wait_bar(&rfull[i2 % C::kR], (i2 / C::kR) & 1);
      }
    }
  } else if (warp == 5) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t idesc = idesc_tf32(BN);
      int it = 0;
      bool issued = false;
      for (int j = 0; j < ntiles && ok; ++j) {
        const Tile T = tile(j);
        const int b = j & 1;
        if (j >= 2 && !wait_bar(&tempty[b], ((j >> 1) - 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t acc = tmem + (uint32_t)b * BN;
        for (int i = 0; i < T.nkb; ++i, ++it) {
          const int s = it % C::kS;
          if (!wait_bar(&sfull[s], (it / C::kS) & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t ahi = smem_u32(spl0 + s * C::kSplit);
          const uint32_t alo = ahi + C::kARaw;
          const uint32_t bhi = ahi + 2 * C::kARaw;
          const uint32_t blo = bhi + C::kBRaw;
#pragma unroll
          for (int kk = 0; kk < kBK / 8; ++kk) {
            // 8 float32 of k = 32 bytes along the swizzled row
            const uint32_t o = kk * 32;
            umma_tf32(acc, kdesc(ahi + o), kdesc(bhi + o), idesc, (i > 0 || kk > 0) ? 1u : 0u);
            umma_tf32(acc, kdesc(ahi + o), kdesc(blo + o), idesc, 1u);
            umma_tf32(acc, kdesc(alo + o), kdesc(bhi + o), idesc, 1u);
          }
          issued = true;
          umma_commit(&sempty[s]);
        }
        if (!ok) break;
        umma_commit(&tfull[b]);  // arrives once the tile's MMAs are complete
      }
      if (issued) {
        // every MMA issued is complete before tensor memory is freed
        umma_commit(drain);
        wait_bar(drain, 0);
      }
    }
  } else if (warp >= kConvWarp0) {
    // -------------------------------------------------------------- converters
    const int cw = warp - kConvWarp0, ct = cw * 32 + lane;
    int it = 0;
    for (int j = 0; j < ntiles && ok; ++j) {
      const Tile T = tile(j);
      for (int i = 0; i < T.nkb; ++i, ++it) {
        const int rs = it % C::kR, ss = it % C::kS;
        bool w = wait_bar(&rfull[rs], (it / C::kR) & 1);
        w = w && (it < C::kS || wait_bar(&sempty[ss], ((it / C::kS) - 1) & 1));
        if (!__all_sync(0xffffffffu, w)) {
          ok = false;
          break;
        }
        const unsigned char* ra = raw0 + rs * C::kRaw;
        const unsigned char* rb = ra + C::kARaw;
        unsigned char* ahi = spl0 + ss * C::kSplit;
        unsigned char* alo = ahi + C::kARaw;
        unsigned char* bhi = ahi + 2 * C::kARaw;
        unsigned char* blo = bhi + C::kBRaw;
        if (C::kAMn)
          split_transpose(ra, ahi, alo, kBM / 32, cw, lane);
        else
          split_same(ra, ahi, alo, C::kARaw, ct);
        if (C::kBMn)
          split_transpose(rb, bhi, blo, BN / 32, cw, lane);
        else
          split_same(rb, bhi, blo, C::kBRaw, ct);
        // the generic-proxy writes are visible to the tensor core's reads
        px::fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&rempty[rs]);
          mbar_arrive(&sfull[ss]);
        }
      }
    }
  } else {
    // -------------------------------------------------------------- epilogue (warps 0-3)
    if (KIND == GCOL) zero_share(a.zero, blockIdx.x, gridDim.x, threadIdx.x, 128);
    const int row = warp * 32 + lane;
    for (int j = 0; j < ntiles; ++j) {
      const Tile T = tile(j);
      const int b = j & 1;
      ok = ok && __all_sync(0xffffffffu, wait_bar(&tfull[b], (j >> 1) & 1));
      if (!ok) break;
      tc_fence_after();
      const int m = T.m0 + row;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tmem + (uint32_t)b * BN + (uint32_t)(c * 32) + ((uint32_t)(warp * 32) << 16), r);
        if (T.nkb == 0) continue;
        const int n_first = T.n0 + c * 32;
        if (KIND == FWD) {
          if (a.relu) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float v = __uint_as_float(r[j]);
              if (!(v > 0.f) && v == v) r[j] = 0u;
            }
          }
          if (m < a.c_out) store_row(a.out + ((long long)T.z * a.c_out + m) * a.howo + n_first, r, n_first, a.howo);
        } else if (KIND == GCOL) {
          if (m < a.kdim) store_row(a.out + m * a.out_row + T.z * a.out_img + n_first, r, n_first, a.howo);
        } else {
          if (m >= a.c_out) continue;
          float* dst = a.out + (long long)m * a.kdim + n_first;
          if (n_first + 32 <= a.kdim) {
#pragma unroll
            for (int v = 0; v < 8; ++v)
              atomicAdd(reinterpret_cast<float4*>(dst + v * 4),
                        make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                    __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3])));
          } else {
#pragma unroll
            for (int jj = 0; jj < 32; ++jj)
              if (n_first + jj < a.kdim) atomicAdd(dst + jj, __uint_as_float(r[jj]));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[b]);
    }
  }
  pdl_release();
  tc_fence_before();
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"((uint32_t)C::kTmemCols)
                 : "memory");
}

// ---------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// float32 tensor map, 128-byte swizzle, zero fill outside the tensor.
bool map_f32(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
             const cuuint64_t* strides, const cuuint32_t* box) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, (cuuint32_t)rank, const_cast<void*>(base), dims,
            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// main weights {kdim, c_out}
bool w_map(CUtensorMap* m, const void* w, const Geom& g, cuuint32_t box0, cuuint32_t box1) {
  const cuuint64_t dims[2] = {(cuuint64_t)g.kdim, (cuuint64_t)g.c_out};
  const cuuint64_t strides[1] = {(cuuint64_t)g.kdim * 4};
  const cuuint32_t box[2] = {box0, box1};
  return map_f32(m, w, 2, dims, strides, box);
}

// plane-major map {pixel (true extent), image, row}
bool col_map(CUtensorMap* m, const void* col, const Geom& g, const ColLayout& L, cuuint32_t box_rows) {
  const cuuint64_t dims[3] = {(cuuint64_t)g.howo, (cuuint64_t)g.n, (cuuint64_t)g.kdim};
  const cuuint64_t strides[2] = {(cuuint64_t)L.img * 4, (cuuint64_t)L.row * 4};
  const cuuint32_t box[3] = {32, 1, box_rows};
  return map_f32(m, col, 3, dims, strides, box);
}

// grad_y {pixel, channel, image}
bool gy_map(CUtensorMap* m, const void* gy, const Geom& g, cuuint32_t box_ch) {
  const cuuint64_t dims[3] = {(cuuint64_t)g.howo, (cuuint64_t)g.c_out, (cuuint64_t)g.n};
  const cuuint64_t strides[2] = {(cuuint64_t)g.howo * 4, (cuuint64_t)g.c_out * g.howo * 4};
  const cuuint32_t box[3] = {32, box_ch, 1};
  return map_f32(m, gy, 3, dims, strides, box);
}

int sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return 152;
  return sms;
}

// Persistent launch over the tile grid (gx, gy, gz): one CTA per SM at most.
template <int KIND, int BN>
cudaError_t launch(const CUtensorMap& A, const CUtensorMap& B, Tf32Args a, long long gx, long long gy,
                   long long gz, cudaStream_t s) {
  using C = Cfg<KIND, BN>;
  auto k = tf32_gemm<KIND, BN>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem);
  if (e != cudaSuccess) return e;
  const long long tiles = gx * gy * gz;
  if (tiles <= 0 || tiles > INT_MAX) return cudaErrorInvalidValue;
  a.vgx = (int)gx;
  a.vgy = (int)gy;
  a.vgz = (int)gz;
  const long long sms = sm_count();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(tiles < sms ? tiles : sms));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, k, A, B, a);
  note_launches(1);
  return e;
}

Tf32Args base_args(const Geom& g) {
  Tf32Args a{};
  a.c_out = g.c_out;
  a.kdim = g.kdim;
  a.howo = (int)g.howo;
  a.nimg = g.n;
  return a;
}

}  // namespace

// Every tensor map needs 16-byte aligned rows: kdim and the pixel count are
// multiples of four.
bool tf32_gemm_supported(const Geom& g) {
  return g.kdim % 4 == 0 && g.howo % 4 == 0 && g.howo < INT_MAX && encode_fn() != nullptr;
}

cudaError_t launch_gemm_fwd_tf32(const GemmArgs& ga, cudaStream_t s) {
  const Geom& g = ga.g;
  CUtensorMap A, B;
  if (!w_map(&A, ga.w, g, 32, 128)) return cudaErrorInvalidValue;
  if (!col_map(&B, ga.col, g, ga.col_layout, 32)) return cudaErrorInvalidValue;
  Tf32Args a = base_args(g);
  a.kb_total = (int)ceil_div_ll(g.kdim, kBK);
  a.out = static_cast<float*>(ga.y);
  a.relu = g.relu;
  return launch<FWD, 64>(A, B, a, ceil_div_ll(g.howo, 64), ceil_div_ll(g.c_out, kBM), g.n, s);
}

cudaError_t launch_gemm_gcol_tf32(const GemmArgs& ga, cudaStream_t s) {
  const Geom& g = ga.g;
  CUtensorMap A, B;
  if (!w_map(&A, ga.w, g, 32, 32)) return cudaErrorInvalidValue;
  if (!gy_map(&B, ga.gy, g, 32)) return cudaErrorInvalidValue;
  Tf32Args a = base_args(g);
  a.kb_total = (int)ceil_div_ll(g.c_out, kBK);
  a.out = static_cast<float*>(ga.gcol);
  a.out_row = ga.gcol_layout.row;
  a.out_img = ga.gcol_layout.img;
  a.zero = ga.zero;
  return launch<GCOL, 128>(A, B, a, ceil_div_ll(g.howo, 128), ceil_div_ll(g.kdim, kBM), g.n, s);
}

cudaError_t launch_gemm_gw_tf32(const GemmArgs& ga, cudaStream_t s) {
  const Geom& g = ga.g;
  CUtensorMap A, B;
  if (!gy_map(&A, ga.gy, g, 128)) return cudaErrorInvalidValue;
  if (!col_map(&B, ga.col, g, ga.col_layout, 128)) return cudaErrorInvalidValue;
  Tf32Args a = base_args(g);
  a.qblocks = (int)ceil_div_ll(g.howo, kBK);
  a.kb_total = a.qblocks * g.n;
  a.out = ga.gw;
  const long long tiles = ceil_div_ll(g.kdim, 128) * ceil_div_ll(g.c_out, kBM);
  // about one tile per SM: more splits only add float4 atomics on grad_W
  long long splits = ceil_div_ll(sm_count(), tiles);
  if (splits > a.kb_total) splits = a.kb_total;
  if (splits < 1) splits = 1;
  a.kb_per_split = (int)ceil_div_ll(a.kb_total, splits);
  splits = ceil_div_ll(a.kb_total, a.kb_per_split);
  return launch<GW, 128>(A, B, a, ceil_div_ll(g.kdim, 128), ceil_div_ll(g.c_out, kBM), splits, s);
}

// This file's share of dc_device_error (2 = unreadable).
unsigned int tf32_read_error(int clear) {
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_tf32_error, sizeof(v)) != cudaSuccess) return 2u;
  if (clear && v) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_tf32_error, &zero, sizeof(zero)) != cudaSuccess) return 2u;
  }
  return v;
}

}  // namespace dc
