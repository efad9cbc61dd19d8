// K4 on tensor cores: backward of the offset convolution ("Following a
// deformable layer through DefT", Step 1 of 5, on the explainer page "DefT:
// Boosting Scalability of Deformable Convolution Operations on GPUs") for bf16
// problems with at most kMaxM offset channels.  With goff the completed
// gradient of the offset convolution's output (summed over all channels by K3)
// and one CTA per (band of output rows, slice of 16 input channels):
//
//   weight part  gw_off[m][c][k] += sum_px X[c,k][px] * goff[m][px]
//                X[c,k][px] = x[c] at the window position tap k of pixel px reads
//                (M = 16 channels of one tap, N = offset channels, K = pixels)
//   input part   grad_x[c][q]   += sum_(k,m) w_off[m][c][k] * goff[m][px(q,k)]
//                px(q,k) = the band pixel whose tap k reads window position q
//                (M = 16 channels, N = window positions, K = (tap, offset channel))
//   bias         gb_off[m]      += sum_px goff[m][px]   (slice 0 only)
//
// Both parts are dense mma.sync m16n8k16 contractions (bf16 operands, fp32
// accumulation).  The input part is written as a gather over window positions
// (the im2col of goff), so every grad_x element of the window is produced once
// in registers and added to global memory by one atomic (an 8-byte atomic for
// two adjacent elements when image rows have even length): there is no shared
// grad_x window and no shared-memory atomic.  The weight part's partial sums go
// to a per-image copy laid out in the accumulators' own order (one 16-byte
// atomic per lane and tile), summed over images after K4.  Every fragment
// register is one 32-bit shared load: goff is packed twice (pixel pairs
// [m][px/2], offset-channel pairs [px][m/2]), w_off^T as [(k,c)][m/2], and the
// input window as pixel-pair words (x[q], x[q + stride]) so that the two
// pixels a register holds are one word whenever they lie in the same band row.
#include "dc_band.cuh"

namespace dc {
namespace {

using band::kThreads;
constexpr int kCpc = kGwoSlice;  // channels per CTA: one mma row tile
constexpr int kMaxM = 80;
constexpr int kWarps = kThreads / 32;
constexpr int kMChunk = 5;  // offset-channel n-tiles per pass of the weight part
constexpr int kQGroup = 4;  // window-position n-tiles per unit of the input part

struct TcPlan {
  int R, TW, tiles_w, tiles_h, npx, nslices;
  int rows, cols, npos, nq;  // window (receptive field + 1 column, even), positions, rounded to 8
  int xplane;                // words per channel plane of the pair-packed window
  int pxp, mp8, mp16;        // pixels to 16, offset channels to 8 and 16
  int sa, sb, sw;            // word strides of ga [m][px/2], gb [px][m/2], wa [(k,c)][m/2]
  size_t off_xp, off_ga, off_gb, off_wa, off_pair, off_gpos, smem;
};

__host__ TcPlan make_tc_plan(const Geom& g, int px) {
  const band::Shape sh = band::make_shape(g, 0, px);
  TcPlan p{};
  p.R = sh.R;
  p.TW = sh.TW;
  p.npx = sh.npx;
  p.tiles_w = sh.tiles_w;
  p.tiles_h = sh.tiles_h;
  p.nslices = (g.c_in + kCpc - 1) / kCpc;
  p.rows = sh.rows;
  // one more column, rounded to even: the window starts at an even image
  // column, so the two window positions of an accumulator pair are two
  // adjacent, 8-byte aligned grad_x elements
  p.cols = (sh.cols + 2) & ~1;
  p.npos = p.rows * p.cols;
  p.nq = (p.npos + 7) / 8 * 8;
  p.xplane = band::pad_plane(p.npos);
  p.pxp = (p.npx + 15) / 16 * 16;
  p.mp8 = (g.M + 7) / 8 * 8;
  p.mp16 = (g.M + 15) / 16 * 16;
  p.sa = p.pxp / 2 + 4;
  p.sb = p.mp16 / 2 + 4;
  p.sw = p.mp16 / 2 + 4;
  size_t at = 0;
  p.off_xp = at;
  at += (size_t)kCpc * p.xplane * 4;
  p.off_ga = at;
  at += (size_t)p.mp8 * p.sa * 4;
  p.off_gb = at;
  at += (size_t)(p.pxp + 1) * p.sb * 4;  // last row: zeros (positions no pixel reaches)
  p.off_wa = at;
  at += (size_t)g.K * kCpc * p.sw * 4;
  p.off_pair = at;
  at += (size_t)(p.pxp / 2) * 8;
  p.off_gpos = at;
  at += (size_t)p.pxp * 4;
  p.smem = at;
  return p;
}

// The largest tile (up to 256 pixels) that fits two CTAs per SM and still
// gives the grid at least two CTAs per SM of the GPU's 152: larger tiles stage
// less halo and add fewer grad_w_off partials, but a grid below two CTAs per
// SM leaves K4's tail, which runs after the sampling backward, on few SMs
// (measured: res3 103.8 us per step with 448 CTAs of 112 pixels against
// 107.3 us with 256 CTAs of 196 pixels; the 56 x 56 stack layer 667 ->
// 639 us with 224- instead of 112-pixel tiles).  Problems too small for that
// take the smallest tile that fits (the most CTAs).
__host__ TcPlan pick_tc_plan(const Geom& g) {
  constexpr int kMinGrid = 2 * 152;
  TcPlan fallback{};
  bool have = false;
  for (int px = 2 * band::kBandPx; px >= 32; px /= 2) {
    const TcPlan p = make_tc_plan(g, px);
    if (p.smem > 110 * 1024) continue;
    if ((long long)p.nslices * p.tiles_w * p.tiles_h * g.n >= kMinGrid) return p;
    fallback = p;
    have = true;
  }
  return have ? fallback : make_tc_plan(g, 32);
}

__device__ __forceinline__ void mma16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// Four 8x8 b16 matrices from shared memory; lane l gives the 16-byte row
// (l & 7) of matrix l >> 3.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// The two input values of a pixel pair (2j, 2j+1) at tap offset `tap` as one
// bf16-pair register.  e.x / e.y: window positions of the two pixels (-1 for
// a padding pixel).  When the pair lies in one band row the word at e.x
// already holds both (its high half is the value one column stride further).
__device__ __forceinline__ uint32_t x_pair(const uint32_t* plane, int2 e, int tap, int sw) {
  if (e.x < 0) return 0u;
  uint32_t w = plane[e.x + tap];
  if (e.y < 0) return w & 0xffffu;
  if (e.y != e.x + sw) w = (w & 0xffffu) | (plane[e.y + tap] << 16);
  return w;
}

__global__ void __launch_bounds__(kThreads, 3) k4_offconv_bwd_tc(OffconvBwdArgs a, TcPlan pl) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int s_next_unit;  // work units handed out after each warp's first
  const Geom g = a.g;
  const __nv_bfloat16* __restrict__ x = static_cast<const __nv_bfloat16*>(a.x);
  const unsigned short* __restrict__ w_off = static_cast<const unsigned short*>(a.w_off);
  const int slice = (int)(blockIdx.x % pl.nslices);
  const int tw_idx = (int)(blockIdx.x / pl.nslices);
  const int ho0 = blockIdx.y * pl.R, wo0 = tw_idx * pl.TW;
  const int n = blockIdx.z;
  const int c_begin = slice * kCpc;
  const int ncur = min(g.c_in, c_begin + kCpc) - c_begin;
  const int ylo = ho0 * g.sh - g.ph;
  // window column 0 is image column xlo (even); the receptive field starts xs later
  const int xs = (wo0 * g.sw - g.pw) & 1, xlo = wo0 * g.sw - g.pw - xs;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int M = g.M, K = g.K;
  const long long img = (long long)n * g.c_in * g.hw;
  // grad_w_off partial sums: this image's copy in accumulator order (reduced
  // after K4) when given, else grad_w_off itself
  const bool gwo_frag = a.gw_off_img != nullptr;
  float* gwo = gwo_frag ? a.gw_off_img + (long long)n * gwo_frag_count(M, g.c_in, K) : a.gw_off;

  uint32_t* xp = reinterpret_cast<uint32_t*>(smem + pl.off_xp);      // [kCpc][xplane]
  uint32_t* ga = reinterpret_cast<uint32_t*>(smem + pl.off_ga);      // [mp8][sa]
  uint32_t* gb = reinterpret_cast<uint32_t*>(smem + pl.off_gb);      // [pxp + 1][sb]
  uint32_t* wa = reinterpret_cast<uint32_t*>(smem + pl.off_wa);      // [K * kCpc][sw]
  int2* pair = reinterpret_cast<int2*>(smem + pl.off_pair);          // [pxp / 2]
  int* gpos = reinterpret_cast<int*>(smem + pl.off_gpos);          // [pxp]

  // ---------------------------------------------------------------- prologue (inputs only)
  // pixel-pair table: window positions of pixels 2j and 2j+1
  for (int j = tid; j < pl.pxp / 2; j += kThreads) {
    int2 e = make_int2(-1, -1);
    const int p = 2 * j;
    if (p < pl.npx) {
      const int r = p / pl.TW, c = p - r * pl.TW;
      e.x = r * g.sh * pl.cols + c * g.sw + xs;
      if (p + 1 < pl.npx) {
        const int r1 = (p + 1) / pl.TW, c1 = p + 1 - r1 * pl.TW;
        e.y = r1 * g.sh * pl.cols + c1 * g.sw + xs;
      }
    }
    pair[j] = e;
  }
  // pixel -> offset within one goff plane (-1: padding or outside the output)
  for (int px = tid; px < pl.pxp; px += kThreads) {
    int v = -1;
    if (px < pl.npx) {
      const int r = px / pl.TW;
      const int ho = ho0 + r, wo = wo0 + px - r * pl.TW;
      if (ho < g.ho && wo < g.wo) v = ho * g.wo + wo;
    }
    gpos[px] = v;
  }
  if (tid == 0) s_next_unit = 0;
  // gb's last row stays zero: window positions that no pixel's tap reaches
  for (int j = tid; j < pl.mp16 / 2; j += kThreads) gb[pl.pxp * pl.sb + j] = 0u;
  // input window of the slice as pixel-pair words (x[q], x[q + column stride]),
  // zero outside the image and beyond c_in.  Unit stride with image rows of
  // whole 8-byte quads: a task reads the 4-pixel quad and the next one (for
  // the fifth value) and writes up to four words.
  const bool xquad = g.sw == 1 && (g.w & 3) == 0 && (reinterpret_cast<uintptr_t>(x) & 7) == 0;
  if (xquad) {
    const int q_lo = (xlo >= 0 ? xlo : xlo - 3) / 4;
    const int q_hi = (xlo + pl.cols - 1 >= 0 ? xlo + pl.cols - 1 : xlo + pl.cols - 4) / 4;
    const int nqd = q_hi - q_lo + 1;
    band::Walk3 w;
    w.init(tid, kThreads, pl.rows, nqd);
    while (w.a < kCpc) {
      const int cl = w.a, r = w.b, x0 = 4 * (q_lo + w.c);
      w.next();
      const int c = c_begin + cl, yy = ylo + r;
      uint2 cur = make_uint2(0u, 0u);
      uint32_t nxt = 0u;
      if (c < g.c_in && yy >= 0 && yy < g.h) {
        const __nv_bfloat16* row = x + img + (long long)c * g.hw + (long long)yy * g.w;
        if (x0 >= 0 && x0 < g.w) cur = *reinterpret_cast<const uint2*>(row + x0);
        if (x0 + 4 >= 0 && x0 + 4 < g.w) nxt = *reinterpret_cast<const uint32_t*>(row + x0 + 4);
      }
      const uint32_t wv[4] = {cur.x, __byte_perm(cur.x, cur.y, 0x5432), cur.y,
                              __byte_perm(cur.y, nxt, 0x5432)};
      uint32_t* dst = xp + cl * pl.xplane + r * pl.cols;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int q = x0 + i - xlo;
        if (q >= 0 && q < pl.cols) dst[q] = wv[i];
      }
    }
  } else {
    constexpr int kB = 8;
    const int total = kCpc * pl.npos;
    band::Walk3 w;
    w.init(tid, kThreads, pl.rows, pl.cols);
    for (int base = tid; base < total; base += kThreads * kB) {
      uint32_t v[kB];
      int at[kB];
#pragma unroll
      for (int u = 0; u < kB; ++u) {
        v[u] = 0u;
        at[u] = -1;
        if (w.a < kCpc) {
          at[u] = w.a * pl.xplane + w.b * pl.cols + w.c;
          const int c = c_begin + w.a, yy = ylo + w.b, xx = xlo + w.c;
          if (c < g.c_in && yy >= 0 && yy < g.h) {
            const __nv_bfloat16* row = x + img + (long long)c * g.hw + (long long)yy * g.w;
            if (xx >= 0 && xx < g.w) v[u] = band::bf16_bits(row + xx);
            if (xx + g.sw >= 0 && xx + g.sw < g.w) v[u] |= band::bf16_bits(row + xx + g.sw) << 16;
          }
          w.next();
        }
      }
#pragma unroll
      for (int u = 0; u < kB; ++u)
        if (at[u] >= 0) xp[at[u]] = v[u];
    }
  }
  // w_off^T as [(k, c)][offset-channel pair] words, zero for m >= M or c >= c_in.
  // A full slice with aligned rows reads each offset channel's contiguous run
  // w_off[m][c_begin ..][*] as uint4 and scatters the halves.
  const bool wvec = c_begin + kCpc <= g.c_in && ((g.c_in * K) & 7) == 0 &&
                    (reinterpret_cast<uintptr_t>(w_off) & 15) == 0;
  if (wvec) {
    for (int idx = tid; idx < K * kCpc * pl.sw; idx += kThreads) wa[idx] = 0u;
    __syncthreads();
    unsigned short* wh = reinterpret_cast<unsigned short*>(wa);
    const int span8 = kCpc * K / 8, total = M * span8;
    for (int idx = tid; idx < total; idx += kThreads) {
      const int m = idx / span8, q = idx - m * span8;
      const uint4 v = *reinterpret_cast<const uint4*>(w_off + ((long long)m * g.c_in + c_begin) * K + 8 * q);
      const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
      int cl = (8 * q) / K, k = 8 * q - cl * K;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        wh[((k * kCpc + cl) * pl.sw) * 2 + m] =
            (unsigned short)((e & 1) ? (vw[e >> 1] >> 16) : (vw[e >> 1] & 0xffffu));
        if (++k == K) {
          k = 0;
          ++cl;
        }
      }
    }
  } else {
    constexpr int kB = 4;
    const int wpr = pl.mp16 / 2;  // words per row
    const int total = K * kCpc * wpr;
    const long long mstride = (long long)g.c_in * K;
    band::Walk2 w;
    w.init(tid, kThreads, wpr);
    for (int base = tid; base < total; base += kThreads * kB) {
      unsigned short lo[kB], hi[kB];
      int at[kB];
#pragma unroll
      for (int u = 0; u < kB; ++u) {
        lo[u] = hi[u] = 0;
        at[u] = -1;
        if (w.a < K * kCpc) {
          const int row = w.a, j = w.b;
          const int k = row / kCpc, cl = row - k * kCpc;
          at[u] = row * pl.sw + j;
          if (cl < ncur) {
            const long long o = (long long)(c_begin + cl) * K + k;
            if (2 * j < M) lo[u] = w_off[(2 * j) * mstride + o];
            if (2 * j + 1 < M) hi[u] = w_off[(2 * j + 1) * mstride + o];
          }
          w.next();
        }
      }
#pragma unroll
      for (int u = 0; u < kB; ++u)
        if (at[u] >= 0) wa[at[u]] = (uint32_t)lo[u] | ((uint32_t)hi[u] << 16);
    }
  }
  // the offset gradient is K3's output; grad_x / grad_w_off / grad_b_off were
  // cleared by the GCOL GEMM before K3 started
  pdl_wait();
  pdl_release();

  __syncthreads();  // gpos

  // ---------------------------------------------------------------- the band's offset gradient
  // packed straight from global memory: ga [m][pixel pair] (zero rows m >= M)
  // and gb [pixel][offset-channel pair]; eight loads in flight per thread
  {
    const float* gsrc = a.goff + (long long)n * M * g.howo;
    const int wa_ = pl.pxp / 2, wb_ = pl.mp16 / 2;
    const int nga = pl.mp8 * wa_, total = nga + pl.pxp * wb_;
    auto gv = [&](int m, int px) {
      const int o = gpos[px];
      return (m < M && o >= 0) ? gsrc[(long long)m * g.howo + o] : 0.f;
    };
    // pixel quads read as float4; a warp covers 8 offset-channel pairs x 4
    // pixel quads (conflicts on the packed stores stay two-way).  Full-width
    // band with 16-byte aligned rows: the band's pixels are one contiguous run
    // of each goff plane.  Tile rows of whole quads (TW and Wo multiples of 4):
    // a quad is four pixels of one tile row, all inside or all outside the
    // output.
    const int nvalid = (min(ho0 + pl.R, g.ho) - ho0) * g.wo;
    const bool aligned = (reinterpret_cast<uintptr_t>(a.goff) & 15) == 0;
    const bool run = pl.TW == g.wo && (g.howo & 3) == 0 && ((ho0 * g.wo) & 3) == 0 &&
                     (nvalid & 3) == 0 && aligned;
    const bool quads = !run && (pl.TW & 3) == 0 && (g.wo & 3) == 0 && aligned;
    const bool vec = run || quads;
    // goff plane offset of the tile's pixel quad p4, -1 outside the output
    auto quad_at = [&](int p4) -> int {
      if (run) return 4 * p4 < nvalid ? ho0 * g.wo + 4 * p4 : -1;
      const int r = (4 * p4) / pl.TW, c = 4 * p4 - r * pl.TW;
      return (4 * p4 < pl.npx && ho0 + r < g.ho && wo0 + c < g.wo) ? (ho0 + r) * g.wo + wo0 + c : -1;
    };
    if (vec) {
      const int pblocks = pl.pxp / 16, nblk = (pl.mp16 / 16) * pblocks;
      for (int blk0 = warp; blk0 < nblk; blk0 += 2 * kWarps) {
        float4 f[2][2];
        int jj[2], pq[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int blk = blk0 + u * kWarps;
          const int jb = blk / pblocks, pb = blk - jb * pblocks;
          jj[u] = jb * 8 + (lane >> 2);
          pq[u] = pb * 4 + (lane & 3);
          f[u][0] = f[u][1] = make_float4(0.f, 0.f, 0.f, 0.f);
          const int o = blk < nblk ? quad_at(pq[u]) : -1;
          if (o >= 0) {
            if (2 * jj[u] < M)
              f[u][0] = *reinterpret_cast<const float4*>(gsrc + (long long)(2 * jj[u]) * g.howo + o);
            if (2 * jj[u] + 1 < M)
              f[u][1] = *reinterpret_cast<const float4*>(gsrc + (long long)(2 * jj[u] + 1) * g.howo + o);
          }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          if (blk0 + u * kWarps >= nblk) break;
          const int j = jj[u], p4 = pq[u];
          const float4 f0 = f[u][0], f1 = f[u][1];
          if (2 * j < pl.mp8) {
            ga[(2 * j) * pl.sa + 2 * p4] = pack2(f0.x, f0.y);
            ga[(2 * j) * pl.sa + 2 * p4 + 1] = pack2(f0.z, f0.w);
          }
          if (2 * j + 1 < pl.mp8) {
            ga[(2 * j + 1) * pl.sa + 2 * p4] = pack2(f1.x, f1.y);
            ga[(2 * j + 1) * pl.sa + 2 * p4 + 1] = pack2(f1.z, f1.w);
          }
          uint32_t* gq = gb + (4 * p4) * pl.sb + j;
          gq[0] = pack2(f0.x, f1.x);
          gq[pl.sb] = pack2(f0.y, f1.y);
          gq[2 * pl.sb] = pack2(f0.z, f1.z);
          gq[3 * pl.sb] = pack2(f0.w, f1.w);
        }
      }
    }
    constexpr int kB = 4;
    for (int base = vec ? total : tid; base < total; base += kThreads * kB) {
      float lo[kB], hi[kB];
      int at[kB];
#pragma unroll
      for (int u = 0; u < kB; ++u) {
        const int idx = base + u * kThreads;
        at[u] = -1;
        lo[u] = hi[u] = 0.f;
        if (idx < nga) {
          const int m = idx / wa_, j = idx - m * wa_;
          at[u] = m * pl.sa + j;
          lo[u] = gv(m, 2 * j);
          hi[u] = gv(m, 2 * j + 1);
        } else if (idx < total) {
          const int r = idx - nga;
          const int px = r / wb_, j = r - px * wb_;
          at[u] = (1 << 30) | (px * pl.sb + j);
          lo[u] = gv(2 * j, px);
          hi[u] = gv(2 * j + 1, px);
        }
      }
#pragma unroll
      for (int u = 0; u < kB; ++u) {
        if (at[u] < 0) continue;
        if (at[u] & (1 << 30))
          gb[at[u] & ((1 << 30) - 1)] = pack2(lo[u], hi[u]);
        else
          ga[at[u]] = pack2(lo[u], hi[u]);
      }
    }
    if (a.gb_off && slice == 0) {
      // bias gradient in fp32: one warp per offset channel
      for (int m = warp; m < M; m += kWarps) {
        float s = 0.f;
        for (int px = lane; px < pl.npx; px += 32) s += gv(m, px);
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) atomicAdd(a.gb_off + m, s);
      }
    }
  }
  __syncthreads();

  // ---------------------------------------------------------------- both contractions
  // work units: the input part in groups of kQGroup position tiles (the
  // larger units, first) and K weight-part units (one tap each); each warp
  // takes its first unit by index and every further one from a shared
  // counter, so warps that drew small units take more of them
  const int qtiles = pl.nq / 8;
  const bool unit_stride = g.sh == 1 && g.sw == 1;
  const int qunits = (qtiles + kQGroup - 1) / kQGroup;
  const int mtiles8 = pl.mp8 / 8;
  const int ksteps = pl.pxp / 16;
  // the pixels 2j, 2j + 1 of every pair share a band row (and are one column
  // stride apart) when the tile is one row or an even number of columns wide
  const bool pairs_in_row = pl.R == 1 || (pl.TW & 1) == 0;
  // grad_x element pairs are 8-byte aligned when image rows have even length
  const bool gx_pairs = (g.w & 1) == 0 && (reinterpret_cast<uintptr_t>(a.gx) & 7) == 0;
  auto next_seq = [&]() {
    int v = 0;
    if (lane == 0) v = atomicAdd(&s_next_unit, 1);
    return __shfl_sync(0xffffffffu, v, 0) + kWarps;
  };
  for (int seq = warp; seq < K + qunits; seq = next_seq()) {
    const int unit = seq < qunits ? K + seq : seq - qunits;
    if (unit < K) {
      // ---- weight part, tap k: rows = 16 channels, columns = offset channels
      const int k = unit;
      const int i = k / g.kw;
      const int tap = i * g.dh * pl.cols + (k - i * g.kw) * g.dw;
      const uint32_t* p0 = xp + gid * pl.xplane;
      const uint32_t* p1 = xp + (gid + 8) * pl.xplane;
      for (int mt0 = 0; mt0 < mtiles8; mt0 += kMChunk) {
        float acc[kMChunk][4];
#pragma unroll
        for (int t = 0; t < kMChunk; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
        // k-steps whose 16 pixels all exist and whose pairs never straddle
        // a band row read each fragment register with one plain load
        const int ks_full = pairs_in_row ? pl.npx / 16 : 0;
        for (int ks = 0; ks < ks_full; ++ks) {
          const int x0 = pair[ks * 8 + tig].x + tap, x1 = pair[ks * 8 + tig + 4].x + tap;
          const uint32_t a0 = p0[x0], a1 = p1[x0], a2 = p0[x1], a3 = p1[x1];
#pragma unroll
          for (int t = 0; t < kMChunk; ++t) {
            if (mt0 + t >= mtiles8) break;
            const uint32_t* b = ga + ((mt0 + t) * 8 + gid) * pl.sa + ks * 8 + tig;
            mma16816(acc[t], a0, a1, a2, a3, b[0], b[4]);
          }
        }
        for (int ks = ks_full; ks < ksteps; ++ks) {
          const int2 e0 = pair[ks * 8 + tig], e1 = pair[ks * 8 + tig + 4];
          const uint32_t a0 = x_pair(p0, e0, tap, g.sw), a1 = x_pair(p1, e0, tap, g.sw);
          const uint32_t a2 = x_pair(p0, e1, tap, g.sw), a3 = x_pair(p1, e1, tap, g.sw);
#pragma unroll
          for (int t = 0; t < kMChunk; ++t) {
            if (mt0 + t >= mtiles8) break;
            const uint32_t* b = ga + ((mt0 + t) * 8 + gid) * pl.sa + ks * 8 + tig;
            mma16816(acc[t], a0, a1, a2, a3, b[0], b[4]);
          }
        }
#pragma unroll
        for (int t = 0; t < kMChunk; ++t) {
          if (mt0 + t >= mtiles8) break;
          if (gwo_frag) {
            // the accumulator tile as one 16-byte atomic per lane (lanes whose
            // four elements are all padding hold zeros and skip it)
            if (gid < ncur && (mt0 + t) * 8 + 2 * tig < M)
              atomicAdd(reinterpret_cast<float4*>(gwo + ((long long)(slice * K + k) * mtiles8 + mt0 + t) * 128 +
                                                  lane * 4),
                        make_float4(acc[t][0], acc[t][1], acc[t][2], acc[t][3]));
            continue;
          }
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const int cl = gid + (h >> 1) * 8;
            const int m = (mt0 + t) * 8 + 2 * tig + (h & 1);
            if (cl < ncur && m < M)
              atomicAdd(gwo + ((long long)m * g.c_in + c_begin + cl) * K + k, acc[t][h]);
          }
        }
      }
    } else {
      // ---- input part: rows = 16 channels, columns = window positions,
      // reduction over (tap, offset channel); the pixel each position reads
      // through tap k is found on the fly.  Fragments come from ldmatrix: one
      // x4 load gives the A fragment, another the B fragments of two position
      // tiles (each lane addresses one 16-byte row: lane & 7 picks the row,
      // lane >> 3 the matrix).  Two accumulator chains (even and odd
      // offset-channel blocks) halve the dependent mma sequence.
      const int nt0 = (unit - K) * kQGroup;
      // this lane's ldmatrix row of the B matrices: position tile 2 * tp + (lane >> 4)
      int lqr[kQGroup / 2], lqc[kQGroup / 2];
#pragma unroll
      for (int tp = 0; tp < kQGroup / 2; ++tp) {
        const int q = (nt0 + 2 * tp + (lane >> 4)) * 8 + (lane & 7);
        lqr[tp] = -(1 << 20);  // no pixel
        lqc[tp] = 0;
        if (q < pl.npos) {
          lqr[tp] = q / pl.cols;
          lqc[tp] = q - lqr[tp] * pl.cols - xs;
        }
      }
      const uint32_t gb_lane = smem_addr(gb) + ((lane >> 3) & 1) * 16;
      const uint32_t wa_lane =
          smem_addr(wa) + ((lane & 7) + ((lane >> 3) & 1) * 8) * pl.sw * 4 + (lane >> 4) * 16;
      const int nmc = pl.mp16 / 16;
      float acc[2][kQGroup][4];
#pragma unroll
      for (int s = 0; s < 2; ++s)
#pragma unroll
        for (int t = 0; t < kQGroup; ++t) acc[s][t][0] = acc[s][t][1] = acc[s][t][2] = acc[s][t][3] = 0.f;
      for (int i = 0, k = 0; i < g.kh; ++i) {
        for (int j = 0; j < g.kw; ++j, ++k) {
          uint32_t brow[kQGroup / 2];
#pragma unroll
          for (int tp = 0; tp < kQGroup / 2; ++tp) {
            const int r = lqr[tp] - i * g.dh, c = lqc[tp] - j * g.dw;
            int px = pl.pxp;
            if (unit_stride) {
              if (r >= 0 && r < pl.R && c >= 0 && c < pl.TW) px = r * pl.TW + c;
            } else if (r >= 0 && c >= 0 && r % g.sh == 0 && c % g.sw == 0 && r / g.sh < pl.R &&
                       c / g.sw < pl.TW) {
              px = (r / g.sh) * pl.TW + c / g.sw;
            }
            brow[tp] = gb_lane + px * pl.sb * 4;
          }
          const uint32_t arow = wa_lane + k * kCpc * pl.sw * 4;
#pragma unroll
          for (int mc = 0; mc < kMaxM / 16; ++mc) {
            if (mc >= nmc) break;
            uint32_t a0, a1, a2, a3;
            ldsm_x4(arow + mc * 32, a0, a1, a2, a3);
#pragma unroll
            for (int tp = 0; tp < kQGroup / 2; ++tp) {
              uint32_t b0, b1, b2, b3;
              ldsm_x4(brow[tp] + mc * 32, b0, b1, b2, b3);
              mma16816(acc[mc & 1][2 * tp], a0, a1, a2, a3, b0, b1);
              mma16816(acc[mc & 1][2 * tp + 1], a0, a1, a2, a3, b2, b3);
            }
          }
        }
      }
#pragma unroll
      for (int t = 0; t < kQGroup; ++t)
#pragma unroll
        for (int h = 0; h < 4; ++h) acc[0][t][h] += acc[1][t][h];
#pragma unroll
      for (int t = 0; t < kQGroup; ++t) {
        if (nt0 + t >= qtiles) break;
        // window positions q0 = 8 * tile + 2 * tig and q0 + 1 of accumulator
        // columns 2 * tig, 2 * tig + 1: one window row (cols and npos are even)
        const int q0 = (nt0 + t) * 8 + 2 * tig;
        if (q0 >= pl.npos) continue;
        const int qrow = q0 / pl.cols, qcol = q0 - qrow * pl.cols;
        const int yy = ylo + qrow, xx = xlo + qcol;
        if (yy < 0 || yy >= g.h) continue;
        float* dst = a.gx + img + (long long)c_begin * g.hw + (long long)yy * g.w + xx;
        if (gx_pairs) {
          // xx is even and the image width even: both columns lie in the image
          // or both outside; one 8-byte atomic per channel
          if (xx < 0 || xx >= g.w) continue;
          if (gid < ncur && (acc[0][t][0] != 0.f || acc[0][t][1] != 0.f))
            atomicAdd(reinterpret_cast<float2*>(dst + (long long)gid * g.hw),
                      make_float2(acc[0][t][0], acc[0][t][1]));
          if (gid + 8 < ncur && (acc[0][t][2] != 0.f || acc[0][t][3] != 0.f))
            atomicAdd(reinterpret_cast<float2*>(dst + (long long)(gid + 8) * g.hw),
                      make_float2(acc[0][t][2], acc[0][t][3]));
          continue;
        }
#pragma unroll
        for (int hc = 0; hc < 2; ++hc) {
          if (xx + hc < 0 || xx + hc >= g.w) continue;
          if (gid < ncur && acc[0][t][hc] != 0.f) atomicAdd(dst + hc + (long long)gid * g.hw, acc[0][t][hc]);
          if (gid + 8 < ncur && acc[0][t][2 + hc] != 0.f)
            atomicAdd(dst + hc + (long long)(gid + 8) * g.hw, acc[0][t][2 + hc]);
        }
      }
    }
  }
}

// grad_w_off = sum over images of the per-image partials (in K4's accumulator
// order): one thread per float4 of that order, eight images' loads in flight,
// each element stored to its place in grad_w_off
__global__ void __launch_bounds__(kThreads) gw_off_reduce(const float* __restrict__ img_part,
                                                          float* __restrict__ gw_off, int nimg,
                                                          long long count, int M, int c_in, int K) {
  pdl_wait();  // the partials are complete once K4 (and the GEMM after it) finished
  const long long c4 = count / 4;
  const float4* src = reinterpret_cast<const float4*>(img_part);
  for (long long e = blockIdx.x * (long long)kThreads + threadIdx.x; e < c4;
       e += (long long)gridDim.x * kThreads) {
    float s[4] = {0.f, 0.f, 0.f, 0.f};
    int n = 0;
    for (; n + 8 <= nimg; n += 8) {
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = src[(long long)(n + u) * c4 + e];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        s[0] += v[u].x;
        s[1] += v[u].y;
        s[2] += v[u].z;
        s[3] += v[u].w;
      }
    }
    for (; n < nimg; ++n) {
      const float4 v = src[(long long)n * c4 + e];
      s[0] += v.x;
      s[1] += v.y;
      s[2] += v.z;
      s[3] += v.w;
    }
    long long d[4];
    gwo_frag_dest4((int)e, M, c_in, K, d);
#pragma unroll
    for (int h = 0; h < 4; ++h)
      if (d[h] >= 0) gw_off[d[h]] = s[h];
  }
}

}  // namespace

cudaError_t launch_gw_off_reduce(const OffconvBwdArgs& a, cudaStream_t s) {
  const long long count = gwo_frag_count(a.g.M, a.g.c_in, a.g.K);
  long long blocks = (count / 4 + kThreads - 1) / kThreads;
  if (blocks > 152 * 4) blocks = 152 * 4;
  if (blocks < 1) blocks = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, gw_off_reduce, (const float*)a.gw_off_img, a.gw_off,
                                     a.g.n, count, a.g.M, a.g.c_in, a.g.K);
  note_launches(1);
  return e;
}

bool offconv_bwd_tc_supported(const Geom& g, dc_dtype dt) { return dt == DC_BF16 && g.M <= kMaxM; }

size_t offconv_bwd_tc_smem_bytes(const Geom& g) { return pick_tc_plan(g).smem; }

cudaError_t launch_offconv_bwd_tc(const OffconvBwdArgs& a, cudaStream_t s) {
  const TcPlan pl = pick_tc_plan(a.g);
  cudaError_t e = cudaFuncSetAttribute(k4_offconv_bwd_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)pl.smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(pl.nslices * pl.tiles_w), (unsigned)pl.tiles_h, (unsigned)a.g.n);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, k4_offconv_bwd_tc, a, pl);
  note_launches(1);
  return e;
}

}  // namespace dc
