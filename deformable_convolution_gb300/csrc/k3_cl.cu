// K3, channels-last: backward of the bilinear sampling step.
//
// Derivatives of the layer of the explainer page "DefT: Boosting Scalability
// of Deformable Convolution Operations on GPUs" ("The argument in one glance":
// offset convolution -> four-neighbour bilinear blend -> main convolution),
// given gcol, the gradient of the deformed map:
//   grad_x at corner j of sample s    += w_j(s) * gcol[s]           (per channel)
//   grad_offset (dy, dx) of sample s   = sum_j (wy_j, wx_j) * D_j(s),
//     D_j(s) = sum_c gcol[s][c] * x[corner j of s][c]
// with (wy) = (-(1-lx), -lx, 1-lx, lx) and (wx) = (-(1-ly), 1-ly, -ly, ly)
// for corners (00, 01, 10, 11): the derivatives of the blend with respect to
// the sampling coordinate, the lower corner being floor(p) (right-sided at
// integer coordinates).
//
// GB300 mapping, one offset group, channels-last.  The kernel is persistent
// and warp-specialised, tiles of TH x TW output pixels, the C_in channels
// split over `csplit` independent CTAs per tile.  Per tile, TMA brings two
// boxes into shared memory (double-buffered): x's window from the NHWC copy
// (the window of the fused forward stage, 128-byte swizzle) and the tile's
// slice of gcol, which is pixel-major (gcol[n][pixel][tap][channel], written
// by the tensor-core GEMM), so the tile's samples are one 5-D box.
//   P warps (4)  per tile: the sampling taps from the given offsets and every
//                (sample, corner) pair that lands in the window and in the
//                image, bucketed by window position (counts and ranks from
//                shared-memory atomics, a scan, a scatter); D_j(s) = 0 for
//                the corners outside the image;
//   S warps (12) per tile: lanes in groups of cpc / 16 (sixteen channels
//                each, two 8-channel pieces half a slice apart; eight
//                channels for 64-channel slices); the bucketed pairs are
//                split evenly over the groups and walked in batches of 4
//                (8): per pair, the sample's gcol
//                slice from shared memory, w * gcol accumulated in registers
//                (packed fp32 FMAs) for the current position (added to a
//                float32 NHWC buffer with vector float atomics when the
//                position changes) and the lanes' partial dot products with x
//                at that position, which one transposing butterfly per batch
//                sums over the group (D_j(s)); then per sample its offset
//                gradient from its four
//                D_j, added with float atomics (the CTAs of a tile each hold
//                a slice of the channels).  Samples whose corners leave the
//                window read x from global memory and add their corners'
//                gradients directly.
// The order of the pairs within a position follows the atomics, so grad_x is
// summed in a run-dependent order (as it is anyway across tiles, whose
// windows overlap).  A separate kernel writes grad_x (NCHW) from the NHWC
// buffer.  All waits are bounded mbarrier waits.
#include <limits.h>

#include "dc_band.cuh"
#include "dc_tma.cuh"

namespace dc {

// Raised by this file's bounded waits (read by dc_device_error).
__device__ unsigned int g_cl3_error;

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kPWarps = 4;
constexpr int kSWarps = kWarps - kPWarps;
constexpr int kPThreads = kPWarps * 32;
constexpr int kSThreads = kSWarps * 32;
constexpr int kMaxIPT = 4;  // samples per P thread and tile
constexpr size_t kSmemBudget = 225 * 1024;
constexpr int kRefMargin = 3;

struct K3Plan {
  int TH, TW, tiles_h, tiles_w, tiles;
  int rows, cols, npos;     // staged window; its positions
  int csplit, cpc, chunks;  // CTAs per tile (independent), channels per CTA, 64-channel chunks
  int npx, items;           // pixels per tile; samples per tile (npx * K)
  uint32_t win_bytes, gc_bytes, chunk_pitch;
  size_t off_stage, off_gc, off_tap, off_syx, off_ent, off_pst, off_cnt, off_pix, off_itab, off_otab,
      off_D, off_slow, off_oin, off_bar, smem;
  int grid;
};

__host__ K3Plan k3_plan_for(const Geom& g, int margin, int TH, int TW, int csplit, int sms) {
  K3Plan p{};
  p.TH = TH;
  p.TW = TW;
  p.npx = TH * TW;
  p.items = p.npx * g.K;
  p.tiles_h = (int)ceil_div_ll(g.ho, TH);
  p.tiles_w = (int)ceil_div_ll(g.wo, TW);
  p.tiles = g.n * p.tiles_h * p.tiles_w;
  p.rows = (TH - 1) * g.sh + (g.kh - 1) * g.dh + 1 + 2 * margin;
  p.cols = (TW - 1) * g.sw + (g.kw - 1) * g.dw + 1 + 2 * margin;
  p.npos = p.rows * p.cols;
  p.csplit = csplit;
  p.cpc = g.c_in / csplit;
  p.chunks = p.cpc / 64;
  p.chunk_pitch = ((uint32_t)p.rows * p.cols * 128u + 1023u) / 1024u * 1024u;
  p.win_bytes = (uint32_t)p.chunks * p.rows * p.cols * 128u;
  p.gc_bytes = (uint32_t)p.items * p.cpc * 2u;
  size_t at = 0;
  p.off_stage = at;  // two window buffers
  at += 2 * (size_t)p.chunks * p.chunk_pitch;
  p.off_gc = at;  // two gcol buffers [items][cpc]
  at += 2 * (((size_t)p.gc_bytes + 1023) / 1024 * 1024);
  p.off_tap = at;  // [2][items] int4 {ly, lx, -, kind}
  at += 2 * (size_t)p.items * 16;
  p.off_syx = at;  // [2][items] int2 {y0, x0} of the upper-left corner
  at += 2 * (size_t)p.items * 8;
  p.off_ent = at;  // [2][items * 4] int2 {item * 4 + corner | position << 16, w}, by position
  at += 2 * (size_t)p.items * 4 * 8;
  p.off_pst = at;  // [2][npos + 1] bucket starts
  at += 2 * (size_t)(p.npos + 1) * 4;
  p.off_cnt = at;  // [npos + 1] bucket counts (P only)
  at += (size_t)(p.npos + 1) * 4;
  p.off_pix = at;  // [npos] window position -> pixel offset from the window's corner, wy * W + wx
  at += (size_t)p.npos * 4;
  at = (at + 15) / 16 * 16;
  p.off_itab = at;  // [items] int4 {row, column of the tap in the window w/o margin, pixel row | col << 16, k | p << 16}
  at += (size_t)p.items * 16;
  p.off_otab = at;  // [M * npx] int2 {offset-map element from the tile's first, pixel row | col << 16}
  at += (size_t)g.M * p.npx * 8;
  p.off_D = at;  // [2][items * 4] D_j(s) (S; P writes the zeros of corners outside the image)
  at += 2 * (size_t)p.items * 4 * 4;
  p.off_slow = at;  // [2][items + 1] samples read from global memory (count first)
  at += 2 * (size_t)(p.items + 1) * 4;
  at = (at + 15) / 16 * 16;
  p.off_oin = at;  // [2][M][npx] the tile's offsets (prefetched a tile ahead)
  at += 2 * (size_t)g.M * p.npx * 4;
  at = (at + 7) / 8 * 8;
  p.off_bar = at;  // wfull[2], wempty[2], tfull[2], tempty[2]
  at += 8 * 8;
  p.smem = at + 1024;
  const int slots = sms / csplit * csplit;
  const int ctas = p.tiles * csplit;
  p.grid = ctas < slots ? ctas : slots;
  return p;
}

__host__ bool k3_fits(const K3Plan& p) {
  return p.smem <= kSmemBudget && p.rows <= 256 && p.cols <= 256 && p.items <= kPThreads * kMaxIPT &&
         p.npos < 65536 && p.items * 4 < 65536;
}

__host__ K3Plan k3_best(const Geom& g, int margin, int sms) {
  // cost per CTA-tile: per (sample, corner) pair a fixed part and the
  // channel work, per window position the x load and the gradient's atomics
  static const int cand[][2] = {{2, 8}, {4, 8}, {2, 16}, {8, 8}, {4, 16}};
  K3Plan best{};
  double best_cost = 0.0;
  for (int csplit = 1; csplit <= 4; csplit *= 2) {
    if (g.c_in % csplit != 0 || (g.c_in / csplit) % 64 != 0) continue;
    for (const auto& c : cand) {
      const K3Plan p = k3_plan_for(g, margin, c[0], c[1], csplit, sms);
      if (!k3_fits(p)) continue;
      const double per_tile = (double)p.items * 4 * (24.0 + p.cpc / 8.0) + (double)p.npos * p.cpc / 16.0;
      const double cost = (double)ceil_div_ll((long long)p.tiles * csplit, p.grid) * per_tile;
      if (best.npx == 0 || cost < best_cost) {
        best = p;
        best_cost = cost;
      }
    }
  }
  return best;
}

__host__ K3Plan k3_make_plan(const Geom& g, int margin, int sms) {
  const K3Plan ref = k3_best(g, kRefMargin, sms);
  if (ref.npx != 0) {
    const K3Plan p = k3_plan_for(g, margin, ref.TH, ref.TW, ref.csplit, sms);
    if (k3_fits(p)) return p;
  }
  return k3_best(g, margin, sms);
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ uint32_t line_off(uint32_t pos) { return (pos << 7) | ((pos & 7u) << 4); }

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(px::smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void p_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kPThreads) : "memory"); }
__device__ __forceinline__ bool p_sync_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, 1, %2, p;\n"
      " selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(kPThreads)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void s_sync() { asm volatile("bar.sync 2, %0;" ::"n"(kSThreads) : "memory"); }

// CPL consecutive bf16 channels (4, 8 or 16 bytes) as floats
template <int CPL>
__device__ __forceinline__ void unpack_bf(const uint32_t* w, float* f) {
#pragma unroll
  for (int i = 0; i < CPL / 2; ++i) {
    f[2 * i] = bf_lo(w[i]);
    f[2 * i + 1] = bf_hi(w[i]);
  }
}

template <int CPL>
__device__ __forceinline__ void ldg_bf(const __nv_bfloat16* p, float* f) {
  uint32_t w[CPL / 2];
  if constexpr (CPL == 8) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
    w[0] = v.x;
    w[1] = v.y;
    w[2] = v.z;
    w[3] = v.w;
  } else if constexpr (CPL == 4) {
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
    w[0] = v.x;
    w[1] = v.y;
  } else {
    w[0] = __ldg(reinterpret_cast<const unsigned int*>(p));
  }
  unpack_bf<CPL>(w, f);
}

// the raw words of CPL consecutive bf16 channels in shared memory (plain
// loads: the compiler may schedule them freely between the barriers)
template <int CPL>
__device__ __forceinline__ void lds_words(const unsigned char* p, uint32_t* w) {
  if constexpr (CPL == 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    w[0] = v.x;
    w[1] = v.y;
    w[2] = v.z;
    w[3] = v.w;
  } else if constexpr (CPL == 4) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    w[0] = v.x;
    w[1] = v.y;
  } else {
    w[0] = *reinterpret_cast<const uint32_t*>(p);
  }
}

// One butterfly step of a transposing warp reduction: lanes with bit `o` set
// keep the upper half of v[0 .. 2H-1] and add their partner's copy of it,
// the others the lower half.
template <int H>
__device__ __forceinline__ void xstep(float* v, int lane, int o) {
  const bool upper = (lane & o) != 0;
#pragma unroll
  for (int i = 0; i < H; ++i) {
    const float send = upper ? v[i] : v[i + H];
    const float keep = upper ? v[i + H] : v[i];
    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
  }
}

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{.reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2,%3};\n mov.b64 rb, {%4,%5};\n"
      " mov.b64 rc, {%6,%7};\n fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0,%1}, rd;}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

__device__ __forceinline__ float2 bf2(uint32_t w) { return make_float2(bf_lo(w), bf_hi(w)); }

// Sums each of NBV (a power of two, at most L) per-lane values over a group
// of L consecutive lanes: lane l of the group returns the total of
// v[l >> log2(L / NBV)].
template <int NBV, int L>
__device__ __forceinline__ float group_sum_t(float* v, int lane) {
  if constexpr (NBV >= 8) xstep<NBV / 2>(v, lane, L / 2);
  if constexpr (NBV >= 4) xstep<(NBV >= 8 ? NBV / 4 : NBV / 2)>(v, lane, NBV >= 8 ? L / 4 : L / 2);
  if constexpr (NBV >= 2) xstep<1>(v, lane, L / NBV);
  float r = v[0];
#pragma unroll
  for (int o = L / (2 * NBV); o >= 1; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
  return r;
}

// float atomics on CPL consecutive floats (vector reductions at L2); nothing
// in the kernel reads the target, so no compiler memory barrier
template <int CPL>
__device__ __forceinline__ void red_add(float* p, const float* v) {
  if constexpr (CPL >= 4) {
#pragma unroll
    for (int i = 0; i < CPL; i += 4)
      asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p + i), "f"(v[i]),
                   "f"(v[i + 1]), "f"(v[i + 2]), "f"(v[i + 3]));
  } else {
    asm volatile("red.global.add.v2.f32 [%0], {%1, %2};" ::"l"(p), "f"(v[0]), "f"(v[1]));
  }
}

struct K3Args {
  Geom g;
  const __nv_bfloat16* xc;  // x, NHWC
  const float* off;         // offsets [n][M][Ho][Wo]
  float* gx;                // grad_x accumulator, NHWC float32 (cleared beforehand)
  float* goff;              // offset gradient [n][M][Ho][Wo] (cleared beforehand)
  int margin;
};

struct TileXY {
  int n, ho0, wo0, ylo, xlo;
};

__device__ __forceinline__ TileXY tile_xy(int t, const K3Plan& pl, const Geom& g, int margin) {
  TileXY r;
  const int per_img = pl.tiles_h * pl.tiles_w;
  r.n = t / per_img;
  const int rr = t - r.n * per_img;
  const int th = rr / pl.tiles_w, tw = rr - th * pl.tiles_w;
  r.ho0 = th * pl.TH;
  r.wo0 = tw * pl.TW;
  r.ylo = r.ho0 * g.sh - g.ph - margin;
  r.xlo = r.wo0 * g.sw - g.pw - margin;
  return r;
}

__device__ __forceinline__ void tma_load_5d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0,
                                            int c1, int c2, int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%3, %4, %5, %6, %7}], [%2];" ::"r"(px::smem_u32(dst)),
      "l"(map), "r"(px::smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
      : "memory");
}

template <int CPL>
__global__ void __launch_bounds__(kThreads, 1)
    k3_cl_bwd(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap gmap,
              K3Args a, K3Plan pl) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = px::align1024(smem_raw);
  const Geom g = a.g;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int K = g.K, M = g.M, C = g.c_in;
  const uint32_t stage_pitch = (uint32_t)pl.chunks * pl.chunk_pitch;
  const uint32_t gc_pitch = (pl.gc_bytes + 1023u) / 1024u * 1024u;
  int4* tap0 = reinterpret_cast<int4*>(smem + pl.off_tap);
  int2* syx0 = reinterpret_cast<int2*>(smem + pl.off_syx);
  int2* ent0 = reinterpret_cast<int2*>(smem + pl.off_ent);
  int* pixoff = reinterpret_cast<int*>(smem + pl.off_pix);
  const int4* itab = reinterpret_cast<const int4*>(smem + pl.off_itab);
  const int2* otab = reinterpret_cast<const int2*>(smem + pl.off_otab);
  int* pst0 = reinterpret_cast<int*>(smem + pl.off_pst);
  int* cnt = reinterpret_cast<int*>(smem + pl.off_cnt);
  float* D0 = reinterpret_cast<float*>(smem + pl.off_D);
  int* slow0 = reinterpret_cast<int*>(smem + pl.off_slow);
  float* oin = reinterpret_cast<float*>(smem + pl.off_oin);
  uint64_t* wfull = reinterpret_cast<uint64_t*>(smem + pl.off_bar);
  uint64_t* wempty = wfull + 2;
  uint64_t* tfull = wfull + 4;
  uint64_t* tempty = wfull + 6;
  const int rank = (int)(blockIdx.x % pl.csplit);
  const int cbeg = rank * pl.cpc;
  const int t0 = blockIdx.x / pl.csplit, tstep = gridDim.x / pl.csplit;
  const int items = pl.items, npos = pl.npos;

  // x's window and the tile's gcol slice, completing on wfull[s]
  auto issue = [&](int t, int s) {
    const TileXY tx = tile_xy(t, pl, g, a.margin);
    px::mbar_expect_tx(&wfull[s], pl.win_bytes + pl.gc_bytes);
    unsigned char* dst = smem + pl.off_stage + (size_t)s * stage_pitch;
    for (int ch = 0; ch < pl.chunks; ++ch)
      px::tma_load_4d(dst + (size_t)ch * pl.chunk_pitch, &xmap, &wfull[s], cbeg + ch * 64, tx.xlo,
                      tx.ylo, tx.n);
    tma_load_5d(smem + pl.off_gc + (size_t)s * gc_pitch, &gmap, &wfull[s], cbeg, 0, tx.wo0, tx.ho0,
                tx.n);
  };

  if (tid == 0) {
    for (int q = 0; q < 2; ++q) {
      px::mbar_init(&wfull[q], 1);
      px::mbar_init(&wempty[q], kSWarps);
      px::mbar_init(&tfull[q], 1);
      px::mbar_init(&tempty[q], kSWarps);
    }
    px::fence_mbar_init();
  }
  // tile-independent index tables (no divisions in the per-tile loops)
  for (int q = tid; q < npos; q += kThreads) {
    const int wy = q / pl.cols;
    pixoff[q] = wy * g.w + (q - wy * pl.cols);
  }
  for (int it = tid; it < items; it += kThreads) {
    const int p = it / K, k = it - p * K;
    const int pr = p / pl.TW, pc = p - pr * pl.TW;
    const int ki = k / g.kw, kj = k - ki * g.kw;
    reinterpret_cast<int4*>(smem + pl.off_itab)[it] =
        make_int4(pr * g.sh + ki * g.dh, pc * g.sw + kj * g.dw, pr | (pc << 16), k | (p << 16));
  }
  for (int e = tid; e < M * pl.npx; e += kThreads) {
    const int m = e / pl.npx, p = e - m * pl.npx;
    const int pr = p / pl.TW, pc = p - pr * pl.TW;
    reinterpret_cast<int2*>(smem + pl.off_otab)[e] =
        make_int2((int)((long long)m * g.howo + (long long)pr * g.wo + pc), pr | (pc << 16));
  }
  __syncthreads();
  // x's NHWC copy, the offsets and gcol come from earlier kernels on the stream
  pdl_wait();

  if (warp < kPWarps) {
    // ============================================================ P warps
    int issued[2] = {0, 0};
    if (tid == 0) {
      for (int q = 0; q < 2; ++q)
        if (t0 + q * tstep < pl.tiles) {
          issue(t0 + q * tstep, q);
          ++issued[q];
        }
    }
    auto prefetch_off = [&](int t, int buf) {
      if (t >= pl.tiles) return;
      const TileXY tq = tile_xy(t, pl, g, a.margin);
      float* dsto = oin + (size_t)buf * M * pl.npx;
      const float* first = a.off + (long long)tq.n * M * g.howo + (long long)tq.ho0 * g.wo + tq.wo0;
      for (int e = tid; e < M * pl.npx; e += kPThreads) {
        const int2 ot = otab[e];
        if (tq.ho0 + (ot.y & 0xffff) < g.ho && tq.wo0 + (ot.y >> 16) < g.wo) {
          const float* src = first + ot.x;
          asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(px::smem_u32(dsto + e)), "l"(src)
                       : "memory");
        } else {
          dsto[e] = 0.f;
        }
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
    };
    prefetch_off(t0, 0);
    for (int i = 0, t = t0; t < pl.tiles; ++i, t += tstep) {
      const int s = i & 1;
      const uint32_t par = (uint32_t)(i >> 1) & 1u;
      const TileXY tx = tile_xy(t, pl, g, a.margin);
      bool ok = true;
      if (i >= 2) ok = px::mbar_wait(&tempty[s], par ^ 1u, &g_cl3_error);
      asm volatile("cp.async.wait_group 0;" ::: "memory");
      if (!p_sync_and(ok)) break;
      prefetch_off(t + tstep, s ^ 1);
      const float* offs = oin + (size_t)s * M * pl.npx;  // [M][npx]
      int4* tap = tap0 + (size_t)s * items;
      int2* syx = syx0 + (size_t)s * items;
      int2* ent = ent0 + (size_t)s * items * 4;
      int* pst = pst0 + (size_t)s * (npos + 1);
      int* slow = slow0 + (size_t)s * (items + 1);
      float* Dz = D0 + (size_t)s * items * 4;  // S's D table of this tile
      if (tid == 0) slow[0] = 0;
      for (int e = tid; e <= npos; e += kPThreads) cnt[e] = 0;
      p_sync();
      // -------------------------------------------------- taps; bucket counts and ranks
      uint32_t pr[kMaxIPT][4];  // position | rank << 16 per corner, or ~0u
#pragma unroll
      for (int u = 0; u < kMaxIPT; ++u) {
        const int it = tid + u * kPThreads;
#pragma unroll
        for (int j = 0; j < 4; ++j) pr[u][j] = ~0u;
        if (it >= items) continue;
        const int4 ie = itab[it];
        const int k = ie.w & 0xffff, p = ie.w >> 16;
        int4 tp = make_int4(0, 0, 0, 3);  // kind 3: pixel outside the output
        if (tx.ho0 + (ie.z & 0xffff) < g.ho && tx.wo0 + (ie.z >> 16) < g.wo) {
          const float by = (float)(tx.ho0 * g.sh - g.ph + ie.x);
          const float bx = (float)(tx.wo0 * g.sw - g.pw + ie.y);
          const float pyf = by + offs[(2 * k) * pl.npx + p];
          const float pxf = bx + offs[(2 * k + 1) * pl.npx + p];
          tp.w = 1;  // kind 1: no corner touches the image
          if (touches_image(pyf, pxf, g.h, g.w)) {
            const float fy = floorf(pyf), fx = floorf(pxf);
            const int y0 = (int)fy, x0 = (int)fx;
            tp.x = __float_as_int(pyf - fy);
            tp.y = __float_as_int(pxf - fx);
            syx[it] = make_int2(y0, x0);
            const int ry = y0 - tx.ylo, rx = x0 - tx.xlo;
            if (ry >= 0 && ry + 1 < pl.rows && rx >= 0 && rx + 1 < pl.cols) {
              tp.w = 0;  // kind 0: corners in the window
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const int yy = y0 + (j >> 1), xx = x0 + (j & 1);
                if (yy >= 0 && yy < g.h && xx >= 0 && xx < g.w) {
                  const int pos = (ry + (j >> 1)) * pl.cols + rx + (j & 1);
                  pr[u][j] = (uint32_t)pos | ((uint32_t)atomicAdd(&cnt[pos], 1) << 16);
                } else {
                  Dz[it * 4 + j] = 0.f;  // no pair: D_j(s) = 0 (S writes the others)
                }
              }
            } else {
              tp.w = 2;  // kind 2: corners read from global memory
              slow[1 + atomicAdd(&slow[0], 1)] = it;
            }
          }
        }
        tap[it] = tp;
      }
      p_sync();
      if (warp == 0) {
        // ------------------------------------------------ bucket starts (exclusive scan)
        int carry = 0;
        for (int b0 = 0; b0 < npos; b0 += 32) {
          const int e = b0 + lane;
          const int v = e < npos ? cnt[e] : 0;
          int inc = v;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += u;
          }
          if (e < npos) pst[e] = carry + inc - v;
          carry += __shfl_sync(0xffffffffu, inc, 31);
        }
        if (lane == 0) pst[npos] = carry;
      }
      p_sync();
      // -------------------------------------------------- scatter into the buckets
#pragma unroll
      for (int u = 0; u < kMaxIPT; ++u) {
        const int it = tid + u * kPThreads;
        if (it >= items) continue;
        const int4 tp = tap[it];
        const float ly = __int_as_float(tp.x), lx = __int_as_float(tp.y);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t v = pr[u][j];
          if (v == ~0u) continue;
          const int pos = (int)(v & 0xffffu);
          const float wy = (j >> 1) ? ly : 1.0f - ly, wx = (j & 1) ? lx : 1.0f - lx;
          ent[pst[pos] + (int)(v >> 16)] =
              make_int2((it * 4 + j) | (pos << 16), __float_as_int(__fmul_rn(wy, wx)));
        }
      }
      p_sync();
      if (tid == 0) mbar_arrive(&tfull[s]);
      // the next tile's boxes into the buffers of the tile before, once S is done with them
      const int tn = t + tstep;
      if (i >= 1 && tn < pl.tiles && tid == 0) {
        if (px::mbar_wait(&wempty[s ^ 1], (uint32_t)((i - 1) >> 1) & 1u, &g_cl3_error)) {
          issue(tn, s ^ 1);
          ++issued[s ^ 1];
        }
      }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    // no copy may be in flight when the CTA exits (the S warps wait for each
    // one, unless they gave up); a buffer's copies complete in order
    if (tid == 0) {
      for (int q = 0; q < 2; ++q)
        if (issued[q] > 0) px::mbar_wait(&wfull[q], (uint32_t)(issued[q] - 1) & 1u, &g_cl3_error);
    }
  } else {
    // ============================================================ S warps
    // lane l holds channels cbeg + l * CPL .. + CPL - 1
    const int sw = warp - kPWarps;
    const int cl = lane * CPL;

    const uint32_t row_bytes = (uint32_t)pl.cpc * 2u;
    for (int i = 0, t = t0; t < pl.tiles; ++i, t += tstep) {
      const int s = i & 1;
      const uint32_t par = (uint32_t)(i >> 1) & 1u;
      bool ok = px::mbar_wait(&tfull[s], par, &g_cl3_error);
      ok = ok && px::mbar_wait(&wfull[s], par, &g_cl3_error);
      if (!__all_sync(0xffffffffu, ok)) break;
      const TileXY tx = tile_xy(t, pl, g, a.margin);
      const int4* tap = tap0 + (size_t)s * items;
      const int2* syx = syx0 + (size_t)s * items;
      const int2* ent = ent0 + (size_t)s * items * 4;
      const int* pst = pst0 + (size_t)s * (npos + 1);
      const int* slow = slow0 + (size_t)s * (items + 1);
      float* Dt = D0 + (size_t)s * items * 4;
      const unsigned char* xsm0 = smem + pl.off_stage + (size_t)s * stage_pitch;
      const unsigned char* gsm0 = smem + pl.off_gc + (size_t)s * gc_pitch;
      const unsigned char* gsm = gsm0 + cl * 2;
      float* gximg = a.gx + (long long)tx.n * g.hw * C + cbeg + cl;
      // every D_j(s) the offset gradients read is written once this tile:
      // by the pair walk, the global path, or (corners outside the image) P
      // ---------------------------------------------- pairs, by window position
      // Lanes in groups of L = cpc / W, W channels each (16 when the slice has
      // 128 or more channels: a pair's fixed work is shared by twice the
      // channels and its two halves are independent chains).  Lane l of a
      // group holds the 8-channel pieces l * 8 + v * cpc / 2 (v < W / 8), so
      // each 16-byte load of 8 lanes covers one contiguous 128 bytes; every group
      // walks its own contiguous run of the bucketed pairs (the runs split
      // them evenly over the CTA's groups), NB pairs per batch: per pair the
      // gradient at its position accumulates in registers (added to the NHWC
      // buffer when the position changes) and the lanes' partial dot products
      // with x at that position are kept; one transposing butterfly per batch
      // sums them over the group.
      {
        constexpr int W = CPL >= 4 ? 16 : 8;  // channels per lane
        constexpr int NV = W / 8;              // 16-byte pieces per lane
        constexpr int LW = CPL * 32 / W;       // lanes per group
        constexpr int GW = 32 / LW;            // groups per warp
        constexpr int NB = W == 16 ? 4 : 8;  // pairs per batch (registers)
        const int glw = lane & (LW - 1);
        const int gidw = sw * GW + (lane / LW);
        // piece v: channels cp[v] .. + 7 of the slice; its x line offset in
        // the window (chunk) and 16-byte piece within the swizzled line
        int cp[NV];
        uint32_t xo[NV], xpv[NV];
#pragma unroll
        for (int v = 0; v < NV; ++v) {
          cp[v] = v * (LW * 8) + glw * 8;
          xo[v] = (uint32_t)(cp[v] >> 6) * pl.chunk_pitch;
          xpv[v] = (uint32_t)((cp[v] & 63) >> 3) << 4;
        }
        const int E = pst[npos];
        const int ngroups = kSWarps * GW;
        const int ebeg = (int)((long long)E * gidw / ngroups);
        const int eend = (int)((long long)E * (gidw + 1) / ngroups);
        const int minlen = E / ngroups, maxlen = (E + ngroups - 1) / ngroups;
        const uint32_t gs = px::smem_u32(gsm0);
        const uint32_t xs = px::smem_u32(xsm0);
        float* gxrow = a.gx + (((long long)tx.n * g.h + tx.ylo) * g.w + tx.xlo) * C + cbeg;
        int cur = -1;
        float2 xv[W / 2], acc[W / 2];
#pragma unroll
        for (int c = 0; c < W / 2; ++c) xv[c] = acc[c] = make_float2(0.f, 0.f);
        // the group's gradient at `pos` into the NHWC buffer (vector float atomics)
        auto flush = [&](int pos) {
          float* dst = gxrow + (long long)pixoff[pos] * C;
#pragma unroll
          for (int v = 0; v < NV; ++v) red_add<8>(dst + cp[v], reinterpret_cast<const float*>(acc + 4 * v));
        };
        // the sample's gcol slice of a pair (NV 16-byte pieces)
        auto row = [&](const int2 en, uint4* gw) {
          const uint32_t ra = gs + (uint32_t)((en.x & 0xffff) >> 2) * row_bytes;
#pragma unroll
          for (int v = 0; v < NV; ++v)
            asm("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                : "=r"(gw[v].x), "=r"(gw[v].y), "=r"(gw[v].z), "=r"(gw[v].w)
                : "r"(ra + (uint32_t)(cp[v] * 2)));
        };
        // one pair: its gradient at the current position, its partial dot product
        auto pair = [&](const int2 en, const uint4* gw, bool valid, float& dpj) {
          const int pos = (int)((uint32_t)en.x >> 16);
          if (valid && pos != cur) {
            if (cur >= 0) flush(cur);
            cur = pos;
            const uint32_t lo = line_off((uint32_t)cur);
#pragma unroll
            for (int v = 0; v < NV; ++v) {
              uint4 xw;
              asm("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                  : "=r"(xw.x), "=r"(xw.y), "=r"(xw.z), "=r"(xw.w)
                  : "r"(xs + xo[v] + (lo ^ xpv[v])));
              xv[4 * v] = bf2(xw.x);
              xv[4 * v + 1] = bf2(xw.y);
              xv[4 * v + 2] = bf2(xw.z);
              xv[4 * v + 3] = bf2(xw.w);
            }
#pragma unroll
            for (int c = 0; c < W / 2; ++c) acc[c] = make_float2(0.f, 0.f);
          }
          const float w = __int_as_float(en.y);
          const float2 w2 = make_float2(w, w);
          float dsum = 0.f;
#pragma unroll
          for (int v = 0; v < NV; ++v) {
            const float2 g0 = bf2(gw[v].x), g1 = bf2(gw[v].y), g2 = bf2(gw[v].z), g3 = bf2(gw[v].w);
            acc[4 * v] = ffma2(w2, g0, acc[4 * v]);
            acc[4 * v + 1] = ffma2(w2, g1, acc[4 * v + 1]);
            acc[4 * v + 2] = ffma2(w2, g2, acc[4 * v + 2]);
            acc[4 * v + 3] = ffma2(w2, g3, acc[4 * v + 3]);
            float2 d2 = ffma2(g0, xv[4 * v], make_float2(0.f, 0.f));
            d2 = ffma2(g1, xv[4 * v + 1], d2);
            d2 = ffma2(g2, xv[4 * v + 2], d2);
            d2 = ffma2(g3, xv[4 * v + 3], d2);
            dsum += d2.x + d2.y;
          }
          dpj = dsum;
        };
        // the batch's dot products summed over the group, to the D table
        auto finish = [&](float* dp, int b) {
          const float dsum = group_sum_t<NB, LW>(dp, lane);
          constexpr int kSh = (LW / NB) == 1 ? 0 : ((LW / NB) == 2 ? 1 : ((LW / NB) == 4 ? 2 : 3));
          const int e = ebeg + b + (glw >> kSh);
          if ((glw & ((1 << kSh) - 1)) == 0 && e < eend) Dt[ent[e].x & 0xffff] = dsum;
        };
        // full batches (every group has NB pairs left), software-pipelined:
        // the next batch's pairs load while this one computes; then one
        // checked tail
        const int fullb = minlen / NB * NB;
        int2 enn[NB];
        if (fullb > 0) {
#pragma unroll
          for (int j = 0; j < NB; ++j) enn[j] = ent[ebeg + j];
        }
        for (int b = 0; b < fullb; b += NB) {
          int2 en[NB];
          uint4 gw[NB][NV];
#pragma unroll
          for (int j = 0; j < NB; ++j) {
            en[j] = enn[j];
            row(en[j], gw[j]);
          }
          if (b + NB < fullb) {
#pragma unroll
            for (int j = 0; j < NB; ++j) enn[j] = ent[ebeg + b + NB + j];
          }
          float dp[NB];
#pragma unroll
          for (int j = 0; j < NB; ++j) pair(en[j], gw[j], true, dp[j]);
          finish(dp, b);
        }
        if (fullb < maxlen) {
          float dp[NB];
#pragma unroll
          for (int j = 0; j < NB; ++j) {
            const int e = ebeg + fullb + j;
            const bool valid = e < eend;
            const int2 en = valid ? ent[e] : make_int2(0, 0);
            uint4 gw[NV];
            if (valid) {
              row(en, gw);
            } else {
#pragma unroll
              for (int v = 0; v < NV; ++v) gw[v] = make_uint4(0u, 0u, 0u, 0u);
            }
            pair(en, gw, valid, dp[j]);
          }
          finish(dp, fullb);
        }
        if (cur >= 0) flush(cur);
      }
      // ---------------------------------------------- samples outside the window
      const int nslow = slow[0];
      for (int q = sw; q < nslow; q += kSWarps) {
        const int it = slow[1 + q];
        const int4 tp = tap[it];
        const int2 yx = syx[it];
        const float ly = __int_as_float(tp.x), lx = __int_as_float(tp.y);
        float gv[CPL];
        uint32_t gws[CPL / 2];
        lds_words<CPL>(gsm + (size_t)it * row_bytes, gws);
        unpack_bf<CPL>(gws, gv);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int yy = yx.x + (j >> 1), xx = yx.y + (j & 1);
          const bool in = yy >= 0 && yy < g.h && xx >= 0 && xx < g.w;
          float xv[CPL];
          if (in) {
            ldg_bf<CPL>(a.xc + ((long long)tx.n * g.hw + (long long)yy * g.w + xx) * C + cbeg + cl, xv);
          } else {
#pragma unroll
            for (int c = 0; c < CPL; ++c) xv[c] = 0.f;
          }
          float d = 0.f;
#pragma unroll
          for (int c = 0; c < CPL; ++c) d = __fmaf_rn(gv[c], xv[c], d);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
          if (lane == 0) Dt[it * 4 + j] = d;
          if (in) {
            const float wv = __fmul_rn((j >> 1) ? ly : 1.0f - ly, (j & 1) ? lx : 1.0f - lx);
            float v[CPL];
#pragma unroll
            for (int c = 0; c < CPL; ++c) v[c] = wv * gv[c];
            red_add<CPL>(gximg + ((long long)yy * g.w + xx) * C, v);
          }
        }
      }
      // the window and gcol buffers are free for the tile after next
      __syncwarp();
      if (lane == 0) mbar_arrive(&wempty[s]);
      s_sync();
      // ---------------------------------------------- offset gradients
      for (int it = tid - kPThreads; it < items; it += kSThreads) {
        const int4 tp = tap[it];
        if (tp.w == 1 || tp.w == 3) continue;
        const float ly = __int_as_float(tp.x), lx = __int_as_float(tp.y);
        const float d00 = Dt[it * 4], d01 = Dt[it * 4 + 1], d10 = Dt[it * 4 + 2], d11 = Dt[it * 4 + 3];
        const float gy = __fmaf_rn(1.0f - lx, d10 - d00, lx * (d11 - d01));
        const float gxo = __fmaf_rn(1.0f - ly, d01 - d00, ly * (d11 - d10));
        const int4 ie = itab[it];
        const int k = ie.w & 0xffff;
        const long long pix = (long long)(tx.ho0 + (ie.z & 0xffff)) * g.wo + (tx.wo0 + (ie.z >> 16));
        atomicAdd(a.goff + ((long long)tx.n * M + 2 * k) * g.howo + pix, gy);
        atomicAdd(a.goff + ((long long)tx.n * M + 2 * k + 1) * g.howo + pix, gxo);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[s]);
    }
  }
  pdl_release();
}

// grad_x (NCHW) = the NHWC float32 accumulator, transposed through shared
// memory: 64 channels x 32 pixels per CTA, float4 loads along channels and
// stores along pixels.
__global__ void __launch_bounds__(256) nhwc_to_nchw_f32(const float* __restrict__ src,
                                                        float* __restrict__ dst, int C, long long HW) {
  __shared__ float tile[64][33];
  pdl_wait();
  const int n = blockIdx.z, c0 = blockIdx.y * 64;
  const long long p0 = (long long)blockIdx.x * 32;
  const int t = threadIdx.x;
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int e = t + 256 * u;  // 32 pixels x 16 float4 of channels
    const int pp = e >> 4, q = e & 15;
    const long long p = p0 + pp;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (p < HW) v = __ldg(reinterpret_cast<const float4*>(src + ((long long)n * HW + p) * C + c0 + 4 * q));
    tile[4 * q][pp] = v.x;
    tile[4 * q + 1][pp] = v.y;
    tile[4 * q + 2][pp] = v.z;
    tile[4 * q + 3][pp] = v.w;
  }
  __syncthreads();
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int e = t + 256 * u;  // 64 channels x 32 pixels
    const int c = e >> 5, pp = e & 31;
    const long long p = p0 + pp;
    if (p < HW) dst[((long long)n * C + c0 + c) * HW + p] = tile[c][pp];
  }
  pdl_release();
}

cudaError_t launch_pdl3(const void* func, dim3 grid, dim3 block, size_t smem, cudaStream_t s,
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

int sm_count3() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return sms;
}

}  // namespace

bool k3cl_supported(const Geom& g, dc_dtype dt, int margin) {
  if (!cl_supported(g, dt, margin) || g.groups != 1) return false;
  if ((long long)g.M * g.howo >= INT_MAX) return false;  // offset-map index table is 32-bit
  const int sms = sm_count3();
  if (sms <= 0) return false;
  return k3_make_plan(g, margin, sms).npx != 0;
}

cudaError_t launch_k3cl(const K3ClArgs& in, cudaStream_t s) {
  const Geom& g = in.g;
  const int sms = sm_count3();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const K3Plan pl = k3_make_plan(g, in.margin, sms);
  if (pl.npx == 0) return cudaErrorInvalidValue;
  CUtensorMap xmap;
  const unsigned long long dims[4] = {(unsigned long long)g.c_in, (unsigned long long)g.w,
                                      (unsigned long long)g.h, (unsigned long long)g.n};
  const unsigned long long strides[3] = {(unsigned long long)g.c_in * 2,
                                         (unsigned long long)g.w * g.c_in * 2,
                                         (unsigned long long)g.hw * g.c_in * 2};
  const unsigned int box[4] = {64u, (unsigned)pl.cols, (unsigned)pl.rows, 1u};
  if (!make_tmap_bf16(&xmap, in.xc, 4, dims, strides, box, true)) return cudaErrorInvalidValue;
  // gcol[n][pixel][tap][channel] as {channel, tap, column, row, image}; one
  // box = the tile's samples, this CTA's channels
  CUtensorMap gmap;
  const unsigned long long gdims[5] = {(unsigned long long)g.c_in, (unsigned long long)g.K,
                                       (unsigned long long)g.wo, (unsigned long long)g.ho,
                                       (unsigned long long)g.n};
  const unsigned long long row = (unsigned long long)g.K * g.c_in * 2;
  const unsigned long long gstrides[4] = {(unsigned long long)g.c_in * 2, row, row * g.wo,
                                          row * g.wo * g.ho};
  const unsigned int gbox[5] = {(unsigned)pl.cpc, (unsigned)g.K, (unsigned)pl.TW, (unsigned)pl.TH, 1u};
  if (!make_tmap_bf16(&gmap, in.gcol, 5, gdims, gstrides, gbox, false)) return cudaErrorInvalidValue;
  K3Args a{};
  a.g = g;
  a.xc = static_cast<const __nv_bfloat16*>(in.xc);
  a.off = in.off;
  a.gx = in.gx_nhwc;
  a.goff = in.goff;
  a.margin = in.margin;
  const void* func = nullptr;
  switch (pl.cpc / 32) {
    case 2: func = (const void*)k3_cl_bwd<2>; break;
    case 4: func = (const void*)k3_cl_bwd<4>; break;
    case 8: func = (const void*)k3_cl_bwd<8>; break;
    default: return cudaErrorInvalidValue;
  }
  const cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem);
  if (e != cudaSuccess) return e;
  K3Plan plc = pl;
  void* args[] = {&xmap, &gmap, &a, &plc};
  return launch_pdl3(func, dim3((unsigned)pl.grid), dim3(kThreads), pl.smem, s, args);
}

cudaError_t launch_gx_to_nchw(const float* gx_nhwc, float* grad_x, const Geom& g, cudaStream_t s) {
  const float* a = gx_nhwc;
  float* b = grad_x;
  int C = g.c_in;
  long long HW = g.hw;
  void* args[] = {&a, &b, &C, &HW};
  return launch_pdl3((const void*)nhwc_to_nchw_f32,
                     dim3((unsigned)ceil_div_ll(g.hw, 32), (unsigned)(g.c_in / 64), (unsigned)g.n),
                     dim3(256), 0, s, args);
}

// This file's share of dc_device_error.
unsigned int cl3_read_error(int clear) {
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_cl3_error, sizeof(v)) != cudaSuccess) return 2u;
  if (clear && v) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_cl3_error, &zero, sizeof(zero)) != cudaSuccess) return 2u;
  }
  return v;
}

}  // namespace dc
