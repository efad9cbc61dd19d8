// K1, channels-last: fused offset convolution + bilinear sampling over an
// input staged channel-innermost.
//
// Explainer page "DefT: Boosting Scalability of Deformable Convolution
// Operations on GPUs":
//   - "This paper's idea" / "Why it works": the offset convolution and the
//     interpolation read the same input, so they run in one kernel and the
//     offsets are consumed on chip;
//   - "Why it works": tiling by the output's spatial dimensions puts each
//     tile's scattered gathers in shared memory;
//   - "The idea": the tile's input window is padded by a margin sized to the
//     offset distribution; samples whose corners leave it are read from
//     global memory instead.
//
// GB300 mapping.  x is first copied to NHWC (one transpose kernel), so that a
// tile's input window -- its receptive field plus `margin` pixels per side,
// zero outside the image -- is a plain 4-D box: TMA brings it into shared
// memory in 64-channel chunks with the 128-byte swizzle, one 128-byte line
// per (position, chunk).  The kernel is persistent and warp-specialised: one
// CTA (or a cluster of two, each holding half of the channels) per SM, two
// window buffers, and
//   P warps (8)  per tile: the offset convolution on tensor cores (mma.sync
//                m16n8k16, bf16 in, fp32 accumulate; rows = output pixels,
//                columns = offset channels, reduction = (tap, channel); A
//                straight from the swizzled window by ldmatrix, B from the
//                offset weights, which stay resident in shared memory in
//                fragment order for the whole run); with two CTAs per tile
//                the two channel halves' sums meet through distributed shared
//                memory; then offset_out and the tile's table of sampling
//                taps; then the TMA copy of a later tile's window;
//   S warps (8)  per tile, one tile behind P: bilinear sampling with lanes
//                over channels -- C/8 lanes take one (output pixel, tap), each
//                lane eight channels: four 16-byte corner loads (conflict
//                free), the blend in fp32 with the reference roundings, one
//                16-byte store.  The deformed map is pixel-major,
//                col[n][pixel][tap][channel].  Taps whose corners leave the
//                window load them from the NHWC copy in global memory.
// All waits are bounded mbarrier waits.
#include <cooperative_groups.h>
#include <limits.h>

#include "dc_band.cuh"
#include "dc_tma.cuh"

namespace dc {

// Raised by this file's bounded waits (read by dc_device_error).
__device__ unsigned int g_cl_error;

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kPWarps = 8;                 // TMA + offset convolution + tap table
constexpr int kSWarps = kWarps - kPWarps;  // sampling
constexpr int kPThreads = kPWarps * 32;
constexpr size_t kSmemBudget = 225 * 1024;

struct ClPlan {
  int TH, TW;              // output tile
  int tiles_h, tiles_w, tiles;  // tiles per image row / column, all tiles (all images)
  int rows, cols;          // staged window
  int csplit, cpc;         // CTAs per tile (a cluster), channels per CTA
  int nstages;             // window buffers: 2 (the next tile's copy overlaps), or 1
  int chunks;              // 64-channel chunks per CTA
  int npx;                 // TH * TW, a multiple of 16
  int mp, ntiles;          // offset channels padded to 8, their n8 tiles
  int kstl;                // reduction steps of 16 per CTA: K * cpc / 16
  uint32_t stage_bytes;    // bytes one window's TMA copies write: chunks * rows * cols * 128
  uint32_t chunk_pitch;    // rows * cols * 128 rounded up to 1024 (swizzle atoms stay aligned)
  int ntaps;               // tap-table entries per tile: npx * K * G
  size_t off_stage, off_wb, off_offs, off_partk, off_part, off_xbuf, off_taps, off_tab, off_oin, off_bar,
      smem;
  int grid;                // CTAs (a multiple of csplit)
};

__host__ ClPlan cl_plan_for(const Geom& g, int margin, int TH, int TW, int csplit, int sms,
                            int nstages = 2) {
  ClPlan p{};
  p.TH = TH;
  p.TW = TW;
  p.npx = TH * TW;
  p.tiles_h = (int)ceil_div_ll(g.ho, TH);
  p.tiles_w = (int)ceil_div_ll(g.wo, TW);
  p.tiles = g.n * p.tiles_h * p.tiles_w;
  p.rows = (TH - 1) * g.sh + (g.kh - 1) * g.dh + 1 + 2 * margin;
  p.cols = (TW - 1) * g.sw + (g.kw - 1) * g.dw + 1 + 2 * margin;
  p.csplit = csplit;
  p.cpc = g.c_in / csplit;
  p.chunks = p.cpc / 64;
  p.mp = (g.M + 7) / 8 * 8;
  p.ntiles = p.mp / 8;
  p.kstl = g.K * p.cpc / 16;
  p.stage_bytes = (uint32_t)p.chunks * p.rows * p.cols * 128u;
  p.chunk_pitch = ((uint32_t)p.rows * p.cols * 128u + 1023u) / 1024u * 1024u;
  p.ntaps = p.npx * g.K * g.groups;
  size_t at = 0;
  p.nstages = nstages;
  p.off_stage = at;  // window buffers of `chunks` 1024-byte aligned chunks each
  at += (size_t)nstages * p.chunks * p.chunk_pitch;
  p.off_wb = at;  // this CTA's offset weights in B-fragment order [kstl][ntiles][32] uint2
  at += (size_t)p.kstl * p.ntiles * 32 * 8;
  p.off_offs = at;  // offsets [npx][mp] fp32
  at += (size_t)p.npx * p.mp * 4;
  p.off_partk = at;  // the offset convolution's per-slice partial sums [KS][npx][mp]
  at += (size_t)kPWarps * p.npx * p.mp * 4;  // KS <= kPWarps
  p.off_part = at;  // two-CTA tiles: this CTA's partial sums [npx][mp]
  p.off_xbuf = at;
  if (csplit == 2) {
    at += (size_t)p.npx * p.mp * 4;
    p.off_xbuf = at;  // and the peer's, written by the peer, one per tile parity
    at += 2 * (size_t)p.npx * p.mp * 4;
  }
  p.off_taps = at;  // two tap tables [npx][K][G] of 32-byte entries (see the P warps)
  at += 2 * (size_t)p.ntaps * 32;
  p.off_tab = at;  // tap window offsets [K], then b_off [mp]
  at += (size_t)(g.K + 4 + p.mp) * 4;
  at = (at + 15) / 16 * 16;
  p.off_oin = at;  // the tile's given offsets / offset_add [2][M][npx] (prefetched a tile ahead)
  at += 2 * (size_t)g.M * p.npx * 4;
  at = (at + 7) / 8 * 8;
  p.off_bar = at;  // wfull[2], wempty[2], tfull[2], tempty[2], xfull[2]
  at += 10 * 8;
  p.smem = at + 1024;  // alignment slack of the dynamic buffer
  const int slots = sms / csplit * csplit;
  const int ctas = p.tiles * csplit;
  p.grid = ctas < slots ? ctas : slots;
  return p;
}

// Tile shape and channel split, chosen at the default margin so that a
// problem keeps its tiles (and its float32 summation order) whatever
// halo_margin is: one CTA per tile when its offset weights and two windows fit
// in shared memory, else two; among the tiles that fit, the lowest estimate
// of the busiest SM's work -- whole tiles per CTA times (sampling work +
// staging of the window + a fixed cost per tile).  If that shape does not fit
// at the requested margin, the best one that does.
constexpr int kRefMargin = 3;

__host__ ClPlan cl_best(const Geom& g, int margin, int sms) {
  static const int cand[][2] = {{2, 8}, {4, 8}, {2, 16}, {8, 8}, {4, 16}, {2, 32}, {16, 8}, {8, 16}, {4, 32}};
  for (int csplit = 1; csplit <= 2; ++csplit) {
    if ((g.c_in / csplit) % 64 != 0) continue;
    ClPlan best{};
    double best_cost = 0.0;
    for (const auto& c : cand) {
      const ClPlan p = cl_plan_for(g, margin, c[0], c[1], csplit, sms);
      if (p.smem > kSmemBudget || p.rows > 256 || p.cols > 256) continue;
      const double per_tile = (double)p.npx * g.K * p.cpc + 0.5 * (double)p.rows * p.cols * p.cpc +
                              8192.0;
      const double cost = (double)ceil_div_ll((long long)p.tiles * csplit, p.grid) * per_tile;
      if (best.npx == 0 || cost < best_cost) {
        best = p;
        best_cost = cost;
      }
    }
    if (best.npx != 0) return best;
  }
  return ClPlan{};
}

__host__ ClPlan cl_make_plan(const Geom& g, int margin, int sms) {
  const ClPlan ref = cl_best(g, kRefMargin, sms);
  if (ref.npx != 0) {
    // the reference shape at this margin: two window buffers, else one
    for (int ns = 2; ns >= 1; --ns) {
      const ClPlan p = cl_plan_for(g, margin, ref.TH, ref.TW, ref.csplit, sms, ns);
      if (p.smem <= kSmemBudget && p.rows <= 256 && p.cols <= 256) return p;
    }
  }
  return cl_best(g, margin, sms);
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// packed-pair fp32 arithmetic (two lanes of a 64-bit register pair)
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  float2 d;
  asm("{.reg .b64 ra, rb, rd;\n mov.b64 ra, {%2,%3};\n mov.b64 rb, {%4,%5};\n"
      " mul.rn.f32x2 rd, ra, rb;\n mov.b64 {%0,%1}, rd;}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{.reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2,%3};\n mov.b64 rb, {%4,%5};\n"
      " mov.b64 rc, {%6,%7};\n fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0,%1}, rd;}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

// blend of one bf16 channel pair (one word of each corner) with the
// reference roundings (blend4), both channels in one packed-pair chain
__device__ __forceinline__ uint32_t blend_pair2(float2 w00, float2 w01, float2 w10, float2 w11,
                                                uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  float2 s = fmul2(w00, make_float2(bf_lo(a), bf_hi(a)));
  s = ffma2(w01, make_float2(bf_lo(b), bf_hi(b)), s);
  s = ffma2(w10, make_float2(bf_lo(c), bf_hi(c)), s);
  s = ffma2(w11, make_float2(bf_lo(d), bf_hi(d)), s);
  return pack_bf16(s.x, s.y);
}

__device__ __forceinline__ uint4 ld_g16(const __nv_bfloat16* xc, const Geom& g, int n, int y,
                                        int x, int c) {
  if (y < 0 || y >= g.h || x < 0 || x >= g.w) return make_uint4(0u, 0u, 0u, 0u);
  return __ldg(reinterpret_cast<const uint4*>(xc + (((long long)n * g.h + y) * g.w + x) * g.c_in + c));
}

__device__ __forceinline__ uint4 lds16(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ uint2 lds8(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

// byte offset of window line `pos` for 16-byte piece 0 (128-byte swizzle);
// piece j is this XOR (j << 4)
__device__ __forceinline__ uint32_t line_off(uint32_t pos) { return (pos << 7) | ((pos & 7u) << 4); }

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(px::smem_u32(bar)) : "memory");
}

// arrive on the mbarrier at shared::cluster address `addr` (the peer's),
// releasing this thread's earlier writes at cluster scope
__device__ __forceinline__ void mbar_arrive_remote(uint32_t addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(addr) : "memory");
}

// bounded wait that acquires at cluster scope (the peer's writes)
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < px::kSpinLimit; ++i) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(px::smem_u32(bar)), "r"(parity)
        : "memory");
    if (ok) return true;
  }
  atomicOr(&g_cl_error, 1u);
  return false;
}

__device__ __forceinline__ uint32_t mapa(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// barrier of the four P warps only
__device__ __forceinline__ void p_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kPThreads) : "memory"); }

// the same barrier, returning whether v holds in every one of those threads
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

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

struct ClKArgs {
  Geom g;
  const __nv_bfloat16* xc;   // NHWC copy of x
  const uint2* wfrag;        // offset weights in B-fragment order, per channel slice (not in replay)
  const float* b_off;
  const float* off_add;
  const float* off_in;       // replay: sample these offsets, no offset convolution
  __nv_bfloat16* col;        // [n][pixel][tap][channel], or null (offsets only)
  float* off_out;
  unsigned long long* slow_count;
  int margin;
};

struct TileXY {
  int n, ho0, wo0, ylo, xlo;
};

__device__ __forceinline__ TileXY tile_xy(int t, const ClPlan& pl, const Geom& g, int margin) {
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

// A tap-table entry is two int4:
//   [0] corners in the window: the byte offsets of the four corner lines
//       (upper-left, upper-right, lower-left, lower-right) in a window chunk
//       for 16-byte piece 0 (piece j: XOR j << 4); corners read from global
//       memory: {y0, x0, -, -} in the image
//   [1] {ly, lx (float bits), dst, kind}: dst = output row (pixel * K + tap)
//       in the image; kind 0 window, 1 zeros (no corner touches the image),
//       2 global memory (corners outside the window), 3 pixel outside the
//       output (nothing written).

// Work split of the offset convolution over the P warps: NG groups of n8
// tiles (offset channels) x KS slices of the reduction.
template <int NT>
struct OcSplit {
  static constexpr int NG = NT <= 3 ? 1 : (NT <= 5 ? 2 : 4);
  static constexpr int KS = kPWarps / NG;
  static constexpr int NQ = (NT + NG - 1) / NG;  // n8 tiles per warp at most
};

// The offset convolution of one tile over this CTA's channels.  Warp w takes
// the n8 tiles q = w % NG, + NG, ... and the reduction slice w / NG (of
// (tap, 16-channel step) pairs), for every m16 tile of pixels: each A
// fragment (ldmatrix from the swizzled window) serves all its n8 tiles and
// each B fragment (resident fragment-ordered weights) all its m16 tiles.
// The slice's partial sums go to part_k[slice][npx][mp]; the caller adds the
// slices in a fixed order.
template <int NT, int CPS>
__device__ __forceinline__ void offconv_slices(const ClPlan& pl, const Geom& g, int margin,
                                               uint32_t win_u32, uint32_t wb_u32, const int* toff,
                                               float* part_k, int warp, int lane) {
  using S = OcSplit<NT>;
  constexpr int MG = 2;  // m16 tiles per pass
  const int ng = warp % S::NG, ksl = warp / S::NG;
  const int nk = g.K * CPS;
  const int k0 = (int)((long long)nk * ksl / S::KS), k1 = (int)((long long)nk * (ksl + 1) / S::KS);
  const uint32_t half = (uint32_t)(lane >> 4);
  const int MP = pl.mp;
  const int mtiles = pl.npx / 16;
  float* dst = part_k + (size_t)ksl * pl.npx * MP;
  for (int mt0 = 0; mt0 < mtiles; mt0 += MG) {
    int base[MG];
#pragma unroll
    for (int j = 0; j < MG; ++j) {
      const int pr = (mt0 + j < mtiles ? mt0 + j : mt0) * 16 + (lane & 15);
      const int py = pr / pl.TW, pxx = pr - py * pl.TW;
      base[j] = (py * g.sh + margin) * pl.cols + pxx * g.sw + margin;
    }
    float acc[MG][S::NQ][4];
#pragma unroll
    for (int j = 0; j < MG; ++j)
#pragma unroll
      for (int u = 0; u < S::NQ; ++u) acc[j][u][0] = acc[j][u][1] = acc[j][u][2] = acc[j][u][3] = 0.f;
    for (int kk = k0; kk < k1; ++kk) {
      const int k = kk / CPS, cs = kk - k * CPS;
      const int tk = toff[k];
      const uint32_t cb = win_u32 + (uint32_t)(cs >> 2) * pl.chunk_pitch;
      const uint32_t pb = ((uint32_t)((cs & 3) * 2) + half) << 4;
      uint32_t af[MG][4];
#pragma unroll
      for (int j = 0; j < MG; ++j)
        if (mt0 + j < mtiles) px::ldmatrix_x4(af[j], cb + (line_off((uint32_t)(base[j] + tk)) ^ pb));
      uint2 bb[S::NQ];
#pragma unroll
      for (int u = 0; u < S::NQ; ++u) {
        const int q = ng + u * S::NG;
        if (q < NT) bb[u] = lds8(wb_u32 + (uint32_t)(((kk * NT + q) * 32 + lane) * 8));
      }
#pragma unroll
      for (int j = 0; j < MG; ++j)
#pragma unroll
        for (int u = 0; u < S::NQ; ++u)
          if (mt0 + j < mtiles && ng + u * S::NG < NT)
            px::mma_bf16_16816(acc[j][u], af[j], bb[u].x, bb[u].y);
    }
    const int gid = lane >> 2, tig = lane & 3;
#pragma unroll
    for (int j = 0; j < MG; ++j) {
      if (mt0 + j >= mtiles) continue;
      const int r0 = (mt0 + j) * 16 + gid;
#pragma unroll
      for (int u = 0; u < S::NQ; ++u) {
        const int q = ng + u * S::NG;
        if (q >= NT) continue;
        const int m = q * 8 + 2 * tig;
        dst[r0 * MP + m] = acc[j][u][0];
        dst[r0 * MP + m + 1] = acc[j][u][1];
        dst[(r0 + 8) * MP + m] = acc[j][u][2];
        dst[(r0 + 8) * MP + m + 1] = acc[j][u][3];
      }
    }
  }
}

template <int NT, int CPS, bool kReplay>
__global__ void __launch_bounds__(kThreads, 1)
    k1_cl_sample(const __grid_constant__ CUtensorMap xmap, ClKArgs a, ClPlan pl) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = px::align1024(smem_raw);
  const Geom g = a.g;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t stage_pitch = (uint32_t)pl.chunks * pl.chunk_pitch;
  float* offs = reinterpret_cast<float*>(smem + pl.off_offs);  // [npx][mp]
  float* part = reinterpret_cast<float*>(smem + pl.off_part);  // [npx][mp] (two-CTA tiles)
  float* partk = reinterpret_cast<float*>(smem + pl.off_partk);  // [KS][npx][mp]
  float* xbuf = reinterpret_cast<float*>(smem + pl.off_xbuf);  // [2][npx][mp] (peer's)
  int4* taps0 = reinterpret_cast<int4*>(smem + pl.off_taps);   // [2][npx][K][G]
  int* toff = reinterpret_cast<int*>(smem + pl.off_tab);       // [K] window offset of tap k
  float* bsm = reinterpret_cast<float*>(toff + g.K + 4);       // [mp] b_off
  float* oin = reinterpret_cast<float*>(smem + pl.off_oin);    // [2][M][npx]
  uint64_t* wfull = reinterpret_cast<uint64_t*>(smem + pl.off_bar);
  uint64_t* wempty = wfull + 2;
  uint64_t* tfull = wfull + 4;
  uint64_t* tempty = wfull + 6;
  uint64_t* xfull = wfull + 8;
  const int K = g.K, G = g.groups, M = g.M, MP = pl.mp;
  const bool sampling = a.col != nullptr;
  const int rank = pl.csplit == 2 ? (int)cluster_rank() : 0;
  const int peer = rank ^ 1;
  const int cbeg = rank * pl.cpc;  // this CTA's channels [cbeg, cbeg + cpc)
  const int t0 = blockIdx.x / pl.csplit, tstep = gridDim.x / pl.csplit;

  auto issue = [&](int t, int s) {
    const TileXY tx = tile_xy(t, pl, g, a.margin);
    px::mbar_expect_tx(&wfull[s], pl.stage_bytes);
    unsigned char* dst = smem + pl.off_stage + (size_t)s * stage_pitch;
    for (int ch = 0; ch < pl.chunks; ++ch)
      px::tma_load_4d(dst + (size_t)ch * pl.chunk_pitch, &xmap, &wfull[s], cbeg + ch * 64, tx.xlo,
                      tx.ylo, tx.n);
  };

  if (tid == 0) {
    for (int q = 0; q < 2; ++q) {
      px::mbar_init(&wfull[q], 1);
      px::mbar_init(&wempty[q], kSWarps);
      px::mbar_init(&tfull[q], 1);
      px::mbar_init(&tempty[q], kSWarps);
      px::mbar_init(&xfull[q], kPThreads);  // the peer's P threads, one arrival each
    }
    px::fence_mbar_init();
  }
  for (int k = tid; k < K; k += kThreads) {
    const int i = k / g.kw;
    toff[k] = i * g.dh * pl.cols + (k - i * g.kw) * g.dw;
  }
  // per-tile offset inputs (the given offsets in replay mode, else offset_add)
  const float* oin_src = kReplay ? a.off_in : a.off_add;
  // x's NHWC copy, the fragment-ordered weights and offset_add come from the
  // preceding kernels on the stream
  pdl_wait();
  if (!kReplay) {
    // this CTA's offset weights, resident for the whole run
    const uint4* src = reinterpret_cast<const uint4*>(a.wfrag + (size_t)rank * pl.kstl * NT * 32);
    uint4* dst = reinterpret_cast<uint4*>(smem + pl.off_wb);
    for (int e = tid; e < pl.kstl * NT * 16; e += kThreads) dst[e] = __ldg(src + e);
  }
  for (int m = tid; m < MP; m += kThreads) bsm[m] = (!kReplay && a.b_off && m < M) ? a.b_off[m] : 0.f;
  __syncthreads();
  if (pl.csplit == 2) cluster_sync_all();  // the peer's barriers exist before any remote arrive

  if (warp < kPWarps) {
    // ============================================================ P warps
    int issued[2] = {0, 0}, consumed[2] = {0, 0};  // window copies (thread 0)
    if (tid == 0) {
      for (int q = 0; q < pl.nstages; ++q)
        if (t0 + q * tstep < pl.tiles) {
          issue(t0 + q * tstep, q);
          ++issued[q];
        }
    }
    const uint32_t wb_u32 = px::smem_u32(smem + pl.off_wb);
    // asynchronous copies of tile t's per-pixel offset inputs into oin[buf]
    // (zeros outside the output), waited for when the tile is processed
    auto prefetch_oin = [&](int t, int buf) {
      if (!oin_src || t >= pl.tiles) return;
      const TileXY tq = tile_xy(t, pl, g, a.margin);
      float* dsto = oin + (size_t)buf * M * pl.npx;
      for (int e = tid; e < M * pl.npx; e += kPThreads) {
        const int m = e / pl.npx, p = e - m * pl.npx;
        const int ho = tq.ho0 + p / pl.TW, wo = tq.wo0 + p % pl.TW;
        if (ho < g.ho && wo < g.wo) {
          const float* src = oin_src + ((long long)tq.n * M + m) * g.howo + (long long)ho * g.wo + wo;
          asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(px::smem_u32(dsto + e)),
                       "l"(src)
                       : "memory");
        } else {
          dsto[e] = 0.f;
        }
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
    };
    prefetch_oin(t0, 0);
    unsigned long long slow_local = 0;
    for (int i = 0, t = t0; t < pl.tiles; ++i, t += tstep) {
      const int s = i & 1;  // tap table slot (and exchange buffer)
      const uint32_t par = (uint32_t)(i >> 1) & 1u;
      const int ws = pl.nstages == 2 ? s : 0;  // window buffer
      const uint32_t wpar = (uint32_t)(pl.nstages == 2 ? (i >> 1) : i) & 1u;
      const TileXY tx = tile_xy(t, pl, g, a.margin);
      const uint32_t win_u32 = px::smem_u32(smem + pl.off_stage + (size_t)ws * stage_pitch);
      bool ok = px::mbar_wait(&wfull[ws], wpar, &g_cl_error);
      if (ok && tid == 0) ++consumed[ws];
      if (sampling && i >= 2) ok = ok && px::mbar_wait(&tempty[s], par ^ 1u, &g_cl_error);
      // this tile's offset inputs have landed (own copies; the barrier below
      // makes every thread's visible); the next tile's start now
      asm volatile("cp.async.wait_group 0;" ::: "memory");
      if (!p_sync_and(ok)) break;  // a wait expired: every P thread leaves together
      prefetch_oin(t + tstep, s ^ 1);
      const float* oin_t = oin + (size_t)s * M * pl.npx;
      // the copy of the next tile's window (tile i + 1), into the buffer of
      // tile i + 1 - nstages once the S warps are done with that tile: thread
      // 0 polls for that after each phase of this tile and issues it as soon
      // as the buffer is free (the last check waits), so that the window has
      // landed when this tile is done
      const int tn = t + tstep;
      const int jn = i + 1 - pl.nstages;  // the tile that last used that buffer
      bool pend = (sampling || pl.nstages == 1) && jn >= 0 && tn < pl.tiles && tid == 0;
      const int wbn = pl.nstages == 2 ? (s ^ 1) : 0;
      const uint32_t epar = (uint32_t)(pl.nstages == 2 ? (jn >> 1) : jn) & 1u;
      auto try_issue = [&](bool block) {
        // offsets only, one buffer: the P warps themselves read it, so the
        // copy waits for the end of the tile
        if (!pend || (!block && !sampling)) return;
        const bool ready = !sampling || (block ? px::mbar_wait(&wempty[wbn], epar, &g_cl_error)
                                               : px::mbar_try_wait(&wempty[wbn], epar));
        if (ready) {
          issue(tn, wbn);
          ++issued[wbn];
          pend = false;
        } else if (block) {
          pend = false;  // the wait expired (flag raised): no copy
        }
      };
      if (!kReplay) {
        // ---------------------------------------------------- offset convolution
        offconv_slices<NT, CPS>(pl, g, a.margin, win_u32, wb_u32, toff, partk, warp, lane);
        try_issue(false);
        p_sync();
        // the slices' partial sums in a fixed order: this CTA's share of the
        // offsets (to part, and into the peer's exchange buffer) or all of them
        {
          constexpr int KS = OcSplit<NT>::KS;
          float* dstp = pl.csplit == 2 ? part : offs;
          const uint32_t rb = pl.csplit == 2
                                  ? mapa(px::smem_u32(xbuf + (size_t)s * pl.npx * MP), (uint32_t)peer)
                                  : 0u;
          for (int e = tid; e < pl.npx * MP; e += kPThreads) {
            float v = partk[e];
#pragma unroll
            for (int q = 1; q < KS; ++q) v += partk[(size_t)q * pl.npx * MP + e];
            dstp[e] = v;
            if (pl.csplit == 2) st_cluster_f32(rb + (uint32_t)(e * 4), v);
          }
        }
        if (pl.csplit == 2) {
          mbar_arrive_remote(mapa(px::smem_u32(&xfull[s]), (uint32_t)peer));
          try_issue(false);
          const bool okx = mbar_wait_cluster(&xfull[s], par);
          if (!p_sync_and(okx)) break;
          // both halves' sums, identical on both CTAs (a + b == b + a)
          const float* xb = xbuf + (size_t)s * pl.npx * MP;
          for (int e = tid; e < pl.npx * MP; e += kPThreads) offs[e] = part[e] + xb[e];
        }
        p_sync();
        // bias, offset_add; the offsets out (one CTA of a pair)
        for (int e = tid; e < M * pl.npx; e += kPThreads) {
          const int m = e / pl.npx, p = e - m * pl.npx;
          float v = offs[p * MP + m] + bsm[m];
          if (a.off_add) v += oin_t[e];
          const int ho = tx.ho0 + p / pl.TW, wo = tx.wo0 + p % pl.TW;
          if (a.off_out && rank == 0 && ho < g.ho && wo < g.wo)
            a.off_out[((long long)tx.n * M + m) * g.howo + (long long)ho * g.wo + wo] = v;
          offs[p * MP + m] = v;
        }
      } else {
        // the given offsets (prefetched into oin_t)
        for (int e = tid; e < M * pl.npx; e += kPThreads) {
          const int m = e / pl.npx, p = e - m * pl.npx;
          offs[p * MP + m] = oin_t[e];
        }
      }
      p_sync();
      if (!sampling && pl.nstages == 2 && tid == 0 && t + 2 * tstep < pl.tiles) {
        // offsets only: this window is free once the convolution has read it
        issue(t + 2 * tstep, ws);
        ++issued[ws];
      }
      if (sampling) {
        // ---------------------------------------------------- tap table
        int4* taps = taps0 + (size_t)s * pl.ntaps * 2;
        for (int e = tid; e < pl.ntaps; e += kPThreads) {
          const int p = e / (K * G), kg = e - p * (K * G);
          const int k = kg / G, gg = kg - k * G;
          const int ho = tx.ho0 + p / pl.TW, wo = tx.wo0 + p % pl.TW;
          int4 e0 = make_int4(0, 0, 0, 0), e1 = make_int4(0, 0, 0, 3);
          if (ho < g.ho && wo < g.wo) {
            const int ki = k / g.kw, kj = k - ki * g.kw;
            const float by = (float)(ho * g.sh - g.ph + ki * g.dh);
            const float bx = (float)(wo * g.sw - g.pw + kj * g.dw);
            const float pyf = by + offs[p * MP + 2 * (gg * K + k)];
            const float pxf = bx + offs[p * MP + 2 * (gg * K + k) + 1];
            e1.z = (ho * g.wo + wo) * K + k;
            e1.w = 1;
            if (touches_image(pyf, pxf, g.h, g.w)) {
              const float fy = floorf(pyf), fx = floorf(pxf);
              const int y0 = (int)fy, x0 = (int)fx;
              e1.x = __float_as_int(pyf - fy);
              e1.y = __float_as_int(pxf - fx);
              const int ry = y0 - tx.ylo, rx = x0 - tx.xlo;
              if (ry >= 0 && ry + 1 < pl.rows && rx >= 0 && rx + 1 < pl.cols) {
                const uint32_t pos = (uint32_t)(ry * pl.cols + rx);
                e0 = make_int4((int)line_off(pos), (int)line_off(pos + 1), (int)line_off(pos + pl.cols),
                               (int)line_off(pos + pl.cols + 1));
                e1.w = 0;
              } else {
                e0.x = y0;
                e0.y = x0;
                e1.w = 2;
                // counted once over the CTAs of a tile: by the one holding
                // the group's first channel
                const int gc = gg * g.cg;
                if (gc >= cbeg && gc < cbeg + pl.cpc) ++slow_local;
              }
            }
          }
          taps[2 * e] = e0;
          taps[2 * e + 1] = e1;
        }
        p_sync();
        if (tid == 0) mbar_arrive(&tfull[s]);
      }
      try_issue(true);
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    if (tid == 0) {
      // after an expired wait: give the copies still in flight a bounded time
      // to land before the CTA exits (nothing to do after a normal run)
      for (int q = 0; q < 2; ++q)
        for (; consumed[q] < issued[q]; ++consumed[q])
          px::mbar_wait(&wfull[q], (uint32_t)consumed[q] & 1u, &g_cl_error);
    }
    if (a.slow_count) {
      for (int o = 16; o > 0; o >>= 1) slow_local += __shfl_xor_sync(0xffffffffu, slow_local, o);
      if (lane == 0 && slow_local) atomicAdd(a.slow_count, slow_local);
    }
  } else if (sampling) {
    // ============================================================ S warps
    const int sw = warp - kPWarps;
    const int L = pl.cpc / 8;       // lanes per (pixel, tap)
    const int ipw = 32 / L;         // (pixel, tap) items per warp and step
    const int sub = lane / L;
    const int cl = (lane - sub * L) * 8;  // channel offset within this CTA's slice
    const int lg = (cbeg + cl) / g.cg;    // offset group of this lane's channels
    const uint32_t pbits = (uint32_t)((cl & 63) >> 3) << 4;  // 16-byte piece, XOR form
    const int items = pl.npx * K;
    for (int i = 0, t = t0; t < pl.tiles; ++i, t += tstep) {
      const int s = i & 1;
      const uint32_t par = (uint32_t)(i >> 1) & 1u;
      const int ws = pl.nstages == 2 ? s : 0;
      const uint32_t wpar = (uint32_t)(pl.nstages == 2 ? (i >> 1) : i) & 1u;
      bool ok = px::mbar_wait(&tfull[s], par, &g_cl_error);
      ok = ok && px::mbar_wait(&wfull[ws], wpar, &g_cl_error);  // the window's copy, seen here too
      if (!__all_sync(0xffffffffu, ok)) break;
      const TileXY tx = tile_xy(t, pl, g, a.margin);
      const int4* taps = taps0 + (size_t)s * pl.ntaps * 2;
      const uint32_t lbase = px::smem_u32(smem + pl.off_stage + (size_t)ws * stage_pitch) +
                             (uint32_t)(cl >> 6) * pl.chunk_pitch;
      __nv_bfloat16* cimg = a.col + (long long)tx.n * g.howo * K * g.c_in + cbeg + cl;
      const int stride = kSWarps * ipw;
      // two items per lane and iteration: their loads overlap
      for (int it = sw * ipw + sub; it < items; it += 2 * stride) {
        uint4 v[2][4];
        float ly[2], lx[2];
        int dst[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int iu = it + u * stride;
          dst[u] = -1;
          ly[u] = lx[u] = 0.f;
          v[u][0] = v[u][1] = v[u][2] = v[u][3] = make_uint4(0u, 0u, 0u, 0u);
          if (iu < items) {
            const int4 e0 = taps[2 * (iu * G + lg)];
            const int4 e1 = taps[2 * (iu * G + lg) + 1];
            if (e1.w != 3) dst[u] = e1.z;
            ly[u] = __int_as_float(e1.x);
            lx[u] = __int_as_float(e1.y);
            if (e1.w == 0) {
              v[u][0] = lds16(lbase + ((uint32_t)e0.x ^ pbits));
              v[u][1] = lds16(lbase + ((uint32_t)e0.y ^ pbits));
              v[u][2] = lds16(lbase + ((uint32_t)e0.z ^ pbits));
              v[u][3] = lds16(lbase + ((uint32_t)e0.w ^ pbits));
            } else if (e1.w == 2) {
              v[u][0] = ld_g16(a.xc, g, tx.n, e0.x, e0.y, cbeg + cl);
              v[u][1] = ld_g16(a.xc, g, tx.n, e0.x, e0.y + 1, cbeg + cl);
              v[u][2] = ld_g16(a.xc, g, tx.n, e0.x + 1, e0.y, cbeg + cl);
              v[u][3] = ld_g16(a.xc, g, tx.n, e0.x + 1, e0.y + 1, cbeg + cl);
            }
          }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          if (dst[u] < 0) continue;
          const float hy = 1.0f - ly[u], hx = 1.0f - lx[u];
          const float w00 = __fmul_rn(hy, hx), w01 = __fmul_rn(hy, lx[u]);
          const float w10 = __fmul_rn(ly[u], hx), w11 = __fmul_rn(ly[u], lx[u]);
          const float2 q00 = make_float2(w00, w00), q01 = make_float2(w01, w01);
          const float2 q10 = make_float2(w10, w10), q11 = make_float2(w11, w11);
          uint4 o;
          o.x = blend_pair2(q00, q01, q10, q11, v[u][0].x, v[u][1].x, v[u][2].x, v[u][3].x);
          o.y = blend_pair2(q00, q01, q10, q11, v[u][0].y, v[u][1].y, v[u][2].y, v[u][3].y);
          o.z = blend_pair2(q00, q01, q10, q11, v[u][0].z, v[u][1].z, v[u][2].z, v[u][3].z);
          o.w = blend_pair2(q00, q01, q10, q11, v[u][0].w, v[u][1].w, v[u][2].w, v[u][3].w);
          *reinterpret_cast<uint4*>(cimg + (long long)dst[u] * g.c_in) = o;
        }
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&wempty[ws]);
        mbar_arrive(&tempty[s]);
      }
    }
  }
  pdl_release();
  // neither CTA of a pair leaves while the other may still write its buffers
  if (pl.csplit == 2) cluster_sync_all();
}

// NCHW -> NHWC copy of x (bf16): 64 channels x 128 pixels per CTA through
// shared memory.  Thread (channel pair cp, 16-pixel group) loads 2 x 32 bytes
// (its two channels' 16 pixels), packs the channel pairs into 32-bit words
// and writes them to a [pixel][channel pair] tile (lanes run over channel
// pairs: conflict-free); then each thread stores four 16-byte runs of 8
// channels of one pixel.  C % 64 == 0 and H * W % 8 == 0 (cl_supported).
constexpr int kTrPx = 128;
constexpr int kTrPitch = 36;  // words per tile row: 32 channel pairs + 4 (16-byte rows, banks shifted)
__device__ __forceinline__ void nchw_to_nhwc_tile(const __nv_bfloat16* __restrict__ x,
                                                  __nv_bfloat16* __restrict__ xc, int C, long long HW,
                                                  int bx, int by, int bz, uint32_t* tile) {
  const int n = bz, c0 = by * 64;
  const long long p0 = (long long)bx * kTrPx;
  const int t = threadIdx.x;
  {
    const int cp = t & 31, g16 = t >> 5;
    const long long p = p0 + 16 * g16;
    const __nv_bfloat16* r0 = x + ((long long)n * C + c0 + 2 * cp) * HW + p;
    const __nv_bfloat16* r1 = r0 + HW;
    uint4 a0 = make_uint4(0u, 0u, 0u, 0u), a1 = a0, b0 = a0, b1 = a0;
    if (p < HW) {
      a0 = __ldg(reinterpret_cast<const uint4*>(r0));
      b0 = __ldg(reinterpret_cast<const uint4*>(r1));
    }
    if (p + 8 < HW) {
      a1 = __ldg(reinterpret_cast<const uint4*>(r0 + 8));
      b1 = __ldg(reinterpret_cast<const uint4*>(r1 + 8));
    }
    const uint32_t wa[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const uint32_t wb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
    uint32_t* dst = tile + (16 * g16) * kTrPitch + cp;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      dst[(2 * j) * kTrPitch] = __byte_perm(wa[j], wb[j], 0x5410);      // pixel 2j: (c, c+1)
      dst[(2 * j + 1) * kTrPitch] = __byte_perm(wa[j], wb[j], 0x7632);  // pixel 2j + 1
    }
  }
  __syncthreads();
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int e = t + 256 * u;  // 128 pixels x 8 runs of 8 channels
    const int pp = e >> 3, j = e & 7;
    const long long p = p0 + pp;
    if (p < HW)
      *reinterpret_cast<uint4*>(xc + ((long long)n * HW + p) * C + c0 + 8 * j) =
          *reinterpret_cast<const uint4*>(tile + pp * kTrPitch + 4 * j);
  }
}

// Weight preparation, one launch.  Blocks [0, O): row o of the main weights
// permuted w [o][c][k] -> w' [o][k][c] through shared memory (16-byte loads
// and stores).  Blocks [O, O + ksteps) (unless frag is null): the offset
// weights in mma.m16n8k16 B-fragment order -- for reduction step ks (tap
// k = ks / (C/16), channels 16 * (ks % (C/16)) ..) and n8 tile q of offset
// channels, lane (gid, tig) holds {w(m, c0 + 2tig, k), w(m, c0 + 2tig + 1, k)}
// and the same at c0 + 8, m = 8q + gid; zero for m >= M.  The steps are
// ordered by channel slice (the channels one CTA of a tile holds), then tap.
__device__ __forceinline__ void prep_weights_block(const unsigned short* __restrict__ w,
                                                   unsigned short* __restrict__ wp,
                                                   const unsigned short* __restrict__ w_off,
                                                   uint2* __restrict__ frag, int O, int C, int K,
                                                   int M, int ntiles, int cpc, int wb,
                                                   unsigned short* row) {
  const int CK = C * K;
  if (wb < O) {
    const int o = wb;
    const uint4* src = reinterpret_cast<const uint4*>(w + (long long)o * CK);
    for (int e = threadIdx.x; e < CK / 8; e += blockDim.x) reinterpret_cast<uint4*>(row)[e] = __ldg(src + e);
    __syncthreads();
    uint4* dst = reinterpret_cast<uint4*>(wp + (long long)o * CK);
    for (int e = threadIdx.x; e < CK / 8; e += blockDim.x) {
      const int k = (8 * e) / C, c = 8 * e - k * C;  // 8 channels of tap k
      uint32_t v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        v[j] = (uint32_t)row[(c + 2 * j) * K + k] | ((uint32_t)row[(c + 2 * j + 1) * K + k] << 16);
      dst[e] = make_uint4(v[0], v[1], v[2], v[3]);
    }
  } else if (frag) {
    // reduction step ks of channel slice r (slices of cpc channels, in slice
    // order): tap k, channels r * cpc + 16 * (step within the tap) ..
    const int ks_all = wb - O;
    const int kstl = K * cpc / 16, r = ks_all / kstl, ks = ks_all - r * kstl;
    const int cps = cpc / 16;
    const int k = ks / cps;
    for (int e = threadIdx.x; e < ntiles * 32; e += blockDim.x) {
      const int q = e >> 5, lane = e & 31;
      const int c0 = r * cpc + (ks - k * cps) * 16 + 2 * (lane & 3);
      const int m = q * 8 + (lane >> 2);
      uint2 v = make_uint2(0u, 0u);
      if (m < M) {
        const long long b = (long long)m * C;
        v.x = (uint32_t)w_off[(b + c0) * K + k] | ((uint32_t)w_off[(b + c0 + 1) * K + k] << 16);
        v.y = (uint32_t)w_off[(b + c0 + 8) * K + k] | ((uint32_t)w_off[(b + c0 + 9) * K + k] << 16);
      }
      frag[(long long)ks_all * ntiles * 32 + e] = v;
    }
  }
}

// The channels-last preparation in one launch: blocks [0, nxb) the NHWC copy
// of x (block b: pixel tile b % ntx, channel chunk (b / ntx) % nty, image
// b / (ntx * nty)), the rest the weight layouts (two independent jobs that
// the sampling stage both waits for).
__global__ void __launch_bounds__(256) cl_prep(const __nv_bfloat16* __restrict__ x,
                                               __nv_bfloat16* __restrict__ xc, long long HW, int ntx,
                                               int nty, int nxb, const unsigned short* __restrict__ w,
                                               unsigned short* __restrict__ wp,
                                               const unsigned short* __restrict__ w_off,
                                               uint2* __restrict__ frag, int O, int C, int K, int M,
                                               int ntiles, int cpc) {
  __shared__ __align__(16) uint32_t tile[kTrPx * kTrPitch];
  extern __shared__ __align__(16) unsigned short row[];  // C * K (weight blocks)
  pdl_wait();
  const int b = (int)blockIdx.x;
  if (b < nxb)
    nchw_to_nhwc_tile(x, xc, C, HW, b % ntx, (b / ntx) % nty, b / (ntx * nty), tile);
  else
    prep_weights_block(w, wp, w_off, frag, O, C, K, M, ntiles, cpc, b - nxb, row);
  pdl_release();
}

cudaError_t launch_pdl(const void* func, dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       void** args, int cluster_x = 1) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  unsigned nattr = 1;
  if (cluster_x > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)cluster_x;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    nattr = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = nattr;
  const cudaError_t e = cudaLaunchKernelExC(&cfg, func, args);
  note_launches(1);
  return e;
}

int sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return sms;
}

}  // namespace

namespace {
typedef CUresult (*EncodeTiledFnCl)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                    const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                    const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                    CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFnCl encode_cl() {
  static EncodeTiledFnCl fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFnCl>(f);
  }
  return fn;
}
}  // namespace

namespace {
bool make_tmap_dt(CUtensorMap* m, CUtensorMapDataType dt, const void* base, int rank,
                  const unsigned long long* dims, const unsigned long long* strides_bytes,
                  const unsigned int* box, bool swizzle128) {
  EncodeTiledFnCl fn = encode_cl();
  if (!fn) return false;
  cuuint64_t d[5];
  cuuint64_t st[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) st[i] = strides_bytes[i];
  }
  return fn(m, dt, (cuuint32_t)rank, const_cast<void*>(base), d, st, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

// fp32 tensor map, no swizzle (zero fill outside the tensor).
bool make_tmap_f32(CUtensorMap* m, const void* base, int rank, const unsigned long long* dims,
                   const unsigned long long* strides_bytes, const unsigned int* box) {
  return make_tmap_dt(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, base, rank, dims, strides_bytes, box, false);
}

// bf16 tensor map (zero fill outside the tensor); 128-byte swizzle or none.
bool make_tmap_bf16(CUtensorMap* m, const void* base, int rank, const unsigned long long* dims,
                    const unsigned long long* strides_bytes, const unsigned int* box,
                    bool swizzle128) {
  EncodeTiledFnCl fn = encode_cl();
  if (!fn) return false;
  cuuint64_t d[5];
  cuuint64_t st[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) st[i] = strides_bytes[i];
  }
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(base), d, st,
            bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool cl_supported(const Geom& g, dc_dtype dt, int margin) {
  if (dt != DC_BF16 || g.c_in % 64 != 0 || g.c_in > 256 || g.cg % 8 != 0) return false;
  if (g.hw % 8 != 0 || g.kdim % 8 != 0 || g.howo % 8 != 0 || g.M > 72) return false;
  const int nt = (g.M + 7) / 8;
  if (nt != 3 && nt != 5 && nt != 7 && nt != 9) return false;  // compiled offset-channel tilings
  const int sms = sm_count();
  if (sms <= 0) return false;
  if (g.h > 32000 || g.w > 32000) return false;  // slow-tap coordinates are packed in 15 bits
  const ClPlan p = cl_make_plan(g, margin, sms);
  return p.npx != 0;
}

void cl_tile(const Geom& g, int margin, int* th, int* tw) {
  const ClPlan p = cl_make_plan(g, margin, sm_count() > 0 ? sm_count() : 152);
  *th = p.TH;
  *tw = p.TW;
}

size_t cl_wfrag_bytes(const Geom& g) {
  return (size_t)(g.K * g.c_in / 16) * ((g.M + 7) / 8) * 32 * sizeof(uint2);
}

cudaError_t launch_cl_prep(const void* x, void* xc, const void* w, void* wp, const void* w_off,
                           void* frag, const Geom& g, int margin, cudaStream_t s) {
  const __nv_bfloat16* xp = static_cast<const __nv_bfloat16*>(x);
  __nv_bfloat16* xcp = static_cast<__nv_bfloat16*>(xc);
  const unsigned short* a = static_cast<const unsigned short*>(w);
  unsigned short* b = static_cast<unsigned short*>(wp);
  const unsigned short* c = static_cast<const unsigned short*>(w_off);
  uint2* f = static_cast<uint2*>(frag);
  long long HW = g.hw;
  int ntx = (int)ceil_div_ll(g.hw, kTrPx), nty = g.c_in / 64;
  int nxb = ntx * nty * g.n;
  int O = w ? g.c_out : 0, C = g.c_in, K = g.K, M = g.M, nt = (g.M + 7) / 8;
  const int sms = sm_count();
  // the fragments are ordered by the channel slices the sampling stage's plan uses
  const ClPlan pl = cl_make_plan(g, margin, sms > 0 ? sms : 152);
  int cpc = pl.csplit > 0 ? g.c_in / pl.csplit : g.c_in;
  const long long blocks = (long long)nxb + O + (frag ? g.K * g.c_in / 16 : 0);
  const size_t smem = (size_t)C * K * 2;
  cudaError_t e = cudaFuncSetAttribute((const void*)cl_prep, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  void* args[] = {&xp, &xcp, &HW, &ntx, &nty, &nxb, &a, &b, &c, &f, &O, &C, &K, &M, &nt, &cpc};
  return launch_pdl((const void*)cl_prep, dim3((unsigned)blocks), dim3(256), smem, s, args);
}

cudaError_t launch_cl_sample(const ClArgs& in, cudaStream_t s) {
  const Geom& g = in.g;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const ClPlan pl = cl_make_plan(g, in.margin, sms);
  if (pl.npx == 0) return cudaErrorInvalidValue;
  CUtensorMap xmap;
  const unsigned long long dims[4] = {(unsigned long long)g.c_in, (unsigned long long)g.w,
                                      (unsigned long long)g.h, (unsigned long long)g.n};
  const unsigned long long strides[3] = {(unsigned long long)g.c_in * 2,
                                         (unsigned long long)g.w * g.c_in * 2,
                                         (unsigned long long)g.hw * g.c_in * 2};
  const unsigned int box[4] = {64u, (unsigned)pl.cols, (unsigned)pl.rows, 1u};
  if (!make_tmap_bf16(&xmap, in.xc, 4, dims, strides, box, true)) return cudaErrorInvalidValue;
  ClKArgs a{};
  a.g = g;
  a.xc = static_cast<const __nv_bfloat16*>(in.xc);
  a.wfrag = static_cast<const uint2*>(in.wfrag);
  a.b_off = in.b_off;
  a.off_add = in.off_add;
  a.off_in = in.off_in;
  a.col = static_cast<__nv_bfloat16*>(in.col);
  a.off_out = in.off_out;
  a.slow_count = in.slow_count;
  a.margin = in.margin;
  const bool replay = in.off_in != nullptr;
  const void* func = nullptr;
#define DC_K1CL(NT, CPS)                                                                     \
  if (pl.ntiles == NT && pl.cpc / 16 == CPS)                                                 \
    func = replay ? (const void*)k1_cl_sample<NT, CPS, true> : (const void*)k1_cl_sample<NT, CPS, false>;
  DC_K1CL(3, 4) DC_K1CL(3, 8) DC_K1CL(3, 16)
  DC_K1CL(5, 4) DC_K1CL(5, 8) DC_K1CL(5, 16)
  DC_K1CL(7, 4) DC_K1CL(7, 8) DC_K1CL(7, 16)
  DC_K1CL(9, 4) DC_K1CL(9, 8) DC_K1CL(9, 16)
#undef DC_K1CL
  if (!func) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem);
  if (e != cudaSuccess) return e;
  ClPlan plc = pl;
  void* args[] = {&xmap, &a, &plc};
  return launch_pdl(func, dim3((unsigned)pl.grid), dim3(kThreads), pl.smem, s, args, pl.csplit);
}

// This file's share of dc_device_error: the flag of its bounded waits.
unsigned int cl_read_error(int clear) {
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_cl_error, sizeof(v)) != cudaSuccess) return 2u;
  if (clear && v) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_cl_error, &zero, sizeof(zero)) != cudaSuccess) return 2u;
  }
  return v;
}

}  // namespace dc
