// K1: fused offset convolution + bilinear sampling.
//
// Explainer page "DefT: Boosting Scalability of Deformable Convolution
// Operations on GPUs":
//   - "This paper's idea" / "Why it works": the offset convolution and the
//     interpolation read the same input, so they run in one kernel and the
//     offsets are consumed on chip instead of round-tripping through memory;
//   - "Why it works": tiling by the output's spatial dimensions fits each
//     block's inputs in shared memory;
//   - "The idea": each tile is padded by a margin sized to the (tight,
//     near-zero) offset distribution, so out-of-tile reads are rare; the ones
//     that remain take a guarded path to global memory.
//
// GB300 mapping.  The output is cut into bands of R full-width rows (at most
// 128 pixels).  A thread-block cluster of up to 8 CTAs owns one band of one
// image; CTA r of the cluster owns a slice of CPC input channels.  Each CTA
// stages its channel slice of the band's input halo (receptive field plus
// `margin` pixels per side, zero outside the image) in shared memory once;
// that one copy serves both phases:
//   phase 1  partial offset convolution over the CTA's channels (bf16: mma.sync
//            m16n8k16 tensor-core tiles, fp32 accumulate; fp32: CUDA cores),
//            then the cluster adds the partials through distributed shared
//            memory -- every CTA ends with the band's complete offsets on chip;
//   phase 2  bilinear sampling of the CTA's channels at every tap, from shared
//            memory, or from global memory for taps whose corners leave the
//            staged window.  Rows of the deformed map are written pixel-fastest,
//            so a band's full-width rows land as one contiguous run.
// In replay mode (offsets given) phase 1 is skipped and no cluster is formed.
#include <cooperative_groups.h>

#include "dc_band.cuh"

namespace cg = cooperative_groups;

namespace dc {
namespace {

constexpr int kThreads = 384;  // block size of K1 (12 warps: two CTAs per SM hide more latency)
using band::Tap;
using band::gload;
using band::make_tap;
constexpr int kMaxPx = band::kBandPx;  // largest band (output pixels)
constexpr int kNtMax = 9;              // n8 tiles of offset channels per mma pass
constexpr int kMaxCluster = band::kMaxCluster;
constexpr size_t kSmemBudget = 112 * 1024;

struct Plan {
  int R, TW;              // band: R output rows x TW output columns
  int tiles_w, tiles_h;
  int npx;                // R * TW
  int ps;                 // pixel stride of the per-band offset arrays
  int cpc;                // channels per CTA (multiple of 16)
  int csize;              // CTAs per cluster = channel slices
  int rows, cols;         // staged window
  int plane;              // padded words (bf16 pairs) or floats (fp32) per staged channel (pair)
  int mp;                 // offset channels padded to a multiple of 8
  int qcap;  // capacity of the deferred slow-tap queue
  size_t off_halo, off_w, off_part, off_offs, off_tab, off_q, smem;
};

__host__ size_t plan_bytes(Plan& p, const Geom& g, bool bf16, bool replay) {
  const int units = bf16 ? p.cpc / 2 : p.cpc;  // staged planes
  size_t at = 0;
  p.off_halo = at;
  at += (size_t)units * p.plane * 4;
  p.off_w = at;
  if (!replay) at += bf16 ? (size_t)g.K * (p.cpc / 2) * p.mp * 4 : (size_t)p.cpc * g.K * p.mp * 4;
  p.off_part = at;
  if (!replay) at += (size_t)p.mp * p.ps * 4;
  p.off_offs = at;
  at += (size_t)g.M * p.ps * 4;
  p.off_tab = at;  // pixel table [ps] + tap offsets [K]
  at += (size_t)(p.ps + g.K) * 4;
  {
    int ngroups = 1;  // most offset groups any channel slice touches
    for (int r = 0; r * p.cpc < g.c_in; ++r) {
      const int lo = r * p.cpc, hi = (r + 1) * p.cpc < g.c_in ? (r + 1) * p.cpc : g.c_in;
      const int ng = (hi - 1) / g.cg - lo / g.cg + 1;
      if (ng > ngroups) ngroups = ng;
    }
    p.qcap = p.npx * g.K * (ngroups < 4 ? ngroups : 4);
  }
  p.off_q = at;  // queue counter + entries (overflow is handled in place)
  at += (size_t)(1 + p.qcap) * 4;
  p.smem = at;
  return at;
}

// Largest band (128, 64 or 32 pixels) and widest channel slice (32 or 16, and
// wider when 8 CTAs of 32 would not cover C_in) whose shared memory fits and
// that still give the grid a CTA per SM (else the fitting plan with the most
// CTAs; measured: smaller bands than that only add halo).  (Slices of 16
// double the CTAs per band, but 8-CTA clusters then no longer fit in one wave
// on GB300.)
__host__ Plan make_plan(const Geom& g, dc_dtype dt, int margin, bool replay) {
  constexpr long long kMinGrid = 152;
  const bool bf16 = dt == DC_BF16;
  const int c16 = (g.c_in + 15) / 16 * 16;
  int cmin = 16;
  while ((c16 + cmin - 1) / cmin > kMaxCluster) cmin += 16;
  Plan best{}, most{};
  long long most_grid = 0;
  for (int px = kMaxPx; px >= 32; px /= 2) {
    const band::Shape sh = band::make_shape(g, margin, px);
    for (int cpc = (c16 <= 16 ? 16 : (cmin > 32 ? cmin : 32)); cpc >= cmin; cpc -= 16) {
      Plan p{};
      p.R = sh.R;
      p.TW = sh.TW;
      p.npx = sh.npx;
      p.ps = px + 8;  // rows of the per-band arrays start 8 banks apart
      p.tiles_w = sh.tiles_w;
      p.tiles_h = sh.tiles_h;
      p.rows = sh.rows;
      p.cols = sh.cols;
      p.plane = sh.plane;
      p.mp = (g.M + 7) / 8 * 8;
      p.cpc = cpc;
      p.csize = (g.c_in + cpc - 1) / cpc;
      plan_bytes(p, g, bf16, replay);
      if (best.smem == 0 || p.smem < best.smem) best = p;
      if (p.smem <= kSmemBudget) {
        const long long grid = (long long)p.csize * p.tiles_w * p.tiles_h * g.n;
        if (grid >= kMinGrid) return p;
        if (grid > most_grid) {
          most = p;
          most_grid = grid;
        }
      }
    }
  }
  return most_grid > 0 ? most : best;  // over budget: the caller rejects the problem
}

__device__ __forceinline__ float lo_bf16(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_bf16(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

using band::bf16_bits;

__device__ __forceinline__ void mma_bf16_16816(float* d, const uint32_t* a, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <typename T>
__device__ __forceinline__ float sample_global(const T* plane, const Geom& g, const Tap& t) {
  return blend4(t.ly, t.lx, gload(plane, g, t.y0, t.x0), gload(plane, g, t.y0, t.x0 + 1),
                gload(plane, g, t.y0 + 1, t.x0), gload(plane, g, t.y0 + 1, t.x0 + 1));
}

template <typename T, bool kReplay>
__global__ void __launch_bounds__(kThreads, 2) k1_band_sample(SampleArgs a, Plan pl) {
  extern __shared__ __align__(16) unsigned char smem[];
  constexpr bool kBf16 = sizeof(T) == 2;
  const Geom g = a.g;
  const T* __restrict__ x = static_cast<const T*>(a.x);
  T* __restrict__ col = static_cast<T*>(a.col);

  const int rank = (int)(blockIdx.x % pl.csize);
  const int tw_idx = (int)(blockIdx.x / pl.csize);
  const int band_idx = blockIdx.y;
  const int n = blockIdx.z;
  const int ho0 = band_idx * pl.R, wo0 = tw_idx * pl.TW;
  const int c_begin = rank * pl.cpc;
  const int c_end = min(g.c_in, c_begin + pl.cpc);
  const int g_begin = c_begin / g.cg;
  const int ylo = ho0 * g.sh - g.ph - a.margin;
  const int xlo = wo0 * g.sw - g.pw - a.margin;
  const int tid = threadIdx.x;
  const int PL = pl.plane;
  const int npx = pl.npx;
  const int PS = pl.ps;
  const long long img = (long long)n * g.c_in * g.hw;

  uint32_t* xw = reinterpret_cast<uint32_t*>(smem + pl.off_halo);  // staged input words
  float* offs = reinterpret_cast<float*>(smem + pl.off_offs);      // [M][PS]
  int* pix = reinterpret_cast<int*>(smem + pl.off_tab);            // (row << 16 | col) in band
  int* tapoff = pix + PS;                                          // window offset of tap k
  int* nslow = reinterpret_cast<int*>(smem + pl.off_q);            // deferred slow taps
  int* slowq = nslow + 1;
  if (tid == 0) *nslow = 0;
  // x, the weights and offset_add may come from the previous kernel on the
  // stream, and the column and offsets it may still be reading are rewritten
  pdl_wait();

  band::fill_pixel_table(pix, npx, pl.TW);
  for (int k = tid; k < g.K; k += kThreads) {
    const int i = k / g.kw;
    tapoff[k] = i * g.dh * pl.cols + (k - i * g.kw) * g.dw;
  }

  // ---------------------------------------------------------------- stage halo
  band::stage_window<T>(x, g, img, c_begin, pl.cpc, ylo, xlo, pl.rows, pl.cols, PL, xw);

  if (!kReplay) {
    // -------------------------------------------------------------- weights
    const T* __restrict__ w_off = static_cast<const T*>(a.w_off);
    const bool wvec = kBf16 && c_begin + pl.cpc <= g.c_in && ((g.c_in * g.K) & 7) == 0 &&
                      ((pl.cpc * g.K) & 7) == 0 && (reinterpret_cast<uintptr_t>(w_off) & 15) == 0;
    if (wvec) {
      // each offset channel's slice w_off[m][c_begin ..][*] is one contiguous,
      // 16-byte aligned run: read it as uint4 (eight weights), write the
      // halves of the channel-pair words; padding rows m >= M are zero
      uint32_t* wb = reinterpret_cast<uint32_t*>(smem + pl.off_w);  // [K][cpc/2][mp]
      unsigned short* wh = reinterpret_cast<unsigned short*>(wb);
      const int cpp = pl.cpc / 2;
      const unsigned short* wsrc = reinterpret_cast<const unsigned short*>(w_off);
      const int span8 = pl.cpc * g.K / 8, total = g.M * span8;
      for (int base = tid; base < total; base += 2 * kThreads) {
        uint4 v[2];
        int mm[2], t0[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int idx = base + u * kThreads;
          mm[u] = -1;
          if (idx < total) {
            const int m = idx / span8, q = idx - m * span8;
            mm[u] = m;
            t0[u] = 8 * q;
            v[u] = *reinterpret_cast<const uint4*>(wsrc + ((long long)m * g.c_in + c_begin) * g.K + 8 * q);
          }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          if (mm[u] < 0) continue;
          const uint32_t vw[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
          int cl = t0[u] / g.K, k = t0[u] - cl * g.K;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const unsigned short h = (unsigned short)((e & 1) ? (vw[e >> 1] >> 16) : (vw[e >> 1] & 0xffffu));
            wh[((k * cpp + (cl >> 1)) * pl.mp + mm[u]) * 2 + (cl & 1)] = h;
            if (++k == g.K) {
              k = 0;
              ++cl;
            }
          }
        }
      }
      for (int idx = tid; idx < g.K * cpp * (pl.mp - g.M); idx += kThreads) {
        const int row = idx / (pl.mp - g.M), m = g.M + idx - row * (pl.mp - g.M);
        wb[row * pl.mp + m] = 0u;
      }
    } else if (kBf16) {
      uint32_t* wb = reinterpret_cast<uint32_t*>(smem + pl.off_w);  // [K][cpc/2][mp]
      const int cpp = pl.cpc / 2;
      const __nv_bfloat16* wsrc = reinterpret_cast<const __nv_bfloat16*>(w_off);
      band::Walk3 w;
      w.init(tid, kThreads, cpp, pl.mp);
      constexpr int kB = 8;
      while (w.a < g.K) {
        uint32_t v[kB];
        int at[kB];
#pragma unroll
        for (int j = 0; j < kB; ++j) {
          v[j] = 0u;
          at[j] = -1;
          if (w.a < g.K) {
            const int k = w.a, cp = w.b, m = w.c;
            const int c0 = c_begin + 2 * cp;
            if (m < g.M && c0 < g.c_in) v[j] = bf16_bits(wsrc + ((long long)m * g.c_in + c0) * g.K + k);
            if (m < g.M && c0 + 1 < g.c_in)
              v[j] |= bf16_bits(wsrc + ((long long)m * g.c_in + c0 + 1) * g.K + k) << 16;
            at[j] = (k * cpp + cp) * pl.mp + m;
            w.next();
          }
        }
#pragma unroll
        for (int j = 0; j < kB; ++j)
          if (at[j] >= 0) wb[at[j]] = v[j];
      }
    } else {
      float* wf = reinterpret_cast<float*>(smem + pl.off_w);  // [cpc][K][mp]
      band::Walk3 w;
      w.init(tid, kThreads, g.K, pl.mp);
      while (w.a < pl.cpc) {
        const int cl = w.a, k = w.b, m = w.c;
        const int c = c_begin + cl;
        float v = 0.f;
        if (m < g.M && c < g.c_in) v = ld_f(w_off + ((long long)m * g.c_in + c) * g.K + k);
        wf[(cl * g.K + k) * pl.mp + m] = v;
        w.next();
      }
    }
    __syncthreads();

    // -------------------------------------------------------------- phase 1
    float* part = reinterpret_cast<float*>(smem + pl.off_part);  // [mp][PS]
    if (kBf16) {
      const uint32_t* wb = reinterpret_cast<const uint32_t*>(smem + pl.off_w);
      const int warp = tid >> 5, lane = tid & 31;
      const int gid = lane >> 2, tig = lane & 3;
      const int mtiles = (npx + 15) / 16;
      const int cpp = pl.cpc / 2;
      for (int mt = warp; mt < mtiles; mt += kThreads / 32) {
        const int r0 = mt * 16 + gid, r1 = r0 + 8;
        const int e0 = pix[r0 < npx ? r0 : 0], e1 = pix[r1 < npx ? r1 : 0];
        const int b0 = ((e0 >> 16) * g.sh + a.margin) * pl.cols + (e0 & 0xffff) * g.sw + a.margin;
        const int b1 = ((e1 >> 16) * g.sh + a.margin) * pl.cols + (e1 & 0xffff) * g.sw + a.margin;
        for (int nt0 = 0; nt0 < pl.mp / 8; nt0 += kNtMax) {
          const int ntn = min(kNtMax, pl.mp / 8 - nt0);
          float acc[kNtMax][4];
#pragma unroll
          for (int t = 0; t < kNtMax; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
          for (int k = 0; k < g.K; ++k) {
            const int toff = tapoff[k];
            for (int cpb = 0; cpb < cpp; cpb += 8) {
              uint32_t af[4];
              const uint32_t* xa = xw + (cpb + tig) * PL + toff;
              af[0] = xa[b0];
              af[1] = xa[b1];
              af[2] = xa[4 * PL + b0];
              af[3] = xa[4 * PL + b1];
              const uint32_t* wk = wb + ((k * cpp) + cpb + tig) * pl.mp + nt0 * 8 + gid;
#pragma unroll
              for (int t = 0; t < kNtMax; ++t)
                if (t < ntn) mma_bf16_16816(acc[t], af, wk[t * 8], wk[4 * pl.mp + t * 8]);
            }
          }
#pragma unroll
          for (int t = 0; t < kNtMax; ++t) {
            if (t >= ntn) continue;
            const int m = (nt0 + t) * 8 + 2 * tig;
            if (r0 < npx) {
              part[m * PS + r0] = acc[t][0];
              part[(m + 1) * PS + r0] = acc[t][1];
            }
            if (r1 < npx) {
              part[m * PS + r1] = acc[t][2];
              part[(m + 1) * PS + r1] = acc[t][3];
            }
          }
        }
      }
    } else {
      const float* wf = reinterpret_cast<const float*>(smem + pl.off_w);
      const float* xf = reinterpret_cast<const float*>(xw);
      constexpr int kMc = 12;
      const int ngrp = (g.M + kMc - 1) / kMc;
      band::Walk2 w;
      w.init(tid, kThreads, npx);
      while (w.a < ngrp) {
        const int m0 = w.a * kMc, px = w.b;
        const int e = pix[px];
        const int base = ((e >> 16) * g.sh + a.margin) * pl.cols + (e & 0xffff) * g.sw + a.margin;
        float acc[kMc];
#pragma unroll
        for (int t = 0; t < kMc; ++t) acc[t] = 0.f;
        for (int cl = 0; cl < pl.cpc; ++cl) {
          const float* xc = xf + cl * PL + base;
          const float* wc = wf + cl * g.K * pl.mp + m0;
          for (int k = 0; k < g.K; ++k) {
            const float xv = xc[tapoff[k]];
            const float4* wv = reinterpret_cast<const float4*>(wc + k * pl.mp);
#pragma unroll
            for (int t4 = 0; t4 < kMc / 4; ++t4) {
              if (m0 + 4 * t4 >= pl.mp) break;
              const float4 w4 = wv[t4];
              acc[4 * t4 + 0] = __fmaf_rn(w4.x, xv, acc[4 * t4 + 0]);
              acc[4 * t4 + 1] = __fmaf_rn(w4.y, xv, acc[4 * t4 + 1]);
              acc[4 * t4 + 2] = __fmaf_rn(w4.z, xv, acc[4 * t4 + 2]);
              acc[4 * t4 + 3] = __fmaf_rn(w4.w, xv, acc[4 * t4 + 3]);
            }
          }
        }
#pragma unroll
        for (int t = 0; t < kMc; ++t)
          if (m0 + t < g.M) part[(m0 + t) * PS + px] = acc[t];
        w.next();
      }
    }

    // -------------------------------------------------------------- cluster reduction
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    {
      // this CTA reduces its share of the (m, px) items (four per round, their
      // remote loads all in flight) and writes each sum into every peer's
      // offset array, so each partial is read once in the whole cluster
      const int items = g.M * npx;
      const int i_begin = (int)((long long)items * rank / pl.csize);
      const int i_end = (int)((long long)items * (rank + 1) / pl.csize);
      band::Walk2 w;
      w.init(i_begin + tid, kThreads, npx);
      int idx = i_begin + tid;
      while (idx < i_end) {
        int mm[4], pp[4];
        float v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          mm[j] = -1;
          v[j] = 0.f;
          if (idx < i_end) {
            mm[j] = w.a;
            pp[j] = w.b;
            w.next();
            idx += kThreads;
          }
        }
        for (int r = 0; r < pl.csize; ++r) {
          const float* rp = cluster.map_shared_rank(part, r);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (mm[j] >= 0) v[j] += rp[mm[j] * PS + pp[j]];
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (mm[j] < 0) continue;
          const int m = mm[j], px = pp[j];
          float vv = v[j];
          const int e = pix[px];
          const int ho = ho0 + (e >> 16), wo = wo0 + (e & 0xffff);
          if (ho < g.ho && wo < g.wo) {
            if (a.b_off) vv += a.b_off[m];
            const long long oi = ((long long)n * g.M + m) * g.howo + (long long)ho * g.wo + wo;
            if (a.off_add) vv += a.off_add[oi];
            if (a.off_out) a.off_out[oi] = vv;
          }
          for (int r = 0; r < pl.csize; ++r) cluster.map_shared_rank(offs, r)[m * PS + px] = vv;
        }
      }
    }
    cluster.sync();  // every CTA's offsets are complete; peers are done reading partials
  } else {
    __syncthreads();  // pixel table
    band::Walk2 w;
    w.init(tid, kThreads, npx);
    while (w.a < g.M) {
      const int m = w.a, px = w.b;
      const int e = pix[px];
      const int ho = ho0 + (e >> 16), wo = wo0 + (e & 0xffff);
      float v = 0.f;
      if (ho < g.ho && wo < g.wo)
        v = a.off_in[((long long)n * g.M + m) * g.howo + (long long)ho * g.wo + wo];
      offs[m * PS + px] = v;
      w.next();
    }
    __syncthreads();
  }

  pdl_release();  // the forward GEMM may set up while the sampling runs
  if (!kReplay && col == nullptr) return;  // offset convolution only (no sampling)

  // ---------------------------------------------------------------- slow-path count
  if (a.slow_count && rank == 0) {
    unsigned long long local = 0;
    band::Walk2 w;
    w.init(tid, kThreads, npx);
    while (w.a < g.K) {
      const int k = w.a, px = w.b;
      const int e = pix[px];
      const int ho = ho0 + (e >> 16), wo = wo0 + (e & 0xffff);
      if (ho < g.ho && wo < g.wo) {
        const int i = k / g.kw, j = k - (k / g.kw) * g.kw;
        const float by = (float)(ho * g.sh - g.ph + i * g.dh);
        const float bx = (float)(wo * g.sw - g.pw + j * g.dw);
        for (int gg = 0; gg < g.groups; ++gg) {
          const Tap t = make_tap(by + offs[(2 * (gg * g.K + k)) * PS + px],
                                 bx + offs[(2 * (gg * g.K + k) + 1) * PS + px], g, ylo, xlo,
                                 pl.rows, pl.cols);
          if (t.inside && !t.fast) ++local;
        }
      }
      w.next();
    }
    for (int o = 16; o > 0; o >>= 1) local += __shfl_xor_sync(0xffffffffu, local, o);
    if ((tid & 31) == 0 && local) atomicAdd(a.slow_count, local);
  }

  // ---------------------------------------------------------------- phase 2
  const long long cstride = (long long)g.K * a.col_layout.row;  // next channel's row
  band::Walk2 w;
  w.init(tid, kThreads, npx);
  while (w.a < g.K) {
    const int k = w.a, px = w.b;
    w.next();
    const int e = pix[px];
    const int ho = ho0 + (e >> 16), wo = wo0 + (e & 0xffff);
    if (ho >= g.ho || wo >= g.wo) continue;
    const int i = k / g.kw, j = k - i * g.kw;
    const float by = (float)(ho * g.sh - g.ph + i * g.dh);
    const float bx = (float)(wo * g.sw - g.pw + j * g.dw);
    T* crow = col + (long long)k * a.col_layout.row + (long long)n * a.col_layout.img +
              (long long)ho * g.wo + wo;
    // channels in runs that share one offset group (one sampling point)
    int c = c_begin;
    for (int gg = g_begin; c < c_end; ++gg) {
      const int run_end = min(c_end, (gg + 1) * g.cg);
      const Tap t = make_tap(by + offs[(2 * (gg * g.K + k)) * PS + px],
                             bx + offs[(2 * (gg * g.K + k) + 1) * PS + px], g, ylo, xlo, pl.rows,
                             pl.cols);
      const int sbase = (t.y0 - ylo) * pl.cols + (t.x0 - xlo);
      if (t.inside && !t.fast) {
        // out-of-window tap: queued for the cooperative pass below, so that
        // this warp does not wait on global memory for one lane
        const int qi = atomicAdd(nslow, 1);
        if (qi < pl.qcap) {
          slowq[qi] = px | (k << 8) | ((gg - g_begin) << 16);
          c = run_end;
        }
      }
      while (c < run_end) {
        const int rel = c - c_begin;
        if (kBf16 && !(rel & 1) && c + 1 < run_end) {
          float s0 = 0.f, s1 = 0.f;
          if (t.inside) {
            if (t.fast) {
              const uint32_t* wp = xw + (rel >> 1) * PL + sbase;
              const uint32_t w00 = wp[0], w01 = wp[1], w10 = wp[pl.cols], w11 = wp[pl.cols + 1];
              s0 = blend4(t.ly, t.lx, lo_bf16(w00), lo_bf16(w01), lo_bf16(w10), lo_bf16(w11));
              s1 = blend4(t.ly, t.lx, hi_bf16(w00), hi_bf16(w01), hi_bf16(w10), hi_bf16(w11));
            } else {
              s0 = sample_global(x + img + (long long)c * g.hw, g, t);
              s1 = sample_global(x + img + (long long)(c + 1) * g.hw, g, t);
            }
          }
          crow[(long long)c * cstride] = from_f<T>(s0);
          crow[(long long)(c + 1) * cstride] = from_f<T>(s1);
          c += 2;
        } else {
          float s = 0.f;
          if (t.inside) {
            if (t.fast) {
              const int pos = sbase;
              s = blend4(t.ly, t.lx, band::staged<T>(xw, PL, rel, pos),
                         band::staged<T>(xw, PL, rel, pos + 1),
                         band::staged<T>(xw, PL, rel, pos + pl.cols),
                         band::staged<T>(xw, PL, rel, pos + pl.cols + 1));
            } else {
              s = sample_global(x + img + (long long)c * g.hw, g, t);
            }
          }
          crow[(long long)c * cstride] = from_f<T>(s);
          c += 1;
        }
      }
    }
  }

  // ---------------------------------------------------------------- deferred slow taps
  // all lanes together: one (queued tap, channel) pair per thread, corners read
  // from global memory with the same blend as the on-chip path
  __syncthreads();
  const int nq = min(*nslow, pl.qcap);
  for (int task = tid; task < nq * pl.cpc; task += kThreads) {
    const int ent = task / pl.cpc, jj = task - ent * pl.cpc;
    const int code = slowq[ent];
    const int px = code & 0xff, k = (code >> 8) & 0xff, gg = g_begin + (code >> 16);
    const int c = max(c_begin, gg * g.cg) + jj;
    if (c >= min(c_end, (gg + 1) * g.cg)) continue;
    const int e = pix[px];
    const int ho = ho0 + (e >> 16), wo = wo0 + (e & 0xffff);
    const int i = k / g.kw, j = k - i * g.kw;
    const Tap t = make_tap((float)(ho * g.sh - g.ph + i * g.dh) + offs[(2 * (gg * g.K + k)) * PS + px],
                           (float)(wo * g.sw - g.pw + j * g.dw) + offs[(2 * (gg * g.K + k) + 1) * PS + px],
                           g, ylo, xlo, pl.rows, pl.cols);
    col[(long long)k * a.col_layout.row + (long long)n * a.col_layout.img + (long long)ho * g.wo + wo +
        (long long)c * cstride] = from_f<T>(sample_global(x + img + (long long)c * g.hw, g, t));
  }
}

template <typename T, bool kReplay>
cudaError_t launch_t(const SampleArgs& a, const Plan& pl, cudaStream_t s) {
  auto kern = k1_band_sample<T, kReplay>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)pl.smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(pl.csize * pl.tiles_w), (unsigned)pl.tiles_h, (unsigned)a.g.n);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  unsigned nattr = 0;
  // early start behind whatever precedes on the stream: the kernel waits for
  // it before its first global-memory access
  attr[nattr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[nattr].val.programmaticStreamSerializationAllowed = 1;
  ++nattr;
  if (!kReplay) {
    attr[nattr].id = cudaLaunchAttributeClusterDimension;
    attr[nattr].val.clusterDim.x = (unsigned)pl.csize;
    attr[nattr].val.clusterDim.y = 1;
    attr[nattr].val.clusterDim.z = 1;
    ++nattr;
  }
  cfg.attrs = attr;
  cfg.numAttrs = nattr;
  e = cudaLaunchKernelEx(&cfg, kern, a, pl);
  note_launches(1);
  return e;
}

}  // namespace

size_t sample_smem_bytes(const Geom& g, dc_dtype dt, int margin) {
  return make_plan(g, dt, margin, false).smem;
}

void sample_band(const Geom& g, dc_dtype dt, int margin, int* R, int* TW) {
  const Plan p = make_plan(g, dt, margin, false);
  *R = p.R;
  *TW = p.TW;
}

cudaError_t launch_sample(const SampleArgs& a, dc_dtype dt, cudaStream_t s) {
  const bool replay = a.off_in != nullptr;
  const Plan pl = make_plan(a.g, dt, a.margin, replay);
  if (dt == DC_BF16)
    return replay ? launch_t<__nv_bfloat16, true>(a, pl, s) : launch_t<__nv_bfloat16, false>(a, pl, s);
  return replay ? launch_t<float, true>(a, pl, s) : launch_t<float, false>(a, pl, s);
}

}  // namespace dc
