// K3: backward of the bilinear sampling step.
//
// Derivatives of the layer of the explainer page "DefT: Boosting Scalability
// of Deformable Convolution Operations on GPUs" ("The argument in one glance":
// offset convolution -> four-neighbour bilinear blend -> main convolution),
// given gcol, the gradient of the deformed map from the main-convolution GEMM:
//   grad_x[b][c] at the four corners += corner weight * gcol
//   grad_offset (dy) += sum_{c in slice, group} gcol * ((1-lx)(v10-v00) + lx(v11-v01))
//   grad_offset (dx) += sum_{c in slice, group} gcol * ((1-ly)(v01-v00) + ly(v11-v10))
// The lower corner is floor(p), so at integer coordinates the offset gradient
// is the right-sided difference.  The kernel also writes the deformed map
// (the replayed forward sample) that the weight-gradient GEMM consumes.  The
// offset convolution's own backward runs afterwards in K4 on the completed
// offset gradient.
//
// GB300 mapping: a CTA owns a band of full-width output rows of one image and
// a slice of 16 input channels (no cluster: slices only meet in the offset
// gradient, which each CTA adds to global memory with fire-and-forget float
// reductions).  It stages its slice of the band's input window (receptive
// field + margin) once and accumulates grad_x over the same window in shared
// memory.  bf16 problems whose gcol comes from the tensor-core GEMM accumulate
// in 32-bit fixed point (integer shared-memory atomics, several times faster
// than float ones) with a per-CTA scale derived from the largest |gcol| of the
// tiles it reads; other problems accumulate floats.  Taps whose corners leave
// the window are queued and processed by all lanes together from global
// memory.  The window is flushed to grad_x with float atomics (neighbouring
// bands' windows overlap).
#include <type_traits>

#include "dc_band.cuh"

namespace dc {
namespace {

using band::kThreads;
using band::Tap;
using band::gload;
using band::make_tap;
constexpr int kMaxPx = band::kBandPx;
constexpr size_t kSmemBudget = 72 * 1024;  // three CTAs per SM

struct Plan {
  int R, TW, tiles_w, tiles_h, npx;
  int ps;  // pixel stride of the per-band offset arrays
  int cpc, csize;  // channels per CTA, number of channel slices
  int rows, cols, plane;
  int qcap;  // capacity of the deferred slow-tap queue
  int ml;    // offset channels staged per CTA (2K per offset group of its slice)
  size_t off_halo, off_gx, off_offs, off_part, off_tab, off_q, smem;
};

// Largest band (128, 64 or 32 pixels) whose shared memory fits and that
// still gives the grid at least two CTAs per SM (else the fitting band with
// the most CTAs), with slices of 16 channels: staged input, grad_x window,
// offsets, this CTA's partial offset gradient, pixel table and the slow-tap
// queue.
__host__ Plan make_plan(const Geom& g, dc_dtype dt, int margin) {
  constexpr long long kMinGrid = 2 * 152;
  const bool bf16 = dt == DC_BF16;
  const int cpc = 16;
  Plan best{}, most{};
  long long most_grid = 0;
  for (int px = kMaxPx; px >= 32; px /= 2) {
    const band::Shape sh = band::make_shape(g, margin, px);
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
    p.cpc = cpc;
    p.csize = (g.c_in + cpc - 1) / cpc;  // channel slices
    size_t at = 0;
    p.off_halo = at;
    at += (size_t)(bf16 ? cpc / 2 : cpc) * p.plane * 4;
    p.off_gx = at;
    at += (size_t)cpc * p.plane * 4;
    int ngroups = 1;  // most offset groups any channel slice touches
    for (int r = 0; r * cpc < g.c_in; ++r) {
      const int lo = r * cpc, hi = (r + 1) * cpc < g.c_in ? (r + 1) * cpc : g.c_in;
      const int ng = (hi - 1) / g.cg - lo / g.cg + 1;
      if (ng > ngroups) ngroups = ng;
    }
    p.ml = 2 * g.K * ngroups;  // offset channels a CTA reads: its own groups only
    p.off_offs = at;
    at += (size_t)p.ml * p.ps * 4;
    p.off_part = at;
    at += (size_t)p.ml * p.ps * 4;
    p.off_tab = at;  // pixel table [ps] + tap offsets [K]
    at += (size_t)(p.ps + g.K) * 4;
    p.qcap = p.npx * g.K * (ngroups < 4 ? ngroups : 4);
    p.off_q = at;  // queue counter + entries (overflow is handled in place)
    at += (size_t)(1 + p.qcap) * 4;
    p.smem = at;
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
  return most_grid > 0 ? most : best;  // over budget: the caller rejects the problem
}

__device__ __forceinline__ void gadd(float* plane, const Geom& g, int y, int x, float v) {
  if (y >= 0 && y < g.h && x >= 0 && x < g.w) atomicAdd(plane + (long long)y * g.w + x, v);
}

__device__ __forceinline__ float lo_bf16(uint32_t w) { return __uint_as_float(w << 16); }

// gcol is bf16 when it comes from the tensor-core GEMM (the fixed-point
// path), fp32 otherwise
template <bool kFixed>
using GcolT = typename std::conditional<kFixed, __nv_bfloat16, float>::type;

__device__ __forceinline__ float ldg_f(const float* p) { return __ldg(p); }
__device__ __forceinline__ float ldg_f(const __nv_bfloat16* p) { return __bfloat162float(__ldg(p)); }

// round(ws * gc) as an int, for |ws * gc| < 2^22: adding 1.5 * 2^23 puts the
// rounded integer in the low mantissa bits (one rounding, to nearest even)
__device__ __forceinline__ int to_fixed(float ws, float gc) {
  return __float_as_int(__fmaf_rn(ws, gc, 12582912.0f)) - 0x4B400000;
}
__device__ __forceinline__ float hi_bf16(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Sampling backward of one on-chip tap over `count` consecutive channels of
// the slice starting at slice channel `cl0`: reads gcol, the four staged
// corners, writes the replayed sample, adds the offset-gradient terms to
// sdy/sdx and scatters the corner weights times gcol into the grad_x window
// (shared-memory atomics).  Loads of a batch of channels are issued before any
// of the batch's atomics.  bf16: channel pairs share one corner word load.
template <typename T, bool kFixed>
__device__ __forceinline__ void band_bwd_run(const uint32_t* __restrict__ xw, int PL, int cols,
                                             int sbase, int cl0, int count,
                                             const GcolT<kFixed>* __restrict__ gp, long long gstride,
                                             T* cp, long long cstride, float* gxp, float ly,
                                             float lx, float w00, float w01, float w10, float w11,
                                             float& sA, float& sB, float& sC) {
  // offset-gradient terms as three sums over the run's channels, combined
  // once per tap by the caller: sA = sum gc (v10 - v00), sB = sum gc (v11 - v01),
  // sC = sum gc (v01 - v00); the fourth difference v11 - v10 is b + c - a
  auto one = [&](float gc, float v00, float v01, float v10, float v11, int ch) {
    sA = __fmaf_rn(gc, v10 - v00, sA);
    sB = __fmaf_rn(gc, v11 - v01, sB);
    sC = __fmaf_rn(gc, v01 - v00, sC);
    if (cp) cp[(long long)ch * cstride] = from_f<T>(blend4(ly, lx, v00, v01, v10, v11));
  };
  auto scatter = [&](float gc, int ch) {
    if (kFixed) {
      // fixed point: the weights arrive pre-scaled; integer shared-memory
      // atomics are several times faster than float ones
      int* q = reinterpret_cast<int*>(gxp) + ch * PL;
      atomicAdd(q, to_fixed(w00, gc));
      atomicAdd(q + 1, to_fixed(w01, gc));
      atomicAdd(q + cols, to_fixed(w10, gc));
      atomicAdd(q + cols + 1, to_fixed(w11, gc));
    } else {
      float* q = gxp + ch * PL;
      atomicAdd(q, w00 * gc);
      atomicAdd(q + 1, w01 * gc);
      atomicAdd(q + cols, w10 * gc);
      atomicAdd(q + cols + 1, w11 * gc);
    }
  };
  int ch = 0;
  if (sizeof(T) == 2) {
    const uint32_t* xs = xw + sbase;
    if (cl0 & 1) {  // odd start: high half of a pair word
      const uint32_t* wp = xs + (cl0 >> 1) * PL;
      const float gc = ldg_f(gp);
      one(gc, hi_bf16(wp[0]), hi_bf16(wp[1]), hi_bf16(wp[cols]), hi_bf16(wp[cols + 1]), 0);
      scatter(gc, 0);
      ch = 1;
    }
    constexpr int kPairs = 4;  // 8 channels per batch
    for (; ch + 2 * kPairs <= count; ch += 2 * kPairs) {
      uint32_t a00[kPairs], a01[kPairs], a10[kPairs], a11[kPairs];
      float g0[kPairs], g1[kPairs];
#pragma unroll
      for (int u = 0; u < kPairs; ++u) {
        const uint32_t* wp = xs + ((cl0 + ch) >> 1) * PL + u * PL;
        a00[u] = wp[0];
        a01[u] = wp[1];
        a10[u] = wp[cols];
        a11[u] = wp[cols + 1];
        g0[u] = ldg_f(gp + (long long)(ch + 2 * u) * gstride);
        g1[u] = ldg_f(gp + (long long)(ch + 2 * u + 1) * gstride);
      }
#pragma unroll
      for (int u = 0; u < kPairs; ++u) {
        one(g0[u], lo_bf16(a00[u]), lo_bf16(a01[u]), lo_bf16(a10[u]), lo_bf16(a11[u]), ch + 2 * u);
        one(g1[u], hi_bf16(a00[u]), hi_bf16(a01[u]), hi_bf16(a10[u]), hi_bf16(a11[u]), ch + 2 * u + 1);
      }
#pragma unroll
      for (int u = 0; u < kPairs; ++u) {
        scatter(g0[u], ch + 2 * u);
        scatter(g1[u], ch + 2 * u + 1);
      }
    }
    for (; ch < count; ++ch) {
      const int cl = cl0 + ch;
      const uint32_t* wp = xs + (cl >> 1) * PL;
      const float gc = ldg_f(gp + (long long)ch * gstride);
      if (cl & 1)
        one(gc, hi_bf16(wp[0]), hi_bf16(wp[1]), hi_bf16(wp[cols]), hi_bf16(wp[cols + 1]), ch);
      else
        one(gc, lo_bf16(wp[0]), lo_bf16(wp[1]), lo_bf16(wp[cols]), lo_bf16(wp[cols + 1]), ch);
      scatter(gc, ch);
    }
  } else {
    const float* xs = reinterpret_cast<const float*>(xw) + sbase + cl0 * PL;
    constexpr int kB = 8;
    for (; ch + kB <= count; ch += kB) {
      float v00[kB], v01[kB], v10[kB], v11[kB], gc[kB];
#pragma unroll
      for (int u = 0; u < kB; ++u) {
        const float* wp = xs + (ch + u) * PL;
        v00[u] = wp[0];
        v01[u] = wp[1];
        v10[u] = wp[cols];
        v11[u] = wp[cols + 1];
        gc[u] = ldg_f(gp + (long long)(ch + u) * gstride);
      }
#pragma unroll
      for (int u = 0; u < kB; ++u) one(gc[u], v00[u], v01[u], v10[u], v11[u], ch + u);
#pragma unroll
      for (int u = 0; u < kB; ++u) scatter(gc[u], ch + u);
    }
    for (; ch < count; ++ch) {
      const float* wp = xs + ch * PL;
      const float gc = ldg_f(gp + (long long)ch * gstride);
      one(gc, wp[0], wp[1], wp[cols], wp[cols + 1], ch);
      scatter(gc, ch);
    }
  }
}


template <typename T, bool kFixed>
__global__ void __launch_bounds__(kThreads, 3) k3_band_bwd(BwdArgs a, Plan pl) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int s_gmax;
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
  const int ncur = c_end - c_begin;
  const int g_begin = c_begin / g.cg;
  const int ylo = ho0 * g.sh - g.ph - a.margin;
  const int xlo = wo0 * g.sw - g.pw - a.margin;
  const int tid = threadIdx.x;
  const int PL = pl.plane;
  const int npx = pl.npx;
  const int PS = pl.ps;
  const int M = g.M;
  const long long img = (long long)n * g.c_in * g.hw;

  uint32_t* xw = reinterpret_cast<uint32_t*>(smem + pl.off_halo);
  float* gxs = reinterpret_cast<float*>(smem + pl.off_gx);     // [cpc][PL] grad_x window
  // offsets and partial offset gradient of this slice's offset groups only:
  // local row 2 * ((gg - g_begin) * K + k) (+1 for dx)
  float* offs = reinterpret_cast<float*>(smem + pl.off_offs);  // [ml][PS]
  float* part = reinterpret_cast<float*>(smem + pl.off_part);  // [ml][PS]
  const int ml = 2 * g.K * ((c_end - 1) / g.cg - g_begin + 1);
  const int m_base = 2 * g.K * g_begin;  // global offset channel of local row 0
  int* pix = reinterpret_cast<int*>(smem + pl.off_tab);        // (row << 16 | col) in band
  int* tapoff = pix + PS;                                      // window offset of tap k
  int* nslow = reinterpret_cast<int*>(smem + pl.off_q);        // deferred slow taps
  int* slowq = nslow + 1;

  // ---------------------------------------------------------------- staging
  band::fill_pixel_table(pix, npx, pl.TW);
  for (int k = tid; k < g.K; k += kThreads) {
    const int i = k / g.kw;
    tapoff[k] = i * g.dh * pl.cols + (k - i * g.kw) * g.dw;
  }
  band::stage_window<T>(x, g, img, c_begin, pl.cpc, ylo, xlo, pl.rows, pl.cols, PL, xw);
  for (int idx = tid; idx < pl.cpc * PL; idx += kThreads) gxs[idx] = 0.f;
  for (int idx = tid; idx < ml * PS; idx += kThreads) part[idx] = 0.f;
  if (tid == 0) {
    *nslow = 0;
    s_gmax = 0;
  }
  __syncthreads();
  {
    band::Walk2 w;
    w.init(tid, kThreads, npx);
    while (w.a < ml) {
      const int m = w.a, px = w.b;
      const int e = pix[px];
      const int ho = ho0 + (e >> 16), wo = wo0 + (e & 0xffff);
      float v = 0.f;
      if (ho < g.ho && wo < g.wo)
        v = a.off[((long long)n * M + m_base + m) * g.howo + (long long)ho * g.wo + wo];
      offs[m * PS + px] = v;
      w.next();
    }
  }
  __syncthreads();
  // x and the offsets come from the forward call; gcol and the cleared
  // grad_x / offset-gradient buffers come from the GCOL GEMM just before
  pdl_wait();
  pdl_release();

  // fixed-point scale of the grad_x window: every contribution is
  // |corner weight * gcol| <= G (the largest |gcol| of the GCOL tiles that
  // cover this slice's rows and this band's pixels, weights <= 1), and a
  // window element receives at most K * npx of them.  2^S keeps every sum
  // below 2^30 and every single contribution below 2^21 (the range of
  // to_fixed); the rounding error per contribution is 2^-(S+1) <= G * 2^-22.
  float fscale = 1.f, finv = 1.f;
  bool poison = false;  // a non-finite gcol in range: the window flushes NaN
  if (kFixed) {
    const int ty0 = (c_begin * g.K) / 128, ty1 = (c_end * g.K - 1) / 128;
    const int p_lo = ho0 * g.wo + wo0;
    const int p_hi = (min(ho0 + pl.R, g.ho) - 1) * g.wo + min(wo0 + pl.TW, g.wo) - 1;
    const int tx0 = p_lo / 128, tx1 = p_hi / 128;
    const int ntx = tx1 - tx0 + 1, nent = (ty1 - ty0 + 1) * ntx * 4;
    for (int i = tid; i < nent; i += kThreads) {
      const int e = i & 3, r = i >> 2;
      const int ty = ty0 + r / ntx, tx = tx0 + r - (r / ntx) * ntx;
      const float v = a.gmax[(((long long)n * a.gmax_ty + ty) * a.gmax_tx + tx) * 4 + e];
      atomicMax(&s_gmax, __float_as_int(v));  // |values|: their bits order like the floats
                                              // (a NaN sorts above inf)
    }
    __syncthreads();
    const float G = __int_as_float(s_gmax);
    if (!(G <= 3.402823466e38f)) {
      poison = true;
    } else {
      int eg;
      frexpf(G, &eg);  // G < 2^eg
      const int units = g.K * npx;
      const int lg = 32 - __clz(units > 1 ? units - 1 : 1);  // ceil(log2(K * npx))
      int S = min(30 - (eg + lg), 21 - eg);
      S = max(-126, min(126, S));
      fscale = ldexpf(1.0f, S);
      finv = ldexpf(1.0f, -S);
    }
  }

  // ---------------------------------------------------------------- sampling backward
  {
    const long long gstride = (long long)g.K * a.gcol_layout.row;
    const long long cstride = (long long)g.K * a.col_layout.row;
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
      const long long qo = (long long)ho * g.wo + wo;
      const GcolT<kFixed>* grow = static_cast<const GcolT<kFixed>*>(a.gcol) +
                                  (long long)k * a.gcol_layout.row + (long long)n * a.gcol_layout.img + qo;
      T* crow = col ? col + (long long)k * a.col_layout.row + (long long)n * a.col_layout.img + qo : nullptr;
      int c = c_begin;
      for (int gg = g_begin; c < c_end; ++gg) {
        const int run_end = min(c_end, (gg + 1) * g.cg);
        const Tap t = make_tap(by + offs[(2 * ((gg - g_begin) * g.K + k)) * PS + px],
                               bx + offs[(2 * ((gg - g_begin) * g.K + k) + 1) * PS + px], g, ylo, xlo,
                               pl.rows, pl.cols);
        const int sbase = (t.y0 - ylo) * pl.cols + (t.x0 - xlo);
        const float hy = 1.0f - t.ly, hx = 1.0f - t.lx;
        const float w00 = hy * hx, w01 = hy * t.lx, w10 = t.ly * hx, w11 = t.ly * t.lx;
        float sdy = 0.f, sdx = 0.f;
        float sA = 0.f, sB = 0.f, sC = 0.f;  // on-chip run sums (see band_bwd_run)
        if (t.inside && !t.fast) {
          // out-of-window tap: queued for the cooperative pass below, so that
          // this warp does not wait on global memory for one lane
          const int qi = atomicAdd(nslow, 1);
          if (qi < pl.qcap) {
            slowq[qi] = px | (k << 8) | ((gg - g_begin) << 16);
            c = run_end;
          }
        }
        if (!t.inside) {
          if (crow)
            for (; c < run_end; ++c) crow[(long long)c * cstride] = from_f<T>(0.f);
          c = run_end;
        }
        if (c < run_end && !t.fast) {
          // queue full: this out-of-window tap is handled here, from global memory
          for (; c < run_end; ++c) {
            const float gc = ldg_f(grow + (long long)c * gstride);
            const T* xp = x + img + (long long)c * g.hw;
            const float v00 = gload(xp, g, t.y0, t.x0), v01 = gload(xp, g, t.y0, t.x0 + 1);
            const float v10 = gload(xp, g, t.y0 + 1, t.x0), v11 = gload(xp, g, t.y0 + 1, t.x0 + 1);
            float* gq = a.gx + img + (long long)c * g.hw;
            gadd(gq, g, t.y0, t.x0, w00 * gc);
            gadd(gq, g, t.y0, t.x0 + 1, w01 * gc);
            gadd(gq, g, t.y0 + 1, t.x0, w10 * gc);
            gadd(gq, g, t.y0 + 1, t.x0 + 1, w11 * gc);
            sdy = __fmaf_rn(gc, hx * (v10 - v00) + t.lx * (v11 - v01), sdy);
            sdx = __fmaf_rn(gc, hy * (v01 - v00) + t.ly * (v11 - v10), sdx);
            if (crow) crow[(long long)c * cstride] = from_f<T>(blend4(t.ly, t.lx, v00, v01, v10, v11));
          }
        }
        if (c < run_end) {
          // on-chip tap: gcol, corners, blend, offset-gradient terms, scatter
          const GcolT<kFixed>* gp = grow + (long long)c * gstride;
          T* cp = crow ? crow + (long long)c * cstride : nullptr;
          float* gxp = gxs + (c - c_begin) * PL + sbase;
          if constexpr (kFixed)
            band_bwd_run<T, true>(xw, PL, pl.cols, sbase, c - c_begin, run_end - c, gp, gstride, cp,
                                  cstride, gxp, t.ly, t.lx, w00 * fscale, w01 * fscale,
                                  w10 * fscale, w11 * fscale, sA, sB, sC);
          else
            band_bwd_run<T, false>(xw, PL, pl.cols, sbase, c - c_begin, run_end - c, gp, gstride,
                                   cp, cstride, gxp, t.ly, t.lx, w00, w01, w10, w11, sA, sB, sC);
          c = run_end;
        }
        // dy term: hx (v10 - v00) + lx (v11 - v01); dx term: hy (v01 - v00) + ly (v11 - v10)
        sdy += hx * sA + t.lx * sB;
        sdx += hy * sC + t.ly * (sB + sC - sA);
        part[(2 * ((gg - g_begin) * g.K + k)) * PS + px] = sdy;
        part[(2 * ((gg - g_begin) * g.K + k) + 1) * PS + px] = sdx;
      }
    }
  }

  // ---------------------------------------------------------------- deferred slow taps
  // all lanes together: one (queued tap, channel) pair per thread, corners and
  // grad_x updates in global memory, offset-gradient terms added to `part`
  __syncthreads();
  {
    const int nq = min(*nslow, pl.qcap);
    const long long gstride = (long long)g.K * a.gcol_layout.row;
    const long long cstride = (long long)g.K * a.col_layout.row;
    for (int task = tid; task < nq * pl.cpc; task += kThreads) {
      const int ent = task / pl.cpc, jj = task - ent * pl.cpc;
      const int code = slowq[ent];
      const int px = code & 0xff, k = (code >> 8) & 0xff, gg = g_begin + (code >> 16);
      const int c = max(c_begin, gg * g.cg) + jj;
      if (c >= min(c_end, (gg + 1) * g.cg)) continue;
      const int e = pix[px];
      const int ho = ho0 + (e >> 16), wo = wo0 + (e & 0xffff);
      const int i = k / g.kw, j = k - i * g.kw;
      const Tap t = make_tap((float)(ho * g.sh - g.ph + i * g.dh) + offs[(2 * ((gg - g_begin) * g.K + k)) * PS + px],
                             (float)(wo * g.sw - g.pw + j * g.dw) + offs[(2 * ((gg - g_begin) * g.K + k) + 1) * PS + px],
                             g, ylo, xlo, pl.rows, pl.cols);
      const long long qo = (long long)ho * g.wo + wo;
      const float gc = ldg_f(static_cast<const GcolT<kFixed>*>(a.gcol) + (long long)k * a.gcol_layout.row + (long long)n * a.gcol_layout.img +
                             qo + (long long)c * gstride);
      const T* xp = x + img + (long long)c * g.hw;
      const float v00 = gload(xp, g, t.y0, t.x0), v01 = gload(xp, g, t.y0, t.x0 + 1);
      const float v10 = gload(xp, g, t.y0 + 1, t.x0), v11 = gload(xp, g, t.y0 + 1, t.x0 + 1);
      const float hy = 1.0f - t.ly, hx = 1.0f - t.lx;
      float* gp = a.gx + img + (long long)c * g.hw;
      gadd(gp, g, t.y0, t.x0, hy * hx * gc);
      gadd(gp, g, t.y0, t.x0 + 1, hy * t.lx * gc);
      gadd(gp, g, t.y0 + 1, t.x0, t.ly * hx * gc);
      gadd(gp, g, t.y0 + 1, t.x0 + 1, t.ly * t.lx * gc);
      atomicAdd(part + (2 * ((gg - g_begin) * g.K + k)) * PS + px, gc * (hx * (v10 - v00) + t.lx * (v11 - v01)));
      atomicAdd(part + (2 * ((gg - g_begin) * g.K + k) + 1) * PS + px, gc * (hy * (v01 - v00) + t.ly * (v11 - v10)));
      if (col)
        col[(long long)k * a.col_layout.row + (long long)n * a.col_layout.img + qo + (long long)c * cstride] =
            from_f<T>(blend4(t.ly, t.lx, v00, v01, v10, v11));
    }
  }

  // ---------------------------------------------------------------- offset gradient
  // this slice's partial sums, added to grad_offset (cleared before the pass);
  // full-width bands with 16-byte aligned rows add float4 quads
  __syncthreads();
  {
    const int nvalid = (min(ho0 + pl.R, g.ho) - ho0) * g.wo;
    const bool vec = pl.TW == g.wo && (g.howo & 3) == 0 && ((ho0 * g.wo) & 3) == 0 &&
                     (nvalid & 3) == 0 && (PS & 3) == 0 &&
                     (reinterpret_cast<uintptr_t>(a.goff) & 15) == 0;
    if (vec) {
      band::Walk2 w;
      w.init(tid, kThreads, nvalid / 4);
      while (w.a < ml) {
        const int m = w.a, p4 = w.b;
        w.next();
        const float4 v = *reinterpret_cast<const float4*>(part + m * PS + 4 * p4);
        if (v.x == 0.f && v.y == 0.f && v.z == 0.f && v.w == 0.f) continue;
        atomicAdd(reinterpret_cast<float4*>(a.goff + ((long long)n * M + m_base + m) * g.howo +
                                            (long long)ho0 * g.wo + 4 * p4),
                  v);
      }
    } else {
      band::Walk2 w;
      w.init(tid, kThreads, npx);
      while (w.a < ml) {
        const int m = w.a, px = w.b;
        w.next();
        const float v = part[m * PS + px];
        if (v == 0.f) continue;
        const int e = pix[px];
        const int ho = ho0 + (e >> 16), wo = wo0 + (e & 0xffff);
        if (ho < g.ho && wo < g.wo)
          atomicAdd(a.goff + ((long long)n * M + m_base + m) * g.howo + (long long)ho * g.wo + wo, v);
      }
    }
  }

  // ---------------------------------------------------------------- flush the grad_x window
  // (neighbouring bands' windows overlap: float atomics).  With image rows of
  // whole 16-byte quads, one float4 atomic per quad of an image row.
  {
    auto value = [&](int at) {
      return kFixed ? (poison ? __int_as_float(0x7fc00000)
                              : (float)reinterpret_cast<const int*>(gxs)[at] * finv)
                    : gxs[at];
    };
    if ((g.w & 3) == 0 && (reinterpret_cast<uintptr_t>(a.gx) & 15) == 0) {
      const int q_lo = (xlo >= 0 ? xlo : xlo - 3) / 4;
      const int q_hi = (xlo + pl.cols - 1 >= 0 ? xlo + pl.cols - 1 : xlo + pl.cols - 4) / 4;
      band::Walk3 w;
      w.init(tid, kThreads, pl.rows, q_hi - q_lo + 1);
      while (w.a < ncur) {
        const int cl = w.a, r = w.b, x0 = 4 * (q_lo + w.c);
        w.next();
        const int yy = ylo + r;
        if (yy < 0 || yy >= g.h || x0 < 0 || x0 >= g.w) continue;
        float v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int q = x0 + i - xlo;
          v[i] = (q >= 0 && q < pl.cols) ? value(cl * PL + r * pl.cols + q) : 0.f;
        }
        if (v[0] == 0.f && v[1] == 0.f && v[2] == 0.f && v[3] == 0.f) continue;
        atomicAdd(reinterpret_cast<float4*>(a.gx + img + (long long)(c_begin + cl) * g.hw +
                                            (long long)yy * g.w + x0),
                  make_float4(v[0], v[1], v[2], v[3]));
      }
    } else {
      band::Walk3 w;
      w.init(tid, kThreads, pl.rows, pl.cols);
      while (w.a < ncur) {
        const int cl = w.a, r = w.b, q = w.c;
        w.next();
        const int yy = ylo + r, xx = xlo + q;
        if (yy < 0 || yy >= g.h || xx < 0 || xx >= g.w) continue;
        const float v = value(cl * PL + r * pl.cols + q);
        if (v != 0.f) atomicAdd(a.gx + img + (long long)(c_begin + cl) * g.hw + (long long)yy * g.w + xx, v);
      }
    }
  }
}

template <typename T, bool kFixed>
cudaError_t launch_t(const BwdArgs& a, const Plan& pl, cudaStream_t s) {
  auto kern = k3_band_bwd<T, kFixed>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)pl.smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(pl.csize * pl.tiles_w), (unsigned)pl.tiles_h, (unsigned)a.g.n);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, a, pl);
  note_launches(1);
  return e;
}

}  // namespace

size_t bwd_smem_bytes(const Geom& g, dc_dtype dt, int margin) {
  return make_plan(g, dt, margin).smem;
}

cudaError_t launch_band_bwd(const BwdArgs& a, dc_dtype dt, cudaStream_t s) {
  const Plan pl = make_plan(a.g, dt, a.margin);
  if (dt == DC_BF16)
    return a.gmax ? launch_t<__nv_bfloat16, true>(a, pl, s) : launch_t<__nv_bfloat16, false>(a, pl, s);
  return launch_t<float, false>(a, pl, s);
}

}  // namespace dc
