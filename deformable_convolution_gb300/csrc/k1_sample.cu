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
// One CTA owns a TH x TW tile of output pixels of one image.  The input halo
// of that tile (receptive field plus `margin` pixels on every side) is staged
// in shared memory a chunk of channels at a time, zero-filled outside the
// image.  Pass 1 accumulates the offset convolution for the tile's pixels over
// all channel chunks; pass 2 restages each chunk and samples every (channel,
// tap, pixel) from shared memory, or from global memory for taps whose corners
// leave the staged window.  The deformed map is written with pixels fastest
// (coalesced), one row per (channel, tap).
#include "dc_common.cuh"

namespace dc {
namespace {

constexpr int kThreads = 256;
constexpr int kTH = 8, kTW = 16;       // output tile
constexpr int kTilePx = kTH * kTW;
constexpr int kAccMax = 8;              // offset accumulators per thread

struct Window {
  int y_lo, x_lo, rows, cols;
};

__host__ __device__ inline Window make_window(const Geom& g, int ho0, int wo0, int margin) {
  Window w;
  w.y_lo = ho0 * g.sh - g.ph - margin;
  w.x_lo = wo0 * g.sw - g.pw - margin;
  w.rows = (kTH - 1) * g.sh + (g.kh - 1) * g.dh + 1 + 2 * margin;
  w.cols = (kTW - 1) * g.sw + (g.kw - 1) * g.dw + 1 + 2 * margin;
  return w;
}

__host__ __device__ inline int chunk_channels(const Geom& g, int margin, size_t elt) {
  // channels per staged chunk: keep the halo chunk near 48 KB
  Window w = make_window(g, 0, 0, margin);
  long long per_c = (long long)w.rows * w.cols * (long long)elt;
  long long cc = (48 * 1024) / per_c;
  if (cc < 1) cc = 1;
  if (cc > g.c_in) cc = g.c_in;
  if (cc > 32) cc = 32;
  return (int)cc;
}

__host__ __device__ inline int offset_chunk(const Geom& g) {
  // offset channels computed per pass so that each thread holds <= kAccMax
  int mc = kAccMax * kThreads / kTilePx;
  return mc < g.M ? mc : g.M;
}

template <typename T>
__device__ void stage_halo(const T* __restrict__ x, const Geom& g, int n, int c0, int cc,
                           const Window& win, T* xs) {
  const int plane = win.rows * win.cols;
  const int total = cc * plane;
  for (int idx = threadIdx.x; idx < total; idx += kThreads) {
    const int cl = idx / plane;
    const int rem = idx - cl * plane;
    const int r = rem / win.cols;
    const int q = rem - r * win.cols;
    const int c = c0 + cl;
    const int yy = win.y_lo + r, xx = win.x_lo + q;
    T v = from_f<T>(0.0f);
    if (c < g.c_in && yy >= 0 && yy < g.h && xx >= 0 && xx < g.w)
      v = x[(((long long)n * g.c_in + c) * g.h + yy) * g.w + xx];
    xs[idx] = v;
  }
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
    k1_fused_sample(SampleArgs a, int tiles_w, int cc, int mc) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const Geom g = a.g;
  const T* __restrict__ x = static_cast<const T*>(a.x);
  T* __restrict__ col = static_cast<T*>(a.col);

  const int n = blockIdx.y;
  const int tile = blockIdx.x;
  const int ho0 = (tile / tiles_w) * kTH;
  const int wo0 = (tile % tiles_w) * kTW;
  const Window win = make_window(g, ho0, wo0, a.margin);
  const int plane = win.rows * win.cols;

  // shared memory: [offsets: kTilePx x M floats][w_off chunk: mc x cc x K floats][halo: cc x plane T]
  float* offs = reinterpret_cast<float*>(smem_raw);
  float* wsm = offs + (size_t)kTilePx * g.M;
  T* xs = reinterpret_cast<T*>(wsm + (size_t)mc * cc * g.K);

  const long long howo = g.howo;

  // ---------------------------------------------------------------- pass 1
  if (a.off_in == nullptr) {
    const T* __restrict__ w_off = static_cast<const T*>(a.w_off);
    for (int m0 = 0; m0 < g.M; m0 += mc) {
      const int mcur = min(mc, g.M - m0);
      float acc[kAccMax];
#pragma unroll
      for (int r = 0; r < kAccMax; ++r) acc[r] = 0.0f;
      for (int c0 = 0; c0 < g.c_in; c0 += cc) {
        const int ccur = min(cc, g.c_in - c0);
        __syncthreads();
        stage_halo<T>(x, g, n, c0, cc, win, xs);
        for (int idx = threadIdx.x; idx < mcur * cc * g.K; idx += kThreads) {
          const int mm = idx / (cc * g.K);
          const int rem = idx - mm * cc * g.K;
          const int cl = rem / g.K;
          const int k = rem - cl * g.K;
          float v = 0.0f;
          if (cl < ccur)
            v = ld_f(w_off + ((long long)(m0 + mm) * g.c_in + c0 + cl) * g.K + k);
          wsm[idx] = v;
        }
        __syncthreads();
#pragma unroll
        for (int r = 0; r < kAccMax; ++r) {
          const int pair = threadIdx.x + r * kThreads;
          if (pair >= kTilePx * mcur) break;
          const int mm = pair / kTilePx;
          const int px = pair - mm * kTilePx;
          const int ty = px / kTW, tx = px - (px / kTW) * kTW;
          if (ho0 + ty >= g.ho || wo0 + tx >= g.wo) continue;
          float s = acc[r];
          for (int cl = 0; cl < ccur; ++cl) {
            const T* xp = xs + cl * plane + (ty * g.sh + a.margin) * win.cols + tx * g.sw + a.margin;
            const float* wp = wsm + (mm * cc + cl) * g.K;
            for (int i = 0; i < g.kh; ++i)
              for (int j = 0; j < g.kw; ++j)
                s = __fmaf_rn(wp[i * g.kw + j], to_f(xp[i * g.dh * win.cols + j * g.dw]), s);
          }
          acc[r] = s;
        }
      }
      // finish: bias, external shift, write to smem and to the offset output
#pragma unroll
      for (int r = 0; r < kAccMax; ++r) {
        const int pair = threadIdx.x + r * kThreads;
        if (pair >= kTilePx * mcur) break;
        const int mm = pair / kTilePx;
        const int px = pair - mm * kTilePx;
        const int ty = px / kTW, tx = px - (px / kTW) * kTW;
        const int ho = ho0 + ty, wo = wo0 + tx;
        if (ho >= g.ho || wo >= g.wo) continue;
        const int m = m0 + mm;
        float v = acc[r];
        if (a.b_off) v += a.b_off[m];
        const long long oi = ((long long)n * g.M + m) * howo + (long long)ho * g.wo + wo;
        if (a.off_add) v += a.off_add[oi];
        offs[px * g.M + m] = v;
        if (a.off_out) a.off_out[oi] = v;
      }
    }
  } else {
    for (int idx = threadIdx.x; idx < kTilePx * g.M; idx += kThreads) {
      const int m = idx / kTilePx;
      const int px = idx - m * kTilePx;
      const int ho = ho0 + px / kTW, wo = wo0 + px % kTW;
      float v = 0.0f;
      if (ho < g.ho && wo < g.wo)
        v = a.off_in[((long long)n * g.M + m) * howo + (long long)ho * g.wo + wo];
      offs[px * g.M + m] = v;
    }
  }
  __syncthreads();

  // count the (pixel, tap, group) sampling points that leave the staged window
  if (a.slow_count) {
    unsigned long long local = 0;
    for (int pair = threadIdx.x; pair < kTilePx * g.K; pair += kThreads) {
      const int k = pair / kTilePx;
      const int px = pair - k * kTilePx;
      const int ty = px / kTW, tx = px % kTW;
      if (ho0 + ty >= g.ho || wo0 + tx >= g.wo) continue;
      const int i = k / g.kw, j = k - (k / g.kw) * g.kw;
      for (int gg = 0; gg < g.groups; ++gg) {
        const float py = (float)((ho0 + ty) * g.sh - g.ph + i * g.dh) + offs[px * g.M + 2 * (gg * g.K + k)];
        const float pxf = (float)((wo0 + tx) * g.sw - g.pw + j * g.dw) + offs[px * g.M + 2 * (gg * g.K + k) + 1];
        if (!touches_image(py, pxf, g.h, g.w)) continue;
        const int y0 = (int)floorf(py) - win.y_lo, x0 = (int)floorf(pxf) - win.x_lo;
        if (y0 < 0 || y0 + 1 >= win.rows || x0 < 0 || x0 + 1 >= win.cols) ++local;
      }
    }
    for (int o = 16; o > 0; o >>= 1) local += __shfl_xor_sync(0xffffffffu, local, o);
    if ((threadIdx.x & 31) == 0 && local) atomicAdd(a.slow_count, local);
  }

  // ---------------------------------------------------------------- pass 2
  for (int c0 = 0; c0 < g.c_in; c0 += cc) {
    const int ccur = min(cc, g.c_in - c0);
    __syncthreads();
    stage_halo<T>(x, g, n, c0, cc, win, xs);
    __syncthreads();
    for (int pair = threadIdx.x; pair < kTilePx * g.K; pair += kThreads) {
      const int k = pair / kTilePx;
      const int px = pair - k * kTilePx;
      const int ty = px / kTW, tx = px % kTW;
      const int ho = ho0 + ty, wo = wo0 + tx;
      if (ho >= g.ho || wo >= g.wo) continue;
      const int i = k / g.kw, j = k - (k / g.kw) * g.kw;
      const float by = (float)(ho * g.sh - g.ph + i * g.dh);
      const float bx = (float)(wo * g.sw - g.pw + j * g.dw);
      const long long q = (long long)n * a.col_layout.img + (long long)ho * g.wo + wo;
      int gcur = -1;
      float ly = 0.f, lx = 0.f;
      int y0 = 0, x0 = 0;
      bool inside = false, fast = false;
      for (int cl = 0; cl < ccur; ++cl) {
        const int c = c0 + cl;
        const int gg = c / g.cg;
        if (gg != gcur) {
          gcur = gg;
          const float py = by + offs[px * g.M + 2 * (gg * g.K + k)];
          const float pxf = bx + offs[px * g.M + 2 * (gg * g.K + k) + 1];
          inside = touches_image(py, pxf, g.h, g.w);
          if (inside) {
            const float fy = floorf(py), fx = floorf(pxf);
            ly = py - fy;
            lx = pxf - fx;
            y0 = (int)fy;
            x0 = (int)fx;
            const int ry = y0 - win.y_lo, rx = x0 - win.x_lo;
            fast = ry >= 0 && ry + 1 < win.rows && rx >= 0 && rx + 1 < win.cols;
          }
        }
        float s = 0.0f;
        if (inside) {
          float v00, v01, v10, v11;
          if (fast) {
            const T* p = xs + cl * plane + (y0 - win.y_lo) * win.cols + (x0 - win.x_lo);
            v00 = to_f(p[0]);
            v01 = to_f(p[1]);
            v10 = to_f(p[win.cols]);
            v11 = to_f(p[win.cols + 1]);
          } else {
            const T* base = x + ((long long)n * g.c_in + c) * g.hw;
            const bool r0 = y0 >= 0 && y0 < g.h, r1 = y0 + 1 >= 0 && y0 + 1 < g.h;
            const bool q0 = x0 >= 0 && x0 < g.w, q1 = x0 + 1 >= 0 && x0 + 1 < g.w;
            v00 = (r0 && q0) ? ld_f(base + (long long)y0 * g.w + x0) : 0.0f;
            v01 = (r0 && q1) ? ld_f(base + (long long)y0 * g.w + x0 + 1) : 0.0f;
            v10 = (r1 && q0) ? ld_f(base + (long long)(y0 + 1) * g.w + x0) : 0.0f;
            v11 = (r1 && q1) ? ld_f(base + (long long)(y0 + 1) * g.w + x0 + 1) : 0.0f;
          }
          s = blend4(ly, lx, v00, v01, v10, v11);
        }
        col[(long long)(c * g.K + k) * a.col_layout.row + q] = from_f<T>(s);
      }
    }
  }
}

template <typename T>
size_t smem_for(const Geom& g, int margin, int cc, int mc) {
  Window w = make_window(g, 0, 0, margin);
  return (size_t)kTilePx * g.M * 4 + (size_t)mc * cc * g.K * 4 +
         (size_t)cc * w.rows * w.cols * sizeof(T);
}

}  // namespace

size_t sample_smem_bytes(const Geom& g, dc_dtype dt, int margin) {
  const size_t elt = dt == DC_BF16 ? 2 : 4;
  const int cc = chunk_channels(g, margin, elt);
  const int mc = offset_chunk(g);
  return dt == DC_BF16 ? smem_for<__nv_bfloat16>(g, margin, cc, mc)
                       : smem_for<float>(g, margin, cc, mc);
}

cudaError_t launch_sample(const SampleArgs& a, dc_dtype dt, cudaStream_t s) {
  const Geom& g = a.g;
  const int tiles_h = (int)ceil_div_ll(g.ho, kTH), tiles_w = (int)ceil_div_ll(g.wo, kTW);
  const size_t elt = dt == DC_BF16 ? 2 : 4;
  const int cc = chunk_channels(g, a.margin, elt);
  const int mc = offset_chunk(g);
  const size_t smem = sample_smem_bytes(g, dt, a.margin);
  dim3 grid(tiles_h * tiles_w, g.n);
  cudaError_t e;
  if (dt == DC_BF16) {
    auto k = k1_fused_sample<__nv_bfloat16>;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k<<<grid, kThreads, smem, s>>>(a, tiles_w, cc, mc);
    note_launches(1);
  } else {
    auto k = k1_fused_sample<float>;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k<<<grid, kThreads, smem, s>>>(a, tiles_w, cc, mc);
    note_launches(1);
  }
  return cudaGetLastError();
}

}  // namespace dc
