// Offset statistics for choosing the tile margin.
//
// The explainer page "DefT: Boosting Scalability of Deformable Convolution
// Operations on GPUs" pads each tile's input window by just enough margin for
// the offsets that occur, sized from their measured distribution ("Why it
// works", "The idea").  The band kernels take the margin as a plan parameter;
// this kernel measures, from the offsets a forward call returned, how much
// margin each sampling tap needs, as a histogram over whole pixels.
//
// A tap reads the rows floor(py) and floor(py) + 1 (columns likewise).  Its
// band stages the band's receptive field plus m pixels on each side, so the
// tap needs m >= the distance by which those rows and columns pass the
// field's edges.  The band is the one the fused stage uses for the problem
// (R output rows x TW columns at the problem's current margin).  Taps whose
// sampling point lies entirely outside the image read nothing and need no
// margin.  With margin m and the same band shape, exactly the taps of the bins
// above m take the slow path.
#include "dc_common.cuh"

namespace dc {
namespace {

constexpr int kBins = DC_MARGIN_BINS;
constexpr int kThreads = 256;

// extra pixels beyond [lo, lo + extent) that the pair (c, c + 1) needs
__device__ __forceinline__ int beyond(float p, int lo, int extent) {
  const float c = floorf(p);
  const float before = (float)lo - c, after = c + 2.0f - (float)(lo + extent);
  const float m = fmaxf(0.0f, fmaxf(before, after));
  return m >= (float)(kBins - 1) ? kBins - 1 : (int)m;
}

__global__ void __launch_bounds__(kThreads) margin_histogram(const float* __restrict__ off, Geom g,
                                                             int R, int TW,
                                                             unsigned long long* hist) {
  const int in_rows = (R - 1) * g.sh + (g.kh - 1) * g.dh + 1;
  const int in_cols = (TW - 1) * g.sw + (g.kw - 1) * g.dw + 1;
  __shared__ unsigned int h[kBins];
  for (int b = threadIdx.x; b < kBins; b += kThreads) h[b] = 0u;
  __syncthreads();
  const long long taps_per_img = (long long)g.groups * g.K * g.howo;
  const long long total = (long long)g.n * taps_per_img;
  for (long long t = blockIdx.x * (long long)kThreads + threadIdx.x; t < total;
       t += (long long)gridDim.x * kThreads) {
    const long long n = t / taps_per_img;
    const long long r = t - n * taps_per_img;
    const int gk = (int)(r / g.howo);
    const int q = (int)(r - (long long)gk * g.howo);
    const int k = gk % g.K;
    const int i = k / g.kw, j = k - i * g.kw;
    const int ho = q / g.wo, wo = q - ho * g.wo;
    const float* o = off + ((long long)n * g.M + 2 * gk) * g.howo + q;
    const float dy = o[0], dx = o[g.howo];
    const float py = (float)(ho * g.sh - g.ph + i * g.dh) + dy;
    const float px = (float)(wo * g.sw - g.pw + j * g.dw) + dx;
    int bin = 0;
    if (!(py == py) || !(px == px)) {
      bin = kBins - 1;
    } else if (touches_image(py, px, g.h, g.w)) {
      const int ylo = (ho / R) * R * g.sh - g.ph, xlo = (wo / TW) * TW * g.sw - g.pw;
      bin = max(beyond(py, ylo, in_rows), beyond(px, xlo, in_cols));
    }
    atomicAdd(&h[bin], 1u);
  }
  __syncthreads();
  for (int b = threadIdx.x; b < kBins; b += kThreads)
    if (h[b]) atomicAdd(hist + b, (unsigned long long)h[b]);
}

}  // namespace

cudaError_t launch_margin_histogram(const float* offset, const Geom& g, int R, int TW,
                                    unsigned long long* hist, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(hist, 0, kBins * sizeof(unsigned long long), s);
  if (e != cudaSuccess) return e;
  const long long total = (long long)g.n * g.groups * g.K * g.howo;
  long long blocks = (total + kThreads - 1) / kThreads;
  if (blocks > 152 * 8) blocks = 152 * 8;
  if (blocks < 1) blocks = 1;
  margin_histogram<<<(unsigned)blocks, kThreads, 0, s>>>(offset, g, R, TW, hist);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace dc
