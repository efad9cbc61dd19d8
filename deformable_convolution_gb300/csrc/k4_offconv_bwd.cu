// K4: backward of the offset convolution ("Following a deformable layer
// through DefT", Step 1 of 5, on the explainer page "DefT: Boosting
// Scalability of Deformable Convolution Operations on GPUs": a small standard
// convolution over the same input).  With goff the gradient of its output:
//   grad_x[b][c][y][x] += sum_{m,i,j} goff[b][m][ho][wo] * w_off[m][c][i][j]
//                         over (ho, wo) with ho*sh - ph + i*dh = y, likewise x
//   grad_w_off[m][c][i][j] = sum_{b,q} goff[b][m][q] * xbar[b][c](tap (i,j) of q)
//   grad_b_off[m]          = sum_{b,q} goff[b][m][q]
#include "dc_common.cuh"

namespace dc {
namespace {

constexpr int kThreads = 256;

// grad_x += conv^T(goff, w_off); one thread per input element, gathering.
template <typename T>
__global__ void __launch_bounds__(kThreads) k4_input_grad(OffconvBwdArgs a) {
  const Geom g = a.g;
  const T* __restrict__ w_off = static_cast<const T*>(a.w_off);
  const long long total = (long long)g.n * g.c_in * g.hw;
  for (long long idx = (long long)blockIdx.x * kThreads + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * kThreads) {
    const int xx = (int)(idx % g.w);
    long long t = idx / g.w;
    const int yy = (int)(t % g.h);
    t /= g.h;
    const int c = (int)(t % g.c_in);
    const int b = (int)(t / g.c_in);
    float s = 0.0f;
    for (int i = 0; i < g.kh; ++i) {
      const int ny = yy + g.ph - i * g.dh;
      if (ny < 0 || ny % g.sh) continue;
      const int ho = ny / g.sh;
      if (ho >= g.ho) continue;
      for (int j = 0; j < g.kw; ++j) {
        const int nx = xx + g.pw - j * g.dw;
        if (nx < 0 || nx % g.sw) continue;
        const int wo = nx / g.sw;
        if (wo >= g.wo) continue;
        const float* gp = a.goff + (long long)b * g.M * g.howo + (long long)ho * g.wo + wo;
        const T* wp = w_off + ((long long)c * g.kh + i) * g.kw + j;
        for (int m = 0; m < g.M; ++m)
          s = __fmaf_rn(gp[(long long)m * g.howo], ld_f(wp + (long long)m * g.c_in * g.K), s);
      }
    }
    a.gx[idx] += s;
  }
}

// grad_w_off and grad_b_off: one block per (m, c) reduces over all images and
// output pixels for the K taps at once.
template <typename T>
__global__ void __launch_bounds__(kThreads) k4_weight_grad(OffconvBwdArgs a) {
  const Geom g = a.g;
  const T* __restrict__ x = static_cast<const T*>(a.x);
  const int m = blockIdx.x / g.c_in;
  const int c = blockIdx.x % g.c_in;
  constexpr int kMaxTaps = 49;
  float acc[kMaxTaps];
  for (int k = 0; k < kMaxTaps; ++k) acc[k] = 0.0f;
  float bias = 0.0f;
  const long long total = (long long)g.n * g.howo;
  for (long long idx = threadIdx.x; idx < total; idx += kThreads) {
    const int b = (int)(idx / g.howo);
    const long long q = idx % g.howo;
    const int ho = (int)(q / g.wo), wo = (int)(q % g.wo);
    const float go = a.goff[((long long)b * g.M + m) * g.howo + q];
    bias += go;
    const T* plane = x + ((long long)b * g.c_in + c) * g.hw;
    for (int i = 0; i < g.kh; ++i) {
      const int yy = ho * g.sh - g.ph + i * g.dh;
      const bool rin = yy >= 0 && yy < g.h;
      for (int j = 0; j < g.kw; ++j) {
        const int xx = wo * g.sw - g.pw + j * g.dw;
        const float v = (rin && xx >= 0 && xx < g.w) ? ld_f(plane + (long long)yy * g.w + xx) : 0.0f;
        acc[i * g.kw + j] = __fmaf_rn(go, v, acc[i * g.kw + j]);
      }
    }
  }
  __shared__ float red[kThreads / 32];
  for (int k = 0; k <= g.K; ++k) {
    float v = k < g.K ? acc[k] : bias;
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    if (threadIdx.x == 0) {
      float s = 0.0f;
      for (int w = 0; w < kThreads / 32; ++w) s += red[w];
      if (k < g.K)
        a.gw_off[((long long)m * g.c_in + c) * g.K + k] = s;
      else if (a.gb_off && c == 0)
        a.gb_off[m] = s;
    }
  }
}

}  // namespace

cudaError_t launch_offconv_bwd(const OffconvBwdArgs& a, dc_dtype dt, cudaStream_t s) {
  const Geom& g = a.g;
  long long blocks = ceil_div_ll((long long)g.n * g.c_in * g.hw, kThreads);
  if (blocks > 152LL * 16) blocks = 152LL * 16;
  const unsigned wblocks = (unsigned)(g.M * g.c_in);
  if (dt == DC_BF16) {
    k4_input_grad<__nv_bfloat16><<<(unsigned)blocks, kThreads, 0, s>>>(a);
    k4_weight_grad<__nv_bfloat16><<<wblocks, kThreads, 0, s>>>(a);
  } else {
    k4_input_grad<float><<<(unsigned)blocks, kThreads, 0, s>>>(a);
    k4_weight_grad<float><<<wblocks, kThreads, 0, s>>>(a);
  }
  note_launches(2);
  return cudaGetLastError();
}

}  // namespace dc
