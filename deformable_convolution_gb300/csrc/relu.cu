// ReLU between stacked deformable layers, forward and backward.
//
// Explainer page "DefT: Boosting Scalability of Deformable Convolution
// Operations on GPUs", "What people did before, and where it broke" (adding
// deformable layers throughout a ResNet) and "Why it works / Fixing the
// slowest stage lifts the whole layer" (training time of a fully deformable
// ResNet): the layers of such a network are separated by ReLU activations,
// so a training step over a stack of layers needs the activation and its
// gradient between them.  Both are pure streams over HBM: 16-byte loads and
// stores, a grid of a few CTAs per SM striding over the tensor.
#include "dc_common.cuh"

namespace dc {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;  // 16-byte vectors per thread in flight

// +0 where the value is <= 0, else the value: NaN stays NaN (it is not <= 0),
// as a training run wants it to; the hardware may return its canonical NaN.
__device__ __forceinline__ float relu1(float v) {
  return __uint_as_float(v <= 0.f ? 0u : __float_as_uint(v));
}
__device__ __forceinline__ __nv_bfloat16 relu1(__nv_bfloat16 v) {
  const unsigned short b = *reinterpret_cast<const unsigned short*>(&v);
  const unsigned short r = __uint_as_float((uint32_t)b << 16) <= 0.f ? (unsigned short)0 : b;
  return *reinterpret_cast<const __nv_bfloat16*>(&r);
}

// out = max(y, 0) elementwise (NaN stays NaN); out may be y.  Whole 16-byte
// chunks are vectorised, the last count % (16 / sizeof(T)) elements are not.
template <typename T>
__global__ void __launch_bounds__(kThreads, 6) relu_fwd_kernel(const T* y, T* out,
                                                            long long count) {
  pdl_wait();
  constexpr int kVec = 16 / sizeof(T);
  const long long nvec = count / kVec;
  const long long stride = (long long)gridDim.x * blockDim.x;
  const long long t0 = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  // kUnroll vectors per thread in flight at once (loads first, then stores)
  for (long long i0 = t0; i0 < nvec; i0 += kUnroll * stride) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const long long i = i0 + u * stride;
      if (i < nvec) v[u] = reinterpret_cast<const uint4*>(y)[i];
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const long long i = i0 + u * stride;
      if (i >= nvec) break;
      uint32_t* w = reinterpret_cast<uint32_t*>(&v[u]);
      if (sizeof(T) == 2) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          // compare the floats the two bf16 halves widen to; keep a half's
          // bits unless it is <= 0 (so NaN is kept)
          const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xffff0000u);
          w[e] = (lo <= 0.f ? 0u : (w[e] & 0xffffu)) | (hi <= 0.f ? 0u : (w[e] & 0xffff0000u));
        }
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) w[e] = __uint_as_float(w[e]) <= 0.f ? 0u : w[e];
      }
      reinterpret_cast<uint4*>(out)[i] = v[u];
    }
  }
  for (long long i = nvec * kVec + t0; i < count; i += stride) out[i] = relu1(y[i]);
  pdl_release();
}

// grad_in = grad_out where act > 0, else 0, rounded to T (nearest even).
// act is the activation's output (positive exactly where its input was).
template <typename T>
__global__ void __launch_bounds__(kThreads, 6) relu_bwd_kernel(const T* __restrict__ act,
                                                            const float* __restrict__ gout,
                                                            T* __restrict__ gin, long long count) {
  pdl_wait();
  const long long nvec = count / 8;
  const long long stride = (long long)gridDim.x * blockDim.x;
  const long long t0 = (long long)blockIdx.x * blockDim.x + threadIdx.x;
#pragma unroll 2
  for (long long i = t0; i < nvec; i += stride) {
    const float4 g0 = reinterpret_cast<const float4*>(gout)[2 * i];
    const float4 g1 = reinterpret_cast<const float4*>(gout)[2 * i + 1];
    const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
    float a[8];
    if (sizeof(T) == 2) {
      const uint4 v = reinterpret_cast<const uint4*>(act)[i];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        a[2 * e] = __uint_as_float(w[e] << 16);
        a[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
      }
    } else {
      const float4 v0 = reinterpret_cast<const float4*>(act)[2 * i];
      const float4 v1 = reinterpret_cast<const float4*>(act)[2 * i + 1];
      a[0] = v0.x; a[1] = v0.y; a[2] = v0.z; a[3] = v0.w;
      a[4] = v1.x; a[5] = v1.y; a[6] = v1.z; a[7] = v1.w;
    }
    if (sizeof(T) == 2) {
      uint4 o;
      uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        __nv_bfloat162 b2 = __floats2bfloat162_rn(a[2 * e] > 0.f ? g[2 * e] : 0.f,
                                                  a[2 * e + 1] > 0.f ? g[2 * e + 1] : 0.f);
        ow[e] = *reinterpret_cast<uint32_t*>(&b2);
      }
      reinterpret_cast<uint4*>(gin)[i] = o;
    } else {
      float o[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = a[e] > 0.f ? g[e] : 0.f;
      reinterpret_cast<float4*>(gin)[2 * i] = make_float4(o[0], o[1], o[2], o[3]);
      reinterpret_cast<float4*>(gin)[2 * i + 1] = make_float4(o[4], o[5], o[6], o[7]);
    }
  }
  for (long long i = nvec * 8 + t0; i < count; i += stride)
    gin[i] = from_f<T>(to_f(act[i]) > 0.f ? gout[i] : 0.f);
  pdl_release();
}

template <typename K, typename... A>
cudaError_t launch_stream_kernel(K kern, long long count, cudaStream_t s, A... args) {
  int sms = 0, dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // 8 CTAs of 256 threads per SM (the SM's full 2048 threads), fewer for
  // small tensors
  long long blocks = ceil_div_ll(ceil_div_ll(count, 8), kThreads);
  if (blocks > 8LL * sms) blocks = 8LL * sms;
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
  e = cudaLaunchKernelEx(&cfg, kern, args..., count);
  note_launches(1);
  return e;
}

}  // namespace

cudaError_t launch_relu_fwd(const void* y, void* out, long long count, dc_dtype dt,
                            cudaStream_t s) {
  if (dt == DC_BF16)
    return launch_stream_kernel(relu_fwd_kernel<__nv_bfloat16>, count, s,
                                static_cast<const __nv_bfloat16*>(y), static_cast<__nv_bfloat16*>(out));
  return launch_stream_kernel(relu_fwd_kernel<float>, count, s, static_cast<const float*>(y),
                              static_cast<float*>(out));
}

cudaError_t launch_relu_bwd(const void* act, const float* gout, void* gin, long long count,
                            dc_dtype dt, cudaStream_t s) {
  if (dt == DC_BF16)
    return launch_stream_kernel(relu_bwd_kernel<__nv_bfloat16>, count, s,
                                static_cast<const __nv_bfloat16*>(act), gout,
                                static_cast<__nv_bfloat16*>(gin));
  return launch_stream_kernel(relu_bwd_kernel<float>, count, s, static_cast<const float*>(act), gout,
                              static_cast<float*>(gin));
}

}  // namespace dc
