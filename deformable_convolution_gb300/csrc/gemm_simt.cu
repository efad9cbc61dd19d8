// Main-convolution GEMMs on CUDA cores (fp32 arithmetic).
//
// Explainer page "DefT: Boosting Scalability of Deformable Convolution
// Operations on GPUs", "The argument in one glance / This paper's idea": the
// main convolution over the deformed map stays a plain dense GEMM.  With the
// column layout [kdim][image][pixel]:
//   forward  y[b][o][q]     = sum_r w[o][r] * col[r][b][q]
//   backward gcol[r][b][q]  = sum_o w[o][r] * gy[b][o][q]
//            gw[o][r]      += sum_{b,q} gy[b][o][q] * col[r][b][q]
// This file serves the shapes whose rows are not 16-byte aligned, float32
// (C_in * K or Ho * Wo not a multiple of 4) and bf16 (not a multiple of 8);
// other problems use the tcgen05 kernels of gemm_tc.cu (bf16) and
// gemm_tf32.cu (float32, three-product TF32 split).
#include "dc_common.cuh"

namespace dc {
namespace {

constexpr int BM = 64, BN = 64, BK = 16, TM = 4, TN = 4;
constexpr int kThreads = (BM / TM) * (BN / TN);  // 256

// C[m][nn] = sum_k A(m, k) * B(k, nn), one batch entry per blockIdx.z.
// Element (m, k) of A is at A + z*a_z + m*a_m + k*a_k; likewise B and C.
struct StridedGemm {
  int M, N, K;
  long long a_z, a_m, a_k;
  long long b_z, b_k, b_n;
  long long c_z, c_m, c_n;
  int atomic;  // 1: atomically add fp32 into C, 0: store
  ZeroArgs zero;  // buffers this launch clears as a side job (GCOL)
  int ksplit;     // K ranges per batch entry along blockIdx.z (needs atomic when > 1)
  int relu;       // stores only: max(value, 0), NaN kept (the forward's fused activation)
};

template <typename TA, typename TB, typename TC>
__global__ void __launch_bounds__(kThreads)
    gemm_simt_kernel(StridedGemm p, const TA* __restrict__ A, const TB* __restrict__ B, TC* C) {
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  const int ks = p.ksplit > 1 ? p.ksplit : 1;
  const int z = blockIdx.z / ks;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  // this CTA's K range (whole BK blocks)
  const int kchunk = (int)ceil_div_ll(ceil_div_ll(p.K, ks), BK) * BK;
  const int k_begin = (int)(blockIdx.z % ks) * kchunk;
  const int k_end = min(p.K, k_begin + kchunk);
  {
    const long long nparts = (long long)gridDim.x * gridDim.y * gridDim.z;
    const long long part = blockIdx.x + (long long)gridDim.x * (blockIdx.y + (long long)gridDim.y * blockIdx.z);
    zero_share(p.zero, part, nparts, threadIdx.x, kThreads);
  }
  const TA* Az = A + (long long)z * p.a_z;
  const TB* Bz = B + (long long)z * p.b_z;
  const int tid = threadIdx.x;
  const int tr = tid / (BN / TN), tc = tid % (BN / TN);
  float acc[TM][TN];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TN; ++j) acc[i][j] = 0.0f;

  for (int k0 = k_begin; k0 < k_end; k0 += BK) {
    // stage A tile (BM x BK) and B tile (BK x BN); lanes run along whichever
    // index is contiguous in memory
    for (int idx = tid; idx < BM * BK; idx += kThreads) {
      int mm, kk;
      if (p.a_m == 1) { mm = idx % BM; kk = idx / BM; } else { kk = idx % BK; mm = idx / BK; }
      const int m = m0 + mm, k = k0 + kk;
      As[kk][mm] = (m < p.M && k < k_end) ? ld_f(Az + m * p.a_m + k * p.a_k) : 0.0f;
    }
    for (int idx = tid; idx < BK * BN; idx += kThreads) {
      int nn, kk;
      if (p.b_n == 1) { nn = idx % BN; kk = idx / BN; } else { kk = idx % BK; nn = idx / BK; }
      const int nidx = n0 + nn, k = k0 + kk;
      Bs[kk][nn] = (nidx < p.N && k < k_end) ? ld_f(Bz + k * p.b_k + nidx * p.b_n) : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float av[TM], bv[TN];
#pragma unroll
      for (int i = 0; i < TM; ++i) av[i] = As[kk][tr * TM + i];
#pragma unroll
      for (int j = 0; j < TN; ++j) bv[j] = Bs[kk][tc * TN + j];
#pragma unroll
      for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = __fmaf_rn(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
  TC* Cz = C + (long long)z * p.c_z;
#pragma unroll
  for (int i = 0; i < TM; ++i) {
    const int m = m0 + tr * TM + i;
    if (m >= p.M) continue;
#pragma unroll
    for (int j = 0; j < TN; ++j) {
      const int nidx = n0 + tc * TN + j;
      if (nidx >= p.N) continue;
      TC* dst = Cz + m * p.c_m + nidx * p.c_n;
      if (p.atomic) {
        atomicAdd(reinterpret_cast<float*>(dst), acc[i][j]);
      } else {
        float v = acc[i][j];
        if (p.relu && !(v > 0.f) && v == v) v = 0.f;
        *dst = from_f<TC>(v);
      }
    }
  }
}

template <typename TA, typename TB, typename TC>
cudaError_t run(const StridedGemm& p, int batch, const void* A, const void* B, void* C,
                cudaStream_t s) {
  if (p.M <= 0 || p.N <= 0 || batch <= 0) return cudaSuccess;
  const int ks = p.ksplit > 1 ? p.ksplit : 1;
  dim3 grid((unsigned)ceil_div_ll(p.N, BN), (unsigned)ceil_div_ll(p.M, BM), (unsigned)(batch * ks));
  gemm_simt_kernel<TA, TB, TC><<<grid, kThreads, 0, s>>>(
      p, static_cast<const TA*>(A), static_cast<const TB*>(B), static_cast<TC*>(C));
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_fwd_simt(const GemmArgs& a, dc_dtype dt, cudaStream_t s) {
  const Geom& g = a.g;
  StridedGemm p{};
  p.M = g.c_out; p.N = (int)g.howo; p.K = g.kdim;
  p.a_z = 0; p.a_m = g.kdim; p.a_k = 1;
  p.b_z = a.col_layout.img; p.b_k = a.col_layout.row; p.b_n = 1;
  p.c_z = (long long)g.c_out * g.howo; p.c_m = g.howo; p.c_n = 1;
  p.atomic = 0;
  p.relu = g.relu;
  if (dt == DC_BF16)
    return run<__nv_bfloat16, __nv_bfloat16, __nv_bfloat16>(p, g.n, a.w, a.col, a.y, s);
  return run<float, float, float>(p, g.n, a.w, a.col, a.y, s);
}

cudaError_t launch_gemm_gcol_simt(const GemmArgs& a, dc_dtype dt, cudaStream_t s) {
  const Geom& g = a.g;
  StridedGemm p{};
  p.M = g.kdim; p.N = (int)g.howo; p.K = g.c_out;
  p.a_z = 0; p.a_m = 1; p.a_k = g.kdim;
  p.b_z = (long long)g.c_out * g.howo; p.b_k = g.howo; p.b_n = 1;
  p.c_z = a.gcol_layout.img; p.c_m = a.gcol_layout.row; p.c_n = 1;
  p.atomic = 0;
  p.zero = a.zero;
  if (dt == DC_BF16)
    return run<__nv_bfloat16, __nv_bfloat16, float>(p, g.n, a.w, a.gy, a.gcol, s);
  return run<float, float, float>(p, g.n, a.w, a.gy, a.gcol, s);
}

cudaError_t launch_gemm_gw_simt(const GemmArgs& a, dc_dtype dt, cudaStream_t s) {
  // gw[o][r] += sum_q gy[b][o][q] * col[r][b][q]; batch entries (images) are
  // reduced with fp32 atomics into the zeroed gw.
  const Geom& g = a.g;
  StridedGemm p{};
  p.M = g.c_out; p.N = g.kdim; p.K = (int)g.howo;
  p.a_z = (long long)g.c_out * g.howo; p.a_m = g.howo; p.a_k = 1;
  p.b_z = a.col_layout.img; p.b_k = 1; p.b_n = a.col_layout.row;
  p.c_z = 0; p.c_m = g.kdim; p.c_n = 1;
  p.atomic = 1;
  // split the pixel reduction until about two CTAs per SM run (at least 128
  // pixels per CTA): small problems would otherwise leave most SMs idle
  {
    const long long tiles = ceil_div_ll(p.N, BN) * ceil_div_ll(p.M, BM) * g.n;
    long long ks = ceil_div_ll(304, tiles);
    const long long kmax = p.K / 128 > 1 ? p.K / 128 : 1;
    if (ks > kmax) ks = kmax;
    if (ks < 1) ks = 1;
    p.ksplit = (int)ks;
  }
  if (dt == DC_BF16)
    return run<__nv_bfloat16, __nv_bfloat16, float>(p, g.n, a.gy, a.col, a.gw, s);
  return run<float, float, float>(p, g.n, a.gy, a.col, a.gw, s);
}

}  // namespace dc
