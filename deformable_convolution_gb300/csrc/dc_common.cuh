// Shared definitions of the CUDA library (device helpers, derived geometry,
// kernel launch entry points).  Nothing here is visible through the C ABI.
#pragma once

#include <climits>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "deform_conv.h"

namespace dc {

// Layer geometry with the derived sizes every kernel needs.
struct Geom {
  int n, c_in, h, w, c_out, kh, kw;
  int sh, sw, ph, pw, dh, dw;
  int groups;
  int ho, wo;
  int K;     // taps per filter, kh * kw
  int M;     // offset channels, 2 * groups * K
  int cg;    // input channels per offset group
  int kdim;  // main-GEMM reduction length, c_in * K
  long long hw, howo;
  int relu;  // forward: the main GEMM's epilogue writes max(y, 0) (NaN kept)
  int in_relu;  // backward: grad_x masked by x > 0 and written in the problem dtype
};

// Pitches of the deformed map ("column") buffer [kdim][n][howo(+pad)]:
// element (row r, image b, pixel q) lives at r * row + b * img + q.
struct ColLayout {
  long long row;
  long long img;
};

__host__ __device__ inline long long ceil_div_ll(long long a, long long b) {
  return (a + b - 1) / b;
}

__device__ __forceinline__ float ld_f(const float* p) { return *p; }
__device__ __forceinline__ float ld_f(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}
__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T>
__device__ __forceinline__ T from_f(float v);
template <>
__device__ __forceinline__ float from_f<float>(float v) {
  return v;
}
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// Bilinear blend of the four corners around a fractional point ("Why it fell
// short": four neighbouring pixels averaged by weight).  Every caller goes
// through this one sequence of roundings, so the on-chip and global-memory
// paths of a kernel give bitwise identical samples.
__device__ __forceinline__ float blend4(float ly, float lx, float v00, float v01,
                                        float v10, float v11) {
  const float hy = 1.0f - ly, hx = 1.0f - lx;
  float s = __fmul_rn(__fmul_rn(hy, hx), v00);
  s = __fmaf_rn(__fmul_rn(hy, lx), v01, s);
  s = __fmaf_rn(__fmul_rn(ly, hx), v10, s);
  s = __fmaf_rn(__fmul_rn(ly, lx), v11, s);
  return s;
}

// A sampling point can touch the image only if -1 <= p < extent on both axes
// (p = -1 still gives the right-sided derivative a nonzero value at row 0);
// outside, the sample and both of its derivatives are zero.  NaN is outside.
__device__ __forceinline__ bool touches_image(float py, float px, int H, int W) {
  return py >= -1.0f && py < (float)H && px >= -1.0f && px < (float)W;
}

// Programmatic dependent launch.  A kernel launched with the programmatic
// stream serialization attribute may start while its predecessor on the
// stream is finishing; it must call pdl_wait() before touching anything the
// predecessor writes (or reads and this kernel overwrites).  pdl_wait() is a
// no-op for kernels launched without the attribute.  pdl_release() lets this
// kernel's own dependent start its prologue; every kernel calls it only after
// its own pdl_wait(), so a dependent's prologue may read anything produced two
// or more launches earlier.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_release() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- launchers
// All return the launch's cudaError_t; the ABI layer maps it to a status.

// Host-side count of kernels enqueued by this library (dc_launch_count).
void note_launches(unsigned n);

struct SampleArgs {
  Geom g;
  const void* x;
  const void* w_off;
  const float* b_off;
  const float* off_add;
  const float* off_in;  // non-null: sample these offsets, skip the offset conv
  void* col;
  ColLayout col_layout;
  float* off_out;  // may be null: offsets are then kept on chip only
  unsigned long long* slow_count;
  int margin;
};
cudaError_t launch_sample(const SampleArgs& a, dc_dtype dt, cudaStream_t s);
size_t sample_smem_bytes(const Geom& g, dc_dtype dt, int margin);
// band (output rows R x columns TW) the fused stage tiles with at this margin
void sample_band(const Geom& g, dc_dtype dt, int margin, int* R, int* TW);

// Buffers a kernel zeroes as a side job (up to six float arrays); CTA `part`
// of `nparts` clears its share of each, float4 where aligned.
struct ZeroArgs {
  float* p[6];
  long long n[6];
};

__device__ __forceinline__ void zero_share(const ZeroArgs& z, long long part, long long nparts,
                                           int tid, int nthreads) {
#pragma unroll
  for (int i = 0; i < 6; ++i) {
    if (!z.p[i] || z.n[i] <= 0) continue;
    const long long chunk = (ceil_div_ll(z.n[i], nparts) + 3) / 4 * 4;
    const long long lo = part * chunk;
    long long hi = lo + chunk;
    if (hi > z.n[i]) hi = z.n[i];
    float* p = z.p[i];
    long long e = lo + 4LL * tid;
    for (; e + 4 <= hi; e += 4LL * nthreads)
      *reinterpret_cast<float4*>(p + e) = make_float4(0.f, 0.f, 0.f, 0.f);
    for (; e < hi; ++e) p[e] = 0.f;
  }
}

// Main-convolution GEMMs on the column layout (batched over images).
struct GemmArgs {
  Geom g;
  const void* w;      // [c_out][kdim]
  const void* col;    // column buffer, dtype
  ColLayout col_layout;
  const void* gy;     // [n][c_out][howo], dtype
  void* y;            // [n][c_out][howo], dtype (forward)
  void* gcol;         // column-layout gradient: bf16 from the tensor-core GEMM, else fp32
  ColLayout gcol_layout;
  float* gw;          // [c_out][kdim] fp32, accumulated with atomics (backward)
  float* gw_perm;     // channels-last GW: when given, the gradient is added in w' order
                      // ([c_out][tap][c], float4 atomics) here instead of into gw
  ZeroArgs zero;      // GCOL kernels clear these (the backward's atomic targets)
  float* gmax;        // tensor-core GCOL: max |gcol| per 128 x 128 tile (4 floats each), or null
  // tensor-core GW: after K4, gw_off = sum over images of gwo_img (count
  // floats per image, in the order of gwo_frag_dest4); null = nothing to reduce
  const float* gwo_img;
  float* gw_off;
  long long gwo_count;
};
// Tensor-core (tcgen05, bf16) versions; need tc_gemm_supported(g).
bool tc_gemm_supported(const Geom& g);
cudaError_t launch_gemm_fwd_tc(const GemmArgs& a, cudaStream_t s);
cudaError_t launch_gemm_gcol_tc(const GemmArgs& a, cudaStream_t s);
cudaError_t launch_gemm_gw_tc(const GemmArgs& a, cudaStream_t s);
// The same on the pixel-major map (channels-last path): `w` is w'[o][tap][c],
// `col` / `gcol` are col[n][pixel][tap][c]; GW writes grad_w[o][c][tap].
cudaError_t launch_gemm_fwd_cl(const GemmArgs& a, cudaStream_t s);
cudaError_t launch_gemm_gcol_cl(const GemmArgs& a, cudaStream_t s);
cudaError_t launch_gemm_gw_cl(const GemmArgs& a, cudaStream_t s);
// Forward GEMM with its B operand sampled in shared memory from x and the
// offsets (bf16, tensor cores; no column buffer): y = w * map(x, off).
bool fwd_sampled_supported(const Geom& g);
cudaError_t launch_fwd_sampled_tc(const Geom& g, const void* x, const void* w, const float* off,
                                  void* y, cudaStream_t s);
// float32 problems on the tensor cores (tcgen05 kind::tf32, three-product
// split); need tf32_gemm_supported(g): kdim and the pixel count multiples of 4.
bool tf32_gemm_supported(const Geom& g);
cudaError_t launch_gemm_fwd_tf32(const GemmArgs& a, cudaStream_t s);
cudaError_t launch_gemm_gcol_tf32(const GemmArgs& a, cudaStream_t s);
cudaError_t launch_gemm_gw_tf32(const GemmArgs& a, cudaStream_t s);
// CUDA-core (fp32 arithmetic) versions, any layout pitch.
cudaError_t launch_gemm_fwd_simt(const GemmArgs& a, dc_dtype dt, cudaStream_t s);
cudaError_t launch_gemm_gcol_simt(const GemmArgs& a, dc_dtype dt, cudaStream_t s);
cudaError_t launch_gemm_gw_simt(const GemmArgs& a, dc_dtype dt, cudaStream_t s);

// Backward of the sampling step (K3): grad_x and the offset gradient goff
// (float atomics into buffers cleared beforehand) and the replayed deformed map.
struct BwdArgs {
  Geom g;
  const void* x;
  const float* off;
  const void* gcol;  // bf16 when gmax is given (tensor-core GCOL), else fp32
  ColLayout gcol_layout;
  void* col;  // may be null: deformed map not written
  ColLayout col_layout;
  float* gx;
  float* goff;
  int margin;
  // max |gcol| per 128 x 128 tile of the GCOL GEMM (4 floats per tile, tiles
  // [image][row tile][pixel tile]); when given, K3 accumulates its grad_x window
  // in fixed point scaled from it, else in float
  const float* gmax;
  int gmax_tx, gmax_ty;  // pixel tiles per image, row tiles
};
cudaError_t launch_band_bwd(const BwdArgs& a, dc_dtype dt, cudaStream_t s);
size_t bwd_smem_bytes(const Geom& g, dc_dtype dt, int margin);

// Backward of the offset convolution (K4) from the completed goff: adds into
// grad_x, grad_w_off and grad_b_off (cleared beforehand).
struct OffconvBwdArgs {
  Geom g;
  const void* x;
  const void* w_off;
  const float* goff;
  float* gx;
  float* gw_off;
  float* gb_off;  // may be null
  // tensor-core kernel: per-image partial sums of grad_w_off, gwo_frag_count
  // floats per image in the order below (cleared by GCOL), reduced into gw_off
  // by the grad_W GEMM's tail or launch_gw_off_reduce
  float* gw_off_img;
};

// The tensor-core K4 adds its grad_w_off partials in the order of its mma
// accumulators, [channel slice of 16][tap][offset-channel tile of 8][lane][4],
// so that a warp's partial of one tile is 512 contiguous bytes (one 16-byte
// atomic per lane) instead of 32 scattered floats per instruction.
constexpr int kGwoSlice = 16;

__host__ __device__ inline long long gwo_frag_count(int M, int c_in, int K) {
  return (long long)((c_in + kGwoSlice - 1) / kGwoSlice) * K * ((M + 7) / 8) * 128;
}

// grad_w_off [M][C_in][K] indices of the four elements 4 * e4 .. 4 * e4 + 3
// of that order (one lane's accumulator tile); -1 for the padding (offset
// channel >= M or input channel >= C_in).  Accumulator element h of lane l
// holds row (l >> 2) + 8 * (h >> 1) (the channel within the slice) and column
// 2 * (l & 3) + (h & 1) (the offset channel within the tile).  32-bit index
// arithmetic: one image's partials are far below 2^31 floats.
__host__ __device__ inline void gwo_frag_dest4(int e4, int M, int c_in, int K, long long d[4]) {
  const int lane = e4 & 31, r = e4 >> 5;
  const int mtiles = (M + 7) / 8;
  const int sk = r / mtiles, mt = r - sk * mtiles;
  const int slice = sk / K, k = sk - slice * K;
  const int m0 = mt * 8 + 2 * (lane & 3);
  const int c0 = slice * kGwoSlice + (lane >> 2);
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    const int m = m0 + (h & 1), c = c0 + 8 * (h >> 1);
    d[h] = (m < M && c < c_in) ? ((long long)m * c_in + c) * K + k : -1;
  }
}
cudaError_t launch_offconv_bwd(const OffconvBwdArgs& a, dc_dtype dt, cudaStream_t s);
size_t offconv_bwd_smem_bytes(const Geom& g, dc_dtype dt);
// histogram of the margin each sampling tap needs (DC_MARGIN_BINS bins)
cudaError_t launch_margin_histogram(const float* offset, const Geom& g, int R, int TW,
                                    unsigned long long* hist, cudaStream_t s);
// tensor-core variant (bf16, few offset channels), chosen by launch_offconv_bwd
bool offconv_bwd_tc_supported(const Geom& g, dc_dtype dt);
size_t offconv_bwd_tc_smem_bytes(const Geom& g);
cudaError_t launch_offconv_bwd_tc(const OffconvBwdArgs& a, cudaStream_t s);
// gw_off = sum over images of gw_off_img (launched after the grad_W GEMM)
cudaError_t launch_gw_off_reduce(const OffconvBwdArgs& a, cudaStream_t s);

// ---------------------------------------------------------------- channels-last path
// bf16 problems with C_in % 64 == 0 (C_in <= 256), 8 | C_in / G, H*W % 8 == 0
// and the tensor-core GEMMs' alignment run on x copied to NHWC and a
// pixel-major deformed map col[n][pixel][tap][channel] (row = n*Ho*Wo + pixel,
// kdim = K*C_in elements per row, tap-major); the main weights are permuted
// to w'[o][tap][channel] to match.
bool cl_supported(const Geom& g, dc_dtype dt, int margin);
void cl_tile(const Geom& g, int margin, int* th, int* tw);  // output tile of the sampling stage
size_t cl_wfrag_bytes(const Geom& g);  // w_off in mma B-fragment order
struct ClArgs {
  Geom g;
  const void* xc;      // x, NHWC bf16
  const void* wfrag;   // launch_cl_prep_woff's output (ignored in replay mode)
  const float* b_off;
  const float* off_add;
  const float* off_in;  // non-null: sample these offsets (replay), no offset convolution
  void* col;            // pixel-major deformed map, or null: offsets only
  float* off_out;
  unsigned long long* slow_count;
  int margin;
};
// In one launch: x (NCHW) to its NHWC copy xc; w [o][c][tap] -> w' [o][tap][c]
// (w non-null); w_off in mma B-fragment order (frag non-null).
cudaError_t launch_cl_prep(const void* x, void* xc, const void* w, void* wp, const void* w_off,
                           void* frag, const Geom& g, int margin, cudaStream_t s);
cudaError_t launch_cl_sample(const ClArgs& a, cudaStream_t s);
unsigned int cl_read_error(int clear);
// Backward of the sampling step on the channels-last path (one offset group):
// grad_x accumulated into an NHWC float32 buffer, the offset gradient into
// goff (both cleared beforehand); then launch_gx_to_nchw writes grad_x.
bool k3cl_supported(const Geom& g, dc_dtype dt, int margin);
struct K3ClArgs {
  Geom g;
  const void* xc;    // x, NHWC bf16
  const float* off;  // offsets [n][M][Ho][Wo]
  const void* gcol;  // pixel-major gradient of the deformed map, bf16
  float* gx_nhwc;    // [n][H][W][C_in] float32
  float* goff;
  int margin;
};
cudaError_t launch_k3cl(const K3ClArgs& a, cudaStream_t s);
cudaError_t launch_gx_to_nchw(const float* gx_nhwc, float* grad_x, const Geom& g, cudaStream_t s);
unsigned int cl3_read_error(int clear);
unsigned int tf32_read_error(int clear);
// Backward of the offset convolution on the channels-last path (one offset
// group, K <= 9 taps): the input part adds into the NHWC grad_x buffer's
// values and writes grad_x (NCHW) whole; the weight part writes per-chunk
// partial sums into `part` (k4cl_part_bytes), which the reduce kernel adds
// into grad_w_off and grad_b_off (overwritten).
bool k4cl_supported(const Geom& g);
size_t k4cl_part_bytes(const Geom& g);
struct K4ClArgs {
  Geom g;
  const void* xc;       // x, NHWC bf16
  const void* w_off;    // [M][C_in][K] bf16
  const float* goff;    // [n][M][Ho][Wo]
  const float* gx_nhwc; // the sampling backward's grad_x, NHWC float32
  const void* x;        // x, NCHW bf16 (the ReLU mask when g.in_relu)
  void* grad_x;         // [n][C_in][H][W] float32, or bf16 masked by x > 0 when g.in_relu
  float* grad_w_off;    // [M][C_in][K]
  float* grad_b_off;    // [M] or null
  float* part;          // workspace, k4cl_part_bytes
  const float* gw_perm; // grad_w in w' order [C_out][K][C_in] (the GEMM's), or null
  float* grad_w;        // [C_out][C_in][K], written from gw_perm by the reduce kernel
  int c_out;
};
cudaError_t launch_k4cl_input(const K4ClArgs& a, cudaStream_t s);
cudaError_t launch_k4cl_weight(const K4ClArgs& a, cudaStream_t s);
cudaError_t launch_k4cl_reduce(const K4ClArgs& a, cudaStream_t s);
unsigned int k4cl_read_error(int clear);
bool make_tmap_f32(CUtensorMap* m, const void* base, int rank, const unsigned long long* dims,
                   const unsigned long long* strides_bytes, const unsigned int* box);
bool make_tmap_bf16(CUtensorMap* m, const void* base, int rank, const unsigned long long* dims,
                    const unsigned long long* strides_bytes, const unsigned int* box,
                    bool swizzle128);

// ReLU between stacked layers: out = max(y, 0); gin = gout where act > 0
// (rounded to the dtype), else 0.  16-byte aligned pointers.
cudaError_t launch_relu_fwd(const void* y, void* out, long long count, dc_dtype dt, cudaStream_t s);
cudaError_t launch_relu_bwd(const void* act, const float* gout, void* gin, long long count,
                            dc_dtype dt, cudaStream_t s);

}  // namespace dc
