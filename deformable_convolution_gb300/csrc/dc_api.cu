// The C ABI (include/deform_conv.h): argument checks, workspace plan and the
// launch sequences of the forward and backward passes.
//
// Forward ("The argument in one glance / This paper's idea" on the explainer
// page "DefT: Boosting Scalability of Deformable Convolution Operations on
// GPUs"): K1 fuses the offset convolution with the bilinear interpolation and
// writes the deformed map; the main convolution is a separate dense GEMM over
// that map.  Backward: a GEMM gives the deformed map's gradient (and clears
// the buffers the later kernels accumulate into); K3 scatters it into grad_x,
// accumulates the offset gradient and replays the deformed map; K4 runs the
// offset convolution's backward; a second GEMM gives the main weights'
// gradient from the replayed map.
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "dc_common.cuh"

namespace dc {

static std::atomic<unsigned long long> g_launches{0};
void note_launches(unsigned n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

// Per-launch timing (dc_kernel_timing): when enabled, every kernel the ABI
// enqueues is bracketed by two CUDA events on its stream; dc_kernel_times
// reads the records of the calls made since timing was (re)enabled.  Off by
// default; events are host/driver objects, no device memory is allocated.
namespace {
constexpr int kMaxTimed = 256;
struct TimedLaunch {
  const char* name;
  cudaEvent_t a, b;
};
std::mutex g_timing_mu;
std::atomic<bool> g_timing{false};  // read without the lock on every launch
TimedLaunch g_timed[kMaxTimed];
int g_ntimed = 0;
int g_nevents = 0;  // event pairs created so far (reused across calls)

// Test hook (dc_test_fail_launches): launches still to fail without being made.
std::atomic<int> g_fail_launches{0};

template <typename F>
cudaError_t timed(const char* name, cudaStream_t s, F&& launch) {
  if (g_fail_launches.load(std::memory_order_relaxed) > 0 &&
      g_fail_launches.fetch_sub(1, std::memory_order_relaxed) > 0)
    return cudaErrorLaunchFailure;  // injected: nothing is enqueued
  int slot = -1;
  if (g_timing.load(std::memory_order_relaxed)) {
    std::lock_guard<std::mutex> lock(g_timing_mu);
    if (g_timing.load(std::memory_order_relaxed) && g_ntimed < kMaxTimed) {
      slot = g_ntimed++;
      if (slot >= g_nevents) {
        if (cudaEventCreate(&g_timed[slot].a) != cudaSuccess ||
            cudaEventCreate(&g_timed[slot].b) != cudaSuccess)
          return cudaErrorUnknown;
        g_nevents = slot + 1;
      }
      g_timed[slot].name = name;
    }
  }
  if (slot >= 0) cudaEventRecord(g_timed[slot].a, s);
  const cudaError_t e = launch();
  if (slot >= 0) cudaEventRecord(g_timed[slot].b, s);
  return e;
}
}  // namespace

cudaError_t launch_gemm_fwd(const GemmArgs& a, dc_dtype dt, cudaStream_t s);
cudaError_t launch_gemm_gcol(const GemmArgs& a, dc_dtype dt, cudaStream_t s);
cudaError_t launch_gemm_gw(const GemmArgs& a, dc_dtype dt, cudaStream_t s);

namespace {

constexpr int kDefaultMargin = 3;
constexpr int kMaxMargin = 64;
constexpr int kMaxTaps = 49;
constexpr size_t kMaxSmem = 225 * 1024;  // dynamic shared memory per CTA on sm_103a is 227 KB

size_t elt_size(dc_dtype dt) { return dt == DC_BF16 ? 2 : 4; }

long long round_up(long long v, long long m) { return (v + m - 1) / m * m; }

dc_status make_geom(const dc_problem* p, Geom* g, int* margin) {
  if (!p) return DC_ERR_INVALID_ARG;
  if (p->n <= 0 || p->c_in <= 0 || p->h <= 0 || p->w <= 0 || p->c_out <= 0 || p->kh <= 0 ||
      p->kw <= 0 || p->stride_h <= 0 || p->stride_w <= 0 || p->pad_h < 0 || p->pad_w < 0 ||
      p->dil_h <= 0 || p->dil_w <= 0 || p->offset_groups <= 0 ||
      p->c_in % p->offset_groups != 0)
    return DC_ERR_INVALID_ARG;
  if (p->dtype != DC_F32 && p->dtype != DC_BF16) return DC_ERR_INVALID_ARG;
  if (p->halo_margin < -1) return DC_ERR_INVALID_ARG;
  if (p->out_relu != 0 && p->out_relu != 1) return DC_ERR_INVALID_ARG;
  if (p->in_relu != 0 && p->in_relu != 1) return DC_ERR_INVALID_ARG;
  const long long eh = (long long)p->h + 2LL * p->pad_h - (long long)p->dil_h * (p->kh - 1) - 1;
  const long long ew = (long long)p->w + 2LL * p->pad_w - (long long)p->dil_w * (p->kw - 1) - 1;
  if (eh < 0 || ew < 0) return DC_ERR_INVALID_ARG;
  g->n = p->n;
  g->c_in = p->c_in;
  g->h = p->h;
  g->w = p->w;
  g->c_out = p->c_out;
  g->kh = p->kh;
  g->kw = p->kw;
  g->sh = p->stride_h;
  g->sw = p->stride_w;
  g->ph = p->pad_h;
  g->pw = p->pad_w;
  g->dh = p->dil_h;
  g->dw = p->dil_w;
  g->groups = p->offset_groups;
  g->ho = (int)(eh / p->stride_h + 1);
  g->wo = (int)(ew / p->stride_w + 1);
  g->K = p->kh * p->kw;
  g->M = 2 * p->offset_groups * g->K;
  g->cg = p->c_in / p->offset_groups;
  g->kdim = p->c_in * g->K;
  g->hw = (long long)p->h * p->w;
  g->howo = (long long)g->ho * g->wo;
  g->relu = p->out_relu;
  g->in_relu = p->in_relu;
  // limits of this build
  if (g->K > kMaxTaps) return DC_ERR_UNSUPPORTED;
  if ((long long)p->c_in * g->K > (1LL << 30) || (long long)p->n * p->c_in * g->hw > (1LL << 40) ||
      g->howo * p->n > (1LL << 31))
    return DC_ERR_UNSUPPORTED;
  *margin = p->halo_margin < 0 ? kDefaultMargin : p->halo_margin;
  if (*margin > kMaxMargin) return DC_ERR_UNSUPPORTED;
  if (!cl_supported(*g, p->dtype, *margin) && sample_smem_bytes(*g, p->dtype, *margin) > kMaxSmem)
    return DC_ERR_UNSUPPORTED;
  return DC_OK;
}

// Workspace carve-up.  The column buffer keeps each image's pixel run padded
// to a multiple of 8 elements so that every row starts 16-byte aligned.
// The channels-last path (bf16, see cl_supported) adds x's NHWC copy, the
// permuted main weights and the fragment-ordered offset weights, and keeps
// the deformed map pixel-major (col[n][pixel][tap][channel], no padding).
struct Plan {
  bool cl;
  bool k3cl;  // channels-last sampling backward (pixel-major gcol, NHWC grad_x accumulator)
  bool k4cl;  // channels-last offset-convolution backward (writes grad_x from that accumulator)
  ColLayout col, gcol;
  size_t col_off, gcol_off, off_off, gmax_off, gwo_img_off, xc_off, wp_off, wfrag_off, gxc_off, k4part_off,
      gwp_off, gxr_off,
      total;
  int gmax_tx, gmax_ty;
};

Plan make_plan(const Geom& g, dc_dtype dt, int backward, int margin) {
  Plan pl{};
  pl.cl = cl_supported(g, dt, margin);
  pl.k3cl = backward && pl.cl && k3cl_supported(g, dt, margin);
  pl.k4cl = pl.k3cl && k4cl_supported(g);
  const long long pitch = round_up(g.howo, 8);
  pl.col.img = pitch;
  pl.col.row = pitch * g.n;
  pl.gcol = pl.col;
  size_t at = 0;
  auto take = [&](size_t bytes) {
    const size_t here = at;
    at = (size_t)round_up((long long)(at + bytes), 256);
    return here;
  };
  pl.col_off = take((size_t)g.kdim * pl.col.row * elt_size(dt));
  pl.off_off = take((size_t)g.n * g.M * g.howo * sizeof(float));
  if (pl.cl) {
    pl.xc_off = take((size_t)g.n * g.hw * g.c_in * 2);
    pl.wp_off = take((size_t)g.c_out * g.kdim * 2);
    pl.wfrag_off = take(cl_wfrag_bytes(g));
  }
  // gcol: bf16 from the tensor-core GEMM (K3 then scales it into fixed point),
  // fp32 from the CUDA-core GEMM
  const size_t gcol_elt = dt == DC_BF16 && tc_gemm_supported(g) ? 2 : sizeof(float);
  pl.gcol_off = backward ? take((size_t)g.kdim * pl.gcol.row * gcol_elt) : 0;
  // per-tile max |gcol| written by the tensor-core GCOL GEMM (128 x 128 tiles)
  pl.gmax_tx = (int)ceil_div_ll(g.howo, 128);
  pl.gmax_ty = (int)ceil_div_ll(g.kdim, 128);
  pl.gmax_off = backward ? take((size_t)g.n * pl.gmax_tx * pl.gmax_ty * 4 * sizeof(float)) : 0;
  // per-image grad_w_off partials of the tensor-core offset-conv backward
  // (one image's bands add into one copy: far fewer atomics per address), in
  // the kernel's accumulator order
  pl.gxc_off = pl.k3cl ? take((size_t)g.n * g.hw * g.c_in * sizeof(float)) : 0;
  pl.k4part_off = pl.k4cl ? take(k4cl_part_bytes(g)) : 0;
  // grad_w in w' order, permuted by the offset-convolution backward's reduce
  pl.gwp_off = pl.k4cl ? take((size_t)g.c_out * g.kdim * sizeof(float)) : 0;
  pl.gwo_img_off = backward && !pl.k4cl && offconv_bwd_tc_supported(g, dt)
                       ? take((size_t)g.n * gwo_frag_count(g.M, g.c_in, g.K) * sizeof(float))
                       : 0;
  // float32 grad_x ahead of the fused ReLU backward (in_relu) where the
  // kernels accumulate into grad_x itself; last, so the regions before it are
  // where the forward pass put them
  pl.gxr_off = backward && g.in_relu && !pl.k4cl ? take((size_t)g.n * g.c_in * g.hw * sizeof(float)) : 0;
  pl.total = at;
  return pl;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

dc_status cuda_status(cudaError_t e) { return e == cudaSuccess ? DC_OK : DC_ERR_CUDA; }

}  // namespace

namespace {
// The channels-last sampling stage: in one launch x to NHWC, the main weights
// permuted (when `w` is given) and w_off in mma fragment order (unless in
// replay mode); then K1 over the staged windows.
dc_status cl_stage(const Geom& g, int margin, const Plan& pl, char* wsb, const void* x,
                   const void* w_off, const void* w, const float* b_off, const float* off_add,
                   const float* off_in, void* col, float* off_out, unsigned long long* slow,
                   cudaStream_t s) {
  // x to NHWC and (unless replaying without new weights) the weight layouts
  const bool weights = !off_in || w;
  dc_status st = cuda_status(timed("cl_prep", s, [&] {
    return launch_cl_prep(x, wsb + pl.xc_off, weights ? w : nullptr, wsb + pl.wp_off, w_off,
                          weights && !off_in ? wsb + pl.wfrag_off : nullptr, g, margin, s);
  }));
  if (st != DC_OK) return st;
  ClArgs ca{};
  ca.g = g;
  ca.xc = wsb + pl.xc_off;
  ca.wfrag = wsb + pl.wfrag_off;
  ca.b_off = off_in ? nullptr : b_off;
  ca.off_add = off_in ? nullptr : off_add;
  ca.off_in = off_in;
  ca.col = col;
  ca.off_out = off_out;
  ca.slow_count = slow;
  ca.margin = margin;
  const char* name = col ? "k1_cl_sample" : "k1_cl_offsets";
  return cuda_status(timed(name, s, [&] { return launch_cl_sample(ca, s); }));
}
}  // namespace
}  // namespace dc

using namespace dc;

namespace dc {
namespace {

// The backward pass; with reuse_map the deformed map the forward pass left in
// the workspace feeds the weight-gradient GEMM and K3 does not replay it.
dc_status backward(const dc_problem* prob, const void* x, const void* w_off, const void* w,
                   const float* offset, const void* grad_y, void* grad_x, float* grad_w_off,
                   float* grad_b_off, float* grad_w, float* grad_offset, void* ws,
                   size_t ws_bytes, void* stream, bool reuse_map) {
  Geom g;
  int margin;
  dc_status st = make_geom(prob, &g, &margin);
  if (st != DC_OK) return st;
  if (!x || !w_off || !w || !offset || !grad_y || !grad_x || !grad_w_off || !grad_w)
    return DC_ERR_INVALID_ARG;
  if (bwd_smem_bytes(g, prob->dtype, margin) > kMaxSmem ||
      offconv_bwd_smem_bytes(g, prob->dtype) > kMaxSmem)
    return DC_ERR_UNSUPPORTED;
  const void* ptrs[] = {x, w_off, w, offset, grad_y, grad_x, grad_w_off, grad_b_off, grad_w,
                        grad_offset, ws};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return DC_ERR_UNSUPPORTED;
  const Plan pl = make_plan(g, prob->dtype, 1, margin);
  if (!ws || ws_bytes < pl.total) return DC_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* wsb = static_cast<char*>(ws);
  float* goff = grad_offset ? grad_offset : reinterpret_cast<float*>(wsb + pl.off_off);
  // float32 grad_x: the caller's buffer, or with in_relu the scratch the
  // ReLU backward reads at the end (the channels-last offset-convolution
  // backward applies it while writing grad_x and needs neither)
  float* gx32 = pl.gxr_off ? reinterpret_cast<float*>(wsb + pl.gxr_off) : static_cast<float*>(grad_x);
  if (pl.cl && !reuse_map) {
    // the pixel-major map for the weight-gradient GEMM, sampled at the given
    // offsets, and the permuted weights
    st = cl_stage(g, margin, pl, wsb, x, w_off, w, nullptr, nullptr, offset, wsb + pl.col_off,
                  nullptr, nullptr, s);
    if (st != DC_OK) return st;
  }

  // gradient of the deformed map: gcol = w^T grad_y
  GemmArgs ga{};
  ga.g = g;
  ga.w = w;
  ga.col = wsb + pl.col_off;
  ga.col_layout = pl.col;
  ga.gy = grad_y;
  ga.gcol = wsb + pl.gcol_off;
  ga.gcol_layout = pl.gcol;
  ga.gw = grad_w;
  // the GCOL launch also clears the buffers later kernels accumulate into (on
  // the channels-last path grad_x's NHWC accumulator: grad_x is written whole
  // from it)
  float* gxc = pl.k3cl ? reinterpret_cast<float*>(wsb + pl.gxc_off) : nullptr;
  if (pl.k3cl) ga.w = wsb + pl.wp_off;
  ga.zero.p[0] = pl.k3cl ? gxc : gx32;
  ga.zero.n[0] = (long long)g.n * g.c_in * g.hw;
  float* gw_perm = pl.k4cl ? reinterpret_cast<float*>(wsb + pl.gwp_off) : nullptr;
  ga.zero.p[1] = pl.k4cl ? gw_perm : grad_w;
  ga.zero.n[1] = (long long)g.c_out * g.kdim;
  ga.zero.p[2] = grad_w_off;
  ga.zero.n[2] = (long long)g.M * g.kdim;
  ga.zero.p[3] = grad_b_off;
  ga.zero.n[3] = grad_b_off ? g.M : 0;
  ga.zero.p[4] = goff;
  ga.zero.n[4] = (long long)g.n * g.M * g.howo;
  float* gwo_img = pl.gwo_img_off ? reinterpret_cast<float*>(wsb + pl.gwo_img_off) : nullptr;
  ga.zero.p[5] = gwo_img;
  ga.zero.n[5] = gwo_img ? (long long)g.n * gwo_frag_count(g.M, g.c_in, g.K) : 0;
  // the tensor-core GCOL GEMM also reports max |gcol| per tile, from which K3
  // scales its fixed-point grad_x accumulation
  const bool tc_gcol = prob->dtype == DC_BF16 && tc_gemm_supported(g);
  ga.gmax = tc_gcol && !pl.k3cl ? reinterpret_cast<float*>(wsb + pl.gmax_off) : nullptr;
  st = cuda_status(timed("gemm_gcol", s, [&] {
    return pl.k3cl ? launch_gemm_gcol_cl(ga, s) : launch_gemm_gcol(ga, prob->dtype, s);
  }));
  if (st != DC_OK) return st;
  ga.w = w;

  if (pl.k3cl) {
    // sampling backward over the staged NHWC windows, then grad_x from the
    // NHWC accumulator
    K3ClArgs ka{};
    ka.g = g;
    ka.xc = wsb + pl.xc_off;
    ka.off = offset;
    ka.gcol = ga.gcol;
    ka.gx_nhwc = gxc;
    ka.goff = goff;
    ka.margin = margin;
    st = cuda_status(timed("k3_cl_bwd", s, [&] { return launch_k3cl(ka, s); }));
    if (st != DC_OK) return st;
    if (pl.k4cl) {
      // offset-convolution backward: the weight part's chunk partials (it
      // also lays out w_off for the input part), then grad_x (NCHW) written
      // whole from the NHWC accumulator plus the input part; the partials
      // are summed after the weight-gradient GEMM
      K4ClArgs k4{};
      k4.g = g;
      k4.xc = wsb + pl.xc_off;
      k4.w_off = w_off;
      k4.goff = goff;
      k4.gx_nhwc = gxc;
      k4.x = x;
      k4.grad_x = grad_x;
      k4.grad_w_off = grad_w_off;
      k4.grad_b_off = grad_b_off;
      k4.part = reinterpret_cast<float*>(wsb + pl.k4part_off);
      k4.gw_perm = gw_perm;
      k4.grad_w = grad_w;
      k4.c_out = g.c_out;
      st = cuda_status(timed("k4cl_weight", s, [&] { return launch_k4cl_weight(k4, s); }));
      if (st != DC_OK) return st;
      st = cuda_status(timed("k4cl_input", s, [&] { return launch_k4cl_input(k4, s); }));
      if (st != DC_OK) return st;
      ga.gw_perm = gw_perm;
      st = cuda_status(timed("gemm_gw", s, [&] { return launch_gemm_gw_cl(ga, s); }));
      if (st != DC_OK) return st;
      return cuda_status(timed("k4cl_reduce", s, [&] { return launch_k4cl_reduce(k4, s); }));
    }
    st = cuda_status(timed("gx_to_nchw", s, [&] { return launch_gx_to_nchw(gxc, gx32, g, s); }));
    if (st != DC_OK) return st;
  }

  // sampling backward; replays the deformed map for grad_w
  BwdArgs ba{};
  ba.g = g;
  ba.x = x;
  ba.off = offset;
  ba.gcol = ga.gcol;
  ba.gcol_layout = pl.gcol;
  ba.col = (reuse_map || pl.cl) ? nullptr : wsb + pl.col_off;
  ba.col_layout = pl.col;
  ba.gx = gx32;
  ba.goff = goff;
  ba.margin = margin;
  ba.gmax = ga.gmax;
  ba.gmax_tx = pl.gmax_tx;
  ba.gmax_ty = pl.gmax_ty;
  if (!pl.k3cl) {
    st = cuda_status(timed("k3_band_bwd", s, [&] { return launch_band_bwd(ba, prob->dtype, s); }));
    if (st != DC_OK) return st;
  }

  // offset-convolution backward on the completed offset gradient
  OffconvBwdArgs oa{};
  oa.g = g;
  oa.x = x;
  oa.w_off = w_off;
  oa.goff = goff;
  oa.gx = gx32;
  oa.gw_off = grad_w_off;
  oa.gb_off = grad_b_off;
  oa.gw_off_img = gwo_img;
  st = cuda_status(timed("k4_offconv_bwd", s, [&] { return launch_offconv_bwd(oa, prob->dtype, s); }));
  if (st != DC_OK) return st;

  // main weight gradient from the replayed map; the tensor-core GEMM also sums
  // K4's per-image grad_w_off partials once K4 is done (its CTAs wait for K4
  // before exiting anyway), else a small kernel does
  const bool gw_reduces = gwo_img && tc_gcol;
  if (gw_reduces) {
    ga.gwo_img = gwo_img;
    ga.gw_off = grad_w_off;
    ga.gwo_count = gwo_frag_count(g.M, g.c_in, g.K);
  }
  st = cuda_status(timed("gemm_gw", s, [&] {
    return pl.cl ? launch_gemm_gw_cl(ga, s) : launch_gemm_gw(ga, prob->dtype, s);
  }));
  if (st != DC_OK) return st;
  if (gwo_img && !gw_reduces) {
    // grad_w_off from K4's per-image partials
    st = cuda_status(timed("gw_off_reduce", s, [&] { return launch_gw_off_reduce(oa, s); }));
    if (st != DC_OK) return st;
  }
  if (!pl.gxr_off) return DC_OK;
  // the ReLU backward of the layer before, on the completed grad_x
  return cuda_status(timed("relu_bwd", s, [&] {
    return launch_relu_bwd(x, gx32, grad_x, (long long)g.n * g.c_in * g.hw, prob->dtype, s);
  }));
}

}  // namespace
}  // namespace dc

extern "C" {

dc_status dc_test_fail_launches(int count) {
  if (count < 0) return DC_ERR_INVALID_ARG;
  g_fail_launches.store(count, std::memory_order_relaxed);
  return DC_OK;
}

int dc_out_h(const dc_problem* prob) {
  Geom g;
  int m;
  return make_geom(prob, &g, &m) == DC_OK ? g.ho : 0;
}

int dc_out_w(const dc_problem* prob) {
  Geom g;
  int m;
  return make_geom(prob, &g, &m) == DC_OK ? g.wo : 0;
}

dc_status deform_conv_workspace_size(const dc_problem* prob, int backward, size_t* bytes) {
  if (!bytes) return DC_ERR_INVALID_ARG;
  Geom g;
  int margin;
  const dc_status st = make_geom(prob, &g, &margin);
  if (st != DC_OK) return st;
  if (backward && (bwd_smem_bytes(g, prob->dtype, margin) > kMaxSmem ||
                   offconv_bwd_smem_bytes(g, prob->dtype) > kMaxSmem))
    return DC_ERR_UNSUPPORTED;
  *bytes = make_plan(g, prob->dtype, backward ? 1 : 0, margin).total;
  return DC_OK;
}

dc_status deform_conv_fwd(const dc_problem* prob, const void* x, const void* w_off,
                          const float* b_off, const void* w, const float* offset_add, void* y,
                          float* offset_out, unsigned long long* slowpath_count, void* ws,
                          size_t ws_bytes, void* stream) {
  Geom g;
  int margin;
  dc_status st = make_geom(prob, &g, &margin);
  if (st != DC_OK) return st;
  if (!x || !w_off || !w || !y) return DC_ERR_INVALID_ARG;
  const void* ptrs[] = {x, w_off, b_off, w, offset_add, y, offset_out, slowpath_count, ws};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return DC_ERR_UNSUPPORTED;
  const Plan pl = make_plan(g, prob->dtype, 0, margin);
  if (!ws || ws_bytes < pl.total) return DC_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* wsb = static_cast<char*>(ws);

  if (pl.cl) {
    st = cl_stage(g, margin, pl, wsb, x, w_off, w, b_off, offset_add, nullptr, wsb + pl.col_off,
                  offset_out, slowpath_count, s);
    if (st != DC_OK) return st;
    GemmArgs ga{};
    ga.g = g;
    ga.w = wsb + pl.wp_off;
    ga.col = wsb + pl.col_off;
    ga.y = y;
    return cuda_status(timed("gemm_fwd", s, [&] { return launch_gemm_fwd_cl(ga, s); }));
  }
  SampleArgs sa{};
  sa.g = g;
  sa.x = x;
  sa.w_off = w_off;
  sa.b_off = b_off;
  sa.off_add = offset_add;
  sa.off_in = nullptr;
  sa.col = wsb + pl.col_off;
  sa.col_layout = pl.col;
  sa.off_out = offset_out;
  sa.slow_count = slowpath_count;
  sa.margin = margin;
  st = cuda_status(timed("k1_band_sample", s, [&] { return launch_sample(sa, prob->dtype, s); }));
  if (st != DC_OK) return st;

  GemmArgs ga{};
  ga.g = g;
  ga.w = w;
  ga.col = sa.col;
  ga.col_layout = pl.col;
  ga.y = y;
  return cuda_status(timed("gemm_fwd", s, [&] { return launch_gemm_fwd(ga, prob->dtype, s); }));
}

dc_status deform_conv_bwd(const dc_problem* prob, const void* x, const void* w_off, const void* w,
                          const float* offset, const void* grad_y, void* grad_x,
                          float* grad_w_off, float* grad_b_off, float* grad_w,
                          float* grad_offset, void* ws, size_t ws_bytes, void* stream) {
  return dc::backward(prob, x, w_off, w, offset, grad_y, grad_x, grad_w_off, grad_b_off, grad_w,
                      grad_offset, ws, ws_bytes, stream, false);
}

dc_status deform_conv_bwd_after_fwd(const dc_problem* prob, const void* x, const void* w_off,
                                    const void* w, const float* offset, const void* grad_y,
                                    void* grad_x, float* grad_w_off, float* grad_b_off,
                                    float* grad_w, float* grad_offset, void* ws, size_t ws_bytes,
                                    void* stream) {
  return dc::backward(prob, x, w_off, w, offset, grad_y, grad_x, grad_w_off, grad_b_off, grad_w,
                      grad_offset, ws, ws_bytes, stream, true);
}

dc_status deform_conv_sample(const dc_problem* prob, const void* x, const void* w_off,
                             const float* b_off, const float* offset_add, const float* offset_in,
                             void* col, float* offset_out, unsigned long long* slowpath_count,
                             void* ws, size_t ws_bytes, void* stream) {
  Geom g;
  int margin;
  dc_status st = make_geom(prob, &g, &margin);
  if (st != DC_OK) return st;
  if (!x || !col || (!offset_in && !w_off)) return DC_ERR_INVALID_ARG;
  const void* ptrs[] = {x, w_off, b_off, offset_add, offset_in, col, offset_out, slowpath_count, ws};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return DC_ERR_UNSUPPORTED;
  const Plan pl = make_plan(g, prob->dtype, 0, margin);
  if (!ws || ws_bytes < pl.total) return DC_ERR_WORKSPACE;
  if (pl.cl)
    return cl_stage(g, margin, pl, static_cast<char*>(ws), x, w_off, nullptr, b_off, offset_add,
                    offset_in, col, offset_out, slowpath_count, static_cast<cudaStream_t>(stream));
  SampleArgs sa{};
  sa.g = g;
  sa.x = x;
  sa.w_off = w_off;
  sa.b_off = offset_in ? nullptr : b_off;
  sa.off_add = offset_in ? nullptr : offset_add;
  sa.off_in = offset_in;
  sa.col = col;
  sa.col_layout.img = g.howo;
  sa.col_layout.row = g.howo * g.n;
  sa.off_out = offset_out;
  sa.slow_count = slowpath_count;
  sa.margin = margin;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return cuda_status(timed("k1_band_sample", s, [&] { return launch_sample(sa, prob->dtype, s); }));
}

dc_status deform_conv_offsets(const dc_problem* prob, const void* x, const void* w_off,
                              const float* b_off, const float* offset_add, float* offset_out,
                              void* ws, size_t ws_bytes, void* stream) {
  Geom g;
  int margin;
  dc_status st = make_geom(prob, &g, &margin);
  if (st != DC_OK) return st;
  if (!x || !w_off || !offset_out) return DC_ERR_INVALID_ARG;
  const void* ptrs[] = {x, w_off, b_off, offset_add, offset_out, ws};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return DC_ERR_UNSUPPORTED;
  const Plan pl = make_plan(g, prob->dtype, 0, margin);
  if (!ws || ws_bytes < pl.total) return DC_ERR_WORKSPACE;
  if (pl.cl)
    return cl_stage(g, margin, pl, static_cast<char*>(ws), x, w_off, nullptr, b_off, offset_add,
                    nullptr, nullptr, offset_out, nullptr, static_cast<cudaStream_t>(stream));
  SampleArgs sa{};
  sa.g = g;
  sa.x = x;
  sa.w_off = w_off;
  sa.b_off = b_off;
  sa.off_add = offset_add;
  sa.col = nullptr;  // K1 stops after the offset convolution
  sa.off_out = offset_out;
  sa.margin = margin;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return cuda_status(timed("k1_offsets", s, [&] { return launch_sample(sa, prob->dtype, s); }));
}

dc_status deform_conv_fwd_sampled_gemm(const dc_problem* prob, const void* x, const void* w_off,
                                       const float* b_off, const void* w,
                                       const float* offset_add, void* y, float* offset_out,
                                       void* stream) {
  Geom g;
  int margin;
  dc_status st = make_geom(prob, &g, &margin);
  if (st != DC_OK) return st;
  if (!x || !w_off || !w || !y || !offset_out) return DC_ERR_INVALID_ARG;
  if (prob->dtype != DC_BF16 || !fwd_sampled_supported(g)) return DC_ERR_UNSUPPORTED;
  const void* ptrs[] = {x, w_off, b_off, w, offset_add, y, offset_out};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return DC_ERR_UNSUPPORTED;
  SampleArgs sa{};
  sa.g = g;
  sa.x = x;
  sa.w_off = w_off;
  sa.b_off = b_off;
  sa.off_add = offset_add;
  sa.col = nullptr;  // K1 stops after the offset convolution
  sa.off_out = offset_out;
  sa.margin = margin;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = cuda_status(timed("k1_offsets", s, [&] { return launch_sample(sa, prob->dtype, s); }));
  if (st != DC_OK) return st;
  return cuda_status(timed("gemm_fwd_sampled", s, [&] {
    return launch_fwd_sampled_tc(g, x, w, offset_out, y, s);
  }));
}

dc_status deform_conv_margin_histogram(const dc_problem* prob, const float* offset,
                                       unsigned long long* hist, void* stream) {
  Geom g;
  int margin;
  dc_status st = make_geom(prob, &g, &margin);
  if (st != DC_OK) return st;
  if (!offset || !hist) return DC_ERR_INVALID_ARG;
  int R, TW;
  if (cl_supported(g, prob->dtype, margin))
    cl_tile(g, margin, &R, &TW);
  else
    sample_band(g, prob->dtype, margin, &R, &TW);
  return cuda_status(
      launch_margin_histogram(offset, g, R, TW, hist, static_cast<cudaStream_t>(stream)));
}

int dc_suggest_margin(const dc_problem* prob, const unsigned long long* hist,
                      double max_slow_fraction, int for_backward) {
  if (!prob || !hist || !(max_slow_fraction >= 0.0 && max_slow_fraction <= 1.0)) return -1;
  dc_problem q = *prob;
  q.halo_margin = 0;
  Geom g;
  int m0;
  if (make_geom(&q, &g, &m0) != DC_OK) return -1;
  unsigned long long total = 0;
  for (int b = 0; b < DC_MARGIN_BINS; ++b) total += hist[b];
  // smallest m with (taps needing more than m) <= fraction * total
  int m = DC_MARGIN_BINS - 1;
  unsigned long long above = 0;
  for (int b = DC_MARGIN_BINS - 1; b >= 1; --b) {
    above += hist[b];  // taps needing b or more
    if ((double)above > max_slow_fraction * (double)total) break;
    m = b - 1;
  }
  if (m > kMaxMargin) m = kMaxMargin;
  auto fits = [&](int mm) {
    if (sample_smem_bytes(g, q.dtype, mm) > kMaxSmem) return false;
    return !for_backward || bwd_smem_bytes(g, q.dtype, mm) <= kMaxSmem;
  };
  while (m > 0 && !fits(m)) --m;
  return m;
}

int dc_col_layout(const dc_problem* prob) {
  Geom g;
  int margin;
  if (make_geom(prob, &g, &margin) != DC_OK) return -1;
  return cl_supported(g, prob->dtype, margin) ? DC_COL_PIXEL_MAJOR : DC_COL_PLANE_MAJOR;
}

dc_status dc_sample_tile(const dc_problem* prob, int* tile_h, int* tile_w) {
  Geom g;
  int margin;
  const dc_status st = make_geom(prob, &g, &margin);
  if (st != DC_OK) return st;
  if (!tile_h || !tile_w) return DC_ERR_INVALID_ARG;
  if (cl_supported(g, prob->dtype, margin))
    cl_tile(g, margin, tile_h, tile_w);
  else
    sample_band(g, prob->dtype, margin, tile_h, tile_w);
  return DC_OK;
}

dc_status dc_relu_fwd(const void* y, void* out, size_t count, dc_dtype dtype, void* stream) {
  if (dtype != DC_F32 && dtype != DC_BF16) return DC_ERR_INVALID_ARG;
  if (count == 0) return DC_OK;
  if (!y || !out) return DC_ERR_INVALID_ARG;
  if (!aligned16(y) || !aligned16(out)) return DC_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return cuda_status(timed("relu_fwd", s, [&] {
    return launch_relu_fwd(y, out, (long long)count, dtype, s);
  }));
}

dc_status dc_relu_bwd(const void* act, const float* grad_out, void* grad_in, size_t count,
                      dc_dtype dtype, void* stream) {
  if (dtype != DC_F32 && dtype != DC_BF16) return DC_ERR_INVALID_ARG;
  if (count == 0) return DC_OK;
  if (!act || !grad_out || !grad_in) return DC_ERR_INVALID_ARG;
  if (!aligned16(act) || !aligned16(grad_out) || !aligned16(grad_in)) return DC_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return cuda_status(timed("relu_bwd", s, [&] {
    return launch_relu_bwd(act, grad_out, grad_in, (long long)count, dtype, s);
  }));
}

const char* dc_status_string(dc_status status) {
  switch (status) {
    case DC_OK: return "DC_OK: success";
    case DC_ERR_INVALID_ARG: return "DC_ERR_INVALID_ARG: invalid problem size or missing argument";
    case DC_ERR_UNSUPPORTED: return "DC_ERR_UNSUPPORTED: no path for this problem (alignment, dtype or size)";
    case DC_ERR_WORKSPACE: return "DC_ERR_WORKSPACE: workspace missing or too small";
    case DC_ERR_CUDA: return "DC_ERR_CUDA: a CUDA launch or runtime call failed";
    case DC_ERR_TIMEOUT: return "DC_ERR_TIMEOUT: a bounded device wait expired";
  }
  return "unknown dc_status";
}

void dc_kernel_timing(int enable) {
  std::lock_guard<std::mutex> lock(g_timing_mu);
  g_timing.store(enable != 0, std::memory_order_relaxed);
  g_ntimed = 0;
}

int dc_kernel_times(const char** names, float* ms, int capacity) {
  std::lock_guard<std::mutex> lock(g_timing_mu);
  const int n = g_ntimed < capacity ? g_ntimed : capacity;
  for (int i = 0; i < n; ++i) {
    float t = -1.f;
    if (cudaEventSynchronize(g_timed[i].b) != cudaSuccess ||
        cudaEventElapsedTime(&t, g_timed[i].a, g_timed[i].b) != cudaSuccess)
      t = -1.f;
    if (names) names[i] = g_timed[i].name;
    if (ms) ms[i] = t;
  }
  g_ntimed = 0;
  return n;
}

unsigned long long dc_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char* dc_build_info(void) {
  return "deformable_convolution_gb300: sm_103a, CUDA "
#define DC_STR2(x) #x
#define DC_STR(x) DC_STR2(x)
         DC_STR(__CUDACC_VER_MAJOR__) "." DC_STR(__CUDACC_VER_MINOR__);
}

}  // extern "C"

namespace dc {

// GEMM dispatch: bf16 problems whose rows are 16-byte aligned run on the
// tensor cores; float32 problems (whose tolerance a bf16/tf32 contraction would
// not hold) and unaligned shapes run on CUDA cores.
cudaError_t launch_gemm_fwd(const GemmArgs& a, dc_dtype dt, cudaStream_t s) {
  if (dt == DC_BF16 && tc_gemm_supported(a.g)) return launch_gemm_fwd_tc(a, s);
  if (dt == DC_F32 && tf32_gemm_supported(a.g)) return launch_gemm_fwd_tf32(a, s);
  return launch_gemm_fwd_simt(a, dt, s);
}
cudaError_t launch_gemm_gcol(const GemmArgs& a, dc_dtype dt, cudaStream_t s) {
  if (dt == DC_BF16 && tc_gemm_supported(a.g)) return launch_gemm_gcol_tc(a, s);
  if (dt == DC_F32 && tf32_gemm_supported(a.g)) return launch_gemm_gcol_tf32(a, s);
  return launch_gemm_gcol_simt(a, dt, s);
}
cudaError_t launch_gemm_gw(const GemmArgs& a, dc_dtype dt, cudaStream_t s) {
  if (dt == DC_BF16 && tc_gemm_supported(a.g)) return launch_gemm_gw_tc(a, s);
  if (dt == DC_F32 && tf32_gemm_supported(a.g)) return launch_gemm_gw_tf32(a, s);
  return launch_gemm_gw_simt(a, dt, s);
}

}  // namespace dc
