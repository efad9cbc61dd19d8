/*
 * deform_conv.h -- C ABI of the GB300 (sm_103a) deformable convolution layer.
 *
 * The layer follows the explainer page "DefT: Boosting Scalability of
 * Deformable Convolution Operations on GPUs" (ASPLOS 2023):
 *   - "The argument in one glance / What people did": three operators -- an
 *     offset convolution, a bilinear interpolation that builds the deformed
 *     feature map, and the main convolution over that map;
 *   - "Following a deformable layer through DefT", Step 1 of 5: a fractional
 *     (y, x) offset for every filter position at every output location, added
 *     to the base sampling coordinate;
 *   - "The argument in one glance / Why it fell short": each displaced sample
 *     blends its four neighbouring pixels by their bilinear weights;
 *   - "This paper's idea" / "Why it works": the offset convolution and the
 *     interpolation run fused in one kernel over an output-spatial tile whose
 *     input halo, padded by a margin sized to the offset distribution, is staged
 *     on chip; the main convolution stays a separate dense GEMM.
 * Written out: y[n,o,p0] = sum_{c,k} w[o,c,k] * xbar[n,c](p0*s - pad + k*dil +
 * dp[n,g(c),k,p0]), with xbar read by bilinear interpolation and zero outside
 * the image.
 *
 * Conventions (the page fixes none of these; they are this library's):
 *   - All tensors are dense, contiguous, row-major, on the current CUDA device.
 *     x, y: NCHW.  w: [C_out, C_in, Kh, Kw].  w_off: [2*G*Kh*Kw, C_in, Kh, Kw].
 *     x, y, w and w_off are in the problem's dtype; b_off, offsets and every
 *     gradient are float32.
 *   - The offset convolution uses the main convolution's kernel size, stride,
 *     padding and dilation and has a bias b_off, so its output grid is the
 *     output grid [N, 2*G*Kh*Kw, Ho, Wo].
 *   - Offset channel 2*(g*Kh*Kw + k) is the row shift and 2*(g*Kh*Kw + k) + 1
 *     the column shift of tap k = i*Kw + j in offset group g; input channel c
 *     belongs to group c / (C_in / G).
 *   - Corners outside [0,H) x [0,W) contribute zero.  At an integer sampling
 *     coordinate the lower corner is floor(p), so offset gradients there are
 *     right-sided differences.
 *   - Ownership: the caller allocates every buffer, including the workspace.
 *     The library allocates no device memory, keeps no per-call state, and
 *     never synchronises; all work is enqueued on `stream` (a cudaStream_t; 0
 *     is the legacy default stream).  Calls on different streams must not
 *     share a workspace.
 *   - Errors: arguments are checked on the host before anything is launched.
 *     A non-DC_OK status means nothing was enqueued, except DC_ERR_CUDA from a
 *     launch, after which earlier kernels of the same call may have run.
 *   - Pointers must be 16-byte aligned.  Gradient outputs are overwritten.
 */
#ifndef DEFORM_CONV_H_
#define DEFORM_CONV_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DC_OK = 0,
  DC_ERR_INVALID_ARG = 1, /* bad size, C_in % G != 0, Ho or Wo < 1, NULL required pointer */
  DC_ERR_UNSUPPORTED = 2, /* valid problem this build has no path for (alignment, dtype, size) */
  DC_ERR_WORKSPACE = 3,   /* workspace pointer NULL or smaller than the query returned */
  DC_ERR_CUDA = 4,        /* a CUDA launch or runtime call failed */
  DC_ERR_TIMEOUT = 5      /* a bounded on-device wait expired (reported by dc_device_error) */
} dc_status;

typedef enum { DC_F32 = 0, DC_BF16 = 1 } dc_dtype;

/* Geometry of one deformable layer.  halo_margin is the number of extra pixels
 * the fused sampling kernel stages around each output tile's receptive field
 * ("The idea": tile padding sized to the offset distribution); -1 selects the
 * library default (3 px).  It changes speed only, never results: taps that
 * fall outside the staged tile are read from global memory.
 * out_relu (0 or 1): the forward calls write y = max(conv, 0) instead of the
 * convolution, a following ReLU fused into the main GEMM's epilogue; the
 * result is bit for bit dc_relu_fwd of the plain forward (NaN kept, -0 -> +0).
 * The backward calls ignore it: their grad_y is the gradient with respect to
 * the convolution's output, as without it.
 * in_relu (0 or 1): x is the output of a ReLU, x = max(z, 0), and the backward
 * calls return the gradient with respect to z instead of x:
 * grad_x[i] = x[i] > 0 ? dL/dx[i] : 0, written in the problem dtype (the
 * grad_x buffer of a bf16 problem then holds bf16 elements), what
 * dc_relu_bwd(x, dL/dx) gives for the float32 dL/dx the call computes -- the
 * previous layer's ReLU backward fused into this layer's grad_x epilogue.  The backward workspace query counts it (problems
 * off the channels-last backward need a float32 grad_x scratch); the forward
 * calls ignore it. */
typedef struct {
  int n, c_in, h, w, c_out, kh, kw;
  int stride_h, stride_w, pad_h, pad_w, dil_h, dil_w;
  int offset_groups;
  dc_dtype dtype;
  int halo_margin;
  int out_relu;
  int in_relu;
} dc_problem;

/* Output height/width of the problem (0 if the problem is invalid). */
int dc_out_h(const dc_problem* prob);
int dc_out_w(const dc_problem* prob);

/* Bytes of device workspace deform_conv_fwd (backward = 0) or deform_conv_bwd
 * (backward = 1) needs for this problem.  Writes *bytes; returns
 * DC_ERR_INVALID_ARG / DC_ERR_UNSUPPORTED for problems the calls would reject. */
dc_status deform_conv_workspace_size(const dc_problem* prob, int backward, size_t* bytes);

/* Forward pass of the whole layer ("What people did": offset convolution ->
 * bilinear interpolation -> main convolution; the first two fused, "This
 * paper's idea").
 *   x          [N, C_in, H, W]                 dtype, required
 *   w_off      [2GK, C_in, Kh, Kw]             dtype, required (offset conv weights)
 *   b_off      [2GK]                           float32, NULL = zero bias
 *   w          [C_out, C_in, Kh, Kw]           dtype, required (main weights)
 *   offset_add [N, 2GK, Ho, Wo]                float32, NULL = none; added to the
 *                                              offset-conv output before sampling
 *   y          [N, C_out, Ho, Wo]              dtype, required, overwritten
 *   offset_out [N, 2GK, Ho, Wo]                float32, NULL = not returned; the
 *                                              offsets used (input to the backward)
 *   slowpath_count  one unsigned 64-bit counter, NULL = not counted; the number
 *                   of taps read outside the staged tile is ADDED to it
 *   ws, ws_bytes    workspace from deform_conv_workspace_size(prob, 0, ...)
 * Accumulation is float32 for both dtypes; bf16 outputs are rounded to nearest
 * even. */
dc_status deform_conv_fwd(const dc_problem* prob, const void* x, const void* w_off,
                          const float* b_off, const void* w, const float* offset_add,
                          void* y, float* offset_out, unsigned long long* slowpath_count,
                          void* ws, size_t ws_bytes, void* stream);

/* Backward pass: gradients of sum(y * grad_y) at the saved offsets.
 *   x, w_off, w   as in the forward pass
 *   offset        [N, 2GK, Ho, Wo] float32, required: offset_out of the forward
 *   grad_y        [N, C_out, Ho, Wo] dtype, required
 *   grad_x        [N, C_in, H, W] float32, required (sampling + offset-conv paths);
 *                 the problem dtype, masked by x > 0, when prob->in_relu = 1
 *   grad_w_off    [2GK, C_in, Kh, Kw] float32, required
 *   grad_b_off    [2GK] float32, NULL = not returned
 *   grad_w        [C_out, C_in, Kh, Kw] float32, required
 *   grad_offset   [N, 2GK, Ho, Wo] float32, NULL = not returned; gradient with
 *                 respect to the offsets (equivalently to offset_add)
 *   ws, ws_bytes  workspace from deform_conv_workspace_size(prob, 1, ...)
 * Float32 atomics make grad_x, grad_w and grad_w_off reproducible only up to
 * summation order. */
dc_status deform_conv_bwd(const dc_problem* prob, const void* x, const void* w_off,
                          const void* w, const float* offset, const void* grad_y,
                          void* grad_x, float* grad_w_off, float* grad_b_off,
                          float* grad_w, float* grad_offset, void* ws, size_t ws_bytes,
                          void* stream);

/* The backward pass when the workspace still holds the forward pass's
 * deformed map ("What people did before, and where it broke": the unrolled
 * map the interpolation materialises): the weight-gradient GEMM reads that map
 * and the sampling backward does not replay it.  Arguments as in
 * deform_conv_bwd; `ws` must be the workspace the deform_conv_fwd call for
 * these x, w_off and offsets used (any halo_margin), not rewritten since --
 * a training step that keeps its forward workspace until the backward.  The
 * library cannot check this: a stale map gives a wrong grad_w only. */
dc_status deform_conv_bwd_after_fwd(const dc_problem* prob, const void* x, const void* w_off,
                                    const void* w, const float* offset, const void* grad_y,
                                    void* grad_x, float* grad_w_off, float* grad_b_off,
                                    float* grad_w, float* grad_offset, void* ws, size_t ws_bytes,
                                    void* stream);

/* Layout of the deformed feature map for a problem (dc_col_layout):
 *   DC_COL_PLANE_MAJOR  col[C_in*Kh*Kw][N][Ho*Wo]: row c*Kh*Kw + k holds channel
 *                       c sampled at tap k for every output pixel;
 *   DC_COL_PIXEL_MAJOR  col[N][Ho*Wo][Kh*Kw][C_in]: for each output pixel and
 *                       tap, the C_in channels are contiguous.
 * bf16 problems with C_in a multiple of 64 (at most 256), C_in / G a multiple
 * of 8, H*W, C_in*Kh*Kw and Ho*Wo multiples of 8 take the channels-last path
 * (pixel-major map, x staged from an NHWC copy); all others the plane-major
 * one.  Returns -1 for an invalid problem. */
#define DC_COL_PLANE_MAJOR 0
#define DC_COL_PIXEL_MAJOR 1
int dc_col_layout(const dc_problem* prob);

/* Output tile (tile_h rows x tile_w columns of output pixels) over which the
 * fused sampling stage stages its input window for this problem and margin
 * (the window is the tile's receptive field plus halo_margin pixels per side).
 * DC_ERR_INVALID_ARG for an invalid problem or NULL outputs. */
dc_status dc_sample_tile(const dc_problem* prob, int* tile_h, int* tile_w);

/* The fused offset-convolution + bilinear-interpolation stage alone ("This
 * paper's idea": the kernel whose arithmetic intensity the fusion raises),
 * returning the deformed feature map ("What people did before, and where it
 * broke": the unrolled map the interpolation materialises).
 *   col        dtype, required, C_in*Kh*Kw*N*Ho*Wo elements in the problem's
 *              layout (dc_col_layout)
 *   offset_add, b_off, offset_out, slowpath_count as in deform_conv_fwd
 *   ws, ws_bytes  workspace from deform_conv_workspace_size(prob, 0, ...)
 *              (the channels-last path keeps x's NHWC copy there)
 * If `offset_in` is non-NULL the offset convolution is skipped and those
 * offsets [N, 2GK, Ho, Wo] are sampled instead (w_off and b_off are ignored). */
dc_status deform_conv_sample(const dc_problem* prob, const void* x, const void* w_off,
                             const float* b_off, const float* offset_add,
                             const float* offset_in, void* col, float* offset_out,
                             unsigned long long* slowpath_count, void* ws, size_t ws_bytes,
                             void* stream);

/* The offset convolution alone ("Following a deformable layer through DefT",
 * Step 1 of 5: a small standard convolution over the input that predicts one
 * (dy, dx) per tap and output pixel), written to HBM.  This is the first
 * kernel of the unfused pipeline that the page contrasts with the fused one
 * ("What people did before, and where it broke": offsets round-trip through
 * memory before the interpolation reads them); deform_conv_sample with
 * offset_in = these offsets is the second.  Same kernel as the fused stage,
 * stopping before the interpolation.
 *   x, w_off, b_off, offset_add  as in deform_conv_fwd
 *   offset_out   [N, 2GK, Ho, Wo] float32, required
 *   ws, ws_bytes workspace from deform_conv_workspace_size(prob, 0, ...)
 * Errors: DC_ERR_INVALID_ARG for a NULL x, w_off or offset_out,
 * DC_ERR_UNSUPPORTED for a pointer that is not 16-byte aligned,
 * DC_ERR_WORKSPACE for a missing or short workspace. */
dc_status deform_conv_offsets(const dc_problem* prob, const void* x, const void* w_off,
                              const float* b_off, const float* offset_add, float* offset_out,
                              void* ws, size_t ws_bytes, void* stream);

/* The forward pass with the deformed map never written to memory: the
 * offset convolution (as deform_conv_offsets, offsets to offset_out), then one
 * tensor-core kernel that samples each 64 x 64 tile of the map from x and the
 * offsets straight into shared memory as the main GEMM's B operand and
 * multiplies it by w.  This is the fusion of interpolation and main
 * convolution that the explainer page argues against ("This paper's idea":
 * the main convolution should stay a separate, library-grade GEMM), provided
 * to measure that trade-off.  Same sampling arithmetic and MMA order as
 * deform_conv_fwd for the same offsets.
 *   x, w_off, b_off, w, offset_add, y, offset_out  as in deform_conv_fwd
 *     (y, offset_out required)
 * No workspace.  Asynchronous on `stream`.  Errors: DC_ERR_INVALID_ARG for a
 * NULL x, w_off, w, y or offset_out or an invalid problem;
 * DC_ERR_UNSUPPORTED unless the problem is bf16 with C_in*Kh*Kw and Ho*Wo
 * multiples of 8 (the tensor-core GEMM's alignment) or for a pointer that is
 * not 16-byte aligned. */
dc_status deform_conv_fwd_sampled_gemm(const dc_problem* prob, const void* x, const void* w_off,
                                       const float* b_off, const void* w,
                                       const float* offset_add, void* y, float* offset_out,
                                       void* stream);

/* Margin statistics ("Why it works" / "The idea" on the explainer page: each
 * tile is padded by just enough margin for the offsets that occur, measured
 * from their distribution).  From the offsets a forward call returned, counts
 * for every sampling tap (image, offset group, tap, output pixel) the margin
 * in whole pixels its band's staged window needs to serve it on chip: how far
 * the two rows and two columns it reads pass the edges of the band's
 * receptive field, for the bands the fused stage uses with prob's current
 * halo_margin.  Taps that sample entirely outside the image count as 0;
 * needs of DC_MARGIN_BINS - 1 or more (and NaN positions) go to the last bin.
 * With the same band shape, the taps of the bins above a margin m are exactly
 * those the forward pass reads from global memory (its slowpath_count).
 *   offset  [N, 2GK, Ho, Wo] float32 device pointer, required
 *   hist    DC_MARGIN_BINS unsigned 64-bit device counters, required,
 *           overwritten (cleared on the stream, then accumulated)
 * Asynchronous on `stream`; allocates nothing.  Errors: DC_ERR_INVALID_ARG
 * for NULL pointers or an invalid problem. */
#define DC_MARGIN_BINS 64
dc_status deform_conv_margin_histogram(const dc_problem* prob, const float* offset,
                                       unsigned long long* hist, void* stream);

/* Host helper: the smallest halo_margin m whose slow-path fraction, by the
 * histogram (a HOST copy of deform_conv_margin_histogram's output), is at most
 * max_slow_fraction: the taps in bins above m over all taps.  The result is
 * lowered to the largest margin this build can stage for `prob` (forward, and
 * backward too when for_backward != 0).  A margin large enough to make the
 * fused stage pick smaller bands changes the shape the histogram assumed;
 * measuring again at the new margin closes the loop.  Returns -1 for an
 * invalid problem, histogram or fraction (outside [0, 1]). */
int dc_suggest_margin(const dc_problem* prob, const unsigned long long* hist,
                      double max_slow_fraction, int for_backward);

/* Forward pass without a caller-provided workspace.  The paper has no
 * counterpart to this entry point; it exists for callers that cannot allocate
 * device memory -- loops that must not allocate once running, plug-ins whose
 * host framework owns all device memory, call sites that could not handle an
 * allocation failure.  Arguments and results are those of deform_conv_fwd
 * minus ws/ws_bytes.
 *   - Scratch: a fixed array of DC_NOALLOC_SCRATCH_BYTES inside this library,
 *     held on every GPU that loads the library until the process exits.
 *     Problems whose forward workspace (deform_conv_workspace_size(prob, 0))
 *     exceeds it are rejected with DC_ERR_WORKSPACE before anything runs.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *   - Every call looks up the array's address on the current device
 *     (cudaGetSymbolAddress, a host-side query that allocates nothing; the
 *     first one on a device may load this library's module there): make the
 *     first call on each device before any stream capture.
 *   - Every call on a device shares the one array and leaves its contents
 *     behind; nothing there needs to start at zero.  Calls whose work
 *     overlaps on the GPU (other streams, other host threads) race on the
 *     array: serialise them. */
#define DC_NOALLOC_SCRATCH_BYTES (32u << 20)
dc_status deform_conv_fwd_noalloc(const dc_problem* prob, const void* x, const void* w_off,
                                  const float* b_off, const void* w, const float* offset_add,
                                  void* y, float* offset_out,
                                  unsigned long long* slowpath_count, void* stream);

/* ReLU between stacked deformable layers.  The explainer page's networks
 * stack deformable layers throughout a ResNet ("What people did before, and
 * where it broke": adding deformable layers; "Why it works / Fixing the
 * slowest stage lifts the whole layer": training a fully deformable ResNet),
 * whose convolutions are separated by ReLU activations; a training step over
 * such a stack needs the activation and its gradient between layers.
 *   dc_relu_fwd: out[i] = y[i] <= 0 ? 0 : y[i] (NaN stays NaN).  y and out are
 *     `count` elements of `dtype`; out may equal y (in place).
 *   dc_relu_bwd: grad_in[i] = act[i] > 0 ? grad_out[i] : 0, rounded to dtype
 *     (nearest even).  act is the activation's OUTPUT (`dtype`, positive
 *     exactly where its input was; NaN gives a zero gradient), grad_out float32
 *     (the next layer's grad_x),
 *     grad_in `dtype` (the previous layer's grad_y).
 * Device pointers, 16-byte aligned (else DC_ERR_UNSUPPORTED); NULL or a bad
 * dtype gives DC_ERR_INVALID_ARG; count 0 does nothing.  Asynchronous on
 * `stream`; allocates nothing. */
dc_status dc_relu_fwd(const void* y, void* out, size_t count, dc_dtype dtype, void* stream);
dc_status dc_relu_bwd(const void* act, const float* grad_out, void* grad_in, size_t count,
                      dc_dtype dtype, void* stream);

/* Static description of a status code. */
const char* dc_status_string(dc_status status);

/* Library build description (architecture, version). */
const char* dc_build_info(void);

/* DC_ERR_TIMEOUT if a bounded on-device wait of this library's kernels has
 * expired since the flag was last cleared on the current device, else DC_OK
 * (DC_ERR_CUDA if the flag cannot be read).  Synchronises with the device.
 * clear != 0 resets the flag.  An expired wait means the kernel skipped the
 * rest of its work: its outputs are not valid. */
dc_status dc_device_error(int clear);

/* Test hooks for the failure paths (no counterpart on the explainer page;
 * they exist so that tests can drive the error reporting without a fault).
 *
 * dc_selftest_wait_timeout enqueues on `stream` (a cudaStream_t, NULL = the
 * default stream) one kernel whose single thread polls, at most `spins`
 * times (1 .. 2^20), an mbarrier that nothing arrives on, then raises the
 * device error flag exactly as an expired wait of the layer's kernels does:
 * the next dc_device_error reports DC_ERR_TIMEOUT.  The kernel holds no
 * copies and no tensor memory, so the expiry leaves the context usable.
 * Returns DC_ERR_INVALID_ARG for spins out of range, DC_ERR_CUDA if the
 * launch fails.
 *
 * dc_test_fail_launches(n): the next n kernel launches of the layer entry
 * points (deform_conv_fwd, _bwd, _sample, _offsets and their variants) are
 * not made and the call returns DC_ERR_CUDA, as for a failed launch; n = 0
 * cancels.  Process-wide, like the timing record below; DC_ERR_INVALID_ARG
 * for n < 0. */
dc_status dc_selftest_wait_timeout(unsigned int spins, void* stream);
dc_status dc_test_fail_launches(int count);

/* Kernel timing (tracing).  dc_kernel_timing(1) starts recording: every
 * kernel (and the backward pass's group of memsets) enqueued by the calls that
 * follow is bracketed by two CUDA events on its stream, up to 256 launches;
 * dc_kernel_timing(0) stops.  Timing is off by default; it must not be enabled
 * while a stream is being captured into a CUDA graph.  dc_kernel_times waits
 * for the recorded launches, writes up to `capacity` (static name, duration in
 * ms) pairs in launch order (-1 for a launch that could not be timed), returns
 * how many it wrote and clears the record.  names or ms may be NULL.
 * The record is process-wide (shared by every host thread and device): it is
 * the one piece of state this library keeps across calls, outside the
 * no-state rule above, and exists only while timing is enabled. */
void dc_kernel_timing(int enable);
int dc_kernel_times(const char** names, float* ms, int capacity);

/* Number of kernels this library has enqueued in this process so far (host
 * counter, incremented per launch; memsets are not counted).  Lets a caller
 * count the launches of a region of work, e.g. of a captured CUDA graph. */
unsigned long long dc_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* DEFORM_CONV_H_ */
