// Forward pass for callers that cannot allocate device memory.
//
// Some callers have no way to hand the library a workspace: code that must
// not allocate once it is running (real-time or embedded loops), plug-ins
// whose host framework owns every byte of device memory, or call sites where
// an allocation failure could not be handled.  deform_conv_fwd_noalloc runs
// the ordinary forward pass with its scratch (the deformed feature map and
// the offsets) in a fixed array that belongs to this library instead of a
// caller-provided workspace.  The explainer page on DefT has no counterpart
// to this entry point; it is an interface convenience only.
//
// The array is a file-scope __device__ object, so every GPU that loads the
// library holds DC_NOALLOC_SCRATCH_BYTES of it until the process exits.  Host
// code cannot use its name as a device address; every call looks the address
// up with cudaGetSymbolAddress on the current device (a host-side query that
// allocates nothing).  Nothing is cached, so a device reset or another
// context on the device, which can place the array elsewhere, never leaves a
// stale address behind.
#include "dc_common.cuh"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[DC_NOALLOC_SCRATCH_BYTES];

}  // namespace

extern "C" dc_status deform_conv_fwd_noalloc(const dc_problem* prob, const void* x,
                                             const void* w_off, const float* b_off,
                                             const void* w, const float* offset_add, void* y,
                                             float* offset_out,
                                             unsigned long long* slowpath_count,
                                             void* stream) {
  size_t need = 0;
  const dc_status st = deform_conv_workspace_size(prob, 0, &need);
  if (st != DC_OK) return st;
  if (need > (size_t)DC_NOALLOC_SCRATCH_BYTES) return DC_ERR_WORKSPACE;
  // the array's address on the current device, looked up on every call
  void* scratch = nullptr;
  if (cudaGetSymbolAddress(&scratch, g_noalloc_scratch) != cudaSuccess || !scratch)
    return DC_ERR_CUDA;
  // Nothing in the forward workspace has to start at zero: every byte the
  // kernels read there was written earlier in the same call.
  return deform_conv_fwd(prob, x, w_off, b_off, w, offset_add, y, offset_out, slowpath_count,
                         scratch, (size_t)DC_NOALLOC_SCRATCH_BYTES, stream);
}
