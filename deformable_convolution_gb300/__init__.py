"""GB300-native deformable convolution layer (sm_103a CUDA behind a C ABI).

The layer is the one the explainer page "DefT: Boosting Scalability of
Deformable Convolution Operations on GPUs" describes: an offset convolution,
a bilinear-interpolation gather that builds the deformed feature map (the two
fused in one kernel), and the main convolution over that map.

``binding`` mirrors ``include/deform_conv.h`` one function per entry point;
``workloads`` holds the seeded synthetic inputs used by the tests and the
benchmark.  The library is built in-tree by ``_native.build()``.
"""
from .binding import (DC_BF16, DC_F32, DcError, Problem, backward, deform_conv_bwd,
                      deform_conv_fwd, deform_conv_sample, deform_conv_workspace_size,
                      forward, workspace)

__all__ = ["DC_BF16", "DC_F32", "DcError", "Problem", "backward", "deform_conv_bwd",
           "deform_conv_fwd", "deform_conv_sample", "deform_conv_workspace_size",
           "forward", "workspace"]
