"""The forward entry point that allocates nothing (deform_conv_fwd_noalloc).

It serves callers that cannot allocate device memory (loops that must not
allocate once running, plug-ins whose host framework owns all device memory):
its scratch is a fixed array inside the library instead of a workspace.  It
must give what the ordinary deform_conv_fwd gives, call after call, even
though every call reuses the same array.  This file is collected last so a
run that stops at its first failure has run every other test before it."""
import pytest
import torch

from deformable_convolution_gb300 import binding as B
from deformable_convolution_gb300 import workloads as W


pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


def _inputs(wl, seed):
    d = W.generate(wl, seed=seed)
    return {k: (None if v is None else v.cuda()) for k, v in d.items()}


@pytest.mark.parametrize("name", ["res3_bf16", "tiny_f32"])
def test_noalloc_matches_workspace_forward_twice(name):
    wl = W.WORKLOADS[name]
    p = wl.problem()
    assert B.deform_conv_workspace_size(p, False) <= B.NOALLOC_SCRATCH_BYTES
    s = p.shapes()
    for call, seed in enumerate((11, 12)):  # two calls in a row, different inputs
        d = _inputs(wl, seed)
        y_ref, off_ref = B.forward(p, d["x"], d["w_off"], d["b_off"], d["w"], d["offset_add"])
        y = torch.full(s["y"], float("nan"), dtype=p.torch_dtype, device="cuda")
        off = torch.full(s["offset"], float("nan"), dtype=torch.float32, device="cuda")
        B.deform_conv_fwd_noalloc(p, d["x"], d["w_off"], d["b_off"], d["w"], d["offset_add"],
                                  y, off)
        torch.cuda.synchronize()
        # the same kernels on the same problem: bit for bit, so that a stale
        # byte left in the shared array by an earlier call would show
        assert torch.equal(_bits(y), _bits(y_ref)), call
        assert torch.equal(off, off_ref), call


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def test_noalloc_large_problem_then_small_one():
    """A call on a large problem leaves its map in the shared array; the next,
    smaller problem reads only what it writes itself."""
    wl = W.WORKLOADS["res3_bf16"]
    big, small = wl.problem(), wl.problem(1)
    d = _inputs(wl, 13)
    y_big = torch.empty(big.shapes()["y"], dtype=big.torch_dtype, device="cuda")
    B.deform_conv_fwd_noalloc(big, d["x"], d["w_off"], d["b_off"], d["w"], d["offset_add"], y_big)
    one = {k: (None if v is None else (v[:1].contiguous() if k in ("x", "offset_add") else v))
           for k, v in d.items()}
    y_ref, off_ref = B.forward(small, one["x"], one["w_off"], one["b_off"], one["w"],
                               one["offset_add"])
    y = torch.empty_like(y_ref)
    off = torch.empty_like(off_ref)
    B.deform_conv_fwd_noalloc(small, one["x"], one["w_off"], one["b_off"], one["w"],
                              one["offset_add"], y, off)
    torch.cuda.synchronize()
    assert torch.equal(_bits(y), _bits(y_ref))
    assert torch.equal(off, off_ref)


def test_noalloc_rejects_problems_beyond_its_scratch():
    # the early-layer workload needs far more than the fixed scratch array;
    # the call must refuse it on the host, before any launch
    p = W.WORKLOADS["early_bf16"].problem()
    assert B.deform_conv_workspace_size(p, False) > B.NOALLOC_SCRATCH_BYTES
    x = torch.empty(p.shapes()["x"], dtype=p.torch_dtype, device="cuda")
    w_off = torch.empty(p.shapes()["w_off"], dtype=p.torch_dtype, device="cuda")
    w = torch.empty(p.shapes()["w"], dtype=p.torch_dtype, device="cuda")
    y = torch.empty(p.shapes()["y"], dtype=p.torch_dtype, device="cuda")
    with pytest.raises(B.DcError) as e:
        B.deform_conv_fwd_noalloc(p, x, w_off, None, w, None, y)
    assert e.value.status == B.DC_ERR_WORKSPACE
