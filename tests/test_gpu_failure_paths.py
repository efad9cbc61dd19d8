"""Failure reporting on the GPU, driven without a fault: a bounded wait that
runs out (an mbarrier nothing arrives on, a few polls) must surface as
DC_ERR_TIMEOUT through dc_device_error and leave the context usable; an
injected launch failure must surface as DC_ERR_CUDA with nothing enqueued,
and the next call must run normally."""
import pytest
import torch

from deformable_convolution_gb300 import binding as B
from deformable_convolution_gb300 import workloads as W

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

DC_OK, DC_ERR_INVALID_ARG, DC_ERR_CUDA, DC_ERR_TIMEOUT = 0, 1, 4, 5


def test_expired_wait_is_reported_as_timeout_and_cleared():
    assert B.device_error(clear=True) == DC_OK
    assert B.selftest_wait_timeout(0) == DC_ERR_INVALID_ARG
    assert B.selftest_wait_timeout(64) == DC_OK
    torch.cuda.synchronize()
    assert B.device_error() == DC_ERR_TIMEOUT
    assert B.device_error(clear=True) == DC_ERR_TIMEOUT  # read, then cleared
    assert B.device_error() == DC_OK
    # the context still works: a layer runs and its wait flag stays clear
    wl = W.WORKLOADS["tiny_f32"]
    p = wl.problem()
    d = {k: (None if v is None else v.cuda()) for k, v in W.generate(wl).items()}
    y, off = B.forward(p, d["x"], d["w_off"], d["b_off"], d["w"], d["offset_add"])
    torch.cuda.synchronize()
    assert torch.isfinite(y).all()
    assert B.device_error() == DC_OK


def test_injected_launch_failure_returns_cuda_error_without_launching():
    wl = W.WORKLOADS["tiny_f32"]
    p = wl.problem()
    d = {k: (None if v is None else v.cuda()) for k, v in W.generate(wl).items()}
    s = p.shapes()
    y = torch.full(s["y"], 7.0, dtype=p.torch_dtype, device="cuda")
    off = torch.empty(s["offset"], dtype=torch.float32, device="cuda")
    ws = B.workspace(p, False, "cuda")
    torch.cuda.synchronize()
    before = B.launch_count()
    assert B.test_fail_launches(-1) == DC_ERR_INVALID_ARG
    assert B.test_fail_launches(1) == DC_OK
    with pytest.raises(B.DcError) as err:
        B.deform_conv_fwd(p, d["x"], d["w_off"], d["b_off"], d["w"], d["offset_add"], y, off, None, ws)
    assert err.value.status == DC_ERR_CUDA
    torch.cuda.synchronize()
    assert B.launch_count() == before          # nothing was launched
    assert torch.all(y == 7.0)                 # and nothing was written
    # the injection is used up: the next call runs
    B.deform_conv_fwd(p, d["x"], d["w_off"], d["b_off"], d["w"], d["offset_add"], y, off, None, ws)
    torch.cuda.synchronize()
    assert B.launch_count() > before
    assert not torch.all(y == 7.0)
    assert B.test_fail_launches(0) == DC_OK
