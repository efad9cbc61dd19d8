"""GPU parity of the training stack: deformable layers with ReLU between them
(the networks the explainer page "DefT: Boosting Scalability of Deformable
Convolution Operations on GPUs" trains: deformable layers throughout a ResNet,
"What people did before, and where it broke" and "Why it works / Fixing the
slowest stage lifts the whole layer").

The oracle runs the stack layer by layer in fp64 on image 0; each activation
and each gradient between layers is stored in the layers' dtype (bf16) on both
sides, so the oracle rounds it the same way (to float32, then to bf16,
nearest even).  The CUDA path is compared layer by layer at the oracle's
inputs (forward, backward at the oracle's float32 offsets, the ReLU kernels
bit for bit, and the backward with the ReLU below fused), then as a chain
through the stack runner on the one-image slice and at full batch (forward
output of image 0, and the top layer's weight gradient, which depends on no
offset gradient)."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from deformable_convolution_gb300 import binding as B
from deformable_convolution_gb300 import stack as S
from deformable_convolution_gb300 import workloads as W

from parity import TOL, f64, oracle_problem, rel_err

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


# The forward with the following ReLU fused into its main GEMM's epilogue
# (out_relu) is bit for bit dc_relu_fwd of the plain forward, on every
# forward GEMM: the channels-last tcgen05 GEMM (per-image tiles, and tiles over
# the flat pixel index of all images with chunks crossing image boundaries),
# the plane-major bf16 tcgen05 GEMM, the float32 TF32 GEMM, the CUDA-core GEMM
# (rows that are not 16-byte aligned) and the sampled-operand forward.
FUSED_RELU_CASES = [
    ((2, 64, 20, 24, 32, 3, 3, 1, 1, 1, 1), B.DC_BF16, "fwd"),
    ((8, 64, 36, 36, 136, 3, 3, 1, 1, 1, 1), B.DC_BF16, "fwd"),
    ((2, 16, 12, 10, 24, 3, 3, 1, 1, 1, 2), B.DC_BF16, "fwd"),
    ((2, 12, 10, 14, 40, 3, 3, 1, 1, 1, 1), B.DC_F32, "fwd"),
    ((1, 5, 17, 19, 7, 3, 3, 1, 1, 1, 1), B.DC_F32, "fwd"),
    ((2, 16, 12, 10, 24, 3, 3, 1, 1, 1, 2), B.DC_BF16, "sampled"),
]


@pytest.mark.parametrize("geom,dtype,entry", FUSED_RELU_CASES)
def test_fused_relu_forward_is_relu_of_the_forward(geom, dtype, entry):
    import dataclasses
    n, c_in, h, w, c_out, kh, kw, s, pad, dil, groups = geom
    p = B.Problem(n, c_in, h, w, c_out, kh, kw, s, pad, dil, groups, dtype)
    pr = dataclasses.replace(p, out_relu=1)
    g = torch.Generator().manual_seed(31 + c_in + c_out)
    sh = p.shapes()
    dt = p.torch_dtype
    x = torch.randn(sh["x"], generator=g).to(dt).cuda()
    w_off = (0.05 * torch.randn(sh["w_off"], generator=g)).to(dt).cuda()
    b_off = torch.zeros(sh["b_off"]).cuda()
    wm = (torch.randn(sh["w"], generator=g) / (c_in * kh * kw) ** 0.5).to(dt).cuda()
    outs = []
    for q in (p, pr):
        y = torch.empty(sh["y"], dtype=dt, device="cuda")
        off = torch.empty(sh["offset"], dtype=torch.float32, device="cuda")
        if entry == "sampled":
            B.deform_conv_fwd_sampled_gemm(q, x, w_off, b_off, wm, None, y, off)
        else:
            ws = B.workspace(q, False, "cuda")
            B.deform_conv_fwd(q, x, w_off, b_off, wm, None, y, off, None, ws)
        outs.append(y)
    ref = torch.empty_like(outs[0])
    B.dc_relu_fwd(outs[0], ref)
    torch.cuda.synchronize()
    bits = torch.int16 if dtype == B.DC_BF16 else torch.int32
    assert (outs[0] < 0).any() and (outs[0] > 0).any()
    assert torch.equal(outs[1].view(bits), ref.view(bits))


# The backward through the ReLU below (in_relu): grad_x in the layer's dtype,
# +0 where x is not above zero and elsewhere the float32 grad_x rounded as
# dc_relu_bwd rounds it.  Where the channels-last offset-convolution backward
# writes grad_x, it applies the ReLU in that store (16-byte rows, and a row
# length that is not a multiple of four: the per-element store; 64 and 128
# channels per CTA); the others (a channels-last problem with stride 2, the
# plane-major ones) accumulate grad_x in a float32 scratch and run the ReLU
# kernel.  Columns: geometry, dtype, channels-last, ReLU in the grad_x store.
FUSED_RELU_BWD_CASES = [
    ((2, 64, 20, 24, 32, 3, 3, 1, 1, 1, 1), B.DC_BF16, True, True),
    ((2, 64, 20, 22, 32, 3, 3, 1, 1, 1, 1), B.DC_BF16, True, True),
    ((1, 128, 16, 32, 40, 3, 3, 1, 1, 1, 1), B.DC_BF16, True, True),
    ((1, 128, 18, 32, 40, 3, 3, 2, 1, 1, 1), B.DC_BF16, True, False),
    ((2, 16, 12, 10, 24, 3, 3, 1, 1, 1, 2), B.DC_BF16, False, False),
    ((2, 12, 10, 14, 40, 3, 3, 1, 1, 1, 1), B.DC_F32, False, False),
    ((1, 5, 17, 19, 7, 3, 3, 1, 1, 1, 1), B.DC_F32, False, False),
]


@pytest.mark.parametrize("geom,dtype,channels_last,in_store", FUSED_RELU_BWD_CASES)
def test_fused_relu_backward_is_relu_bwd_of_the_backward(geom, dtype, channels_last, in_store):
    import dataclasses
    n, c_in, h, w, c_out, kh, kw, s, pad, dil, groups = geom
    p = B.Problem(n, c_in, h, w, c_out, kh, kw, s, pad, dil, groups, dtype)
    pr = dataclasses.replace(p, in_relu=1)
    assert (B.col_layout(p) == B.DC_COL_PIXEL_MAJOR) == channels_last
    g = torch.Generator().manual_seed(53 + c_in + w)
    sh = p.shapes()
    dt = p.torch_dtype
    x = torch.relu(torch.randn(sh["x"], generator=g)).to(dt).cuda()  # a ReLU's output
    w_off = (0.05 * torch.randn(sh["w_off"], generator=g)).to(dt).cuda()
    wm = (torch.randn(sh["w"], generator=g) / (c_in * kh * kw) ** 0.5).to(dt).cuda()
    off = (0.7 * torch.randn(sh["offset"], generator=g)).cuda()
    gy = torch.randn(sh["y"], generator=g).to(dt).cuda()
    plain = B.backward(p, x, w_off, wm, off, gy)
    B.kernel_timing(True)
    fused = B.backward(pr, x, w_off, wm, off, gy)
    names = [k for k, _ in B.kernel_times()]
    B.kernel_timing(False)
    ref = torch.empty_like(x)
    B.dc_relu_bwd(x, plain["grad_x"], ref)
    torch.cuda.synchronize()
    assert fused["grad_x"].dtype == dt
    # a separate ReLU kernel only where grad_x is not written by the
    # channels-last offset-convolution backward
    assert ("relu_bwd" in names) == (not in_store), names
    assert ("k4cl_input" in names) == in_store, names
    got, want = fused["grad_x"].double().cpu(), ref.double().cpu()
    masked = x.cpu() <= 0
    assert masked.any() and (~masked).any()
    bits = torch.int16 if dtype == B.DC_BF16 else torch.int32
    assert torch.all(fused["grad_x"].cpu()[masked].view(bits) == 0)  # +0
    # float32 atomics sum grad_x in a run-dependent order: the float32 values
    # differ by summation rounding (1e-5 of the tensor's scale bounds it,
    # cancellation included), then by one bf16 rounding step at most
    scale = float(want.abs().max())
    assert scale > 0
    rel = 2.0 ** -7 if dtype == B.DC_BF16 else 0.0
    assert torch.all((got - want).abs() <= rel * torch.maximum(got.abs(), want.abs()) + 1e-5 * scale)
    for k in ("grad_w", "grad_w_off", "grad_b_off", "grad_offset"):
        assert rel_err(f64(fused[k]), f64(plain[k])) <= 1e-4, k


def to_bf16_via_f32(a):
    """fp64 -> float32 -> bf16 (nearest even at each step), back as fp64."""
    return torch.from_numpy(np.asarray(a, dtype=np.float64)).float().to(torch.bfloat16).double().numpy()


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("count", [1, 7, 8, 4099, 1 << 20])
def test_relu_kernels_match_the_definition(dtype, count):
    gen = torch.Generator().manual_seed(count)
    y = (torch.randn(count, generator=gen) * 3).to(dtype)
    special = torch.tensor([0.0, -0.0, float("nan"), float("inf"), -float("inf"), 1e-30, -1e-30],
                           dtype=dtype)
    y[:min(count, special.numel())] = special[:min(count, special.numel())]
    g = torch.randn(count, generator=gen)
    yd, gd = y.cuda(), g.cuda()
    out = torch.empty_like(yd)
    B.dc_relu_fwd(yd, out)
    gin = torch.empty_like(yd)
    B.dc_relu_bwd(out, gd, gin)
    inplace = yd.clone()
    B.dc_relu_fwd(inplace, inplace)
    torch.cuda.synchronize()
    want = torch.from_numpy(oracle.relu(y.double().numpy())).to(dtype)
    bits = torch.int16 if dtype == torch.bfloat16 else torch.int32
    nan = torch.isnan(want)
    for got in (out.cpu(), inplace.cpu()):
        # NaN stays NaN (the hardware may return its canonical NaN); every
        # other element bit for bit, +0 for the zeros
        assert torch.equal(torch.isnan(got), nan)
        assert torch.equal(got.view(bits)[~nan], want.view(bits)[~nan])
    gwant = torch.from_numpy(oracle.relu_grad(want.double().numpy(), g.double().numpy()))
    gwant = gwant.float().to(dtype)
    assert torch.equal(gin.cpu().view(bits), gwant.view(bits))


def oracle_stack(p1, x0, layers, gy, backward=True):
    """The stack in fp64 on one image: per layer the oracle's forward, ReLU,
    storage rounding; then (unless backward is False) the backward from the
    top at each layer's float32 offsets, the gradient through the ReLU stored
    rounded as well."""
    op = oracle_problem(p1)
    L = len(layers)
    xs, ys, offs = [f64(x0)], [], []
    for l, q in enumerate(layers):
        y, off = oracle.forward(op, xs[l], f64(q["w_off"]), f64(q["b_off"]), f64(q["w"]))
        ys.append(y)
        offs.append(off.astype(np.float32).astype(np.float64))
        if l + 1 < L:
            xs.append(to_bf16_via_f32(oracle.relu(y)))
    gys = [None] * (L - 1) + [f64(gy)]
    grads = [None] * L
    for l in reversed(range(L) if backward else []):
        q = layers[l]
        grads[l] = oracle.backward(op, xs[l], f64(q["w_off"]), f64(q["w"]), offs[l], gys[l])
        if l > 0:
            gx32 = grads[l]["grad_x"].astype(np.float32).astype(np.float64)
            gys[l - 1] = to_bf16_via_f32(oracle.relu_grad(xs[l], gx32))
    return xs, ys, offs, gys, grads


def test_stack_layer_by_layer_and_chained_on_one_image():
    wl = W.WORKLOADS["stack_bf16"]
    x0, layers, gy = W.generate_stack(wl)
    p1 = wl.problem(1)
    x0, gy = x0[:1].contiguous(), gy[:1].contiguous()
    xs, ys, offs, gys, grads = oracle_stack(p1, x0, layers, gy)
    tol = TOL[p1.dtype]
    dt = p1.torch_dtype
    bf = lambda a: torch.from_numpy(a).to(dt).cuda()  # noqa: E731  (values already bf16)
    dev_layers = [{k: v.cuda() for k, v in q.items()} for q in layers]
    for l, q in enumerate(dev_layers):
        y, off = B.forward(p1, bf(xs[l]), q["w_off"], q["b_off"], q["w"])
        g = B.backward(p1, bf(xs[l]), q["w_off"], q["w"],
                       torch.from_numpy(offs[l]).float().cuda(), bf(gys[l]))
        torch.cuda.synchronize()
        assert rel_err(f64(y), ys[l]) <= tol, l
        assert rel_err(f64(off), offs[l]) <= tol, l
        for k in ("grad_x", "grad_w", "grad_w_off", "grad_b_off", "grad_offset"):
            assert rel_err(f64(g[k]), grads[l][k]) <= tol, (l, k)
        if l + 1 < len(layers):
            act = torch.empty(p1.shapes()["x"], dtype=dt, device="cuda")
            B.dc_relu_fwd(bf(to_bf16_via_f32(ys[l])), act)
            torch.cuda.synchronize()
            assert np.array_equal(f64(act), xs[l + 1]), l
        if l > 0:
            gin = torch.empty(p1.shapes()["y"], dtype=dt, device="cuda")
            B.dc_relu_bwd(bf(xs[l]), torch.from_numpy(grads[l]["grad_x"]).float().cuda(), gin)
            # the same gradient from the backward with the ReLU fused (in_relu)
            gf = B.backward(dataclasses.replace(p1, in_relu=1), bf(xs[l]), q["w_off"], q["w"],
                            torch.from_numpy(offs[l]).float().cuda(), bf(gys[l]))
            torch.cuda.synchronize()
            assert np.array_equal(f64(gin), gys[l - 1]), l
            assert rel_err(f64(gf["grad_x"]), gys[l - 1]) <= tol, l
            assert np.all(f64(gf["grad_x"])[xs[l] <= 0] == 0), l
    # the chain through the stack runner, on the same image
    st = S.Stack(p1, dev_layers, "cuda")
    st.step(x0.cuda(), gy.cuda())
    torch.cuda.synchronize()
    assert rel_err(f64(st.y[-1]), ys[-1]) <= tol
    assert rel_err(f64(st.grads[-1]["grad_w"]), grads[-1]["grad_w"]) <= tol


def test_stack_full_batch_matches_the_oracle_on_image_0():
    wl = W.WORKLOADS["stack_bf16"]
    x0, layers, gy = W.generate_stack(wl)
    p = wl.problem()
    st = S.Stack(p, [{k: v.cuda() for k, v in q.items()} for q in layers], "cuda")
    st.step(x0.cuda(), gy.cuda())
    torch.cuda.synchronize()
    p1 = wl.problem(1)
    _, ys, _, _, _ = oracle_stack(p1, x0[:1].contiguous(), layers, gy[:1].contiguous(),
                                  backward=False)
    assert rel_err(f64(st.y[-1][:1]), ys[-1]) <= TOL[p.dtype]
    assert B.device_error() == 0
