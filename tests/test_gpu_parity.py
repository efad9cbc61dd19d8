"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded inputs, element by element.

Full-size workloads whose oracle run stays within seconds are compared
whole (the tiny layer, the res3-style layer the benchmark times, the res4
layer).  The two largest (early layer, training-stack layer) run on the GPU at
full batch in the benchmark's launch configuration; their forward is compared
on image 0 (batch items are independent), their backward whole."""
import numpy as np
import pytest
import torch

import oracle
from deformable_convolution_gb300 import binding as B
from deformable_convolution_gb300 import workloads as W

from parity import (TOL, check_layer, f64, gpu_backward, gpu_forward, oracle_backward,
                    oracle_forward, oracle_problem, rel_err)

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


@pytest.mark.parametrize("name", ["tiny_f32", "res3_f32", "res3_bf16", "res4_bf16"])
def test_workload_full(name):
    wl = W.WORKLOADS[name]
    p = wl.problem()
    d = W.generate(wl)
    errs = check_layer(p, d)
    print(name, errs)


@pytest.mark.parametrize("name", ["early_bf16", "stack_bf16"])
def test_workload_batch_slice(name):
    """Full batch in the benchmark's launch configuration.  The forward and the
    per-image gradients are compared on image 0 (batch items are
    independent); the weight gradients, which sum over every image (the
    split-K grad_W GEMM, the per-image partials of the offset-convolution
    backward), against the oracle's full-batch backward."""
    wl = W.WORKLOADS[name]
    p = wl.problem()
    d = W.generate(wl)
    tol = TOL[p.dtype]
    one = {k: (None if v is None else (v[:1].contiguous() if k in ("x", "offset_add", "grad_y") else v))
           for k, v in d.items()}
    p1 = wl.problem(1)
    # forward at full batch, image 0 against the oracle
    y, off, _ = gpu_forward(p, d)
    y_ref, off_ref = oracle_forward(p1, one)
    assert rel_err(f64(y[:1]), y_ref) <= tol
    assert rel_err(f64(off[:1]), off_ref) <= tol
    # backward at full batch with the oracle's offsets for every image
    op = oracle_problem(p)
    off_all = oracle.offsets(op, f64(d["x"]), f64(d["w_off"]), f64(d["b_off"]), f64(d["offset_add"]))
    off32 = torch.from_numpy(off_all).float()
    g = gpu_backward(p, d, off32)
    ref = oracle_backward(p, d, off32.double().numpy())
    for k in ("grad_x", "grad_offset"):
        assert rel_err(f64(g[k][:1]), ref[k][:1]) <= tol, k
        assert rel_err(f64(g[k]), ref[k]) <= tol, k
    for k in ("grad_w", "grad_w_off", "grad_b_off"):
        assert rel_err(f64(g[k]), ref[k]) <= tol, k


def random_inputs(p, seed, off_scale=1.5):
    gen = torch.Generator().manual_seed(seed)
    s = p.shapes()
    dt = p.torch_dtype
    x = (torch.rand(s["x"], generator=gen) * 2 - 1).to(dt)
    w_off = (torch.randn(s["w_off"], generator=gen) * off_scale /
             np.sqrt(p.c_in * p.kh * p.kw / 3.0)).to(dt)
    b_off = torch.randn(s["b_off"], generator=gen) * 0.5
    w = (torch.randn(s["w"], generator=gen) / np.sqrt(p.c_in * p.kh * p.kw)).to(dt)
    add = torch.randn(s["offset"], generator=gen) * 0.5
    gy = torch.randn(s["y"], generator=gen).to(dt)
    return dict(x=x, w_off=w_off, b_off=b_off, w=w, offset_add=add, grad_y=gy)


EDGE_GEOMETRIES = [
    # n, c_in, h, w, c_out, kh, kw, stride, pad, dil, groups
    (1, 1, 1, 1, 1, 1, 1, 1, 0, 1, 1),
    (2, 1, 3, 4, 2, 3, 3, 1, 1, 1, 1),
    (1, 2, 5, 3, 3, 3, 3, 2, 1, 1, 2),
    (3, 3, 7, 9, 5, 3, 3, 1, 2, 2, 3),
    (2, 4, 6, 5, 1, 2, 3, (2, 1), (0, 1), (1, 2), 2),
    (1, 5, 17, 19, 7, 3, 3, 1, 1, 1, 1),
    (2, 8, 33, 21, 16, 3, 3, 2, 1, 1, 4),
    (1, 3, 11, 40, 2, 5, 5, 1, 2, 1, 1),
    (1, 16, 9, 130, 24, 3, 3, 1, 1, 1, 2),
    # kdim and the pixel count multiples of 4 (the float32 tensor-core GEMMs),
    # with ragged k-blocks, pixel tiles and output-channel tiles
    (2, 12, 10, 14, 40, 3, 3, 1, 1, 1, 1),
    (1, 20, 12, 12, 136, 3, 3, 1, 1, 1, 2),
]


@pytest.mark.parametrize("geom", EDGE_GEOMETRIES)
@pytest.mark.parametrize("dtype", [B.DC_F32, B.DC_BF16])
def test_edge_geometries(geom, dtype):
    n, c_in, h, w, c_out, kh, kw, s, pad, dil, groups = geom
    p = B.Problem(n, c_in, h, w, c_out, kh, kw, s, pad, dil, groups, dtype)
    check_layer(p, random_inputs(p, 100 + h * w + c_in))


# One offset group per input channel (8 to 16 of them) with margin 0: every
# channel slice of the fused stage and of the sampling backward holds more than
# four offset groups, many of whose taps leave the window, so the deferred
# slow-tap queue (sized for at most four groups per slice) overflows and is
# drained in place.  (Wider many-group problems exceed the shared memory of
# the plane-major kernels and are refused as unsupported.)
@pytest.mark.parametrize("dtype,c_in", [(B.DC_F32, 8), (B.DC_F32, 12), (B.DC_BF16, 8),
                                         (B.DC_BF16, 16)])
def test_slow_tap_queue_overflow(dtype, c_in):
    p = B.Problem(2, c_in, 14, 18, 8, 3, 3, 1, 1, 1, c_in, dtype, 0)
    d = random_inputs(p, 900 + c_in, off_scale=3.0)
    cnt = torch.zeros(1, dtype=torch.int64, device="cuda")
    dd = {k: v.cuda() for k, v in d.items()}
    B.forward(p, dd["x"], dd["w_off"], dd["b_off"], dd["w"], dd["offset_add"], slowpath_count=cnt)
    torch.cuda.synchronize()
    taps = p.n * c_in * p.kh * p.kw * p.ho * p.wo
    assert int(cnt.item()) > taps // 4  # many taps take the global path
    errs = check_layer(p, d)
    print(c_in, errs)


@pytest.mark.parametrize("dtype,c_in,layout", [
    (B.DC_F32, 16, B.DC_COL_PLANE_MAJOR), (B.DC_BF16, 16, B.DC_COL_PLANE_MAJOR),
    (B.DC_BF16, 64, B.DC_COL_PIXEL_MAJOR)])
def test_fast_and_slow_paths_agree_bitwise(dtype, c_in, layout):
    """Margin 0 sends most taps to the global-memory path, a wide margin keeps
    them on chip: sampled at the same offsets, the deformed maps must be
    identical bit for bit (both the plane-major path and the channels-last
    one), and the fused stage's offsets must not depend on the margin."""
    p = B.Problem(2, c_in, 24, 29, 8, 3, 3, 1, 1, 1, 2, dtype)
    assert B.col_layout(p) == layout
    d = random_inputs(p, 7, off_scale=3.0)
    dd = {k: v.cuda() for k, v in d.items()}
    off0 = torch.empty(p.shapes()["offset"], dtype=torch.float32, device="cuda")
    B.deform_conv_offsets(p, dd["x"], dd["w_off"], dd["b_off"], dd["offset_add"], off0)
    cols, counts, offs = [], [], []
    for margin in (0, 2, 12):
        q = B.Problem(2, c_in, 24, 29, 8, 3, 3, 1, 1, 1, 2, dtype, margin)
        assert B.col_layout(q) == layout
        col = torch.empty(B.col_shape(q), dtype=q.torch_dtype, device="cuda")
        cnt = torch.zeros(1, dtype=torch.int64, device="cuda")
        B.deform_conv_sample(q, dd["x"], None, None, None, off0, col, slowpath_count=cnt)
        off = torch.empty_like(off0)
        B.deform_conv_offsets(q, dd["x"], dd["w_off"], dd["b_off"], dd["offset_add"], off)
        torch.cuda.synchronize()
        cols.append(col.cpu())
        counts.append(int(cnt.item()))
        offs.append(off.cpu())
    assert counts[0] > counts[1] > counts[2]
    bits = torch.int16 if dtype else torch.int32
    assert torch.equal(cols[0].view(bits), cols[1].view(bits))
    assert torch.equal(cols[0].view(bits), cols[2].view(bits))
    for o in offs:
        assert rel_err(o.double().numpy(), off0.cpu().double().numpy()) <= 1e-6


@pytest.mark.parametrize("dtype,c_in,groups", [(B.DC_F32, 6, 3), (B.DC_BF16, 6, 3),
                                               (B.DC_BF16, 128, 2), (B.DC_BF16, 64, 4)])
def test_column_matches_oracle(dtype, c_in, groups):
    # 13 x 11 for the plane-major path; the channels-last one needs H*W % 8 == 0
    w = 11 if c_in % 64 else 16
    p = B.Problem(2, c_in, 13, w, 4, 3, 3, 1, 1, 1, groups, dtype)
    d = random_inputs(p, 8)
    dd = {k: v.cuda() for k, v in d.items()}
    col = torch.empty(B.col_shape(p), dtype=p.torch_dtype, device="cuda")
    off = torch.empty(p.shapes()["offset"], dtype=torch.float32, device="cuda")
    B.deform_conv_sample(p, dd["x"], dd["w_off"], dd["b_off"], dd["offset_add"], None, col, off)
    torch.cuda.synchronize()
    op = oracle_problem(p)
    off_ref = oracle.offsets(op, f64(d["x"]), f64(d["w_off"]), f64(d["b_off"]), f64(d["offset_add"]))
    assert rel_err(f64(off), off_ref) <= 1e-5
    # sample both at the same offsets
    col2 = torch.empty_like(col)
    off32 = torch.from_numpy(off_ref).float().cuda()
    B.deform_conv_sample(p, dd["x"], None, None, None, off32, col2)
    torch.cuda.synchronize()
    ref = oracle.column(op, f64(d["x"]), off32.double().cpu().numpy())  # [n, c, k, ho, wo]
    if B.col_layout(p) == B.DC_COL_PIXEL_MAJOR:  # [n][pixel][tap][channel]
        ref = ref.reshape(p.n, p.c_in, 9, p.ho * p.wo).transpose(0, 3, 2, 1)
    else:  # [channel * 9 + tap][n][pixel]
        ref = ref.reshape(p.n, p.c_in * 9, p.ho * p.wo).transpose(1, 0, 2)
    tol = 1e-6 if dtype == B.DC_F32 else 8e-3
    assert rel_err(f64(col2), ref) <= tol


def test_zero_and_integer_offsets():
    p = B.Problem(2, 8, 12, 10, 6, 3, 3, 1, 1, 1, 2, B.DC_F32)
    d = random_inputs(p, 9)
    d["w_off"] = torch.zeros_like(d["w_off"])
    d["offset_add"] = None
    d["b_off"] = torch.zeros_like(d["b_off"])
    check_layer(p, d)
    d["b_off"] = torch.randint(-3, 4, d["b_off"].shape).float()
    check_layer(p, d)


def test_far_outside_offsets():
    p = B.Problem(1, 4, 8, 8, 3, 3, 3, 1, 1, 1, 1, B.DC_F32)
    d = random_inputs(p, 10)
    d["offset_add"] = torch.full(p.shapes()["offset"], 1e4)
    y, off, cnt = gpu_forward(p, d)
    assert torch.count_nonzero(y).item() == 0
    g = gpu_backward(p, d, off.cpu())
    assert torch.count_nonzero(g["grad_offset"]).item() == 0


def test_hand_worked_layer():
    import json
    import os
    gold = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")))
    L = gold["layer"]
    p = B.Problem(1, 1, 2, 3, 1, 1, 1, 1, 0, 1, 1, B.DC_F32)
    x = torch.tensor(gold["plane"], dtype=torch.float32).reshape(1, 1, 2, 3).cuda()
    y, off = B.forward(p, x, torch.zeros(2, 1, 1, 1, device="cuda"),
                       torch.tensor(L["b_off"], device="cuda"),
                       torch.full((1, 1, 1, 1), L["w_main"], device="cuda"))
    assert y.cpu().reshape(2, 3).tolist() == L["y"]


def test_repeated_calls_are_deterministic_forward():
    wl = W.WORKLOADS["res3_bf16"]
    p = wl.problem()
    d = W.generate(wl)
    y1, off1, _ = gpu_forward(p, d)
    y2, off2, _ = gpu_forward(p, d)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    assert torch.equal(off1, off2)


# bf16 problem whose GCOL GEMM runs on the tensor cores (C_in * K and Ho * Wo
# multiples of 8), so K3 accumulates grad_x in fixed point scaled from the
# per-tile max |gcol|; the relative error must not depend on the gradient's
# magnitude
SCALED_PROBLEM = (2, 32, 16, 16, 16, 3, 3, 1, 1, 1, 1)


@pytest.mark.parametrize("scale", [1e-30, 1e-8, 1e6, 1e25])
def test_backward_parity_at_extreme_gradient_scales(scale):
    n, c_in, h, w, c_out, kh, kw, s, pad, dil, groups = SCALED_PROBLEM
    p = B.Problem(n, c_in, h, w, c_out, kh, kw, s, pad, dil, groups, B.DC_BF16)
    d = random_inputs(p, 77)
    d["grad_y"] = (d["grad_y"].float() * scale).to(p.torch_dtype)
    errs = check_layer(p, d)
    print(scale, errs)


def test_backward_non_finite_gradient_propagates():
    n, c_in, h, w, c_out, kh, kw, s, pad, dil, groups = SCALED_PROBLEM
    p = B.Problem(n, c_in, h, w, c_out, kh, kw, s, pad, dil, groups, B.DC_BF16)
    d = random_inputs(p, 78)
    d["grad_y"][0, 3, 5, 7] = float("nan")
    y, off, _ = gpu_forward(p, d)
    g = gpu_backward(p, d, off.cpu())
    assert torch.isnan(g["grad_x"][0]).any()
    # image 1 never sees the NaN: its gradient stays finite
    assert torch.isfinite(g["grad_x"][1]).all()
    assert B.device_error() == 0


@pytest.mark.parametrize("dtype", [B.DC_F32, B.DC_BF16])
def test_unfused_pipeline_matches_fused_stage(dtype):
    """Offsets through HBM (deform_conv_offsets, then deform_conv_sample with
    offset_in) give the fused stage's offsets and deformed map bit for bit,
    and the offsets match the oracle."""
    wl = W.WORKLOADS["res3_bf16" if dtype == B.DC_BF16 else "res3_f32"]
    p = wl.problem()
    d = {k: (None if v is None else v.cuda()) for k, v in W.generate(wl).items()}
    s = p.shapes()
    col_f = torch.empty(B.col_shape(p), dtype=p.torch_dtype, device="cuda")
    off_f = torch.empty(s["offset"], dtype=torch.float32, device="cuda")
    B.deform_conv_sample(p, d["x"], d["w_off"], d["b_off"], d["offset_add"], None, col_f, off_f)
    off_u = torch.empty_like(off_f)
    B.deform_conv_offsets(p, d["x"], d["w_off"], d["b_off"], d["offset_add"], off_u)
    col_u = torch.empty_like(col_f)
    B.deform_conv_sample(p, d["x"], None, None, None, off_u, col_u)
    torch.cuda.synchronize()
    assert torch.equal(off_u, off_f)
    assert torch.equal(col_u.view(torch.int16) if dtype == B.DC_BF16 else col_u,
                       col_f.view(torch.int16) if dtype == B.DC_BF16 else col_f)
    cpu = {k: (None if v is None else v.cpu()) for k, v in d.items()}
    _, off_ref = oracle_forward(p, cpu)
    assert rel_err(f64(off_u), off_ref) <= TOL[dtype]


def _margin_need_reference(p, off, R, TW):
    """Per-tap margin need recomputed on the host from the offsets (float32
    positions, as the kernels form them) for bands of R rows x TW columns."""
    o = off.cpu().numpy().astype(np.float32)
    n, m2, ho, wo = o.shape
    K = p.kh * p.kw
    G = m2 // (2 * K)
    dy = o[:, 0::2].reshape(n, G, K, ho, wo)
    dx = o[:, 1::2].reshape(n, G, K, ho, wo)
    k = np.arange(K)
    i, j = k // p.kw, k % p.kw
    by = (np.arange(ho)[None, :] * p.stride[0] - p.pad[0] + i[:, None] * p.dil[0]).astype(np.float32)
    bx = (np.arange(wo)[None, :] * p.stride[1] - p.pad[1] + j[:, None] * p.dil[1]).astype(np.float32)
    py = by[None, None, :, :, None] + dy
    px = bx[None, None, :, None, :] + dx
    inside = (py >= -1) & (py < p.h) & (px >= -1) & (px < p.w)
    # receptive field of each pixel's band
    ylo = (np.arange(ho) // R * R * p.stride[0] - p.pad[0])[None, None, None, :, None]
    xlo = (np.arange(wo) // TW * TW * p.stride[1] - p.pad[1])[None, None, None, None, :]
    rows = (R - 1) * p.stride[0] + (p.kh - 1) * p.dil[0] + 1
    cols = (TW - 1) * p.stride[1] + (p.kw - 1) * p.dil[1] + 1

    def beyond(pos, lo, extent):
        c = np.floor(pos)
        return np.minimum(np.maximum(0, np.maximum(lo - c, c + 2 - (lo + extent))),
                          B.MARGIN_BINS - 1)
    b = np.where(inside, np.maximum(beyond(py, ylo, rows), beyond(px, xlo, cols)), 0)
    return np.bincount(b.astype(np.int64).ravel(), minlength=B.MARGIN_BINS)


def test_margin_histogram_and_suggested_margin_bound_the_slow_path():
    wl = W.WORKLOADS["res3_bf16"]
    p = wl.problem()
    d = W.generate(wl)
    _, off, _ = gpu_forward(p, d)
    hist = torch.zeros(B.MARGIN_BINS, dtype=torch.int64, device="cuda")
    B.deform_conv_margin_histogram(p, off, hist)
    torch.cuda.synchronize()
    h = hist.cpu().numpy()
    # the histogram is taken for the output tile the fused stage stages
    R, TW = B.sample_tile(p)
    assert np.array_equal(h, _margin_need_reference(p, off, R, TW))
    total = int(h.sum())
    assert total == p.n * p.offset_groups * p.kh * p.kw * off.shape[2] * off.shape[3]
    # at the default margin (3) exactly the taps above bin 3 took the slow path
    _, _, slow3 = gpu_forward(p, d)
    assert slow3 == int(h[4:].sum())
    for frac in (0.0, 0.01, 0.2):
        m = B.dc_suggest_margin(p, h.tolist(), frac, True)
        assert m >= 0
        pm = B.Problem(p.n, p.c_in, p.h, p.w, p.c_out, p.kh, p.kw, p.stride, p.pad, p.dil,
                       p.offset_groups, p.dtype, m)
        # at margin m the stage may stage another tile shape (a wider margin
        # can leave less room): measure again for that shape, which closes the loop
        Rm, TWm = B.sample_tile(pm)
        hm_dev = torch.zeros(B.MARGIN_BINS, dtype=torch.int64, device="cuda")
        B.deform_conv_margin_histogram(pm, off, hm_dev)
        torch.cuda.synchronize()
        hm = hm_dev.cpu().numpy()
        assert np.array_equal(hm, _margin_need_reference(pm, off, Rm, TWm))
        _, _, slow = gpu_forward(pm, d)
        assert slow == int(hm[m + 1:].sum()), (frac, m, slow)
        if (Rm, TWm) == (R, TW):
            assert slow <= frac * total, (frac, m, slow)
        if frac == 0.01:
            check_layer(pm, d)


def test_backward_after_forward_reuses_the_map():
    """deform_conv_bwd_after_fwd takes the deformed map the forward call left
    in the workspace: its gradients match the oracle and the replaying
    backward's.  Two backward runs agree only to bf16 level on grad_x and
    grad_w_off: the offset gradient is summed over channel slices with float
    atomics (order-dependent in the last bit) and then rounded to bf16 for the
    offset-convolution backward's tensor-core contractions."""
    wl = W.WORKLOADS["res3_bf16"]
    p = wl.problem()
    d = {k: (None if v is None else v.cuda()) for k, v in W.generate(wl).items()}
    s = p.shapes()
    ws = B.workspace(p, True, "cuda")
    y = torch.empty(s["y"], dtype=p.torch_dtype, device="cuda")
    off = torch.empty(s["offset"], dtype=torch.float32, device="cuda")
    B.deform_conv_fwd(p, d["x"], d["w_off"], d["b_off"], d["w"], d["offset_add"], y, off, None, ws)

    def bwd(after):
        out = {k: torch.empty(s[sh], dtype=torch.float32, device="cuda") for k, sh in
               (("grad_x", "x"), ("grad_w_off", "w_off"), ("grad_b_off", "b_off"), ("grad_w", "w"),
                ("grad_offset", "offset"))}
        B.deform_conv_bwd(p, d["x"], d["w_off"], d["w"], off, d["grad_y"], out["grad_x"],
                          out["grad_w_off"], out["grad_b_off"], out["grad_w"], out["grad_offset"],
                          ws, after_fwd=after)
        torch.cuda.synchronize()
        return out
    reused = bwd(True)
    replayed = bwd(False)
    for k in ("grad_offset", "grad_w", "grad_b_off"):
        assert rel_err(f64(reused[k]), f64(replayed[k])) <= 1e-5, k
    for k in ("grad_x", "grad_w_off"):
        assert rel_err(f64(reused[k]), f64(replayed[k])) <= 5e-3, k
    cpu = {k: (None if v is None else v.cpu()) for k, v in d.items()}
    ref = oracle_backward(p, cpu, off.cpu().double().numpy())
    for k in ("grad_x", "grad_w", "grad_w_off", "grad_b_off", "grad_offset"):
        assert rel_err(f64(reused[k]), ref[k]) <= TOL[p.dtype], k


# The forward pass with the deformed map sampled straight into the GEMM's
# shared-memory operand (no column buffer): bf16, C_in*Kh*Kw and Ho*Wo
# multiples of 8.  Geometries: offset groups, stride + dilation, a partial
# last k-block and pixel tile with two output-channel tiles.
SAMPLED_GEOMETRIES = [
    (2, 16, 12, 10, 24, 3, 3, 1, 1, 1, 2),
    (1, 8, 17, 16, 8, 3, 3, 2, 2, 2, 1),
    (1, 40, 20, 20, 136, 3, 3, 1, 1, 1, 1),
]


def sampled_forward(p, d):
    dd = {k: (None if v is None else v.cuda()) for k, v in d.items()}
    s = p.shapes()
    y = torch.empty(s["y"], dtype=p.torch_dtype, device="cuda")
    off = torch.empty(s["offset"], dtype=torch.float32, device="cuda")
    B.deform_conv_fwd_sampled_gemm(p, dd["x"], dd["w_off"], dd["b_off"], dd["w"], dd["offset_add"],
                                   y, off)
    torch.cuda.synchronize()
    return y, off


@pytest.mark.parametrize("geom", SAMPLED_GEOMETRIES)
def test_sampled_gemm_forward_matches_oracle_and_two_kernel_path(geom):
    n, c_in, h, w, c_out, kh, kw, s, pad, dil, groups = geom
    p = B.Problem(n, c_in, h, w, c_out, kh, kw, s, pad, dil, groups, B.DC_BF16)
    d = random_inputs(p, 300 + h * w + c_in)
    y, off = sampled_forward(p, d)
    y_ref, off_ref = oracle_forward(p, d)
    assert rel_err(f64(y), y_ref) <= TOL[B.DC_BF16]
    assert rel_err(f64(off), off_ref) <= TOL[B.DC_BF16]
    y2, off2, _ = gpu_forward(p, d)
    assert torch.equal(off, off2)
    # same deformed-map values; the GEMMs may differ in tile width, so the
    # bf16 outputs agree up to a rounding of the fp32 sums
    assert rel_err(f64(y), f64(y2)) <= 1e-2


def test_sampled_gemm_forward_matches_two_kernel_forward_res3():
    """res3 bf16 takes the channels-last path in the two-kernel forward (its
    offset convolution and GEMM sum in another order than the sampled-operand
    kernel's), so the two agree to rounding: offsets to float32 summation
    order, y to a bf16 rounding of the fp32 sums.  Both match the oracle."""
    wl = W.WORKLOADS["res3_bf16"]
    p = wl.problem()
    d = W.generate(wl)
    y, off = sampled_forward(p, d)
    y2, off2, _ = gpu_forward(p, d)
    assert rel_err(f64(off), f64(off2)) <= 1e-5
    assert rel_err(f64(y), f64(y2)) <= 1e-2
    y_ref, _ = oracle_forward(p, d)
    assert rel_err(f64(y), y_ref) <= TOL[B.DC_BF16]


def test_sampled_gemm_forward_early_layer_full_batch():
    """The early layer at full batch, image 0 against the oracle (batch items
    are independent), every image against the two-kernel forward."""
    wl = W.WORKLOADS["early_bf16"]
    p = wl.problem()
    d = W.generate(wl)
    y, off = sampled_forward(p, d)
    one = {k: (None if v is None else (v[:1].contiguous() if k in ("x", "offset_add", "grad_y") else v))
           for k, v in d.items()}
    y_ref, off_ref = oracle_forward(wl.problem(1), one)
    assert rel_err(f64(y[:1]), y_ref) <= TOL[B.DC_BF16]
    assert rel_err(f64(off[:1]), off_ref) <= TOL[B.DC_BF16]
    y2, off2, _ = gpu_forward(p, d)
    assert rel_err(f64(off), f64(off2)) <= 1e-5
    assert rel_err(f64(y), f64(y2)) <= 1e-2


# One offset group, bf16, C_in a multiple of 64: the backward runs the
# channels-last sampling backward (pixel-major gcol from the tensor-core GEMM,
# grad_x gathered per window position into an NHWC accumulator).  Geometries:
# 64 / 128 / 256 channels (2, 4, 8 channels per lane), stride 2, dilation 2
# with a ragged last row of tiles, a 3 x 4 filter; 136 output channels over
# 8 images of 36 x 36 (forward GEMM tiles over the flat pixel index of all
# images, 32-pixel chunks crossing image boundaries, a ragged second half of
# output channels); then margin 0 with wide offsets, where most samples leave
# the window and take the global path.
CL_BACKWARD_GEOMETRIES = [
    (2, 64, 20, 24, 32, 3, 3, 1, 1, 1, 1),
    (1, 128, 18, 32, 40, 3, 3, 2, 1, 1, 1),
    (2, 256, 15, 16, 24, 3, 3, 1, 2, 2, 1),
    (1, 64, 16, 24, 16, 3, 4, 1, 1, 1, 1),
    (8, 64, 36, 36, 136, 3, 3, 1, 1, 1, 1),
]


def backward_kernels(p, d):
    """Names of the kernels one backward call launches."""
    dd = {k: (None if v is None else v.cuda()) for k, v in d.items()}
    s = p.shapes()
    ws = B.workspace(p, True, "cuda")
    off = torch.zeros(s["offset"], dtype=torch.float32, device="cuda")
    out = [torch.empty(s[sh], dtype=torch.float32, device="cuda")
           for sh in ("x", "w_off", "b_off", "w", "offset")]
    torch.cuda.synchronize()
    B.kernel_timing(True)
    B.deform_conv_bwd(p, dd["x"], dd["w_off"], dd["w"], off, dd["grad_y"], *out, ws)
    names = [n for n, _ in B.kernel_times()]
    B.kernel_timing(False)
    return names


@pytest.mark.parametrize("geom", CL_BACKWARD_GEOMETRIES)
def test_channels_last_backward_matches_oracle(geom):
    n, c_in, h, w, c_out, kh, kw, s, pad, dil, groups = geom
    p = B.Problem(n, c_in, h, w, c_out, kh, kw, s, pad, dil, groups, B.DC_BF16)
    assert B.col_layout(p) == B.DC_COL_PIXEL_MAJOR
    d = random_inputs(p, 500 + h * w + c_in)
    assert "k3_cl_bwd" in backward_kernels(p, d)
    errs = check_layer(p, d)
    print(geom, errs)


def test_channels_last_backward_global_path_matches_oracle():
    n, c_in, h, w, c_out, kh, kw, s, pad, dil, groups = CL_BACKWARD_GEOMETRIES[0]
    p = B.Problem(n, c_in, h, w, c_out, kh, kw, s, pad, dil, groups, B.DC_BF16, 0)
    d = random_inputs(p, 600, off_scale=4.0)
    assert "k3_cl_bwd" in backward_kernels(p, d)
    errs = check_layer(p, d)
    print(errs)
