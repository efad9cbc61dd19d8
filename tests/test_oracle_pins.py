"""Pins for the fp64 oracle: each test ties it to something other than itself.

The explainer page "DefT: Boosting Scalability of Deformable Convolution
Operations on GPUs" prints no numeric example, so the pins are closed forms,
library special cases (torch fp64 convolution, scipy's linear interpolation),
brute force on tiny inputs, finite differences, and values worked by hand.
A plausible mistake in the oracle -- a dropped corner, a swapped dy/dx, a wrong
group index, a sign flip in a derivative, a transposed weight -- fails at least
one of them.
"""
import json
import os

import numpy as np
import pytest
import scipy.ndimage as ndi
import torch
import torch.nn.functional as F

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")

GEOMETRIES = [
    # n, c_in, h, w, c_out, kh, kw, stride, pad, dil, groups
    (2, 3, 5, 6, 2, 3, 3, 1, 1, 1, 1),
    (1, 4, 7, 5, 3, 3, 3, 2, 1, 1, 2),
    (2, 4, 9, 8, 2, 3, 3, 1, 2, 2, 4),
    (1, 2, 6, 7, 3, 2, 3, (1, 2), (0, 1), (2, 1), 1),
]


def make_problem(g):
    n, c_in, h, w, c_out, kh, kw, s, pad, d, groups = g
    return oracle.Problem(n, c_in, h, w, c_out, kh, kw, s, pad, d, groups)


def rand_inputs(p, seed, w_off_std=0.1):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((p.n, p.c_in, p.h, p.w))
    w_off = rng.standard_normal((p.n_off, p.c_in, p.kh, p.kw)) * w_off_std
    b_off = rng.standard_normal(p.n_off) * 0.5
    w = rng.standard_normal((p.c_out, p.c_in, p.kh, p.kw))
    gy = rng.standard_normal((p.n, p.c_out, p.ho, p.wo))
    return x, w_off, b_off, w, gy


def torch_conv(p, x, w):
    return F.conv2d(torch.from_numpy(x), torch.from_numpy(w),
                    stride=(p.stride_h, p.stride_w), padding=(p.pad_h, p.pad_w),
                    dilation=(p.dil_h, p.dil_w)).numpy()


def rel_err(a, b):
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


# ---------------------------------------------------------------- hand-worked


def test_hand_worked_samples():
    gold = json.load(open(GOLDEN))
    plane = np.array(gold["plane"], dtype=np.float64)
    for s in gold["samples"]:
        assert oracle.bilinear(plane, s["py"], s["px"]) == s["value"]
        assert oracle.bilinear_closed_form(plane, s["py"], s["px"]) == s["value"]
        if "d_py" in s:
            dy, dx = oracle.bilinear_grad(plane, s["py"], s["px"])
            assert (dy, dx) == (s["d_py"], s["d_px"])


def test_hand_worked_layer():
    L = json.load(open(GOLDEN))["layer"]
    p = oracle.Problem(L["n"], L["c_in"], L["h"], L["w"], L["c_out"], L["kh"],
                       L["kw"], L["stride"], L["pad"], L["dil"], L["groups"])
    x = np.array(json.load(open(GOLDEN))["plane"], dtype=np.float64)[None, None]
    w_off = np.zeros((2, 1, 1, 1))
    w = np.full((1, 1, 1, 1), L["w_main"])
    y, off = oracle.forward(p, x, w_off, np.array(L["b_off"]), w)
    np.testing.assert_array_equal(y[0, 0], np.array(L["y"]))
    np.testing.assert_array_equal(off[0, :, 0, 0], np.array(L["b_off"]))


# ---------------------------------------------------------------- P4 bilinear


def test_bilinear_matches_scipy_and_tent_kernel():
    """Four-corner blend == tent-kernel brute force == scipy linear
    interpolation with zeros beyond the edge, at interior, border, integer and
    far-outside points."""
    rng = np.random.default_rng(1)
    plane = rng.standard_normal((6, 9))
    H, W = plane.shape
    pts = list(zip(rng.uniform(-2.5, H + 1.5, 400), rng.uniform(-2.5, W + 1.5, 400)))
    pts += [(a, b) for a in (-1.0, -0.5, 0.0, 2.0, H - 1.0, H - 0.5, H)
            for b in (-1.0, -0.25, 0.0, 3.0, W - 1.0, W - 0.75, W)]
    pts += [(1e6, 2.0), (-1e6, 2.0), (2.0, 3e7), (-3.5, -4.0), (H + 5.0, W + 5.0)]
    got = np.array([oracle.bilinear(plane, a, b) for a, b in pts])
    tent = np.array([oracle.bilinear_closed_form(plane, a, b) for a, b in pts])
    ref = ndi.map_coordinates(plane, np.array(pts).T, order=1, mode="grid-constant",
                              cval=0.0, prefilter=False)
    np.testing.assert_allclose(got, tent, rtol=0, atol=1e-13)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_bilinear_grad_matches_difference_of_samples():
    """Away from cell edges the derivative is exact for a bilinear function:
    central differences of the sample agree to rounding."""
    rng = np.random.default_rng(2)
    plane = rng.standard_normal((5, 7))
    h = 1e-6
    for _ in range(300):
        a = np.floor(rng.uniform(-1.5, 5.5)) + rng.uniform(0.05, 0.95)
        b = np.floor(rng.uniform(-1.5, 7.5)) + rng.uniform(0.05, 0.95)
        dy, dx = oracle.bilinear_grad(plane, a, b)
        fy = (oracle.bilinear(plane, a + h, b) - oracle.bilinear(plane, a - h, b)) / (2 * h)
        fx = (oracle.bilinear(plane, a, b + h) - oracle.bilinear(plane, a, b - h)) / (2 * h)
        assert abs(dy - fy) < 1e-8 and abs(dx - fx) < 1e-8


# ---------------------------------------------------------------- P1 zero offsets


@pytest.mark.parametrize("g", GEOMETRIES)
def test_zero_offsets_equal_standard_conv(g):
    p = make_problem(g)
    x, _, _, w, gy = rand_inputs(p, 3)
    zeros_off = np.zeros((p.n_off, p.c_in, p.kh, p.kw))
    y, off = oracle.forward(p, x, zeros_off, np.zeros(p.n_off), w)
    assert np.all(off == 0.0)
    ref = torch_conv(p, x, w)
    assert y.shape == ref.shape
    assert rel_err(y, ref) < 1e-12


@pytest.mark.parametrize("g", GEOMETRIES)
def test_zero_offsets_backward_equals_conv_autograd(g):
    """With zero offset-conv weights the gradients of x and of the main weights
    are those of a standard convolution (torch autograd, fp64)."""
    p = make_problem(g)
    x, _, _, w, gy = rand_inputs(p, 4)
    zeros_off = np.zeros((p.n_off, p.c_in, p.kh, p.kw))
    off = np.zeros((p.n, p.n_off, p.ho, p.wo))
    got = oracle.backward(p, x, zeros_off, w, off, gy)
    xt = torch.from_numpy(x).requires_grad_()
    wt = torch.from_numpy(w).requires_grad_()
    yt = F.conv2d(xt, wt, stride=(p.stride_h, p.stride_w), padding=(p.pad_h, p.pad_w),
                  dilation=(p.dil_h, p.dil_w))
    (yt * torch.from_numpy(gy)).sum().backward()
    assert rel_err(got["grad_x"], xt.grad.numpy()) < 1e-12
    assert rel_err(got["grad_w"], wt.grad.numpy()) < 1e-12


# ---------------------------------------------------------------- P2 integer offsets


def shifted_conv_torch(p, x, w, shifts):
    """Reference for integer offsets: tap k reads the zero-padded input at its
    base position plus (dy_k, dx_k), i.e. a sum of shifted 1x1 convolutions.
    Written with torch slicing on a zero-padded copy."""
    big = 64
    xt = F.pad(x, (big, big, big, big))
    y = 0
    for i in range(p.kh):
        for j in range(p.kw):
            dy, dx = shifts[i * p.kw + j]
            r0 = big - p.pad_h + i * p.dil_h + dy
            c0 = big - p.pad_w + j * p.dil_w + dx
            patch = xt[:, :, r0:r0 + p.stride_h * (p.ho - 1) + 1:p.stride_h,
                       c0:c0 + p.stride_w * (p.wo - 1) + 1:p.stride_w]
            y = y + torch.einsum("nchw,oc->nohw", patch, w[:, :, i, j])
    return y


@pytest.mark.parametrize("g", GEOMETRIES[:3])
def test_integer_offsets_equal_shifted_conv(g):
    p = make_problem(g)
    x, _, _, w, gy = rand_inputs(p, 5)
    rng = np.random.default_rng(6)
    K = p.kh * p.kw
    shifts = rng.integers(-3, 4, size=(K, 2))
    b_off = np.zeros(p.n_off)
    for gg in range(p.groups):
        for k in range(K):
            b_off[2 * (gg * K + k)] = shifts[k, 0]
            b_off[2 * (gg * K + k) + 1] = shifts[k, 1]
    zeros_off = np.zeros((p.n_off, p.c_in, p.kh, p.kw))
    y, off = oracle.forward(p, x, zeros_off, b_off, w)
    xt = torch.from_numpy(x).requires_grad_()
    wt = torch.from_numpy(w).requires_grad_()
    ref = shifted_conv_torch(p, xt, wt, shifts)
    assert rel_err(y, ref.detach().numpy()) < 1e-12
    (ref * torch.from_numpy(gy)).sum().backward()
    got = oracle.backward(p, x, zeros_off, w, off, gy)
    assert rel_err(got["grad_x"], xt.grad.numpy()) < 1e-12
    assert rel_err(got["grad_w"], wt.grad.numpy()) < 1e-12


# ---------------------------------------------------------------- P3 half pixel


def test_half_pixel_rows_average_neighbours():
    """dy = 1/2 on every tap: each sample is the mean of two vertically
    adjacent pixels of the zero-padded input."""
    p = oracle.Problem(2, 3, 6, 5, 4, 3, 3, 1, 1, 1, 1)
    x, _, _, w, _ = rand_inputs(p, 7)
    b_off = np.zeros(p.n_off)
    b_off[0::2] = 0.5
    y, _ = oracle.forward(p, x, np.zeros((p.n_off, p.c_in, 3, 3)), b_off, w)
    z = F.pad(torch.from_numpy(x), (p.pad_w, p.pad_w, p.pad_h, p.pad_h + 1))
    zh = 0.5 * (z[:, :, :-1, :] + z[:, :, 1:, :])
    ref = F.conv2d(zh, torch.from_numpy(w)).numpy()
    assert rel_err(y, ref) < 1e-12


# ---------------------------------------------------------------- P5 finite differences


def fd_inputs(p, seed):
    """Random inputs whose every sampling point sits at least 0.2 px inside a
    bilinear cell, so central differences are exact up to rounding."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((p.n, p.c_in, p.h, p.w))
    w_off = rng.standard_normal((p.n_off, p.c_in, p.kh, p.kw)) * 0.05
    b_off = rng.standard_normal(p.n_off) * 0.3
    w = rng.standard_normal((p.c_out, p.c_in, p.kh, p.kw))
    gy = rng.standard_normal((p.n, p.c_out, p.ho, p.wo))
    conv = oracle.offsets(p, x, w_off, b_off)
    target = np.floor(conv) + rng.integers(-1, 2, conv.shape) + rng.uniform(0.2, 0.8, conv.shape)
    add = target - conv
    return x, w_off, b_off, w, add, gy


FD_GEOMETRIES = [
    (2, 3, 5, 6, 2, 3, 3, 1, 1, 1, 1),
    (2, 3, 5, 6, 2, 3, 3, 2, 1, 1, 3),
    (1, 3, 6, 6, 2, 3, 3, 1, 2, 2, 1),
    (1, 2, 5, 6, 2, 2, 3, (2, 1), (1, 0), (1, 2), 2),
]


@pytest.mark.parametrize("g", FD_GEOMETRIES)
def test_backward_matches_finite_differences(g):
    p = make_problem(g)
    x, w_off, b_off, w, add, gy = fd_inputs(p, 11)

    def loss(x, w_off, b_off, w, add):
        y, _ = oracle.forward(p, x, w_off, b_off, w, add)
        return float(np.sum(y * gy))

    _, off = oracle.forward(p, x, w_off, b_off, w, add)
    an = oracle.backward(p, x, w_off, w, off, gy)
    args = dict(x=x, w_off=w_off, b_off=b_off, w=w, add=add)
    names = dict(x="grad_x", w_off="grad_w_off", b_off="grad_b_off", w="grad_w",
                 add="grad_offset")
    rng = np.random.default_rng(12)
    h = 1e-6
    for key, gname in names.items():
        base = args[key]
        flat_idx = rng.choice(base.size, size=min(base.size, 60), replace=False)
        scale = max(np.max(np.abs(an[gname])), 1.0)
        for fi in flat_idx:
            idx = np.unravel_index(fi, base.shape)
            plus = {k: v.copy() for k, v in args.items()}
            minus = {k: v.copy() for k, v in args.items()}
            plus[key][idx] += h
            minus[key][idx] -= h
            fd = (loss(**plus) - loss(**minus)) / (2 * h)
            assert abs(fd - an[gname][idx]) <= 2e-7 * scale, (key, idx, fd, an[gname][idx])


# ---------------------------------------------------------------- P6 adjoint


@pytest.mark.parametrize("g", GEOMETRIES)
def test_scatter_is_adjoint_of_gather(g):
    p = make_problem(g)
    rng = np.random.default_rng(13)
    x = rng.standard_normal((p.n, p.c_in, p.h, p.w))
    off = rng.standard_normal((p.n, p.n_off, p.ho, p.wo)) * 2.0
    u = rng.standard_normal((p.n, p.c_in, p.kh * p.kw, p.ho, p.wo))
    lhs = np.sum(oracle.column(p, x, off) * u)
    rhs = np.sum(x * oracle.column_adjoint(p, off, u))
    assert abs(lhs - rhs) <= 1e-12 * max(abs(lhs), 1.0)


# ---------------------------------------------------------------- P7 groups


@pytest.mark.parametrize("groups", [2, 4])
def test_identical_offsets_in_every_group_equal_one_group(groups):
    p1 = oracle.Problem(2, 4, 7, 6, 3, 3, 3, 1, 1, 1, 1)
    pg = oracle.Problem(2, 4, 7, 6, 3, 3, 3, 1, 1, 1, groups)
    x, w_off, b_off, w, gy = rand_inputs(p1, 14, w_off_std=0.2)
    y1, off1 = oracle.forward(p1, x, w_off, b_off, w)
    w_off_g = np.concatenate([w_off] * groups, axis=0)
    b_off_g = np.concatenate([b_off] * groups)
    yg, offg = oracle.forward(pg, x, w_off_g, b_off_g, w)
    np.testing.assert_allclose(yg, y1, rtol=0, atol=1e-12 * np.max(np.abs(y1)))
    g1 = oracle.backward(p1, x, w_off, w, off1, gy)
    gg = oracle.backward(pg, x, w_off_g, w, offg, gy)
    np.testing.assert_allclose(gg["grad_x"] - 0, g1["grad_x"] - 0, rtol=0,
                               atol=1e-11 * np.max(np.abs(g1["grad_x"])))
    np.testing.assert_allclose(gg["grad_w"], g1["grad_w"], rtol=0,
                               atol=1e-11 * np.max(np.abs(g1["grad_w"])))
    # the offset gradient of the single group is the sum over the copies
    K = 9
    summed = sum(gg["grad_offset"][:, 2 * K * q:2 * K * (q + 1)] for q in range(groups))
    np.testing.assert_allclose(summed, g1["grad_offset"], rtol=0,
                               atol=1e-11 * np.max(np.abs(g1["grad_offset"])))


# ---------------------------------------------------------------- P8 far outside


def test_far_outside_offsets_give_zero():
    p = oracle.Problem(2, 3, 6, 7, 2, 3, 3, 1, 1, 1, 1)
    x, _, _, w, gy = rand_inputs(p, 15)
    b_off = np.full(p.n_off, 1.0)
    b_off[0::2] = -(p.h + p.w + 3 * p.kh + 5.0)
    zeros_off = np.zeros((p.n_off, p.c_in, 3, 3))
    y, off = oracle.forward(p, x, zeros_off, b_off, w)
    assert np.all(y == 0.0)
    g = oracle.backward(p, x, zeros_off, w, off, gy)
    assert np.all(g["grad_offset"] == 0.0)
    assert np.all(g["grad_x"] == 0.0)
    assert np.all(g["grad_w"] == 0.0)


# ---------------------------------------------------------------- P9 kink convention


def test_zero_offset_gradient_is_right_sided_difference():
    p = oracle.Problem(2, 3, 5, 6, 2, 3, 3, 1, 1, 1, 1)
    x, _, _, w, gy = rand_inputs(p, 16)
    off = np.zeros((p.n, p.n_off, p.ho, p.wo))
    g = oracle.backward(p, x, np.zeros((p.n_off, p.c_in, 3, 3)), w, off, gy)
    # gradient of the deformed map: sum over output channels
    gcol = np.einsum("ock,nohw->nckhw", w.reshape(p.c_out, p.c_in, 9), gy)
    xp = np.pad(x, ((0, 0), (0, 0), (2, 2), (2, 2)))
    for i in range(3):
        for j in range(3):
            k = i * 3 + j
            r0, c0 = 2 - 1 + i, 2 - 1 + j  # base position in the padded copy
            v00 = xp[:, :, r0:r0 + p.ho, c0:c0 + p.wo]
            v10 = xp[:, :, r0 + 1:r0 + 1 + p.ho, c0:c0 + p.wo]
            v01 = xp[:, :, r0:r0 + p.ho, c0 + 1:c0 + 1 + p.wo]
            want_y = np.sum(gcol[:, :, k] * (v10 - v00), axis=1)
            want_x = np.sum(gcol[:, :, k] * (v01 - v00), axis=1)
            np.testing.assert_allclose(g["grad_offset"][:, 2 * k], want_y, rtol=0, atol=1e-12)
            np.testing.assert_allclose(g["grad_offset"][:, 2 * k + 1], want_x, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- P10 translation


def test_integer_translation_of_offsets_shifts_the_input():
    p = oracle.Problem(1, 3, 9, 10, 2, 3, 3, 1, 1, 1, 1)
    x, w_off, b_off, w, _ = rand_inputs(p, 17)
    rng = np.random.default_rng(18)
    off = rng.standard_normal((p.n, p.n_off, p.ho, p.wo))
    a, b = 2, -1
    # the rows and columns that the shifted copy cannot hold are set to zero,
    # so the identity below is exact
    x[:, :, :a, :] = 0.0
    x[:, :, :, p.w + b:] = 0.0
    shifted = off.copy()
    shifted[:, 0::2] += a
    shifted[:, 1::2] += b
    col_a = oracle.column(p, x, shifted)
    xs = np.zeros_like(x)  # xs[r, c] = x[r + a, c + b], zero where that is outside
    xs[:, :, :p.h - a, -b:] = x[:, :, a:, :p.w + b]
    col_b = oracle.column(p, xs, off)
    np.testing.assert_allclose(col_a, col_b, rtol=0, atol=1e-13)


def test_rejects_bad_problems():
    x = np.zeros((1, 3, 4, 4))
    with pytest.raises(ValueError):
        oracle.offsets(oracle.Problem(1, 3, 4, 4, 2, groups=2), x,
                       np.zeros((36, 3, 3, 3)))
    with pytest.raises(ValueError):
        oracle.offsets(oracle.Problem(1, 3, 1, 4, 2, kh=3, kw=3, pad=0), x[:, :, :1],
                       np.zeros((18, 3, 3, 3)))


# ---------------------------------------------------------------- cell decision


def test_cell_is_decided_on_the_float32_coordinate():
    """floor() of a sampling coordinate is an integer decision and is taken on
    the float32 value base + shift (the kernels' precision).  A shift that is
    just below 1 in fp64 but rounds to 1.0 in float32 puts the sample in the
    next cell: the offset gradient is the right-sided difference there."""
    p = oracle.Problem(1, 1, 8, 3, 1, 1, 1, 1, 0, 1, 1)
    rng = np.random.default_rng(19)
    x = rng.standard_normal((1, 1, 8, 3))
    w = np.ones((1, 1, 1, 1))
    gy = np.zeros((1, 1, 8, 3))
    gy[0, 0, 3, 1] = 1.0
    off = np.zeros((1, 2, 8, 3))
    shift = 0.99999999
    off[0, 0, 3, 1] = shift
    assert np.floor(np.float32(3) + np.float32(shift)) == 4.0
    assert np.floor(3 + shift) == 3.0
    g = oracle.backward(p, x, np.zeros((2, 1, 1, 1)), w, off, gy)
    assert g["grad_offset"][0, 0, 3, 1] == x[0, 0, 5, 1] - x[0, 0, 4, 1]
    # the sample itself is continuous across the line
    col = oracle.column(p, x, off)
    assert abs(col[0, 0, 0, 3, 1] - x[0, 0, 4, 1]) < 1e-7


# ---------------------------------------------------------------- offset convolution (Step 1 of 5)

OFFSET_GEOMETRIES = GEOMETRIES + [
    # kh != kw with per-axis stride, padding and dilation, several offset groups
    (2, 6, 7, 9, 2, 2, 3, (2, 1), (1, 0), (1, 2), 2),
    (1, 8, 6, 5, 2, 3, 2, 1, (2, 1), (2, 1), 4),
]


def torch_conv_bias(p, x, w, b):
    return F.conv2d(x, w, b, stride=(p.stride_h, p.stride_w), padding=(p.pad_h, p.pad_w),
                    dilation=(p.dil_h, p.dil_w))


@pytest.mark.parametrize("g", OFFSET_GEOMETRIES)
def test_offset_convolution_equals_torch_conv(g):
    """Step 1 of 5 ("Following a deformable layer through DefT"): the offsets
    are a standard convolution of the input, with the main convolution's
    kernel size, stride, padding and dilation and a bias (reading C1), plus
    offset_add.  Nonzero random w_off, compared with torch's fp64 conv2d."""
    p = make_problem(g)
    x, w_off, b_off, w, _ = rand_inputs(p, 21, w_off_std=1.0)
    add = np.random.default_rng(22).standard_normal((p.n, p.n_off, p.ho, p.wo))
    got = oracle.offsets(p, x, w_off, b_off, add)
    ref = torch_conv_bias(p, torch.from_numpy(x), torch.from_numpy(w_off),
                          torch.from_numpy(b_off)).numpy() + add
    assert got.shape == ref.shape
    assert rel_err(got, ref) < 1e-12
    _, off = oracle.forward(p, x, w_off, b_off, w, add)
    assert np.array_equal(off, got)


@pytest.mark.parametrize("g", OFFSET_GEOMETRIES)
def test_offset_convolution_backward_equals_conv_autograd(g):
    """The offset convolution's part of the backward -- grad_w_off, grad_b_off
    and its term of grad_x -- is torch autograd of the same fp64 conv2d,
    driven by the oracle's offset gradient.  The sampling term of grad_x is
    removed by a second run at the same offsets with w_off = 0 (the offset
    gradient depends only on the offsets, so it is identical)."""
    p = make_problem(g)
    x, w_off, b_off, w, gy = rand_inputs(p, 23, w_off_std=0.3)
    _, off = oracle.forward(p, x, w_off, b_off, w)
    full = oracle.backward(p, x, w_off, w, off, gy)
    samp = oracle.backward(p, x, np.zeros_like(w_off), w, off, gy)
    assert np.array_equal(full["grad_offset"], samp["grad_offset"])
    xt = torch.from_numpy(x).requires_grad_()
    wt = torch.from_numpy(w_off).requires_grad_()
    bt = torch.from_numpy(b_off).requires_grad_()
    o = torch_conv_bias(p, xt, wt, bt)
    (o * torch.from_numpy(full["grad_offset"])).sum().backward()
    assert rel_err(full["grad_w_off"], wt.grad.numpy()) < 1e-12
    assert rel_err(full["grad_b_off"], bt.grad.numpy()) < 1e-12
    assert rel_err(full["grad_x"] - samp["grad_x"], xt.grad.numpy()) < 1e-10


# ---------------------------------------------------------------- channel -> offset group

GROUP_GEOMETRIES = [
    # n, c_in, h, w, c_out, kh, kw, stride, pad, dil, groups -- every group has Cg > 1
    (2, 8, 6, 7, 3, 3, 3, 1, 1, 1, 2),
    (1, 8, 7, 6, 2, 3, 3, 2, 1, 1, 4),
    (2, 6, 5, 6, 2, 2, 3, 1, (1, 0), (1, 2), 3),
]


@pytest.mark.parametrize("g", GROUP_GEOMETRIES)
def test_offset_groups_split_the_channels_into_contiguous_blocks(g):
    """Offset group q serves input channels [q*Cg, (q+1)*Cg) (reading C3).
    The main convolution is linear over input channels, so with a distinct
    random offset field per group the layer is the sum, over q, of a
    one-group layer on channel block q that samples at group q's offsets; the
    gradients of x, of w and of the offsets are the blocks' gradients side by
    side.  The one-group runs never evaluate the channel-to-group index."""
    p = make_problem(g)
    G, Cg, K = p.groups, p.c_in // p.groups, p.kh * p.kw
    rng = np.random.default_rng(24)
    x = rng.standard_normal((p.n, p.c_in, p.h, p.w))
    w = rng.standard_normal((p.c_out, p.c_in, p.kh, p.kw))
    gy = rng.standard_normal((p.n, p.c_out, p.ho, p.wo))
    add = rng.standard_normal((p.n, p.n_off, p.ho, p.wo)) * 1.5
    y, off = oracle.forward(p, x, np.zeros((p.n_off, p.c_in, p.kh, p.kw)), None, w, add)
    full = oracle.backward(p, x, np.zeros((p.n_off, p.c_in, p.kh, p.kw)), w, off, gy)
    y_sum = np.zeros_like(y)
    for q in range(G):
        blk = slice(q * Cg, (q + 1) * Cg)
        om = slice(2 * q * K, 2 * (q + 1) * K)
        p1 = oracle.Problem(p.n, Cg, p.h, p.w, p.c_out, p.kh, p.kw,
                            (p.stride_h, p.stride_w), (p.pad_h, p.pad_w),
                            (p.dil_h, p.dil_w), 1)
        zero_w = np.zeros((2 * K, Cg, p.kh, p.kw))
        yq, offq = oracle.forward(p1, x[:, blk], zero_w, None, w[:, blk], add[:, om])
        bq = oracle.backward(p1, x[:, blk], zero_w, w[:, blk], offq, gy)
        y_sum += yq
        assert rel_err(full["grad_x"][:, blk], bq["grad_x"]) < 1e-12
        assert rel_err(full["grad_w"][:, blk], bq["grad_w"]) < 1e-12
        assert rel_err(full["grad_offset"][:, om], bq["grad_offset"]) < 1e-12
    assert rel_err(y, y_sum) < 1e-12


# ---------------------------------------------------------------- activation between layers


def test_relu_and_its_gradient_by_hand():
    """Values worked by hand: negatives and both zeros go to +0, positives
    pass, NaN passes; the gradient flows only where the output is positive."""
    y = np.array([-2.5, -0.0, 0.0, 1e-30, 3.0, np.nan, -np.inf, np.inf])
    r = oracle.relu(y)
    assert r[:5].tolist() == [0.0, 0.0, 0.0, 1e-30, 3.0]
    assert np.isnan(r[5]) and r[6] == 0.0 and r[7] == np.inf
    assert not np.signbit(r[1])
    g = np.array([1.0, 2.0, 3.0, 4.0, 5.0, 6.0, 7.0, 8.0])
    assert oracle.relu_grad(r, g).tolist() == [0.0, 0.0, 0.0, 4.0, 5.0, 0.0, 0.0, 8.0]


def test_elementwise_parity_bound_catches_what_the_tensor_bound_misses():
    """The parity helper's per-element bound: an error in a small element that
    the max-normalised measure lets through is caught; exact and relative
    errors within the bound pass."""
    from parity import elementwise_err, rel_err
    ref = np.array([1000.0, 1.0, -3.0])
    got = ref.copy()
    got[1] += 6.0  # 0.6 % of the tensor's maximum, 600 % of the element
    assert rel_err(got, ref) <= 2e-2
    assert elementwise_err(got, ref, 2e-2) > 1.0
    assert elementwise_err(ref, ref, 2e-2) == 0.0
    ok = ref * (1 + 1e-2)  # 1 % relative everywhere
    assert elementwise_err(ok, ref, 2e-2) <= 1.0
    assert elementwise_err(np.zeros(3), np.zeros(3), 2e-2) == 0.0
