"""Host-side contract of the C ABI: builds, loads, exports every declared
symbol, and rejects bad arguments on the host before launching anything.
None of these tests needs a GPU (no call here reaches a kernel launch)."""
import ctypes
import os
import re

import pytest

from deformable_convolution_gb300 import _native, binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(",
                            text, flags=re.M)
    return sorted(set(names))


def test_library_builds_and_exports_every_declared_symbol():
    _native.build()
    lib = ctypes.CDLL(_native.LIB_PATH)
    names = declared_functions()
    assert "deform_conv_fwd" in names and "deform_conv_bwd" in names
    for name in names:
        assert hasattr(lib, name), name
    assert set(B.EXPORTED_SYMBOLS) == set(names)


def test_build_info_and_status_strings():
    assert "sm_103a" in B.build_info()
    for s in range(6):
        assert B.status_string(s).startswith("DC_")


def problem(**kw):
    base = dict(n=2, c_in=4, h=9, w=7, c_out=3)
    base.update(kw)
    return B.Problem(**base)


def ws_size(p, backward=False):
    out = ctypes.c_size_t(0)
    st = p.c_struct()
    return B.lib().deform_conv_workspace_size(ctypes.byref(st), int(backward), ctypes.byref(out)), out.value


@pytest.mark.parametrize("kw,status", [
    (dict(c_in=5, offset_groups=2), B.DC_ERR_INVALID_ARG),
    (dict(n=0), B.DC_ERR_INVALID_ARG),
    (dict(h=1, pad=0), B.DC_ERR_INVALID_ARG),
    (dict(stride=0), B.DC_ERR_INVALID_ARG),
    (dict(dtype=7), B.DC_ERR_INVALID_ARG),
    (dict(halo_margin=-2), B.DC_ERR_INVALID_ARG),
    (dict(out_relu=2), B.DC_ERR_INVALID_ARG),
    (dict(in_relu=-1), B.DC_ERR_INVALID_ARG),
    (dict(kh=9, kw=9, pad=4), B.DC_ERR_UNSUPPORTED),
    (dict(halo_margin=1000), B.DC_ERR_UNSUPPORTED),
])
def test_invalid_problems_are_rejected(kw, status):
    st, _ = ws_size(problem(**kw))
    assert st == status
    assert B.out_hw(problem(**kw)) == (0, 0)


def test_output_size_and_workspace():
    p = problem(h=9, w=7, stride=(2, 1), pad=(1, 0), dil=(1, 2))
    assert B.out_hw(p) == ((9 + 2 - 2 - 1) // 2 + 1, (7 - 4 - 1) + 1)
    st, fwd = ws_size(p)
    assert st == B.DC_OK and fwd > 0
    st, bwd = ws_size(p, True)
    assert st == B.DC_OK and bwd > fwd


def _call_fwd(p, ptrs, ws_bytes):
    st = p.c_struct()
    vp = ctypes.c_void_p
    return B.lib().deform_conv_fwd(ctypes.byref(st), *[vp(v) if v else None for v in ptrs],
                                   ctypes.c_size_t(ws_bytes), None)


@pytest.mark.parametrize("kw", [dict(dtype=B.DC_F32), dict(dtype=B.DC_BF16, offset_groups=2)])
def test_in_relu_backward_workspace_holds_a_float32_grad_x(kw):
    # problems off the channels-last backward accumulate grad_x in a float32
    # scratch at the workspace's end, which the ReLU backward then reads; the
    # forward workspace and every region before it are unchanged
    import dataclasses
    p = problem(**kw)
    q = dataclasses.replace(p, in_relu=1)
    scratch = p.n * p.c_in * p.h * p.w * 4
    assert ws_size(q, False) == ws_size(p, False)
    (s0, b0), (s1, b1) = ws_size(p, True), ws_size(q, True)
    assert s0 == s1 == B.DC_OK
    assert scratch <= b1 - b0 < scratch + 256


def test_fwd_argument_checks_fail_before_any_launch():
    # fake, never dereferenced device addresses: every check below happens on
    # the host before the first launch
    p = problem()
    _, need = ws_size(p)
    good = [0x10000 * (i + 1) for i in range(9)]  # x w_off b_off w add y off slow ws
    bad = list(good)
    bad[0] = 0
    assert _call_fwd(p, bad, need) == B.DC_ERR_INVALID_ARG
    bad = list(good)
    bad[3] += 4
    assert _call_fwd(p, bad, need) == B.DC_ERR_UNSUPPORTED
    assert _call_fwd(p, good, need - 1) == B.DC_ERR_WORKSPACE
    bad = list(good)
    bad[8] = 0
    assert _call_fwd(p, bad, need) == B.DC_ERR_WORKSPACE
    assert _call_fwd(problem(c_in=3, offset_groups=2), good, need) == B.DC_ERR_INVALID_ARG


def test_bwd_argument_checks_fail_before_any_launch():
    p = problem()
    _, need = ws_size(p, True)
    st = p.c_struct()
    vp = ctypes.c_void_p
    ptrs = [vp(0x10000 * (i + 1)) for i in range(11)]
    ptrs[5] = None  # grad_x missing
    rc = B.lib().deform_conv_bwd(ctypes.byref(st), *ptrs, ctypes.c_size_t(need), None)
    assert rc == B.DC_ERR_INVALID_ARG
    ptrs = [vp(0x10000 * (i + 1)) for i in range(11)]
    rc = B.lib().deform_conv_bwd(ctypes.byref(st), *ptrs, ctypes.c_size_t(need // 2), None)
    assert rc == B.DC_ERR_WORKSPACE


def test_offsets_argument_checks_fail_before_any_launch():
    p = problem()
    st = p.c_struct()
    vp = ctypes.c_void_p
    good = [0x10000 * (i + 1) for i in range(6)]  # x w_off b_off add offset_out ws
    _, need = ws_size(p, False)

    def call(ptrs, ws_bytes=need):
        return B.lib().deform_conv_offsets(ctypes.byref(st), *[vp(v) if v else None for v in ptrs],
                                           ctypes.c_size_t(ws_bytes), None)
    for missing in (0, 1, 4):  # x, w_off and offset_out are required
        bad = list(good)
        bad[missing] = 0
        assert call(bad) == B.DC_ERR_INVALID_ARG
    bad = list(good)
    bad[4] += 8
    assert call(bad) == B.DC_ERR_UNSUPPORTED
    bad = list(good)
    bad[5] = 0
    assert call(bad) == B.DC_ERR_WORKSPACE
    assert call(good, need - 1) == B.DC_ERR_WORKSPACE


def test_sampled_gemm_forward_argument_checks_fail_before_any_launch():
    vp = ctypes.c_void_p
    good = [0x10000 * (i + 1) for i in range(7)]  # x w_off b_off w add y offset_out

    def call(p, ptrs):
        st = p.c_struct()
        return B.lib().deform_conv_fwd_sampled_gemm(ctypes.byref(st),
                                                    *[vp(v) if v else None for v in ptrs], None)
    pb = B.Problem(2, 16, 8, 8, 16, 3, 3, 1, 1, 1, 1, B.DC_BF16)
    for missing in (0, 1, 3, 5, 6):  # x, w_off, w, y and offset_out are required
        bad = list(good)
        bad[missing] = 0
        assert call(pb, bad) == B.DC_ERR_INVALID_ARG
    bad = list(good)
    bad[6] += 8
    assert call(pb, bad) == B.DC_ERR_UNSUPPORTED
    # tensor-core path only: bf16, C_in*Kh*Kw and Ho*Wo multiples of 8
    assert call(B.Problem(2, 16, 8, 8, 16, 3, 3, 1, 1, 1, 1, B.DC_F32), good) == B.DC_ERR_UNSUPPORTED
    assert call(B.Problem(2, 16, 7, 7, 16, 3, 3, 1, 1, 1, 1, B.DC_BF16), good) == B.DC_ERR_UNSUPPORTED


def _hist(**bins):
    h = [0] * B.MARGIN_BINS
    for k, v in bins.items():
        h[int(k[1:])] = v
    return h


def test_suggest_margin_from_histogram():
    p = problem()
    # every tap needs 2 pixels: margin 2, whatever the allowed fraction
    assert B.dc_suggest_margin(p, _hist(b2=1000), 0.0, False) == 2
    assert B.dc_suggest_margin(p, _hist(b2=1000), 0.5, False) == 2
    # 10 % of the taps need 5: allowed at 10 %, not at 5 %
    h = _hist(b1=900, b5=100)
    assert B.dc_suggest_margin(p, h, 0.10, False) == 1
    assert B.dc_suggest_margin(p, h, 0.05, False) == 5
    assert B.dc_suggest_margin(p, _hist(), 0.0, False) == 0  # no taps at all
    assert B.dc_suggest_margin(p, h, -0.1, False) == -1
    assert B.dc_suggest_margin(p, h, 1.5, False) == -1
    assert B.dc_suggest_margin(problem(n=0), h, 0.1, False) == -1


def test_suggested_margin_is_one_the_build_can_stage():
    # a wide layer with a far-out tail: the ideal margin (62) does not fit in
    # shared memory, so the helper lowers it to the largest one that does
    p = problem(n=1, c_in=256, h=56, w=56, c_out=256, dtype=B.DC_BF16)
    m = B.dc_suggest_margin(p, _hist(b1=10, b62=10), 0.0, True)
    assert 0 <= m < 62
    ok = B.Problem(1, 256, 56, 56, 256, dtype=B.DC_BF16, halo_margin=m)
    assert ws_size(ok, True)[0] == B.DC_OK
    too_big = B.Problem(1, 256, 56, 56, 256, dtype=B.DC_BF16, halo_margin=m + 1)
    assert ws_size(too_big, True)[0] != B.DC_OK or ws_size(too_big, False)[0] != B.DC_OK


def test_bwd_after_fwd_argument_checks_fail_before_any_launch():
    p = problem()
    _, need = ws_size(p, True)
    st = p.c_struct()
    vp = ctypes.c_void_p
    ptrs = [vp(0x10000 * (i + 1)) for i in range(11)]
    ptrs[4] = None  # grad_y missing
    rc = B.lib().deform_conv_bwd_after_fwd(ctypes.byref(st), *ptrs, ctypes.c_size_t(need), None)
    assert rc == B.DC_ERR_INVALID_ARG
    ptrs = [vp(0x10000 * (i + 1)) for i in range(11)]
    rc = B.lib().deform_conv_bwd_after_fwd(ctypes.byref(st), *ptrs, ctypes.c_size_t(need - 1), None)
    assert rc == B.DC_ERR_WORKSPACE
