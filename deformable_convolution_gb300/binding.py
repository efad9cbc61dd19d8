"""Thin Python binding of the C ABI in ``include/deform_conv.h``.

Argument marshalling only: every function here checks tensor shapes and
dtypes, passes raw device pointers and the current CUDA stream to the library
and turns a non-OK status into ``DcError``.  All arithmetic runs in the CUDA
kernels of ``libdeformconv.so``; nothing here computes any part of the layer.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import torch

from . import _native

DC_OK, DC_ERR_INVALID_ARG, DC_ERR_UNSUPPORTED, DC_ERR_WORKSPACE, DC_ERR_CUDA, DC_ERR_TIMEOUT = range(6)
DC_F32, DC_BF16 = 0, 1
_TORCH_DTYPE = {DC_F32: torch.float32, DC_BF16: torch.bfloat16}

# every symbol include/deform_conv.h declares
EXPORTED_SYMBOLS = (
    "dc_out_h", "dc_out_w", "deform_conv_workspace_size", "deform_conv_fwd",
    "deform_conv_bwd", "deform_conv_sample", "dc_status_string", "dc_build_info",
    "dc_launch_count", "deform_conv_fwd_noalloc", "dc_device_error", "dc_kernel_timing",
    "dc_kernel_times", "deform_conv_offsets", "deform_conv_margin_histogram", "dc_suggest_margin",
    "deform_conv_bwd_after_fwd", "deform_conv_fwd_sampled_gemm", "dc_relu_fwd", "dc_relu_bwd",
    "dc_col_layout", "dc_sample_tile", "dc_selftest_wait_timeout", "dc_test_fail_launches",
)
DC_COL_PLANE_MAJOR, DC_COL_PIXEL_MAJOR = 0, 1
MARGIN_BINS = 64
NOALLOC_SCRATCH_BYTES = 32 << 20


class DcProblem(ctypes.Structure):
    """Mirror of ``dc_problem``."""
    _fields_ = [(name, ctypes.c_int) for name in (
        "n", "c_in", "h", "w", "c_out", "kh", "kw", "stride_h", "stride_w",
        "pad_h", "pad_w", "dil_h", "dil_w", "offset_groups", "dtype", "halo_margin", "out_relu",
        "in_relu")]


class DcError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}")


_configured = False


def lib() -> ctypes.CDLL:
    global _configured
    L = _native.load()
    if not _configured:
        vp, sz, i = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
        pp = ctypes.POINTER(DcProblem)
        L.dc_out_h.argtypes = [pp]
        L.dc_out_h.restype = i
        L.dc_out_w.argtypes = [pp]
        L.dc_out_w.restype = i
        L.deform_conv_workspace_size.argtypes = [pp, i, ctypes.POINTER(sz)]
        L.deform_conv_workspace_size.restype = i
        L.deform_conv_fwd.argtypes = [pp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.deform_conv_fwd.restype = i
        L.deform_conv_bwd.argtypes = [pp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.deform_conv_bwd.restype = i
        L.deform_conv_bwd_after_fwd.argtypes = [pp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.deform_conv_bwd_after_fwd.restype = i
        L.deform_conv_sample.argtypes = [pp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.deform_conv_sample.restype = i
        L.dc_col_layout.argtypes = [pp]
        L.dc_col_layout.restype = i
        L.dc_sample_tile.argtypes = [pp, ctypes.POINTER(i), ctypes.POINTER(i)]
        L.dc_sample_tile.restype = i
        L.deform_conv_offsets.argtypes = [pp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.deform_conv_offsets.restype = i
        L.deform_conv_fwd_sampled_gemm.argtypes = [pp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.deform_conv_fwd_sampled_gemm.restype = i
        L.deform_conv_margin_histogram.argtypes = [pp, vp, vp, vp]
        L.deform_conv_margin_histogram.restype = i
        L.dc_suggest_margin.argtypes = [pp, ctypes.POINTER(ctypes.c_ulonglong), ctypes.c_double, i]
        L.dc_suggest_margin.restype = i
        L.dc_status_string.argtypes = [i]
        L.dc_status_string.restype = ctypes.c_char_p
        L.dc_build_info.argtypes = []
        L.dc_build_info.restype = ctypes.c_char_p
        L.deform_conv_fwd_noalloc.argtypes = [pp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.deform_conv_fwd_noalloc.restype = i
        L.dc_kernel_timing.argtypes = [i]
        L.dc_kernel_timing.restype = None
        L.dc_kernel_times.argtypes = [ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_float), i]
        L.dc_kernel_times.restype = i
        L.dc_device_error.argtypes = [i]
        L.dc_device_error.restype = i
        L.dc_selftest_wait_timeout.argtypes = [ctypes.c_uint, vp]
        L.dc_selftest_wait_timeout.restype = i
        L.dc_test_fail_launches.argtypes = [i]
        L.dc_test_fail_launches.restype = i
        L.dc_relu_fwd.argtypes = [vp, vp, sz, i, vp]
        L.dc_relu_fwd.restype = i
        L.dc_relu_bwd.argtypes = [vp, vp, vp, sz, i, vp]
        L.dc_relu_bwd.restype = i
        L.dc_launch_count.argtypes = []
        L.dc_launch_count.restype = ctypes.c_ulonglong
        _configured = True
    return L


def status_string(status: int) -> str:
    return lib().dc_status_string(int(status)).decode()


def build_info() -> str:
    return lib().dc_build_info().decode()


def device_error(clear: bool = False) -> int:
    """DC_ERR_TIMEOUT if a bounded device wait expired (synchronises)."""
    return int(lib().dc_device_error(1 if clear else 0))


def selftest_wait_timeout(spins: int, stream=None) -> int:
    """Test hook: a kernel whose bounded wait on an mbarrier nothing arrives on
    expires after `spins` polls (the next device_error() is DC_ERR_TIMEOUT)."""
    return int(lib().dc_selftest_wait_timeout(spins, _stream(stream)))


def test_fail_launches(count: int) -> int:
    """Test hook: the next `count` launches of the layer entry points fail
    with DC_ERR_CUDA without being made (0 cancels)."""
    return int(lib().dc_test_fail_launches(count))


def kernel_timing(enable: bool) -> None:
    """Start/stop CUDA-event timing of every launch the library enqueues."""
    lib().dc_kernel_timing(1 if enable else 0)


def kernel_times(capacity: int = 256):
    """[(kernel name, ms)] of the launches recorded since timing was enabled
    (waits for them); clears the record."""
    names = (ctypes.c_char_p * capacity)()
    ms = (ctypes.c_float * capacity)()
    n = lib().dc_kernel_times(names, ms, capacity)
    return [(names[i].decode(), float(ms[i])) for i in range(n)]


def launch_count() -> int:
    return int(lib().dc_launch_count())


@dataclass(frozen=True)
class Problem:
    """One deformable layer: NCHW input, 3x3-style kernel geometry, dtype."""
    n: int
    c_in: int
    h: int
    w: int
    c_out: int
    kh: int = 3
    kw: int = 3
    stride: tuple = (1, 1)
    pad: tuple = (1, 1)
    dil: tuple = (1, 1)
    offset_groups: int = 1
    dtype: int = DC_F32
    halo_margin: int = -1
    out_relu: int = 0  # 1: the forward writes relu(y) (a following ReLU fused into its epilogue)
    in_relu: int = 0   # 1: x = relu(z); the backward writes dL/dz in the dtype as grad_x

    def __post_init__(self):
        for f in ("stride", "pad", "dil"):
            v = getattr(self, f)
            if isinstance(v, int):
                object.__setattr__(self, f, (v, v))

    def c_struct(self) -> DcProblem:
        return DcProblem(self.n, self.c_in, self.h, self.w, self.c_out, self.kh, self.kw,
                         self.stride[0], self.stride[1], self.pad[0], self.pad[1],
                         self.dil[0], self.dil[1], self.offset_groups, self.dtype,
                         self.halo_margin, self.out_relu, self.in_relu)

    @property
    def torch_dtype(self):
        return _TORCH_DTYPE[self.dtype]

    @property
    def ho(self):
        return (self.h + 2 * self.pad[0] - self.dil[0] * (self.kh - 1) - 1) // self.stride[0] + 1

    @property
    def wo(self):
        return (self.w + 2 * self.pad[1] - self.dil[1] * (self.kw - 1) - 1) // self.stride[1] + 1

    @property
    def n_off(self):
        return 2 * self.offset_groups * self.kh * self.kw

    def shapes(self):
        return dict(x=(self.n, self.c_in, self.h, self.w),
                    w_off=(self.n_off, self.c_in, self.kh, self.kw),
                    b_off=(self.n_off,),
                    w=(self.c_out, self.c_in, self.kh, self.kw),
                    offset=(self.n, self.n_off, self.ho, self.wo),
                    y=(self.n, self.c_out, self.ho, self.wo),
                    col=(self.c_in * self.kh * self.kw, self.n, self.ho * self.wo))

    # (the deformed map's shape depends on the path the library takes for the
    # problem: binding.col_shape)


def _ptr(t, name, shape=None, dtype=None, optional=False):
    if t is None:
        if optional:
            return None
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name}: expected {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(status, what):
    if status != DC_OK:
        raise DcError(status, what)


def deform_conv_workspace_size(p: Problem, backward: bool) -> int:
    out = ctypes.c_size_t(0)
    st = p.c_struct()
    _check(lib().deform_conv_workspace_size(ctypes.byref(st), 1 if backward else 0,
                                            ctypes.byref(out)), "deform_conv_workspace_size")
    return int(out.value)


def out_hw(p: Problem):
    st = p.c_struct()
    return lib().dc_out_h(ctypes.byref(st)), lib().dc_out_w(ctypes.byref(st))


def deform_conv_fwd(p: Problem, x, w_off, b_off, w, offset_add, y, offset_out=None,
                    slowpath_count=None, ws=None, stream=None):
    s = p.shapes()
    dt, f32 = p.torch_dtype, torch.float32
    st = p.c_struct()
    ws_ptr = _ptr(ws, "ws", dtype=torch.uint8)
    _check(lib().deform_conv_fwd(
        ctypes.byref(st), _ptr(x, "x", s["x"], dt), _ptr(w_off, "w_off", s["w_off"], dt),
        _ptr(b_off, "b_off", s["b_off"], f32, True), _ptr(w, "w", s["w"], dt),
        _ptr(offset_add, "offset_add", s["offset"], f32, True), _ptr(y, "y", s["y"], dt),
        _ptr(offset_out, "offset_out", s["offset"], f32, True),
        _ptr(slowpath_count, "slowpath_count", (1,), torch.int64, True),
        ws_ptr, ctypes.c_size_t(ws.numel()), _stream(stream)), "deform_conv_fwd")


def deform_conv_fwd_noalloc(p: Problem, x, w_off, b_off, w, offset_add, y, offset_out=None,
                            slowpath_count=None, stream=None):
    """Forward pass with the library's fixed scratch array instead of a
    workspace (for callers that cannot allocate device memory)."""
    s = p.shapes()
    dt, f32 = p.torch_dtype, torch.float32
    st = p.c_struct()
    _check(lib().deform_conv_fwd_noalloc(
        ctypes.byref(st), _ptr(x, "x", s["x"], dt), _ptr(w_off, "w_off", s["w_off"], dt),
        _ptr(b_off, "b_off", s["b_off"], f32, True), _ptr(w, "w", s["w"], dt),
        _ptr(offset_add, "offset_add", s["offset"], f32, True), _ptr(y, "y", s["y"], dt),
        _ptr(offset_out, "offset_out", s["offset"], f32, True),
        _ptr(slowpath_count, "slowpath_count", (1,), torch.int64, True),
        _stream(stream)), "deform_conv_fwd_noalloc")


def deform_conv_bwd(p: Problem, x, w_off, w, offset, grad_y, grad_x, grad_w_off, grad_b_off,
                    grad_w, grad_offset=None, ws=None, stream=None, after_fwd=False):
    """after_fwd: `ws` still holds the deformed map of the deform_conv_fwd call
    for these inputs (deform_conv_bwd_after_fwd); the map is not replayed.
    grad_x is float32, or of the problem dtype when ``p.in_relu``."""
    s = p.shapes()
    dt, f32 = p.torch_dtype, torch.float32
    st = p.c_struct()
    ws_ptr = _ptr(ws, "ws", dtype=torch.uint8)
    fn = lib().deform_conv_bwd_after_fwd if after_fwd else lib().deform_conv_bwd
    _check(fn(
        ctypes.byref(st), _ptr(x, "x", s["x"], dt), _ptr(w_off, "w_off", s["w_off"], dt),
        _ptr(w, "w", s["w"], dt), _ptr(offset, "offset", s["offset"], f32),
        _ptr(grad_y, "grad_y", s["y"], dt), _ptr(grad_x, "grad_x", s["x"], dt if p.in_relu else f32),
        _ptr(grad_w_off, "grad_w_off", s["w_off"], f32),
        _ptr(grad_b_off, "grad_b_off", s["b_off"], f32, True),
        _ptr(grad_w, "grad_w", s["w"], f32),
        _ptr(grad_offset, "grad_offset", s["offset"], f32, True),
        ws_ptr, ctypes.c_size_t(ws.numel()), _stream(stream)), "deform_conv_bwd")


def col_layout(p: Problem) -> int:
    """DC_COL_PLANE_MAJOR or DC_COL_PIXEL_MAJOR (the deformed map's layout)."""
    st = p.c_struct()
    v = int(lib().dc_col_layout(ctypes.byref(st)))
    if v < 0:
        raise DcError(DC_ERR_INVALID_ARG, "dc_col_layout")
    return v


def col_shape(p: Problem):
    """Shape of the deformed map in the problem's layout."""
    if col_layout(p) == DC_COL_PIXEL_MAJOR:
        return (p.n, p.ho * p.wo, p.kh * p.kw, p.c_in)
    return (p.c_in * p.kh * p.kw, p.n, p.ho * p.wo)


def sample_tile(p: Problem):
    """(tile_h, tile_w): the output tile the sampling stage stages a window for."""
    st = p.c_struct()
    th, tw = ctypes.c_int(0), ctypes.c_int(0)
    _check(lib().dc_sample_tile(ctypes.byref(st), ctypes.byref(th), ctypes.byref(tw)),
           "dc_sample_tile")
    return th.value, tw.value


def deform_conv_sample(p: Problem, x, w_off, b_off, offset_add, offset_in, col,
                       offset_out=None, slowpath_count=None, ws=None, stream=None):
    s = p.shapes()
    dt, f32 = p.torch_dtype, torch.float32
    st = p.c_struct()
    if ws is None:
        ws = workspace(p, False, x.device)
    _check(lib().deform_conv_sample(
        ctypes.byref(st), _ptr(x, "x", s["x"], dt),
        _ptr(w_off, "w_off", s["w_off"], dt, True),
        _ptr(b_off, "b_off", s["b_off"], f32, True),
        _ptr(offset_add, "offset_add", s["offset"], f32, True),
        _ptr(offset_in, "offset_in", s["offset"], f32, True),
        _ptr(col, "col", col_shape(p), dt),
        _ptr(offset_out, "offset_out", s["offset"], f32, True),
        _ptr(slowpath_count, "slowpath_count", (1,), torch.int64, True),
        _ptr(ws, "ws", dtype=torch.uint8), ctypes.c_size_t(ws.numel()),
        _stream(stream)), "deform_conv_sample")


def deform_conv_offsets(p: Problem, x, w_off, b_off, offset_add, offset_out, ws=None,
                        stream=None):
    s = p.shapes()
    dt, f32 = p.torch_dtype, torch.float32
    st = p.c_struct()
    if ws is None:
        ws = workspace(p, False, x.device)
    _check(lib().deform_conv_offsets(
        ctypes.byref(st), _ptr(x, "x", s["x"], dt), _ptr(w_off, "w_off", s["w_off"], dt),
        _ptr(b_off, "b_off", s["b_off"], f32, True),
        _ptr(offset_add, "offset_add", s["offset"], f32, True),
        _ptr(offset_out, "offset_out", s["offset"], f32),
        _ptr(ws, "ws", dtype=torch.uint8), ctypes.c_size_t(ws.numel()),
        _stream(stream)), "deform_conv_offsets")


def deform_conv_fwd_sampled_gemm(p: Problem, x, w_off, b_off, w, offset_add, y, offset_out,
                                 stream=None):
    s = p.shapes()
    dt, f32 = p.torch_dtype, torch.float32
    st = p.c_struct()
    _check(lib().deform_conv_fwd_sampled_gemm(
        ctypes.byref(st), _ptr(x, "x", s["x"], dt), _ptr(w_off, "w_off", s["w_off"], dt),
        _ptr(b_off, "b_off", s["b_off"], f32, True), _ptr(w, "w", s["w"], dt),
        _ptr(offset_add, "offset_add", s["offset"], f32, True), _ptr(y, "y", s["y"], dt),
        _ptr(offset_out, "offset_out", s["offset"], f32), _stream(stream)),
        "deform_conv_fwd_sampled_gemm")


def deform_conv_margin_histogram(p: Problem, offset, hist, stream=None):
    st = p.c_struct()
    _check(lib().deform_conv_margin_histogram(
        ctypes.byref(st), _ptr(offset, "offset", p.shapes()["offset"], torch.float32),
        _ptr(hist, "hist", (MARGIN_BINS,), torch.int64), _stream(stream)),
        "deform_conv_margin_histogram")


def dc_suggest_margin(p: Problem, hist_host, max_slow_fraction: float, for_backward: bool) -> int:
    """hist_host: MARGIN_BINS counts on the host (any integer sequence)."""
    arr = (ctypes.c_ulonglong * MARGIN_BINS)(*[int(v) for v in hist_host])
    st = p.c_struct()
    return int(lib().dc_suggest_margin(ctypes.byref(st), arr, float(max_slow_fraction),
                                       int(bool(for_backward))))


def _dc_dtype(t):
    for k, v in _TORCH_DTYPE.items():
        if t.dtype == v:
            return k
    raise ValueError(f"unsupported dtype {t.dtype}")


def dc_relu_fwd(y, out, stream=None):
    """out = max(y, 0) (float32 or bfloat16 tensors of one shape; out may be y)."""
    if out.shape != y.shape or out.dtype != y.dtype:
        raise ValueError("y and out must have the same shape and dtype")
    _check(lib().dc_relu_fwd(_ptr(y, "y"), _ptr(out, "out"), ctypes.c_size_t(y.numel()),
                             _dc_dtype(y), _stream(stream)), "dc_relu_fwd")


def dc_relu_bwd(act, grad_out, grad_in, stream=None):
    """grad_in = grad_out where act > 0 else 0, in act's dtype; grad_out float32."""
    if grad_out.shape != act.shape or grad_in.shape != act.shape or grad_in.dtype != act.dtype:
        raise ValueError("act, grad_out and grad_in must have one shape; grad_in act's dtype")
    _check(lib().dc_relu_bwd(_ptr(act, "act"), _ptr(grad_out, "grad_out", dtype=torch.float32),
                             _ptr(grad_in, "grad_in"), ctypes.c_size_t(act.numel()),
                             _dc_dtype(act), _stream(stream)), "dc_relu_bwd")


# ---------------------------------------------------------------- conveniences
# Allocate outputs with torch (device memory is PyTorch's job) and call the ABI.

def workspace(p: Problem, backward: bool, device="cuda"):
    return torch.empty(max(deform_conv_workspace_size(p, backward), 1), dtype=torch.uint8,
                       device=device)


def forward(p: Problem, x, w_off, b_off, w, offset_add=None, ws=None, stream=None,
            slowpath_count=None):
    """Returns (y, offsets)."""
    s = p.shapes()
    y = torch.empty(s["y"], dtype=p.torch_dtype, device=x.device)
    off = torch.empty(s["offset"], dtype=torch.float32, device=x.device)
    if ws is None:
        ws = workspace(p, False, x.device)
    deform_conv_fwd(p, x, w_off, b_off, w, offset_add, y, off, slowpath_count, ws, stream)
    return y, off


def backward(p: Problem, x, w_off, w, offset, grad_y, ws=None, stream=None):
    """Returns dict(grad_x, grad_w_off, grad_b_off, grad_w, grad_offset)."""
    s = p.shapes()
    dev = x.device
    out = dict(grad_x=torch.empty(s["x"], dtype=p.torch_dtype if p.in_relu else torch.float32,
                                  device=dev),
               grad_w_off=torch.empty(s["w_off"], dtype=torch.float32, device=dev),
               grad_b_off=torch.empty(s["b_off"], dtype=torch.float32, device=dev),
               grad_w=torch.empty(s["w"], dtype=torch.float32, device=dev),
               grad_offset=torch.empty(s["offset"], dtype=torch.float32, device=dev))
    if ws is None:
        ws = workspace(p, True, dev)
    deform_conv_bwd(p, x, w_off, w, offset, grad_y, out["grad_x"], out["grad_w_off"],
                    out["grad_b_off"], out["grad_w"], out["grad_offset"], ws, stream)
    return out
