"""Deformable convolution oracle: fp64 CPU statement of the layer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The CUDA library and
its Python binding never import it, and it imports nothing from them.

The arithmetic lives in ``deform_conv_oracle.c`` (plain C, fp64, OpenMP over
disjoint outputs); this module compiles it with gcc and marshals numpy arrays.
Every function follows the explainer page "DefT: Boosting Scalability of
Deformable Convolution Operations on GPUs":

* ``offsets``   -- "Following a deformable layer through DefT", Step 1 of 5:
  the offset convolution gives a fractional (y, x) shift for every filter
  position at every output location.
* ``column``    -- "The argument in one glance / Why it fell short": bilinear
  blend of the four pixels around each displaced tap, written into the
  deformed (unrolled) feature map.
* ``forward``   -- "The argument in one glance / What people did": offset
  convolution, interpolation, then the main convolution over the deformed map.
* ``backward``  -- exact derivative of ``forward`` (the page names training
  time as a result; the gradient of the definition is written out in the C
  file).
* ``bilinear`` / ``bilinear_closed_form`` / ``bilinear_grad`` -- the single
  sample, as the four-corner blend and, independently, as the tent-kernel sum
  over every pixel.
* ``relu`` / ``relu_grad`` -- the activation between stacked layers of the
  networks the page trains ("What people did before, and where it broke":
  deformable layers throughout a ResNet) and its derivative, elementwise in
  numpy.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "deform_conv_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liborc_deform_conv.so")
_lock = threading.Lock()
_lib = None


class OracleProblem(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int) for name in (
        "n", "c_in", "h", "w", "c_out", "kh", "kw",
        "stride_h", "stride_w", "pad_h", "pad_w", "dil_h", "dil_w", "groups")]


def build(force: bool = False) -> str:
    """Compile the oracle's shared library with gcc (OpenMP)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        dp = ctypes.POINTER(ctypes.c_double)
        pp = ctypes.POINTER(OracleProblem)
        lib.orc_check.argtypes = [pp]
        lib.orc_offsets.argtypes = [pp, dp, dp, dp, dp, dp]
        lib.orc_column.argtypes = [pp, dp, dp, dp]
        lib.orc_column_adjoint.argtypes = [pp, dp, dp, dp]
        lib.orc_forward.argtypes = [pp, dp, dp, dp, dp, dp, dp, dp]
        lib.orc_backward.argtypes = [pp, dp, dp, dp, dp, dp, dp, dp, dp, dp, dp]
        lib.orc_bilinear.argtypes = [dp, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_double, ctypes.c_double]
        lib.orc_bilinear.restype = ctypes.c_double
        lib.orc_bilinear_closed_form.argtypes = lib.orc_bilinear.argtypes
        lib.orc_bilinear_closed_form.restype = ctypes.c_double
        lib.orc_bilinear_grad.argtypes = [dp, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_double, ctypes.c_double, dp, dp]
        lib.orc_num_threads.restype = ctypes.c_int
        _lib = lib
        return lib


def num_threads() -> int:
    """Host threads the oracle's parallel loops use."""
    return int(_load().orc_num_threads())


class Problem:
    """Layer geometry: NCHW input, [C_out, C_in, Kh, Kw] weights."""

    def __init__(self, n, c_in, h, w, c_out, kh=3, kw=3, stride=1, pad=1,
                 dil=1, groups=1):
        sh, sw = (stride, stride) if np.isscalar(stride) else stride
        ph, pw = (pad, pad) if np.isscalar(pad) else pad
        dh, dw = (dil, dil) if np.isscalar(dil) else dil
        self.n, self.c_in, self.h, self.w, self.c_out = n, c_in, h, w, c_out
        self.kh, self.kw = kh, kw
        self.stride_h, self.stride_w = sh, sw
        self.pad_h, self.pad_w = ph, pw
        self.dil_h, self.dil_w = dh, dw
        self.groups = groups

    @property
    def ho(self):
        return (self.h + 2 * self.pad_h - self.dil_h * (self.kh - 1) - 1) // self.stride_h + 1

    @property
    def wo(self):
        return (self.w + 2 * self.pad_w - self.dil_w * (self.kw - 1) - 1) // self.stride_w + 1

    @property
    def n_off(self):
        return 2 * self.groups * self.kh * self.kw

    def c_struct(self) -> OracleProblem:
        return OracleProblem(self.n, self.c_in, self.h, self.w, self.c_out,
                             self.kh, self.kw, self.stride_h, self.stride_w,
                             self.pad_h, self.pad_w, self.dil_h, self.dil_w,
                             self.groups)


def _arr(a, shape=None):
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    if shape is not None and a.shape != tuple(shape):
        raise ValueError(f"expected shape {tuple(shape)}, got {a.shape}")
    return a


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _call(fn, *args):
    rc = fn(*args)
    if rc != 0:
        raise ValueError(f"oracle rejected the problem (code {rc})")


def offsets(p: Problem, x, w_off, b_off=None, offset_add=None):
    """Offset convolution output [N, 2GK, Ho, Wo] (Step 1 of 5)."""
    lib = _load()
    x = _arr(x, (p.n, p.c_in, p.h, p.w))
    w_off = _arr(w_off, (p.n_off, p.c_in, p.kh, p.kw))
    b_off = None if b_off is None else _arr(b_off, (p.n_off,))
    add = None if offset_add is None else _arr(offset_add, (p.n, p.n_off, p.ho, p.wo))
    out = np.empty((p.n, p.n_off, p.ho, p.wo))
    st = p.c_struct()
    _call(lib.orc_offsets, ctypes.byref(st), _ptr(x), _ptr(w_off), _ptr(b_off),
          _ptr(add), _ptr(out))
    return out


def column(p: Problem, x, off):
    """Deformed map [N, C_in, Kh*Kw, Ho, Wo] sampled at the given offsets."""
    lib = _load()
    x = _arr(x, (p.n, p.c_in, p.h, p.w))
    off = _arr(off, (p.n, p.n_off, p.ho, p.wo))
    out = np.empty((p.n, p.c_in, p.kh * p.kw, p.ho, p.wo))
    st = p.c_struct()
    _call(lib.orc_column, ctypes.byref(st), _ptr(x), _ptr(off), _ptr(out))
    return out


def column_adjoint(p: Problem, off, gcol):
    """Adjoint of ``column`` with respect to x: [N, C_in, H, W]."""
    lib = _load()
    off = _arr(off, (p.n, p.n_off, p.ho, p.wo))
    gcol = _arr(gcol, (p.n, p.c_in, p.kh * p.kw, p.ho, p.wo))
    out = np.empty((p.n, p.c_in, p.h, p.w))
    st = p.c_struct()
    _call(lib.orc_column_adjoint, ctypes.byref(st), _ptr(off), _ptr(gcol), _ptr(out))
    return out


def forward(p: Problem, x, w_off, b_off, w, offset_add=None):
    """Whole layer.  Returns (y [N, C_out, Ho, Wo], offsets [N, 2GK, Ho, Wo])."""
    lib = _load()
    x = _arr(x, (p.n, p.c_in, p.h, p.w))
    w_off = _arr(w_off, (p.n_off, p.c_in, p.kh, p.kw))
    b_off = None if b_off is None else _arr(b_off, (p.n_off,))
    w = _arr(w, (p.c_out, p.c_in, p.kh, p.kw))
    add = None if offset_add is None else _arr(offset_add, (p.n, p.n_off, p.ho, p.wo))
    y = np.empty((p.n, p.c_out, p.ho, p.wo))
    off = np.empty((p.n, p.n_off, p.ho, p.wo))
    st = p.c_struct()
    _call(lib.orc_forward, ctypes.byref(st), _ptr(x), _ptr(w_off), _ptr(b_off),
          _ptr(w), _ptr(add), _ptr(y), _ptr(off))
    return y, off


def backward(p: Problem, x, w_off, w, off, grad_y):
    """Gradients of sum(y * grad_y) at the saved offsets ``off``.

    Returns a dict with grad_x, grad_w_off, grad_b_off, grad_w and grad_offset
    (the gradient with respect to the total offsets, i.e. to offset_add)."""
    lib = _load()
    x = _arr(x, (p.n, p.c_in, p.h, p.w))
    w_off = _arr(w_off, (p.n_off, p.c_in, p.kh, p.kw))
    w = _arr(w, (p.c_out, p.c_in, p.kh, p.kw))
    off = _arr(off, (p.n, p.n_off, p.ho, p.wo))
    gy = _arr(grad_y, (p.n, p.c_out, p.ho, p.wo))
    out = dict(grad_x=np.empty((p.n, p.c_in, p.h, p.w)),
               grad_w_off=np.empty((p.n_off, p.c_in, p.kh, p.kw)),
               grad_b_off=np.empty((p.n_off,)),
               grad_w=np.empty((p.c_out, p.c_in, p.kh, p.kw)),
               grad_offset=np.empty((p.n, p.n_off, p.ho, p.wo)))
    st = p.c_struct()
    _call(lib.orc_backward, ctypes.byref(st), _ptr(x), _ptr(w_off), _ptr(w),
          _ptr(off), _ptr(gy), _ptr(out["grad_x"]), _ptr(out["grad_w_off"]),
          _ptr(out["grad_b_off"]), _ptr(out["grad_w"]), _ptr(out["grad_offset"]))
    return out


def _plane(plane):
    plane = _arr(plane)
    if plane.ndim != 2:
        raise ValueError("expected one H x W plane")
    return plane


def bilinear(plane, py, px):
    """Four-corner bilinear sample of one plane; zero outside the image."""
    plane = _plane(plane)
    return float(_load().orc_bilinear(_ptr(plane), plane.shape[0], plane.shape[1],
                                      float(py), float(px)))


def bilinear_closed_form(plane, py, px):
    """Tent-kernel sum over every pixel of the plane (independent statement)."""
    plane = _plane(plane)
    return float(_load().orc_bilinear_closed_form(
        _ptr(plane), plane.shape[0], plane.shape[1], float(py), float(px)))


def bilinear_grad(plane, py, px):
    """(dS/dpy, dS/dpx) with the lower corner at floor(p)."""
    plane = _plane(plane)
    dy = ctypes.c_double()
    dx = ctypes.c_double()
    _load().orc_bilinear_grad(_ptr(plane), plane.shape[0], plane.shape[1],
                              float(py), float(px), ctypes.byref(dy), ctypes.byref(dx))
    return float(dy.value), float(dx.value)


def relu(y):
    """max(y, 0) elementwise; NaN stays NaN (it is not <= 0)."""
    y = np.asarray(y, dtype=np.float64)
    return np.where(y <= 0.0, 0.0, y)


def relu_grad(act, g):
    """Gradient through the activation given its OUTPUT act: g where act > 0,
    else 0 (act > 0 exactly where the input was > 0)."""
    act = np.asarray(act, dtype=np.float64)
    return np.where(act > 0.0, np.asarray(g, dtype=np.float64), 0.0)
