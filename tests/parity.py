"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
and the fp64 oracle on the same seeded inputs and compare them.

Error measure (per output tensor): max_i |gpu_i - ref_i| / max_i |ref_i|,
i.e. the largest deviation relative to the tensor's scale.  Bars: 1e-4 for
float32 problems, 2e-2 for bf16 inputs with float32 accumulation."""
import numpy as np
import torch

import oracle
from deformable_convolution_gb300 import binding as B

TOL = {B.DC_F32: 1e-4, B.DC_BF16: 2e-2}


def oracle_problem(p: B.Problem) -> oracle.Problem:
    return oracle.Problem(p.n, p.c_in, p.h, p.w, p.c_out, p.kh, p.kw, p.stride, p.pad,
                          p.dil, p.offset_groups)


def f64(t):
    return None if t is None else t.detach().to("cpu", torch.float64).numpy()


def rel_err(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    scale = np.max(np.abs(ref)) if ref.size else 0.0
    if scale == 0.0:
        return float(np.max(np.abs(got))) if got.size else 0.0
    return float(np.max(np.abs(got - ref)) / scale)


def elementwise_err(got, ref, tol):
    """Largest violation ratio of the per-element bound
    |got - ref| <= tol * (|ref| + max|ref| / 4): relative for large elements,
    a quarter of the tensor-wide bound for small ones (<= 1 passes)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    scale = np.max(np.abs(ref)) if ref.size else 0.0
    if scale == 0.0:
        return 0.0 if not got.size or np.max(np.abs(got)) == 0.0 else float("inf")
    bound = tol * (np.abs(ref) + 0.25 * scale)
    return float(np.max(np.abs(got - ref) / bound))


def to_dev(d):
    return {k: (None if v is None else v.cuda()) for k, v in d.items()}


def gpu_forward(p, d, margin=None, count=True):
    if margin is not None:
        p = B.Problem(p.n, p.c_in, p.h, p.w, p.c_out, p.kh, p.kw, p.stride, p.pad, p.dil,
                      p.offset_groups, p.dtype, margin)
    dd = to_dev(d)
    cnt = torch.zeros(1, dtype=torch.int64, device="cuda") if count else None
    y, off = B.forward(p, dd["x"], dd["w_off"], dd["b_off"], dd["w"], dd["offset_add"],
                       slowpath_count=cnt)
    torch.cuda.synchronize()
    return y, off, (int(cnt.item()) if count else None)


def gpu_backward(p, d, offsets_f32):
    dd = to_dev(d)
    g = B.backward(p, dd["x"], dd["w_off"], dd["w"], offsets_f32.cuda().contiguous(),
                   dd["grad_y"])
    torch.cuda.synchronize()
    return g


def oracle_forward(p, d):
    return oracle.forward(oracle_problem(p), f64(d["x"]), f64(d["w_off"]), f64(d["b_off"]),
                          f64(d["w"]), f64(d["offset_add"]))


def oracle_backward(p, d, off64):
    return oracle.backward(oracle_problem(p), f64(d["x"]), f64(d["w_off"]), f64(d["w"]),
                           off64, f64(d["grad_y"]))


def check_layer(p, d, tol=None, margin=None, check_bwd=True):
    """Forward and backward parity of one problem; returns the error table."""
    tol = TOL[p.dtype] if tol is None else tol
    y, off, _ = gpu_forward(p, d, margin)
    y_ref, off_ref = oracle_forward(p, d)
    errs = {"y": rel_err(f64(y), y_ref), "offset": rel_err(f64(off), off_ref)}
    if check_bwd:
        # both sides take the same float32 offsets (the oracle's, rounded)
        off32 = torch.from_numpy(off_ref).float()
        g = gpu_backward(p, d, off32)
        ref = oracle_backward(p, d, off32.double().numpy())
        for k in ("grad_x", "grad_w", "grad_w_off", "grad_b_off", "grad_offset"):
            errs[k] = rel_err(f64(g[k]), ref[k])
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"parity failed (tol {tol}): {errs}"
    # and element by element: small outputs may not hide large relative errors
    # behind the tensor's maximum
    elem = {"y": elementwise_err(f64(y), y_ref, tol)}
    if check_bwd:
        for k in ("grad_x", "grad_w", "grad_w_off", "grad_b_off", "grad_offset"):
            elem[k] = elementwise_err(f64(g[k]), ref[k], tol)
    bad = {k: v for k, v in elem.items() if not v <= 1.0}
    assert not bad, f"elementwise parity failed (tol {tol}): {elem}"
    return errs
