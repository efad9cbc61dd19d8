"""Seeded synthetic inputs for the deformable layer (tests and benchmark).

This module only draws random numbers and sets their scales; it holds none
of the layer's arithmetic, and both the CUDA path and the oracle consume its
output.  Each workload stands in for a layer shape of the networks the
explainer page "DefT: Boosting Scalability of Deformable Convolution
Operations on GPUs" evaluates on ("The evaluation": deformable Mask R-CNN on
COCO, all-deformable ResNet-18 on ImageNet); those datasets and trained
weights are not available, so inputs are random with the stated
distributions.

Recipe (one ``torch.Generator(seed)`` on the CPU, draws in this order):
  1. x: uniform(-1, 1), or max(N(0, 1), 0) for the post-ReLU workloads;
  2. w_off ~ N(0, s^2) with s = sigma / sqrt(C_in * Kh * Kw * Var(x)), so the
     offset convolution's output has standard deviation ~sigma at interior
     pixels; b_off = -E[x] * sum_{c,i,j} w_off[m, c, i, j] removes the mean a
     non-centred input gives (zero for centred x);
  3. w ~ N(0, gain / (Kh * Kw * C_in)), gain 1 (gain 2 for the training
     stack: He initialisation, which keeps a ReLU network's activations at
     the scale of its input from layer to layer);
  4. offset_add: each element independently, with probability
     ``outlier_p``, is +-``outlier_px`` (uniform sign), else 0;
  5. grad_y ~ N(0, 1).
bf16 workloads round x, w_off and w to bf16 (round to nearest even) once;
both sides of every comparison receive the same rounded values.

Stacks of layers (``generate_stack``): layer 0 is ``generate(wl)``; layer l
draws its w_off, b_off and w by the same recipe from seed ``wl.seed + 1000 *
l``.  The offset weights of every layer are scaled for a post-ReLU N(0, 1)
input, the distribution a He-initialised layer's ReLU output keeps
approximately; grad_y at the stack's output is layer 0's draw.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

from .binding import DC_BF16, DC_F32, Problem


@dataclass(frozen=True)
class Workload:
    name: str
    n: int
    c_in: int
    c_out: int
    h: int
    w: int
    k: int = 3
    stride: int = 1
    pad: int = 1
    dil: int = 1
    groups: int = 1
    dtype: int = DC_F32
    sigma: float = 1.0          # target offset standard deviation (px)
    relu_x: bool = False        # x = max(N(0,1), 0) instead of U(-1, 1)
    outlier_p: float = 0.0
    outlier_px: float = 0.0
    layers: int = 1
    w_gain: float = 1.0         # variance gain of the main weights
    seed: int = 0

    def problem(self, n=None, halo_margin=-1) -> Problem:
        return Problem(self.n if n is None else n, self.c_in, self.h, self.w, self.c_out,
                       self.k, self.k, self.stride, self.pad, self.dil, self.groups,
                       self.dtype, halo_margin)

    @property
    def dtype_name(self):
        return "bf16" if self.dtype == DC_BF16 else "f32"


WORKLOADS = {
    # tiny layer: N1 C16->16 32x32, 3x3 s1 p1 d1, one offset group, fp32
    "tiny_f32": Workload("tiny_f32", 1, 16, 16, 32, 32, seed=0),
    # ResNet-50 res3-style: N8 C128->128 28x28, offsets ~N(0,1) px + 1% outliers at +-8 px
    "res3_f32": Workload("res3_f32", 8, 128, 128, 28, 28, outlier_p=0.01, outlier_px=8.0,
                         seed=1),
    "res3_bf16": Workload("res3_bf16", 8, 128, 128, 28, 28, dtype=DC_BF16, outlier_p=0.01,
                          outlier_px=8.0, seed=1),
    # detector-resolution res4: N2 C256->256 50x84, offsets ~N(0, 2) px, post-ReLU input
    "res4_bf16": Workload("res4_bf16", 2, 256, 256, 50, 84, dtype=DC_BF16, sigma=2.0,
                          relu_x=True, seed=2),
    # early layer: N16 C64->64 112x112, pad 2, dilation 2, 4 offset groups, offsets ~N(0, 1.5)
    "early_bf16": Workload("early_bf16", 16, 64, 64, 112, 112, pad=2, dil=2, groups=4,
                           dtype=DC_BF16, sigma=1.5, seed=3),
    # one layer of the 4-layer training stack: N8 C256->256 56x56, offsets ~N(0, 1)
    # (the whole stack: 4 such layers with ReLU between them, He-initialised)
    "stack_bf16": Workload("stack_bf16", 8, 256, 256, 56, 56, dtype=DC_BF16, relu_x=True,
                           layers=4, w_gain=2.0, seed=4),
}


def generate(wl: Workload, n=None, seed=None):
    """CPU tensors for one layer: x, w_off, b_off, w, offset_add, grad_y.

    x, w_off and w come back in the workload's dtype; b_off, offset_add and
    grad_y are float32 (grad_y in the workload's dtype)."""
    n = wl.n if n is None else n
    gen = torch.Generator().manual_seed(wl.seed if seed is None else seed)
    p = wl.problem(n)
    K = wl.k * wl.k
    if wl.relu_x:
        x = torch.randn(p.shapes()["x"], generator=gen).clamp_min_(0.0)
        mean, var = 1.0 / math.sqrt(2 * math.pi), 0.5 - 1.0 / (2 * math.pi)
    else:
        x = torch.rand(p.shapes()["x"], generator=gen) * 2.0 - 1.0
        mean, var = 0.0, 1.0 / 3.0
    s = wl.sigma / math.sqrt(wl.c_in * K * var)
    w_off = torch.randn(p.shapes()["w_off"], generator=gen) * s
    w = torch.randn(p.shapes()["w"], generator=gen) * math.sqrt(wl.w_gain / (K * wl.c_in))
    tdt = p.torch_dtype
    x, w_off, w = x.to(tdt), w_off.to(tdt), w.to(tdt)
    b_off = (-mean * w_off.float().sum(dim=(1, 2, 3))).contiguous()
    offset_add = None
    if wl.outlier_p > 0:
        shape = p.shapes()["offset"]
        hit = torch.rand(shape, generator=gen) < wl.outlier_p
        sign = torch.where(torch.rand(shape, generator=gen) < 0.5, -1.0, 1.0)
        offset_add = (hit.float() * sign * wl.outlier_px).contiguous()
    grad_y = torch.randn(p.shapes()["y"], generator=gen).to(tdt)
    return dict(x=x, w_off=w_off, b_off=b_off, w=w, offset_add=offset_add, grad_y=grad_y)


def generate_stack(wl: Workload, n=None):
    """Inputs of a stack of ``wl.layers`` layers with ReLU between them:
    (x of layer 0, [dict(w_off, b_off, w) per layer], grad_y at the output).
    Every layer has C_in = C_out and keeps the spatial size, so that a layer's
    output is the next layer's input."""
    p = wl.problem(n)
    if p.c_in != p.c_out or (p.ho, p.wo) != (p.h, p.w):
        raise ValueError("a stack needs layers that keep the channel count and size")
    first = generate(wl, n)
    layers = [{k: first[k] for k in ("w_off", "b_off", "w")}]
    for l in range(1, wl.layers):
        d = generate(wl, 1, seed=wl.seed + 1000 * l)
        layers.append({k: d[k] for k in ("w_off", "b_off", "w")})
    return first["x"], layers, first["grad_y"]


def conv_flops(p: Problem) -> float:
    """Conv-equivalent flops of one forward pass: the main convolution plus the
    offset convolution, 2 * P * C_in * K * (C_out + 2GK)."""
    P = p.n * p.ho * p.wo
    return 2.0 * P * p.c_in * p.kh * p.kw * (p.c_out + p.n_off)
