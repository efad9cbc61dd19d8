"""Training step over a stack of deformable layers with ReLU between them.

The explainer page "DefT: Boosting Scalability of Deformable Convolution
Operations on GPUs" measures whole networks built from deformable layers
("What people did before, and where it broke": deformable layers added
throughout a ResNet; "Why it works / Fixing the slowest stage lifts the whole
layer": training time of a fully deformable ResNet).  This module chains the C
ABI's calls for such a stack: per layer the forward (``deform_conv_fwd``) and
the backward that reuses the forward's deformed map
(``deform_conv_bwd_after_fwd``), with the ReLU between layers fused on both
sides: in the forward into the layer's main GEMM epilogue (``out_relu``, bit
for bit ``dc_relu_fwd`` of the plain output), in the backward into the grad_x
store of the layer above (``in_relu``, what ``dc_relu_bwd`` gives for the
float32 grad_x).
Marshalling only: buffers come from PyTorch, every step of the arithmetic runs
in the library's kernels.

Layer l's input is x[l] (x[0] is the caller's); x[l + 1] = relu(y[l]), which
the forward of layer l writes directly; y is kept for the last layer.  The
backward runs from the top: layer l's grad_y is the caller's grad_y for the
last layer, else relu'(x[l + 1]) * grad_x[l + 1], rounded to the dtype, which
the backward of layer l + 1 writes directly; grad_x (float32) is kept for
layer 0.
"""
from __future__ import annotations

import dataclasses

import torch

from . import binding as B


class Stack:
    """Buffers and calls of one forward + backward over ``len(params)`` layers.

    p: the layer problem (every layer has this geometry, C_in = C_out and the
       output size equal to the input size); params: per layer a dict with
       w_off, b_off, w (device tensors, p's dtype; b_off float32).  Each layer
       keeps its own backward workspace, so that its backward finds the
       deformed map its forward wrote."""

    def __init__(self, p: B.Problem, params, device):
        s = p.shapes()
        if s["x"] != s["y"]:
            raise ValueError("stacked layers need C_in = C_out and an unchanged size")
        self.p, self.params, self.L = p, params, len(params)
        self.p_relu = dataclasses.replace(p, out_relu=1)  # forward with the ReLU fused
        self.p_grelu = dataclasses.replace(p, in_relu=1)  # backward through the ReLU below
        dt, f32 = p.torch_dtype, torch.float32
        self.x = [None] + [torch.empty(s["x"], dtype=dt, device=device) for _ in range(self.L - 1)]
        self.y = [torch.empty(s["y"], dtype=dt, device=device) for _ in range(self.L)]
        self.off = [torch.empty(s["offset"], dtype=f32, device=device) for _ in range(self.L)]
        self.ws = [B.workspace(self.p_grelu if l else p, True, device) for l in range(self.L)]
        self.gx = [torch.empty(s["x"], dtype=f32, device=device)]
        self.gy = [torch.empty(s["y"], dtype=dt, device=device) for _ in range(self.L - 1)] + [None]
        self.grads = [dict(grad_w_off=torch.empty(s["w_off"], dtype=f32, device=device),
                           grad_b_off=torch.empty(s["b_off"], dtype=f32, device=device),
                           grad_w=torch.empty(s["w"], dtype=f32, device=device))
                      for _ in range(self.L)]

    def forward(self, x0, offset_add=None):
        """Runs every layer's forward; returns the last layer's output y."""
        self.x[0] = x0
        for l in range(self.L):
            q, last = self.params[l], l + 1 == self.L
            B.deform_conv_fwd(self.p if last else self.p_relu, self.x[l], q["w_off"], q["b_off"],
                              q["w"], offset_add if l == 0 else None,
                              self.y[l] if last else self.x[l + 1], self.off[l], None, self.ws[l])
        return self.y[-1]

    def backward(self, grad_y):
        """Runs every layer's backward from the top; returns grad_x of layer 0.
        Weight gradients land in ``self.grads[l]``."""
        self.gy[-1] = grad_y
        for l in reversed(range(self.L)):
            self.backward_layer(l)
        return self.gx[0]

    def backward_layer(self, l, stream=None):
        """Layer l's backward: its weight gradients, and layer l - 1's grad_y
        through the ReLU between them (grad_x itself for layer 0)."""
        q, g = self.params[l], self.grads[l]
        B.deform_conv_bwd(self.p_grelu if l else self.p, self.x[l], q["w_off"], q["w"],
                          self.off[l], self.gy[l], self.gy[l - 1] if l else self.gx[0],
                          g["grad_w_off"], g["grad_b_off"], g["grad_w"], None, self.ws[l],
                          stream, after_fwd=True)

    def step(self, x0, grad_y, offset_add=None):
        self.forward(x0, offset_add)
        return self.backward(grad_y)
