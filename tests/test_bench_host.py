"""Host logic of bench.py that needs no GPU: the packed host/device buffers of
the end-to-end measurement (each group of tensors moves in one copy), and the
recorded DRAM-traffic table's tie to the kernel sources it was measured on."""
import hashlib
import os

import torch

import bench


def test_packed_views_are_aligned_disjoint_and_cover_every_tensor():
    specs = [("x", (8, 128, 28, 28), torch.bfloat16), ("b_off", (18,), torch.float32),
             ("w", (128, 128, 3, 3), torch.bfloat16), ("offset_add", (8, 18, 28, 28), torch.float32)]
    buf, views = bench._packed(specs, "cpu", False)
    base = buf.data_ptr()
    spans = []
    for name, shape, dt in specs:
        v = views[name]
        assert tuple(v.shape) == shape and v.dtype == dt and v.is_contiguous()
        off = v.data_ptr() - base
        assert off % 256 == 0  # the library wants 16-byte aligned pointers
        spans.append((off, off + v.numel() * v.element_size()))
    spans.sort()
    assert all(a[1] <= b[0] for a, b in zip(spans, spans[1:]))
    assert spans[-1][1] <= buf.numel()
    # writes through one view leave the others untouched
    for _, t in views.items():
        t.zero_()
    views["b_off"].fill_(3.0)
    assert float(views["offset_add"].abs().sum()) == 0.0 and float(views["b_off"].sum()) == 54.0


def test_traffic_records_name_existing_kernel_sources():
    csrc = os.path.join(bench.ROOT, "deformable_convolution_gb300", "csrc")
    for (workload, kernel), rec in bench.TRAFFIC.items():
        assert kernel in bench.KERNEL_SOURCES, kernel
        path = os.path.join(csrc, bench.KERNEL_SOURCES[kernel])
        assert os.path.exists(path), path
        assert rec["bytes"] > 0 and len(rec["source"]) == 16
        int(rec["source"], 16)
        # a stale record reads as null, never as another source's figure
        assert bench.source_hash(path) == hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]
