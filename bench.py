"""Benchmark of the deformable convolution layer (forward + backward) on GB300.

One step = one forward and one backward pass of the layer over one batch of
synthetic input, through the C ABI (offset convolution + bilinear sampling
fused in K1, main convolution GEMM, and the backward kernels).  Inputs are
resident in HBM when the timed region starts; L2 is flushed (a 256 MiB write,
outside the timed events) before every timed step.  The step is captured once
in a CUDA graph and replayed.

Prints one JSON line.  ``--impl reference`` times the fp64 CPU oracle instead
(the reference arm: a deliberately slow, obviously correct program on the host
cores), on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "deform-conv layer fwd+bwd ms and GFLOP/s; sampling-stage HBM GB/s vs GB300 peak"
FLUSH_BYTES = 256 << 20


def fp32_alu_tflops(dev):
    """FFMA peak of the part: SMs (from the device) x 128 fp32 lanes x 2 flop
    x the maximum SM clock (MEASURED_PEAKS.json's sm_max_mhz, else 2070 MHz)."""
    import torch
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = measured_peaks()[0].get("sm_max_mhz", 2070.0)
    return sms * 128 * 2 * mhz * 1e6 / 1e12, sms, mhz

# Nominal dense TF32 : bf16 tensor rate of the part (1.1 : 2.25 PFLOP/s).
TF32_PER_BF16 = 1.1 / 2.25


def tf32_path(p):
    """True when a float32 problem's GEMMs run on the tensor cores (kind::tf32):
    the library takes that path when kdim and the output pixel count are
    multiples of 4 (16-byte rows for every tensor map)."""
    return (p.c_in * p.kh * p.kw) % 4 == 0 and (p.ho * p.wo) % 4 == 0


# DRAM traffic of one launch from an ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum), keyed by (workload, kernel); valid only while the
# kernel's source file hashes to the recorded value (else reported as null).
TRAFFIC = {
    # ncu sections capture of one training step of the stack (cold caches),
    # one launch each (layer 3 of the timed step); writes that stay in the
    # 126 MB L2 are not counted (k4cl_input: layer 3's store with the ReLU
    # below fused, whose bf16 output stays in L2 for the next backward).
    ("stack_bf16", "k3_cl_bwd"): {"bytes": 171687424, "source": "02a91a919a0f90c2"},
    ("stack_bf16", "k1_cl_sample"): {"bytes": 69400064, "source": "cbee7b1732934ddc"},
    ("stack_bf16", "k4cl_input"): {"bytes": 40613888, "source": "1f46bd658bb5b517"},
    ("stack_bf16", "k4cl_weight"): {"bytes": 14768640, "source": "1f46bd658bb5b517"},
    ("stack_bf16", "gemm_fwd"): {"bytes": 120043008, "source": "d21b94d0b4d051a4"},
    ("stack_bf16", "gemm_gcol"): {"bytes": 97627136, "source": "d21b94d0b4d051a4"},
    ("stack_bf16", "gemm_gw"): {"bytes": 133967104, "source": "d21b94d0b4d051a4"},
}
KERNEL_SOURCES = {
    "k1_band_sample": "k1_sample.cu", "k3_band_bwd": "k3_band_bwd.cu",
    "k1_cl_sample": "k1_cl.cu", "k3_cl_bwd": "k3_cl.cu", "k4cl_input": "k4_cl.cu",
    "k4cl_weight": "k4_cl.cu",
    # bf16 workloads run the offset-convolution backward on tensor cores
    "k4_offconv_bwd": "k4_offconv_bwd_tc.cu",
    "gemm_fwd": "gemm_tc.cu", "gemm_gcol": "gemm_tc.cu", "gemm_gw": "gemm_tc.cu",
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="stack_bf16")
    ap.add_argument("--single-layer", action="store_true",
                    help="one layer of a stacked workload instead of the whole stack")
    ap.add_argument("--no-ablations", action="store_true")
    ap.add_argument("--eager", action="store_true", help="no CUDA graph")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="budget of the oracle's CPU-baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--roofline-iters", type=int, default=200)
    ap.add_argument("--e2e-iters", type=int, default=20)
    ap.add_argument("--only", choices=["stage", "offsets", "replay", "step"],
                    help="profiling runs: launch only the sampling stage (fused, offsets only, or "
                         "sampling at given offsets) or the whole step, warm-up + steps times on "
                         "layer 0's inputs, eagerly, and print the device time per call")
    return ap.parse_args()


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if os.environ.get("DC_BENCH_GLOO") is None else "gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, v, device):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def source_hash(path):
    return hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi samples (200 ms) of the SM clock and throttle reasons."""
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.uuid = uuid
        self.proc = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        self.proc.wait()
        self.out.flush()
        rows = []
        with open(self.out.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                if self.uuid and parts[0] != self.uuid:
                    continue
                rows.append(parts)
        os.unlink(self.out.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def oracle_sample(wl, rows=None):
    """The oracle, as it stands, on image 0 of the workload (fwd + bwd in
    fp64), optionally on its first `rows` input rows only (same per-pixel
    work, for bounded samples).  Returns (run, flops per run, description)."""
    import oracle
    from deformable_convolution_gb300 import workloads as W
    d = W.generate(wl)
    p1 = wl.problem(1)
    h = p1.h if rows is None else max(1, min(p1.h, rows))
    p1 = type(p1)(1, p1.c_in, h, p1.w, p1.c_out, p1.kh, p1.kw, p1.stride, p1.pad, p1.dil,
                  p1.offset_groups, p1.dtype)
    s = p1.shapes()
    ho, wo = s["y"][2], s["y"][3]

    def crop(k, v):
        if v is None:
            return None
        if k == "x":
            return v[:1, :, :h]
        if k in ("offset_add", "grad_y"):
            return v[:1, :, :ho, :wo]
        return v
    one = {k: crop(k, v) for k, v in d.items()}
    op = oracle.Problem(1, p1.c_in, h, p1.w, p1.c_out, p1.kh, p1.kw, p1.stride, p1.pad,
                        p1.dil, p1.offset_groups)
    f64 = lambda t: None if t is None else t.contiguous().double().numpy()  # noqa: E731
    args = [f64(one[k]) for k in ("x", "w_off", "b_off", "w", "offset_add")]
    gy = f64(one["grad_y"])

    def run():
        y, off = oracle.forward(op, *args)
        oracle.backward(op, args[0], args[1], args[3], off, gy)
    what = f"image 0 of {wl.name} (N=1 of {wl.n})" + (
        f", input rows 0..{h - 1} of {wl.h}" if h < wl.h else "")
    return run, 3 * W.conv_flops(p1), what


def cpu_baseline(wl, seconds, stacked=False):
    """The oracle on image 0 of the workload (fwd + bwd), repeated until
    `seconds` have passed (at least once).  For a stack: image 0 of its first
    layer (every layer has the same shape, so the per-image, per-layer rate
    is the stack's rate)."""
    import oracle
    run, flops, what = oracle_sample(wl)
    if stacked:
        what = f"layer 1 of {wl.layers}, " + what
    runs, t0 = 0, time.perf_counter()
    while True:
        run()
        runs += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    per = el / runs
    return {"value": flops / per / 1e9, "unit": "GFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"{what}, fwd+bwd in fp64, {runs} run(s), {per * 1e3:.0f} ms each",
            "ms_per_image": per * 1e3}


REFERENCE_BUDGET_S = 120.0  # whole --impl reference run (warm-up + timed steps)


def run_reference(args, world, rank):
    """The oracle as the reference arm: each step is a bounded sample of the
    workload (image 0, cropped to the rows that keep the whole run within
    REFERENCE_BUDGET_S seconds), timed on the host cores."""
    import oracle
    from deformable_convolution_gb300 import workloads as W
    if rank != 0:
        return
    wl = W.WORKLOADS[args.workload]
    stacked = wl.layers > 1 and not args.single_layer
    run, _, _ = oracle_sample(wl)
    t0 = time.perf_counter()
    run()
    t_full = time.perf_counter() - t0
    per_step = REFERENCE_BUDGET_S / max(1, args.steps + args.warmup)
    rows = wl.h if t_full <= per_step else max(1, int(wl.h * per_step / t_full))
    run, flops, what = oracle_sample(wl, rows)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    el = time.perf_counter() - t0
    ms = el / max(1, args.steps) * 1e3
    gflops = flops / (ms / 1e3) / 1e9
    sample = f"{what}, fwd+bwd in fp64 per step"
    if stacked:
        # every layer of the stack has this shape: the rate of one layer's
        # sample is the stack's rate
        sample = f"layer 1 of {wl.layers}, " + sample
    line = {"impl": "reference", "metric": METRIC, "value": gflops, "unit": "GFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(job_config(wl, stacked), step=sample),
            "cpu_baseline": {"value": gflops, "unit": "GFLOP/s", "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": gflops, "unit": "GFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "flops_per_step": flops}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    import torch

    from deformable_convolution_gb300 import workloads as W

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = W.WORKLOADS[args.workload]
    stacked = wl.layers > 1 and not args.single_layer
    if args.only:
        run_only(args, wl, stacked, dev)
        return
    job = StackJob(wl, dev) if stacked else LayerJob(wl, dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    ms_step, graph_used, launches_per_step, wall, clocks = time_steps(job, args, world, dev,
                                                                      stream, flush)
    value = job.flops_step * world / (ms_step / 1e3) / 1e9
    line = {"metric": METRIC, "value": value, "unit": "GFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": wl.dtype_name, "data": "synthetic",
            "config": dict(job.config(), l2="flushed (256 MiB write) before every timed step",
                           graph=graph_used, parallelism=f"replicas x{world}"),
            "flops_per_step": job.flops_step, "wall_s_timed_region": wall,
            "gpu_launches": launches_per_step * args.steps, "clocks": clocks}

    if rank == 0:
        p, t = job.p, job.t
        kernels = kernel_breakdown(p, wl, job.step, dev, stream, flush)
        dom = dict(kernels[0])
        line["roofline"] = {k: dom[k] for k in ("kernel", "bound", "achieved", "peak", "unit", "frac",
                                                "traffic", "ms_per_launch", "peak_source")
                            if k in dom}
        line["roofline"]["note"] = "dominant kernel of the step (longest per-launch time)"
        line["kernels"] = kernels
        line["sampling_stage"] = k1_roofline(p, t, dev, stream, flush, wl, args.roofline_iters)
        if stacked:
            line["standard_conv_ratio"] = standard_conv_reference(job, dev, stream, flush,
                                                                  ms_step, args.roofline_iters // 4)
            line["offset_std_per_layer"] = job.offset_std()
        if not args.no_ablations:
            line["unfused_ablation"] = unfused_ablation(p, t, dev, stream, flush,
                                                        args.roofline_iters)
            sga = sampled_gemm_ablation(p, t, dev, stream, flush, args.roofline_iters)
            if sga is not None:
                line["sampled_gemm_ablation"] = sga
        line["margin"] = margin_report(p, t, dev)
        line["e2e"] = (e2e_stack(job, dev, stream, args.e2e_iters) if stacked
                       else e2e(p, job.d, dev, stream, job.flops_step, args.e2e_iters))
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(wl, args.cpu_seconds, stacked)
            line["cpu_baseline"].pop("ms_per_image", None)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_only(args, wl, stacked, dev):
    """A short eager run of one piece of the path, for profilers: the sampling
    stage three ways (deform_conv_sample fused, deform_conv_offsets, or
    deform_conv_sample at offsets given) on layer 0's inputs, or the whole
    step."""
    import torch

    from deformable_convolution_gb300 import binding as B
    job = StackJob(wl, dev) if stacked else LayerJob(wl, dev)
    p, t = job.p, job.t
    s = p.shapes()
    col = torch.empty(B.col_shape(p), dtype=p.torch_dtype, device=dev)
    off = torch.empty(s["offset"], dtype=torch.float32, device=dev)
    ws = B.workspace(p, False, dev)
    B.deform_conv_offsets(p, t["x"], t["w_off"], t["b_off"], t["offset_add"], off, ws=ws)
    launch = {
        "stage": lambda: B.deform_conv_sample(p, t["x"], t["w_off"], t["b_off"], t["offset_add"],
                                              None, col, off, ws=ws),
        "offsets": lambda: B.deform_conv_offsets(p, t["x"], t["w_off"], t["b_off"],
                                                 t["offset_add"], off, ws=ws),
        "replay": lambda: B.deform_conv_sample(p, t["x"], None, None, None, off, col, ws=ws),
        "step": job.step,
    }[args.only]
    for _ in range(args.warmup):
        launch()
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.steps):
        launch()
    b.record()
    torch.cuda.synchronize(dev)
    print(json.dumps({"only": args.only, "workload": wl.name, "stacked": stacked,
                      "ms_per_call": a.elapsed_time(b) / max(1, args.steps)}), flush=True)


def job_config(wl, stacked):
    """The `config` object of the JSON line (the workload, with its sizes)."""
    c = {"workload": (f"{wl.name} x{wl.layers} layers, ReLU between (training step)" if stacked
                      else wl.name),
         "layers": wl.layers if stacked else 1, "n": wl.n, "c_in": wl.c_in, "c_out": wl.c_out,
         "h": wl.h, "w": wl.w, "k": wl.k, "stride": wl.stride, "pad": wl.pad, "dil": wl.dil,
         "offset_groups": wl.groups}
    if stacked:
        c["offsets"] = (f"N(0,{wl.sigma}) px (offset weights scaled for a post-ReLU N(0,1) "
                        "input in every layer; measured std per layer in offset_std_per_layer)")
        c["init"] = "He (main weights N(0, 2/(9 C_in)))"
        c["backward"] = ("deform_conv_bwd_after_fwd per layer, the ReLU between layers fused into "
                         "the grad_x store of the layer above (in_relu)")
        c["forward"] = "deform_conv_fwd per layer, the ReLU between layers fused into its GEMM epilogue (out_relu)"
    else:
        c["offsets"] = f"N(0,{wl.sigma}) px" + (
            f" + {wl.outlier_p:.0%} outliers at +-{wl.outlier_px} px" if wl.outlier_p else "")
        c["backward"] = ("deform_conv_bwd_after_fwd (reuses the forward's deformed map from the "
                         "shared workspace)")
    return c


class LayerJob:
    """One forward + backward of one layer (the backward reusing the forward's
    deformed map from the shared workspace)."""

    def __init__(self, wl, dev):
        import torch

        from deformable_convolution_gb300 import binding as B
        from deformable_convolution_gb300 import workloads as W
        self.wl, self.p = wl, wl.problem()
        self.d = W.generate(wl)
        self.t = t = {k: (None if v is None else v.to(dev)) for k, v in self.d.items()}
        p, s = self.p, self.p.shapes()
        f32 = torch.float32
        self.y = torch.empty(s["y"], dtype=p.torch_dtype, device=dev)
        self.off = torch.empty(s["offset"], dtype=f32, device=dev)
        self.g = {k: torch.empty(s[sh], dtype=f32, device=dev) for k, sh in
                  (("gx", "x"), ("gwo", "w_off"), ("gbo", "b_off"), ("gw", "w"), ("goff", "offset"))}
        self.ws = B.workspace(p, True, dev)
        self.flops_step = 3 * W.conv_flops(p)

        def step():
            B.deform_conv_fwd(p, t["x"], t["w_off"], t["b_off"], t["w"], t["offset_add"], self.y,
                              self.off, None, self.ws)
            g = self.g
            B.deform_conv_bwd(p, t["x"], t["w_off"], t["w"], self.off, t["grad_y"], g["gx"],
                              g["gwo"], g["gbo"], g["gw"], g["goff"], self.ws, after_fwd=True)
        self.step = step

    def config(self):
        return job_config(self.wl, False)


class StackJob:
    """The training step of a stack of deformable layers with ReLU between
    them: every layer's forward, then every layer's backward from the top
    (each reusing its forward's deformed map), through the C ABI."""

    def __init__(self, wl, dev):
        from deformable_convolution_gb300 import stack as S
        from deformable_convolution_gb300 import workloads as W
        self.wl, self.p = wl, wl.problem()
        x0, layers, gy = W.generate_stack(wl)
        self.x0, self.gy = x0.to(dev), gy.to(dev)
        self.params = [{k: v.to(dev) for k, v in q.items()} for q in layers]
        self.host = (x0, layers, gy)
        self.stack = S.Stack(self.p, self.params, dev)
        # layer 0's inputs, for the single-kernel measurements
        q = self.params[0]
        self.t = {"x": self.x0, "w_off": q["w_off"], "b_off": q["b_off"], "w": q["w"],
                  "offset_add": None, "grad_y": self.gy}
        self.flops_step = 3 * W.conv_flops(self.p) * wl.layers
        self.step = lambda: self.stack.step(self.x0, self.gy)

    def config(self):
        return job_config(self.wl, True)

    def offset_std(self):
        import torch
        self.stack.forward(self.x0)
        torch.cuda.synchronize()
        return [float(o.std()) for o in self.stack.off]


def time_steps(job, args, world, dev, stream, flush):
    """W warm-up steps, then K timed steps (each a CUDA-graph replay of the
    whole step unless --eager) between barriers and synchronisations, each
    step bracketed by its own CUDA events on the launching stream after an
    L2 flush.  Returns (max-over-ranks ms per step, graph used, launches per
    step, wall seconds of the timed region, clock record)."""
    import torch

    from deformable_convolution_gb300 import binding as B
    launches_before = B.launch_count()
    with torch.cuda.stream(stream):
        job.step()  # first call (attributes, module load) outside any capture
    torch.cuda.synchronize(dev)
    launches_per_step = B.launch_count() - launches_before
    graph = None
    if not args.eager:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            job.step()
        torch.cuda.synchronize(dev)

    def run_step():
        if graph is not None:
            graph.replay()
        else:
            job.step()

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            flush.fill_(1)
            run_step()
    torch.cuda.synchronize(dev)

    props = torch.cuda.get_device_properties(dev)
    uuid = "GPU-" + str(props.uuid) if hasattr(props, "uuid") else None
    sampler = ClockSampler(uuid)
    sampler.start()
    time.sleep(0.3)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            starts[i].record(stream)
            run_step()
            ends[i].record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    wall = time.perf_counter() - wall0
    clocks = sampler.stop()
    total_ms = sum(a.elapsed_time(b) for a, b in zip(starts, ends))
    total_ms = max_over_ranks(world, total_ms, dev)
    return total_ms / args.steps, graph is not None, launches_per_step, wall, clocks


def standard_conv_reference(job, dev, stream, flush, ms_deform, iters):
    """The same stack with zero offsets, i.e. a standard convolution, run through
    torch.nn.functional.conv2d (cuDNN) with ReLU between layers, forward and
    backward (gradients of the input and of every weight), in the same dtype.
    A measurement reference only, never part of the library: the ratio of the
    deformable step to it is the on-box counterpart of the explainer page's
    roughly 4x slowdown of a deformable layer against a standard one ("The
    argument in one glance / Problem")."""
    import torch
    import torch.nn.functional as F
    p = job.p
    torch.backends.cudnn.benchmark = True
    ws = [q["w"].detach().clone().requires_grad_() for q in job.params]
    xin = job.x0.detach().clone().requires_grad_()
    gy = job.gy

    def run():
        h = xin
        for l, w in enumerate(ws):
            h = F.conv2d(h, w, stride=p.stride, padding=p.pad, dilation=p.dil)
            if l + 1 < len(ws):
                h = F.relu(h)
        torch.autograd.grad(h, [xin] + ws, gy)

    with torch.cuda.stream(stream):
        for _ in range(5):
            run()
        torch.cuda.synchronize(dev)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(max(iters, 10))]
        for a, b in ev:
            flush.fill_(11)
            a.record(stream)
            run()
            b.record(stream)
    torch.cuda.synchronize(dev)
    ms = statistics.median(a.elapsed_time(b) for a, b in ev)
    return {"standard_ms_per_step": ms, "deformable_ms_per_step": ms_deform,
            "ratio": ms_deform / ms, "page_ratio": "about 4x (deformable vs standard layer)",
            "how": "torch.nn.functional.conv2d (cuDNN, benchmark mode) + relu, autograd "
                   "backward to the input and all weights, same dtype, CUDA events, median; "
                   "a measurement reference only"}


def traffic_for(workload, kernel):
    rec = TRAFFIC.get((workload, kernel))
    if not rec:
        return None
    src = os.path.join(ROOT, "deformable_convolution_gb300", "csrc", KERNEL_SOURCES[kernel])
    return rec["bytes"] if rec["source"] == source_hash(src) else None


def kernel_costs(p, has_add):
    """Algorithmic bytes (HBM-bound kernels) or flops (GEMMs) of one launch of
    each kernel of the forward + backward step."""
    elt = 2 if p.dtype == 1 else 4
    P = p.n * p.ho * p.wo
    kdim = p.c_in * p.kh * p.kw
    x_b = p.n * p.c_in * p.h * p.w * elt
    off_b = p.n_off * P * 4
    gemm = 2.0 * p.c_out * kdim * P
    gx_b = p.n * p.c_in * p.h * p.w * 4
    # gcol is bf16 from the tensor-core GEMM (bf16 problems), fp32 otherwise; the
    # step's backward reuses the forward's deformed map, so K3 writes no map
    gcol_elt = 2 if p.dtype == 1 else 4
    k3 = (x_b + off_b + kdim * P * gcol_elt  # read x, offsets, gcol
          + gx_b + off_b)                     # write grad_x, grad_offset
    k4 = (x_b + off_b + p.n_off * kdim * elt  # read x, grad_offset, w_off
          + 2 * gx_b                          # add into grad_x (read + write)
          + p.n_off * (kdim + 1) * 4)         # write grad_w_off, grad_b_off
    # channels-last path (bf16, C_in a multiple of 64): x copied to NHWC once
    # per layer; the backward kernels read that copy
    w_b = p.c_out * kdim * elt
    woff_b = p.n_off * kdim * elt
    k4cl_chunks = 152 // max(1, p.c_in // 64)
    return {
        "k1_band_sample": ("hbm", k1_bytes(p, has_add)),
        "k1_cl_sample": ("hbm", k1_bytes(p, has_add)),
        "k1_cl_offsets": ("hbm", x_b + woff_b + off_b * (2 if has_add else 1)),
        # x to its NHWC copy, w permuted, w_off laid out: one launch
        "cl_prep": ("hbm", 2 * x_b + 2 * w_b + 2 * woff_b),
        "gemm_fwd": ("tensor", gemm), "gemm_gcol": ("tensor", gemm), "gemm_gw": ("tensor", gemm),
        "k3_band_bwd": ("hbm", k3),
        # read x (NHWC), offsets, gcol; grad_x into the NHWC float32 buffer, goff
        "k3_cl_bwd": ("hbm", k3),
        "gx_to_nchw": ("hbm", 2 * gx_b),
        "k4_offconv_bwd": ("hbm", k4),
        # input part: read goff, w_off and the NHWC grad_x buffer, write grad_x
        # (float32; through the fused ReLU read x, write bf16: the same bytes)
        "k4cl_input": ("hbm", off_b + woff_b + 2 * gx_b),
        # weight part: read x (NHWC) and goff, write the chunk partials
        "k4cl_weight": ("hbm", x_b + off_b + k4cl_chunks * p.n_off * (kdim + 1) * 4),
        "k4cl_reduce": ("hbm", (k4cl_chunks + 1) * p.n_off * (kdim + 1) * 4),
        # per-image grad_w_off partials of the tensor-core K4, summed
        "gw_off_reduce": ("hbm", (p.n + 1) * p.n_off * kdim * 4),
        # ReLU between stacked layers: read y, write the next input; read the
        # next input and its grad_x (fp32), write grad_y
        "relu_fwd": ("hbm", 2 * p.n * p.c_out * p.ho * p.wo * elt),
        "relu_bwd": ("hbm", p.n * p.c_out * p.ho * p.wo * (2 * elt + 4)),
    }


def kernel_breakdown(p, wl, step, dev, stream, flush, iters=40):
    """Every kernel of the step timed with CUDA events on its stream (the
    library's dc_kernel_timing), eager launches, L2 flushed before each step."""
    import torch

    from deformable_convolution_gb300 import binding as B
    with torch.cuda.stream(stream):
        for _ in range(3):
            flush.fill_(5)
            step()
        torch.cuda.synchronize(dev)
        B.kernel_timing(True)
        for _ in range(iters):
            flush.fill_(9)
            step()
    torch.cuda.synchronize(dev)
    recs = B.kernel_times()
    B.kernel_timing(False)
    tot, cnt = {}, {}
    for name, ms in recs:
        if ms >= 0:
            tot[name] = tot.get(name, 0.0) + ms
            cnt[name] = cnt.get(name, 0) + 1
    costs = kernel_costs(p, wl.outlier_p > 0)
    peaks, src = measured_peaks()
    step_ms = sum(tot[k] / cnt[k] for k in tot)
    out = []
    for name in tot:
        ms = tot[name] / cnt[name]
        bound, amount = costs.get(name, ("hbm", 0.0))
        if bound == "tensor" and p.dtype != 1 and tf32_path(p):
            # float32 problems with 16-byte aligned rows: tcgen05 kind::tf32,
            # three products per multiply (hi*hi + hi*lo + lo*hi)
            achieved = amount / (ms / 1e3) / 1e12
            peak, unit = peaks["bf16_tflops"] * TF32_PER_BF16 / 3, "TFLOP/s"
            peak_src = (f"derived: {src} bf16_tflops (burst) x nominal tf32/bf16 "
                        f"{TF32_PER_BF16:.3f} / 3 products")
        elif bound == "tensor" and p.dtype != 1:
            # other float32 problems run the GEMMs on CUDA cores: FFMA peak of the part
            bound = "alu"
            achieved = amount / (ms / 1e3) / 1e12
            peak, sms, mhz = fp32_alu_tflops(dev)
            unit = "TFLOP/s"
            peak_src = f"derived: {sms} SMs x 128 fp32 lanes x 2 flop x {mhz:.0f} MHz"
        elif bound == "tensor":
            achieved = amount / (ms / 1e3) / 1e12
            # each GEMM launch is timed on its own (tens of microseconds),
            # not as a seconds-long loop: the burst peak applies
            peak, unit = peaks["bf16_tflops"], "TFLOP/s"
            peak_src = f"{src} (bf16_tflops, burst)"
        else:
            achieved = amount / (ms / 1e3) / 1e9
            peak, unit = peaks["hbm_gbs"], "GB/s"
            peak_src = f"{src} (hbm_gbs)"
        out.append({"kernel": name, "ms_per_launch": ms, "share": ms / step_ms, "bound": bound,
                    "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
                    "peak_source": peak_src,
                    ("algorithmic_flops" if bound == "tensor" else "algorithmic_bytes"): amount,
                    "traffic": traffic_for(wl.name, name)})
    out.sort(key=lambda r: -r["ms_per_launch"])
    return out


def k1_bytes(p, has_add):
    """Algorithmic bytes of one K1 launch: read x and w_off once, write the
    deformed map and the fp32 offsets (and read offset_add when given)."""
    elt = 2 if p.dtype == 1 else 4
    P = p.n * p.ho * p.wo
    b = p.n * p.c_in * p.h * p.w * elt + p.n_off * p.c_in * p.kh * p.kw * elt
    b += p.c_in * p.kh * p.kw * P * elt + p.n_off * P * 4
    if has_add:
        b += p.n_off * P * 4
    return b


def k1_roofline(p, t, dev, stream, flush, wl, iters=200):
    """K1 (the fused sampling stage) timed alone: one launch captured in a CUDA
    graph, replayed between L2 flushes, CUDA events on the launching stream."""
    import torch

    from deformable_convolution_gb300 import binding as B
    col = torch.empty(B.col_shape(p), dtype=p.torch_dtype, device=dev)
    off = torch.empty(p.shapes()["offset"], dtype=torch.float32, device=dev)
    ws = B.workspace(p, False, dev)

    def launch():
        B.deform_conv_sample(p, t["x"], t["w_off"], t["b_off"], t["offset_add"], None, col, off,
                             ws=ws)

    with torch.cuda.stream(stream):
        launch()
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        launch()
    with torch.cuda.stream(stream):
        for _ in range(5):
            flush.fill_(3)
            graph.replay()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(iters)]
        torch.cuda.synchronize(dev)
        for a, b in ev:
            flush.fill_(7)
            a.record(stream)
            graph.replay()
            b.record(stream)
    torch.cuda.synchronize(dev)
    ms = sum(a.elapsed_time(b) for a, b in ev) / iters
    nbytes = k1_bytes(p, t["offset_add"] is not None)
    peaks, src = measured_peaks()
    achieved = nbytes / (ms / 1e3) / 1e9
    cl = B.col_layout(p) == B.DC_COL_PIXEL_MAJOR
    name = "k1_cl_sample" if cl else "k1_band_sample"
    traffic = traffic_for(wl.name, name)
    what = ("cl_prep (x to NHWC, weight layouts) + k1_cl_sample (offset conv + bilinear "
            "sampling), one deform_conv_sample call" if cl
            else "k1_band_sample (offset conv + bilinear sampling)")
    return {"kernel": what, "bound": "hbm",
            "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / peaks["hbm_gbs"], "peak_source": f"{src} (hbm_gbs, burst)",
            "traffic": traffic, "algorithmic_bytes": nbytes, "ms_per_launch": ms}


def time_graph(launch, dev, stream, flush, iters):
    """Average device time of `launch` captured in a CUDA graph and replayed
    between L2 flushes (CUDA events on the launching stream)."""
    import torch
    with torch.cuda.stream(stream):
        launch()
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        launch()
    with torch.cuda.stream(stream):
        for _ in range(5):
            flush.fill_(3)
            graph.replay()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(iters)]
        torch.cuda.synchronize(dev)
        for a, b in ev:
            flush.fill_(7)
            a.record(stream)
            graph.replay()
            b.record(stream)
    torch.cuda.synchronize(dev)
    return sum(a.elapsed_time(b) for a, b in ev) / iters


def unfused_ablation(p, t, dev, stream, flush, iters=200):
    """The pages' comparison, on this GPU: the fused stage (offset convolution
    and interpolation in one kernel, offsets kept on chip) against the unfused
    pipeline (offset convolution -> offsets in HBM -> interpolation), each
    timed alone between L2 flushes.  Arithmetic intensity = the stage's flops
    (offset convolution + 4-corner blends) / its algorithmic HBM bytes."""
    import torch

    from deformable_convolution_gb300 import binding as B
    s = p.shapes()
    col = torch.empty(B.col_shape(p), dtype=p.torch_dtype, device=dev)
    off = torch.empty(s["offset"], dtype=torch.float32, device=dev)
    ws = B.workspace(p, False, dev)
    add = t["offset_add"]
    fused = time_graph(lambda: B.deform_conv_sample(p, t["x"], t["w_off"], t["b_off"], add, None,
                                                    col, off, ws=ws), dev, stream, flush, iters)
    k_off = time_graph(lambda: B.deform_conv_offsets(p, t["x"], t["w_off"], t["b_off"], add, off,
                                                     ws=ws), dev, stream, flush, iters)
    k_smp = time_graph(lambda: B.deform_conv_sample(p, t["x"], None, None, None, off, col, ws=ws),
                       dev, stream, flush, iters)
    elt = 2 if p.dtype == 1 else 4
    P = p.n * p.ho * p.wo
    kdim = p.c_in * p.kh * p.kw
    x_b, w_b = p.n * p.c_in * p.h * p.w * elt, p.n_off * kdim * elt
    off_b, col_b = p.n_off * P * 4, kdim * P * elt
    add_b = off_b if add is not None else 0
    flops = 2.0 * P * kdim * p.n_off + 8.0 * P * kdim  # offset conv + blends
    bytes_fused = x_b + w_b + add_b + col_b + off_b
    bytes_unfused = (x_b + w_b + add_b + off_b) + (x_b + off_b + col_b)
    return {"fused_us": fused * 1e3, "unfused_offsets_us": k_off * 1e3,
            "unfused_sampler_us": k_smp * 1e3, "unfused_us": (k_off + k_smp) * 1e3,
            "speedup": (k_off + k_smp) / fused,
            "ai_fused": flops / bytes_fused, "ai_unfused": flops / bytes_unfused,
            "note": "fused: one K1 launch; unfused: offsets-only K1 then the sampler reading "
                    "offsets from HBM; both write the offsets and the deformed map"}


def sampled_gemm_ablation(p, t, dev, stream, flush, iters=200):
    """The forward pass two ways, each timed alone between L2 flushes: the
    library's path (fused offset convolution + interpolation writing the
    deformed map, then the tensor-core GEMM reading it) against the sampled-
    operand GEMM (offsets-only K1, then one kernel that samples each map tile
    into shared memory as the GEMM's B operand: the map never reaches memory).
    The explainer page argues for the first (the GEMM stays a separate, tuned
    kernel); the second removes the map's write and read."""
    import torch

    from deformable_convolution_gb300 import binding as B
    if p.dtype != 1:
        return None
    s = p.shapes()
    y = torch.empty(s["y"], dtype=p.torch_dtype, device=dev)
    off = torch.empty(s["offset"], dtype=torch.float32, device=dev)
    ws = B.workspace(p, False, dev)
    add = t["offset_add"]
    two = time_graph(lambda: B.deform_conv_fwd(p, t["x"], t["w_off"], t["b_off"], t["w"], add, y,
                                               off, None, ws), dev, stream, flush, iters)
    one = time_graph(lambda: B.deform_conv_fwd_sampled_gemm(p, t["x"], t["w_off"], t["b_off"],
                                                            t["w"], add, y, off),
                     dev, stream, flush, iters)
    P = p.n * p.ho * p.wo
    kdim = p.c_in * p.kh * p.kw
    col_b = kdim * P * 2
    return {"map_in_hbm_us": two * 1e3, "sampled_operand_us": one * 1e3, "speedup": two / one,
            "map_bytes_avoided": 2 * col_b,
            "note": "map_in_hbm: K1 (offset conv + sampling, map to memory) + tensor-core GEMM; "
                    "sampled_operand: offsets-only K1 + one GEMM whose sampling warps write each "
                    "64x64 map tile into its shared-memory B operand"}


def margin_report(p, t, dev):
    """Slow-path fraction of the timed configuration's margin, measured by the
    forward's own counter, and the margin the offset statistics suggest for at
    most 1 % slow taps."""
    import torch

    from deformable_convolution_gb300 import binding as B
    cnt = torch.zeros(1, dtype=torch.int64, device=dev)
    y, off = B.forward(p, t["x"], t["w_off"], t["b_off"], t["w"], t["offset_add"],
                       slowpath_count=cnt)
    hist = torch.zeros(B.MARGIN_BINS, dtype=torch.int64, device=dev)
    B.deform_conv_margin_histogram(p, off, hist)
    torch.cuda.synchronize(dev)
    h = [int(v) for v in hist.cpu().tolist()]
    total = sum(h)
    return {"halo_margin": p.halo_margin if p.halo_margin >= 0 else 3,
            "slow_fraction": int(cnt.item()) / max(1, total),
            "suggested_for_1pct": B.dc_suggest_margin(p, h, 0.01, True), "taps": total}


def _packed(specs, device, pinned):
    """One buffer holding several tensors (256-byte aligned views), so that a
    group of them moves between host and device in one copy."""
    import torch
    at, place = 0, {}
    for name, shape, dt in specs:
        nbytes = math.prod(shape) * torch.empty((), dtype=dt).element_size()
        at = (at + 255) // 256 * 256
        place[name] = (at, nbytes, shape, dt)
        at += nbytes
    buf = torch.empty(max(at, 1), dtype=torch.uint8, device=device, pin_memory=pinned)
    views = {n: buf[o:o + nb].view(dt).view(shape) for n, (o, nb, shape, dt) in place.items()}
    return buf, views


def _timed_runs(step, stream, dev, iters, runs=3):
    """ms per step of `iters` steps timed with CUDA events on `stream`, three
    times: the median, and every run (the host link is shared with other work
    on the machine, so a single run can catch a slow moment)."""
    import statistics

    import torch
    out = []
    for _ in range(runs):
        with torch.cuda.stream(stream):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(iters):
                step()
            b.record(stream)
        torch.cuda.synchronize(dev)
        out.append(a.elapsed_time(b) / iters)
    return statistics.median(out), out


def e2e_stack(job, dev, stream, iters=10):
    """The stack's training step through the ABI with host buffers: every step
    uploads layer 0's input, every layer's weights and grad_y from pinned host
    memory and reads back the last layer's output, grad_x of layer 0 and every
    layer's weight gradients.  One CUDA graph per step over two streams:
    layer 0's input and weights go up first on the compute stream, alone, so
    the forward starts as early as the link allows; then, on a copy stream
    while layer 0's forward runs, the other layers' weights (the next
    forward waits for them) and grad_y (the backward waits for it); the
    output comes back on the copy stream while the backward runs, and each
    layer's weight gradients come back on it as soon as that layer's
    backward is done.  Each group of tensors is one packed buffer on both
    sides, so each group is one copy."""
    import torch

    from deformable_convolution_gb300 import binding as B
    st, p, L = job.stack, job.p, job.wl.layers
    s = p.shapes()
    f32, dt = torch.float32, p.torch_dtype
    x0h, layers_h, gyh = job.host
    groups = {"in0": [("x", tuple(s["x"]), dt)] + [(f"{k}0", tuple(v.shape), v.dtype)
                                                   for k, v in layers_h[0].items()],
              "wrest": [(f"{k}{l}", tuple(v.shape), v.dtype) for l in range(1, L)
                        for k, v in layers_h[l].items()],
              "gyin": [("gy", tuple(s["y"]), dt)],
              "yout": [("y", tuple(s["y"]), dt)], "gx": [("gx", tuple(s["x"]), f32)]}
    for l in range(L):
        groups[f"g{l}"] = [("grad_w_off", tuple(s["w_off"]), f32),
                           ("grad_b_off", tuple(s["b_off"]), f32), ("grad_w", tuple(s["w"]), f32)]
    hbuf, dbuf, hv, dv = {}, {}, {}, {}
    for gname, specs in groups.items():
        hbuf[gname], hv[gname] = _packed(specs, "cpu", True)
        dbuf[gname], dv[gname] = _packed(specs, dev, False)
    hv["in0"]["x"].copy_(x0h)
    hv["gyin"]["gy"].copy_(gyh)
    for l in range(L):
        for k, v in layers_h[l].items():
            hv["in0" if l == 0 else "wrest"][f"{k}{l}"].copy_(v)
    params = [{k: dv["in0" if l == 0 else "wrest"][f"{k}{l}"] for k in ("w_off", "b_off", "w")}
              for l in range(L)]
    saved = st.params, st.grads
    st.params = params
    st.grads = [dv[f"g{l}"] for l in range(L)]
    up = ("in0", "wrest", "gyin")
    h2d = sum(b.numel() for g, b in hbuf.items() if g in up)
    d2h = sum(b.numel() for g, b in hbuf.items() if g not in up)
    cs = torch.cuda.Stream(device=dev)
    e_in0, e_wrest, e_gy = torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event()
    e_fwd = torch.cuda.Event()
    e_layer = [torch.cuda.Event() for _ in range(L)]
    x_dev, gy_dev = dv["in0"]["x"], dv["gyin"]["gy"]

    def one():
        cur = torch.cuda.current_stream(dev)
        dbuf["in0"].copy_(hbuf["in0"], non_blocking=True)
        e_in0.record(cur)
        cs.wait_event(e_in0)
        with torch.cuda.stream(cs):
            if L > 1:
                dbuf["wrest"].copy_(hbuf["wrest"], non_blocking=True)
                e_wrest.record(cs)
            dbuf["gyin"].copy_(hbuf["gyin"], non_blocking=True)
            e_gy.record(cs)
        st.x[0] = x_dev
        q = st.params[0]
        # layers below the last write relu(y) into the next layer's input (fused)
        B.deform_conv_fwd(st.p_relu if L > 1 else p, x_dev, q["w_off"], q["b_off"], q["w"], None,
                          st.x[1] if L > 1 else st.y[0], st.off[0], None, st.ws[0])
        if L > 1:
            cur.wait_event(e_wrest)
        for l in range(1, L):
            q, last = st.params[l], l + 1 == L
            B.deform_conv_fwd(p if last else st.p_relu, st.x[l], q["w_off"], q["b_off"], q["w"], None,
                              st.y[l] if last else st.x[l + 1], st.off[l], None, st.ws[l])
        e_fwd.record(cur)
        cs.wait_event(e_fwd)
        with torch.cuda.stream(cs):
            # the output straight into its pinned host view (the backward
            # reads the forward's workspace, not y)
            hv["yout"]["y"].copy_(st.y[-1], non_blocking=True)
        cur.wait_event(e_gy)
        st.gy[-1] = gy_dev
        for l in reversed(range(L)):
            st.backward_layer(l)  # layer l - 1's grad_y through the ReLU, fused
            e_layer[l].record(cur)
            cs.wait_event(e_layer[l])
            with torch.cuda.stream(cs):
                hbuf[f"g{l}"].copy_(dbuf[f"g{l}"], non_blocking=True)
        # one tensor: straight into its pinned host view, no packing copy
        hv["gx"]["gx"].copy_(st.gx[0], non_blocking=True)
        cur.wait_stream(cs)

    with torch.cuda.stream(stream):
        for _ in range(2):
            one()
    torch.cuda.synchronize(dev)
    step, how = one, "CUDA graph per step"
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            one()
        torch.cuda.synchronize(dev)
        step = graph.replay
    except RuntimeError as e:  # capture refused: the same two-stream step, launched eagerly
        torch.cuda.synchronize(dev)
        how = f"eager launches (graph capture failed: {str(e).splitlines()[0][:120]})"
    with torch.cuda.stream(stream):
        for _ in range(2):
            step()
        torch.cuda.synchronize(dev)
    ms, runs = _timed_runs(step, stream, dev, iters)
    # the read-back is complete: the host copies equal the device buffers
    assert torch.equal(hv["yout"]["y"], st.y[-1].cpu()), "e2e read-back mismatch"
    assert torch.equal(hv["g0"]["grad_w"], dv["g0"]["grad_w"].cpu()), "e2e read-back mismatch"
    st.params, st.grads = saved
    return {"value": job.flops_step / (ms / 1e3) / 1e9, "unit": "GFLOP/s", "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "runs_ms_per_step": runs, "timing": f"median of {len(runs)} runs of {iters} steps",
            "method": how + ": layer 0's input and weights up on the compute stream first, then "
                            "the other layers' weights and grad_y up on a copy stream during "
                            "layer 0's forward; the output, each layer's weight gradients (as soon "
                            "as its backward is done) and grad_x of layer 0 back, packed groups"}


def e2e(p, d, dev, stream, flops_step, iters=20):
    """Same metric through the ABI with host buffers: every step copies its
    inputs from pinned host memory and reads all outputs back.  The step is
    one CUDA graph over two streams: grad_y's upload and the read-back of the
    forward's outputs (y, offsets) run on a copy stream beside the compute,
    the forward's inputs go up before the forward and the gradients come
    back after the backward.  Each group of tensors lives in one packed
    buffer on both sides, so each group is one copy.  Each replay is a whole
    step: every copy of every step happens inside the timed region."""
    import torch

    from deformable_convolution_gb300 import binding as B
    s = p.shapes()
    f32, dt = torch.float32, p.torch_dtype
    fwd_in = [(k, tuple(v.shape), v.dtype) for k, v in d.items() if v is not None and k != "grad_y"]
    groups = {
        "in": fwd_in,
        "gy": [("grad_y", tuple(d["grad_y"].shape), d["grad_y"].dtype)],
        "fwd_out": [("y", tuple(s["y"]), dt), ("off", tuple(s["offset"]), f32)],
        "bwd_out": [("gx", tuple(s["x"]), f32), ("gwo", tuple(s["w_off"]), f32),
                    ("gbo", tuple(s["b_off"]), f32), ("gw", tuple(s["w"]), f32),
                    ("goff", tuple(s["offset"]), f32)],
    }
    hbuf, dbuf, hv, dv = {}, {}, {}, {}
    for gname, specs in groups.items():
        hbuf[gname], h = _packed(specs, "cpu", True)
        dbuf[gname], g = _packed(specs, dev, False)
        hv.update(h)
        dv.update(g)
    for k, v in d.items():
        if v is not None:
            hv[k].copy_(v)
    devt = {k: (dv[k] if v is not None else None) for k, v in d.items()}
    outs = {k: dv[k] for k in ("y", "off", "gx", "gwo", "gbo", "gw", "goff")}
    ws = B.workspace(p, True, dev)
    h2d = sum(v.numel() * v.element_size() for v in d.values() if v is not None)
    d2h = sum(v.numel() * v.element_size() for v in outs.values())
    cs = torch.cuda.Stream(device=dev)
    e_gy = torch.cuda.Event()
    e_fwd = torch.cuda.Event()

    def one():
        # fork: the copy stream uploads grad_y while the forward runs
        cs.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(cs):
            dbuf["gy"].copy_(hbuf["gy"], non_blocking=True)
            e_gy.record(cs)
        dbuf["in"].copy_(hbuf["in"], non_blocking=True)
        B.deform_conv_fwd(p, devt["x"], devt["w_off"], devt["b_off"], devt["w"],
                          devt["offset_add"], outs["y"], outs["off"], None, ws)
        e_fwd.record(torch.cuda.current_stream(dev))
        # the forward's outputs come back while the backward runs (both only read them)
        cs.wait_event(e_fwd)
        with torch.cuda.stream(cs):
            hbuf["fwd_out"].copy_(dbuf["fwd_out"], non_blocking=True)
        torch.cuda.current_stream(dev).wait_event(e_gy)
        B.deform_conv_bwd(p, devt["x"], devt["w_off"], devt["w"], outs["off"], devt["grad_y"],
                          outs["gx"], outs["gwo"], outs["gbo"], outs["gw"], outs["goff"], ws,
                          after_fwd=True)
        hbuf["bwd_out"].copy_(dbuf["bwd_out"], non_blocking=True)
        # join
        torch.cuda.current_stream(dev).wait_stream(cs)

    with torch.cuda.stream(stream):
        for _ in range(3):
            one()
    torch.cuda.synchronize(dev)
    step = one
    how = "CUDA graph per step"
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            one()
        torch.cuda.synchronize(dev)
        step = graph.replay
    except RuntimeError as e:  # capture refused: the same two-stream step, launched eagerly
        torch.cuda.synchronize(dev)
        how = f"eager launches (graph capture failed: {str(e).splitlines()[0][:120]})"
    with torch.cuda.stream(stream):
        for _ in range(3):
            step()
        torch.cuda.synchronize(dev)
    ms, runs = _timed_runs(step, stream, dev, iters)
    # the read-back is complete: the last step's y and grad_x on the host equal
    # the device copies
    assert torch.equal(hv["y"], outs["y"].cpu()), "e2e read-back mismatch"
    assert torch.equal(hv["gx"], outs["gx"].cpu()), "e2e read-back mismatch"
    return {"value": flops_step / (ms / 1e3) / 1e9, "unit": "GFLOP/s", "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "runs_ms_per_step": runs, "timing": f"median of {len(runs)} runs of {iters} steps",
            "method": how + ": forward inputs up (one packed copy), forward, backward, gradients "
                            "back (one packed copy) on the compute stream; grad_y up and y/offsets "
                            "back on a copy stream beside it"}


if __name__ == "__main__":
    main()
