#!/usr/bin/env python
"""Benchmark of the attention forward path on the ANDREA-120M-shaped SSSL workload.

One step = one forward call per layer of the 12-layer stack (B=32, H=12, T=1024, D=64; windows
512, 512, 512, 1024 repeated three times), each layer with its own seeded inputs. The metric is
TFLOP/s over unmasked score entries only (4*D FLOPs per entry), summed over the layers.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0). `--impl reference` times the float64 CPU oracle on the host
cores on a bounded sample of the same workload (the reference arm of this comparison).
Multi-GPU (torchrun): every rank runs its own replica of the workload (weak scaling, no
collective on the data path); the timed region is bracketed by barriers and the slowest rank's
time is reported.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from sliding_window_attention_04_b300 import configs  # noqa: E402
from sliding_window_attention_04_b300.inputs import layer_seed, make_qkv  # noqa: E402

METRIC = "attention fwd TFLOP/s (unmasked FLOPs, SSSL mix) and % of B300 dense-BF16 peak"
WORKLOAD_INDEX = 2  # ANDREA-120M shape
FALLBACK_PEAK_TFLOPS = 1800.0


FWD_SOURCES = ("attn_api.cu", "attn_common.cuh", "attn_fwd_simple.cuh", "attn_fwd_ws.cuh", "ptx.cuh")


def kernel_hash() -> str:
    """Hash of the forward's CUDA sources: ties committed ncu counters to the kernel they were taken on."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sliding_window_attention_04_b300", "csrc")
    for name in FWD_SOURCES:
        h.update(name.encode())
        h.update(open(os.path.join(csrc, name), "rb").read())
    return h.hexdigest()[:16]


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0.0)), "measured"
    return FALLBACK_PEAK_TFLOPS, 1400.0, "fallback"


def traffic_per_launch():
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this kernel."""
    p = os.path.join(ROOT, "profiles", "attn_fwd_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    if d.get("kernel_hash") != kernel_hash():
        return None
    return d.get("dram_bytes_per_launch")


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons in the background during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def wait_ready(self, timeout: float = 10.0):
        """Block until the sampler has printed its first sample, so that its start-up (which can stall the
        GPU for milliseconds) lies before the timed region, then let one more interval pass."""
        t0 = time.time()
        while self.proc is not None and not self.lines and time.time() - t0 < timeout:
            time.sleep(0.02)
        time.sleep(0.25)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, flag in zip(names, parts[5:9]):
                if flag.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def build_inputs(w, device):
    """Per-layer seeded inputs: pinned host copies (for the end-to-end leg) and device copies."""
    host, dev = [], []
    for li, _ in enumerate(w.layers):
        q, k, v = make_qkv(w.B, w.T, w.H, w.D, seed=layer_seed(w.index, li))
        hq = [t.pin_memory() for t in (q, k, v)]
        host.append(hq)
        dev.append([t.to(device, non_blocking=True) for t in hq])
    torch.cuda.synchronize(device)
    return host, dev


def oracle_sample_rows(w, budget_s: float) -> int:
    """How many batch rows of every layer the float64 oracle can do in about `budget_s` seconds:
    calibrated on up to sixteen batch rows of the first layer (a second, warm call; fewer rows keep too
    few of the oracle's threads busy and overestimate the time per row), scaled to every layer by its
    unmasked score entries."""
    import oracle

    nc = min(w.B, 16)
    q, k, v = make_qkv(nc, w.T, w.H, w.D, seed=layer_seed(w.index, 0))
    w0 = w.layers[0].window
    oracle.attn_fwd(q, k, v, window=w0, causal=True, rope_base=w.rope_base, eps=w.eps)  # warm-up
    t0 = time.perf_counter()
    oracle.attn_fwd(q, k, v, window=w0, causal=True, rope_base=w.rope_base, eps=w.eps)
    per_row = (time.perf_counter() - t0) / nc
    weight = sum(configs.n_unmasked(w.T, l.window) for l in w.layers) / configs.n_unmasked(w.T, w0)
    return int(max(1, min(w.B, budget_s / max(per_row * weight, 1e-9))))


L2_BYTES = 126 * 2 ** 20


def needs_flush(w) -> bool:
    """True when a step's inputs (each layer its own q, k, v) are less than twice the L2 capacity: the
    timed steps are then separated by an L2 flush instead of relying on the step's own size."""
    return len(w.layers) * 3 * 2 * w.B * w.T * w.H * w.D < 2 * L2_BYTES


def config_dict(w):
    step_gb = len(w.layers) * 3 * 2 * w.B * w.T * w.H * w.D / 1e9
    if needs_flush(w):
        l2 = (f"flushed: a step reads {step_gb * 1e3:.1f} MB of inputs, less than twice the 126 MiB L2, so "
              f"each timed step is its own CUDA-graph replay between CUDA events, preceded (outside the "
              f"events) by a {2 * L2_BYTES >> 20} MiB write that evicts L2")
        launch = "each timed step one CUDA-graph replay of the step (captured, replayed once untimed)"
    else:
        l2 = (f"no flush: a step reads {step_gb:.2f} GB of inputs, each layer its own, more than twice the "
              f"126 MiB L2")
        launch = "the K timed steps as one CUDA graph (captured, replayed once untimed, then once timed)"
    return {"workload": w.name, "B": w.B, "H": w.H, "T": w.T, "D": w.D,
            "layers": f"{len(w.layers)} layers, windows " + ",".join(str(l.window) for l in w.layers),
            "qk_norm_eps": w.eps, "rope_base": w.rope_base, "mask": "causal + sliding window (W=T/2 on S)",
            "l2": l2,
            "launch": launch,
            "parallelism": "replicas (one full workload per GPU)"}


def max_over_ranks(values, dist=None, device=None):
    """Per-rank timings -> their maximum over all ranks (the slowest rank sets the job's time)."""
    if dist is None:
        return [float(x) for x in values]
    t = torch.tensor([float(x) for x in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def whole_job_tflops(flops_per_rank_step, steps, world, elapsed_ms):
    """Whole-job throughput: every rank runs its own replica (weak scaling), so the job does world
    times the work of one rank in the max-over-ranks time."""
    return flops_per_rank_step * steps * world / (elapsed_ms / 1e3) / 1e12


def run_reference(args, w, rank):
    """The reference arm: the float64 oracle on the host cores, a bounded sample per step."""
    import oracle

    if rank != 0:
        return
    cores = oracle.num_threads()
    per_step_budget = max(0.05, 120.0 / max(1, args.steps + args.warmup))
    # sample unit: one batch row (all 12 heads, full T) of one layer, cycling through the layers
    inputs = []
    for li, layer in enumerate(w.layers):
        q, k, v = make_qkv(w.B, w.T, w.H, w.D, seed=layer_seed(w.index, li))
        inputs.append((q[:1].clone(), k[:1].clone(), v[:1].clone(), layer))
    q, k, v, layer = inputs[0]
    oracle.attn_fwd(q, k, v, window=layer.window, causal=True, rope_base=w.rope_base, eps=w.eps)
    t0 = time.perf_counter()
    oracle.attn_fwd(q, k, v, window=layer.window, causal=True, rope_base=w.rope_base, eps=w.eps)
    unit_s = time.perf_counter() - t0
    n_units = max(1, int(per_step_budget / max(unit_s, 1e-9)))
    total_flops, total_s = 0, 0.0
    for step in range(args.warmup + args.steps):
        flops = 0
        t0 = time.perf_counter()
        for u in range(n_units):
            q, k, v, layer = inputs[(step * n_units + u) % len(inputs)]
            oracle.attn_fwd(q, k, v, window=layer.window, causal=layer.causal, rope_base=w.rope_base, eps=w.eps)
            flops += configs.attn_flops(1, w.H, w.T, w.D, layer.window, layer.causal)
        dt = time.perf_counter() - t0
        if step >= args.warmup:
            total_flops += flops
            total_s += dt
    value = total_flops / total_s / 1e12
    sample = (f"{n_units} x (one batch row, all {w.H} heads, T={w.T}) per step, cycling through the "
              f"{len(w.layers)} layers of the workload")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_s / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(w),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


BWD_METRIC = "attention bwd TFLOP/s (2.5x the unmasked forward FLOPs, SSSL mix) and % of B300 dense-BF16 peak"


def run_backward(args, w, rank, local_rank, world):
    """The backward of every layer (dq, dk, dv from the forward's out, lse and a seeded dout), timed
    like the forward: the K steps as CUDA-graph replays with device-resident inputs."""
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=device)
    from sliding_window_attention_04_b300 import attn

    attn.attn_init(local_rank)
    host, dev = build_inputs(w, device)
    douts, outs, lses, grads = [], [], [], []
    for li, layer in enumerate(w.layers):
        douts.append(make_qkv(w.B, w.T, w.H, w.D, seed=layer_seed(w.index, li) + 7919)[2].to(device))
        o, l = attn.attn_fwd(dev[li][0], dev[li][1], dev[li][2], window=layer.window, causal=layer.causal,
                             rope_base=w.rope_base, eps=w.eps)
        outs.append(o)
        lses.append(l)
        grads.append(tuple(torch.empty(dev[li][0].shape, dtype=torch.float32, device=device) for _ in range(3)))
    ws = torch.empty(attn.attn_bwd_workspace_bytes(w.B, w.H, w.H, w.T, w.D), dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    step_flops = 2.5 * sum(configs.attn_flops(w.B, w.H, w.T, w.D, l.window, l.causal) for l in w.layers)

    def step(strm):
        for li, layer in enumerate(w.layers):
            dq, dk, dv = grads[li]
            attn.attn_bwd(dev[li][0], dev[li][1], dev[li][2], outs[li], lses[li], douts[li], window=layer.window,
                          causal=layer.causal, rope_base=w.rope_base, eps=w.eps, workspace=ws, dq=dq, dk=dk, dv=dv,
                          stream=strm)

    for _ in range(args.warmup):
        step(stream)
    torch.cuda.synchronize(device)
    st = attn.attn_device_status()
    if st != 0:
        raise SystemExit(f"device status after warm-up: {attn.status_string(st)}")
    # inputs of a layer: q, k, v, out, dout (5 x B T H D bf16); the workspace is rewritten every call
    step_in_bytes = len(w.layers) * 5 * 2 * w.B * w.T * w.H * w.D
    flush = step_in_bytes < 2 * L2_BYTES
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(device)
    cap.wait_stream(stream)
    with torch.cuda.graph(graph, stream=cap):
        for _ in range(1 if flush else args.steps):
            step(cap)
    stream.wait_stream(cap)
    graph.replay()
    scrub = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=device) if flush else None
    torch.cuda.synchronize(device)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps if flush else 1)]
    sampler = ClockSampler(local_rank)
    sampler.start()
    sampler.wait_ready()
    if dist:
        dist.barrier()
    torch.cuda.synchronize(device)
    for e0, e1 in evs:
        if flush:
            scrub.fill_(1)
        e0.record(stream)
        graph.replay()
        e1.record(stream)
    torch.cuda.synchronize(device)
    if dist:
        dist.barrier()
    clocks = sampler.stop()
    elapsed_ms = sum(e0.elapsed_time(e1) for e0, e1 in evs)
    st = attn.attn_device_status()
    if st != 0:
        raise SystemExit(f"device status after the timed region: {attn.status_string(st)}")
    (elapsed_ms,) = max_over_ranks([elapsed_ms], dist, device)
    value = whole_job_tflops(step_flops, args.steps, world, elapsed_ms)
    peak, peak_sustained, peak_kind = peaks()
    if rank == 0:
        cfg = config_dict(w)
        cfg["pass"] = "backward: prologue pass, tcgen05 main kernel, finalize pass per layer"
        cfg["l2"] = (f"flushed between steps ({step_in_bytes / 1e6:.0f} MB of inputs per step)" if flush else
                     f"no flush: a step reads {step_in_bytes / 1e9:.2f} GB of inputs, each layer its own")
        line = {
            "metric": BWD_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": cfg,
            "pct_of_peak": value / world / peak * 100.0,
            "roofline": {"bound": "tensor", "achieved": value / world, "peak": peak, "unit": "TFLOP/s",
                         "frac": value / world / peak, "traffic": None,
                         "peak_kind": f"{peak_kind} dense bf16 burst (sustained {peak_sustained})",
                         "kernel": "attn_bwd (three launches per layer)",
                         "achieved_basis": "2.5 x unmasked forward FLOPs per layer / the layer's three launches"},
            "gpu_launches": 3 * args.steps * len(w.layers),
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


POLAR_METRIC = ("Polar Express effective TFLOP/s (the listing's 5 steps in full, Muon matrix groups of the ANDREA-120M "
                "shape) and % of B300 dense-BF16 peak")


def run_polar(args, rank, local_rank, world):
    """Muon's orthogonalisation of one optimiser step on the ANDREA-120M shape (12 layers, n_embd 768):
    the attention projections (48 matrices of 768 x 768), the MLP input (12 x 3072 x 768, tall) and output
    (12 x 768 x 3072, wide) matrices, each group one batched polar_express call (5 steps), bf16."""
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=device)
    from sliding_window_attention_04_b300 import attn, polar

    attn.attn_init(local_rank)
    groups = [(48, 768, 768), (12, 3072, 768), (12, 768, 3072)]
    bufs = []
    flops = 0
    for gi, (bt, m, n) in enumerate(groups):
        g = torch.randn(bt, m, n, generator=torch.Generator().manual_seed(555 + gi)).to(torch.bfloat16).to(device)
        out = torch.empty_like(g)
        ws = torch.empty(polar.workspace_bytes(bt, m, n), dtype=torch.uint8, device=device)
        bufs.append((g, out, ws))
        s, l = min(m, n), max(m, n)
        flops += bt * 5 * (4 * s * s * l + 2 * s ** 3)
    # what the tensor cores execute: the symmetric products A and B only on and above the diagonal
    executed = sum(5 * polar.step_flops(bt, m, n) for bt, m, n in groups)
    if not executed > 0:
        raise SystemExit("pe_step_flops returned no count")
    stream = torch.cuda.current_stream(device)

    def step(strm):
        for g, out, ws in bufs:
            polar.polar_express(g, out=out, workspace=ws, stream=strm)

    for _ in range(args.warmup):
        step(stream)
    torch.cuda.synchronize(device)
    if attn.attn_device_status() != 0:
        raise SystemExit("device status after warm-up")
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(device)
    cap.wait_stream(stream)
    with torch.cuda.graph(graph, stream=cap):
        for _ in range(args.steps):
            step(cap)
    stream.wait_stream(cap)
    graph.replay()
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local_rank)
    sampler.start()
    sampler.wait_ready()
    if dist:
        dist.barrier()
    torch.cuda.synchronize(device)
    e0.record(stream)
    graph.replay()
    e1.record(stream)
    torch.cuda.synchronize(device)
    if dist:
        dist.barrier()
    clocks = sampler.stop()
    elapsed_ms = e0.elapsed_time(e1)
    if attn.attn_device_status() != 0:
        raise SystemExit("device status after the timed region")
    (elapsed_ms,) = max_over_ranks([elapsed_ms], dist, device)
    value = whole_job_tflops(flops, args.steps, world, elapsed_ms)
    achieved = whole_job_tflops(executed, args.steps, world, elapsed_ms) / world
    peak, peak_sustained, peak_kind = peaks()
    n_launch = args.steps * sum(2 + 5 * 3 for _ in groups)  # two normalisation passes, three GEMMs a step
    if rank == 0:
        line = {
            "metric": POLAR_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "Muon groups of the ANDREA-120M shape: 48 x 768x768, 12 x 3072x768, "
                                   "12 x 768x3072, 5 Polar Express steps each",
                       "flops": "value: the listing's count, 4 s^2 l + 2 s^3 per matrix and step (s, l = min, max "
                                "of its sides); roofline: the FLOPs executed (pe_step_flops: A and B, being "
                                "symmetric, only on and above the diagonal)",
                       "executed_gflop_per_step": executed / 1e9, "listing_gflop_per_step": flops / 1e9,
                       "l2": "no flush: a step reads 141 MB of matrices plus their products",
                       "launch": "the K timed steps as one CUDA graph (captured, replayed once untimed, then timed)"},
            "pct_of_peak": achieved / peak * 100.0,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "traffic": None,
                         "peak_kind": f"{peak_kind} dense bf16 burst (sustained {peak_sustained})",
                         "kernel": "gemm_kernel (three per step; achieved over the whole step, normalisation "
                                   "passes and gaps included)"},
            "gpu_launches": n_launch,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--cpu-budget-s", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=0,
                    help="run only the first N layers of the workload (profiling captures); 0 = all")
    ap.add_argument("--workload", default="",
                    help="another workload by name prefix (extra measurements and captures; the bench "
                         "line is the ANDREA-120M workload)")
    ap.add_argument("--pass", dest="which", choices=["fwd", "bwd", "fwd_ve", "polar"], default="fwd",
                    help="bwd: time attn_bwd (dq, dk, dv from out, lse, dout) on the same layers instead of "
                         "the forward; fwd_ve: the forward with the value-embedding gate on every layer "
                         "(attn_fwd_ve); extra measurements, the bench line is the forward")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    w = configs.by_name(args.workload) if args.workload else configs.workloads()[WORKLOAD_INDEX]
    if args.layers > 0:
        import dataclasses

        w = dataclasses.replace(w, layers=list(w.layers[:args.layers]))

    if args.impl == "reference":
        run_reference(args, w, rank)
        return

    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.which == "bwd":
        run_backward(args, w, rank, local_rank, world)
        return
    if args.which == "polar":
        run_polar(args, rank, local_rank, world)
        return
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=device)

    from sliding_window_attention_04_b300 import attn

    attn.attn_init(local_rank)
    host, dev = build_inputs(w, device)
    outs = [torch.empty_like(d[0]) for d in dev]
    lses = [torch.empty((w.B, w.H, w.T), dtype=torch.float32, device=device) for _ in dev]
    stream = torch.cuda.current_stream(device)
    step_flops = sum(configs.attn_flops(w.B, w.H, w.T, w.D, l.window, l.causal) for l in w.layers)

    gates = None
    if args.which == "fwd_ve":
        # per layer: value embeddings like v, the block input x [B, T, H*D] (the gate reads its first 32
        # channels) and the gate weights [H, 32], all seeded
        gates = []
        for li, _ in enumerate(w.layers):
            gen = torch.Generator().manual_seed(layer_seed(w.index, li) + 104729)
            ve = make_qkv(w.B, w.T, w.H, w.D, seed=layer_seed(w.index, li) + 7907)[2].to(device)
            xg = torch.randn(w.B, w.T, w.H * w.D, generator=gen).to(torch.bfloat16).to(device)
            wg = (torch.randn(w.H, 32, generator=gen) * 0.3).to(torch.bfloat16).to(device)
            gws = torch.empty(attn.attn_fwd_ve_workspace_bytes(w.B, w.H, w.T), dtype=torch.uint8, device=device)
            gates.append((ve, xg, wg, gws))

    def step(strm):
        for li, layer in enumerate(w.layers):
            if gates is None:
                attn.attn_fwd(dev[li][0], dev[li][1], dev[li][2], window=layer.window, causal=layer.causal,
                              rope_base=w.rope_base, eps=w.eps, out=outs[li], lse=lses[li], stream=strm)
            else:
                ve, xg, wg, gws = gates[li]
                attn.attn_fwd_ve(dev[li][0], dev[li][1], dev[li][2], ve, xg, wg, window=layer.window,
                                 causal=layer.causal, rope_base=w.rope_base, eps=w.eps, out=outs[li], lse=lses[li],
                                 workspace=gws, stream=strm)

    for _ in range(args.warmup):
        step(stream)
    torch.cuda.synchronize(device)
    st = attn.attn_device_status()
    if st != 0:
        raise SystemExit(f"device status after warm-up: {attn.status_string(st)}")

    # ---- timed region: K steps, device-resident inputs ----
    # The steps are captured into a CUDA graph, replayed once untimed, then timed: the host's per-call
    # work (argument checks, ticket slot, launch) stays out of the measurement and the kernels run back
    # to back. Large steps: one graph of all K steps, one pair of events around its replay (events
    # recorded inside a graph cannot be timed, so the average launch duration is the replay's time
    # over its launches, inter-kernel gaps included). Small steps: one graph of one step, K replays,
    # each between its own pair of events and after an L2-evicting write outside them.
    flush = needs_flush(w)
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(device)
    cap.wait_stream(stream)
    with torch.cuda.graph(graph, stream=cap):
        for _ in range(1 if flush else args.steps):
            step(cap)
    stream.wait_stream(cap)
    graph.replay()
    scrub = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=device) if flush else None
    torch.cuda.synchronize(device)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps if flush else 1)]
    sampler = ClockSampler(local_rank)
    sampler.start()
    sampler.wait_ready()
    if dist:
        dist.barrier()
    torch.cuda.synchronize(device)
    for e0, e1 in evs:
        if flush:
            scrub.fill_(1)
        e0.record(stream)
        graph.replay()
        e1.record(stream)
    torch.cuda.synchronize(device)
    if dist:
        dist.barrier()
    clocks = sampler.stop()
    elapsed_ms = sum(e0.elapsed_time(e1) for e0, e1 in evs)
    kernel_ms = elapsed_ms  # every launch of the graph is this kernel, back to back
    st = attn.attn_device_status()
    if st != 0:
        raise SystemExit(f"device status after the timed region: {attn.status_string(st)}")
    elapsed_ms, kernel_ms = max_over_ranks([elapsed_ms, kernel_ms], dist, device)

    n_launch = args.steps * len(w.layers) * (2 if gates is not None else 1)
    value = whole_job_tflops(step_flops, args.steps, world, elapsed_ms)
    achieved = step_flops * args.steps / (kernel_ms / 1e3) / 1e12  # per GPU, kernel time only
    peak, peak_sustained, peak_kind = peaks()

    # ---- end to end through the public API: pinned host -> device, compute, device -> host ----
    # Three streams and two device buffer sets, as a caller of the stream-taking API pipelines layers:
    # layer l + 1's inputs copy in while layer l computes and layer l - 1's results copy out (PCIe
    # carries both directions at once). Events order each buffer's reuse.
    h_out = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs]
    h_lse = [torch.empty(l.shape, dtype=l.dtype, pin_memory=True) for l in lses]
    d_in = [[torch.empty_like(dev[0][i]) for i in range(3)] for _ in range(2)]
    d_out = [torch.empty_like(outs[0]) for _ in range(2)]
    d_lse = [torch.empty_like(lses[0]) for _ in range(2)]
    s_in, s_back = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in_ready", "in_free", "out_ready", "out_free")}
    seq = [0]

    def e2e_step():
        for li, layer in enumerate(w.layers):
            b = seq[0] & 1
            first_use = seq[0] < 2
            seq[0] += 1
            if not first_use:
                s_in.wait_event(ev["in_free"][b])
            with torch.cuda.stream(s_in):
                for i in range(3):
                    d_in[b][i].copy_(host[li][i], non_blocking=True)
            ev["in_ready"][b].record(s_in)
            stream.wait_event(ev["in_ready"][b])
            if not first_use:
                stream.wait_event(ev["out_free"][b])
            attn.attn_fwd(d_in[b][0], d_in[b][1], d_in[b][2], window=layer.window, causal=layer.causal,
                          rope_base=w.rope_base, eps=w.eps, out=d_out[b], lse=d_lse[b], stream=stream)
            ev["in_free"][b].record(stream)
            ev["out_ready"][b].record(stream)
            s_back.wait_event(ev["out_ready"][b])
            with torch.cuda.stream(s_back):
                h_out[li].copy_(d_out[b], non_blocking=True)
                h_lse[li].copy_(d_lse[b], non_blocking=True)
            ev["out_free"][b].record(s_back)

    e2e_step()
    torch.cuda.synchronize(device)
    if dist:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_stream(stream)  # the copies start after e0
    for _ in range(args.e2e_steps):
        e2e_step()
    stream.wait_stream(s_back)  # e1 after the last result has reached the host
    stream.wait_stream(s_in)
    e1.record(stream)
    torch.cuda.synchronize(device)
    e2e_ms = e0.elapsed_time(e1)
    (e2e_ms,) = max_over_ranks([e2e_ms], dist, device)
    if dist:
        dist.barrier()
    e2e_value = whole_job_tflops(step_flops, args.e2e_steps, world, e2e_ms)
    h2d = sum(t.numel() * t.element_size() for hl in host for t in hl)
    d2h = sum(t.numel() * t.element_size() for t in h_out + h_lse)

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    cpu = None
    if not args.no_cpu_baseline and world == 1:
        import oracle

        nb = oracle_sample_rows(w, args.cpu_budget_s)
        cores = oracle.num_threads()
        flops = sum(configs.attn_flops(nb, w.H, w.T, w.D, l.window, l.causal) for l in w.layers)
        samples = []  # inputs generated outside the timed part
        for li, layer in enumerate(w.layers):
            q, k, v = make_qkv(w.B, w.T, w.H, w.D, seed=layer_seed(w.index, li))
            samples.append((q[:nb].clone(), k[:nb].clone(), v[:nb].clone(), layer))
        t0 = time.perf_counter()
        for q, k, v, layer in samples:
            oracle.attn_fwd(q, k, v, window=layer.window, causal=layer.causal, rope_base=w.rope_base, eps=w.eps)
        cpu_s = time.perf_counter() - t0
        cpu = {"value": flops / cpu_s / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": f"batch rows 0..{nb - 1} of every layer (all {w.H} heads, T={w.T}); "
                         f"{flops / 1e9:.2f} GFLOP in {cpu_s:.1f} s"}

    cfg = config_dict(w)
    if gates is not None:
        cfg["pass"] = ("forward with the value-embedding gate on every layer (attn_fwd_ve: gate-factor pass + "
                       "attention kernel, two launches per layer); e2e is the plain forward")
    line = {
        "metric": METRIC if gates is None else METRIC + ", value-embedding gate on every layer",
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": cfg,
        "pct_of_peak": value / world / peak * 100.0,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic_per_launch(),
                     "peak_kind": f"{peak_kind} dense bf16 burst (sustained {peak_sustained})",
                     "kernel": "attn_fwd (one launch per layer)",
                     "achieved_basis": "algorithmic unmasked FLOPs per launch / mean launch time (CUDA events "
                                       "around the graph replays of the timed launches, gaps between "
                                       "launches of a replay included)"},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": args.e2e_steps},
        "gpu_launches": n_launch,
        "clocks": clocks,
        "kernel_hash": kernel_hash(),
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
