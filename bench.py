#!/usr/bin/env python
"""Benchmark of the MoE layer forward pass on B300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload moe256] [--impl ours|reference]

A step is one whole forward pass (gate, dispatch, experts, combine, losses) over
one batch of seeded synthetic inputs already resident in HBM, through the
one-call entry point ``moe_forward``: K steps bracketed by CUDA events on the
launching stream give ``ms_per_step`` and the metric, routed tokens per second
(T tokens per step / step time).  A second timed region of K steps runs
``moe_forward_timed`` (the same call with CUDA events at its stage boundaries) for
the per-stage times and the expert FFN's roofline: an event between two kernels
makes the later one wait for the earlier to finish before its setup starts, so
that region is a little slower and is reported beside the first
(``stages_region``).  Multi-GPU (torchrun, one process
per GPU): every rank runs its own batch (weak scaling, data parallel); the
reported time is the max over ranks.

Also reported: an end-to-end number through ``moe_forward`` with pinned host
buffers (copies of x and eps in and of y and the losses out inside the timed
region, double-buffered on copy streams), SM clocks sampled during the timed
region, and the fp64 oracle timed on the host cores over a bounded sample
(``cpu_baseline``).  ``--impl reference`` times only the oracle (the reference
arm).
"""
from __future__ import annotations

import argparse
import dataclasses
import math
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from sparsely_gated_mixture_03_b300 import synthetic as S  # noqa: E402

METRIC = "MoE fwd routed tokens/s; expert-FFN TFLOP/s as % of B300 bf16 peak"
UNIT = "tokens/s"
# DRAM bytes (read + write) of one expert-FFN launch, from an ncu capture of the kernel
# as it now stands, keyed by (workload, kernel); a workload or kernel without a
# capture reports null.
FFN_TRAFFIC = {
    ("moe256", "ffn_pair_tc_kernel"): 1.0564e9,     # 687.0 MB read + 369.3 MB written
    ("moe256", "ffn_swap_tc_kernel"): 1.2013e9,     # tiles sized to the expert's rows
}


def max_over_ranks(value: float, dist, device) -> float:
    """The largest of every rank's `value` (the step time of the slowest rank), or
    `value` itself without a process group.  `device` holds the reduction buffer
    ("cuda" under NCCL, "cpu" under gloo)."""
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        j = json.load(open(p))
        return dict(hbm_gbs=j["hbm_gbs"], bf16_tflops=j["bf16_tflops"],
                    bf16_tflops_sustained=j.get("bf16_tflops_sustained"), source="measured")
    return dict(hbm_gbs=6400.0, bf16_tflops=1800.0, bf16_tflops_sustained=1400.0, source="fallback")


class ClockSampler:
    """nvidia-smi SM clock / throttle-reason samples every 100 ms while running;
    summary() keeps the samples taken inside [t0, t1] (host wall clock)."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0=None, t1=None):
        """Samples inside [t0, t1]; the file is read once and kept for later windows."""
        if getattr(self, "rows", None) is None:
            self.rows = self._read()
        rows = self.rows
        inside = [r for r in rows if t0 is None or (t0 - 0.05 <= r["ts"] <= t1 + 0.05)]
        window = "timed region"
        if not inside and rows:       # a timed region shorter than the sampling period
            mid = 0.5 * (t0 + t1)
            inside = sorted(rows, key=lambda r: abs(r["ts"] - mid))[:2]
            window = "nearest samples to a timed region shorter than 100 ms"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        reasons = set()
        for r in inside:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in inside),
                "sm_max_mhz": max(r["smax"] for r in inside),
                "power_w_max": max(r["power"] for r in inside), "samples": len(inside),
                "window": window, "reasons": sorted(reasons)}

    def _read(self):
        rows = []
        if self.path and os.path.exists(self.path):
            for line in open(self.path):
                f = [x.strip() for x in line.split(",")]
                if len(f) < 10:
                    continue
                try:
                    ts = time.mktime(time.strptime(f[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    ts += float("0." + f[0].split(".")[1]) if "." in f[0] else 0.0
                    rows.append(dict(ts=ts, sm=float(f[2]), smax=float(f[3]), power=float(f[4]),
                                     hw=f[6], hwt=f[7], swt=f[8], swp=f[9]))
                except (ValueError, IndexError):
                    continue
            os.unlink(self.path)
        return rows


def cpu_baseline(shape, inp, budget_s=12.0):
    """The fp64 oracle on the host cores over a bounded sample of the same
    workload: gate + experts + combine for the first S tokens of the batch
    (rows are independent; the batch-level CV^2 of two n-vectors is
    negligible).  S is calibrated so the timed run takes about budget_s."""
    from oracle import moe_oracle as O
    try:
        from threadpoolctl import threadpool_info
        cores = max([i.get("num_threads", 1) for i in threadpool_info()] + [1])
    except Exception:  # noqa: BLE001
        cores = os.cpu_count()
    host = {k: (None if v is None else v.detach().to("cpu", torch.float64).numpy())
            for k, v in inp.items()}

    def run(s):
        rows = np.arange(s)
        t0 = time.perf_counter()
        O.moe_forward_rows(host["x"], host["W_g"], host["W_noise"], host["eps"], host["W_in"],
                           host["W_out"], shape.k, rows, 0.0, host["b_g"])
        return time.perf_counter() - t0

    s = min(256, shape.T)
    t = run(s)
    s = int(min(shape.T, max(s, s * budget_s / max(t, 1e-3))))
    reps, t = 0, 0.0
    while t < budget_s and reps < 100:     # the whole batch is short: repeat it
        t += run(s)
        reps += 1
    return {"value": reps * s / t, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"fp64 oracle gate+experts+combine on the first {s} of {shape.T} tokens "
                      f"of the {shape.name} workload, {reps} time(s) ({t:.1f} s)"}


def reference_arm(args, shape):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    inp = S.make_flat_inputs(shape, seed=1000, device="cpu")
    from oracle import moe_oracle as O
    host = {k: (None if v is None else v.to(torch.float64).numpy()) for k, v in inp.items()}
    per_step = max(64, min(shape.T, 1024))
    rows = np.arange(per_step)

    def step():
        O.moe_forward_rows(host["x"], host["W_g"], host["W_noise"], host["eps"], host["W_in"],
                           host["W_out"], shape.k, rows, 0.0, host["b_g"])
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = per_step / dt
    try:
        from threadpoolctl import threadpool_info
        cores = max([i.get("num_threads", 1) for i in threadpool_info()] + [1])
    except Exception:  # noqa: BLE001
        cores = os.cpu_count()
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": shape.name, "T": shape.T, "d": shape.d,
                                            "n": shape.n, "h": shape.h, "k": shape.k},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{per_step} of {shape.T} tokens per step"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def ffn_flags(args):
    import sparsely_gated_mixture_03_b300 as moe
    f = {"auto": 0, "rows": moe.FLAG_FFN_ROW_TILES, "sized": moe.FLAG_FFN_SIZED_TILES}[args.ffn_tiles]
    return f | (moe.FLAG_SWITCH_GATE if getattr(args, "switch", False) else 0)


def ffn_row_tiles(args, R, n):
    """Whether the expert FFN runs 256-row tiles (the library's default) or tiles
    sized to each expert's rows (asked for with --ffn-tiles sized)."""
    return args.ffn_tiles != "sized"


def ffn_tiles_name(args, R, n):
    return "256-row tiles" if ffn_row_tiles(args, R, n) else "tiles sized to each expert's rows"



def hier_bench(args, shape):
    """The hierarchical layer (128 groups x 128 experts): whole-call time of
    moe_hier_forward per step, on one GPU (a secondary measurement line)."""
    import sparsely_gated_mixture_03_b300 as moe
    torch.cuda.set_device(0)
    inp = S.make_hier_inputs(shape, seed=1000, device="cuda")
    cfg = moe.make_hier_config(shape.T, shape.d, shape.a, shape.b, shape.h, shape.k1, shape.k2,
                               flags=ffn_flags(args))
    ws = moe.alloc_hier_workspace(cfg)
    T, d = shape.T, shape.d
    y = torch.empty((T, d), dtype=torch.float32, device="cuda")
    losses = torch.empty(3, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        moe.moe_hier_forward(cfg, inp["x"], inp["W_g1"], inp["W_noise1"], inp["eps1"],
                             inp["W_g2"], inp["W_noise2"], inp["eps2"], inp["W_in"],
                             inp["W_out"], y, losses, workspace=ws, stream=stream)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert moe.moe_get_device_error() == 0
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clk:
        torch.cuda.synchronize()
        launches0 = moe.moe_launch_counter()
        w0 = time.time()
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        w1 = time.time()
        launches = moe.moe_launch_counter() - launches0
    ms = e0.elapsed_time(e1) / args.steps
    K = shape.k1 * shape.k2
    ffn_flops = 4.0 * T * K * d * shape.h
    line = {"metric": METRIC, "value": T / (ms * 1e-3), "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) inputs and N(0,1/fan_in) weights)",
            "config": {"workload": shape.name, "T": T, "d": d, "a": shape.a, "b": shape.b,
                       "h": shape.h, "k1": shape.k1, "k2": shape.k2,
                       "ffn_tiles": ffn_tiles_name(args, T * K, shape.a * shape.b),
                       "l2": "inputs larger than L2 (expert weights %d GB)"
                             % (2 * shape.a * shape.b * d * shape.h * 2 // 2**30)},
            "gpu_launches": int(launches), "clocks": clk.summary(w0, w1),
            "expert_ffn_flops_per_step": ffn_flops,
            "whole_step_tflops_of_expert_ffn": ffn_flops / (ms * 1e-3) / 1e12}
    print(json.dumps(line))


# FP32 FFMA peak of a B300: 148 SMs x 128 FP32 lanes x 2 flops x the 2032 MHz maximum
# SM clock (the CUDA-core GEMMs of the backward are bound by it).
FP32_FFMA_TFLOPS = 148 * 128 * 2 * 2.032e9 / 1e12


def backward_bench(args, shape):
    """The backward pass (moe_backward: forward recompute and every gradient) per
    step over one batch resident in HBM, on one GPU (a secondary measurement line)."""
    import sparsely_gated_mixture_03_b300 as moe
    torch.cuda.set_device(0)
    inp = S.make_flat_inputs(shape, seed=1000, device="cuda")
    T, d, n, h, k = shape.T, shape.d, shape.n, shape.h, shape.k
    cfg = moe.make_config(T, d, n, h, k, shape.x_dtype, shape.expert_dtype)
    ws = moe.alloc_backward_workspace(cfg)
    dy = torch.randn((T, d), generator=torch.Generator().manual_seed(7)).to("cuda")
    f = dict(device="cuda", dtype=torch.float32)
    out = [torch.empty((T, d), **f), torch.empty((d, n), **f), torch.empty((d, n), **f), None,
           torch.empty((n, d, h), **f), torch.empty((n, h, d), **f)]
    stream = torch.cuda.current_stream()
    steps_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]

    def step(ev=None):
        a = (cfg, inp["x"], inp["W_g"], inp["W_noise"], inp["eps"], inp["b_g"], inp["W_in"],
             inp["W_out"], dy, *out, ws)
        if ev is None:
            moe.moe_backward(*a, stream=stream)
        else:
            moe.moe_backward_timed(*a, ev, stream=stream)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert moe.moe_get_device_error() == 0
    with ClockSampler(0) as clk:
        # K plain moe_backward steps for the metric, then K with CUDA events at the stage
        # boundaries for the stage times (as in the forward bench)
        torch.cuda.synchronize()
        launches0 = moe.moe_launch_counter()
        w0 = time.time()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for i in range(args.steps):
            step()
        end.record(stream)
        torch.cuda.synchronize()
        w1 = time.time()
        launches = moe.moe_launch_counter() - launches0
        for i in range(args.steps):
            step(steps_ev[i])
        torch.cuda.synchronize()
    names = ["forward_recompute", "combine_and_gate_backward", "expert_data_gradients",
             "expert_weight_gradients", "gate_weight_gradients"]
    st = {nm: statistics.mean(ev[i].elapsed_time(ev[i + 1]) for ev in steps_ev)
          for i, nm in enumerate(names)}
    ms = start.elapsed_time(end) / args.steps
    ms_instrumented = statistics.mean(ev[0].elapsed_time(ev[5]) for ev in steps_ev)
    R = T * k
    expert_flops = 8.0 * R * d * h          # dU, dX_perm, dW_out, dW_in: 2 R d h each
    gate_flops = 6.0 * T * d * n            # dW_g, dW_noise, the gate's share of dx
    wgrad_flops = 4.0 * R * d * h           # dW_out, dW_in
    tc = shape.expert_dtype == torch.bfloat16 and d % 256 == 0 and h % 256 == 0
    pk = peaks()
    if tc:
        # the tensor-core weight gradients are bound by HBM: they read hidden, dE, x_perm
        # and dU (bf16) once and write both fp32 gradients (ncu: DRAM 75 % of peak, tensor
        # pipe 43 %); achieved = these algorithmic bytes / the stage's event time
        wgrad_bytes = 2.0 * R * (h + d) * 2 + 2.0 * n * h * d * 4
        ach = wgrad_bytes / (st["expert_weight_gradients"] * 1e-3) / 1e9
        peak, unit, bound = pk["hbm_gbs"], "GB/s", "hbm"
    else:
        ach = wgrad_flops / (st["expert_weight_gradients"] * 1e-3) / 1e12
        peak, unit, bound = FP32_FFMA_TFLOPS, "TFLOP/s", "alu"
    line = {"metric": "MoE backward (forward recompute + all gradients) tokens/s",
            "value": T / (ms * 1e-3), "unit": UNIT, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if shape.expert_dtype == torch.bfloat16 else "f32",
            "data": "synthetic (seeded N(0,1) inputs, dy and N(0,1/fan_in) weights)",
            "config": {"workload": shape.name, "T": T, "d": d, "n": n, "h": h, "k": k,
                       "l2": "inputs larger than L2"},
            "gpu_launches": int(launches), "clocks": clk.summary(w0, w1),
            "stages": {nm: {"ms": v} for nm, v in st.items()},
            "stages_region": {"ms_per_step": ms_instrumented,
                              "note": "K more steps through moe_backward_timed: CUDA events "
                                      "at the stage boundaries, the source of stages and roofline"},
            "roofline": {"kernel": "expert weight gradients (%s)"
                                   % ("ffn_wgrad_tc_kernel" if tc else "grouped_gemm_kernel"),
                         "bound": bound, "achieved": ach, "peak": peak, "unit": unit,
                         "frac": ach / peak, "traffic": None,
                         "peak_source": (pk["source"] + " HBM copy") if tc else
                                        "derived: 148 SMs x 128 FP32 lanes x 2 x 2032 MHz"},
            "expert_weight_gradient_tflops": wgrad_flops / (st["expert_weight_gradients"] * 1e-3) / 1e12,
            "expert_gradient_flops": expert_flops, "gate_gradient_flops": gate_flops}
    print(json.dumps(line))


def batchwise_bench(args, shape):
    """The layer with the batchwise top-m gate (moe_batchwise_forward) per step over one
    batch resident in HBM, on one GPU (a secondary measurement line)."""
    import sparsely_gated_mixture_03_b300 as moe
    torch.cuda.set_device(0)
    inp = S.make_flat_inputs(shape, seed=1000, device="cuda")
    T, d, n, h, k = shape.T, shape.d, shape.n, shape.h, shape.k
    cfg = moe.make_config(T, d, n, h, k, shape.x_dtype, shape.expert_dtype)
    ws = moe.alloc_batchwise_workspace(cfg)
    y = torch.empty((T, d), dtype=torch.float32, device="cuda")
    losses = torch.empty(3, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        moe.moe_batchwise_forward(cfg, inp["x"], inp["W_g"], inp["W_noise"], inp["eps"],
                                  inp["b_g"], inp["W_in"], inp["W_out"], y, losses, workspace=ws,
                                  stream=stream)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert moe.moe_get_device_error() == 0
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clk:
        torch.cuda.synchronize()
        launches0 = moe.moe_launch_counter()
        w0 = time.time()
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        w1 = time.time()
        launches = moe.moe_launch_counter() - launches0
    ms = e0.elapsed_time(e1) / args.steps
    line = {"metric": "MoE fwd routed tokens/s (batchwise top-m gate)", "value": T / (ms * 1e-3),
            "unit": UNIT, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if shape.expert_dtype == torch.bfloat16 else "f32",
            "data": "synthetic (seeded N(0,1) inputs and N(0,1/fan_in) weights)",
            "config": {"workload": shape.name + "-batchwise", "T": T, "d": d, "n": n, "h": h,
                       "k": k, "rows_per_expert": k * T // n, "l2": "inputs larger than L2"},
            "gpu_launches": int(launches), "clocks": clk.summary(w0, w1)}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="moe256", choices=sorted(S.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--host-noise", action="store_true",
                    help="pass the gate noise in as eps (copied from the host in e2e) instead "
                         "of letting the layer draw it on the device")
    ap.add_argument("--batchwise", action="store_true",
                    help="time the layer with the batchwise top-m gate instead")
    ap.add_argument("--backward", action="store_true",
                    help="time the backward pass (moe_backward) instead of the forward")
    ap.add_argument("--switch", action="store_true",
                    help="the Switch gate (softmax over all n logits, k = 1, the Switch loss)")
    ap.add_argument("--capacity-factor", type=float, default=0.0,
                    help="per-expert capacity of ceil(F T k / n) routed rows (0: none, the "
                         "layer as the paper defines it)")
    ap.add_argument("--ffn-tiles", default="auto", choices=["auto", "rows", "sized"],
                    help="tile kind of the expert FFN: the library's default (auto, 256-row "
                         "tiles) or forced, for comparison")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    shape = S.WORKLOADS[args.workload]
    if args.switch:      # Switch routing: one expert per token, the softmax over all n
        if not isinstance(shape, S.FlatShape):
            ap.error("--switch applies to the flat workloads")
        shape = dataclasses.replace(shape, k=1, name=shape.name + "-switch-k1")
    if args.batchwise:
        if not isinstance(shape, S.FlatShape) or args.impl != "ours":
            ap.error("--batchwise times this library's flat layer")
        batchwise_bench(args, shape)
        return
    if args.backward:
        if not isinstance(shape, S.FlatShape) or args.impl != "ours":
            ap.error("--backward times this library's flat layer")
        backward_bench(args, shape)
        return
    if isinstance(shape, S.HierShape):
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the reference arm times the "
                              "oracle on the flat workloads only"}))
            return
        hier_bench(args, shape)
        return
    if args.impl == "reference":
        reference_arm(args, shape)
        return

    import sparsely_gated_mixture_03_b300 as moe
    from sparsely_gated_mixture_03_b300 import shards
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    def barrier():
        if dist is not None:
            dist.barrier()

    dev = "cuda"
    inp = S.make_flat_inputs(shape, seed=1000 + rank, device=dev)
    capacity = (math.ceil(args.capacity_factor * shape.T * shape.k / shape.n)
                if args.capacity_factor > 0 else 0)
    # the layer draws its gate noise on the device (one standard normal per token and
    # expert, a counter-based generator seeded per rank) unless --host-noise passes eps in
    noise_flag = 0 if args.host_noise else moe.FLAG_DEVICE_NOISE
    cfg = moe.make_config(shape.T, shape.d, shape.n, shape.h, shape.k, shape.x_dtype,
                          shape.expert_dtype, flags=ffn_flags(args) | noise_flag,
                          capacity=capacity, noise_seed=1000 + rank)
    ws = moe.alloc_workspace(cfg)
    eps_in = None if noise_flag else inp["eps"]
    T, d, n, h, k = shape.T, shape.d, shape.n, shape.h, shape.k
    R = T * k
    y = torch.empty((T, d), dtype=torch.float32, device=dev)
    losses = torch.empty(3, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    names = ["gate", "dispatch", "expert_ffn", "combine", "losses"]
    # data parallel (N > 1): the balancing losses are those of the whole job's batch, so
    # every step all-reduces the rank's [importance; load] (2n floats) and forms the
    # losses from the totals (moe_losses_from_sums)
    sums = torch.empty(2 * n, dtype=torch.float32, device=dev)
    cfg_all = moe.make_config(T * world, d, n, h, k, shape.x_dtype, shape.expert_dtype,
                              flags=ffn_flags(args), capacity=capacity)

    def step(ev=None):
        if ev is None:
            moe.moe_forward(cfg, inp["x"], inp["W_g"], inp["W_noise"], eps_in, inp["b_g"],
                            inp["W_in"], inp["W_out"], y, losses, importance=sums[:n],
                            load=sums[n:], workspace=ws, stream=stream)
        else:       # the same call, with CUDA events at its stage boundaries
            moe.moe_forward_timed(cfg, inp["x"], inp["W_g"], inp["W_noise"], eps_in,
                                  inp["b_g"], inp["W_in"], inp["W_out"], y, losses, ev,
                                  importance=sums[:n], load=sums[n:], workspace=ws,
                                  stream=stream)
        if dist is not None:
            shards.global_losses(cfg_all, sums, losses, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert moe.moe_get_device_error() == 0

    # ---- timed region: K whole steps of the call a user makes (moe_forward) ----------------
    dev_index = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[local]
                    if os.environ.get("CUDA_VISIBLE_DEVICES") else local)
    with ClockSampler(dev_index) as clk:
        barrier()
        torch.cuda.synchronize()
        launches0 = moe.moe_launch_counter()
        w0 = time.time()
        start = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for i in range(args.steps):
            step()
        end = torch.cuda.Event(enable_timing=True)
        end.record(stream)              # after the last step's all-reduce at N > 1
        torch.cuda.synchronize()
        w1 = time.time()
        barrier()
        launches = moe.moe_launch_counter() - launches0
        ms = start.elapsed_time(end) / args.steps

        # ---- second timed region: the same K steps with CUDA events at the stage
        # boundaries (moe_forward_timed), for the stage times and the roofline kernel's
        # duration; an event between two kernels makes the second wait for the first to
        # finish instead of starting its setup early, so this region runs a little slower
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
        barrier()
        torch.cuda.synchronize()
        w2 = time.time()
        for i in range(args.steps):
            step(evs[i])
        end2 = torch.cuda.Event(enable_timing=True)
        end2.record(stream)
        torch.cuda.synchronize()
        w3 = time.time()
        barrier()
    clocks = clk.summary(w0, w1)
    clocks_stages = clk.summary(w2, w3)
    ms_instrumented = evs[0][0].elapsed_time(end2) / args.steps
    stage_ms = {s: sum(ev[i].elapsed_time(ev[i + 1]) for ev in evs) / args.steps
                for i, s in enumerate(names)}
    assert moe.moe_get_device_error() == 0
    ms = max_over_ranks(ms, dist, dev)
    ms_instrumented = max_over_ranks(ms_instrumented, dist, dev)
    value = world * T / (ms * 1e-3)

    pk = peaks()
    ffn_flops = 4.0 * T * k * d * h
    ffn_tflops = ffn_flops / (stage_ms["expert_ffn"] * 1e-3) / 1e12
    xb = 2 if shape.x_dtype == torch.bfloat16 else 4
    eb = 2 if shape.expert_dtype == torch.bfloat16 else 4
    # algorithmic bytes of the memory-bound stages (each tensor read or written once)
    gate_bytes = T * d * xb + 2 * d * n * 4 + T * n * 4 + R * 8 + T + n * 4
    if noise_flag:
        gate_bytes += T * n * 4          # the drawn noise, written once and read by the gate
    dispatch_bytes = R * 4 + T * d * xb + R * d * xb + (n + 1) * 4 + 2 * R * 4
    combine_bytes = R * d * eb + R * 8 + T * d * 4
    stages = {}
    for s in names:
        stages[s] = {"ms": stage_ms[s]}
    for s, b in (("gate", gate_bytes), ("dispatch", dispatch_bytes), ("combine", combine_bytes)):
        gbs = b / (stage_ms[s] * 1e-3) / 1e9
        stages[s].update(algorithmic_bytes=b, gbs=gbs, hbm_frac=gbs / pk["hbm_gbs"])
    gate_flops = 2.0 * T * d * 2 * n
    stages["gate"]["tflops_fp32_equiv"] = gate_flops / (stage_ms["gate"] * 1e-3) / 1e12
    stages["gate"]["tensor_tflops_bf16"] = 3 * gate_flops / (stage_ms["gate"] * 1e-3) / 1e12
    # the peak of the clock regime the timed region ran in: the sustained bf16 figure
    # (measured under the power cap) when the clock record shows sw_power_cap active,
    # else the burst figure; both fractions are reported
    capped = "sw_power_cap" in clocks_stages.get("reasons", [])
    sustained = pk.get("bf16_tflops_sustained")
    tc_peak = sustained if capped and sustained else pk["bf16_tflops"]
    tc_peak_source = (pk["source"] + (" bf16 sustained (sw_power_cap active in the stages' timed region)"
                                      if capped and sustained else " bf16 burst"))
    stages["expert_ffn"].update(flops=ffn_flops, tflops=ffn_tflops,
                                tensor_frac=ffn_tflops / tc_peak,
                                tensor_frac_of_burst=ffn_tflops / pk["bf16_tflops"])

    # ---- end to end through the public API with host buffers -------------------------
    # every step copies its x (and with --host-noise its eps) in from pinned host memory
    # and its y and losses out; copies run on their own streams, double-buffered, so the
    # copies of one step overlap the compute of its neighbours
    def fwd(xx, ee, yy, ll):
        moe.moe_forward(cfg, xx, inp["W_g"], inp["W_noise"], ee, inp["b_g"], inp["W_in"],
                        inp["W_out"], yy, ll, importance=sums[:n], load=sums[n:], workspace=ws,
                        stream=stream)
        if dist is not None:
            shards.global_losses(cfg_all, sums, ll, stream=stream)

    x_host = inp["x"].cpu().pin_memory()
    eps_host = None if noise_flag else inp["eps"].cpu().pin_memory()
    y_host = [torch.empty((T, d), dtype=torch.float32).pin_memory() for _ in range(2)]
    l_host = [torch.empty(3, dtype=torch.float32).pin_memory() for _ in range(2)]
    x_dev = [torch.empty_like(inp["x"]) for _ in range(2)]
    eps_dev = [None if noise_flag else torch.empty_like(inp["eps"]) for _ in range(2)]
    y_dev = [torch.empty((T, d), dtype=torch.float32, device=dev) for _ in range(2)]
    l_dev = [torch.empty(3, dtype=torch.float32, device=dev) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def e2e_run(nsteps):
        done_in = [torch.cuda.Event() for _ in range(nsteps)]
        done_fwd = [torch.cuda.Event() for _ in range(nsteps)]
        done_out = [torch.cuda.Event() for _ in range(nsteps)]
        for i in range(nsteps):
            b = i % 2
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(done_fwd[i - 2])      # buffer b's inputs consumed
                x_dev[b].copy_(x_host, non_blocking=True)
                if eps_host is not None:
                    eps_dev[b].copy_(eps_host, non_blocking=True)
                done_in[i].record(s_in)
            stream.wait_event(done_in[i])
            if i >= 2:
                stream.wait_event(done_out[i - 2])        # buffer b's outputs copied out
            fwd(x_dev[b], eps_dev[b], y_dev[b], l_dev[b])
            done_fwd[i].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done_fwd[i])
                y_host[b].copy_(y_dev[b], non_blocking=True)
                l_host[b].copy_(l_dev[b], non_blocking=True)
                done_out[i].record(s_out)
        torch.cuda.synchronize()
    e2e_run(3)
    e2e_steps = max(3, min(args.steps, 50))
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    e2e_run(e2e_steps)
    e2e_ms = (time.perf_counter() - t0) * 1e3 / e2e_steps
    e2e_ms = max_over_ranks(e2e_ms, dist, dev)
    assert moe.moe_get_device_error() == 0

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if shape.expert_dtype == torch.bfloat16 else "f32",
        "data": "synthetic (seeded N(0,1) inputs and N(0,1/fan_in) weights of the pages' layer shape)",
        "config": {"workload": shape.name, "T": T, "d": d, "n": n, "h": h, "k": k,
                   "gate_dtype": "f32", "parallelism": f"dp{world}" if world > 1 else "single",
                   "losses": ("whole batch: all-reduce of 2n floats per step" if world > 1
                              else "whole batch"),
                   "ffn_tiles": ffn_tiles_name(args, R, n),
                   "capacity": capacity if capacity else "none",
                   "noise": ("eps passed in (host copies in e2e)" if args.host_noise else
                             "drawn on the device by the layer (MOE_FLAG_DEVICE_NOISE, one "
                             "standard normal per token and expert, seed 1000 + rank)"),
                   "l2": "inputs larger than L2 (expert weights %d MB; x and eps %d MB)"
                         % (2 * n * d * h * eb // 2**20, (T * d * xb + T * n * 4) // 2**20)},
        "gpu_launches": int(launches),
        "clocks": clocks,
        "stages": stages,
        "stages_region": {"ms_per_step": ms_instrumented, "clocks": clocks_stages,
                          "note": "K more steps through moe_forward_timed: CUDA events at the "
                                  "stage boundaries, the source of stages and roofline"},
        "expert_ffn_tflops": ffn_tflops,
        "roofline": {"kernel": "expert_ffn (%s)" % ("ffn_pair_tc_kernel" if ffn_row_tiles(args, R, n)
                                                     else "ffn_swap_tc_kernel"),
                     "bound": "tensor",
                     "achieved": ffn_tflops, "peak": tc_peak, "unit": "TFLOP/s",
                     "frac": ffn_tflops / tc_peak,
                     "frac_of_burst": ffn_tflops / pk["bf16_tflops"],
                     "traffic": FFN_TRAFFIC.get((shape.name, "ffn_pair_tc_kernel"
                                                 if ffn_row_tiles(args, R, n)
                                                 else "ffn_swap_tc_kernel")),
                     "peak_source": tc_peak_source},
        "e2e": {"value": world * T / (e2e_ms * 1e-3), "unit": UNIT,
                "h2d_bytes_per_step": int(x_host.numel() * x_host.element_size()
                                          + (0 if eps_host is None else eps_host.numel() * 4)),
                "d2h_bytes_per_step": int(y_host[0].numel() * 4 + 12)},
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(shape, inp)
    print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
