#!/usr/bin/env python3
"""Benchmark of exact tiled attention on GB300: one step = forward + backward of the
training-shaped workload (B=8, H=16, n=4096, d=128, bf16, no mask), i.e. every kernel of
the path: forward (online softmax, writes O and LSE), backward preprocessing (D = rowsum
dO∘O, cleared dQ accumulator), backward (recomputed P, dS; dQ, dK, dV) and dQ
postprocessing.

Prints ONE JSON line (rank 0).  FLOPs per step are counted the standard way: forward
4·B·H·n²·d, backward 2.5 times that (10·B·H·n²·d), no mask so no causal factor.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (float64 numpy, materialised scores) on a bounded
sample of the same workload.  Under torchrun with N > 1 every rank runs its own replica of
the workload (weak scaling; the path needs no collective).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import select
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

# the oracle's BLAS threads: every host core this process may run on
_CORES = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, str(_CORES))

METRIC = "attention fwd/bwd TFLOP/s and % of GB300 dense BF16 peak at n=4096–65536"
WORKLOAD = "train_bf16_d128"
B, H, N_TOK, D = 8, 16, 4096, 128
C_SCALE = 1.0 / D ** 0.5
FWD_FLOP = 4.0 * B * H * N_TOK * N_TOK * D
BWD_FLOP = 2.5 * FWD_FLOP
STEP_FLOP = FWD_FLOP + BWD_FLOP
L2_BYTES = 129 * 2**20


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), \
            float(p["hbm_gbs"]), "measured"
    return 1900.0, 1700.0, 6800.0, "fallback"


def kernel_source_digest():
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_io_aware_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.startswith(("bwd_tc", "dq_tc", "tile", "ptx")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode())
                h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(path=None):
    """DRAM bytes per attn_bwd call (its two launches) from the committed ncu summary, or
    None if the summary is missing or was taken from different kernel sources."""
    path = path or os.path.join(ROOT, "profiles", "bwd_tc_train_bf16_d128.md")
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            text = line.strip().strip("`")
            if "=" in text and text.startswith(("dram_bytes_per_launch", "source_digest")):
                k, v = text.split("=", 1)
                vals[k.strip()] = v.strip().strip("`")
    if vals.get("source_digest") != kernel_source_digest():
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        if self.proc is not None:
            # nvidia-smi takes a while to start: wait (at most 5 s) for its first sample, taken
            # before the timed region and dropped, so that the region is sampled from its start
            ready, _, _ = select.select([self.proc.stdout], [], [], 5.0)
            if ready:
                self.proc.stdout.readline()
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "lines", []):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(n_gpus):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
        return rank, world, local, dist
    return 0, 1, 0, None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(x, dist):
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x, dist):
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------------------ oracle
def time_oracle(heads: int):
    from oracle import attention as ref
    from oracle import masks
    from synth import draw_head, workload
    import numpy as np
    wl = workload(WORKLOAD)
    mk = masks.none(N_TOK)
    rows = np.arange(N_TOK)
    inputs = [tuple(draw_head(wl, t, bh) for t in ("q", "k", "v", "do")) for bh in range(heads)]
    t0 = time.perf_counter()
    for q, k, v, g in inputs:
        a = mk(0, rows)
        ref.forward_rows(q, k, v, wl.c, a)
        ref.backward_head(q, k, v, wl.c, a, g)
    dt = time.perf_counter() - t0
    return 14.0 * N_TOK * N_TOK * D * heads, dt


def cpu_baseline(heads=24):
    flop, dt = time_oracle(heads)
    return {"value": flop / dt / 1e12, "unit": "TFLOP/s", "cores": _CORES, "kind": "oracle",
            "sample": f"{heads} of {B * H} heads of {WORKLOAD} (n={N_TOK}, d={D}), forward + "
                      f"backward in float64 numpy, {dt:.2f} s"}


def run_reference(args):
    rank, world, local, dist = dist_setup(args.gpus)
    if rank != 0:
        return
    heads = 1
    for _ in range(args.warmup):
        time_oracle(heads)
    times = []
    for _ in range(args.steps):
        flop, dt = time_oracle(heads)
        times.append(dt)
    total = sum(times)
    value = flop * args.steps / total / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{WORKLOAD}: B={B} H={H} n={N_TOK} d={D} bf16-rounded inputs, "
                               "no mask, forward + backward", "sample_heads_per_step": heads},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": _CORES, "kind": "oracle",
                         "sample": f"{heads} head per step of {B * H}"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------ GPU
def run_ours(args):
    import torch
    rank, world, local, dist = dist_setup(args.gpus)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    from exact_io_aware_gb300.build import build
    if rank == 0:
        build()
    barrier(dist)
    import exact_io_aware_gb300 as ea
    ea.load()

    g = torch.Generator(device=dev)
    g.manual_seed(3 + rank)
    shape = (B, H, N_TOK, D)
    q, k, v, do = (torch.randn(shape, device=dev, dtype=torch.float32, generator=g)
                   .to(torch.bfloat16) for _ in range(4))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N_TOK), device=dev, dtype=torch.float32)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(ea.attn_bwd_workspace_bytes(torch.bfloat16, B, H, N_TOK, D),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        ea.attn_fwd(q, k, v, C_SCALE, o=o, lse=lse, stream=stream)
        ea.attn_bwd(q, k, v, o, lse, do, C_SCALE, dq=dq, dk=dk, dv=dv, workspace=ws,
                    stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if ea.attn_device_status(stream) != ea.ATTN_OK:
        raise SystemExit("device status not clean after warm-up")

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    barrier(dist)
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index) as clk:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for i in range(args.steps):
            ev[i][0].record(stream)
            ea.attn_fwd(q, k, v, C_SCALE, o=o, lse=lse, stream=stream)
            ev[i][1].record(stream)
            ea.attn_bwd(q, k, v, o, lse, do, C_SCALE, dq=dq, dk=dk, dv=dv, workspace=ws,
                        stream=stream)
            ev[i][2].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize(dev)
    barrier(dist)
    status = ea.attn_device_status(stream)
    total_ms = t_start.elapsed_time(t_end)
    fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    bwd_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    total_ms = max_over_ranks(total_ms, dist)
    ms_per_step = total_ms / args.steps
    value = world * STEP_FLOP * args.steps / (total_ms / 1e3) / 1e12

    # End to end through the public API: every step copies its inputs from pinned host memory
    # to the device and its results back to pinned host memory, inside the timed region.  The
    # steps are pipelined the way a training input pipeline runs: two device sets of inputs and
    # outputs, the host-to-device copies of step i+1 and the device-to-host copies of step i-1
    # on their own streams while step i computes (the link carries both directions at once).
    h_in = [t.cpu().pin_memory() for t in (q, k, v, do)]
    h_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (o, lse, dq, dk, dv)]
    e2e_steps = max(2, min(args.steps, 30))
    sets = []
    for _ in range(2):
        d_in = [torch.empty_like(t) for t in (q, k, v, do)]
        d_out = [torch.empty_like(t) for t in (o, lse, dq, dk, dv)]
        d_ws = torch.empty_like(ws)
        sets.append((d_in, d_out, d_ws))
    s_h2d = torch.cuda.Stream(dev)
    s_d2h = torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of set b copied in
    ev_done = [torch.cuda.Event() for _ in range(2)]  # step on set b computed
    ev_out = [torch.cuda.Event() for _ in range(2)]   # outputs of set b copied out

    def e2e_run(nsteps, e_start=None, e_end=None):
        if e_start is not None:
            e_start.record(stream)
            s_h2d.wait_stream(stream)
            s_d2h.wait_stream(stream)
        for i in range(nsteps):
            b = i % 2
            d_in, d_out, d_ws = sets[b]
            if i >= 2:
                s_h2d.wait_event(ev_done[b])  # the step two back has read this set's inputs
            with torch.cuda.stream(s_h2d):
                for h, d_ in zip(h_in, d_in):
                    d_.copy_(h, non_blocking=True)
            ev_in[b].record(s_h2d)
            stream.wait_event(ev_in[b])
            if i >= 2:
                stream.wait_event(ev_out[b])  # its outputs are on the host
            qq, kk, vv, gg = d_in
            oo, ll, dqq, dkk, dvv = d_out
            ea.attn_fwd(qq, kk, vv, C_SCALE, o=oo, lse=ll, stream=stream)
            ea.attn_bwd(qq, kk, vv, oo, ll, gg, C_SCALE, dq=dqq, dk=dkk, dv=dvv, workspace=d_ws,
                        stream=stream)
            ev_done[b].record(stream)
            s_d2h.wait_event(ev_done[b])
            with torch.cuda.stream(s_d2h):
                for h, d_ in zip(h_out, d_out):
                    h.copy_(d_, non_blocking=True)
            ev_out[b].record(s_d2h)
        if e_end is not None:
            stream.wait_stream(s_d2h)
            e_end.record(stream)

    e2e_run(2)
    torch.cuda.synchronize(dev)
    barrier(dist)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_run(e2e_steps, e0, e1)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dist)
    e2e_value = world * STEP_FLOP * e2e_steps / (e2e_ms / 1e3) / 1e12
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = sum(t.numel() * t.element_size() for t in h_out)
    # the copied-back results are the step's results
    if not torch.equal(h_out[2][0, 0, :4].to(dev), sets[(e2e_steps - 1) % 2][1][2][0, 0, :4]):
        raise SystemExit("end-to-end results did not reach the host")

    if rank != 0:
        return
    burst, sustained, hbm, kind = peaks()
    dominant = "bwd" if bwd_ms >= fwd_ms else "fwd"
    dom_ms = bwd_ms if dominant == "bwd" else fwd_ms
    dom_flop = BWD_FLOP if dominant == "bwd" else FWD_FLOP
    achieved = dom_flop / (dom_ms / 1e3) / 1e12
    roof = {
        "bound": "tensor", "achieved": achieved, "peak": burst, "unit": "TFLOP/s",
        "frac": achieved / burst,
        "traffic": profiled_traffic() if dominant == "bwd" else None,
        "kernel": ("attn_bwd, timed as the whole call: dq_tc_kernel<bf16, d=128> (dQ and "
                   "the row table of LSE and D) then bwd_tc_kernel<bf16, d=128> (dK, dV)"
                   if dominant == "bwd"
                   else "fwd_tc_kernel<bf16, d=128, b=128>"),
        "peak_source": f"bf16_tflops burst ({kind}); kernel launches of a few ms",
        "algorithmic": f"{dom_flop:.4g} FLOP per launch = "
                       + ("10" if dominant == "bwd" else "4") + "·B·H·n²·d",
    }
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": f"{WORKLOAD}: B={B} H={H} n={N_TOK} d={D} bf16, no mask, c=1/sqrt(d), "
                        "forward + backward per step",
            "B": B, "H": H, "n": N_TOK, "d": D, "mask": "none", "kv_block": 128,
            "l2": "inputs larger than L2 (q, k, v, dO: 128 MiB each; 129 MiB L2), no flush",
            "pct_of_dense_bf16_peak": 100.0 * value / world / burst,
            "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
            "fwd_tflops": FWD_FLOP / (fwd_ms / 1e3) / 1e12,
            "bwd_tflops": BWD_FLOP / (bwd_ms / 1e3) / 1e12,
            "device_status": status,
        },
        "roofline": roof,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "pipelining": "two device sets; H2D of the next step and D2H of the previous "
                              "one on their own streams while a step computes"},
        "gpu_launches": 3 * args.steps,  # attn_fwd: 1 launch; attn_bwd: 2
        "clocks": clk.summary(),
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("at least 3 warm-up steps")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
