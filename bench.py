#!/usr/bin/env python3
"""Benchmark of exact tiled attention on GB300.

Headline step = forward + backward of the training-shaped workload (B=8, H=16, n=4096,
d=128, bf16, no mask): three launches, every kernel of the path: the forward (online
softmax; writes O and LSE), the dQ kernel (recomputes P and dS per query tile, computes
D = rowsum(dO∘O) and writes the row table) and the dK/dV kernel (recomputes P and dS per key
tile).  FLOPs per step are counted the standard way: forward 4·B·H·n²·d, backward 2.5 times
that (10·B·H·n²·d), no mask so no causal factor.

After the headline, the line's "workloads" list times every other configuration of the
metric's range (n = 4096 ... 65536) the same way, each with its own roofline fraction and the
oracle timed on a bounded sample beside it: the long-context causal forwards (n = 16384 and
65536), the fp16 overflow shapes (d = 16 and 64, literal and hot scale), the block-sparse
bitmap shape (bf16 and float32), the causal training shape and the small float32 shape.

Prints ONE JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--no-legs]

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
        if name.startswith(("bwd_tc", "dq_tc", "tile", "ptx", "dropout")):
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
        # the same against the power-capped sustained rate, for a reader comparing runs whose
        # clock record shows the cap active (frac above stays against the burst figure)
        "peak_sustained": sustained,
        "frac_of_sustained": achieved / sustained,
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
    if world == 1 and not args.no_legs:
        with ClockSampler(dev.index) as clk_legs:
            line["workloads"] = run_legs(dev, stream, burst, hbm, line["clocks"].get("sm_max_mhz"))
        line["workloads_clocks"] = clk_legs.summary()
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------ other workloads
# (workload, passes): every configuration of the metric's range beside the headline.
LEGS = [
    ("longctx_bf16_n16384", "fwd"),
    ("longctx_bf16_n65536", "fwd"),
    ("overflow_f16_d16", "fwd"),
    ("overflow_f16_d16_hot", "fwd"),
    ("overflow_f16_d64", "fwd"),
    ("overflow_f16_d64_hot", "fwd"),
    ("bitmap_bf16", "fwd+bwd"),
    ("bitmap_f32", "fwd+bwd"),
    ("train_bf16_d128_causal", "fwd+bwd"),
    ("small_causal_f32", "fwd+bwd"),
]
MUFU_EX2_PER_CLK_SM = 32   # ex2.approx results per clock per SM (probed on this part)
FFMA_PER_CLK_SM = 128      # float32 FMA lanes per SM
N_SM = 152


def leg_workload(name):
    from synth import workload
    if name == "train_bf16_d128_causal":
        return workload("train_bf16_d128").with_(name=name, mask="causal")
    return workload(name)


def leg_mask(wl):
    """(kappa, allowed [n, n] bool or None, device words or None)."""
    import numpy as np
    import torch
    if wl.mask == "bitmap":
        from synth import bitmap_mask, pack_bitmap
        allowed = bitmap_mask(wl.n, wl.seed)
        bits = torch.from_numpy(pack_bitmap(allowed).view(np.int32)).cuda()
        return float(allowed.mean()), allowed, bits
    return (0.5 if wl.mask == "causal" else 1.0), None, None


def oracle_leg(wl, passes, allowed, row_budget=512):
    """The oracle on a bounded sample of one head of the workload: (FLOP, seconds, sample).
    Forward-only legs take evenly spaced query rows of head 0 (all keys they see); legs with a
    backward take the whole head (the key gradients need every row)."""
    import numpy as np
    from oracle import attention as ref
    from oracle import masks
    from synth import draw_head
    n, d = wl.n, wl.d
    if allowed is not None:
        mk = masks.dense(allowed)
    else:
        mk = masks.for_kind(wl.mask, n)
    q, k, v = (draw_head(wl, t, 0) for t in ("q", "k", "v"))
    if passes == "fwd":
        rows = np.unique(np.linspace(0, n - 1, min(n, row_budget)).astype(np.int64))
        a = mk(0, rows)
        t0 = time.perf_counter()
        ref.forward_rows(q[rows], k, v, wl.c, a)
        dt = time.perf_counter() - t0
        flop = 4.0 * float(a.sum()) * d
        return flop, dt, f"{rows.size} evenly spaced query rows of 1 of {wl.heads} heads, forward"
    g = draw_head(wl, "do", 0)
    rows = np.arange(n)
    a = mk(0, rows)
    t0 = time.perf_counter()
    ref.forward_rows(q, k, v, wl.c, a)
    ref.backward_head(q, k, v, wl.c, a, g)
    dt = time.perf_counter() - t0
    return 14.0 * float(a.sum()) * d, dt, f"1 of {wl.heads} heads, forward + backward"


def time_calls(fn, iters, flush, stream):
    """Mean CUDA-event time (ms) of fn() over iters calls, L2 flushed before each call."""
    import torch
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    evs = []
    for i in range(iters):
        flush.fill_(float(i))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        evs.append((e0, e1))
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in evs)


def run_legs(dev, stream, burst, hbm, sm_mhz_max):
    """Every other configuration of the metric's range, timed as the headline is (CUDA events
    on the launching stream, L2 flushed between calls), with its roofline fractions and the
    oracle on a bounded sample beside it."""
    import torch
    import exact_io_aware_gb300 as ea
    flush = torch.empty(64 * 2**20, dtype=torch.float32, device=dev)  # 256 MiB > L2
    dts = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
    clock_ghz = (sm_mhz_max or 2070.0) / 1e3
    mufu_peak = MUFU_EX2_PER_CLK_SM * N_SM * clock_ghz * 1e9        # ex2 per second
    ffma_peak = 2.0 * FFMA_PER_CLK_SM * N_SM * clock_ghz * 1e9 / 1e12  # float32 TFLOP/s
    out = []
    for name, passes in LEGS:
        wl = leg_workload(name)
        kappa, allowed, bits = leg_mask(wl)
        g = torch.Generator(device=dev)
        g.manual_seed(wl.seed)
        shape = (wl.B, wl.H, wl.n, wl.d)
        dt = dts[wl.dtype]
        q, k, v, do = (torch.randn(shape, device=dev, generator=g) for _ in range(4))
        q = (q * wl.q_scale).to(dt)
        k, v, do = k.to(dt), v.to(dt), do.to(dt)
        o = torch.empty_like(q)
        lse = torch.empty(shape[:3], device=dev, dtype=torch.float32)
        kvb = wl.kv_block
        pairs = wl.heads * wl.n * wl.n * kappa
        fwd_flop = 4.0 * pairs * wl.d
        bwd_flop = 2.5 * fwd_flop
        iters = 5 if wl.n >= 65536 else 20

        def fwd():
            ea.attn_fwd(q, k, v, wl.c, mask=wl.mask, mask_bits=bits, kv_block=kvb, o=o, lse=lse,
                        stream=stream)

        fwd_ms = time_calls(fwd, iters, flush, stream)
        leg = {"workload": name, "B": wl.B, "H": wl.H, "n": wl.n, "d": wl.d, "dtype": wl.dtype,
               "mask": wl.mask, "kappa": kappa, "passes": passes, "fwd_ms": fwd_ms,
               "fwd_tflops": fwd_flop / (fwd_ms / 1e3) / 1e12}
        splits = ea.attn_fwd_split_count(dt, wl.B, wl.H, wl.n, wl.d, kvb)
        best_fwd_ms = fwd_ms
        if splits > 1:
            ws = torch.empty(max(16, ea.attn_fwd_split_workspace_bytes(dt, wl.B, wl.H, wl.n, wl.d,
                                                                         splits)),
                             dtype=torch.uint8, device=dev)

            def fwd_split():
                ea.attn_fwd_split(q, k, v, wl.c, mask=wl.mask, mask_bits=bits, kv_block=kvb,
                                  num_splits=splits, o=o, lse=lse, workspace=ws, stream=stream)

            leg["fwd_split_ms"] = time_calls(fwd_split, iters, flush, stream)
            leg["fwd_split_shares"] = splits
            best_fwd_ms = min(fwd_ms, leg["fwd_split_ms"])
        step_ms = best_fwd_ms
        step_flop = fwd_flop
        if passes == "fwd+bwd":
            fwd()
            dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
            ws_b = torch.empty(ea.attn_bwd_workspace_bytes(dt, wl.B, wl.H, wl.n, wl.d),
                               dtype=torch.uint8, device=dev)

            def bwd():
                ea.attn_bwd(q, k, v, o, lse, do, wl.c, mask=wl.mask, mask_bits=bits, kv_block=kvb,
                            dq=dq, dk=dk, dv=dv, workspace=ws_b, stream=stream)

            bwd_ms = time_calls(bwd, iters, flush, stream)
            leg["bwd_ms"] = bwd_ms
            leg["bwd_tflops"] = bwd_flop / (bwd_ms / 1e3) / 1e12
            step_ms += bwd_ms
            step_flop += bwd_flop
        leg["status"] = ea.attn_device_status(stream)
        leg["tflops"] = step_flop / (step_ms / 1e3) / 1e12
        e = 4 if wl.dtype == "f32" else 2
        fwd_bytes = wl.heads * (4.0 * wl.n * wl.d * e + 4.0 * wl.n)
        frac = {}
        if wl.dtype == "f32":
            frac["fp32_alu"] = leg["tflops"] / ffma_peak
        else:
            frac["tensor"] = leg["tflops"] / burst
        frac["hbm_fwd"] = fwd_bytes / (best_fwd_ms / 1e3) / 1e9 / hbm
        frac["mufu_fwd"] = pairs / (best_fwd_ms / 1e3) / mufu_peak
        bound = max(frac, key=frac.get)
        leg["roofline"] = {
            "fractions": frac, "highest": bound,
            "peaks": {"tensor_tflops": burst, "hbm_gbs": hbm, "fp32_alu_tflops": ffma_peak,
                      "mufu_ex2_per_s": mufu_peak},
            "peak_source": "tensor and HBM measured (MEASURED_PEAKS.json); float32 FMA and ex2 "
                           "rates = per-SM unit counts x 152 SMs x the maximum SM clock",
            "algorithmic": "FLOP 4·B·H·n²·d·κ forward (2.5x backward); forward bytes "
                           "4·n·d·e + 4n per head; one exp2 per allowed (query, key) pair",
        }
        try:
            flop_c, dt_c, sample = oracle_leg(wl, passes, allowed)
            leg["cpu_baseline"] = {"value": flop_c / dt_c / 1e12, "unit": "TFLOP/s",
                                   "cores": _CORES, "kind": "oracle",
                                   "sample": f"{sample}, {dt_c:.2f} s"}
        except MemoryError:
            leg["cpu_baseline"] = None
        out.append(leg)
        del q, k, v, do, o, lse
        torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-legs", action="store_true",
                    help="time the headline step only (no other workloads)")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("at least 3 warm-up steps")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
