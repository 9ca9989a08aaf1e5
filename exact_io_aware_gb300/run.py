"""Run the attention forward/backward on a synthetic problem and time it.

For profilers (ncu) and for timing one shape or one named workload:

    python -m exact_io_aware_gb300.run --B 1 --H 64 --n 4096 --d 128 --iters 2
    python -m exact_io_aware_gb300.run --workload longctx_bf16_n65536 --iters 5

Inputs are seeded N(0,1) tensors generated on the device (the workload's query scale
applied); a bitmap workload uses the seeded allowed-key sets of ``synth``.  Prints the mean
CUDA-event time of the forward and backward calls after one untimed call, with TFLOP/s
counted the standard way (forward 4·B·H·n²·d·κ, backward 2.5 times that; κ = 1/2 causal,
popcount/n² for a bitmap).
"""
from __future__ import annotations

import argparse
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main(argv=None):
    import numpy as np
    import torch

    import exact_io_aware_gb300 as ea

    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default=None, help="named workload from synth.CONFIGS")
    ap.add_argument("--B", type=int, default=1)
    ap.add_argument("--H", type=int, default=64)
    ap.add_argument("--n", type=int, default=4096)
    ap.add_argument("--d", type=int, default=128)
    ap.add_argument("--dtype", choices=["f16", "bf16", "f32"], default="bf16")
    ap.add_argument("--mask", choices=["none", "causal"], default="none")
    ap.add_argument("--kv-block", type=int, default=0)
    ap.add_argument("--iters", type=int, default=2)
    ap.add_argument("--fwd-only", action="store_true")
    ap.add_argument("--splits", type=int, default=None,
                    help="forward through attn_fwd_split with this many key shares (0 = library choice)")
    ap.add_argument("--dropout", type=float, default=0.0, help="drop probability (0 = none)")
    ap.add_argument("--n-kv", type=int, default=0,
                    help="keys of a key/value cache (forward of --n query rows through attn_fwd_kv)")
    ap.add_argument("--fp8", action="store_true", help="forward through attn_fwd_fp8 (E4M3 inputs)")
    ap.add_argument("--fp8-blocks", action="store_true",
                    help="with --fp8: attn_fp8_quantize (timed apart) + attn_fwd_fp8_blocks")
    ap.add_argument("--rotate", action="store_true",
                    help="with --fp8-blocks: incoherent processing of Q and K")
    ap.add_argument("--vdim", type=int, default=0, help="value width v (default: d)")
    ap.add_argument("--json", action="store_true", help="print one JSON line")
    a = ap.parse_args(argv)

    B, H, n, d, dtype, mask, kvb, qs = a.B, a.H, a.n, a.d, a.dtype, a.mask, a.kv_block, 1.0
    c = d ** -0.5
    bits = None
    kappa = 0.5 if mask == "causal" else 1.0
    fwd_only = a.fwd_only
    name = "custom"
    if a.workload:
        from synth import bitmap_mask, pack_bitmap, workload
        wl = workload(a.workload)
        B, H, n, d, dtype, mask, c, qs = wl.B, wl.H, wl.n, wl.d, wl.dtype, wl.mask, wl.c, wl.q_scale
        kvb = a.kv_block or wl.kv_block
        fwd_only = fwd_only or "bwd" not in wl.passes
        name = wl.name
        kappa = 0.5 if mask == "causal" else 1.0
        if mask == "bitmap":
            allowed = bitmap_mask(n, wl.seed)
            kappa = float(allowed.mean())
            bits = torch.from_numpy(pack_bitmap(allowed).view(np.int32)).cuda()
    dt = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}[dtype]
    ea.load()
    if a.n_kv:
        return _run_kv(a, B, H, n, a.n_kv, d, dt, mask, c, kvb)
    if a.fp8:
        return _run_fp8(a, B, H, n, d, mask, c)
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    shape = (B, H, n, d)
    vd = a.vdim or d
    q, k = (torch.randn(shape, device="cuda", generator=g) for _ in range(2))
    v, do = (torch.randn((B, H, n, vd), device="cuda", generator=g) for _ in range(2))
    q = (q * qs).to(dt)
    k, v, do = k.to(dt), v.to(dt), do.to(dt)
    o = torch.empty_like(v)
    lse = torch.empty(shape[:3], device="cuda", dtype=torch.float32)
    ws = torch.empty(ea.attn_bwd_workspace_bytes(dt, *shape), dtype=torch.uint8, device="cuda")
    splits, fws = 1, None
    if a.splits is not None:
        splits = a.splits or ea.attn_fwd_split_count(dt, *shape, kv_block=kvb)
        fws = torch.empty(max(16, ea.attn_fwd_split_workspace_bytes(dt, *shape, splits)),
                          dtype=torch.uint8, device="cuda")
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(a.iters + 1)]
    for e in ev:
        e[0].record()
        if a.splits is None:
            ea.attn_fwd(q, k, v, c, mask=mask, mask_bits=bits, kv_block=kvb, o=o, lse=lse,
                        dropout_p=a.dropout, seed=1234)
        else:
            ea.attn_fwd_split(q, k, v, c, mask=mask, mask_bits=bits, kv_block=kvb, o=o, lse=lse,
                              num_splits=splits, workspace=fws)
        e[1].record()
        if not fwd_only:
            ea.attn_bwd(q, k, v, o, lse, do, c, mask=mask, mask_bits=bits, kv_block=kvb,
                        workspace=ws, dropout_p=a.dropout, seed=1234)
        e[2].record()
    torch.cuda.synchronize()
    status = ea.attn_device_status()
    fwd_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in ev[1:]]))
    bwd_ms = float(np.mean([e[1].elapsed_time(e[2]) for e in ev[1:]])) if not fwd_only else None
    # forward: S (width d) and P V (width v); backward: S, dK, dQ (d) and dP, dV (v)
    fl = 2.0 * B * H * n * n * (d + vd) * kappa
    fl_b = 2.0 * B * H * n * n * (3 * d + 2 * vd) * kappa
    out = {"workload": name, "B": B, "H": H, "n": n, "d": d, "v": vd, "dtype": dtype, "mask": mask,
           "kv_block": kvb, "splits": splits, "dropout": a.dropout, "kappa": kappa, "fwd_ms": fwd_ms,
           "fwd_tflops": fl / (fwd_ms / 1e3) / 1e12, "status": status}
    if bwd_ms is not None:
        out.update(bwd_ms=bwd_ms, bwd_tflops=fl_b / (bwd_ms / 1e3) / 1e12)
    if a.json:
        print(json.dumps(out))
    else:
        print(" ".join(f"{k}={v:.4g}" if isinstance(v, float) else f"{k}={v}" for k, v in out.items()))
    return 0 if status == ea.ATTN_OK else 1


def _run_fp8(a, B, H, n, d, mask, c):
    """FP8 forward on N(0,1) inputs quantized per tensor; time and TFLOP/s."""
    import numpy as np
    import torch

    import exact_io_aware_gb300 as ea
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    xs = [torch.randn((B, H, n, d), device="cuda", generator=g) for _ in range(3)]
    o = torch.empty((B, H, n, d), device="cuda", dtype=torch.bfloat16)
    lse = torch.empty((B, H, n), device="cuda", dtype=torch.float32)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(a.iters + 1)]
    quant_ms = None
    if a.fp8_blocks:
        xb = [x.to(torch.bfloat16) for x in xs]
        signs = None
        if a.rotate:
            signs = (torch.randint(0, 2, (d,), device="cuda", generator=g) * 2 - 1).to(torch.int8)
        ops = None
        for e in ev:
            e[0].record()
            ops = ea.attn_fp8_quantize(*xb, signs=signs)
            e[1].record()
            ea.attn_fwd_fp8_blocks(*ops, c, mask=mask, o=o, lse=lse)
            e[2].record()
        torch.cuda.synchronize()
        quant_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in ev[1:]]))
        ms = float(np.mean([e[1].elapsed_time(e[2]) for e in ev[1:]]))
    else:
        scales = [float(x.abs().max()) / 448.0 for x in xs]
        q8, k8, v8 = ((x / s).to(torch.float8_e4m3fn) for x, s in zip(xs, scales))
        vt8 = v8.transpose(2, 3).contiguous()
        for e in ev:
            e[0].record()
            ea.attn_fwd_fp8(q8, k8, vt8, c, *scales, mask=mask, o=o, lse=lse)
            e[1].record()
        torch.cuda.synchronize()
        ms = float(np.mean([e[0].elapsed_time(e[1]) for e in ev[1:]]))
    status = ea.attn_device_status()
    kappa = 0.5 if mask == "causal" else 1.0
    out = {"workload": "fp8_blocks" if a.fp8_blocks else "fp8", "B": B, "H": H, "n": n, "d": d,
           "dtype": "e4m3", "mask": mask, "rotate": bool(a.rotate),
           "fwd_ms": ms, "fwd_tflops": 4.0 * B * H * n * n * d * kappa / (ms / 1e3) / 1e12,
           "status": status}
    if quant_ms is not None:
        qbytes = 3 * B * H * n * d * 3 + 3 * 4 * B * H * ((n + 127) // 128)  # read 2 B, write 1 B
        out.update(quant_ms=quant_ms, quant_gbs=qbytes / (quant_ms / 1e3) / 1e9)
    print(json.dumps(out) if a.json else " ".join(f"{k}={v}" for k, v in out.items()))
    return 0 if status == ea.ATTN_OK else 1


def _run_kv(a, B, H, nq, nk, d, dt, mask, c, kvb):
    """Forward of nq query rows against an nk-key cache; time and K/V bytes streamed."""
    import numpy as np
    import torch

    import exact_io_aware_gb300 as ea
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    q = torch.randn((B, H, nq, d), device="cuda", generator=g).to(dt)
    k = torch.randn((B, H, nk, d), device="cuda", generator=g).to(dt)
    v = torch.randn((B, H, nk, d), device="cuda", generator=g).to(dt)
    splits = a.splits if a.splits else ea.attn_fwd_kv_split_count(dt, B, H, nq, nk, d, kvb)
    ws = torch.empty(max(16, ea.attn_fwd_split_workspace_bytes(dt, B, H, nq, d, splits)),
                     dtype=torch.uint8, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((B, H, nq), device="cuda", dtype=torch.float32)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(a.iters + 1)]
    for e in ev:
        e[0].record()
        ea.attn_fwd_kv(q, k, v, c, mask=mask, kv_block=kvb, num_splits=splits, o=o, lse=lse,
                       workspace=ws)
        e[1].record()
    torch.cuda.synchronize()
    status = ea.attn_device_status()
    ms = float(np.mean([e[0].elapsed_time(e[1]) for e in ev[1:]]))
    if mask == "causal":  # query i sees keys <= i + nk - nq
        pairs = sum(max(0, min(nk, i + nk - nq + 1)) for i in range(nq))
    else:
        pairs = nq * nk
    kv_bytes = 2 * B * H * nk * d * q.element_size()
    out = {"workload": "kv_cache", "B": B, "H": H, "n_q": nq, "n_kv": nk, "d": d,
           "dtype": str(dt).split(".")[-1], "mask": mask, "splits": splits, "fwd_ms": ms,
           "fwd_tflops": 4.0 * B * H * pairs * d / (ms / 1e3) / 1e12,
           "kv_gbs": kv_bytes / (ms / 1e3) / 1e9, "kv_bytes": kv_bytes, "status": status}
    print(json.dumps(out) if a.json else " ".join(f"{k}={v}" for k, v in out.items()))
    return 0 if status == ea.ATTN_OK else 1


if __name__ == "__main__":
    sys.exit(main())
