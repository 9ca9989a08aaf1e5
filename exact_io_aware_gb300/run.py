"""Run the attention forward/backward on a synthetic problem a few times.

Meant for profilers (ncu) and quick timing of one shape:

    python -m exact_io_aware_gb300.run --B 1 --H 64 --n 4096 --d 128 --dtype bf16 \\
        --mask none --iters 2

Inputs are seeded N(0,1) tensors generated on the device.  Prints the device time of the
last forward and backward call.
"""
from __future__ import annotations

import argparse
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main(argv=None):
    import torch

    import exact_io_aware_gb300 as ea

    ap = argparse.ArgumentParser()
    ap.add_argument("--B", type=int, default=1)
    ap.add_argument("--H", type=int, default=64)
    ap.add_argument("--n", type=int, default=4096)
    ap.add_argument("--d", type=int, default=128)
    ap.add_argument("--dtype", choices=["f16", "bf16", "f32"], default="bf16")
    ap.add_argument("--mask", choices=["none", "causal"], default="none")
    ap.add_argument("--kv-block", type=int, default=0)
    ap.add_argument("--iters", type=int, default=2)
    ap.add_argument("--fwd-only", action="store_true")
    a = ap.parse_args(argv)
    dt = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}[a.dtype]
    ea.load()
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    shape = (a.B, a.H, a.n, a.d)
    q, k, v, do = (torch.randn(shape, device="cuda", generator=g).to(dt) for _ in range(4))
    c = a.d ** -0.5
    o = torch.empty_like(q)
    lse = torch.empty(shape[:3], device="cuda", dtype=torch.float32)
    ws = torch.empty(ea.attn_bwd_workspace_bytes(dt, *shape), dtype=torch.uint8, device="cuda")
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    for _ in range(a.iters):
        ev[0].record()
        ea.attn_fwd(q, k, v, c, mask=a.mask, kv_block=a.kv_block, o=o, lse=lse)
        ev[1].record()
        if not a.fwd_only:
            ea.attn_bwd(q, k, v, o, lse, do, c, mask=a.mask, kv_block=a.kv_block, workspace=ws)
        ev[2].record()
    torch.cuda.synchronize()
    status = ea.attn_device_status()
    print(f"fwd {ev[0].elapsed_time(ev[1]):.3f} ms  bwd {ev[1].elapsed_time(ev[2]):.3f} ms  "
          f"status {status}")
    return 0 if status == ea.ATTN_OK else 1


if __name__ == "__main__":
    sys.exit(main())
