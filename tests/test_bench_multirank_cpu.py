"""The bench's multi-rank plumbing on CPU with two gloo ranks (no GPU).

bench.py runs one rank per GPU under torchrun; every rank joins the barriers around the timed
region, the timed span is the maximum over ranks and the processed work the sum.  Here two
processes on the gloo backend check those reductions, and the reference arm launched by
torchrun with two ranks prints exactly one JSON line (rank 0) while rank 1 exits cleanly.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench

    r, w, _, dist = bench.dist_setup(world)
    bench.barrier(dist)
    mx = bench.max_over_ranks(1.5 + r, dist)
    sm = bench.sum_over_ranks(10.0 * (r + 1), dist)
    bench.barrier(dist)
    with open(os.path.join(out, f"rank{r}.json"), "w") as f:
        json.dump({"rank": r, "world": w, "max": mx, "sum": sm}, f)
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_max_and_sum(tmp_path):
    import torch.multiprocessing as mp

    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    for r in range(2):
        got = json.load(open(tmp_path / f"rank{r}.json"))
        assert got == {"rank": r, "world": 2, "max": 2.5, "sum": 30.0}


def test_reference_arm_under_torchrun_two_ranks():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "3"]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-3000:]
    lines = [l for l in out.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
