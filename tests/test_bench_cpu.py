"""Host-side pieces of bench.py: the profiled-traffic lookup and the reference arm's JSON line."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _summary(tmp_path, digest, value="1234567"):
    p = tmp_path / "summary.md"
    p.write_text("# capture\n\n"
                 f"`dram_bytes_per_launch = {value}`\n"
                 f"`source_digest = {digest}`\n")
    return str(p)


def test_traffic_read_when_sources_match(tmp_path):
    path = _summary(tmp_path, bench.kernel_source_digest())
    assert bench.profiled_traffic(path) == 1234567.0


def test_traffic_null_when_sources_changed(tmp_path):
    assert bench.profiled_traffic(_summary(tmp_path, "0000000000000000")) is None
    assert bench.profiled_traffic(str(tmp_path / "missing.md")) is None


def test_committed_summary_parses():
    # the committed summary carries both keys (whether its digest is current is not asserted:
    # it goes stale by design whenever the kernels change before the next capture)
    path = os.path.join(ROOT, "profiles", "bwd_tc_train_bf16_d128.md")
    text = open(path).read()
    assert "dram_bytes_per_launch = " in text and "source_digest = " in text


def test_reference_arm_prints_one_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "3"], capture_output=True, text=True,
                         timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_every_leg_names_a_workload_and_counts_allowed_pairs():
    import numpy as np
    from synth import bitmap_mask
    for name, passes in bench.LEGS:
        wl = bench.leg_workload(name)
        assert wl.name == name and passes in ("fwd", "fwd+bwd")
    assert bench.leg_workload("train_bf16_d128_causal").mask == "causal"
    # causal fwd+bwd over the whole head: 14 FLOP per allowed pair per column, n(n+1)/2 pairs
    wl = bench.leg_workload("small_causal_f32")
    flop, dt, sample = bench.oracle_leg(wl, "fwd+bwd", None)
    assert flop == 14.0 * (256 * 257 / 2) * 64 and dt > 0 and "forward + backward" in sample
    # forward-only legs sample evenly spaced rows; the last row sees every key
    wl = bench.leg_workload("longctx_bf16_n16384")
    flop, _, sample = bench.oracle_leg(wl, "fwd", None, row_budget=3)
    assert flop == 4.0 * (1 + 8192 + 16384) * 128 and sample.startswith("3 evenly spaced")
    wl = bench.leg_workload("bitmap_f32")
    allowed = bitmap_mask(wl.n, wl.seed)
    flop, _, _ = bench.oracle_leg(wl, "fwd", allowed, row_budget=2)
    assert flop == 4.0 * (allowed[0].sum() + allowed[-1].sum()) * 64
    assert 0.3 < float(np.mean(allowed)) < 0.5
