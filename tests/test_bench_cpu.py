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
