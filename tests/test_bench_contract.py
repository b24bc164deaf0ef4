"""The bench's output contract on CPU, no GPU: the reference arm (the oracle
timed on the host cores) prints one JSON line with the keys the harness reads,
and the FFN traffic figure is reported only while the kernel sources are the
ones its ncu capture was taken on."""
import hashlib
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_reference_arm_json_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0",
                          "--cpu-budget", "0.5"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert d["steps"] == 1 and d["warmup"] >= 3          # warm-up is never below three steps
    assert d["scaling"] == "weak" and d["n_gpus"] == 1
    assert "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_traffic_only_for_the_captured_sources(tmp_path, monkeypatch):
    src = tmp_path / "kernel.cu"
    src.write_text("// one version of a kernel\n")
    sha = hashlib.sha256(src.read_bytes()).hexdigest()
    prof = tmp_path / "profile.md"
    prof.write_text("# a capture\n\n- traffic_bytes_per_launch: 1000\n- algorithmic_bytes_per_launch: 990\n"
                    "- active_experts: 3\n- sources_sha256: %s\n" % sha)
    monkeypatch.setattr(bench, "FFN_PROFILE", str(prof))
    monkeypatch.setattr(bench, "FFN_SOURCES", [str(src)])
    assert bench.ffn_traffic_capture() == (1000.0, 990.0, 3)
    src.write_text("// the kernel changed since the capture\n")
    assert bench.ffn_traffic_capture() is None
    monkeypatch.setattr(bench, "FFN_PROFILE", str(tmp_path / "missing.md"))
    assert bench.ffn_traffic_capture() is None
