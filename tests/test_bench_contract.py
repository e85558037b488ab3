"""The JSON line bench.py prints: the reference arm (the CPU oracle, no GPU
needed) and the GPU arm, run as subprocesses with a few steps."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*args, timeout=600):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                       capture_output=True, text=True, timeout=timeout)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def _common(line):
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config"):
        assert key in line, key
    assert line["value"] > 0 and line["ms_per_step"] > 0
    assert line["higher_is_better"] is True
    assert line["unit"] == "TFLOP/s"
    assert "workload" in line["config"]


def test_reference_arm_line():
    line = _bench("--impl", "reference", "--steps", "2", "--warmup", "3", "--ref-seconds", "2")
    _common(line)
    assert line["impl"] == "reference" and line["dtype"] == "f64"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"]
    assert cb["sample"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


@pytest.mark.gpu
def test_gpu_arm_line():
    import __graft_entry__
    __graft_entry__.build()
    line = _bench("--steps", "5", "--warmup", "3", "--cpu-seconds", "1")
    _common(line)
    assert line["n_gpus"] == 1 and line["dtype"] == "bf16"
    assert line["config"]["calls_per_step"] == 768
    for key, bound, unit in (("roofline", "tensor", "TFLOP/s"),
                             ("roofline_window", "hbm", "GB/s")):
        rf = line[key]
        assert rf["bound"] == bound and rf["unit"] == unit
        assert 0 < rf["achieved"] and 0 < rf["peak"]
        assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-3
        # A number far above the measured peak would mean the kernel skipped work.
        assert rf["frac"] < 1.2
    # the per-kernel pass accounts for the whole step (isolated kernels run
    # no faster than the step's back-to-back launches)
    kinds = line["per_kind"]
    assert kinds["full_causal"]["calls"] == 384 and kinds["window_128"]["calls"] == 384
    assert sum(k["ms_per_step"] for k in kinds.values()) > 0.9 * line["ms_per_step"]
    e2e = line["e2e"]
    assert 0 < e2e["value"] < 1.05 * line["value"]
    assert e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert line["gpu_launches"] == 768 * line["steps"]
    assert "sm_mhz" in line["clocks"] and "reasons" in line["clocks"]
    pair = line["layer_pair"]
    assert pair["value"] > 0 and pair["full_causal"]["bound"] == "tensor"
    assert 0 < pair["window_128"]["frac"] < 1.2 and 0 < pair["full_causal"]["frac"] < 1.2
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1
