"""bench.py on the GPU: one short run of the default workload prints one JSON line with every
field the benchmark contract names, with values that fit together (the value is the work over
the measured time, the roofline fraction is achieved over peak, our own kernels ran)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu


def _run(*args):
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "5", "--warmup", "3", "--e2e-steps", "4",
           "--skip-cpu", *args]
    out = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    return json.loads(lines[0])


def test_default_line_carries_the_contract_fields():
    d = _run("--skip-decode")
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "clocks", "gpu_launches", "e2e", "bandwidth"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["device_status"] == 0
    assert d["gpu_launches"] >= d["steps"]
    # valid-token TFLOP/s of the ramp: 1.0337 TFLOP per call
    assert d["value"] == pytest.approx(1.033677438976 / (d["ms_per_step"] * 1e-3), rel=1e-6)
    r = d["roofline"]
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"], rel=1e-9)
    assert 0.05 < r["frac"] < 1.5
    assert r["other_roof"]["bound"] == "hbm"
    e = d["e2e"]
    assert e["unit"] == d["unit"] and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert e["ms_per_step"] > d["ms_per_step"]          # the copies are inside the end-to-end time
    assert d["padding_gap_pct"] == pytest.approx(
        100.0 * (d["ms_no_topk_length"] / d["ms_topk_length_passed"] - 1.0), abs=1e-6)


def test_decode_line_names_the_hbm_roof():
    d = _run("--config", "decode", "--skip-e2e", "--no-clocks")
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(d["bandwidth"]["hbm_gbs"]["algorithmic"], rel=1e-9)
