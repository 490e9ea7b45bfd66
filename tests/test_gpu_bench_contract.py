"""The benchmark's output contract: one JSON line with the required keys,
consistent with itself (value and ms_per_step, roofline fraction, launch
count), for the default workload, the MLA step and the oracle arm."""

import json
import subprocess
import sys
from pathlib import Path

import pytest

pytestmark = pytest.mark.gpu

ROOT = Path(__file__).resolve().parents[1]
KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
        "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e",
        "gpu_launches", "clocks"}


def _run(*args):
    out = subprocess.run([sys.executable, str(ROOT / "bench.py"), *args], cwd=ROOT,
                         capture_output=True, text=True, timeout=900)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    return json.loads(lines[0])


@pytest.mark.parametrize("extra", [[], ["--mla"]])
def test_bench_line(extra):
    d = _run("--steps", "50", "--warmup", "3", "--stage-steps", "5", "--e2e-steps", "5",
             "--no-cpu-baseline", *extra)
    assert KEYS <= d.keys()
    assert d["n_gpus"] == 1 and d["steps"] == 50 and d["warmup"] == 3
    assert d["scaling"] == "weak" and d["higher_is_better"] is True
    assert abs(d["value"] * d["ms_per_step"] * 1e-3 - 1.0) < 1e-6  # steps/s over one GPU
    r = d["roofline"]
    assert r["bound"] in ("hbm", "tensor") and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    assert 0 < r["frac"] < 1.5
    assert d["gpu_launches"] >= 3 * d["steps"]
    e = d["e2e"]
    assert e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0 and e["value"] > 0
    assert d["config"]["workload"]


@pytest.mark.parametrize("extra", [[], ["--mla"]])
def test_reference_arm_line(extra):
    d = _run("--impl", "reference", "--steps", "3", "--warmup", "3", *extra)
    assert d["impl"] == "reference"
    # the oracle alone: the library's shared object is never loaded on this arm
    assert "liboracle.so" in d["loaded_libraries"]
    assert "libpks.so" not in d["loaded_libraries"]
    assert {"metric", "value", "unit", "ms_per_step", "cpu_baseline", "e2e"} <= d.keys()
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
