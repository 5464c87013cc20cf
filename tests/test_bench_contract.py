"""The one-line JSON that bench.py prints: every key the benchmark contract
asks for, with consistent values, for the reference arm (the CPU oracle; runs
anywhere) and for the library's own arm (needs the GPU).  The tiny workload
keeps both runs to seconds."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

BASE_KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
             "scaling", "vs_baseline", "dtype", "data", "config", "e2e", "cpu_baseline"}


def _run(*args, timeout=600):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, capture_output=True,
                       text=True, timeout=timeout)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.strip().splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


def _check_common(d, steps, warmup):
    assert BASE_KEYS <= set(d), BASE_KEYS - set(d)
    assert d["n_gpus"] == 1 and d["steps"] == steps and d["warmup"] == warmup
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["vs_baseline"] is None
    assert d["unit"] == "TFLOP/s" and d["value"] > 0 and d["ms_per_step"] > 0
    assert d["config"]["workload"].startswith("tiny")
    assert d["data"] == "synthetic"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0 and cb["sample"]


def test_reference_arm_line():
    d = _run("--impl", "reference", "--config", "tiny", "--steps", "2", "--warmup", "1")
    _check_common(d, 2, 1)
    assert d["impl"] == "reference" and d["dtype"] == "f64"
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


@pytest.mark.gpu
def test_own_arm_line():
    from gpu_util import need_gpu
    need_gpu()
    d = _run("--config", "tiny", "--steps", "3", "--warmup", "3")
    _check_common(d, 3, 3)
    assert "impl" not in d or d["impl"] != "reference"
    assert d["dtype"] == "bf16"
    roof = d["roofline"]
    assert roof["bound"] == "tensor" and roof["unit"] == "TFLOP/s" and roof["peak"] > 0
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-9
    clocks = d["clocks"]
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(clocks)
    # 4 certification launches + 1 attention launch per timed step
    assert d["gpu_launches"] == 5 * d["steps"]
    assert d["device_error_word"] == 0 and d["certified_heads"] == "2/2"
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["unit"] == d["unit"]
    # Q, K, V in and O out, bf16 [1, 2, 256, 64]
    assert e2e["h2d_bytes_per_step"] == 3 * 2 * 256 * 64 * 2 and e2e["d2h_bytes_per_step"] == 2 * 256 * 64 * 2
    for leg in ("online", "online_lazy", "backward", "chunked"):
        assert leg in d
