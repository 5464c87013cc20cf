"""The CPU legs of bench.py (the reference arm and the cpu_baseline sample)
run the oracle alone: they must not import the CUDA library's binding, whose
import loads (or builds) libclis.so.  Checked in a fresh interpreter, so that
nothing imported by other tests hides an import."""
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_PROBE = r"""
import argparse, io, json, sys, contextlib
sys.path.insert(0, ROOT)
import bench
from certified_fixed_stabilizer_gb300.workloads import WORKLOADS
w = WORKLOADS["tiny"]
args = argparse.Namespace(gpus=1, steps=1, warmup=1, variant="auto", config="tiny")
buf = io.StringIO()
with contextlib.redirect_stdout(buf):
    bench.run_reference(args, w, w.H)
line = json.loads(buf.getvalue().strip().splitlines()[-1])
assert line["impl"] == "reference" and line["value"] > 0, line
import torch
q = torch.zeros(1, 2, 256, 64, dtype=torch.bfloat16)
heads, rows = bench.cpu_sample_plan(q, q, q, w, target_s=0.05)
bench.oracle_sample_step(q, q, q, w, heads, rows)
loaded = sorted(m for m in sys.modules if m.startswith("certified_fixed_stabilizer_gb300"))
print(json.dumps(loaded))
"""


def test_reference_arm_does_not_import_the_binding():
    env = dict(os.environ, WORLD_SIZE="1", RANK="0")
    r = subprocess.run([sys.executable, "-c", f"ROOT = {ROOT!r}\n" + _PROBE], cwd=ROOT, capture_output=True,
                       text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-3000:]
    import json
    loaded = json.loads(r.stdout.strip().splitlines()[-1])
    # Only the package and its input generator, which holds no arithmetic of the method.
    assert "certified_fixed_stabilizer_gb300.clis" not in loaded, loaded
    assert "certified_fixed_stabilizer_gb300.build" not in loaded, loaded
    assert set(loaded) <= {"certified_fixed_stabilizer_gb300", "certified_fixed_stabilizer_gb300.workloads"}, loaded
