"""The library from plain C: tests/c_abi_example.c (no Python in the compute
path, no torch) is compiled against include/clis.h and libclis.so, run on
inputs written here, and its outputs are compared with the oracle -- the fused
forward, the no-allocation certification, the KV-chunk forms (causal chunks
at their key offsets), the FP8 P.V path and the forward on host buffers
(clis_attention_host)."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
from certified_fixed_stabilizer_gb300 import clis
from certified_fixed_stabilizer_gb300.workloads import WORKLOADS, make_inputs
from gpu_util import assert_close_to_oracle, flat, need_gpu

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _nvcc():
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    p = os.path.join(cuda, "bin", "nvcc")
    return p if os.path.exists(p) else (shutil.which("nvcc") or "nvcc")


@pytest.fixture(scope="module")
def c_program(tmp_path_factory):
    need_gpu()
    clis.load_library()  # builds libclis.so if needed
    libdir = os.path.dirname(clis.library_path())
    exe = str(tmp_path_factory.mktemp("c_abi") / "c_abi_example")
    subprocess.run([_nvcc(), "-O2", "-o", exe, os.path.join(ROOT, "tests", "c_abi_example.c"),
                    "-I" + os.path.join(ROOT, "include"), "-L" + libdir, "-lclis", "-Xlinker", "-rpath=" + libdir,
                    "-lcudart", "-lm"], check=True, capture_output=True, text=True)
    return exe


@pytest.mark.parametrize("causal,mode", [(False, "fused"), (True, "fused"), (False, "noalloc"), (True, "chunks"),
                                         (False, "chunks"), (False, "fp8"), (False, "host"), (True, "host")])
def test_c_program_matches_oracle(c_program, tmp_path, causal, mode):
    w = WORKLOADS["causal" if causal else "480p"]
    H, N = 3, 777
    q, k, v = make_inputs(w, device="cpu", N=N, H=H)
    for name, t in (("q", q), ("k", k), ("v", v)):
        t.contiguous().view(torch.int16).numpy().tofile(str(tmp_path / f"{name}.bin"))
    r = subprocess.run([c_program, str(tmp_path), str(w.B), str(H), str(N), str(w.d), str(int(causal)), mode],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    o = torch.from_numpy(np.fromfile(str(tmp_path / "o.bin"), dtype=np.int16)).view(torch.bfloat16)
    lse2 = np.fromfile(str(tmp_path / "lse2.bin"), dtype=np.float32)
    certs = torch.from_numpy(np.fromfile(str(tmp_path / "certs.bin"), dtype=np.int32))
    ref, rlse = oracle.attention(flat(q), flat(k), flat(v), w.softmax_scale(), causal=causal, with_lse2=True)
    got = o.float().numpy().reshape(ref.shape)
    if mode == "fp8":
        # E4M3 P.V on 777 keys: against the CPU model of the same roundings, and
        # against the oracle within the E4M3 error model (mean 0.05 / sqrt(Nk)).
        import rounding_model as rm
        from gpu_util import head_errors
        for h in range(ref.shape[0]):
            e, _, flip = rm.certified_forward_fp8pv(*(flat(t)[h].double().numpy() for t in (q, k, v)),
                                                    w.softmax_scale(), with_flip_bound=True)
            sc = max(1.0, np.abs(e).max())
            assert np.maximum(np.abs(got[h] - e) - np.abs(e) * 2.0 ** -8, 0).max() / sc <= 2 * flip / sc + 1e-4
        mx, mn = head_errors(got, ref)
        assert mn.max() <= 0.05 / np.sqrt(N) and mx.max() <= 2e-2, (mx.max(), mn.max())
    else:
        assert_close_to_oracle(got, ref, f"C program causal={causal} {mode}")
    if mode == "host":
        assert np.isnan(lse2).all()  # no lse2 on this path
    else:
        np.testing.assert_allclose(lse2.reshape(rlse.shape), rlse, atol=2e-3, rtol=0)
    _, ocerts = oracle.certify(q, k, v, clis.scale_log2_for(w.d))
    for g, c in zip(clis.decode_certs(certs.reshape(-1, clis.CERT_WORDS)), ocerts):
        for key in ("certified", "G", "A", "C", "reason"):
            assert g[key] == c[key], (key, g, c)
