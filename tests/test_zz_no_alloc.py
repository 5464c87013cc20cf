"""clis_certify_noalloc: certification for callers that cannot allocate.

Some callers of this library run where cudaMalloc is off limits (a plugin
inside another runtime that owns all device memory, a serving loop whose
memory was planned up front).  clis_certify_noalloc gives them the same
certification using a fixed scratch array inside the library.  These tests
call it through the C ABI and check it against clis_certify (which takes a
caller workspace) on two calls in a row, so a second call that inherits the
first call's scratch contents must still be right.  The file sorts last so a
run that stops at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from certified_fixed_stabilizer_gb300 import clis
from certified_fixed_stabilizer_gb300.workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 4 << 20  # CLIS_NOALLOC_SCRATCH_BYTES in include/clis.h
CLIS_ERR_WORKSPACE = 4


def _noalloc(q, k, v, sl2):
    BH = q.shape[0] * q.shape[1]
    # Outputs start as garbage so a stale or skipped write cannot pass.
    kbar = torch.full((BH, q.shape[-1]), float("nan"), device=q.device)
    certs = torch.full((BH, clis.CERT_WORDS), -7, dtype=torch.int32, device=q.device)
    return clis.clis_certify_noalloc(q, k, v, sl2, kbar=kbar, certs=certs)


def _check_same(q, k, v, sl2):
    ref_kbar, ref_certs = clis.clis_certify(q, k, v, sl2)
    kbar, certs = _noalloc(q, k, v, sl2)
    torch.cuda.synchronize()
    np.testing.assert_allclose(kbar.cpu().numpy(), ref_kbar.cpu().numpy(), rtol=2e-5, atol=2e-5)
    got, ref = clis.decode_certs(certs), clis.decode_certs(ref_certs)
    for g, r in zip(got, ref):
        for key in ("certified", "reason", "G", "A", "C"):
            assert g[key] == r[key], (key, g, r)
        for key in ("B_h", "kappa", "qmax"):
            assert abs(g[key] - r[key]) <= 1e-4 * max(abs(r[key]), 1e-30), (key, g, r)
    return got


def test_noalloc_matches_workspace_entry_point_twice():
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a visible CUDA device")
    dev = torch.device("cuda:0")
    # Call 1: mixed-certification heads (outliers in a quarter of them).
    w = WORKLOADS["mixed"]
    q, k, v = make_inputs(w, device=dev, N=5000)
    got1 = _check_same(q, k, v, clis.scale_log2_for(w.d))
    assert 0 < sum(c["certified"] for c in got1) < len(got1)
    # Call 2, straight after: other data and a different shape (d = 64, fewer
    # rows), so scratch left over from call 1 is laid out differently.
    w2 = WORKLOADS["tiny"]
    q2, k2, v2 = make_inputs(w2, device=dev, N=1500, seed=9)
    got2 = _check_same(q2, k2, v2, clis.scale_log2_for(w2.d))
    assert all(c["certified"] for c in got2)
    assert clis.clis_get_device_error() == 0


def test_noalloc_rejects_shapes_beyond_its_scratch():
    """A shape needing more than the fixed scratch is refused before any launch
    (the pointers below are never touched)."""
    s = clis.Shape(B=1, H=64, Nq=75600, Nk=600000, d=128)
    for t in "qkv":
        setattr(s, f"{t}_sn", 128)
        setattr(s, f"{t}_sh", 600000 * 128)
        setattr(s, f"{t}_sb", 64 * 600000 * 128)
    assert clis.clis_certify_workspace_size(s) > SCRATCH_BYTES
    fake = 0x100000
    st = clis.load_library().clis_certify_noalloc(ctypes.byref(s), fake, fake, fake, 0.1, 1, 2, fake, fake, None,
                                                  None)
    assert st == CLIS_ERR_WORKSPACE
