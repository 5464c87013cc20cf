"""clis_certify_noalloc: certification for callers that cannot allocate.

Some callers of this library run where cudaMalloc is off limits (a plugin
inside another runtime that owns all device memory, a serving loop whose
memory was planned up front).  clis_certify_noalloc gives them the same
certification using a fixed scratch array inside the library.  These tests
call it through the C ABI and check it against clis_certify (which takes a
caller workspace) on two calls in a row, so a second call that inherits the
first call's scratch contents must still be right.  Both entry points run
the same deterministic kernels, so their outputs must be identical bit for
bit; the integer results are also checked against the CPU oracle.  The file
sorts last so a run that stops at the first failure has already run every
other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from certified_fixed_stabilizer_gb300 import clis
from certified_fixed_stabilizer_gb300.workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 4 << 20  # CLIS_NOALLOC_SCRATCH_BYTES in include/clis.h
CLIS_ERR_UNSUPPORTED = 2
CLIS_ERR_WORKSPACE = 4


def _garbage_outputs(q):
    BH, d, N = q.shape[0] * q.shape[1], q.shape[-1], q.shape[-2]
    # Outputs start as garbage so a stale or skipped write cannot pass.
    kbar = torch.full((BH, d), float("nan"), device=q.device)
    certs = torch.full((BH, clis.CERT_WORDS), -7, dtype=torch.int32, device=q.device)
    mu = torch.full((BH * N,), float("nan"), device=q.device)
    return kbar, certs, mu


def _check_same(q, k, v, sl2):
    ref_kbar, ref_certs, ref_mu = _garbage_outputs(q)
    clis.clis_certify(q, k, v, sl2, kbar=ref_kbar, certs=ref_certs, mu=ref_mu)
    kbar, certs, mu = _garbage_outputs(q)
    clis.clis_certify_noalloc(q, k, v, sl2, kbar=kbar, certs=certs, mu=mu)
    torch.cuda.synchronize()
    # Bit for bit: same kernels, same order of every sum.
    assert torch.equal(kbar.view(torch.int32), ref_kbar.view(torch.int32))
    assert torch.equal(certs, ref_certs)
    assert torch.equal(mu.view(torch.int32), ref_mu.view(torch.int32))
    got = clis.decode_certs(certs)
    # And against the CPU oracle: flags, reasons and G, A, C exactly, kbar to
    # fp32 summation error.
    okbar, oc = oracle.certify(q, k, v, sl2)
    for h, (g, o) in enumerate(zip(got, oc)):
        for key in ("certified", "reason", "G", "A", "C"):
            assert g[key] == o[key], (h, key, g, o)
    np.testing.assert_allclose(kbar.cpu().double().numpy(), okbar, rtol=2e-5, atol=2e-5)
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


def _shape(H, N, d):
    s = clis.Shape(B=1, H=H, Nq=N, Nk=N, d=d)
    for t in "qkv":
        setattr(s, f"{t}_sn", d)
        setattr(s, f"{t}_sh", N * d)
        setattr(s, f"{t}_sb", H * N * d)
    return s


def test_noalloc_rejects_shapes_beyond_its_scratch():
    """A shape needing more than the fixed scratch is refused before any launch
    (the pointers below are never touched)."""
    s = _shape(64, 600000, 128)
    assert clis.clis_certify_workspace_size(s) > SCRATCH_BYTES
    fake = 0x100000
    st = clis.load_library().clis_certify_noalloc(ctypes.byref(s), fake, fake, fake, 0.1, 1, 2, fake, fake, None,
                                                  None)
    assert st == CLIS_ERR_WORKSPACE


def test_noalloc_reports_argument_errors_before_the_scratch_size():
    """An unsupported head dimension is reported as such even when the shape
    would also need more scratch than the library holds."""
    s = _shape(64, 600000, 256)
    assert clis.clis_certify_workspace_size(s) > SCRATCH_BYTES
    fake = 0x100000
    lib = clis.load_library()
    assert lib.clis_certify_noalloc(ctypes.byref(s), fake, fake, fake, 0.1, 1, 2, fake, fake, None,
                                    None) == CLIS_ERR_UNSUPPORTED
    assert lib.clis_certify(ctypes.byref(s), fake, fake, fake, 0.1, 1, 2, fake, fake, None, None, 0,
                            None) == CLIS_ERR_UNSUPPORTED
