"""Long sequences: 262,144 tokens in one head (the pages' longest LLM context,
Table 3), forward and backward through the C ABI.

Row indices, tile counts and accumulator offsets run into the millions here,
so this catches index arithmetic that only overflows or wraps at size.  The
oracle evaluates sampled rows (each needs one pass over all keys): forward
outputs and dQ rows; dK obeys sum_j dK_j = 0 at any size.
"""
import dataclasses
import os

import numpy as np
import pytest
import torch

import oracle
from certified_fixed_stabilizer_gb300 import clis
from certified_fixed_stabilizer_gb300.workloads import WORKLOADS, make_dout, make_inputs, sample_rows
from gpu_util import assert_close_to_oracle, assert_grads_close, flat, need_gpu

pytestmark = pytest.mark.gpu

N_LONG = 262144


@pytest.fixture(scope="module", autouse=True)
def _setup():
    need_gpu()
    oracle.set_num_threads(os.cpu_count() or 1)
    clis.clis_clear_device_error()
    yield


@pytest.fixture(autouse=True)
def _device_error_word_stays_clear():
    yield
    code = clis.clis_get_device_error()
    clis.clis_clear_device_error()
    assert code == 0, f"device error word {code:#x}"


def _inputs(causal):
    w = dataclasses.replace(WORKLOADS["causal" if causal else "480p"], B=1)
    q, k, v = make_inputs(w, device=need_gpu(), N=N_LONG, H=1, seed=21)
    return w, q, k, v


@pytest.mark.parametrize("causal", [False, True])
def test_long_sequence_forward_and_certificate(causal):
    w, q, k, v = _inputs(causal)
    sl2 = clis.scale_log2_for(w.d)
    o, kbar, certs = clis.attention(q, k, v, causal=causal, return_certs=True)
    torch.cuda.synchronize()
    _, ocerts = oracle.certify(q.cpu(), k.cpu(), v.cpu(), sl2)
    got = clis.decode_certs(certs)
    for g, r in zip(got, ocerts):
        assert not r["band"]
        for key in ("certified", "G", "A", "C", "reason"):
            assert g[key] == r[key], (key, g, r)
    assert got[0]["A"] == 18 + got[0]["G"]  # ceil(log2 262144) = 18
    rows = sample_rows(N_LONG, 24, seed=5)
    ref = oracle.attention(flat(q).cpu(), flat(k).cpu(), flat(v).cpu(), w.softmax_scale(), causal=causal, rows=rows)
    assert_close_to_oracle(flat(o)[:, rows].float().cpu().numpy(), ref, f"forward N=262144 causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_long_sequence_backward(causal):
    w, q, k, v = _inputs(causal)
    do = make_dout(q.shape, device=q.device, seed=21)
    o, lse2 = clis.attention_fwd_lse(q, k, v, causal=causal)
    dq, dk, dv = clis.attention_bwd(q, k, v, o, do, lse2, causal=causal)
    torch.cuda.synchronize()
    rows = sample_rows(N_LONG, 12, seed=6)
    ref = oracle.attention_bwd_dq_rows(flat(q).cpu(), flat(k).cpu(), flat(v).cpu(), flat(do).cpu(),
                                       w.softmax_scale(), rows, causal=causal)
    assert_grads_close(flat(dq)[:, rows].float().cpu().numpy(), ref, "dq", f"backward N=262144 causal={causal}")
    dkf = flat(dk).double()
    assert torch.isfinite(dkf).all() and torch.isfinite(flat(dv).float()).all()
    colsum = dkf.sum(dim=1).abs().max().item()
    mag = dkf.abs().sum(dim=1).max().item()
    assert colsum <= 1e-2 * mag, colsum / mag
