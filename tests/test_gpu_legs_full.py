"""The benchmark's extra legs at full size, in the launch configuration
bench.py times, against the oracle on seed-chosen rows (always row 0, N-1 and
the ragged last tile): the ring-step form with K/V in eight chunks (720p; the
causal shape through the causal chunk entry point) and the FP8 P.V path on the
mixed workload (its 48 certified heads take E4M3, the 16 injected heads the
online BF16 path)."""
import os

import numpy as np
import pytest
import torch

import oracle
from certified_fixed_stabilizer_gb300 import clis
from certified_fixed_stabilizer_gb300.workloads import WORKLOADS, make_inputs, sample_rows
from gpu_util import assert_close_to_oracle, flat, need_gpu

pytestmark = pytest.mark.gpu


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


def _bench_bounds(N, n_chunks=8):
    """The chunk boundaries bench.py uses (multiples of 8 inside the sequence)."""
    bounds = [round(i * N / n_chunks) for i in range(n_chunks + 1)]
    return [b - b % 8 if 0 < b < N else b for b in bounds]


@pytest.mark.parametrize("name,rows_per_head", [("720p", 16), ("causal", 48)])
def test_chunked_leg_full_size(name, rows_per_head):
    dev = need_gpu()
    w = WORKLOADS[name]
    q, k, v = make_inputs(w, device=dev)
    sl2 = clis.scale_log2_for(w.d)
    BH, N = w.heads, w.N
    mu = torch.empty(BH * N, device=dev)
    kbar, certs = clis.clis_certify(q, k, v, sl2, mu=mu)
    o_acc = torch.empty((BH * N, w.d), device=dev)
    l_acc = torch.empty(BH * N, device=dev)
    m_acc = torch.empty(BH * N, device=dev)
    bounds = _bench_bounds(N)
    for i, (a, b) in enumerate(zip(bounds[:-1], bounds[1:])):
        if w.causal:
            clis.clis_attn_fwd_chunk_causal(q, k[:, :, a:b], v[:, :, a:b], sl2, o_acc, l_acc, m_acc, a, kbar=kbar,
                                            certs=certs, first=(i == 0), mu=mu)
        else:
            clis.clis_attn_fwd_chunk(q, k[:, :, a:b], v[:, :, a:b], sl2, o_acc, l_acc, m_acc, kbar=kbar,
                                     certs=certs, first=(i == 0), mu=mu)
    lse2 = torch.empty(BH * N, device=dev)
    out = clis.clis_attn_chunk_finalize(q, o_acc, l_acc, m_acc, lse2=lse2)
    torch.cuda.synchronize()
    rows = sample_rows(N, rows_per_head, seed=3)
    ref, rlse = oracle.attention(flat(q).cpu(), flat(k).cpu(), flat(v).cpu(), w.softmax_scale(), causal=w.causal,
                                 rows=rows, with_lse2=True)
    assert_close_to_oracle(flat(out)[:, rows].float().cpu().numpy(), ref, f"{name} chunked x8")
    np.testing.assert_allclose(lse2.reshape(BH, N)[:, rows].cpu().numpy(), rlse, atol=2e-3, rtol=0)


def test_fp8pv_leg_mixed_full_size():
    dev = need_gpu()
    w = WORKLOADS["mixed"]
    q, k, v = make_inputs(w, device=dev)
    sl2 = clis.scale_log2_for(w.d)
    mu = torch.empty(w.heads * w.N, device=dev)
    kbar, certs = clis.clis_certify(q, k, v, sl2, mu=mu)
    vt8 = clis.clis_v_to_e4m3(v)
    out = clis.clis_attn_fwd_fp8pv(q, k, v, vt8, sl2, kbar=kbar, certs=certs, mu=mu)
    torch.cuda.synchronize()
    cs = clis.decode_certs(certs)
    assert sum(c["certified"] and c["B_h"] <= 8 and c["G"] <= 8 for c in cs) == 48
    rows = sample_rows(w.N, 32, seed=4)
    ref, _ = oracle.attention(flat(q).cpu(), flat(k).cpu(), flat(v).cpu(), w.softmax_scale(), rows=rows,
                              with_lse2=True)
    assert_close_to_oracle(flat(out)[:, rows].float().cpu().numpy(), ref, "mixed fp8 P.V")


def test_backward_leg_720p_full_size():
    """The backward as the bench times it at 720p (from a forward that wrote
    lse2): dQ on seed-chosen rows of three heads against the oracle's row-wise
    dQ, and two identities over every head: sum_j dV_j = sum_i dO_i (each row's
    softmax weights sum to 1) and sum_j dK_j = 0 (each row's dS sums to 0)."""
    from certified_fixed_stabilizer_gb300.workloads import make_dout
    from gpu_util import assert_grads_close
    dev = need_gpu()
    w = WORKLOADS["720p"]
    q, k, v = make_inputs(w, device=dev)
    do = make_dout(q.shape, device=dev)
    o, lse2 = clis.attention_fwd_lse(q, k, v)
    dq, dk, dv = clis.attention_bwd(q, k, v, o, do, lse2)
    torch.cuda.synchronize()
    heads, rows = [0, 21, 39], sample_rows(w.N, 8, seed=7)
    ref = oracle.attention_bwd_dq_rows(flat(q)[heads].cpu(), flat(k)[heads].cpu(), flat(v)[heads].cpu(),
                                       flat(do)[heads].cpu(), w.softmax_scale(), rows)
    assert_grads_close(flat(dq)[heads][:, rows].float().cpu().numpy(), ref, "dq", "720p backward")
    # sum_j dV_j = sum_i dO_i up to two roundings, each unbiased and at most 2^-9
    # of its term: P to bf16 inside the product and each dV_j to bf16.  Summed
    # over tens of thousands of independent terms they grow like the square
    # root of the count, so the difference is compared with the column's own
    # random-walk scale sqrt(sum_i dO_i^2) (a 0.1% slip in dV's scale moves it
    # by about that scale times 1e-3).
    dvf, dof = flat(dv).double(), flat(do).double()
    err = (dvf.sum(dim=1) - dof.sum(dim=1)).abs()                      # [BH, d]
    scale = dof.pow(2).sum(dim=1).sqrt()                               # [BH, d]
    from gpu_util import report
    report("720p backward sum dV", worst_ratio=float((err / scale).max()), worst_err=float(err.max()))
    assert (err <= 1e-3 * scale).all(), float((err / scale).max())
    dkf = flat(dk).double()
    assert torch.isfinite(dkf).all()
    assert (dkf.sum(dim=1).abs().amax(dim=1) <= 1e-2 * dkf.abs().sum(dim=1).amax(dim=1)).all()
