"""Grouped-query and multi-query attention through broadcast K/V strides.

The query heads of a group share one key/value head: the key/value heads are
folded into the batch and K, V get head stride 0 (clis.grouped_query_views, no
copy).  Checks, against the oracle on the same keys and values repeated per
query head: the certificates (flags and the integers G, A, C bit-exact), the
forward output and lse2; and bit-identity with the same call on a materialised
repeated K/V (the kernels read the same values through the broadcast map).
The backward sums each group's dK and dV inside the dK/dV kernel: checked
against the oracle's gradients on repeated K/V summed over each group.
"""
import dataclasses
import os

import numpy as np
import pytest
import torch

import oracle
from certified_fixed_stabilizer_gb300 import clis
from certified_fixed_stabilizer_gb300.workloads import WORKLOADS, make_inputs
from certified_fixed_stabilizer_gb300.workloads import make_dout
from gpu_util import assert_close_to_oracle, assert_grads_close, flat, need_gpu

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


CASES = [  # B, H (query heads), H_kv, N, d, causal
    (2, 8, 2, 1000, 128, False),
    (2, 8, 2, 1000, 128, True),
    (1, 8, 1, 777, 64, False),      # multi-query
    (3, 6, 3, 513, 128, True),
]


def _inputs(B, H, Hkv, N, d, causal, seed):
    dev = need_gpu()
    w = dataclasses.replace(WORKLOADS["causal" if causal else "480p"], B=B, d=d)
    q, _, _ = make_inputs(w, device=dev, N=N, H=H, seed=seed)
    _, k, v = make_inputs(w, device=dev, N=N, H=Hkv, seed=seed + 1)
    return q, k, v


@pytest.mark.parametrize("B,H,Hkv,N,d,causal", CASES)
def test_grouped_query_forward_matches_oracle(B, H, Hkv, N, d, causal):
    q, k, v = _inputs(B, H, Hkv, N, d, causal, seed=40 + H + N)
    g = H // Hkv
    o, kbar, certs = clis.attention(q, k, v, causal=causal, return_certs=True)
    torch.cuda.synchronize()
    assert o.shape == q.shape
    krep, vrep = (t.repeat_interleave(g, dim=1) for t in (k, v))  # [B, H, N, d]: head h uses h // g
    ref, _ = oracle.attention(flat(q).cpu(), flat(krep).cpu(), flat(vrep).cpu(), d ** -0.5, causal=causal,
                              with_lse2=True)
    what = f"GQA B={B} H={H} H_kv={Hkv} N={N} d={d} causal={causal}"
    assert_close_to_oracle(flat(o).float().cpu().numpy(), ref, what)
    sl2 = clis.scale_log2_for(d)
    _, ocerts = oracle.certify(q.cpu(), krep.cpu(), vrep.cpu(), sl2)
    for hd, (gc, oc) in enumerate(zip(clis.decode_certs(certs), ocerts)):
        if not oc["band"]:
            for key in ("certified", "G", "A", "C", "reason"):
                assert gc[key] == oc[key], (what, hd, key, gc, oc)
    # The same call on materialised repeated K/V gives the same bits.
    o2, _, certs2 = clis.attention(q, krep.contiguous(), vrep.contiguous(), causal=causal, return_certs=True)
    torch.cuda.synchronize()
    assert torch.equal(o, o2), what
    assert torch.equal(certs, certs2), what


def test_grouped_query_lse2_and_views():
    B, H, Hkv, N, d = 2, 8, 2, 640, 128
    q, k, v = _inputs(B, H, Hkv, N, d, False, seed=77)
    qf, kf, vf, _ = clis.grouped_query_views(q, k, v)
    assert qf.shape == (B * Hkv, H // Hkv, N, d) and kf.stride(1) == 0 and vf.stride(1) == 0
    assert qf.data_ptr() == q.data_ptr() and kf.data_ptr() == k.data_ptr()
    sl2 = clis.scale_log2_for(d)
    lse2 = torch.empty(B * H * N, device=q.device)
    kbar, certs = clis.clis_certify(qf, kf, vf, sl2)
    o = clis.clis_attn_fwd(qf, kf, vf, sl2, kbar=kbar, certs=certs, lse2=lse2)
    torch.cuda.synchronize()
    krep, vrep = (t.repeat_interleave(H // Hkv, dim=1) for t in (k, v))
    ref, rlse = oracle.attention(flat(q).cpu(), flat(krep).cpu(), flat(vrep).cpu(), d ** -0.5, with_lse2=True)
    assert_close_to_oracle(o.reshape(B * H, N, d).float().cpu().numpy(), ref, "GQA views")
    np.testing.assert_allclose(lse2.reshape(B * H, N).cpu().numpy(), rlse, atol=2e-3, rtol=0)


@pytest.mark.parametrize("B,H,Hkv,N,d,causal", [(1, 4, 1, 300, 128, False), (2, 6, 2, 257, 128, True),
                                                 (1, 8, 2, 200, 64, False)])
def test_grouped_query_backward_matches_oracle(B, H, Hkv, N, d, causal):
    q, k, v = _inputs(B, H, Hkv, N, d, causal, seed=90 + H + N)
    g = H // Hkv
    do = make_dout(q.shape, device=q.device, seed=5)
    o, lse2 = clis.attention_fwd_lse(q, k, v, causal=causal)
    dq, dk, dv = clis.attention_bwd(q, k, v, o, do, lse2, causal=causal)
    torch.cuda.synchronize()
    assert dk.shape == k.shape and dv.shape == v.shape and dq.shape == q.shape
    krep, vrep = (t.repeat_interleave(g, dim=1) for t in (k, v))
    rdq, rdk, rdv = oracle.attention_bwd(flat(q).cpu(), flat(krep).cpu(), flat(vrep).cpu(), flat(do).cpu(),
                                         d ** -0.5, causal=causal)
    what = f"GQA backward B={B} H={H} H_kv={Hkv} N={N} d={d} causal={causal}"
    # The group's gradients summed: reference [B*H_kv, N, d].
    rdk = np.asarray(rdk).reshape(B * Hkv, g, N, d).sum(axis=1)
    rdv = np.asarray(rdv).reshape(B * Hkv, g, N, d).sum(axis=1)
    assert_grads_close(flat(dq).float().cpu().numpy(), rdq, "dq", what)
    assert_grads_close(flat(dk).float().cpu().numpy(), rdk, "dk", what)
    assert_grads_close(flat(dv).float().cpu().numpy(), rdv, "dv", what)
    # Deterministic: a second run gives the same bits.
    dq2, dk2, dv2 = clis.attention_bwd(q, k, v, o, do, lse2, causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(dk, dk2) and torch.equal(dv, dv2) and torch.equal(dq, dq2)


def test_grouped_query_autograd():
    B, H, Hkv, N, d = 1, 4, 2, 256, 128
    q, k, v = _inputs(B, H, Hkv, N, d, True, seed=11)
    q, k, v = (t.clone().requires_grad_() for t in (q, k, v))
    o = clis.attention_autograd(q, k, v, causal=True)
    o.float().sum().backward()
    assert q.grad.shape == q.shape and k.grad.shape == k.shape and v.grad.shape == v.shape
    assert all(torch.isfinite(t.grad.float()).all() for t in (q, k, v))


def test_grouped_query_fp8pv_and_chunks_match_repeated_layout():
    """The FP8 P.V path and the ring-step chunk form read broadcast K/V like
    the forward: bit-identical to the same calls on materialised repeats."""
    B, H, Hkv, N, d = 1, 4, 1, 4608, 128
    q, k, v = _inputs(B, H, Hkv, N, d, False, seed=23)
    krep, vrep = (t.repeat_interleave(H // Hkv, dim=1).contiguous() for t in (k, v))
    o8 = clis.attention(q, k, v, pv="fp8")
    o8r = clis.attention(q, krep, vrep, pv="fp8")
    torch.cuda.synchronize()
    assert torch.equal(o8, o8r)
    qf, kf, vf, _ = clis.grouped_query_views(q, k, v)
    sl2 = clis.scale_log2_for(d)
    outs = []
    for kk, vv, qq in ((kf, vf, qf), (krep.view(B * Hkv, H // Hkv, N, d), vrep.view(B * Hkv, H // Hkv, N, d), qf)):
        mu = torch.empty(B * H * N, device=q.device)
        kbar, certs = clis.clis_certify(qq, kk, vv, sl2, mu=mu)
        o_acc = torch.empty((B * H * N, d), device=q.device)
        l_acc = torch.empty(B * H * N, device=q.device)
        m_acc = torch.empty(B * H * N, device=q.device)
        for i, (a, b) in enumerate(((0, 2048), (2048, N))):
            clis.clis_attn_fwd_chunk(qq, kk[:, :, a:b], vv[:, :, a:b], sl2, o_acc, l_acc, m_acc, kbar=kbar,
                                     certs=certs, first=(i == 0), mu=mu)
        outs.append(clis.clis_attn_chunk_finalize(qq, o_acc, l_acc, m_acc))
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])
