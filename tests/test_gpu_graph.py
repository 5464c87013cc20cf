"""The library's calls captured in a CUDA graph.

Every entry point is asynchronous on the given stream and allocates no device
memory, so certify + forward, the KV-chunk form and the backward can be
captured once and replayed.  A replay on new inputs written into the captured
buffers must give results bit-identical to eager calls on the same inputs (the
kernels are deterministic), and the eager results are checked against the
oracle, so the graph path inherits their parity.
"""
import dataclasses
import os

import numpy as np
import pytest
import torch

import oracle
from certified_fixed_stabilizer_gb300 import clis
from certified_fixed_stabilizer_gb300.workloads import WORKLOADS, make_dout, make_inputs
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


def _capture(fn):
    """Warm up on a side stream, then capture fn() into a graph; returns (graph, outputs)."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        outs = fn()
    return g, outs


def _inputs(name, seed, N, H):
    w = WORKLOADS[name]
    w = dataclasses.replace(w, B=min(w.B, 2))
    return w, make_inputs(w, device=need_gpu(), seed=seed, N=N, H=H)


@pytest.mark.parametrize("name,causal", [("480p", False), ("mixed", False), ("causal", True)])
def test_certify_and_forward_replay_bit_identical(name, causal):
    N, H = 1000, 4
    w, (q, k, v) = _inputs(name, 1, N, H)
    sl2 = clis.scale_log2_for(w.d)
    BH = q.shape[0] * q.shape[1]
    kbar = torch.empty((BH, w.d), dtype=torch.float32, device=q.device)
    certs = torch.empty((BH, clis.CERT_WORDS), dtype=torch.int32, device=q.device)
    mu = torch.empty(BH * N, dtype=torch.float32, device=q.device)
    lse2 = torch.empty(BH * N, dtype=torch.float32, device=q.device)
    o = torch.empty_like(q)

    def step():
        clis.clis_certify(q, k, v, sl2, kbar=kbar, certs=certs, mu=mu)
        clis.clis_attn_fwd(q, k, v, sl2, kbar=kbar, certs=certs, causal=causal, out=o, lse2=lse2, mu=mu)
        return o

    g, _ = _capture(step)
    for seed in (2, 3):
        _, (q2, k2, v2) = _inputs(name, seed, N, H)
        q.copy_(q2), k.copy_(k2), v.copy_(v2)
        g.replay()
        torch.cuda.synchronize()
        got_o, got_l, got_c = o.clone(), lse2.clone(), certs.clone()
        step()  # eager on the same buffers
        torch.cuda.synchronize()
        assert torch.equal(got_c, certs)
        assert torch.equal(got_o, o), f"{name} seed {seed}: replayed O differs from eager"
        assert torch.equal(got_l, lse2)
        ref = oracle.attention(flat(q).cpu(), flat(k).cpu(), flat(v).cpu(), w.softmax_scale(), causal=causal)
        assert_close_to_oracle(flat(got_o).float().cpu().numpy(), ref, f"graph {name} seed {seed}")


def test_chunked_forward_replay_bit_identical():
    """Certify + three KV chunks + finalize, captured as one graph."""
    N, H = 900, 3
    w, (q, k, v) = _inputs("mixed", 4, N, H)
    sl2 = clis.scale_log2_for(w.d)
    BH = q.shape[0] * q.shape[1]
    dev = q.device
    kbar = torch.empty((BH, w.d), dtype=torch.float32, device=dev)
    certs = torch.empty((BH, clis.CERT_WORDS), dtype=torch.int32, device=dev)
    mu = torch.empty(BH * N, dtype=torch.float32, device=dev)
    o_acc = torch.empty((BH * N, w.d), dtype=torch.float32, device=dev)
    l_acc = torch.empty(BH * N, dtype=torch.float32, device=dev)
    m_acc = torch.empty(BH * N, dtype=torch.float32, device=dev)
    o = torch.empty_like(q)
    bounds = [0, 296, 600, N]

    def step():
        clis.clis_certify(q, k, v, sl2, kbar=kbar, certs=certs, mu=mu)
        for i, (a, b) in enumerate(zip(bounds[:-1], bounds[1:])):
            clis.clis_attn_fwd_chunk(q, k[:, :, a:b], v[:, :, a:b], sl2, o_acc, l_acc, m_acc, kbar=kbar,
                                     certs=certs, first=(i == 0), mu=mu)
        clis.clis_attn_chunk_finalize(q, o_acc, l_acc, m_acc, out=o)
        return o

    g, _ = _capture(step)
    _, (q2, k2, v2) = _inputs("mixed", 5, N, H)
    q.copy_(q2), k.copy_(k2), v.copy_(v2)
    g.replay()
    torch.cuda.synchronize()
    got = o.clone()
    step()
    torch.cuda.synchronize()
    assert torch.equal(got, o)
    ref = oracle.attention(flat(q).cpu(), flat(k).cpu(), flat(v).cpu(), w.softmax_scale())
    assert_close_to_oracle(flat(got).float().cpu().numpy(), ref, "graph chunked")


def test_backward_replay_bit_identical():
    N, H = 700, 2
    w, (q, k, v) = _inputs("causal", 6, N, H)
    do = make_dout(q.shape, device=q.device, seed=6)
    bufs = {}

    def step():
        o, lse2 = clis.attention_fwd_lse(q, k, v, causal=True)
        dq, dk, dv = clis.attention_bwd(q, k, v, o, do, lse2, causal=True)
        bufs.update(o=o, dq=dq, dk=dk, dv=dv)
        return dq, dk, dv

    g, (dq, dk, dv) = _capture(step)
    _, (q2, k2, v2) = _inputs("causal", 7, N, H)
    q.copy_(q2), k.copy_(k2), v.copy_(v2)
    do.copy_(make_dout(q.shape, device=q.device, seed=7))
    g.replay()
    torch.cuda.synchronize()
    got = [t.clone() for t in (dq, dk, dv)]
    ref = step()
    torch.cuda.synchronize()
    for a, b, name in zip(got, ref, ("dq", "dk", "dv")):
        assert torch.equal(a, b), f"replayed {name} differs from eager"
    assert np.isfinite(torch.stack([t.float().abs().max() for t in got]).cpu().numpy()).all()
