"""Many short work tiles: hundreds of heads of a few hundred tokens.

Each persistent CTA then runs several rounds of work tiles with one or two KV
steps each, so barrier phases, the alternating KV sweep direction of odd
rounds and the hand-over of TMEM and shared-memory slots between tiles are
exercised thousands of times per launch (the dedicated parity tests have at
most a few rounds).  Outputs are checked head by head against the fp64 oracle
(every head, all rows), for every forward variant, the KV-chunk form and the
backward.
"""
import dataclasses
import os

import numpy as np
import pytest
import torch

import oracle
from certified_fixed_stabilizer_gb300 import clis
from certified_fixed_stabilizer_gb300.workloads import WORKLOADS, make_dout, make_inputs
from gpu_util import assert_close_to_oracle, assert_grads_close, flat, need_gpu

pytestmark = pytest.mark.gpu

B, H = 8, 40  # 320 heads; one or two 256-row work tiles each


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


def _inputs(causal, N, seed):
    w = dataclasses.replace(WORKLOADS["causal" if causal else "480p"], B=B)
    q, k, v = make_inputs(w, device=need_gpu(), N=N, H=H, seed=seed)
    return w, q, k, v


@pytest.mark.parametrize("causal,N", [(False, 200), (False, 300), (True, 300)])
@pytest.mark.parametrize("variant", ["auto", "online", "online_lazy"])
def test_forward_many_short_tiles(causal, N, variant):
    w, q, k, v = _inputs(causal, N, seed=31 + N)
    o = clis.attention(q, k, v, causal=causal, variant=variant)
    torch.cuda.synchronize()
    ref = oracle.attention(flat(q).cpu(), flat(k).cpu(), flat(v).cpu(), w.softmax_scale(), causal=causal)
    assert_close_to_oracle(flat(o).float().cpu().numpy(), ref, f"{B}x{H} heads N={N} causal={causal} {variant}")


def test_chunked_forward_many_short_tiles():
    N = 300
    w, q, k, v = _inputs(False, N, seed=41)
    sl2 = clis.scale_log2_for(w.d)
    BH = B * H
    dev = q.device
    mu = torch.empty(BH * N, dtype=torch.float32, device=dev)
    kbar, certs = clis.clis_certify(q, k, v, sl2, mu=mu)
    o_acc = torch.empty((BH * N, w.d), dtype=torch.float32, device=dev)
    l_acc = torch.empty(BH * N, dtype=torch.float32, device=dev)
    m_acc = torch.empty(BH * N, dtype=torch.float32, device=dev)
    for i, (a, b) in enumerate(((0, 104), (104, 232), (232, N))):
        clis.clis_attn_fwd_chunk(q, k[:, :, a:b], v[:, :, a:b], sl2, o_acc, l_acc, m_acc, kbar=kbar, certs=certs,
                                 first=(i == 0), mu=mu)
    o = clis.clis_attn_chunk_finalize(q, o_acc, l_acc, m_acc)
    torch.cuda.synchronize()
    ref = oracle.attention(flat(q).cpu(), flat(k).cpu(), flat(v).cpu(), w.softmax_scale())
    assert_close_to_oracle(flat(o).float().cpu().numpy(), ref, f"{B}x{H} heads N={N} KV in 3 chunks")


@pytest.mark.parametrize("causal", [False, True])
def test_backward_many_short_tiles(causal):
    N = 300
    w, q, k, v = _inputs(causal, N, seed=51)
    do = make_dout(q.shape, device=q.device, seed=51)
    o, lse2 = clis.attention_fwd_lse(q, k, v, causal=causal)
    dq, dk, dv = clis.attention_bwd(q, k, v, o, do, lse2, causal=causal)
    torch.cuda.synchronize()
    refs = oracle.attention_bwd(flat(q).cpu(), flat(k).cpu(), flat(v).cpu(), flat(do).cpu(), w.softmax_scale(),
                                causal=causal)
    what = f"backward {B}x{H} heads N={N} causal={causal}"
    for g, r, name in zip((dq, dk, dv), refs, ("dq", "dk", "dv")):
        assert_grads_close(flat(g).float().cpu().numpy(), r, name, what)
