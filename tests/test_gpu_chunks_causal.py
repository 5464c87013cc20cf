"""Causal KV-chunk (ring-step) form, clis_attn_fwd_chunk_causal, against the
oracle (CLiS: Table 7's ring columns and Figure 6's ring step, in the causal
setting of Table 3).

The keys and values of each causal head arrive in chunks; each call merges
one chunk into fp32 accumulators, query i seeing chunk key j iff
key_offset + j <= i.  The finalized output must be the oracle's causal
attention over the whole sequence, whatever the split: chunk boundaries inside
a 128-key tile and inside a 256-row query block, a one-key chunk, chunks in
any order after the first.  Certified rows keep their fixed stabiliser in
every chunk (m_acc never changes), so their partials add with no rescaling.
"""
import dataclasses
import os

import numpy as np
import pytest
import torch

import oracle
from certified_fixed_stabilizer_gb300 import clis
from certified_fixed_stabilizer_gb300.workloads import WORKLOADS, make_inputs
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


def _inputs(N, H=4, seed=0, late=False, dtype=torch.bfloat16, d=128):
    w = dataclasses.replace(WORKLOADS["causal"], B=1, d=d)
    q, k, v = make_inputs(w, device=need_gpu(), N=N, H=H, seed=seed, dtype=dtype)
    if late:
        k = k.clone()
        k[:, 1::2, N - 100:] *= 8  # odd heads: large keys at the end, so they fail as heads
        k = k.contiguous()
    return w, q, k, v


def _chunked_causal(q, k, v, bounds, variant, kbar=None, certs=None, tiles=None, order=None, mu=None):
    """Runs the chunks [bounds[i], bounds[i+1]) (first the one at key 0, then
    the others in `order`), finalizes, returns (out, lse2, m_after_first, m_acc)."""
    sl2 = clis.scale_log2_for(q.shape[-1])
    BH, Nq, d = q.shape[0] * q.shape[1], q.shape[2], q.shape[3]
    o_acc = torch.full((BH * Nq, d), float("nan"), device=q.device)
    l_acc = torch.full((BH * Nq,), float("nan"), device=q.device)
    m_acc = torch.full((BH * Nq,), float("nan"), device=q.device)
    chunks = list(zip(bounds[:-1], bounds[1:]))
    order = order or list(range(len(chunks)))
    assert order[0] == 0
    m_first = None
    for n, i in enumerate(order):
        a, b = chunks[i]
        clis.clis_attn_fwd_chunk_causal(q, k[:, :, a:b], v[:, :, a:b], sl2, o_acc, l_acc, m_acc, a, kbar=kbar,
                                        certs=certs, tile_certs=tiles, first=(n == 0), variant=variant, mu=mu)
        if n == 0:
            m_first = m_acc.clone()
    l2 = torch.full((BH * Nq,), float("nan"), device=q.device)
    out = clis.clis_attn_chunk_finalize(q, o_acc, l_acc, m_acc, lse2=l2)
    torch.cuda.synchronize()
    return out, l2, m_first, m_acc


def _oracle(q, k, v):
    return oracle.attention(flat(q).cpu(), flat(k).cpu(), flat(v).cpu(), q.shape[-1] ** -0.5, causal=True,
                            with_lse2=True)


SPLITS = {
    # inside a 128-key tile and a 256-row block; a one-key chunk; a ragged end
    "ragged": [0, 300, 301, 700, 1100, 1500],
    # two chunks split inside the second 128-key tile of the second query block
    "two": [0, 389, 1500],
    # chunk boundaries on 256-row block edges
    "blocks": [0, 256, 512, 1024, 1500],
}


@pytest.mark.parametrize("variant", ["auto", "online", "online_lazy", "certified"])
@pytest.mark.parametrize("split", sorted(SPLITS))
def test_causal_chunks_match_oracle(variant, split):
    w, q, k, v = _inputs(1500, seed=31)
    sl2 = clis.scale_log2_for(w.d)
    kbar, certs = clis.clis_certify(q, k, v, sl2)
    flags = [c["certified"] for c in clis.decode_certs(certs)]
    assert all(flags)
    out, l2, m_first, m_acc = _chunked_causal(q, k, v, SPLITS[split], variant, kbar, certs)
    ref, rlse = _oracle(q, k, v)
    assert_close_to_oracle(flat(out).float().cpu().numpy(), ref, f"causal chunks {split}/{variant}")
    np.testing.assert_allclose(l2.cpu().numpy().reshape(rlse.shape), rlse, atol=2e-3, rtol=0)
    if variant in ("auto", "certified"):
        # The fixed stabiliser written by the first chunk is never changed.
        assert torch.equal(m_first, m_acc)


def test_causal_chunks_in_any_order():
    """After the chunk holding key 0, the other chunks may come in any order
    (each row's rescaling or plain addition does not depend on it)."""
    w, q, k, v = _inputs(1500, seed=32)
    sl2 = clis.scale_log2_for(w.d)
    kbar, certs = clis.clis_certify(q, k, v, sl2)
    ref, _ = _oracle(q, k, v)
    for variant in ("auto", "online"):
        out, _, _, _ = _chunked_causal(q, k, v, SPLITS["ragged"], variant, kbar, certs, order=[0, 4, 2, 3, 1])
        assert_close_to_oracle(flat(out).float().cpu().numpy(), ref, f"causal chunks reversed/{variant}")


def test_causal_single_chunk_is_the_fused_forward():
    """One chunk holding every key, then the finalize: the same tiles, the same
    arithmetic and the same final divide as clis_attn_fwd, bit for bit."""
    w, q, k, v = _inputs(1300, seed=33, late=True)
    sl2 = clis.scale_log2_for(w.d)
    kbar, certs = clis.clis_certify(q, k, v, sl2)
    flags = [c["certified"] for c in clis.decode_certs(certs)]
    assert 0 < sum(flags) < len(flags)
    lse2 = torch.empty(q.shape[0] * q.shape[1] * q.shape[2], device=q.device)
    fused = clis.clis_attn_fwd(q, k, v, sl2, kbar=kbar, certs=certs, causal=True, lse2=lse2)
    out, l2, _, _ = _chunked_causal(q, k, v, [0, 1300], "auto", kbar, certs)
    assert torch.equal(out, fused)
    assert torch.equal(l2, lse2)


def test_causal_chunks_with_per_prefix_certificates():
    """Heads whose last keys are large fail as heads; with the per-prefix flags
    their early query blocks still take the fixed stabiliser in every chunk.
    Output against the oracle; certified blocks' stabilisers never change."""
    w, q, k, v = _inputs(1500, seed=34, late=True)
    sl2 = clis.scale_log2_for(w.d)
    mu = torch.empty(q.shape[0] * q.shape[1] * q.shape[2], device=q.device)
    kbar, certs, tiles = clis.clis_certify_tiles(q, k, v, sl2, mu=mu)
    flags = [c["certified"] for c in clis.decode_certs(certs)]
    assert 0 < sum(flags) < len(flags)
    t = tiles.cpu().numpy()
    failed = [h for h, f in enumerate(flags) if not f]
    assert t[failed].sum() > 0  # some blocks of failed heads certify by their prefix
    out, l2, m_first, m_acc = _chunked_causal(q, k, v, SPLITS["ragged"], "auto", kbar, certs, tiles=tiles, mu=mu)
    ref, rlse = _oracle(q, k, v)
    assert_close_to_oracle(flat(out).float().cpu().numpy(), ref, "causal chunks per-prefix")
    np.testing.assert_allclose(l2.cpu().numpy().reshape(rlse.shape), rlse, atol=2e-3, rtol=0)
    N = q.shape[2]
    mf, ma = m_first.view(-1, N), m_acc.view(-1, N)
    for h in range(t.shape[0]):
        for b in range(t.shape[1]):
            if t[h, b]:
                rows = slice(256 * b, min(N, 256 * b + 256))
                assert torch.equal(mf[h, rows], ma[h, rows]), (h, b)
    # The same flags in one call (clis_attn_fwd_tiles) give the same result
    # within the output tolerance.
    one = clis.clis_attn_fwd_tiles(q, k, v, sl2, kbar, certs, tiles, mu=mu)
    torch.cuda.synchronize()
    assert_close_to_oracle(flat(one).float().cpu().numpy(), ref, "per-prefix fused")


def test_causal_chunks_deterministic_and_fp16():
    w, q, k, v = _inputs(900, seed=35, dtype=torch.float16, d=64)
    sl2 = clis.scale_log2_for(w.d)
    kbar, certs = clis.clis_certify(q, k, v, sl2, exp_fmt="fp16")
    bounds = [0, 129, 400, 401, 900]
    a = _chunked_causal(q, k, v, bounds, "auto", kbar, certs)
    b = _chunked_causal(q, k, v, bounds, "auto", kbar, certs)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    ref, _ = _oracle(q, k, v)
    assert_close_to_oracle(flat(a[0]).float().cpu().numpy(), ref, "causal chunks fp16 d=64")
