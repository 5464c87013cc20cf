"""Per-prefix certificates of causal heads (clis_certify_tiles) and the causal
forward that uses them (clis_attn_fwd_tiles), against the oracle.

Causal-LLM-shaped heads get their last 100 keys scaled by 8 in some heads:
those heads fail the per-head certificate, while every query block whose
prefix ends before the scaled keys still certifies.  Checked: the per-head
certificates and the per-block flags bit-exact against the oracle (blocks in
the oracle's rounding band excluded), the output against the oracle, and that
each block took the path its flag names (bit-identical to the forced
certified or the online kernel on that block's rows).
"""
import dataclasses
import os

import numpy as np
import pytest
import torch

import oracle
from certified_fixed_stabilizer_gb300 import clis
from certified_fixed_stabilizer_gb300.workloads import WORKLOADS, injected_heads_present, make_inputs, sample_rows
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


def _inputs(N, seed, d=128, dtype=torch.bfloat16):
    w = dataclasses.replace(WORKLOADS["causal"], B=2, d=d)
    q, k, v = make_inputs(w, device=need_gpu(), N=N, H=4, seed=seed, dtype=dtype)
    k = k.clone()
    k[:, 1::2, N - 100:] *= 8  # heads 1 and 3 of each batch: large keys at the end
    return w, q, k.contiguous(), v


@pytest.mark.parametrize("N", [2048, 1000])
def test_tile_certificates_match_oracle(N):
    w, q, k, v = _inputs(N, seed=70 + N)
    sl2 = clis.scale_log2_for(w.d)
    kbar, certs, tiles = clis.clis_certify_tiles(q, k, v, sl2)
    kbar2, certs2 = clis.clis_certify(q, k, v, sl2)
    torch.cuda.synchronize()
    assert torch.equal(certs, certs2) and torch.equal(kbar, kbar2)  # same pass, same per-head result
    ocert, oband, oB = oracle.certify_prefix_tiles(q.cpu(), k.cpu(), v.cpu(), sl2)
    _, heads = oracle.certify(q.cpu(), k.cpu(), v.cpu(), sl2)
    g = tiles.cpu().numpy().astype(np.int32)
    assert g.shape == ocert.shape
    keep = oband == 0
    np.testing.assert_array_equal(g[keep], ocert[keep])
    for h, (gc, oc) in enumerate(zip(clis.decode_certs(certs), heads)):
        if not oc["band"]:
            assert gc["certified"] == oc["certified"], h
        if gc["certified"]:
            assert g[h].all(), h  # a certified head certifies every block
    # the scaled heads fail as heads but keep their early blocks
    failed = [h for h, c in enumerate(heads) if not c["certified"]]
    assert failed and all(g[h, 0] == 1 and g[h, -1] == 0 for h in failed)


def test_tile_certified_forward_takes_each_blocks_path():
    N = 2048
    w, q, k, v = _inputs(N, seed=81)
    sl2 = clis.scale_log2_for(w.d)
    mu = torch.empty(q.shape[0] * q.shape[1] * N, dtype=torch.float32, device=q.device)
    kbar, certs, tiles = clis.clis_certify_tiles(q, k, v, sl2, mu=mu)
    o = clis.clis_attn_fwd_tiles(q, k, v, sl2, kbar, certs, tiles, mu=mu)
    forced = clis.clis_attn_fwd(q, k, v, sl2, kbar=kbar, certs=certs, causal=True, variant="certified", mu=mu)
    online = clis.clis_attn_fwd(q, k, v, sl2, kbar=kbar, certs=certs, causal=True, variant="online")
    torch.cuda.synchronize()
    ref = oracle.attention(flat(q).cpu(), flat(k).cpu(), flat(v).cpu(), w.softmax_scale(), causal=True)
    assert_close_to_oracle(flat(o).float().cpu().numpy(), ref, f"causal N={N} with per-prefix certificates")
    of, ff, nf = flat(o), flat(forced), flat(online)
    t = tiles.cpu().numpy()
    n_fixed = 0
    for h in range(t.shape[0]):
        for b in range(t.shape[1]):
            rows = slice(256 * b, min(N, 256 * (b + 1)))
            want = ff if t[h, b] else nf
            assert torch.equal(of[h, rows], want[h, rows]), (h, b, int(t[h, b]))
            n_fixed += int(t[h, b])
    heads_cert = sum(c["certified"] for c in clis.decode_certs(certs))
    # more blocks run certified than the per-head decision alone would allow
    assert n_fixed > heads_cert * t.shape[1]


def test_fp16_tiles_respect_the_fp16_budget():
    """FP16 data: blocks take the fixed stabiliser only under a budget C <= 15
    (certification with the FP16 exp2 format); with a BF16-format certificate the
    tile flags are ignored and the output equals the online kernel's."""
    N = 1024
    w, q, k, v = _inputs(N, seed=91, dtype=torch.float16)
    q = q * 0.25  # exact in binary16; keeps the early blocks' bounds under 2^15
    sl2 = clis.scale_log2_for(w.d)
    online = clis.clis_attn_fwd(q, k, v, sl2, causal=True, variant="online")
    kb, cs, tl = clis.clis_certify_tiles(q, k, v, sl2, exp_fmt="bf16")
    # heads whose bound exceeds the FP16 limit: neither their BF16-budget head
    # certificate nor their block flags may put them on the fixed stabiliser
    guarded = [h for h, c in enumerate(clis.decode_certs(cs)) if c["B_h"] > 15]
    o = clis.clis_attn_fwd_tiles(q, k, v, sl2, kb, cs, tl)
    torch.cuda.synchronize()
    assert guarded and tl.cpu().numpy()[guarded].any()
    for h in guarded:
        assert torch.equal(flat(o)[h], flat(online)[h])
    kb16, cs16, tl16 = clis.clis_certify_tiles(q, k, v, sl2, exp_fmt="fp16")
    o16 = clis.clis_attn_fwd_tiles(q, k, v, sl2, kb16, cs16, tl16)
    torch.cuda.synchronize()
    failed16 = [h for h, c in enumerate(clis.decode_certs(cs16)) if not c["certified"]]
    assert failed16 and tl16.cpu().numpy()[failed16, 0].all()  # FP16 budget: early blocks still certify
    ref = oracle.attention(flat(q).cpu(), flat(k).cpu(), flat(v).cpu(), w.softmax_scale(), causal=True)
    assert_close_to_oracle(flat(o16).float().cpu().numpy(), ref, "fp16 causal with per-prefix certificates")


def test_causal_late_workload_full_size():
    """The bench's causal workload with late large keys in 32 of 128 heads, at full
    size: block flags bit-exact against the oracle, the injected heads keep most
    of their blocks, and sampled output rows match the oracle."""
    w = WORKLOADS["causal_late"]
    q, k, v = make_inputs(w, device=need_gpu())
    sl2 = clis.scale_log2_for(w.d)
    mu = torch.empty(w.heads * w.N, dtype=torch.float32, device=q.device)
    kbar, certs, tiles = clis.clis_certify_tiles(q, k, v, sl2, mu=mu)
    o = clis.clis_attn_fwd_tiles(q, k, v, sl2, kbar, certs, tiles, mu=mu)
    torch.cuda.synchronize()
    ocert, oband, _ = oracle.certify_prefix_tiles(q.cpu(), k.cpu(), v.cpu(), sl2)
    g = tiles.cpu().numpy().astype(np.int32)
    keep = oband == 0
    np.testing.assert_array_equal(g[keep], ocert[keep])
    injected = injected_heads_present(w)
    dc = clis.decode_certs(certs)
    assert len(injected) == 32 and not any(dc[h]["certified"] for h in injected)
    assert all(g[h, :-1].all() and g[h, -1] == 0 for h in injected)  # only the last block holds the large keys
    rows = sample_rows(w.N, 24, seed=7)
    ref = oracle.attention(flat(q).cpu(), flat(k).cpu(), flat(v).cpu(), w.softmax_scale(), causal=True, rows=rows)
    assert_close_to_oracle(flat(o)[:, rows].float().cpu().numpy(), ref, "causal_late with per-prefix certificates")


@pytest.mark.parametrize("N", [1, 255, 256, 257, 513])
def test_tiles_degenerate_and_ragged_sizes(N):
    """One block (N = 1, 255, 256), a second block of a single row (257) and a
    ragged third block (513): flags bit-exact against the oracle, and the output
    of the per-prefix forward against the oracle."""
    w = dataclasses.replace(WORKLOADS["causal"], B=2)
    q, k, v = make_inputs(w, device=need_gpu(), N=N, H=3, seed=200 + N)
    k = k.clone()
    k[:, 1, -1:] *= 64  # head 1 of each batch: its last key is far out
    k = k.contiguous()
    sl2 = clis.scale_log2_for(w.d)
    kbar, certs, tiles = clis.clis_certify_tiles(q, k, v, sl2)
    o = clis.clis_attn_fwd_tiles(q, k, v, sl2, kbar, certs, tiles)
    torch.cuda.synchronize()
    assert tiles.shape == (6, -(-N // 256))
    ocert, oband, _ = oracle.certify_prefix_tiles(q.cpu(), k.cpu(), v.cpu(), sl2)
    g = tiles.cpu().numpy().astype(np.int32)
    keep = oband == 0
    np.testing.assert_array_equal(g[keep], ocert[keep])
    ref = oracle.attention(flat(q).cpu(), flat(k).cpu(), flat(v).cpu(), w.softmax_scale(), causal=True)
    assert_close_to_oracle(flat(o).float().cpu().numpy(), ref, f"causal N={N} with per-prefix certificates")
