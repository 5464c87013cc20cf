"""GPU attention backward vs the fp64 oracle, through the C ABI.

The GPU side runs its own forward (certify + fused kernel, giving O and
lse2) and then clis_attn_bwd; the oracle computes the exact gradients of
sum(dO * O) from q, k, v and dO alone.  Bounds per head and gradient are in
gpu_util.GRAD_TOL (derived in tests/test_bwd_tolerance.py).
"""
import dataclasses
import os

import numpy as np
import pytest
import torch

import oracle
from certified_fixed_stabilizer_gb300 import clis
from certified_fixed_stabilizer_gb300.workloads import WORKLOADS, make_dout, make_inputs
from gpu_util import assert_grads_close, flat, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    need_gpu()
    oracle.set_num_threads(os.cpu_count() or 1)
    clis.clis_clear_device_error()
    yield


@pytest.fixture(autouse=True)
def _device_error_word_stays_clear():
    """Every test must leave the kernels' error word at 0 (no wait ran out)."""
    yield
    code = clis.clis_get_device_error()
    clis.clis_clear_device_error()
    assert code == 0, f"device error word {code:#x}"


def _inputs(B, H, Nq, Nk, d, causal, dtype=torch.bfloat16, seed=0):
    """Workload distributions: the causal-LLM recipe for causal cases, the DiT
    recipe otherwise (the tiny workload's recipe for d = 64)."""
    dev = need_gpu()
    w = WORKLOADS["causal" if causal else ("480p" if d == 128 else "tiny")]
    w = dataclasses.replace(w, B=B, d=d)
    q, k, v = make_inputs(w, device=dev, seed=seed, N=Nq, H=H, dtype=dtype)
    if Nk != Nq:
        _, k, v = make_inputs(w, device=dev, seed=seed + 1, N=Nk, H=H, dtype=dtype)
    do = make_dout(q.shape, device=dev, seed=seed, dtype=dtype)
    return q, k, v, do


def _gpu_grads(q, k, v, do, causal, variant="auto"):
    o, lse2 = clis.attention_fwd_lse(q, k, v, causal=causal, variant=variant)
    dq, dk, dv = clis.attention_bwd(q, k, v, o, do, lse2, causal=causal)
    torch.cuda.synchronize()
    return dq, dk, dv


def _check(got, q, k, v, do, causal, what):
    ref = oracle.attention_bwd(q.cpu(), k.cpu(), v.cpu(), do.cpu(), q.shape[-1] ** -0.5, causal=causal)
    for g, r, name in zip(got, ref, ("dq", "dk", "dv")):
        assert_grads_close(flat(g).float().cpu().numpy(), r, name, what)


CASES = [
    # B, H, Nq, Nk, d, causal
    (1, 2, 300, 300, 64, True),
    (1, 2, 300, 300, 64, False),
    (1, 2, 700, 700, 128, True),      # several tiles, ragged tail
    (2, 1, 517, 389, 128, False),     # Nq != Nk, both ragged
    (1, 1, 128, 128, 128, True),      # one tile, diagonal only
    (2, 2, 333, 333, 128, True),
    (1, 2, 1, 257, 128, False),       # one query row
    (1, 1, 1000, 129, 64, False),     # one key past a full tile
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal", CASES)
def test_backward_matches_oracle(B, H, Nq, Nk, d, causal):
    q, k, v, do = _inputs(B, H, Nq, Nk, d, causal)
    _check(_gpu_grads(q, k, v, do, causal), q, k, v, do, causal, f"bwd {B}x{H}x{Nq}x{Nk}x{d} c={causal}")


def test_backward_alone_from_oracle_forward():
    """O and lse2 from the oracle (rounded as the forward would emit them):
    isolates the backward kernels from the forward."""
    q, k, v, do = _inputs(1, 2, 640, 640, 128, True, seed=3)
    ref_o, ref_lse2 = oracle.attention(q.cpu(), k.cpu(), v.cpu(), q.shape[-1] ** -0.5, causal=True, with_lse2=True)
    o = torch.from_numpy(ref_o).float().reshape(q.shape).to(torch.bfloat16).to(q.device)
    lse2 = torch.from_numpy(ref_lse2).float().reshape(-1).to(q.device)
    got = clis.attention_bwd(q, k, v, o, do, lse2, causal=True)
    torch.cuda.synchronize()
    _check(got, q, k, v, do, True, "bwd from oracle O, lse2")


@pytest.mark.parametrize("variant", ["online", "online_lazy", "certified"])
def test_backward_after_each_forward_path(variant):
    """lse2 is the same row statistic on every forward path."""
    q, k, v, do = _inputs(1, 2, 520, 520, 128, True, seed=5)
    _check(_gpu_grads(q, k, v, do, True, variant), q, k, v, do, True, f"bwd after {variant}")


@pytest.mark.parametrize("d,causal", [(128, True), (64, True), (64, False)])
def test_backward_fp16(d, causal):
    q, k, v, do = _inputs(1, 2, 600, 600, d, causal, dtype=torch.float16, seed=7)
    _check(_gpu_grads(q, k, v, do, causal), q, k, v, do, causal, f"bwd fp16 d={d} causal={causal}")


def test_backward_strided_layout():
    """[B, N, H, d] storage viewed as [B, H, N, d]: dq, dk, dv come back with
    the strides of q, k, v."""
    q0, k0, v0, do0 = _inputs(2, 3, 384, 384, 128, False, seed=9)
    q, k, v, do = (t.transpose(1, 2).contiguous().transpose(1, 2) for t in (q0, k0, v0, do0))
    assert q.stride() != q0.stride()
    dq, dk, dv = _gpu_grads(q, k, v, do, False)
    assert dq.stride() == q.stride() and dk.stride() == k.stride() and dv.stride() == v.stride()
    _check((dq, dk, dv), q0, k0, v0, do0, False, "bwd strided")


def test_backward_is_deterministic():
    q, k, v, do = _inputs(1, 4, 900, 900, 128, True, seed=11)
    a = _gpu_grads(q, k, v, do, True)
    b = _gpu_grads(q, k, v, do, True)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_no_queries_gives_zero_key_gradients():
    dev = need_gpu()
    q = torch.empty(1, 2, 0, 128, dtype=torch.bfloat16, device=dev)
    k = torch.randn(1, 2, 200, 128, device=dev).to(torch.bfloat16)
    v = torch.randn(1, 2, 200, 128, device=dev).to(torch.bfloat16)
    dk = torch.full_like(k, 7.0)
    dv = torch.full_like(v, 7.0)
    lse2 = torch.empty(0, dtype=torch.float32, device=dev)
    clis.clis_attn_bwd(q, k, v, q, q, lse2, 0.1, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dk) == 0 and torch.count_nonzero(dv) == 0


def test_autograd_function():
    q, k, v, do = _inputs(1, 2, 400, 400, 64, True, seed=13)
    qr, kr, vr = (t.clone().requires_grad_(True) for t in (q, k, v))
    o = clis.attention_autograd(qr, kr, vr, causal=True)
    o.backward(do)
    torch.cuda.synchronize()
    _check((qr.grad, kr.grad, vr.grad), q, k, v, do, True, "autograd")


def test_causal_full_size_sampled_heads():
    """The causal LLM workload at full size (B=4, H=32, N=8192, d=128): every
    gradient of two seed-chosen heads against the oracle, and for all heads
    the identity sum_j dK_j = 0 (rows of the softmax Jacobian sum to zero)."""
    dev = need_gpu()
    w = WORKLOADS["causal"]
    q, k, v = make_inputs(w, device=dev)
    do = make_dout(q.shape, device=dev)
    dq, dk, dv = _gpu_grads(q, k, v, do, True)
    g = torch.Generator().manual_seed(2024)
    heads = sorted({0, int(torch.randint(1, w.B * w.H, (1,), generator=g))})
    for bh in heads:
        b, h = divmod(bh, w.H)
        sl = (slice(b, b + 1), slice(h, h + 1))
        _check((dq[sl], dk[sl], dv[sl]), q[sl], k[sl], v[sl], do[sl], True, f"causal full-size head {bh}")
    dkf = flat(dk).float()
    colsum = dkf.sum(dim=1).abs().amax(dim=1)
    mag = dkf.abs().sum(dim=1).amax(dim=1)
    assert torch.all(colsum <= 2e-2 * mag), (colsum / mag).max().item()
