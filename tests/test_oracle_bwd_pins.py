"""Pins for the oracle's attention backward (no GPU needed).

The gradients are checked against things other than the backward code:
numerical differentiation of the forward oracle (itself pinned by
tests/test_oracle_pins.py) in fp64, a 40-digit mpmath differentiation of an
independently written loss, closed forms (one key, identical keys, the first
causal row, the last causal key) and identities (sum over keys of dK is zero,
key-shift invariance).  A dropped D_i term, a wrong sign, a missing scale, a
transposed mask or a swapped operand fails at least one of them.
"""
import numpy as np
import pytest
import torch


def _rand(rng, *shape, scale=1.0):
    return rng.standard_normal(shape) * scale


def _loss(oracle_mod, q, k, v, g, scale, causal):
    return float(np.sum(oracle_mod.attention(q, k, v, scale, causal=causal) * g))


@pytest.mark.parametrize("causal,shape", [(False, (2, 6, 9, 8)), (True, (2, 7, 7, 8)), (False, (1, 1, 5, 3))])
def test_gradients_match_finite_differences(oracle_mod, causal, shape):
    BH, Nq, Nk, d = shape
    rng = np.random.default_rng(5 + Nq)
    q, g = _rand(rng, BH, Nq, d), _rand(rng, BH, Nq, d)
    k, v = _rand(rng, BH, Nk, d, scale=0.8), _rand(rng, BH, Nk, d)
    scale = 0.45
    dq, dk, dv = oracle_mod.attention_bwd(q, k, v, g, scale, causal=causal)
    h = 1e-5
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            old = x[idx]
            x[idx] = old + h
            lp = _loss(oracle_mod, q, k, v, g, scale, causal)
            x[idx] = old - h
            lm = _loss(oracle_mod, q, k, v, g, scale, causal)
            x[idx] = old
            num[idx] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(grad, num, rtol=1e-6, atol=1e-8, err_msg=f"d{name}")


def test_gradients_match_high_precision_differentiation(oracle_mod):
    """Loss written out in mpmath at 40 digits, differentiated numerically by
    mpmath.diff (which refines its step at that precision)."""
    import mpmath
    mpmath.mp.dps = 40
    rng = np.random.default_rng(11)
    Nq, Nk, d, scale = 3, 4, 3, 0.6
    q, g = _rand(rng, 1, Nq, d), _rand(rng, 1, Nq, d)
    k, v = _rand(rng, 1, Nk, d), _rand(rng, 1, Nk, d)
    for causal in (False, True):
        if causal:
            k, v = k[:, :Nq], v[:, :Nq]
        nk = k.shape[1]

        def loss(qm, km, vm):
            tot = mpmath.mpf(0)
            for i in range(Nq):
                keys = range(i + 1) if causal else range(nk)
                w = [mpmath.exp(scale * mpmath.fsum(qm[i][c] * km[j][c] for c in range(d))) for j in keys]
                z = mpmath.fsum(w)
                for c in range(d):
                    oc = mpmath.fsum(wj * vm[j][c] for wj, j in zip(w, keys)) / z
                    tot += mpmath.mpf(float(g[0, i, c])) * oc
            return tot

        base = [[[mpmath.mpf(float(t[0, r, c])) for c in range(d)] for r in range(t.shape[1])] for t in (q, k, v)]
        dq, dk, dv = oracle_mod.attention_bwd(q, k, v, g, scale, causal=causal)
        for which, grad in enumerate((dq, dk, dv)):
            for r in range(grad.shape[1]):
                for c in range(d):
                    def f(x, which=which, r=r, c=c):
                        args = [[row[:] for row in m] for m in base]
                        args[which][r][c] = x
                        return loss(*args)
                    ref = float(mpmath.diff(f, base[which][r][c]))
                    assert abs(grad[0, r, c] - ref) <= 1e-12 * max(1.0, abs(ref)), (causal, which, r, c)


def test_single_key_has_no_query_or_key_gradient(oracle_mod):
    rng = np.random.default_rng(2)
    q, g = _rand(rng, 2, 5, 4), _rand(rng, 2, 5, 4)
    k, v = _rand(rng, 2, 1, 4), _rand(rng, 2, 1, 4)
    dq, dk, dv = oracle_mod.attention_bwd(q, k, v, g, 0.9)
    assert np.all(dq == 0.0) and np.all(dk == 0.0)
    np.testing.assert_allclose(dv[:, 0], g.sum(axis=1), rtol=0, atol=1e-13)


def test_identical_keys_give_uniform_weights(oracle_mod):
    rng = np.random.default_rng(3)
    Nk = 6
    q, g = _rand(rng, 1, 4, 5), _rand(rng, 1, 4, 5)
    k = np.repeat(_rand(rng, 1, 1, 5), Nk, axis=1)
    v = _rand(rng, 1, Nk, 5)
    dq, dk, dv = oracle_mod.attention_bwd(q, k, v, g, 0.7)
    np.testing.assert_allclose(dq, 0.0, atol=1e-13)
    for j in range(Nk):
        np.testing.assert_allclose(dv[0, j], g[0].sum(axis=0) / Nk, atol=1e-13)
    # With equal keys every row's weights are 1/Nk, so dK_j = scale/Nk * sum_i (dO_i.v_j - D_i) q_i.
    D = np.einsum("ic,jc->ij", g[0], v[0]).mean(axis=1)
    for j in range(Nk):
        ref = 0.7 / Nk * ((g[0] @ v[0, j]) - D) @ q[0]
        np.testing.assert_allclose(dk[0, j], ref, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_key_gradients_sum_to_zero(oracle_mod, causal):
    """Each row of the softmax Jacobian times dP sums to zero, so sum_j dK_j = 0."""
    rng = np.random.default_rng(4)
    q, g = _rand(rng, 3, 40, 16), _rand(rng, 3, 40, 16)
    k, v = _rand(rng, 3, 40, 16, scale=1.5), _rand(rng, 3, 40, 16)
    _, dk, _ = oracle_mod.attention_bwd(q, k, v, g, 0.3, causal=causal)
    assert np.abs(dk.sum(axis=1)).max() <= 1e-12 * np.abs(dk).max() * 40


def test_key_shift_leaves_gradients_unchanged(oracle_mod):
    rng = np.random.default_rng(6)
    q, g = _rand(rng, 2, 12, 8), _rand(rng, 2, 12, 8)
    k, v = _rand(rng, 2, 15, 8), _rand(rng, 2, 15, 8)
    a = oracle_mod.attention_bwd(q, k, v, g, 0.5)
    b = oracle_mod.attention_bwd(q, k + _rand(rng, 2, 1, 8, scale=3.0), v, g, 0.5)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, rtol=1e-10, atol=1e-12)


def test_causal_first_row_and_last_key(oracle_mod):
    """Row 0 sees only key 0 (weight 1): dQ_0 = 0.  Key N-1 is seen only by
    row N-1: dV_{N-1} = P_{N-1,N-1} dO_{N-1}."""
    rng = np.random.default_rng(7)
    N, d, scale = 9, 6, 0.8
    q, g = _rand(rng, 1, N, d), _rand(rng, 1, N, d)
    k, v = _rand(rng, 1, N, d), _rand(rng, 1, N, d)
    dq, dk, dv = oracle_mod.attention_bwd(q, k, v, g, scale, causal=True)
    assert np.all(dq[0, 0] == 0.0)
    s = scale * (k[0] @ q[0, N - 1])
    p_last = np.exp(s[-1] - s.max()) / np.exp(s - s.max()).sum()
    np.testing.assert_allclose(dv[0, N - 1], p_last * g[0, N - 1], rtol=1e-12)
    # Masking the wrong side would give key 0 the gradient of row 0 alone.
    assert np.abs(dv[0, 0] - g[0, 0]).max() > 1e-3


@pytest.mark.parametrize("fmt", ["bf16", "fp16"])
def test_half_precision_inputs_decode_exactly(oracle_mod, fmt):
    dt = torch.bfloat16 if fmt == "bf16" else torch.float16
    gen = torch.Generator().manual_seed(8)
    q, k, v, g = (torch.randn(2, 1, 10, 8, generator=gen).to(dt) for _ in range(4))
    got = oracle_mod.attention_bwd(q, k, v, g, 0.35, causal=True)
    ref = oracle_mod.attention_bwd(*(t.double().numpy().reshape(2, 10, 8) for t in (q, k, v, g)), 0.35, causal=True)
    for x, y in zip(got, ref):
        np.testing.assert_array_equal(x, y)


def test_no_queries_gives_zero_key_gradients(oracle_mod):
    rng = np.random.default_rng(9)
    q, g = np.zeros((1, 0, 4)), np.zeros((1, 0, 4))
    k, v = _rand(rng, 1, 3, 4), _rand(rng, 1, 3, 4)
    dq, dk, dv = oracle_mod.attention_bwd(q, k, v, g, 1.0)
    assert dq.shape == (1, 0, 4) and np.all(dk == 0.0) and np.all(dv == 0.0)


def test_backward_rejects_bad_arguments(oracle_mod):
    rng = np.random.default_rng(10)
    q = _rand(rng, 1, 4, 4)
    k = _rand(rng, 1, 5, 4)
    with pytest.raises(ValueError):
        oracle_mod.attention_bwd(q, k, k, q, 1.0, causal=True)  # causal needs Nq == Nk
    with pytest.raises(ValueError):
        oracle_mod.attention_bwd(q, k[:, :0], k[:, :0], q, 1.0)  # no keys
    with pytest.raises(ValueError):
        oracle_mod.attention_bwd(q, k, k, q[:, :3], 1.0)  # do shape


@pytest.mark.parametrize("causal", [False, True])
def test_dq_rows_equal_full_backward_rows(oracle_mod, causal):
    """The row-sampled dQ routine (used at sizes the full backward cannot
    reach) reproduces the pinned full backward's dQ rows exactly."""
    rng = np.random.default_rng(12)
    q, g = _rand(rng, 2, 23, 8), _rand(rng, 2, 23, 8)
    k, v = _rand(rng, 2, 23, 8), _rand(rng, 2, 23, 8)
    dq, _, _ = oracle_mod.attention_bwd(q, k, v, g, 0.4, causal=causal)
    rows = [0, 5, 22, 11]
    got = oracle_mod.attention_bwd_dq_rows(q, k, v, g, 0.4, rows, causal=causal)
    np.testing.assert_allclose(got, dq[:, rows], rtol=1e-13, atol=1e-15)
    tq, tk, tv, tg = (torch.from_numpy(t.astype(np.float32)).to(torch.bfloat16) for t in (q, k, v, g))
    got16 = oracle_mod.attention_bwd_dq_rows(tq, tk, tv, tg, 0.4, rows, causal=causal)
    ref16, _, _ = oracle_mod.attention_bwd(tq, tk, tv, tg, 0.4, causal=causal)
    np.testing.assert_allclose(got16, ref16[:, rows], rtol=1e-13, atol=1e-15)
