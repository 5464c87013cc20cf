"""Pins for the CPU oracle (no GPU needed).

Each test checks the oracle against something other than itself: values
fixed by the floating-point format definitions, hand-built heads whose
certificate is known in closed form, brute-force high-precision evaluation on
tiny inputs, and identities of softmax attention (shift invariance of
Algorithm 1 step 2, N_k = 1, identical keys, dominant key, causal prefix).
A plausible slip in the oracle (a dropped centring, a wrong index range in
the causal mask, a transposed operand, a missing scale) fails at least one.
"""
import math
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

import torch  # noqa: E402


def _bf16(a):
    return torch.tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


# ---------------------------------------------------------------- Figure 3 ----

def test_format_limits_match_golden_and_libraries(oracle_mod):
    for fmt, mx, fl, ce in _read_golden("format_limits.txt"):
        U = oracle_mod.format_log2_max(fmt)
        assert math.floor(U) == int(fl) and math.ceil(U) == int(ce)
        assert abs(2.0 ** U - float(mx)) <= 1e-12 * float(mx)
    # independent library values of the same maxima
    assert abs(2.0 ** oracle_mod.format_log2_max("fp16") - float(np.finfo(np.float16).max)) < 1e-9
    assert abs(2.0 ** oracle_mod.format_log2_max("fp32") / float(np.finfo(np.float32).max) - 1) < 1e-14
    assert abs(2.0 ** oracle_mod.format_log2_max("bf16") / torch.finfo(torch.bfloat16).max - 1) < 1e-14
    assert abs(2.0 ** oracle_mod.format_log2_max("e4m3") - torch.finfo(torch.float8_e4m3fn).max) < 1e-9


def test_exp2_limits_in_each_format(oracle_mod):
    """exp2(floor U) is finite in the format, exp2(floor U + 1) overflows."""
    Uh = math.floor(oracle_mod.format_log2_max("fp16"))
    with np.errstate(over="ignore"):
        assert np.isfinite(np.exp2(np.float16(Uh)))
        assert np.isinf(np.exp2(np.float16(Uh + 1)))
        Uf = math.floor(oracle_mod.format_log2_max("fp32"))
        assert np.isfinite(np.exp2(np.float32(Uf)))
        assert np.isinf(np.exp2(np.float32(Uf + 1)))
    Ub = math.floor(oracle_mod.format_log2_max("bf16"))
    t = torch.exp2(torch.tensor([float(Ub), float(Ub + 1)], dtype=torch.bfloat16))
    assert torch.isfinite(t[0]) and torch.isinf(t[1])
    # E4M3 has no infinity: 2^8 = 256 is exact, 2^9 = 512 lies beyond its largest
    # value 448 (torch's conversion gives NaN there, a saturating one 448).
    U8 = math.floor(oracle_mod.format_log2_max("e4m3"))
    t8 = torch.tensor([2.0 ** U8, 2.0 ** (U8 + 1)]).to(torch.float8_e4m3fn).float()
    assert t8[0].item() == 256.0 and not (abs(t8[1].item()) <= 448.0)


# ------------------------------------------------------- Algorithm 1, 5-7 ----

def test_ceil_log2_count_golden(oracle_mod):
    for n, a in _read_golden("ceil_log2_counts.txt"):
        assert oracle_mod.ceil_log2_count(int(n)) == int(a), n


@pytest.mark.parametrize("m,G", [
    (0.0, 0), (0.5, 0), (1.0, 0), (1.0 + 2.0 ** -7, 1), (2.0, 1), (2.5, 2), (3.0, 2),
    (4.0, 2), (4096.0, 12), (4096.0 * (1 + 2.0 ** -7), 13), (2.0 ** -130, 0),
    (65504.0, 16), (2.0 ** 127, 127),
])
def test_v_exponent_table(oracle_mod, m, G):
    assert oracle_mod.v_exponent(m) == G


def test_exponent_budget_closed_forms(oracle_mod):
    for A in range(0, 60):
        # BF16 exp outputs, FP32 accumulator: min(127, 128 - A - 1) = 127 - A
        assert oracle_mod.exponent_budget("bf16", "fp32", A) == 127 - A
        assert oracle_mod.exponent_budget("fp32", "fp32", A) == 127 - A
        assert oracle_mod.exponent_budget("bf16", "bf16", A) == 127 - A
        assert oracle_mod.exponent_budget("fp16", "fp32", A) == min(15, 127 - A)
        assert oracle_mod.exponent_budget("bf16", "fp16", A) == 15 - A
        assert oracle_mod.exponent_budget("fp16", "fp16", A) == 15 - A
        # E4M3 exp outputs (the FP8 P.V path), FP32 accumulator: min(8, 127 - A)
        assert oracle_mod.exponent_budget("e4m3", "fp32", A) == min(8, 127 - A)


# ------------------------------------------------- hand-built boundary heads ----

def _head(keys, queries, values=None):
    keys = np.asarray(keys, dtype=np.float32)
    queries = np.asarray(queries, dtype=np.float32)
    if values is None:
        values = np.zeros_like(keys)
    q = _bf16(queries)[None]
    k = _bf16(keys)[None]
    v = _bf16(values)[None]
    # the hand-built values must be exact in bf16
    assert np.array_equal(k[0].float().numpy(), keys)
    assert np.array_equal(q[0].float().numpy(), queries)
    return q, k, v


def _pm_keys(d, kappa, offset=0.0):
    """Keys offset +- kappa e_1 (twice): mean exactly `offset`, centred norms exactly kappa."""
    e = np.zeros(d, dtype=np.float32)
    e[0] = kappa
    base = np.full(d, offset, dtype=np.float32)
    return np.stack([base + e, base - e, base + e, base - e])


def test_boundary_head_tie_certifies(oracle_mod):
    d = 64
    q0 = np.zeros(d, dtype=np.float32)
    q0[0] = 2000.0
    q, k, v = _head(_pm_keys(d, 1.0), [q0])
    kbar, certs = oracle_mod.certify(q, k, v, scale_log2=1.0 / 16)
    c = certs[0]
    # N_k = 4 -> ceil(log2) = 2, V = 0 -> G = 0, A = 2, C = 127 - 2 = 125
    assert (c["G"], c["A"], c["C"]) == (0, 2, 125)
    assert c["kappa"] == 1.0 and c["qmax"] == 2000.0 and c["B_h"] == 125.0
    assert c["certified"] == 1 and c["reason"] == 0 and c["band"] == 1
    assert np.all(kbar == 0.0)


def test_boundary_head_just_above_fails(oracle_mod):
    d = 64
    q0 = np.zeros(d, dtype=np.float32)
    q0[0] = 2008.0            # B_h = 125.5 > C = 125
    q, k, v = _head(_pm_keys(d, 1.0), [q0])
    _, certs = oracle_mod.certify(q, k, v, scale_log2=1.0 / 16)
    c = certs[0]
    assert c["B_h"] == 125.5 and c["certified"] == 0 and c["reason"] == 1


def test_boundary_heads_under_the_e4m3_budget(oracle_mod):
    """With E4M3 exp outputs the budget is min(8, 127 - A) = 8: B_h = 8 exactly
    certifies (the tie), B_h = 8.0625 fails, and the same heads certify easily
    under the BF16 budget (C = 125)."""
    d = 64
    for qv, B, ok in ((128.0, 8.0, 1), (129.0, 8.0625, 0)):
        q0 = np.zeros(d, dtype=np.float32)
        q0[0] = qv
        q, k, v = _head(_pm_keys(d, 1.0), [q0])
        _, c8 = oracle_mod.certify(q, k, v, scale_log2=1.0 / 16, exp_fmt="e4m3")
        _, cb = oracle_mod.certify(q, k, v, scale_log2=1.0 / 16)
        assert c8[0]["C"] == 8 and c8[0]["B_h"] == B and c8[0]["certified"] == ok, c8[0]
        assert cb[0]["C"] == 125 and cb[0]["certified"] == 1


def test_centering_is_applied(oracle_mod):
    """Keys offset by a large common vector: kappa must still be exactly 1.
    An oracle that forgot to centre (Alg. 1 step 2) would report ~||offset||."""
    d = 64
    q0 = np.zeros(d, dtype=np.float32)
    q0[0] = 2000.0
    q, k, v = _head(_pm_keys(d, 1.0, offset=3.0), [q0])
    kbar, certs = oracle_mod.certify(q, k, v, scale_log2=1.0 / 16)
    assert certs[0]["kappa"] == 1.0 and certs[0]["certified"] == 1
    assert np.all(kbar == 3.0)


def test_asymmetric_kappa(oracle_mod):
    """Keys {0, 0, 0, 4 e_1}: mean e_1, centred norms 1, 1, 1, 3 -> kappa = 3.
    Query (3, 4, 0, ...) has norm 5, so B_h = scale_log2 * 15."""
    d = 8
    keys = np.zeros((4, d), dtype=np.float32)
    keys[3, 0] = 4.0
    qv = np.zeros((2, d), dtype=np.float32)
    qv[0, :2] = [3.0, 4.0]
    qv[1, :2] = [1.0, 1.0]
    vals = np.zeros((4, d), dtype=np.float32)
    vals[2, 5] = -3.0          # max |V| = 3 -> G = 2
    q, k, v = _head(keys, qv, vals)
    kbar, certs = oracle_mod.certify(q, k, v, scale_log2=0.5)
    c = certs[0]
    assert kbar[0, 0] == 1.0 and np.all(kbar[0, 1:] == 0)
    assert c["kappa"] == 3.0 and c["qmax"] == 5.0 and c["B_h"] == 7.5
    assert (c["G"], c["A"], c["C"]) == (2, 4, 123)
    assert c["vmax"] == 3.0 and c["certified"] == 1


def test_equal_keys_kappa_zero(oracle_mod):
    d = 16
    keys = np.tile(np.linspace(-2, 2, d, dtype=np.float32), (5, 1))
    keys = _bf16(keys).float().numpy()
    q, k, v = _head(keys, np.ones((3, d), dtype=np.float32) * 100)
    _, certs = oracle_mod.certify(q, k, v, scale_log2=1.0)
    assert certs[0]["kappa"] == 0.0 and certs[0]["B_h"] == 0.0 and certs[0]["certified"] == 1


def test_g_from_v_and_budget_shrinks(oracle_mod):
    """V max exactly 2^12 -> G = 12; one ulp above -> 13; C drops accordingly."""
    d = 8
    keys = _pm_keys(d, 1.0)
    for vm, G in [(4096.0, 12), (4128.0, 13), (1.0, 0), (0.75, 0)]:
        vals = np.zeros((4, d), dtype=np.float32)
        vals[1, 3] = -vm
        q, k, v = _head(keys, [np.ones(d, dtype=np.float32)], vals)
        _, certs = oracle_mod.certify(q, k, v, scale_log2=1.0)
        c = certs[0]
        assert c["G"] == G and c["A"] == 2 + G and c["C"] == 125 - G


@pytest.mark.parametrize("where", ["q", "k", "v"])
@pytest.mark.parametrize("bad", [float("nan"), float("inf"), -float("inf")])
def test_nonfinite_inputs_fail(oracle_mod, where, bad):
    d = 8
    keys = _pm_keys(d, 1.0)
    qv = np.ones((2, d), dtype=np.float32)
    vals = np.ones((4, d), dtype=np.float32)
    arrs = {"q": qv, "k": keys, "v": vals}
    arrs[where] = arrs[where].copy()
    arrs[where][1, 2] = bad
    q = _bf16(arrs["q"])[None]
    k = _bf16(arrs["k"])[None]
    v = _bf16(arrs["v"])[None]
    _, certs = oracle_mod.certify(q, k, v, scale_log2=1.0)
    assert certs[0]["certified"] == 0 and certs[0]["reason"] == 2
    assert (certs[0]["G"], certs[0]["A"], certs[0]["C"]) == (0, 0, 0)


def test_fp16_budget_decides(oracle_mod):
    """With FP16 exp outputs, C = min(15, 127 - A): B_h = 15 certifies, 15.5 fails."""
    d = 8
    keys = _pm_keys(d, 1.0)
    for qx, cert in [(15.0, 1), (15.5, 0)]:
        q0 = np.zeros(d, dtype=np.float32)
        q0[0] = qx
        q, k, v = _head(keys, [q0])
        _, c = oracle_mod.certify(q, k, v, scale_log2=1.0, exp_fmt="fp16")
        assert c[0]["C"] == 15 and c[0]["certified"] == cert


# ------------------------------------------------------------ attention ----

def _brute(q, k, v, scale, causal):
    """Unstabilised softmax attention in 50-digit arithmetic, pure Python."""
    import mpmath
    mpmath.mp.dps = 50
    BH, Nq, d = q.shape
    Nk = k.shape[1]
    out = np.zeros((BH, Nq, d))
    lse2 = np.zeros((BH, Nq))
    for h in range(BH):
        for i in range(Nq):
            js = range(i + 1) if causal else range(Nk)
            ws = []
            for j in js:
                s = mpmath.fsum(mpmath.mpf(float(q[h, i, c])) * mpmath.mpf(float(k[h, j, c]))
                                for c in range(d))
                ws.append(mpmath.exp(mpmath.mpf(scale) * s))
            tot = mpmath.fsum(ws)
            for c in range(d):
                out[h, i, c] = float(mpmath.fsum(w * mpmath.mpf(float(v[h, j, c]))
                                                 for w, j in zip(ws, js)) / tot)
            lse2[h, i] = float(mpmath.log(tot, 2))
    return out, lse2


@pytest.mark.parametrize("causal", [False, True])
def test_attention_matches_brute_force(oracle_mod, causal):
    rng = np.random.default_rng(1)
    BH, N, d = 2, 7, 5
    q = rng.normal(size=(BH, N, d)) * 2
    k = rng.normal(size=(BH, N, d)) * 2 + rng.normal(size=(BH, 1, d))
    v = rng.normal(size=(BH, N, d))
    scale = 0.7
    out, lse2 = oracle_mod.attention(q, k, v, scale, causal=causal, with_lse2=True)
    ref, ref_lse2 = _brute(q, k, v, scale, causal)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse2, ref_lse2, rtol=0, atol=1e-12)


def test_attention_bf16_input_path_matches_brute_force(oracle_mod):
    rng = np.random.default_rng(2)
    q = _bf16(rng.normal(size=(1, 4, 6)))
    k = _bf16(rng.normal(size=(1, 9, 6)) + 1.5)
    v = _bf16(rng.normal(size=(1, 9, 6)))
    out = oracle_mod.attention(q, k, v, 0.5)
    ref, _ = _brute(q.double().numpy(), k.double().numpy(), v.double().numpy(), 0.5, False)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_shift_invariance(oracle_mod):
    """softmax(q K^T) = softmax(q (K - 1 c^T)^T) (the identity behind Alg. 1 step 2)."""
    rng = np.random.default_rng(3)
    q = rng.normal(size=(3, 16, 8))
    k = rng.normal(size=(3, 33, 8))
    v = rng.normal(size=(3, 33, 8))
    c = rng.normal(size=(3, 1, 8)) * 10
    a = oracle_mod.attention(q, k, v, 0.4)
    b = oracle_mod.attention(q, k - c, v, 0.4)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-11)


def test_single_key_returns_its_value(oracle_mod):
    rng = np.random.default_rng(4)
    q = rng.normal(size=(2, 5, 8)) * 30
    k = rng.normal(size=(2, 1, 8)) * 30
    v = rng.normal(size=(2, 1, 8))
    out = oracle_mod.attention(q, k, v, 1.0)
    assert np.array_equal(out, np.broadcast_to(v, out.shape))


def test_identical_keys_give_mean_value(oracle_mod):
    rng = np.random.default_rng(5)
    q = rng.normal(size=(1, 6, 8))
    k = np.tile(rng.normal(size=(1, 1, 8)), (1, 40, 1))
    v = rng.normal(size=(1, 40, 8))
    out = oracle_mod.attention(q, k, v, 0.3)
    np.testing.assert_allclose(out, np.broadcast_to(v.mean(axis=1, keepdims=True), out.shape),
                               rtol=0, atol=1e-14)


def test_dominant_key_selects_its_value(oracle_mod):
    rng = np.random.default_rng(6)
    d = 8
    q = np.zeros((1, 1, d))
    q[0, 0, 2] = 1.0
    k = rng.normal(size=(1, 20, d)) * 0.1
    k[0, 13, 2] = 60.0          # score 60 vs ~0.1: weight of the rest ~ 20 e^-59
    v = rng.normal(size=(1, 20, d))
    out = oracle_mod.attention(q, k, v, 1.0)
    np.testing.assert_allclose(out[0, 0], v[0, 13], rtol=0, atol=1e-15)


def test_scale_enters_as_multiplier_of_scores(oracle_mod):
    rng = np.random.default_rng(7)
    q = rng.normal(size=(1, 5, 4))
    k = rng.normal(size=(1, 11, 4))
    v = rng.normal(size=(1, 11, 4))
    a = oracle_mod.attention(q, k, v, 0.25)
    b = oracle_mod.attention(q, k * 0.25, v, 1.0)     # 0.25 scaling is exact in fp64
    np.testing.assert_array_equal(a, b)
    c = oracle_mod.attention(q, k, v, 1.0)
    assert np.max(np.abs(a - c)) > 1e-3


def test_causal_rows_equal_prefix_attention(oracle_mod):
    rng = np.random.default_rng(8)
    N, d = 12, 4
    q = rng.normal(size=(1, N, d))
    k = rng.normal(size=(1, N, d))
    v = rng.normal(size=(1, N, d))
    out = oracle_mod.attention(q, k, v, 0.9, causal=True)
    assert np.array_equal(out[0, 0], v[0, 0])
    for i in range(N):
        ref = oracle_mod.attention(q[:, i:i + 1], k[:, :i + 1], v[:, :i + 1], 0.9)
        np.testing.assert_allclose(out[0, i], ref[0, 0], rtol=0, atol=1e-15)


def test_row_selection_matches_full(oracle_mod):
    rng = np.random.default_rng(9)
    q = rng.normal(size=(2, 30, 8))
    k = rng.normal(size=(2, 25, 8))
    v = rng.normal(size=(2, 25, 8))
    full, lf = oracle_mod.attention(q, k, v, 0.5, with_lse2=True)
    rows = [0, 7, 29, 3]
    part, lp = oracle_mod.attention(q, k, v, 0.5, rows=rows, with_lse2=True)
    np.testing.assert_array_equal(part, full[:, rows])
    np.testing.assert_array_equal(lp, lf[:, rows])


def test_rejects_bad_arguments(oracle_mod):
    q = np.zeros((1, 3, 4))
    k = np.zeros((1, 5, 4))
    with pytest.raises(ValueError):
        oracle_mod.attention(q, k, k, 1.0, causal=True)     # causal needs Nq == Nk
    with pytest.raises(ValueError):
        oracle_mod.attention(q, k, k, 1.0, rows=[3])        # row out of range


# ---------------------------------------------------------- input formats ----

def test_decode_every_fp16_and_bf16_pattern(oracle_mod):
    """The oracle's reading of all 65,536 bit patterns of each input format
    equals numpy's float16 and torch's bfloat16 conversions (NaN patterns
    decode to NaN)."""
    bits = np.arange(1 << 16, dtype=np.uint16)
    ref16 = bits.view(np.float16).astype(np.float64)
    refb = torch.from_numpy(bits.astype(np.int16)).view(torch.bfloat16).double().numpy()
    got16 = np.array([oracle_mod.decode(int(b), "fp16") for b in bits])
    gotb = np.array([oracle_mod.decode(int(b), "bf16") for b in bits])
    for got, ref in ((got16, ref16), (gotb, refb)):
        nan = np.isnan(ref)
        assert np.array_equal(np.isnan(got), nan)
        assert np.array_equal(got[~nan], ref[~nan])


def test_fp16_inputs_match_brute_force_and_certify(oracle_mod):
    rng = np.random.default_rng(12)
    q = rng.normal(size=(2, 5, 6)).astype(np.float16)
    k = (rng.normal(size=(2, 7, 6)) * 3 + 1).astype(np.float16)
    v = rng.normal(size=(2, 7, 6)).astype(np.float16)
    out = oracle_mod.attention(q, k, v, 0.6)
    ref, _ = _brute(q.astype(np.float64), k.astype(np.float64), v.astype(np.float64), 0.6, False)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    # FP16 exp2 outputs: C = min(15, 127 - A); a head with B_h between 15 and 125 fails
    d = 8
    keys = _pm_keys(d, 1.0)
    q0 = np.zeros((1, d), dtype=np.float32)
    q0[0, 0] = 20.0
    kb, certs = oracle_mod.certify(q0[None].astype(np.float16), keys[None].astype(np.float16),
                                   np.zeros((1, 4, d), dtype=np.float16), 1.0, exp_fmt="fp16")
    assert certs[0]["B_h"] == 20.0 and certs[0]["C"] == 15 and certs[0]["certified"] == 0
    _, certs = oracle_mod.certify(q0[None].astype(np.float16), keys[None].astype(np.float16),
                                  np.zeros((1, 4, d), dtype=np.float16), 1.0, exp_fmt="bf16")
    assert certs[0]["C"] == 125 and certs[0]["certified"] == 1
    # an fp16 infinity is non-finite input
    vbad = np.zeros((1, 4, d), dtype=np.float16)
    vbad[0, 2, 3] = np.float16(np.inf)
    _, certs = oracle_mod.certify(q0[None].astype(np.float16), keys[None].astype(np.float16), vbad, 1.0)
    assert certs[0]["reason"] == 2


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_centred_scores_have_nonnegative_row_max_and_stay_within_bound(oracle_mod, seed):
    """With mu_i = scale_log2 * q_i . kbar, row i's exp2 arguments are
    scale_log2 * q_i . (k_j - kbar).  kbar is the key mean, so they average to
    zero over j: the row maximum is >= 0 and the row sum of 2^x is >= 1 (the
    no-underflow reading for non-causal rows).  And every argument lies in
    [-B_h, B_h], the certificate's Cauchy-Schwarz bound (Algorithm 1 step 4)."""
    rng = np.random.default_rng(100 + seed)
    BH, N, d = 3, 300, 64
    bias = rng.standard_normal((BH, 1, d)) * 2.0
    q = _bf16(rng.standard_normal((BH, N, d)) * (0.5 + seed))
    k = _bf16(rng.standard_normal((BH, N, d)) * 0.7 + bias)
    v = _bf16(rng.standard_normal((BH, N, d)))
    sl2 = 0.125 * 1.4426950408889634
    kbar, certs = oracle_mod.certify(q, k, v, sl2)
    qf, kf = q.double().numpy(), k.double().numpy()
    for h in range(BH):
        x = sl2 * (qf[h] @ (kf[h] - kbar[h]).T)
        assert x.max(axis=1).min() >= -1e-9
        assert np.exp2(x).sum(axis=1).min() >= 1.0 - 1e-12
        assert np.abs(x).max() <= certs[h]["B_h"] * (1 + 1e-12)
        assert np.abs(x).max() >= 0.25 * certs[h]["B_h"]  # and not vacuous (a few-fold inflated B_h fails)


# ---------------------------------------------------------------------------
# Per-prefix certificates of causal heads (one per block of query rows)


def _prefix_head(a, b, c, d=64, N=512):
    """Keys of rows 0-255 at +-a e1 in pairs and of rows 256-511 at +-b e1, so kbar = 0
    exactly and the prefix maxima of ||k - kbar|| are a (first block) and b (second);
    every query is c e1.  V = 0.5 everywhere (G = 0)."""
    k = torch.zeros(1, N, d)
    k[0, 0:256:2, 0], k[0, 1:256:2, 0] = a, -a
    k[0, 256::2, 0], k[0, 257::2, 0] = b, -b
    q = torch.zeros(1, N, d)
    q[0, :, 0] = c
    v = torch.full((1, N, d), 0.5)
    return tuple(t.to(torch.bfloat16) for t in (q, k, v))


@pytest.mark.parametrize("c,first_certified", [(59.0, 1), (59.25, 0)])
def test_prefix_tiles_hand_built(oracle_mod, c, first_certified):
    """N = 512, G = 0: A = 9, C = 127 - 9 = 118.  B_0 = c * 2 and B_1 = c * 8 with
    scale_log2 = 1: c = 59 puts block 0 exactly on the budget (a tie certifies) while
    the head (B_h = 472) fails; c = 59.25 fails block 0 as well."""
    q, k, v = _prefix_head(2.0, 8.0, c)
    cert, band, B = oracle_mod.certify_prefix_tiles(q, k, v, 1.0)
    _, heads = oracle_mod.certify(q, k, v, 1.0)
    assert heads[0]["C"] == 118 and heads[0]["certified"] == 0 and heads[0]["B_h"] == c * 8
    np.testing.assert_array_equal(B[0], [c * 2, c * 8])
    np.testing.assert_array_equal(cert[0], [first_certified, 0])


def test_prefix_tiles_bound_every_visible_exponent(oracle_mod):
    """What a block certificate promises, checked by enumeration: in a certified
    block every causal exp2 argument scale_log2 q_i . (k_j - kbar), j <= i, lies in
    [-C, C]; and the block bounds never exceed the head's bound."""
    gen = torch.Generator().manual_seed(17)
    BH, N, d, T = 6, 96, 16, 16
    q = torch.randn(BH, N, d, generator=gen)
    k = torch.randn(BH, N, d, generator=gen) * 0.5
    k[:, 72:] += 10.0  # the last quarter of the keys sits far from the rest
    v = torch.randn(BH, N, d, generator=gen)
    q, k, v = (t.to(torch.bfloat16) for t in (q, k, v))
    sl2 = 0.9
    cert, _, B = oracle_mod.certify_prefix_tiles(q, k, v, sl2, tile_rows=T)
    kbar, heads = oracle_mod.certify(q, k, v, sl2)
    qd, kd = q.double().numpy(), k.double().numpy()
    n_cert = 0
    for h in range(BH):
        C = heads[h]["C"]
        assert np.all(B[h] <= heads[h]["B_h"] * (1 + 1e-12))
        if heads[h]["certified"]:
            assert cert[h].all()
        x = sl2 * qd[h] @ (kd[h] - kbar[h]).T
        for b in range(cert.shape[1]):
            rows = range(b * T, min(N, (b + 1) * T))
            worst = max(np.abs(x[i, :i + 1]).max() for i in rows)
            assert worst <= B[h, b] * (1 + 1e-12)
            if cert[h, b]:
                n_cert += 1
                assert worst <= C
    # the far keys only enter the last blocks' prefixes: early blocks certify, late ones not,
    # and no head certifies as a whole
    assert 0 < n_cert < cert.size
    assert not any(hd["certified"] for hd in heads)


def test_prefix_tiles_nonfinite_head(oracle_mod):
    q, k, v = _prefix_head(1.0, 1.0, 1.0)
    q = q.clone()
    q[0, 300, 5] = float("nan")  # a row of the second block
    cert, _, B = oracle_mod.certify_prefix_tiles(q, k, v, 1.0)
    assert not cert.any() and np.all(np.isinf(B))
