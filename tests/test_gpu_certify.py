"""GPU certification pass (Algorithm 1) vs the fp64 oracle, through the C ABI.

Flags, reasons and the integers G, A, C must match bit for bit; kappa, B_h and
qmax are upward-rounded fp32 bounds and must sit within a relative 1e-4 of the
oracle's exact values; kbar within fp32 summation error.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from certified_fixed_stabilizer_gb300 import clis
from certified_fixed_stabilizer_gb300.workloads import WORKLOADS, injected_heads, make_inputs
from gpu_util import need_gpu

pytestmark = pytest.mark.gpu

INT_KEYS = ("certified", "reason", "G", "A", "C")


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


def _compare(q, k, v, sl2, exp_fmt="bf16", acc_fmt="fp32", expect_no_band=True):
    kbar, certs = clis.clis_certify(q, k, v, sl2, exp_fmt=exp_fmt, acc_fmt=acc_fmt)
    torch.cuda.synchronize()
    g = clis.decode_certs(certs)
    okbar, oc = oracle.certify(q, k, v, sl2, exp_fmt, acc_fmt)
    BH = q.shape[0] * q.shape[1]
    assert len(g) == BH or BH == 0
    for h in range(BH):
        for key in INT_KEYS:
            assert g[h][key] == oc[h][key], (h, key, g[h], oc[h])
        if oc[h]["reason"] == 2:
            continue
        if expect_no_band:
            assert oc[h]["band"] == 0, f"head {h} sits within rounding of the decision boundary"
        for key in ("kappa", "qmax", "B_h"):
            ref = oc[h][key]
            assert abs(g[h][key] - ref) <= 1e-4 * max(ref, 1e-30), (h, key, g[h][key], ref)
        assert g[h]["qmax"] >= oc[h]["qmax"]              # upward rounding of an exact quantity
        assert g[h]["kappa"] >= oc[h]["kappa"] * (1 - 1e-5)
    if BH:
        kb = kbar.cpu().double().numpy()
        np.testing.assert_allclose(kb, okbar, rtol=2e-5, atol=2e-5)
    return g, oc


@pytest.mark.parametrize("name", ["tiny", "480p", "720p", "mixed", "causal", "causal_late"])
def test_workload_certificates_match_oracle(name):
    dev = need_gpu()
    w = WORKLOADS[name]
    q, k, v = make_inputs(w, device=dev)
    sl2 = clis.scale_log2_for(w.d)
    g, oc = _compare(q, k, v, sl2)
    flags = [c["certified"] for c in g]
    if w.inject_frac > 0:  # mixed: 16 of 64 heads; causal_late: 32 of 128
        inj = set(injected_heads(w))
        assert len(inj) == {"mixed": 16, "causal_late": 32}[name]
        assert flags == [0 if h in inj else 1 for h in range(w.heads)]
        for h in inj:
            assert g[h]["G"] == 12 and g[h]["reason"] == 1
    else:
        assert all(flags), flags


def _head_tensors(dev, keys, queries, values=None, d=64):
    keys = np.asarray(keys, dtype=np.float32)
    queries = np.asarray(queries, dtype=np.float32)
    if values is None:
        values = np.zeros_like(keys)

    def t(a):
        a = np.asarray(a, dtype=np.float32)
        full = np.zeros((a.shape[0], d), dtype=np.float32)
        full[:, :a.shape[1]] = a
        x = torch.tensor(full).to(torch.bfloat16)
        assert np.array_equal(x.float().numpy(), full)
        return x.reshape(1, 1, *full.shape).to(dev)
    return t(queries), t(keys), t(values)


def _pm_keys(d, kappa, offset=0.0):
    e = np.zeros(d, dtype=np.float32)
    e[0] = kappa
    base = np.full(d, offset, dtype=np.float32)
    return np.stack([base + e, base - e, base + e, base - e])


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("qx,offset,cert", [(2000.0, 0.0, 1), (2008.0, 0.0, 0), (2000.0, 3.0, 1),
                                             (2008.0, -5.0, 0)])
def test_boundary_heads_bit_exact(d, qx, offset, cert):
    """B_h = C exactly certifies (tie), B_h = C + 0.5 fails; a common key offset
    must not change kappa.  All values are exact, so the GPU's directed
    rounding is exact too."""
    dev = need_gpu()
    q0 = np.zeros(d, dtype=np.float32)
    q0[0] = qx
    q, k, v = _head_tensors(dev, _pm_keys(d, 1.0, offset), [q0], d=d)
    g, oc = _compare(q, k, v, 1.0 / 16, expect_no_band=False)
    assert g[0]["certified"] == cert and g[0]["C"] == 125
    assert g[0]["kappa"] == 1.0 and g[0]["qmax"] == qx and g[0]["B_h"] == qx / 16


def test_equal_keys_and_fp16_budget():
    dev = need_gpu()
    d = 64
    keys = np.tile(np.linspace(-2, 2, d, dtype=np.float32), (5, 1))
    keys = torch.tensor(keys).to(torch.bfloat16).float().numpy()
    q, k, v = _head_tensors(dev, keys, np.ones((3, d), dtype=np.float32) * 100, d=d)
    g, _ = _compare(q, k, v, 1.0, expect_no_band=False)
    assert g[0]["kappa"] == 0.0 and g[0]["B_h"] == 0.0 and g[0]["certified"] == 1
    for qx, cert in [(15.0, 1), (15.5, 0)]:
        q0 = np.zeros(d, dtype=np.float32)
        q0[0] = qx
        q, k, v = _head_tensors(dev, _pm_keys(d, 1.0), [q0], d=d)
        g, _ = _compare(q, k, v, 1.0, exp_fmt="fp16", expect_no_band=False)
        assert g[0]["C"] == 15 and g[0]["certified"] == cert
    for ef, af, C in [("bf16", "fp16", 13), ("fp32", "fp32", 125), ("fp16", "fp16", 13)]:
        q, k, v = _head_tensors(dev, _pm_keys(d, 1.0), [np.ones(d, dtype=np.float32)], d=d)
        g, _ = _compare(q, k, v, 1.0, exp_fmt=ef, acc_fmt=af, expect_no_band=False)
        assert g[0]["C"] == C


@pytest.mark.parametrize("vm,G", [(4096.0, 12), (4128.0, 13), (1.0, 0), (0.75, 0), (3.0, 2)])
def test_v_exponent_bit_exact(vm, G):
    dev = need_gpu()
    d = 128
    vals = np.zeros((4, d), dtype=np.float32)
    vals[1, 3] = -vm
    q, k, v = _head_tensors(dev, _pm_keys(d, 1.0), [np.ones(d, dtype=np.float32)], vals, d=d)
    g, _ = _compare(q, k, v, 1.0, expect_no_band=False)
    assert g[0]["G"] == G and g[0]["A"] == 2 + G


@pytest.mark.parametrize("where", ["q", "k", "v"])
@pytest.mark.parametrize("bad", [float("nan"), float("inf"), -float("inf")])
def test_nonfinite_inputs_fail_certification(where, bad):
    dev = need_gpu()
    w = WORKLOADS["tiny"]
    q, k, v = make_inputs(w, device=dev, N=700)
    t = {"q": q, "k": k, "v": v}[where]
    t[0, 1, 517, 5] = bad
    g, oc = _compare(q, k, v, clis.scale_log2_for(w.d))
    assert g[1]["reason"] == 2 and g[1]["certified"] == 0 and g[0]["certified"] == 1


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Nq,Nk", [(1, 1), (5, 3), (1023, 1025), (3001, 1000), (0, 17), (2048, 4099)])
def test_ragged_sizes(d, Nq, Nk):
    dev = need_gpu()
    g = torch.Generator(device=dev)
    g.manual_seed(Nq * 7 + Nk)
    q = (torch.randn(2, 3, Nq, d, generator=g, device=dev)).to(torch.bfloat16)
    k = (torch.randn(2, 3, Nk, d, generator=g, device=dev) * 0.7 + 1.5).to(torch.bfloat16)
    v = (torch.randn(2, 3, Nk, d, generator=g, device=dev) * 3).to(torch.bfloat16)
    _compare(q, k, v, clis.scale_log2_for(d))


def test_strided_layout():
    """[B, N, H, d] storage viewed as [B, H, N, d]: non-default strides."""
    dev = need_gpu()
    g = torch.Generator(device=dev)
    g.manual_seed(5)
    base = (torch.randn(2, 1500, 4, 128, generator=g, device=dev) + 0.3).to(torch.bfloat16)
    q = base.permute(0, 2, 1, 3)
    k = (base * 0.5 + 1).permute(0, 2, 1, 3)
    v = base.flip(1).permute(0, 2, 1, 3)
    assert q.stride(2) == 4 * 128
    _compare(q, k, v, clis.scale_log2_for(128))


def test_deterministic():
    dev = need_gpu()
    w = WORKLOADS["480p"]
    q, k, v = make_inputs(w, device=dev, H=4)
    sl2 = clis.scale_log2_for(w.d)
    a = clis.clis_certify(q, k, v, sl2)
    b = clis.clis_certify(q, k, v, sl2)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("name", ["tiny", "mixed"])
def test_per_row_stabilisers(name):
    """mu_i = scale_log2 * (q_i . kbar) from the certification pass, against the
    same formula in fp64 with the oracle's kbar (|error| well below one exp2
    unit: mu is a shift, any fixed value is exact in real arithmetic)."""
    dev = need_gpu()
    w = WORKLOADS[name]
    q, k, v = make_inputs(w, device=dev, N=3000 if name == "mixed" else None)
    sl2 = clis.scale_log2_for(w.d)
    mu = torch.full((q.shape[0] * q.shape[1] * q.shape[2],), float("nan"), device=dev)
    clis.clis_certify(q, k, v, sl2, mu=mu)
    torch.cuda.synchronize()
    okbar, _ = oracle.certify(q, k, v, sl2)
    qf = oracle.bf16_bits_to_f64(oracle.as_bf16_bits(q)).reshape(okbar.shape[0], -1, w.d)
    ref = sl2 * np.einsum("hnd,hd->hn", qf, okbar)
    got = mu.cpu().double().numpy().reshape(ref.shape)
    scale = sl2 * np.linalg.norm(qf, axis=2) * np.linalg.norm(okbar, axis=1)[:, None]
    assert np.all(np.abs(got - ref) <= 1e-5 * scale + 1e-6)


@pytest.mark.parametrize("name,N,H", [("tiny", None, None), ("480p", 5000, 4), ("mixed", 3000, 8), ("causal", 2000, 4)])
def test_fp16_certificates_match_oracle(name, N, H):
    """FP16 data certified with the FP16 exp2 budget (U_exp = 15.9993, Figure 3):
    flags, G, A, C bit-exact vs the oracle."""
    dev = need_gpu()
    w = WORKLOADS[name]
    q, k, v = make_inputs(w, device=dev, N=N, H=H, dtype=torch.float16)
    g, oc = _compare(q, k, v, clis.scale_log2_for(w.d), exp_fmt="fp16")
    assert all(c["C"] <= 15 for c in g if c["reason"] != 2)
    if name == "causal":   # B_h ~ 23 > 15: every head fails the FP16 budget
        assert not any(c["certified"] for c in g)


@pytest.mark.parametrize("vm,G", [(4096.0, 12), (4100.0, 13), (1.0, 0), (0.5, 0), (3.0, 2), (65504.0, 16)])
def test_fp16_v_exponent_bit_exact(vm, G):
    dev = need_gpu()
    d = 64
    keys = np.stack([np.eye(1, d, 0)[0], -np.eye(1, d, 0)[0]] * 2).astype(np.float32)
    vals = np.zeros((4, d), dtype=np.float32)
    vals[1, 3] = -vm
    q = torch.tensor(np.ones((1, d), np.float32)).to(torch.float16).reshape(1, 1, 1, d).to(dev)
    k = torch.tensor(keys).to(torch.float16).reshape(1, 1, 4, d).to(dev)
    v = torch.tensor(vals).to(torch.float16).reshape(1, 1, 4, d).to(dev)
    g, _ = _compare(q, k, v, 1.0, expect_no_band=False)
    assert g[0]["G"] == G and g[0]["A"] == 2 + G


@pytest.mark.parametrize("where", ["q", "k", "v"])
def test_fp16_nonfinite_inputs_fail_certification(where):
    dev = need_gpu()
    w = WORKLOADS["480p"]   # B_h ~ 5.5: clean heads certify under the FP16 budget
    q, k, v = make_inputs(w, device=dev, N=700, H=2, dtype=torch.float16)
    t = {"q": q, "k": k, "v": v}[where]
    t[0, 1, 300, 9] = float("inf")
    g, oc = _compare(q, k, v, clis.scale_log2_for(w.d), exp_fmt="fp16")
    assert g[1]["reason"] == 2 and g[0]["certified"] == 1


def test_workspace_contents_do_not_leak_between_calls():
    """The norms pass combines the quarter-chunk maxima of a chunk with atomicMax
    in the caller's workspace, after the k-bar step has cleared them.  A workspace
    holding garbage (all bits set) or the maxima of larger inputs must give the
    same certificates as a fresh one."""
    dev = need_gpu()
    w = WORKLOADS["480p"]
    q, k, v = make_inputs(w, device=dev, H=3, N=3000)
    sl2 = clis.scale_log2_for(w.d)
    ref_kbar, ref_certs = clis.clis_certify(q, k, v, sl2)
    ws = torch.empty(max(256, clis.clis_certify_workspace_size(clis.make_shape(q, k, v))), dtype=torch.uint8,
                     device=dev)
    ws.fill_(255)
    kb1, c1 = clis.clis_certify(q, k, v, sl2, workspace=ws)
    clis.clis_certify(q * 64, k * 64, v * 64, sl2, workspace=ws)
    kb2, c2 = clis.clis_certify(q, k, v, sl2, workspace=ws)
    torch.cuda.synchronize()
    for kb, c in ((kb1, c1), (kb2, c2)):
        assert torch.equal(kb, ref_kbar)
        assert torch.equal(c, ref_certs)


@pytest.mark.parametrize("H", [2, 7, 13])
def test_long_heads_with_prefix_flags(H):
    """Heads of 40,000 keys at d = 64: 40 column-sum chunks and 157 query blocks
    each, the last ones ragged.  Head 0 has its last 64 keys scaled by 16: it
    fails as a head while its earlier query blocks certify by their prefix.
    Certificates, kbar, mu and the per-prefix flags against the oracle."""
    dev = need_gpu()
    N, d = 40000, 64
    g = torch.Generator(device=dev)
    g.manual_seed(100 + H)
    q = (torch.randn(1, H, N, d, generator=g, device=dev) * 0.5).to(torch.bfloat16)
    k = (torch.randn(1, H, N, d, generator=g, device=dev) * 0.7 + 1.5).to(torch.bfloat16)
    v = (torch.randn(1, H, N, d, generator=g, device=dev) * 3).to(torch.bfloat16)
    k[0, 0, N - 64:] *= 16  # exactly the last 256-row block's keys (rows 39,936 on)
    sl2 = clis.scale_log2_for(d)
    gc, oc = _compare(q, k, v, sl2)
    assert [c["certified"] for c in gc] == [0] + [1] * (H - 1)
    mu = torch.full((H * N,), float("nan"), device=dev)
    kbar, certs, tiles = clis.clis_certify_tiles(q, k, v, sl2, mu=mu)
    kbar2, certs2 = clis.clis_certify(q, k, v, sl2)
    torch.cuda.synchronize()
    assert torch.equal(kbar, kbar2) and torch.equal(certs, certs2)
    ocert, oband, _ = oracle.certify_prefix_tiles(q.cpu(), k.cpu(), v.cpu(), sl2)
    t = tiles.cpu().numpy().astype(np.int32)
    assert not oband.any()
    np.testing.assert_array_equal(t, ocert)
    assert t[0, :-1].all() and t[0, -1] == 0 and t[1:].all()
    okbar, _ = oracle.certify(q, k, v, sl2)
    qf = oracle.bf16_bits_to_f64(oracle.as_bf16_bits(q)).reshape(H, N, d)
    ref = sl2 * np.einsum("hnd,hd->hn", qf, okbar)
    got = mu.cpu().double().numpy().reshape(ref.shape)
    scale = sl2 * np.linalg.norm(qf, axis=2) * np.linalg.norm(okbar, axis=1)[:, None]
    assert np.all(np.abs(got - ref) <= 1e-5 * scale + 1e-6)

