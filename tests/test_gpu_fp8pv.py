"""FP8 P.V path (clis_v_to_e4m3 + clis_attn_fwd_fp8pv) against the oracle and
against a CPU rounding model of the same E4M3 roundings.

The FP8 path is one step below Figure 3's FP16 row: P and V in E4M3 for the
P.V product (kind::f8f6f4), everything else as on the certified BF16 path.
Checked: the V^T conversion bit for bit against torch's E4M3 rounding; forced
FP8 output element by element against tests/rounding_model.py's FP8 model
(what remains is fp32 summation order and the E4M3 roundings it tips over)
and against the fp64 oracle (within the acceptance bar from 4096 keys on);
AUTO sends eligible heads (certified, B_h <= min(8, C), G <= 8, Nk >= 4096)
to FP8 and every other head through the unchanged BF16 kernel path, bit for
bit; ragged and full-size shapes.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import rounding_model as rm
from certified_fixed_stabilizer_gb300 import clis
from certified_fixed_stabilizer_gb300.workloads import WORKLOADS, injected_heads_present, make_inputs, sample_rows
from gpu_util import assert_close_to_oracle, flat, need_gpu, report

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


def _fp8_eligible(c, Nk):
    return bool(c["certified"]) and c["B_h"] <= min(8, c["C"]) and c["G"] <= 8 and Nk >= 4096


def _run(q, k, v, variant="auto", lse=False):
    sl2 = clis.scale_log2_for(q.shape[-1])
    mu = torch.empty(q.shape[0] * q.shape[1] * q.shape[2], device=q.device)
    kbar, certs = clis.clis_certify(q, k, v, sl2, mu=mu)
    vt8 = clis.clis_v_to_e4m3(v)
    l2 = torch.empty_like(mu) if lse else None
    out = clis.clis_attn_fwd_fp8pv(q, k, v, vt8, sl2, kbar=kbar, certs=certs, variant=variant, mu=mu, lse2=l2)
    torch.cuda.synchronize()
    return out, l2, kbar, certs, mu


def test_v_conversion_matches_e4m3_rounding():
    dev = need_gpu()
    w = WORKLOADS["480p"]
    for N in (1000, 128, 3):
        _, _, v = make_inputs(w, device=dev, N=N, H=3, seed=N)
        vt8 = clis.clis_v_to_e4m3(v)
        torch.cuda.synchronize()
        pitch = -(-N // 16) * 16
        assert vt8.shape == (3, 128, pitch)
        ref = flat(v).cpu().float().transpose(1, 2).contiguous().to(torch.float8_e4m3fn).view(torch.uint8)
        got = vt8.cpu()
        assert torch.equal(got[:, :, :N], ref)
        assert torch.count_nonzero(got[:, :, N:]) == 0


def _model_errors(got, q, k, v, scale):
    """Worst per-head (max excess over half a bf16 ulp, mean abs) of the GPU
    output against the FP8 rounding model, divided by max(1, max |model|)."""
    qf, kf, vf = (flat(t).double().cpu().numpy() for t in (q, k, v))
    worst_excess, worst_mean = 0.0, 0.0
    for h in range(qf.shape[0]):
        e, _ = rm.certified_forward_fp8pv(qf[h], kf[h], vf[h], scale)
        sc = max(1.0, np.abs(e).max())
        worst_excess = max(worst_excess, np.maximum(np.abs(got[h] - e) - np.abs(e) * 2.0 ** -8, 0.0).max() / sc)
        worst_mean = max(worst_mean, np.abs(got[h] - rm.bf16(e)).mean() / sc)
    return worst_excess, worst_mean


@pytest.mark.parametrize("N", [4500, 2000, 513])
def test_forced_fp8_matches_rounding_model(N):
    """Element by element against the FP8 model; what remains is fp32 order,
    the hardware exp2 and the E4M3 roundings those tip over (one E4M3 step is
    2^-3 of a weight, shared by the rest of the row's thousands of keys).
    Against the oracle: the bar from 4096 keys on (AUTO's threshold), and
    below that the error model's 0.05 / sqrt(Nk) for the mean."""
    dev = need_gpu()
    w = WORKLOADS["480p"]
    q, k, v = make_inputs(w, device=dev, N=N, H=4, seed=40 + N)
    out, l2, _, certs, _ = _run(q, k, v, "certified", lse=True)
    got = flat(out).float().cpu().numpy()
    excess, mean = _model_errors(got, q, k, v, w.softmax_scale())
    report(f"fp8pv forced N={N} vs model", max_excess=excess, mean=mean)
    assert excess <= 1e-3 and mean <= 1e-5, (excess, mean)
    ref, rlse = oracle.attention(flat(q).cpu(), flat(k).cpu(), flat(v).cpu(), w.softmax_scale(), with_lse2=True)
    if N >= 4096:
        assert_close_to_oracle(got, ref, f"fp8pv forced N={N}")
    else:
        from gpu_util import head_errors
        mx, mn = head_errors(got, ref)
        report(f"fp8pv forced N={N} vs oracle", max_abs=float(mx.max()), mean_abs=float(mn.max()))
        assert mn.max() <= 0.05 / np.sqrt(N) and mx.max() <= 2e-2, (mx.max(), mn.max())
    np.testing.assert_allclose(l2.cpu().numpy().reshape(rlse.shape), rlse, atol=2e-3, rtol=0)


def test_auto_routes_heads_by_eligibility():
    """Mixed heads: injected (uncertified) heads and certified heads; eligible
    heads equal the forced FP8 output, the others the BF16 kernel's, bit for bit."""
    dev = need_gpu()
    w = WORKLOADS["mixed"]
    N = 4500
    q, k, v = make_inputs(w, device=dev, N=N, H=8)
    out, _, kbar, certs, mu = _run(q, k, v, "auto")
    forced, _, _, _, _ = _run(q, k, v, "certified")
    sl2 = clis.scale_log2_for(w.d)
    bf = clis.clis_attn_fwd(q, k, v, sl2, kbar=kbar, certs=certs, mu=mu)
    torch.cuda.synchronize()
    cs = clis.decode_certs(certs)
    elig = [_fp8_eligible(c, N) for c in cs]
    assert 0 < sum(elig) < len(elig)
    # The same rule from the oracle's certificate under the E4M3 budget (Algorithm 1
    # with exp_fmt = E4M3: C = min(8, 127 - A)), independent of the GPU's numbers.
    _, oc = oracle.certify(q.cpu(), k.cpu(), v.cpu(), sl2, exp_fmt="e4m3")
    for h, (e, c) in enumerate(zip(elig, oc)):
        if not c["band"]:
            assert e == (bool(c["certified"]) and c["G"] <= 8 and N >= 4096), (h, c)
    fo, ff, fb = flat(out), flat(forced), flat(bf)
    for h, e in enumerate(elig):
        assert torch.equal(fo[h], ff[h] if e else fb[h]), (h, e)
    ref, _ = oracle.attention(flat(q).cpu(), flat(k).cpu(), flat(v).cpu(), w.softmax_scale(), with_lse2=True)
    assert_close_to_oracle(fo.float().cpu().numpy(), ref, "fp8pv auto mixed")
    assert set(injected_heads_present(w, 8)) <= {h for h, e in enumerate(elig) if not e}


def test_auto_keeps_short_heads_on_bf16():
    """Below 4096 keys no head takes E4M3 in AUTO: the output is the BF16
    kernel's, bit for bit."""
    dev = need_gpu()
    w = WORKLOADS["480p"]
    q, k, v = make_inputs(w, device=dev, N=3000, H=3)
    out, _, kbar, certs, mu = _run(q, k, v, "auto")
    bf = clis.clis_attn_fwd(q, k, v, clis.scale_log2_for(w.d), kbar=kbar, certs=certs, mu=mu)
    torch.cuda.synchronize()
    assert torch.equal(out, bf)


@pytest.mark.parametrize("Nk", [4095, 4096])
def test_auto_key_count_threshold(Nk):
    """AUTO takes E4M3 from 4096 keys on: 4095 keys give the BF16 kernel's
    output, 4096 the forced FP8 output, bit for bit."""
    dev = need_gpu()
    w = WORKLOADS["480p"]
    q, _, _ = make_inputs(w, device=dev, N=600, H=2, seed=51)
    _, k, v = make_inputs(w, device=dev, N=Nk, H=2, seed=52)
    out, _, kbar, certs, mu = _run(q, k, v, "auto")
    forced, _, _, _, _ = _run(q, k, v, "certified")
    bf = clis.clis_attn_fwd(q, k, v, clis.scale_log2_for(w.d), kbar=kbar, certs=certs, mu=mu)
    torch.cuda.synchronize()
    assert all(c["certified"] and c["B_h"] <= 8 for c in clis.decode_certs(certs))
    assert torch.equal(out, forced if Nk >= 4096 else bf)
    assert not torch.equal(forced, bf)


@pytest.mark.parametrize("Nq,Nk", [(1, 1), (127, 129), (1000, 300), (257, 1025)])
def test_ragged_shapes(Nq, Nk):
    """Forced FP8 on ragged shapes (a single key, partial tiles, Nq != Nk),
    against the FP8 model."""
    dev = need_gpu()
    w = WORKLOADS["480p"]
    q, _, _ = make_inputs(w, device=dev, N=Nq, H=2, seed=Nq)
    _, k, v = make_inputs(w, device=dev, N=Nk, H=2, seed=Nk + 1)
    out, _, _, _, _ = _run(q, k, v, "certified")
    excess, mean = _model_errors(flat(out).float().cpu().numpy(), q, k, v, w.softmax_scale())
    report(f"fp8pv ragged {Nq}x{Nk} vs model", max_excess=excess, mean=mean)
    assert excess <= 1e-3 and mean <= 1e-5, (excess, mean)


def test_full_720p_sampled_rows():
    """The 720p workload in the launch configuration the benchmark times, on
    seed-chosen rows of three heads."""
    dev = need_gpu()
    w = WORKLOADS["720p"]
    q, k, v = make_inputs(w, device=dev)
    out, _, _, certs, _ = _run(q, k, v, "auto")
    assert all(_fp8_eligible(c, w.N) for c in clis.decode_certs(certs))
    rows = sample_rows(w.N, 48, seed=5)
    heads = [0, 17, 39]
    got = flat(out)[heads][:, rows].float().cpu().numpy()
    ref, _ = oracle.attention(flat(q)[heads].cpu(), flat(k)[heads].cpu(), flat(v)[heads].cpu(), w.softmax_scale(),
                              rows=rows, with_lse2=True)
    assert_close_to_oracle(got, ref, "fp8pv 720p sampled")


def test_attention_call_with_fp8_pv():
    """The public attention() call with pv="fp8" is certify + conversion +
    clis_attn_fwd_fp8pv, bit for bit."""
    dev = need_gpu()
    w = WORKLOADS["480p"]
    q, k, v = make_inputs(w, device=dev, N=5000, H=2, seed=61)
    out = clis.attention(q, k, v, pv="fp8")
    ref, _, _, _, _ = _run(q, k, v, "auto")
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    with pytest.raises(ValueError):
        clis.attention(q, k, v, causal=True, pv="fp8")
    # Under 4096 keys no head takes E4M3 in AUTO: the call skips the conversion and
    # gives the BF16 result, bit for bit.
    qs, ks, vs = (t[:, :, :3000] for t in (q, k, v))
    o_small = clis.attention(qs, ks, vs, pv="fp8")
    o_bf16 = clis.attention(qs, ks, vs)
    torch.cuda.synchronize()
    assert torch.equal(o_small, o_bf16)


def test_ring_step_chunks_with_fp8_pv():
    """The ring-step form with E4M3 P.V: K/V of 480p-distributed heads in three
    chunks of 4096 keys and more (each converted on its own), merged into the
    fp32 accumulators; AUTO sends every head to E4M3 (chunks of at least 4096
    keys) and the result meets the bar against the oracle; forced FP8 on one
    chunk holding every key equals clis_attn_fwd_fp8pv, bit for bit."""
    dev = need_gpu()
    w = WORKLOADS["480p"]
    N = 13000
    q, k, v = make_inputs(w, device=dev, N=N, H=3, seed=71)
    sl2 = clis.scale_log2_for(w.d)
    mu = torch.empty(3 * N, device=dev)
    kbar, certs = clis.clis_certify(q, k, v, sl2, mu=mu)
    BHN = 3 * N

    def run(bounds, variant):
        o_acc = torch.full((BHN, w.d), float("nan"), device=dev)
        l_acc = torch.full((BHN,), float("nan"), device=dev)
        m_acc = torch.full((BHN,), float("nan"), device=dev)
        for i, (a, b) in enumerate(zip(bounds[:-1], bounds[1:])):
            kc, vc = k[:, :, a:b], v[:, :, a:b]
            clis.clis_attn_fwd_chunk_fp8pv(q, kc, vc, clis.clis_v_to_e4m3(vc), sl2, o_acc, l_acc, m_acc, kbar=kbar,
                                           certs=certs, first=(i == 0), variant=variant, mu=mu)
        lse2 = torch.empty(BHN, device=dev)
        out = clis.clis_attn_chunk_finalize(q, o_acc, l_acc, m_acc, lse2=lse2)
        torch.cuda.synchronize()
        return out, lse2

    out, lse2 = run([0, 4096, 8400, N], "auto")
    ref, rlse = oracle.attention(flat(q).cpu(), flat(k).cpu(), flat(v).cpu(), w.softmax_scale(), with_lse2=True)
    assert_close_to_oracle(flat(out).float().cpu().numpy(), ref, "fp8pv ring step")
    np.testing.assert_allclose(lse2.cpu().numpy().reshape(rlse.shape), rlse, atol=2e-3, rtol=0)
    one, _ = run([0, N], "certified")
    fused, _, _, _, _ = _run(q, k, v, "certified")
    assert torch.equal(one, fused)
