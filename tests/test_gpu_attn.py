"""GPU attention forward vs the fp64 oracle, through the C ABI.

Bar (per head, errors divided by max(1, max |O_ref|)): max-abs <= 1e-2 and
mean-abs <= 1e-3 against the fp64 two-pass softmax; the certified (CLiS) and
online paths must also agree with each other on certified heads.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from certified_fixed_stabilizer_gb300 import clis
from certified_fixed_stabilizer_gb300.workloads import (WORKLOADS, injected_heads, make_inputs,
                                                        sample_rows)
from gpu_util import assert_close_to_oracle, assert_paths_agree, flat, need_gpu

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


def _run(q, k, v, causal, variant, lse2=False, softmax_scale=None, exp_fmt=None):
    sl2 = clis.scale_log2_for(q.shape[-1], softmax_scale)
    if exp_fmt is None:
        exp_fmt = "fp16" if q.dtype == torch.float16 else "bf16"
    kbar, certs = clis.clis_certify(q, k, v, sl2, exp_fmt=exp_fmt)
    l2 = None
    if lse2:
        l2 = torch.full((q.shape[0] * q.shape[1] * q.shape[2],), float("nan"), device=q.device)
    out = clis.clis_attn_fwd(q, k, v, sl2, kbar=kbar, certs=certs, causal=causal, variant=variant, lse2=l2)
    torch.cuda.synchronize()
    return out, l2, certs


def _oracle(q, k, v, causal, rows=None, softmax_scale=None):
    scale = (1.0 / np.sqrt(q.shape[-1])) if softmax_scale is None else softmax_scale
    return oracle.attention(flat(q), flat(k), flat(v), scale, causal=causal, rows=rows, with_lse2=True)


@pytest.mark.parametrize("variant", ["auto", "online", "certified", "online_lazy"])
def test_tiny_full_parity(variant):
    dev = need_gpu()
    w = WORKLOADS["tiny"]
    q, k, v = make_inputs(w, device=dev)
    out, l2, certs = _run(q, k, v, w.causal, variant, lse2=True)
    ref, rlse = _oracle(q, k, v, w.causal)
    assert_close_to_oracle(out.float().cpu().numpy(), ref, f"tiny/{variant}")
    np.testing.assert_allclose(l2.cpu().numpy().reshape(rlse.shape), rlse, atol=1e-3, rtol=0)
    assert all(c["certified"] for c in clis.decode_certs(certs))


@pytest.mark.parametrize("name,rows_per_head", [("480p", 48), ("720p", 24), ("mixed", 48), ("causal", 64)])
def test_workload_sampled_parity(name, rows_per_head):
    """Full-size workloads, the launch configuration the benchmark times;
    the oracle evaluates seed-chosen rows (always 0, N-1 and the ragged tail)."""
    dev = need_gpu()
    w = WORKLOADS[name]
    q, k, v = make_inputs(w, device=dev)
    rows = sample_rows(w.N, rows_per_head, seed=1)
    ref, rlse = _oracle(q, k, v, w.causal, rows=rows)
    for variant in ("online_lazy", "auto", "online"):
        out, l2, certs = _run(q, k, v, w.causal, variant, lse2=True)
        got = flat(out)[:, rows].float().cpu().numpy()
        assert_close_to_oracle(got, ref, f"{name}/{variant}")
        g2 = l2.reshape(w.heads, w.N)[:, rows].cpu().numpy()
        np.testing.assert_allclose(g2, rlse, atol=2e-3, rtol=0)
        assert torch.isfinite(out).all()
        if variant == "auto":
            auto_out = out
    flags = [c["certified"] for c in clis.decode_certs(certs)]
    if name == "mixed":
        assert sum(flags) == 48
        for h in injected_heads(w):
            assert flags[h] == 0
    else:
        assert all(flags)
    # certified and online paths agree on certified heads (whole tensors)
    cert_heads = [h for h, f in enumerate(flags) if f]
    assert_paths_agree(flat(auto_out)[cert_heads], flat(out)[cert_heads], name)


CASES = [
    # (B, H, Nq, Nk, d, causal)
    (1, 2, 1, 1, 64, False),
    (1, 2, 1, 1, 128, True),
    (2, 3, 129, 129, 64, True),
    (1, 2, 257, 1000, 128, False),
    (1, 2, 1000, 257, 128, False),
    (2, 2, 700, 700, 128, True),
    (1, 3, 513, 513, 64, False),
    (1, 1, 2000, 2000, 128, True),
    (3, 1, 300, 4097, 64, False),
    (1, 4, 20000, 100, 128, False),   # one KV step per work tile, several tiles per CTA
    (2, 3, 9000, 1, 64, False),       # a single key
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal", CASES)
@pytest.mark.parametrize("variant", ["auto", "online", "online_lazy"])
def test_ragged_shapes(B, H, Nq, Nk, d, causal, variant):
    dev = need_gpu()
    g = torch.Generator(device=dev)
    g.manual_seed(B * 1000003 + H * 1009 + Nq * 31 + Nk + d)
    q = torch.randn(B, H, Nq, d, generator=g, device=dev).to(torch.bfloat16)
    k = (torch.randn(B, H, Nk, d, generator=g, device=dev) + torch.randn(d, generator=g, device=dev)).to(
        torch.bfloat16)
    v = torch.randn(B, H, Nk, d, generator=g, device=dev).to(torch.bfloat16)
    out, l2, _ = _run(q, k, v, causal, variant, lse2=True)
    ref, rlse = _oracle(q, k, v, causal)
    assert_close_to_oracle(out.float().cpu().numpy(), ref, f"{(B, H, Nq, Nk, d, causal)}/{variant}")
    np.testing.assert_allclose(l2.cpu().numpy().reshape(rlse.shape), rlse, atol=2e-3, rtol=0)


def test_strided_tensors_and_guard_bands():
    """Q/K/V/O stored as [B, N, H, d] (non-default strides) with O inside a larger
    buffer whose canary bytes must survive: no write outside O's rows."""
    dev = need_gpu()
    B, H, N, d = 2, 3, 777, 128
    g = torch.Generator(device=dev)
    g.manual_seed(11)
    q = torch.randn(B, N, H, d, generator=g, device=dev).to(torch.bfloat16).permute(0, 2, 1, 3)
    k = (torch.randn(B, N, H, d, generator=g, device=dev) + 2).to(torch.bfloat16).permute(0, 2, 1, 3)
    v = torch.randn(B, N, H, d, generator=g, device=dev).to(torch.bfloat16).permute(0, 2, 1, 3)
    pad = 4096
    canary = torch.full((pad * 2 + B * N * H * d,), -12345.0, device=dev).to(torch.bfloat16)
    o = canary[pad:pad + B * N * H * d].view(B, N, H, d).permute(0, 2, 1, 3)
    o.fill_(0)
    sl2 = clis.scale_log2_for(d)
    kbar, certs = clis.clis_certify(q, k, v, sl2)
    clis.clis_attn_fwd(q, k, v, sl2, kbar=kbar, certs=certs, out=o)
    torch.cuda.synchronize()
    assert torch.all(canary[:pad] == -12345.0) and torch.all(canary[-pad:] == -12345.0)
    ref, _ = _oracle(q, k, v, False)
    assert_close_to_oracle(o.float().cpu().numpy().reshape(ref.shape), ref, "strided")


def test_empty_query_launches_nothing():
    dev = need_gpu()
    q = torch.empty(1, 2, 0, 64, dtype=torch.bfloat16, device=dev)
    k = torch.randn(1, 2, 10, 64, device=dev).to(torch.bfloat16)
    out = clis.clis_attn_fwd(q, k, k, clis.scale_log2_for(64), variant="online")
    assert out.shape == q.shape


def test_softmax_scale_is_honoured():
    dev = need_gpu()
    g = torch.Generator(device=dev)
    g.manual_seed(3)
    q = torch.randn(1, 2, 300, 64, generator=g, device=dev).to(torch.bfloat16)
    k = torch.randn(1, 2, 300, 64, generator=g, device=dev).to(torch.bfloat16)
    v = torch.randn(1, 2, 300, 64, generator=g, device=dev).to(torch.bfloat16)
    out, _, _ = _run(q, k, v, False, "auto", softmax_scale=0.5)
    ref, _ = _oracle(q, k, v, False, softmax_scale=0.5)
    assert_close_to_oracle(out.float().cpu().numpy(), ref, "scale=0.5")


def test_host_tensors_end_to_end():
    """The public attention() call with pinned host tensors (the e2e path)."""
    need_gpu()
    w = WORKLOADS["tiny"]
    q, k, v = (t.pin_memory() for t in make_inputs(w, device="cpu"))
    out = clis.attention(q, k, v)
    assert out.device.type == "cpu"
    ref, _ = _oracle(q, k, v, False)
    assert_close_to_oracle(out.float().numpy(), ref, "host e2e")


def test_lazy_rescale_with_growing_maxima():
    """Keys whose scores grow along the sequence force the lazy online path to
    rescale in many blocks (the row maximum keeps outgrowing the stale one by
    more than 8): parity must hold there too, and in causal rows."""
    dev = need_gpu()
    g = torch.Generator(device=dev)
    g.manual_seed(21)
    B, H, N, d = 1, 2, 1500, 128
    q = torch.randn(B, H, N, d, generator=g, device=dev)
    ramp = torch.linspace(0, 6, N, device=dev)[:, None]
    k = torch.randn(B, H, N, d, generator=g, device=dev) * ramp + q.mean(dim=2, keepdim=True) * ramp
    v = torch.randn(B, H, N, d, generator=g, device=dev)
    q, k, v = (t.to(torch.bfloat16) for t in (q, k, v))
    for causal in (False, True):
        for variant in ("online_lazy", "online"):
            out, l2, _ = _run(q, k, v, causal, variant, lse2=True)
            ref, rlse = _oracle(q, k, v, causal)
            assert_close_to_oracle(out.float().cpu().numpy(), ref, f"growing/{variant}/{causal}")
            np.testing.assert_allclose(l2.cpu().numpy().reshape(rlse.shape), rlse, atol=2e-3, rtol=0)


def test_stabilisers_from_certification_match_in_kernel_ones():
    """clis_attn_fwd with mu from clis_certify vs the kernel computing mu itself."""
    dev = need_gpu()
    w = WORKLOADS["causal"]
    q, k, v = make_inputs(w, device=dev, N=2000, H=4)
    sl2 = clis.scale_log2_for(w.d)
    mu = torch.empty(q.shape[0] * q.shape[1] * q.shape[2], device=dev)
    kbar, certs = clis.clis_certify(q, k, v, sl2, mu=mu)
    a = clis.clis_attn_fwd(q, k, v, sl2, kbar=kbar, certs=certs, causal=True, mu=mu)
    b = clis.clis_attn_fwd(q, k, v, sl2, kbar=kbar, certs=certs, causal=True)
    torch.cuda.synchronize()
    assert_paths_agree(flat(a), flat(b), "mu from certify")
    ref, _ = _oracle(q, k, v, True)
    assert_close_to_oracle(flat(a).float().cpu().numpy(), ref, "mu from certify vs oracle")


@pytest.mark.parametrize("causal", [False, True])
def test_host_path_pipelined_over_head_groups(causal):
    """attention() with pinned host tensors splits the heads into groups that
    cross the batch boundary; the result matches the device path and the oracle."""
    dev = need_gpu()
    g = torch.Generator(device="cpu")
    g.manual_seed(17)
    B, H, N, d = 2, 3, 900, 128
    q = torch.randn(B, H, N, d, generator=g).to(torch.bfloat16).pin_memory()
    k = (torch.randn(B, H, N, d, generator=g) * 0.5 + 0.3).to(torch.bfloat16).pin_memory()
    v = torch.randn(B, H, N, d, generator=g).to(torch.bfloat16).pin_memory()
    host = clis.attention(q, k, v, causal=causal, groups=4)
    assert host.device.type == "cpu" and host.shape == q.shape
    dev_out = clis.attention(q.to(dev), k.to(dev), v.to(dev), causal=causal)
    torch.cuda.synchronize()
    assert_paths_agree(flat(host.to(dev)), flat(dev_out), "host vs device")
    ref, _ = _oracle(q, k, v, causal)
    assert_close_to_oracle(host.float().numpy().reshape(ref.shape), ref, "host pipelined")


def test_host_path_back_to_back_non_blocking_calls():
    """Consecutive non-blocking host calls with the same shapes reuse one set of
    staging buffers and overlap (a call's copies of a head group wait only for
    the previous call's kernels on that group): each call's output must be
    its own inputs' attention, including a call whose certificates are asked
    for (copied out on the caller's stream) between two others."""
    dev = need_gpu()
    g = torch.Generator(device="cpu")
    g.manual_seed(23)
    B, H, N, d = 1, 6, 1500, 128
    ins, outs = [], []
    for i in range(4):
        q = torch.randn(B, H, N, d, generator=g).to(torch.bfloat16).pin_memory()
        k = (torch.randn(B, H, N, d, generator=g) * 0.5 + 0.2 * i).to(torch.bfloat16).pin_memory()
        v = torch.randn(B, H, N, d, generator=g).to(torch.bfloat16).pin_memory()
        ins.append((q, k, v))
    certs = None
    for i, (q, k, v) in enumerate(ins):
        o = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
        if i == 2:
            _, _, certs = clis.attention(q, k, v, groups=3, out=o, non_blocking=True, return_certs=True)
        else:
            clis.attention(q, k, v, groups=3, out=o, non_blocking=True)
        outs.append(o)
    torch.cuda.synchronize()
    for i, ((q, k, v), o) in enumerate(zip(ins, outs)):
        dev_out, _, dcerts = clis.attention(q.to(dev), k.to(dev), v.to(dev), return_certs=True)
        torch.cuda.synchronize()
        assert_paths_agree(flat(o.to(dev)), flat(dev_out), f"back-to-back call {i}")
        if i == 2:
            assert torch.equal(certs, dcerts)
    ref, _ = _oracle(*ins[3], False)
    assert_close_to_oracle(outs[3].float().numpy().reshape(ref.shape), ref, "back-to-back last call")


def test_host_plan_workspace_and_argument_checks():
    """clis_host_plan_workspace_size covers staging for every head, k-bar,
    certificates, stabilisers and two certification scratch areas; the
    forward's pointer and workspace checks return their statuses (nothing is
    queued); the certificates sit where include/clis.h says."""
    import ctypes
    dev = need_gpu()
    B, H, N, d = 2, 3, 1000, 128
    g = torch.Generator(device="cpu")
    g.manual_seed(41)
    q, k, v = (torch.randn(B, H, N, d, generator=g).to(torch.bfloat16).pin_memory() for _ in range(3))
    o = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    plan = clis.HostPlan(q, k, v, o, groups=2, device=dev)
    n = ctypes.c_size_t(0)
    lib = clis.load_library()
    assert lib.clis_host_plan_workspace_size(plan.handle, ctypes.byref(n)) == 0
    n = n.value
    per_group = clis.clis_certify_workspace_size(clis.make_shape(q[:1], k[:1], v[:1]))
    assert n % 256 == 0 and n >= 4 * B * H * N * d * 2 + B * H * (d * 4 + 32 + N * 4) + 2 * per_group
    vp, ws = ctypes.c_void_p, plan.workspace
    args = [vp(t.data_ptr()) for t in (q, k, v, o)]
    for i in range(4):
        bad = list(args)
        bad[i] = None
        assert lib.clis_attention_host(plan.handle, *bad, 0.1, 0, vp(ws.data_ptr()), n, None) == 1
    assert lib.clis_attention_host(plan.handle, *args, 0.1, 0, None, n, None) == 4
    assert lib.clis_attention_host(plan.handle, *args, 0.1, 0, vp(ws.data_ptr()), n - 1, None) == 4
    assert lib.clis_attention_host(plan.handle, *args, 0.1, 0, vp(ws.data_ptr() + 16), n, None) == 3
    # A real call, then the certificates from the workspace against clis_certify.
    clis.clis_attention_host(plan, q, k, v, o, clis.scale_log2_for(d))
    plan.wait()
    torch.cuda.synchronize()
    off = (B * H * d * 4 + 255) // 256 * 256
    certs = ws[off:off + B * H * clis.CERT_WORDS * 4].view(torch.int32).view(B * H, clis.CERT_WORDS)
    kbar = ws[:B * H * d * 4].view(torch.float32).view(B * H, d)
    dkbar, dcerts = clis.clis_certify(q.to(dev), k.to(dev), v.to(dev), clis.scale_log2_for(d))
    torch.cuda.synchronize()
    assert torch.equal(certs, dcerts) and torch.equal(kbar, dkbar)
    ref = clis.attention(q.to(dev), k.to(dev), v.to(dev))
    torch.cuda.synchronize()
    assert_paths_agree(flat(o.to(dev)), flat(ref), "plan call")
    plan.destroy()


def test_host_path_follows_work_queued_on_the_current_stream():
    """Host inputs filled by asynchronous copies queued on the current stream
    (behind a long kernel) are read only after those copies: the call's input
    copies follow the caller's stream."""
    dev = need_gpu()
    w = WORKLOADS["480p"]
    q, k, v = make_inputs(w, device=dev, N=1200, H=4, seed=31)
    hosts = [torch.zeros(q.shape, dtype=q.dtype, pin_memory=True) for _ in range(3)]
    a = torch.randn(8192, 8192, device=dev)
    torch.cuda.synchronize()
    cur = torch.cuda.current_stream()
    for _ in range(3):
        a = a @ a / 8192.0  # a few milliseconds of work ahead of the copies
    for h, t in zip(hosts, (q, k, v)):
        h.copy_(t, non_blocking=True)
    out = clis.attention(*hosts, groups=2)
    torch.cuda.synchronize()
    ref = clis.attention(q, k, v)
    torch.cuda.synchronize()
    assert_paths_agree(flat(out.to(dev)), flat(ref), "host inputs from queued copies")
    del a, cur


def test_outputs_are_deterministic():
    dev = need_gpu()
    w = WORKLOADS["mixed"]
    q, k, v = make_inputs(w, device=dev, N=3000)
    a, _, _ = _run(q, k, v, False, "auto")
    b, _, _ = _run(q, k, v, False, "auto")
    assert torch.equal(a, b)


def test_bounded_wait_times_out_and_context_survives():
    """A kernel wait on a barrier that nothing arrives on gives up after its
    limit, reports through the device error word, and the next launches run
    normally (failure detection without a GPU fault)."""
    dev = need_gpu()
    clis.clis_clear_device_error()
    clis.clis_debug_wait_selftest(2000)
    code = clis.clis_get_device_error()
    assert code & (1 << 8), code
    clis.clis_clear_device_error()
    assert clis.clis_get_device_error() == 0
    w = WORKLOADS["tiny"]
    q, k, v = make_inputs(w, device=dev)
    out, _, _ = _run(q, k, v, False, "auto")
    ref, _ = _oracle(q, k, v, False)
    assert_close_to_oracle(out.float().cpu().numpy(), ref, "after selftest")
    assert clis.clis_get_device_error() == 0


def _chunked(q, k, v, bounds, variant, kbar=None, certs=None, lse2=True):
    sl2 = clis.scale_log2_for(q.shape[-1])
    BH, Nq, d = q.shape[0] * q.shape[1], q.shape[2], q.shape[3]
    o_acc = torch.full((BH * Nq, d), float("nan"), device=q.device)
    l_acc = torch.full((BH * Nq,), float("nan"), device=q.device)
    m_acc = torch.full((BH * Nq,), float("nan"), device=q.device)
    m_first = None
    for i, (a, b) in enumerate(zip(bounds[:-1], bounds[1:])):
        clis.clis_attn_fwd_chunk(q, k[:, :, a:b], v[:, :, a:b], sl2, o_acc, l_acc, m_acc, kbar=kbar, certs=certs,
                                 first=(i == 0), variant=variant)
        if i == 0:
            m_first = m_acc.clone()
    l2 = torch.full((BH * Nq,), float("nan"), device=q.device) if lse2 else None
    out = clis.clis_attn_chunk_finalize(q, o_acc, l_acc, m_acc, lse2=l2)
    torch.cuda.synchronize()
    return out, l2, m_first, m_acc


@pytest.mark.parametrize("variant", ["auto", "online", "online_lazy", "certified"])
def test_kv_chunk_merge_matches_full_attention(variant):
    """Ring-step form: K/V split into unequal chunks (with ragged ends), each
    merged into fp32 accumulators; the result must match the oracle on the
    whole sequence.  Certified heads keep the same shift in every chunk (their
    partials add with no rescaling)."""
    dev = need_gpu()
    w = WORKLOADS["mixed"]
    q, k, v = make_inputs(w, device=dev, N=4100, H=8)
    sl2 = clis.scale_log2_for(w.d)
    kbar, certs = clis.clis_certify(q, k, v, sl2)
    bounds = [0, 1300, 2048, 2049, 4100]
    if variant == "certified":
        heads = [h for h, c in enumerate(clis.decode_certs(certs)) if c["certified"]]
    else:
        heads = list(range(w.B * 8))
    out, l2, m_first, m_acc = _chunked(q, k, v, bounds, variant, kbar, certs)
    ref, rlse = _oracle(q, k, v, False)
    got = flat(out).float().cpu().numpy()
    assert_close_to_oracle(got[heads], ref[heads], f"chunked/{variant}")
    g2 = l2.cpu().numpy().reshape(rlse.shape)
    np.testing.assert_allclose(g2[heads], rlse[heads], atol=2e-3, rtol=0)
    flags = [c["certified"] for c in clis.decode_certs(certs)]
    assert 0 < sum(flags) < len(flags)
    if variant in ("auto", "certified"):
        rows = q.shape[2]
        for h, f in enumerate(flags):
            if f:  # fixed stabiliser: the shift never changed across chunks
                assert torch.equal(m_first[h * rows:(h + 1) * rows], m_acc[h * rows:(h + 1) * rows])


def test_kv_chunk_merge_is_deterministic():
    """Certified heads merge chunks with in-memory vector adds: one add per
    accumulator element per launch, so two identical passes agree bit for
    bit (mixed heads: the online ones read-modify-write)."""
    dev = need_gpu()
    w = WORKLOADS["mixed"]
    q, k, v = make_inputs(w, device=dev, N=5000, H=8)
    kbar, certs = clis.clis_certify(q, k, v, clis.scale_log2_for(w.d))
    bounds = [0, 700, 2500, 2501, 5000]
    a = _chunked(q, k, v, bounds, "auto", kbar, certs)
    b = _chunked(q, k, v, bounds, "auto", kbar, certs)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1]) and torch.equal(a[3], b[3])


def test_kv_chunk_single_chunk_equals_fused():
    dev = need_gpu()
    w = WORKLOADS["480p"]
    q, k, v = make_inputs(w, device=dev, N=3000, H=3)
    sl2 = clis.scale_log2_for(w.d)
    kbar, certs = clis.clis_certify(q, k, v, sl2)
    fused = clis.clis_attn_fwd(q, k, v, sl2, kbar=kbar, certs=certs)
    out, _, _, _ = _chunked(q, k, v, [0, 3000], "auto", kbar, certs, lse2=False)
    assert_paths_agree(flat(out), flat(fused), "single chunk")



@pytest.mark.parametrize("variant", ["auto", "online", "certified", "online_lazy"])
def test_fp16_full_parity(variant):
    """FP16 data with the 480p distributions (B_h ~ 5.5, within the FP16 budget
    C = 15), all rows checked.  (The tiny workload's B_h ~ 20 exceeds it: with
    fp16 data those heads do not certify.)"""
    dev = need_gpu()
    w = WORKLOADS["480p"]
    q, k, v = make_inputs(w, device=dev, N=777, H=2, dtype=torch.float16)
    out, l2, certs = _run(q, k, v, False, variant, lse2=True)
    assert out.dtype == torch.float16
    ref, rlse = _oracle(q, k, v, False)
    assert_close_to_oracle(out.float().cpu().numpy(), ref, f"fp16/{variant}")
    np.testing.assert_allclose(l2.cpu().numpy().reshape(rlse.shape), rlse, atol=1e-3, rtol=0)
    c = clis.decode_certs(certs)
    assert all(x["certified"] and x["C"] == 15 for x in c)


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal", [(1, 2, 1, 1, 64, False), (2, 3, 129, 129, 64, True),
                                                (1, 2, 1000, 257, 128, False), (2, 2, 700, 700, 128, True),
                                                (1, 4, 20000, 100, 128, False)])
@pytest.mark.parametrize("variant", ["auto", "online", "online_lazy"])
def test_fp16_ragged_shapes(B, H, Nq, Nk, d, causal, variant):
    dev = need_gpu()
    g = torch.Generator(device=dev)
    g.manual_seed(B * 7919 + H * 131 + Nq + Nk * 3 + d)
    q = torch.randn(B, H, Nq, d, generator=g, device=dev).half()
    k = (torch.randn(B, H, Nk, d, generator=g, device=dev) * 0.5 + 0.7).half()
    v = torch.randn(B, H, Nk, d, generator=g, device=dev).half()
    out, l2, _ = _run(q, k, v, causal, variant, lse2=True)
    ref, rlse = _oracle(q, k, v, causal)
    assert_close_to_oracle(out.float().cpu().numpy(), ref, f"fp16 {(B, H, Nq, Nk, d, causal)}/{variant}")
    np.testing.assert_allclose(l2.cpu().numpy().reshape(rlse.shape), rlse, atol=2e-3, rtol=0)


def test_fp16_auto_guard_with_bf16_budget():
    """Heads certified with the BF16 budget (B_h ~ 23 <= 127 - A) but not the FP16
    one: in AUTO with fp16 data they must run online softmax (fixed-stabiliser
    p would reach 2^23 and overflow FP16)."""
    dev = need_gpu()
    w = WORKLOADS["causal"]
    q, k, v = make_inputs(w, device=dev, N=1500, H=2, dtype=torch.float16)
    out, _, certs = _run(q, k, v, False, "auto", exp_fmt="bf16")
    c = clis.decode_certs(certs)
    assert all(x["certified"] for x in c) and all(x["B_h"] > 15 for x in c)
    assert torch.isfinite(out).all()
    ref, _ = _oracle(q, k, v, False)
    assert_close_to_oracle(out.float().cpu().numpy(), ref, "fp16 guard")


def test_fp16_kv_chunks():
    dev = need_gpu()
    w = WORKLOADS["480p"]
    q, k, v = make_inputs(w, device=dev, N=3000, H=3, dtype=torch.float16)
    sl2 = clis.scale_log2_for(w.d)
    kbar, certs = clis.clis_certify(q, k, v, sl2, exp_fmt="fp16")
    out, l2, _, _ = _chunked(q, k, v, [0, 1000, 1001, 3000], "auto", kbar, certs)
    assert out.dtype == torch.float16
    ref, rlse = _oracle(q, k, v, False)
    assert_close_to_oracle(flat(out).float().cpu().numpy(), ref, "fp16 chunked")
