"""Benchmark of the CLiS attention-forward hot path on GB300.

One step = the whole path over one batch of synthetic inputs resident in HBM:
clis_certify (Algorithm 1, four kernels) + clis_attn_fwd (AUTO: certified
heads on the fixed-stabiliser path, the rest on online softmax).  The metric
is attention-forward TFLOP/s, FLOP = 4 B H Nq Nk d (halved for causal).

Prints ONE JSON line (rank 0).  Default workload: the 720p Wan-2.2-shaped DiT
self-attention (B=1, H=40, N=75,600, d=128, non-causal).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
  python bench.py --impl reference ...   # the CPU fp64 oracle on a sample

Under torchrun each rank runs its own copy of the workload on its own GPU
(heads are independent: no collective on the data path; weak scaling).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from certified_fixed_stabilizer_gb300.workloads import WORKLOADS, make_dout, make_inputs, sample_rows  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
NOMINAL_BF16_TFLOPS = 2250.0       # GB300 dense BF16, vendor nominal
TENSOR_FLOP_PER_CLK_SM = 8192.0    # 2*128*128*16 FLOP per 64 cycles (tcgen05 kind::f16, measured)
METRIC = "attention fwd TFLOP/s (BF16, 1xGB300); CLiS step = certification + fused attention (AUTO)"


def config_dict(w, H, variant):
    in_bytes = 3 * w.B * H * w.N * w.d * 2
    l2 = ("flushed between steps (256 MB write)" if in_bytes < 2 * L2_BYTES
          else "inputs larger than L2 (Q, K, V %.0f MB each)" % (in_bytes / 3 / 1e6))
    return {"workload": workload_desc(w, H), "B": w.B, "H": H, "N": w.N, "d": w.d,
            "causal": w.causal, "variant": variant, "seed": w.seed, "l2": l2}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", default="720p", choices=sorted(WORKLOADS))
    ap.add_argument("--heads", type=int, default=None, help="override H (profiling runs)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--variant", default="auto", choices=["auto", "online", "certified", "online_lazy"])
    ap.add_argument("--dtype", default="bf16", choices=["bf16", "fp16"],
                    help="element type of Q, K, V, P and O (fp16 certifies with the FP16 exp2 budget)")
    ap.add_argument("--extras", default="all", choices=["all", "none", "backward", "chunks", "e2e", "tiles", "fp8", "gqa"],
                    help="legs after the headline step: all (online variants, ring-step chunks, backward, e2e, "
                         "CPU baseline, per-prefix certificates for causal configs, FP8 P.V for non-causal BF16 "
                         "configs, grouped-query attention with a quarter of the key/value heads for causal "
                         "configs), none, or only the backward, the ring-step chunks, the e2e leg, the per-prefix "
                         "leg, the FP8 P.V leg or the grouped-query leg (profiling runs)")
    ap.add_argument("--no-extras", action="store_true", help="same as --extras none")
    return ap.parse_args()


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def workload_desc(w, H):
    return (f"{w.name}: B={w.B} H={H} N={w.N} d={w.d} causal={w.causal} "
            f"({w.note})")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ------------------------------------------------------------------ CPU legs

def oracle_sample_step(q, k, v, w, heads, rows):
    """Oracle work for one sampled step: certification of the sampled heads
    (full length) and attention on `rows` of each sampled head."""
    import oracle
    # scale_log2 = softmax scale * log2(e), formed here so that the oracle legs
    # import nothing from the CUDA library's binding.
    sl2 = w.softmax_scale() * math.log2(math.e)
    qs, ks, vs = (t.reshape(-1, t.shape[2], t.shape[3])[heads] for t in (q, k, v))
    oracle.certify(qs, ks, vs, sl2)
    oracle.attention(qs, ks, vs, w.softmax_scale(), causal=w.causal, rows=rows)


def sample_flops(w, n_heads, rows):
    if w.causal:
        return sum(4.0 * (r + 1) * w.d for r in rows) * n_heads
    return 4.0 * len(rows) * w.N * w.d * n_heads


def cpu_sample_plan(q, k, v, w, target_s):
    """Pick a bounded sample (heads 0..1 and seed-chosen rows, or more heads when
    all their rows fit) taking about target_s."""
    import oracle
    oracle.build()
    oracle.set_num_threads(os.cpu_count() or 1)
    heads = [0, 1] if w.heads > 1 else [0]
    # A step costs a + b * rows: a is the certification over all keys, b one row's
    # attention.  Two probes separate the two so the sample lands near target_s.
    dts = []
    for n_probe in (32, 128):
        t0 = time.perf_counter()
        oracle_sample_step(q, k, v, w, heads, sample_rows(w.N, n_probe, seed=2))
        dts.append(time.perf_counter() - t0)
    per_row = max((dts[1] - dts[0]) / 96, 1e-6)
    fixed = max(dts[0] - 32 * per_row, 0.0)
    n = int(min(w.N, max(32, (target_s - fixed) / per_row)))
    total_heads = q.shape[0] * q.shape[1]
    if n >= w.N and total_heads > len(heads):
        # Every row of the sampled heads fits in the budget: sample more heads.
        t_all_rows = fixed + per_row * w.N
        nh = int(min(total_heads, max(len(heads), len(heads) * target_s / max(t_all_rows, 1e-6))))
        heads = list(range(nh))
    return heads, sample_rows(w.N, n, seed=2)


def run_reference(args, w, H):
    """--impl reference: the CPU oracle, as it stands, on a bounded sample."""
    ws, rank, _ = dist_setup()
    if rank != 0:
        return
    import oracle
    q, k, v = make_inputs(w, device="cuda" if torch.cuda.is_available() else "cpu", H=H)
    q, k, v = (t.cpu() for t in (q, k, v))
    heads, rows = cpu_sample_plan(q, k, v, w, target_s=4.0)
    for _ in range(args.warmup):
        oracle_sample_step(q, k, v, w, heads, rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_sample_step(q, k, v, w, heads, rows)
    dt = (time.perf_counter() - t0) / args.steps
    flops = sample_flops(w, len(heads), rows)
    val = flops / dt / 1e12
    sample = (f"certification of heads 0-{heads[-1]} ({len(heads)} of {q.shape[0] * q.shape[1]}) over all {w.N} "
              f"keys + attention rows ({len(rows)} seed-chosen query rows per head incl. 0 and N-1) of those heads")
    line = {
        "impl": "reference", "metric": METRIC, "value": val,
        "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": config_dict(w, H, args.variant),
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU legs

def main():
    args = parse()
    w = WORKLOADS[args.config]
    H = args.heads or w.H
    if args.impl == "reference":
        return run_reference(args, w, H)

    from certified_fixed_stabilizer_gb300 import clis
    ws, rank, local = dist_setup()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()

    dt = torch.float16 if args.dtype == "fp16" else torch.bfloat16
    exp_fmt = args.dtype
    q, k, v = make_inputs(w, device=dev, H=H, dtype=dt)
    heads = w.B * H
    flops = w.flops() * H / w.H
    sl2 = clis.scale_log2_for(w.d)
    shape = clis.make_shape(q, k, v)
    kbar = torch.empty((heads, w.d), dtype=torch.float32, device=dev)
    certs = torch.empty((heads, clis.CERT_WORDS), dtype=torch.int32, device=dev)
    wsp = torch.empty(max(256, clis.clis_certify_workspace_size(shape)), dtype=torch.uint8, device=dev)
    out = torch.empty_like(q)
    mu = torch.empty(heads * w.N, dtype=torch.float32, device=dev)  # per-row stabilisers
    in_bytes = 3 * q.numel() * q.element_size()
    needs_flush = in_bytes < 2 * L2_BYTES
    flush_buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if needs_flush else None

    def step(variant):
        if variant in ("auto", "certified"):
            clis.clis_certify(q, k, v, sl2, kbar=kbar, certs=certs, workspace=wsp, mu=mu, exp_fmt=exp_fmt)
        clis.clis_attn_fwd(q, k, v, sl2, kbar=kbar, certs=certs, causal=w.causal, variant=variant, out=out,
                           mu=mu)

    def timed_loop(variant, steps, warmup):
        for _ in range(warmup):
            step(variant)
        torch.cuda.synchronize()
        barrier(ws)
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
               torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for e0, e1, e2 in ev:
            if flush_buf is not None:
                flush_buf.zero_()
            e0.record(stream)
            if variant in ("auto", "certified"):
                clis.clis_certify(q, k, v, sl2, kbar=kbar, certs=certs, workspace=wsp, mu=mu, exp_fmt=exp_fmt)
            e1.record(stream)
            clis.clis_attn_fwd(q, k, v, sl2, kbar=kbar, certs=certs, causal=w.causal, variant=variant,
                               out=out, mu=mu)
            e2.record(stream)
        torch.cuda.synchronize()
        barrier(ws)
        torch.cuda.synchronize()
        step_ms = [e0.elapsed_time(e2) for e0, _, e2 in ev]
        cert_ms = [e0.elapsed_time(e1) for e0, e1, _ in ev]
        attn_ms = [e1.elapsed_time(e2) for _, e1, e2 in ev]
        return sum(step_ms), cert_ms, attn_ms

    clis.clis_clear_device_error()
    with ClockSampler(local) as cs:
        total_ms, cert_ms, attn_ms = timed_loop(args.variant, args.steps, args.warmup)
    clocks = cs.summary()
    total_ms = max_over_ranks(total_ms, ws)
    ms_per_step = total_ms / args.steps
    value = ws * flops / (ms_per_step * 1e-3) / 1e12
    attn_avg_ms = statistics.mean(attn_ms)
    cert_avg_ms = statistics.mean(cert_ms)
    n_cert = sum(c["certified"] for c in clis.decode_certs(certs))
    dev_err = clis.clis_get_device_error()

    peaks, peak_src = measured_peaks()
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    clock_peak = (TENSOR_FLOP_PER_CLK_SM * n_sm * clocks["sm_mhz"] * 1e6 / 1e12) if clocks["sm_mhz"] else None
    peak_tf = peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops"))
    achieved = flops / (attn_avg_ms * 1e-3) / 1e12
    traffic = None
    tfile = os.path.join(ROOT, "profiles", "attn_fwd_traffic.json")
    if os.path.exists(tfile):
        with open(tfile) as f:
            tinfo = json.load(f)
        if tinfo.get("config") == args.config and tinfo.get("kernel_rev") == kernel_rev():
            traffic = tinfo.get("bytes_per_launch")

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": args.dtype, "data": "synthetic",
        "config": config_dict(w, H, args.variant),
        "gpu_launches": args.steps * (5 if args.variant in ("auto", "certified") else 1),
        "certified_heads": f"{n_cert}/{heads}",
        "device_error_word": dev_err,
        "attention_only": {"value": achieved, "unit": "TFLOP/s", "ms": attn_avg_ms,
                           "median_ms": statistics.median(attn_ms)},
        "certify": {"ms": cert_avg_ms, "median_ms": statistics.median(cert_ms),
                    "gbs_algorithmic": in_bytes / (cert_avg_ms * 1e-3) / 1e9,
                    "gbs_moved": (in_bytes * 4 / 3) / (cert_avg_ms * 1e-3) / 1e9,
                    "frac_of_hbm_peak_moved": (in_bytes * 4 / 3) / (cert_avg_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                    "hbm_peak_gbs": peaks["hbm_gbs"]},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": achieved / peak_tf, "traffic": traffic,
                     "kernel": "attn_fwd_kernel<%d,%d,%d>" % (w.d, 1 if w.causal else 0, 1 if args.dtype == "fp16" else 0),
                     "peak_source": f"{peak_src} bf16_tflops_sustained (cuBLAS, seconds-long loop)",
                     # Two more denominators: the vendor's nominal dense BF16 figure, and the
                     # tensor pipe's instruction rate (a 128x128x16 MMA per 64 cycles per SM,
                     # measured) at the SM clock seen during the timed region.
                     "frac_of_nominal": achieved / NOMINAL_BF16_TFLOPS,
                     "nominal_peak": NOMINAL_BF16_TFLOPS,
                     "frac_of_clock_peak": (achieved / clock_peak) if clock_peak else None,
                     "clock_peak": clock_peak},
        "clocks": clocks,
    }

    extras = "none" if args.no_extras else args.extras
    if extras in ("all", "e2e"):
        # (Timed right after the headline step, in the same thermal and power
        # state, before the other legs heat the chip.)
        # End to end through the public call (clis.attention) with pinned host
        # buffers, which marshals them to the C ABI's clis_attention_host: every
        # step copies Q, K, V in, computes and copies O out, the library
        # pipelining head groups over a copy-in, two compute and a copy-out stream.
        qh, kh, vh = (t.cpu().pin_memory() for t in (q, k, v))
        oh = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)

        def e2e_step():
            clis.attention(qh, kh, vh, causal=w.causal, variant=args.variant, device=dev, out=oh,
                           non_blocking=True)

        for _ in range(max(1, args.warmup)):
            e2e_step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_e2e = max(1, min(args.steps, 10))
        with ClockSampler(local) as cs_e2e:
            e0.record(stream)
            e0.synchronize()  # the first step's copies are queued after the start mark
            for _ in range(n_e2e):
                e2e_step()
            stream.wait_event(clis.host_done_event(dev))  # after the last step's output copy
            e1.record(stream)
            torch.cuda.synchronize()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1) / n_e2e, ws)
        line["e2e"] = {"value": ws * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                       "h2d_bytes_per_step": in_bytes, "d2h_bytes_per_step": out.numel() * out.element_size(),
                       "ms_per_step": e2e_ms, "api": "certified_fixed_stabilizer_gb300.clis.attention -> clis_attention_host (C ABI, host buffers)",
                       "clocks": cs_e2e.summary()}
        del qh, kh, vh, oh
    if extras == "all":
        # Online-softmax baseline (same kernel skeleton, every head on the online path).
        on_total, _, on_attn = timed_loop("online", args.steps, args.warmup)
        line["online"] = {"value": flops / (statistics.mean(on_attn) * 1e-3) / 1e12, "unit": "TFLOP/s",
                          "ms": statistics.mean(on_attn)}
        line["certified_speedup_vs_online"] = statistics.mean(on_attn) / attn_avg_ms
        # FA4-style online baseline: rescale only when a row maximum grows by > 8.
        _, _, lz_attn = timed_loop("online_lazy", args.steps, args.warmup)
        line["online_lazy"] = {"value": flops / (statistics.mean(lz_attn) * 1e-3) / 1e12, "unit": "TFLOP/s",
                               "ms": statistics.mean(lz_attn)}
        line["certified_speedup_vs_online_lazy"] = statistics.mean(lz_attn) / attn_avg_ms
    if extras in ("all", "fp8") and not w.causal and args.dtype == "bf16" and w.d == 128:
        # FP8 P.V (E4M3 P and V for eligible certified heads; the others as in the
        # headline step).  A reduced-precision leg beside the BF16 headline: step =
        # certification + V -> E4M3 transpose + attention.
        vt8 = torch.empty((heads, w.d, -(-w.N // 16) * 16), dtype=torch.uint8, device=dev)
        fev = []
        for i in range(args.warmup + args.steps):
            if flush_buf is not None:
                flush_buf.zero_()
            e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
            e0.record(stream)
            clis.clis_certify(q, k, v, sl2, kbar=kbar, certs=certs, workspace=wsp, mu=mu, exp_fmt=exp_fmt)
            clis.clis_v_to_e4m3(v, vt8)
            e1.record(stream)
            clis.clis_attn_fwd_fp8pv(q, k, v, vt8, sl2, kbar=kbar, certs=certs, out=out, mu=mu)
            e2.record(stream)
            if i >= args.warmup:
                fev.append((e0, e1, e2))
        torch.cuda.synchronize()
        f_step = statistics.mean(a.elapsed_time(c) for a, _, c in fev)
        f_attn = statistics.mean(b.elapsed_time(c) for _, b, c in fev)
        n_f8 = sum(1 for c in clis.decode_certs(certs)
                   if c["certified"] and c["B_h"] <= min(8, c["C"]) and c["G"] <= 8 and w.N >= 4096)
        line["fp8_pv"] = {
            "value": flops / (f_step * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": f_step,
            "attention_only": flops / (f_attn * 1e-3) / 1e12, "attention_ms": f_attn,
            "prepass_ms": f_step - f_attn, "fp8_heads": f"{n_f8}/{heads}",
            "speedup_vs_bf16_attention": attn_avg_ms / f_attn,
            "precision": "P and V in E4M3 for the P.V product (kind::f8f6f4); Q K^T in BF16; fp32 accumulators"}
        del vt8
    if extras in ("all", "tiles") and w.causal:
        # Per-prefix certificates (clis_certify_tiles + clis_attn_fwd_tiles): query
        # blocks of heads that fail as a whole still take the fixed stabiliser
        # when their prefix certifies.  Same inputs, same timing as the step.
        nqb = -(-w.N // 256)
        tiles = torch.empty((heads, nqb), dtype=torch.uint8, device=dev)
        tev = []
        for i in range(args.warmup + args.steps):
            e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
            e0.record(stream)
            clis.clis_certify_tiles(q, k, v, sl2, kbar=kbar, certs=certs, tile_certs=tiles, workspace=wsp, mu=mu,
                                    exp_fmt=exp_fmt)
            e1.record(stream)
            clis.clis_attn_fwd_tiles(q, k, v, sl2, kbar, certs, tiles, out=out, mu=mu)
            e2.record(stream)
            if i >= args.warmup:
                tev.append((e0, e1, e2))
        torch.cuda.synchronize()
        t_step = statistics.mean(a.elapsed_time(c) for a, _, c in tev)
        t_attn = statistics.mean(b.elapsed_time(c) for _, b, c in tev)
        n_heads_cert = sum(c["certified"] for c in clis.decode_certs(certs))
        line["per_prefix"] = {
            "value": flops / (t_step * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": t_step,
            "attention_only": flops / (t_attn * 1e-3) / 1e12,
            "certified_blocks": f"{int(tiles.sum().item())}/{heads * nqb}",
            "blocks_of_certified_heads": f"{n_heads_cert * nqb}/{heads * nqb}",
            "speedup_vs_per_head_step": ms_per_step / t_step}
    if extras in ("all", "chunks"):
        # Ring-step form: K/V in 8 chunks, each merged into fp32 accumulators
        # (clis_attn_fwd_chunk), then clis_attn_chunk_finalize.  Certified heads
        # add their partials with no rescaling; online heads rescale per chunk.
        # Causal configs use clis_attn_fwd_chunk_causal: chunk c holds keys
        # bounds[c] .. bounds[c+1] - 1, and query blocks ending before its first
        # key are not launched.
        n_chunks = 8
        bounds = [round(i * w.N / n_chunks) for i in range(n_chunks + 1)]
        bounds = [b - b % 8 if 0 < b < w.N else b for b in bounds]
        o_acc = torch.empty((heads * w.N, w.d), dtype=torch.float32, device=dev)
        l_acc = torch.empty((heads * w.N,), dtype=torch.float32, device=dev)
        m_acc = torch.empty((heads * w.N,), dtype=torch.float32, device=dev)

        fp8_chunks = not w.causal and args.dtype == "bf16" and w.d == 128
        vt8s = ([torch.empty((heads, w.d, -(-(b - a) // 16) * 16), dtype=torch.uint8, device=dev)
                 for a, b in zip(bounds[:-1], bounds[1:])] if fp8_chunks else [])

        def chunk_pass(variant):
            for i, (a, b) in enumerate(zip(bounds[:-1], bounds[1:])):
                if variant == "fp8" and b - a >= 4096:
                    # FP8 P.V: each chunk's V converted to E4M3 as it arrives, then merged.
                    # (A chunk under 4096 keys runs BF16 on every head, so it is merged
                    # as in the certified pass, without a conversion.)
                    kc, vc = k[:, :, a:b], v[:, :, a:b]
                    clis.clis_v_to_e4m3(vc, vt8s[i])
                    clis.clis_attn_fwd_chunk_fp8pv(q, kc, vc, vt8s[i], sl2, o_acc, l_acc, m_acc, kbar=kbar,
                                                   certs=certs, first=(i == 0), mu=mu)
                elif w.causal:
                    clis.clis_attn_fwd_chunk_causal(q, k[:, :, a:b], v[:, :, a:b], sl2, o_acc, l_acc, m_acc, a,
                                                    kbar=kbar, certs=certs, first=(i == 0), variant=variant,
                                                    mu=mu)
                else:
                    clis.clis_attn_fwd_chunk(q, k[:, :, a:b], v[:, :, a:b], sl2, o_acc, l_acc, m_acc,
                                             kbar=kbar, certs=certs, first=(i == 0),
                                             variant="auto" if variant == "fp8" else variant, mu=mu)
            clis.clis_attn_chunk_finalize(q, o_acc, l_acc, m_acc, out=out)

        chunked = {"chunks": n_chunks, "causal": w.causal}
        for variant in ("auto", "online") + (("fp8",) if fp8_chunks else ()):
            for _ in range(args.warmup):
                chunk_pass(variant)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(args.steps):
                chunk_pass(variant)
            e1.record(stream)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / args.steps
            chunked[{"auto": "certified", "online": "online", "fp8": "certified_fp8_pv"}[variant]] = {
                "value": flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms": ms}
        chunked["certified_speedup_vs_online"] = chunked["online"]["ms"] / chunked["certified"]["ms"]
        if fp8_chunks:
            # (head, chunk) pairs on E4M3: eligible certified heads, chunks of 4096 keys or more.
            n_elig = sum(1 for c in clis.decode_certs(certs)
                         if c["certified"] and c["B_h"] <= min(8, c["C"]) and c["G"] <= 8)
            n_big = sum(1 for a, b in zip(bounds[:-1], bounds[1:]) if b - a >= 4096)
            chunked["certified_fp8_pv"]["fp8_head_chunks"] = f"{n_elig * n_big}/{heads * n_chunks}"
        line["chunked"] = chunked
        del o_acc, l_acc, m_acc, vt8s
    if extras in ("all", "backward"):
        # Backward (clis_attn_bwd: row dots, dK/dV kernel, dQ kernel) on the same
        # inputs, from a forward that also wrote lse2, for a seeded dO.  FLOPs
        # are the backward's five matmuls: 2.5 x the forward's count.
        lse2 = torch.empty(heads * w.N, dtype=torch.float32, device=dev)
        clis.clis_certify(q, k, v, sl2, kbar=kbar, certs=certs, workspace=wsp, mu=mu, exp_fmt=exp_fmt)
        clis.clis_attn_fwd(q, k, v, sl2, kbar=kbar, certs=certs, causal=w.causal, variant=args.variant, out=out,
                           mu=mu, lse2=lse2)
        dout = make_dout(q.shape, device=dev, dtype=dt)
        dq, dk, dv = (torch.empty_like(t) for t in (q, k, v))
        bws = torch.empty(max(256, clis.clis_attn_bwd_workspace_size(clis.make_shape(q, k, v, out))),
                          dtype=torch.uint8, device=dev)

        def bwd_step():
            clis.clis_attn_bwd(q, k, v, out, dout, lse2, sl2, causal=w.causal, dq=dq, dk=dk, dv=dv, workspace=bws)

        for _ in range(args.warmup):
            bwd_step()
        torch.cuda.synchronize()
        bev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for e0, e1 in bev:
            if flush_buf is not None:
                flush_buf.zero_()
            e0.record(stream)
            bwd_step()
            e1.record(stream)
        torch.cuda.synchronize()
        bwd_ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in bev)
        bwd_tf = 2.5 * flops / (bwd_ms * 1e-3) / 1e12
        line["backward"] = {"value": bwd_tf, "unit": "TFLOP/s", "ms": bwd_ms, "frac_of_peak": bwd_tf / peak_tf,
                            "launches_per_step": 3, "flops": "five matmuls (2.5x the forward's count)",
                            "fwd_plus_bwd_ms": attn_avg_ms + cert_avg_ms + bwd_ms}
        del dout, dq, dk, dv, bws, lse2
    if extras in ("all", "gqa") and w.causal and heads % (4 * w.B) == 0:
        # Grouped-query attention (the LLM training shape with one key/value head
        # per four query heads): Q as the headline's, K and V the first quarter of
        # the heads of each batch entry, shared through zero head strides.
        # Certification + forward, and the backward (whose dK/dV kernel sums each
        # group), on the same FLOP counts as the headline.
        hkv = heads // w.B // 4
        kg, vg = k[:, :hkv].contiguous(), v[:, :hkv].contiguous()
        qf, kf, vf, of = clis.grouped_query_views(q, kg, vg, out)
        lse2 = torch.empty(heads * w.N, dtype=torch.float32, device=dev)
        dout = make_dout(q.shape, device=dev, dtype=dt)
        dq, dkg, dvg = torch.empty_like(q), torch.empty_like(kg), torch.empty_like(vg)
        dqf, dkf, dvf, dof = clis.grouped_query_views(dq, dkg, dvg, dout)
        gws = torch.empty(max(256, clis.clis_certify_workspace_size(clis.make_shape(qf, kf, vf))), dtype=torch.uint8,
                          device=dev)
        bws = torch.empty(max(256, clis.clis_attn_bwd_workspace_size(clis.make_shape(qf, kf, vf, of))),
                          dtype=torch.uint8, device=dev)

        def gqa_fwd():
            clis.clis_certify(qf, kf, vf, sl2, kbar=kbar, certs=certs, workspace=gws, mu=mu, exp_fmt=exp_fmt)
            clis.clis_attn_fwd(qf, kf, vf, sl2, kbar=kbar, certs=certs, causal=True, variant=args.variant, out=of,
                               mu=mu, lse2=lse2)

        def gqa_bwd():
            clis.clis_attn_bwd(qf, kf, vf, of, dof, lse2, sl2, causal=True, dq=dqf, dk=dkf, dv=dvf, workspace=bws)

        res = {}
        for name, fn in (("forward", gqa_fwd), ("backward", gqa_bwd)):
            for _ in range(args.warmup):
                fn()
            torch.cuda.synchronize()
            gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(args.steps)]
            for e0, e1 in gev:
                if flush_buf is not None:
                    flush_buf.zero_()
                e0.record(stream)
                fn()
                e1.record(stream)
            torch.cuda.synchronize()
            ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in gev)
            mult = 2.5 if name == "backward" else 1.0
            res[name] = {"value": mult * flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms": ms}
        line["grouped_query"] = {"kv_heads_per_batch": hkv, "query_heads_per_kv_head": 4,
                                 "forward_step": res["forward"], "backward": res["backward"]}
        del kg, vg, lse2, dout, dq, dkg, dvg, gws, bws
    if rank == 0 and ws == 1 and extras == "all":
        # CPU baseline: the oracle on a bounded sample of this workload.
        import oracle
        qc, kc, vc = (t.cpu() for t in (q, k, v))
        hs, rows = cpu_sample_plan(qc, kc, vc, w, target_s=15.0)
        t0 = time.perf_counter()
        oracle_sample_step(qc, kc, vc, w, hs, rows)
        dt = time.perf_counter() - t0
        line["cpu_baseline"] = {
            "value": sample_flops(w, len(hs), rows) / dt / 1e12, "unit": "TFLOP/s",
            "cores": oracle.num_threads(), "kind": "oracle",
            "sample": (f"heads 0-{hs[-1]} ({len(hs)} of {qc.shape[0] * qc.shape[1]}): certification "
                       f"over all {w.N} keys + attention for {len(rows)} seed-chosen query rows per head; "
                       f"{dt:.1f} s")}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def kernel_rev() -> str:
    """Hash of the attention kernel source: a stored traffic figure only applies
    to the kernel it was captured from."""
    import hashlib
    p = os.path.join(ROOT, "certified_fixed_stabilizer_gb300", "csrc", "attn_fwd.cu")
    with open(p, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


if __name__ == "__main__":
    main()
