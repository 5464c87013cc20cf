"""Seeded synthetic inputs for CLiS attention forward.

This module holds the workload definitions and random-number recipes only:
shapes, value distributions, seeds, head selection for injected outliers and
sampled query rows.  It contains none of the method's arithmetic, so both the
CUDA path and the CPU oracle can consume what it produces.

The paper measures on Wan 2.2 / LTX-2 video DiT self-attention and causal LLM
training (Tables 1, 3, 7, 8); none of those models or datasets is available,
so these tensors stand in for them with the paper's shapes (H=40, S=75,600,
D=128 at 720p x 81 frames, Table 7; 32,760 tokens at 480p x 81 frames,
Table 8) and simple Gaussian value distributions.

Layout of every tensor: [B, H, N, d], bf16 (or fp16 on request), d contiguous.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    q_sigma: float        # Q ~ q_sigma * N(0, 1)
    k_sigma: float        # K ~ k_sigma * N(0, 1) + per-head bias
    bias_sigma: float     # per-head key bias vector ~ N(0, bias_sigma^2), shared by all keys
    v_sigma: float = 1.0  # V ~ v_sigma * N(0, 1)
    inject_frac: float = 0.0   # fraction of (b, h) heads that get outliers
    outlier_frac: float = 0.0  # fraction of key rows scaled in an injected head
    outlier_scale: float = 64.0
    v_inject_max: float = 4096.0  # largest |V| entry planted in an injected head
    late_outliers: bool = False   # outlier keys are the head's last rows instead of random ones
    seed: int = 0
    note: str = field(default="", compare=False)

    @property
    def heads(self) -> int:
        return self.B * self.H

    def flops(self) -> float:
        """4 * B * H * Nq * Nk * d, halved for the causal mask (both matmuls only)."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2.0 if self.causal else f

    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


WORKLOADS = {
    # Tiny correctness case: the CPU oracle finishes it in about a second.
    "tiny": Workload("tiny", B=1, H=2, N=256, d=64, causal=False,
                     q_sigma=1.0, k_sigma=1.0, bias_sigma=2.0,
                     note="Q,K,V ~ N(0,1), per-head key offset ~ N(0,4)"),
    # Wan-2.2-shaped 480p DiT self-attention: 21x30x52 latent grid.
    "480p": Workload("480p", B=1, H=20, N=32760, d=128, causal=False,
                     q_sigma=0.5, k_sigma=0.5, bias_sigma=2.0,
                     note="Q,K ~ 0.5 N(0,1), key bias ~ N(0,4), V ~ N(0,1)"),
    # Wan-2.2-shaped 720p DiT self-attention: 21x45x80 latent grid (81 frames, 1280x720).
    "720p": Workload("720p", B=1, H=40, N=75600, d=128, causal=False,
                     q_sigma=0.5, k_sigma=0.5, bias_sigma=2.0,
                     note="same distributions as 480p"),
    # Mixed certification: a seed-chosen 25% of heads get 0.1% outlier keys (x64)
    # and V entries up to 2^12, so they fail certification.
    "mixed": Workload("mixed", B=2, H=32, N=24576, d=128, causal=False,
                      q_sigma=0.5, k_sigma=0.5, bias_sigma=2.0,
                      inject_frac=0.25, outlier_frac=0.001,
                      note="480p distributions plus outlier injection in 16 of 64 heads"),
    # Causal-LLM training-shaped forward.
    "causal": Workload("causal", B=4, H=32, N=8192, d=128, causal=True,
                       q_sigma=1.0, k_sigma=1.0, bias_sigma=math.sqrt(2.0),
                       note="Q,K ~ N(0,1), key bias ~ N(0,2), V ~ N(0,1), causal"),
    # The causal shape with large keys at the end of a seed-chosen 25% of heads
    # (the last 1% of rows x 64, plus the mixed workload's V entries): those heads
    # fail the per-head certificate, while every query block whose prefix ends
    # before the large keys certifies by its prefix (clis_certify_tiles).
    "causal_late": Workload("causal_late", B=4, H=32, N=8192, d=128, causal=True,
                            q_sigma=1.0, k_sigma=1.0, bias_sigma=math.sqrt(2.0),
                            inject_frac=0.25, outlier_frac=0.01, late_outliers=True,
                            note="causal distributions, last 1% of keys x64 in 32 of 128 heads"),
}


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def injected_heads(w: Workload) -> list[int]:
    """Seed-chosen flat (b*H + h) indices of heads that receive outliers."""
    n = int(round(w.inject_frac * w.heads))
    if n == 0:
        return []
    g = _gen("cpu", w.seed + 7919)
    return sorted(torch.randperm(w.heads, generator=g)[:n].tolist())


def make_inputs(w: Workload, device="cpu", seed: int | None = None, N: int | None = None,
                H: int | None = None, dtype=torch.bfloat16):
    """Generate (q, k, v) tensors of shape [B, H, N, d] for workload ``w``.

    Values are drawn in fp32 with a seeded torch.Generator on ``device`` and
    rounded to ``dtype`` (bf16 by default, or fp16; nearest even).  ``N`` /
    ``H`` override the sequence length / head count (reduced-size copies of a
    workload for tests and profiling; injected heads are then chosen among the
    heads that exist).
    """
    seed = w.seed if seed is None else seed
    N = w.N if N is None else N
    H = w.H if H is None else H
    dev = torch.device(device)
    g = _gen(dev, seed)
    shape = (w.B, H, N, w.d)
    q = torch.empty(shape, dtype=dtype, device=dev)
    k = torch.empty(shape, dtype=dtype, device=dev)
    v = torch.empty(shape, dtype=dtype, device=dev)
    # One head at a time keeps the fp32 temporaries small at 720p.
    for b in range(w.B):
        for h in range(H):
            bias = torch.randn(w.d, generator=g, device=dev) * w.bias_sigma
            q[b, h] = (torch.randn(N, w.d, generator=g, device=dev) * w.q_sigma).to(dtype)
            k[b, h] = (torch.randn(N, w.d, generator=g, device=dev) * w.k_sigma + bias).to(dtype)
            v[b, h] = (torch.randn(N, w.d, generator=g, device=dev) * w.v_sigma).to(dtype)
    if w.inject_frac > 0:
        _inject(w, q, k, v, seed)
    return q, k, v


def make_dout(shape, device="cpu", seed: int = 0, dtype=torch.bfloat16, sigma: float = 1.0):
    """Upstream gradient dO ~ sigma * N(0, 1) of the given [B, H, N, d] shape
    (the backward's input; a training loss would supply it)."""
    g = _gen(torch.device(device), seed + 65537)
    return (torch.randn(tuple(shape), generator=g, device=device) * sigma).to(dtype)


def _inject(w: Workload, q, k, v, seed: int) -> None:
    """Plant outlier keys (x outlier_scale, exact in bf16 for a power of two)
    and large V entries (magnitude uniform in [1, v_inject_max], one entry
    exactly +-v_inject_max) into the heads chosen by :func:`injected_heads`."""
    H, N = k.shape[1], k.shape[2]
    g = _gen("cpu", seed + 104729)
    n_out = max(1, math.ceil(w.outlier_frac * N))
    for flat in injected_heads(w):
        b, h = divmod(flat, w.H)
        if h >= H:
            continue
        rows = torch.randperm(N, generator=g)[:n_out]
        if w.late_outliers:
            rows = torch.arange(N - n_out, N)
        rows = rows.to(k.device)
        k[b, h, rows] = (k[b, h, rows].float() * w.outlier_scale).to(k.dtype)
        n_v = 8
        vr = torch.randint(0, N, (n_v,), generator=g)
        vc = torch.randint(0, w.d, (n_v,), generator=g)
        mag = 1.0 + torch.rand(n_v, generator=g) * (w.v_inject_max - 1.0)
        sgn = torch.where(torch.rand(n_v, generator=g) < 0.5, -1.0, 1.0)
        vals = mag * sgn
        vals[0] = w.v_inject_max * sgn[0]
        for t in range(n_v):
            v[b, h, int(vr[t]), int(vc[t])] = float(vals[t])


def injected_heads_present(w: Workload, H: int | None = None) -> list[int]:
    """Flat head indices that actually received outliers for head count ``H``."""
    H = w.H if H is None else H
    out = []
    for flat in injected_heads(w):
        b, h = divmod(flat, w.H)
        if h < H:
            out.append(b * H + h)
    return out


def sample_rows(N: int, n: int, seed: int = 0, tile: int = 128) -> list[int]:
    """Seed-chosen query rows for sampled checks: always rows 0 and N-1, the
    first row of the last (possibly ragged) 128-row tile and its neighbours,
    plus uniformly drawn rows; sorted, unique."""
    base = {0, N - 1}
    last_tile = (N - 1) // tile * tile
    base.update({last_tile, min(N - 1, last_tile + 1), max(0, last_tile - 1)})
    g = _gen("cpu", seed + 31337)
    extra = torch.randint(0, N, (max(0, n - len(base)),), generator=g).tolist()
    return sorted(base.union(extra))
