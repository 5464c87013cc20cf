"""Rounding model of the certified forward and of the backward kernels (test
infrastructure; CPU, numpy fp64).

The kernels compute in fp32 and round to the input format (bf16) at a few
fixed points.  This module applies exactly those roundings to an otherwise
fp64 computation, so its results differ from the kernels' only by fp32
accumulation order and the hardware exp2 (relative 1e-6 or less on any
intermediate) and by the bf16 roundings those differences tip over.  It is
written from the arithmetic each kernel performs, not from the kernels' code,
and is used two ways: to derive the fp64-oracle tolerances (how far these
roundings alone move a result from the exact one) and, in the tight GPU
checks, as the element-wise reference for the kernels themselves.

Rounding points:
  forward (certified path): p = exp2(scale_log2 * s - mu_i) with
      mu_i = scale_log2 * (q_i . kbar); P rounded to bf16 for the P V product;
      row sum l of the unrounded p; O = O_acc / l rounded to bf16 once;
      lse2 = mu_i + log2 l in fp32.
  backward: P = exp2(scale_log2 * s - lse2_i) from the given lse2; P rounded
      to bf16 for dV = P^T dO; dS = P (dP - D_i) with the unrounded P, rounded
      to bf16 for dQ = scale dS K and dK = scale dS^T Q; D_i = dO_i . O_i from
      the given (bf16) O; dQ, dK, dV rounded to bf16 once at the end (the
      functions below return them before that last rounding).
"""
from __future__ import annotations

import numpy as np
import torch

LOG2E = 1.4426950408889634


def bf16(x) -> np.ndarray:
    """Round to the nearest bf16 value (ties to even); returns float64."""
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).double().numpy()


def _mask(x: np.ndarray, causal: bool) -> np.ndarray:
    if not causal:
        return x
    nq, nk = x.shape
    return np.where(np.arange(nk)[None, :] <= np.arange(nq)[:, None], x, -np.inf)


def certified_forward(q, k, v, scale: float, causal: bool):
    """One head: (O as bf16 values, lse2 as fp32 values), both float64 arrays."""
    sl2 = scale * LOG2E
    mu = sl2 * (q @ k.mean(axis=0))
    p = np.exp2(_mask(sl2 * (q @ k.T) - mu[:, None], causal))
    l = p.sum(axis=1)
    o = bf16((bf16(p) @ v) / l[:, None])
    lse2 = (mu + np.log2(l)).astype(np.float32).astype(np.float64)
    return o, lse2


def backward(q, k, v, o, g, lse2, scale: float, causal: bool):
    """One head: dQ, dK, dV before their final rounding to bf16 (float64)."""
    sl2 = scale * LOG2E
    P = np.exp2(_mask(sl2 * (q @ k.T) - lse2[:, None], causal))
    D = (g * o).sum(axis=1, keepdims=True)
    dV = bf16(P).T @ g
    dS = bf16(P * (g @ v.T - D))
    return scale * (dS @ k), scale * (dS.T @ q), dV


def e4m3(x) -> np.ndarray:
    """Round to the nearest E4M3 value (ties to even), saturating at +-448."""
    x = np.clip(np.asarray(x, dtype=np.float32), -448.0, 448.0)
    return torch.from_numpy(x).to(torch.float8_e4m3fn).float().double().numpy()


def certified_forward_fp8pv(q, k, v, scale: float, rows=None, with_flip_bound=False):
    """One head, no mask, on the FP8 P.V path: p = exp2(scale_log2 * s - mu_i)
    rounded to E4M3 for the P V product with V rounded to E4M3, the row sum of
    the unrounded p, O rounded to bf16.  Returns (O before its final rounding,
    lse2) for the given rows (default all).

    with_flip_bound: also return how far one E4M3 rounding decision that goes
    the other way can move an output: one E4M3 step (at most 2^-3 of the
    weight) times the largest normalised weight p_ij / l_i of the head times
    max |V|.  A kernel whose fp32 p differs from this model's by a few ulp
    takes the other rounding now and then; with few keys per row one such
    decision dominates the difference."""
    sl2 = scale * LOG2E
    qr = q if rows is None else q[rows]
    mu = sl2 * (qr @ k.mean(axis=0))
    p = np.exp2(sl2 * (qr @ k.T) - mu[:, None])
    l = p.sum(axis=1)
    o = (e4m3(p) @ e4m3(v)) / l[:, None]
    if with_flip_bound:
        flip = 2.0 ** -3 * float((p / l[:, None]).max()) * float(np.abs(v).max())
        return o, mu + np.log2(l), flip
    return o, mu + np.log2(l)
