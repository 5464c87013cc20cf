"""Helpers shared by the GPU parity tests (comparison only, no method arithmetic)."""
import numpy as np
import pytest
import torch

MAX_ABS = 1e-2   # bf16 output vs fp64 oracle, per element (spec tolerance)
MEAN_ABS = 1e-3  # mean over a head


def need_gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a visible CUDA device")
    return torch.device("cuda:0")


def flat(t):
    """[B, H, N, d] -> [B*H, N, d] (contiguous copy on the same device)."""
    return t.reshape(-1, t.shape[-2], t.shape[-1])


def head_errors(got: np.ndarray, ref: np.ndarray):
    """Per-head (max, mean) abs error, divided by max(1, max |ref|) of the head.

    Heads whose outputs reach 2^12 (planted large V entries) cannot meet an
    absolute 1e-2 in bf16; dividing by the head's output magnitude keeps the
    bound absolute for ordinary heads and relative for those."""
    got = got.reshape(ref.shape[0], -1).astype(np.float64)
    ref = ref.reshape(ref.shape[0], -1)
    scale = np.maximum(1.0, np.abs(ref).max(axis=1))
    err = np.abs(got - ref) / scale[:, None]
    return err.max(axis=1), err.mean(axis=1)


def report(what: str, **values):
    """Append measured errors to the JSON-lines file named by CLIS_PARITY_REPORT (if set)."""
    import json
    import os
    path = os.environ.get("CLIS_PARITY_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"case": what, **values}) + "\n")


def assert_close_to_oracle(got: np.ndarray, ref: np.ndarray, what: str = ""):
    mx, mn = head_errors(got, ref)
    report(what, max_abs=float(mx.max()), mean_abs=float(mn.max()))
    assert np.all(np.isfinite(got)), f"{what}: non-finite outputs"
    assert mx.max() <= MAX_ABS, f"{what}: max abs err {mx.max():.3e} (head {mx.argmax()})"
    assert mn.max() <= MEAN_ABS, f"{what}: mean abs err {mn.max():.3e} (head {mn.argmax()})"
    return mx.max(), mn.max()


def assert_paths_agree(a, b, what: str = ""):
    """Certified and online outputs (same heads) agree within the oracle bound,
    per head, errors divided by max(1, max |b|) of the head: two bf16 results
    may differ by one bf16 ulp, which is 2^-6 for |O| in [2, 4)."""
    a = a.reshape(a.shape[0], -1).float()
    b = b.reshape(b.shape[0], -1).float()
    scale = torch.clamp(b.abs().amax(dim=1), min=1.0)
    err = (a - b).abs() / scale[:, None]
    mx, mn = err.amax().item(), err.mean(dim=1).amax().item()
    assert mx <= MAX_ABS, f"{what}: paths differ by {mx:.3e} (max)"
    assert mn <= MEAN_ABS, f"{what}: paths differ by {mn:.3e} (mean)"


# Gradients (dQ, dK, dV) vs the fp64 oracle, per head, errors divided by the
# head's max |ref| of that gradient: (max, mean) bounds per gradient.  The
# kernels round P and dS to the input format before the matmuls and the
# outputs once more; tests/test_bwd_tolerance.py applies exactly those
# roundings on the CPU and shows they alone stay within half of these bounds.
# dQ gets the widest bound: dQ_i = scale sum_j dS_ij k_j where the keys share
# a large per-head bias that cancels in exact arithmetic (sum_j dS_ij = 0) but
# not in the bf16-rounded dS (up to 4.1e-2 of max |dQ| over 320 diffuse heads).
# dK's bound covers causal heads whose early rows one key dominates: the
# certified forward gives that key's weight 2^x its bf16 rounding, so O and
# D_i = dO_i . O_i are off by up to 2^-9 relative and the key's dK collects it
# from every such row (up to 1.9e-2 of max |dK| over 320 short causal heads).
GRAD_TOL = {"dq": (9e-2, 5e-3), "dk": (4e-2, 2e-3), "dv": (1.2e-2, 2e-3)}


def grad_errors(got: np.ndarray, ref: np.ndarray):
    """Per-head (max, mean) abs error divided by the head's max |ref|."""
    got = got.reshape(ref.shape[0], -1).astype(np.float64)
    ref = ref.reshape(ref.shape[0], -1)
    scale = np.maximum(np.abs(ref).max(axis=1), 1e-30)
    err = np.abs(got - ref) / scale[:, None]
    return err.max(axis=1), err.mean(axis=1)


def assert_grads_close(got: np.ndarray, ref: np.ndarray, which: str, what: str = ""):
    """which: "dq", "dk" or "dv" (selects the bound)."""
    tmax, tmean = GRAD_TOL[which]
    mx, mn = grad_errors(got, ref)
    report(f"{what} {which}", max_rel=float(mx.max()), mean_rel=float(mn.max()))
    assert np.all(np.isfinite(got)), f"{what} {which}: non-finite gradients"
    assert mx.max() <= tmax, f"{what} {which}: max err {mx.max():.3e} of max|ref| (head {mx.argmax()})"
    assert mn.max() <= tmean, f"{what} {which}: mean err {mn.max():.3e} of max|ref| (head {mn.argmax()})"
    return mx.max(), mn.max()


# Tight check of the backward kernels against tests/rounding_model.py, which
# applies the kernels' own bf16 roundings to an fp64 computation from the same
# O and lse2.  What remains is fp32 accumulation order and the hardware exp2
# (relative 1e-6 or so on P and dP), plus the bf16 roundings of P and dS that
# those tip over and the final rounding of each gradient.  Per head and
# gradient, errors divided by the head's max |reference|:
#   max over elements of (|got - e| - 2^-8 |e|), e the model's gradient before
#   its final rounding (2^-8 |e| covers that rounding): TIGHT_TOL[.][0];
#   mean over elements of |got - bf16(e)|: TIGHT_TOL[.][1].
# tests/test_bwd_tolerance.py derives them: relative noise of 1e-5 (five times
# the fp32 error estimate) on P and dP before the roundings stays within them
# on the short-causal and diffuse populations, while a 3% slip in one gradient
# or a D_i dropped from a few rows exceeds them (the fp64-oracle bounds of
# GRAD_TOL let both pass).
TIGHT_TOL = {"dq": (1e-2, 5e-4), "dk": (5e-3, 5e-4), "dv": (5e-3, 5e-4)}


def tight_errors(got: np.ndarray, model: np.ndarray):
    """Per-head (max excess over half an ulp, mean abs) error of bf16 `got`
    against the rounding model's unrounded gradient, divided by max |model|."""
    import torch
    got = got.reshape(model.shape[0], -1).astype(np.float64)
    e = model.reshape(model.shape[0], -1)
    eb = torch.from_numpy(e.astype(np.float32)).to(torch.bfloat16).double().numpy()
    scale = np.maximum(np.abs(e).max(axis=1), 1e-30)
    excess = np.maximum(np.abs(got - e) - np.abs(e) * 2.0 ** -8, 0.0) / scale[:, None]
    mean = np.abs(got - eb).mean(axis=1) / scale
    return excess.max(axis=1), mean


def assert_grads_tight(got: np.ndarray, model: np.ndarray, which: str, what: str = ""):
    tmax, tmean = TIGHT_TOL[which]
    mx, mn = tight_errors(got, model)
    report(f"{what} {which} tight", max_excess=float(mx.max()), mean_rel=float(mn.max()))
    assert np.all(np.isfinite(got)), f"{what} {which}: non-finite gradients"
    assert mx.max() <= tmax, f"{what} {which}: max excess {mx.max():.3e} of max|model| (head {mx.argmax()})"
    assert mn.max() <= tmean, f"{what} {which}: mean err {mn.max():.3e} of max|model| (head {mn.argmax()})"
    return mx.max(), mn.max()
