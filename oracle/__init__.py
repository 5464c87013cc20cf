"""CPU fp64 oracle for CLiS attention forward -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never touches it, and the two share no code.

What it computes (each routine cites the passage it follows):

* :func:`certify` -- Algorithm 1 steps 1-7 of "CLiS: Plug-and-Play Attention
  Acceleration for Video Diffusion on TPUs via Certified Stabilization"
  (k-bar, centred-key norm bound kappa, score bound B_h, V exponent G,
  accumulator exponent A, exponent budget C), then the certification decision
  (all inputs finite and B_h <= C; the step after 7 is lost from the pages, so
  this is a stated reading).
* :func:`attention` -- plain softmax attention, O_i = sum_j softmax_j(scale *
  q_i.k_j) v_j, computed in fp64 with two passes per row.  A fixed stabiliser
  cancels exactly in real arithmetic, so this definition is the result both
  CLiS kernels must reproduce.
* :func:`attention_bwd` -- gradients dQ, dK, dV of sum_i dO_i . O_i for the
  same attention, by the plain chain rule through softmax (the pages give no
  backward algorithm; their causal LLM training results, Table 3, need one).

The arithmetic lives in ``clis_oracle.c``; this module only builds it with
gcc and marshals numpy arrays.  Every function here is pinned by the
``-m "not gpu"`` tests in ``tests/test_oracle_pins.py`` (brute force,
closed forms, identities, hand-built boundary heads).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "clis_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libclis_oracle.so")

FMT = {"fp16": 0, "bf16": 1, "fp32": 2, "e4m3": 3}

_lib = None
_lock = threading.Lock()


class OracleCert(ctypes.Structure):
    _fields_ = [
        ("certified", ctypes.c_int32),
        ("G", ctypes.c_int32),
        ("A", ctypes.c_int32),
        ("C", ctypes.c_int32),
        ("reason", ctypes.c_int32),
        ("band", ctypes.c_int32),
        ("B_h", ctypes.c_double),
        ("kappa", ctypes.c_double),
        ("qmax", ctypes.c_double),
        ("vmax", ctypes.c_double),
    ]


def build(force: bool = False) -> str:
    """Compile clis_oracle.c into a shared library with gcc (-O2, OpenMP)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64, i32, dbl, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
        lib.oracle_certify.argtypes = [i64, i64, i64, i64, vp, vp, vp, i32, dbl, i32, i32, vp, vp]
        lib.oracle_certify.restype = i32
        lib.oracle_certify_prefix_tiles.argtypes = [i64, i64, i64, i64, vp, vp, vp, i32, dbl, i32, i32, vp, vp,
                                                    vp]
        lib.oracle_certify_prefix_tiles.restype = i32
        for name in ("oracle_attn_bf16", "oracle_attn_fp16", "oracle_attn_f64"):
            f = getattr(lib, name)
            f.argtypes = [i64, i64, i64, i64, vp, vp, vp, dbl, i32, i64, vp, vp, vp]
            f.restype = i32
        for name in ("oracle_attn_bwd_bf16", "oracle_attn_bwd_fp16", "oracle_attn_bwd_f64"):
            f = getattr(lib, name)
            f.argtypes = [i64, i64, i64, i64, vp, vp, vp, vp, dbl, i32, vp, vp, vp]
            f.restype = i32
        lib.oracle_attn_bwd_dq_rows.argtypes = [i32, i64, i64, i64, i64, vp, vp, vp, vp, dbl, i32, i64, vp, vp]
        lib.oracle_attn_bwd_dq_rows.restype = i32
        lib.oracle_format_log2_max.argtypes = [i32]
        lib.oracle_format_log2_max.restype = dbl
        lib.oracle_ceil_log2_count.argtypes = [i64]
        lib.oracle_ceil_log2_count.restype = ctypes.c_int32
        lib.oracle_v_exponent.argtypes = [dbl]
        lib.oracle_v_exponent.restype = ctypes.c_int32
        lib.oracle_exponent_budget.argtypes = [i32, i32, ctypes.c_int32]
        lib.oracle_exponent_budget.restype = ctypes.c_int32
        lib.oracle_decode.argtypes = [ctypes.c_uint16, i32]
        lib.oracle_decode.restype = dbl
        lib.oracle_num_threads.restype = i32
        lib.oracle_set_num_threads.argtypes = [i32]
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


IN_FMT = {"bf16": 0, "fp16": 1}


def as_bits(x):
    """bf16 / fp16 torch tensor (any device), numpy float16 array or uint16 bf16
    bit array -> (contiguous uint16 numpy bits, input format name)."""
    if isinstance(x, np.ndarray):
        if x.dtype == np.float16:
            return np.ascontiguousarray(x).view(np.uint16), "fp16"
        if x.dtype != np.uint16:
            raise TypeError("expected bf16 bit patterns as uint16 or a float16 array")
        return np.ascontiguousarray(x), "bf16"
    import torch
    if x.dtype not in (torch.bfloat16, torch.float16):
        raise TypeError("expected a bfloat16 or float16 tensor")
    fmt = "bf16" if x.dtype == torch.bfloat16 else "fp16"
    return x.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16), fmt


def as_bf16_bits(x) -> np.ndarray:
    """bf16 torch tensor (any device) or uint16 array -> contiguous uint16 numpy bits."""
    bits, fmt = as_bits(x)
    if fmt != "bf16":
        raise TypeError("expected bf16 data")
    return bits


def decode(bits: int, fmt: str) -> float:
    """One bf16 / fp16 bit pattern -> its exact value (as the oracle reads it)."""
    return _load().oracle_decode(int(bits), IN_FMT[fmt])


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _heads_first(a: np.ndarray) -> np.ndarray:
    """[..., N, d] -> contiguous [prod(...), N, d] (works for N = 0)."""
    lead = int(np.prod(a.shape[:-2])) if a.ndim > 2 else 1
    return np.ascontiguousarray(a.reshape(lead, a.shape[-2], a.shape[-1]))


# --- Figure 3 limits and Algorithm 1 steps 5-7 as scalar functions ----------

def format_log2_max(fmt: str) -> float:
    """U for a format: log2 of its largest finite value (exp2 limit, Figure 3)."""
    return _load().oracle_format_log2_max(FMT[fmt])


def ceil_log2_count(n: int) -> int:
    """Least a >= 0 with 2^a >= n (the ceil(log2 N_k) of Algorithm 1 step 6)."""
    return _load().oracle_ceil_log2_count(n)


def v_exponent(m: float) -> int:
    """G = ceil(log2 max(1, m)) (Algorithm 1 step 5)."""
    return _load().oracle_v_exponent(m)


def exponent_budget(exp_fmt: str, acc_fmt: str, A: int) -> int:
    """C = min(floor(U_exp), ceil(U_acc - A) - 1) (Algorithm 1 step 7)."""
    return _load().oracle_exponent_budget(FMT[exp_fmt], FMT[acc_fmt], A)


def certify(q, k, v, scale_log2: float, exp_fmt: str = "bf16", acc_fmt: str = "fp32"):
    """Algorithm 1 for every head.

    q: [BH, Nq, d], k, v: [BH, Nk, d] (bf16 or fp16 tensors, or uint16 bf16 bit
    arrays; a leading [B, H] pair is flattened).  Returns (kbar [BH, d] float64,
    list of dicts with certified, G, A, C, reason, band, B_h, kappa, qmax, vmax).
    """
    (qb, fq), (kb, fk), (vb, fv) = (as_bits(t) for t in (q, k, v))
    if not fq == fk == fv:
        raise TypeError("q, k, v must share one format")
    qb, kb, vb = (_heads_first(a) for a in (qb, kb, vb))
    d = qb.shape[-1]
    BH, Nq, Nk = qb.shape[0], qb.shape[1], kb.shape[1]
    kbar = np.zeros((BH, d), dtype=np.float64)
    certs = (OracleCert * max(BH, 1))()
    rc = _load().oracle_certify(BH, Nq, Nk, d, _ptr(qb), _ptr(kb), _ptr(vb), IN_FMT[fq],
                                float(scale_log2), FMT[exp_fmt], FMT[acc_fmt],
                                _ptr(kbar), ctypes.cast(certs, ctypes.c_void_p))
    if rc != 0:
        raise ValueError(f"oracle_certify rejected its arguments (rc={rc})")
    out = []
    for h in range(BH):
        c = certs[h]
        out.append({f: getattr(c, f) for f, _ in OracleCert._fields_})
    return kbar, out


def certify_prefix_tiles(q, k, v, scale_log2: float, tile_rows: int = 256, exp_fmt: str = "bf16",
                         acc_fmt: str = "fp32"):
    """Per-prefix certificates of causal heads (Nq == Nk), one per block of
    ``tile_rows`` query rows: block b is certified when every input of the head
    is finite and B_b = scale_log2 * max_{i in b} ||q_i|| * max_{j <= last row of
    b} ||k_j - kbar|| <= C, the head's budget.  Returns (certified, band, B),
    each [BH, ceil(N / tile_rows)] (int32, int32, float64)."""
    (qb, fq), (kb, fk), (vb, fv) = (as_bits(t) for t in (q, k, v))
    if not fq == fk == fv:
        raise TypeError("q, k, v must share one format")
    qb, kb, vb = (_heads_first(a) for a in (qb, kb, vb))
    BH, N, d = qb.shape
    if kb.shape[1] != N:
        raise ValueError("per-prefix certificates are for causal heads (Nq == Nk)")
    nb = -(-N // tile_rows)
    cert = np.zeros((BH, nb), dtype=np.int32)
    band = np.zeros((BH, nb), dtype=np.int32)
    B = np.zeros((BH, nb), dtype=np.float64)
    rc = _load().oracle_certify_prefix_tiles(BH, N, d, int(tile_rows), _ptr(qb), _ptr(kb), _ptr(vb), IN_FMT[fq],
                                             float(scale_log2), FMT[exp_fmt], FMT[acc_fmt], _ptr(cert), _ptr(band),
                                             _ptr(B))
    if rc != 0:
        raise ValueError(f"oracle_certify_prefix_tiles rejected its arguments (rc={rc})")
    return cert, band, B


def attention(q, k, v, scale: float, causal: bool = False, rows=None,
              with_lse2: bool = False):
    """fp64 softmax attention (two passes per row).

    q: [BH, Nq, d], k, v: [BH, Nk, d] as bf16 / fp16 tensors, uint16 bf16 bits,
    or float64 arrays (then the inputs are used as given).  ``scale`` multiplies
    q.k inside exp (natural base).  ``rows``: query indices to evaluate (the
    same for every head) or None for all.  Returns out [BH, n_rows, d] and,
    if requested, lse2 [BH, n_rows] = log2 sum_j exp(scale q_i.k_j).
    """
    f64 = isinstance(q, np.ndarray) and q.dtype == np.float64
    if f64:
        qa, ka, va = (np.ascontiguousarray(t, dtype=np.float64) for t in (q, k, v))
        fn = _load().oracle_attn_f64
    else:
        (qa, fq), (ka, fk), (va, fv) = (as_bits(t) for t in (q, k, v))
        if not fq == fk == fv:
            raise TypeError("q, k, v must share one format")
        fn = _load().oracle_attn_fp16 if fq == "fp16" else _load().oracle_attn_bf16
    qa, ka, va = (_heads_first(a) for a in (qa, ka, va))
    d = qa.shape[-1]
    BH, Nq, Nk = qa.shape[0], qa.shape[1], ka.shape[1]
    if rows is None:
        n_rows, rows_arr = Nq, None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n_rows = rows_arr.shape[0]
    out = np.zeros((BH, n_rows, d), dtype=np.float64)
    lse2 = np.zeros((BH, n_rows), dtype=np.float64) if with_lse2 else None
    rc = fn(BH, Nq, Nk, d, _ptr(qa), _ptr(ka), _ptr(va), float(scale), int(bool(causal)),
            n_rows, _ptr(rows_arr) if rows_arr is not None else None, _ptr(out),
            _ptr(lse2) if lse2 is not None else None)
    if rc != 0:
        raise ValueError(f"oracle attention rejected its arguments (rc={rc})")
    return (out, lse2) if with_lse2 else out


def attention_bwd(q, k, v, do, scale: float, causal: bool = False):
    """fp64 gradients (dq, dk, dv) of L = sum(O * do) for O = attention(q, k, v).

    Inputs as for :func:`attention` (``do`` has q's shape and format).  Returns
    three float64 arrays, heads first: dq [BH, Nq, d], dk and dv [BH, Nk, d].
    """
    f64 = isinstance(q, np.ndarray) and q.dtype == np.float64
    if f64:
        qa, ka, va, ga = (np.ascontiguousarray(t, dtype=np.float64) for t in (q, k, v, do))
        fn = _load().oracle_attn_bwd_f64
    else:
        (qa, fq), (ka, fk), (va, fv), (ga, fg) = (as_bits(t) for t in (q, k, v, do))
        if not fq == fk == fv == fg:
            raise TypeError("q, k, v, do must share one format")
        fn = _load().oracle_attn_bwd_fp16 if fq == "fp16" else _load().oracle_attn_bwd_bf16
    qa, ka, va, ga = (_heads_first(a) for a in (qa, ka, va, ga))
    if ga.shape != qa.shape:
        raise ValueError("do must have q's shape")
    BH, Nq, d = qa.shape
    Nk = ka.shape[1]
    dq = np.zeros((BH, Nq, d), dtype=np.float64)
    dk = np.zeros((BH, Nk, d), dtype=np.float64)
    dv = np.zeros((BH, Nk, d), dtype=np.float64)
    rc = fn(BH, Nq, Nk, d, _ptr(qa), _ptr(ka), _ptr(va), _ptr(ga), float(scale), int(bool(causal)),
            _ptr(dq), _ptr(dk), _ptr(dv))
    if rc != 0:
        raise ValueError(f"oracle attention_bwd rejected its arguments (rc={rc})")
    return dq, dk, dv


def attention_bwd_dq_rows(q, k, v, do, scale: float, rows, causal: bool = False):
    """fp64 dQ of sum(O * do) for the given query rows only: [BH, len(rows), d].

    Each row needs only its own scores, so this reaches sizes where the full
    backward (dK, dV need every row) does not."""
    f64 = isinstance(q, np.ndarray) and q.dtype == np.float64
    if f64:
        qa, ka, va, ga = (np.ascontiguousarray(t, dtype=np.float64) for t in (q, k, v, do))
        el = 1
    else:
        (qa, fq), (ka, fk), (va, fv), (ga, fg) = (as_bits(t) for t in (q, k, v, do))
        if not fq == fk == fv == fg:
            raise TypeError("q, k, v, do must share one format")
        el = 2 if fq == "fp16" else 0
    qa, ka, va, ga = (_heads_first(a) for a in (qa, ka, va, ga))
    if ga.shape != qa.shape:
        raise ValueError("do must have q's shape")
    BH, Nq, d = qa.shape
    rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    dq = np.zeros((BH, rows_arr.shape[0], d), dtype=np.float64)
    rc = _load().oracle_attn_bwd_dq_rows(el, BH, Nq, ka.shape[1], d, _ptr(qa), _ptr(ka), _ptr(va), _ptr(ga),
                                         float(scale), int(bool(causal)), rows_arr.shape[0], _ptr(rows_arr),
                                         _ptr(dq))
    if rc != 0:
        raise ValueError(f"oracle attention_bwd_dq_rows rejected its arguments (rc={rc})")
    return dq


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(n)
