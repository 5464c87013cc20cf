"""ctypes binding of libclis.so -- argument marshalling only.

Function names match the C ABI in ``include/clis.h``.  Tensors are torch
tensors used purely as device (or pinned host) memory; every step of the
computation runs in the library's CUDA kernels.  If the library is missing,
importing this module raises: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

from . import build as _build

LOG2E = 1.4426950408889634

FMT = {"fp16": 0, "bf16": 1, "fp32": 2}
VARIANT = {"auto": 0, "online": 1, "certified": 2, "online_lazy": 3}
DTYPE = {torch.bfloat16: 0, torch.float16: 1}
STATUS = {0: "CLIS_OK", 1: "CLIS_ERR_INVALID_ARG", 2: "CLIS_ERR_UNSUPPORTED", 3: "CLIS_ERR_MISALIGNED",
          4: "CLIS_ERR_WORKSPACE", 5: "CLIS_ERR_CUDA", 6: "CLIS_ERR_TIMEOUT"}


class ClisError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS.get(status, status)} ({clis_status_string(status)})")


class Shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "B", "H", "Nq", "Nk", "d",
        "q_sb", "q_sh", "q_sn", "k_sb", "k_sh", "k_sn",
        "v_sb", "v_sh", "v_sn", "o_sb", "o_sh", "o_sn", "dtype")]


class Cert(ctypes.Structure):
    _fields_ = [("certified", ctypes.c_int32), ("G", ctypes.c_int32), ("A", ctypes.c_int32),
                ("C", ctypes.c_int32), ("reason", ctypes.c_int32), ("B_h", ctypes.c_float),
                ("kappa", ctypes.c_float), ("qmax", ctypes.c_float)]


CERT_WORDS = ctypes.sizeof(Cert) // 4  # a certificate is 8 32-bit words

_lib = None


def library_path() -> str:
    return _build.LIB


def load_library():
    """Load libclis.so (building it first when nvcc is available and it is stale)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path) or _build._stale():
        _build.build()
    lib = ctypes.CDLL(path)
    vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    sp = ctypes.POINTER(Shape)
    lib.clis_certify_workspace_size.argtypes = [sp, ctypes.POINTER(sz)]
    lib.clis_certify_workspace_size.restype = i32
    lib.clis_certify.argtypes = [sp, vp, vp, vp, f32, i32, i32, vp, vp, vp, vp, sz, vp]
    lib.clis_certify.restype = i32
    lib.clis_certify_noalloc.argtypes = [sp, vp, vp, vp, f32, i32, i32, vp, vp, vp, vp]
    lib.clis_certify_noalloc.restype = i32
    lib.clis_certify_tiles.argtypes = [sp, vp, vp, vp, f32, i32, i32, vp, vp, vp, vp, vp, sz, vp]
    lib.clis_certify_tiles.restype = i32
    lib.clis_attn_fwd_tiles.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, f32, i32, i32, vp]
    lib.clis_attn_fwd_tiles.restype = i32
    lib.clis_attn_fwd.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, f32, i32, i32, vp]
    lib.clis_attn_fwd.restype = i32
    lib.clis_status_string.argtypes = [i32]
    lib.clis_status_string.restype = ctypes.c_char_p
    lib.clis_get_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
    lib.clis_get_device_error.restype = i32
    lib.clis_clear_device_error.argtypes = []
    lib.clis_clear_device_error.restype = i32
    lib.clis_attn_fwd_chunk.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, f32, i32, i32, vp]
    lib.clis_attn_fwd_chunk.restype = i32
    lib.clis_attn_fwd_chunk_causal.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, f32, ctypes.c_int64, i32,
                                               i32, vp]
    lib.clis_attn_fwd_chunk_causal.restype = i32
    lib.clis_v_e4m3_size.argtypes = [sp, ctypes.POINTER(sz)]
    lib.clis_v_e4m3_size.restype = i32
    lib.clis_v_to_e4m3.argtypes = [sp, vp, vp, vp]
    lib.clis_v_to_e4m3.restype = i32
    lib.clis_attn_fwd_fp8pv.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, f32, i32, vp]
    lib.clis_attn_fwd_fp8pv.restype = i32
    lib.clis_attn_fwd_chunk_fp8pv.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, f32, i32, i32, vp]
    lib.clis_attn_fwd_chunk_fp8pv.restype = i32
    lib.clis_attn_chunk_finalize.argtypes = [sp, vp, vp, vp, vp, vp, vp]
    lib.clis_attn_chunk_finalize.restype = i32
    lib.clis_debug_wait_selftest.argtypes = [ctypes.c_uint32, vp]
    lib.clis_debug_wait_selftest.restype = i32
    lib.clis_attn_bwd_workspace_size.argtypes = [sp, ctypes.POINTER(sz)]
    lib.clis_attn_bwd_workspace_size.restype = i32
    lib.clis_attn_bwd.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, f32, i32, vp, sz, vp]
    lib.clis_attn_bwd.restype = i32
    lib.clis_host_plan_create.argtypes = [sp, i32, i32, ctypes.POINTER(vp)]
    lib.clis_host_plan_create.restype = i32
    lib.clis_host_plan_workspace_size.argtypes = [vp, ctypes.POINTER(sz)]
    lib.clis_host_plan_workspace_size.restype = i32
    lib.clis_attention_host.argtypes = [vp, vp, vp, vp, vp, f32, i32, vp, sz, vp]
    lib.clis_attention_host.restype = i32
    lib.clis_host_plan_wait.argtypes = [vp, vp]
    lib.clis_host_plan_wait.restype = i32
    lib.clis_host_plan_destroy.argtypes = [vp]
    lib.clis_host_plan_destroy.restype = i32
    _lib = lib
    return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def make_shape(q, k, v, o=None) -> Shape:
    """Shape and element strides of [B, H, N, d] tensors (d must be contiguous)."""
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o)):
        if t is None:
            continue
        if t.dim() != 4 or t.dtype not in DTYPE:
            raise ValueError(f"{name} must be a 4-D bfloat16 or float16 tensor [B, H, N, d]")
        if t.dtype != q.dtype:
            raise ValueError("q, k, v and o must share one dtype")
        if t.stride(-1) != 1:
            raise ValueError(f"{name} must have a contiguous last dimension")
    B, H, Nq, d = q.shape
    s = Shape(B=B, H=H, Nq=Nq, Nk=k.shape[2], d=d, dtype=DTYPE[q.dtype],
              q_sb=q.stride(0), q_sh=q.stride(1), q_sn=q.stride(2),
              k_sb=k.stride(0), k_sh=k.stride(1), k_sn=k.stride(2),
              v_sb=v.stride(0), v_sh=v.stride(1), v_sn=v.stride(2))
    if o is not None:
        s.o_sb, s.o_sh, s.o_sn = o.stride(0), o.stride(1), o.stride(2)
    return s


def clis_status_string(status: int) -> str:
    return load_library().clis_status_string(int(status)).decode()


def clis_certify_workspace_size(shape: Shape) -> int:
    n = ctypes.c_size_t(0)
    st = load_library().clis_certify_workspace_size(ctypes.byref(shape), ctypes.byref(n))
    if st != 0:
        raise ClisError("clis_certify_workspace_size", st)
    return n.value


def clis_certify(q, k, v, scale_log2: float, exp_fmt: str = "bf16", acc_fmt: str = "fp32",
                 kbar=None, certs=None, workspace=None, stream=None, mu=None):
    """Certification pre-pass.  Returns (kbar float32 [B*H, d], certs int32 [B*H, 8]);
    decode certificates with :func:`decode_certs`.  If ``mu`` (float32 [B*H*Nq])
    is given it receives the per-row stabilisers."""
    lib = load_library()
    shape = make_shape(q, k, v)
    BH, d = shape.B * shape.H, shape.d
    dev = q.device
    if kbar is None:
        kbar = torch.empty((max(BH, 1), d), dtype=torch.float32, device=dev)
    if certs is None:
        certs = torch.empty((max(BH, 1), CERT_WORDS), dtype=torch.int32, device=dev)
    need = clis_certify_workspace_size(shape)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    st = lib.clis_certify(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), float(scale_log2),
                          FMT[exp_fmt], FMT[acc_fmt], _ptr(kbar), _ptr(certs), _ptr(mu), _ptr(workspace),
                          workspace.numel(), _stream(stream))
    if st != 0:
        raise ClisError("clis_certify", st)
    return kbar, certs


def clis_certify_noalloc(q, k, v, scale_log2: float, exp_fmt: str = "bf16", acc_fmt: str = "fp32",
                         kbar=None, certs=None, stream=None, mu=None):
    """clis_certify without a workspace argument: the library's own fixed scratch
    (CLIS_NOALLOC_SCRATCH_BYTES) stands in for it.  Returns (kbar, certs)."""
    lib = load_library()
    shape = make_shape(q, k, v)
    BH, d = shape.B * shape.H, shape.d
    if kbar is None:
        kbar = torch.empty((max(BH, 1), d), dtype=torch.float32, device=q.device)
    if certs is None:
        certs = torch.empty((max(BH, 1), CERT_WORDS), dtype=torch.int32, device=q.device)
    st = lib.clis_certify_noalloc(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), float(scale_log2), FMT[exp_fmt],
                                  FMT[acc_fmt], _ptr(kbar), _ptr(certs), _ptr(mu), _stream(stream))
    if st != 0:
        raise ClisError("clis_certify_noalloc", st)
    return kbar, certs


def clis_certify_tiles(q, k, v, scale_log2: float, exp_fmt: str = "bf16", acc_fmt: str = "fp32",
                       kbar=None, certs=None, tile_certs=None, workspace=None, stream=None, mu=None):
    """clis_certify plus per-prefix certificates of causal heads (Nq == Nk): one
    uint8 flag per block of 256 query rows.  Returns (kbar, certs, tile_certs
    uint8 [B*H, ceil(Nq / 256)])."""
    lib = load_library()
    shape = make_shape(q, k, v)
    BH, d = shape.B * shape.H, shape.d
    dev = q.device
    if kbar is None:
        kbar = torch.empty((max(BH, 1), d), dtype=torch.float32, device=dev)
    if certs is None:
        certs = torch.empty((max(BH, 1), CERT_WORDS), dtype=torch.int32, device=dev)
    if tile_certs is None:
        tile_certs = torch.empty((max(BH, 1), max(1, -(-shape.Nq // 256))), dtype=torch.uint8, device=dev)
    need = clis_certify_workspace_size(shape)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    st = lib.clis_certify_tiles(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), float(scale_log2),
                                FMT[exp_fmt], FMT[acc_fmt], _ptr(kbar), _ptr(certs), _ptr(mu), _ptr(tile_certs),
                                _ptr(workspace), workspace.numel(), _stream(stream))
    if st != 0:
        raise ClisError("clis_certify_tiles", st)
    return kbar, certs, tile_certs


def clis_attn_fwd_tiles(q, k, v, scale_log2: float, kbar, certs, tile_certs, out=None, lse2=None, stream=None,
                        mu=None):
    """Causal AUTO forward that lets query blocks certified by their prefix
    (clis_certify_tiles) take the fixed stabiliser; returns ``out``."""
    lib = load_library()
    if out is None:
        out = torch.empty_like(q, memory_format=torch.contiguous_format)
    shape = make_shape(q, k, v, out)
    st = lib.clis_attn_fwd_tiles(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse2),
                                 _ptr(kbar), _ptr(certs), _ptr(tile_certs), _ptr(mu), float(scale_log2), 1,
                                 VARIANT["auto"], _stream(stream))
    if st != 0:
        raise ClisError("clis_attn_fwd_tiles", st)
    return out


def clis_attn_fwd(q, k, v, scale_log2: float, kbar=None, certs=None, causal: bool = False,
                  variant: str = "auto", out=None, lse2=None, stream=None, mu=None):
    """Fused attention forward; returns ``out`` (bf16, shape of q)."""
    lib = load_library()
    if out is None:
        out = torch.empty_like(q, memory_format=torch.contiguous_format)
    shape = make_shape(q, k, v, out)
    st = lib.clis_attn_fwd(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse2),
                           _ptr(kbar), _ptr(certs), _ptr(mu), float(scale_log2), int(bool(causal)),
                           VARIANT[variant], _stream(stream))
    if st != 0:
        raise ClisError("clis_attn_fwd", st)
    return out


def clis_v_e4m3_size(shape: Shape) -> int:
    n = ctypes.c_size_t(0)
    st = load_library().clis_v_e4m3_size(ctypes.byref(shape), ctypes.byref(n))
    if st != 0:
        raise ClisError("clis_v_e4m3_size", st)
    return n.value


def clis_v_to_e4m3(v, vt8=None, stream=None):
    """E4M3 transpose of V for the FP8 P.V path: uint8 [B*H, d, pitch],
    pitch = Nk rounded up to 16."""
    lib = load_library()
    shape = make_shape(v, v, v)
    B, H, Nk, d = v.shape
    pitch = -(-Nk // 16) * 16
    if vt8 is None:
        vt8 = torch.empty((B * H, d, pitch), dtype=torch.uint8, device=v.device)
    st = lib.clis_v_to_e4m3(ctypes.byref(shape), _ptr(v), _ptr(vt8), _stream(stream))
    if st != 0:
        raise ClisError("clis_v_to_e4m3", st)
    return vt8


def clis_attn_fwd_fp8pv(q, k, v, vt8, scale_log2: float, kbar=None, certs=None, variant: str = "auto", out=None,
                        lse2=None, stream=None, mu=None):
    """Attention forward whose eligible certified heads run P.V in E4M3
    (vt8 from clis_v_to_e4m3); returns ``out``."""
    lib = load_library()
    if out is None:
        out = torch.empty_like(q, memory_format=torch.contiguous_format)
    shape = make_shape(q, k, v, out)
    st = lib.clis_attn_fwd_fp8pv(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(vt8), _ptr(out), _ptr(lse2),
                                 _ptr(kbar), _ptr(certs), _ptr(mu), float(scale_log2), VARIANT[variant],
                                 _stream(stream))
    if st != 0:
        raise ClisError("clis_attn_fwd_fp8pv", st)
    return out


def clis_attn_fwd_chunk_fp8pv(q, k, v, vt8, scale_log2: float, o_acc, l_acc, m_acc, kbar=None, certs=None,
                              first: bool = False, variant: str = "auto", stream=None, mu=None):
    """clis_attn_fwd_chunk with the FP8 P.V path; vt8 = clis_v_to_e4m3 of this chunk's v."""
    lib = load_library()
    shape = make_shape(q, k, v)
    st = lib.clis_attn_fwd_chunk_fp8pv(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(vt8), _ptr(o_acc),
                                       _ptr(l_acc), _ptr(m_acc), _ptr(kbar), _ptr(certs), _ptr(mu),
                                       float(scale_log2), int(bool(first)), VARIANT[variant], _stream(stream))
    if st != 0:
        raise ClisError("clis_attn_fwd_chunk_fp8pv", st)


def clis_attn_fwd_chunk(q, k, v, scale_log2: float, o_acc, l_acc, m_acc, kbar=None, certs=None,
                        first: bool = False, variant: str = "auto", stream=None, mu=None):
    """Merge one KV chunk (k, v: [B, H, Nk_chunk, d]) into fp32 accumulators
    o_acc [B*H*Nq, d], l_acc [B*H*Nq], m_acc [B*H*Nq]."""
    lib = load_library()
    shape = make_shape(q, k, v)
    st = lib.clis_attn_fwd_chunk(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(o_acc), _ptr(l_acc),
                                 _ptr(m_acc), _ptr(kbar), _ptr(certs), _ptr(mu), float(scale_log2),
                                 int(bool(first)),
                                 VARIANT[variant], _stream(stream))
    if st != 0:
        raise ClisError("clis_attn_fwd_chunk", st)


def clis_attn_fwd_chunk_causal(q, k, v, scale_log2: float, o_acc, l_acc, m_acc, key_offset: int, kbar=None,
                               certs=None, tile_certs=None, first: bool = False, variant: str = "auto", stream=None,
                               mu=None):
    """Merge one causal KV chunk (k, v: [B, H, Nk_chunk, d], keys key_offset ..
    key_offset + Nk_chunk - 1 of each head) into the accumulators, as
    clis_attn_fwd_chunk does; query i sees chunk key j iff key_offset + j <= i."""
    lib = load_library()
    shape = make_shape(q, k, v)
    st = lib.clis_attn_fwd_chunk_causal(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(o_acc), _ptr(l_acc),
                                        _ptr(m_acc), _ptr(kbar), _ptr(certs), _ptr(tile_certs), _ptr(mu),
                                        float(scale_log2), int(key_offset), int(bool(first)), VARIANT[variant],
                                        _stream(stream))
    if st != 0:
        raise ClisError("clis_attn_fwd_chunk_causal", st)


def clis_attn_chunk_finalize(q, o_acc, l_acc, m_acc, out=None, lse2=None, stream=None):
    """o = o_acc / l_acc (bf16, shape of q), optional lse2 = m_acc + log2 l_acc."""
    lib = load_library()
    if out is None:
        out = torch.empty_like(q, memory_format=torch.contiguous_format)
    shape = make_shape(q, q, q, out)
    st = lib.clis_attn_chunk_finalize(ctypes.byref(shape), _ptr(o_acc), _ptr(l_acc), _ptr(m_acc), _ptr(out),
                                      _ptr(lse2), _stream(stream))
    if st != 0:
        raise ClisError("clis_attn_chunk_finalize", st)
    return out


def clis_attn_bwd_workspace_size(shape: Shape) -> int:
    n = ctypes.c_size_t(0)
    st = load_library().clis_attn_bwd_workspace_size(ctypes.byref(shape), ctypes.byref(n))
    if st != 0:
        raise ClisError("clis_attn_bwd_workspace_size", st)
    return n.value


def _like(t):
    """Empty tensor with t's shape and strides (the backward writes dq, dk, dv
    with the strides of q, k, v)."""
    return torch.empty_strided(t.shape, t.stride(), dtype=t.dtype, device=t.device)


def clis_attn_bwd(q, k, v, o, dout, lse2, scale_log2: float, causal: bool = False, dq=None, dk=None, dv=None,
                  workspace=None, stream=None):
    """Attention backward; returns (dq, dk, dv) with the strides of q, k, v.

    o: the forward output; dout: its gradient, with o's strides; lse2: the
    forward's fp32 row statistic [B*H*Nq]."""
    lib = load_library()
    if dout.stride() != o.stride():
        dout = torch.empty_strided(o.shape, o.stride(), dtype=o.dtype, device=o.device).copy_(dout)
    dq = _like(q) if dq is None else dq
    dk = _like(k) if dk is None else dk
    dv = _like(v) if dv is None else dv
    for name, g, t in (("dq", dq, q), ("dk", dk, k), ("dv", dv, v)):
        if g.stride() != t.stride() or g.shape != t.shape or g.dtype != t.dtype:
            raise ValueError(f"{name} must have the shape, strides and dtype of {name[1]}")
    shape = make_shape(q, k, v, o)
    if workspace is None:
        workspace = torch.empty(max(1, clis_attn_bwd_workspace_size(shape)), dtype=torch.uint8, device=q.device)
    st = lib.clis_attn_bwd(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse2),
                           _ptr(dq), _ptr(dk), _ptr(dv), float(scale_log2), int(bool(causal)), _ptr(workspace),
                           workspace.numel(), _stream(stream))
    if st != 0:
        raise ClisError("clis_attn_bwd", st)
    return dq, dk, dv


def attention_fwd_lse(q, k, v, softmax_scale: float | None = None, causal: bool = False, variant: str = "auto",
                      out=None):
    """Forward that also returns the row statistic the backward needs:
    (o, lse2), lse2 fp32 [B*H*Nq].  k, v may have fewer heads than q
    (grouped-query attention, see :func:`grouped_query_views`)."""
    if k.shape[1] != q.shape[1]:
        o = torch.empty_like(q, memory_format=torch.contiguous_format) if out is None else out
        qf, kf, vf, of = grouped_query_views(q, k, v, o)
        _, lse2 = attention_fwd_lse(qf, kf, vf, softmax_scale, causal, variant, out=of)
        return o, lse2
    sl2 = scale_log2_for(q.shape[-1], softmax_scale)
    lse2 = torch.empty(q.shape[0] * q.shape[1] * q.shape[2], dtype=torch.float32, device=q.device)
    kbar = certs = mu = None
    if variant in ("auto", "certified"):
        mu = torch.empty_like(lse2)
        kbar, certs = clis_certify(q, k, v, sl2, mu=mu, exp_fmt=_exp_fmt(q))
    o = clis_attn_fwd(q, k, v, sl2, kbar=kbar, certs=certs, causal=causal, variant=variant, mu=mu, lse2=lse2,
                      out=out)
    return o, lse2


def attention_bwd(q, k, v, o, dout, lse2, softmax_scale: float | None = None, causal: bool = False):
    """(dq, dk, dv) for the attention whose forward gave (o, lse2).  With k, v
    of fewer heads than q (grouped-query attention) dk and dv have k's and v's
    shape: each holds the sum over its group's query heads, accumulated in the
    kernel (K and V pass as broadcast views, dK and dV as broadcast views of
    tensors shaped like k and v)."""
    sl2 = scale_log2_for(q.shape[-1], softmax_scale)
    if k.shape[1] == q.shape[1]:
        return clis_attn_bwd(q, k, v, o, dout, lse2, sl2, causal=causal)
    if dout.stride() != o.stride():
        dout = torch.empty_strided(o.shape, o.stride(), dtype=o.dtype, device=o.device).copy_(dout)
    dq = torch.empty_strided(q.shape, q.stride(), dtype=q.dtype, device=q.device)
    dk = torch.empty_strided(k.shape, k.stride(), dtype=k.dtype, device=k.device)
    dv = torch.empty_strided(v.shape, v.stride(), dtype=v.dtype, device=v.device)
    qf, kf, vf, of = grouped_query_views(q, k, v, o)
    dqf, dkf, dvf, dof = grouped_query_views(dq, dk, dv, dout)
    clis_attn_bwd(qf, kf, vf, of, dof, lse2, sl2, causal=causal, dq=dqf, dk=dkf, dv=dvf)
    return dq, dk, dv


class AttentionFunction(torch.autograd.Function):
    """Autograd wrapper: CLiS forward (certify + fused kernel), backward
    through clis_attn_bwd.  Device tensors only."""

    @staticmethod
    def forward(ctx, q, k, v, softmax_scale, causal, variant):
        o, lse2 = attention_fwd_lse(q, k, v, softmax_scale, causal, variant)
        ctx.save_for_backward(q, k, v, o, lse2)
        ctx.softmax_scale, ctx.causal = softmax_scale, causal
        return o

    @staticmethod
    def backward(ctx, dout):
        q, k, v, o, lse2 = ctx.saved_tensors
        dq, dk, dv = attention_bwd(q, k, v, o, dout, lse2, ctx.softmax_scale, ctx.causal)
        return dq, dk, dv, None, None, None


def attention_autograd(q, k, v, softmax_scale: float | None = None, causal: bool = False, variant: str = "auto"):
    """Differentiable CLiS attention (training): o = attention(q, k, v)."""
    return AttentionFunction.apply(q, k, v, softmax_scale, causal, variant)


def clis_get_device_error() -> int:
    code = ctypes.c_uint32(0)
    st = load_library().clis_get_device_error(ctypes.byref(code))
    if st not in (0, 6):
        raise ClisError("clis_get_device_error", st)
    return code.value


def clis_clear_device_error() -> None:
    st = load_library().clis_clear_device_error()
    if st != 0:
        raise ClisError("clis_clear_device_error", st)


def clis_debug_wait_selftest(limit_us: int = 1000, stream=None) -> None:
    """Launch the bounded-wait self-test kernel (see include/clis.h)."""
    st = load_library().clis_debug_wait_selftest(int(limit_us), _stream(stream))
    if st != 0:
        raise ClisError("clis_debug_wait_selftest", st)


def decode_certs(certs) -> list[dict]:
    """int32 [BH, 8] certificate words -> list of dicts (host copy)."""
    c = certs.detach().to("cpu").contiguous()
    ints = c[:, :5].tolist()
    floats = c[:, 5:8].view(torch.float32).tolist()
    out = []
    for i, f in zip(ints, floats):
        out.append({"certified": i[0], "G": i[1], "A": i[2], "C": i[3], "reason": i[4],
                    "B_h": f[0], "kappa": f[1], "qmax": f[2]})
    return out


def scale_log2_for(d: int, softmax_scale: float | None = None) -> float:
    """scale_log2 = softmax_scale * log2(e), default softmax_scale = 1/sqrt(d)."""
    s = (1.0 / math.sqrt(d)) if softmax_scale is None else softmax_scale
    return s * LOG2E


def certify(q, k, v, softmax_scale: float | None = None, **kw):
    return clis_certify(q, k, v, scale_log2_for(q.shape[-1], softmax_scale), **kw)


def _exp_fmt(q) -> str:
    return "fp16" if q.dtype == torch.float16 else "bf16"


def grouped_query_views(q, k, v, out=None):
    """Views for grouped-query / multi-query attention: q [B, H, Nq, d] and k, v
    [B, H_kv, Nk, d] with H a multiple of H_kv (query head h uses key/value head
    h // (H / H_kv)).  Returns (q', k', v', out') of shape [B * H_kv, H / H_kv, N, d]
    over the same memory: the key/value heads are folded into the batch and K, V
    get head stride 0, so every query head of a group reads its group's keys and
    values (no copy).  The certificate of folded head (b', j) sits at index
    b' * (H / H_kv) + j = b * H + h, as without folding."""
    B, H, Nq, d = q.shape
    Hkv = k.shape[1]
    if v.shape[1] != Hkv or H % Hkv:
        raise ValueError("k and v need the same number of heads, dividing q's")
    g = H // Hkv
    views = []
    for t, heads, bcast in ((q, H, False), (k, Hkv, True), (v, Hkv, True), (out, H, False)):
        if t is None:
            views.append(None)
            continue
        sb, sh, sn, sd = t.stride()
        if sb != heads * sh and t.shape[0] > 1:
            raise ValueError("the batch stride must span the heads (sb == H * sh) to fold them")
        n = t.shape[2]
        if bcast:
            views.append(t.as_strided((B * Hkv, g, n, d), (sh, 0, sn, sd)))
        else:
            views.append(t.as_strided((B * Hkv, g, n, d), (g * sh, sh, sn, sd)))
    return tuple(views)


def attention(q, k, v, softmax_scale: float | None = None, causal: bool = False,
              variant: str = "auto", return_certs: bool = False, device=None, out=None,
              groups: int | None = None, non_blocking: bool = False, pv: str = "bf16"):
    """CLiS attention forward: certification pre-pass, then the fused kernel.

    q, k, v: bf16 or fp16 [B, H, N, d].  Device tensors are processed in place
    on the current stream.  Host tensors (pinned for overlap) go through the
    library's clis_attention_host on ``device`` (default cuda:0), which writes
    the result to ``out`` (a contiguous host tensor, allocated if None): heads
    are processed in ``groups`` groups (by default about one group per 2 TFLOP
    of attention work, at least 8, at most one per head), with copies in and
    out on two streams of the library's and the kernels on two more
    (alternating groups), so that the copies of one group overlap the compute
    of another and one group's kernel can start on SMs the previous one has
    left idle (heads are independent).  The input copies follow the work
    already queued on the current stream.  The call returns once ``out`` is
    filled, unless ``non_blocking``: then it returns after queueing, and the
    caller waits for :func:`host_done_event` (or synchronises the device)
    before reading ``out`` or changing q, k, v.  The plan (streams, events)
    and its device workspace (staging for every head) are kept for the next
    call with the same shapes, so consecutive non-blocking calls overlap: a
    call's copies of a head group start as soon as the previous call's
    kernels on that group are done.

    ``pv="fp8"`` (device tensors, bf16, d = 128, no mask, variant "auto" or
    "certified") runs the FP8 P.V path: V's E4M3 transpose, then
    clis_attn_fwd_fp8pv, where heads within the E4M3 budget multiply P and V
    in E4M3 and every other head runs as with ``pv="bf16"``.

    k and v may have fewer heads than q (grouped-query or multi-query
    attention, device tensors): see :func:`grouped_query_views`; the output
    has q's shape.
    """
    if pv not in ("bf16", "fp8"):
        raise ValueError(f"pv must be 'bf16' or 'fp8', not {pv!r}")
    if k.shape[1] != q.shape[1]:
        if q.device.type == "cpu":
            raise ValueError("grouped key/value heads take device tensors")
        if out is None:
            out = torch.empty_like(q, memory_format=torch.contiguous_format)
        qf, kf, vf, of = grouped_query_views(q, k, v, out)
        res = attention(qf, kf, vf, softmax_scale, causal, variant, return_certs, out=of, pv=pv)
        return (out,) + tuple(res[1:]) if return_certs else out
    if pv == "fp8" and variant == "auto" and k.shape[2] < 4096:
        # No head takes E4M3 under 4096 keys (the accuracy rule of clis_attn_fwd_fp8pv),
        # and every other head runs exactly as in clis_attn_fwd: skip the conversion.
        pv = "bf16"
    if pv == "fp8":
        if q.device.type == "cpu" or causal or variant not in ("auto", "certified"):
            raise ValueError("pv='fp8' takes device tensors, no mask and variant 'auto' or 'certified'")
        sl2 = scale_log2_for(q.shape[-1], softmax_scale)
        mu = torch.empty(q.shape[0] * q.shape[1] * q.shape[2], dtype=torch.float32, device=q.device)
        kbar, certs = clis_certify(q, k, v, sl2, mu=mu)
        res = clis_attn_fwd_fp8pv(q, k, v, clis_v_to_e4m3(v), sl2, kbar=kbar, certs=certs, variant=variant,
                                  out=out, mu=mu)
        return (res, kbar, certs) if return_certs else res
    if q.device.type == "cpu":
        return _attention_host(q, k, v, softmax_scale, causal, variant, return_certs,
                               torch.device(device or "cuda:0"), out, groups, non_blocking)
    sl2 = scale_log2_for(q.shape[-1], softmax_scale)
    kbar = certs = mu = None
    if variant in ("auto", "certified"):
        mu = torch.empty(q.shape[0] * q.shape[1] * q.shape[2], dtype=torch.float32, device=q.device)
        kbar, certs = clis_certify(q, k, v, sl2, mu=mu, exp_fmt=_exp_fmt(q))
    res = clis_attn_fwd(q, k, v, sl2, kbar=kbar, certs=certs, causal=causal, variant=variant, mu=mu,
                        out=out)
    if return_certs:
        return res, kbar, certs
    return res


class HostPlan:
    """A clis_host_plan_t (streams and per-group events of the host-memory
    forward for one shape on one device) with its device workspace."""

    def __init__(self, q, k, v, out, causal: bool = False, groups: int = 0, device=None):
        lib = load_library()
        self.device = torch.device(device or "cuda:0")
        self.shape = make_shape(q, k, v, out)
        self.handle = ctypes.c_void_p()
        with torch.cuda.device(self.device):
            st = lib.clis_host_plan_create(ctypes.byref(self.shape), int(bool(causal)), int(groups),
                                           ctypes.byref(self.handle))
            if st != 0:
                raise ClisError("clis_host_plan_create", st)
            n = ctypes.c_size_t(0)
            st = lib.clis_host_plan_workspace_size(self.handle, ctypes.byref(n))
            if st != 0:
                raise ClisError("clis_host_plan_workspace_size", st)
            self.workspace = torch.empty(max(n.value, 256), dtype=torch.uint8, device=self.device)
            self.side = torch.cuda.Stream(device=self.device)  # records the completion events

    def wait(self, stream=None) -> None:
        """clis_host_plan_wait: ``stream`` waits for the latest call's last copy out."""
        st = load_library().clis_host_plan_wait(self.handle, _stream(stream))
        if st != 0:
            raise ClisError("clis_host_plan_wait", st)

    def destroy(self) -> None:
        """Waits for the plan's queued work (the workspace tensor is freed through
        torch, which does not see the plan's streams), then releases the plan."""
        if self.handle:
            self.wait(self.side)
            self.side.synchronize()
            load_library().clis_host_plan_destroy(self.handle)
            self.handle = ctypes.c_void_p()

    def __del__(self):
        try:
            self.destroy()
        except Exception:  # interpreter shutdown: the library may be gone already
            pass


def clis_attention_host(plan: HostPlan, q, k, v, out, scale_log2: float, variant: str = "auto", stream=None):
    """One forward of host tensors q, k, v into out (dense [B, H, N, d], the
    plan's shape; pinned for asynchronous copies) with ``plan``: copies in,
    certification, attention and copies out pipelined over head groups inside
    the library.  Queued, not waited for: ``plan.wait(stream)`` orders a
    stream after it."""
    st = load_library().clis_attention_host(plan.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(out), float(scale_log2),
                                            VARIANT[variant], _ptr(plan.workspace), plan.workspace.numel(),
                                            _stream(stream))
    if st != 0:
        raise ClisError("clis_attention_host", st)
    return out


# Per device: the plan of the host-tensor path (kept for the next call with
# the same shapes, so that consecutive calls overlap) and the event after the
# latest call's last output copy.
_host_plans: dict = {}
_host_done: dict = {}


def _attention_host(q, k, v, softmax_scale, causal, variant, return_certs, dev, out, groups, non_blocking):
    q, k, v = (t.contiguous() for t in (q, k, v))
    B, H, Nq, d = q.shape
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, pin_memory=q.is_pinned())
    elif not out.is_contiguous():
        raise ValueError("out must be a contiguous host tensor")
    sl2 = scale_log2_for(d, softmax_scale)
    g = 0 if groups is None else int(groups)
    key = (tuple(q.shape), tuple(k.shape), q.dtype, bool(causal), g)
    with torch.cuda.device(dev):
        plan = _host_plans.get(dev)
        if plan is None or plan.key != key:
            if plan is not None:
                torch.cuda.synchronize(dev)  # the old workspace may still be in use
                plan.destroy()
            plan = _host_plans[dev] = HostPlan(q, k, v, out, causal, g, dev)
            plan.key = key
        cur = torch.cuda.current_stream(dev)
        clis_attention_host(plan, q, k, v, out, sl2, variant, stream=cur)
        # The caller's stream is not made to wait, so that its next call's copies
        # can start while this call's last groups still run.
        plan.wait(plan.side)
        done = _host_done[dev] = torch.cuda.Event()
        done.record(plan.side)
        kbar = certs = None
        if return_certs and variant in ("auto", "certified") and B * H > 0 and Nq > 0:
            # k-bar at the start of the workspace, the certificates at the next
            # multiple of 256 bytes (include/clis.h), copied on the caller's
            # stream once every kernel of the call has run.
            plan.wait(cur)
            BH, ws = B * H, plan.workspace
            nk = BH * d * 4
            off = (nk + 255) // 256 * 256
            kbar = ws[:nk].view(torch.float32).view(BH, d).clone()
            certs = ws[off:off + BH * CERT_WORDS * 4].view(torch.int32).view(BH, CERT_WORDS).clone()
    if not non_blocking:
        done.synchronize()
    if return_certs:
        return out, kbar, certs
    return out


def host_done_event(device=None):
    """The event after the last output copy of the most recent host-tensor
    attention() call on ``device`` (default cuda:0), or None: a stream that
    waits for it (``stream.wait_event(...)``) is ordered after that call's
    output, and ``.synchronize()`` waits for it on the host."""
    return _host_done.get(torch.device(device or "cuda:0"))


load_library()
