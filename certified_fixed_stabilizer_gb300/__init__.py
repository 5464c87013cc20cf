"""CLiS (Certified Loop-invariant Stabilization) attention for GB300.

The compute lives in ``libclis.so`` (CUDA for sm_103a, C ABI declared in
``include/clis.h``).  :mod:`certified_fixed_stabilizer_gb300.clis` is the thin
ctypes binding with the same function names; it is imported on first use so
that ``workloads`` can be used on machines without the built library.  Using
any binding name without the built library raises an error: there is no CPU
fallback.
"""
from __future__ import annotations

import importlib

_BINDING_NAMES = {
    "clis_certify", "clis_certify_workspace_size", "clis_certify_noalloc", "clis_certify_tiles", "clis_attn_fwd",
    "clis_attn_fwd_tiles",
    "clis_status_string", "clis_get_device_error", "clis_clear_device_error",
    "ClisError", "attention", "certify", "Cert", "VARIANT", "FMT", "STATUS",
    "library_path", "load_library", "decode_certs", "make_shape", "scale_log2_for",
    "Shape", "CERT_WORDS", "LOG2E", "clis_debug_wait_selftest", "clis_attn_fwd_chunk", "clis_attn_fwd_chunk_causal",
    "clis_attn_chunk_finalize", "clis_v_e4m3_size", "clis_v_to_e4m3", "clis_attn_fwd_fp8pv", "clis_attn_fwd_chunk_fp8pv",
    "clis_attn_bwd", "clis_attn_bwd_workspace_size", "attention_bwd", "attention_fwd_lse", "attention_autograd",
    "AttentionFunction", "host_done_event", "grouped_query_views", "clis_attention_host",
    "HostPlan",
}


def __getattr__(name):
    if name in _BINDING_NAMES:
        mod = importlib.import_module(".clis", __name__)
        return getattr(mod, name)
    raise AttributeError(name)
