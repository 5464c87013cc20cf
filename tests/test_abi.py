"""Host-side checks of the C ABI (no GPU): the library loads, exports every
symbol include/clis.h declares, and rejects bad arguments with the documented
status codes before touching the GPU (every call here fails validation, so
nothing is launched)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "clis.h")


@pytest.fixture(scope="module")
def clis():
    from certified_fixed_stabilizer_gb300 import clis as mod
    return mod


def _declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"CLIS_API\s+[\w\s\*]*?\b(clis_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared_symbols()
    for n in ("clis_certify_workspace_size", "clis_certify", "clis_attn_fwd", "clis_status_string",
              "clis_get_device_error", "clis_clear_device_error", "clis_debug_wait_selftest",
              "clis_attn_fwd_chunk", "clis_attn_chunk_finalize", "clis_certify_noalloc",
              "clis_attn_bwd_workspace_size", "clis_attn_bwd", "clis_certify_tiles", "clis_attn_fwd_tiles",
              "clis_attn_fwd_chunk_causal", "clis_v_e4m3_size", "clis_v_to_e4m3", "clis_attn_fwd_fp8pv",
              "clis_attn_fwd_chunk_fp8pv", "clis_host_plan_create", "clis_host_plan_workspace_size",
              "clis_attention_host", "clis_host_plan_wait", "clis_host_plan_destroy"):
        assert n in names


@pytest.mark.parametrize("lang,std", [("c", "-std=c99"), ("c", "-std=c11"), ("c++", "-std=c++11")])
def test_header_compiles_standalone(tmp_path, lang, std):
    """include/clis.h needs no CUDA or C++ headers: plain C99 and C++11 accept it."""
    import shutil
    import subprocess
    cc = shutil.which("gcc" if lang == "c" else "g++")
    if cc is None:
        pytest.skip("no host compiler")
    src = tmp_path / ("t.c" if lang == "c" else "t.cpp")
    src.write_text('#include "clis.h"\nint main(void) { clis_shape_t s; (void)s; return (int)CLIS_OK; }\n')
    r = subprocess.run([cc, std, "-Wall", "-Wextra", "-Werror", "-fsyntax-only", "-I" + os.path.dirname(HEADER),
                        str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_library_exports_every_declared_symbol(clis):
    lib = ctypes.CDLL(clis.library_path())
    for n in _declared_symbols():
        assert hasattr(lib, n), n


def test_wait_selftest_rejects_bad_limits(clis):
    lib = clis.load_library()
    assert lib.clis_debug_wait_selftest(0, None) == 1
    assert lib.clis_debug_wait_selftest(2_000_000, None) == 1


def test_status_strings(clis):
    for code in range(7):
        s = clis.clis_status_string(code)
        assert isinstance(s, str) and s and s != "unknown status"
    assert clis.clis_status_string(99) == "unknown status"


def _shape(clis, B=1, H=2, Nq=300, Nk=300, d=128):
    s = clis.Shape(B=B, H=H, Nq=Nq, Nk=Nk, d=d)
    for t in "qkvo":
        setattr(s, f"{t}_sn", d)
        setattr(s, f"{t}_sh", (Nq if t in "qo" else Nk) * d)
        setattr(s, f"{t}_sb", H * (Nq if t in "qo" else Nk) * d)
    return s


FAKE = 0x10000  # never dereferenced: every call below fails validation first


def _certify(clis, shape, q=FAKE, k=FAKE, v=FAKE, scale=0.1, ef=1, af=2, kbar=FAKE, certs=FAKE,
             ws=FAKE, ws_bytes=1 << 30):
    lib = clis.load_library()
    vp = ctypes.c_void_p
    return lib.clis_certify(ctypes.byref(shape) if shape is not None else None, vp(q), vp(k), vp(v), scale,
                            ef, af, vp(kbar), vp(certs), None, vp(ws), ws_bytes, None)


def _attn(clis, shape, q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse2=None, kbar=FAKE, certs=FAKE, scale=0.1,
          causal=0, variant=0):
    lib = clis.load_library()
    vp = ctypes.c_void_p
    return lib.clis_attn_fwd(ctypes.byref(shape) if shape is not None else None, vp(q), vp(k), vp(v), vp(o),
                             vp(lse2), vp(kbar), vp(certs), None, scale, causal, variant, None)


def test_workspace_size_is_host_only_and_grows(clis):
    a = clis.clis_certify_workspace_size(_shape(clis, Nk=1000))
    b = clis.clis_certify_workspace_size(_shape(clis, Nk=100000))
    assert 0 < a < b
    assert a % 256 == 0


def test_certify_rejects_bad_arguments(clis):
    OK_INVALID, UNSUP, MIS, WS = 1, 2, 3, 4
    assert _certify(clis, None) == OK_INVALID
    assert _certify(clis, _shape(clis), q=0) == OK_INVALID
    assert _certify(clis, _shape(clis), scale=0.0) == OK_INVALID
    assert _certify(clis, _shape(clis), scale=float("nan")) == OK_INVALID
    assert _certify(clis, _shape(clis), scale=-1.0) == OK_INVALID
    assert _certify(clis, _shape(clis), ef=7) == OK_INVALID
    assert _certify(clis, _shape(clis, Nk=0)) == OK_INVALID
    assert _certify(clis, _shape(clis, d=96)) == UNSUP
    assert _certify(clis, _shape(clis), k=FAKE + 8) == MIS
    s = _shape(clis)
    s.k_sn = 132
    assert _certify(clis, s) == MIS
    assert _certify(clis, _shape(clis), ws=0) == WS
    assert _certify(clis, _shape(clis), ws_bytes=16) == WS
    assert _certify(clis, _shape(clis), ws=FAKE + 16) == MIS


def test_attn_rejects_bad_arguments(clis):
    INV, UNSUP, MIS = 1, 2, 3
    assert _attn(clis, None) == INV
    assert _attn(clis, _shape(clis), o=0) == INV
    assert _attn(clis, _shape(clis), kbar=0) == INV               # AUTO needs kbar
    assert _attn(clis, _shape(clis), certs=0) == INV              # AUTO needs certificates
    assert _attn(clis, _shape(clis), certs=0, variant=2, scale=0) == INV
    assert _attn(clis, _shape(clis), variant=5) == INV
    assert _attn(clis, _shape(clis), causal=2) == INV
    assert _attn(clis, _shape(clis, Nq=300, Nk=400), causal=1) == UNSUP
    assert _attn(clis, _shape(clis, d=256)) == UNSUP
    bad = _shape(clis)
    bad.dtype = 7
    assert _attn(clis, bad) == INV
    assert _certify(clis, bad) == INV
    assert _attn(clis, _shape(clis), o=FAKE + 2) == MIS
    assert _attn(clis, _shape(clis), lse2=FAKE + 2) == MIS
    lib = clis.load_library()
    vp = ctypes.c_void_p
    s = _shape(clis)
    assert lib.clis_attn_fwd(ctypes.byref(s), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), None, vp(FAKE), vp(FAKE),
                             vp(FAKE + 2), 0.1, 0, 0, None) == MIS          # mu misaligned
    s = _shape(clis)
    s.o_sn = 129
    assert _attn(clis, s) == INV or _attn(clis, s) == MIS
    s = _shape(clis)
    s.q_sh = 12
    assert _attn(clis, s) == MIS


def test_written_tensors_must_not_alias(clis):
    """A zero head or batch stride may broadcast K and V (grouped-query
    attention) but never an output: O in the forward and the chunk finalize,
    dQ/dK/dV (written with the Q/K/V strides) in the backward -- except dK and
    dV when K and V are broadcast over the heads together, where the kernel
    sums each group and writes every row once."""
    INV = 1
    s = _shape(clis)
    s.o_sh = 0
    assert _attn(clis, s) == INV
    s = _shape(clis, B=2, H=1)
    s.o_sb = 0
    assert _attn(clis, s) == INV
    lib = clis.load_library()
    vp = ctypes.c_void_p
    s = _shape(clis)
    s.o_sh = 0
    assert lib.clis_attn_chunk_finalize(ctypes.byref(s), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), None, None) == INV
    for t in "qkv":  # one of Q, K, V alone with head stride 0: its gradient rows would alias
        s = _shape(clis)
        setattr(s, f"{t}_sh", 0)
        assert _bwd(clis, s) == INV, t
    s = _shape(clis, B=2)  # K and V broadcast over the batch
    s.k_sb = s.v_sb = 0
    assert _bwd(clis, s) == INV
    s = _shape(clis)       # K and V broadcast over the heads together: grouped-query, allowed
    s.k_sh = s.v_sh = 0
    assert _bwd(clis, s, dq=FAKE + 8) == 3


def test_broadcast_kv_passes_the_forward_checks(clis):
    """K and V with head stride 0 (the grouped-query fold) pass the shape and
    stride checks, which come first: the calls below get as far as the
    deliberately misaligned pointer."""
    MIS = 3
    s = _shape(clis)
    s.k_sh = s.v_sh = 0
    assert _attn(clis, s, o=FAKE + 2) == MIS
    assert _certify(clis, s, k=FAKE + 8) == MIS
    assert clis.clis_certify_workspace_size(s) > 0


def test_chunk_entry_points_reject_bad_arguments(clis):
    lib = clis.load_library()
    vp = ctypes.c_void_p
    s = _shape(clis)
    call = lambda **kw: lib.clis_attn_fwd_chunk(ctypes.byref(s), vp(kw.get("q", FAKE)), vp(FAKE), vp(FAKE),
                                                vp(kw.get("oa", FAKE)), vp(kw.get("la", FAKE)), vp(FAKE), vp(FAKE),
                                                vp(FAKE), None, kw.get("scale", 0.1), kw.get("first", 0),
                                                kw.get("variant", 0), None)
    assert call(oa=0) == 1
    assert call(first=3) == 1
    assert call(scale=-1.0) == 1
    assert call(variant=9) == 1
    assert call(oa=FAKE + 4) == 3
    assert call(la=FAKE + 2) == 3
    assert lib.clis_attn_chunk_finalize(ctypes.byref(s), vp(FAKE), vp(FAKE), vp(FAKE), vp(0), None, None) == 1
    s2 = _shape(clis, d=80)
    assert lib.clis_attn_chunk_finalize(ctypes.byref(s2), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), None, None) == 2


def test_causal_chunk_entry_point_rejects_bad_arguments(clis):
    """Causal KV chunks: the chunk must lie inside the query range, only the
    chunk holding key 0 may be first, per-prefix flags need AUTO (all rejected
    on the host; the fake pointers are never touched)."""
    lib = clis.load_library()
    vp = ctypes.c_void_p
    s = _shape(clis, Nq=1000, Nk=300)

    def call(off, first=0, tiles=None, variant=0, oa=FAKE):
        return lib.clis_attn_fwd_chunk_causal(ctypes.byref(s), vp(FAKE), vp(FAKE), vp(FAKE), vp(oa), vp(FAKE),
                                              vp(FAKE), vp(FAKE), vp(FAKE), tiles, None, 0.1, off, first, variant,
                                              None)
    assert call(-1) == 1                      # negative key offset
    assert call(256, first=1) == 1            # a first chunk that does not hold key 0
    assert call(701) == 2                     # keys past the last query row
    assert call(0, tiles=vp(FAKE), variant=1) == 1  # per-prefix flags outside AUTO
    assert call(0, first=2) == 1
    assert call(100, oa=0) == 1
    assert call(100, oa=FAKE + 4) == 3


def test_fp8pv_entry_points_reject_bad_arguments(clis):
    """FP8 P.V: d = 128 and BF16 data only, AUTO or CERTIFIED_FORCED only, a
    V^T buffer required (rejected on the host; fake pointers never touched)."""
    lib = clis.load_library()
    vp = ctypes.c_void_p

    def call(s, vt8=FAKE, variant=0):
        return lib.clis_attn_fwd_fp8pv(ctypes.byref(s), vp(FAKE), vp(FAKE), vp(FAKE), vp(vt8), vp(FAKE), None,
                                       vp(FAKE), vp(FAKE), None, 0.1, variant, None)
    assert call(_shape(clis, d=64)) == 2
    s16 = _shape(clis)
    s16.dtype = 1
    assert call(s16) == 2
    assert call(_shape(clis), variant=1) == 1
    assert call(_shape(clis), variant=3) == 1
    assert call(_shape(clis), vt8=0) == 1
    assert call(_shape(clis), vt8=FAKE + 8) == 3
    assert lib.clis_v_to_e4m3(ctypes.byref(s16), vp(FAKE), vp(FAKE), None) == 2

    def chunk(s, vt8=FAKE, variant=0):
        return lib.clis_attn_fwd_chunk_fp8pv(ctypes.byref(s), vp(FAKE), vp(FAKE), vp(FAKE), vp(vt8), vp(FAKE),
                                             vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), None, 0.1, 1, variant, None)
    assert chunk(_shape(clis, d=64)) == 2
    assert chunk(s16) == 2
    assert chunk(_shape(clis), variant=1) == 1
    assert chunk(_shape(clis), vt8=0) == 1
    assert chunk(_shape(clis), vt8=FAKE + 8) == 3
    assert lib.clis_v_to_e4m3(ctypes.byref(_shape(clis)), vp(FAKE), vp(0), None) == 1
    n = ctypes.c_size_t(0)
    assert lib.clis_v_e4m3_size(ctypes.byref(_shape(clis, Nk=1000)), ctypes.byref(n)) == 0
    assert n.value == 1 * 2 * 128 * 1008


def test_tile_entry_points_reject_bad_arguments(clis):
    """Per-prefix certificates: causal (Nq == Nk) only, AUTO only, tile flags required
    (rejected on the host, before any launch; the fake pointers are never touched)."""
    lib = clis.load_library()
    vp = ctypes.c_void_p
    s = _shape(clis)
    cert = lambda shape, tiles=FAKE: lib.clis_certify_tiles(ctypes.byref(shape), vp(FAKE), vp(FAKE), vp(FAKE), 0.1,
                                                            1, 2, vp(FAKE), vp(FAKE), None, vp(tiles), vp(FAKE),
                                                            1 << 20, None)
    assert cert(s, tiles=0) == 1
    assert cert(_shape(clis, Nq=300, Nk=400)) == 2
    attn = lambda shape, causal=1, variant=0, tiles=FAKE: lib.clis_attn_fwd_tiles(
        ctypes.byref(shape), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), None, vp(FAKE), vp(FAKE), vp(tiles), None,
        0.1, causal, variant, None)
    assert attn(s, tiles=0) == 1
    assert attn(s, causal=0) == 1
    assert attn(s, variant=1) == 1
    assert attn(_shape(clis, Nq=300, Nk=400)) == 2


def _bwd(clis, shape=None, ws_bytes=1 << 20, scale=0.1, causal=0, **ptrs):
    lib = clis.load_library()
    vp = ctypes.c_void_p
    s = shape if shape is not None else _shape(clis)
    args = [vp(ptrs.get(n, FAKE)) for n in ("q", "k", "v", "o", "do", "lse2", "dq", "dk", "dv")]
    return lib.clis_attn_bwd(ctypes.byref(s), *args, scale, causal, vp(ptrs.get("ws", FAKE)), ws_bytes, None)


def test_bwd_workspace_size(clis):
    assert clis.clis_attn_bwd_workspace_size(_shape(clis, Nq=300)) == 2560  # 2 heads x 300 rows x 4 B -> 256s
    assert clis.clis_attn_bwd_workspace_size(_shape(clis, Nq=0)) == 0
    with pytest.raises(clis.ClisError):
        clis.clis_attn_bwd_workspace_size(_shape(clis, d=96))


def test_bwd_rejects_bad_arguments(clis):
    INV, UNSUP, MIS, WS = 1, 2, 3, 4
    for name in ("q", "k", "v", "o", "do", "lse2", "dq", "dk", "dv"):
        assert _bwd(clis, **{name: 0}) == INV, name
    assert _bwd(clis, scale=0.0) == INV
    assert _bwd(clis, scale=float("inf")) == INV
    assert _bwd(clis, causal=2) == INV
    assert _bwd(clis, _shape(clis, Nq=300, Nk=200), causal=1) == UNSUP
    assert _bwd(clis, _shape(clis, d=256)) == UNSUP
    bad = _shape(clis)
    bad.dtype = 3
    assert _bwd(clis, bad) == INV
    assert _bwd(clis, dq=FAKE + 8) == MIS
    assert _bwd(clis, do=FAKE + 2) == MIS
    assert _bwd(clis, lse2=FAKE + 2) == MIS
    assert _bwd(clis, ws=0) == WS
    assert _bwd(clis, ws_bytes=2559) == WS
    assert _bwd(clis, ws=FAKE + 8) == WS
    s = _shape(clis)
    s.o_sn = 132
    assert _bwd(clis, s) == MIS


def test_binding_has_no_cpu_fallback(clis):
    """The binding exposes only library calls: no torch or numpy attention."""
    src = open(os.path.join(ROOT, "certified_fixed_stabilizer_gb300", "clis.py")).read()
    assert "oracle" not in src
    assert "softmax" not in src.replace("softmax_scale", "")



def _plan(clis, shape, causal=0, groups=0):
    h = ctypes.c_void_p()
    st = clis.load_library().clis_host_plan_create(ctypes.byref(shape) if shape is not None else None, causal,
                                                   groups, ctypes.byref(h))
    return st, h


def test_host_plan_rejects_bad_arguments(clis):
    """clis_host_plan_create checks everything before any CUDA call."""
    lib = clis.load_library()
    INVALID, UNSUP = 1, 2
    assert lib.clis_host_plan_create(ctypes.byref(_shape(clis)), 0, 0, None) == INVALID
    assert _plan(clis, None)[0] == INVALID
    assert _plan(clis, _shape(clis), causal=2)[0] == INVALID
    assert _plan(clis, _shape(clis), groups=-1)[0] == INVALID
    assert _plan(clis, _shape(clis, Nk=0))[0] == INVALID
    s = _shape(clis)
    s.dtype = 5
    assert _plan(clis, s)[0] == INVALID
    assert _plan(clis, _shape(clis, d=96))[0] == UNSUP
    assert _plan(clis, _shape(clis, Nq=300, Nk=400), causal=1)[0] == UNSUP
    for field, val in (("k_sn", 136), ("q_sh", 300 * 128 + 8), ("o_sb", 0), ("v_sh", 0)):
        s = _shape(clis, B=2)
        setattr(s, field, val)
        st, h = _plan(clis, s)
        assert st == UNSUP and not h.value, field  # not dense
    vp = ctypes.c_void_p
    assert lib.clis_attention_host(None, vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), 0.1, 0, vp(FAKE), 1 << 30,
                                   None) == INVALID
    assert lib.clis_host_plan_wait(None, None) == INVALID
    assert lib.clis_host_plan_workspace_size(None, None) == INVALID
    assert lib.clis_host_plan_destroy(None) == 0


@pytest.mark.parametrize("B,H,Nq,Nk", [(0, 3, 300, 300), (1, 2, 0, 5)])
def test_host_plan_with_nothing_to_compute(clis, B, H, Nq, Nk):
    """B*H = 0 or Nq = 0: a plan without streams (no CUDA call), a workspace of
    0 bytes, calls that queue nothing; the scale and variant are still checked."""
    lib = clis.load_library()
    st, h = _plan(clis, _shape(clis, B=B, H=H, Nq=Nq, Nk=Nk))
    assert st == 0 and h.value
    n = ctypes.c_size_t(123)
    assert lib.clis_host_plan_workspace_size(h, ctypes.byref(n)) == 0 and n.value == 0
    vp = ctypes.c_void_p
    assert lib.clis_attention_host(h, None, None, None, None, 0.1, 0, None, 0, None) == 0
    assert lib.clis_attention_host(h, None, None, None, None, 0.0, 0, None, 0, None) == 1
    assert lib.clis_attention_host(h, None, None, None, None, 0.1, 9, None, 0, None) == 1
    assert lib.clis_host_plan_wait(h, None) == 0
    assert lib.clis_host_plan_destroy(h) == 0
    del vp
