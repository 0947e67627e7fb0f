"""CPU tests of the C ABI: libfa.so builds for sm_103a, loads, exports every function that
include/fa.h declares, and rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from exact_attention_81_gb300 import build
    build.build()
    import exact_attention_81_gb300 as fa
    return fa.load_library()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "fa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_header_symbols_exported(lib):
    names = _declared_functions()
    assert "fa_fwd" in names and "fa_fwd_varlen" in names and "fa_fwd_kvcache" in names
    for n in names:
        assert hasattr(lib, n), f"libfa.so does not export {n}"


def test_struct_layout(lib):
    from exact_attention_81_gb300._binding import BwdParams, FwdParams
    assert lib.fa_fwd_params_size() == ctypes.sizeof(FwdParams)
    assert lib.fa_bwd_params_size() == ctypes.sizeof(BwdParams)


def _bwd_params(**kw):
    from exact_attention_81_gb300._binding import BwdParams
    p = BwdParams()
    for name in ("q", "k", "v", "o", "dout", "lse", "dq", "dk", "dv"):
        setattr(p, name, 4096)
    p.B, p.Nq, p.Nk, p.Hq, p.Hkv, p.d = 1, 128, 128, 4, 2, 128
    for name in ("q_strides", "o_strides", "do_strides", "dq_strides"):
        getattr(p, name)[:] = [128 * 4 * 128, 4 * 128, 128]
    for name in ("k_strides", "v_strides", "dk_strides", "dv_strides"):
        getattr(p, name)[:] = [128 * 2 * 128, 2 * 128, 128]
    p.scale, p.causal, p.dtype = 0.088, 1, 0
    p.workspace, p.workspace_bytes = 4096, 1 << 30
    for k, v in kw.items():
        setattr(p, k, v)
    return p


@pytest.mark.parametrize("change,status", [
    ({"d": 100}, 2), ({"d": 264}, 2), ({"dtype": 3}, 2), ({"Hkv": 3}, 1), ({"scale": 0.0}, 1),
    ({"dout": None}, 1),
    ({"lse": None}, 1), ({"dk": 4100}, 1), ({"workspace": None}, 4), ({"workspace_bytes": 16}, 4),
    ({"workspace": 4096 + 64}, 4), ({"B": 0}, 0),
])
def test_bwd_rejects_bad_arguments(lib, change, status):
    assert lib.fa_bwd(ctypes.byref(_bwd_params(**change)), None) == status


def test_bwd_workspace_size(lib):
    ws = lib.fa_bwd_workspace_size
    assert ws(2, 1000, 4, 128) == (2 * 1000 * 4 * 128 * 4 + ((2 * 4 * 1000 * 4 + 255) // 256) * 256
                                   + 256)  # 2 x 4 x 8 block counters
    # width 256 (d 136..256): the transposed accumulator [B, Hq, d, Nq rounded up to 4] and
    # counters per (b, h, 64-query block, d half)
    assert ws(2, 1001, 4, 256) == (2 * 4 * 256 * 1004 * 4 + ((2 * 4 * 1001 * 4 + 255) // 256) * 256
                                   + 1024)  # 2 x 4 x 16 x 2 counters
    assert ws(0, 10, 4, 128) == 0


def _params(**kw):
    from exact_attention_81_gb300._binding import FwdParams
    p = FwdParams()
    p.q = p.k = p.v = p.o = 4096
    p.lse = 4096
    p.B, p.Nq, p.Nk, p.Hq, p.Hkv, p.d = 1, 128, 128, 4, 2, 128
    for name in ("q_strides", "k_strides", "v_strides", "o_strides"):
        getattr(p, name)[:] = [128 * 4 * 128, 4 * 128, 128]
    p.scale = 0.088
    p.causal = 0
    for k, v in kw.items():
        setattr(p, k, v)
    return p


@pytest.mark.parametrize("change,status", [
    ({"d": 100}, 2), ({"d": 264}, 2), ({"d": 252}, 2), ({"d": 0}, 2), ({"d": 4}, 2), ({"dtype": 2}, 2), ({"dtype": -1}, 2), ({"Hkv": 3}, 1), ({"Hq": 0}, 1), ({"B": -1}, 1),
    ({"scale": 0.0}, 1), ({"scale": float("nan")}, 1), ({"scale": -1.0}, 1),
    ({"q": 4098}, 1), ({"o": 4100}, 1), ({"lse": 4098}, 1), ({"q": None}, 1),
    ({"k": None}, 1), ({"Nq": -5}, 1),
])
def test_fwd_rejects_bad_arguments(lib, change, status):
    p = _params(**change)
    assert lib.fa_fwd(ctypes.byref(p), None) == status


def _mod(**kw):
    from exact_attention_81_gb300._binding import ScoreMod
    m = ScoreMod()
    for k, v in kw.items():
        setattr(m, k, v)
    return m


@pytest.mark.parametrize("mod", [
    dict(softcap=-0.5), dict(softcap=float("nan")), dict(softcap=float("inf")),
    dict(alibi_slopes=4097), dict(alibi_slopes=4096, alibi_batch_stride=-1),
])
def test_fwd_rejects_bad_score_mod(lib, mod):
    p = _params()
    p.mod = _mod(**mod)
    assert lib.fa_fwd(ctypes.byref(p), None) == 1


def test_fwd_rejects_misaligned_stride(lib):
    p = _params()
    p.q_strides[1] = 4 * 128 + 4  # not a multiple of 8 elements
    assert lib.fa_fwd(ctypes.byref(p), None) == 1


def test_fwd_empty_batch_is_noop(lib):
    assert lib.fa_fwd(ctypes.byref(_params(B=0)), None) == 0
    assert lib.fa_fwd(ctypes.byref(_params(Nq=0)), None) == 0
    assert lib.fa_fwd(None, None) == 1


def test_varlen_rejects_bad_arguments(lib):
    f = lib.fa_fwd_varlen
    good = dict(q=4096, k=4096, v=4096, o=4096, lse=4096, cq=4096, ck=4096, B=2, mq=10, mk=10,
                tq=20, tk=20, Hq=4, Hkv=2, d=64, scale=0.1, causal=1, dtype=0)

    def call(**kw):
        a = dict(good, **kw)
        return f(a["q"], a["k"], a["v"], a["o"], a["lse"], a["cq"], a["ck"], a["B"], a["mq"],
                 a["mk"], a["tq"], a["tk"], a["Hq"], a["Hkv"], a["d"], a["scale"], a["causal"],
                 a["dtype"], a.get("mod"), None)

    assert call(d=84) == 2
    assert call(d=264) == 2
    assert call(dtype=3) == 2
    assert call(Hkv=3) == 1
    assert call(cq=None) == 1
    assert call(q=4097) == 1
    assert call(tq=-1) == 1
    assert call(B=0) == 0
    assert call(tq=0) == 0
    assert call(mod=ctypes.byref(_mod(softcap=-1.0))) == 1
    assert call(mod=ctypes.byref(_mod(alibi_slopes=4098))) == 1


def test_kvcache_rejects_bad_arguments(lib):
    strides = (ctypes.c_int64 * 3)(1024 * 8 * 128, 8 * 128, 128)

    def call(**kw):
        a = dict(q=4096, kc=4096, vc=4096, lens=4096, B=2, L=1024, Hq=32, Hkv=8, d=128,
                 scale=0.1, ns=0, ws=4096, wsb=1 << 30, o=4096, lse=4096, dtype=0)
        a.update(kw)
        return lib.fa_fwd_kvcache(a["q"], a["kc"], a["vc"], a["lens"], a["B"], a["L"], a["Hq"],
                                  a["Hkv"], a["d"], strides, a["scale"], a["ns"], a["ws"],
                                  a["wsb"], a["o"], a["lse"], a["dtype"], a.get("mod"),
                                  a.get("ex"), None)

    # any group size passes host validation (without a GPU the call then stops at the
    # device lookup, never at an argument check)
    for hq, hkv in ((32, 2), (32, 1), (24, 8), (12, 2)):
        assert call(Hq=hq, Hkv=hkv) not in (1, 2, 4)
    assert call(dtype=5) == 2
    assert call(d=36) == 2
    assert call(d=264) == 2                 # decode serves d up to 256
    assert call(Hkv=5) == 1
    assert call(ns=-1) == 1
    assert call(lens=None) == 1
    assert call(ws=None) == 4
    need = lib.fa_fwd_kvcache_workspace_size(2, 32, 1024, 128, 0)
    assert call(wsb=need - 1) == 4
    assert call(ws=4096 + 16) == 4          # workspace must be 256-byte aligned
    assert call(B=0) == 0
    assert call(mod=ctypes.byref(_mod(softcap=float("inf")))) == 1
    from exact_attention_81_gb300._binding import KvCacheExtras

    def ex(**kw):
        e = KvCacheExtras()
        for k, v in kw.items():
            setattr(e, k, v)
        return ctypes.byref(e)
    assert call(ex=ex(k_new=4096)) == 1                                  # v_new missing
    assert call(ex=ex(rotary_cos=4096, rotary_sin=4096, rotary_dim=64,
                      rotary_positions=10)) == 1                         # rotary without append
    assert call(ex=ex(k_new=4096, v_new=4096, rotary_cos=4096, rotary_sin=4096,
                      rotary_dim=63, rotary_positions=10)) == 1          # odd rotary_dim
    assert call(ex=ex(k_new=4096, v_new=4096, rotary_cos=4096, rotary_sin=4096,
                      rotary_dim=256, rotary_positions=10)) == 1         # rotary_dim > d
    assert call(ex=ex(block_table=4096, block_table_stride=8, page_size=100,
                      num_pages=4)) == 1                                 # page not 128-multiple
    assert call(ex=ex(block_table=4096, block_table_stride=4, page_size=128,
                      num_pages=4)) == 1                                 # table shorter than Lmax
    assert call(mod=ctypes.byref(_mod(alibi_slopes=4096, alibi_batch_stride=-32))) == 1


def test_kvcache_fp8_rejects_bad_arguments(lib):
    strides = (ctypes.c_int64 * 3)(1024 * 8 * 128, 8 * 128, 128)

    def call(**kw):
        a = dict(q=4096, kc=4096, vc=4096, lens=4096, B=2, L=1024, Hq=32, Hkv=8, d=128,
                 scale=0.1, ns=0, kd=None, vd=None, ws=4096, wsb=1 << 30, o=4096, lse=4096)
        a.update(kw)
        return lib.fa_fwd_kvcache_fp8(a["q"], a["kc"], a["vc"], a["lens"], a["B"], a["L"],
                                      a["Hq"], a["Hkv"], a["d"], strides, a["scale"], a["ns"],
                                      a["kd"], a["vd"], a["ws"], a["wsb"], a["o"], a["lse"],
                                      a.get("mod"), a.get("ex"), None)

    assert call(d=8) == 2                   # E4M3 rows: d a multiple of 16
    assert call(d=24) == 2
    assert call(d=272) == 2
    assert call(Hq=32, Hkv=1) not in (1, 2, 4)   # MQA 32:1 passes host validation
    assert call(kd=4098) == 1               # descale pointers 4-byte aligned
    assert call(vd=4097) == 1
    assert call(lens=None) == 1
    assert call(ws=None) == 4
    assert call(B=0) == 0
    from exact_attention_81_gb300._binding import KvCacheExtras
    e = KvCacheExtras()
    e.k_new, e.v_new = 4096, 4096
    assert call(ex=ctypes.byref(e)) == 2    # no append into an E4M3 cache


def test_workspace_size(lib):
    ws = lib.fa_fwd_kvcache_workspace_size
    # automatic chunking: ~16 splits of a full-length cache, chunk >= 256, multiple of 128
    assert ws(64, 32, 32768, 128, 0) == 64 * 32 * 16 * 129 * 4
    assert ws(1, 1, 100, 64, 0) == ((1 * 1 * 1 * 65 * 4 + 255) // 256) * 256
    assert ws(2, 4, 1000, 64, 3) == 2 * 4 * 3 * 65 * 4 // 256 * 256 + (256 if (2 * 4 * 3 * 65 * 4) % 256 else 0)
    assert ws(0, 4, 100, 64, 0) == 0
    assert ws(2, 4, 100, 64, -1) == 0


def test_status_strings(lib):
    lib.fa_status_string.restype = ctypes.c_char_p
    for s in range(7):
        assert lib.fa_status_string(s).decode().startswith("FA_")


def test_fp8_rejects_bad_arguments(lib):
    """fa_fwd_fp8 validates before any CUDA call: dtype must be E4M3, d a multiple of 16 up
    to 128, 8-bit strides multiples of 16, a large enough 256-byte-aligned workspace."""
    from exact_attention_81_gb300._binding import FwdParams
    B, Nq, Nk, Hq, Hkv, d = 2, 100, 300, 4, 2, 128

    def call(ws=4096, wsb=1 << 30, **kw):
        p = FwdParams()
        for name in ("q", "k", "v", "o", "lse"):
            setattr(p, name, 4096)
        p.B, p.Nq, p.Nk, p.Hq, p.Hkv, p.d = B, Nq, Nk, Hq, Hkv, d
        p.q_strides[:] = [Nq * Hq * d, Hq * d, d]
        p.k_strides[:] = p.v_strides[:] = [Nk * Hkv * d, Hkv * d, d]
        p.o_strides[:] = [Nq * Hq * d, Hq * d, d]
        p.scale, p.causal, p.dtype = 0.088, 1, 2
        for key, val in kw.items():
            if key.endswith("_strides"):
                getattr(p, key)[:] = val
            else:
                setattr(p, key, val)
        return lib.fa_fwd_fp8(ctypes.byref(p), None, None, None, ws, wsb, None)

    assert call(dtype=0) == 2                      # bf16 inputs: use fa_fwd
    assert call(d=120) == 2 and call(d=144) == 2 and call(d=8) == 2
    assert call(q_strides=[Nq * Hq * d, Hq * d + 8, d]) == 1   # 8-bit stride not % 16
    assert call(k=4104) == 1                       # misaligned pointer
    assert call(ws=None) == 4
    need = lib.fa_fwd_fp8_workspace_size(B, Nk, Hkv, d)
    assert need == ((B * Hkv * d * 304 + 255) // 256) * 256   # keys padded to 304
    assert call(wsb=need - 1) == 4
    assert call(ws=4096 + 128) == 4                # workspace not 256-byte aligned
    assert call(B=0) == 0 and call(Nq=0) == 0      # nothing to do
    assert lib.fa_fwd_fp8_workspace_size(0, 10, 2, 128) == 0


def test_varlen_fp8_rejects_bad_arguments(lib):
    """fa_fwd_varlen_fp8 validates before any CUDA call: d a multiple of 16 up to 128, at
    most 65535 sequences, aligned pointers, a large enough 256-byte-aligned workspace (the
    transposed V with every sequence from a 16-aligned column)."""
    B, total_q, total_k, Hq, Hkv, d = 3, 500, 700, 4, 2, 128

    def call(ws=4096, wsb=1 << 30, **kw):
        a = dict(q=4096, k=4096, v=4096, o=4096, lse=4096, cu_q=4096, cu_k=4096, B=B,
                 max_q=300, max_k=400, total_q=total_q, total_k=total_k, Hq=Hq, Hkv=Hkv, d=d)
        a.update(kw)
        return lib.fa_fwd_varlen_fp8(a["q"], a["k"], a["v"], a["o"], a["lse"], a["cu_q"],
                                     a["cu_k"], a["B"], a["max_q"], a["max_k"], a["total_q"],
                                     a["total_k"], a["Hq"], a["Hkv"], a["d"], 0.088, 1, None,
                                     None, None, None, ws, wsb, None)

    assert call(d=120) == 2 and call(d=144) == 2 and call(d=8) == 2
    assert call(B=70000) == 1                      # more sequences than a grid dimension
    assert call(Hq=3) == 1                         # Hq not a multiple of Hkv
    assert call(k=4104) == 1 and call(cu_k=4098) == 1   # misaligned pointers
    assert call(ws=None) == 4
    need = lib.fa_fwd_varlen_fp8_workspace_size(B, total_k, Hkv, d)
    assert need == ((Hkv * d * (704 + 16 * (B + 1)) + 255) // 256) * 256
    assert call(wsb=need - 1) == 4
    assert call(ws=4096 + 128) == 4                # workspace not 256-byte aligned
    assert call(B=0) == 0 and call(total_q=0) == 0     # nothing to do
    assert lib.fa_fwd_varlen_fp8_workspace_size(0, 10, 2, 128) == 0


def test_host_call_rejects_bad_arguments(lib):
    """fa_fwd_host validates before any CUDA call: 1..64 ranges, contiguous layouts, device
    buffers present and aligned."""
    from exact_attention_81_gb300._binding import FwdParams
    B, Nq, Nk, Hq, Hkv, d = 2, 300, 300, 4, 2, 64

    def call(chunks=4, bufs=(4096, 4096, 4096, 4096, 4096), **kw):
        p = FwdParams()
        for name in ("q", "k", "v", "o", "lse"):
            setattr(p, name, 8192)
        p.B, p.Nq, p.Nk, p.Hq, p.Hkv, p.d = B, Nq, Nk, Hq, Hkv, d
        p.q_strides[:] = p.o_strides[:] = [Nq * Hq * d, Hq * d, d]
        p.k_strides[:] = p.v_strides[:] = [Nk * Hkv * d, Hkv * d, d]
        p.scale, p.causal, p.dtype = 0.1, 1, 0
        for key, val in kw.items():
            if key.endswith("_strides"):
                getattr(p, key)[:] = val
            else:
                setattr(p, key, val)
        return lib.fa_fwd_host(ctypes.byref(p), *bufs, chunks, None)

    assert call(chunks=0) == 1 and call(chunks=65) == 1
    assert call(q_strides=[Nq * Hq * d, Hq * d + 8, d]) == 1      # not contiguous
    assert call(k_strides=[Nk * Hkv * d * 2, Hkv * d, d]) == 1    # batch stride padded
    assert call(bufs=(None, 4096, 4096, 4096, 4096)) == 1
    assert call(bufs=(4096, 4096, 4096, 4104, 4096)) == 1         # device O misaligned
    assert call(d=100) == 2 and call(dtype=2) == 2
    assert call(B=0) == 0
