"""fp64 CPU oracle for exact attention -- Python side (ctypes over attn_oracle.c).

TEST INFRASTRUCTURE ONLY.  The product path (the CUDA library and its Python
binding) never imports this module; only the tests, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` do.  It shares no code with the CUDA
path: the C source is compiled here with gcc into ``oracle/_build``.

Every function takes bf16 or fp16 inputs (torch tensors, or their 16-bit patterns as
numpy ``uint16`` with ``elem`` = 0 for bf16, 1 for fp16) so that the oracle reads
exactly the numbers the GPU reads, widens them exactly to double and computes the
plain definition of attention
("FlashAttention 1-4 详解", section 原算法: S = Q K^T, P = softmax(scale * S),
O = P V; plus the natural-log log-sum-exp of each row of scaled scores).

Every function also takes the score modifiers of "flash-attention" (capabilities table:
sliding window, ALiBi, softcap): ``window=(left, right)`` (negative = unbounded; causal
sets right = 0), ``softcap`` (0 = off) and ``alibi_slopes`` (fp32 ``[Hq]`` or ``[B, Hq]``),
read as described in attn_oracle.c.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile attn_oracle.c with gcc (plain -O2, IEEE double, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            lib = ctypes.CDLL(path)
            p = ctypes.c_void_p
            i = ctypes.c_int
            i64 = ctypes.c_int64
            d = ctypes.c_double
            mod = [i, i, d, p, i64]  # window_left, window_right, softcap, alibi, alibi_sb
            lib.oracle_fwd.argtypes = [p, p, p, i, i, i, i, i, i, p, p, p, d, i, p, p, i,
                                       i] + mod
            lib.oracle_fwd_rows.argtypes = [p, p, p, i, i, i, i, i, i, p, p, p, d, i, p, i64,
                                            p, p, i, i] + mod
            lib.oracle_fwd_varlen.argtypes = [p, p, p, p, p, i, i, i, i, p, p, p, d, i, p, p, i,
                                              i] + mod
            lib.oracle_fwd_kvcache.argtypes = [p, p, p, p, i, i, i, i, i, p, p, p, d, p, p, i,
                                               i] + mod
            lib.oracle_row_probs.argtypes = [p, p, p, i, i, i, i, i, i, p, p, p, d, i, i, i, i,
                                             p, i] + mod
            lib.oracle_rotary.argtypes = [p, i64, i64, i, p, p, p, i, i, p, i]
            lib.oracle_bwd.argtypes = [p, p, p, p, i, i, i, i, i, i, p, p, p, p, d, i, p, p, p,
                                       p, p, i, i] + mod
            lib.oracle_bwd.restype = ctypes.c_int
            lib.oracle_round16.argtypes = [p, i64, p, i]
            for f in (lib.oracle_fwd, lib.oracle_fwd_rows, lib.oracle_fwd_varlen,
                      lib.oracle_fwd_kvcache, lib.oracle_row_probs, lib.oracle_rotary,
                      lib.oracle_round16):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _threads(n):
    return int(n) if n else (os.cpu_count() or 1)


_ELEM = {"torch.bfloat16": 0, "torch.float16": 1}


def _elem_of(a, default=0) -> int:
    return _ELEM.get(str(getattr(a, "dtype", "")), default)


def _bits(a) -> np.ndarray:
    """Accept a numpy uint16 array or a torch bf16 / fp16 tensor; return uint16 bits."""
    if str(getattr(a, "dtype", "")) in _ELEM:
        import torch  # local: only the tests hand torch tensors in
        a = a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("oracle inputs are 16-bit float bit patterns (uint16)")
    return a


def _common_elem(*ts, elem=None) -> int:
    if elem is not None:
        return int(elem)
    kinds = {_elem_of(t) for t in ts}
    if len(kinds) != 1:
        raise TypeError("q, k and v must share one element type")
    return kinds.pop()


class _Mod:
    """Marshalled score modifiers; keeps the slope array alive for the call."""

    def __init__(self, B, Hq, window=(-1, -1), softcap=0.0, alibi_slopes=None):
        wl, wr = (-1, -1) if window is None else window
        self.wl, self.wr = int(wl), int(wr)
        self.softcap = float(softcap or 0.0)
        self.slopes = None
        self.sb = 0
        if alibi_slopes is not None:
            a = alibi_slopes
            if hasattr(a, "detach"):
                a = a.detach().cpu().numpy()
            a = np.asarray(a)
            if a.dtype != np.float32:
                raise TypeError("ALiBi slopes are fp32")
            if a.ndim == 1 and a.shape[0] == Hq:
                self.sb = 0
            elif a.ndim == 2 and a.shape == (B, Hq):
                self.sb = Hq
            else:
                raise ValueError("ALiBi slopes must be [Hq] or [B, Hq]")
            self.slopes = np.ascontiguousarray(a.astype(np.float64))

    def args(self):
        ptr = _ptr(self.slopes) if self.slopes is not None else None
        return (self.wl, self.wr, self.softcap, ptr, self.sb)


def _strides4(a: np.ndarray):
    """(b, n, h) element strides of a contiguous [B, N, H, d] array."""
    s = [x // a.itemsize for x in a.strides]
    return (ctypes.c_int64 * 3)(s[0], s[1], s[2])


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def attention(q, k, v, scale: float, causal: bool = False, nthreads: int | None = None,
              elem=None, window=(-1, -1), softcap=0.0, alibi_slopes=None):
    """Dense attention.  q [B,Nq,Hq,d], k/v [B,Nk,Hkv,d] (bf16 or fp16).

    Returns (O [B,Nq,Hq,d] float64, LSE [B,Hq,Nq] float64).
    """
    el = _common_elem(q, k, v, elem=elem)
    q, k, v = _bits(q), _bits(k), _bits(v)
    B, Nq, Hq, d = q.shape
    _, Nk, Hkv, _ = k.shape
    mod = _Mod(B, Hq, window, softcap, alibi_slopes)
    o = np.zeros((B, Nq, Hq, d), np.float64)
    lse = np.zeros((B, Hq, Nq), np.float64)
    rc = _load().oracle_fwd(_ptr(q), _ptr(k), _ptr(v), B, Nq, Nk, Hq, Hkv, d, _strides4(q),
                            _strides4(k), _strides4(v), float(scale), int(bool(causal)),
                            _ptr(o), _ptr(lse), _threads(nthreads), el, *mod.args())
    if rc != 0:
        raise ValueError("oracle_fwd rejected its arguments")
    return o, lse


def attention_rows(q, k, v, rows, scale: float, causal: bool = False,
                   nthreads: int | None = None, elem=None, window=(-1, -1), softcap=0.0,
                   alibi_slopes=None):
    """Dense attention on selected rows; rows is an (n, 3) int array of (b, h, i).

    Returns (O [n, d] float64, LSE [n] float64).
    """
    el = _common_elem(q, k, v, elem=elem)
    q, k, v = _bits(q), _bits(k), _bits(v)
    B, Nq, Hq, d = q.shape
    _, Nk, Hkv, _ = k.shape
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 3))
    n = rows.shape[0]
    mod = _Mod(B, Hq, window, softcap, alibi_slopes)
    o = np.zeros((n, d), np.float64)
    lse = np.zeros((n,), np.float64)
    rc = _load().oracle_fwd_rows(_ptr(q), _ptr(k), _ptr(v), B, Nq, Nk, Hq, Hkv, d,
                                 _strides4(q), _strides4(k), _strides4(v), float(scale),
                                 int(bool(causal)), _ptr(rows), n, _ptr(o), _ptr(lse),
                                 _threads(nthreads), el, *mod.args())
    if rc != 0:
        raise ValueError("oracle_fwd_rows rejected its arguments")
    return o, lse


def attention_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, scale: float, causal: bool = False,
                     nthreads: int | None = None, elem=None, window=(-1, -1), softcap=0.0,
                     alibi_slopes=None):
    """Packed varlen attention.  q [total_q,Hq,d], k/v [total_k,Hkv,d].

    Returns (O [total_q,Hq,d] float64, LSE [Hq,total_q] float64).
    """
    el = _common_elem(q, k, v, elem=elem)
    q, k, v = _bits(q), _bits(k), _bits(v)
    cu_q = np.ascontiguousarray(np.asarray(cu_seqlens_q, dtype=np.int32))
    cu_k = np.ascontiguousarray(np.asarray(cu_seqlens_k, dtype=np.int32))
    B = cu_q.shape[0] - 1
    total_q, Hq, d = q.shape
    Hkv = k.shape[1]

    def st3(a):
        s = [x // a.itemsize for x in a.strides]
        return (ctypes.c_int64 * 3)(0, s[0], s[1])

    mod = _Mod(B, Hq, window, softcap, alibi_slopes)
    o = np.zeros((total_q, Hq, d), np.float64)
    lse = np.zeros((Hq, total_q), np.float64)
    rc = _load().oracle_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_q), _ptr(cu_k), B, Hq,
                                   Hkv, d, st3(q), st3(k), st3(v), float(scale),
                                   int(bool(causal)), _ptr(o), _ptr(lse), _threads(nthreads),
                                   el, *mod.args())
    if rc != 0:
        raise ValueError("oracle_fwd_varlen rejected its arguments")
    return o, lse


def attention_kvcache(q, k_cache, v_cache, cache_seqlens, scale: float,
                      nthreads: int | None = None, elem=None, window=(-1, -1), softcap=0.0,
                      alibi_slopes=None):
    """Single-query decode.  q [B,1,Hq,d], caches [B,Lmax,Hkv,d], lengths [B].

    Returns (O [B,Hq,d] float64, LSE [B,Hq] float64).
    """
    el = _common_elem(q, k_cache, v_cache, elem=elem)
    q, kc, vc = _bits(q), _bits(k_cache), _bits(v_cache)
    lens = np.ascontiguousarray(np.asarray(cache_seqlens, dtype=np.int32))
    B, _, Hq, d = q.shape
    _, Lmax, Hkv, _ = kc.shape
    mod = _Mod(B, Hq, window, softcap, alibi_slopes)
    o = np.zeros((B, Hq, d), np.float64)
    lse = np.zeros((B, Hq), np.float64)
    rc = _load().oracle_fwd_kvcache(_ptr(q), _ptr(kc), _ptr(vc), _ptr(lens), B, Lmax, Hq, Hkv,
                                    d, _strides4(q), _strides4(kc), _strides4(vc),
                                    float(scale), _ptr(o), _ptr(lse), _threads(nthreads), el,
                                    *mod.args())
    if rc != 0:
        raise ValueError("oracle_fwd_kvcache rejected its arguments")
    return o, lse


def row_probs(q, k, v, b: int, h: int, i: int, scale: float, causal: bool = False, elem=None,
              window=(-1, -1), softcap=0.0, alibi_slopes=None):
    """Softmax probabilities P[i, :] of one dense row (zeros on invisible keys)."""
    el = _common_elem(q, k, v, elem=elem)
    q, k, v = _bits(q), _bits(k), _bits(v)
    B, Nq, Hq, d = q.shape
    _, Nk, Hkv, _ = k.shape
    mod = _Mod(B, Hq, window, softcap, alibi_slopes)
    p = np.zeros((Nk,), np.float64)
    rc = _load().oracle_row_probs(_ptr(q), _ptr(k), _ptr(v), B, Nq, Nk, Hq, Hkv, d,
                                  _strides4(q), _strides4(k), _strides4(v), float(scale),
                                  int(bool(causal)), b, h, i, _ptr(p), el, *mod.args())
    if rc != 0:
        raise ValueError("oracle_row_probs rejected its arguments")
    return p


# --------------------------------------------------------------------------
# KV-cache extras ("flash-attention", section 1: the decode call appends the new key and
# value to the cache in place and applies rotary in the same step; capabilities table,
# KV cache row: in-place append, paged KV).


def round16(x, elem: int = 0) -> np.ndarray:
    """fp32 values -> bf16 (elem 0) or fp16 (elem 1) bit patterns, round to nearest even."""
    x = np.ascontiguousarray(np.asarray(x, np.float32))
    out = np.zeros(x.shape, np.uint16)
    if _load().oracle_round16(_ptr(x), x.size, _ptr(out), int(elem)) != 0:
        raise ValueError("oracle_round16 rejected its arguments")
    return out


def rotary(x, positions, cos, sin, interleaved: bool = False, elem=None) -> np.ndarray:
    """Rotary embedding of vectors x [..., d] (16-bit) at integer positions [...] with fp32
    tables cos/sin [P, rotary_dim / 2]; returns uint16 bits of the same shape."""
    el = _common_elem(x, elem=elem)
    xb = _bits(x)
    d = xb.shape[-1]
    rows = xb.reshape(-1, d)
    pos = np.ascontiguousarray(np.asarray(positions, np.int32).reshape(-1))
    cos = np.ascontiguousarray(np.asarray(cos, np.float32))
    sin = np.ascontiguousarray(np.asarray(sin, np.float32))
    if pos.shape[0] != rows.shape[0] or cos.shape != sin.shape or cos.ndim != 2:
        raise ValueError("rotary: one position per row and tables [P, rotary_dim / 2]")
    if pos.size and (pos.min() < 0 or pos.max() >= cos.shape[0]):
        raise ValueError("rotary: position outside the tables")
    out = np.zeros(rows.shape, np.uint16)
    rc = _load().oracle_rotary(_ptr(rows), d, rows.shape[0], d, _ptr(pos), _ptr(cos),
                               _ptr(sin), 2 * cos.shape[1], int(bool(interleaved)),
                               _ptr(out), el)
    if rc != 0:
        raise ValueError("oracle_rotary rejected its arguments")
    return out.reshape(xb.shape)


def kvcache_step(q, k_cache, v_cache, cache_seqlens, scale: float, k_new=None, v_new=None,
                 rotary_cos=None, rotary_sin=None, rotary_interleaved: bool = False,
                 block_table=None, nthreads: int | None = None, elem=None, window=(-1, -1),
                 softcap=0.0, alibi_slopes=None):
    """One decode step against a KV cache, the way the decode call reads it:

    1. with k_new / v_new ([B, 1, Hkv, d]): the new key (rotated when tables are given)
       and value are written at logical row cache_seqlens[b] of sequence b, and the query
       is rotated at the same position;
    2. the query attends to logical rows [0, cache_seqlens[b] (+ 1 after an append)).

    Contiguous caches are [B, Lmax, Hkv, d]; paged ones (block_table [B, nblk] int32) are
    [num_pages, page_size, Hkv, d], logical row r of sequence b being row r % page_size of
    page block_table[b, r // page_size].

    Returns (O [B, Hq, d] float64, LSE [B, Hq] float64, k_cache, v_cache) with the caches
    after the append as uint16 bits in the caller's layout.
    """
    el = _common_elem(q, k_cache, v_cache, elem=elem)
    qb, kc, vc = _bits(q).copy(), _bits(k_cache).copy(), _bits(v_cache).copy()
    lens = np.asarray(cache_seqlens, np.int64).reshape(-1).copy()
    B, _, Hq, d = qb.shape
    Hkv = kc.shape[2]
    bt = None if block_table is None else np.asarray(block_table, np.int64)
    if bt is None:
        Lmax = kc.shape[1]
    else:
        page = kc.shape[1]
        Lmax = bt.shape[1] * page

    def locate(b, r):
        """(page or batch index, row) of logical row r of sequence b."""
        if bt is None:
            return b, r
        pg = int(bt[b, r // page])
        if pg < 0 or pg >= kc.shape[0]:
            raise ValueError("block table entry outside the cache")
        return pg, r % page

    if (k_new is None) != (v_new is None):
        raise ValueError("k_new and v_new go together")
    if rotary_cos is not None and k_new is None:
        raise ValueError("rotary applies to an appended key")
    if np.any(lens < 0) or np.any(lens > Lmax):
        raise ValueError("cache length outside [0, Lmax]")
    if k_new is not None:
        kn, vn = _bits(k_new).copy(), _bits(v_new).copy()
        if np.any(lens + 1 > Lmax):
            raise ValueError("no room for the appended row")
        if rotary_cos is not None:
            kn = rotary(kn, np.repeat(lens, Hkv).reshape(B, 1, Hkv), rotary_cos, rotary_sin,
                        rotary_interleaved, elem=el)
            qb = rotary(qb, np.repeat(lens, Hq).reshape(B, 1, Hq), rotary_cos, rotary_sin,
                        rotary_interleaved, elem=el)
        for b in range(B):
            i0, r = locate(b, int(lens[b]))
            kc[i0, r] = kn[b, 0]
            vc[i0, r] = vn[b, 0]
        lens = lens + 1
    if bt is None:
        kl, vl = kc, vc
    else:
        kl = np.full((B, Lmax, Hkv, d), 0x7fc0, np.uint16)  # NaN in both 16-bit types
        vl = kl.copy()
        for b in range(B):
            for r in range(int(lens[b])):
                i0, rr = locate(b, r)
                kl[b, r] = kc[i0, rr]
                vl[b, r] = vc[i0, rr]
    o, lse = attention_kvcache(qb, kl, vl, lens.astype(np.int32), scale, nthreads, el,
                               window=window, softcap=softcap, alibi_slopes=alibi_slopes)
    return o, lse, kc, vc


# --------------------------------------------------------------------------
# Backward pass ("flash-attention", sections 2.3 and 4: gradients recomputed from q, k, v,
# out and softmax_lse; "FlashAttention 1-4 详解", FlashAttention 2 backward).


def attention_bwd(q, k, v, dout, scale: float, causal: bool = False,
                  nthreads: int | None = None, elem=None, window=(-1, -1), softcap=0.0,
                  alibi_slopes=None):
    """Gradients of dense attention for the upstream gradient dout [B,Nq,Hq,d].

    Returns (dQ [B,Nq,Hq,d], dK [B,Nk,Hkv,d], dV [B,Nk,Hkv,d], LSE [B,Hq,Nq],
    D [B,Hq,Nq]) in float64, D_i = dO_i . O_i.
    """
    el = _common_elem(q, k, v, dout, elem=elem)
    q, k, v, dout = _bits(q), _bits(k), _bits(v), _bits(dout)
    B, Nq, Hq, d = q.shape
    _, Nk, Hkv, _ = k.shape
    if dout.shape != q.shape:
        raise ValueError("dout must have the shape of q")
    mod = _Mod(B, Hq, window, softcap, alibi_slopes)
    dq = np.zeros((B, Nq, Hq, d), np.float64)
    dk = np.zeros((B, Nk, Hkv, d), np.float64)
    dv = np.zeros((B, Nk, Hkv, d), np.float64)
    lse = np.zeros((B, Hq, Nq), np.float64)
    D = np.zeros((B, Hq, Nq), np.float64)
    rc = _load().oracle_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), B, Nq, Nk, Hq, Hkv, d,
                            _strides4(q), _strides4(k), _strides4(v), _strides4(dout),
                            float(scale), int(bool(causal)), _ptr(dq), _ptr(dk), _ptr(dv),
                            _ptr(lse), _ptr(D), _threads(nthreads), el, *mod.args())
    if rc != 0:
        raise ValueError("oracle_bwd rejected its arguments")
    return dq, dk, dv, lse, D


def attention_varlen_bwd(q, k, v, dout, cu_seqlens_q, cu_seqlens_k, scale: float,
                         causal: bool = False, nthreads: int | None = None, elem=None,
                         window=(-1, -1), softcap=0.0, alibi_slopes=None):
    """Gradients of packed varlen attention: each sequence is an independent dense problem
    (capabilities table, varlen row), so this applies attention_bwd sequence by sequence.
    q, dout [total_q, Hq, d]; k, v [total_k, Hkv, d].  Returns (dQ, dK, dV) float64 in the
    packed layouts."""
    import torch  # local: only the tests hand torch tensors in
    cu_q = [int(x) for x in np.asarray(cu_seqlens_q).reshape(-1)]
    cu_k = [int(x) for x in np.asarray(cu_seqlens_k).reshape(-1)]
    dq = np.zeros(tuple(q.shape), np.float64)
    dk = np.zeros(tuple(k.shape), np.float64)
    dv = np.zeros(tuple(v.shape), np.float64)
    for b in range(len(cu_q) - 1):
        a, e = cu_q[b], cu_q[b + 1]
        ka, ke = cu_k[b], cu_k[b + 1]
        if e == a or ke == ka:
            continue  # no queries or no keys: every gradient of the sequence is 0
        sl = None
        if alibi_slopes is not None:
            sl = np.asarray(alibi_slopes.detach().cpu() if hasattr(alibi_slopes, "detach")
                            else alibi_slopes, np.float32)
            sl = sl[b] if sl.ndim == 2 else sl
        g = attention_bwd(q[a:e].unsqueeze(0).contiguous(), k[ka:ke].unsqueeze(0).contiguous(),
                          v[ka:ke].unsqueeze(0).contiguous(),
                          dout[a:e].unsqueeze(0).contiguous(), scale, causal, nthreads, elem,
                          window=window, softcap=softcap, alibi_slopes=sl)
        dq[a:e], dk[ka:ke], dv[ka:ke] = g[0][0], g[1][0], g[2][0]
    return dq, dk, dv


# ---------------------------------------------------------------------------------------
# FP8 inputs ("FlashAttention 1-4 详解", FlashAttention 3 engineering notes: FP8 tensor
# cores in the forward pass).  The 8-bit code is E4M3 as torch.float8_e4m3fn stores it:
# sign bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0 holds the
# subnormals m/8 * 2^-6; S.1111.111 is NaN; there is no infinity (largest value 448).

def e4m3_values() -> np.ndarray:
    """The 256 E4M3 code points as float64 (NaN for the two NaN codes)."""
    out = np.empty(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        e = (code >> 3) & 0xF
        m = code & 0x7
        if e == 0xF and m == 0x7:
            out[code] = np.nan
        elif e == 0:
            out[code] = sign * (m / 8.0) * 2.0 ** (1 - 7)
        else:
            out[code] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return out


def _u8(a) -> np.ndarray:
    """Accept a numpy uint8 array or a torch float8_e4m3fn / uint8 tensor; return codes."""
    if hasattr(a, "detach"):
        import torch  # local: only the tests hand torch tensors in
        t = a.detach().cpu().contiguous()
        if t.dtype != torch.uint8:
            t = t.view(torch.uint8)
        a = t.numpy()
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint8:
        raise TypeError("FP8 oracle inputs are E4M3 codes (uint8)")
    return a


def e4m3_to_bf16_bits(codes) -> np.ndarray:
    """E4M3 codes -> bf16 bit patterns of the same values.  Exact: a finite E4M3 value has
    at most 4 significant bits and an exponent in [-9, 8], both inside bf16."""
    v = e4m3_values()[_u8(codes)].astype(np.float32)
    bits = v.view(np.uint32)
    finite = np.isfinite(v)
    if np.any(bits[finite] & 0xFFFF):
        raise ValueError("E4M3 value not exact in bf16")
    return (bits >> 16).astype(np.uint16)


def attention_kvcache_fp8(q, k_cache, v_cache, cache_seqlens, scale: float, k_descale=None,
                          v_descale=None, nthreads: int | None = None, window=(-1, -1),
                          softcap=0.0, alibi_slopes=None):
    """Single-query decode of a bf16 query q [B,1,Hq,d] against E4M3 caches [B,Lmax,Hkv,d]
    with descale factors per (batch, kv head) ([B, Hkv] fp32, None = 1): the attended keys
    and values are dk * K and dv * V.  The plain decode definition with the score scale
    scale * dk on the decoded cache, and O times dv (O is linear in V).  Returns
    (O [B,Hq,d], LSE [B,Hq]) in float64."""
    qb = _bits(q)
    kb, vb = e4m3_to_bf16_bits(k_cache), e4m3_to_bf16_bits(v_cache)
    lens = np.asarray(cache_seqlens, dtype=np.int32).reshape(-1)
    B, _, Hq, d = qb.shape
    Hkv = kb.shape[2]
    G = Hq // Hkv

    def desc(x):
        if x is None:
            return np.ones((B, Hkv), dtype=np.float64)
        if hasattr(x, "detach"):
            x = x.detach().cpu().numpy()
        return np.asarray(x, dtype=np.float32).astype(np.float64).reshape(B, Hkv)

    dk, dv = desc(k_descale), desc(v_descale)
    slopes = None
    if alibi_slopes is not None:
        s_ = alibi_slopes.detach().cpu().numpy() if hasattr(alibi_slopes, "detach") \
            else np.asarray(alibi_slopes)
        slopes = np.broadcast_to(s_.astype(np.float32), (B, Hq))
    o_all = np.empty((B, Hq, d))
    lse_all = np.empty((B, Hq))
    for b in range(B):
        for g in range(Hkv):
            h0, h1 = g * G, (g + 1) * G  # the query heads of kv head g
            sigma = float(np.float32(scale)) * dk[b, g]
            o, lse = attention_kvcache(np.ascontiguousarray(qb[b:b + 1, :, h0:h1]),
                                       np.ascontiguousarray(kb[b:b + 1, :, g:g + 1]),
                                       np.ascontiguousarray(vb[b:b + 1, :, g:g + 1]),
                                       lens[b:b + 1], sigma, nthreads, elem=0, window=window,
                                       softcap=softcap,
                                       alibi_slopes=None if slopes is None else
                                       np.ascontiguousarray(slopes[b, h0:h1]))
            o_all[b, h0:h1] = o[0] * dv[b, g]
            lse_all[b, h0:h1] = lse[0]
    return o_all, lse_all


def attention_fp8(q, k, v, scale: float, causal: bool = False, q_descale=None,
                  k_descale=None, v_descale=None, nthreads: int | None = None,
                  window=(-1, -1), softcap=0.0, alibi_slopes=None):
    """Dense attention of E4M3 inputs q [B,Nq,Hq,d], k/v [B,Nk,Hkv,d] with descale factors
    per (batch, kv head) ([B, Hkv] fp32, None = 1): the values attended are dq * Q, dk * K
    and dv * V.  So the scores are (scale * dq * dk) q.k, the plain definition with that
    score scale, and O is dv times the attention of the unscaled V (O is linear in V; the
    LSE does not depend on V).  Returns (O [B,Nq,Hq,d], LSE [B,Hq,Nq]) in float64."""
    qb, kb, vb = (e4m3_to_bf16_bits(t) for t in (q, k, v))
    B, Nq, Hq, d = qb.shape
    Hkv = kb.shape[2]
    G = Hq // Hkv

    def desc(x):
        if x is None:
            return np.ones((B, Hkv), dtype=np.float64)
        if hasattr(x, "detach"):
            x = x.detach().cpu().numpy()
        return np.asarray(x, dtype=np.float32).astype(np.float64).reshape(B, Hkv)

    dq, dk, dv = desc(q_descale), desc(k_descale), desc(v_descale)
    slopes = None
    if alibi_slopes is not None:
        s = alibi_slopes.detach().cpu().numpy() if hasattr(alibi_slopes, "detach") \
            else np.asarray(alibi_slopes)
        slopes = np.broadcast_to(s.astype(np.float32), (B, Hq))
    o_all = np.empty((B, Nq, Hq, d))
    lse_all = np.empty((B, Hq, Nq))
    for b in range(B):
        for g in range(Hkv):
            hs = slice(g * G, (g + 1) * G)
            sigma = float(np.float32(scale)) * dq[b, g] * dk[b, g]
            o, lse = attention(np.ascontiguousarray(qb[b:b + 1, :, hs]),
                               np.ascontiguousarray(kb[b:b + 1, :, g:g + 1]),
                               np.ascontiguousarray(vb[b:b + 1, :, g:g + 1]), sigma, causal,
                               nthreads, elem=0, window=window, softcap=softcap,
                               alibi_slopes=None if slopes is None else
                               np.ascontiguousarray(slopes[b, hs]))
            o_all[b, :, hs] = o[0] * dv[b, g]
            lse_all[b, hs] = lse[0]
    return o_all, lse_all
