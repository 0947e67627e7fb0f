"""ctypes binding over libfa.so (the C ABI in include/fa.h).

Argument marshalling only: it checks tensor types, reads pointers, shapes and strides,
allocates outputs with torch when the caller does not pass them, and calls the C entry
point of the same name on the current CUDA stream.  Every step of the attention itself
runs in the library's CUDA kernels.  If libfa.so is missing or fails to load, every call
raises; there is no fallback.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfa.so")

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_CUDA = 3
FA_ERR_WORKSPACE = 4
FA_ERR_TIMEOUT = 5
FA_ERR_CONCURRENT = 6

FA_BF16 = 0
FA_FP16 = 1
FA_E4M3 = 2
_DTYPE = {torch.bfloat16: FA_BF16, torch.float16: FA_FP16}


class FAError(RuntimeError):
    """A libfa call returned a non-zero fa_status."""

    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = int(status)
        msg = f"{where}: {status_string(self.status)}"
        if detail:
            msg += f" [{detail}]"
        super().__init__(msg)


class ScoreMod(ctypes.Structure):
    """Mirror of fa_score_mod (sliding window, softcap, ALiBi; zero-filled = none)."""

    _fields_ = [
        ("use_window", ctypes.c_int),
        ("window_left", ctypes.c_int),
        ("window_right", ctypes.c_int),
        ("softcap", ctypes.c_float),
        ("alibi_slopes", ctypes.c_void_p),
        ("alibi_batch_stride", ctypes.c_int64),
    ]


class KvCacheExtras(ctypes.Structure):
    """Mirror of fa_kvcache_extras (in-place append, rotary, paged cache)."""

    _fields_ = [
        ("k_new", ctypes.c_void_p),
        ("v_new", ctypes.c_void_p),
        ("new_strides", ctypes.c_int64 * 3),
        ("rotary_cos", ctypes.c_void_p),
        ("rotary_sin", ctypes.c_void_p),
        ("rotary_dim", ctypes.c_int),
        ("rotary_positions", ctypes.c_int),
        ("rotary_interleaved", ctypes.c_int),
        ("block_table", ctypes.c_void_p),
        ("block_table_stride", ctypes.c_int),
        ("page_size", ctypes.c_int),
        ("num_pages", ctypes.c_int),
    ]


class FwdParams(ctypes.Structure):
    """Mirror of fa_fwd_params."""

    _fields_ = [
        ("q", ctypes.c_void_p),
        ("k", ctypes.c_void_p),
        ("v", ctypes.c_void_p),
        ("o", ctypes.c_void_p),
        ("lse", ctypes.c_void_p),
        ("B", ctypes.c_int),
        ("Nq", ctypes.c_int),
        ("Nk", ctypes.c_int),
        ("Hq", ctypes.c_int),
        ("Hkv", ctypes.c_int),
        ("d", ctypes.c_int),
        ("q_strides", ctypes.c_int64 * 3),
        ("k_strides", ctypes.c_int64 * 3),
        ("v_strides", ctypes.c_int64 * 3),
        ("o_strides", ctypes.c_int64 * 3),
        ("scale", ctypes.c_float),
        ("causal", ctypes.c_int),
        ("dtype", ctypes.c_int),
        ("mod", ScoreMod),
    ]


class BwdParams(ctypes.Structure):
    """Mirror of fa_bwd_params."""

    _fields_ = [
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("o", ctypes.c_void_p), ("dout", ctypes.c_void_p), ("lse", ctypes.c_void_p),
        ("dq", ctypes.c_void_p), ("dk", ctypes.c_void_p), ("dv", ctypes.c_void_p),
        ("B", ctypes.c_int), ("Nq", ctypes.c_int), ("Nk", ctypes.c_int), ("Hq", ctypes.c_int),
        ("Hkv", ctypes.c_int), ("d", ctypes.c_int),
        ("q_strides", ctypes.c_int64 * 3), ("k_strides", ctypes.c_int64 * 3),
        ("v_strides", ctypes.c_int64 * 3), ("o_strides", ctypes.c_int64 * 3),
        ("do_strides", ctypes.c_int64 * 3), ("dq_strides", ctypes.c_int64 * 3),
        ("dk_strides", ctypes.c_int64 * 3), ("dv_strides", ctypes.c_int64 * 3),
        ("scale", ctypes.c_float), ("causal", ctypes.c_int), ("dtype", ctypes.c_int),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("deterministic", ctypes.c_int),
        ("mod", ScoreMod),
    ]


_lib = None
_lock = threading.Lock()


def load_library(path: str | None = None):
    """Load libfa.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"{p} not found: build it with `python -m exact_attention_81_gb300.build`")
        lib = ctypes.CDLL(p)
        vp, i, i64, f, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                             ctypes.c_size_t)
        lib.fa_fwd.argtypes = [ctypes.POINTER(FwdParams), vp]
        lib.fa_fwd.restype = i
        pmod = ctypes.POINTER(ScoreMod)
        lib.fa_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, i,
                                      i, pmod, vp]
        lib.fa_fwd_varlen.restype = i
        lib.fa_fwd_kvcache_workspace_size.argtypes = [i, i, i, i, i]
        lib.fa_fwd_kvcache_workspace_size.restype = sz
        lib.fa_fwd_kvcache.argtypes = [vp, vp, vp, vp, i, i, i, i, i, ctypes.POINTER(i64), f, i,
                                       vp, sz, vp, vp, i, pmod, ctypes.POINTER(KvCacheExtras),
                                       vp]
        lib.fa_fwd_kvcache.restype = i
        lib.fa_fwd_kvcache_fp8.argtypes = [vp, vp, vp, vp, i, i, i, i, i, ctypes.POINTER(i64), f,
                                           i, vp, vp, vp, sz, vp, vp, pmod,
                                           ctypes.POINTER(KvCacheExtras), vp]
        lib.fa_fwd_kvcache_fp8.restype = i
        lib.fa_get_last_device_error.argtypes = [vp]
        lib.fa_get_last_device_error.restype = i
        lib.fa_status_string.argtypes = [i]
        lib.fa_status_string.restype = ctypes.c_char_p
        lib.fa_last_cuda_error.argtypes = []
        lib.fa_last_cuda_error.restype = ctypes.c_char_p
        lib.fa_set_wait_timeout_ns.argtypes = [ctypes.c_ulonglong]
        lib.fa_set_wait_timeout_ns.restype = None
        lib.fa_set_fault_injection.argtypes = [ctypes.c_int]
        lib.fa_set_fault_injection.restype = None
        lib.fa_set_cta_pairs.argtypes = [ctypes.c_int]
        lib.fa_set_cta_pairs.restype = None
        lib.fa_fwd_host.argtypes = [ctypes.POINTER(FwdParams), vp, vp, vp, vp, vp, i, vp]
        lib.fa_fwd_host.restype = i
        lib.fa_fwd_fp8_workspace_size.argtypes = [i, i, i, i]
        lib.fa_fwd_fp8_workspace_size.restype = sz
        lib.fa_fwd_fp8.argtypes = [ctypes.POINTER(FwdParams), vp, vp, vp, vp, sz, vp]
        lib.fa_fwd_fp8.restype = i
        lib.fa_fwd_varlen_fp8_workspace_size.argtypes = [i, i, i, i]
        lib.fa_fwd_varlen_fp8_workspace_size.restype = sz
        lib.fa_fwd_varlen_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f,
                                          i, pmod, vp, vp, vp, vp, sz, vp]
        lib.fa_fwd_varlen_fp8.restype = i
        lib.fa_fwd_params_size.argtypes = []
        lib.fa_fwd_params_size.restype = sz
        lib.fa_bwd.argtypes = [ctypes.POINTER(BwdParams), vp]
        lib.fa_bwd.restype = i
        lib.fa_bwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i,
                                      i, i, i, f, i, i, vp, sz, i, pmod, vp]
        lib.fa_bwd_varlen.restype = i
        lib.fa_bwd_workspace_size.argtypes = [i, i, i, i]
        lib.fa_bwd_workspace_size.restype = sz
        lib.fa_bwd_params_size.argtypes = []
        lib.fa_bwd_params_size.restype = sz
        if lib.fa_fwd_params_size() != ctypes.sizeof(FwdParams):
            raise RuntimeError("fa_fwd_params layout mismatch between libfa.so and the binding")
        if lib.fa_bwd_params_size() != ctypes.sizeof(BwdParams):
            raise RuntimeError("fa_bwd_params layout mismatch between libfa.so and the binding")
        if path is None:
            _lib = lib
        return lib


def status_string(status: int) -> str:
    return load_library().fa_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != FA_OK:
        detail = load_library().fa_last_cuda_error().decode() if status == FA_ERR_CUDA else ""
        raise FAError(status, where, detail)


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t) -> int | None:
    return None if t is None else int(t.data_ptr())


def _require_bf16_cuda(name, t, ndim, dtype=None):
    """A bf16 or fp16 CUDA tensor of `ndim` dimensions (of `dtype` when given)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype not in _DTYPE or not t.is_cuda:
        raise TypeError(f"{name} must be a bf16 or fp16 CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must have the element type of q ({dtype})")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions")
    if t.numel() > 0 and t.stride(-1) != 1:
        raise ValueError(f"{name} must have unit stride in the head dimension")


def default_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)


def _score_mod(B, Hq, device, window_size=None, softcap=0.0, alibi_slopes=None) -> ScoreMod:
    """fa_score_mod from the Python arguments.  window_size = (left, right), negative =
    unbounded; alibi_slopes an fp32 CUDA tensor [Hq] or [B, Hq] (kept alive by the caller)."""
    m = ScoreMod()
    if window_size is not None:
        wl, wr = (int(x) for x in window_size)
        if wl >= 0 or wr >= 0:
            m.use_window, m.window_left, m.window_right = 1, wl, wr
    m.softcap = float(softcap or 0.0)
    if alibi_slopes is not None:
        a = alibi_slopes
        if not isinstance(a, torch.Tensor) or a.dtype != torch.float32 or not a.is_cuda:
            raise TypeError("alibi_slopes must be an fp32 CUDA tensor")
        if a.device != device:
            raise ValueError("alibi_slopes must be on the device of q")
        if a.dim() == 1 and a.shape[0] == Hq and a.is_contiguous():
            m.alibi_batch_stride = 0
        elif a.dim() == 2 and tuple(a.shape) == (B, Hq) and a.stride(1) == 1:
            m.alibi_batch_stride = a.stride(0)
        else:
            raise ValueError("alibi_slopes must be [Hq] or [B, Hq] with unit stride over heads")
        m.alibi_slopes = a.data_ptr()
    return m


def fa_fwd(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
           stream=None, window_size=None, softcap: float = 0.0, alibi_slopes=None):
    """Dense attention.  q [B,Nq,Hq,d], k/v [B,Nk,Hkv,d] (bf16 or fp16, CUDA).

    window_size (left, right), softcap and alibi_slopes are the score modifiers of
    fa_score_mod.  Returns (out [B,Nq,Hq,d], lse [B,Hq,Nq] fp32).
    """
    _require_bf16_cuda("q", q, 4)
    _require_bf16_cuda("k", k, 4, q.dtype)
    _require_bf16_cuda("v", v, 4, q.dtype)
    B, Nq, Hq, d = q.shape
    Nk, Hkv = k.shape[1], k.shape[2]
    if tuple(k.shape) != (B, Nk, Hkv, d) or tuple(v.shape) != (B, Nk, Hkv, d):
        raise ValueError("k and v must be [B, Nk, Hkv, d] matching q")
    if out is None:
        out = torch.empty((B, Nq, Hq, d), dtype=q.dtype, device=q.device)
    else:
        _require_bf16_cuda("out", out, 4, q.dtype)
        if tuple(out.shape) != (B, Nq, Hq, d):
            raise ValueError("out must be [B, Nq, Hq, d]")
    if lse is None:
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device)
    elif lse.dtype != torch.float32 or tuple(lse.shape) != (B, Hq, Nq) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [B, Hq, Nq] tensor")
    p = FwdParams()
    p.q, p.k, p.v, p.o, p.lse = _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse)
    p.B, p.Nq, p.Nk, p.Hq, p.Hkv, p.d = B, Nq, Nk, Hq, Hkv, d
    for name, t in (("q_strides", q), ("k_strides", k), ("v_strides", v), ("o_strides", out)):
        getattr(p, name)[:] = list(t.stride()[:3])
    p.scale = default_scale(d) if scale is None else float(scale)
    p.causal = int(bool(causal))
    p.dtype = _DTYPE[q.dtype]
    p.mod = _score_mod(B, Hq, q.device, window_size, softcap, alibi_slopes)
    _check(load_library().fa_fwd(ctypes.byref(p), _stream_handle(stream)), "fa_fwd")
    return out, lse


def fa_fwd_host(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
                device_buffers=None, chunks: int = 8, stream=None, window_size=None,
                softcap: float = 0.0, alibi_slopes=None, device=None):
    """fa_fwd on host tensors: q [B,Nq,Hq,d], k/v [B,Nk,Hkv,d] contiguous, pinned CPU bf16 /
    fp16.  Copies in, computes and copies O and LSE out with the copies overlapping the
    computation (see fa_fwd_host in fa.h).  device_buffers: (q, k, v, o, lse) CUDA tensors
    of the same shapes (allocated if None).  Returns (out, lse) pinned CPU tensors; they hold
    the results once `stream` (default: the current stream) has reached the call."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype not in _DTYPE or t.is_cuda or t.dim() != 4 or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous 4-D bf16 / fp16 CPU tensor")
    dev = torch.device("cuda") if device is None else torch.device(device)
    if dev.index is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    B, Nq, Hq, d = q.shape
    Nk, Hkv = k.shape[1], k.shape[2]
    if tuple(k.shape) != (B, Nk, Hkv, d) or tuple(v.shape) != (B, Nk, Hkv, d):
        raise ValueError("k and v must be [B, Nk, Hkv, d] matching q")
    if out is None:
        out = torch.empty((B, Nq, Hq, d), dtype=q.dtype, pin_memory=True)
    if lse is None:
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, pin_memory=True)
    if device_buffers is None:
        device_buffers = (torch.empty(q.shape, dtype=q.dtype, device=dev),
                          torch.empty(k.shape, dtype=q.dtype, device=dev),
                          torch.empty(v.shape, dtype=q.dtype, device=dev),
                          torch.empty(out.shape, dtype=q.dtype, device=dev),
                          torch.empty(lse.shape, dtype=torch.float32, device=dev))
    p = FwdParams()
    p.q, p.k, p.v, p.o, p.lse = _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse)
    p.B, p.Nq, p.Nk, p.Hq, p.Hkv, p.d = B, Nq, Nk, Hq, Hkv, d
    for name, t in (("q_strides", q), ("k_strides", k), ("v_strides", v), ("o_strides", out)):
        getattr(p, name)[:] = list(t.stride()[:3])
    p.scale = default_scale(d) if scale is None else float(scale)
    p.causal = int(bool(causal))
    p.dtype = _DTYPE[q.dtype]
    p.mod = _score_mod(B, Hq, dev, window_size, softcap, alibi_slopes)
    st = load_library().fa_fwd_host(ctypes.byref(p), *[_ptr(t) for t in device_buffers],
                                    int(chunks), _stream_handle(stream))
    _check(st, "fa_fwd_host")
    return out, lse


def fa_fwd_fp8_workspace_size(B: int, Nk: int, Hkv: int, d: int) -> int:
    return int(load_library().fa_fwd_fp8_workspace_size(B, Nk, Hkv, d))


def fa_fwd_fp8(q, k, v, causal: bool = False, scale: float | None = None, q_descale=None,
               k_descale=None, v_descale=None, out=None, lse=None, workspace=None, stream=None,
               window_size=None, softcap: float = 0.0, alibi_slopes=None):
    """FP8 dense attention.  q [B,Nq,Hq,d], k/v [B,Nk,Hkv,d] torch.float8_e4m3fn (CUDA),
    d a multiple of 16 up to 128; q/k/v_descale fp32 [B, Hkv] CUDA tensors or None (= 1).
    Returns (out [B,Nq,Hq,d] bf16, lse [B,Hq,Nq] fp32)."""
    f8 = torch.float8_e4m3fn
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != f8 or not t.is_cuda or t.dim() != 4:
            raise TypeError(f"{name} must be a 4-D torch.float8_e4m3fn CUDA tensor")
        if t.stride(3) != 1:
            raise ValueError(f"{name} must have a unit-stride head dimension")
    B, Nq, Hq, d = q.shape
    Nk, Hkv = k.shape[1], k.shape[2]
    if tuple(k.shape) != (B, Nk, Hkv, d) or tuple(v.shape) != (B, Nk, Hkv, d):
        raise ValueError("k and v must be [B, Nk, Hkv, d] matching q")
    keep = []
    ptrs = []
    for name, t in (("q_descale", q_descale), ("k_descale", k_descale), ("v_descale", v_descale)):
        if t is None:
            ptrs.append(None)
            continue
        if t.dtype != torch.float32 or not t.is_cuda or t.numel() != B * Hkv:
            raise TypeError(f"{name} must be an fp32 CUDA tensor of B * Hkv elements")
        t = t.contiguous()
        keep.append(t)
        ptrs.append(_ptr(t))
    if out is None:
        out = torch.empty((B, Nq, Hq, d), dtype=torch.bfloat16, device=q.device)
    elif out.dtype != torch.bfloat16 or tuple(out.shape) != (B, Nq, Hq, d) or out.stride(3) != 1:
        raise ValueError("out must be a bf16 [B, Nq, Hq, d] tensor with unit-stride d")
    if lse is None:
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device)
    elif lse.dtype != torch.float32 or tuple(lse.shape) != (B, Hq, Nq) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [B, Hq, Nq] tensor")
    need = fa_fwd_fp8_workspace_size(B, Nk, Hkv, d)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    p = FwdParams()
    p.q, p.k, p.v, p.o, p.lse = _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse)
    p.B, p.Nq, p.Nk, p.Hq, p.Hkv, p.d = B, Nq, Nk, Hq, Hkv, d
    for name, t in (("q_strides", q), ("k_strides", k), ("v_strides", v), ("o_strides", out)):
        getattr(p, name)[:] = list(t.stride()[:3])
    p.scale = default_scale(d) if scale is None else float(scale)
    p.causal = int(bool(causal))
    p.dtype = FA_E4M3
    p.mod = _score_mod(B, Hq, q.device, window_size, softcap, alibi_slopes)
    st = load_library().fa_fwd_fp8(ctypes.byref(p), *ptrs, _ptr(workspace), workspace.numel(),
                                   _stream_handle(stream))
    _check(st, "fa_fwd_fp8")
    return out, lse


def fa_fwd_varlen_fp8_workspace_size(B: int, total_k: int, Hkv: int, d: int) -> int:
    return int(load_library().fa_fwd_varlen_fp8_workspace_size(B, total_k, Hkv, d))


def fa_fwd_varlen_fp8(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int,
                      max_seqlen_k: int, causal: bool = False, scale: float | None = None,
                      q_descale=None, k_descale=None, v_descale=None, out=None, lse=None,
                      workspace=None, stream=None, window_size=None, softcap: float = 0.0,
                      alibi_slopes=None):
    """FP8 attention over packed sequences.  q [total_q,Hq,d], k/v [total_k,Hkv,d]
    torch.float8_e4m3fn (CUDA, contiguous), cu_seqlens int32 [B+1], d a multiple of 16 up
    to 128; q/k/v_descale fp32 [B, Hkv] CUDA tensors or None (= 1).
    Returns (out [total_q,Hq,d] bf16, lse [Hq,total_q] fp32)."""
    f8 = torch.float8_e4m3fn
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != f8 or not t.is_cuda or t.dim() != 3 or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous 3-D torch.float8_e4m3fn CUDA tensor")
    for name, t in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k)):
        if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous int32 CUDA tensor")
    total_q, Hq, d = q.shape
    total_k, Hkv = k.shape[0], k.shape[1]
    if tuple(k.shape) != (total_k, Hkv, d) or tuple(v.shape) != (total_k, Hkv, d):
        raise ValueError("k and v must be [total_k, Hkv, d] matching q")
    B = cu_seqlens_q.numel() - 1
    if cu_seqlens_k.numel() != B + 1:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must have the same length")
    keep = []
    ptrs = []
    for name, t in (("q_descale", q_descale), ("k_descale", k_descale), ("v_descale", v_descale)):
        if t is None:
            ptrs.append(None)
            continue
        if t.dtype != torch.float32 or not t.is_cuda or t.numel() != B * Hkv:
            raise TypeError(f"{name} must be an fp32 CUDA tensor of B * Hkv elements")
        t = t.contiguous()
        keep.append(t)
        ptrs.append(_ptr(t))
    if out is None:
        out = torch.empty((total_q, Hq, d), dtype=torch.bfloat16, device=q.device)
    elif out.dtype != torch.bfloat16 or tuple(out.shape) != (total_q, Hq, d) or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 [total_q, Hq, d] tensor")
    if lse is None:
        lse = torch.empty((Hq, total_q), dtype=torch.float32, device=q.device)
    elif lse.dtype != torch.float32 or tuple(lse.shape) != (Hq, total_q) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [Hq, total_q] tensor")
    need = fa_fwd_varlen_fp8_workspace_size(B, total_k, Hkv, d)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    sc = default_scale(d) if scale is None else float(scale)
    mod = _score_mod(B, Hq, q.device, window_size, softcap, alibi_slopes)
    st = load_library().fa_fwd_varlen_fp8(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
        B, int(max_seqlen_q), int(max_seqlen_k), total_q, total_k, Hq, Hkv, d, sc,
        int(bool(causal)), ctypes.byref(mod), *ptrs, _ptr(workspace), workspace.numel(),
        _stream_handle(stream))
    _check(st, "fa_fwd_varlen_fp8")
    return out, lse


def fa_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, max_seqlen_k: int,
                  causal: bool = False, scale: float | None = None, out=None, lse=None,
                  stream=None, window_size=None, softcap: float = 0.0, alibi_slopes=None):
    """Packed varlen attention.  q [total_q,Hq,d], k/v [total_k,Hkv,d], cu_seqlens int32 [B+1].

    Returns (out [total_q,Hq,d] bf16, lse [Hq,total_q] fp32).
    """
    _require_bf16_cuda("q", q, 3)
    _require_bf16_cuda("k", k, 3, q.dtype)
    _require_bf16_cuda("v", v, 3, q.dtype)
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous for the varlen call")
    for name, t in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k)):
        if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous int32 CUDA tensor")
    total_q, Hq, d = q.shape
    total_k, Hkv = k.shape[0], k.shape[1]
    B = cu_seqlens_q.numel() - 1
    if cu_seqlens_k.numel() != B + 1:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must have the same length")
    if out is None:
        out = torch.empty((total_q, Hq, d), dtype=q.dtype, device=q.device)
    else:
        _require_bf16_cuda("out", out, 3, q.dtype)
    if lse is None:
        lse = torch.empty((Hq, total_q), dtype=torch.float32, device=q.device)
    sc = default_scale(d) if scale is None else float(scale)
    mod = _score_mod(B, Hq, q.device, window_size, softcap, alibi_slopes)
    st = load_library().fa_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                                      _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), B,
                                      int(max_seqlen_q), int(max_seqlen_k), total_q, total_k, Hq,
                                      Hkv, d, sc, int(bool(causal)), _DTYPE[q.dtype],
                                      ctypes.byref(mod), _stream_handle(stream))
    _check(st, "fa_fwd_varlen")
    return out, lse


def fa_fwd_kvcache_workspace_size(B: int, Hq: int, Lmax: int, d: int, num_splits: int = 0) -> int:
    return int(load_library().fa_fwd_kvcache_workspace_size(B, Hq, Lmax, d, num_splits))


def _kv_extras(q, k_cache, B, Hkv, d, k_new, v_new, rotary_cos, rotary_sin,
               rotary_interleaved, block_table):
    """fa_kvcache_extras from the Python arguments, or None when none is used."""
    if k_new is None and v_new is None and rotary_cos is None and block_table is None:
        return None
    ex = KvCacheExtras()
    if (k_new is None) != (v_new is None):
        raise ValueError("k_new and v_new go together")
    if k_new is not None:
        for name, t in (("k_new", k_new), ("v_new", v_new)):
            _require_bf16_cuda(name, t, 4, q.dtype)
            if tuple(t.shape) != (B, 1, Hkv, d):
                raise ValueError(f"{name} must be [B, 1, Hkv, d]")
        if k_new.stride() != v_new.stride():
            raise ValueError("k_new and v_new must share strides")
        ex.k_new, ex.v_new = k_new.data_ptr(), v_new.data_ptr()
        ex.new_strides[:] = list(k_new.stride()[:3])
    if (rotary_cos is None) != (rotary_sin is None):
        raise ValueError("rotary_cos and rotary_sin go together")
    if rotary_cos is not None:
        for name, t in (("rotary_cos", rotary_cos), ("rotary_sin", rotary_sin)):
            if t.dtype != torch.float32 or not t.is_cuda or t.dim() != 2 or not t.is_contiguous():
                raise TypeError(f"{name} must be a contiguous fp32 CUDA tensor [P, rotary_dim/2]")
        if rotary_cos.shape != rotary_sin.shape:
            raise ValueError("rotary_cos and rotary_sin must have the same shape")
        ex.rotary_cos, ex.rotary_sin = rotary_cos.data_ptr(), rotary_sin.data_ptr()
        ex.rotary_positions, ex.rotary_dim = rotary_cos.shape[0], 2 * rotary_cos.shape[1]
        ex.rotary_interleaved = int(bool(rotary_interleaved))
    if block_table is not None:
        if block_table.dtype != torch.int32 or not block_table.is_cuda or block_table.dim() != 2 \
                or block_table.stride(1) != 1 or block_table.shape[0] != B:
            raise TypeError("block_table must be an int32 CUDA tensor [B, blocks_per_seq]")
        ex.block_table = block_table.data_ptr()
        ex.block_table_stride = block_table.stride(0)
        ex.page_size = k_cache.shape[1]
        ex.num_pages = k_cache.shape[0]
    return ex


def fa_fwd_kvcache(q, k_cache, v_cache, cache_seqlens, scale: float | None = None,
                   num_splits: int = 0, workspace=None, out=None, lse=None, stream=None,
                   window_size=None, softcap: float = 0.0, alibi_slopes=None, k_new=None,
                   v_new=None, rotary_cos=None, rotary_sin=None, rotary_interleaved=False,
                   block_table=None):
    """Single-query decode.  q [B,1,Hq,d], caches [B,Lmax,Hkv,d] (paged: [num_pages,
    page_size, Hkv, d] with block_table int32 [B, blocks_per_seq]), cache_seqlens int32 [B].

    k_new / v_new [B,1,Hkv,d] are appended in place at row cache_seqlens[b] first (the
    caches are modified); rotary_cos / rotary_sin fp32 [P, rotary_dim/2] turn the query and
    the new key at that position.  Returns (out [B,1,Hq,d], lse [B,Hq] fp32).
    """
    _require_bf16_cuda("q", q, 4)
    _require_bf16_cuda("k_cache", k_cache, 4, q.dtype)
    _require_bf16_cuda("v_cache", v_cache, 4, q.dtype)
    if k_cache.stride() != v_cache.stride() or k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache must share shape and strides")
    if cache_seqlens.dtype != torch.int32 or not cache_seqlens.is_cuda:
        raise TypeError("cache_seqlens must be an int32 CUDA tensor")
    if not q.is_contiguous():
        raise ValueError("q must be contiguous")
    B, _, Hq, d = q.shape
    Hkv = k_cache.shape[2]
    Lmax = k_cache.shape[1] if block_table is None else block_table.shape[1] * k_cache.shape[1]
    ex = _kv_extras(q, k_cache, B, Hkv, d, k_new, v_new, rotary_cos, rotary_sin,
                    rotary_interleaved, block_table)
    if out is None:
        out = torch.empty((B, 1, Hq, d), dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    need = fa_fwd_kvcache_workspace_size(B, Hq, Lmax, d, num_splits)
    if workspace is None:
        workspace = torch.empty((max(need, 256),), dtype=torch.uint8, device=q.device)
    strides = (ctypes.c_int64 * 3)(*k_cache.stride()[:3])
    sc = default_scale(d) if scale is None else float(scale)
    mod = _score_mod(B, Hq, q.device, window_size, softcap, alibi_slopes)
    st = load_library().fa_fwd_kvcache(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(cache_seqlens),
                                       B, Lmax, Hq, Hkv, d, strides, sc, int(num_splits),
                                       _ptr(workspace), workspace.numel(), _ptr(out), _ptr(lse),
                                       _DTYPE[q.dtype], ctypes.byref(mod),
                                       None if ex is None else ctypes.byref(ex),
                                       _stream_handle(stream))
    _check(st, "fa_fwd_kvcache")
    return out, lse


def fa_fwd_kvcache_fp8(q, k_cache, v_cache, cache_seqlens, k_descale=None, v_descale=None,
                       scale: float | None = None, num_splits: int = 0, workspace=None,
                       out=None, lse=None, stream=None, window_size=None, softcap: float = 0.0,
                       alibi_slopes=None, block_table=None):
    """Single-query decode over an E4M3 KV cache.  q [B,1,Hq,d] bf16; caches [B,Lmax,Hkv,d]
    torch.float8_e4m3fn (paged: [num_pages, page_size, Hkv, d] with block_table);
    k_descale / v_descale fp32 [B, Hkv] CUDA tensors or None (= 1).  d a multiple of 16 up
    to 256.  Returns (out [B,1,Hq,d] bf16, lse [B,Hq] fp32)."""
    _require_bf16_cuda("q", q, 4)
    if q.dtype != torch.bfloat16:
        raise TypeError("q must be bf16 for an E4M3 cache")
    for name, t in (("k_cache", k_cache), ("v_cache", v_cache)):
        if t.dtype != torch.float8_e4m3fn or not t.is_cuda or t.dim() != 4:
            raise TypeError(f"{name} must be a 4-D torch.float8_e4m3fn CUDA tensor")
    if k_cache.stride() != v_cache.stride() or k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache must share shape and strides")
    if cache_seqlens.dtype != torch.int32 or not cache_seqlens.is_cuda:
        raise TypeError("cache_seqlens must be an int32 CUDA tensor")
    if not q.is_contiguous():
        raise ValueError("q must be contiguous")
    B, _, Hq, d = q.shape
    Hkv = k_cache.shape[2]
    Lmax = k_cache.shape[1] if block_table is None else block_table.shape[1] * k_cache.shape[1]
    ex = _kv_extras(q, k_cache, B, Hkv, d, None, None, None, None, False, block_table)
    keep, ptrs = [], []
    for name, t in (("k_descale", k_descale), ("v_descale", v_descale)):
        if t is None:
            ptrs.append(None)
            continue
        if t.dtype != torch.float32 or not t.is_cuda or t.numel() != B * Hkv:
            raise TypeError(f"{name} must be an fp32 CUDA tensor of B * Hkv elements")
        t = t.contiguous()
        keep.append(t)
        ptrs.append(_ptr(t))
    if out is None:
        out = torch.empty((B, 1, Hq, d), dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    need = fa_fwd_kvcache_workspace_size(B, Hq, Lmax, d, num_splits)
    if workspace is None:
        workspace = torch.empty((max(need, 256),), dtype=torch.uint8, device=q.device)
    strides = (ctypes.c_int64 * 3)(*k_cache.stride()[:3])
    sc = default_scale(d) if scale is None else float(scale)
    mod = _score_mod(B, Hq, q.device, window_size, softcap, alibi_slopes)
    st = load_library().fa_fwd_kvcache_fp8(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(cache_seqlens), B, Lmax, Hq, Hkv, d,
        strides, sc, int(num_splits), ptrs[0], ptrs[1], _ptr(workspace), workspace.numel(),
        _ptr(out), _ptr(lse), ctypes.byref(mod), None if ex is None else ctypes.byref(ex),
        _stream_handle(stream))
    _check(st, "fa_fwd_kvcache_fp8")
    return out, lse


def fa_bwd_workspace_size(B: int, Nq: int, Hq: int, d: int) -> int:
    return int(load_library().fa_bwd_workspace_size(B, Nq, Hq, d))


def fa_bwd(q, k, v, out, lse, dout, causal: bool = False, scale: float | None = None,
           dq=None, dk=None, dv=None, workspace=None, stream=None, deterministic=False,
           window_size=None, softcap: float = 0.0, alibi_slopes=None):
    """Backward of fa_fwd: q/out/dout [B,Nq,Hq,d], k/v [B,Nk,Hkv,d] (bf16 or fp16, CUDA),
    lse [B,Hq,Nq] fp32 from the forward call.  deterministic fixes the order in which the
    key blocks add into dQ.  Returns (dq, dk, dv)."""
    _require_bf16_cuda("q", q, 4)
    for name, t in (("k", k), ("v", v), ("out", out), ("dout", dout)):
        _require_bf16_cuda(name, t, 4, q.dtype)
    B, Nq, Hq, d = q.shape
    Nk, Hkv = k.shape[1], k.shape[2]
    if tuple(k.shape) != (B, Nk, Hkv, d) or tuple(v.shape) != (B, Nk, Hkv, d):
        raise ValueError("k and v must be [B, Nk, Hkv, d] matching q")
    if tuple(out.shape) != tuple(q.shape) or tuple(dout.shape) != tuple(q.shape):
        raise ValueError("out and dout must have the shape of q")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, Hq, Nq) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [B, Hq, Nq] tensor")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for name, t, ref in (("dq", dq, q), ("dk", dk, k), ("dv", dv, v)):
        _require_bf16_cuda(name, t, 4, q.dtype)
        if t.shape != ref.shape:
            raise ValueError(f"{name} must have the shape of {name[1:]}")
    need = fa_bwd_workspace_size(B, Nq, Hq, d)
    if workspace is None:
        workspace = torch.empty((max(need, 256),), dtype=torch.uint8, device=q.device)
    p = BwdParams()
    p.q, p.k, p.v, p.o, p.dout = _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout)
    p.lse, p.dq, p.dk, p.dv = _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv)
    p.B, p.Nq, p.Nk, p.Hq, p.Hkv, p.d = B, Nq, Nk, Hq, Hkv, d
    for name, t in (("q_strides", q), ("k_strides", k), ("v_strides", v), ("o_strides", out),
                    ("do_strides", dout), ("dq_strides", dq), ("dk_strides", dk),
                    ("dv_strides", dv)):
        getattr(p, name)[:] = list(t.stride()[:3])
    p.scale = default_scale(d) if scale is None else float(scale)
    p.causal = int(bool(causal))
    p.dtype = _DTYPE[q.dtype]
    p.workspace, p.workspace_bytes = _ptr(workspace), workspace.numel()
    p.deterministic = int(bool(deterministic))
    p.mod = _score_mod(B, Hq, q.device, window_size, softcap, alibi_slopes)
    _check(load_library().fa_bwd(ctypes.byref(p), _stream_handle(stream)), "fa_bwd")
    return dq, dk, dv


def fa_bwd_varlen(q, k, v, out, lse, dout, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int,
                  max_seqlen_k: int, causal: bool = False, scale: float | None = None, dq=None,
                  dk=None, dv=None, workspace=None, stream=None, deterministic=False,
                  window_size=None, softcap: float = 0.0, alibi_slopes=None):
    """Backward of fa_fwd_varlen: q/out/dout [total_q,Hq,d], k/v [total_k,Hkv,d] contiguous,
    lse [Hq,total_q] fp32 from the forward call.  Returns (dq, dk, dv)."""
    _require_bf16_cuda("q", q, 3)
    for name, t in (("k", k), ("v", v), ("out", out), ("dout", dout)):
        _require_bf16_cuda(name, t, 3, q.dtype)
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out), ("dout", dout)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous for the varlen call")
    total_q, Hq, d = q.shape
    total_k, Hkv = k.shape[0], k.shape[1]
    B = cu_seqlens_q.numel() - 1
    if lse.dtype != torch.float32 or tuple(lse.shape) != (Hq, total_q) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [Hq, total_q] tensor")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = fa_bwd_workspace_size(B, int(max_seqlen_q), Hq, d)
    if workspace is None:
        workspace = torch.empty((max(need, 256),), dtype=torch.uint8, device=q.device)
    sc = default_scale(d) if scale is None else float(scale)
    mod = _score_mod(B, Hq, q.device, window_size, softcap, alibi_slopes)
    st = load_library().fa_bwd_varlen(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
        _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), B, int(max_seqlen_q), int(max_seqlen_k),
        total_q, total_k, Hq, Hkv, d, sc, int(bool(causal)), _DTYPE[q.dtype], _ptr(workspace),
        workspace.numel(), int(bool(deterministic)), ctypes.byref(mod), _stream_handle(stream))
    _check(st, "fa_bwd_varlen")
    return dq, dk, dv


def get_last_device_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error status."""
    return int(load_library().fa_get_last_device_error(_stream_handle(stream)))


def set_wait_timeout_ns(ns: int):
    """Limit on device-side waits for later launches (0 = default)."""
    load_library().fa_set_wait_timeout_ns(int(ns))


def set_fault_injection(withhold_loads: bool):
    """Testing aid: later kernels issue no loads, so their waits run into the limit."""
    load_library().fa_set_fault_injection(int(bool(withhold_loads)))


def set_cta_pairs(enable: bool):
    """Run the 16-bit forward at head dimensions 72..128 on CTA pairs, or on the single-CTA
    kernel (the default) (process-wide, for later calls)."""
    load_library().fa_set_cta_pairs(int(bool(enable)))


# Names of the upstream Python API ("flash-attention", section 1), mapped onto the C calls.
def flash_attn_func(q, k, v, dropout_p: float = 0.0, softmax_scale=None, causal=False,
                    window_size=(-1, -1), softcap=0.0, alibi_slopes=None, return_lse=False):
    if dropout_p != 0.0:
        raise NotImplementedError("dropout is not part of this forward path")
    o, lse = fa_fwd(q, k, v, causal=causal, scale=softmax_scale, window_size=window_size,
                    softcap=softcap, alibi_slopes=alibi_slopes)
    return (o, lse) if return_lse else o


def flash_attn_varlen_func(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k,
                           dropout_p: float = 0.0, softmax_scale=None, causal=False,
                           window_size=(-1, -1), softcap=0.0, alibi_slopes=None,
                           return_lse=False):
    if dropout_p != 0.0:
        raise NotImplementedError("dropout is not part of this forward path")
    o, lse = fa_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k,
                           causal=causal, scale=softmax_scale, window_size=window_size,
                           softcap=softcap, alibi_slopes=alibi_slopes)
    return (o, lse) if return_lse else o


def flash_attn_with_kvcache(q, k_cache, v_cache, k=None, v=None, rotary_cos=None,
                            rotary_sin=None, cache_seqlens=None, block_table=None,
                            softmax_scale=None, causal=True, window_size=(-1, -1), softcap=0.0,
                            rotary_interleaved=False, alibi_slopes=None, num_splits=0,
                            return_lse=False):
    # With one query per sequence, bottom-right causal alignment lets it see the whole
    # visible prefix, so `causal` does not change the result.
    o, lse = fa_fwd_kvcache(q, k_cache, v_cache, cache_seqlens, scale=softmax_scale,
                            num_splits=num_splits, window_size=window_size, softcap=softcap,
                            alibi_slopes=alibi_slopes, k_new=k, v_new=v, rotary_cos=rotary_cos,
                            rotary_sin=rotary_sin, rotary_interleaved=rotary_interleaved,
                            block_table=block_table)
    return (o, lse) if return_lse else o
