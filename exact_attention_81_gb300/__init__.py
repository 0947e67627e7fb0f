"""Exact fused attention forward for GB300 (sm_103a).

O = softmax(scale * Q K^T) V and the per-row log-sum-exp, computed tile by tile with the
online-softmax recurrence in hand-written CUDA kernels (libfa.so, C ABI in include/fa.h).
This package is the thin Python binding: ``fa_fwd`` (dense, batched, GQA, causal),
``fa_fwd_varlen`` (packed sequences), ``fa_fwd_kvcache`` (single-query split-KV decode)
and ``fa_bwd`` (gradients of ``fa_fwd``), plus the upstream-style names
``flash_attn_func``, ``flash_attn_varlen_func`` and ``flash_attn_with_kvcache``.  Build the library with
``python -m exact_attention_81_gb300.build``.
"""
from ._binding import (  # noqa: F401
    FA_BF16,
    FA_E4M3,
    FA_FP16,
    FA_ERR_CUDA,
    FA_ERR_INVALID_ARG,
    FA_ERR_TIMEOUT,
    FA_ERR_CONCURRENT,
    FA_ERR_UNSUPPORTED,
    FA_ERR_WORKSPACE,
    FA_OK,
    FAError,
    fa_bwd,
    fa_bwd_varlen,
    fa_bwd_workspace_size,
    fa_fwd,
    fa_fwd_fp8,
    fa_fwd_fp8_workspace_size,
    fa_fwd_varlen_fp8,
    fa_fwd_varlen_fp8_workspace_size,
    fa_fwd_kvcache_fp8,
    fa_fwd_host,
    fa_fwd_kvcache,
    fa_fwd_kvcache_workspace_size,
    fa_fwd_varlen,
    flash_attn_func,
    flash_attn_varlen_func,
    flash_attn_with_kvcache,
    get_last_device_error,
    load_library,
    set_cta_pairs,
    set_fault_injection,
    set_wait_timeout_ns,
    status_string,
)
