"""Helpers shared by the GPU parity tests: tolerances and comparisons.

The bar for every call (dense, varlen, decode) is the one the exact-attention forward
pass is held to: max|O - O_ref| <= 1e-2, mean|O - O_ref| <= 1e-3 and
max|LSE - LSE_ref| <= 1e-3, with O_ref and LSE_ref from the fp64 oracle on the same
bf16 inputs.  Rows that see no key must give O = 0 exactly and LSE = -inf.

By default the bounds apply to the raw differences.  A test may pass allowance=True when
its outputs are dominated by a few keys (steep ALiBi slopes, narrow windows, softcaps that
saturate): O is then close to one value row, and a 16-bit output cannot come closer to
O_ref than half an ulp of the output type (an exact O of 3 is already 0.0078 from its
nearest bf16).  With the allowance, half an ulp at max(|O|, |O_ref|) is taken off each
element's difference before the bounds apply.  The flash-attention page (section 5, tests)
judges an implementation against a PyTorch baseline that rounds its output the same way.

With FA_PARITY_LOG set to a file path, every comparison appends one JSON line with the
raw and the allowance-adjusted errors and the test it came from.
"""
from __future__ import annotations

import json
import os

import numpy as np
import torch

O_MAX_TOL = 1e-2
O_MEAN_TOL = 1e-3
LSE_TOL = 1e-3


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


# significand bits (with the implicit one) and smallest normal exponent
_FORMAT = {torch.bfloat16: (8, -126), torch.float16: (11, -14)}


def half_ulp(x: np.ndarray, dtype) -> np.ndarray:
    """Half the spacing of `dtype` (bf16 / fp16) around each |x| (subnormals: the fixed
    spacing at the smallest exponent); 0 for other types."""
    fmt = _FORMAT.get(dtype)
    ax = np.abs(np.asarray(x, np.float64))
    if fmt is None:
        return np.zeros_like(ax)
    bits, emin = fmt
    e = np.maximum(np.floor(np.log2(np.where(ax > 0, ax, 1.0))), emin)
    return np.exp2(e - bits)


def _log(rec):
    path = os.environ.get("FA_PARITY_LOG")
    if not path:
        return
    rec = dict(rec, test=os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0])
    with open(path, "a") as f:
        f.write(json.dumps(rec) + "\n")


def compare(o_gpu, lse_gpu, o_ref, lse_ref, what="", allowance=False):
    """o_* [..., d] and lse_* [...] with the same row order (o.shape[:-1] == lse.shape).

    Asserts the bounds on the raw differences, or on the differences beyond half an ulp
    of the output type when allowance=True.  Returns the errors it measured."""
    out_dtype = o_gpu.dtype if isinstance(o_gpu, torch.Tensor) else None
    o = to_np(o_gpu) if isinstance(o_gpu, torch.Tensor) else np.asarray(o_gpu, np.float64)
    lse = to_np(lse_gpu) if isinstance(lse_gpu, torch.Tensor) else np.asarray(lse_gpu, np.float64)
    o_ref = np.asarray(o_ref, np.float64)
    lse_ref = np.asarray(lse_ref, np.float64)
    assert o.shape == o_ref.shape, f"{what}: O shape {o.shape} vs {o_ref.shape}"
    assert lse.shape == lse_ref.shape, f"{what}: LSE shape {lse.shape} vs {lse_ref.shape}"
    assert o.shape[:-1] == lse.shape, f"{what}: O rows {o.shape[:-1]} vs LSE rows {lse.shape}"
    assert np.all(np.isfinite(o)), f"{what}: non-finite O"
    empty = ~np.isfinite(lse_ref)
    assert np.array_equal(~np.isfinite(lse), empty), f"{what}: -inf LSE rows differ"
    assert np.all(lse[empty] == -np.inf), f"{what}: empty rows must have LSE = -inf"
    if empty.any():
        assert np.all(o[empty] == 0.0), f"{what}: empty rows must have O = 0"
    raw = np.abs(o - o_ref)
    raw_max = float(raw.max(initial=0.0))
    raw_mean = float(raw.mean()) if raw.size else 0.0
    rep = np.maximum(half_ulp(o, out_dtype), half_ulp(o_ref, out_dtype))
    adj = np.maximum(raw - rep, 0.0)
    del rep
    adj_max = float(adj.max(initial=0.0))
    adj_mean = float(adj.mean()) if adj.size else 0.0
    del adj
    fin = ~empty
    max_l = float(np.abs(lse[fin] - lse_ref[fin]).max(initial=0.0))
    _log({"what": what, "allowance": bool(allowance), "elements": int(raw.size),
          "raw_max_abs_o": raw_max, "raw_mean_abs_o": raw_mean, "adj_max_abs_o": adj_max,
          "adj_mean_abs_o": adj_mean, "max_abs_lse": max_l})
    max_o, mean_o = (adj_max, adj_mean) if allowance else (raw_max, raw_mean)
    tag = " (beyond half an ulp)" if allowance else ""
    assert max_o <= O_MAX_TOL, f"{what}: max|dO|{tag} = {max_o:.3e} > {O_MAX_TOL}"
    assert mean_o <= O_MEAN_TOL, f"{what}: mean|dO|{tag} = {mean_o:.3e} > {O_MEAN_TOL}"
    assert max_l <= LSE_TOL, f"{what}: max|dLSE| = {max_l:.3e} > {LSE_TOL}"
    return {"max_abs_o": max_o, "mean_abs_o": mean_o, "max_abs_lse": max_l,
            "raw_max_abs_o": raw_max, "raw_mean_abs_o": raw_mean}


def sample_rows(B, H, N, n, seed, must=()):
    """(b, h, i) triples: tile edges of every (b, h) subset plus random rows."""
    rng = np.random.default_rng(seed)
    rows = set(tuple(r) for r in must)
    edges = [0, 1, 127, 128, 129, 255, 256, N // 2, N - 129, N - 128, N - 2, N - 1]
    for b in range(B):
        for h in range(H):
            for i in rng.choice(edges, size=2, replace=False):
                if 0 <= i < N:
                    rows.add((b, h, int(i)))
    while len(rows) < n + len(must):
        rows.add((int(rng.integers(B)), int(rng.integers(H)), int(rng.integers(N))))
    return np.array(sorted(rows), dtype=np.int32)


def dense_rows(o, lse):
    """Dense O [B,N,H,d] and LSE [B,H,N] -> row-aligned O [B,H,N,d] and LSE."""
    if isinstance(o, torch.Tensor):
        return o.permute(0, 2, 1, 3), lse
    return np.transpose(o, (0, 2, 1, 3)), lse


def varlen_rows(o, lse):
    """Varlen O [T,H,d] and LSE [H,T] -> row-aligned O [H,T,d] and LSE."""
    if isinstance(o, torch.Tensor):
        return o.permute(1, 0, 2), lse
    return np.transpose(o, (1, 0, 2)), lse
