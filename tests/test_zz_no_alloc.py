"""fa_fwd_kvcache_noalloc: the split-KV decode entry point for callers that cannot allocate
device memory (it keeps its partials in a scratch array compiled into libfa.so instead of a
caller workspace).  Called here through the C ABI and checked against fa_fwd_kvcache, the
entry point that takes a workspace, on two calls in a row.  Kept in a file of its own that
pytest collects last."""
import ctypes
import math

import numpy as np
import pytest
import torch

from exact_attention_81_gb300 import (FA_ERR_WORKSPACE, FA_OK, fa_fwd_kvcache,
                                      fa_fwd_kvcache_workspace_size, get_last_device_error,
                                      load_library)
from exact_attention_81_gb300.inputs import kvcache_inputs
from tests.parity_util import LSE_TOL, O_MAX_TOL, O_MEAN_TOL

pytestmark = pytest.mark.gpu
DEV = "cuda"
SCRATCH_MAX = 64 << 20


def _noalloc_fn():
    lib = load_library()
    f = lib.fa_fwd_kvcache_noalloc
    vp, i = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [vp, vp, vp, vp, i, i, i, i, i, ctypes.POINTER(ctypes.c_int64), ctypes.c_float,
                  i, vp, vp, vp]
    f.restype = i
    return f


def _call_noalloc(f, q, kc, vc, lens, num_splits=0):
    B, _, Hq, d = q.shape
    Lmax, Hkv = kc.shape[1], kc.shape[2]
    o = torch.empty((B, 1, Hq, d), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=DEV)
    strides = (ctypes.c_int64 * 3)(*kc.stride()[:3])
    st = f(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), lens.data_ptr(), B, Lmax, Hq, Hkv, d,
           strides, float(np.float32(1 / math.sqrt(d))), num_splits, o.data_ptr(),
           lse.data_ptr(), torch.cuda.current_stream().cuda_stream)
    return st, o, lse


def _close(o, lse, o_ref, lse_ref):
    err = (o.float() - o_ref.float()).abs()
    assert err.max().item() <= O_MAX_TOL and err.mean().item() <= O_MEAN_TOL
    fin = torch.isfinite(lse_ref)
    assert torch.equal(torch.isfinite(lse), fin)
    assert (lse[fin] - lse_ref[fin]).abs().max().item() <= LSE_TOL


def test_noalloc_matches_workspace_entry_point_twice():
    f = _noalloc_fn()
    cases = [
        dict(lens=[4096, 1, 3000, 128, 129, 2047, 0, 4000], Hq=32, Hkv=8, d=128, seed=901),
        dict(lens=[17, 900, 4096, 2], Hq=16, Hkv=8, d=64, seed=902),
    ]
    for c in cases:  # two calls in a row; the second finds the first one's partials
        q, kc, vc, lens = kvcache_inputs(len(c["lens"]), 4096, c["Hq"], c["Hkv"], c["d"],
                                         seed=c["seed"], lengths=torch.tensor(c["lens"]),
                                         device=DEV)
        o_ref, lse_ref = fa_fwd_kvcache(q, kc, vc, lens)
        st, o, lse = _call_noalloc(f, q, kc, vc, lens)
        assert st == FA_OK
        assert get_last_device_error() == FA_OK
        _close(o, lse, o_ref, lse_ref)


def test_noalloc_rejects_calls_beyond_its_scratch():
    f = _noalloc_fn()
    B, Hq, Hkv, Lmax, d = 128, 64, 8, 32768, 128
    assert fa_fwd_kvcache_workspace_size(B, Hq, Lmax, d, 0) > SCRATCH_MAX
    strides = (ctypes.c_int64 * 3)(Lmax * Hkv * d, Hkv * d, d)
    dummy = 1 << 20  # never dereferenced: the size check comes first
    st = f(dummy, dummy, dummy, dummy, B, Lmax, Hq, Hkv, d, strides, 0.088, 0, dummy, dummy,
           None)
    assert st == FA_ERR_WORKSPACE
