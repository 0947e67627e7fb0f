"""fa_fwd_kvcache_noalloc: the split-KV decode entry point for callers that cannot allocate
device memory (it keeps its partials in a scratch array compiled into libfa.so instead of a
caller workspace).  Called here through the C ABI and checked bit for bit against
fa_fwd_kvcache, the entry point that takes a workspace (same kernels, same splits), on calls
in a row that reuse the scratch with different layouts, and against the fp64 oracle at head
dimensions 96 and 256.  Kept in a file of its own that pytest collects last."""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle.oracle as ORACLE
from exact_attention_81_gb300 import (FA_ERR_WORKSPACE, FA_OK, fa_fwd_kvcache,
                                      fa_fwd_kvcache_workspace_size, get_last_device_error,
                                      load_library)
from exact_attention_81_gb300.inputs import kvcache_inputs
from tests.parity_util import compare

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


CASES = {
    "wide": dict(lens=[4096, 1, 3000, 128, 129, 2047, 0, 4000], Lmax=4096, Hq=32, Hkv=8,
                 d=128, seed=901, splits=0),
    "small": dict(lens=[17, 900, 4096, 2], Lmax=4096, Hq=16, Hkv=8, d=64, seed=902, splits=0),
    "d96_splits3": dict(lens=[1000, 3, 2500, 513], Lmax=2560, Hq=8, Hkv=2, d=96, seed=903,
                        splits=3),
    "d256": dict(lens=[2048, 77, 1500], Lmax=2048, Hq=16, Hkv=2, d=256, seed=904, splits=0),
}


def _inputs(c):
    return kvcache_inputs(len(c["lens"]), c["Lmax"], c["Hq"], c["Hkv"], c["d"], seed=c["seed"],
                          lengths=torch.tensor(c["lens"]), device=DEV)


def test_noalloc_matches_workspace_entry_point_bit_for_bit():
    """Calls in a row on the one scratch array: a large layout, a small one, the large one
    again (it finds the small call's partials in the scratch), an explicit split count, and
    the width-256 instance.  Each output equals fa_fwd_kvcache's with the same num_splits."""
    f = _noalloc_fn()
    for name in ["wide", "small", "wide", "d96_splits3", "d256", "wide"]:
        c = CASES[name]
        q, kc, vc, lens = _inputs(c)
        o_ref, lse_ref = fa_fwd_kvcache(q, kc, vc, lens, num_splits=c["splits"])
        st, o, lse = _call_noalloc(f, q, kc, vc, lens, num_splits=c["splits"])
        assert st == FA_OK, name
        assert get_last_device_error() == FA_OK
        assert torch.equal(o, o_ref), name
        assert torch.equal(lse, lse_ref), name


@pytest.mark.parametrize("name", ["d96_splits3", "d256"])
def test_noalloc_matches_oracle(name):
    f = _noalloc_fn()
    c = CASES[name]
    q, kc, vc, lens = _inputs(c)
    st, o, lse = _call_noalloc(f, q, kc, vc, lens, num_splits=c["splits"])
    assert st == FA_OK
    assert get_last_device_error() == FA_OK
    o_ref, lse_ref = ORACLE.attention_kvcache(q.cpu(), kc.cpu(), vc.cpu(), lens.cpu(),
                                              float(np.float32(1 / math.sqrt(c["d"]))))
    compare(o[:, 0], lse, o_ref, lse_ref, f"noalloc {name}")


def test_noalloc_rejects_calls_beyond_its_scratch():
    f = _noalloc_fn()
    B, Hq, Hkv, Lmax, d = 128, 64, 8, 32768, 128
    assert fa_fwd_kvcache_workspace_size(B, Hq, Lmax, d, 0) > SCRATCH_MAX
    strides = (ctypes.c_int64 * 3)(Lmax * Hkv * d, Hkv * d, d)
    dummy = 1 << 20  # never dereferenced: the size check comes first
    st = f(dummy, dummy, dummy, dummy, B, Lmax, Hq, Hkv, d, strides, 0.088, 0, dummy, dummy,
           None)
    assert st == FA_ERR_WORKSPACE
