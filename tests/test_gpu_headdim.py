"""GPU parity for head dimensions other than 64 and 128 (any multiple of 8 up to 128): the
kernels run at width 64 or 128 and the tensor maps give the columns past d as zeros, so
the scores are unchanged and only d columns are stored.  Dense, varlen, decode (with the
KV-cache extras) and backward against the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

import oracle.oracle as ORACLE
from exact_attention_81_gb300 import (FA_OK, fa_bwd, fa_fwd, fa_fwd_kvcache, fa_fwd_varlen,
                                      get_last_device_error)
from exact_attention_81_gb300.inputs import bf16_normal, dense_inputs, kvcache_inputs, varlen_inputs
from tests.parity_util import compare, dense_rows, varlen_rows
from tests.test_gpu_backward import _check as _check_bwd

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _scale(d):
    return float(np.float32(1 / math.sqrt(d)))


@pytest.mark.parametrize("d", [8, 32, 40, 72, 96, 112])
@pytest.mark.parametrize("causal", [False, True])
def test_dense_head_dims(d, causal):
    q, k, v = dense_inputs(2, 300, 333, 4, 2, d, seed=800 + d, device=DEV)
    o, lse = fa_fwd(q, k, v, causal=causal)
    assert get_last_device_error() == FA_OK
    assert o.shape[-1] == d
    o_ref, lse_ref = ORACLE.attention(q.cpu(), k.cpu(), v.cpu(), _scale(d), causal)
    compare(*dense_rows(o, lse), *dense_rows(o_ref, lse_ref), f"dense d={d} causal={causal}")


def test_dense_head_dim_strided_output_untouched_padding():
    """O is written only in its d columns: a wider buffer's other columns keep their
    contents (the padding of the kernel is never stored)."""
    d = 96
    q, k, v = dense_inputs(1, 200, 200, 2, 2, d, seed=810, device=DEV)
    big = torch.full((1, 200, 2, 128), 7.0, dtype=torch.bfloat16, device=DEV)
    out = big[..., :d]
    fa_fwd(q, k, v, causal=True, out=out)
    assert get_last_device_error() == FA_OK
    assert torch.all(big[..., d:] == 7.0)
    o_ref, lse_ref = ORACLE.attention(q.cpu(), k.cpu(), v.cpu(), _scale(d), True)
    lse = fa_fwd(q, k, v, causal=True)[1]
    compare(*dense_rows(out, lse), *dense_rows(o_ref, lse_ref), "strided d=96")


@pytest.mark.parametrize("d,mod", [(96, dict(softcap=20.0)), (40, dict(window_size=(50, 0))),
                                   (72, dict(window_size=(100, 3), softcap=5.0))])
def test_dense_head_dims_with_modifiers(d, mod):
    q, k, v = dense_inputs(1, 400, 400, 4, 4, d, seed=820 + d, device=DEV)
    o, lse = fa_fwd(q, k, v, **mod)
    assert get_last_device_error() == FA_OK
    o_ref, lse_ref = ORACLE.attention(q.cpu(), k.cpu(), v.cpu(), _scale(d), False,
                                      window=mod.get("window_size", (-1, -1)),
                                      softcap=mod.get("softcap", 0.0))
    compare(*dense_rows(o, lse), *dense_rows(o_ref, lse_ref), f"d={d} {mod}")


def test_dense_head_dim_fp16():
    d = 96
    q, k, v = dense_inputs(2, 256, 256, 4, 2, d, seed=830, device=DEV, dtype=torch.float16)
    o, lse = fa_fwd(q, k, v, causal=True)
    assert get_last_device_error() == FA_OK
    o_ref, lse_ref = ORACLE.attention(q.cpu(), k.cpu(), v.cpu(), _scale(d), True)
    compare(*dense_rows(o, lse), *dense_rows(o_ref, lse_ref), "fp16 d=96")


@pytest.mark.parametrize("d", [32, 96])
def test_varlen_head_dims(d):
    sq, sk = [5, 0, 333, 129], [7, 3, 333, 200]
    q, k, v, cu_q, cu_k = varlen_inputs(sq, sk, 4, 2, d, seed=840 + d, device=DEV)
    o, lse = fa_fwd_varlen(q, k, v, cu_q, cu_k, max(sq), max(sk), causal=True)
    assert get_last_device_error() == FA_OK
    o_ref, lse_ref = ORACLE.attention_varlen(q.cpu(), k.cpu(), v.cpu(), cu_q.cpu(), cu_k.cpu(),
                                             _scale(d), True)
    compare(*varlen_rows(o, lse), *varlen_rows(o_ref, lse_ref), f"varlen d={d}")


@pytest.mark.parametrize("d,group", [(32, 4), (96, 8), (96, 1), (48, 2)])
def test_decode_head_dims(d, group):
    lens = torch.tensor([1, 127, 1000, 2048, 0, 513], dtype=torch.int32)
    q, kc, vc, lens = kvcache_inputs(len(lens), 2048, 2 * group, 2, d, seed=850 + d + group,
                                     lengths=lens, device=DEV)
    o, lse = fa_fwd_kvcache(q, kc, vc, lens)
    assert get_last_device_error() == FA_OK
    assert o.shape[-1] == d
    o_ref, lse_ref = ORACLE.attention_kvcache(q.cpu(), kc.cpu(), vc.cpu(), lens.cpu(), _scale(d))
    compare(o[:, 0], lse, o_ref, lse_ref, f"decode d={d} G={group}")


def test_decode_head_dim_append_rotary():
    d, rd = 96, 64
    B, Lmax, Hq, Hkv = 4, 1024, 8, 2
    lens = torch.tensor([0, 5, 700, 1023], dtype=torch.int32, device=DEV)
    q = bf16_normal((B, 1, Hq, d), 860, DEV)
    kc = bf16_normal((B, Lmax, Hkv, d), 861, DEV)
    vc = bf16_normal((B, Lmax, Hkv, d), 862, DEV)
    kn = bf16_normal((B, 1, Hkv, d), 863, DEV)
    vn = bf16_normal((B, 1, Hkv, d), 864, DEV)
    ang = np.arange(1100)[:, None] * (10000.0 ** (-np.arange(rd // 2) / (rd // 2)))[None, :]
    cos, sin = (torch.from_numpy(f(ang).astype(np.float32)).to(DEV) for f in (np.cos, np.sin))
    kc0, vc0 = kc.clone(), vc.clone()
    o, lse = fa_fwd_kvcache(q, kc, vc, lens, k_new=kn, v_new=vn, rotary_cos=cos, rotary_sin=sin,
                            rotary_interleaved=True)
    assert get_last_device_error() == FA_OK
    o_ref, l_ref, k_ref, v_ref = ORACLE.kvcache_step(
        q.cpu(), kc0.cpu(), vc0.cpu(), lens.cpu().numpy(), _scale(d), k_new=kn.cpu(),
        v_new=vn.cpu(), rotary_cos=cos.cpu().numpy(), rotary_sin=sin.cpu().numpy(),
        rotary_interleaved=True)
    bits = lambda t: t.cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bits(kc), k_ref) and np.array_equal(bits(vc), v_ref)
    compare(o[:, 0], lse, o_ref, l_ref, "decode d=96 append + rotary 64")


@pytest.mark.parametrize("d,causal", [(32, True), (96, False), (96, True), (48, True)])
def test_backward_head_dims(d, causal):
    q, k, v = dense_inputs(1, 300, 300, 4, 2, d, seed=870 + d, device=DEV)
    do = bf16_normal((1, 300, 4, d), seed=871 + d, device=DEV)
    _check_bwd(q, k, v, do, _scale(d), causal, f"bwd d={d} causal={causal}")


# Head dimensions above 128 (forward only): the wide kernel, one 128-row sub-tile per work
# tile with S double-buffered in TMEM and K / V moved as d halves.

@pytest.mark.parametrize("d,causal", [(256, False), (256, True), (192, True), (136, False),
                                      (248, True)])
def test_dense_wide_head_dims(d, causal):
    q, k, v = dense_inputs(2, 333, 300, 4, 2, d, seed=880 + d, device=DEV)
    o, lse = fa_fwd(q, k, v, causal=causal)
    assert get_last_device_error() == FA_OK
    assert o.shape[-1] == d
    o_ref, lse_ref = ORACLE.attention(q.cpu(), k.cpu(), v.cpu(), _scale(d), causal)
    compare(*dense_rows(o, lse), *dense_rows(o_ref, lse_ref), f"wide d={d} causal={causal}")


def test_dense_wide_long_causal():
    """Many K/V steps per tile (both S buffers, the ring wrapping many times, rescales)."""
    d = 256
    q, k, v = dense_inputs(1, 1100, 1100, 2, 1, d, seed=890, device=DEV)
    o, lse = fa_fwd(q, k, v, causal=True)
    assert get_last_device_error() == FA_OK
    o_ref, lse_ref = ORACLE.attention(q.cpu(), k.cpu(), v.cpu(), _scale(d), True)
    compare(*dense_rows(o, lse), *dense_rows(o_ref, lse_ref), "wide d=256 N=1100 causal")


def test_dense_wide_fp16_gqa():
    d = 256
    q, k, v = dense_inputs(2, 256, 640, 8, 2, d, seed=891, device=DEV, dtype=torch.float16)
    o, lse = fa_fwd(q, k, v, causal=False)
    assert get_last_device_error() == FA_OK
    o_ref, lse_ref = ORACLE.attention(q.cpu(), k.cpu(), v.cpu(), _scale(d), False)
    compare(*dense_rows(o, lse), *dense_rows(o_ref, lse_ref), "wide fp16 GQA")


@pytest.mark.parametrize("mod", [dict(window_size=(100, 20)), dict(softcap=15.0),
                                 dict(window_size=(300, -1), softcap=8.0, alibi=True)])
def test_dense_wide_modifiers(mod):
    d, Hq = 256, 4
    mod = dict(mod)
    slopes = None
    if mod.pop("alibi", False):
        slopes = torch.tensor(2.0 ** (-8.0 * np.arange(1, Hq + 1) / Hq), dtype=torch.float32)
    q, k, v = dense_inputs(1, 500, 500, Hq, 2, d, seed=892, device=DEV)
    o, lse = fa_fwd(q, k, v, causal=True, alibi_slopes=None if slopes is None else
                    slopes.to(DEV), **mod)
    assert get_last_device_error() == FA_OK
    o_ref, lse_ref = ORACLE.attention(q.cpu(), k.cpu(), v.cpu(), _scale(d), True,
                                      window=mod.get("window_size", (-1, -1)),
                                      softcap=mod.get("softcap", 0.0), alibi_slopes=slopes)
    compare(*dense_rows(o, lse), *dense_rows(o_ref, lse_ref), f"wide {sorted(mod)}")


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_wide_head_dims(causal):
    d = 256
    sq, sk = [5, 0, 333, 129, 1], [7, 3, 333, 200, 0]
    q, k, v, cu_q, cu_k = varlen_inputs(sq, sk, 4, 2, d, seed=893, device=DEV)
    o, lse = fa_fwd_varlen(q, k, v, cu_q, cu_k, max(sq), max(sk), causal=causal)
    assert get_last_device_error() == FA_OK
    o_ref, lse_ref = ORACLE.attention_varlen(q.cpu(), k.cpu(), v.cpu(), cu_q.cpu(), cu_k.cpu(),
                                             _scale(d), causal)
    compare(*varlen_rows(o, lse), *varlen_rows(o_ref, lse_ref), f"varlen wide causal={causal}")


def test_head_dims_past_256_not_served_by_backward():
    """The backward serves d up to 256 (above 128 the wide kernel, tested in
    test_gpu_backward_wide.py); a larger d is refused before any launch."""
    from exact_attention_81_gb300 import FAError
    d = 264
    q, k, v = dense_inputs(1, 128, 128, 2, 2, d, seed=894, device=DEV)
    lse = torch.zeros((1, 2, 128), dtype=torch.float32, device=DEV)
    with pytest.raises(FAError):
        fa_bwd(q, k, v, torch.zeros_like(q), lse, torch.ones_like(q))


@pytest.mark.parametrize("d,group,dtype", [
    (256, 8, torch.bfloat16), (256, 4, torch.bfloat16), (256, 2, torch.float16),
    (192, 8, torch.bfloat16), (136, 1, torch.bfloat16), (248, 4, torch.float16)])
def test_decode_wide_head_dims(d, group, dtype):
    """Width-256 decode; a group of 8 runs as two work items of 4 heads on the same rows."""
    lens = torch.tensor([1, 127, 128, 1000, 3071, 0, 513, 3072], dtype=torch.int32)
    q, kc, vc, lens = kvcache_inputs(len(lens), 3072, 2 * group, 2, d, seed=900 + d + group,
                                     lengths=lens, device=DEV, dtype=dtype)
    o, lse = fa_fwd_kvcache(q, kc, vc, lens)
    assert get_last_device_error() == FA_OK
    assert o.shape[-1] == d
    o_ref, lse_ref = ORACLE.attention_kvcache(q.cpu(), kc.cpu(), vc.cpu(), lens.cpu(), _scale(d))
    compare(o[:, 0], lse, o_ref, lse_ref, f"decode d={d} G={group} {dtype}")


@pytest.mark.parametrize("num_splits", [1, 3, 7])
def test_decode_wide_explicit_splits(num_splits):
    lens = torch.tensor([2000, 1, 129, 1024], dtype=torch.int32)
    q, kc, vc, lens = kvcache_inputs(len(lens), 2048, 16, 2, 256, seed=910 + num_splits,
                                     lengths=lens, device=DEV)
    o, lse = fa_fwd_kvcache(q, kc, vc, lens, num_splits=num_splits)
    assert get_last_device_error() == FA_OK
    o_ref, lse_ref = ORACLE.attention_kvcache(q.cpu(), kc.cpu(), vc.cpu(), lens.cpu(),
                                              _scale(256))
    compare(o[:, 0], lse, o_ref, lse_ref, f"decode d=256 splits={num_splits}")
