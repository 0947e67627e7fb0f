"""GPU parity of the score modifiers (sliding window, softcap, ALiBi) against the fp64
oracle: dense, varlen and decode calls, windows that straddle tile edges or hide every key
of a row, per-head and per-(batch, head) ALiBi slopes, all three modifiers at once."""
import math

import numpy as np
import pytest
import torch

import oracle.oracle as ORACLE
from exact_attention_81_gb300 import (FA_OK, fa_fwd, fa_fwd_kvcache, fa_fwd_varlen,
                                      get_last_device_error)
from exact_attention_81_gb300.inputs import (WORKLOADS, dense_inputs, kvcache_inputs,
                                             varlen_inputs)
from tests.parity_util import compare, dense_rows, sample_rows, varlen_rows

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _scale(d):
    return float(np.float32(1 / math.sqrt(d)))


def _slopes(Hq, B=None):
    """ALiBi-style geometric slopes 2^(-8 h / Hq); per batch entry shifted when B is given."""
    base = 2.0 ** (-8.0 * np.arange(1, Hq + 1) / Hq)
    if B is None:
        return torch.tensor(base, dtype=torch.float32)
    return torch.tensor(np.stack([base * (1.0 + 0.25 * b) for b in range(B)]),
                        dtype=torch.float32)


def _dense(B, Nq, Nk, Hq, Hkv, d, causal, seed, dtype=torch.bfloat16, scale=None,
           allowance=False, **mod):
    q, k, v = dense_inputs(B, Nq, Nk, Hq, Hkv, d, seed=seed, device=DEV, dtype=dtype)
    sc = _scale(d) if scale is None else scale
    what = f"dense B={B} Nq={Nq} Nk={Nk} causal={causal} {sorted(mod)}"
    slopes = mod.pop("alibi_slopes", None)
    o, lse = fa_fwd(q, k, v, causal=causal, scale=sc, alibi_slopes=None if slopes is None
                    else slopes.to(DEV), **mod)
    assert get_last_device_error() == FA_OK
    window = mod.get("window_size", (-1, -1))
    o_ref, lse_ref = ORACLE.attention(q.cpu(), k.cpu(), v.cpu(), sc, causal, window=window,
                                      softcap=mod.get("softcap", 0.0), alibi_slopes=slopes)
    return compare(*dense_rows(o, lse), *dense_rows(o_ref, lse_ref), what, allowance=allowance)


@pytest.mark.parametrize("window,causal", [
    ((100, 0), False), ((256, 256), False), ((0, 0), False), ((127, 129), False),
    ((-1, 300), False), ((1000, -1), False), ((300, -1), True), ((5, 7), True),
])
def test_window_dense(window, causal):
    _dense(2, 700, 700, 4, 2, 128, causal, seed=500 + window[0], window_size=window)


@pytest.mark.parametrize("Nq,Nk,window", [
    (300, 900, (200, 50)), (900, 300, (100, 10)), (129, 1000, (0, 0)), (1000, 129, (64, -1)),
])
def test_window_unequal_lengths(Nq, Nk, window):
    """Bottom-right alignment; with Nq > Nk the first rows' windows hold no key."""
    _dense(1, Nq, Nk, 2, 1, 64, False, seed=510 + Nq, window_size=window)


@pytest.mark.parametrize("softcap,causal,d,scale", [
    (30.0, True, 128, None), (5.0, False, 128, 0.5), (2.0, True, 64, None), (50.0, False, 64, 1.0),
])
def test_softcap_dense(softcap, causal, d, scale):
    _dense(2, 517, 517, 4, 2, d, causal, seed=520 + d, scale=scale, softcap=softcap)


@pytest.mark.parametrize("per_batch,causal,Nq,Nk,allowance", [
    (False, True, 640, 640, False), (True, False, 333, 777, False),
    (False, False, 777, 333, True), (True, True, 256, 1024, False),
])
def test_alibi_dense(per_batch, causal, Nq, Nk, allowance):
    """allowance: with Nq > Nk and no causal mask the rows past the keys sit far from every
    key, the steepest slopes leave nearly all of P on the nearest key, and O is within a
    few bf16 ulps of one value row (raw max |dO| 1.07e-2, 3.0e-3 beyond half an ulp)."""
    Hq, B = 8, 2
    slopes = _slopes(Hq, B if per_batch else None)
    _dense(B, Nq, Nk, Hq, 2, 128, causal, seed=530 + Nq, allowance=allowance,
           alibi_slopes=slopes)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_all_modifiers_dense(dtype):
    _dense(2, 600, 650, 8, 4, 128, True, seed=540, dtype=dtype, window_size=(200, -1),
           softcap=20.0, alibi_slopes=_slopes(8, 2))


def test_modifiers_varlen():
    sq = [5, 0, 333, 128, 129, 700]
    sk = [7, 3, 333, 400, 200, 700]
    Hq, Hkv, d = 4, 2, 128
    q, k, v, cu_q, cu_k = varlen_inputs(sq, sk, Hq, Hkv, d, seed=550, device=DEV)
    slopes = _slopes(Hq, len(sq))
    for causal, mod in [(True, dict(window_size=(64, -1))), (False, dict(softcap=10.0)),
                        (True, dict(alibi_slopes=slopes)),
                        (False, dict(window_size=(150, 20), softcap=8.0, alibi_slopes=slopes))]:
        sl = mod.get("alibi_slopes")
        kw = dict(mod, alibi_slopes=None if sl is None else sl.to(DEV))
        o, lse = fa_fwd_varlen(q, k, v, cu_q, cu_k, max(sq), max(sk), causal=causal, **kw)
        assert get_last_device_error() == FA_OK
        o_ref, lse_ref = ORACLE.attention_varlen(
            q.cpu(), k.cpu(), v.cpu(), cu_q.cpu(), cu_k.cpu(), _scale(d), causal,
            window=mod.get("window_size", (-1, -1)), softcap=mod.get("softcap", 0.0),
            alibi_slopes=sl)
        compare(*varlen_rows(o, lse), *varlen_rows(o_ref, lse_ref), f"varlen {causal} {mod}")


@pytest.mark.parametrize("d,group", [(128, 4), (128, 8), (64, 1), (128, 1), (256, 8), (192, 4)])
@pytest.mark.parametrize("mod", ["window", "softcap", "alibi", "all"])
def test_modifiers_decode(d, group, mod):
    lens = torch.tensor([1, 127, 128, 129, 1000, 3000, 0, 4096], dtype=torch.int32)
    B, Hkv = len(lens), 2
    Hq = Hkv * group
    q, kc, vc, lens = kvcache_inputs(B, 4096, Hq, Hkv, d, seed=560 + d + group, lengths=lens,
                                     device=DEV)
    slopes = _slopes(Hq, B)
    kw = {"window": dict(window_size=(700, -1)), "softcap": dict(softcap=15.0),
          "alibi": dict(alibi_slopes=slopes),
          "all": dict(window_size=(1500, 0), softcap=4.0, alibi_slopes=slopes)}[mod]
    sl = kw.get("alibi_slopes")
    o, lse = fa_fwd_kvcache(q, kc, vc, lens, **dict(kw, alibi_slopes=None if sl is None
                                                     else sl.to(DEV)))
    assert get_last_device_error() == FA_OK
    o_ref, lse_ref = ORACLE.attention_kvcache(q.cpu(), kc.cpu(), vc.cpu(), lens.cpu(), _scale(d),
                                              window=kw.get("window_size", (-1, -1)),
                                              softcap=kw.get("softcap", 0.0), alibi_slopes=sl)
    compare(o[:, 0], lse, o_ref, lse_ref, f"decode d={d} G={group} {mod}")


@pytest.mark.parametrize("wl", [0, 1, 255, 256, 257, 2047])
def test_decode_window_chunk_edges(wl):
    """Left bounds on and around 128-key block and chunk edges (chunks of 256 keys here)."""
    lens = torch.tensor([4096, 2049, 2048, 300, 1], dtype=torch.int32)
    q, kc, vc, lens = kvcache_inputs(len(lens), 4096, 8, 2, 128, seed=570 + wl, lengths=lens,
                                     device=DEV)
    o, lse = fa_fwd_kvcache(q, kc, vc, lens, window_size=(wl, -1))
    assert get_last_device_error() == FA_OK
    o_ref, lse_ref = ORACLE.attention_kvcache(q.cpu(), kc.cpu(), vc.cpu(), lens.cpu(),
                                              _scale(128), window=(wl, -1))
    compare(o[:, 0], lse, o_ref, lse_ref, f"decode window {wl}")


@pytest.mark.parametrize("Lmax,wl,num_splits", [(4097, 4095, 0), (4097, 300, 0),
                                                (9000, 5000, 3), (700, 699, 0)])
def test_decode_window_within_workspace(Lmax, wl, num_splits):
    """The window's key range is split within the chunk count the workspace was sized for
    (auto chunking is not monotone in the length: 4096 keys give 16 chunks, 4097 give 11);
    the workspace is allocated to exactly fa_fwd_kvcache_workspace_size."""
    from exact_attention_81_gb300 import fa_fwd_kvcache_workspace_size
    lens = torch.tensor([Lmax, Lmax - 1, wl + 1, wl, 1], dtype=torch.int32)
    Hq, Hkv, d = 8, 2, 128
    q, kc, vc, lens = kvcache_inputs(len(lens), Lmax, Hq, Hkv, d, seed=590 + wl, lengths=lens,
                                     device=DEV)
    need = fa_fwd_kvcache_workspace_size(len(lens), Hq, Lmax, d, num_splits)
    buf = torch.full((need + (1 << 20),), 0x7F, dtype=torch.uint8, device=DEV)
    o, lse = fa_fwd_kvcache(q, kc, vc, lens, num_splits=num_splits, workspace=buf[:need],
                            window_size=(wl, -1))
    assert get_last_device_error() == FA_OK
    assert torch.all(buf[need:] == 0x7F), "partials written past the workspace"
    o_ref, lse_ref = ORACLE.attention_kvcache(q.cpu(), kc.cpu(), vc.cpu(), lens.cpu(),
                                              _scale(d), window=(wl, -1))
    compare(o[:, 0], lse, o_ref, lse_ref, f"decode Lmax={Lmax} window {wl}")


def test_full_size_causal8k_sliding_window():
    """The causal 8k workload with a 4096-key sliding window: sampled rows."""
    w = WORKLOADS["causal8k"]
    q, k, v = dense_inputs(w.B, w.Nq, w.Nk, w.Hq, w.Hkv, w.d, seed=w.seed, device=DEV)
    o, lse = fa_fwd(q, k, v, causal=True, window_size=(4096, 0))
    assert get_last_device_error() == FA_OK
    rows = sample_rows(w.B, w.Hq, w.Nq, 120, seed=w.seed + 7,
                       must=[(0, 0, 4095), (0, 0, 4096), (1, 31, 8191)])
    o_ref, lse_ref = ORACLE.attention_rows(q.cpu(), k.cpu(), v.cpu(), rows, w.scale, True,
                                           window=(4096, 0))
    r = torch.as_tensor(rows, dtype=torch.long)
    compare(o[r[:, 0], r[:, 2], r[:, 1]], lse[r[:, 0], r[:, 1], r[:, 2]], o_ref, lse_ref,
            "causal8k window 4096")


def test_full_size_causal8k_softcap_alibi():
    w = WORKLOADS["causal8k"]
    q, k, v = dense_inputs(w.B, w.Nq, w.Nk, w.Hq, w.Hkv, w.d, seed=w.seed, device=DEV)
    slopes = _slopes(w.Hq)
    o, lse = fa_fwd(q, k, v, causal=True, softcap=30.0, alibi_slopes=slopes.to(DEV))
    assert get_last_device_error() == FA_OK
    rows = sample_rows(w.B, w.Hq, w.Nq, 80, seed=w.seed + 8)
    o_ref, lse_ref = ORACLE.attention_rows(q.cpu(), k.cpu(), v.cpu(), rows, w.scale, True,
                                           softcap=30.0, alibi_slopes=slopes)
    r = torch.as_tensor(rows, dtype=torch.long)
    compare(o[r[:, 0], r[:, 2], r[:, 1]], lse[r[:, 0], r[:, 1], r[:, 2]], o_ref, lse_ref,
            "causal8k softcap + ALiBi")


def test_plain_window_matches_plain_kernels():
    """Windows that hide nothing take the plain kernels: bit-identical results."""
    q, k, v = dense_inputs(1, 1000, 1000, 4, 2, 128, seed=580, device=DEV)
    o1, l1 = fa_fwd(q, k, v, causal=True)
    o2, l2 = fa_fwd(q, k, v, window_size=(-1, 0))
    o3, l3 = fa_fwd(q, k, v, causal=True, window_size=(5000, -1))  # general kernel
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    compare(*dense_rows(o3, l3), *dense_rows(o1.double().cpu().numpy(), l1.double().cpu().numpy()),
            "wide window vs causal")


@pytest.mark.parametrize("d,dtype,window,Nq,Nk", [
    (128, torch.bfloat16, (-1, -1), 2048, 2048), (64, torch.float16, (-1, -1), 1500, 1900),
    (128, torch.bfloat16, (500, -1), 1300, 1300), (256, torch.bfloat16, (-1, -1), 900, 900),
])
def test_alibi_only_causal_long_rows(d, dtype, window, Nq, Nk):
    """ALiBi without a softcap runs its own instance: on the tiles whose keys all lie at or
    before the row's position the bias is built as a linear function of the column.  Long
    causal rows put most tiles on that path; slopes from 1 down to 2^-3 (steeper than the
    usual geometric set) make the bias dominate the scores."""
    Hq, Hkv = 4, 1
    slopes = torch.tensor([1.0, 0.5, 0.25, 0.125], dtype=torch.float32)
    # allowance: a slope of 1 leaves 1 - 1/e of a row's probability on its last key, so O
    # is close to one value row and rounds like it
    _dense(1, Nq, Nk, Hq, Hkv, d, True, seed=560 + d + Nq, dtype=dtype, window_size=window,
           allowance=True, alibi_slopes=slopes)
