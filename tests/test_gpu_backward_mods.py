"""GPU parity of the backward pass with the score modifiers (sliding window, softcap,
ALiBi) against the fp64 oracle, under the same bar as the plain backward: for each of dQ,
dK and dV the error is at most twice that of a PyTorch baseline in the input precision
(+1e-4).  The baseline applies the modifiers in fp32 on the input-precision scores, then
the softmax in fp32 rounded to the input type, and is differentiated by autograd."""
import math

import numpy as np
import pytest
import torch

import oracle.oracle as ORACLE
from exact_attention_81_gb300 import (FA_OK, fa_bwd, fa_bwd_varlen, fa_fwd, fa_fwd_varlen,
                                      get_last_device_error)
from exact_attention_81_gb300.inputs import bf16_normal, dense_inputs, varlen_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _scale(d):
    return float(np.float32(1 / math.sqrt(d)))


def _slopes(Hq, B=None):
    base = 2.0 ** (-8.0 * np.arange(1, Hq + 1) / Hq)
    if B is None:
        return torch.tensor(base, dtype=torch.float32)
    return torch.tensor(np.stack([base * (1.0 + 0.25 * b) for b in range(B)]),
                        dtype=torch.float32)


def _visible(Nq, Nk, wl, wr):
    """Key j is visible to query i when pos - wl <= j <= pos + wr, pos = i + Nk - Nq
    (negative bounds are unbounded)."""
    pos = torch.arange(Nq)[:, None] + (Nk - Nq)
    j = torch.arange(Nk)[None, :]
    vis = torch.ones(Nq, Nk, dtype=torch.bool)
    if wl >= 0:
        vis &= j >= pos - wl
    if wr >= 0:
        vis &= j <= pos + wr
    return vis, (pos - j).abs()


def _baseline(q, k, v, do, scale, wl, wr, softcap, slopes):
    dt = q.dtype
    B, Nq, Hq, _ = q.shape
    Nk, Hkv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    qq = q.cpu().permute(0, 2, 1, 3).detach().requires_grad_()
    kk = k.cpu().permute(0, 2, 1, 3).detach().requires_grad_()
    vv = v.cpu().permute(0, 2, 1, 3).detach().requires_grad_()
    s = (torch.matmul(qq, kk.repeat_interleave(G, 1).transpose(-1, -2)) * scale).float()
    if softcap > 0:
        s = softcap * torch.tanh(s / softcap)
    vis, dist = _visible(Nq, Nk, wl, wr)
    if slopes is not None:
        sl = slopes.reshape(-1, Hq) if slopes.dim() == 2 else slopes.reshape(1, Hq)
        s = s - sl[:, :, None, None] * dist.float()
    s = s.masked_fill(~vis, float("-inf"))
    p = torch.softmax(s, dim=-1).nan_to_num(0.0).to(dt)
    o = torch.matmul(p, vv.repeat_interleave(G, 1))
    o.backward(do.cpu().permute(0, 2, 1, 3))
    return (qq.grad.permute(0, 2, 1, 3), kk.grad.permute(0, 2, 1, 3),
            vv.grad.permute(0, 2, 1, 3))


def _bar(what, grads, ref, base):
    for name, g, r, b in zip(("dQ", "dK", "dV"), grads, ref, base):
        g = g.double().cpu().numpy()
        assert np.all(np.isfinite(g)), f"{what}: non-finite {name}"
        e_gpu = float(np.abs(g - r).max())
        e_base = float(np.abs(b.double().numpy() - r).max())
        assert e_gpu <= 2 * e_base + 1e-4, \
            f"{what}: max|d{name}| = {e_gpu:.3e} > 2 x baseline {e_base:.3e}"


def _dense(B, Nq, Nk, Hq, Hkv, d, causal, seed, dtype=torch.bfloat16, deterministic=False,
           window=(-1, -1), softcap=0.0, slopes=None):
    q, k, v = dense_inputs(B, Nq, Nk, Hq, Hkv, d, seed=seed, device=DEV, dtype=dtype)
    do = bf16_normal((B, Nq, Hq, d), seed=seed + 1, device=DEV, dtype=dtype)
    sc = _scale(d)
    kw = dict(window_size=window, softcap=softcap,
              alibi_slopes=None if slopes is None else slopes.to(DEV))
    o, lse = fa_fwd(q, k, v, causal=causal, scale=sc, **kw)
    grads = fa_bwd(q, k, v, o, lse, do, causal=causal, scale=sc, deterministic=deterministic,
                   **kw)
    assert get_last_device_error() == FA_OK
    ref = ORACLE.attention_bwd(q.cpu(), k.cpu(), v.cpu(), do.cpu(), sc, causal, window=window,
                               softcap=softcap, alibi_slopes=slopes)[:3]
    wl, wr = window
    if causal:
        wr = 0
    base = _baseline(q, k, v, do, sc, wl, wr, softcap, slopes)
    what = f"bwd B={B} Nq={Nq} Nk={Nk} causal={causal} window={window} softcap={softcap}"
    _bar(what, grads, ref, base)
    if deterministic:
        again = fa_bwd(q, k, v, o, lse, do, causal=causal, scale=sc, deterministic=True, **kw)
        assert all(torch.equal(a, b) for a, b in zip(grads, again)), \
            f"{what}: deterministic backward differs between calls"
    return grads


@pytest.mark.parametrize("window,causal", [
    ((100, 0), False), ((256, 256), False), ((0, 0), False), ((127, 129), False),
    ((-1, 300), False), ((1000, -1), False), ((300, -1), True), ((5, 7), True),
])
def test_window_backward(window, causal):
    _dense(2, 700, 700, 4, 2, 128, causal, seed=900 + window[0], window=window)


@pytest.mark.parametrize("Nq,Nk,window", [
    (300, 900, (200, 50)), (900, 300, (100, 10)), (129, 1000, (0, 0)), (1000, 129, (64, -1)),
])
def test_window_backward_unequal_lengths(Nq, Nk, window):
    """Bottom-right alignment; with Nq > Nk the first rows' windows hold no key and their
    dQ is exactly 0."""
    dq, _, _ = _dense(1, Nq, Nk, 2, 1, 64, False, seed=910 + Nq, window=window)
    vis, _ = _visible(Nq, Nk, *window)
    empty = ~vis.any(dim=1)
    if empty.any():
        assert torch.all(dq[:, empty.to(DEV)] == 0)


@pytest.mark.parametrize("softcap,causal,d", [(30.0, True, 128), (5.0, False, 128),
                                              (2.0, True, 64), (50.0, False, 64)])
def test_softcap_backward(softcap, causal, d):
    _dense(2, 517, 517, 4, 2, d, causal, seed=920 + d, softcap=softcap)


@pytest.mark.parametrize("per_batch,causal", [(False, True), (True, False), (True, True)])
def test_alibi_backward(per_batch, causal):
    B, Hq = 2, 8
    slopes = _slopes(Hq, B if per_batch else None)
    _dense(B, 400, 600, Hq, 2, 128, causal, seed=930 + per_batch, slopes=slopes)


def test_all_modifiers_backward_fp16():
    _dense(2, 640, 640, 8, 2, 128, False, seed=940, dtype=torch.float16, window=(200, 30),
           softcap=20.0, slopes=_slopes(8, 2))


@pytest.mark.parametrize("window,causal", [((300, -1), True), ((150, 40), False),
                                           ((0, 0), False)])
def test_window_backward_deterministic(window, causal):
    """With a left window bound the key blocks that reach a query block start past block 0;
    the deterministic order still covers them once each, in a fixed order."""
    _dense(2, 900, 900, 4, 2, 128, causal, seed=950 + window[0], deterministic=True,
           window=window, softcap=10.0)


@pytest.mark.parametrize("d", [64, 96])
def test_modifiers_backward_head_dims(d):
    _dense(1, 333, 333, 4, 4, d, True, seed=960 + d, window=(100, -1), softcap=15.0,
           slopes=_slopes(4))


def test_varlen_backward_modifiers():
    sq = [5, 0, 333, 128, 129, 700, 1]
    sk = [7, 3, 333, 400, 200, 700, 0]
    Hq, Hkv, d = 4, 2, 128
    window, softcap, slopes = (120, 16), 12.0, _slopes(Hq, len(sq))
    q, k, v, cu_q, cu_k = varlen_inputs(sq, sk, Hq, Hkv, d, seed=970, device=DEV)
    do = bf16_normal(tuple(q.shape), seed=971, device=DEV)
    sc = _scale(d)
    kw = dict(window_size=window, softcap=softcap, alibi_slopes=slopes.to(DEV))
    o, lse = fa_fwd_varlen(q, k, v, cu_q, cu_k, max(sq), max(sk), causal=False, scale=sc, **kw)
    grads = fa_bwd_varlen(q, k, v, o, lse, do, cu_q, cu_k, max(sq), max(sk), causal=False,
                          scale=sc, **kw)
    assert get_last_device_error() == FA_OK
    ref = ORACLE.attention_varlen_bwd(q.cpu(), k.cpu(), v.cpu(), do.cpu(), cu_q.cpu(),
                                      cu_k.cpu(), sc, False, window=window, softcap=softcap,
                                      alibi_slopes=slopes)
    base = [torch.zeros(t.shape, dtype=t.dtype) for t in (q, k, v)]
    cq, ck = cu_q.tolist(), cu_k.tolist()
    for b in range(len(sq)):
        a, e, ka, ke = cq[b], cq[b + 1], ck[b], ck[b + 1]
        if e == a or ke == ka:
            continue
        g = _baseline(q[a:e].unsqueeze(0), k[ka:ke].unsqueeze(0), v[ka:ke].unsqueeze(0),
                      do[a:e].unsqueeze(0), sc, window[0], window[1], softcap, slopes[b])
        base[0][a:e], base[1][ka:ke], base[2][ka:ke] = g[0][0], g[1][0], g[2][0]
    _bar("varlen with modifiers", grads, ref, base)


@pytest.mark.parametrize("deterministic,Nq,Nk", [(False, 1024, 1024), (True, 700, 1100)])
def test_alibi_only_backward_long_rows(deterministic, Nq, Nk):
    """ALiBi without a softcap: blocks whose queries all sit at or after their keys build the
    bias as a linear function of the query (the ALiBi instance's packed path)."""
    slopes = torch.tensor([1.0, 0.5, 0.25, 0.125], dtype=torch.float32)
    _dense(1, Nq, Nk, 4, 2, 128, True, seed=970 + Nq, deterministic=deterministic,
           slopes=slopes)
