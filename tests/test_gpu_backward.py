"""GPU parity of the backward pass (fa_bwd) against the fp64 oracle.

The forward bounds have no stated counterpart for gradients, so the bar is the pages' own
("flash-attention", section 5, tests: the error of the fused kernel is at most twice the
error of a PyTorch baseline run in the input precision): for each of dQ, dK and dV,
    max |g_gpu - g_oracle| <= 2 * max |g_baseline - g_oracle| + 1e-4,
where the baseline is the same attention written with torch ops on the CPU in bf16 / fp16
(matmuls in the input type, softmax in fp32 then rounded, as upstream's reference does)
and differentiated by autograd.  Query rows that see no key must get dQ = 0 exactly.
"""
import math

import numpy as np
import pytest
import torch

import oracle.oracle as ORACLE
from exact_attention_81_gb300 import (FA_OK, fa_bwd, fa_bwd_varlen, fa_fwd, fa_fwd_varlen,
                                      get_last_device_error)
from exact_attention_81_gb300.inputs import WORKLOADS, bf16_normal, dense_inputs, varlen_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _mask(Nq, Nk):
    i = torch.arange(Nq)[:, None]
    j = torch.arange(Nk)[None, :]
    return j <= i + (Nk - Nq)


def _baseline(q, k, v, do, scale, causal):
    """PyTorch attention in the input precision on the CPU, differentiated by autograd."""
    dt = q.dtype
    Hq, Hkv = q.shape[2], k.shape[2]
    G = Hq // Hkv
    qq = q.cpu().permute(0, 2, 1, 3).detach().requires_grad_()
    kk = k.cpu().permute(0, 2, 1, 3).detach().requires_grad_()
    vv = v.cpu().permute(0, 2, 1, 3).detach().requires_grad_()
    s = torch.matmul(qq, kk.repeat_interleave(G, 1).transpose(-1, -2)) * scale
    if causal:
        s = s.masked_fill(~_mask(q.shape[1], k.shape[1]), float("-inf"))
    p = torch.softmax(s.float(), dim=-1).nan_to_num(0.0).to(dt)
    o = torch.matmul(p, vv.repeat_interleave(G, 1))
    o.backward(do.cpu().permute(0, 2, 1, 3))
    return (qq.grad.permute(0, 2, 1, 3), kk.grad.permute(0, 2, 1, 3),
            vv.grad.permute(0, 2, 1, 3))


def _check(q, k, v, do, scale, causal, what, deterministic=False):
    o, lse = fa_fwd(q, k, v, causal=causal, scale=scale)
    dq, dk, dv = fa_bwd(q, k, v, o, lse, do, causal=causal, scale=scale,
                        deterministic=deterministic)
    assert get_last_device_error() == FA_OK
    ref = ORACLE.attention_bwd(q.cpu(), k.cpu(), v.cpu(), do.cpu(), scale, causal)[:3]
    base = _baseline(q, k, v, do, scale, causal)
    report = {}
    for name, g, r, b in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref, base):
        g = g.double().cpu().numpy()
        b = b.double().numpy()
        assert np.all(np.isfinite(g)), f"{what}: non-finite {name}"
        e_gpu = float(np.abs(g - r).max())
        e_base = float(np.abs(b - r).max())
        report[name] = (e_gpu, e_base)
        assert e_gpu <= 2 * e_base + 1e-4, \
            f"{what}: max|d{name}| = {e_gpu:.3e} > 2 x baseline {e_base:.3e}"
    return report, (dq, dk, dv)


@pytest.mark.parametrize("case", [
    # B, Nq, Nk, Hq, Hkv, d, causal, dtype
    (1, 128, 128, 1, 1, 128, False, torch.bfloat16),
    (2, 256, 256, 4, 2, 128, True, torch.bfloat16),
    (1, 300, 300, 2, 2, 64, True, torch.bfloat16),
    (1, 200, 517, 4, 1, 128, True, torch.bfloat16),
    (2, 384, 384, 8, 2, 128, False, torch.float16),
    (1, 129, 1000, 2, 2, 128, False, torch.bfloat16),
    (1, 640, 640, 2, 1, 64, False, torch.float16),
])
def test_backward(case):
    B, Nq, Nk, Hq, Hkv, d, causal, dt = case
    q, k, v = dense_inputs(B, Nq, Nk, Hq, Hkv, d, seed=700 + Nq + d, device=DEV, dtype=dt)
    do = bf16_normal((B, Nq, Hq, d), seed=710 + Nq, device=DEV, dtype=dt)
    _check(q, k, v, do, float(np.float32(1 / math.sqrt(d))), causal, f"bwd {case}")


@pytest.mark.parametrize("case", [
    (2, 700, 700, 4, 2, 128, True), (1, 300, 900, 4, 1, 128, True), (2, 513, 513, 2, 2, 64, False)])
def test_backward_deterministic(case):
    """deterministic=True: the key blocks add into dQ in a fixed order, so two calls give
    bit-identical gradients, within the same bar against the oracle."""
    B, Nq, Nk, Hq, Hkv, d, causal = case
    q, k, v = dense_inputs(B, Nq, Nk, Hq, Hkv, d, seed=730 + Nq, device=DEV)
    do = bf16_normal((B, Nq, Hq, d), seed=731 + Nq, device=DEV)
    scale = float(np.float32(1 / math.sqrt(d)))
    _, g1 = _check(q, k, v, do, scale, causal, f"deterministic {case}", deterministic=True)
    o, lse = fa_fwd(q, k, v, causal=causal, scale=scale)
    for _ in range(2):
        g2 = fa_bwd(q, k, v, o, lse, do, causal=causal, scale=scale, deterministic=True)
        assert get_last_device_error() == FA_OK
        for a, b in zip(g1, g2):
            assert torch.equal(a, b), "deterministic backward differs between calls"


def test_backward_rows_without_keys():
    """Causal with Nq > Nk (bottom-right): query rows i < Nq - Nk see no key, their dQ is
    exactly 0 and they add nothing to dK and dV."""
    B, Nq, Nk, H, d = 1, 700, 130, 2, 128
    q, k, v = dense_inputs(B, Nq, Nk, H, H, d, seed=722, device=DEV)
    do = bf16_normal((B, Nq, H, d), seed=723, device=DEV)
    _, (dq, dk, dv) = _check(q, k, v, do, 0.088, True, "bwd Nq > Nk")
    assert torch.all(dq[:, :Nq - Nk] == 0), "rows that see no key must have dQ = 0"


def test_backward_full_size_one_head():
    """The causal 8k workload: the gradients of head (0, 0), whose dK / dV depend only on
    that head (no GQA), against the oracle and the baseline on that head alone."""
    w = WORKLOADS["causal8k"]
    q, k, v = dense_inputs(w.B, w.Nq, w.Nk, w.Hq, w.Hkv, w.d, seed=w.seed, device=DEV)
    do = bf16_normal((w.B, w.Nq, w.Hq, w.d), seed=w.seed + 9, device=DEV)
    o, lse = fa_fwd(q, k, v, causal=True)
    dq, dk, dv = fa_bwd(q, k, v, o, lse, do, causal=True)
    assert get_last_device_error() == FA_OK
    sl = (slice(0, 1), slice(None), slice(0, 1))
    q1, k1, v1, do1 = (t[sl].contiguous() for t in (q, k, v, do))
    ref = ORACLE.attention_bwd(q1.cpu(), k1.cpu(), v1.cpu(), do1.cpu(), w.scale, True)[:3]
    base = _baseline(q1, k1, v1, do1, w.scale, True)
    for name, g, r, b in zip(("dQ", "dK", "dV"), (dq[sl], dk[sl], dv[sl]), ref, base):
        e_gpu = float(np.abs(g.double().cpu().numpy() - r).max())
        e_base = float(np.abs(b.double().numpy() - r).max())
        assert e_gpu <= 2 * e_base + 1e-4, f"causal8k {name}: {e_gpu:.3e} vs {e_base:.3e}"


def _baseline_varlen(q, k, v, do, cu_q, cu_k, scale, causal):
    """The PyTorch baseline sequence by sequence, in the packed layouts."""
    outs = [torch.zeros(t.shape, dtype=t.dtype) for t in (q, k, v)]
    cq, ck = cu_q.tolist(), cu_k.tolist()
    for b in range(len(cq) - 1):
        a, e, ka, ke = cq[b], cq[b + 1], ck[b], ck[b + 1]
        if e == a or ke == ka:
            continue
        g = _baseline(q[a:e].unsqueeze(0), k[ka:ke].unsqueeze(0), v[ka:ke].unsqueeze(0),
                      do[a:e].unsqueeze(0), scale, causal)
        outs[0][a:e], outs[1][ka:ke], outs[2][ka:ke] = g[0][0], g[1][0], g[2][0]
    return outs


@pytest.mark.parametrize("causal,deterministic,dt", [(True, False, torch.bfloat16),
                                                     (False, False, torch.bfloat16),
                                                     (True, True, torch.bfloat16),
                                                     (True, False, torch.float16)])
def test_backward_varlen(causal, deterministic, dt):
    sq = [5, 0, 333, 128, 129, 700, 1]
    sk = [7, 3, 333, 400, 200, 700, 0]
    Hq, Hkv, d = 4, 2, 128
    q, k, v, cu_q, cu_k = varlen_inputs(sq, sk, Hq, Hkv, d, seed=740, device=DEV, dtype=dt)
    do = bf16_normal(tuple(q.shape), seed=741, device=DEV, dtype=dt)
    scale = float(np.float32(1 / math.sqrt(d)))
    o, lse = fa_fwd_varlen(q, k, v, cu_q, cu_k, max(sq), max(sk), causal=causal, scale=scale)
    g = fa_bwd_varlen(q, k, v, o, lse, do, cu_q, cu_k, max(sq), max(sk), causal=causal,
                      scale=scale, deterministic=deterministic)
    assert get_last_device_error() == FA_OK
    ref = ORACLE.attention_varlen_bwd(q.cpu(), k.cpu(), v.cpu(), do.cpu(), cu_q.cpu(),
                                      cu_k.cpu(), scale, causal)
    base = _baseline_varlen(q.cpu(), k.cpu(), v.cpu(), do.cpu(), cu_q.cpu(), cu_k.cpu(), scale,
                            causal)
    for name, a, r, b in zip(("dQ", "dK", "dV"), g, ref, base):
        a = a.double().cpu().numpy()
        e_gpu = float(np.abs(a - r).max())
        e_base = float(np.abs(b.double().numpy() - r).max())
        assert e_gpu <= 2 * e_base + 1e-4, f"varlen {name}: {e_gpu:.3e} vs {e_base:.3e}"
    # sequences without keys give dQ = 0; keys no query sees give dK = dV = 0
    assert torch.all(g[0][cu_q[6]:cu_q[7]] == 0)
    assert torch.all(g[1][cu_k[1]:cu_k[2]] == 0) and torch.all(g[2][cu_k[1]:cu_k[2]] == 0)
    if deterministic:
        g2 = fa_bwd_varlen(q, k, v, o, lse, do, cu_q, cu_k, max(sq), max(sk), causal=causal,
                           scale=scale, deterministic=True)
        assert all(torch.equal(x, y) for x, y in zip(g, g2))
