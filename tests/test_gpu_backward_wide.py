"""GPU parity of the backward pass at head dimensions 136..256 (the wide kernel: units per
d half, 64-query steps, a transposed dQ accumulator) against the fp64 oracle, under the
plain backward's bar: for each of dQ, dK and dV the error is at most twice that of a
PyTorch baseline in the input precision (+1e-4).  Dense (causal or not, GQA, ragged
lengths, both 16-bit types), deterministic order, varlen and the score modifiers."""
import math

import numpy as np
import pytest
import torch

import oracle.oracle as ORACLE
from exact_attention_81_gb300 import (FA_OK, fa_bwd, fa_bwd_varlen, fa_fwd, fa_fwd_varlen,
                                      get_last_device_error)
from exact_attention_81_gb300.inputs import bf16_normal, dense_inputs, varlen_inputs
from tests.test_gpu_backward import _baseline_varlen, _check
from tests.test_gpu_backward_mods import _dense, _slopes

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _scale(d):
    return float(np.float32(1 / math.sqrt(d)))


@pytest.mark.parametrize("case", [
    # B, Nq, Nk, Hq, Hkv, d, causal, dtype
    (1, 128, 128, 1, 1, 256, False, torch.bfloat16),
    (2, 300, 300, 4, 2, 192, True, torch.bfloat16),   # ragged: 300 = 4 x 64 + 44 queries
    (1, 200, 517, 4, 1, 256, True, torch.bfloat16),   # Nq < Nk, MQA
    (1, 517, 200, 2, 2, 136, True, torch.bfloat16),   # Nq > Nk: leading rows see no key
    (2, 257, 257, 2, 1, 248, False, torch.float16),
    (1, 640, 640, 2, 2, 256, True, torch.float16),
])
def test_backward_wide(case):
    B, Nq, Nk, Hq, Hkv, d, causal, dt = case
    q, k, v = dense_inputs(B, Nq, Nk, Hq, Hkv, d, seed=1700 + Nq + d, device=DEV, dtype=dt)
    do = bf16_normal((B, Nq, Hq, d), seed=1710 + Nq, device=DEV, dtype=dt)
    _, (dq, _, _) = _check(q, k, v, do, _scale(d), causal, f"wide bwd {case}")
    if causal and Nq > Nk:
        assert torch.all(dq[:, :Nq - Nk] == 0), "rows that see no key must have dQ = 0"


@pytest.mark.parametrize("case", [(2, 700, 700, 4, 2, 256, True), (1, 300, 900, 4, 1, 192, True),
                                  (1, 513, 513, 2, 2, 160, False)])
def test_backward_wide_deterministic(case):
    """deterministic=True: bit-identical gradients between calls, within the bar."""
    B, Nq, Nk, Hq, Hkv, d, causal = case
    q, k, v = dense_inputs(B, Nq, Nk, Hq, Hkv, d, seed=1730 + Nq, device=DEV)
    do = bf16_normal((B, Nq, Hq, d), seed=1731 + Nq, device=DEV)
    sc = _scale(d)
    _, g1 = _check(q, k, v, do, sc, causal, f"wide deterministic {case}", deterministic=True)
    o, lse = fa_fwd(q, k, v, causal=causal, scale=sc)
    for _ in range(2):
        g2 = fa_bwd(q, k, v, o, lse, do, causal=causal, scale=sc, deterministic=True)
        assert get_last_device_error() == FA_OK
        for a, b in zip(g1, g2):
            assert torch.equal(a, b), "deterministic backward differs between calls"


@pytest.mark.parametrize("causal,deterministic", [(True, False), (False, True)])
def test_backward_wide_varlen(causal, deterministic):
    sq = [5, 0, 333, 128, 129, 450, 1]
    sk = [7, 3, 333, 400, 200, 450, 0]
    Hq, Hkv, d = 4, 2, 192
    q, k, v, cu_q, cu_k = varlen_inputs(sq, sk, Hq, Hkv, d, seed=1740, device=DEV)
    do = bf16_normal(tuple(q.shape), seed=1741, device=DEV)
    sc = _scale(d)
    o, lse = fa_fwd_varlen(q, k, v, cu_q, cu_k, max(sq), max(sk), causal=causal, scale=sc)
    g = fa_bwd_varlen(q, k, v, o, lse, do, cu_q, cu_k, max(sq), max(sk), causal=causal,
                      scale=sc, deterministic=deterministic)
    assert get_last_device_error() == FA_OK
    ref = ORACLE.attention_varlen_bwd(q.cpu(), k.cpu(), v.cpu(), do.cpu(), cu_q.cpu(),
                                      cu_k.cpu(), sc, causal)
    base = _baseline_varlen(q.cpu(), k.cpu(), v.cpu(), do.cpu(), cu_q.cpu(), cu_k.cpu(), sc,
                            causal)
    for name, a, r, b in zip(("dQ", "dK", "dV"), g, ref, base):
        a = a.double().cpu().numpy()
        e_gpu = float(np.abs(a - r).max())
        e_base = float(np.abs(b.double().numpy() - r).max())
        assert e_gpu <= 2 * e_base + 1e-4, f"wide varlen {name}: {e_gpu:.3e} vs {e_base:.3e}"
    assert torch.all(g[0][cu_q[6]:cu_q[7]] == 0)
    assert torch.all(g[1][cu_k[1]:cu_k[2]] == 0) and torch.all(g[2][cu_k[1]:cu_k[2]] == 0)
    if deterministic:
        g2 = fa_bwd_varlen(q, k, v, o, lse, do, cu_q, cu_k, max(sq), max(sk), causal=causal,
                           scale=sc, deterministic=True)
        assert all(torch.equal(x, y) for x, y in zip(g, g2))


@pytest.mark.parametrize("mod", ["window", "softcap", "alibi", "all"])
def test_backward_wide_modifiers(mod):
    Hq, B = 4, 2
    kw = {"window": dict(window=(150, 20)), "softcap": dict(softcap=20.0),
          "alibi": dict(slopes=_slopes(Hq)),
          "all": dict(window=(200, -1), softcap=10.0, slopes=_slopes(Hq, B))}[mod]
    _dense(B, 333, 333, Hq, 2, 256, mod in ("alibi", "all"), seed=1750 + len(mod), **kw)
