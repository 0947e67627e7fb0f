"""Pins for the fp64 oracle: checks against facts fixed outside the oracle itself.

Each ``pin_*`` function takes an oracle module (``oracle.oracle`` or a copy built
from a mutated source) and raises ``AssertionError`` when the oracle disagrees with
what the pages and the mathematics fix:

* a library routine it does not call (``torch.nn.functional.scaled_dot_product_attention``
  and ``torch.logsumexp`` in float64);
* closed forms (uniform scores, a single visible key, constant V, two keys, rows
  with no visible key, the hard-max limit);
* invariants (rows of P sum to one, shift of every key by one vector, joint
  permutation of keys and values, GQA as MHA with repeated K/V heads, varlen as
  per-sequence dense, decode as dense with one query, sampled rows as full rows);
* an independent algorithm: the tiled online-softmax recurrence of
  "FlashAttention 1-4 详解", section Online Softmax 数学推导 (running max m,
  running sum l, rescaled accumulator), written here in numpy with the scale and
  the causal mask added, which must reach the same result as the oracle's direct
  two-pass softmax.

The same battery runs against deliberately broken copies of the oracle
(tests/test_oracle.py) to show that a plausible slip in it fails a pin.
"""
from __future__ import annotations

import math

import numpy as np
import torch
import torch.nn.functional as F

from exact_attention_81_gb300.inputs import bf16_normal, dense_inputs, varlen_inputs


def _f64(t: torch.Tensor) -> torch.Tensor:
    return t.to(torch.float64)


def _np(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).numpy()


def _bottom_right_mask(Nq, Nk):
    i = torch.arange(Nq)[:, None]
    j = torch.arange(Nk)[None, :]
    return j <= i + (Nk - Nq)


def _library_attention(q, k, v, scale, causal):
    """float64 torch SDPA + logsumexp; q [B,Nq,Hq,d] -> (O [B,Nq,Hq,d], LSE [B,Hq,Nq])."""
    Hq, Hkv = q.shape[2], k.shape[2]
    G = Hq // Hkv
    qq = _f64(q).permute(0, 2, 1, 3)
    kk = _f64(k).permute(0, 2, 1, 3).repeat_interleave(G, dim=1)
    vv = _f64(v).permute(0, 2, 1, 3).repeat_interleave(G, dim=1)
    mask = _bottom_right_mask(q.shape[1], k.shape[1]) if causal else None
    o = F.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask, scale=scale)
    scores = torch.matmul(qq, kk.transpose(-1, -2)) * scale
    if mask is not None:
        scores = scores.masked_fill(~mask, float("-inf"))
    lse = torch.logsumexp(scores, dim=-1)
    return o.permute(0, 2, 1, 3).numpy(), lse.numpy()


def _close(a, b, tol, what):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    fin = np.isfinite(b)
    assert np.array_equal(np.isfinite(a), fin), f"{what}: finiteness differs"
    assert np.array_equal(a[~fin], b[~fin]), f"{what}: infinite entries differ"
    if fin.any():
        err = np.max(np.abs(a[fin] - b[fin]))
        assert err <= tol, f"{what}: max abs error {err:.3e} > {tol:.1e}"


# --------------------------------------------------------------------------
# library cross-check

LIB_CASES = [
    # B, Nq, Nk, Hq, Hkv, d, causal
    (1, 64, 64, 2, 2, 16, False),
    (2, 37, 37, 4, 2, 64, True),
    (1, 50, 80, 4, 1, 32, True),  # Nq < Nk: bottom-right causal alignment
    (1, 70, 45, 2, 2, 16, False),
    (1, 130, 130, 2, 2, 128, True),
]


def pin_library(O, cases=LIB_CASES):
    for n, (B, Nq, Nk, Hq, Hkv, d, causal) in enumerate(cases):
        q, k, v = dense_inputs(B, Nq, Nk, Hq, Hkv, d, seed=50 + n)
        scale = 1.0 / math.sqrt(d)
        o, lse = O.attention(q, k, v, scale, causal)
        o_ref, lse_ref = _library_attention(q, k, v, scale, causal)
        _close(o, o_ref, 1e-11, f"O vs torch SDPA case {n}")
        _close(lse, lse_ref, 1e-11, f"LSE vs torch logsumexp case {n}")


# --------------------------------------------------------------------------
# closed forms

def pin_uniform_scores(O):
    """Q = 0: every visible key scores 0, so O is the mean of the visible V rows and
    LSE = ln(#visible)."""
    B, N, H, d = 1, 40, 2, 16
    _, k, v = dense_inputs(B, N, N, H, H, d, seed=7)
    q = torch.zeros((B, N, H, d), dtype=torch.bfloat16)
    vv = _np(v)
    for causal in (False, True):
        o, lse = O.attention(q, k, v, 0.25, causal)
        for i in range(N):
            n_vis = i + 1 if causal else N
            for h in range(H):
                _close(o[0, i, h], vv[0, :n_vis, h].mean(axis=0), 1e-13, "uniform O")
                _close(lse[0, h, i], math.log(n_vis), 1e-13, "uniform LSE")


def pin_single_key(O):
    """Causal row 0 sees key 0 only: O = v_0, LSE = scale * q_0 . k_0."""
    B, N, H, d = 2, 9, 3, 32
    q, k, v = dense_inputs(B, N, N, H, H, d, seed=8)
    scale = 0.3
    o, lse = O.attention(q, k, v, scale, True)
    qq, kk, vv = _np(q), _np(k), _np(v)
    for b in range(B):
        for h in range(H):
            _close(o[b, 0, h], vv[b, 0, h], 1e-14, "single-key O")
            s0 = scale * float(np.dot(qq[b, 0, h], kk[b, 0, h]))
            _close(lse[b, h, 0], s0, 1e-12, "single-key LSE")


def pin_constant_v(O):
    """All value rows equal to c: O = c for every row, whatever the scores."""
    B, Nq, Nk, H, d = 1, 20, 33, 2, 16
    q, k, _ = dense_inputs(B, Nq, Nk, H, H, d, seed=9)
    c = bf16_normal((1, 1, H, d), seed=10)
    v = c.expand(B, Nk, H, d).contiguous()
    for causal in (False, True):
        o, _ = O.attention(q, k, v, 0.2, causal)
        _close(o, np.broadcast_to(_np(c), o.shape), 1e-14, "constant-V O")


def pin_two_keys(O):
    """Two keys: P = (sigmoid(s0 - s1), sigmoid(s1 - s0)), LSE = logaddexp(s0, s1)."""
    B, Nq, Nk, H, d = 1, 6, 2, 2, 8
    q, k, v = dense_inputs(B, Nq, Nk, H, H, d, seed=11)
    scale = 0.7
    o, lse = O.attention(q, k, v, scale, False)
    qq, kk, vv = _np(q), _np(k), _np(v)
    for i in range(Nq):
        for h in range(H):
            s0 = scale * float(np.dot(qq[0, i, h], kk[0, 0, h]))
            s1 = scale * float(np.dot(qq[0, i, h], kk[0, 1, h]))
            p0 = 1.0 / (1.0 + math.exp(s1 - s0))
            p1 = 1.0 / (1.0 + math.exp(s0 - s1))
            _close(o[0, i, h], p0 * vv[0, 0, h] + p1 * vv[0, 1, h], 1e-13, "two-key O")
            _close(lse[0, h, i], np.logaddexp(s0, s1), 1e-13, "two-key LSE")


def pin_empty_rows(O):
    """Causal with Nq > Nk (bottom-right): the first Nq - Nk rows see no key and give
    O = 0, LSE = -inf; the others see i - (Nq - Nk) + 1 keys."""
    B, Nq, Nk, H, d = 1, 12, 5, 1, 16
    q, k, v = dense_inputs(B, Nq, Nk, H, H, d, seed=12)
    o, lse = O.attention(q, k, v, 0.25, True)
    for i in range(Nq - Nk):
        assert np.all(o[0, i] == 0.0), "empty row O must be 0"
        assert lse[0, 0, i] == -np.inf, "empty row LSE must be -inf"
    # the last row sees every key: equal to the non-causal last row
    o_nc, lse_nc = O.attention(q, k, v, 0.25, False)
    _close(o[0, -1], o_nc[0, -1], 1e-14, "last causal row")
    _close(lse[0, 0, -1], lse_nc[0, 0, -1], 1e-14, "last causal row LSE")


def pin_hard_max(O):
    """A large scale makes the softmax a hard max: O tends to the value row of the
    best key, within sum_{j != *} exp(-(s* - s_j)) * max|v|."""
    B, N, H, d = 1, 24, 1, 16
    q, k, v = dense_inputs(B, N, N, H, H, d, seed=13)
    scale = 40.0
    o, lse = O.attention(q, k, v, scale, False)
    qq, kk, vv = _np(q), _np(k), _np(v)
    for i in range(N):
        s = scale * (kk[0, :, 0] @ qq[0, i, 0])
        j = int(np.argmax(s))
        gap = np.sort(s)[-1] - s
        bound = np.sum(np.exp(-gap[gap > 0])) * np.max(np.abs(vv)) * 2 + 1e-12
        err = np.max(np.abs(o[0, i, 0] - vv[0, j, 0]))
        assert err <= bound, f"hard-max row {i}: {err:.3e} > {bound:.3e}"
        assert s[j] <= lse[0, 0, i] <= s[j] + math.log(N) + 1e-12, "hard-max LSE bounds"


# --------------------------------------------------------------------------
# invariants

def pin_probs(O):
    """Rows of P sum to one, P_j / P_0 = exp(s_j - s_0), invisible keys get 0."""
    B, N, H, d = 1, 30, 2, 16
    q, k, v = dense_inputs(B, N, N, H, H, d, seed=14)
    scale = 0.25
    qq, kk = _np(q), _np(k)
    for causal in (False, True):
        for i in (0, 7, N - 1):
            p = O.row_probs(q, k, v, 0, 1, i, scale, causal)
            n_vis = i + 1 if causal else N
            assert abs(p.sum() - 1.0) <= 1e-14, "P row must sum to 1"
            assert np.all(p[n_vis:] == 0.0), "invisible keys must have P = 0"
            s = scale * (kk[0, :n_vis, 1] @ qq[0, i, 1])
            _close(p[:n_vis] / p[0], np.exp(s - s[0]), 1e-12, "P ratios")


def pin_shift(O):
    """Adding one vector u to every key leaves O unchanged and shifts LSE by
    scale * q . u (keys and u are small integers, so K + u is exact in bf16)."""
    B, N, H, d = 1, 25, 2, 16
    g = torch.Generator().manual_seed(15)
    q = bf16_normal((B, N, H, d), seed=16)
    k = torch.randint(-8, 9, (B, N, H, d), generator=g).to(torch.bfloat16)
    u = torch.randint(-8, 9, (1, 1, H, d), generator=g).to(torch.bfloat16)
    v = bf16_normal((B, N, H, d), seed=17)
    k2 = (k.float() + u.float()).to(torch.bfloat16)
    assert torch.equal(k2.float(), k.float() + u.float())
    scale = 0.125
    for causal in (False, True):
        o1, l1 = O.attention(q, k, v, scale, causal)
        o2, l2 = O.attention(q, k2, v, scale, causal)
        _close(o2, o1, 1e-12, "shifted-keys O")
        qu = scale * np.einsum("bnhd,hd->bhn", _np(q), _np(u)[0, 0])
        _close(l2, l1 + qu, 1e-11, "shifted-keys LSE")


def pin_permutation(O):
    """Non-causal attention does not depend on the order of the (key, value) pairs."""
    B, Nq, Nk, H, d = 2, 17, 29, 2, 32
    q, k, v = dense_inputs(B, Nq, Nk, H, H, d, seed=18)
    perm = torch.randperm(Nk, generator=torch.Generator().manual_seed(19))
    o1, l1 = O.attention(q, k, v, 0.2, False)
    o2, l2 = O.attention(q, k[:, perm].contiguous(), v[:, perm].contiguous(), 0.2, False)
    _close(o2, o1, 1e-13, "permuted O")
    _close(l2, l1, 1e-13, "permuted LSE")


def pin_gqa(O):
    """GQA with Hq = G * Hkv equals MHA with each K/V head repeated G times."""
    B, N, Hq, Hkv, d = 2, 21, 8, 2, 16
    q, k, v = dense_inputs(B, N, N, Hq, Hkv, d, seed=20)
    G = Hq // Hkv
    kr = k.repeat_interleave(G, dim=2).contiguous()
    vr = v.repeat_interleave(G, dim=2).contiguous()
    for causal in (False, True):
        o1, l1 = O.attention(q, k, v, 0.25, causal)
        o2, l2 = O.attention(q, kr, vr, 0.25, causal)
        _close(o1, o2, 0.0, "GQA vs repeated-head MHA O")
        _close(l1, l2, 0.0, "GQA vs repeated-head MHA LSE")


def pin_varlen(O):
    """A packed varlen batch equals each sequence run on its own (dense)."""
    sq = [5, 0, 19, 33, 1]
    sk = [7, 3, 19, 20, 1]
    Hq, Hkv, d = 4, 2, 16
    q, k, v, cu_q, cu_k = varlen_inputs(sq, sk, Hq, Hkv, d, seed=21)
    for causal in (False, True):
        o, lse = O.attention_varlen(q, k, v, cu_q, cu_k, 0.25, causal)
        for b in range(len(sq)):
            a, e = int(cu_q[b]), int(cu_q[b + 1])
            ka, ke = int(cu_k[b]), int(cu_k[b + 1])
            if e == a:
                continue
            qb = q[a:e].unsqueeze(0).contiguous()
            kb = k[ka:ke].unsqueeze(0).contiguous()
            vb = v[ka:ke].unsqueeze(0).contiguous()
            if ke == ka:
                assert np.all(o[a:e] == 0.0) and np.all(lse[:, a:e] == -np.inf)
                continue
            ob, lb = O.attention(qb, kb, vb, 0.25, causal)
            _close(o[a:e], ob[0], 0.0, f"varlen seq {b} O")
            _close(lse[:, a:e], lb[0], 0.0, f"varlen seq {b} LSE")


def pin_kvcache(O):
    """Decode over the first L_b cache rows equals dense attention with one query and
    Nk = L_b; NaN rows past L_b never reach the result."""
    B, Lmax, Hq, Hkv, d = 3, 40, 4, 2, 16
    lens = [40, 1, 23]
    q = bf16_normal((B, 1, Hq, d), seed=22)
    kc = bf16_normal((B, Lmax, Hkv, d), seed=23)
    vc = bf16_normal((B, Lmax, Hkv, d), seed=24)
    for b, n in enumerate(lens):
        kc[b, n:] = float("nan")
        vc[b, n:] = float("nan")
    o, lse = O.attention_kvcache(q, kc, vc, lens, 0.25)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    for b, n in enumerate(lens):
        ob, lb = O.attention(q[b:b + 1].contiguous(), kc[b:b + 1, :n].contiguous(),
                             vc[b:b + 1, :n].contiguous(), 0.25, False)
        _close(o[b], ob[0, 0], 0.0, f"decode batch {b} O")
        _close(lse[b], lb[0, :, 0], 0.0, f"decode batch {b} LSE")


def pin_rows(O):
    """Row sampling returns exactly the rows of the full computation."""
    B, N, Hq, Hkv, d = 2, 33, 4, 2, 16
    q, k, v = dense_inputs(B, N, N, Hq, Hkv, d, seed=25)
    o, lse = O.attention(q, k, v, 0.25, True)
    rows = np.array([[0, 0, 0], [1, 3, 32], [0, 2, 17], [1, 1, 5]], np.int32)
    orow, lrow = O.attention_rows(q, k, v, rows, 0.25, True)
    for n, (b, h, i) in enumerate(rows):
        _close(orow[n], o[b, i, h], 0.0, "sampled row O")
        _close(lrow[n], lse[b, h, i], 0.0, "sampled row LSE")


def online_softmax_attention(q, k, v, scale, causal, Br, Bc):
    """Tiled forward with the online-softmax recurrence (numpy, fp64), following the
    update rules m_new = max(m, rowmax(S_ij)), P~ = exp(S_ij - m_new),
    l_new = e^{m - m_new} l + rowsum(P~), O_new = e^{m - m_new} O + P~ V_j and the
    final O / l, with the scale applied to S and masked entries set to -inf."""
    qq, kk, vv = _np(q), _np(k), _np(v)
    B, Nq, Hq, d = qq.shape
    Nk, Hkv = kk.shape[1], kk.shape[2]
    G = Hq // Hkv
    O_out = np.zeros((B, Nq, Hq, d))
    L_out = np.zeros((B, Hq, Nq))
    for b in range(B):
        for h in range(Hq):
            Q = qq[b, :, h]
            K = kk[b, :, h // G]
            V = vv[b, :, h // G]
            for i0 in range(0, Nq, Br):
                Qi = Q[i0:i0 + Br]
                rows = np.arange(i0, i0 + Qi.shape[0])
                m = np.full(Qi.shape[0], -np.inf)
                l = np.zeros(Qi.shape[0])
                Oi = np.zeros((Qi.shape[0], d))
                for j0 in range(0, Nk, Bc):
                    Kj, Vj = K[j0:j0 + Bc], V[j0:j0 + Bc]
                    S = scale * (Qi @ Kj.T)
                    if causal:
                        cols = np.arange(j0, j0 + Kj.shape[0])
                        S = np.where(cols[None, :] <= rows[:, None] + (Nk - Nq), S, -np.inf)
                    m_new = np.maximum(m, S.max(axis=1))
                    safe = np.where(np.isfinite(m_new), m_new, 0.0)
                    P = np.exp(S - safe[:, None])
                    alpha = np.where(np.isfinite(m), np.exp(m - safe), 0.0)
                    l = alpha * l + P.sum(axis=1)
                    Oi = alpha[:, None] * Oi + P @ Vj
                    m = m_new
                with np.errstate(invalid="ignore", divide="ignore"):
                    O_out[b, i0:i0 + Br, h] = np.where(l[:, None] > 0, Oi / np.where(
                        l > 0, l, 1.0)[:, None], 0.0)
                    L_out[b, h, i0:i0 + Br] = np.where(l > 0, m + np.log(np.where(
                        l > 0, l, 1.0)), -np.inf)
    return O_out, L_out


def pin_recurrence(O):
    """The oracle's direct softmax and the tiled online recurrence agree."""
    cases = [(1, 70, 70, 2, 1, 16, True, 16, 16), (2, 45, 61, 2, 2, 32, False, 16, 16),
             (1, 150, 150, 1, 1, 64, True, 128, 128), (1, 30, 50, 2, 2, 16, True, 16, 32)]
    for n, (B, Nq, Nk, Hq, Hkv, d, causal, Br, Bc) in enumerate(cases):
        q, k, v = dense_inputs(B, Nq, Nk, Hq, Hkv, d, seed=30 + n)
        scale = 1.0 / math.sqrt(d)
        o, lse = O.attention(q, k, v, scale, causal)
        o2, l2 = online_softmax_attention(q, k, v, scale, causal, Br, Bc)
        _close(o, o2, 1e-12, f"recurrence case {n} O")
        _close(lse, l2, 1e-12, f"recurrence case {n} LSE")


def pin_lse_recompute(O):
    """P recomputed from the saved LSE, P = exp(scale * S - LSE), has unit row sums
    and reproduces O = P V (the relation the backward pass relies on)."""
    B, N, H, d = 1, 48, 2, 32
    q, k, v = dense_inputs(B, N, N, H, H, d, seed=40)
    scale = 1.0 / math.sqrt(d)
    o, lse = O.attention(q, k, v, scale, True)
    qq, kk, vv = _np(q), _np(k), _np(v)
    for h in range(H):
        S = scale * qq[0, :, h] @ kk[0, :, h].T
        S = np.where(_bottom_right_mask(N, N).numpy(), S, -np.inf)
        P = np.exp(S - lse[0, h][:, None])
        _close(P.sum(axis=1), np.ones(N), 1e-12, "recomputed P row sums")
        _close(P @ vv[0, :, h], o[0, :, h], 1e-12, "recomputed O")


def pin_library_fp16(O):
    """fp16 inputs: the same library cross-check (torch converts fp16 to float64)."""
    for n, (B, Nq, Nk, Hq, Hkv, d, causal) in enumerate(LIB_CASES[:3]):
        q, k, v = dense_inputs(B, Nq, Nk, Hq, Hkv, d, seed=60 + n, dtype=torch.float16)
        scale = 1.0 / math.sqrt(d)
        o, lse = O.attention(q, k, v, scale, causal)
        o_ref, lse_ref = _library_attention(q, k, v, scale, causal)
        _close(o, o_ref, 1e-11, f"fp16 O vs torch SDPA case {n}")
        _close(lse, lse_ref, 1e-11, f"fp16 LSE vs torch logsumexp case {n}")


def pin_fp16_values(O):
    """One visible key (causal row 0) built from special binary16 values -- normal,
    subnormal, largest finite, negative: O = v_0 exactly and LSE = scale q_0 . k_0, with
    the values converted by torch."""
    vals = [1.0, -2.0, 65504.0, 2.0 ** -24, 0.333251953125, -6.103515625e-05, 1.5, -0.0]
    v0 = torch.tensor(vals, dtype=torch.float16)
    q0 = torch.tensor([0.5, -1.0, 2.0 ** -14, 3.0, 0.0, 1.0, -0.25, 2.0], dtype=torch.float16)
    k0 = torch.tensor([1.0, 0.5, 1024.0, -0.125, 7.0, 2.0 ** -10, 4.0, -1.5], dtype=torch.float16)
    q = torch.zeros((1, 2, 1, 8), dtype=torch.float16)
    k = torch.zeros((1, 2, 1, 8), dtype=torch.float16)
    v = torch.zeros((1, 2, 1, 8), dtype=torch.float16)
    q[0, 0, 0], k[0, 0, 0], v[0, 0, 0] = q0, k0, v0
    o, lse = O.attention(q, k, v, 0.5, True)
    _close(o[0, 0, 0], v0.double().numpy(), 0.0, "fp16 single-key O")
    _close(lse[0, 0, 0], 0.5 * float((q0.double() * k0.double()).sum()), 1e-12,
           "fp16 single-key LSE")


# --------------------------------------------------------------------------
# score modifiers: sliding window, softcap, ALiBi ("flash-attention", capabilities table:
# causal / sliding window / ALiBi / softcap).  The pages name these and give no formulas;
# the readings pinned here are: with pos = i + Nk - Nq, key j is visible when
# pos - wl <= j <= pos + wr (negative bound = unbounded); the scaled score z becomes
# c * tanh(z / c) under a softcap c; ALiBi then adds -slope * |pos - j|.

def _visible_count(pos, Nk, wl, wr):
    lo = 0 if wl < 0 else max(pos - wl, 0)
    hi = Nk - 1 if wr < 0 else min(pos + wr, Nk - 1)
    return lo, max(hi - lo + 1, 0)


def pin_window_uniform(O):
    """Q = 0 under a window: O is the mean of the visible V rows and LSE = ln(#visible);
    rows whose window holds no key give O = 0, LSE = -inf."""
    for (Nq, Nk, wl, wr) in [(30, 30, 4, 0), (30, 30, 3, 5), (12, 40, 7, 2), (40, 12, 0, 3),
                             (25, 25, 0, 0), (20, 33, -1, 6), (20, 33, 9, -1)]:
        H, d = 2, 16
        _, k, v = dense_inputs(1, Nq, Nk, H, H, d, seed=200 + Nq + wl)
        q = torch.zeros((1, Nq, H, d), dtype=torch.bfloat16)
        o, lse = O.attention(q, k, v, 0.5, False, window=(wl, wr))
        vv = _np(v)
        for i in range(Nq):
            lo, n = _visible_count(i + Nk - Nq, Nk, wl, wr)
            for h in range(H):
                if n == 0:
                    assert np.all(o[0, i, h] == 0.0) and lse[0, h, i] == -np.inf, "empty window"
                    continue
                _close(o[0, i, h], vv[0, lo:lo + n, h].mean(axis=0), 1e-13, "window mean O")
                _close(lse[0, h, i], math.log(n), 1e-13, "window LSE")


def pin_window_diagonal(O):
    """Window (0, 0): each row sees only the key at its own position, so O = v_pos and
    LSE = scale * q_i . k_pos."""
    B, Nq, Nk, H, d = 1, 10, 14, 2, 16
    q, k, v = dense_inputs(B, Nq, Nk, H, H, d, seed=210)
    o, lse = O.attention(q, k, v, 0.4, False, window=(0, 0))
    qq, kk, vv = _np(q), _np(k), _np(v)
    for i in range(Nq):
        pos = i + Nk - Nq
        for h in range(H):
            _close(o[0, i, h], vv[0, pos, h], 1e-14, "diagonal O")
            _close(lse[0, h, i], 0.4 * float(np.dot(qq[0, i, h], kk[0, pos, h])), 1e-12,
                   "diagonal LSE")


def pin_window_library(O):
    """Random inputs under a band mask: torch SDPA (float64) with the boolean mask of the
    visible keys; windows that cover everything reduce to the unmasked / causal results."""
    for n, (Nq, Nk, wl, wr) in enumerate([(33, 33, 5, 2), (20, 45, 10, 0), (45, 20, 3, 4),
                                          (64, 64, 0, 7)]):
        H, d = 2, 32
        q, k, v = dense_inputs(1, Nq, Nk, H, H, d, seed=220 + n)
        o, lse = O.attention(q, k, v, 0.2, False, window=(wl, wr))
        pos = torch.arange(Nq)[:, None] + (Nk - Nq)
        j = torch.arange(Nk)[None, :]
        band = (j >= pos - wl) & (j <= pos + wr)
        qq, kk, vv = (_f64(t).permute(0, 2, 1, 3) for t in (q, k, v))
        scores = (qq @ kk.transpose(-1, -2) * 0.2).masked_fill(~band, float("-inf"))
        lse_ref = torch.logsumexp(scores, dim=-1)
        rows = band.any(dim=1)
        o_ref = F.scaled_dot_product_attention(qq[:, :, rows], kk, vv, attn_mask=band[rows],
                                               scale=0.2)
        _close(o[0][rows.numpy()], o_ref.permute(0, 2, 1, 3)[0].numpy(), 1e-12, "band O")
        _close(lse, lse_ref.numpy(), 1e-12, "band LSE")
    q, k, v = dense_inputs(1, 30, 30, 2, 2, 16, seed=230)
    for causal, win in [(False, (30, 30)), (True, (-1, -1)), (False, (-1, 0)), (False, (99, 0))]:
        o1, l1 = O.attention(q, k, v, 0.3, causal, window=win)
        o2, l2 = O.attention(q, k, v, 0.3, causal or win[1] == 0)
        _close(o1, o2, 0.0, f"window {win} vs plain O")
        _close(l1, l2, 0.0, f"window {win} vs plain LSE")


def pin_softcap_limits(O):
    """Softcap: Q = 0 keeps every score at 0 (uniform); a very large cap changes nothing
    measurable; keys with scores far above the cap all saturate at the cap, so they share
    the probability equally: LSE = log(m e^c + (n - m)) with the other keys at score 0."""
    _, k, v = dense_inputs(1, 9, 9, 1, 1, 16, seed=240)
    q0 = torch.zeros((1, 9, 1, 16), dtype=torch.bfloat16)
    _, l0 = O.attention(q0, k, v, 0.5, False, softcap=3.0)
    _close(l0, np.full((1, 1, 9), math.log(9)), 1e-13, "softcap uniform LSE")
    q, k, v = dense_inputs(1, 17, 23, 2, 2, 16, seed=241)
    o1, l1 = O.attention(q, k, v, 0.25, True, softcap=1e6)
    o2, l2 = O.attention(q, k, v, 0.25, True)
    _close(o1, o2, 1e-9, "large softcap O")
    _close(l1, l2, 1e-9, "large softcap LSE")
    # keys 0..2 along +e0 with huge scores, keys 3..7 orthogonal (score 0)
    n, m, cap = 8, 3, 2.5
    q = torch.zeros((1, 1, 1, 8), dtype=torch.bfloat16)
    k = torch.zeros((1, n, 1, 8), dtype=torch.bfloat16)
    v = torch.zeros((1, n, 1, 8), dtype=torch.bfloat16)
    q[0, 0, 0, 0] = 64.0
    for j in range(m):
        k[0, j, 0, 0] = 32.0 * (j + 1)
    for j in range(m, n):
        k[0, j, 0, 1 + (j - m) % 7] = 1.0
    for j in range(n):
        v[0, j, 0, j % 8] = 1.0
    o, lse = O.attention(q, k, v, 1.0, False, softcap=cap)
    z = m * math.exp(cap) + (n - m)
    _close(lse[0, 0, 0], math.log(z), 1e-12, "saturated softcap LSE")
    p_hi, p_lo = math.exp(cap) / z, 1.0 / z
    _close(o[0, 0, 0], np.array([p_hi if j < m else p_lo for j in range(n)]), 1e-12,
           "saturated softcap O")


def _alibi_geometric(pos, lo, hi, a):
    """sum_{j=lo}^{hi-1} e^{-a |pos - j|} by geometric series (lo <= pos < hi assumed)."""
    left = pos - lo            # keys below pos: distances 1..left
    right = hi - 1 - pos       # keys above pos: distances 1..right
    r = math.exp(-a)
    g = lambda n: r * (1.0 - r ** n) / (1.0 - r) if n > 0 else 0.0
    return 1.0 + g(left) + g(right)


def pin_alibi_geometric(O):
    """Q = 0 with ALiBi: P_j = e^{-a |pos - j|} / Z with Z a two-sided geometric sum, so with
    one-hot V rows O reproduces P; per-(batch, head) slopes read with their batch stride."""
    B, Nq, Nk, H = 2, 6, 8, 3
    d = 16
    slopes = np.array([[0.5, 0.25, 1.0], [0.125, 2.0, 0.75]], np.float32)
    q = torch.zeros((B, Nq, H, d), dtype=torch.bfloat16)
    k = bf16_normal((B, Nk, H, d), seed=250)
    v = torch.zeros((B, Nk, H, d), dtype=torch.bfloat16)
    for j in range(Nk):
        v[:, j, :, j] = 1.0
    for causal in (False, True):
        o, lse = O.attention(q, k, v, 0.3, causal, alibi_slopes=slopes)
        for b in range(B):
            for h in range(H):
                a = float(slopes[b, h])
                for i in range(Nq):
                    pos = i + Nk - Nq
                    hi = pos + 1 if causal else Nk
                    zsum = _alibi_geometric(pos, 0, hi, a)
                    _close(lse[b, h, i], math.log(zsum), 1e-13, "ALiBi geometric LSE")
                    p = np.array([math.exp(-a * abs(pos - j)) / zsum if j < hi else 0.0
                                  for j in range(Nk)])
                    _close(o[b, i, h, :Nk], p, 1e-13, "ALiBi geometric P")
    o1, l1 = O.attention(q, k, v, 0.3, True, alibi_slopes=np.zeros(H, np.float32))
    o2, l2 = O.attention(q, k, v, 0.3, True)
    _close(o1, o2, 0.0, "zero-slope ALiBi O")
    _close(l1, l2, 0.0, "zero-slope ALiBi LSE")


def pin_alibi_library(O):
    """Random inputs with ALiBi: torch SDPA (float64) with the additive bias
    -a |pos - j| as a float mask, causal and not, Nq != Nk, GQA."""
    for n, (Nq, Nk, causal) in enumerate([(40, 40, True), (25, 50, False), (50, 30, True)]):
        Hq, Hkv, d = 4, 2, 32
        q, k, v = dense_inputs(1, Nq, Nk, Hq, Hkv, d, seed=260 + n)
        slopes = (2.0 ** -np.arange(1, Hq + 1)).astype(np.float32)
        o, lse = O.attention(q, k, v, 0.2, causal, alibi_slopes=slopes)
        pos = torch.arange(Nq)[:, None] + (Nk - Nq)
        j = torch.arange(Nk)[None, :]
        bias = -torch.tensor(slopes, dtype=torch.float64)[:, None, None] * (pos - j).abs()
        if causal:
            bias = bias.masked_fill(~(j <= pos), float("-inf"))
        qq = _f64(q).permute(0, 2, 1, 3)
        kk = _f64(k).permute(0, 2, 1, 3).repeat_interleave(Hq // Hkv, dim=1)
        vv = _f64(v).permute(0, 2, 1, 3).repeat_interleave(Hq // Hkv, dim=1)
        lse_ref = torch.logsumexp(qq @ kk.transpose(-1, -2) * 0.2 + bias, dim=-1)
        rows = torch.isfinite(lse_ref[0, 0])
        o_ref = F.scaled_dot_product_attention(qq[:, :, rows], kk, vv,
                                               attn_mask=bias[None][:, :, rows], scale=0.2)
        _close(o[0][rows.numpy()], o_ref.permute(0, 2, 1, 3)[0].numpy(), 1e-12, "ALiBi O")
        _close(lse, lse_ref.numpy(), 1e-12, "ALiBi LSE")


def pin_mod_bruteforce(O):
    """All three modifiers at once on tiny rows, brute force in plain Python: window,
    then softcap on the scaled score, then the ALiBi bias, then the softmax."""
    B, Nq, Nk, H, d = 1, 5, 7, 2, 4
    q, k, v = dense_inputs(B, Nq, Nk, H, H, d, seed=270)
    qq, kk, vv = _np(q), _np(k), _np(v)
    scale, cap, wl, wr = 0.9, 1.5, 3, 1
    slopes = np.array([0.3, 0.7], np.float32)
    o, lse = O.attention(q, k, v, scale, False, window=(wl, wr), softcap=cap,
                         alibi_slopes=slopes)
    for i in range(Nq):
        pos = i + Nk - Nq
        for h in range(H):
            zs, vs = [], []
            for j in range(Nk):
                if not (pos - wl <= j <= pos + wr):
                    continue
                zdot = sum(float(qq[0, i, h, c]) * float(kk[0, j, h, c]) for c in range(d))
                z = cap * math.tanh(scale * zdot / cap) - float(slopes[h]) * abs(pos - j)
                zs.append(z)
                vs.append(vv[0, j, h])
            mx = max(zs)
            w = [math.exp(z - mx) for z in zs]
            tot = sum(w)
            _close(lse[0, h, i], mx + math.log(tot), 1e-12, "brute-force LSE")
            _close(o[0, i, h], sum(wj * vj for wj, vj in zip(w, vs)) / tot, 1e-12,
                   "brute-force O")


def pin_mod_paths(O):
    """Decode with modifiers equals dense attention of one query at the last position of
    a sequence of cache_seqlens[b] keys; varlen with modifiers equals per-sequence dense."""
    B, Lmax, Hq, Hkv, d = 3, 40, 4, 2, 16
    lens = [40, 1, 23]
    q = bf16_normal((B, 1, Hq, d), seed=280)
    kc = bf16_normal((B, Lmax, Hkv, d), seed=281)
    vc = bf16_normal((B, Lmax, Hkv, d), seed=282)
    slopes = np.array([[0.1, 0.2, 0.3, 0.4], [0.5, 0.6, 0.7, 0.8], [0.05, 0.0, 1.0, 0.25]],
                      np.float32)
    for kw in [dict(window=(5, -1)), dict(softcap=2.0), dict(alibi_slopes=slopes),
               dict(window=(17, 0), softcap=1.0, alibi_slopes=slopes)]:
        o, lse = O.attention_kvcache(q, kc, vc, lens, 0.25, **kw)
        for b, n in enumerate(lens):
            kwb = dict(kw)
            if "alibi_slopes" in kw:
                kwb["alibi_slopes"] = slopes[b]
            ob, lb = O.attention(q[b:b + 1].contiguous(), kc[b:b + 1, :n].contiguous(),
                                 vc[b:b + 1, :n].contiguous(), 0.25, False, **kwb)
            _close(o[b], ob[0, 0], 0.0, f"decode {kw.keys()} batch {b} O")
            _close(lse[b], lb[0, :, 0], 0.0, f"decode {kw.keys()} batch {b} LSE")
    sq, sk = [5, 0, 19, 33], [7, 3, 19, 20]
    q, k, v, cu_q, cu_k = varlen_inputs(sq, sk, 4, 2, 16, seed=283)
    for causal, kw in [(False, dict(window=(4, 2))), (True, dict(softcap=1.5)),
                       (True, dict(alibi_slopes=slopes[0], window=(6, -1)))]:
        o, lse = O.attention_varlen(q, k, v, cu_q, cu_k, 0.25, causal, **kw)
        for b in range(len(sq)):
            a, e = int(cu_q[b]), int(cu_q[b + 1])
            ka, ke = int(cu_k[b]), int(cu_k[b + 1])
            if e == a:
                continue
            ob, lb = O.attention(q[a:e].unsqueeze(0).contiguous(),
                                 k[ka:ke].unsqueeze(0).contiguous(),
                                 v[ka:ke].unsqueeze(0).contiguous(), 0.25, causal, **kw)
            _close(o[a:e], ob[0], 0.0, f"varlen mod seq {b} O")
            _close(lse[:, a:e], lb[0], 0.0, f"varlen mod seq {b} LSE")


# --------------------------------------------------------------------------
# KV-cache extras: rounding to the cache type, rotary embedding, in-place append, paged
# caches ("flash-attention", section 1 and capabilities table, KV cache row).  Readings:
# the new key and value of a decode step go to logical row cache_seqlens[b]; rotary turns
# dimension pairs (i, i + r/2) (or (2i, 2i+1) interleaved) of q and the new key by the
# table angle of that same position; results are rounded once to the element type.

def _spacing(x, dtype):
    """One ulp of the 16-bit type at |x| (normal range)."""
    bits = 8 if dtype == torch.bfloat16 else 11
    ax = np.abs(x)
    return np.exp2(np.floor(np.log2(np.where(ax > 0, ax, 1.0))) - (bits - 1))


def _to64(bits, dtype):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(dtype).double().numpy()


def _rope_tables(P, half):
    inv = 10000.0 ** (-np.arange(half) / half)
    ang = np.arange(P)[:, None] * inv[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


def pin_round16_library(O):
    """fp32 -> bf16 / fp16 rounding equals torch's conversion (round to nearest even),
    including ties, subnormals and overflow to inf."""
    rng = np.random.default_rng(5)
    x = (rng.normal(size=50000) * 10.0 ** rng.integers(-9, 6, size=50000)).astype(np.float32)
    special = np.array([65504, 65519.99, 65520, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26,
                        2.0 ** -14, -0.0, 1e30, np.inf, -np.inf, 1 + 2.0 ** -8,
                        1 + 3 * 2.0 ** -8, 1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11], np.float32)
    x = np.concatenate([x, special])
    for elem, dt in ((0, torch.bfloat16), (1, torch.float16)):
        ref = torch.from_numpy(x).to(dt).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(O.round16(x, elem), ref), f"round16 elem {elem} vs torch"


def pin_rotary(O):
    """Rotary: angle 0 is the identity and a quarter turn maps (x_a, x_b) to (-x_b, x_a)
    exactly; random angles agree with the rotation evaluated in float64 to one ulp of the
    element type (fixes the sign, the pairing and the table row); interleaved pairs equal
    half-split pairs after the matching permutation of dimensions; dimensions past
    rotary_dim are copied."""
    rd, half, d = 48, 24, 64
    cos, sin = _rope_tables(128, half)
    for elem, dt in ((0, torch.bfloat16), (1, torch.float16)):
        x = bf16_normal((6, 4, d), seed=300 + elem, dtype=dt)
        xb = x.view(torch.int16).numpy().view(np.uint16)
        x64 = x.double().numpy()
        pos = np.repeat(np.array([0, 1, 5, 17, 100, 3], np.int32)[:, None], 4, axis=1)
        y = O.rotary(x, pos, cos, sin)
        assert np.array_equal(y[0], xb[0]), "position 0 is not the identity"
        assert np.array_equal(y[..., rd:], xb[..., rd:]), "dimensions past rotary_dim changed"
        cq, sq = np.zeros((1, half), np.float32), np.ones((1, half), np.float32)
        yq = _to64(O.rotary(x, np.zeros((6, 4), np.int32), cq, sq), dt)
        assert np.array_equal(yq[..., :half], -x64[..., half:rd]), "quarter turn, first half"
        assert np.array_equal(yq[..., half:rd], x64[..., :half]), "quarter turn, second half"
        c, s_ = cos[pos].astype(np.float64), sin[pos].astype(np.float64)
        xa, xc = x64[..., :half], x64[..., half:rd]
        exact = np.concatenate([xa * c - xc * s_, xa * s_ + xc * c], axis=-1)
        got = _to64(y, dt)[..., :rd]
        assert np.all(np.abs(got - exact) <= _spacing(exact, dt)), "rotation vs float64"
        perm = np.concatenate([np.arange(0, rd, 2), np.arange(1, rd, 2), np.arange(rd, d)])
        xi = x[..., torch.from_numpy(np.argsort(perm))].contiguous()  # interleaved layout
        yi = O.rotary(xi, pos, cos, sin, interleaved=True)
        assert np.array_equal(yi[..., perm], y), "interleaved vs half-split pairs"


def _kv_case(seed, B=3, Lmax=40, Hq=4, Hkv=2, d=16):
    q = bf16_normal((B, 1, Hq, d), seed=seed)
    kc = bf16_normal((B, Lmax, Hkv, d), seed=seed + 1)
    vc = bf16_normal((B, Lmax, Hkv, d), seed=seed + 2)
    kn = bf16_normal((B, 1, Hkv, d), seed=seed + 3)
    vn = bf16_normal((B, 1, Hkv, d), seed=seed + 4)
    return q, kc, vc, kn, vn


def pin_kv_append(O):
    """Append: the caches change only at row cache_seqlens[b], which holds the new key and
    value; the query then sees that row (decode over length + 1).  Rotary turns the new key
    and the query by the angle of position cache_seqlens[b]: with tables that turn only
    that row by a quarter, both come out as exact quarter turns."""
    q, kc, vc, kn, vn = _kv_case(310)
    lens = [0, 17, 39]
    o, lse, kc2, vc2 = O.kvcache_step(q, kc, vc, lens, 0.25, k_new=kn, v_new=vn)
    ke, ve = kc.clone(), vc.clone()
    for b, n in enumerate(lens):
        ke[b, n], ve[b, n] = kn[b, 0], vn[b, 0]
    bits = lambda t: t.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(kc2, bits(ke)) and np.array_equal(vc2, bits(ve)), "appended caches"
    o_ref, l_ref = O.attention_kvcache(q, ke, ve, [n + 1 for n in lens], 0.25)
    _close(o, o_ref, 0.0, "append O")
    _close(lse, l_ref, 0.0, "append LSE")
    half = 8
    cos, sin = np.ones((64, half), np.float32), np.zeros((64, half), np.float32)
    for n in lens:
        cos[n], sin[n] = 0.0, 1.0
    o, lse, kc3, _ = O.kvcache_step(q, kc, vc, lens, 0.25, k_new=kn, v_new=vn, rotary_cos=cos,
                                    rotary_sin=sin)
    quarter = lambda t: torch.cat([-t[..., half:], t[..., :half]], dim=-1)
    kq = ke.clone()
    for b, n in enumerate(lens):
        kq[b, n] = quarter(kn[b, 0])
    assert np.array_equal(kc3, bits(kq)), "rotated key not a quarter turn at its position"
    o_ref, l_ref = O.attention_kvcache(quarter(q).contiguous(), kq, ve, [n + 1 for n in lens],
                                       0.25)
    _close(o, o_ref, 0.0, "rotary append O")
    _close(lse, l_ref, 0.0, "rotary append LSE")


def pin_kv_paged(O):
    """A paged cache (pages of 8 rows in a shuffled pool, block table per sequence) gives
    the same step as the contiguous cache it holds, before and after an append, with the
    score modifiers too; the appended row lands in the page the table names."""
    q, kc, vc, kn, vn = _kv_case(320)
    B, Lmax, Hkv, d = kc.shape
    P, nblk = 8, Lmax // 8
    rng = np.random.default_rng(321)
    order = rng.permutation(B * nblk + 3)[:B * nblk].reshape(B, nblk).astype(np.int32)
    kp = torch.full((B * nblk + 3, P, Hkv, d), float("nan"), dtype=torch.bfloat16)
    vp = kp.clone()
    for b in range(B):
        for j in range(nblk):
            kp[order[b, j]] = kc[b, j * P:(j + 1) * P]
            vp[order[b, j]] = vc[b, j * P:(j + 1) * P]
    lens = [0, 23, 39]
    cos, sin = _rope_tables(64, 8)
    for kw in [dict(), dict(window=(9, -1), softcap=3.0)]:
        o1, l1, k1, v1 = O.kvcache_step(q, kc, vc, lens, 0.3, k_new=kn, v_new=vn,
                                        rotary_cos=cos, rotary_sin=sin, **kw)
        o2, l2, k2, v2 = O.kvcache_step(q, kp, vp, lens, 0.3, k_new=kn, v_new=vn,
                                        rotary_cos=cos, rotary_sin=sin, block_table=order, **kw)
        _close(o2, o1, 0.0, "paged O")
        _close(l2, l1, 0.0, "paged LSE")
        for b in range(B):
            for j in range(nblk):
                assert np.array_equal(k2[order[b, j]], k1[b, j * P:(j + 1) * P]), "paged keys"
                assert np.array_equal(v2[order[b, j]], v1[b, j * P:(j + 1) * P]), "paged values"
        o3, l3, _, _ = O.kvcache_step(q, kp, vp, lens, 0.3, block_table=order, **kw)
        o4, l4 = O.attention_kvcache(q, kc, vc, lens, 0.3, **kw)
        _close(o3, o4, 0.0, "paged without append O")
        _close(l3, l4, 0.0, "paged without append LSE")


# --------------------------------------------------------------------------
# Backward pass: the chain rule through O = P V, P = softmax(scale Q K^T).

BWD_CASES = [
    # B, Nq, Nk, Hq, Hkv, d, causal
    (1, 33, 33, 2, 2, 16, False),
    (2, 40, 40, 4, 2, 32, True),
    (1, 20, 45, 4, 1, 16, True),   # Nq < Nk, bottom-right causal
    (1, 45, 20, 2, 2, 16, True),   # Nq > Nk: leading rows see no key
    (1, 130, 130, 1, 1, 64, True),
]


def pin_bwd_library(O):
    """float64 torch autograd through scaled_dot_product_attention (a library routine the
    oracle does not call), GQA as repeated heads, bottom-right causal mask."""
    for n, (B, Nq, Nk, Hq, Hkv, d, causal) in enumerate(BWD_CASES):
        q, k, v = dense_inputs(B, Nq, Nk, Hq, Hkv, d, seed=400 + n)
        do = bf16_normal((B, Nq, Hq, d), seed=410 + n)
        scale = 1.0 / math.sqrt(d)
        dq, dk, dv, lse, D = O.attention_bwd(q, k, v, do, scale, causal)
        G = Hq // Hkv
        qq = _f64(q).permute(0, 2, 1, 3).requires_grad_()
        kk = _f64(k).permute(0, 2, 1, 3).requires_grad_()
        vv = _f64(v).permute(0, 2, 1, 3).requires_grad_()
        mask = _bottom_right_mask(Nq, Nk) if causal else None
        rows = mask.any(dim=1) if causal else torch.ones(Nq, dtype=torch.bool)
        out = F.scaled_dot_product_attention(qq[:, :, rows], kk.repeat_interleave(G, dim=1),
                                             vv.repeat_interleave(G, dim=1),
                                             attn_mask=None if mask is None else mask[rows],
                                             scale=scale)
        out.backward(_f64(do).permute(0, 2, 1, 3)[:, :, rows])
        _close(dq, qq.grad.permute(0, 2, 1, 3).numpy(), 1e-11, f"dQ vs autograd case {n}")
        _close(dk, kk.grad.permute(0, 2, 1, 3).numpy(), 1e-11, f"dK vs autograd case {n}")
        _close(dv, vv.grad.permute(0, 2, 1, 3).numpy(), 1e-11, f"dV vs autograd case {n}")
        o_f, l_f = O.attention(q, k, v, scale, causal)
        _close(lse, l_f, 1e-12, f"backward LSE vs forward case {n}")
        D_ref = np.einsum("bnhd,bnhd->bhn", _np(do), o_f)
        _close(D, D_ref, 1e-11, f"D = rowsum(dO * O) case {n}")


def pin_bwd_closed_forms(O):
    """sum_j dV_j = sum of dO over rows that see a key (each row of P sums to one);
    constant V rows give dP_ij = D_i, so dS = 0 and dQ = dK = 0; causal row 0 sees one key,
    so its dQ is 0; shifting every key by one vector (an exact bf16 shift) changes no
    gradient; GQA gradients equal MHA with repeated K/V heads, dK and dV summed per group."""
    B, N, Hq, Hkv, d = 1, 30, 4, 2, 16
    q, k, v = dense_inputs(B, N, N, Hq, Hkv, d, seed=420)
    do = bf16_normal((B, N, Hq, d), seed=421)
    for causal in (False, True):
        dq, dk, dv, _, _ = O.attention_bwd(q, k, v, do, 0.3, causal)
        G = Hq // Hkv
        tot = _np(do).reshape(B, N, Hkv, G, d).sum(axis=(1, 3))
        _close(dv.sum(axis=1), tot, 1e-11, "sum of dV")
        if causal:
            _close(dq[:, 0], np.zeros((B, Hq, d)), 1e-14, "causal row 0 dQ")
    c = bf16_normal((1, 1, Hkv, d), seed=422)
    vc = c.expand(B, N, Hkv, d).contiguous()
    dq, dk, dv, _, _ = O.attention_bwd(q, k, vc, do, 0.3, True)
    _close(dq, np.zeros_like(dq), 1e-13, "constant V gives dQ = 0")
    _close(dk, np.zeros_like(dk), 1e-13, "constant V gives dK = 0")
    gen = torch.Generator().manual_seed(423)
    ki = torch.randint(-8, 9, (B, N, Hkv, d), generator=gen).to(torch.bfloat16)
    u = torch.randint(-8, 9, (1, 1, Hkv, d), generator=gen).to(torch.bfloat16)
    ks = (ki.float() + u.float()).to(torch.bfloat16)
    assert torch.equal(ks.float(), ki.float() + u.float()), "setup: the shift must be exact"
    g1 = O.attention_bwd(q, ki, v, do, 0.05, True)
    g2 = O.attention_bwd(q, ks, v, do, 0.05, True)
    for a, b_, name in zip(g1[:3], g2[:3], ("dQ", "dK", "dV")):
        _close(a, b_, 1e-11, f"{name} under a key shift")
    g1 = O.attention_bwd(q, k, v, do, 0.3, True)
    kr = k.repeat_interleave(Hq // Hkv, dim=2).contiguous()
    vr = v.repeat_interleave(Hq // Hkv, dim=2).contiguous()
    dq2, dk2, dv2, _, _ = O.attention_bwd(q, kr, vr, do, 0.3, True)
    _close(g1[0], dq2, 1e-12, "GQA dQ vs MHA")
    _close(g1[1], dk2.reshape(B, N, Hkv, Hq // Hkv, d).sum(axis=3), 1e-12, "GQA dK vs MHA")
    _close(g1[2], dv2.reshape(B, N, Hkv, Hq // Hkv, d).sum(axis=3), 1e-12, "GQA dV vs MHA")



def pin_bwd_modifiers(O):
    """Backward with the score modifiers: float64 torch autograd through the explicit
    attention (z = scale q.k, softcap c tanh(z / c), ALiBi -slope |pos - j|, window mask,
    softmax, P V); every row sees at least one key."""
    cases = [
        dict(Nq=33, Nk=33, causal=False, window=(5, 2)),
        dict(Nq=30, Nk=30, causal=True, softcap=2.0),
        dict(Nq=20, Nk=45, causal=True, alibi=True),
        dict(Nq=40, Nk=40, causal=False, window=(9, 3), softcap=1.5, alibi=True),
    ]
    for n, c in enumerate(cases):
        B, Hq, Hkv, d = 2, 4, 2, 16
        Nq, Nk = c["Nq"], c["Nk"]
        q, k, v = dense_inputs(B, Nq, Nk, Hq, Hkv, d, seed=430 + n)
        do = bf16_normal((B, Nq, Hq, d), seed=440 + n)
        scale, cap = 0.35, c.get("softcap", 0.0)
        slopes = np.array([[0.3, 0.1, 0.7, 0.05], [0.2, 0.5, 0.01, 0.9]], np.float32) \
            if c.get("alibi") else None
        wl, wr = c.get("window", (-1, -1))
        dq, dk, dv, _, _ = O.attention_bwd(q, k, v, do, scale, c["causal"], window=(wl, wr),
                                           softcap=cap, alibi_slopes=slopes)
        G = Hq // Hkv
        qq = _f64(q).permute(0, 2, 1, 3).requires_grad_()
        kk = _f64(k).permute(0, 2, 1, 3).requires_grad_()
        vv = _f64(v).permute(0, 2, 1, 3).requires_grad_()
        z = torch.matmul(qq, kk.repeat_interleave(G, 1).transpose(-1, -2)) * scale
        if cap > 0:
            z = cap * torch.tanh(z / cap)
        pos = torch.arange(Nq)[:, None] + (Nk - Nq)
        j = torch.arange(Nk)[None, :]
        if slopes is not None:
            z = z - torch.tensor(slopes, dtype=torch.float64)[:, :, None, None] * \
                (pos - j).abs().double()
        vis = torch.ones(Nq, Nk, dtype=torch.bool)
        if wl >= 0:
            vis &= j >= pos - wl
        if wr >= 0 or c["causal"]:
            vis &= j <= pos + (0 if c["causal"] else wr)
        assert bool(vis.any(dim=1).all()), "setup: every row must see a key"
        p = torch.softmax(z.masked_fill(~vis, float("-inf")), dim=-1)
        torch.matmul(p, vv.repeat_interleave(G, 1)).backward(_f64(do).permute(0, 2, 1, 3))
        _close(dq, qq.grad.permute(0, 2, 1, 3).numpy(), 1e-11, f"modifier dQ case {n}")
        _close(dk, kk.grad.permute(0, 2, 1, 3).numpy(), 1e-11, f"modifier dK case {n}")
        _close(dv, vv.grad.permute(0, 2, 1, 3).numpy(), 1e-11, f"modifier dV case {n}")


def _e4m3_codes(shape, seed):
    """Random E4M3 codes with exponent fields 0..8 (subnormals up to 3.75 in magnitude, so
    that the scores stay small enough for an absolute 1e-12 comparison)."""
    g = np.random.default_rng(seed)
    sign = g.integers(0, 2, size=shape) << 7
    exp = g.integers(0, 9, size=shape) << 3
    man = g.integers(0, 8, size=shape)
    return (sign | exp | man).astype(np.uint8)


def pin_e4m3_decode(O):
    """The E4M3 decoder against torch.float8_e4m3fn for all 256 codes, and the exact
    re-encoding of every finite value as bf16."""
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = O.e4m3_values()
    assert np.array_equal(np.isnan(got), np.isnan(ref)), "E4M3 NaN codes"
    fin = ~np.isnan(ref)
    assert np.array_equal(got[fin], ref[fin]), "E4M3 values differ from torch.float8_e4m3fn"
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x38] == 1.0
    bits = O.e4m3_to_bf16_bits(np.arange(256, dtype=np.uint8)[fin])
    back = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64)
    assert np.array_equal(back.numpy(), ref[fin]), "bf16 re-encoding not exact"


def pin_fp8_bruteforce(O):
    """FP8 attention against the definition written out in torch float64 on values decoded
    by torch: scores scale * (dq q).(dk k), bottom-right causal mask, softmax, P (dv V)."""
    for n, (B, Nq, Nk, Hq, Hkv, d, causal) in enumerate(
            [(2, 7, 9, 4, 2, 16, True), (1, 11, 5, 2, 1, 8, False), (2, 9, 9, 6, 3, 32, True)]):
        q, k, v = (_e4m3_codes(s, 600 + 3 * n + i) for i, s in enumerate(
            [(B, Nq, Hq, d), (B, Nk, Hkv, d), (B, Nk, Hkv, d)]))
        g = np.random.default_rng(610 + n)
        dq, dk, dv = (g.uniform(0.02, 0.5, size=(B, Hkv)).astype(np.float32) for _ in range(3))
        scale = 0.3
        o, lse = O.attention_fp8(q, k, v, scale, causal, dq, dk, dv)
        val = lambda c: torch.from_numpy(c).view(torch.float8_e4m3fn).to(torch.float64)
        G = Hq // Hkv
        qq = val(q) * torch.from_numpy(dq.astype(np.float64)).repeat_interleave(G, 1)[:, None, :, None]
        kk = (val(k) * torch.from_numpy(dk.astype(np.float64))[:, None, :, None]).repeat_interleave(G, 2)
        vv = (val(v) * torch.from_numpy(dv.astype(np.float64))[:, None, :, None]).repeat_interleave(G, 2)
        z = torch.einsum("bihc,bjhc->bhij", qq, kk) * float(np.float32(scale))
        if causal:
            z = z.masked_fill(~_bottom_right_mask(Nq, Nk), float("-inf"))
        ref_lse = torch.logsumexp(z, dim=-1)
        ref_o = torch.einsum("bhij,bjhc->bihc", torch.softmax(z, dim=-1).nan_to_num(0.0), vv)
        _close(o, ref_o.numpy(), 1e-12, f"fp8 case {n} O")
        fin = torch.isfinite(ref_lse).numpy()
        _close(lse[fin], ref_lse.numpy()[fin], 1e-12, f"fp8 case {n} LSE")


def pin_fp8_kvcache_bruteforce(O):
    """Decode over E4M3 caches against the definition written out in torch float64 on
    values decoded by torch: for each sequence and query head, scores scale * q.(dk k) over
    the first cache_seqlens[b] rows of its kv head, softmax, P (dv V); the empty sequence
    gives O = 0 and LSE = -inf."""
    for n, (B, Lmax, Hq, Hkv, d, lens) in enumerate(
            [(3, 9, 4, 2, 16, [5, 9, 0]), (2, 12, 3, 3, 32, [1, 12]), (1, 7, 8, 1, 16, [7])]):
        k, v = (_e4m3_codes((B, Lmax, Hkv, d), 640 + 2 * n + i) for i in range(2))
        g = np.random.default_rng(650 + n)
        q = g.standard_normal((B, 1, Hq, d)).astype(np.float32)
        qbits = (q.view(np.uint32) >> 16).astype(np.uint16)  # truncated to bf16 bits
        dk, dv = (g.uniform(0.02, 0.5, size=(B, Hkv)).astype(np.float32) for _ in range(2))
        scale = 0.4
        o, lse = O.attention_kvcache_fp8(qbits, k, v, np.array(lens, np.int32), scale, dk, dv)
        val = lambda c: torch.from_numpy(c).view(torch.float8_e4m3fn).to(torch.float64)
        qq = torch.from_numpy((qbits.astype(np.uint32) << 16).view(np.float32).astype(np.float64))
        G = Hq // Hkv
        for b in range(B):
            for h in range(Hq):
                kv = h // G
                L = lens[b]
                if L == 0:
                    assert np.all(o[b, h] == 0.0) and lse[b, h] == -np.inf, "empty sequence"
                    continue
                kk = val(k)[b, :L, kv] * float(dk[b, kv])
                vv = val(v)[b, :L, kv] * float(dv[b, kv])
                z = (kk @ qq[b, 0, h]) * float(np.float32(scale))
                ref_lse = torch.logsumexp(z, 0)
                ref_o = torch.softmax(z, 0) @ vv
                _close(o[b, h], ref_o.numpy(), 1e-12, f"fp8 decode case {n} O b{b} h{h}")
                _close(np.array([lse[b, h]]), np.array([float(ref_lse)]), 1e-12,
                       f"fp8 decode case {n} LSE b{b} h{h}")


ALL_PINS = [pin_library, pin_library_fp16, pin_fp16_values, pin_uniform_scores, pin_single_key, pin_constant_v, pin_two_keys,
            pin_empty_rows, pin_hard_max, pin_probs, pin_shift, pin_permutation, pin_gqa,
            pin_varlen, pin_kvcache, pin_rows, pin_recurrence, pin_lse_recompute,
            pin_window_uniform, pin_window_diagonal, pin_window_library, pin_softcap_limits,
            pin_alibi_geometric, pin_alibi_library, pin_mod_bruteforce, pin_mod_paths,
            pin_round16_library, pin_rotary, pin_kv_append, pin_kv_paged, pin_bwd_library,
            pin_bwd_closed_forms, pin_bwd_modifiers, pin_e4m3_decode, pin_fp8_bruteforce,
            pin_fp8_kvcache_bruteforce]
