"""GPU parity of the FP8 forward (fa_fwd_fp8 and, over packed sequences, fa_fwd_varlen_fp8:
E4M3 Q, K, V with per-(batch, kv head) descale factors, bf16 O) and of the decode call over E4M3 caches (fa_fwd_kvcache_fp8)
against the fp64 oracle.

The pages fix no tolerance for FP8.  The bar is their own test criterion ("flash-attention",
section 5, tests): the kernel's O error is at most twice that of a PyTorch baseline in the
input precision (+1e-4) -- fp32 scores and softmax of the decoded inputs, P rounded to E4M3
for the P V product (the kernel's only 8-bit rounding besides the inputs), normalised by the
fp32 row sum -- both in the maximum and in the mean; the LSE, computed from unrounded scores
on both sides, within 1e-3.  The decode over E4M3 caches rounds nothing beyond its inputs,
so it takes the 16-bit decode bar (tests.parity_util)."""
import math

import numpy as np
import pytest
import torch

import oracle.oracle as ORACLE
from exact_attention_81_gb300 import FA_OK, fa_fwd_fp8, fa_fwd_varlen_fp8, get_last_device_error
from exact_attention_81_gb300.inputs import fp8_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _baseline(q, k, v, dq, dk, dv, scale, causal, window=(-1, -1), softcap=0.0):
    B, Nq, Hq, d = q.shape
    Nk, Hkv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    qf = q.cpu().float() * dq.cpu().repeat_interleave(G, 1)[:, None, :, None]
    kf = (k.cpu().float() * dk.cpu()[:, None, :, None]).repeat_interleave(G, 2)
    vf = (v.cpu().float() * dv.cpu()[:, None, :, None]).repeat_interleave(G, 2)
    s = torch.einsum("bihc,bjhc->bhij", qf, kf) * scale
    if softcap > 0:
        s = softcap * torch.tanh(s / softcap)
    pos = torch.arange(Nq)[:, None] + (Nk - Nq)
    j = torch.arange(Nk)[None, :]
    vis = torch.ones(Nq, Nk, dtype=torch.bool)
    wl, wr = window
    if causal:
        wr = 0
    if wl >= 0:
        vis &= j >= pos - wl
    if wr >= 0:
        vis &= j <= pos + wr
    s = s.masked_fill(~vis, float("-inf"))
    m = s.amax(dim=-1, keepdim=True).clamp_min(-1e30)
    p = torch.exp(s - m)
    l = p.sum(dim=-1, keepdim=True)
    p8 = p.to(torch.float8_e4m3fn).float()
    o = torch.einsum("bhij,bjhc->bihc", p8, vf) / l.permute(0, 2, 1, 3).clamp_min(1e-30)
    return o.double().numpy()


def _check(B, Nq, Nk, Hq, Hkv, d, causal, seed, what, descales=True, **mod):
    q, k, v, dq, dk, dv = fp8_inputs(B, Nq, Nk, Hq, Hkv, d, seed, device=DEV)
    if not descales:
        dq = dk = dv = torch.ones((B, Hkv), dtype=torch.float32, device=DEV)
    scale = float(np.float32(1 / math.sqrt(d)))
    o, lse = fa_fwd_fp8(q, k, v, causal=causal, scale=scale,
                        q_descale=dq if descales else None, k_descale=dk if descales else None,
                        v_descale=dv if descales else None, **mod)
    assert get_last_device_error() == FA_OK
    window = mod.get("window_size", (-1, -1))
    softcap = mod.get("softcap", 0.0)
    o_ref, lse_ref = ORACLE.attention_fp8(q.cpu(), k.cpu(), v.cpu(), scale, causal, dq.cpu(),
                                          dk.cpu(), dv.cpu(), window=window, softcap=softcap)
    base = _baseline(q, k, v, dq, dk, dv, scale, causal, window, softcap)
    g = o.double().cpu().numpy()
    assert np.all(np.isfinite(g)), f"{what}: non-finite O"
    e_gpu, e_base = np.abs(g - o_ref), np.abs(base - o_ref)
    assert e_gpu.max() <= 2 * e_base.max() + 1e-4, \
        f"{what}: max |dO| {e_gpu.max():.3e} > 2 x baseline {e_base.max():.3e}"
    assert e_gpu.mean() <= 2 * e_base.mean() + 1e-4, \
        f"{what}: mean |dO| {e_gpu.mean():.3e} > 2 x baseline {e_base.mean():.3e}"
    l = lse.double().cpu().numpy()
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(l), fin), f"{what}: LSE finiteness"
    assert np.abs(l[fin] - lse_ref[fin]).max(initial=0.0) <= 1e-3, f"{what}: LSE"
    return e_gpu.max(), e_base.max()


@pytest.mark.parametrize("case", [
    # B, Nq, Nk, Hq, Hkv, d, causal
    (1, 128, 128, 1, 1, 128, False),
    (2, 512, 512, 8, 2, 128, True),
    (2, 700, 700, 4, 4, 128, False),
    (1, 300, 900, 4, 1, 128, True),
    (1, 900, 300, 2, 2, 128, True),
    (2, 333, 517, 4, 2, 64, False),
    (1, 256, 256, 2, 1, 32, True),
])
def test_fp8(case):
    _check(*case, seed=sum(case[:6]) + 17, what=f"fp8 {case}")


def test_fp8_no_descales():
    _check(1, 400, 400, 4, 2, 128, True, seed=5, what="fp8 without descales", descales=False)


@pytest.mark.parametrize("mod", [dict(window_size=(256, 0)), dict(softcap=10.0),
                                 dict(window_size=(100, 30), softcap=5.0)])
def test_fp8_modifiers(mod):
    _check(2, 600, 600, 4, 2, 128, False, seed=23, what=f"fp8 {mod}", **mod)


def _varlen_fp8(sq, sk, Hq, Hkv, d, causal, seed, **mod):
    """Packed sequences through fa_fwd_varlen_fp8, each sequence checked under the bar of
    _check against the dense FP8 oracle of that sequence alone.  Returns the per-sequence
    inputs and outputs."""
    per = [fp8_inputs(1, nq, nk, Hq, Hkv, d, seed + b, device=DEV) for b, (nq, nk) in
           enumerate(zip(sq, sk))]
    q = torch.cat([t[0][0] for t in per]).contiguous()
    k = torch.cat([t[1][0] for t in per]).contiguous()
    v = torch.cat([t[2][0] for t in per]).contiguous()
    dq, dk, dv = (torch.cat([t[i] for t in per]).contiguous() for i in (3, 4, 5))
    cu_q = torch.tensor([0] + list(np.cumsum(sq)), dtype=torch.int32, device=DEV)
    cu_k = torch.tensor([0] + list(np.cumsum(sk)), dtype=torch.int32, device=DEV)
    scale = float(np.float32(1 / math.sqrt(d)))
    o, lse = fa_fwd_varlen_fp8(q, k, v, cu_q, cu_k, max(sq), max(sk), causal=causal,
                               scale=scale, q_descale=dq, k_descale=dk, v_descale=dv, **mod)
    assert get_last_device_error() == FA_OK
    window = mod.get("window_size", (-1, -1))
    softcap = mod.get("softcap", 0.0)
    for b, (nq, nk) in enumerate(zip(sq, sk)):
        qb, kb, vb, dqb, dkb, dvb = per[b]
        ob = o[int(cu_q[b]):int(cu_q[b + 1])].double().cpu().numpy()[None]
        lb = lse[:, int(cu_q[b]):int(cu_q[b + 1])].double().cpu().numpy()[None]
        if nq == 0:
            continue
        if nk == 0:
            assert np.all(ob == 0) and np.all(lb == -np.inf), f"sequence {b}: empty keys"
            continue
        o_ref, lse_ref = ORACLE.attention_fp8(qb.cpu(), kb.cpu(), vb.cpu(), scale, causal,
                                              dqb.cpu(), dkb.cpu(), dvb.cpu(), window=window,
                                              softcap=softcap)
        base = _baseline(qb, kb, vb, dqb, dkb, dvb, scale, causal, window, softcap)
        what = f"varlen fp8 sequence {b} ({nq} x {nk})"
        assert np.all(np.isfinite(ob)), f"{what}: non-finite O"
        e_gpu, e_base = np.abs(ob - o_ref), np.abs(base - o_ref)
        assert e_gpu.max() <= 2 * e_base.max() + 1e-4, \
            f"{what}: max |dO| {e_gpu.max():.3e} > 2 x baseline {e_base.max():.3e}"
        assert e_gpu.mean() <= 2 * e_base.mean() + 1e-4, \
            f"{what}: mean |dO| {e_gpu.mean():.3e} > 2 x baseline {e_base.mean():.3e}"
        fin = np.isfinite(lse_ref)
        assert np.array_equal(np.isfinite(lb), fin), f"{what}: LSE finiteness"
        assert np.abs(lb[fin] - lse_ref[fin]).max(initial=0.0) <= 1e-3, f"{what}: LSE"
    return per, o, lse


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_varlen(causal):
    # sequence starts that are not multiples of 16 (the transposed V gives each its own
    # 16-aligned column), an empty key range, Nq != Nk within a sequence, GQA
    _varlen_fp8([37, 1, 300, 129, 64, 200], [37, 0, 333, 129, 17, 450], 4, 2, 128, causal,
                seed=1900)


@pytest.mark.parametrize("d", [64, 96])
def test_fp8_varlen_head_dims(d):
    _varlen_fp8([100, 257, 3], [150, 257, 40], 2, 1, d, True, seed=1910 + d)


def test_fp8_varlen_window():
    _varlen_fp8([300, 45, 512], [300, 90, 700], 4, 4, 128, False, seed=1920,
                window_size=(100, 20))


def test_fp8_varlen_softcap():
    _varlen_fp8([130, 7, 400], [260, 7, 400], 4, 2, 128, True, seed=1925, softcap=10.0)


def test_fp8_varlen_one_sequence_equals_dense():
    """One sequence: the same kernel over the same K / V tiles as fa_fwd_fp8, bit for bit."""
    per, o, lse = _varlen_fp8([333], [517], 4, 2, 128, True, seed=1930)
    q, k, v, dq, dk, dv = per[0]
    scale = float(np.float32(1 / math.sqrt(128)))
    o_d, lse_d = fa_fwd_fp8(q, k, v, causal=True, scale=scale, q_descale=dq, k_descale=dk,
                            v_descale=dv)
    assert torch.equal(o, o_d[0]), "varlen O differs from the dense call"
    assert torch.equal(lse, lse_d[0]), "varlen LSE differs from the dense call"


def test_fp8_empty_keys_and_rows_without_keys():
    """Nk = 0: O = 0, LSE = -inf.  Causal with Nq > Nk: the first rows see no key."""
    q, k, v, dq, dk, dv = fp8_inputs(1, 64, 1, 2, 2, 128, 31, device=DEV)
    o, lse = fa_fwd_fp8(q, k[:, :0].contiguous(), v[:, :0].contiguous(), q_descale=dq,
                        k_descale=dk, v_descale=dv)
    assert get_last_device_error() == FA_OK
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))
    _check(1, 500, 200, 2, 2, 128, True, seed=32, what="fp8 Nq > Nk causal")


def test_fp8_full_size_head():
    """The causal 8k shape (B=2, H=32, N=8192): every head computed; head (0, 0) against
    the oracle and the baseline."""
    B, N, H, d = 2, 8192, 32, 128
    q, k, v, dq, dk, dv = fp8_inputs(B, N, N, H, H, d, 41, device=DEV)
    scale = float(np.float32(1 / math.sqrt(d)))
    o, lse = fa_fwd_fp8(q, k, v, causal=True, scale=scale, q_descale=dq, k_descale=dk,
                        v_descale=dv)
    assert get_last_device_error() == FA_OK
    sl = (slice(0, 1), slice(None), slice(0, 1))
    q1, k1, v1 = (t[sl].contiguous() for t in (q, k, v))
    d1 = [x[0:1, 0:1].contiguous() for x in (dq, dk, dv)]
    o_ref, lse_ref = ORACLE.attention_fp8(q1.cpu(), k1.cpu(), v1.cpu(), scale, True,
                                          *(x.cpu() for x in d1))
    base = _baseline(q1, k1, v1, *d1, scale, True)
    g = o[sl].double().cpu().numpy()
    e_gpu, e_base = np.abs(g - o_ref), np.abs(base - o_ref)
    assert e_gpu.max() <= 2 * e_base.max() + 1e-4 and e_gpu.mean() <= 2 * e_base.mean() + 1e-4
    assert np.abs(lse[0:1, 0:1].double().cpu().numpy() - lse_ref).max() <= 1e-3


# ---- decode over E4M3 caches (fa_fwd_kvcache_fp8): the cache is decoded exactly and every
# product is in fp32, as in the 16-bit decode, so the 16-bit decode bar applies.

def _decode_fp8(d, group, lens, seed, Lmax=3072, Hkv=2, descales=True, num_splits=0, **mod):
    from exact_attention_81_gb300 import fa_fwd_kvcache_fp8
    from exact_attention_81_gb300.inputs import kvcache_fp8_inputs
    from tests.parity_util import compare
    q, kc, vc, lens, dk, dv = kvcache_fp8_inputs(len(lens), Lmax, Hkv * group, Hkv, d, seed,
                                                 lens, device=DEV)
    if not descales:
        dk = dv = None
    scale = float(np.float32(1 / math.sqrt(d)))
    sl = mod.get("alibi_slopes")
    kw = dict(mod, alibi_slopes=None if sl is None else sl.to(DEV))
    o, lse = fa_fwd_kvcache_fp8(q, kc, vc, lens, k_descale=dk, v_descale=dv, scale=scale,
                                num_splits=num_splits, **kw)
    assert get_last_device_error() == FA_OK
    o_ref, lse_ref = ORACLE.attention_kvcache_fp8(
        q.cpu(), kc.cpu(), vc.cpu(), lens.cpu().numpy(), scale,
        None if dk is None else dk.cpu(), None if dv is None else dv.cpu(),
        window=mod.get("window_size", (-1, -1)), softcap=mod.get("softcap", 0.0),
        alibi_slopes=sl)
    # allowance without descales: the codes were drawn as N(0,1) / (0.25..0.375), so the
    # undescaled values and O are several times larger (|O| up to ~4, where half a bf16
    # ulp is 0.0156); measured 4e-7 beyond half an ulp, 1.5e-2 raw
    compare(o[:, 0], lse, o_ref, lse_ref, f"fp8 decode d={d} G={group} {mod}",
            allowance=not descales)
    return q, kc, vc, lens, dk, dv, o, lse


@pytest.mark.parametrize("d,group", [(128, 4), (128, 8), (128, 1), (64, 2), (96, 4),
                                     (256, 2), (256, 8), (192, 4), (16, 1), (128, 16),
                                     (128, 6), (256, 32)])
def test_decode_fp8(d, group):
    _decode_fp8(d, group, [1, 127, 128, 1000, 3071, 0, 513, 3072], 700 + d + group)


def test_decode_fp8_without_descales_and_explicit_splits():
    _decode_fp8(128, 4, [2000, 1, 129, 1024], 760, Lmax=2048, descales=False)
    _decode_fp8(128, 4, [2000, 1, 129, 1024], 761, Lmax=2048, num_splits=5)


@pytest.mark.parametrize("mod", ["window", "softcap", "alibi", "all"])
def test_decode_fp8_modifiers(mod):
    slopes = torch.tensor(2.0 ** (-8.0 * np.arange(1, 9) / 8), dtype=torch.float32)
    kw = {"window": dict(window_size=(700, -1)), "softcap": dict(softcap=15.0),
          "alibi": dict(alibi_slopes=slopes),
          "all": dict(window_size=(1500, 0), softcap=4.0, alibi_slopes=slopes)}[mod]
    _decode_fp8(128, 4, [1, 127, 128, 129, 1000, 3000, 0, 3072], 770, **kw)


@pytest.mark.parametrize("d", [128, 256])
def test_decode_fp8_paged(d):
    """The same E4M3 caches as shuffled pages of 128 rows through a block table."""
    from exact_attention_81_gb300 import fa_fwd_kvcache_fp8
    from exact_attention_81_gb300.inputs import kvcache_fp8_inputs
    from tests.parity_util import compare
    B, Lmax, Hq, Hkv, page = 4, 1024, 8, 2, 128
    lens = [1, 300, 1024, 640]
    q, kc, vc, lens_t, dk, dv = kvcache_fp8_inputs(B, Lmax, Hq, Hkv, d, 780 + d, lens,
                                                   device=DEV)
    nblk = Lmax // page
    perm = np.random.default_rng(781).permutation(B * nblk + 3)[:B * nblk]
    table = torch.from_numpy(perm.reshape(B, nblk).astype(np.int32)).to(DEV)
    pages = []
    for c in (kc, vc):
        p8 = torch.zeros((B * nblk + 3, page, Hkv, d), dtype=torch.uint8, device=DEV)
        p8[table.reshape(-1).long()] = c.view(torch.uint8).reshape(B * nblk, page, Hkv, d)
        pages.append(p8.view(torch.float8_e4m3fn))
    scale = float(np.float32(1 / math.sqrt(d)))
    o, lse = fa_fwd_kvcache_fp8(q, pages[0], pages[1], lens_t, k_descale=dk, v_descale=dv,
                                scale=scale, block_table=table, window_size=(400, -1))
    assert get_last_device_error() == FA_OK
    o_ref, lse_ref = ORACLE.attention_kvcache_fp8(q.cpu(), kc.cpu(), vc.cpu(), np.array(lens),
                                                  scale, dk.cpu(), dv.cpu(), window=(400, -1))
    compare(o[:, 0], lse, o_ref, lse_ref, f"fp8 decode paged d={d}")
