"""GPU parity of the decode-step extras against the fp64 oracle: in-place append of the new
key and value (caches compared bit for bit), rotary embedding of the query and the new key
(both pair layouts), paged caches through a shuffled block table, together with windows
and softcap; refused appends are flagged and write nothing out of place."""
import math

import numpy as np
import pytest
import torch

import oracle.oracle as ORACLE
from exact_attention_81_gb300 import (FA_ERR_INVALID_ARG, FA_OK, fa_fwd_kvcache,
                                      get_last_device_error)
from exact_attention_81_gb300.inputs import bf16_normal
from tests.parity_util import compare

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _scale(d):
    return float(np.float32(1 / math.sqrt(d)))


def _rope(P, rot_dim):
    half = rot_dim // 2
    inv = 10000.0 ** (-np.arange(half) / half)
    ang = np.arange(P)[:, None] * inv[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _case(B, Lmax, Hq, Hkv, d, seed, dtype=torch.bfloat16):
    q = bf16_normal((B, 1, Hq, d), seed, DEV, dtype)
    kc = bf16_normal((B, Lmax, Hkv, d), seed + 1, DEV, dtype)
    vc = bf16_normal((B, Lmax, Hkv, d), seed + 2, DEV, dtype)
    kn = bf16_normal((B, 1, Hkv, d), seed + 3, DEV, dtype)
    vn = bf16_normal((B, 1, Hkv, d), seed + 4, DEV, dtype)
    return q, kc, vc, kn, vn


def _paged(kc, vc, page, seed, spare=5):
    """The same caches as shuffled pages of `page` rows: (k_pages, v_pages, block_table)."""
    B, Lmax, Hkv, d = kc.shape
    nblk = Lmax // page
    rng = np.random.default_rng(seed)
    table = rng.permutation(B * nblk + spare)[:B * nblk].reshape(B, nblk).astype(np.int32)
    kp = torch.zeros((B * nblk + spare, page, Hkv, d), dtype=kc.dtype, device=DEV)
    vp = torch.zeros_like(kp)
    t = torch.from_numpy(table).to(DEV).long()
    kp[t.reshape(-1)] = kc.reshape(B * nblk, page, Hkv, d)
    vp[t.reshape(-1)] = vc.reshape(B * nblk, page, Hkv, d)
    return kp, vp, torch.from_numpy(table).to(DEV)


def _step(q, kc, vc, lens, **kw):
    """GPU call and oracle on copies of the same caches; returns both results and caches."""
    kc0, vc0 = kc.clone(), vc.clone()
    o, lse = fa_fwd_kvcache(q, kc, vc, lens, **kw)
    st = get_last_device_error()
    okw = {}
    for name in ("k_new", "v_new"):
        if kw.get(name) is not None:
            okw[name] = kw[name].cpu()
    for name in ("rotary_cos", "rotary_sin", "block_table"):
        if kw.get(name) is not None:
            okw[name] = kw[name].cpu().numpy()
    for name in ("window_size", "softcap", "rotary_interleaved"):
        if name in kw:
            okw["window" if name == "window_size" else name] = kw[name]
    ref = ORACLE.kvcache_step(q.cpu(), kc0.cpu(), vc0.cpu(), lens.cpu().numpy(),
                              _scale(q.shape[-1]), **okw)
    return st, o, lse, ref


@pytest.mark.parametrize("d,group,dtype", [(128, 4, torch.bfloat16), (128, 8, torch.bfloat16),
                                           (64, 1, torch.bfloat16), (128, 4, torch.float16)])
def test_append(d, group, dtype):
    B, Lmax, Hkv = 8, 2048, 2
    q, kc, vc, kn, vn = _case(B, Lmax, Hkv * group, Hkv, d, 600 + d + group, dtype)
    lens = torch.tensor([0, 1, 127, 128, 1000, 2046, 2047, 300], dtype=torch.int32, device=DEV)
    st, o, lse, (o_ref, l_ref, k_ref, v_ref) = _step(q, kc, vc, lens, k_new=kn, v_new=vn)
    assert st == FA_OK
    assert np.array_equal(_bits(kc), k_ref) and np.array_equal(_bits(vc), v_ref)
    compare(o[:, 0], lse, o_ref, l_ref, f"append d={d} G={group} {dtype}")


@pytest.mark.parametrize("rot_dim,interleaved,dtype", [
    (128, False, torch.bfloat16), (64, False, torch.bfloat16), (128, True, torch.bfloat16),
    (32, True, torch.float16), (128, False, torch.float16)])
def test_append_rotary(rot_dim, interleaved, dtype):
    B, Lmax, Hq, Hkv, d = 6, 1024, 16, 4, 128
    q, kc, vc, kn, vn = _case(B, Lmax, Hq, Hkv, d, 610 + rot_dim, dtype)
    lens = torch.tensor([0, 5, 511, 512, 1000, 1023], dtype=torch.int32, device=DEV)
    cos, sin = (torch.from_numpy(t).to(DEV) for t in _rope(1100, rot_dim))
    st, o, lse, (o_ref, l_ref, k_ref, v_ref) = _step(
        q, kc, vc, lens, k_new=kn, v_new=vn, rotary_cos=cos, rotary_sin=sin,
        rotary_interleaved=interleaved)
    assert st == FA_OK
    assert np.array_equal(_bits(kc), k_ref), "rotated keys differ from the oracle's"
    assert np.array_equal(_bits(vc), v_ref)
    compare(o[:, 0], lse, o_ref, l_ref, f"rotary {rot_dim} interleaved={interleaved} {dtype}")


@pytest.mark.parametrize("page", [128, 256])
@pytest.mark.parametrize("extra", ["none", "append", "append_rotary", "window", "window_softcap"])
def test_paged(page, extra):
    B, Lmax, Hq, Hkv, d = 6, 2048, 32, 8, 128
    q, kc, vc, kn, vn = _case(B, Lmax, Hq, Hkv, d, 620 + page)
    kp, vp, table = _paged(kc, vc, page, 621 + page)
    lens = torch.tensor([1, 200, 1024, 1500, 2047, 0], dtype=torch.int32, device=DEV)
    cos, sin = (torch.from_numpy(t).to(DEV) for t in _rope(2100, d))
    kw = {"none": {}, "append": dict(k_new=kn, v_new=vn),
          "append_rotary": dict(k_new=kn, v_new=vn, rotary_cos=cos, rotary_sin=sin),
          "window": dict(window_size=(300, -1)),
          "window_softcap": dict(k_new=kn, v_new=vn, window_size=(777, -1), softcap=10.0)}[extra]
    st, o, lse, (o_ref, l_ref, k_ref, v_ref) = _step(q, kp, vp, lens, block_table=table, **kw)
    assert st == FA_OK
    assert np.array_equal(_bits(kp), k_ref) and np.array_equal(_bits(vp), v_ref)
    compare(o[:, 0], lse, o_ref, l_ref, f"paged {page} {extra}")


@pytest.mark.parametrize("group,extra", [(8, "append_rotary"), (8, "window_softcap"),
                                         (4, "append"), (2, "none")])
def test_paged_wide(group, extra):
    """Width-256 decode through a shuffled block table with the step's extras."""
    B, Lmax, Hkv, d = 4, 1024, 2, 256
    q, kc, vc, kn, vn = _case(B, Lmax, Hkv * group, Hkv, d, 630 + group)
    kp, vp, table = _paged(kc, vc, 128, 631 + group)
    lens = torch.tensor([1, 300, 1023, 640], dtype=torch.int32, device=DEV)
    cos, sin = (torch.from_numpy(t).to(DEV) for t in _rope(1100, 128))
    kw = {"none": {}, "append": dict(k_new=kn, v_new=vn),
          "append_rotary": dict(k_new=kn, v_new=vn, rotary_cos=cos, rotary_sin=sin),
          "window_softcap": dict(k_new=kn, v_new=vn, window_size=(333, -1), softcap=12.0)}[extra]
    st, o, lse, (o_ref, l_ref, k_ref, v_ref) = _step(q, kp, vp, lens, block_table=table, **kw)
    assert st == FA_OK
    assert np.array_equal(_bits(kp), k_ref) and np.array_equal(_bits(vp), v_ref)
    compare(o[:, 0], lse, o_ref, l_ref, f"paged d=256 G={group} {extra}")


def test_refused_append_is_flagged_and_writes_nothing():
    """A sequence already at Lmax has no room: flagged, its rows untouched; the others are
    appended and attended as usual in the same call."""
    B, Lmax, Hq, Hkv, d = 4, 512, 8, 2, 128
    q, kc, vc, kn, vn = _case(B, Lmax, Hq, Hkv, d, 630)
    lens = torch.tensor([10, 512, 300, 0], dtype=torch.int32, device=DEV)
    kc0, vc0 = kc.clone(), vc.clone()
    o, lse = fa_fwd_kvcache(q, kc, vc, lens, k_new=kn, v_new=vn)
    assert get_last_device_error() == FA_ERR_INVALID_ARG
    assert torch.equal(kc[1], kc0[1]) and torch.equal(vc[1], vc0[1])
    sel = [0, 2, 3]
    o_ref, l_ref, k_ref, v_ref = ORACLE.kvcache_step(
        q[sel].cpu(), kc0[sel].cpu(), vc0[sel].cpu(), lens[sel].cpu().numpy(), _scale(d),
        k_new=kn[sel].cpu(), v_new=vn[sel].cpu())
    assert np.array_equal(_bits(kc[sel]), k_ref) and np.array_equal(_bits(vc[sel]), v_ref)
    compare(o[sel, 0], lse[sel], o_ref, l_ref, "appends next to a refused one")


def test_bad_block_table_entry_is_flagged():
    """A table entry outside the page pool reads back as zeros and is flagged."""
    B, Lmax, Hq, Hkv, d = 2, 512, 8, 2, 128
    q, kc, vc, _, _ = _case(B, Lmax, Hq, Hkv, d, 640)
    kp, vp, table = _paged(kc, vc, 128, 641)
    table[1, 2] = 1 << 20
    lens = torch.tensor([512, 512], dtype=torch.int32, device=DEV)
    fa_fwd_kvcache(q, kp, vp, lens, block_table=table)
    assert get_last_device_error() == FA_ERR_INVALID_ARG
