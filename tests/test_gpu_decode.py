"""GPU parity of the split-KV decode path (fa_fwd_kvcache) against the fp64 oracle.

Cache rows at or past each sequence's length are NaN, so any read of them into the
result shows up as a non-finite output."""
import math

import numpy as np
import pytest
import torch

import oracle.oracle as ORACLE
from exact_attention_81_gb300 import (FA_ERR_INVALID_ARG, FA_OK, fa_fwd,
                                      fa_fwd_kvcache, fa_fwd_kvcache_workspace_size,
                                      get_last_device_error)
from exact_attention_81_gb300.inputs import WORKLOADS, kvcache_inputs
from tests.parity_util import compare

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _check(q, kc, vc, lens, num_splits, what, batches=None):
    o, lse = fa_fwd_kvcache(q, kc, vc, lens, num_splits=num_splits)
    assert get_last_device_error() == FA_OK
    d = q.shape[-1]
    scale = float(np.float32(1 / math.sqrt(d)))
    if batches is None:
        batches = list(range(q.shape[0]))
    bsel = torch.tensor(batches, dtype=torch.long)
    o_ref, lse_ref = ORACLE.attention_kvcache(q[bsel].cpu(), kc[bsel.to(kc.device)].cpu(),
                                              vc[bsel.to(vc.device)].cpu(),
                                              lens.cpu()[bsel], scale)
    return compare(o[bsel, 0], lse[bsel], o_ref, lse_ref, what), o, lse


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("group", [1, 2, 4, 8, 16, 32])
def test_decode_small(d, group):
    Hkv = 2
    Hq = Hkv * group
    lens = torch.tensor([1, 127, 128, 129, 1000, 255, 256, 2000, 0, 513], dtype=torch.int32)
    q, kc, vc, lens = kvcache_inputs(len(lens), 2048, Hq, Hkv, d, seed=500 + d + group,
                                     lengths=lens, device=DEV)
    _check(q, kc, vc, lens, 0, f"decode d={d} G={group}")


@pytest.mark.parametrize("d,Hq,Hkv", [(128, 24, 8), (128, 12, 2), (64, 40, 4), (256, 16, 1),
                                       (256, 24, 4), (128, 32, 1), (96, 20, 4)])
def test_decode_any_group(d, Hq, Hkv):
    """Group sizes that are not a power of two (3, 6, 10, 5) and MQA groups of 16 and 32:
    the query heads of a kv head run as several work items of up to 8 heads (4 at d > 128)
    that share its K/V stream."""
    lens = torch.tensor([1, 129, 1000, 2047, 0, 640], dtype=torch.int32)
    q, kc, vc, lens = kvcache_inputs(len(lens), 2048, Hq, Hkv, d, seed=550 + Hq + d,
                                     lengths=lens, device=DEV)
    _check(q, kc, vc, lens, 0, f"decode d={d} Hq={Hq} Hkv={Hkv}")
    _check(q, kc, vc, lens, 5, f"decode d={d} Hq={Hq} Hkv={Hkv} 5 splits")


@pytest.mark.parametrize("num_splits", [1, 2, 3, 7, 16, 100])
def test_decode_split_counts(num_splits):
    """Any number of splits gives the oracle result (the LSE-weighted merge is exact)."""
    lens = torch.tensor([3000, 1, 4095, 4096, 2048, 1537], dtype=torch.int32)
    q, kc, vc, lens = kvcache_inputs(len(lens), 4096, 16, 4, 128, seed=600, lengths=lens,
                                     device=DEV)
    _check(q, kc, vc, lens, num_splits, f"splits={num_splits}")


def test_decode_one_split_equals_dense():
    """With one split the decode output matches the dense path on the visible prefix."""
    n = 700
    lens = torch.tensor([n], dtype=torch.int32)
    q, kc, vc, lens = kvcache_inputs(1, 1024, 8, 2, 128, seed=610, lengths=lens, device=DEV)
    o, lse = fa_fwd_kvcache(q, kc, vc, lens, num_splits=1)
    od, ld = fa_fwd(q, kc[:, :n].contiguous(), vc[:, :n].contiguous(), causal=False)
    assert (o.float() - od.float()).abs().max().item() <= 1e-2
    assert (lse - ld[:, :, 0]).abs().max().item() <= 1e-3


def test_decode_deterministic():
    lens = torch.tensor([3333, 10, 2222], dtype=torch.int32)
    q, kc, vc, lens = kvcache_inputs(3, 4096, 32, 8, 128, seed=620, lengths=lens, device=DEV)
    o1, l1 = fa_fwd_kvcache(q, kc, vc, lens)
    o2, l2 = fa_fwd_kvcache(q, kc, vc, lens)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_decode_bad_length_flagged():
    lens = torch.tensor([100, 5000], dtype=torch.int32)  # 5000 > Lmax
    q, kc, vc, _ = kvcache_inputs(2, 1024, 4, 1, 64, seed=630, lengths=[100, 1024], device=DEV)
    fa_fwd_kvcache(q, kc, vc, lens.to(DEV))
    assert get_last_device_error() == FA_ERR_INVALID_ARG
    assert get_last_device_error() == FA_OK


def test_decode_workspace_size_is_checked():
    from exact_attention_81_gb300 import FAError
    lens = torch.tensor([100, 200], dtype=torch.int32)
    q, kc, vc, lens = kvcache_inputs(2, 512, 4, 1, 64, seed=640, lengths=lens, device=DEV)
    need = fa_fwd_kvcache_workspace_size(2, 4, 512, 64, 0)
    ws = torch.empty(need - 256, dtype=torch.uint8, device=DEV)
    with pytest.raises(FAError):
        fa_fwd_kvcache(q, kc, vc, lens, workspace=ws)


def test_decode_full_size_workload():
    """The decode workload at full size (B = 64, Hq = 32, Hkv = 8, caches of 32768 rows,
    lengths uniform in [1024, 32768]), in the benchmark's launch configuration: all 64
    batch entries against the oracle (each entry's visible prefix copied to the host), raw
    max and mean |O - O_ref| and max |LSE - LSE_ref| over the whole output."""
    w = WORKLOADS["decode"]
    q, kc, vc, lens = kvcache_inputs(w.B, w.Nk, w.Hq, w.Hkv, w.d, seed=w.seed, device=DEV)
    o, lse = fa_fwd_kvcache(q, kc, vc, lens)
    assert get_last_device_error() == FA_OK
    scale = float(np.float32(1 / math.sqrt(w.d)))
    lh = lens.cpu()
    o_ref = np.empty((w.B, w.Hq, w.d))
    lse_ref = np.empty((w.B, w.Hq))
    for b in range(w.B):
        n = int(lh[b])
        ob, lb = ORACLE.attention_kvcache(q[b:b + 1].cpu(), kc[b:b + 1, :n].cpu(),
                                          vc[b:b + 1, :n].cpu(), lh[b:b + 1], scale)
        o_ref[b], lse_ref[b] = ob[0], lb[0]
    stats = compare(o[:, 0], lse, o_ref, lse_ref, "decode full size")
    print(f"decode: raw max|dO| {stats['raw_max_abs_o']:.3e}, mean|dO| "
          f"{stats['raw_mean_abs_o']:.3e}, max|dLSE| {stats['max_abs_lse']:.3e} over "
          f"{o.numel()} elements")
