"""GPU parity of the fp16 paths (dense, varlen, decode) against the fp64 oracle, which
reads the same binary16 bit patterns."""
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
F16 = torch.float16


@pytest.mark.parametrize("case", [
    (1, 256, 256, 1, 1, 64, False),
    (2, 300, 300, 2, 2, 128, True),
    (1, 100, 700, 4, 1, 128, True),
    (2, 517, 517, 8, 2, 64, True),
    (1, 129, 383, 3, 3, 128, False),
])
def test_dense_fp16(case):
    B, Nq, Nk, Hq, Hkv, d, causal = case
    q, k, v = dense_inputs(B, Nq, Nk, Hq, Hkv, d, seed=3000 + Nq + d, device=DEV, dtype=F16)
    o, lse = fa_fwd(q, k, v, causal=causal)
    assert get_last_device_error() == FA_OK
    assert o.dtype == F16
    o_ref, lse_ref = ORACLE.attention(q.cpu(), k.cpu(), v.cpu(),
                                      float(np.float32(1 / math.sqrt(d))), causal)
    compare(*dense_rows(o, lse), *dense_rows(o_ref, lse_ref), f"fp16 dense {case}")


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_fp16(causal):
    sq = [5, 0, 333, 128, 129, 256]
    sk = [7, 3, 333, 128, 200, 256]
    q, k, v, cu_q, cu_k = varlen_inputs(sq, sk, 4, 2, 128, seed=33, device=DEV, dtype=F16)
    o, lse = fa_fwd_varlen(q, k, v, cu_q, cu_k, max(sq), max(sk), causal=causal)
    assert get_last_device_error() == FA_OK
    o_ref, lse_ref = ORACLE.attention_varlen(q.cpu(), k.cpu(), v.cpu(), cu_q.cpu(), cu_k.cpu(),
                                             float(np.float32(1 / math.sqrt(128))), causal)
    compare(*varlen_rows(o, lse), *varlen_rows(o_ref, lse_ref), "fp16 varlen")


@pytest.mark.parametrize("d,group", [(64, 4), (128, 1), (128, 4), (128, 8)])
def test_decode_fp16(d, group):
    lens = torch.tensor([1, 127, 128, 129, 1000, 2000, 0, 513], dtype=torch.int32)
    q, kc, vc, lens = kvcache_inputs(len(lens), 2048, 2 * group, 2, d, seed=700 + d + group,
                                     lengths=lens, device=DEV, dtype=F16)
    o, lse = fa_fwd_kvcache(q, kc, vc, lens)
    assert get_last_device_error() == FA_OK
    assert o.dtype == F16
    o_ref, lse_ref = ORACLE.attention_kvcache(q.cpu(), kc.cpu(), vc.cpu(), lens.cpu(),
                                              float(np.float32(1 / math.sqrt(d))))
    compare(o[:, 0], lse, o_ref, lse_ref, f"fp16 decode d={d} G={group}")


def test_full_size_causal8k_fp16():
    """The causal 8k workload drawn in fp16, sampled rows against the oracle."""
    w = WORKLOADS["causal8k"]
    q, k, v = dense_inputs(w.B, w.Nq, w.Nk, w.Hq, w.Hkv, w.d, seed=w.seed, device=DEV, dtype=F16)
    o, lse = fa_fwd(q, k, v, causal=True)
    assert get_last_device_error() == FA_OK
    rows = sample_rows(w.B, w.Hq, w.Nq, 120, seed=w.seed + 1)
    o_ref, lse_ref = ORACLE.attention_rows(q.cpu(), k.cpu(), v.cpu(), rows, w.scale, True)
    r = torch.as_tensor(rows, dtype=torch.long)
    compare(o[r[:, 0], r[:, 2], r[:, 1]], lse[r[:, 0], r[:, 1], r[:, 2]], o_ref, lse_ref,
            "fp16 causal8k")
