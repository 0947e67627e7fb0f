"""fa_fwd_host: the forward with host (pinned) tensors, copies overlapped with the
computation by query ranges.  Its O and LSE are bit-identical to fa_fwd on the same inputs
(each range is computed over the same key tiles in the same order), for causal calls (key
prefixes per range), non-causal calls (whole batch entries), Nq != Nk and the score
modifiers; one case against the oracle."""
import math

import numpy as np
import pytest
import torch

import oracle.oracle as ORACLE
from exact_attention_81_gb300 import FA_OK, fa_fwd, fa_fwd_host, get_last_device_error
from exact_attention_81_gb300.inputs import dense_inputs
from tests.parity_util import compare, dense_rows

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _host(t):
    return t.cpu().contiguous().pin_memory()


@pytest.mark.parametrize("case", [
    # B, Nq, Nk, Hq, Hkv, d, causal, chunks, modifiers
    (2, 1000, 1000, 4, 2, 128, True, 4, {}),
    (2, 1000, 1000, 4, 2, 128, True, 1, {}),
    (1, 777, 1500, 2, 1, 64, True, 8, {}),
    (1, 1500, 700, 2, 2, 128, True, 5, {}),
    (3, 500, 600, 4, 4, 96, False, 4, {}),
    (2, 900, 900, 4, 2, 128, False, 3, dict(window_size=(200, 0))),
    (2, 640, 640, 8, 2, 128, True, 4, dict(softcap=20.0, alibi=True)),
    (2, 512, 512, 4, 2, 256, True, 2, {}),
])
def test_host_matches_device_call(case):
    B, Nq, Nk, Hq, Hkv, d, causal, chunks, mod = case
    mod = dict(mod)
    if mod.pop("alibi", False):
        mod["alibi_slopes"] = torch.rand((B, Hq), dtype=torch.float32, device=DEV) * 0.5
    q, k, v = dense_inputs(B, Nq, Nk, Hq, Hkv, d, seed=990 + Nq, device=DEV)
    o_ref, l_ref = fa_fwd(q, k, v, causal=causal, **mod)
    assert get_last_device_error() == FA_OK
    o, lse = fa_fwd_host(_host(q), _host(k), _host(v), causal=causal, chunks=chunks, **mod)
    torch.cuda.current_stream().synchronize()
    assert get_last_device_error() == FA_OK
    assert torch.equal(o, o_ref.cpu()), f"{case}: O differs from fa_fwd"
    assert torch.equal(lse, l_ref.cpu()), f"{case}: LSE differs from fa_fwd"


def test_host_against_oracle():
    B, N, H, d = 2, 700, 4, 128
    q, k, v = dense_inputs(B, N, N, H, 2, d, seed=1001, device=DEV)
    o, lse = fa_fwd_host(_host(q), _host(k), _host(v), causal=True, chunks=6)
    torch.cuda.current_stream().synchronize()
    assert get_last_device_error() == FA_OK
    scale = float(np.float32(1 / math.sqrt(d)))
    o_ref, lse_ref = ORACLE.attention(q.cpu(), k.cpu(), v.cpu(), scale, True)
    compare(*dense_rows(o, lse), *dense_rows(o_ref, lse_ref), "fa_fwd_host causal")


def test_host_calls_back_to_back_reuse_buffers():
    """Two calls on the same stream with the same device buffers: the second's copies in
    wait for the first's computation, so both results are right."""
    B, N, H, d = 1, 800, 2, 128
    ins = [dense_inputs(B, N, N, H, H, d, seed=1010 + s, device=DEV) for s in range(2)]
    bufs = tuple(torch.empty((B, N, H, d), dtype=torch.bfloat16, device=DEV) for _ in range(4)) + \
        (torch.empty((B, H, N), dtype=torch.float32, device=DEV),)
    outs = [fa_fwd_host(*(_host(t) for t in x), causal=True, device_buffers=bufs, chunks=4)
            for x in ins]
    torch.cuda.current_stream().synchronize()
    for x, (o, lse) in zip(ins, outs):
        o_ref, l_ref = fa_fwd(*x, causal=True)
        assert torch.equal(o, o_ref.cpu()) and torch.equal(lse, l_ref.cpu())
