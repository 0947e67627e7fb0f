"""GPU parity of the dense and varlen prefill path (libfa.so through its C ABI) against the
fp64 oracle, on seeded inputs, element by element: small cases with ragged tails and
degenerate shapes, and the full-size workloads in the benchmark's launch configuration."""
import math

import numpy as np
import pytest
import torch

import oracle.oracle as ORACLE
from exact_attention_81_gb300 import (FA_OK, fa_fwd, fa_fwd_varlen, get_last_device_error)
from exact_attention_81_gb300.inputs import (WORKLOADS, dense_inputs, varlen_inputs,
                                             workload_inputs)
from tests.parity_util import compare, dense_rows, varlen_rows

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _run_dense(q, k, v, causal, scale=None):
    o, lse = fa_fwd(q, k, v, causal=causal, scale=scale)
    assert get_last_device_error() == FA_OK
    return o, lse


def _oracle_dense(q, k, v, causal, scale):
    return ORACLE.attention(q.cpu(), k.cpu(), v.cpu(), scale, causal)


# ------------------------------------------------------------------ small, full compare

DENSE_CASES = [
    # B, Nq, Nk, Hq, Hkv, d, causal
    (1, 256, 256, 1, 1, 64, False),
    (1, 256, 256, 1, 1, 64, True),
    (2, 300, 300, 2, 2, 128, False),   # ragged tail (300 = 2*128 + 44)
    (2, 300, 300, 2, 2, 128, True),
    (1, 1, 1, 1, 1, 128, False),       # single row, single key
    (1, 1, 1, 1, 1, 64, True),
    (1, 100, 700, 2, 1, 128, True),    # Nq < Nk, bottom-right causal
    (1, 700, 100, 2, 2, 64, True),     # Nq > Nk: leading rows see no key
    (1, 129, 383, 3, 3, 128, False),
    (2, 517, 517, 8, 2, 128, True),    # GQA 4:1, several tiles + tail
    (1, 384, 384, 8, 1, 64, False),    # MQA 8:1
    (1, 640, 640, 4, 4, 128, True),
    (3, 64, 200, 4, 2, 64, False),
]


@pytest.mark.parametrize("case", DENSE_CASES, ids=lambda c: "B{}_q{}_k{}_h{}x{}_d{}_{}".format(
    c[0], c[1], c[2], c[3], c[4], c[5], "causal" if c[6] else "full"))
def test_dense_small(case):
    B, Nq, Nk, Hq, Hkv, d, causal = case
    q, k, v = dense_inputs(B, Nq, Nk, Hq, Hkv, d, seed=2000 + Nq + Nk + d, device=DEV)
    scale = 1.0 / math.sqrt(d)
    o, lse = _run_dense(q, k, v, causal)
    o_ref, lse_ref = _oracle_dense(q, k, v, causal, float(np.float32(scale)))
    compare(*dense_rows(o, lse), *dense_rows(o_ref, lse_ref), f"dense {case}")


def test_tiny_workload_and_golden_rows():
    """The tiny workload (1 x 256 x 1 head, d = 64) in full, plus the stored oracle rows."""
    import json
    import os
    w = WORKLOADS["tiny"]
    # drawn from the CPU generator, as the stored rows were (CPU and CUDA streams differ)
    q, k, v = (t.to(DEV) for t in workload_inputs(w, device="cpu"))
    o, lse = _run_dense(q, k, v, w.causal)
    o_ref, lse_ref = _oracle_dense(q, k, v, w.causal, w.scale)
    compare(*dense_rows(o, lse), *dense_rows(o_ref, lse_ref), "tiny")
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "tiny_rows.json")))
    rows = g["rows"]
    compare(o[0, rows, 0], lse[0, 0, rows], np.array(g["o"]), np.array(g["lse"]), "golden rows")


def test_scale_argument():
    q, k, v = dense_inputs(1, 200, 200, 2, 2, 128, seed=77, device=DEV)
    for scale in (0.03, 0.5):
        o, lse = _run_dense(q, k, v, True, scale=scale)
        o_ref, lse_ref = _oracle_dense(q, k, v, True, float(np.float32(scale)))
        compare(*dense_rows(o, lse), *dense_rows(o_ref, lse_ref), f"scale {scale}")


def test_strided_views_and_guard_bands():
    """Non-contiguous q/k/v/o views (a slice of a larger buffer) are honoured, and nothing
    outside the output view is written."""
    B, N, H, d = 2, 260, 3, 128
    big_q = torch.randn(B, N, H + 2, d, device=DEV).to(torch.bfloat16)
    big_k = torch.randn(B, N, H + 1, d, device=DEV).to(torch.bfloat16)
    big_v = torch.randn(B, N, H + 1, d, device=DEV).to(torch.bfloat16)
    q, k, v = big_q[:, :, 1:H + 1], big_k[:, :, :H], big_v[:, :, 1:]
    guard = torch.full((B, N + 16, H + 2, d), 7.0, device=DEV, dtype=torch.bfloat16)
    out = guard[:, 8:N + 8, 1:H + 1]
    o, lse = fa_fwd(q, k, v, causal=True, out=out)
    assert get_last_device_error() == FA_OK
    o_ref, lse_ref = _oracle_dense(q.contiguous(), k.contiguous(), v.contiguous(), True,
                                   float(np.float32(1 / math.sqrt(d))))
    compare(*dense_rows(o, lse), *dense_rows(o_ref, lse_ref), "strided")
    mask = torch.ones_like(guard, dtype=torch.bool)
    mask[:, 8:N + 8, 1:H + 1] = False
    assert torch.all(guard[mask] == 7.0), "write outside the output view"


def test_empty_keys():
    q, _, _ = dense_inputs(2, 50, 1, 2, 2, 64, seed=5, device=DEV)
    k = torch.empty((2, 0, 2, 64), dtype=torch.bfloat16, device=DEV)
    o, lse = _run_dense(q, k, k, False)
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))


def test_deterministic():
    q, k, v = dense_inputs(2, 777, 777, 4, 2, 128, seed=9, device=DEV)
    o1, l1 = _run_dense(q, k, v, True)
    o2, l2 = _run_dense(q, k, v, True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


# ------------------------------------------------------------------ varlen

VARLEN_CASES = [
    ([5, 0, 19, 333, 1, 128, 129, 256], [7, 3, 19, 333, 1, 128, 200, 256], 4, 2, 128),
    ([1000, 17, 600], [1000, 17, 600], 2, 2, 64),
    ([0, 0], [5, 0], 2, 1, 128),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("case", VARLEN_CASES)
def test_varlen(case, causal):
    sq, sk, Hq, Hkv, d = case
    q, k, v, cu_q, cu_k = varlen_inputs(sq, sk, Hq, Hkv, d, seed=31, device=DEV)
    total_q = q.shape[0]
    o_buf = torch.full((total_q + 8, Hq, d), 3.0, dtype=torch.bfloat16, device=DEV)
    out = o_buf[4:total_q + 4]
    o, lse = fa_fwd_varlen(q, k, v, cu_q, cu_k, max(sq), max(sk), causal=causal, out=out)
    assert get_last_device_error() == FA_OK
    o_ref, lse_ref = ORACLE.attention_varlen(q.cpu(), k.cpu(), v.cpu(), cu_q.cpu(), cu_k.cpu(),
                                             float(np.float32(1 / math.sqrt(d))), causal)
    if total_q:
        compare(*varlen_rows(o, lse), *varlen_rows(o_ref, lse_ref),
                f"varlen {case} causal={causal}")
    assert torch.all(o_buf[:4] == 3.0) and torch.all(o_buf[total_q + 4:] == 3.0)


@pytest.mark.parametrize("d", [64, 128])
def test_varlen_staged_and_direct_row_stores(d):
    """Sequences of 31..223 rows: a softmax warp whose 32 rows all lie in its sequence
    stages O in shared memory and writes it with TMA stores, the others store their rows
    one by one.  Each sequence matches the oracle, and the rows around the output (and of
    the neighbouring sequences) are untouched."""
    sq = [31, 32, 33, 95, 96, 97, 160, 223]
    Hq, Hkv = 4, 2
    q, k, v, cu_q, cu_k = varlen_inputs(sq, sq, Hq, Hkv, d, seed=57 + d, device=DEV)
    total_q = q.shape[0]
    o_buf = torch.full((total_q + 8, Hq, d), 5.0, dtype=torch.bfloat16, device=DEV)
    out = o_buf[4:total_q + 4]
    o, lse = fa_fwd_varlen(q, k, v, cu_q, cu_k, max(sq), max(sq), causal=True, out=out)
    assert get_last_device_error() == FA_OK
    o_ref, lse_ref = ORACLE.attention_varlen(q.cpu(), k.cpu(), v.cpu(), cu_q.cpu(), cu_k.cpu(),
                                             float(np.float32(1 / math.sqrt(d))), True)
    compare(*varlen_rows(o, lse), *varlen_rows(o_ref, lse_ref), f"varlen staged d={d}")
    assert torch.all(o_buf[:4] == 5.0) and torch.all(o_buf[total_q + 4:] == 5.0)


@pytest.mark.parametrize("d", [40, 96])
@pytest.mark.parametrize("causal", [False, True])
def test_staged_stores_into_padded_view(d, causal):
    """O as a view of a wider buffer (an extra head before it, columns past d, rows around
    it): the staged TMA stores write d columns of the view's rows and heads only, for a
    sub-tile whose last warp holds a partial row block (223 = 128 + 64 + 31 rows)."""
    B, N, H = 2, 223, 3
    q, k, v = dense_inputs(B, N, N, H, H, d, seed=61 + d, device=DEV)
    dw = 64 if d <= 56 else 128
    buf = torch.full((B, N + 16, H + 1, dw), 7.0, dtype=torch.bfloat16, device=DEV)
    out = buf[:, 8:N + 8, 1:, :d]
    o, lse = fa_fwd(q, k, v, causal=causal, out=out)
    assert get_last_device_error() == FA_OK
    o_ref, lse_ref = _oracle_dense(q, k, v, causal, float(np.float32(1 / math.sqrt(d))))
    compare(*dense_rows(o, lse), *dense_rows(o_ref, lse_ref), f"padded view d={d}")
    mask = torch.ones_like(buf, dtype=torch.bool)
    mask[:, 8:N + 8, 1:, :d] = False
    assert torch.all(buf[mask] == 7.0), "write outside the output view"


def test_varlen_matches_dense():
    """A one-sequence varlen call equals the dense call bit for bit."""
    q, k, v = dense_inputs(1, 500, 500, 4, 2, 128, seed=41, device=DEV)
    o_d, l_d = _run_dense(q, k, v, True)
    cu = torch.tensor([0, 500], dtype=torch.int32, device=DEV)
    o_v, l_v = fa_fwd_varlen(q[0], k[0], v[0], cu, cu, 500, 500, causal=True)
    assert torch.equal(o_v, o_d[0]) and torch.equal(l_v, l_d[0])


def test_varlen_bad_cu_seqlens_flagged():
    """Out-of-range prefix sums on the device are reported, not followed."""
    from exact_attention_81_gb300 import FA_ERR_INVALID_ARG
    q, k, v, _, _ = varlen_inputs([10, 10], [10, 10], 2, 2, 64, seed=3, device=DEV)
    bad = torch.tensor([0, 10, 40], dtype=torch.int32, device=DEV)  # ends past total
    fa_fwd_varlen(q, k, v, bad, bad, 30, 30)
    assert get_last_device_error() == FA_ERR_INVALID_ARG
    assert get_last_device_error() == FA_OK


# ------------------------------------------------------------------ half tiles

def _half_tile_case(which, sm):
    # (B, Nq, Nk, Hq, Hkv, d): tile count just above the SM count and not a multiple of it,
    # so the last partial wave runs as half tiles; ragged last query blocks whose second
    # half is empty, and a ragged last key tile.
    if which == "ragged_rows":
        hq = (sm + 10 + 1) // 2  # 2 query blocks (256 rows) per head
        return 1, 300, 300, hq, hq, 128
    hq = sm // 6 + 1           # 3 query blocks per head, 2 batch entries
    return 2, 600, 1000, hq, 1, 64


@pytest.mark.parametrize("which", ["ragged_rows", "mqa_ragged_keys"])
def test_half_tiles_last_wave(which):
    """Without a mask, the tiles of the last, partial wave are split into two half tiles
    (one 128-row sub-tile each); every row is computed as in a whole tile, so the output
    equals the varlen call (which never splits tiles) bit for bit, and the oracle."""
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    B, Nq, Nk, Hq, Hkv, d = _half_tile_case(which, sm)
    tiles = B * Hq * ((Nq + 255) // 256)
    assert tiles > sm and tiles % sm != 0
    q, k, v = dense_inputs(B, Nq, Nk, Hq, Hkv, d, seed=4100 + Nq + d, device=DEV)
    o, lse = _run_dense(q, k, v, False)
    cu_q = torch.arange(0, (B + 1) * Nq, Nq, dtype=torch.int32, device=DEV)
    cu_k = torch.arange(0, (B + 1) * Nk, Nk, dtype=torch.int32, device=DEV)
    o_v, l_v = fa_fwd_varlen(q.reshape(B * Nq, Hq, d), k.reshape(B * Nk, Hkv, d),
                             v.reshape(B * Nk, Hkv, d), cu_q, cu_k, Nq, Nk, causal=False)
    assert get_last_device_error() == FA_OK
    assert torch.equal(o_v.reshape(B, Nq, Hq, d), o)
    assert torch.equal(l_v.reshape(Hq, B, Nq).permute(1, 0, 2), lse)  # varlen LSE: (Hq, total_q)
    o_ref, lse_ref = _oracle_dense(q, k, v, False, float(np.float32(1 / math.sqrt(d))))
    compare(*dense_rows(o, lse), *dense_rows(o_ref, lse_ref), f"half tiles {which}")


# ------------------------------------------------------------------ full-size workloads

@pytest.mark.parametrize("name", ["dense2k", "causal8k", "gqa16k"])
def test_full_size_workload(name):
    """The benchmark workloads at full size, in the benchmark's launch configuration, every
    output element against the oracle (threaded over all host cores): raw max and mean
    |O - O_ref| over the whole workload and max |LSE - LSE_ref| over all of its rows."""
    w = WORKLOADS[name]
    q, k, v = workload_inputs(w, device=DEV)
    o, lse = _run_dense(q, k, v, w.causal)
    o_ref, lse_ref = _oracle_dense(q, k, v, w.causal, w.scale)
    stats = compare(*dense_rows(o, lse), *dense_rows(o_ref, lse_ref), name)
    print(f"{name}: raw max|dO| {stats['raw_max_abs_o']:.3e}, mean|dO| "
          f"{stats['raw_mean_abs_o']:.3e}, max|dLSE| {stats['max_abs_lse']:.3e} over "
          f"{o.numel()} elements")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("direction", ["rising", "falling"])
def test_row_max_jumps_across_tiles(direction, causal):
    """Key norms that rise (or fall) steeply along the sequence make each row's maximum
    jump by far more than a factor 2^8 from one 128-key tile to the next (or never grow
    after the first tile): both the rescale and the keep-the-reference paths of the online
    softmax are exercised."""
    B, N, H, d = 1, 700, 2, 64
    q, k, v = dense_inputs(B, N, N, H, H, d, seed=91, device=DEV)
    ramp = torch.linspace(0.2, 6.0, N, device=DEV)
    if direction == "falling":
        ramp = ramp.flip(0)
    k = (k.float() * ramp[None, :, None, None]).to(torch.bfloat16)
    scale = 0.9
    o, lse = _run_dense(q, k, v, causal, scale=scale)
    o_ref, lse_ref = _oracle_dense(q, k, v, causal, float(np.float32(scale)))
    compare(*dense_rows(o, lse), *dense_rows(o_ref, lse_ref), f"max jumps {direction}")


# ------------------------------------------------------------------ CTA pairs

PAIR_CASES = [
    # B, Nq, Nk, Hq, Hkv, d, causal: work tiles of 512 rows, sub-tiles of 256 over two CTAs
    (1, 256, 256, 1, 1, 128, False),    # one sub-tile
    (1, 100, 100, 1, 1, 128, True),     # the odd CTA of the pair holds no valid row
    (2, 700, 700, 4, 2, 128, True),     # 2 work tiles, ragged second (700 = 512 + 188)
    (1, 1300, 1300, 2, 2, 96, False),   # d = 96, three tiles, ragged
    (1, 333, 1000, 8, 1, 128, True),    # Nq < Nk (bottom-right), MQA
    (1, 1000, 333, 2, 2, 80, True),     # Nq > Nk: leading rows see no key
]


@pytest.mark.parametrize("case", PAIR_CASES, ids=lambda c: "B{}_q{}_k{}_h{}x{}_d{}_{}".format(
    c[0], c[1], c[2], c[3], c[4], c[5], "causal" if c[6] else "full"))
def test_cta_pairs_and_single_cta_against_oracle(case):
    """The width-128 forward on CTA pairs and on the single-CTA kernel (the default), each
    against the oracle; each selection is deterministic and the two agree bit for bit."""
    from exact_attention_81_gb300 import set_cta_pairs
    B, Nq, Nk, Hq, Hkv, d, causal = case
    q, k, v = dense_inputs(B, Nq, Nk, Hq, Hkv, d, seed=3000 + Nq + d, device=DEV)
    o_ref, lse_ref = _oracle_dense(q, k, v, causal, float(np.float32(1 / math.sqrt(d))))
    outs = []
    try:
        for pairs in (True, False):
            set_cta_pairs(pairs)
            o, lse = _run_dense(q, k, v, causal)
            compare(*dense_rows(o, lse), *dense_rows(o_ref, lse_ref), f"pairs={pairs} {case}")
            o2, l2 = _run_dense(q, k, v, causal)
            assert torch.equal(o, o2) and torch.equal(lse, l2)
            outs.append((o, lse))
    finally:
        set_cta_pairs(False)
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


@pytest.mark.parametrize("causal", [False, True])
def test_cta_pairs_varlen(causal):
    from exact_attention_81_gb300 import set_cta_pairs
    sq = [5, 0, 700, 256, 257, 1100, 1]
    sk = [9, 4, 700, 300, 257, 1100, 1]
    q, k, v, cu_q, cu_k = varlen_inputs(sq, sk, 4, 2, 128, seed=77, device=DEV)
    o_ref, lse_ref = ORACLE.attention_varlen(q.cpu(), k.cpu(), v.cpu(), cu_q.cpu(), cu_k.cpu(),
                                             float(np.float32(1 / math.sqrt(128))), causal)
    try:
        for pairs in (True, False):
            set_cta_pairs(pairs)
            o, lse = fa_fwd_varlen(q, k, v, cu_q, cu_k, max(sq), max(sk), causal=causal)
            assert get_last_device_error() == FA_OK
            compare(*varlen_rows(o, lse), *varlen_rows(o_ref, lse_ref), f"pairs={pairs} varlen")
    finally:
        set_cta_pairs(False)
