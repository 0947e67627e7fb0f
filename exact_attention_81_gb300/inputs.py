"""Seeded synthetic inputs for the attention forward path.

This module holds the workload shapes and the random-number recipes only: no
attention arithmetic.  Both sides of every parity check (the CUDA library and the
CPU oracle) read the tensors made here.

Recipe: Q, K, V entries are iid N(0, 1) drawn in float32 from a seeded
``torch.Generator`` and rounded to bf16 (round-to-nearest-even by ``.to``).
Decode cache lengths are integers uniform in [1024, 32768] from a CPU generator;
cache rows at or past a sequence's length are filled with NaN so that a read past
the visible prefix shows up in the output.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str  # "dense" or "kvcache"
    B: int
    Hq: int
    Hkv: int
    Nq: int
    Nk: int  # dense: key length; kvcache: padded cache length Lmax
    d: int
    causal: bool
    seed: int

    @property
    def scale(self) -> float:
        # 1/sqrt(d) rounded once to float32: the value handed to the kernels.
        return float(torch.tensor(1.0 / math.sqrt(self.d), dtype=torch.float32))


# The five workloads of the exact-attention forward pass (bf16, iid N(0,1)).
WORKLOADS = {
    "tiny": Workload("tiny", "dense", 1, 1, 1, 256, 256, 64, False, 1001),
    "dense2k": Workload("dense2k", "dense", 4, 16, 16, 2048, 2048, 128, False, 1002),
    "causal8k": Workload("causal8k", "dense", 2, 32, 32, 8192, 8192, 128, True, 1003),
    "gqa16k": Workload("gqa16k", "dense", 1, 32, 8, 16384, 16384, 128, True, 1004),
    "decode": Workload("decode", "kvcache", 64, 32, 8, 1, 32768, 128, False, 1005),
    # a smaller decode case (537 MB of cache) for profiling captures
    "decode16": Workload("decode16", "kvcache", 16, 32, 8, 1, 8192, 128, False, 1006),
    # the causal 8k shape at head dimension 256 (half the heads: the same bytes per token)
    "causal8k_d256": Workload("causal8k_d256", "dense", 2, 16, 16, 8192, 8192, 256, True, 1007),
    # the decode shape at head dimension 256 (half the batch: the same cache bytes)
    "decode_d256": Workload("decode_d256", "kvcache", 32, 32, 8, 1, 32768, 256, False, 1008),
    # profiling captures: the causal 8k shape with one batch entry (192 MB of Q/K/V, above
    # the 129 MB L2) and the decode shape with 16 sequences (2.1 GB of cache)
    "causal8k_b1": Workload("causal8k_b1", "dense", 1, 32, 32, 8192, 8192, 128, True, 1009),
    "decode_b16": Workload("decode_b16", "kvcache", 16, 32, 8, 1, 32768, 128, False, 1010),
}


def bf16_normal(shape, seed: int, device="cpu", dtype=torch.bfloat16) -> torch.Tensor:
    """iid N(0,1) float32 draws from a seeded generator, rounded to bf16 (or fp16)."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return torch.randn(tuple(shape), dtype=torch.float32, generator=g, device=device).to(dtype)


def dense_inputs(B, Nq, Nk, Hq, Hkv, d, seed, device="cpu", dtype=torch.bfloat16):
    """Q [B,Nq,Hq,d], K/V [B,Nk,Hkv,d] in the (batch, seqlen, nheads, headdim) layout."""
    q = bf16_normal((B, Nq, Hq, d), seed, device, dtype)
    k = bf16_normal((B, Nk, Hkv, d), seed + 7919, device, dtype)
    v = bf16_normal((B, Nk, Hkv, d), seed + 15823, device, dtype)
    return q, k, v


def workload_inputs(w: Workload, device="cpu", seed=None, dtype=torch.bfloat16):
    s = w.seed if seed is None else seed
    return dense_inputs(w.B, w.Nq, w.Nk, w.Hq, w.Hkv, w.d, s, device, dtype)


def varlen_inputs(seqlens_q, seqlens_k, Hq, Hkv, d, seed, device="cpu", dtype=torch.bfloat16):
    """Packed Q [total_q,Hq,d], K/V [total_k,Hkv,d] and int32 prefix sums [B+1]."""
    sq = torch.tensor([0] + list(seqlens_q), dtype=torch.int64)
    sk = torch.tensor([0] + list(seqlens_k), dtype=torch.int64)
    cu_q = torch.cumsum(sq, 0).to(torch.int32)
    cu_k = torch.cumsum(sk, 0).to(torch.int32)
    tq, tk = int(cu_q[-1]), int(cu_k[-1])
    q = bf16_normal((tq, Hq, d), seed, device, dtype)
    k = bf16_normal((tk, Hkv, d), seed + 7919, device, dtype)
    v = bf16_normal((tk, Hkv, d), seed + 15823, device, dtype)
    return q, k, v, cu_q.to(device), cu_k.to(device)


def decode_lengths(B, lo=1024, hi=32768, seed=1005) -> torch.Tensor:
    """Per-sequence cache lengths, integers uniform in [lo, hi] (CPU generator)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64).to(torch.int32)


def kvcache_inputs(B, Lmax, Hq, Hkv, d, seed, lengths=None, device="cpu", poison=True,
                   dtype=torch.bfloat16):
    """Q [B,1,Hq,d], padded caches [B,Lmax,Hkv,d], lengths int32 [B].

    Rows at or past lengths[b] are NaN when ``poison`` is set.  The cache is drawn
    one batch entry at a time to bound the float32 temporary.
    """
    if lengths is None:
        lengths = decode_lengths(B, seed=seed)
    lengths = torch.as_tensor(lengths, dtype=torch.int32).cpu()
    q = bf16_normal((B, 1, Hq, d), seed, device, dtype)
    kc = torch.empty((B, Lmax, Hkv, d), dtype=dtype, device=device)
    vc = torch.empty((B, Lmax, Hkv, d), dtype=dtype, device=device)
    for b in range(B):
        kc[b] = bf16_normal((Lmax, Hkv, d), seed * 1000003 + 2 * b + 1, device, dtype)
        vc[b] = bf16_normal((Lmax, Hkv, d), seed * 1000003 + 2 * b + 2, device, dtype)
        if poison:
            n = int(lengths[b])
            kc[b, n:] = float("nan")
            vc[b, n:] = float("nan")
    return q, kc, vc, lengths.to(device)


def kvcache_workload_inputs(w: Workload, device="cpu", seed=None):
    """Inputs of a decode workload: lengths uniform in [Lmax/32, Lmax] (the decode
    workload's [1024, 32768]) from a CPU generator seeded like the tensors."""
    s = w.seed if seed is None else seed
    lens = decode_lengths(w.B, lo=max(1, w.Nk // 32), hi=w.Nk, seed=s)
    return kvcache_inputs(w.B, w.Nk, w.Hq, w.Hkv, w.d, seed=s, lengths=lens, device=device)


def kvcache_workload_entry(w: Workload, b: int, device="cpu", seed=None):
    """Batch entry b of kvcache_workload_inputs(w) without drawing the others:
    (q [1,1,Hq,d], k_cache [1,Lmax,Hkv,d], v_cache [1,Lmax,Hkv,d], length)."""
    s = w.seed if seed is None else seed
    lens = decode_lengths(w.B, lo=max(1, w.Nk // 32), hi=w.Nk, seed=s)
    q = bf16_normal((w.B, 1, w.Hq, w.d), s, device)[b:b + 1]
    kc = bf16_normal((w.Nk, w.Hkv, w.d), s * 1000003 + 2 * b + 1, device).unsqueeze(0)
    vc = bf16_normal((w.Nk, w.Hkv, w.d), s * 1000003 + 2 * b + 2, device).unsqueeze(0)
    n = int(lens[b])
    kc[0, n:] = float("nan")
    vc[0, n:] = float("nan")
    return q, kc, vc, int(lens[b])


def fp8_inputs(B, Nq, Nk, Hq, Hkv, d, seed, device="cpu", descale=0.25):
    """E4M3 Q, K, V [B, N, H, d] and their descale factors [B, Hkv]: iid N(0, 1) values
    divided by a per-(batch, kv head) factor (``descale`` times 1.0 .. 1.5) and rounded to
    torch.float8_e4m3fn, so that factor * code ~ N(0, 1).  Returns (q, k, v, dq, dk, dv)."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    fs = [descale * (1.0 + 0.5 * torch.rand((B, Hkv), generator=g)) for _ in range(3)]
    out = []
    for n, h, f in ((Nq, Hq, fs[0]), (Nk, Hkv, fs[1]), (Nk, Hkv, fs[2])):
        x = torch.randn((B, n, h, d), generator=g)
        per_head = f.repeat_interleave(h // Hkv, dim=1) if h != Hkv else f
        out.append((x / per_head[:, None, :, None]).to(torch.float8_e4m3fn).to(device))
    return (*out, *(f.to(torch.float32).to(device) for f in fs))


def kvcache_fp8_inputs(B, Lmax, Hq, Hkv, d, seed, lengths, device="cpu", poison=True,
                       descale=0.25):
    """A bf16 query [B,1,Hq,d] and E4M3 caches [B,Lmax,Hkv,d] with descale factors [B, Hkv]:
    iid N(0, 1) values divided by a per-(batch, kv head) factor (``descale`` times
    1.0 .. 1.5) and rounded to torch.float8_e4m3fn.  Rows at or past lengths[b] hold the
    E4M3 NaN code when ``poison`` is set.  Returns (q, k_cache, v_cache, lengths int32,
    k_descale, v_descale)."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    lengths = torch.as_tensor(lengths, dtype=torch.int32).cpu()
    q = torch.randn((B, 1, Hq, d), generator=g).to(torch.bfloat16)
    fs = [descale * (1.0 + 0.5 * torch.rand((B, Hkv), generator=g)) for _ in range(2)]
    caches = []
    for f in fs:
        c = torch.empty((B, Lmax, Hkv, d), dtype=torch.uint8)
        for b in range(B):  # one batch entry at a time bounds the float32 temporary
            x = torch.randn((Lmax, Hkv, d), generator=g) / f[b][None, :, None]
            c[b] = x.to(torch.float8_e4m3fn).view(torch.uint8)
            if poison:
                c[b, int(lengths[b]):] = 0x7F
        caches.append(c.view(torch.float8_e4m3fn).to(device))
    return (q.to(device), caches[0], caches[1], lengths.to(device),
            fs[0].to(torch.float32).to(device), fs[1].to(torch.float32).to(device))
