"""CPU tests of the seeded input generators (no attention arithmetic involved)."""
import torch

from exact_attention_81_gb300.inputs import (Workload, decode_lengths, kvcache_workload_entry,
                                             kvcache_workload_inputs)


def test_decode_entry_matches_full_draw():
    w = Workload("t", "kvcache", 5, 8, 2, 1, 640, 64, False, 77)
    q, kc, vc, lens = kvcache_workload_inputs(w)
    for b in (0, 3, 4):
        qb, kb, vb, n = kvcache_workload_entry(w, b)
        assert n == int(lens[b])
        assert torch.equal(qb, q[b:b + 1])
        assert torch.equal(kb[:, :n], kc[b:b + 1, :n]) and torch.equal(vb[:, :n], vc[b:b + 1, :n])
        assert torch.isnan(kb[:, n:].float()).all() and torch.isnan(kc[b, n:].float()).all()


def test_decode_lengths_range_and_seed():
    a = decode_lengths(64, seed=1005)
    assert torch.equal(a, decode_lengths(64, seed=1005))
    assert int(a.min()) >= 1024 and int(a.max()) <= 32768
