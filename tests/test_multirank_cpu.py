"""The N > 1 path of bench.py on CPU: two gloo ranks (the driver launches one process per
GPU under torchrun).  Each rank runs the whole workload (weak scaling, no collective on the
data path); the job's step time is the slowest rank's and the job value counts every
rank's work."""
import multiprocessing as mp
import os
import socket

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [1.5, 2.0][rank]  # rank 1 is the slow one
    ms = bench.max_over_ranks(local_ms, dist, "cpu")
    value = bench.job_value(1.0e12, ms, world, 1e12)
    dist.barrier()
    dist.destroy_process_group()
    out.put((rank, ms, value))


def test_two_ranks_max_time_and_weak_scaling_value():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, value in results:
        assert ms == pytest.approx(2.0)              # slowest rank
        assert value == pytest.approx(2 * 1.0 / 2.0e-3)  # 2 ranks x 1 TFLOP per 2 ms


def test_single_process_is_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.25, None, "cpu") == 1.25
    assert bench.job_value(5e11, 1.0, 1, 1e12) == pytest.approx(500.0)


def _shard_worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    from exact_attention_81_gb300.inputs import WORKLOADS
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = bench.shard_workload(WORKLOADS["causal8k"], world, rank)
    local_ms = [0.5, 0.4][rank]
    ms = bench.max_over_ranks(local_ms, dist, "cpu")
    value = bench.job_value(bench.flops(w), ms, world, 1e12)
    dist.barrier()
    dist.destroy_process_group()
    out.put((rank, w.Hq, w.Hkv, w.seed, bench.flops(w), ms, value))


def test_two_ranks_head_sharding_strong_scaling():
    """--shard: each rank takes half the kv heads (and their query heads) of the one
    workload; the job value is the whole workload's FLOPs over the slowest rank's time."""
    import sys
    sys.path.insert(0, ROOT)
    import bench
    from exact_attention_81_gb300.inputs import WORKLOADS
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    total = bench.flops(WORKLOADS["causal8k"])
    assert sum(r[4] for r in results) == pytest.approx(total)
    assert {r[1] for r in results} == {16} and {r[2] for r in results} == {16}
    assert results[0][3] != results[1][3]  # own inputs per rank
    for rank, hq, hkv, seed, work, ms, value in results:
        assert ms == pytest.approx(0.5)
        assert value == pytest.approx(total / 0.5e-3 / 1e12)


@pytest.mark.parametrize("name,world", [("causal8k", 8), ("gqa16k", 8), ("decode", 4),
                                        ("dense2k", 4)])
def test_shards_partition_the_heads(name, world):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    from exact_attention_81_gb300.inputs import WORKLOADS
    w = WORKLOADS[name]
    parts = [bench.shard_workload(w, world, r) for r in range(world)]
    assert sum(p.Hkv for p in parts) == w.Hkv and sum(p.Hq for p in parts) == w.Hq
    assert all(p.Hq // p.Hkv == w.Hq // w.Hkv for p in parts)  # groups stay whole
    with pytest.raises(ValueError):
        bench.shard_workload(w, w.Hkv + 1, 0)
