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
