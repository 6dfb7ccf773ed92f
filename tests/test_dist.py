"""The N > 1 path of bench.py on the CPU: two gloo ranks. Each rank runs its
own replica of the workload; the only cross-rank traffic is the timing
aggregation (barrier, max of the step times, sum of the work)."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    secs = bench.max_over_ranks(0.5 + rank, world)       # slowest rank decides the time
    work = bench.sum_over_ranks(100.0 * (rank + 1), world)  # the whole job's work
    bench.barrier(world)
    out.put((rank, secs, work))
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_rank_aggregation_over_gloo(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, secs, work in res:
        assert secs == 0.5 + (world - 1)
        assert work == 100.0 * world * (world + 1) / 2


def test_single_rank_aggregation_is_identity():
    import bench
    assert bench.max_over_ranks(1.25, 1) == 1.25
    assert bench.sum_over_ranks(3.0, 1) == 3.0
