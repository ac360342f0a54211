"""The multi-GPU bench path is N independent replicas: the only cross-rank
operations are the start/stop barriers and the max-over-ranks of the step time.
Exercised here with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, values, out):
    import sys
    import torch.distributed as dist
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    assert bench.dist_env() == (world, rank, rank)
    bench.barrier(world)
    out[rank] = bench.max_over_ranks(values[rank], world)
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_max_over_ranks_gloo(world):
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    values = [1.25, 3.5][:world]
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, values, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert dict(out) == {r: max(values) for r in range(world)}


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(2.0, 1) == 2.0
    bench.barrier(1)
