"""The multi-rank bench path on CPU: two gloo ranks, each with its own step
time, agree on the slowest rank's time and on the whole-job throughput."""

import os

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [2.0, 3.0][rank]
    ms_max, value = bench.aggregate_over_ranks(ms, 6.0, world)
    out[rank] = (ms_max, value)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation():
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    # both ranks see the max time (3 ms) and 2 ranks x 6 units / 3 ms
    for r in range(2):
        assert res[r][0] == pytest.approx(3.0)
        assert res[r][1] == pytest.approx(2 * 6.0 / 3e-3)


def test_single_rank_aggregation():
    import bench
    assert bench.aggregate_over_ranks(4.0, 8.0, 1) == (4.0, 2000.0)
