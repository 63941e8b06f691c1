"""bench.py's multi-rank aggregation on CPU: two gloo ranks, each a replica with
its own time; every rank must see the slowest time and the whole-job rate."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    m = bench.max_over_ranks(times[rank], world)
    v = bench.whole_job_gbs(8e9, m, world)
    out[rank] = (m, v)
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_max_over_ranks_and_whole_job_rate(world):
    times = [0.5, 0.8]
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank, args=(world, port, times, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        m, v = res[r]
        assert m == pytest.approx(0.8)
        assert v == pytest.approx(world * 8e9 / 0.8 / 1e9)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(1.25, 1) == 1.25
    assert bench.whole_job_gbs(2e9, 1.0, 1) == pytest.approx(2.0)
