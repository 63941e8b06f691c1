"""The tensor-parallel load's partition (hicache_tp_share), on the CPU: the
ranks' parts tile the pairs exactly once, in the caller's order, and differ in
size by one pair at most; bad arguments are refused.  Then two gloo ranks
replay the method's data flow on host arrays -- each loads only its part with
the oracle, layer by layer, and the parts are exchanged with all_gather -- and
every rank ends with exactly the oracle's load of all the pairs."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import tiered_kv_cache_gb300 as hc


@pytest.mark.parametrize("tp", [1, 2, 3, 5, 8, 16])
def test_parts_tile_the_pairs_once_in_order(tp):
    for n in list(range(0, 40)) + [511, 512, 513, 65_537, (1 << 40) - 1]:
        parts = [hc.tp_share(n, tp, r) for r in range(tp)]
        assert parts[0][0] == 0
        for (f0, c0), (f1, _) in zip(parts, parts[1:]):
            assert f0 + c0 == f1                       # contiguous, in order
        assert parts[-1][0] + parts[-1][1] == n        # every pair once
        sizes = [c for _, c in parts]
        assert max(sizes) - min(sizes) <= 1
        assert all(c >= 0 for c in sizes)
        assert [f for f, _ in parts] == [n * r // tp for r in range(tp)]


@pytest.mark.parametrize("args", [(10, 0, 0), (10, 17, 0), (10, 4, 4), (10, 4, -1), (-1, 4, 0), (1 << 40, 2, 0)])
def test_bad_partition_arguments_are_refused(args):
    with pytest.raises(hc.HiCacheError) as e:
        hc.tp_share(*args)
    assert e.value.status == "INVALID_ARG"


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _tp_rank(rank, world, port, layout, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    o = oracle.Oracle()
    B, L, P, R, Dp, Hp, n = 1, 5, 4, 24, 40, 32, 13
    rng = np.random.default_rng(900)                  # the same draws on every rank
    host = rng.integers(0, 1 << 16, B * L * Hp * P * R, dtype=np.uint16)   # the shared, replicated latent
    dp = rng.choice(Dp, n, replace=False)
    hp = rng.choice(Hp, n, replace=False)
    mine = [np.full((Dp * P, R), 0xBEEF, np.uint16) for _ in range(B * L)]
    parts = [hc.tp_share(n, world, r) for r in range(world)]
    first, count = parts[rank]
    for layer in range(L):
        # this rank reads only its part of the layer over its host link ...
        o.load(mine, host, B, L, P, R, Hp, dp[first:first + count], hp[first:first + count], layout, layer)
        # ... and the parts reach every rank (all_gather of each rank's loaded rows)
        rows = mine[layer].reshape(Dp, P * R)[dp[first:first + count]]
        got = [None] * world
        dist.all_gather_object(got, rows)
        for q, (fq, cq) in enumerate(parts):
            if cq:
                mine[layer].reshape(Dp, P * R)[dp[fq:fq + cq]] = got[q]
    want = [np.full((Dp * P, R), 0xBEEF, np.uint16) for _ in range(B * L)]
    o.load(want, host, B, L, P, R, Hp, dp, hp, layout)
    out[rank] = all(np.array_equal(a, b) for a, b in zip(mine, want))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("layout", [0, 1, 2, 3])
def test_two_ranks_partition_and_gather_equal_the_full_load(layout):
    world, port = 2, _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_tp_rank, args=(world, port, layout, out), nprocs=world, join=True)
        res = dict(out)
    assert res == {0: True, 1: True}
