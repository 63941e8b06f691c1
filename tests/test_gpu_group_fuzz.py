"""Seeded random buffer groups: 1-4 pools with random buffer counts, row sizes
and element sizes, random pages and operations (group calls and group plans);
every pool compared byte for byte with the oracle's transfer of that pool
(GB300)."""
import numpy as np
import pytest
import torch

import tiered_kv_cache_gb300 as hc
from tiered_kv_cache_gb300 import workloads as wl

import gpu_helpers as gh

pytestmark = pytest.mark.gpu

TEN_S = 10_000_000


def draw(seed):
    rng = np.random.default_rng(5000 + seed)
    L = int(rng.integers(1, 6))
    P = int(rng.choice([1, 2, 5, 16, 64]))
    Dp = int(rng.integers(4, 36))
    Hps = []
    kinds = []
    for _ in range(int(rng.integers(1, hc.MAX_GROUP + 1))):
        es = int(rng.choice([1, 2, 4, 8]))
        row_bytes = 16 * int(rng.choice([1, 2, 3, 8, 9, 36, 72, 128]))
        kinds.append((int(rng.integers(1, 3)), row_bytes // es, es))
        Hps.append(int(rng.integers(4, 36)))
    n = int(rng.integers(0, min(Dp, min(Hps)) + 1))
    if rng.random() < 0.5:
        dp = wl.fragmented_pages(rng, Dp, n, max_run=int(rng.integers(1, 5)))
    else:
        dp = rng.choice(Dp, n, replace=False)
    hp = rng.choice(min(Hps), n, replace=False)
    return dict(L=L, P=P, Dp=Dp, Hps=Hps, kinds=kinds, dp=dp, hp=hp, layout=int(rng.integers(0, 4)),
                op=str(rng.choice(["backup", "load", "load_layer", "pipelined", "plan_all", "plan_layer",
                                   "plan_graph"])),
                layer=int(rng.integers(0, L)))


@pytest.mark.parametrize("seed", range(150 * gh.SOAK))
def test_random_group(seed):
    c = draw(seed)
    L, P, Dp, layout, dp, hp = c["L"], c["P"], c["Dp"], c["layout"], c["dp"], c["hp"]
    rng = np.random.default_rng(seed)
    sizes = [B * L * h * P * R * es for (B, R, es), h in zip(c["kinds"], c["Hps"])]
    mem = hc.PinnedHost(sum(sizes))
    pools, bufsets, off = [], [], 0
    for (B, R, es), h, nbytes in zip(c["kinds"], c["Hps"], sizes):
        pools.append(hc.Pool(L, B, P, R, h, layout, elem_bytes=es, host_ptr=mem.ptr + off, host_bytes=nbytes))
        bufsets.append(gh.random_device_bufs(B, L, P, R, Dp, es, seed=seed * 7 + off % 31))
        off += nbytes
    kvs = [hc.DeviceKV(b, Dp) for b in bufsets]
    for pool in pools:
        pool.host_array(np.uint8)[:] = rng.integers(0, 256, pool.nbytes, dtype=np.uint8)
    torch.cuda.synchronize()
    host0 = [pool.host_array(np.uint8).copy() for pool in pools]
    dev0 = [gh.to_np(b, es) for b, (B, R, es) in zip(bufsets, c["kinds"])]
    s = torch.cuda.Stream()
    if c["op"] == "backup":
        hc.group_transfer(pools, kvs, dp, hp, hc.BACKUP, layout=layout, stream=s)
    elif c["op"] == "load":
        hc.group_transfer(pools, kvs, dp, hp, hc.LOAD, layout=layout, stream=s)
    elif c["op"] == "load_layer":
        hc.group_transfer(pools, kvs, dp, hp, hc.LOAD, layer=c["layer"], layout=layout, stream=s)
    elif c["op"] == "pipelined":
        hc.group_load_pipelined(pools, kvs, dp, hp, layout=layout, stream=s)
    else:
        plan = hc.group_plan(pools, dp, hp, Dp)
        if c["op"] == "plan_all":
            plan.execute(kvs, layout=layout, stream=s)
        elif c["op"] == "plan_layer":
            plan.execute(kvs, layer=c["layer"], layout=layout, stream=s)
        else:
            plan.load_layers(kvs, layout=layout, stream=s)
        hc.wait(s, TEN_S)
        plan.close()
    hc.wait(s, TEN_S)
    for i, (pool, bufs, (B, R, es), h) in enumerate(zip(pools, bufsets, c["kinds"], c["Hps"])):
        want_host = host0[i].view(gh.NP_DT[es]).copy()
        want_dev = [x.copy() for x in dev0[i]]
        if c["op"] == "backup":
            gh.orc().backup(dev0[i], want_host, B, L, P, R, h, dp, hp, layout)
        else:
            layer = c["layer"] if c["op"] in ("load_layer", "plan_layer") else -1
            gh.orc().load(want_dev, host0[i].view(gh.NP_DT[es]), B, L, P, R, h, dp, hp, layout, layer)
        assert np.array_equal(pool.host_array(gh.NP_DT[es]), want_host), (c, i)
        got = gh.to_np(bufs, es)
        for k in range(B * L):
            assert np.array_equal(got[k], want_dev[k]), (c, i, k)
        if c["op"] == "pipelined":
            for layer in range(L):
                done, target = pool.pipeline_status(layer)
                assert done == target, (c, i, layer)
    for pool in pools:
        pool.close()
