"""Seeded random sequences of every kind of call -- backup, load, per-layer
load, pipelined (plain and allocation-free), fused backup + load, plans
(per-layer, chained per-layer, graph replay), group calls and group plans
(graph replay, chained per-layer), a one-rank tensor-parallel load -- on two
pools that share the page numbering, all on one stream.
A shadow copy of the device buffers and host pools is updated by the oracle in
the same order; at the end every byte must agree (GB300)."""
import ctypes

import numpy as np
import pytest
import torch

import tiered_kv_cache_gb300 as hc

import gpu_helpers as gh

pytestmark = pytest.mark.gpu

TEN_S = 10_000_000
OPS = ["backup", "load", "load_layer", "pipelined", "noalloc", "fused", "plan_layers", "plan_graph",
       "plan_chained", "tp1", "group_backup", "group_load", "group_layer", "group_pipelined",
       "group_plan_graph", "group_plan_chained"]


def _noalloc(pool, kv, dp, hp, stream):
    rc = hc.library().hicache_load_pipelined_noalloc(pool.handle, ctypes.byref(kv.struct),
                                                     hc._ptr(hc._idx(dp)), hc._ptr(hc._idx(hp)), len(dp),
                                                     hc.LAYOUT_POOL, hc._stream(stream))
    hc._check(rc)


@pytest.mark.parametrize("seed", range(100 * gh.SOAK))
def test_random_call_sequence(seed):
    rng = np.random.default_rng(9000 + seed)
    L, P, Dp, Hp = int(rng.integers(1, 5)), int(rng.choice([1, 4, 16])), 24, 24
    layout = int(rng.integers(0, 4))
    kinds = [(int(rng.integers(1, 3)), 64, 2), (1, 16 * int(rng.integers(1, 4)), 1)]
    sizes = [B * L * Hp * P * R * es for B, R, es in kinds]
    mem = hc.PinnedHost(sum(sizes))
    pools, bufsets, off = [], [], 0
    for (B, R, es), nbytes in zip(kinds, sizes):
        pools.append(hc.Pool(L, B, P, R, Hp, layout, elem_bytes=es, host_ptr=mem.ptr + off, host_bytes=nbytes))
        bufsets.append(gh.random_device_bufs(B, L, P, R, Dp, es, seed=seed * 11 + off % 13))
        off += nbytes
    kvs = [hc.DeviceKV(b, Dp) for b in bufsets]
    for pool in pools:
        pool.host_array(np.uint8)[:] = rng.integers(0, 256, pool.nbytes, dtype=np.uint8)
    torch.cuda.synchronize()
    dev = [gh.to_np(b, es) for b, (B, R, es) in zip(bufsets, kinds)]
    host = [pool.host_array(gh.NP_DT[es]).copy() for pool, (B, R, es) in zip(pools, kinds)]
    o = gh.orc()
    st = torch.cuda.Stream()

    def shadow(i, op, dp, hp, layer=-1):
        B, R, es = kinds[i]
        if op == "backup":
            o.backup(dev[i], host[i], B, L, P, R, Hp, dp, hp, layout)
        else:
            o.load(dev[i], host[i], B, L, P, R, Hp, dp, hp, layout, layer)

    def pairs(n):
        return rng.permutation(Dp)[:n], rng.permutation(Hp)[:n]

    plans = []
    for step in range(30):
        op = str(rng.choice(OPS))
        i = int(rng.integers(0, 2))
        pool, kv = pools[i], kvs[i]
        dp, hp = pairs(int(rng.integers(0, 10)))
        layer = int(rng.integers(0, L))
        if op == "backup":
            pool.backup(kv, dp, hp, stream=st)
            shadow(i, "backup", dp, hp)
        elif op == "load":
            pool.load(kv, dp, hp, stream=st)
            shadow(i, "load", dp, hp)
        elif op == "load_layer":
            pool.load_layer(kv, dp, hp, layer, stream=st)
            shadow(i, "load", dp, hp, layer)
        elif op == "pipelined":
            pool.load_pipelined(kv, dp, hp, stream=st)
            shadow(i, "load", dp, hp)
        elif op == "noalloc":
            _noalloc(pool, kv, dp, hp, st)
            shadow(i, "load", dp, hp)
        elif op == "fused":
            # a backup and a load with no page in common on either side
            d, h = rng.permutation(Dp), rng.permutation(Hp)
            k = int(rng.integers(0, 8))
            pool.backup_load(kv, d[:k], h[:k], d[k:2 * k], h[k:2 * k], stream=st)
            shadow(i, "backup", d[:k], h[:k])
            shadow(i, "load", d[k:2 * k], h[k:2 * k])
        elif op == "plan_layers":
            plan = pool.plan(dp, hp, Dp, hc.LOAD)
            for l in rng.permutation(L)[:int(rng.integers(1, L + 1))]:
                plan.load_layer(kv, int(l), stream=st)
                shadow(i, "load", dp, hp, int(l))
            plan.close()
        elif op == "plan_graph":
            plan = pool.plan(dp, hp, Dp, hc.LOAD)
            for _ in range(int(rng.integers(1, 3))):
                plan.load_layers(kv, stream=st)
                shadow(i, "load", dp, hp)
            plans.append(plan)                 # kept until the stream is done
        elif op == "plan_chained":
            # layers first..last in order, one chained call each: a chain from
            # layer 0, or calls that start mid-way (each a new chain)
            plan = pool.plan(dp, hp, Dp, hc.LOAD)
            first = 0 if rng.random() < 0.7 else int(rng.integers(0, L))
            last = int(rng.integers(first, L))
            for l in range(first, last + 1):
                plan.load_layer_chained(kv, l, stream=st)
                shadow(i, "load", dp, hp, l)
            plans.append(plan)                 # kept until the stream is done
        elif op == "tp1":
            # a tensor-parallel load with this pool as the group's only rank
            hc.tp_load_pipelined(pool, [kv], [pool.layer_counters()], 0, dp, hp, stream=st)
            shadow(i, "load", dp, hp)
        elif op == "group_backup":
            hc.group_transfer(pools, kvs, dp, hp, hc.BACKUP, stream=st)
            shadow(0, "backup", dp, hp)
            shadow(1, "backup", dp, hp)
        elif op == "group_load":
            hc.group_transfer(pools, kvs, dp, hp, hc.LOAD, stream=st)
            shadow(0, "load", dp, hp)
            shadow(1, "load", dp, hp)
        elif op == "group_layer":
            hc.group_transfer(pools, kvs, dp, hp, hc.LOAD, layer=layer, stream=st)
            shadow(0, "load", dp, hp, layer)
            shadow(1, "load", dp, hp, layer)
        elif op == "group_pipelined":
            hc.group_load_pipelined(pools, kvs, dp, hp, stream=st)
            shadow(0, "load", dp, hp)
            shadow(1, "load", dp, hp)
        elif op == "group_plan_chained":
            gplan = hc.group_plan(pools, dp, hp, Dp)
            for l in range(0, int(rng.integers(0, L)) + 1):
                gplan.load_layer_chained(kvs, l, stream=st)
                shadow(0, "load", dp, hp, l)
                shadow(1, "load", dp, hp, l)
            plans.append(gplan)                # kept until the stream is done
        else:
            gplan = hc.group_plan(pools, dp, hp, Dp)
            gplan.load_layers(kvs, stream=st)
            shadow(0, "load", dp, hp)
            shadow(1, "load", dp, hp)
            plans.append(gplan)                # kept until the stream is done
    hc.wait(st, TEN_S)
    for plan in plans:
        plan.close()
    for i, (pool, bufs, (B, R, es)) in enumerate(zip(pools, bufsets, kinds)):
        assert np.array_equal(pool.host_array(gh.NP_DT[es]), host[i]), (seed, i)
        got = gh.to_np(bufs, es)
        for k in range(B * L):
            assert np.array_equal(got[k], dev[i][k]), (seed, i, k)
        for layer in range(L):
            done, target = pool.pipeline_status(layer)
            assert done == target, (seed, i, layer)
    for pool in pools:
        pool.close()
