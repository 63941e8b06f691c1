"""Per-layer waits after seeded random sequences of every kind of load: plain
per-layer, all layers, fused backup + load, plan (one layer, all layers, graph
replay, chained), pipelined (plain and allocation-free), one-rank
tensor-parallel, and group calls.  Before each load the device buffers are
refilled with a sentinel; after it a compute stream waits for each loaded layer
(hicache_wait_layer, or the layer's CUDA event from hicache_layer_event) and
the stand-in attention adds up the layer.  Each load is held back behind a
sleep kernel on its stream, so that a wait which does not wait for it lets the
attention read the sentinel.  Every sum must be that of the loaded
data, whatever the load before it was (GB300)."""
import ctypes

import numpy as np
import pytest
import torch

import tiered_kv_cache_gb300 as hc
from tiered_kv_cache_gb300 import workloads as wl

import gpu_helpers as gh

pytestmark = pytest.mark.gpu

TEN_S = 10_000_000
KINDS = ["layer", "all", "fused", "plan_layer", "plan_all", "plan_graph", "plan_chained", "pipelined",
         "noalloc", "tp1", "group_layer", "group_all", "group_pipelined", "group_plan_all"]


@pytest.mark.parametrize("seed", range(12 * gh.SOAK))
def test_waits_after_random_loads(seed):
    rng = np.random.default_rng(7000 + seed)
    B, L, P, R, Dp, Hp, n = 1, 6, 32, 576, 96, 96, 40
    dp = wl.fragmented_pages(rng, Dp // 2, n)           # loads go below Dp / 2
    hp = np.arange(n)
    bdp, bhp = np.arange(Dp // 2, Dp // 2 + 4), np.arange(Hp - 4, Hp)    # a fused call's backup
    bufs = gh.random_device_bufs(B, L, P, R, Dp, seed=seed)
    mem = hc.PinnedHost(B * L * Hp * P * R * 2)
    pool = hc.Pool(L, B, P, R, Hp, "page_first", host_ptr=mem.ptr, host_bytes=mem.nbytes)
    host = pool.host_array(np.uint8)
    host[:] = rng.integers(0, 256, host.size, dtype=np.uint8)
    kv = hc.DeviceKV(bufs, Dp)
    want = [np.zeros((Dp * P, R), np.uint16) for _ in range(B * L)]
    gh.orc().load(want, host.view(np.uint16), B, L, P, R, Hp, dp, hp, 1)
    expect = [int(want[layer].reshape(Dp, -1)[dp].reshape(-1).view(np.uint32).astype(np.uint64)
                  .sum(dtype=np.uint64)) for layer in range(L)]
    plan = pool.plan(dp, hp, Dp, hc.LOAD)
    gplan = hc.group_plan([pool], dp, hp, Dp)
    xfer, comp = torch.cuda.Stream(), torch.cuda.Stream()

    def noalloc():
        hc._check(hc.library().hicache_load_pipelined_noalloc(
            pool.handle, ctypes.byref(kv.struct), hc._ptr(hc._idx(dp)), hc._ptr(hc._idx(hp)), len(dp),
            hc.LAYOUT_POOL, hc._stream(xfer)))

    for step in range(8):
        kind = str(rng.choice(KINDS))
        gh.sentinel_fill(bufs, 0)
        torch.cuda.synchronize()
        with torch.cuda.stream(xfer):
            torch.cuda._sleep(1_000_000)     # the load starts late: a wait that passes early reads the sentinel
        layers = list(range(L))
        if kind == "layer":
            layers = sorted(rng.choice(L, int(rng.integers(1, L + 1)), replace=False).tolist())
            for layer in layers:
                pool.load_layer(kv, dp, hp, layer, stream=xfer)
        elif kind == "all":
            pool.load(kv, dp, hp, stream=xfer)
        elif kind == "fused":
            pool.backup_load(kv, bdp, bhp, dp, hp, stream=xfer)
        elif kind == "plan_layer":
            layers = [int(rng.integers(0, L))]
            plan.execute(kv, layer=layers[0], stream=xfer)
        elif kind == "plan_all":
            plan.execute(kv, stream=xfer)
        elif kind == "plan_graph":
            plan.load_layers(kv, stream=xfer)
        elif kind == "plan_chained":
            for layer in range(L):
                plan.load_layer_chained(kv, layer, stream=xfer)
        elif kind == "pipelined":
            pool.load_pipelined(kv, dp, hp, stream=xfer)
        elif kind == "noalloc":
            noalloc()
        elif kind == "tp1":
            hc.tp_load_pipelined(pool, [kv], [pool.layer_counters()], 0, dp, hp, stream=xfer)
        elif kind == "group_layer":
            layers = [int(rng.integers(0, L))]
            hc.group_transfer([pool], [kv], dp, hp, hc.LOAD, layer=layers[0], stream=xfer)
        elif kind == "group_all":
            hc.group_transfer([pool], [kv], dp, hp, hc.LOAD, stream=xfer)
        elif kind == "group_pipelined":
            hc.group_load_pipelined([pool], [kv], dp, hp, stream=xfer)
        else:
            gplan.execute([kv], stream=xfer)
        sums = torch.zeros(L, dtype=torch.int64, device="cuda")
        by_event = bool(rng.integers(0, 2))
        for layer in layers:
            if by_event:
                gh.stream_wait_event(comp, pool.layer_event(layer))
            else:
                pool.wait_layer(layer, comp)
            hc.layer_checksum(kv, pool, dp, layer, sums.data_ptr() + 8 * layer, stream=comp)
        hc.wait(comp, TEN_S)
        hc.wait(xfer, TEN_S)
        got = sums.cpu().numpy().view(np.uint64)
        for layer in layers:
            assert int(got[layer]) == expect[layer], (seed, step, kind, by_event, layer)
    plan.close()
    gplan.close()
    pool.close()
    del host
    mem.free()
