"""Pipelined loads: every layer in one launch, each layer signalled on the
device as it lands.  The counting is checked first without any wait; the
tests that wait on it use a bounded host wait, so a counting error fails a
test instead of blocking a stream for good."""
import numpy as np
import pytest
import torch

import tiered_kv_cache_gb300 as hc
from tiered_kv_cache_gb300 import build as hc_build
from tiered_kv_cache_gb300 import workloads as wl

import gpu_helpers as gh

pytestmark = pytest.mark.gpu
LAYOUTS = list(hc.LAYOUTS.values())
TEN_S = 10_000_000


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    hc_build.build()
    torch.cuda.init()


@pytest.mark.parametrize("layout", LAYOUTS, ids=list(hc.LAYOUTS))
def test_pipelined_load_parity_and_counts(layout):
    B, L, P, R, Dp, Hp, n = 2, 5, 16, 128, 64, 64, 30
    rng = np.random.default_rng(300 + layout)
    dp = wl.fragmented_pages(rng, Dp, n)
    hp = rng.choice(Hp, n, replace=False)
    bufs = gh.random_device_bufs(B, L, P, R, Dp, seed=300)
    with hc.Pool(L, B, P, R, Hp, layout) as pool:
        host = pool.host_array(np.uint8)
        host[:] = rng.integers(0, 256, host.size, dtype=np.uint8)
        gh.sentinel_fill(bufs)
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        c0 = hc.launch_count()
        for rep in range(2):                   # the counts accumulate over loads
            pool.load_pipelined(hc.DeviceKV(bufs, Dp), dp, hp, stream=s)
        s.synchronize()
        assert hc.launch_count() - c0 == 2
        targets = set()
        for layer in range(L):
            done, target = pool.pipeline_status(layer)
            assert done == target and target > 0, (layer, done, target)
            targets.add(target)
        assert len(targets) == 1               # every layer has the same tiles
        want = [np.full((Dp * P, R), 0x5A5A, np.uint16) for _ in range(B * L)]
        gh.orc().load(want, host.view(np.uint16), B, L, P, R, Hp, dp, hp, layout)
        got = gh.to_np(bufs, 2)
        for k in range(B * L):
            assert np.array_equal(got[k], want[k])


def test_compute_waits_for_each_layer():
    """The stand-in attention on a second stream, behind wait_layer per layer,
    sees every layer fully loaded; the transfer is one launch."""
    B, L, P, R, Dp, Hp, n = 1, 12, 64, 576, 128, 128, 100
    rng = np.random.default_rng(310)
    dp = wl.fragmented_pages(rng, Dp, n)
    hp = np.arange(n)
    bufs = gh.random_device_bufs(B, L, P, R, Dp, seed=310)
    with hc.Pool(L, B, P, R, Hp, "page_first") as pool:
        host = pool.host_array(np.uint8)
        host[:] = rng.integers(0, 256, host.size, dtype=np.uint8)
        gh.sentinel_fill(bufs, 0)
        torch.cuda.synchronize()
        kv = hc.DeviceKV(bufs, Dp)
        xfer, comp = torch.cuda.Stream(), torch.cuda.Stream()
        sums = torch.zeros(L, dtype=torch.int64, device="cuda")
        plan = pool.plan(dp, hp, Dp, hc.LOAD)
        c0 = hc.launch_count()
        plan.load_pipelined(kv, stream=xfer)
        assert hc.launch_count() - c0 == 1
        for layer in range(L):
            pool.wait_layer(layer, comp)
            hc.layer_checksum(kv, pool, dp, layer, sums.data_ptr() + 8 * layer, stream=comp)
        hc.wait(comp, TEN_S)
        hc.wait(xfer, TEN_S)
        want = [np.zeros((Dp * P, R), np.uint16) for _ in range(B * L)]
        gh.orc().load(want, host.view(np.uint16), B, L, P, R, Hp, dp, hp, 1)
        got = sums.cpu().numpy().view(np.uint64)
        for layer in range(L):
            words = want[layer].reshape(Dp, -1)[dp].reshape(-1).view(np.uint32)
            assert int(got[layer]) == int(words.astype(np.uint64).sum(dtype=np.uint64)), layer
        plan.close()


def test_layer_events_of_counted_loads():
    """After a pipelined load (and an allocation-free one), each layer's event,
    asked for right after the call, holds the stand-in attention until that
    layer has landed; after a plain per-layer load it is that load's event."""
    import ctypes
    B, L, P, R, Dp, Hp, n = 1, 12, 64, 576, 128, 128, 100
    rng = np.random.default_rng(330)
    dp = wl.fragmented_pages(rng, Dp, n)
    hp = np.arange(n)
    bufs = gh.random_device_bufs(B, L, P, R, Dp, seed=330)
    with hc.Pool(L, B, P, R, Hp, "page_first") as pool:
        host = pool.host_array(np.uint8)
        host[:] = rng.integers(0, 256, host.size, dtype=np.uint8)
        kv = hc.DeviceKV(bufs, Dp)
        want = [np.zeros((Dp * P, R), np.uint16) for _ in range(B * L)]
        gh.orc().load(want, host.view(np.uint16), B, L, P, R, Hp, dp, hp, 1)
        expect = [int(want[layer].reshape(Dp, -1)[dp].reshape(-1).view(np.uint32).astype(np.uint64)
                      .sum(dtype=np.uint64)) for layer in range(L)]
        xfer, comp = torch.cuda.Stream(), torch.cuda.Stream()

        def noalloc():
            hc._check(hc.library().hicache_load_pipelined_noalloc(
                pool.handle, ctypes.byref(kv.struct), hc._ptr(hc._idx(dp)), hc._ptr(hc._idx(hp)), len(dp),
                hc.LAYOUT_POOL, hc._stream(xfer)))

        for load in (lambda: pool.load_pipelined(kv, dp, hp, stream=xfer), noalloc,
                     lambda: [pool.load_layer(kv, dp, hp, layer, stream=xfer) for layer in range(L)]):
            gh.sentinel_fill(bufs, 0)
            torch.cuda.synchronize()
            sums = torch.zeros(L, dtype=torch.int64, device="cuda")
            with torch.cuda.stream(xfer):
                torch.cuda._sleep(1_000_000)     # the load starts late: an early wait reads the sentinel
            load()
            for layer in range(L):
                gh.stream_wait_event(comp, pool.layer_event(layer))
                hc.layer_checksum(kv, pool, dp, layer, sums.data_ptr() + 8 * layer, stream=comp)
            hc.wait(comp, TEN_S)
            hc.wait(xfer, TEN_S)
            got = sums.cpu().numpy().view(np.uint64)
            assert [int(x) for x in got] == expect


def test_waits_follow_a_load_of_every_layer():
    """A load of every layer -- hicache_load, a fused backup + load, a plan's
    or a group's load of every layer -- is the last load of each layer: after
    an earlier pipelined load (whose counts are all in), hicache_wait_layer and
    the layer event both hold the stand-in attention until the new load is in."""
    B, L, P, R, Dp, Hp, n = 1, 12, 64, 576, 256, 256, 100
    rng = np.random.default_rng(350)
    dp = wl.fragmented_pages(rng, Dp // 2, n)             # loads: device pages below Dp / 2
    hp = np.arange(n)
    bdp, bhp = np.arange(Dp // 2, Dp // 2 + 8), np.arange(Hp - 8, Hp)   # the fused call's backup
    bufs = gh.random_device_bufs(B, L, P, R, Dp, seed=350)
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
    loads = {
        "load": lambda: pool.load(kv, dp, hp, stream=xfer),
        "backup_load": lambda: pool.backup_load(kv, bdp, bhp, dp, hp, stream=xfer),
        "plan": lambda: plan.execute(kv, stream=xfer),
        "group": lambda: hc.group_transfer([pool], [kv], dp, hp, hc.LOAD, stream=xfer),
        "group_plan": lambda: gplan.execute([kv], stream=xfer),
    }
    for name, load in loads.items():
        for by_event in (False, True):
            pool.load_pipelined(kv, dp, hp, stream=xfer)       # counts met: a stale wait passes at once
            hc.wait(xfer, TEN_S)
            gh.sentinel_fill(bufs, 0)
            torch.cuda.synchronize()
            sums = torch.zeros(L, dtype=torch.int64, device="cuda")
            with torch.cuda.stream(xfer):
                torch.cuda._sleep(1_000_000)     # the load starts late: an early wait reads the sentinel
            load()
            for layer in range(L):
                if by_event:
                    gh.stream_wait_event(comp, pool.layer_event(layer))
                else:
                    pool.wait_layer(layer, comp)
                hc.layer_checksum(kv, pool, dp, layer, sums.data_ptr() + 8 * layer, stream=comp)
            hc.wait(comp, TEN_S)
            hc.wait(xfer, TEN_S)
            got = sums.cpu().numpy().view(np.uint64)
            assert [int(x) for x in got] == expect, (name, by_event)
    plan.close()
    gplan.close()
    pool.close()
    del host
    mem.free()


def test_wait_layer_follows_the_last_load_kind_and_stream_rule():
    B, L, P, R, Dp, Hp = 1, 3, 4, 64, 8, 8
    bufs = [torch.zeros((Dp * P, R), dtype=torch.int16, device="cuda") for _ in range(B * L)]
    with hc.Pool(L, B, P, R, Hp, "layer_first") as pool:
        pool.host_array()[:] = 7
        kv = hc.DeviceKV(bufs, Dp)
        s1, s2, comp = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        with torch.cuda.stream(s1):
            torch.cuda._sleep(int(2e8))                     # keep s1 busy for ~0.1 s
        pool.load_pipelined(kv, [1], [2], stream=s1)
        with pytest.raises(hc.HiCacheError) as e:          # still running on s1: not on s2
            pool.load_pipelined(kv, [1], [2], stream=s2)
        assert e.value.status == "INVALID_ARG"
        pool.load_layer(kv, [3], [4], 1, stream=s2)         # an event-signalled load of layer 1
        for layer in range(L):
            pool.wait_layer(layer, comp)
        with torch.cuda.stream(comp):
            a = torch.stack([b[1 * P:2 * P].sum() for b in bufs])
            c = bufs[1][3 * P:4 * P].sum()
        hc.wait(comp, TEN_S)
        assert torch.all(a == 7 * P * R) and int(c) == 7 * P * R
        hc.wait(s1, TEN_S)
        pool.load_pipelined(kv, [5], [2], stream=s2)        # s1's load is done: s2 may go on
        for layer in range(L):
            pool.wait_layer(layer, comp)
        with torch.cuda.stream(comp):
            d = torch.stack([b[5 * P:6 * P].sum() for b in bufs])
        hc.wait(comp, TEN_S)
        assert torch.all(d == 7 * P * R)


def test_pipelined_load_split_over_several_launches():
    """4,000 scattered one-token pages are more runs than one launch holds: the
    pipelined load is split, each launch adds its tiles to every layer's count,
    and each layer is waited for correctly."""
    B, L, P, R, Dp, Hp, n = 2, 3, 1, 8, 9000, 9000, 4000
    rng = np.random.default_rng(320)
    dp, hp = rng.permutation(Dp)[:n], rng.permutation(Hp)[:n]
    bufs = gh.random_device_bufs(B, L, P, R, Dp, seed=320)
    with hc.Pool(L, B, P, R, Hp, "page_first_direct") as pool:
        host = pool.host_array(np.uint8)
        host[:] = rng.integers(0, 256, host.size, dtype=np.uint8)
        gh.sentinel_fill(bufs, 0)
        torch.cuda.synchronize()
        kv = hc.DeviceKV(bufs, Dp)
        xfer, comp = torch.cuda.Stream(), torch.cuda.Stream()
        c0 = hc.launch_count()
        pool.load_pipelined(kv, dp, hp, stream=xfer)
        assert hc.launch_count() - c0 >= 3
        hc.wait(xfer, TEN_S)
        for layer in range(L):
            done, target = pool.pipeline_status(layer)
            assert done == target > 0
        want = [np.zeros((Dp * P, R), np.uint16) for _ in range(B * L)]
        gh.orc().load(want, host.view(np.uint16), B, L, P, R, Hp, dp, hp, 2)
        got = gh.to_np(bufs, 2)
        for k in range(B * L):
            assert np.array_equal(got[k], want[k])
        sums = torch.zeros(L, dtype=torch.int64, device="cuda")
        for layer in range(L):
            pool.wait_layer(layer, comp)
            hc.layer_checksum(kv, pool, dp, layer, sums.data_ptr() + 8 * layer, stream=comp)
        hc.wait(comp, TEN_S)
        got_s = sums.cpu().numpy().view(np.uint64)
        for layer in range(L):
            words = np.concatenate([want[b * L + layer].reshape(Dp, -1)[dp].reshape(-1).view(np.uint32)
                                    for b in range(B)])
            assert int(got_s[layer]) == int(words.astype(np.uint64).sum(dtype=np.uint64))


@pytest.mark.parametrize("ctas", [1, 7, 300])
def test_tile_counter_covers_every_tile_and_resets(ctas):
    """CTAs take tiles from the pool's scheduler word: with 1, 7 or 300 CTAs
    every tile is moved, and three loads in a row each start from tile 0 (a
    scheduler left non-zero would skip the first tiles of the next load)."""
    B, L, P, R, Dp, Hp, n = 2, 6, 8, 256, 96, 96, 40
    rng = np.random.default_rng(700 + ctas)
    bufs = gh.random_device_bufs(B, L, P, R, Dp, seed=701)
    with hc.Pool(L, B, P, R, Hp, "page_first", launch_ctas=ctas) as pool:
        host = pool.host_array(np.uint8)
        kv = hc.DeviceKV(bufs, Dp)
        s = torch.cuda.Stream()
        for call in range(3):
            dp, hp = rng.permutation(Dp)[:n], rng.permutation(Hp)[:n]
            host[:] = rng.integers(0, 256, host.size, dtype=np.uint8)
            gh.sentinel_fill(bufs)
            torch.cuda.synchronize()
            pool.load_pipelined(kv, dp, hp, stream=s)
            hc.wait(s, TEN_S)
            want = [np.full((Dp * P, R), 0x5A5A, np.uint16) for _ in range(B * L)]
            gh.orc().load(want, host.view(np.uint16), B, L, P, R, Hp, dp, hp, 1)
            got = gh.to_np(bufs, 2)
            for k in range(B * L):
                assert np.array_equal(got[k], want[k]), (call, k)
            for layer in range(L):
                done, target = pool.pipeline_status(layer)
                assert done == target


def test_pipelined_loads_refuse_a_capturing_stream():
    """A pipelined load raises each layer's target on the host when it is
    enqueued, so a captured call (replayed any number of times, or never) would
    leave the per-layer waits wrong.  Every pipelined entry point refuses a
    capturing stream with INVALID_ARG and enqueues nothing."""
    B, L, P, R, Dp, Hp, n = 1, 3, 16, 64, 32, 32, 8
    rng = np.random.default_rng(330)
    dp = rng.choice(Dp, n, replace=False)
    hp = rng.choice(Hp, n, replace=False)
    bufs = gh.random_device_bufs(B, L, P, R, Dp, seed=330)
    kv = hc.DeviceKV(bufs, Dp)
    with hc.Pool(L, B, P, R, Hp, "page_first") as pool:
        s = torch.cuda.Stream()
        pool.load_pipelined(kv, dp, hp, stream=s)          # a plain call first
        s.synchronize()
        plan = pool.plan(dp, hp, Dp, hc.LOAD)
        before = [pool.pipeline_status(layer) for layer in range(L)]
        marker = torch.zeros(1, dtype=torch.int32, device="cuda")
        torch.cuda.synchronize()
        c0 = hc.launch_count()
        codes = []
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for call in (lambda: pool.load_pipelined(kv, dp, hp, stream=s),
                         lambda: plan.load_pipelined(kv, stream=s),
                         lambda: hc.group_load_pipelined([pool], [kv], dp, hp, stream=s)):
                try:
                    call()
                    codes.append(0)
                except hc.HiCacheError as e:
                    codes.append(e.code)
            marker.add_(1)                                 # keeps the captured graph non-empty
        assert codes == [-1, -1, -1]
        assert hc.launch_count() == c0
        g.replay()
        torch.cuda.synchronize()
        assert int(marker.item()) == 1
        assert [pool.pipeline_status(layer) for layer in range(L)] == before
        plan.close()


def test_a_captured_load_of_every_layer_leaves_the_waits():
    """hicache_load captured into a CUDA graph: the replay moves the pages,
    and the per-layer waits still refer to the last load enqueued outside the
    capture (they neither fail nor wait on the graph)."""
    B, L, P, R, Dp, Hp, n = 1, 4, 16, 64, 48, 48, 10
    rng = np.random.default_rng(360)
    dp = rng.permutation(Dp)[:n]
    hp = np.arange(n)
    bufs = gh.random_device_bufs(B, L, P, R, Dp, seed=360)
    with hc.Pool(L, B, P, R, Hp, "page_first") as pool:
        host = pool.host_array(np.uint8)
        host[:] = rng.integers(0, 256, host.size, dtype=np.uint8)
        kv = hc.DeviceKV(bufs, Dp)
        s, comp = torch.cuda.Stream(), torch.cuda.Stream()
        pool.load_layer(kv, dp, hp, 0, stream=s)
        torch.cuda.synchronize()
        gh.sentinel_fill(bufs, 0)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            pool.load(kv, dp, hp, stream=s)
        g.replay()
        torch.cuda.synchronize()
        for layer in range(L):
            pool.wait_layer(layer, comp)
            gh.stream_wait_event(comp, pool.layer_event(layer))
        comp.synchronize()
        want = [np.zeros((Dp * P, R), np.uint16) for _ in range(B * L)]
        gh.orc().load(want, host.view(np.uint16), B, L, P, R, Hp, dp, hp, 1)
        got = gh.to_np(bufs, 2)
        for k in range(B * L):
            assert np.array_equal(got[k], want[k]), k
