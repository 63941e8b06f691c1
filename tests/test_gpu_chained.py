"""Per-layer loads chained on one stream (hicache_plan_load_layer_chained):
each layer's kernel starts as the previous layer's drains, and each layer is
signalled by a device counter that its CTAs count into.  Every device buffer
must equal the oracle's load, each layer's count must reach its target (read
and checked before any stream wait relies on it), and the stand-in attention
behind each layer's wait must see the layer complete."""
import numpy as np
import pytest
import torch

import tiered_kv_cache_gb300 as hc
from tiered_kv_cache_gb300 import build as hc_build
from tiered_kv_cache_gb300 import workloads as wl

import gpu_helpers as gh

pytestmark = pytest.mark.gpu
TEN_S = 10_000_000


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    hc_build.build()
    torch.cuda.init()


def oracle_load(host, B, L, P, R, Hp, Dp, dp, hp, layout, sentinel=0x5A5A):
    want = [np.full((Dp * P, R), sentinel, np.uint16) for _ in range(B * L)]
    gh.orc().load(want, host.view(np.uint16), B, L, P, R, Hp, dp, hp, layout)
    return want


@pytest.mark.parametrize("layout", list(hc.LAYOUTS))
@pytest.mark.parametrize("shape", [(2, 6, 16, 128, 64, 48, 30), (1, 5, 1, 8, 9000, 9000, 4000)],
                         ids=["pages16", "one_token_pages_split_launches"])
def test_chained_layers_equal_the_oracle(layout, shape):
    B, L, P, R, Dp, Hp, n = shape
    lay = hc.LAYOUTS[layout]
    rng = np.random.default_rng(1200 + lay + n)
    dp = rng.permutation(Dp)[:n] if P == 1 else wl.fragmented_pages(rng, Dp, n)
    hp = rng.choice(Hp, n, replace=False)
    bufs = gh.random_device_bufs(B, L, P, R, Dp, seed=1200)
    kv = hc.DeviceKV(bufs, Dp)
    with hc.Pool(L, B, P, R, Hp, layout) as pool:
        host = pool.host_array(np.uint8)
        host[:] = rng.integers(0, 256, host.size, dtype=np.uint8)
        want = oracle_load(host, B, L, P, R, Hp, Dp, dp, hp, lay)
        plan = pool.plan(dp, hp, Dp, hc.LOAD)
        xfer = torch.cuda.Stream()
        for rep in range(2):
            gh.sentinel_fill(bufs)
            torch.cuda.synchronize()
            c0 = hc.launch_count()
            for layer in range(L):
                plan.load_layer_chained(kv, layer, stream=xfer)
            hc.wait(xfer, TEN_S)
            assert hc.launch_count() - c0 >= L
            for layer in range(L):
                done, target = pool.pipeline_status(layer)
                assert done == target and target > 0, (rep, layer, done, target)
            got = gh.to_np(bufs, 2)
            for k in range(B * L):
                assert np.array_equal(got[k], want[k]), (rep, k)
        # waited per layer on a compute stream, with the stand-in attention reading each layer
        gh.sentinel_fill(bufs)
        torch.cuda.synchronize()
        comp = torch.cuda.Stream()
        sums = torch.zeros(L, dtype=torch.int64, device="cuda")
        for layer in range(L):
            plan.load_layer_chained(kv, layer, stream=xfer)
            pool.wait_layer(layer, comp)
            hc.layer_checksum(kv, pool, dp, layer, sums.data_ptr() + 8 * layer, stream=comp)
        hc.wait(comp, TEN_S)
        hc.wait(xfer, TEN_S)
        after = torch.zeros_like(sums)
        for layer in range(L):
            hc.layer_checksum(kv, pool, dp, layer, after.data_ptr() + 8 * layer)
        torch.cuda.synchronize()
        assert torch.equal(sums, after)
        got = gh.to_np(bufs, 2)
        for k in range(B * L):
            assert np.array_equal(got[k], want[k]), ("waited", k)
        # and waited on each layer's CUDA event, taken right after its chained
        # call (the event fires once the layer's count is in)
        gh.sentinel_fill(bufs)
        torch.cuda.synchronize()
        sums.zero_()
        for layer in range(L):
            plan.load_layer_chained(kv, layer, stream=xfer)
            gh.stream_wait_event(comp, pool.layer_event(layer))
            hc.layer_checksum(kv, pool, dp, layer, sums.data_ptr() + 8 * layer, stream=comp)
        hc.wait(comp, TEN_S)
        hc.wait(xfer, TEN_S)
        torch.cuda.synchronize()
        assert torch.equal(sums, after), "a layer event fired before its layer landed"
        plan.close()


def test_chain_breaks_and_restarts_stay_correct():
    """Layers out of order start a new chain (a plain wait for earlier work);
    another stream is refused while the chain is open; the result is the
    oracle's load whatever the order."""
    B, L, P, R, Dp, Hp, n = 2, 5, 16, 64, 40, 40, 17
    rng = np.random.default_rng(1300)
    dp = wl.fragmented_pages(rng, Dp, n)
    hp = rng.choice(Hp, n, replace=False)
    bufs = gh.random_device_bufs(B, L, P, R, Dp, seed=1300)
    kv = hc.DeviceKV(bufs, Dp)
    with hc.Pool(L, B, P, R, Hp, "page_first") as pool:
        host = pool.host_array(np.uint8)
        host[:] = rng.integers(0, 256, host.size, dtype=np.uint8)
        want = oracle_load(host, B, L, P, R, Hp, Dp, dp, hp, hc.PAGE_FIRST)
        plan = pool.plan(dp, hp, Dp, hc.LOAD)
        s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
        gh.sentinel_fill(bufs)
        torch.cuda.synchronize()
        for layer in (0, 1, 3, 2):
            plan.load_layer_chained(kv, layer, stream=s1)
        with pytest.raises(hc.HiCacheError) as e:            # the chain on s1 is still open
            plan.load_layer_chained(kv, 4, stream=s2)
        assert e.value.status == "INVALID_ARG"
        plan.load_layer_chained(kv, 4, stream=s1)             # the last layer closes it
        hc.wait(s1, TEN_S)
        plan.load_layer_chained(kv, 0, stream=s2)             # and another stream may follow
        hc.wait(s2, TEN_S)
        got = gh.to_np(bufs, 2)
        for k in range(B * L):
            assert np.array_equal(got[k], want[k]), k
        plan.close()


def test_chained_refusals_enqueue_nothing():
    B, L, P, R, Dp, Hp = 1, 3, 16, 64, 32, 32
    base = torch.zeros((Dp * P + 16, R), dtype=torch.int16, device="cuda")
    overlapping = [base[0:Dp * P], base[16:16 + Dp * P], torch.zeros((Dp * P, R), dtype=torch.int16,
                                                                          device="cuda")]
    with hc.Pool(L, B, P, R, Hp, "layer_first") as pool:
        plan = pool.plan(np.arange(4), np.arange(4), Dp, hc.LOAD)
        before = [pool.pipeline_status(layer) for layer in range(L)]
        c0 = hc.launch_count()
        with pytest.raises(hc.HiCacheError) as e:
            plan.load_layer_chained(hc.DeviceKV(overlapping, Dp), 0)
        assert e.value.status == "INVALID_ARG" and "overlap" in str(e.value)
        ok = [torch.zeros((Dp * P, R), dtype=torch.int16, device="cuda") for _ in range(L)]
        with pytest.raises(hc.HiCacheError):
            plan.load_layer_chained(hc.DeviceKV(ok, Dp), L)
        backup_plan = pool.plan(np.arange(4), np.arange(4), Dp, hc.BACKUP)
        with pytest.raises(hc.HiCacheError):
            backup_plan.load_layer_chained(hc.DeviceKV(ok, Dp), 0)
        s = torch.cuda.Stream()
        marker = torch.zeros(1, dtype=torch.int32, device="cuda")
        g = torch.cuda.CUDAGraph()
        code = 0
        with torch.cuda.graph(g, stream=s):
            try:
                plan.load_layer_chained(hc.DeviceKV(ok, Dp), 0, stream=s)
            except hc.HiCacheError as err:
                code = err.code
            marker.add_(1)
        assert code == -1
        assert hc.launch_count() == c0
        assert [pool.pipeline_status(layer) for layer in range(L)] == before
        plan.close()
        backup_plan.close()


@pytest.mark.parametrize("layout", ["page_first", "layer_first"])
def test_chained_group_layers_equal_the_oracle(layout):
    """An MLA latent (576 bf16), an fp8 indexer key (128) and fp32 scales (4):
    one chained group launch per layer; each pool's buffers equal the oracle's
    load of that pool, and each pool's counters reach their targets."""
    lay = hc.LAYOUTS[layout]
    L, P, Dp, Hp, n = 6, 16, 48, 40, 21
    kinds = [(576, 2), (128, 1), (4, 4)]
    rng = np.random.default_rng(1400 + lay)
    dp = wl.fragmented_pages(rng, Dp, n)
    hp = rng.choice(Hp, n, replace=False)
    sizes = [L * Hp * P * R * es for R, es in kinds]
    mem = hc.PinnedHost(sum(sizes))
    pools, bufsets, kvs, off = [], [], [], 0
    for (R, es), nbytes in zip(kinds, sizes):
        pools.append(hc.Pool(L, 1, P, R, Hp, layout, elem_bytes=es, host_ptr=mem.ptr + off, host_bytes=nbytes))
        bufs = [torch.full((Dp * P, R * es), 0x77, dtype=torch.uint8, device="cuda").view(gh.TORCH_DT[es])
                for _ in range(L)]
        bufsets.append(bufs)
        kvs.append(hc.DeviceKV(bufs, Dp))
        h = pools[-1].host_array(np.uint8)
        h[:] = rng.integers(0, 256, h.size, dtype=np.uint8)
        off += nbytes
    plan = hc.group_plan(pools, dp, hp, Dp)
    xfer, comp = torch.cuda.Stream(), torch.cuda.Stream()
    sums = torch.zeros((len(kinds), L), dtype=torch.int64, device="cuda")
    torch.cuda.synchronize()
    c0 = hc.launch_count()
    for layer in range(L):
        plan.load_layer_chained(kvs, layer, stream=xfer)
    hc.wait(xfer, TEN_S)
    assert hc.launch_count() - c0 == L
    for pool in pools:
        for layer in range(L):
            done, target = pool.pipeline_status(layer)
            assert done == target and target > 0
    for layer in range(L):                      # again, waited per layer on the device
        plan.load_layer_chained(kvs, layer, stream=xfer)
        for i, (pool, kv) in enumerate(zip(pools, kvs)):
            pool.wait_layer(layer, comp)
            hc.layer_checksum(kv, pool, dp, layer, sums[i].data_ptr() + 8 * layer, stream=comp)
    hc.wait(comp, TEN_S)
    hc.wait(xfer, TEN_S)
    after = torch.zeros_like(sums)
    for i, (pool, bufs, (R, es)) in enumerate(zip(pools, bufsets, kinds)):
        want = [np.full((Dp * P, R), 0, gh.NP_DT[es]) for _ in range(L)]
        for w in want:
            w.view(np.uint8)[:] = 0x77
        gh.orc().load(want, pool.host_array(gh.NP_DT[es]), 1, L, P, R, Hp, dp, hp, lay)
        got = gh.to_np(bufs, es)
        for layer in range(L):
            assert np.array_equal(got[layer], want[layer]), (i, layer)
            hc.layer_checksum(kvs[i], pool, dp, layer, after[i].data_ptr() + 8 * layer)
    torch.cuda.synchronize()
    assert torch.equal(sums, after)
    # and waited on each pool's layer event, from sentinel-filled buffers
    for bufs in bufsets:
        for b in bufs:
            b.view(torch.uint8).fill_(0x77)
    torch.cuda.synchronize()
    ev_sums = torch.zeros_like(sums)
    for layer in range(L):
        plan.load_layer_chained(kvs, layer, stream=xfer)
        for i, (pool, kv) in enumerate(zip(pools, kvs)):
            gh.stream_wait_event(comp, pool.layer_event(layer))
            hc.layer_checksum(kv, pool, dp, layer, ev_sums[i].data_ptr() + 8 * layer, stream=comp)
    hc.wait(comp, TEN_S)
    hc.wait(xfer, TEN_S)
    torch.cuda.synchronize()
    assert torch.equal(ev_sums, after), "a layer event fired before its layer landed"
    plan.close()
    for pool in pools:
        pool.close()
    mem.free()


def test_counted_loads_share_one_stream_at_a_time():
    """Chained per-layer calls count into the same per-layer counters as
    pipelined loads, and counts from two loads cannot be told apart: a counted
    load on another stream is refused while a chain is open or a pipelined load
    is still running, and accepted once they are done."""
    B, L, P, R, Dp, Hp, n = 1, 4, 16, 64, 32, 32, 9
    rng = np.random.default_rng(1800)
    dp = rng.choice(Dp, n, replace=False)
    hp = rng.choice(Hp, n, replace=False)
    bufs = gh.random_device_bufs(B, L, P, R, Dp, seed=1800)
    kv = hc.DeviceKV(bufs, Dp)
    with hc.Pool(L, B, P, R, Hp, "page_first") as pool:
        host = pool.host_array(np.uint8)
        host[:] = rng.integers(0, 256, host.size, dtype=np.uint8)
        plan = pool.plan(dp, hp, Dp, hc.LOAD)
        s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
        for layer in range(2):                            # a chain left open on s1
            plan.load_layer_chained(kv, layer, stream=s1)
        hc.wait(s1, TEN_S)
        with pytest.raises(hc.HiCacheError) as e:
            pool.load_pipelined(kv, dp, hp, stream=s2)
        assert e.value.status == "INVALID_ARG" and "chained" in str(e.value)
        for layer in range(2, L):                         # closing the chain
            plan.load_layer_chained(kv, layer, stream=s1)
        hc.wait(s1, TEN_S)
        pool.load_pipelined(kv, dp, hp, stream=s2)        # now accepted
        hc.wait(s2, TEN_S)
        # a pipelined load still queued on s2 (behind a sleep) refuses a chain on s1
        with torch.cuda.stream(s2):
            torch.cuda._sleep(int(2e8))
        pool.load_pipelined(kv, dp, hp, stream=s2)
        with pytest.raises(hc.HiCacheError) as e:
            plan.load_layer_chained(kv, 0, stream=s1)
        assert e.value.status == "INVALID_ARG"
        hc.wait(s2, 60_000_000)
        for layer in range(L):
            plan.load_layer_chained(kv, layer, stream=s1)
        hc.wait(s1, TEN_S)
        for layer in range(L):
            done, target = pool.pipeline_status(layer)
            assert done == target, layer
        # every load moved the same pages from the same host pool: the moved rows
        # must be what the oracle's load puts there (the others are unchanged)
        got = gh.to_np(bufs, 2)
        want = [g.copy() for g in got]
        gh.orc().load(want, host.view(np.uint16), B, L, P, R, Hp, dp, hp, hc.PAGE_FIRST)
        for k in range(B * L):
            assert np.array_equal(got[k], want[k]), k
        plan.close()
