"""GPU path vs the oracle, element by element, through the C ABI (GB300).

Small shapes compare whole pools; they span several 16 KiB tiles with ragged
tails, rows of 16 B to 2 KiB, 1-, 2- and 4-byte elements, one to three buffers,
every layout, backup / load / per-layer load / plans.  The five workload shapes
are checked at their full sizes in test_gpu_workloads.py."""
import numpy as np
import pytest
import torch

import tiered_kv_cache_gb300 as hc
from tiered_kv_cache_gb300 import build as hc_build
from tiered_kv_cache_gb300 import workloads as wl

import fullsize as fs
import gpu_helpers as gh

pytestmark = pytest.mark.gpu

LAYOUTS = list(hc.LAYOUTS.values())


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    hc_build.build()
    torch.cuda.init()


# (name, B, L, P, R, es, Dp, Hp, n, pattern)
SHAPES = [
    ("gqa_p16", 2, 2, 16, 128, 2, 64, 128, 12, "random"),
    ("mla_like", 1, 5, 8, 576, 2, 40, 48, 17, "runs"),
    ("row16B_3buf", 3, 3, 3, 8, 2, 30, 31, 11, "random"),
    ("fp8_rows48B", 2, 4, 5, 48, 1, 24, 24, 9, "runs"),
    ("fp32_rows48B", 2, 3, 4, 12, 4, 24, 26, 8, "random"),
    ("ragged_tiles", 2, 2, 64, 72, 2, 60, 64, 40, "contiguous"),
    ("one_layer", 2, 1, 16, 64, 2, 32, 32, 10, "runs"),
    ("one_token_pages", 1, 6, 1, 256, 2, 64, 80, 33, "random"),
]


def indices(pattern, Dp, Hp, n, seed):
    rng = np.random.default_rng(seed)
    if pattern == "random":
        return rng.choice(Dp, n, replace=False), rng.choice(Hp, n, replace=False)
    if pattern == "contiguous":
        return np.arange(n) + (Dp - n) // 2, np.arange(n) + 1
    dp = wl.fragmented_pages(rng, Dp, n, max_run=4)
    hp = np.sort(rng.choice(Hp, n, replace=False))
    hp[: n // 2] = np.arange(n // 2) + 2      # half of it contiguous on the host too
    hp = np.unique(hp)
    while len(hp) < n:
        extra = rng.choice(Hp, n - len(hp), replace=False)
        hp = np.unique(np.concatenate([hp, extra]))
    return dp, hp[:n]


@pytest.mark.parametrize("shape", SHAPES, ids=[s[0] for s in SHAPES])
@pytest.mark.parametrize("layout", LAYOUTS, ids=list(hc.LAYOUTS))
def test_backup_load_parity(shape, layout):
    name, B, L, P, R, es, Dp, Hp, n, pattern = shape
    dp, hp = indices(pattern, Dp, Hp, n, seed=len(name) + layout)
    bufs = gh.random_device_bufs(B, L, P, R, Dp, es, seed=7 + layout)
    with hc.Pool(L, B, P, R, Hp, layout, elem_bytes=es) as pool:
        gh.check_backup(pool, bufs, dp, hp, layout, B, L, P, R, Hp, es)
        gh.check_load(pool, bufs, dp, hp, layout, B, L, P, R, Hp, es)
        for layer in sorted({0, L - 1, L // 2}):
            gh.check_load(pool, bufs, dp, hp, layout, B, L, P, R, Hp, es, layer=layer, seed=layer + 3)


@pytest.mark.parametrize("layout", LAYOUTS, ids=list(hc.LAYOUTS))
def test_tiny_gqa_backup_then_load(layout):
    """The tiny GQA pool: back up 12 random device pages into 12 random host
    pages, sentinel-fill the device, load into 12 fresh random device pages."""
    s = wl.TINY_GQA
    B, L, P, R, Dp, Hp = s.num_buffers, s.num_layers, s.page_size, s.row_elems, s.device_pages, s.host_pages
    rng = wl.index_rng(s.seed)
    src = wl.distinct_pages(rng, Dp, 12)
    hp = wl.distinct_pages(rng, Hp, 12)
    dst = wl.distinct_pages(rng, Dp, 12)
    vals = [t.view(torch.int16) for t in wl.kv_values(s, device="cuda")]
    with hc.Pool(L, B, P, R, Hp, layout) as pool:
        gh.check_backup(pool, vals, src, hp, layout, B, L, P, R, Hp, 2)
        host_before = pool.host_array().copy()
        orig = gh.to_np(vals, 2)
        gh.sentinel_fill(vals, 0xFF)
        kv = hc.DeviceKV(vals, Dp)
        pool.load(kv, dst, hp, layout)
        torch.cuda.synchronize()
        want = [np.full((Dp * P, R), 0xFFFF, np.uint16) for _ in range(B * L)]
        gh.orc().load(want, host_before, B, L, P, R, Hp, dst, hp, layout)
        got = gh.to_np(vals, 2)
        for k in range(B * L):
            assert np.array_equal(got[k], want[k])
            for s_, d_ in zip(src, dst):   # round trip: the pages came back
                assert np.array_equal(got[k][d_ * P:(d_ + 1) * P], orig[k][s_ * P:(s_ + 1) * P])


@pytest.mark.parametrize("layout", LAYOUTS, ids=list(hc.LAYOUTS))
def test_plan_execute_matches_direct_calls(layout):
    B, L, P, R, Dp, Hp, n = 2, 4, 16, 128, 48, 64, 20
    dp, hp = indices("runs", Dp, Hp, n, seed=5)
    bufs = gh.random_device_bufs(B, L, P, R, Dp, seed=11)
    with hc.Pool(L, B, P, R, Hp, layout) as pool:
        plan = pool.plan(dp, hp, Dp, hc.BACKUP)
        pn, pr = plan.info()
        assert pn == n and pr == len(hc.prepass(Hp, Dp, dp, hp, hc.BACKUP))
        host = pool.host_array(np.uint8)
        host[:] = 0x11
        kv = hc.DeviceKV(bufs, Dp)
        plan.execute(kv)
        torch.cuda.synchronize()
        want = np.full(host.size, 0x11, np.uint8).view(np.uint16)
        gh.orc().backup(gh.to_np(bufs, 2), want, B, L, P, R, Hp, dp, hp, layout)
        assert np.array_equal(host.view(np.uint16), want)
        # a load plan executed layer by layer equals one all-layer load
        lplan = pool.plan(dp, hp, Dp, hc.LOAD)
        host[:] = np.random.default_rng(2).integers(0, 256, host.size, dtype=np.uint8)
        gh.sentinel_fill(bufs)
        s = torch.cuda.Stream()
        for layer in range(L):
            lplan.execute(kv, layer=layer, stream=s)
        s.synchronize()
        want = [np.full((Dp * P, R), 0x5A5A, np.uint16) for _ in range(B * L)]
        gh.orc().load(want, host.view(np.uint16), B, L, P, R, Hp, dp, hp, layout)
        got = gh.to_np(bufs, 2)
        for k in range(B * L):
            assert np.array_equal(got[k], want[k])
        with pytest.raises(hc.HiCacheError):      # per-layer execution of a backup plan
            plan.execute(kv, layer=0)
        plan.close()
        lplan.close()


@pytest.mark.parametrize("layout", LAYOUTS, ids=list(hc.LAYOUTS))
def test_plan_load_layer_touches_one_layer(layout):
    """hicache_plan_load_layer equals the oracle's load of that layer alone and
    leaves the other layers as they were; its layer event gates a stream."""
    B, L, P, R, Dp, Hp, n = 2, 5, 8, 64, 40, 50, 17
    dp, hp = indices("runs", Dp, Hp, n, seed=41)
    bufs = gh.random_device_bufs(B, L, P, R, Dp, seed=42)
    with hc.Pool(L, B, P, R, Hp, layout) as pool:
        host = pool.host_array(np.uint8)
        host[:] = np.random.default_rng(43).integers(0, 256, host.size, dtype=np.uint8)
        kv = hc.DeviceKV(bufs, Dp)
        lplan = pool.plan(dp, hp, Dp, hc.LOAD)
        s, comp = torch.cuda.Stream(), torch.cuda.Stream()
        for layer in (3, 0):
            gh.sentinel_fill(bufs)
            torch.cuda.synchronize()
            lplan.load_layer(kv, layer, stream=s)
            pool.wait_layer(layer, comp)
            hc.wait(comp, 10_000_000)
            want = [np.full((Dp * P, R), 0x5A5A, np.uint16) for _ in range(B * L)]
            gh.orc().load(want, host.view(np.uint16), B, L, P, R, Hp, dp, hp, layout, layer)
            got = gh.to_np(bufs, 2)
            for k in range(B * L):
                assert np.array_equal(got[k], want[k]), (layer, k)
        c0 = hc.launch_count()
        for bad in (-1, L):
            with pytest.raises(hc.HiCacheError):
                lplan.load_layer(kv, bad, stream=s)
        bplan = pool.plan(dp, hp, Dp, hc.BACKUP)
        with pytest.raises(hc.HiCacheError):
            bplan.load_layer(kv, 0, stream=s)
        assert hc.launch_count() == c0
        bplan.close()
        lplan.close()


def test_one_launch_per_call_and_errors_enqueue_nothing():
    B, L, P, R, Dp, Hp = 2, 32, 16, 1024, 64, 64
    bufs = [torch.zeros((Dp * P, R), dtype=torch.int16, device="cuda") for _ in range(B * L)]
    kv = hc.DeviceKV(bufs, Dp)
    with hc.Pool(L, B, P, R, Hp, "layer_first") as pool:
        for n in (1, 2, 3, 4, 37, 64):
            rng = np.random.default_rng(n)
            c0 = hc.launch_count()
            pool.load(kv, rng.choice(Dp, n, replace=False), rng.choice(Hp, n, replace=False))
            assert hc.launch_count() - c0 == 1
        c0 = hc.launch_count()
        pool.backup(kv, [], [])                     # n == 0: nothing launched
        assert hc.launch_count() == c0
        bad = [
            (([0, Dp], [0, 1]), "INDEX_RANGE"),
            (([0, 1], [Hp, 1]), "INDEX_RANGE"),
            (([-1], [0]), "INDEX_RANGE"),
            (([3, 3], [0, 1]), "DUPLICATE_INDEX"),  # load writes device page 3 twice
        ]
        for (dp, hp), status in bad:
            with pytest.raises(hc.HiCacheError) as e:
                pool.load(kv, dp, hp)
            assert e.value.status == status
        with pytest.raises(hc.HiCacheError) as e:   # backup writes host page 5 twice
            pool.backup(kv, [0, 1], [5, 5])
        assert e.value.status == "DUPLICATE_INDEX"
        with pytest.raises(hc.HiCacheError) as e:
            pool.load_layer(kv, [0], [0], L)
        assert e.value.status == "INVALID_ARG"
        with pytest.raises(hc.HiCacheError) as e:
            pool.load(kv, [0], [0], layout=9)
        assert e.value.status == "INVALID_ARG"
        misaligned = hc.DeviceKV([bufs[0].data_ptr() + 8] + [b.data_ptr() for b in bufs[1:]], Dp)
        with pytest.raises(hc.HiCacheError) as e:
            pool.load(misaligned, [0], [0])
        assert e.value.status == "ALIGNMENT"
        assert hc.launch_count() == c0
        # the failed calls changed nothing
        torch.cuda.synchronize()
        assert all(int(b.abs().sum()) == 0 for b in bufs[:2])


def test_zero_page_layer_load_still_records_event():
    B, L, P, R, Dp, Hp = 1, 3, 4, 64, 8, 8
    bufs = [torch.zeros((Dp * P, R), dtype=torch.int16, device="cuda") for _ in range(B * L)]
    with hc.Pool(L, B, P, R, Hp, "page_first") as pool:
        s = torch.cuda.Stream()
        pool.load_layer(hc.DeviceKV(bufs, Dp), [], [], 1, stream=s)
        assert pool.layer_event(1) != 0
        pool.wait_layer(1, torch.cuda.current_stream())
        torch.cuda.synchronize()


def test_pool_rejects_pageable_and_accepts_torch_pinned():
    B, L, P, R, Hp = 1, 2, 4, 64, 4
    nbytes = B * L * Hp * P * R * 2
    pageable = np.zeros(nbytes // 2 + 64, np.uint16)
    addr = (pageable.ctypes.data + 15) // 16 * 16
    with pytest.raises(hc.HiCacheError) as e:
        hc.Pool(L, B, P, R, Hp, "layer_first", host_ptr=addr, host_bytes=nbytes)
    assert e.value.status == "NOT_PINNED"
    pinned = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    bufs = gh.random_device_bufs(B, L, P, R, 6, seed=3)
    with hc.Pool(L, B, P, R, Hp, "page_first", host_ptr=pinned.data_ptr(), host_bytes=nbytes) as pool:
        gh.check_backup(pool, bufs, [5, 0, 2], [1, 3, 0], 1, B, L, P, R, Hp, 2)


def test_thp_host_pool():
    B, L, P, R, Dp, Hp = 2, 4, 16, 256, 32, 40
    bufs = gh.random_device_bufs(B, L, P, R, Dp, seed=9)
    dp, hp = indices("runs", Dp, Hp, 24, seed=9)
    with hc.Pool(L, B, P, R, Hp, "page_first_direct", thp=True) as pool:
        gh.check_backup(pool, bufs, dp, hp, 2, B, L, P, R, Hp, 2)
        gh.check_load(pool, bufs, dp, hp, 2, B, L, P, R, Hp, 2)


def test_wait_times_out_without_cancelling():
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        torch.cuda._sleep(int(1.5e9))               # a kernel that spins ~1 s, then ends
    with pytest.raises(hc.HiCacheError) as e:
        hc.wait(s, timeout_us=2000)
    assert e.value.status == "TIMEOUT"
    hc.wait(s, timeout_us=-1)                       # still completes
    hc.wait(s, timeout_us=0)


def test_layer_events_gate_compute():
    """Per-layer loads on a transfer stream, each followed by the stand-in
    attention on a compute stream that waited on that layer's event: every
    checksum must see its layer fully loaded."""
    B, L, P, R, Dp, Hp, n = 1, 8, 64, 576, 96, 96, 80
    rng = np.random.default_rng(4)
    dp = wl.fragmented_pages(rng, Dp, n)
    hp = np.arange(n)
    bufs = gh.random_device_bufs(B, L, P, R, Dp, seed=4)
    with hc.Pool(L, B, P, R, Hp, "page_first") as pool:
        host = pool.host_array(np.uint8)
        host[:] = rng.integers(0, 256, host.size, dtype=np.uint8)
        gh.sentinel_fill(bufs, 0)
        torch.cuda.synchronize()
        kv = hc.DeviceKV(bufs, Dp)
        sums = torch.zeros(L, dtype=torch.int64, device="cuda")
        xfer, comp = torch.cuda.Stream(), torch.cuda.Stream()
        plan = pool.plan(dp, hp, Dp, hc.LOAD)
        for layer in range(L):
            plan.execute(kv, layer=layer, stream=xfer)
            pool.wait_layer(layer, comp)
            hc.layer_checksum(kv, pool, dp, layer, sums.data_ptr() + 8 * layer, reps=1, stream=comp)
        comp.synchronize()
        want = [np.zeros((Dp * P, R), np.uint16) for _ in range(B * L)]
        gh.orc().load(want, host.view(np.uint16), B, L, P, R, Hp, dp, hp, 1)
        got = sums.cpu().numpy().view(np.uint64)
        for layer in range(L):
            words = np.concatenate([want[b * L + layer].reshape(Dp, -1)[dp].reshape(-1).view(np.uint32)
                                    for b in range(B)])
            assert int(got[layer]) == int(words.astype(np.uint64).sum(dtype=np.uint64)), layer


def test_bidirectional_streams():
    """Backup of request A on one stream while request B loads on another."""
    B, L, P, R, Dp, Hp, n = 2, 6, 16, 512, 64, 64, 24
    rng = np.random.default_rng(8)
    perm = rng.permutation(Dp)
    a_dev, b_dev = perm[:n], perm[n:2 * n]
    a_host, b_host = np.arange(n), np.arange(n, 2 * n)
    for layout in LAYOUTS:
        bufs = gh.random_device_bufs(B, L, P, R, Dp, seed=20 + layout)
        with hc.Pool(L, B, P, R, Hp, layout) as pool:
            host = pool.host_array(np.uint8)
            host[:] = rng.integers(0, 256, host.size, dtype=np.uint8)
            host0 = host.copy()
            dev0 = gh.to_np(bufs, 2)
            kv = hc.DeviceKV(bufs, Dp)
            s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
            pool.backup(kv, a_dev, a_host, stream=s1)
            pool.load(kv, b_dev, b_host, stream=s2)
            torch.cuda.synchronize()
            want_host = host0.view(np.uint16).copy()
            gh.orc().backup(dev0, want_host, B, L, P, R, Hp, a_dev, a_host, layout)
            want_dev = [x.copy() for x in dev0]
            gh.orc().load(want_dev, host0.view(np.uint16), B, L, P, R, Hp, b_dev, b_host, layout)
            assert np.array_equal(host.view(np.uint16), want_host)
            got = gh.to_np(bufs, 2)
            for k in range(B * L):
                assert np.array_equal(got[k], want_dev[k])


@pytest.mark.parametrize("layout", LAYOUTS, ids=list(hc.LAYOUTS))
@pytest.mark.parametrize("sizes", [(24, 24), (30, 7), (5, 40), (0, 12), (12, 0)], ids=str)
def test_backup_load_fused(layout, sizes):
    """One launch that backs up request A and loads request B equals the
    oracle's backup of A followed by its load of B (they touch disjoint pages)."""
    nb_, nl_ = sizes
    B, L, P, R, Dp, Hp = 2, 5, 16, 256, 96, 96
    rng = np.random.default_rng(31 + layout + nb_)
    perm = rng.permutation(Dp)
    a_dev, b_dev = perm[:nb_], perm[nb_:nb_ + nl_]
    hperm = rng.permutation(Hp)
    a_host, b_host = np.sort(hperm[:nb_]), hperm[nb_:nb_ + nl_]
    bufs = gh.random_device_bufs(B, L, P, R, Dp, seed=40 + layout)
    with hc.Pool(L, B, P, R, Hp, layout) as pool:
        host = pool.host_array(np.uint8)
        host[:] = rng.integers(0, 256, host.size, dtype=np.uint8)
        host0 = host.copy()
        dev0 = gh.to_np(bufs, 2)
        kv = hc.DeviceKV(bufs, Dp)
        c0 = hc.launch_count()
        pool.backup_load(kv, a_dev, a_host, b_dev, b_host)
        torch.cuda.synchronize()
        assert hc.launch_count() - c0 == (1 if nb_ + nl_ else 0)
        want_host = host0.view(np.uint16).copy()
        gh.orc().backup(dev0, want_host, B, L, P, R, Hp, a_dev, a_host, layout)
        want_dev = [x.copy() for x in dev0]
        gh.orc().load(want_dev, host0.view(np.uint16), B, L, P, R, Hp, b_dev, b_host, layout)
        assert np.array_equal(host.view(np.uint16), want_host)
        got = gh.to_np(bufs, 2)
        for k in range(B * L):
            assert np.array_equal(got[k], want_dev[k])


def test_backup_load_rejects_hazards():
    B, L, P, R, Dp, Hp = 1, 2, 4, 64, 16, 16
    bufs = [torch.zeros((Dp * P, R), dtype=torch.int16, device="cuda") for _ in range(B * L)]
    kv = hc.DeviceKV(bufs, Dp)
    with hc.Pool(L, B, P, R, Hp, "layer_first") as pool:
        c0 = hc.launch_count()
        with pytest.raises(hc.HiCacheError) as e:     # the load overwrites a page the backup reads
            pool.backup_load(kv, [1, 2], [0, 1], [5, 2], [8, 9])
        assert e.value.status == "INVALID_ARG" and "device page 2" in str(e.value)
        with pytest.raises(hc.HiCacheError) as e:     # the load reads a host page the backup writes
            pool.backup_load(kv, [1, 2], [0, 1], [5, 6], [1, 9])
        assert e.value.status == "INVALID_ARG" and "host page 1" in str(e.value)
        with pytest.raises(hc.HiCacheError) as e:     # the usual checks still apply to each side
            pool.backup_load(kv, [1, 2], [3, 3], [5, 6], [8, 9])
        assert e.value.status == "DUPLICATE_INDEX"
        assert hc.launch_count() == c0


@pytest.mark.parametrize("layout", [0, 1, 2], ids=["layer_first", "page_first", "page_first_direct"])
def test_heterogeneous_buffer_sets_as_pools_in_one_allocation(layout):
    """Buffers of different row sizes (an MLA latent of 576 bf16, an fp8
    indexer key of 128 bytes, an fp32 scale row of 4 values): one pool per
    buffer kind, carved out of a single pinned allocation.  With the buffer dim
    outermost in these layouts, the sub-pools side by side are exactly the
    mixed host pool; every sub-pool matches the oracle."""
    L, P, Dp, Hp, n = 6, 16, 40, 48, 14
    kinds = [(576, 2), (128, 1), (4, 4)]          # (row elements, element bytes)
    sizes = [L * Hp * P * R * es for R, es in kinds]
    total = sum(sizes)
    mem = hc.PinnedHost(total)
    rng = np.random.default_rng(50 + layout)
    dp = wl.fragmented_pages(rng, Dp, n, max_run=3)
    hp = rng.choice(Hp, n, replace=False)
    off = 0
    pools, bufsets = [], []
    for (R, es), nbytes in zip(kinds, sizes):
        pools.append(hc.Pool(L, 1, P, R, Hp, layout, elem_bytes=es, host_ptr=mem.ptr + off,
                             host_bytes=nbytes))
        bufsets.append(gh.random_device_bufs(1, L, P, R, Dp, es, seed=off % 97))
        off += nbytes
    s = torch.cuda.Stream()
    for pool, bufs, (R, es) in zip(pools, bufsets, kinds):
        pool.host_array(np.uint8)[:] = 0x3C
        pool.backup(hc.DeviceKV(bufs, Dp), dp, hp, stream=s)
    s.synchronize()
    for pool, bufs, (R, es) in zip(pools, bufsets, kinds):
        want = np.full(pool.nbytes, 0x3C, np.uint8).view(gh.NP_DT[es])
        gh.orc().backup(gh.to_np(bufs, es), want, 1, L, P, R, Hp, dp, hp, layout)
        assert np.array_equal(pool.host_array(gh.NP_DT[es]), want), (R, es)
    # and back, per layer, into fresh device pages
    dst = rng.permutation(Dp)[:n]
    for pool, bufs, (R, es) in zip(pools, bufsets, kinds):
        gh.sentinel_fill(bufs, 0x77)
        for layer in range(L):
            pool.load_layer(hc.DeviceKV(bufs, Dp), dst, hp, layer, stream=s)
    s.synchronize()
    for pool, bufs, (R, es) in zip(pools, bufsets, kinds):
        want = [np.zeros((Dp * P, R), gh.NP_DT[es]) for _ in range(L)]
        for w in want:
            w.view(np.uint8)[:] = 0x77
        gh.orc().load(want, pool.host_array(gh.NP_DT[es]), 1, L, P, R, Hp, dst, hp, layout)
        got = gh.to_np(bufs, es)
        for k in range(L):
            assert np.array_equal(got[k], want[k]), (R, es, k)
    for pool in pools:
        pool.close()


@pytest.mark.parametrize("layout", LAYOUTS, ids=list(hc.LAYOUTS))
def test_more_runs_than_one_launch_holds(layout):
    """4,000 scattered one-token pages are 4,000 runs: more than one launch's
    parameter block takes, so the call is split into several launches; the
    result must still equal the oracle, for one direction and for the fused
    backup + load."""
    B, L, P, R, Dp, Hp = 2, 3, 1, 8, 9000, 9000
    rng = np.random.default_rng(60 + layout)
    perm = rng.permutation(Dp)
    hperm = rng.permutation(Hp)
    n = 4000
    dp, hp = perm[:n], hperm[:n]
    bufs = gh.random_device_bufs(B, L, P, R, Dp, seed=61)
    with hc.Pool(L, B, P, R, Hp, layout) as pool:
        nruns = len(hc.prepass(Hp, Dp, dp, hp, hc.BACKUP))
        assert nruns > 1536
        c0 = hc.launch_count()
        gh.check_backup(pool, bufs, dp, hp, layout, B, L, P, R, Hp, 2)
        assert hc.launch_count() - c0 >= 2
        gh.check_load(pool, bufs, dp, hp, layout, B, L, P, R, Hp, 2)
        # fused, both directions over the launch capacity
        a_dev, b_dev = perm[:n], perm[n:2 * n]
        a_host, b_host = hperm[:n], hperm[n:2 * n]
        host = pool.host_array(np.uint8)
        host[:] = rng.integers(0, 256, host.size, dtype=np.uint8)
        host0 = host.copy()
        dev0 = gh.to_np(bufs, 2)
        c0 = hc.launch_count()
        pool.backup_load(hc.DeviceKV(bufs, Dp), a_dev, a_host, b_dev, b_host)
        torch.cuda.synchronize()
        assert hc.launch_count() - c0 >= 3
        want_host = host0.view(np.uint16).copy()
        gh.orc().backup(dev0, want_host, B, L, P, R, Hp, a_dev, a_host, layout)
        want_dev = [x.copy() for x in dev0]
        gh.orc().load(want_dev, host0.view(np.uint16), B, L, P, R, Hp, b_dev, b_host, layout)
        assert np.array_equal(host.view(np.uint16), want_host)
        got = gh.to_np(bufs, 2)
        for k in range(B * L):
            assert np.array_equal(got[k], want_dev[k])


def test_maximum_buffer_count():
    """B * L = 512 device buffers, the most one call takes (a 256-layer K/V pool)."""
    B, L, P, R, Dp, Hp, n = 2, 256, 2, 8, 12, 12, 7
    rng = np.random.default_rng(70)
    dp, hp = rng.choice(Dp, n, replace=False), rng.choice(Hp, n, replace=False)
    bufs = gh.random_device_bufs(B, L, P, R, Dp, seed=70)
    for layout in LAYOUTS:
        with hc.Pool(L, B, P, R, Hp, layout) as pool:
            gh.check_backup(pool, bufs, dp, hp, layout, B, L, P, R, Hp, 2)
            gh.check_load(pool, bufs, dp, hp, layout, B, L, P, R, Hp, 2)
            gh.check_load(pool, bufs, dp, hp, layout, B, L, P, R, Hp, 2, layer=L - 1)
    with pytest.raises(hc.HiCacheError):
        hc.Pool(257, 2, P, R, Hp, "layer_first")


def test_backup_thread_and_load_thread_share_a_pool():
    """A backup thread and a load thread (the pages' dedicated submitters), each
    with its own stream, calling one pool at the same time; results equal the
    oracle's for the same pairs."""
    import threading
    B, L, P, R, Dp, Hp = 2, 4, 16, 128, 128, 128
    rng = np.random.default_rng(80)
    perm, hperm = rng.permutation(Dp), rng.permutation(Hp)
    bufs = gh.random_device_bufs(B, L, P, R, Dp, seed=80)
    jobs_b = [(perm[i * 8:(i + 1) * 8], hperm[i * 8:(i + 1) * 8]) for i in range(6)]        # backups
    jobs_l = [(perm[64 + i * 8:64 + (i + 1) * 8], hperm[64 + i * 8:64 + (i + 1) * 8]) for i in range(6)]
    with hc.Pool(L, B, P, R, Hp, "page_first_direct") as pool:
        host = pool.host_array(np.uint8)
        host[:] = rng.integers(0, 256, host.size, dtype=np.uint8)
        host0, dev0 = host.copy(), gh.to_np(bufs, 2)
        kv = hc.DeviceKV(bufs, Dp)
        errors = []

        def worker(jobs, fn):
            try:
                st = torch.cuda.Stream()
                for dp, hp in jobs:
                    for layer in range(L) if fn == "load_layer" else [None]:
                        if fn == "backup":
                            pool.backup(kv, dp, hp, stream=st)
                        else:
                            pool.load_layer(kv, dp, hp, layer, stream=st)
                hc.wait(st)
            except Exception as e:  # reported below
                errors.append(e)
        ts = [threading.Thread(target=worker, args=(jobs_b, "backup")),
              threading.Thread(target=worker, args=(jobs_l, "load_layer"))]
        for t in ts:
            t.start()
        for t in ts:
            t.join()
        assert not errors, errors
        want_host = host0.view(np.uint16).copy()
        want_dev = [x.copy() for x in dev0]
        for dp, hp in jobs_b:
            gh.orc().backup(dev0, want_host, B, L, P, R, Hp, dp, hp, 2)
        for dp, hp in jobs_l:
            gh.orc().load(want_dev, host0.view(np.uint16), B, L, P, R, Hp, dp, hp, 2)
        assert np.array_equal(host.view(np.uint16), want_host)
        got = gh.to_np(bufs, 2)
        for k in range(B * L):
            assert np.array_equal(got[k], want_dev[k])


def test_layer_first_contiguous_equals_plain_range_copies():
    """In layer_first with pages contiguous on both sides, a backup is one range
    copy per (buffer, layer): the same bytes a plain cudaMemcpyAsync of each
    buffer's range into the host pool gives (the library-routine special case)."""
    B, L, P, R, Dp, Hp, n, d0, h0 = 2, 5, 16, 256, 64, 80, 24, 9, 31
    bufs = gh.random_device_bufs(B, L, P, R, Dp, seed=400)
    dp, hp = np.arange(d0, d0 + n), np.arange(h0, h0 + n)
    with hc.Pool(L, B, P, R, Hp, "layer_first") as pool:
        host = pool.host_array(np.uint8)
        host[:] = 0
        c0 = hc.launch_count()
        pool.backup(hc.DeviceKV(bufs, Dp), dp, hp)
        torch.cuda.synchronize()
        assert hc.launch_count() - c0 == 1
        got = host.copy()
        assert hc.segment_count(L, B, P, R, Hp, "layer_first", dp, hp) == B * L
        # the same ranges with the copy engine
        host[:] = 0
        row = R * 2
        dst = torch.from_numpy(host)
        for b in range(B):
            for l in range(L):
                off = ((b * L + l) * Hp * P + h0 * P) * row
                src = bufs[b * L + l].view(torch.uint8).reshape(-1)[d0 * P * row:(d0 + n) * P * row]
                dst[off:off + n * P * row].copy_(src, non_blocking=True)
        torch.cuda.synchronize()
        assert np.array_equal(got, host)


@pytest.mark.parametrize("layout", LAYOUTS, ids=list(hc.LAYOUTS))
def test_plan_load_layers_graph_replay(layout):
    """The per-layer loads of a plan replayed from a CUDA graph equal the
    oracle's load, fire every layer's event (a compute stream waits on each and
    reads the layer), count their launches on every replay, and re-capture for
    other device buffers."""
    B, L, P, R, Dp, Hp, n = 2, 5, 8, 64, 40, 48, 15
    dp, hp = indices("runs", Dp, Hp, n, seed=61)
    with hc.Pool(L, B, P, R, Hp, layout) as pool:
        host = pool.host_array(np.uint8)
        host[:] = np.random.default_rng(62).integers(0, 256, host.size, dtype=np.uint8)
        plan = pool.plan(dp, hp, Dp, hc.LOAD)
        s, comp = torch.cuda.Stream(), torch.cuda.Stream()
        sums = torch.zeros(L, dtype=torch.int64, device="cuda")
        want = [np.full((Dp * P, R), 0x5A5A, np.uint16) for _ in range(B * L)]
        gh.orc().load(want, host.view(np.uint16), B, L, P, R, Hp, dp, hp, layout)
        for bufset_seed in (63, 64):          # the second buffer set forces a re-capture
            bufs = gh.random_device_bufs(B, L, P, R, Dp, seed=bufset_seed)
            kv = hc.DeviceKV(bufs, Dp)
            for rep in range(2):
                gh.sentinel_fill(bufs)
                torch.cuda.synchronize()
                c0 = hc.launch_count()
                plan.load_layers(kv, stream=s)
                assert hc.launch_count() - c0 == L
                sums.zero_()
                for layer in range(L):
                    pool.wait_layer(layer, comp)
                    hc.layer_checksum(kv, pool, dp, layer, sums.data_ptr() + 8 * layer, stream=comp)
                hc.wait(comp, 10_000_000)
                hc.wait(s, 10_000_000)
                got = gh.to_np(bufs, 2)
                for k in range(B * L):
                    assert np.array_equal(got[k], want[k]), (bufset_seed, rep, k)
                for layer in range(L):
                    words = np.concatenate([want[b * L + layer].reshape(Dp, -1)[dp].reshape(-1).view(np.uint32)
                                            for b in range(B)])
                    assert int(sums[layer].item()) & (2**64 - 1) == int(words.astype(np.uint64).sum(dtype=np.uint64))
        # consecutive layers may run at once: overlapping buffers are refused
        big = torch.empty(B * L * Dp * P * R + R, dtype=torch.int16, device="cuda")
        step = Dp * P * R - R                    # each buffer starts one row before the last ends
        shared = [big[i * step:i * step + Dp * P * R].view(Dp * P, R) for i in range(B * L)]
        c0 = hc.launch_count()
        with pytest.raises(hc.HiCacheError, match="overlap"):
            plan.load_layers(hc.DeviceKV(shared, Dp), stream=s)
        assert hc.launch_count() == c0
        with pytest.raises(hc.HiCacheError):      # a backup plan has no per-layer loads
            bplan = pool.plan(dp, hp, Dp, hc.BACKUP)
            try:
                bplan.load_layers(kv, stream=s)
            finally:
                bplan.close()
        plan.close()


def test_plan_load_layers_of_an_empty_plan_records_every_event():
    """A plan of no pages replays a graph of event records alone: no launch,
    and every layer's event still fires behind the stream's earlier work."""
    B, L, P, R, Dp, Hp = 1, 3, 4, 32, 8, 8
    bufs = gh.random_device_bufs(B, L, P, R, Dp, seed=70)
    with hc.Pool(L, B, P, R, Hp, "layer_first") as pool:
        kv = hc.DeviceKV(bufs, Dp)
        plan = pool.plan(np.zeros(0, np.int64), np.zeros(0, np.int64), Dp, hc.LOAD)
        s, comp = torch.cuda.Stream(), torch.cuda.Stream()
        with torch.cuda.stream(s):
            torch.cuda._sleep(int(5e7))
        c0 = hc.launch_count()
        plan.load_layers(kv, stream=s)
        assert hc.launch_count() == c0
        for layer in range(L):
            pool.wait_layer(layer, comp)
        hc.wait(comp, 10_000_000)
        assert s.query()
        plan.close()


@pytest.mark.parametrize("layout", LAYOUTS, ids=list(hc.LAYOUTS))
def test_plan_load_layers_graph_with_split_layers(layout):
    """A plan of 4,000 scattered one-token pages needs several launches per
    layer.  In the graph every launch may start while the one before it drains
    (the next chunk of a layer, or the next layer) and ends after it.  The
    replay must equal the oracle's load, three times over."""
    B, L, P, R, Dp, Hp, n = 2, 3, 1, 8, 9000, 9000, 4000
    rng = np.random.default_rng(80 + layout)
    dp, hp = rng.permutation(Dp)[:n], rng.permutation(Hp)[:n]
    bufs = gh.random_device_bufs(B, L, P, R, Dp, seed=81)
    with hc.Pool(L, B, P, R, Hp, layout) as pool:
        host = pool.host_array(np.uint8)
        host[:] = rng.integers(0, 256, host.size, dtype=np.uint8)
        plan = pool.plan(dp, hp, Dp, hc.LOAD)
        kv = hc.DeviceKV(bufs, Dp)
        s = torch.cuda.Stream()
        want = [np.full((Dp * P, R), 0x5A5A, np.uint16) for _ in range(B * L)]
        gh.orc().load(want, host.view(np.uint16), B, L, P, R, Hp, dp, hp, layout)
        for rep in range(3):
            gh.sentinel_fill(bufs)
            torch.cuda.synchronize()
            c0 = hc.launch_count()
            plan.load_layers(kv, stream=s)
            assert hc.launch_count() - c0 >= 2 * L
            hc.wait(s, 10_000_000)
            got = gh.to_np(bufs, 2)
            for k in range(B * L):
                assert np.array_equal(got[k], want[k]), (rep, k)
        plan.close()


def test_plan_load_layers_last_event_means_every_layer():
    """The event of layer l fires only once layers 0..l have all landed, even
    though a layer's kernel may start before the previous one ends: a compute
    stream that waits on the last layer's event alone reads every layer
    complete (64K-token MLA load, where layer kernels overlap the most)."""
    s_ = wl.MLA_LATENT
    B, L, P, R, Hp = s_.num_buffers, s_.num_layers, s_.page_size, s_.row_elems, s_.host_pages
    Dp = s_.device_pages
    t = wl.mla_transfer(s_, 65536)
    bufs = gh.random_device_bufs(B, L, P, R, Dp, seed=90)
    with hc.Pool(L, B, P, R, Hp, "page_first") as pool:
        host = pool.host_array(np.uint8)
        host[:] = np.random.default_rng(91).integers(0, 256, host.size, dtype=np.uint8)
        plan = pool.plan(t.device_pages, t.host_pages, Dp, hc.LOAD)
        kv = hc.DeviceKV(bufs, Dp)
        s, comp = torch.cuda.Stream(), torch.cuda.Stream()
        sums = torch.zeros(L, dtype=torch.int64, device="cuda")
        # the expected per-layer sums, from a plain all-layer load checked
        # against the oracle in every device buffer
        mirror = fs.DeviceMirror(bufs)
        mirror.pull(bufs)
        pool.load(kv, t.device_pages, t.host_pages)
        torch.cuda.synchronize()
        fs.oracle_load(mirror.np, host.view(np.uint16), B, L, P, R, Hp, t.device_pages, t.host_pages,
                       hc.PAGE_FIRST)
        mirror.compare(bufs, "all-layer load of 64K tokens")
        mirror.close()
        for layer in range(L):
            hc.layer_checksum(kv, pool, t.device_pages, layer, sums.data_ptr() + 8 * layer)
        torch.cuda.synchronize()
        want = sums.clone()
        for rep in range(4):
            gh.sentinel_fill(bufs)
            sums.zero_()
            torch.cuda.synchronize()
            plan.load_layers(kv, stream=s)
            pool.wait_layer(L - 1, comp)
            for layer in range(L):
                hc.layer_checksum(kv, pool, t.device_pages, layer, sums.data_ptr() + 8 * layer, stream=comp)
            hc.wait(comp, 10_000_000)
            hc.wait(s, 10_000_000)
            assert torch.equal(sums, want), rep
        plan.close()
    del bufs
    torch.cuda.empty_cache()


@pytest.mark.parametrize("op", ["load", "fused"])
def test_split_call_is_complete_for_the_next_work_on_the_stream(op):
    """The launches of a split call overlap one another, yet work queued behind
    the call on the same stream sees every launch of it finished: a checksum of
    every loaded page, queued right after, equals the oracle's.  The last launch
    is the smallest, so it would finish first if it did not wait for the one
    before it."""
    B, L, P, R, Dp, Hp, n = 2, 3, 1, 8, 9000, 9000, 4000
    rng = np.random.default_rng(95)
    perm, hperm = rng.permutation(Dp), rng.permutation(Hp)
    dp, hp = perm[:n], hperm[:n]
    bufs = gh.random_device_bufs(B, L, P, R, Dp, seed=96)
    with hc.Pool(L, B, P, R, Hp, "layer_first") as pool:
        host = pool.host_array(np.uint8)
        host[:] = rng.integers(0, 256, host.size, dtype=np.uint8)
        want = [np.full((Dp * P, R), 0x5A5A, np.uint16) for _ in range(B * L)]
        gh.orc().load(want, host.view(np.uint16), B, L, P, R, Hp, dp, hp, hc.LAYER_FIRST)
        expect = [int(np.concatenate([want[b * L + l].reshape(Dp, -1)[dp].reshape(-1).view(np.uint32)
                                      for b in range(B)]).astype(np.uint64).sum(dtype=np.uint64))
                  for l in range(L)]
        kv = hc.DeviceKV(bufs, Dp)
        s = torch.cuda.Stream()
        sums = torch.zeros(L, dtype=torch.int64, device="cuda")
        for rep in range(5):
            gh.sentinel_fill(bufs)
            sums.zero_()
            torch.cuda.synchronize()
            c0 = hc.launch_count()
            if op == "load":
                pool.load(kv, dp, hp, stream=s)
            else:                              # a backup of other pages fused with the load
                pool.backup_load(kv, perm[n:2 * n], hperm[n:2 * n], dp, hp, stream=s)
            assert hc.launch_count() - c0 >= 3
            for layer in range(L):
                hc.layer_checksum(kv, pool, dp, layer, sums.data_ptr() + 8 * layer, stream=s)
            hc.wait(s, 10_000_000)
            got = [int(v) & (2**64 - 1) for v in sums.tolist()]
            assert got == expect, rep


@pytest.mark.parametrize("layout", LAYOUTS, ids=list(hc.LAYOUTS))
def test_layer_load_right_after_a_backup_of_the_same_pages(layout):
    """A one-layer load starts early behind the kernel before it and must wait
    for it before touching memory.  Here that kernel is a backup that reads the
    very device pages the load overwrites (and lets the next launch in during
    its last tiles): the backup must still see the old contents, and every
    layer load must land, for each layer in turn, on one stream."""
    B, L, P, R, Dp, Hp, n = 2, 4, 16, 128, 64, 96, 40
    rng = np.random.default_rng(130 + layout)
    dp = rng.permutation(Dp)[:n]
    h_old = rng.permutation(Hp)[:n]
    h_new = np.setdiff1d(np.arange(Hp), h_old)[:n]
    bufs = gh.random_device_bufs(B, L, P, R, Dp, seed=131 + layout)
    with hc.Pool(L, B, P, R, Hp, layout) as pool:
        host = pool.host_array(np.uint8)
        host[:] = rng.integers(0, 256, host.size, dtype=np.uint8)
        kv = hc.DeviceKV(bufs, Dp)
        s = torch.cuda.Stream()
        for layer in range(L):
            torch.cuda.synchronize()
            dev0 = gh.to_np(bufs, 2)
            host0 = host.view(np.uint16).copy()
            pool.backup(kv, dp, h_old, stream=s)            # reads pages dp of every layer
            pool.load_layer(kv, dp, h_new, layer, stream=s)  # overwrites pages dp of one layer
            hc.wait(s, 10_000_000)
            want_host = host0.copy()
            gh.orc().backup(dev0, want_host, B, L, P, R, Hp, dp, h_old, layout)
            assert np.array_equal(host.view(np.uint16), want_host), layer
            want_dev = [x.copy() for x in dev0]
            gh.orc().load(want_dev, want_host, B, L, P, R, Hp, dp, h_new, layout, layer)
            got = gh.to_np(bufs, 2)
            for k in range(B * L):
                assert np.array_equal(got[k], want_dev[k]), (layer, k)
