"""Buffer groups on the GPU: several pools with different row shapes, sharing
the page numbering, moved in one launch (hicache_group_transfer).  Every pool
of the group must match the oracle's own transfer of that pool."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import tiered_kv_cache_gb300 as hc
from tiered_kv_cache_gb300 import workloads as wl

import gpu_helpers as gh

pytestmark = pytest.mark.gpu

LAYOUTS = list(hc.LAYOUTS.values())
TEN_S = 10_000_000
# (buffers, row elements, element bytes): an MLA latent of 576 bf16, an fp8
# indexer key of 128, and its fp32 scales (4 per row, 16 bytes)
NSA_KINDS = [(1, 576, 2), (1, 128, 1), (1, 4, 4)]


class Group:
    """Pools carved from one pinned allocation, with their device buffers."""

    def __init__(self, kinds, L, P, Dp, Hp, layout, seed, hps=None):
        self.kinds, self.L, self.P, self.Dp = kinds, L, P, Dp
        self.hps = hps or [Hp] * len(kinds)
        sizes = [B * L * h * P * R * es for (B, R, es), h in zip(kinds, self.hps)]
        self.mem = hc.PinnedHost(sum(sizes))
        self.pools, self.bufs, off = [], [], 0
        for (B, R, es), h, nbytes in zip(kinds, self.hps, sizes):
            self.pools.append(hc.Pool(L, B, P, R, h, layout, elem_bytes=es, host_ptr=self.mem.ptr + off,
                                      host_bytes=nbytes))
            self.bufs.append(gh.random_device_bufs(B, L, P, R, Dp, es, seed=seed + off % 89))
            off += nbytes
        self.kvs = [hc.DeviceKV(b, Dp) for b in self.bufs]

    def close(self):
        for p in self.pools:
            p.close()


def _want_backup(grp, dp, hp, layout, fill):
    out = []
    for pool, bufs, (B, R, es), h in zip(grp.pools, grp.bufs, grp.kinds, grp.hps):
        want = np.full(pool.nbytes, fill, np.uint8).view(gh.NP_DT[es])
        gh.orc().backup(gh.to_np(bufs, es), want, B, grp.L, grp.P, R, h, dp, hp, layout)
        out.append(want)
    return out


def _want_load(grp, dp, hp, layout, fill, layer=-1):
    out = []
    for pool, (B, R, es), h in zip(grp.pools, grp.kinds, grp.hps):
        want = [np.zeros((grp.Dp * grp.P, R), gh.NP_DT[es]) for _ in range(B * grp.L)]
        for w in want:
            w.view(np.uint8)[:] = fill
        gh.orc().load(want, pool.host_array(gh.NP_DT[es]), B, grp.L, grp.P, R, h, dp, hp, layout, layer)
        out.append(want)
    return out


@pytest.mark.parametrize("layout", LAYOUTS, ids=list(hc.LAYOUTS))
def test_group_backup_and_load_match_the_oracle_in_one_launch(layout):
    L, P, Dp, Hp, n = 6, 16, 40, 48, 14
    grp = Group(NSA_KINDS, L, P, Dp, Hp, layout, seed=60 + layout)
    rng = np.random.default_rng(61 + layout)
    dp = wl.fragmented_pages(rng, Dp, n, max_run=3)
    hp = rng.choice(Hp, n, replace=False)
    s = torch.cuda.Stream()
    for pool in grp.pools:
        pool.host_array(np.uint8)[:] = 0x3C
    torch.cuda.synchronize()
    c0 = hc.launch_count()
    hc.group_transfer(grp.pools, grp.kvs, dp, hp, hc.BACKUP, stream=s)
    assert hc.launch_count() - c0 == 1
    hc.wait(s, TEN_S)
    for pool, want, (B, R, es) in zip(grp.pools, _want_backup(grp, dp, hp, layout, 0x3C), grp.kinds):
        assert np.array_equal(pool.host_array(gh.NP_DT[es]), want), (R, es)
    # all layers back into other device pages, one launch
    dst = rng.permutation(Dp)[:n]
    for bufs in grp.bufs:
        gh.sentinel_fill(bufs, 0x77)
    torch.cuda.synchronize()
    c0 = hc.launch_count()
    hc.group_transfer(grp.pools, grp.kvs, dst, hp, hc.LOAD, stream=s)
    assert hc.launch_count() - c0 == 1
    hc.wait(s, TEN_S)
    for bufs, want, (B, R, es) in zip(grp.bufs, _want_load(grp, dst, hp, layout, 0x77), grp.kinds):
        got = gh.to_np(bufs, es)
        for k in range(B * L):
            assert np.array_equal(got[k], want[k]), (R, es, k)
    grp.close()


@pytest.mark.parametrize("layout", LAYOUTS, ids=list(hc.LAYOUTS))
def test_group_layer_loads_touch_one_layer_and_record_every_pool_event(layout):
    L, P, Dp, Hp, n = 5, 8, 32, 40, 11
    kinds = [(2, 64, 2), (1, 32, 1), (1, 8, 2)]       # K,V beside two single-buffer kinds
    grp = Group(kinds, L, P, Dp, Hp, layout, seed=70 + layout)
    rng = np.random.default_rng(71 + layout)
    for pool in grp.pools:
        pool.host_array(np.uint8)[:] = rng.integers(0, 256, pool.nbytes, dtype=np.uint8)
    dp = rng.permutation(Dp)[:n]
    hp = wl.fragmented_pages(rng, Hp, n, max_run=4)
    s, comp = torch.cuda.Stream(), torch.cuda.Stream()
    sums = torch.zeros(len(kinds), dtype=torch.int64, device="cuda")
    for layer in (4, 1):
        for bufs in grp.bufs:
            gh.sentinel_fill(bufs, 0x5A)
        torch.cuda.synchronize()
        c0 = hc.launch_count()
        hc.group_transfer(grp.pools, grp.kvs, dp, hp, hc.LOAD, layer=layer, stream=s)
        assert hc.launch_count() - c0 == 1
        # every pool's layer event gates a compute stream that reads the layer
        sums.zero_()
        for i, (pool, kv) in enumerate(zip(grp.pools, grp.kvs)):
            pool.wait_layer(layer, comp)
            hc.layer_checksum(kv, pool, dp, layer, sums.data_ptr() + 8 * i, stream=comp)
        hc.wait(comp, TEN_S)
        for i, (bufs, want, (B, R, es)) in enumerate(
                zip(grp.bufs, _want_load(grp, dp, hp, layout, 0x5A, layer), grp.kinds)):
            got = gh.to_np(bufs, es)
            for k in range(B * L):
                assert np.array_equal(got[k], want[k]), (layer, R, k)
            words = np.concatenate([want[b * L + layer].reshape(Dp, -1)[dp].reshape(-1).view(np.uint32)
                                    for b in range(B)])
            assert int(sums[i].item()) & (2**64 - 1) == int(words.astype(np.uint64).sum(dtype=np.uint64))
    grp.close()


def test_group_of_one_equals_the_single_pool_call():
    L, P, Dp, Hp, n = 4, 16, 24, 24, 9
    grp = Group([(2, 128, 2)], L, P, Dp, Hp, "page_first", seed=80)
    rng = np.random.default_rng(81)
    dp, hp = rng.permutation(Dp)[:n], rng.permutation(Hp)[:n]
    pool = grp.pools[0]
    pool.host_array(np.uint8)[:] = 0
    hc.group_transfer(grp.pools, grp.kvs, dp, hp, hc.BACKUP)
    torch.cuda.synchronize()
    a = pool.host_array(np.uint8).copy()
    pool.host_array(np.uint8)[:] = 0
    pool.backup(grp.kvs[0], dp, hp)
    torch.cuda.synchronize()
    assert np.array_equal(a, pool.host_array(np.uint8))
    grp.close()


def test_group_with_more_runs_than_one_launch_holds():
    """Scattered one-page runs beyond one launch's table: the group call is
    split, every pool still matches the oracle."""
    L, P, Dp, Hp, n = 2, 1, 6000, 6000, 2500
    grp = Group(NSA_KINDS, L, P, Dp, Hp, "page_first_direct", seed=90)
    rng = np.random.default_rng(91)
    dp, hp = rng.permutation(Dp)[:n], rng.permutation(Hp)[:n]
    for pool in grp.pools:
        pool.host_array(np.uint8)[:] = 0xA5
    torch.cuda.synchronize()
    c0 = hc.launch_count()
    hc.group_transfer(grp.pools, grp.kvs, dp, hp, hc.BACKUP)
    assert hc.launch_count() - c0 >= 2
    torch.cuda.synchronize()
    for pool, want, (B, R, es) in zip(grp.pools, _want_backup(grp, dp, hp, 2, 0xA5), grp.kinds):
        assert np.array_equal(pool.host_array(gh.NP_DT[es]), want), (R, es)
    grp.close()


def test_group_rejects_mismatches_and_enqueues_nothing():
    L, P, Dp, Hp = 3, 8, 16, 16
    grp = Group(NSA_KINDS, L, P, Dp, Hp, "layer_first", seed=95, hps=[16, 16, 12])
    dp, hp = np.arange(4), np.arange(4)
    other_l = hc.Pool(L + 1, 1, P, 64, Hp, "layer_first")
    other_p = hc.Pool(L, 1, P * 2, 64, Hp, "layer_first")
    other_lay = hc.Pool(L, 1, P, 64, Hp, "page_first")
    kv_l = hc.DeviceKV(gh.random_device_bufs(1, L + 1, P, 64, Dp), Dp)
    kv_p = hc.DeviceKV(gh.random_device_bufs(1, L, P * 2, 64, Dp), Dp)
    kv_lay = hc.DeviceKV(gh.random_device_bufs(1, L, P, 64, Dp), Dp)
    c0 = hc.launch_count()
    bad = [
        ([], [], dp, hp, hc.BACKUP, -1),                                        # no pools
        (grp.pools + [other_lay, other_lay], grp.kvs + [kv_lay, kv_lay], dp, hp, hc.BACKUP, -1),  # 5 pools
        (grp.pools[:1] + [other_l], grp.kvs[:1] + [kv_l], dp, hp, hc.BACKUP, -1),  # layers differ
        (grp.pools[:1] + [other_p], grp.kvs[:1] + [kv_p], dp, hp, hc.BACKUP, -1),  # page sizes differ
        (grp.pools[:1] + [other_lay], grp.kvs[:1] + [kv_lay], dp, hp, hc.BACKUP, -1),  # layouts differ
        (grp.pools[:1] * 2, grp.kvs[:1] * 2, dp, hp, hc.BACKUP, -1),            # a pool twice
        ([grp.pools[0], grp.pools[1]], [grp.kvs[0], grp.kvs[0]], dp, hp, hc.LOAD, -1),  # buffers shared
        (grp.pools, grp.kvs, dp, hp, hc.BACKUP, 0),                             # per-layer backup
        (grp.pools, grp.kvs, dp, hp, hc.LOAD, L),                               # layer out of range
        (grp.pools, grp.kvs, dp, np.array([0, 1, 2, 13]), hc.LOAD, -1),         # past the smallest pool
        (grp.pools, grp.kvs, np.array([0, 1, 2, 16]), hp, hc.BACKUP, -1),        # past the device pool
        (grp.pools, grp.kvs, np.array([0, 1, 1, 2]), hp, hc.LOAD, -1),           # duplicate destination
        (grp.pools, grp.kvs, dp, hp, 7, -1),                                     # no such direction
    ]
    for pools, kvs, d, h, direction, layer in bad:
        with pytest.raises((hc.HiCacheError, ValueError)):
            hc.group_transfer(pools, kvs, d, h, direction, layer=layer)
    assert hc.launch_count() == c0
    hc.group_transfer(grp.pools, grp.kvs, dp, hp, hc.BACKUP, layer=-1)   # the same call, valid
    torch.cuda.synchronize()
    assert hc.launch_count() == c0 + 1
    for p in (other_l, other_p, other_lay):
        p.close()
    grp.close()


@pytest.mark.parametrize("layout", LAYOUTS, ids=list(hc.LAYOUTS))
def test_pipelined_group_matches_the_oracle_and_counts(layout):
    """Every layer of three pools in one launch; each pool equals the oracle's
    load, every pool's per-layer counts reach their targets, and a second load
    in a row (the scheduler words back at zero) is right too."""
    L, P, Dp, Hp, n = 5, 16, 40, 48, 13
    kinds = [(1, 576, 2), (2, 64, 1), (1, 4, 4)]
    grp = Group(kinds, L, P, Dp, Hp, layout, seed=110 + layout)
    rng = np.random.default_rng(111 + layout)
    s = torch.cuda.Stream()
    for call in range(2):
        for pool in grp.pools:
            pool.host_array(np.uint8)[:] = rng.integers(0, 256, pool.nbytes, dtype=np.uint8)
        dp = wl.fragmented_pages(rng, Dp, n, max_run=3)
        hp = rng.choice(Hp, n, replace=False)
        for bufs in grp.bufs:
            gh.sentinel_fill(bufs, 0x5A)
        torch.cuda.synchronize()
        c0 = hc.launch_count()
        hc.group_load_pipelined(grp.pools, grp.kvs, dp, hp, stream=s)
        assert hc.launch_count() - c0 == 1
        hc.wait(s, TEN_S)
        for bufs, want, (B, R, es) in zip(grp.bufs, _want_load(grp, dp, hp, layout, 0x5A), grp.kinds):
            got = gh.to_np(bufs, es)
            for k in range(B * L):
                assert np.array_equal(got[k], want[k]), (call, R, k)
        for pool in grp.pools:
            for layer in range(L):
                done, target = pool.pipeline_status(layer)
                assert done == target > 0
    grp.close()


def test_pipelined_group_layers_gate_compute():
    """Compute on a second stream waits for each pool's layer alone and reads
    it: the checksums taken behind the waits equal those taken afterwards."""
    L, P, Dp, Hp, n = 8, 16, 64, 64, 40
    grp = Group(NSA_KINDS, L, P, Dp, Hp, "page_first", seed=120)
    rng = np.random.default_rng(121)
    for pool in grp.pools:
        pool.host_array(np.uint8)[:] = rng.integers(0, 256, pool.nbytes, dtype=np.uint8)
    dp, hp = rng.permutation(Dp)[:n], rng.permutation(Hp)[:n]
    xfer, comp = torch.cuda.Stream(), torch.cuda.Stream()
    sums = torch.zeros((len(NSA_KINDS), L), dtype=torch.int64, device="cuda")
    for pool in grp.pools:                     # counts are checked before any wait relies on them
        assert all(pool.pipeline_status(layer)[0] == pool.pipeline_status(layer)[1] for layer in range(L))
    hc.group_load_pipelined(grp.pools, grp.kvs, dp, hp, stream=xfer)
    for layer in range(L):
        for i, (pool, kv) in enumerate(zip(grp.pools, grp.kvs)):
            pool.wait_layer(layer, comp)
            hc.layer_checksum(kv, pool, dp, layer, sums[i].data_ptr() + 8 * layer, stream=comp)
    hc.wait(comp, TEN_S)
    hc.wait(xfer, TEN_S)
    after = torch.zeros_like(sums)
    for i, (pool, kv) in enumerate(zip(grp.pools, grp.kvs)):
        for layer in range(L):
            hc.layer_checksum(kv, pool, dp, layer, after[i].data_ptr() + 8 * layer)
    torch.cuda.synchronize()
    assert torch.equal(sums, after)
    grp.close()


def test_pipelined_group_split_over_several_launches():
    L, P, Dp, Hp, n = 3, 1, 8000, 8000, 3000
    grp = Group(NSA_KINDS, L, P, Dp, Hp, "page_first_direct", seed=130)
    rng = np.random.default_rng(131)
    for pool in grp.pools:
        pool.host_array(np.uint8)[:] = rng.integers(0, 256, pool.nbytes, dtype=np.uint8)
    dp, hp = rng.permutation(Dp)[:n], rng.permutation(Hp)[:n]
    for bufs in grp.bufs:
        gh.sentinel_fill(bufs, 0x5A)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    c0 = hc.launch_count()
    hc.group_load_pipelined(grp.pools, grp.kvs, dp, hp, stream=s)
    assert hc.launch_count() - c0 >= 3
    hc.wait(s, TEN_S)
    for bufs, want, (B, R, es) in zip(grp.bufs, _want_load(grp, dp, hp, 2, 0x5A), grp.kinds):
        got = gh.to_np(bufs, es)
        for k in range(B * L):
            assert np.array_equal(got[k], want[k]), (R, k)
    for pool in grp.pools:
        for layer in range(L):
            done, target = pool.pipeline_status(layer)
            assert done == target
    grp.close()


def test_pipelined_group_stream_rule():
    """While a pool's pipelined load runs on one stream, a group that holds
    that pool may not start a pipelined load on another (nothing enqueued)."""
    L, P, Dp, Hp, n = 2, 8, 16, 16, 4
    grp = Group(NSA_KINDS, L, P, Dp, Hp, "page_first", seed=140)
    dp, hp = np.arange(n), np.arange(n)
    a, b = torch.cuda.Stream(), torch.cuda.Stream()
    with torch.cuda.stream(a):
        torch.cuda._sleep(int(2e8))           # keeps stream a busy for ~0.1 s
    grp.pools[1].load_pipelined(grp.kvs[1], dp, hp, stream=a)
    c0 = hc.launch_count()
    with pytest.raises(hc.HiCacheError):
        hc.group_load_pipelined(grp.pools, grp.kvs, dp, hp, stream=b)
    assert hc.launch_count() == c0
    hc.group_load_pipelined(grp.pools, grp.kvs, dp, hp, stream=a)   # same stream: fine
    hc.wait(a, TEN_S)
    for pool in grp.pools:
        for layer in range(L):
            done, target = pool.pipeline_status(layer)
            assert done == target
    grp.close()


def test_group_at_the_buffer_limit_and_beyond():
    """Four pools of 128 layers each: 512 device buffers, the most one launch
    takes; every pool matches the oracle.  A fifth buffer set is refused."""
    L, P, Dp, Hp, n = 128, 2, 12, 12, 5
    kinds = [(1, 8, 2), (1, 16, 1), (1, 4, 4), (1, 64, 2)]
    grp = Group(kinds, L, P, Dp, Hp, "page_first", seed=150)
    rng = np.random.default_rng(151)
    dp, hp = rng.permutation(Dp)[:n], rng.permutation(Hp)[:n]
    for pool in grp.pools:
        pool.host_array(np.uint8)[:] = 0x3C
    torch.cuda.synchronize()
    c0 = hc.launch_count()
    hc.group_transfer(grp.pools, grp.kvs, dp, hp, hc.BACKUP)
    torch.cuda.synchronize()
    assert hc.launch_count() - c0 == 1
    for pool, want, (B, R, es) in zip(grp.pools, _want_backup(grp, dp, hp, 1, 0x3C), grp.kinds):
        assert np.array_equal(pool.host_array(gh.NP_DT[es]), want), (R, es)
    extra = Group([(2, 8, 2)], L, P, Dp, Hp, "page_first", seed=152)   # 256 more buffers
    c0 = hc.launch_count()
    with pytest.raises(hc.HiCacheError):
        hc.group_transfer(grp.pools[:3] + extra.pools, grp.kvs[:3] + extra.kvs, dp, hp, hc.BACKUP)
    assert hc.launch_count() == c0
    extra.close()
    grp.close()


def test_empty_group_call_launches_nothing_and_layer_calls_still_record_events():
    L, P, Dp, Hp = 3, 4, 8, 8
    grp = Group(NSA_KINDS, L, P, Dp, Hp, "layer_first", seed=160)
    empty = np.zeros(0, np.int64)
    s, comp = torch.cuda.Stream(), torch.cuda.Stream()
    with torch.cuda.stream(s):
        torch.cuda._sleep(int(5e7))           # the events below must wait for this
    c0 = hc.launch_count()
    hc.group_transfer(grp.pools, grp.kvs, empty, empty, hc.BACKUP, stream=s)
    hc.group_transfer(grp.pools, grp.kvs, empty, empty, hc.LOAD, layer=2, stream=s)
    hc.group_load_pipelined(grp.pools, grp.kvs, empty, empty, stream=s)
    assert hc.launch_count() == c0
    for pool in grp.pools:                   # recorded on s, behind the sleep
        pool.wait_layer(2, comp)
    hc.wait(comp, TEN_S)
    assert s.query()
    grp.close()


def test_group_backup_thread_and_pipelined_load_thread():
    """A backup thread and a load thread calling one group at once, each on its
    own stream: group backups of one set of pages, pipelined group loads of
    another; both equal the oracle's per-pool results for the same pairs."""
    import threading
    L, P, Dp, Hp = 4, 8, 96, 96
    grp = Group(NSA_KINDS, L, P, Dp, Hp, "page_first_direct", seed=170)
    rng = np.random.default_rng(171)
    perm, hperm = rng.permutation(Dp), rng.permutation(Hp)
    jobs_b = [(perm[i * 6:(i + 1) * 6], hperm[i * 6:(i + 1) * 6]) for i in range(5)]
    jobs_l = [(perm[48 + i * 6:48 + (i + 1) * 6], hperm[48 + i * 6:48 + (i + 1) * 6]) for i in range(5)]
    for pool in grp.pools:
        pool.host_array(np.uint8)[:] = rng.integers(0, 256, pool.nbytes, dtype=np.uint8)
    torch.cuda.synchronize()
    host0 = [pool.host_array(np.uint8).copy() for pool in grp.pools]
    dev0 = [gh.to_np(bufs, es) for bufs, (B, R, es) in zip(grp.bufs, grp.kinds)]
    errors = []

    def worker(jobs, load):
        try:
            st = torch.cuda.Stream()
            for dp, hp in jobs:
                if load:
                    hc.group_load_pipelined(grp.pools, grp.kvs, dp, hp, stream=st)
                else:
                    hc.group_transfer(grp.pools, grp.kvs, dp, hp, hc.BACKUP, stream=st)
            hc.wait(st, TEN_S)
        except Exception as e:  # reported below
            errors.append(e)
    ts = [threading.Thread(target=worker, args=(jobs_b, False)),
          threading.Thread(target=worker, args=(jobs_l, True))]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert not errors, errors
    for i, (pool, bufs, (B, R, es)) in enumerate(zip(grp.pools, grp.bufs, grp.kinds)):
        want_host = host0[i].view(gh.NP_DT[es]).copy()
        want_dev = [x.copy() for x in dev0[i]]
        for dp, hp in jobs_b:
            gh.orc().backup(dev0[i], want_host, B, L, P, R, Hp, dp, hp, 2)
        for dp, hp in jobs_l:
            gh.orc().load(want_dev, host0[i].view(gh.NP_DT[es]), B, L, P, R, Hp, dp, hp, 2)
        assert np.array_equal(pool.host_array(gh.NP_DT[es]), want_host), R
        got = gh.to_np(bufs, es)
        for k in range(B * L):
            assert np.array_equal(got[k], want_dev[k]), (R, k)
        for layer in range(L):
            done, target = pool.pipeline_status(layer)
            assert done == target
    grp.close()


@pytest.mark.parametrize("layout", LAYOUTS, ids=list(hc.LAYOUTS))
def test_group_plan_execute_and_graph_replay_match_the_oracle(layout):
    """A group plan loads every layer at once, one layer, or every layer
    layer by layer from a CUDA graph; each pool equals the oracle's load of that
    pool, every pool's layer events fire, a second buffer set re-captures, and
    overlapping buffers are refused before anything is enqueued."""
    L, P, Dp, Hp, n = 5, 8, 36, 40, 13
    kinds = [(1, 576, 2), (2, 64, 1), (1, 4, 4)]
    grp = Group(kinds, L, P, Dp, Hp, layout, seed=110 + layout)
    rng = np.random.default_rng(111 + layout)
    for pool in grp.pools:
        pool.host_array(np.uint8)[:] = rng.integers(0, 256, pool.nbytes, dtype=np.uint8)
    dp = wl.fragmented_pages(rng, Dp, n, max_run=3)
    hp = rng.choice(Hp, n, replace=False)
    plan = hc.group_plan(grp.pools, dp, hp, Dp)
    s, comp = torch.cuda.Stream(), torch.cuda.Stream()
    want_all = _want_load(grp, dp, hp, layout, 0x6B)

    def check(want):
        for bufs, w, (B, R, es) in zip(grp.bufs, want, kinds):
            got = gh.to_np(bufs, es)
            for k in range(B * L):
                assert np.array_equal(got[k], w[k]), (R, es, k)

    # every layer at once: one launch
    for bufs in grp.bufs:
        gh.sentinel_fill(bufs, 0x6B)
    torch.cuda.synchronize()
    c0 = hc.launch_count()
    plan.execute(grp.kvs, stream=s)
    assert hc.launch_count() - c0 == 1
    hc.wait(s, TEN_S)
    check(want_all)
    # one layer
    for bufs in grp.bufs:
        gh.sentinel_fill(bufs, 0x6B)
    torch.cuda.synchronize()
    plan.execute(grp.kvs, layer=3, stream=s)
    for pool in grp.pools:
        pool.wait_layer(3, comp)
    hc.wait(comp, TEN_S)
    hc.wait(s, TEN_S)
    check(_want_load(grp, dp, hp, layout, 0x6B, layer=3))
    # layer by layer from a graph, for two buffer sets
    for seed in (112, 113):
        if seed == 113:
            grp.bufs = [gh.random_device_bufs(B, L, P, R, Dp, es, seed=seed + i)
                        for i, (B, R, es) in enumerate(kinds)]
            grp.kvs = [hc.DeviceKV(b, Dp) for b in grp.bufs]
        for rep in range(2):
            for bufs in grp.bufs:
                gh.sentinel_fill(bufs, 0x6B)
            torch.cuda.synchronize()
            c0 = hc.launch_count()
            plan.load_layers(grp.kvs, stream=s)
            assert hc.launch_count() - c0 == L
            for pool in grp.pools:
                pool.wait_layer(L - 1, comp)
            hc.wait(comp, TEN_S)
            hc.wait(s, TEN_S)
            check(want_all)
    # two pools' buffers overlapping: refused, nothing enqueued
    big = torch.empty(Dp * P * 576 * 2 * L + 64, dtype=torch.uint8, device="cuda")
    lat = [big[i * Dp * P * 1152:(i + 1) * Dp * P * 1152].view(torch.int16).view(Dp * P, 576) for i in range(L)]
    fp8 = [big[16 + i * Dp * P * 64:16 + (i + 1) * Dp * P * 64].view(Dp * P, 64) for i in range(2 * L)]
    bad = [hc.DeviceKV(lat, Dp), hc.DeviceKV(fp8, Dp), grp.kvs[2]]
    c0 = hc.launch_count()
    with pytest.raises(hc.HiCacheError, match="overlap"):
        plan.load_layers(bad, stream=s)
    assert hc.launch_count() == c0
    plan.close()
    grp.close()


def test_group_plan_graph_with_split_layers():
    """A group plan of 3,000 scattered one-token pages needs several launches
    per layer; the graph replay still equals the oracle for every pool."""
    L, P, Dp, Hp, n = 3, 1, 6000, 6000, 3000
    kinds = [(1, 576, 2), (1, 128, 1), (1, 4, 4)]
    grp = Group(kinds, L, P, Dp, Hp, "page_first", seed=120)
    rng = np.random.default_rng(121)
    for pool in grp.pools:
        pool.host_array(np.uint8)[:] = rng.integers(0, 256, pool.nbytes, dtype=np.uint8)
    dp, hp = rng.permutation(Dp)[:n], rng.permutation(Hp)[:n]
    plan = hc.group_plan(grp.pools, dp, hp, Dp)
    s = torch.cuda.Stream()
    want = _want_load(grp, dp, hp, hc.PAGE_FIRST, 0x2E)
    for rep in range(2):
        for bufs in grp.bufs:
            gh.sentinel_fill(bufs, 0x2E)
        torch.cuda.synchronize()
        c0 = hc.launch_count()
        plan.load_layers(grp.kvs, stream=s)
        assert hc.launch_count() - c0 >= 2 * L
        hc.wait(s, TEN_S)
        for bufs, w, (B, R, es) in zip(grp.bufs, want, kinds):
            got = gh.to_np(bufs, es)
            for k in range(B * L):
                assert np.array_equal(got[k], w[k]), (rep, R, k)
    plan.close()
    grp.close()
