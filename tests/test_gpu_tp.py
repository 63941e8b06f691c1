"""The tensor-parallel load of a replicated latent (hicache_tp_load_pipelined)
with the ranks of a group stood in for by pools on one GPU: each rank's pool
over the same host memory, each with its own device buffers and counters.
Every rank's launch reads only its part of the pages and stores it into every
rank's buffers; afterwards each rank's buffers equal the oracle's load of ALL
the pages, and each rank's per-layer counters reach their targets (read and
checked before any stream wait relies on them).  No launch waits for another,
so the stand-in ranks run one after another or side by side on one GPU."""
import numpy as np
import pytest
import torch

import tiered_kv_cache_gb300 as hc
from tiered_kv_cache_gb300 import build as hc_build
from tiered_kv_cache_gb300 import workloads as wl

import fullsize as fs
import gpu_helpers as gh

pytestmark = pytest.mark.gpu
TEN_S = 10_000_000


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    hc_build.build()
    torch.cuda.init()


def group(tp, L, B, P, R, Hp, Dp, layout, mem, es=2):
    pools = [hc.Pool(L, B, P, R, Hp, layout, elem_bytes=es, host_ptr=mem.ptr, host_bytes=mem.nbytes)
             for _ in range(tp)]
    bufs = [[torch.empty((Dp * P, R * es), dtype=torch.uint8, device="cuda").view(gh.TORCH_DT[es])
             for _ in range(B * L)] for _ in range(tp)]
    kvs = [hc.DeviceKV(b, Dp) for b in bufs]
    return pools, bufs, kvs, [p.layer_counters() for p in pools]


def run_group(pools, kvs, counters, dp, hp, streams=None):
    c0 = hc.launch_count()
    for r, pool in enumerate(pools):
        hc.tp_load_pipelined(pool, kvs, counters, r, dp, hp, stream=None if streams is None else streams[r])
    return hc.launch_count() - c0


@pytest.mark.parametrize("layout", list(hc.LAYOUTS))
@pytest.mark.parametrize("tp,n", [(1, 23), (2, 23), (3, 23), (8, 23), (3, 2), (4, 0)])
def test_every_rank_ends_with_the_full_load(layout, tp, n):
    B, L, P, R, Dp, Hp = 2, 5, 16, 72, 48, 40
    lay = hc.LAYOUTS[layout]
    rng = np.random.default_rng(1000 + 7 * tp + n + lay)
    dp = wl.fragmented_pages(rng, Dp, n) if n else np.zeros(0, np.int64)
    hp = rng.choice(Hp, n, replace=False).astype(np.int64)
    mem = hc.PinnedHost(B * L * Hp * P * R * 2)
    pools, bufs, kvs, counters = group(tp, L, B, P, R, Hp, Dp, layout, mem)
    host = pools[0].host_array(np.uint16)
    host[:] = rng.integers(0, 1 << 16, host.size, dtype=np.uint16)
    for b in bufs:
        gh.sentinel_fill(b, 0xC3)
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in range(tp)]          # the ranks side by side
    launches = run_group(pools, kvs, counters, dp, hp, streams)
    assert launches == sum(1 for r in range(tp) if hc.tp_share(n, tp, r)[1] > 0)
    for s in streams:
        hc.wait(s, TEN_S)
    for p in pools:
        for layer in range(L):
            done, target = p.pipeline_status(layer)
            assert done == target, (layer, done, target)
    want = [np.full((Dp * P, R), 0xC3C3, np.uint16) for _ in range(B * L)]
    gh.orc().load(want, host, B, L, P, R, Hp, dp, hp, lay)
    for r in range(tp):
        got = gh.to_np(bufs[r], 2)
        for k in range(B * L):
            assert np.array_equal(got[k], want[k]), (r, k)
    # again, one stream for all ranks, each rank's layers waited for on its own
    # compute stream behind the counters, with the stand-in attention reading them
    for b in bufs:
        gh.sentinel_fill(b, 0xC3)
    torch.cuda.synchronize()
    xfer = torch.cuda.Stream()
    run_group(pools, kvs, counters, dp, hp, [xfer] * tp)
    comps = [torch.cuda.Stream() for _ in range(tp)]
    sums = torch.zeros((tp, L), dtype=torch.int64, device="cuda")
    for r, p in enumerate(pools):
        for layer in range(L):
            p.wait_layer(layer, comps[r])
            hc.layer_checksum(kvs[r], p, dp, layer, sums[r].data_ptr() + 8 * layer, stream=comps[r])
    for s in comps + [xfer]:
        hc.wait(s, TEN_S)
    for r in range(tp):
        got = gh.to_np(bufs[r], 2)
        for k in range(B * L):
            assert np.array_equal(got[k], want[k]), ("waited", r, k)
    after = torch.zeros_like(sums)
    for r, p in enumerate(pools):
        for layer in range(L):
            hc.layer_checksum(kvs[r], p, dp, layer, after[r].data_ptr() + 8 * layer)
    torch.cuda.synchronize()
    assert torch.equal(sums, after)
    for p in pools:
        p.close()
    del host
    mem.free()


@pytest.mark.parametrize("layout", list(hc.LAYOUTS))
@pytest.mark.parametrize("tp,n", [(2, 23), (3, 23), (8, 23), (8, 5)])
def test_partitioned_backup_of_a_replicated_latent(layout, tp, n):
    """A replicated latent's backup needs no exchange: rank r backs up the
    pairs of hicache_tp_share(n, tp, r) from its own replica into the host
    memory the ranks share, each on its own stream.  The host pool then equals
    the oracle's backup of all n pairs, and so does rank 0 backing up alone."""
    B, L, P, R, Dp, Hp = 1, 5, 16, 72, 48, 40
    lay = hc.LAYOUTS[layout]
    rng = np.random.default_rng(1500 + 7 * tp + n + lay)
    dp = wl.fragmented_pages(rng, Dp, n)
    hp = rng.choice(Hp, n, replace=False).astype(np.int64)
    mem = hc.PinnedHost(B * L * Hp * P * R * 2)
    pools, bufs, kvs, _ = group(tp, L, B, P, R, Hp, Dp, layout, mem)
    src = gh.random_device_bufs(B, L, P, R, Dp, 2, seed=tp * 31 + n)
    for r in range(tp):                                  # identical replicas
        for k in range(B * L):
            bufs[r][k].copy_(src[k])
    host = pools[0].host_array(np.uint16)
    want = np.full(host.size, 0x5A5A, np.uint16)
    gh.orc().backup(gh.to_np(src, 2), want, B, L, P, R, Hp, dp, hp, lay)
    for ranks in (range(tp), [0]):
        host[:] = 0x5A5A
        streams = [torch.cuda.Stream() for _ in range(tp)]
        for r in ranks:
            first, count = hc.tp_share(n, tp, r) if len(ranks) > 1 else (0, n)
            pools[r].backup(kvs[r], dp[first:first + count], hp[first:first + count], stream=streams[r])
        for st in streams:
            hc.wait(st, TEN_S)
        assert np.array_equal(host, want), (len(ranks), tp, n)
    for p in pools:
        p.close()
    del host
    mem.free()


def test_refusals_enqueue_nothing_and_keep_the_targets():
    B, L, P, R, Dp, Hp, tp = 1, 4, 16, 64, 32, 32, 2
    mem = hc.PinnedHost(B * L * Hp * P * R * 2)
    pools, bufs, kvs, counters = group(tp, L, B, P, R, Hp, Dp, "page_first", mem)
    dp, hp = np.arange(6), np.arange(6)
    before = [p.pipeline_status(0) for p in pools]
    c0 = hc.launch_count()
    bad = [
        (lambda: hc.tp_load_pipelined(pools[0], kvs, [counters[0], counters[1] + 2], 0, dp, hp), "ALIGNMENT"),
        (lambda: hc.tp_load_pipelined(pools[0], kvs, counters, 2, dp, hp), "INVALID_ARG"),       # rank
        (lambda: hc.tp_load_pipelined(pools[1], kvs, counters, 1, [0, 0, 1], [0, 1, 2]), "DUPLICATE_INDEX"),
        (lambda: hc.tp_load_pipelined(pools[1], kvs, counters, 1, [0, 1, 40], [0, 1, 2]), "INDEX_RANGE"),
        (lambda: hc.tp_load_pipelined(pools[0], [kvs[0], hc.DeviceKV(bufs[1], Dp - 1)], counters, 0, dp, hp),
         "INVALID_ARG"),                                                                      # unequal pools
    ]
    for call, status in bad:
        with pytest.raises(hc.HiCacheError) as e:
            call()
        assert e.value.status == status, e.value
    # more than 16 ranks; and tp x buffers x layers above the 1024-entry fan-out table
    with pytest.raises(hc.HiCacheError) as e:
        hc.tp_load_pipelined(pools[0], [kvs[0]] * 17, [counters[0]] * 17, 0, dp, hp)
    assert e.value.status == "INVALID_ARG"
    deep = hc.Pool(100, 1, P, R, Hp, "page_first", host_ptr=mem.ptr, host_bytes=mem.nbytes) \
        if mem.nbytes >= 100 * Hp * P * R * 2 else None
    if deep is None:
        mem2 = hc.PinnedHost(100 * Hp * P * R * 2)
        deep = hc.Pool(100, 1, P, R, Hp, "page_first", host_ptr=mem2.ptr, host_bytes=mem2.nbytes)
    deep_kv = hc.DeviceKV([bufs[0][0]] * 100, Dp)
    with pytest.raises(hc.HiCacheError) as e:
        hc.tp_load_pipelined(deep, [deep_kv] * 11, [deep.layer_counters()] * 11, 0, dp, hp)
    assert e.value.status == "INVALID_ARG" and "1024" in str(e.value)
    deep.close()
    assert hc.launch_count() == c0
    assert [p.pipeline_status(0) for p in pools] == before
    for p in pools:
        p.close()
    mem.free()


def test_mla61_64k_eight_ranks_full_size():
    """The MLA latent workload at 64K tokens (1024 pages, 61 layers, 576 bf16
    per row, page_first) split over eight stand-in ranks: every rank's 61
    buffers equal the oracle's load of all 1024 pages, compared whole."""
    s = wl.MLA_LATENT
    t = wl.mla_transfer(s, 65536)
    B, L, P, R, Dp, Hp, tp = s.num_buffers, s.num_layers, s.page_size, s.row_elems, s.device_pages, \
        s.host_pages, 8
    mem = hc.PinnedHost(B * L * Hp * P * R * 2)
    pools, bufs, kvs, counters = group(tp, L, B, P, R, Hp, Dp, "page_first", mem)
    host = pools[0].host_array(np.uint16)
    fs.position_fill(host.view(np.uint32), 61)
    for b in bufs:
        gh.sentinel_fill(b, 0xC3)
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in range(tp)]
    assert run_group(pools, kvs, counters, t.device_pages, t.host_pages, streams) == tp
    for st in streams:
        hc.wait(st, 60_000_000)
    for p in pools:
        assert all(p.pipeline_status(layer)[0] == p.pipeline_status(layer)[1] for layer in range(L))
    mirror = fs.DeviceMirror(bufs[0])
    mirror.fill(0xC3)
    fs.oracle_load(mirror.np, host, B, L, P, R, Hp, t.device_pages, t.host_pages, hc.PAGE_FIRST)
    for r in range(tp):
        mirror.compare(bufs[r], f"rank {r}")
    mirror.close()
    for p in pools:
        p.close()
    del host, bufs, kvs
    mem.free()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("tp", [2, 3])
def test_parts_split_over_several_launches(tp):
    """8,000 scattered one-token pages: each rank's part needs several
    launches (the run table of one launch holds under 1,800 runs), and each
    rank's targets must add up every rank's launches exactly as those ranks
    split them -- the counts reach the targets, and every rank ends with the
    oracle's load."""
    B, L, P, R, Dp, Hp, n = 1, 3, 1, 64, 9000, 9000, 8000
    rng = np.random.default_rng(1900 + tp)
    dp = rng.permutation(Dp)[:n]
    hp = np.sort(rng.choice(Hp, n, replace=False))
    mem = hc.PinnedHost(B * L * Hp * P * R * 2)
    pools, bufs, kvs, counters = group(tp, L, B, P, R, Hp, Dp, "layer_first", mem)
    host = pools[0].host_array(np.uint16)
    host[:] = rng.integers(0, 1 << 16, host.size, dtype=np.uint16)
    for b in bufs:
        gh.sentinel_fill(b, 0xC3)
    torch.cuda.synchronize()
    launches = run_group(pools, kvs, counters, dp, hp, [torch.cuda.Stream() for _ in range(tp)])
    assert launches >= 2 * tp
    torch.cuda.synchronize()
    for p in pools:
        for layer in range(L):
            done, target = p.pipeline_status(layer)
            assert done == target and target > 0, (layer, done, target)
    want = [np.full((Dp * P, R), 0xC3C3, np.uint16) for _ in range(B * L)]
    gh.orc().load(want, host, B, L, P, R, Hp, dp, hp, hc.LAYER_FIRST)
    for r in range(tp):
        got = gh.to_np(bufs[r], 2)
        for k in range(B * L):
            assert np.array_equal(got[k], want[k]), (r, k)
    for p in pools:
        p.close()
    del host
    mem.free()
