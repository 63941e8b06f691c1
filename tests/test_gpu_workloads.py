"""The four large workload shapes at their full sizes, on the GPU, in the launch
configuration the benchmark times (automatic grid).

Full pools are too large for the oracle to redo in seconds, so each transfer is
checked on sampled elements whose host and device offsets come from the oracle
one by one, plus properties that hold at any size: untouched pages keep their
sentinel, a backup followed by a load is the identity, every call of up to
1536 pages is one launch."""
import numpy as np
import pytest
import torch

import tiered_kv_cache_gb300 as hc
from tiered_kv_cache_gb300 import build as hc_build
from tiered_kv_cache_gb300 import workloads as wl

import gpu_helpers as gh

pytestmark = pytest.mark.gpu

SENT16 = 0xC3C3          # never a normal(0,1) bf16 (it is about -390)


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    hc_build.build()
    torch.cuda.init()
    yield
    torch.cuda.empty_cache()


def position_fill(words: np.ndarray, chunk=1 << 26):
    """Host pool words = their own index mod 2^32: a misplaced copy is visible."""
    for off in range(0, words.size, chunk):
        m = min(chunk, words.size - off)
        words[off:off + m] = np.arange(off, off + m, dtype=np.uint64).astype(np.uint32)


def count_equal(a: np.ndarray, value, chunk=1 << 27) -> int:
    return sum(int(np.count_nonzero(a[o:o + chunk] == value)) for o in range(0, a.size, chunk))


def device_pool(shape: wl.KVShape):
    vals = wl.kv_values(shape, device="cuda")
    return [v.view(torch.int16) for v in vals]


def untouched_pages_ok(bufs, P, moved, sentinel16):
    Dp = bufs[0].shape[0] // P
    mask = torch.ones(Dp, dtype=torch.bool, device="cuda")
    mask[torch.as_tensor(np.asarray(moved), device="cuda")] = False
    s = torch.tensor(sentinel16, dtype=torch.int32).to(torch.int16).item()
    for b in bufs:
        rows = b.view(Dp, -1)[mask]
        if rows.numel() and not bool((rows == s).all()):
            return False
    return True


def run_backup_load(pool, bufs, shape, dp, hp, layout, samples=20000, seed=0):
    B, L, P, R, Hp = shape.num_buffers, shape.num_layers, shape.page_size, shape.row_elems, shape.host_pages
    Dp = bufs[0].shape[0] // P
    kv = hc.DeviceKV(bufs, Dp)
    host = pool.host_array(np.uint16)
    # backup
    host.view(np.uint8)[:] = 0xC3
    c0 = hc.launch_count()
    pool.backup(kv, dp, hp, layout)
    torch.cuda.synchronize()
    assert hc.launch_count() - c0 == 1
    assert gh.sampled_host_check(host, bufs, dp, hp, layout, B, L, P, R, Hp, samples, seed)
    moved_words = len(dp) * B * L * P * R
    assert count_equal(host, SENT16) == host.size - moved_words
    # load into sentinel-filled device pages from a position-coded host pool
    keep = [b.clone() for b in bufs]
    position_fill(host.view(np.uint32))
    gh.sentinel_fill(bufs, 0xC3)
    torch.cuda.synchronize()
    c0 = hc.launch_count()
    pool.load(kv, dp, hp, layout)
    torch.cuda.synchronize()
    assert hc.launch_count() - c0 == 1
    assert gh.sampled_host_check(host, bufs, dp, hp, layout, B, L, P, R, Hp, samples, seed + 1)
    assert untouched_pages_ok(bufs, P, dp, SENT16)
    for b, k in zip(bufs, keep):
        b.copy_(k)
    del keep


@pytest.mark.parametrize("shuffled_host", [False, True], ids=["host_contiguous", "host_shuffled"])
def test_llama3_8b_32k_all_layouts(shuffled_host):
    s = wl.LLAMA3_8B
    t = wl.llama_transfer(s, 512, shuffled_host=shuffled_host)
    bufs = device_pool(s)
    with hc.Pool(s.num_layers, s.num_buffers, s.page_size, s.row_elems, s.host_pages,
                 "layer_first") as pool:
        for layout in hc.LAYOUTS.values():
            run_backup_load(pool, bufs, s, t.device_pages, t.host_pages, layout, seed=layout)
        # round trip through the host into other device pages is the identity
        src = t.device_pages
        rest = np.setdiff1d(np.arange(s.device_pages), src)[: len(src)]
        kv = hc.DeviceKV(bufs, s.device_pages)
        for layout in hc.LAYOUTS.values():
            pool.backup(kv, src, t.host_pages, layout)
            pool.load(kv, rest, t.host_pages, layout)
            torch.cuda.synchronize()
            P = s.page_size
            si = torch.as_tensor(src, device="cuda")
            di = torch.as_tensor(rest, device="cuda")
            for b in bufs:
                v = b.view(s.device_pages, -1)
                assert torch.equal(v[si], v[di])
    del bufs
    torch.cuda.empty_cache()


def test_deep78_32k_bidirectional():
    s = wl.DEEP_STRESS
    a, b_req = wl.deep_bidir_transfers(s, 512)
    bufs = device_pool(s)
    B, L, P, R, Hp = s.num_buffers, s.num_layers, s.page_size, s.row_elems, s.host_pages
    kv = hc.DeviceKV(bufs, s.device_pages)
    with hc.Pool(L, B, P, R, Hp, "page_first_direct") as pool:
        host = pool.host_array(np.uint16)
        for layout in hc.LAYOUTS.values():
            position_fill(host.view(np.uint32))
            s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
            c0 = hc.launch_count()
            pool.backup(kv, a.device_pages, a.host_pages, layout, stream=s1)
            pool.load(kv, b_req.device_pages, b_req.host_pages, layout, stream=s2)
            torch.cuda.synchronize()
            assert hc.launch_count() - c0 == 2
            assert gh.sampled_host_check(host, bufs, a.device_pages, a.host_pages, layout, B, L, P, R, Hp,
                                         20000, 10 + layout)
            assert gh.sampled_host_check(host, bufs, b_req.device_pages, b_req.host_pages, layout, B, L, P,
                                         R, Hp, 20000, 20 + layout)
            # the same two requests as one fused launch
            position_fill(host.view(np.uint32))
            c0 = hc.launch_count()
            pool.backup_load(kv, a.device_pages, a.host_pages, b_req.device_pages, b_req.host_pages, layout)
            torch.cuda.synchronize()
            assert hc.launch_count() - c0 == 1
            assert gh.sampled_host_check(host, bufs, a.device_pages, a.host_pages, layout, B, L, P, R, Hp,
                                         20000, 30 + layout)
            assert gh.sampled_host_check(host, bufs, b_req.device_pages, b_req.host_pages, layout, B, L, P,
                                         R, Hp, 20000, 40 + layout)
    del bufs, kv
    torch.cuda.empty_cache()


@pytest.mark.parametrize("tokens", [4096, 16384, 65536])
def test_mla61_per_layer_load_with_events(tokens):
    s = wl.MLA_LATENT
    t = wl.mla_transfer(s, tokens)
    B, L, P, R, Hp = s.num_buffers, s.num_layers, s.page_size, s.row_elems, s.host_pages
    bufs = device_pool(s)
    kv = hc.DeviceKV(bufs, s.device_pages)
    with hc.Pool(L, B, P, R, Hp, "page_first") as pool:
        host = pool.host_array(np.uint16)
        position_fill(host.view(np.uint32))
        gh.sentinel_fill(bufs, 0xC3)
        torch.cuda.synchronize()
        xfer, comp = torch.cuda.Stream(), torch.cuda.Stream()
        sums = torch.zeros(L, dtype=torch.int64, device="cuda")
        plan = pool.plan(t.device_pages, t.host_pages, s.device_pages, hc.LOAD)
        c0 = hc.launch_count()
        for layer in range(L):
            plan.execute(kv, layer=layer, stream=xfer)
            pool.wait_layer(layer, comp)
            hc.layer_checksum(kv, pool, t.device_pages, layer, sums.data_ptr() + 8 * layer, stream=comp)
        torch.cuda.synchronize()
        assert hc.launch_count() - c0 == 2 * L
        assert gh.sampled_host_check(host, bufs, t.device_pages, t.host_pages, 1, B, L, P, R, Hp, 30000, 4)
        assert untouched_pages_ok(bufs, P, t.device_pages, SENT16)
        # the checksums taken behind each layer event equal those taken after
        # everything finished
        after = torch.zeros(L, dtype=torch.int64, device="cuda")
        for layer in range(L):
            hc.layer_checksum(kv, pool, t.device_pages, layer, after.data_ptr() + 8 * layer)
        torch.cuda.synchronize()
        assert torch.equal(sums, after)
        if tokens <= 16384:
            # and both equal the sums of what the oracle loads
            n = len(t.device_pages)
            want = [np.zeros((n * P, R), np.uint16) for _ in range(L)]
            gh.orc().load(want, host, B, L, P, R, Hp, np.arange(n), t.host_pages, 1)
            exp = np.array([w.view(np.uint32).astype(np.uint64).sum() for w in want], np.uint64)
            assert np.array_equal(after.cpu().numpy().view(np.uint64), exp)
        plan.close()
    del bufs, kv
    torch.cuda.empty_cache()


def test_small_mix_one_launch_per_call():
    s = wl.SMALL_MIX
    reqs = wl.small_mix_requests(s)[:300]
    B, L, P, R, Hp = s.num_buffers, s.num_layers, s.page_size, s.row_elems, s.host_pages
    bufs = device_pool(s)
    kv = hc.DeviceKV(bufs, s.device_pages)
    with hc.Pool(L, B, P, R, Hp, "layer_first") as pool:
        host = pool.host_array(np.uint16)
        position_fill(host.view(np.uint32))
        for k, r in enumerate(reqs):
            c0 = hc.launch_count()
            if r.direction == "backup":
                pool.backup(kv, r.device_pages, r.host_pages)
            else:
                pool.load(kv, r.device_pages, r.host_pages)
            torch.cuda.synchronize()
            assert hc.launch_count() - c0 == 1
            assert gh.sampled_host_check(host, bufs, r.device_pages, r.host_pages, 0, B, L, P, R, Hp,
                                         1000, k), k
    del bufs, kv
    torch.cuda.empty_cache()


def untouched_bytes_ok(bufs, P, moved, sentinel8):
    """Every device page not in `moved` still holds the sentinel byte (any dtype)."""
    Dp = bufs[0].shape[0] // P
    mask = torch.ones(Dp, dtype=torch.bool, device="cuda")
    mask[torch.as_tensor(np.asarray(moved), device="cuda")] = False
    for b in bufs:
        rows = b.view(torch.uint8).view(Dp, -1)[mask]
        if rows.numel() and not bool((rows == sentinel8).all()):
            return False
    return True


def test_nsa_group_full_size_per_layer_and_all_layers():
    """An MLA latent (576 bf16), an fp8 indexer key (128) and fp32 scales (4)
    as three pools of one pinned allocation, at 64K tokens: 61 per-layer group
    loads, each gating per-pool checksums through the pools' layer events, then
    one all-layer group backup; every pool checked on sampled oracle offsets."""
    s = wl.MLA_LATENT
    L, P, Dp, Hp = s.num_layers, s.page_size, s.device_pages, s.host_pages
    kinds = [(576, 2), (128, 1), (4, 4)]
    t = wl.mla_transfer(s, 65536)
    dp, hp = t.device_pages, t.host_pages
    sizes = [L * Hp * P * R * es for R, es in kinds]
    mem = hc.PinnedHost(sum(sizes))
    pools, bufsets, kvs, off = [], [], [], 0
    for (R, es), nbytes in zip(kinds, sizes):
        pools.append(hc.Pool(L, 1, P, R, Hp, "page_first", elem_bytes=es, host_ptr=mem.ptr + off,
                             host_bytes=nbytes))
        bufs = [torch.full((Dp * P, R * es), 0xC3, dtype=torch.uint8, device="cuda").view(gh.TORCH_DT[es])
                for _ in range(L)]
        bufsets.append(bufs)
        kvs.append(hc.DeviceKV(bufs, Dp))
        position_fill(pools[-1].host_array(np.uint32))
        off += nbytes
    xfer, comp = torch.cuda.Stream(), torch.cuda.Stream()
    sums = torch.zeros((len(kinds), L), dtype=torch.int64, device="cuda")
    torch.cuda.synchronize()
    c0 = hc.launch_count()
    for layer in range(L):
        hc.group_transfer(pools, kvs, dp, hp, hc.LOAD, layer=layer, stream=xfer)
        for i, (pool, kv) in enumerate(zip(pools, kvs)):
            pool.wait_layer(layer, comp)
            hc.layer_checksum(kv, pool, dp, layer, sums[i].data_ptr() + 8 * layer, stream=comp)
    torch.cuda.synchronize()
    assert hc.launch_count() - c0 == L + len(kinds) * L
    after = torch.zeros_like(sums)
    for i, (pool, kv) in enumerate(zip(pools, kvs)):
        for layer in range(L):
            hc.layer_checksum(kv, pool, dp, layer, after[i].data_ptr() + 8 * layer)
    torch.cuda.synchronize()
    assert torch.equal(sums, after)
    for i, (pool, bufs, (R, es)) in enumerate(zip(pools, bufsets, kinds)):
        host = pool.host_array(gh.NP_DT[es])
        assert gh.sampled_host_check(host, bufs, dp, hp, 1, 1, L, P, R, Hp, 20000, 10 + i), (R, es)
        assert untouched_bytes_ok(bufs, P, dp, 0xC3), (R, es)
    # every layer back to the host in one launch, over a sentinel-filled pool
    for pool in pools:
        pool.host_array(np.uint8)[:] = 0xC3
    c0 = hc.launch_count()
    hc.group_transfer(pools, kvs, dp, hp, hc.BACKUP)
    torch.cuda.synchronize()
    assert hc.launch_count() - c0 == 1
    for i, (pool, bufs, (R, es)) in enumerate(zip(pools, bufsets, kinds)):
        host = pool.host_array(np.uint8)
        assert gh.sampled_host_check(pool.host_array(gh.NP_DT[es]), bufs, dp, hp, 1, 1, L, P, R, Hp, 20000,
                                     20 + i), (R, es)
        moved = len(dp) * L * P * R * es
        assert count_equal(host, 0xC3) >= host.size - moved
    for pool in pools:
        pool.close()
    del bufsets, kvs
    torch.cuda.empty_cache()


def _mem_available_bytes() -> int:
    with open("/proc/meminfo") as f:
        for line in f:
            if line.startswith("MemAvailable:"):
                return int(line.split()[1]) * 1024
    return 0


@pytest.mark.parametrize("layout,B,L", [("layer_first", 1, 1), ("page_first_direct_kv", 2, 2)])
def test_run_past_the_unit_limit_is_split(layout, B, L):
    """The largest unit a launch can index: 2^31 - 1024 vectors of 16 bytes.
    With one-token pages of 1 GiB (every buffer and layer), a run of 34 pages
    contiguous on both sides would make one unit of 34 GiB.  The pre-pass caps
    runs at 31 such pages and the call becomes two launches; every page still
    lands where the oracle's offsets put it (checked page block by page block,
    each block's first and last element placed by the oracle, and on sampled
    elements)."""
    GiB = 1 << 30
    n, Dp, shift = 34, 36, 2
    P, es = 1, 2
    R = GiB // (B * L * es)                 # one page of every buffer and layer = 1 GiB
    dev_free = torch.cuda.mem_get_info()[0]
    if dev_free < (Dp + 4) * GiB or _mem_available_bytes() < 2 * n * GiB:
        pytest.skip("needs 40 GiB of free device memory and 68 GiB of available host memory")
    lay = hc.LAYOUTS[layout]
    o = gh.orc()
    g = torch.Generator(device="cuda")
    g.manual_seed(34)
    bufs = []
    for _ in range(B * L):
        x = torch.empty(Dp * P, R, dtype=torch.int16, device="cuda")
        x.random_(generator=g)
        bufs.append(x)
    kv = hc.DeviceKV(bufs, Dp)
    host_pages = np.arange(n)

    def blocks(dev_pages):
        # (buffer index, device page, host byte offset) of every page block,
        # each block R contiguous elements on both sides per the oracle
        for i, (d, h) in enumerate(zip(dev_pages, host_pages)):
            for b in range(B):
                for l in range(L):
                    h0 = o.host_offset(lay, B, L, P, R, n, b, l, int(h), 0, 0)
                    assert o.host_offset(lay, B, L, P, R, n, b, l, int(h), 0, R - 1) == h0 + R - 1
                    assert o.dev_offset(P, R, int(d), 0, R - 1) == o.dev_offset(P, R, int(d), 0, 0) + R - 1
                    yield b * L + l, int(d), h0 * es

    def same(host_u8, dev_pages):
        for k, d, hb in blocks(dev_pages):
            h = torch.from_numpy(host_u8[hb:hb + R * es]).to("cuda")
            if not torch.equal(h, bufs[k][d].view(torch.uint8)):
                return False
            del h
        return True

    with hc.Pool(L, B, P, R, n, layout) as pool:
        host = pool.host_array(np.uint8)
        src = np.arange(n)
        c0 = hc.launch_count()
        pool.backup(kv, src, host_pages)
        torch.cuda.synchronize()
        assert hc.launch_count() - c0 == 2
        assert same(host, src)
        assert gh.sampled_host_check(host.view(np.uint16), bufs, src, host_pages, lay, B, L, P, R, n, 4000, 1)
        # load into device pages shifted by two, over a sentinel
        keep = [b[:shift].clone() for b in bufs]
        for b in bufs:
            b[shift:].view(torch.uint8).fill_(0xC3)
        dst = src + shift
        c0 = hc.launch_count()
        pool.load(kv, dst, host_pages)
        torch.cuda.synchronize()
        assert hc.launch_count() - c0 == 2
        assert same(host, dst)
        assert gh.sampled_host_check(host.view(np.uint16), bufs, dst, host_pages, lay, B, L, P, R, n, 4000, 2)
        for b, k in zip(bufs, keep):
            assert torch.equal(b[:shift], k)
        del host
    del bufs, kv, keep
    torch.cuda.empty_cache()
