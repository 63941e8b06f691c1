"""The large workload shapes at their full sizes, on the GPU, in the launch
configuration the benchmark times (automatic grid).

Every transfer is compared with the oracle element by element over the WHOLE
host pool and EVERY device buffer: the oracle runs over disjoint groups of the
call's page pairs on all host cores (tests/fullsize.py), so untouched bytes are
checked as well as moved ones.  On top of that: a backup followed by a load is
the identity, per-layer checksums taken behind each layer's signal equal those
of the oracle's result, and every call of up to 1536 pages is one launch."""
import numpy as np
import pytest
import torch

import tiered_kv_cache_gb300 as hc
from tiered_kv_cache_gb300 import build as hc_build
from tiered_kv_cache_gb300 import workloads as wl

import fullsize as fs
import gpu_helpers as gh

pytestmark = pytest.mark.gpu

SENT8 = 0xC3             # 0xC3C3 is never a normal(0,1) bf16 (it is about -390)


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    hc_build.build()
    torch.cuda.init()
    yield
    torch.cuda.empty_cache()


def device_pool(shape: wl.KVShape):
    vals = wl.kv_values(shape, device="cuda")
    return [v.view(torch.int16) for v in vals]


def dims(s: wl.KVShape):
    return s.num_buffers, s.num_layers, s.page_size, s.row_elems, s.host_pages


def check_backup(pool, bufs, mirror, exp_host, s, dp, hp, layout):
    """Backup over a sentinel host pool; the whole pool against the oracle."""
    B, L, P, R, Hp = dims(s)
    host = pool.host_array(np.uint16)
    fs.fill(host.view(np.uint8), SENT8)
    fs.fill(exp_host.view(np.uint8), SENT8)
    c0 = hc.launch_count()
    pool.backup(hc.DeviceKV(bufs, s.device_pages), dp, hp, layout)
    torch.cuda.synchronize()
    assert hc.launch_count() - c0 == 1
    mirror.pull(bufs)
    fs.oracle_backup(mirror.np, exp_host, B, L, P, R, Hp, dp, hp, layout)
    fs.assert_equal(host, exp_host, f"backup, layout {layout}")


def check_load(pool, bufs, mirror, s, dp, hp, layout, salt):
    """Load from a position-coded host pool into sentinel device buffers;
    every device buffer against the oracle."""
    B, L, P, R, Hp = dims(s)
    host = pool.host_array(np.uint16)
    fs.position_fill(host.view(np.uint32), salt)
    gh.sentinel_fill(bufs, SENT8)
    torch.cuda.synchronize()
    c0 = hc.launch_count()
    pool.load(hc.DeviceKV(bufs, s.device_pages), dp, hp, layout)
    torch.cuda.synchronize()
    assert hc.launch_count() - c0 == 1
    mirror.fill(SENT8)
    fs.oracle_load(mirror.np, host, B, L, P, R, Hp, dp, hp, layout)
    mirror.compare(bufs, f"load, layout {layout}")


@pytest.mark.parametrize("shuffled_host", [False, True], ids=["host_contiguous", "host_shuffled"])
def test_llama3_8b_32k_all_layouts(shuffled_host):
    s = wl.LLAMA3_8B
    t = wl.llama_transfer(s, 512, shuffled_host=shuffled_host)
    bufs = device_pool(s)
    keep = [b.clone() for b in bufs]
    mirror = fs.DeviceMirror(bufs)
    B, L, P, R, Hp = dims(s)
    with hc.Pool(L, B, P, R, Hp, "layer_first") as pool:
        exp_host = np.empty_like(pool.host_array(np.uint16))
        for layout in hc.LAYOUTS.values():
            check_backup(pool, bufs, mirror, exp_host, s, t.device_pages, t.host_pages, layout)
            check_load(pool, bufs, mirror, s, t.device_pages, t.host_pages, layout, salt=layout)
            for b, k in zip(bufs, keep):
                b.copy_(k)
        del exp_host
        # round trip through the host into other device pages is the identity
        src = t.device_pages
        rest = np.setdiff1d(np.arange(s.device_pages), src)[: len(src)]
        kv = hc.DeviceKV(bufs, s.device_pages)
        for layout in hc.LAYOUTS.values():
            pool.backup(kv, src, t.host_pages, layout)
            pool.load(kv, rest, t.host_pages, layout)
            torch.cuda.synchronize()
            si = torch.as_tensor(src, device="cuda")
            di = torch.as_tensor(rest, device="cuda")
            for b in bufs:
                v = b.view(s.device_pages, -1)
                assert torch.equal(v[si], v[di])
    mirror.close()
    del bufs, keep
    torch.cuda.empty_cache()


def test_deep78_32k_bidirectional():
    """Backup of request A and load of request B at the same time, on two
    streams and as one fused launch, in every layout: the whole host pool and
    every device buffer against the oracle applying both (they commute: the
    requests are disjoint on both sides)."""
    s = wl.DEEP_STRESS
    a, b_req = wl.deep_bidir_transfers(s, 512)
    bufs = device_pool(s)
    B, L, P, R, Hp = dims(s)
    kv = hc.DeviceKV(bufs, s.device_pages)
    mirror = fs.DeviceMirror(bufs)
    with hc.Pool(L, B, P, R, Hp, "page_first_direct") as pool:
        host = pool.host_array(np.uint16)
        exp_host = np.empty_like(host)
        run = 0
        for layout in hc.LAYOUTS.values():
            for fused in (False, True):
                run += 1
                fs.normal_fill(bufs, 300 + run)          # fresh values, unlike what B loads
                fs.position_fill(host.view(np.uint32), run)
                mirror.pull(bufs)
                fs.copy(exp_host, host)
                c0 = hc.launch_count()
                if fused:
                    pool.backup_load(kv, a.device_pages, a.host_pages, b_req.device_pages, b_req.host_pages,
                                     layout)
                else:
                    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
                    pool.backup(kv, a.device_pages, a.host_pages, layout, stream=s1)
                    pool.load(kv, b_req.device_pages, b_req.host_pages, layout, stream=s2)
                torch.cuda.synchronize()
                assert hc.launch_count() - c0 == (1 if fused else 2)
                fs.oracle_backup(mirror.np, exp_host, B, L, P, R, Hp, a.device_pages, a.host_pages, layout)
                fs.oracle_load(mirror.np, exp_host, B, L, P, R, Hp, b_req.device_pages, b_req.host_pages,
                               layout)
                what = f"layout {layout}, {'fused' if fused else 'two streams'}"
                fs.assert_equal(host, exp_host, what)
                mirror.compare(bufs, what)
        del exp_host, host
    mirror.close()
    del bufs, kv
    torch.cuda.empty_cache()


def layer_sums(mirror, dp, L, Dp):
    """Per-layer sums of the 32-bit words of the given pages (one buffer per
    layer), from the oracle's device buffers: what the stand-in attention adds."""
    out = np.zeros(L, np.uint64)
    for layer in range(L):
        rows = mirror.np[layer].reshape(Dp, -1)[dp]
        out[layer] = rows.view(np.uint32).astype(np.uint64).sum(dtype=np.uint64)
    return out


@pytest.mark.parametrize("tokens", [4096, 16384, 65536])
def test_mla61_per_layer_and_pipelined_loads(tokens):
    """61 per-layer loads, each gating the stand-in attention of its layer
    through the layer's event, then the same load as one pipelined launch and
    as 61 chained per-layer calls, both gated per layer on the device counters:
    every device buffer against the oracle's per-layer loads applied in the
    same order."""
    s = wl.MLA_LATENT
    t = wl.mla_transfer(s, tokens)
    B, L, P, R, Hp = dims(s)
    Dp = s.device_pages
    bufs = device_pool(s)
    kv = hc.DeviceKV(bufs, Dp)
    mirror = fs.DeviceMirror(bufs)
    with hc.Pool(L, B, P, R, Hp, "page_first") as pool:
        host = pool.host_array(np.uint16)
        fs.position_fill(host.view(np.uint32), tokens)
        gh.sentinel_fill(bufs, SENT8)
        torch.cuda.synchronize()
        xfer, comp = torch.cuda.Stream(), torch.cuda.Stream()
        sums = torch.zeros(L, dtype=torch.int64, device="cuda")
        plan = pool.plan(t.device_pages, t.host_pages, Dp, hc.LOAD)
        c0 = hc.launch_count()
        for layer in range(L):
            plan.execute(kv, layer=layer, stream=xfer)
            pool.wait_layer(layer, comp)
            hc.layer_checksum(kv, pool, t.device_pages, layer, sums.data_ptr() + 8 * layer, stream=comp)
        torch.cuda.synchronize()
        assert hc.launch_count() - c0 == 2 * L
        mirror.fill(SENT8)
        for layer in range(L):
            fs.oracle_load(mirror.np, host, B, L, P, R, Hp, t.device_pages, t.host_pages, hc.PAGE_FIRST, layer)
        mirror.compare(bufs, f"per-layer loads of {tokens} tokens")
        # the checksums taken behind each layer's event are those of the oracle's result
        want = layer_sums(mirror, t.device_pages, L, Dp)
        assert np.array_equal(sums.cpu().numpy().view(np.uint64), want)
        # the same load in one pipelined launch, each layer waited for on the device
        gh.sentinel_fill(bufs, SENT8)
        sums.zero_()
        torch.cuda.synchronize()
        c0 = hc.launch_count()
        pool.load_pipelined(kv, t.device_pages, t.host_pages, stream=xfer)
        for layer in range(L):
            pool.wait_layer(layer, comp)
            hc.layer_checksum(kv, pool, t.device_pages, layer, sums.data_ptr() + 8 * layer, stream=comp)
        hc.wait(comp, 30_000_000)
        hc.wait(xfer, 30_000_000)
        assert hc.launch_count() - c0 == 1 + L
        mirror.compare(bufs, f"pipelined load of {tokens} tokens")
        assert np.array_equal(sums.cpu().numpy().view(np.uint64), want)
        # and as 61 chained per-layer calls, each layer waited for on the device
        gh.sentinel_fill(bufs, SENT8)
        sums.zero_()
        torch.cuda.synchronize()
        c0 = hc.launch_count()
        for layer in range(L):
            plan.load_layer_chained(kv, layer, stream=xfer)
            pool.wait_layer(layer, comp)
            hc.layer_checksum(kv, pool, t.device_pages, layer, sums.data_ptr() + 8 * layer, stream=comp)
        hc.wait(comp, 30_000_000)
        hc.wait(xfer, 30_000_000)
        assert hc.launch_count() - c0 == 2 * L
        mirror.compare(bufs, f"chained per-layer loads of {tokens} tokens")
        assert np.array_equal(sums.cpu().numpy().view(np.uint64), want)
        plan.close()
        del host
    mirror.close()
    del bufs, kv
    torch.cuda.empty_cache()


def test_small_mix_all_requests_against_an_oracle_shadow():
    """All 10,000 requests of the mix (1-256 pages, 30% backups) on one stream,
    one launch each.  An oracle shadow of the device pool and the host pool
    applies the same requests in the same order; at five checkpoints (the
    last after every request) the whole host pool and every device buffer are
    compared with the shadow."""
    s = wl.SMALL_MIX
    reqs = wl.small_mix_requests(s)
    assert len(reqs) == 10_000
    B, L, P, R, Hp = dims(s)
    bufs = device_pool(s)
    kv = hc.DeviceKV(bufs, s.device_pages)
    mirror = fs.DeviceMirror(bufs)
    mirror.pull(bufs)
    stream = torch.cuda.Stream()
    with hc.Pool(L, B, P, R, Hp, "layer_first") as pool:
        host = pool.host_array(np.uint16)
        fs.position_fill(host.view(np.uint32), 5)
        shadow_host = np.empty_like(host)
        fs.copy(shadow_host, host)
        checkpoints = {1999, 3999, 5999, 7999, len(reqs) - 1}
        for k, r in enumerate(reqs):
            c0 = hc.launch_count()
            if r.direction == "backup":
                pool.backup(kv, r.device_pages, r.host_pages, stream=stream)
                fs.oracle_backup(mirror.np, shadow_host, B, L, P, R, Hp, r.device_pages, r.host_pages,
                                 hc.LAYER_FIRST)
            else:
                pool.load(kv, r.device_pages, r.host_pages, stream=stream)
                fs.oracle_load(mirror.np, shadow_host, B, L, P, R, Hp, r.device_pages, r.host_pages,
                               hc.LAYER_FIRST)
            assert hc.launch_count() - c0 == 1, k
            if k in checkpoints:
                hc.wait(stream, 60_000_000)
                fs.assert_equal(host, shadow_host, f"host pool after request {k}")
                mirror.compare(bufs, f"device pool after request {k}")
        del host, shadow_host
    mirror.close()
    del bufs, kv
    torch.cuda.empty_cache()


def test_nsa_group_full_size_per_layer_and_all_layers():
    """An MLA latent (576 bf16), an fp8 indexer key (128) and fp32 scales (4)
    as three pools of one pinned allocation, at 64K tokens: 61 per-layer group
    loads, each gating per-pool checksums through the pools' layer events, then
    one all-layer group backup over sentinel host pools.  Every device buffer
    and every host pool against the oracle's transfer of that pool."""
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
        bufs = [torch.full((Dp * P, R * es), SENT8, dtype=torch.uint8, device="cuda").view(gh.TORCH_DT[es])
                for _ in range(L)]
        bufsets.append(bufs)
        kvs.append(hc.DeviceKV(bufs, Dp))
        fs.position_fill(pools[-1].host_array(np.uint32), len(pools))
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
    mirrors = []
    for i, (pool, bufs, (R, es)) in enumerate(zip(pools, bufsets, kinds)):
        m = fs.DeviceMirror(bufs)
        m.fill(SENT8)
        host = pool.host_array(gh.NP_DT[es])
        for layer in range(L):
            fs.oracle_load(m.np, host, 1, L, P, R, Hp, dp, hp, hc.PAGE_FIRST, layer)
        m.compare(bufs, f"per-layer group loads, pool {i}")
        assert np.array_equal(sums[i].cpu().numpy().view(np.uint64), layer_sums(m, dp, L, Dp)), i
        mirrors.append(m)
    # every layer back to the host in one launch, over sentinel host pools
    for pool in pools:
        fs.fill(pool.host_array(np.uint8), SENT8)
    c0 = hc.launch_count()
    hc.group_transfer(pools, kvs, dp, hp, hc.BACKUP)
    torch.cuda.synchronize()
    assert hc.launch_count() - c0 == 1
    for i, (pool, m, (R, es)) in enumerate(zip(pools, mirrors, kinds)):
        host = pool.host_array(gh.NP_DT[es])
        want = np.empty_like(host)
        fs.fill(want.view(np.uint8), SENT8)
        fs.oracle_backup(m.np, want, 1, L, P, R, Hp, dp, hp, hc.PAGE_FIRST)
        fs.assert_equal(host, want, f"group backup, pool {i}")
        m.close()
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
