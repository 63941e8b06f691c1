"""Calls of tens of thousands of pages, the case where the host builds the run
table a chunk at a time while the first launches already run (pairs that come
in host order), where every run has one length (the kernels find a vector's run
by one division), where runs differ in length (a search per warp), and where
the pairs come unsorted (sorted first).  Each call spans many launches; the
whole host pool and every device buffer are compared with the oracle."""
import numpy as np
import pytest
import torch

import tiered_kv_cache_gb300 as hc
from tiered_kv_cache_gb300 import build as hc_build
from tiered_kv_cache_gb300 import workloads as wl

import fullsize as fs
import gpu_helpers as gh

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    hc_build.build()
    torch.cuda.init()
    yield
    torch.cuda.empty_cache()


def pairs(kind, rng, Dp, Hp, n):
    if kind == "sorted_uniform":            # one-token pages fully scattered, host in order
        return rng.permutation(Dp)[:n], np.sort(rng.choice(Hp, n, replace=False))
    if kind == "sorted_mixed":              # device runs of 1..8 pages, host contiguous
        return wl.fragmented_pages(rng, Dp, n), np.arange(n) + 3
    if kind == "unsorted":                  # host pages shuffled
        return rng.permutation(Dp)[:n], rng.permutation(Hp)[:n]
    raise ValueError(kind)


@pytest.mark.parametrize("layout", list(hc.LAYOUTS))
@pytest.mark.parametrize("kind", ["sorted_uniform", "sorted_mixed", "unsorted"])
def test_large_calls_equal_the_oracle(layout, kind):
    B, L, P, R, Dp, Hp, n = 2, 4, 1, 128, 40_000, 40_000, 30_000
    lay = hc.LAYOUTS[layout]
    rng = np.random.default_rng(1500 + 3 * lay + len(kind))
    dp, hp = pairs(kind, rng, Dp, Hp, n)
    bufs = gh.random_device_bufs(B, L, P, R, Dp, seed=1500)
    kv = hc.DeviceKV(bufs, Dp)
    mirror = fs.DeviceMirror(bufs)
    with hc.Pool(L, B, P, R, Hp, layout) as pool:
        host = pool.host_array(np.uint16)
        exp = np.empty_like(host)
        # backup over a sentinel pool
        fs.fill(host.view(np.uint8), 0xC3)
        fs.fill(exp.view(np.uint8), 0xC3)
        c0 = hc.launch_count()
        pool.backup(kv, dp, hp)
        torch.cuda.synchronize()
        assert hc.launch_count() - c0 > 1                   # many launches
        mirror.pull(bufs)
        fs.oracle_backup(mirror.np, exp, B, L, P, R, Hp, dp, hp, lay)
        fs.assert_equal(host, exp, f"backup ({kind})")
        # load from a position-coded pool into sentinel buffers
        fs.position_fill(host.view(np.uint32), 7)
        gh.sentinel_fill(bufs, 0x5A)
        torch.cuda.synchronize()
        pool.load(kv, dp, hp)
        torch.cuda.synchronize()
        mirror.fill(0x5A)
        fs.oracle_load(mirror.np, host, B, L, P, R, Hp, dp, hp, lay)
        mirror.compare(bufs, f"load ({kind})")
        # one layer of it
        gh.sentinel_fill(bufs, 0x5A)
        torch.cuda.synchronize()
        pool.load_layer(kv, dp, hp, 2)
        torch.cuda.synchronize()
        mirror.fill(0x5A)
        fs.oracle_load(mirror.np, host, B, L, P, R, Hp, dp, hp, lay, 2)
        mirror.compare(bufs, f"load of layer 2 ({kind})")
        del host, exp
    mirror.close()


def test_quarter_million_one_token_pages():
    """262,144 one-token pages of 256-byte rows (1 GiB per call, 147 launches),
    host pages in order: load and backup, every byte compared."""
    B, L, P, R = 2, 8, 1, 128
    n = Dp = Hp = 1 << 18
    rng = np.random.default_rng(1600)
    dp, hp = rng.permutation(Dp), np.arange(n)
    bufs = gh.random_device_bufs(B, L, P, R, Dp, seed=1600)
    kv = hc.DeviceKV(bufs, Dp)
    mirror = fs.DeviceMirror(bufs)
    with hc.Pool(L, B, P, R, Hp, "layer_first") as pool:
        host = pool.host_array(np.uint16)
        exp = np.empty_like(host)
        fs.fill(host.view(np.uint8), 0xC3)
        fs.fill(exp.view(np.uint8), 0xC3)
        c0 = hc.launch_count()
        pool.backup(kv, dp, hp)
        torch.cuda.synchronize()
        assert hc.launch_count() - c0 >= 100
        mirror.pull(bufs)
        fs.oracle_backup(mirror.np, exp, B, L, P, R, Hp, dp, hp, hc.LAYER_FIRST)
        fs.assert_equal(host, exp, "backup of 262,144 pages")
        fs.position_fill(host.view(np.uint32), 9)
        gh.sentinel_fill(bufs, 0x5A)
        torch.cuda.synchronize()
        pool.load(kv, dp, hp)
        torch.cuda.synchronize()
        mirror.fill(0x5A)
        fs.oracle_load(mirror.np, host, B, L, P, R, Hp, dp, hp, hc.LAYER_FIRST)
        mirror.compare(bufs, "load of 262,144 pages")
        del host, exp
    mirror.close()
    del bufs, kv
    torch.cuda.empty_cache()
