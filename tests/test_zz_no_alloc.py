"""The allocation-free pipelined load (hicache_load_pipelined_noalloc).

Some callers cannot allocate device memory at the moment they load KV -- their
device memory is all handed out by their own allocator, or the code path must
not call cudaMalloc.  This entry point keeps its per-layer counters in a fixed
array inside the library instead of memory the pool allocated.  The test calls
it through the C ABI twice in a row and checks that every device buffer comes
out exactly as with hicache_load_pipelined, and that waiting per layer works.
This file is collected last so that, if it fails, a run that stops at the first
failure has already run every other test."""
import ctypes

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


def noalloc_load(pool, kv, dp, hp, stream):
    dp = np.ascontiguousarray(dp, dtype=np.int64)
    hp = np.ascontiguousarray(hp, dtype=np.int64)
    return hc.library().hicache_load_pipelined_noalloc(
        pool.handle, ctypes.byref(kv.struct), dp.ctypes.data, hp.ctypes.data, dp.size, hc.LAYOUT_POOL,
        stream.cuda_stream)


@pytest.mark.parametrize("layout", ["layer_first", "page_first_direct"])
def test_noalloc_load_matches_the_allocating_load(layout):
    B, L, P, R, Dp, Hp = 2, 6, 16, 128, 64, 64
    rng = np.random.default_rng(500)
    with hc.Pool(L, B, P, R, Hp, layout) as pool:
        host = pool.host_array(np.uint8)
        host[:] = rng.integers(0, 256, host.size, dtype=np.uint8)
        ref = [torch.zeros((Dp * P, R), dtype=torch.int16, device="cuda") for _ in range(B * L)]
        out = [torch.zeros((Dp * P, R), dtype=torch.int16, device="cuda") for _ in range(B * L)]
        kv_ref, kv_out = hc.DeviceKV(ref, Dp), hc.DeviceKV(out, Dp)
        xfer, comp = torch.cuda.Stream(), torch.cuda.Stream()
        sums = torch.zeros(L, dtype=torch.int64, device="cuda")
        for call in range(2):                       # two calls in a row
            n = 20 + 7 * call
            dp = wl.fragmented_pages(rng, Dp, n)
            hp = rng.choice(Hp, n, replace=False)
            pool.load_pipelined(kv_ref, dp, hp, stream=xfer)          # the allocating entry point
            hc.wait(xfer, TEN_S)
            assert noalloc_load(pool, kv_out, dp, hp, xfer) == 0, hc.library().hicache_last_error()
            sums.zero_()
            for layer in range(L):                  # each layer waited for on its own
                pool.wait_layer(layer, comp)
                hc.layer_checksum(kv_out, pool, dp, layer, sums.data_ptr() + 8 * layer, stream=comp)
            hc.wait(comp, TEN_S)
            hc.wait(xfer, TEN_S)
            for k in range(B * L):
                assert torch.equal(out[k], ref[k]), (call, k)
            got = sums.cpu().numpy().view(np.uint64)
            for layer in range(L):
                words = np.concatenate([ref[b * L + layer].cpu().numpy().reshape(Dp, -1)[dp].reshape(-1)
                                        .view(np.uint32) for b in range(B)])
                assert int(got[layer]) == int(words.astype(np.uint64).sum(dtype=np.uint64)), (call, layer)


def test_noalloc_load_split_over_several_launches_matches():
    """4,000 scattered one-token pages need several launches; two such calls in
    a row give the same device buffers as the allocating entry point."""
    B, L, P, R, Dp, Hp, n = 2, 3, 1, 8, 9000, 9000, 4000
    rng = np.random.default_rng(510)
    with hc.Pool(L, B, P, R, Hp, "page_first") as pool:
        host = pool.host_array(np.uint8)
        host[:] = rng.integers(0, 256, host.size, dtype=np.uint8)
        ref = [torch.zeros((Dp * P, R), dtype=torch.int16, device="cuda") for _ in range(B * L)]
        out = [torch.zeros((Dp * P, R), dtype=torch.int16, device="cuda") for _ in range(B * L)]
        xfer = torch.cuda.Stream()
        for call in range(2):
            dp, hp = rng.permutation(Dp)[:n], rng.permutation(Hp)[:n]
            pool.load_pipelined(hc.DeviceKV(ref, Dp), dp, hp, stream=xfer)
            c0 = hc.launch_count()
            assert noalloc_load(pool, hc.DeviceKV(out, Dp), dp, hp, xfer) == 0
            assert hc.launch_count() - c0 >= 3
            comp = torch.cuda.Stream()
            for layer in range(L):
                pool.wait_layer(layer, comp)
            hc.wait(comp, TEN_S)
            hc.wait(xfer, TEN_S)
            for k in range(B * L):
                assert torch.equal(out[k], ref[k]), (call, k)


def test_noalloc_load_refuses_more_layers_than_it_holds():
    L, P, R, Dp, Hp = 257, 2, 8, 4, 4
    bufs = [torch.zeros((Dp * P, R), dtype=torch.int16, device="cuda") for _ in range(L)]
    with hc.Pool(L, 1, P, R, Hp, "layer_first") as pool:
        c0 = hc.launch_count()
        rc = noalloc_load(pool, hc.DeviceKV(bufs, Dp), [0], [0], torch.cuda.current_stream())
        assert rc == -1
        assert "256" in hc.library().hicache_last_error().decode()
        assert hc.launch_count() == c0


def test_noalloc_load_refuses_a_capturing_stream():
    """Its per-layer targets are raised on the host when the call is enqueued,
    so a captured call would leave the per-layer waits wrong: a capturing
    stream gets INVALID_ARG and nothing is enqueued.  (The first call on the
    device, which looks up the array's address, comes before the capture.)"""
    B, L, P, R, Dp, Hp, n = 1, 3, 16, 64, 32, 32, 8
    rng = np.random.default_rng(530)
    dp = rng.choice(Dp, n, replace=False)
    hp = rng.choice(Hp, n, replace=False)
    bufs = [torch.zeros((Dp * P, R), dtype=torch.int16, device="cuda") for _ in range(B * L)]
    kv = hc.DeviceKV(bufs, Dp)
    with hc.Pool(L, B, P, R, Hp, "layer_first") as pool:
        s = torch.cuda.Stream()
        assert noalloc_load(pool, kv, dp, hp, s) == 0, hc.library().hicache_last_error()
        hc.wait(s, TEN_S)
        marker = torch.zeros(1, dtype=torch.int32, device="cuda")
        torch.cuda.synchronize()
        c0 = hc.launch_count()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            rc = noalloc_load(pool, kv, dp, hp, s)
            marker.add_(1)
        assert rc == -1
        assert b"captur" in hc.library().hicache_last_error()
        assert hc.launch_count() == c0
        g.replay()
        torch.cuda.synchronize()
        assert int(marker.item()) == 1
        # the waits still match the plain call that ran
        comp = torch.cuda.Stream()
        for layer in range(L):
            pool.wait_layer(layer, comp)
        hc.wait(comp, TEN_S)
