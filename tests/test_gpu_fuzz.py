"""Seeded random sweep of shapes, layouts and operations, each compared byte
for byte with the oracle (GB300)."""
import numpy as np
import pytest
import torch

import tiered_kv_cache_gb300 as hc
from tiered_kv_cache_gb300 import build as hc_build
from tiered_kv_cache_gb300 import workloads as wl

import gpu_helpers as gh

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    hc_build.build()
    torch.cuda.init()


def draw(seed):
    rng = np.random.default_rng(1000 + seed)
    es = int(rng.choice([1, 2, 4, 8]))
    row_bytes = 16 * int(rng.choice([1, 2, 3, 5, 8, 9, 16, 36, 64, 72, 128]))
    R = row_bytes // es
    B = int(rng.integers(1, 4))
    L = int(rng.integers(1, 7))
    P = int(rng.choice([1, 2, 3, 7, 16, 64]))
    Dp = int(rng.integers(4, 40))
    Hp = int(rng.integers(4, 40))
    n = int(rng.integers(0, min(Dp, Hp) + 1))
    pattern = rng.choice(["random", "runs", "contiguous"])
    if pattern == "random" or n == 0:
        dp, hp = rng.choice(Dp, n, replace=False), rng.choice(Hp, n, replace=False)
    elif pattern == "runs":
        dp = wl.fragmented_pages(rng, Dp, n, max_run=int(rng.integers(1, 6)))
        hp = np.sort(rng.choice(Hp, n, replace=False))
    else:
        dp, hp = np.arange(n) + int(rng.integers(0, Dp - n + 1)), np.arange(n) + int(rng.integers(0, Hp - n + 1))
    layout = int(rng.integers(0, 4))
    op = str(rng.choice(["backup", "load", "load_layer", "fused"]))
    return dict(es=es, R=R, B=B, L=L, P=P, Dp=Dp, Hp=Hp, dp=dp, hp=hp, layout=layout, op=op,
                layer=int(rng.integers(0, L)), seed=seed)


@pytest.mark.parametrize("seed", range(300 * gh.SOAK))
def test_random_case(seed):
    c = draw(seed)
    B, L, P, R, Dp, Hp, es, layout = (c[k] for k in ("B", "L", "P", "R", "Dp", "Hp", "es", "layout"))
    dp, hp = c["dp"], c["hp"]
    bufs = gh.random_device_bufs(B, L, P, R, Dp, es, seed=seed)
    with hc.Pool(L, B, P, R, Hp, layout, elem_bytes=es) as pool:
        if c["op"] == "backup":
            gh.check_backup(pool, bufs, dp, hp, layout, B, L, P, R, Hp, es)
        elif c["op"] == "load":
            gh.check_load(pool, bufs, dp, hp, layout, B, L, P, R, Hp, es)
        elif c["op"] == "load_layer":
            gh.check_load(pool, bufs, dp, hp, layout, B, L, P, R, Hp, es, layer=c["layer"])
        else:
            # fused: back up the first half of the pairs, load the second half
            k = len(dp) // 2
            host = pool.host_array(np.uint8)
            host[:] = np.random.default_rng(seed).integers(0, 256, host.size, dtype=np.uint8)
            host0 = host.copy().view(gh.NP_DT[es])
            dev0 = gh.to_np(bufs, es)
            pool.backup_load(hc.DeviceKV(bufs, Dp), dp[:k], hp[:k], dp[k:], hp[k:])
            torch.cuda.synchronize()
            want_host = host0.copy()
            gh.orc().backup(dev0, want_host, B, L, P, R, Hp, dp[:k], hp[:k], layout)
            want_dev = [x.copy() for x in dev0]
            gh.orc().load(want_dev, host0, B, L, P, R, Hp, dp[k:], hp[k:], layout)
            assert np.array_equal(host.view(gh.NP_DT[es]), want_host), c
            got = gh.to_np(bufs, es)
            for i in range(B * L):
                assert np.array_equal(got[i], want_dev[i]), (c, i)
