"""The submission engine on the GPU: results equal the oracle applying the
requests one by one in submission order; adjacent hazard-free backup/load pairs
leave as fused launches; dependencies on a caller's stream are honoured."""
import threading

import numpy as np
import pytest
import torch

import tiered_kv_cache_gb300 as hc
from tiered_kv_cache_gb300 import build as hc_build

import gpu_helpers as gh

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    hc_build.build()
    torch.cuda.init()


def oracle_apply(reqs, dev, host, B, L, P, R, Hp, layout):
    for direction, dp, hp in reqs:
        if direction == hc.BACKUP:
            gh.orc().backup(dev, host, B, L, P, R, Hp, dp, hp, layout)
        else:
            gh.orc().load(dev, host, B, L, P, R, Hp, dp, hp, layout)


@pytest.mark.parametrize("seed", range(3))
@pytest.mark.parametrize("layout", [0, 1, 2, 3], ids=list(hc.LAYOUTS))
def test_sequential_semantics_with_hazards(layout, seed):
    """Small pools and many overlapping requests: whether or not the engine
    fuses or holds a request, the outcome is the oracle's in submission order."""
    B, L, P, R, Dp, Hp = 2, 3, 4, 64, 20, 20
    rng = np.random.default_rng(90 + layout + 10 * seed)
    bufs = gh.random_device_bufs(B, L, P, R, Dp, seed=90)
    with hc.Pool(L, B, P, R, Hp, layout) as pool:
        host = pool.host_array(np.uint8)
        host[:] = rng.integers(0, 256, host.size, dtype=np.uint8)
        host0, dev0 = host.view(np.uint16).copy(), gh.to_np(bufs, 2)
        kv = hc.DeviceKV(bufs, Dp)
        reqs = []
        for _ in range(60):
            n = int(rng.integers(1, 7))
            reqs.append((int(rng.integers(0, 2)), rng.choice(Dp, n, replace=False), rng.choice(Hp, n, replace=False)))
        with hc.Engine(pool) as eng:
            tickets = [eng.submit(kv, dp, hp, d) for d, dp, hp in reqs]
            assert tickets == sorted(tickets)
            for t in tickets:
                eng.wait(t)
            launches, fused = eng.stats()
            assert launches + fused == len(reqs)
        oracle_apply(reqs, dev0, host0, B, L, P, R, Hp, layout)
        assert np.array_equal(host.view(np.uint16), host0)
        got = gh.to_np(bufs, 2)
        for k in range(B * L):
            assert np.array_equal(got[k], dev0[k])


def test_backup_and_load_threads_get_fused():
    """A backup thread and a load thread submit hazard-free requests while the
    link is busy: the engine pairs them into fused launches, and the result is
    the oracle's."""
    B, L, P, R, Dp, Hp = 2, 8, 16, 1024, 192, 192
    rng = np.random.default_rng(95)
    bufs = gh.random_device_bufs(B, L, P, R, Dp, seed=95)
    perm, hperm = rng.permutation(Dp), rng.permutation(Hp)
    back = [(hc.BACKUP, perm[i * 12:(i + 1) * 12], hperm[i * 12:(i + 1) * 12]) for i in range(8)]
    load = [(hc.LOAD, perm[96 + i * 12:96 + (i + 1) * 12], hperm[96 + i * 12:96 + (i + 1) * 12]) for i in range(8)]
    with hc.Pool(L, B, P, R, Hp, "layer_first") as pool:
        host = pool.host_array(np.uint8)
        host[:] = rng.integers(0, 256, host.size, dtype=np.uint8)
        host0, dev0 = host.view(np.uint16).copy(), gh.to_np(bufs, 2)
        kv = hc.DeviceKV(bufs, Dp)
        with hc.Engine(pool) as eng:
            # the first request waits on a stream that is busy for ~50 ms, so the
            # threads' requests queue up behind it
            blocker = torch.cuda.Stream()
            with torch.cuda.stream(blocker):
                torch.cuda._sleep(int(1e8))
            first = eng.submit(kv, perm[:96], hperm[:96], hc.BACKUP, after_stream=blocker)
            got_tickets = []

            def submitter(reqs):
                for d, dp, hp in reqs:
                    got_tickets.append(eng.submit(kv, dp, hp, d))
            ts = [threading.Thread(target=submitter, args=(back,)),
                  threading.Thread(target=submitter, args=(load,))]
            for t in ts:
                t.start()
            for t in ts:
                t.join()
            for t in got_tickets + [first]:
                eng.wait(t)
            launches, fused = eng.stats()
        assert fused >= 1, (launches, fused)
        # all requests are hazard-free against each other except the first,
        # which precedes them all: order among the rest does not matter
        oracle_apply([(hc.BACKUP, perm[:96], hperm[:96])] + back + load, dev0, host0, B, L, P, R, Hp, 0)
        assert np.array_equal(host.view(np.uint16), host0)
        got = gh.to_np(bufs, 2)
        for k in range(B * L):
            assert np.array_equal(got[k], dev0[k])


def test_after_stream_dependency_and_wait_on_stream():
    B, L, P, R, Dp, Hp = 1, 2, 4, 64, 8, 8
    bufs = [torch.zeros((Dp * P, R), dtype=torch.int16, device="cuda") for _ in range(B * L)]
    comp = torch.cuda.Stream()
    with hc.Pool(L, B, P, R, Hp, "page_first") as pool:
        pool.host_array()[:] = 0
        kv = hc.DeviceKV(bufs, Dp)
        torch.cuda.synchronize()
        with hc.Engine(pool) as eng:
            with torch.cuda.stream(comp):
                torch.cuda._sleep(int(3e8))          # the "compute" is still running...
                for b in bufs:
                    b[3 * P:4 * P].fill_(1234)       # ...when it writes page 3
            t = eng.submit(kv, [3], [5], hc.BACKUP, after_stream=comp)
            eng.wait(t)
            host = pool.host_array(np.int16)
            assert (host != 0).sum() == L * P * R and set(np.unique(host)) == {0, 1234}
            # a load, then compute that must see it
            t2 = eng.submit(kv, [6], [5], hc.LOAD)
            eng.wait_on_stream(t2, comp)
            with torch.cuda.stream(comp):
                s = torch.stack([b[6 * P:7 * P].float().sum() for b in bufs])
            comp.synchronize()
            assert torch.all(s == 1234.0 * P * R)


def test_refused_requests_are_not_queued():
    B, L, P, R, Dp, Hp = 1, 2, 4, 64, 8, 8
    bufs = [torch.zeros((Dp * P, R), dtype=torch.int16, device="cuda") for _ in range(B * L)]
    with hc.Pool(L, B, P, R, Hp, "layer_first") as pool:
        kv = hc.DeviceKV(bufs, Dp)
        with hc.Engine(pool) as eng:
            with pytest.raises(hc.HiCacheError) as e:
                eng.submit(kv, [0, 0], [1, 2], hc.LOAD)
            assert e.value.status == "DUPLICATE_INDEX"
            with pytest.raises(hc.HiCacheError) as e:
                eng.submit(kv, [9], [1], hc.BACKUP)
            assert e.value.status == "INDEX_RANGE"
            t = eng.submit(kv, [1], [1], hc.BACKUP)
            assert t == 1                               # the refused ones took no ticket
            eng.wait(t)
            with pytest.raises(hc.HiCacheError) as e:
                eng.wait(7)
            assert e.value.status == "INVALID_ARG"
            assert eng.stats() == (1, 0)


@pytest.mark.parametrize("conflict", [False, True], ids=["commutes", "conflicts"])
def test_lookahead_pairs_only_commuting_requests(conflict):
    """Queue: a backup B0 held back by a busy stream, then backups B1, B2 and a
    load L1.  B1 goes out right behind B0; L1 is paired with B2 (or with B1,
    overtaking B2) when it commutes, and otherwise follows alone.  Either way
    the result is the oracle's in submission order."""
    B, L, P, R, Dp, Hp = 2, 8, 16, 1024, 512, 512
    rng = np.random.default_rng(97)
    bufs = gh.random_device_bufs(B, L, P, R, Dp, seed=97)
    perm, hperm = rng.permutation(Dp), rng.permutation(Hp)
    b0 = (hc.BACKUP, perm[:400], hperm[:400])
    b1 = (hc.BACKUP, perm[400:404], hperm[400:404])
    b2 = (hc.BACKUP, perm[404:408], hperm[404:408])
    # the load writes device pages; in the conflicting case one of them is a page B2 reads
    l_dev = np.concatenate([perm[408:411], perm[404:405]]) if conflict else perm[408:412]
    l1 = (hc.LOAD, l_dev, hperm[420:424])
    with hc.Pool(L, B, P, R, Hp, "page_first_direct") as pool:
        host = pool.host_array(np.uint8)
        host[:] = rng.integers(0, 256, host.size, dtype=np.uint8)
        host0, dev0 = host.view(np.uint16).copy(), gh.to_np(bufs, 2)
        kv = hc.DeviceKV(bufs, Dp)
        with hc.Engine(pool) as eng:
            blocker = torch.cuda.Stream()        # holds B0 for ~50 ms while the rest queue
            with torch.cuda.stream(blocker):
                torch.cuda._sleep(int(1e8))
            ts = [eng.submit(kv, b0[1], b0[2], b0[0], after_stream=blocker)]
            ts += [eng.submit(kv, dp, hp, d) for d, dp, hp in (b1, b2, l1)]
            for t in ts:
                eng.wait(t)
            launches, fused = eng.stats()
        assert (launches, fused) == ((4, 0) if conflict else (3, 1))
        oracle_apply([b0, b1, b2, l1], dev0, host0, B, L, P, R, Hp, 2)
        assert np.array_equal(host.view(np.uint16), host0)
        got = gh.to_np(bufs, 2)
        for k in range(B * L):
            assert np.array_equal(got[k], dev0[k])


def test_three_threads_hammer_one_engine():
    """Three threads each submit 80 random requests on their own disjoint
    device and host pages (so the outcome does not depend on how the threads
    interleave) and wait on their own tickets as they go."""
    B, L, P, R, Dp, Hp = 2, 4, 8, 256, 96, 96
    rng = np.random.default_rng(99)
    bufs = gh.random_device_bufs(B, L, P, R, Dp, seed=99)
    dperm, hperm = rng.permutation(Dp), rng.permutation(Hp)
    parts = [(dperm[i::3], hperm[i::3]) for i in range(3)]
    plans = []
    for t, (dpages, hpages) in enumerate(parts):
        r = np.random.default_rng(200 + t)
        reqs = []
        for _ in range(80):
            n = int(r.integers(1, 9))
            reqs.append((int(r.integers(0, 2)), r.choice(dpages, n, replace=False), r.choice(hpages, n, replace=False)))
        plans.append(reqs)
    with hc.Pool(L, B, P, R, Hp, "page_first") as pool:
        host = pool.host_array(np.uint8)
        host[:] = rng.integers(0, 256, host.size, dtype=np.uint8)
        host0, dev0 = host.view(np.uint16).copy(), gh.to_np(bufs, 2)
        kv = hc.DeviceKV(bufs, Dp)
        errors = []
        with hc.Engine(pool) as eng:
            def worker(reqs):
                try:
                    ts = []
                    for k, (d, dp, hp) in enumerate(reqs):
                        ts.append(eng.submit(kv, dp, hp, d))
                        if k % 7 == 6:
                            eng.wait(ts[k - 3])
                    for t in ts:
                        eng.wait(t)
                except Exception as e:  # reported below
                    errors.append(e)
            ths = [threading.Thread(target=worker, args=(p,)) for p in plans]
            for t in ths:
                t.start()
            for t in ths:
                t.join()
            launches, fused = eng.stats()
        assert not errors, errors
        assert launches + fused == 240
        for reqs in plans:
            oracle_apply(reqs, dev0, host0, B, L, P, R, Hp, 1)
        assert np.array_equal(host.view(np.uint16), host0)
        got = gh.to_np(bufs, 2)
        for k in range(B * L):
            assert np.array_equal(got[k], dev0[k])
