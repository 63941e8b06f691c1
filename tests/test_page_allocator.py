"""The LIFO host-page allocator (host-only; no GPU)."""
import numpy as np
import pytest

import tiered_kv_cache_gb300 as hc
from tiered_kv_cache_gb300 import build as hc_build


@pytest.fixture(scope="module", autouse=True)
def built():
    hc_build.build()


def test_fresh_allocator_hands_out_ascending_runs():
    a = hc.PageAllocator(100)
    assert np.array_equal(a.alloc(10), np.arange(10))
    assert np.array_equal(a.alloc(5), np.arange(10, 15))
    assert a.available == 85


def test_lifo_reuses_the_most_recently_freed_pages():
    a = hc.PageAllocator(64)
    x = a.alloc(20)
    y = a.alloc(20)
    a.free(x[3:9])          # freed first
    a.free(y[10:14])        # freed last: handed out first
    got = a.alloc(4)
    assert np.array_equal(got, y[10:14])
    got = a.alloc(6)
    assert np.array_equal(got, x[3:9])
    # then the untouched tail of the pool
    assert np.array_equal(a.alloc(3), np.arange(40, 43))


def test_scattered_free_comes_back_as_merged_runs():
    a = hc.PageAllocator(32)
    a.alloc(32)
    a.free([9, 3, 4, 5, 10, 20])
    got = a.alloc(6)
    assert np.array_equal(got, [3, 4, 5, 9, 10, 20])   # lowest run first, each run ascending
    assert hc.prepass(32, 32, got, got, hc.BACKUP).shape[0] == 3


def test_random_sequences_keep_the_invariants():
    rng = np.random.default_rng(0)
    N = 500
    a = hc.PageAllocator(N)
    held = set()
    for _ in range(2000):
        if held and rng.random() < 0.5:
            k = int(rng.integers(1, len(held) + 1))
            out = rng.choice(sorted(held), k, replace=False)
            a.free(out)
            held -= set(int(x) for x in out)
        else:
            n = int(rng.integers(0, 40))
            if n > N - len(held):
                with pytest.raises(hc.HiCacheError) as e:
                    a.alloc(n)
                assert e.value.status == "NOMEM"
                continue
            got = a.alloc(n)
            assert len(set(got.tolist())) == n and not (set(got.tolist()) & held)
            assert ((got >= 0) & (got < N)).all()
            held |= set(got.tolist())
        assert a.available == N - len(held)
    a.free(sorted(held))
    assert a.available == N


def test_errors_leave_the_allocator_unchanged():
    a = hc.PageAllocator(16)
    x = a.alloc(8)
    with pytest.raises(hc.HiCacheError) as e:
        a.free([x[0], x[0]])
    assert e.value.status == "DUPLICATE_INDEX"
    with pytest.raises(hc.HiCacheError) as e:
        a.free([12])                      # never handed out
    assert e.value.status == "DUPLICATE_INDEX"
    with pytest.raises(hc.HiCacheError) as e:
        a.free([16])
    assert e.value.status == "INDEX_RANGE"
    with pytest.raises(hc.HiCacheError) as e:
        a.alloc(9)
    assert e.value.status == "NOMEM"
    assert a.available == 8
    a.free(x)
    assert a.available == 16
    with pytest.raises(hc.HiCacheError):
        hc.PageAllocator(0)
