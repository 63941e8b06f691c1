"""The host's validation of large calls, split over worker threads: calls of
49,152 pairs or more are scanned in chunks by up to four threads, each with a
bitmap of its own, merged afterwards.  Every error must still be found and
reported exactly as one pass over the pairs reports it, wherever it sits
relative to the parts, and the runs must not change (CPU only)."""
import multiprocessing as mp
import threading

import numpy as np
import pytest

import tiered_kv_cache_gb300 as hc

from test_host_logic import py_runs

N = 100_003                      # above the split threshold, not a multiple of the part count
DP, HP = 3 * N, 2 * N + 7


def scattered(seed, n=N):
    """Host pages in order (as the allocator hands them out), device pages a
    random sample: one-token pages, no runs."""
    rng = np.random.default_rng(seed)
    dp = rng.choice(DP, n, replace=False).astype(np.int64)
    hp = np.sort(rng.choice(HP, n, replace=False)).astype(np.int64)
    return dp, hp


def boundaries(n=N, chunks=(2, 3, 4)):
    """Every pair index next to a boundary of n pairs split into each number of
    `chunks`, and the first and last pair."""
    out = {0, 1, n - 1}
    for parts in chunks:
        for k in range(1, parts):
            b = n * k // parts
            out |= {b - 1, b, b + 1}
    return sorted(out)


# the scan hands out the pairs in 32 chunks: the first pair of each chunk after the first
CHUNK_EDGES = [N * c // 32 for c in range(1, 32)]


def raises(status, fn, *args):
    with pytest.raises(hc.HiCacheError) as e:
        fn(*args)
    assert e.value.status == status, str(e.value)
    return str(e.value)


@pytest.mark.parametrize("seed", range(2))
def test_valid_sets_give_the_plain_runs(seed):
    dp, hp = scattered(seed)
    want = py_runs(dp, hp)
    for direction in (hc.BACKUP, hc.LOAD):
        assert np.array_equal(hc.prepass(HP, DP, dp, hp, direction), want)
    # the pairs shuffled: the sorted path
    perm = np.random.default_rng(seed).permutation(N)
    for direction in (hc.BACKUP, hc.LOAD):
        assert np.array_equal(hc.prepass(HP, DP, dp[perm], hp[perm], direction), want)
    # long runs on both sides
    dp2 = np.arange(N, dtype=np.int64) + 11
    hp2 = np.arange(N, dtype=np.int64) + 5
    for direction in (hc.BACKUP, hc.LOAD):
        assert np.array_equal(hc.prepass(HP, DP, dp2, hp2, direction), py_runs(dp2, hp2))


@pytest.mark.parametrize("pos", boundaries())
def test_range_errors_report_the_first(pos):
    dp, hp = scattered(7)
    bad = dp.copy()
    bad[pos] = DP                                   # one past the end
    msg = raises("INDEX_RANGE", hc.prepass, HP, DP, bad, hp, hc.LOAD)
    assert f"device_pages[{pos}] = {DP}" in msg
    badh = hp.copy()
    badh[pos] = -1
    msg = raises("INDEX_RANGE", hc.prepass, HP, DP, dp, badh, hc.BACKUP)
    assert f"host_pages[{pos}] = -1" in msg
    # a second error in a later part: the earlier one is named
    if pos < N - 10:
        bad[N - 3] = -5
        msg = raises("INDEX_RANGE", hc.prepass, HP, DP, bad, hp, hc.BACKUP)
        assert f"device_pages[{pos}]" in msg


@pytest.mark.parametrize("pos", boundaries())
def test_repeated_destinations_in_and_across_parts(pos):
    dp, hp = scattered(11)
    # a load: device page of pair pos repeated by a pair in another part (the
    # far end) and by its neighbour (the same part, or across a boundary)
    for other in ({0: N - 1}.get(pos, 0), pos - 1 if pos > 0 else 1):
        bad = dp.copy()
        bad[pos] = bad[other]
        msg = raises("DUPLICATE_INDEX", hc.prepass, HP, DP, bad, hp, hc.LOAD)
        assert f"device page {bad[pos]} " in msg
    # a backup in host order: an equal neighbour is the only way to repeat
    if pos > 0:
        badh = hp.copy()
        badh[pos] = badh[pos - 1]
        msg = raises("DUPLICATE_INDEX", hc.prepass, HP, DP, dp, badh, hc.BACKUP)
        assert f"host page {badh[pos]} " in msg
        # ... and the same host page repeated far away, order broken
        badh = hp.copy()
        badh[pos] = hp[0] if pos != 0 else hp[-1]
        raises("DUPLICATE_INDEX", hc.prepass, HP, DP, dp, badh, hc.BACKUP)


@pytest.mark.parametrize("pos", sorted(set(CHUNK_EDGES + [b for b in boundaries() if 0 < b < N - 1])))
def test_order_broken_only_across_a_boundary(pos):
    """Two neighbours swapped: each part on its own may still look sorted, so
    only the check across the boundary sends the call down the sorted path.
    The runs must be those of the sorted pairs either way."""
    dp = np.arange(N, dtype=np.int64) * 2 + 1
    hp = np.arange(N, dtype=np.int64) + 3
    hp[pos - 1], hp[pos] = hp[pos], hp[pos - 1]
    for direction in (hc.BACKUP, hc.LOAD):
        assert np.array_equal(hc.prepass(HP, DP, dp, hp, direction), py_runs(dp, hp))
    # equal host pages, device pages falling across the boundary: a load may do that
    hp = np.arange(N, dtype=np.int64) // 2
    dp = np.arange(N, dtype=np.int64)
    dp[pos - 1], dp[pos] = dp[pos], dp[pos - 1]
    assert np.array_equal(hc.prepass(HP, DP, dp, hp, hc.LOAD), py_runs(dp, hp))


def test_concurrent_callers():
    """Several threads validating large calls at once (the pool serves one;
    the others scan on their own): every result is the plain one."""
    sets = [scattered(100 + k) for k in range(6)]
    wants = [py_runs(dp, hp) for dp, hp in sets]
    errors = []

    def work(k):
        try:
            for rep in range(4):
                dp, hp = sets[(k + rep) % len(sets)]
                got = hc.prepass(HP, DP, dp, hp, hc.LOAD if rep % 2 else hc.BACKUP)
                assert np.array_equal(got, wants[(k + rep) % len(sets)])
                bad = dp.copy()
                bad[N // 2 + k] = bad[k]
                with pytest.raises(hc.HiCacheError):
                    hc.prepass(HP, DP, bad, hp, hc.LOAD)
        except BaseException as e:            # reported on the main thread
            errors.append(e)

    threads = [threading.Thread(target=work, args=(k,)) for k in range(6)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not any(t.is_alive() for t in threads)
    assert not errors, errors[0]


def _child(q):
    dp, hp = scattered(5)
    try:
        q.put(bool(np.array_equal(hc.prepass(HP, DP, dp, hp, hc.LOAD), py_runs(dp, hp))))
    except BaseException as e:
        q.put(repr(e))


@pytest.mark.filterwarnings("ignore:This process .* is multi-threaded:DeprecationWarning")
def test_forked_child_validates_large_calls():
    """A child forked after the workers started has none of them: it must
    start its own, not wait on its parent's."""
    dp, hp = scattered(5)
    hc.prepass(HP, DP, dp, hp, hc.LOAD)                 # the parent's pool exists
    ctx = mp.get_context("fork")
    q = ctx.Queue()
    p = ctx.Process(target=_child, args=(q,))
    p.start()
    p.join(timeout=120)
    if p.is_alive():
        p.kill()
        p.join()
        pytest.fail("the forked child hung in validation")
    assert p.exitcode == 0
    assert q.get(timeout=5) is True


_CHILD = r'''
import os, sys
import numpy as np
sys.path.insert(0, sys.argv[1])
import tiered_kv_cache_gb300 as hc
from test_validate_parts import scattered, HP, DP, N
from test_host_logic import py_runs
dp, hp = scattered(3)
before = len(os.listdir("/proc/self/task"))
assert np.array_equal(hc.prepass(HP, DP, dp, hp, hc.LOAD), py_runs(dp, hp))
started = len(os.listdir("/proc/self/task")) - before
bad = dp.copy()
bad[N // 2] = bad[N // 4]
try:
    hc.prepass(HP, DP, bad, hp, hc.LOAD)
    raise SystemExit("no error")
except hc.HiCacheError as e:
    print(started)
    print(e.status, str(e))
'''


def _run_child(env_threads):
    import os
    import subprocess
    import sys
    tests = os.path.dirname(os.path.abspath(__file__))
    root = os.path.dirname(tests)
    env = dict(os.environ, PYTHONPATH=os.pathsep.join([root, tests]))
    env.pop("HICACHE_VALIDATE_THREADS", None)
    if env_threads:
        env["HICACHE_VALIDATE_THREADS"] = env_threads
    r = subprocess.run([sys.executable, "-c", _CHILD, root], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr[-2000:]
    started, report = r.stdout.strip().split("\n", 1)
    return int(started), report


def test_one_thread_setting_gives_the_same_results():
    """HICACHE_VALIDATE_THREADS=1 keeps large calls on the calling thread:
    its first large call starts no thread, where by default it starts the
    workers, and the runs and the error report are the same either way."""
    import os
    one, report_one = _run_child("1")
    split, report_split = _run_child(None)
    assert one == 0
    if (os.cpu_count() or 1) >= 4:
        assert split >= 1
    assert report_one == report_split
    assert report_one.startswith("DUPLICATE_INDEX ") and "is a load destination twice" in report_one
