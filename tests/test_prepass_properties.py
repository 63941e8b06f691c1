"""Property tests of the pre-pass (validation and run building) on the host:
for any pairs, sorted or not, of any size on either side of the point where
calls start building their runs in chunks, the library either returns the
runs of a plain Python merge of the pairs sorted by (host page, device page),
or refuses with the status a plain reading of the rules gives: an index out
of range first, else a destination named twice."""
import numpy as np
import pytest

import tiered_kv_cache_gb300 as hc

hypothesis = pytest.importorskip("hypothesis")
st = hypothesis.strategies


def reference(dp, hp, Dp, Hp, direction):
    if any(not 0 <= d < Dp for d in dp) or any(not 0 <= h < Hp for h in hp):
        return "INDEX_RANGE"
    dst = hp if direction == hc.BACKUP else dp
    if len(set(dst)) != len(dst):
        return "DUPLICATE_INDEX"
    runs = []
    for h, d in sorted(zip(hp, dp)):
        if runs and h == runs[-1][0] + runs[-1][2] and d == runs[-1][1] + runs[-1][2]:
            runs[-1][2] += 1
        else:
            runs.append([h, d, 1])
    return np.array(runs, np.int64).reshape(-1, 3)


@st.composite
def calls(draw):
    Dp = draw(st.integers(1, 300))
    Hp = draw(st.integers(1, 300))
    n = draw(st.integers(0, 120))
    shape = draw(st.sampled_from(["random", "host_sorted", "runs"]))
    rng = np.random.default_rng(draw(st.integers(0, 2**32 - 1)))
    if shape == "runs" and n <= min(Dp, Hp):
        d0 = int(rng.integers(0, Dp - n + 1))
        h0 = int(rng.integers(0, Hp - n + 1))
        dp, hp = np.arange(d0, d0 + n), np.arange(h0, h0 + n)
        cut = rng.permutation(n)
        dp, hp = dp[cut], hp[cut]
    else:
        dp = rng.integers(-2, Dp + 2, n)
        hp = rng.integers(-2, Hp + 2, n)
        if draw(st.booleans()):                       # mostly valid: clip into range
            dp, hp = np.clip(dp, 0, Dp - 1), np.clip(hp, 0, Hp - 1)
        if shape == "host_sorted":
            order = np.lexsort((dp, hp))
            dp, hp = dp[order], hp[order]
    direction = draw(st.sampled_from([hc.BACKUP, hc.LOAD]))
    return [int(x) for x in dp], [int(x) for x in hp], Dp, Hp, direction


@hypothesis.settings(max_examples=400, deadline=None)
@hypothesis.given(calls())
def test_prepass_matches_a_plain_merge(call):
    dp, hp, Dp, Hp, direction = call
    want = reference(dp, hp, Dp, Hp, direction)
    if isinstance(want, str):
        with pytest.raises(hc.HiCacheError) as e:
            hc.prepass(Hp, Dp, dp, hp, direction)
        assert e.value.status == want
    else:
        assert np.array_equal(hc.prepass(Hp, Dp, dp, hp, direction), want)


@pytest.mark.parametrize("n", [4095, 4096, 4097, 9000])
@pytest.mark.parametrize("direction", [hc.BACKUP, hc.LOAD])
def test_large_sorted_and_unsorted_agree(n, direction):
    """Around the size where a call builds its runs in chunks: the same pairs
    in host order and shuffled reduce to the same runs."""
    rng = np.random.default_rng(n + direction)
    Dp = Hp = 2 * n
    k = n // 3                                                # one long run first, then scattered pages
    rest = rng.permutation(np.setdiff1d(np.arange(Dp), np.arange(7, 7 + k)))[: n - k]
    dp = np.concatenate([np.arange(7, 7 + k), rest])
    hp = np.concatenate([np.arange(k), np.sort(rng.choice(np.arange(k, Hp), n - k, replace=False))])
    a = hc.prepass(Hp, Dp, dp, hp, direction)
    perm = rng.permutation(n)
    b = hc.prepass(Hp, Dp, dp[perm], hp[perm], direction)
    assert np.array_equal(a, b)
    assert np.array_equal(a, reference(list(dp), list(hp), Dp, Hp, direction))
