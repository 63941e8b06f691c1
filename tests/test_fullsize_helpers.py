"""The whole-pool helpers of the full-size GPU tests, on the CPU: the oracle
run over disjoint pair groups on every core gives exactly the oracle's own
single call, and the chunked comparison finds every planted difference."""
import numpy as np
import pytest

import oracle

import fullsize as fs

LAYOUTS = [oracle.LAYER_FIRST, oracle.PAGE_FIRST, oracle.PAGE_FIRST_DIRECT, oracle.PAGE_FIRST_DIRECT_KV]


@pytest.mark.parametrize("layout", LAYOUTS)
def test_split_oracle_equals_one_call(layout):
    B, L, P, R, Dp, Hp, n = 2, 3, 4, 8, 96, 80, 61
    rng = np.random.default_rng(70 + layout)
    dev = [rng.integers(0, 1 << 16, (Dp * P, R), dtype=np.uint16) for _ in range(B * L)]
    dp = rng.choice(Dp, n, replace=False)
    hp = rng.choice(Hp, n, replace=False)
    o = oracle.Oracle()
    size = B * L * Hp * P * R
    one = np.full(size, 7, np.uint16)
    split = one.copy()
    o.backup(dev, one, B, L, P, R, Hp, dp, hp, layout)
    fs.oracle_backup(dev, split, B, L, P, R, Hp, dp, hp, layout)
    assert np.array_equal(one, split)
    for layer in (-1, 1):
        want = [np.full((Dp * P, R), 9, np.uint16) for _ in range(B * L)]
        got = [w.copy() for w in want]
        o.load(want, one, B, L, P, R, Hp, dp, hp, layout, layer)
        fs.oracle_load(got, one, B, L, P, R, Hp, dp, hp, layout, layer)
        assert all(np.array_equal(a, b) for a, b in zip(want, got))


def test_split_oracle_refuses_repeated_destinations():
    dev = [np.zeros((8, 4), np.uint16)]
    host = np.zeros(8 * 4, np.uint16)
    with pytest.raises(AssertionError):
        fs.oracle_backup(dev, host, 1, 1, 1, 4, 8, [0, 1], [3, 3], 0)
    with pytest.raises(AssertionError):
        fs.oracle_load(dev, host, 1, 1, 1, 4, 8, [2, 2], [0, 1], 0)


def test_mismatches_finds_planted_differences(monkeypatch):
    monkeypatch.setattr(fs, "CHUNK", 1000)           # many chunks
    a = np.arange(10_007, dtype=np.uint32)
    b = a.copy()
    assert fs.mismatches(a, b) == (0, -1)
    for i in (9_999, 17, 4_000):
        b[i] ^= 1
    assert fs.mismatches(a, b) == (3, 17)


def test_position_fill_and_copy(monkeypatch):
    monkeypatch.setattr(fs, "CHUNK", 1000)
    w = np.zeros(5_003, np.uint32)
    fs.position_fill(w, 2)
    assert np.array_equal(w, (np.arange(5_003, dtype=np.uint64) + (2 << 20)).astype(np.uint32))
    c = np.empty_like(w)
    fs.copy(c, w)
    assert np.array_equal(c, w)
    fs.fill(c.view(np.uint8), 0xC3)
    assert (c.view(np.uint8) == 0xC3).all()
