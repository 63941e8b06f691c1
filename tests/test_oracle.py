"""The CPU oracle against its pins (no GPU)."""
import pytest

import oracle_pins


@pytest.fixture(scope="module")
def orc():
    import oracle
    return oracle.Oracle()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_golden_files_parse():
    cases = oracle_pins.parse_hand_worked()
    assert {c["name"] for c in cases} == {"swap", "kv_rows", "middle"}
    for c in cases:
        assert set(c["layouts"]) == {"layer_first", "page_first", "page_first_direct",
                                     "page_first_direct_kv"}
    rows = oracle_pins.parse_segment_counts()
    assert {r["expected"] for r in rows} == {39936, 78}


def test_oracle_rejects_bad_arguments(orc):
    import numpy as np
    dev = [np.zeros((4, 2), np.uint16)]
    host = np.zeros(4 * 2, np.uint16)
    with pytest.raises(ValueError):
        orc.backup(dev, host, 1, 1, 2, 2, 2, [0], [2], 0)   # host page out of range
    with pytest.raises(ValueError):
        orc.backup(dev, host, 1, 1, 2, 2, 2, [0], [0], 7)   # unknown layout
    with pytest.raises(ValueError):
        orc.load(dev, host, 1, 1, 2, 2, 2, [0], [0], 0, 1)  # layer out of range


@pytest.mark.parametrize("shape", [(2, 3, 4, 5, 6), (1, 2, 3, 4, 2)])
def test_offset_helpers_follow_the_printed_dims(orc, shape):
    """The single-element offsets the sampled GPU checks use, against numpy's
    row-major flattening of each layout's printed dims (the K/V buffer dim in
    front, reading 3; inside the page for page_first_direct_kv)."""
    import numpy as np
    B, L, P, R, Hp = shape
    Dp = 3
    dims = {0: ((B, L, Hp * P, R), lambda b, l, h, t, e: (b, l, h * P + t, e)),
            1: ((B, Hp * P, L, R), lambda b, l, h, t, e: (b, h * P + t, l, e)),
            2: ((B, Hp, L, P, R), lambda b, l, h, t, e: (b, h, l, t, e)),
            3: ((Hp, B, L, P, R), lambda b, l, h, t, e: (h, b, l, t, e))}
    for layout, (shape_dims, idx) in dims.items():
        for b in range(B):
            for l in range(L):
                for h in range(Hp):
                    for t in range(P):
                        for e in range(R):
                            want = int(np.ravel_multi_index(idx(b, l, h, t, e), shape_dims))
                            assert orc.host_offset(layout, B, L, P, R, Hp, b, l, h, t, e) == want
    for d in range(Dp):
        for t in range(P):
            for e in range(R):
                assert orc.dev_offset(P, R, d, t, e) == int(np.ravel_multi_index((d * P + t, e), (Dp * P, R)))
