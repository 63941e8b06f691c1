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
