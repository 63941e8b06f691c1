"""Pins for the CPU oracle: checks against facts that do not come from the oracle.

Every pin takes an ``oracle.Oracle`` and raises AssertionError when the oracle
disagrees with:
  * host-pool contents worked out by hand from the dims the pages print
    (tests/golden/hand_worked_layouts.txt), for backup and for load;
  * numpy reshape/transpose/fancy-indexing of the stacked device pool, which is
    what a whole-pool backup must reduce to under each layout's printed dims;
  * the segment counts the pages print (tests/golden/segment_counts.txt) and
    the closed forms behind them;
  * invariants: every host element written exactly once when every page moves,
    backup -> load round trip is the identity, untouched memory stays untouched,
    a per-layer load touches only its layer.

The pins are plain functions so that ``test_oracle_mutants.py`` can run them
against deliberately broken builds of the oracle and check that each plausible
mistake is caught by at least one of them.
"""
from __future__ import annotations

import os
import re

import numpy as np

import oracle as orc_mod

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
LAYOUT_IDS = orc_mod.LAYOUTS


# --------------------------------------------------------------------------
# golden parsing
def parse_hand_worked(path=os.path.join(GOLDEN, "hand_worked_layouts.txt")):
    cases = []
    cur = None
    with open(path, encoding="utf-8") as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("case "):
                parts = line.split()
                kv = dict(p.split("=", 1) for p in parts[2:])
                cur = {
                    "name": parts[1],
                    **{k: int(kv[k]) for k in ("B", "L", "P", "R", "Dp", "Hp")},
                    "dev": [int(x) for x in kv["dev"].split(",")],
                    "host": [int(x) for x in kv["host"].split(",")],
                    "layouts": {},
                }
                cases.append(cur)
            else:
                name, *syms = line.split()
                cur["layouts"][name] = syms
    return cases


def parse_segment_counts(path=os.path.join(GOLDEN, "segment_counts.txt")):
    rows = []
    with open(path, encoding="utf-8") as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            lay, B, L, P, R, n, dpat, hpat, exp = line.split()
            rows.append(dict(layout=lay, B=int(B), L=int(L), P=int(P), R=int(R), n=int(n),
                             dev_pattern=dpat, host_pattern=hpat, expected=int(exp)))
    return rows


# --------------------------------------------------------------------------
# helpers
BUF_NAMES = "KV"


def coded_device(B, L, P, R, Dp, dtype=np.uint16):
    """Device buffers whose every element holds a unique non-zero code."""
    bufs = []
    for b in range(B):
        for l in range(L):
            slot = np.arange(Dp * P)[:, None]
            e = np.arange(R)[None, :]
            code = 1 + ((b * L + l) * (Dp * P) + slot) * R + e
            bufs.append(np.ascontiguousarray(code.astype(dtype)))
    return bufs


def code_of(sym, L, P, R, Dp):
    m = re.fullmatch(r"([KV])\.l(\d+)\.s(\d+)\.e(\d+)", sym)
    b = BUF_NAMES.index(m.group(1))
    l, s, e = int(m.group(2)), int(m.group(3)), int(m.group(4))
    return 1 + ((b * L + l) * (Dp * P) + s) * R + e


def host_elems(B, L, P, R, Hp):
    return B * L * Hp * P * R


def stacked(bufs, B, L):
    return np.stack(bufs).reshape(B, L, *bufs[0].shape)


# --------------------------------------------------------------------------
# pins
def pin_hand_worked_backup(o):
    for c in parse_hand_worked():
        B, L, P, R, Dp, Hp = (c[k] for k in ("B", "L", "P", "R", "Dp", "Hp"))
        for lay, syms in c["layouts"].items():
            dev = coded_device(B, L, P, R, Dp)
            host = np.zeros(host_elems(B, L, P, R, Hp), np.uint16)
            o.backup(dev, host, B, L, P, R, Hp, c["dev"], c["host"], LAYOUT_IDS[lay])
            want = np.array([0 if s == "_" else code_of(s, L, P, R, Dp) for s in syms], np.uint16)
            assert want.size == host.size, (c["name"], lay, "golden length")
            assert np.array_equal(host, want), (c["name"], lay, host.tolist(), want.tolist())


def pin_hand_worked_load(o):
    for c in parse_hand_worked():
        B, L, P, R, Dp, Hp = (c[k] for k in ("B", "L", "P", "R", "Dp", "Hp"))
        for lay, syms in c["layouts"].items():
            host = np.array([0 if s == "_" else code_of(s, L, P, R, Dp) for s in syms], np.uint16)
            dev = [np.zeros((Dp * P, R), np.uint16) for _ in range(B * L)]
            o.load(dev, host, B, L, P, R, Hp, c["dev"], c["host"], LAYOUT_IDS[lay])
            want = coded_device(B, L, P, R, Dp)
            moved = np.zeros(Dp * P, bool)
            for d in c["dev"]:
                moved[d * P:(d + 1) * P] = True
            for k in range(B * L):
                w = np.where(moved[:, None], want[k], 0).astype(np.uint16)
                assert np.array_equal(dev[k], w), (c["name"], lay, k)


def pin_load_layer_touches_one_layer(o):
    c = [c for c in parse_hand_worked() if c["name"] == "middle"][0]
    B, L, P, R, Dp, Hp = (c[k] for k in ("B", "L", "P", "R", "Dp", "Hp"))
    for lay, syms in c["layouts"].items():
        host = np.array([0 if s == "_" else code_of(s, L, P, R, Dp) for s in syms], np.uint16)
        for layer in range(L):
            dev = [np.zeros((Dp * P, R), np.uint16) for _ in range(B * L)]
            o.load(dev, host, B, L, P, R, Hp, c["dev"], c["host"], LAYOUT_IDS[lay], layer)
            want = coded_device(B, L, P, R, Dp)
            for b in range(B):
                for l in range(L):
                    got = dev[b * L + l]
                    if l != layer:
                        assert not got.any(), (lay, layer, b, l)
                    else:
                        d = c["dev"][0]
                        assert np.array_equal(got[d * P:(d + 1) * P], want[b * L + l][d * P:(d + 1) * P])


def _numpy_layout(D, P, lay):
    """Whole-pool host image under each printed dims, from the stacked device
    pool D of shape (B, L, Hp*P, R) via numpy reshape/transpose."""
    B, L, S, R = D.shape
    if lay == "layer_first":          # (B, layer, size, kv_dim)
        return D.reshape(-1)
    if lay == "page_first":           # (B, size, layer, kv_dim)
        return D.transpose(0, 2, 1, 3).reshape(-1)
    Hp = S // P
    if lay == "page_first_direct_kv":  # (page_num, B, layer_num, page_size, kv_dim)
        return D.reshape(B, L, Hp, P, R).transpose(2, 0, 1, 3, 4).reshape(-1)
    # (B, page_num, layer_num, page_size, kv_dim)
    return D.reshape(B, L, Hp, P, R).transpose(0, 2, 1, 3, 4).reshape(-1)


def pin_numpy_transpose(o):
    rng = np.random.default_rng(7)
    for (B, L, P, R, Hp, dtype) in [(2, 3, 4, 5, 6, np.uint16), (1, 5, 2, 8, 3, np.uint16),
                                    (2, 2, 3, 2, 4, np.uint32), (1, 1, 1, 1, 1, np.uint8),
                                    (2, 4, 8, 16, 5, np.uint64)]:
        Dp = Hp + 2
        dev = [rng.integers(0, np.iinfo(dtype).max, size=(Dp * P, R), dtype=dtype) for _ in range(B * L)]
        D = np.stack(dev).reshape(B, L, Dp, P, R)
        # pair host page h with device page perm[h]
        perm = rng.permutation(Dp)[:Hp]
        # fancy-index the device pool into host page order, then lay it out
        Dh = D[:, :, perm].reshape(B, L, Hp * P, R)
        for lay, lid in LAYOUT_IDS.items():
            host = np.zeros(host_elems(B, L, P, R, Hp), dtype)
            o.backup(dev, host, B, L, P, R, Hp, perm, np.arange(Hp), lid)
            want = _numpy_layout(Dh, P, lay)
            assert np.array_equal(host, want), (lay, B, L, P, R, Hp, dtype)
            # load it back into a fresh pool at a second permutation
            back = [np.zeros_like(x) for x in dev]
            perm2 = rng.permutation(Dp)[:Hp]
            o.load(back, host, B, L, P, R, Hp, perm2, np.arange(Hp), lid)
            Db = np.stack(back).reshape(B, L, Dp, P, R)
            assert np.array_equal(Db[:, :, perm2], D[:, :, perm]), (lay, "load")


def pin_bijection(o):
    """All Hp pages moved: each host element written once, none twice."""
    rng = np.random.default_rng(11)
    for (B, L, P, R, Hp) in [(2, 3, 4, 8, 5), (1, 4, 2, 16, 7)]:
        Dp = Hp
        dev = coded_device(B, L, P, R, Dp, dtype=np.uint32)
        perm = rng.permutation(Dp)
        for lay, lid in LAYOUT_IDS.items():
            host = np.zeros(host_elems(B, L, P, R, Hp), np.uint32)
            o.backup(dev, host, B, L, P, R, Hp, perm, np.arange(Hp), lid)
            assert (host != 0).all(), (lay, "unwritten host element")
            assert np.array_equal(np.sort(host), np.sort(np.concatenate([x.ravel() for x in dev]))), lay


def pin_roundtrip_and_untouched(o):
    rng = np.random.default_rng(13)
    B, L, P, R, Dp, Hp = 2, 3, 4, 8, 16, 24
    for lay, lid in LAYOUT_IDS.items():
        for n in (0, 1, 5, 12):
            dev = coded_device(B, L, P, R, Dp)
            src = rng.choice(Dp, n, replace=False)
            hp = rng.choice(Hp, n, replace=False)
            host = np.full(host_elems(B, L, P, R, Hp), 0xFFFF, np.uint16)
            o.backup(dev, host, B, L, P, R, Hp, src, hp, lid)
            # host elements not in moved pages keep the sentinel
            touched = np.zeros(host.size, bool)
            for h in hp:
                for b in range(B):
                    for l in range(L):
                        for t in range(P):
                            off = o.host_offset(lid, B, L, P, R, Hp, b, l, int(h), t, 0)
                            touched[off:off + R] = True
            assert (host[~touched] == 0xFFFF).all(), (lay, n)
            assert (host[touched] != 0xFFFF).all(), (lay, n)
            dst = rng.choice(Dp, n, replace=False)
            back = [np.full((Dp * P, R), 0xFFFF, np.uint16) for _ in range(B * L)]
            o.load(back, host, B, L, P, R, Hp, dst, hp, lid)
            for k in range(B * L):
                for s_, d_ in zip(src, dst):
                    assert np.array_equal(back[k][d_ * P:(d_ + 1) * P], dev[k][s_ * P:(s_ + 1) * P])
                mask = np.ones(Dp * P, bool)
                for d_ in dst:
                    mask[d_ * P:(d_ + 1) * P] = False
                assert (back[k][mask] == 0xFFFF).all()


def _runs(dp, hp):
    """Maximal runs of pairs where the device AND the host page both step by
    one, counted on the pairs sorted by (host page, device page)."""
    order = np.lexsort((np.asarray(dp), np.asarray(hp)))
    d, h = np.asarray(dp)[order], np.asarray(hp)[order]
    if len(d) == 0:
        return 0
    return 1 + int(np.sum(~((np.diff(d) == 1) & (np.diff(h) == 1))))


def pin_segment_counts_printed(o):
    rng = np.random.default_rng(17)
    for row in parse_segment_counts():
        n = row["n"]
        dp = np.arange(n) if row["dev_pattern"] == "contiguous" else rng.permutation(4 * n)[:n]
        hp = np.arange(n) if row["host_pattern"] == "contiguous" else rng.permutation(4 * n)[:n]
        Hp = 4 * n
        got = o.segment_count(row["B"], row["L"], row["P"], row["R"], Hp, dp, hp,
                              LAYOUT_IDS[row["layout"]])
        assert got == row["expected"], (row, got)


def pin_segment_count_closed_forms(o):
    rng = np.random.default_rng(19)
    for (B, L, P, R, Dp, Hp, n) in [(2, 5, 4, 8, 64, 64, 20), (1, 3, 1, 4, 16, 32, 9),
                                    (2, 2, 16, 128, 64, 128, 12)]:
        assert L > 1
        for pattern in ("runs", "scattered", "contiguous", "contiguous_shuffled"):
            if pattern == "contiguous":
                dp, hp = np.arange(n) + 3, np.arange(n) + 1
            elif pattern == "contiguous_shuffled":
                # the same pairs in a random call order: still one run
                order = rng.permutation(n)
                dp, hp = (np.arange(n) + 3)[order], (np.arange(n) + 1)[order]
            elif pattern == "scattered":
                dp, hp = rng.choice(Dp, n, replace=False), rng.choice(Hp, n, replace=False)
            else:
                starts = np.sort(rng.choice(Dp // 4, n // 4 + 1, replace=False)) * 4
                dp = np.concatenate([np.arange(s, s + 4) for s in starts])[:n]
                hp = np.arange(n) * 1 + 2
            runs = _runs(dp, hp)
            assert o.segment_count(B, L, P, R, Hp, dp, hp, LAYOUT_IDS["layer_first"]) == B * L * runs
            # more than one layer: page_first_direct(_kv) never merges two pages of a
            # layer, page_first never merges two tokens of a layer
            assert o.segment_count(B, L, P, R, Hp, dp, hp, LAYOUT_IDS["page_first_direct"]) == B * L * n
            assert o.segment_count(B, L, P, R, Hp, dp, hp, LAYOUT_IDS["page_first_direct_kv"]) == B * L * n
            assert o.segment_count(B, L, P, R, Hp, dp, hp, LAYOUT_IDS["page_first"]) == B * L * n * P
            # one layer: page_first rows of one layer are L*R apart on the host
            assert o.segment_count(B, L, P, R, Hp, dp, hp, LAYOUT_IDS["page_first"], 1) == B * n * P
            assert o.segment_count(B, L, P, R, Hp, dp, hp, LAYOUT_IDS["layer_first"], 0) == B * runs
        # a repeated source page (a backup may copy one device page twice): the
        # count does not depend on the order of the arguments
        dp2 = np.array([1, 2, 2, 7]); hp2 = np.array([3, 9, 4, 5])
        for perm in ([0, 1, 2, 3], [2, 0, 3, 1], [3, 2, 1, 0]):
            assert o.segment_count(B, L, P, R, Hp, dp2[perm], hp2[perm], LAYOUT_IDS["layer_first"]) \
                == B * L * _runs(dp2, hp2) == B * L * 3
        # a single layer pool: every layout but page_first_direct_kv degenerates to
        # layer_first's count; page_first_direct_kv still interleaves the buffers
        # inside each page, so only a one-buffer pool merges pages
        dp, hp = rng.choice(Dp, n, replace=False), rng.choice(Hp, n, replace=False)
        for name, lay in LAYOUT_IDS.items():
            want = B * _runs(dp, hp) if (name != "page_first_direct_kv" or B == 1) else B * n
            assert o.segment_count(B, 1, P, R, Hp, dp, hp, lay) == want, name


ALL_PINS = [pin_hand_worked_backup, pin_hand_worked_load, pin_load_layer_touches_one_layer,
            pin_numpy_transpose, pin_bijection, pin_roundtrip_and_untouched,
            pin_segment_counts_printed, pin_segment_count_closed_forms]


def run_all(lib_path=None):
    """Run every pin; returns the names of the pins that failed."""
    lib = orc_mod.load_library(lib_path) if lib_path else orc_mod.load_library()
    o = orc_mod.Oracle(lib)
    failed = []
    for pin in ALL_PINS:
        try:
            pin(o)
        except AssertionError:
            failed.append(pin.__name__)
    return failed
