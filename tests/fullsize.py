"""Whole-pool parity at the workloads' full sizes (test infrastructure).

The oracle is a single-threaded element-by-element loop.  At 4-20 GiB per
transfer the tests run it over disjoint groups of one call's page pairs, one
group per host core.  A call's destinations are distinct (host pages on a
backup, device pages on a load; the library and the oracle both refuse a
repeated destination), so the groups write disjoint elements and together give
exactly the oracle's result for the whole call, in any order.  ctypes drops the
GIL around each oracle call, so plain threads run the groups in parallel.

Besides that split, nothing here computes an offset: fills, copies and
comparisons work on whole arrays cut into equal chunks."""
from __future__ import annotations

import ctypes
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import tiered_kv_cache_gb300 as hc

import gpu_helpers as gh

THREADS = max(1, min(32, os.cpu_count() or 1))
_pool = ThreadPoolExecutor(THREADS)
CHUNK = 1 << 26                       # elements per chunk of a fill or compare


def _parallel(fn, items):
    return list(_pool.map(fn, items))


def _splits(n: int, parts: int):
    parts = max(1, min(parts, n))
    edges = [n * k // parts for k in range(parts + 1)]
    return [(edges[k], edges[k + 1]) for k in range(parts) if edges[k + 1] > edges[k]]


def oracle_backup(dev_np, host_np, B, L, P, R, Hp, dp, hp, layout):
    """The oracle's backup of the pairs (dp[i], hp[i]), run over disjoint pair groups."""
    dp = np.asarray(dp, np.int64)
    hp = np.asarray(hp, np.int64)
    assert len(np.unique(hp)) == len(hp), "a backup's host pages must be distinct"
    o = gh.orc()
    _parallel(lambda ab: o.backup(dev_np, host_np, B, L, P, R, Hp, dp[ab[0]:ab[1]], hp[ab[0]:ab[1]], layout),
              _splits(len(dp), THREADS))


def oracle_load(dev_np, host_np, B, L, P, R, Hp, dp, hp, layout, layer=-1):
    """The oracle's load (every layer, or one) of the pairs, over disjoint pair groups."""
    dp = np.asarray(dp, np.int64)
    hp = np.asarray(hp, np.int64)
    assert len(np.unique(dp)) == len(dp), "a load's device pages must be distinct"
    o = gh.orc()
    _parallel(lambda ab: o.load(dev_np, host_np, B, L, P, R, Hp, dp[ab[0]:ab[1]], hp[ab[0]:ab[1]], layout,
                                layer),
              _splits(len(dp), THREADS))


def fill(a: np.ndarray, value):
    a = a.reshape(-1)
    _parallel(lambda ab: a[ab[0]:ab[1]].fill(value), _splits(a.size, max(1, a.size // CHUNK)))


def copy(dst: np.ndarray, src: np.ndarray):
    d, s = dst.reshape(-1), src.reshape(-1)
    assert d.dtype == s.dtype and d.size == s.size
    _parallel(lambda ab: np.copyto(d[ab[0]:ab[1]], s[ab[0]:ab[1]]), _splits(d.size, max(1, d.size // CHUNK)))


def position_fill(words: np.ndarray, salt: int = 0):
    """32-bit words = (their own index + salt * 2^20) mod 2^32, so any misplaced
    copy shows and two fills with different salts differ everywhere."""
    w = words.reshape(-1)
    assert w.dtype == np.uint32

    def part(ab):
        a, b = ab
        w[a:b] = (np.arange(a, b, dtype=np.uint64) + (salt << 20)).astype(np.uint32)

    _parallel(part, _splits(w.size, max(1, w.size // CHUNK)))


def mismatches(got: np.ndarray, want: np.ndarray) -> tuple[int, int]:
    """(number of differing elements, index of the first), compared chunk by
    chunk on every core; (0, -1) when the arrays are equal."""
    g, w = got.reshape(-1), want.reshape(-1)
    assert g.dtype == w.dtype and g.size == w.size

    def part(ab):
        a, b = ab
        if np.array_equal(g[a:b], w[a:b]):
            return 0, -1
        bad = np.flatnonzero(g[a:b] != w[a:b])
        return int(bad.size), a + int(bad[0])

    res = _parallel(part, _splits(g.size, max(1, g.size // CHUNK)))
    count = sum(c for c, _ in res)
    first = next((f for c, f in res if c), -1)
    return count, first


def assert_equal(got: np.ndarray, want: np.ndarray, what: str):
    count, first = mismatches(got, want)
    assert count == 0, f"{what}: {count} elements differ from the oracle, the first at {first}"


class DeviceMirror:
    """Pinned host copies of a set of device buffers: pull() copies the device
    into them; the oracle then reads or writes them as numpy arrays; compare()
    checks every device buffer against them, on the GPU."""

    def __init__(self, bufs):
        self.shapes = [tuple(b.shape) for b in bufs]
        self.dtypes = [b.dtype for b in bufs]
        sizes = [b.numel() * b.element_size() for b in bufs]
        self.mem = hc.PinnedHost(sum(sizes))
        raw = np.frombuffer((ctypes.c_uint8 * self.mem.nbytes).from_address(self.mem.ptr),
                            dtype=np.uint8)
        self.t, self.np, off = [], [], 0
        for b, nbytes in zip(bufs, sizes):
            u8 = raw[off:off + nbytes]
            t = torch.from_numpy(u8).view(b.dtype).view(b.shape)
            self.t.append(t)
            self.np.append(u8.view(gh.NP_DT[b.element_size()]).reshape(b.shape[0], -1))
            off += nbytes

    def pull(self, bufs):
        for t, b in zip(self.t, bufs):
            t.copy_(b)
        torch.cuda.synchronize()

    def fill(self, byte_value: int):
        for a in self.np:
            fill(a.view(np.uint8), byte_value)

    def compare(self, bufs, what: str):
        """Every device buffer against its mirror, element by element (the
        mirror is uploaded one buffer at a time and compared on the GPU)."""
        bad = []
        for k, (t, b) in enumerate(zip(self.t, bufs)):
            want = t.to(b.device).view(torch.uint8)
            got = b.view(torch.uint8)
            if not torch.equal(want, got):                 # bytes: NaN payloads compare too
                diff = (want != got).view(-1)
                bad.append((k, int(diff.sum()), int(diff.nonzero()[0])))
            del want
        assert not bad, f"{what}: device buffers differ from the oracle (buffer, bytes, first byte): {bad[:4]}"

    def close(self):
        self.t, self.np = [], []
        self.mem.free()


def randomize(bufs, seed: int):
    """Random bit patterns in every device buffer (NaNs and signed zeros included)."""
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    for b in bufs:
        b.view(torch.uint8).random_(0, 256, generator=g)


def normal_fill(bufs, seed: int):
    """bf16 normal(0, 1) values in every device buffer (the workloads' value
    distribution), from a seeded generator."""
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    for b in bufs:
        b.view(torch.bfloat16).normal_(generator=g)
