"""Host-side logic of libhicache, without a GPU: the library loads and exports
every symbol its header declares, the Python structs match the C ABI, and the
validation / pre-pass / segment-count code agrees with the oracle."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import tiered_kv_cache_gb300 as hc
from tiered_kv_cache_gb300 import build as hc_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "hicache.h")


@pytest.fixture(scope="module", autouse=True)
def built():
    hc_build.build()


def declared_functions():
    with open(HEADER, encoding="utf-8") as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(hicache_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol():
    names = declared_functions()
    assert len(names) >= 20
    out = subprocess.run(["nm", "-D", "--defined-only", hc.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (hicache_\w+)", out))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    lib = hc.library()
    for n in names:
        assert getattr(lib, n) is not None


def test_struct_layout_matches_c(tmp_path):
    prog = tmp_path / "sz.c"
    prog.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "hicache.h"\n'
        "int main(void){printf(\"%zu %zu %zu %zu %zu %zu\\n\", sizeof(hicache_pool_desc),"
        " offsetof(hicache_pool_desc,row_elems), offsetof(hicache_pool_desc,host_num_pages),"
        " offsetof(hicache_pool_desc,layout), sizeof(hicache_device_kv),"
        " offsetof(hicache_device_kv,device_num_pages));return 0;}\n")
    exe = tmp_path / "sz"
    subprocess.check_call(["gcc", "-std=c99", f"-I{os.path.join(ROOT, 'include')}", str(prog), "-o", str(exe)])
    vals = [int(x) for x in subprocess.check_output([str(exe)], text=True).split()]
    assert vals == [ctypes.sizeof(hc.PoolDesc), hc.PoolDesc.row_elems.offset,
                    hc.PoolDesc.host_num_pages.offset, hc.PoolDesc.layout.offset,
                    ctypes.sizeof(hc._DeviceKVStruct), hc._DeviceKVStruct.device_num_pages.offset]


def test_fast_division(tmp_path):
    """The multiply-high divider used by the kernels' address decode, run on the
    host (same source) against plain division."""
    prog = tmp_path / "fd.cpp"
    prog.write_text(r'''
#include <cstdio>
#include <cstdint>
#include <random>
#include "hicache_internal.h"
int main() {
  std::mt19937_64 rng(1);
  uint32_t divisors[] = {1,2,3,5,7,16,72,128,576,1000,4608,8192,9216,281088,299520,1048575,
                         (1u<<24), (1u<<25), (1u<<26), (1u<<30)+3u, 2147483647u};
  long bad = 0;
  for (uint32_t d : divisors) {
    hicache::FastDiv f = hicache::make_fastdiv(d);
    for (int k = 0; k < 200000; ++k) {
      uint32_t n = (k < 1000) ? uint32_t(k) : uint32_t(rng() & 0x7fffffffu);
      if (k >= 1000 && k < 2000) n = uint32_t(0x7fffffffu - (k - 1000));
      if (hicache::fast_div(n, f) != n / d) ++bad;
    }
    for (uint32_t m = 1; m < 64 && uint64_t(m) * d < 0x7fffffffu; ++m) {
      uint32_t n = m * d;
      if (hicache::fast_div(n, f) != m || hicache::fast_div(n - 1, f) != m - 1) ++bad;
    }
  }
  printf("%ld\n", bad);
  return 0;
}
''')
    exe = tmp_path / "fd"
    subprocess.check_call(["g++", "-O2", "-std=c++17",
                           f"-I{os.path.join(ROOT, 'tiered_kv_cache_gb300', 'csrc')}", str(prog), "-o", str(exe)])
    assert subprocess.check_output([str(exe)], text=True).strip() == "0"


def py_runs(dp, hp):
    order = np.lexsort((dp, hp))
    out = []
    for h, d in zip(hp[order], dp[order]):
        if out and h == out[-1][0] + out[-1][2] and d == out[-1][1] + out[-1][2]:
            out[-1][2] += 1
        else:
            out.append([h, d, 1])
    return np.array(out, np.int64).reshape(-1, 3)


@pytest.mark.parametrize("seed", range(6))
def test_prepass_runs(seed):
    rng = np.random.default_rng(seed)
    Dp, Hp = 300, 400
    n = int(rng.integers(0, 120))
    if seed % 2:
        starts = np.sort(rng.choice(Dp // 8, n // 8 + 1, replace=False)) * 8
        dp = np.concatenate([np.arange(s, s + 8) for s in starts])[:n]
        hp = (np.arange(n) + 5)
        perm = rng.permutation(n)
        dp, hp = dp[perm], hp[perm]
    else:
        dp = rng.choice(Dp, n, replace=False)
        hp = rng.choice(Hp, n, replace=False)
    for direction in (hc.BACKUP, hc.LOAD):
        runs = hc.prepass(Hp, Dp, dp, hp, direction)
        assert np.array_equal(runs, py_runs(np.asarray(dp, np.int64), np.asarray(hp, np.int64)))
        assert runs[:, 2].sum() == n


def test_prepass_errors():
    with pytest.raises(hc.HiCacheError) as e:
        hc.prepass(10, 10, [0, 10], [0, 1], hc.LOAD)
    assert e.value.status == "INDEX_RANGE"
    with pytest.raises(hc.HiCacheError) as e:
        hc.prepass(10, 10, [0, 1], [0, -1], hc.LOAD)
    assert e.value.status == "INDEX_RANGE"
    with pytest.raises(hc.HiCacheError) as e:       # a backup writes host page 3 twice
        hc.prepass(10, 10, [0, 1], [3, 3], hc.BACKUP)
    assert e.value.status == "DUPLICATE_INDEX"
    with pytest.raises(hc.HiCacheError) as e:       # a load writes device page 2 twice
        hc.prepass(10, 10, [2, 2], [3, 4], hc.LOAD)
    assert e.value.status == "DUPLICATE_INDEX"
    big = np.arange(100)
    with pytest.raises(hc.HiCacheError) as e:       # the sorted path of the same check
        hc.prepass(200, 200, np.concatenate([big, [7]]), np.arange(101), hc.LOAD)
    assert e.value.status == "DUPLICATE_INDEX"
    # repeated sources are allowed in both directions
    assert hc.prepass(10, 10, [2, 2], [3, 4], hc.BACKUP).shape == (2, 3)
    assert hc.prepass(10, 10, [2, 5], [3, 3], hc.LOAD).shape == (2, 3)
    # empty transfer
    assert hc.prepass(10, 10, [], [], hc.LOAD).shape == (0, 3)
    with pytest.raises(hc.HiCacheError) as e:
        hc.prepass(10, 10, [0], [0], 7)
    assert e.value.status == "INVALID_ARG"


def test_segment_count_matches_oracle():
    import oracle
    o = oracle.Oracle()
    rng = np.random.default_rng(3)
    for (B, L, P, R, Hp, Dp) in [(2, 5, 4, 8, 64, 64), (1, 3, 1, 4, 32, 16), (2, 1, 16, 128, 128, 64),
                                 (1, 4, 2, 16, 50, 40)]:
        for trial in range(4):
            n = int(rng.integers(1, min(Dp, Hp) // 2))
            if trial == 0:
                dp, hp = np.arange(n), np.arange(n) + 1
            elif trial == 1:
                dp = rng.choice(Dp, n, replace=False)
                hp = rng.choice(Hp, n, replace=False)
            else:
                s0 = int(rng.integers(0, Dp - n))
                dp = np.arange(s0, s0 + n)
                hp = np.sort(rng.choice(Hp, n, replace=False))
            for lay in hc.LAYOUTS.values():
                for layer in [-1] + list(range(L)):
                    want = o.segment_count(B, L, P, R, Hp, dp, hp, lay, layer)
                    got = hc.segment_count(L, B, P, R, Hp, lay, dp, hp, layer)
                    assert got == want, (B, L, P, R, lay, layer, trial)


def test_segment_count_printed_numbers():
    # 32K tokens, page_size 64, 78 layers, one latent buffer
    dp = np.arange(512)
    assert hc.segment_count(78, 1, 64, 576, 1024, "page_first_direct", dp, dp) == 39936
    assert hc.segment_count(78, 1, 64, 576, 1024, "layer_first", dp, dp) == 78
    scattered = np.random.default_rng(0).permutation(1024)[:512]
    assert hc.segment_count(78, 1, 64, 576, 1024, "page_first_direct", scattered, dp) == 39936
    assert hc.segment_count(78, 1, 64, 576, 1024, "layer_first", scattered, dp) == 78 * 512 \
        - 78 * int(np.sum((np.diff(scattered) == 1)))


def test_validation_before_any_cuda_call():
    """Bad descriptors are rejected on the host, before the library touches CUDA."""
    d = hc.PoolDesc(2, 2, 16, 2, 100, 128, 0, 0, 0, 0)      # 200-byte rows: not a 16-byte multiple
    h = ctypes.c_void_p()
    rc = hc.library().hicache_pool_create(ctypes.byref(d), 4096, 1 << 20, ctypes.byref(h))
    assert rc == -4
    d = hc.PoolDesc(2, 2, 16, 2, 128, 128, 5, 0, 0, 0)      # unknown layout
    assert hc.library().hicache_pool_create(ctypes.byref(d), 4096, 1 << 20, ctypes.byref(h)) == -1
    d = hc.PoolDesc(400, 2, 16, 2, 128, 128, 0, 0, 0, 0)    # B*L above 512
    assert hc.library().hicache_pool_create(ctypes.byref(d), 4096, 1 << 20, ctypes.byref(h)) == -1
    d = hc.PoolDesc(2, 2, 16, 2, 128, 128, 0, 0, 0, 0)      # host pool too small
    assert hc.library().hicache_pool_create(ctypes.byref(d), 4096, 1024, ctypes.byref(h)) == -1
    assert "below" in hc.library().hicache_last_error().decode()
    assert hc.library().hicache_pool_create(ctypes.byref(d), 4104, 1 << 20, ctypes.byref(h)) == -4


@pytest.mark.parametrize("shape", [(2, 3, 4, 8, 5), (1, 4, 2, 16, 3), (3, 1, 2, 8, 4), (1, 1, 3, 8, 4)])
def test_page_span_is_exactly_the_page(shape):
    """A page span holds every element of that host page (and buffer) and
    nothing else, by the oracle's element offsets."""
    import oracle
    o = oracle.Oracle()
    B, L, P, R, Hp = shape
    es = 2
    for name, lid in hc.LAYOUTS.items():
        d = hc._desc(L, B, P, R, Hp, lid, es)
        for h in range(Hp):
            for buf in [-1] + list(range(B)):
                bufs = range(B) if buf < 0 else [buf]
                offs = sorted(o.host_offset(lid, B, L, P, R, Hp, b, l, h, t, e) * es
                              for b in bufs for l in range(L) for t in range(P) for e in range(R))
                contiguous = offs == list(range(offs[0], offs[0] + es * len(offs), es))
                try:
                    off, nb = hc.page_span(d, h, buf)
                except hc.HiCacheError as err:
                    assert err.status == "INVALID_ARG"
                    # refused only where the page (buffer) is not one contiguous span, or
                    # where a single-buffer-only form was asked for several buffers
                    assert not contiguous or (buf < 0 and B > 1), (name, h, buf)
                    continue
                assert contiguous, (name, h, buf)
                assert (off, nb) == (offs[0], es * len(offs)), (name, h, buf)
    with pytest.raises(hc.HiCacheError) as e:
        hc.page_span(hc._desc(2, 2, 4, 8, 5, "page_first"), 5, 0)
    assert e.value.status == "INDEX_RANGE"


def test_group_calls_reject_bad_arguments_before_any_cuda_call():
    """A group call with no pools, too many, NULL arrays or a NULL pool is
    refused on the host; the Python group size matches the header's."""
    with open(os.path.join(ROOT, "include", "hicache.h")) as f:
        hdr = f.read()
    assert int(re.search(r"#define HICACHE_MAX_GROUP (\d+)", hdr).group(1)) == hc.MAX_GROUP
    lib = hc.library()
    kvs = (hc._DeviceKVStruct * 1)()
    none = (ctypes.c_void_p * 1)(None)
    for pools, structs, n in ((none, kvs, 0), (none, kvs, hc.MAX_GROUP + 1), (None, kvs, 1), (none, None, 1),
                              (none, kvs, 1)):
        c0 = hc.launch_count()
        assert lib.hicache_group_transfer(pools, structs, n, None, None, 0, -1, -1, 0, None) == -1
        assert lib.hicache_group_load_pipelined(pools, structs, n, None, None, 0, -1, None) == -1
        assert lib.hicache_last_error()
        assert hc.launch_count() == c0
    for pools, n in ((none, 0), (none, hc.MAX_GROUP + 1), (None, 1), (none, 1)):
        out = ctypes.c_void_p(1)
        assert lib.hicache_group_plan_create(pools, n, None, None, 0, 8, ctypes.byref(out)) == -1
        assert out.value is None and lib.hicache_last_error()
    for call in (lambda: lib.hicache_group_plan_execute(None, kvs, -1, -1, None),
                 lambda: lib.hicache_group_plan_load_layers(None, kvs, -1, None)):
        assert call() == -1
    assert lib.hicache_group_plan_destroy(None) == 0
    with pytest.raises(ValueError):
        hc.group_transfer([object()], [], [0], [0], hc.LOAD)
    with pytest.raises(ValueError):
        hc.group_load_pipelined([], [], [0, 1], [0])


@pytest.mark.parametrize("seed", range(4))
def test_prepass_large_sets(seed):
    """Sets large enough for the radix sort of the pairs and the bitmap
    duplicate check: the runs equal the plain sort-and-merge, and repeated
    destinations are found wherever they sit."""
    rng = np.random.default_rng(300 + seed)
    Dp, Hp, n = 50000, 70000, 6000
    if seed % 2:
        dp = rng.choice(Dp, n, replace=False)
        hp = rng.choice(Hp, n, replace=False)
    else:                                      # runs: both sides step by one in stretches
        starts = np.sort(rng.choice(Dp // 16, n // 16, replace=False)) * 16
        dp = np.concatenate([np.arange(s, s + 16) for s in starts])
        hp = np.arange(dp.size) + 3
        perm = rng.permutation(dp.size)        # the pairs arrive shuffled
        dp, hp = dp[perm], hp[perm]
        n = dp.size
    for direction in (hc.BACKUP, hc.LOAD):
        runs = hc.prepass(Hp, Dp, dp, hp, direction)
        assert np.array_equal(runs, py_runs(np.asarray(dp, np.int64), np.asarray(hp, np.int64)))
        assert runs[:, 2].sum() == n
    # a repeated destination, at the end, in the middle, at the start
    for pos in (n - 1, n // 2, 1):
        bad = np.array(dp, np.int64).copy()
        bad[pos] = bad[pos - 1]
        with pytest.raises(hc.HiCacheError) as e:
            hc.prepass(Hp, Dp, bad, hp, hc.LOAD)
        assert e.value.status == "DUPLICATE_INDEX"
        assert str(bad[pos]) in str(e.value)
        badh = np.array(hp, np.int64).copy()
        badh[pos] = badh[pos - 1]
        with pytest.raises(hc.HiCacheError) as e:
            hc.prepass(Hp, Dp, dp, badh, hc.BACKUP)
        assert e.value.status == "DUPLICATE_INDEX"
    # a failed check leaves nothing behind: the same valid set passes right after
    assert hc.prepass(Hp, Dp, dp, hp, hc.LOAD)[:, 2].sum() == n


def test_prepass_duplicate_check_beyond_the_bitmap():
    """Device pools above 2^27 pages take the sorting duplicate check."""
    Dp = (1 << 28) + 5
    dp = np.array([5, 1 << 27, (1 << 28) + 4, 77] * 10 + [9], np.int64)   # 41 pages, repeats
    with pytest.raises(hc.HiCacheError) as e:
        hc.prepass(100, Dp, dp, np.arange(41), hc.LOAD)
    assert e.value.status == "DUPLICATE_INDEX"
    ok = np.array([(1 << 28) + 4 - k for k in range(41)], np.int64)
    runs = hc.prepass(100, Dp, ok, np.arange(41), hc.LOAD)
    assert np.array_equal(runs, py_runs(ok, np.arange(41, dtype=np.int64)))


def test_index_marshalling_fast_paths():
    """1-D contiguous int64 arrays pass through unchanged; anything else is
    converted; pointers come from the buffer protocol or, for a read-only
    array, from ndarray.ctypes, and are the array's own data address."""
    a = np.arange(5, dtype=np.int64)
    assert hc._idx(a) is a
    for other in ([1, 2, 3], np.arange(4, dtype=np.int32), np.arange(6, dtype=np.int64).reshape(2, 3),
                  np.arange(10, dtype=np.int64)[::2]):
        out = hc._idx(other)
        assert out.dtype == np.int64 and out.ndim == 1 and out.flags.c_contiguous
        assert np.array_equal(out, np.asarray(other).reshape(-1))
    assert hc._ptr(a) == a.ctypes.data
    ro = np.arange(3, dtype=np.int64)
    ro.flags.writeable = False
    assert hc._ptr(ro) == ro.ctypes.data
    assert hc._ptr(a[:0]) is None


def test_large_sorted_calls_are_refused_whole():
    """A large call whose pairs come in host order is validated in full before
    any run is built (so before any launch): a bad index or a repeated
    destination at its very end is refused, and the same pairs minus the bad
    one reduce to the runs of a plain merge."""
    n = 50_000
    rng = np.random.default_rng(1700)
    dp = rng.permutation(n).astype(np.int64)
    hp = np.arange(n, dtype=np.int64)
    runs = hc.prepass(n, n, dp, hp, hc.LOAD)
    assert len(runs) == n - int(np.count_nonzero(np.diff(dp) == 1))
    assert runs[:, 2].sum() == n
    for fix, status in [(lambda d, h: d.__setitem__(-1, n), "INDEX_RANGE"),
                        (lambda d, h: d.__setitem__(-1, -1), "INDEX_RANGE"),
                        (lambda d, h: h.__setitem__(-1, n), "INDEX_RANGE"),
                        (lambda d, h: d.__setitem__(-1, d[0]), "DUPLICATE_INDEX")]:
        d, h = dp.copy(), hp.copy()
        fix(d, h)
        with pytest.raises(hc.HiCacheError) as e:
            hc.prepass(n, n, d, h, hc.LOAD)
        assert e.value.status == status
    # a backup naming the last host page twice
    h = hp.copy()
    h[-1] = h[-2]
    with pytest.raises(hc.HiCacheError) as e:
        hc.prepass(n, n, dp, h, hc.BACKUP)
    assert e.value.status == "DUPLICATE_INDEX"
