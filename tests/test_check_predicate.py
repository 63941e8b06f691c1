"""The bounds-checked build's predicate (check_vector in hicache_internal.h),
compiled for the host with g++ and tried at and around every edge: inside
every extent it passes, one past or one before any extent it names that
extent's check, and the buffer check comes before the device check before the
host check."""
import os
import subprocess

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "tiered_kv_cache_gb300", "csrc")
HARNESS = r'''
#include <cstdio>
#include <cstdint>
#include "hicache_internal.h"
int main() {
  long long v[][6] = {
#include "cases.inc"
  };
  for (auto &c : v)
    std::printf("%d\n", hicache::check_vector(c[0], c[1], c[2], c[3], c[4], c[5]));
  return 0;
}
'''


def expected(bi, nb, doff, dv, hoff, hv):
    if not 0 <= bi < nb:
        return 1
    if not 0 <= doff < dv:
        return 2
    if not 0 <= hoff < hv:
        return 3
    return 0


def test_check_vector_at_every_edge(tmp_path):
    nb, dv, hv = 64, 1 << 31, (1 << 36) + 5
    cases = []
    for bi in (-1, 0, 1, nb - 1, nb, nb + 7):
        for doff in (-1, 0, dv - 1, dv, 1 << 40):
            for hoff in (-(1 << 33), -1, 0, hv - 1, hv):
                cases.append((bi, nb, doff, dv, hoff, hv))
    (tmp_path / "cases.inc").write_text(",\n".join("{%dLL,%dLL,%dLL,%dLL,%dLL,%dLL}" % c for c in cases))
    (tmp_path / "t.cpp").write_text(HARNESS)
    exe = tmp_path / "t"
    subprocess.check_call(["g++", "-std=c++17", "-O1", f"-I{CSRC}", f"-I{tmp_path}", str(tmp_path / "t.cpp"),
                           "-o", str(exe)])
    got = [int(x) for x in subprocess.check_output([str(exe)], text=True).split()]
    assert got == [expected(*c) for c in cases]
    assert 0 < got.count(0) < len(got) and {1, 2, 3} <= set(got)


def test_plain_library_is_not_the_checked_build(monkeypatch):
    import tiered_kv_cache_gb300 as hc
    assert hc.library_path().endswith("libhicache.so")
    assert not hc.checked_build()
    monkeypatch.setenv("HICACHE_CHECKED", "1")
    assert hc.library_path().endswith("libhicache_checked.so")
