"""Each plausible mistake planted in a copy of the oracle fails at least one pin.

The mistakes are planted by text substitution in a temporary copy of the oracle's
C source (never in the oracle itself), built with gcc, and the pins run against
that build in a child process (a mistake that writes out of bounds may crash it;
a crash counts as caught).
"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "hicache_oracle.c")

# (name, original text, mistaken text): one substitution each
MUTANTS = [
    ("lf_dropped_buffer_term", "(((b * L + l) * S) + h * P + t) * R + e", "(((l) * S) + h * P + t) * R + e"),
    ("pf_token_layer_swapped", "(((b * S) + h * P + t) * L + l) * R + e", "(((b * S) + h * P + l) * L + t) * R + e"),
    ("pf_buffer_stride_pages", "(((b * S) + h * P + t) * L + l) * R + e", "(((b * Hp) + h * P + t) * L + l) * R + e"),
    ("pfd_page_layer_swapped", "((((b * Hp + h) * L + l) * P) + t) * R + e", "((((b * L + l) * Hp + h) * P) + t) * R + e"),
    ("pfd_kv_buffer_outside_page", "((((h * B + b) * L + l) * P) + t) * R + e", "((((b * Hp + h) * L + l) * P) + t) * R + e"),
    ("pfd_kv_layer_buffer_swapped", "((((h * B + b) * L + l) * P) + t) * R + e", "((((h * L + l) * B + b) * P) + t) * R + e"),
    ("size_without_page_size", "const int64_t S = Hp * P;", "const int64_t S = Hp;"),
    ("dev_slot_transposed", "return (d * P + t) * R + e;", "return (t * P + d) * R + e;"),
    ("backup_buffer_index", "const uint8_t *src = (const uint8_t *)dev_bufs[b * L + l];",
     "const uint8_t *src = (const uint8_t *)dev_bufs[l * B + b];"),
    ("load_layer_range", "if (layer >= 0) { l_begin = layer; l_end = layer + 1; }\n  for (i = 0; i < n; ++i)\n    if (host_pages[i] < 0 || host_pages[i] >= Hp || dev_pages[i] < 0) return -1;\n  for (i = 0; i < n; ++i) {\n    const int64_t d = dev_pages[i], h = host_pages[i];\n    for (b = 0; b < B; ++b)\n      for (l = l_begin; l < l_end; ++l) {\n        uint8_t",
     "if (layer >= 0) { l_begin = 0; l_end = layer + 1; }\n  for (i = 0; i < n; ++i)\n    if (host_pages[i] < 0 || host_pages[i] >= Hp || dev_pages[i] < 0) return -1;\n  for (i = 0; i < n; ++i) {\n    const int64_t d = dev_pages[i], h = host_pages[i];\n    for (b = 0; b < B; ++b)\n      for (l = l_begin; l < l_end; ++l) {\n        uint8_t"),
    ("segment_host_step", "host == prev_host + R", "host == prev_host + 1"),
    ("segment_slot_step", "slot == prev_slot + 1", "slot == prev_slot + P"),
    ("segment_unsorted", "qsort(order, (size_t)n, sizeof(int64_t), cmp_by_host_then_dev);", ""),
    ("load_reads_wrong_pair", "const int64_t d = dev_pages[i], h = host_pages[i];\n    for (b = 0; b < B; ++b)\n      for (l = l_begin",
     "const int64_t d = dev_pages[i], h = host_pages[n - 1 - i];\n    for (b = 0; b < B; ++b)\n      for (l = l_begin"),
]


@pytest.mark.parametrize("name,orig,bad", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, orig, bad):
    with open(SRC, encoding="utf-8") as f:
        src = f.read()
    assert src.count(orig) == 1, f"mutant {name} no longer matches the oracle source"
    mutated = src.replace(orig, bad)
    csrc = tmp_path / "mutant.c"
    csrc.write_text(mutated, encoding="utf-8")
    lib = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O1", "-std=c99", "-shared", "-fPIC", str(csrc), "-o", str(lib)],
                          stderr=subprocess.DEVNULL)
    code = ("import json, sys; sys.path[:0] = [%r, %r]; import oracle_pins; "
            "print(json.dumps(oracle_pins.run_all(%r)))") % (ROOT, os.path.join(ROOT, "tests"), str(lib))
    proc = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    if proc.returncode != 0:
        return  # crashed (e.g. an out-of-bounds write): caught
    failed = json.loads(proc.stdout.strip().splitlines()[-1])
    assert failed, f"no pin catches mutant {name}"
