"""The C ABI from a plain C program (no Python in the call path)."""
import os
import subprocess

import pytest

from tiered_kv_cache_gb300 import build as hc_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "abi_roundtrip.c")


def compile_c(out_dir):
    lib = hc_build.build()
    cuda = "/usr/local/cuda"
    exe = os.path.join(str(out_dir), "abi_roundtrip")
    libdir = os.path.dirname(lib)
    cmd = ["gcc", "-O1", "-std=c99", "-Wall", f"-I{os.path.join(ROOT, 'include')}", f"-I{cuda}/include",
           SRC, "-o", exe, f"-L{libdir}", "-lhicache", f"-L{cuda}/lib64", "-lcudart",
           f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{cuda}/lib64"]
    subprocess.check_call(cmd)
    return exe


def test_c_program_compiles_and_links(tmp_path):
    assert os.path.exists(compile_c(tmp_path))


@pytest.mark.gpu
def test_c_program_round_trip(tmp_path):
    exe = compile_c(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip() == "ok"
