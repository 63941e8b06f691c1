"""Build libhicache.so in-tree with nvcc for sm_103a (GB300).

Nine translation units, compiled in parallel, linked with the static CUDA
runtime so the library loads on a machine without a GPU driver (and the
kernel file a second time with HICACHE_CHECKED=1 for libhicache_checked.so,
the bounds-checked build):
  csrc/hicache_kernels.cu    transfer and stand-in compute kernels
  csrc/hicache_api.cpp       errors, pinned memory, pools, transfers, events
  csrc/hicache_index.cpp     validation and the index pre-pass (host only)
  csrc/hicache_pipeline.cpp  pipelined loads and per-layer waits
  csrc/hicache_plan.cpp      plans (pre-passed index sets, graph replay)
  csrc/hicache_group.cpp     buffer groups
  csrc/hicache_alloc.cpp     LIFO host-page allocator
  csrc/hicache_engine.cpp    submission engine (queue + worker thread)
  csrc/hicache_tp.cpp        tensor-parallel load of a replicated latent
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libhicache.so")
LIB_CHECKED = os.path.join(HERE, "libhicache_checked.so")   # bounds-checked kernels
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
          f"-I{INCLUDE}", f"-I{CSRC}"]
SOURCES = ["hicache_kernels.cu", "hicache_api.cpp", "hicache_index.cpp", "hicache_pipeline.cpp",
           "hicache_plan.cpp", "hicache_group.cpp", "hicache_alloc.cpp", "hicache_engine.cpp",
           "hicache_tp.cpp"]


def _nvcc() -> str:
    for cand in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        p = os.path.join(cand, "bin", "nvcc") if cand else ""
        if p and os.path.exists(p):
            return p
    p = shutil.which("nvcc")
    if not p:
        raise RuntimeError("nvcc not found (CUDA toolkit required to build libhicache)")
    return p


def _stale(out: str, deps: list[str]) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None,
          checked: bool = True) -> str:
    """Compile and link; returns the path of libhicache.so.  Rebuilds only what
    changed unless ``force``.  With ``checked`` the bounds-checked library
    (libhicache_checked.so: the kernels compiled with HICACHE_CHECKED=1, the
    host objects shared) is built alongside, its kernel file compiled in the
    same parallel batch."""
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".h")]
    headers.append(os.path.join(INCLUDE, "hicache.h"))
    flags = COMMON + (extra_flags or [])
    objs, procs = [], []

    def compile_one(src, o, extra):
        if force or _stale(o, [os.path.join(CSRC, src), __file__] + headers):
            cmd = [nvcc] + ARCH + flags + extra + ["-c", os.path.join(CSRC, src), "-o", o]
            if src.endswith(".cu") and verbose:
                cmd += ["-Xptxas", "-v"]
            procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT,
                                                text=True)))
    for src in SOURCES:
        o = os.path.join(BUILD, src + ".o")
        objs.append(o)
        compile_one(src, o, [])
    checked_obj = os.path.join(BUILD, "hicache_kernels_checked.cu.o")
    if checked:
        compile_one("hicache_kernels.cu", checked_obj, ["-DHICACHE_CHECKED=1"])
    failed = []
    for cmd, p in procs:
        out, _ = p.communicate()
        if verbose and out:
            sys.stdout.write(out)
        if p.returncode != 0:
            failed.append((cmd, out))
    if failed:
        msg = "\n".join(" ".join(c) + "\n" + o for c, o in failed)
        raise RuntimeError("libhicache build failed:\n" + msg)
    _link(nvcc, LIB, objs, force or bool(procs))
    if checked:
        _link(nvcc, LIB_CHECKED, [checked_obj if o.endswith("hicache_kernels.cu.o") else o for o in objs],
              force or bool(procs))
    return LIB


def _link(nvcc, lib, objs, force):
    if force or _stale(lib, objs):
        tmp = lib + f".tmp{os.getpid()}"
        # nodelete: dlclose() leaves the library mapped, since the worker threads
        # of its host-side validation live until the process exits
        cmd = ([nvcc] + ARCH + ["-shared", "-cudart", "static", "-Xlinker", "-z,nodelete", "-o", tmp] + objs
               + ["-lpthread", "-ldl", "-lrt"])
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("libhicache link failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
        os.replace(tmp, lib)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
