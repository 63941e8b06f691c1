"""CPU oracle for the L1 <-> L2 KV page movement (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (``tiered_kv_cache_gb300``)
never does; the two share no code.

The oracle itself is plain C (``hicache_oracle.c``), single-threaded, one element
at a time; this module compiles it with gcc and wraps it with ctypes over numpy
arrays.  See the header of ``hicache_oracle.c`` for the definition it follows
and the page/section each part comes from.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

LAYER_FIRST = 0
PAGE_FIRST = 1
PAGE_FIRST_DIRECT = 2
PAGE_FIRST_DIRECT_KV = 3
LAYOUTS = {"layer_first": LAYER_FIRST, "page_first": PAGE_FIRST,
           "page_first_direct": PAGE_FIRST_DIRECT, "page_first_direct_kv": PAGE_FIRST_DIRECT_KV}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hicache_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle into a shared library with gcc (plain -O2, no tuning)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c99", "-Wall", "-Wextra", "-shared",
                           "-fPIC", src, "-o", tmp])
    os.replace(tmp, out)
    return out


_i64 = ctypes.c_int64
_i32 = ctypes.c_int32
_vp = ctypes.c_void_p


def _bind(lib):
    lib.oracle_host_elem_offset.restype = _i64
    lib.oracle_host_elem_offset.argtypes = [_i32] + [_i64] * 10
    lib.oracle_dev_elem_offset.restype = _i64
    lib.oracle_dev_elem_offset.argtypes = [_i64] * 5
    lib.oracle_backup.restype = ctypes.c_int
    lib.oracle_backup.argtypes = [_vp, _vp] + [_i64] * 6 + [_vp, _vp, _i64, _i32]
    lib.oracle_load.restype = ctypes.c_int
    lib.oracle_load.argtypes = [_vp, _vp] + [_i64] * 6 + [_vp, _vp, _i64, _i32, _i32]
    lib.oracle_segment_count.restype = _i64
    lib.oracle_segment_count.argtypes = [_i64] * 5 + [_vp, _vp, _i64, _i32, _i32]
    return lib


def load_library(path: str | None = None):
    """Load (building first if needed) the oracle library; ``path`` loads a
    specific build, e.g. a deliberately broken copy in a test."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _ptr_array(bufs):
    arr = (ctypes.c_void_p * len(bufs))(*[b.ctypes.data for b in bufs])
    return arr


def _idx(a):
    a = np.ascontiguousarray(np.asarray(a, dtype=np.int64))
    return a


class Oracle:
    """Numpy-facing wrapper.  Device buffers are given as a list of B*L numpy
    arrays (buffer-major: K layers 0..L-1, then V layers), each a contiguous
    ``(Dp*P, R)`` array; the host pool is one flat numpy array."""

    def __init__(self, lib=None):
        self.lib = lib if lib is not None else load_library()

    def host_offset(self, layout, B, L, P, R, Hp, b, l, h, t, e):
        return self.lib.oracle_host_elem_offset(layout, B, L, P, R, Hp, b, l, h, t, e)

    def dev_offset(self, P, R, d, t, e):
        return self.lib.oracle_dev_elem_offset(P, R, d, t, e)

    def backup(self, dev_bufs, host, B, L, P, R, Hp, dev_pages, host_pages, layout):
        es = host.dtype.itemsize
        dp, hp = _idx(dev_pages), _idx(host_pages)
        assert len(dev_bufs) == B * L and all(x.flags.c_contiguous for x in dev_bufs)
        assert host.flags.c_contiguous and dp.shape == hp.shape
        bufs = _ptr_array(dev_bufs)
        rc = self.lib.oracle_backup(bufs, host.ctypes.data, B, L, P, R, Hp, es,
                                    dp.ctypes.data, hp.ctypes.data, dp.size, layout)
        if rc != 0:
            raise ValueError("oracle_backup rejected its arguments")

    def load(self, dev_bufs, host, B, L, P, R, Hp, dev_pages, host_pages, layout, layer=-1):
        es = host.dtype.itemsize
        dp, hp = _idx(dev_pages), _idx(host_pages)
        assert len(dev_bufs) == B * L and all(x.flags.c_contiguous for x in dev_bufs)
        assert host.flags.c_contiguous and dp.shape == hp.shape
        bufs = _ptr_array(dev_bufs)
        rc = self.lib.oracle_load(bufs, host.ctypes.data, B, L, P, R, Hp, es,
                                  dp.ctypes.data, hp.ctypes.data, dp.size, layout, layer)
        if rc != 0:
            raise ValueError("oracle_load rejected its arguments")

    def segment_count(self, B, L, P, R, Hp, dev_pages, host_pages, layout, layer=-1):
        dp, hp = _idx(dev_pages), _idx(host_pages)
        return self.lib.oracle_segment_count(B, L, P, R, Hp, dp.ctypes.data, hp.ctypes.data,
                                             dp.size, layout, layer)
