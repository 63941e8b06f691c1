"""tiered_kv_cache_gb300: L1 (GPU HBM) <-> L2 (pinned host DRAM) paged KV movement
for GB300, as a thin ctypes binding over ``libhicache.so``.

The binding only marshals arguments: every step of a transfer (validation,
pre-pass, kernels) runs in the C/CUDA library.  There is no fallback: if the
library is not built, importing works but every call raises.

Names follow the C ABI in ``include/hicache.h``:
    Pool.backup / Pool.load / Pool.load_layer / Pool.load_pipelined / Pool.backup_load
    Pool.wait_layer / Pool.layer_event
    Pool.plan(...) -> Plan.execute / load_layer / load_layer_chained / load_layers / load_pipelined
    group_transfer / group_load_pipelined / group_plan(...) -> GroupPlan
    Engine (submission engine), PageAllocator (host pages)
    host_alloc / host_free, wait, prepass, segment_count, page_span, layer_checksum
    tp_share / tp_load_pipelined / Pool.layer_counters (tensor-parallel load of a replicated latent)
    stream_copy (roofline probe: plain zero-copy streaming copy)
    checked_build / check_status (the bounds-checked build, HICACHE_CHECKED=1)
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

__all__ = [
    "HiCacheError", "LAYER_FIRST", "PAGE_FIRST", "PAGE_FIRST_DIRECT", "LAYOUT_POOL", "LAYOUTS",
    "BACKUP", "LOAD", "library", "library_path", "PoolDesc", "DeviceKV", "Pool", "Plan", "PinnedHost",
    "PageAllocator", "Engine", "group_transfer", "group_load_pipelined", "group_plan", "GroupPlan",
    "MAX_GROUP", "PAGE_FIRST_DIRECT_KV",
    "host_alloc", "host_free", "wait", "prepass", "segment_count", "layer_checksum", "page_span",
    "launch_count", "version", "stream_copy", "tp_share", "tp_load_pipelined", "checked_build",
    "check_status",
]

LAYOUT_POOL = -1
LAYER_FIRST = 0
PAGE_FIRST = 1
PAGE_FIRST_DIRECT = 2
PAGE_FIRST_DIRECT_KV = 3
LAYOUTS = {"layer_first": LAYER_FIRST, "page_first": PAGE_FIRST,
           "page_first_direct": PAGE_FIRST_DIRECT, "page_first_direct_kv": PAGE_FIRST_DIRECT_KV}
BACKUP = 0
LOAD = 1
HOST_THP = 0x1

STATUS = {0: "OK", -1: "INVALID_ARG", -2: "INDEX_RANGE", -3: "DUPLICATE_INDEX", -4: "ALIGNMENT",
          -5: "NOT_PINNED", -6: "CUDA", -7: "TIMEOUT", -8: "NOMEM"}

_HERE = os.path.dirname(os.path.abspath(__file__))


def library_path() -> str:
    """libhicache.so, or the bounds-checked build libhicache_checked.so when
    the environment sets HICACHE_CHECKED=1 before the library is first loaded."""
    if os.environ.get("HICACHE_CHECKED") == "1":
        return os.path.join(_HERE, "libhicache_checked.so")
    return os.path.join(_HERE, "libhicache.so")


class HiCacheError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"{STATUS.get(code, code)}: {message}")
        self.code = code
        self.status = STATUS.get(code, str(code))


class PoolDesc(ctypes.Structure):
    _fields_ = [("num_layers", ctypes.c_int32), ("num_buffers", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("elem_bytes", ctypes.c_int32),
                ("row_elems", ctypes.c_int64), ("host_num_pages", ctypes.c_int64),
                ("layout", ctypes.c_int32), ("launch_ctas", ctypes.c_int32),
                ("flags", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class _DeviceKVStruct(ctypes.Structure):
    _fields_ = [("buf_ptrs", ctypes.POINTER(ctypes.c_void_p)), ("device_num_pages", ctypes.c_int64)]


_lib = None
_lib_lock = threading.Lock()
_vp, _i32, _i64, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
_P = ctypes.POINTER


def _bind(lib):
    sigs = {
        "hicache_version": (_i32, []),
        "hicache_last_error": (ctypes.c_char_p, []),
        "hicache_launch_count": (_i64, []),
        "hicache_host_alloc": (ctypes.c_int, [_sz, _i32, _P(_vp)]),
        "hicache_host_free": (ctypes.c_int, [_vp]),
        "hicache_pool_create": (ctypes.c_int, [_P(PoolDesc), _vp, _sz, _P(_vp)]),
        "hicache_pool_destroy": (ctypes.c_int, [_vp]),
        "hicache_backup": (ctypes.c_int, [_vp, _P(_DeviceKVStruct), _vp, _vp, _i64, _i32, _vp]),
        "hicache_load": (ctypes.c_int, [_vp, _P(_DeviceKVStruct), _vp, _vp, _i64, _i32, _vp]),
        "hicache_load_layer": (ctypes.c_int, [_vp, _P(_DeviceKVStruct), _vp, _vp, _i64, _i32, _i32, _vp]),
        "hicache_backup_load": (ctypes.c_int, [_vp, _P(_DeviceKVStruct), _vp, _vp, _i64, _vp, _vp, _i64,
                                               _i32, _vp]),
        "hicache_load_pipelined": (ctypes.c_int, [_vp, _P(_DeviceKVStruct), _vp, _vp, _i64, _i32, _vp]),
        "hicache_plan_load_pipelined": (ctypes.c_int, [_vp, _P(_DeviceKVStruct), _i32, _vp]),
        "hicache_load_pipelined_noalloc": (ctypes.c_int, [_vp, _P(_DeviceKVStruct), _vp, _vp, _i64, _i32, _vp]),
        "hicache_pipeline_status": (ctypes.c_int, [_vp, _i32, _P(ctypes.c_uint32), _P(ctypes.c_uint32)]),
        "hicache_group_transfer": (ctypes.c_int, [_P(_vp), _P(_DeviceKVStruct), _i32, _vp, _vp, _i64, _i32,
                                                  _i32, _i32, _vp]),
        "hicache_group_load_pipelined": (ctypes.c_int, [_P(_vp), _P(_DeviceKVStruct), _i32, _vp, _vp, _i64,
                                                        _i32, _vp]),
        "hicache_group_plan_create": (ctypes.c_int, [_P(_vp), _i32, _vp, _vp, _i64, _i64, _P(_vp)]),
        "hicache_group_plan_execute": (ctypes.c_int, [_vp, _P(_DeviceKVStruct), _i32, _i32, _vp]),
        "hicache_group_plan_load_layers": (ctypes.c_int, [_vp, _P(_DeviceKVStruct), _i32, _vp]),
        "hicache_group_plan_load_layer_chained": (ctypes.c_int, [_vp, _P(_DeviceKVStruct), _i32, _i32, _vp]),
        "hicache_group_plan_destroy": (ctypes.c_int, [_vp]),
        "hicache_plan_create": (ctypes.c_int, [_vp, _vp, _vp, _i64, _i64, _i32, _P(_vp)]),
        "hicache_plan_execute": (ctypes.c_int, [_vp, _P(_DeviceKVStruct), _i32, _i32, _vp]),
        "hicache_plan_load_layer": (ctypes.c_int, [_vp, _P(_DeviceKVStruct), _i32, _i32, _vp]),
        "hicache_plan_load_layers": (ctypes.c_int, [_vp, _P(_DeviceKVStruct), _i32, _vp]),
        "hicache_plan_load_layer_chained": (ctypes.c_int, [_vp, _P(_DeviceKVStruct), _i32, _i32, _vp]),
        "hicache_plan_info": (ctypes.c_int, [_vp, _P(_i64), _P(_i64)]),
        "hicache_plan_destroy": (ctypes.c_int, [_vp]),
        "hicache_layer_event": (ctypes.c_int, [_vp, _i32, _P(_vp)]),
        "hicache_wait_layer": (ctypes.c_int, [_vp, _i32, _vp]),
        "hicache_wait": (ctypes.c_int, [_vp, _i64]),
        "hicache_stream_copy": (ctypes.c_int, [_vp, _vp, _sz, _i32, _i32, _vp]),
        "hicache_checked_build": (_i32, []),
        "hicache_check_status": (ctypes.c_int, [_P(ctypes.c_uint64), _P(ctypes.c_uint64), _i32]),
        "hicache_tp_share": (ctypes.c_int, [_i64, _i32, _i32, _P(_i64), _P(_i64)]),
        "hicache_pool_layer_counters": (ctypes.c_int, [_vp, _P(_vp)]),
        "hicache_tp_load_pipelined": (ctypes.c_int, [_vp, _P(_DeviceKVStruct), _P(_vp), _i32, _i32, _vp, _vp,
                                                     _i64, _i32, _vp]),
        "hicache_prepass": (ctypes.c_int, [_i64, _i64, _vp, _vp, _i64, _i32, _P(_i64), _vp, _i64]),
        "hicache_segment_count": (_i64, [_P(PoolDesc), _vp, _vp, _i64, _i32, _i32]),
        "hicache_page_span": (ctypes.c_int, [_P(PoolDesc), _i64, _i32, _P(_i64), _P(_i64)]),
        "hicache_engine_create": (ctypes.c_int, [_vp, _P(_vp)]),
        "hicache_engine_destroy": (ctypes.c_int, [_vp]),
        "hicache_engine_submit": (ctypes.c_int, [_vp, _P(_DeviceKVStruct), _vp, _vp, _i64, _i32, _i32, _i32,
                                                 _vp, _P(ctypes.c_uint64)]),
        "hicache_engine_wait": (ctypes.c_int, [_vp, ctypes.c_uint64, _i64]),
        "hicache_engine_wait_on_stream": (ctypes.c_int, [_vp, ctypes.c_uint64, _vp]),
        "hicache_engine_stats": (ctypes.c_int, [_vp, _P(_i64), _P(_i64)]),
        "hicache_allocator_create": (ctypes.c_int, [_i64, _P(_vp)]),
        "hicache_allocator_destroy": (ctypes.c_int, [_vp]),
        "hicache_allocator_alloc": (ctypes.c_int, [_vp, _i64, _vp]),
        "hicache_allocator_free": (ctypes.c_int, [_vp, _vp, _i64]),
        "hicache_allocator_available": (_i64, [_vp]),
        "hicache_layer_checksum": (ctypes.c_int, [_P(_DeviceKVStruct), _P(PoolDesc), _vp, _i64, _i32,
                                                  _i32, _vp, _vp]),
    }
    for name, (res, args) in sigs.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


def library():
    """The loaded libhicache (raises if it has not been built)."""
    global _lib
    if _lib is None:
        with _lib_lock:
            if _lib is None:
                path = library_path()
                if not os.path.exists(path):
                    raise RuntimeError(
                        f"{path} is missing: build it with tiered_kv_cache_gb300.build.build() "
                        "(there is no fallback path)")
                _lib = _bind(ctypes.CDLL(path))
    return _lib


def _check(rc: int):
    if rc != 0:
        msg = library().hicache_last_error().decode(errors="replace")
        raise HiCacheError(rc, msg)


def _stream(stream) -> int:
    """cudaStream_t handle from None (legacy default), an int, or a torch stream."""
    if stream is None:
        return 0
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def _idx(a) -> np.ndarray:
    if type(a) is np.ndarray and a.dtype == np.int64 and a.ndim == 1 and a.flags.c_contiguous:
        return a
    return np.ascontiguousarray(np.asarray(a, dtype=np.int64).reshape(-1))


def _ptr(a: np.ndarray):
    """Address of a contiguous array's data (None when empty).  Through the
    buffer protocol where the array is writable: a third of the cost of
    ndarray.ctypes, which a small call pays twice."""
    if not a.size:
        return None
    if a.flags.writeable:
        return ctypes.addressof(ctypes.c_char.from_buffer(a))
    return a.ctypes.data


def version() -> int:
    return library().hicache_version()


def launch_count() -> int:
    return library().hicache_launch_count()


def host_alloc(nbytes: int, thp: bool = False) -> int:
    """Page-locked, device-mapped host memory (HICACHE_HOST_THP: mmap + huge
    pages before locking).  Returns the host address."""
    out = ctypes.c_void_p()
    _check(library().hicache_host_alloc(nbytes, HOST_THP if thp else 0, ctypes.byref(out)))
    return out.value


def host_free(ptr: int):
    _check(library().hicache_host_free(ptr))


def wait(stream=None, timeout_us: int = -1):
    """Block until `stream` is idle, for at most timeout_us (raises TIMEOUT)."""
    _check(library().hicache_wait(_stream(stream), timeout_us))

def checked_build() -> bool:
    """True when the loaded library is the bounds-checked build."""
    return bool(library().hicache_checked_build())


def check_status(clear: bool = False):
    """(first failed bounds check, number of failed checks) of the current
    device since the last clear; (0, 0) when every check passed (and always in
    the plain build)."""
    first, count = ctypes.c_uint64(), ctypes.c_uint64()
    _check(library().hicache_check_status(ctypes.byref(first), ctypes.byref(count), int(clear)))
    return first.value, count.value


def tp_share(n: int, tp: int, rank: int):
    """(first, count): the pairs rank `rank` of a tensor-parallel group of tp
    loads out of n, a contiguous part in the caller's order."""
    first, count = ctypes.c_int64(), ctypes.c_int64()
    _check(library().hicache_tp_share(n, tp, rank, ctypes.byref(first), ctypes.byref(count)))
    return first.value, count.value


def tp_load_pipelined(pool, rank_kvs, rank_counters, rank: int, device_pages, host_pages,
                      layout=LAYOUT_POOL, stream=None):
    """This rank's part of a tensor-parallel load of a replicated latent: its
    share of the pages, read from ``pool``'s host memory and stored into every
    rank's buffers (``rank_kvs``), counted into every rank's per-layer
    counters (``rank_counters``: each rank's Pool.layer_counters())."""
    if len(rank_kvs) != len(rank_counters):
        raise ValueError("rank_kvs and rank_counters differ in length")
    dp, hp = _idx(device_pages), _idx(host_pages)
    if dp.size != hp.size:
        raise ValueError("device_pages and host_pages differ in length")
    if isinstance(layout, str):
        layout = LAYOUTS[layout]
    structs = (_DeviceKVStruct * len(rank_kvs))(*[k.struct for k in rank_kvs])
    counters = (ctypes.c_void_p * len(rank_counters))(*rank_counters)
    _check(library().hicache_tp_load_pipelined(pool.handle, structs, counters, len(rank_kvs), rank, _ptr(dp),
                                               _ptr(hp), dp.size, layout, _stream(stream)))


def stream_copy(dst_ptr: int, src_ptr: int, nbytes: int, grid: int = 0, vecs_per_thread: int = 4,
                stream=None):
    """Roofline probe: a plain zero-copy streaming copy of nbytes (no index
    decode) between device memory and/or pinned, mapped host memory."""
    _check(library().hicache_stream_copy(dst_ptr, src_ptr, nbytes, grid, vecs_per_thread, _stream(stream)))


class DeviceKV:
    """B*L device buffer pointers (buffer-major) plus the device pool size in
    pages.  ``tensors`` may be torch tensors (their data_ptr is taken) or raw
    integer addresses; the caller keeps the memory alive."""

    def __init__(self, tensors, device_num_pages: int):
        ptrs = [t if isinstance(t, int) else t.data_ptr() for t in tensors]
        self._arr = (ctypes.c_void_p * len(ptrs))(*ptrs)
        self._tensors = tensors
        self.struct = _DeviceKVStruct(ctypes.cast(self._arr, ctypes.POINTER(ctypes.c_void_p)),
                                      device_num_pages)
        self.ref = ctypes.byref(self.struct)      # made once: every call passes it
        self.device_num_pages = device_num_pages
        self.num_buffers_total = len(ptrs)


def _desc(num_layers, num_buffers, page_size, row_elems, host_num_pages, layout,
          elem_bytes=2, launch_ctas=0) -> PoolDesc:
    if isinstance(layout, str):
        layout = LAYOUTS[layout]
    return PoolDesc(num_layers, num_buffers, page_size, elem_bytes, row_elems, host_num_pages,
                    layout, launch_ctas, 0, 0)


def prepass(host_num_pages: int, device_num_pages: int, device_pages, host_pages, direction: int):
    """Validate a transfer and return its runs as an (r, 3) int64 array of
    (first host page, first device page, page count)."""
    dp, hp = _idx(device_pages), _idx(host_pages)
    if dp.size != hp.size:
        raise ValueError("device_pages and host_pages differ in length")
    nr = ctypes.c_int64()
    out = np.zeros((max(1, dp.size), 3), np.int64)
    _check(library().hicache_prepass(host_num_pages, device_num_pages, _ptr(dp), _ptr(hp), dp.size,
                                     direction, ctypes.byref(nr), out.ctypes.data, out.shape[0]))
    return out[: nr.value].copy()


def segment_count(num_layers, num_buffers, page_size, row_elems, host_num_pages, layout,
                  device_pages, host_pages, layer: int = -1, elem_bytes: int = 2) -> int:
    d = _desc(num_layers, num_buffers, page_size, row_elems, host_num_pages, layout, elem_bytes)
    dp, hp = _idx(device_pages), _idx(host_pages)
    r = library().hicache_segment_count(ctypes.byref(d), _ptr(dp), _ptr(hp), dp.size, d.layout, layer)
    if r < 0:
        _check(int(r))
    return int(r)


def page_span(desc: PoolDesc, host_page: int, buffer: int = -1):
    """(offset, nbytes) of one host page's contiguous span in the host pool."""
    off, nb = ctypes.c_int64(), ctypes.c_int64()
    _check(library().hicache_page_span(ctypes.byref(desc), host_page, buffer, ctypes.byref(off),
                                       ctypes.byref(nb)))
    return off.value, nb.value


def layer_checksum(kv: DeviceKV, pool_or_desc, device_pages, layer: int, out_ptr: int,
                   reps: int = 1, stream=None):
    """Stand-in attention: adds the 32-bit words of `layer` of the given device
    pages (every buffer, `reps` passes) into the device uint64 at out_ptr."""
    desc = pool_or_desc.desc if isinstance(pool_or_desc, Pool) else pool_or_desc
    dp = _idx(device_pages)
    _check(library().hicache_layer_checksum(kv.ref, ctypes.byref(desc), _ptr(dp),
                                            dp.size, layer, reps, out_ptr, _stream(stream)))


MAX_GROUP = 4


def group_transfer(pools, kvs, device_pages, host_pages, direction: int, layer: int = -1,
                   layout=LAYOUT_POOL, stream=None):
    """Move the same page pairs for several pools (buffer kinds with different
    rows that share the page numbering) in one launch.  ``layer`` >= 0 loads
    that layer alone and records its event in every pool."""
    if len(pools) != len(kvs):
        raise ValueError("pools and kvs differ in length")
    dp, hp = _idx(device_pages), _idx(host_pages)
    if dp.size != hp.size:
        raise ValueError("device_pages and host_pages differ in length")
    if isinstance(layout, str):
        layout = LAYOUTS[layout]
    handles = (ctypes.c_void_p * len(pools))(*[p.handle for p in pools])
    structs = (_DeviceKVStruct * len(kvs))(*[k.struct for k in kvs])
    _check(library().hicache_group_transfer(handles, structs, len(pools), _ptr(dp), _ptr(hp), dp.size,
                                            layout, layer, direction, _stream(stream)))


def group_load_pipelined(pools, kvs, device_pages, host_pages, layout=LAYOUT_POOL, stream=None):
    """Every layer of every pool of a group in one launch, layer by layer;
    each pool's wait_layer then waits for that pool's layer alone."""
    if len(pools) != len(kvs):
        raise ValueError("pools and kvs differ in length")
    dp, hp = _idx(device_pages), _idx(host_pages)
    if dp.size != hp.size:
        raise ValueError("device_pages and host_pages differ in length")
    if isinstance(layout, str):
        layout = LAYOUTS[layout]
    handles = (ctypes.c_void_p * len(pools))(*[p.handle for p in pools])
    structs = (_DeviceKVStruct * len(kvs))(*[k.struct for k in kvs])
    _check(library().hicache_group_load_pipelined(handles, structs, len(pools), _ptr(dp), _ptr(hp), dp.size,
                                                  layout, _stream(stream)))


class GroupPlan:
    """A load plan for a buffer group: the page pairs pre-passed once for
    pools that share the page numbering, then loaded every layer at once, one
    layer, or layer by layer from a CUDA graph."""

    def __init__(self, pools, device_pages, host_pages, device_num_pages: int):
        dp, hp = _idx(device_pages), _idx(host_pages)
        if dp.size != hp.size:
            raise ValueError("device_pages and host_pages differ in length")
        handles = (ctypes.c_void_p * len(pools))(*[p.handle for p in pools])
        h = ctypes.c_void_p()
        _check(library().hicache_group_plan_create(handles, len(pools), _ptr(dp), _ptr(hp), dp.size,
                                                   device_num_pages, ctypes.byref(h)))
        self.pools = list(pools)
        self.handle = h.value

    def _kvs(self, kvs):
        if len(kvs) != len(self.pools):
            raise ValueError("one DeviceKV per pool of the plan")
        return (_DeviceKVStruct * len(kvs))(*[k.struct for k in kvs])

    def execute(self, kvs, layer: int = -1, layout=LAYOUT_POOL, stream=None):
        if isinstance(layout, str):
            layout = LAYOUTS[layout]
        _check(library().hicache_group_plan_execute(self.handle, self._kvs(kvs), layout, layer,
                                                    _stream(stream)))

    def load_layers(self, kvs, layout=LAYOUT_POOL, stream=None):
        """Every layer, layer by layer, each followed by its event in every
        pool, replayed from a CUDA graph the plan captures on first use."""
        if isinstance(layout, str):
            layout = LAYOUTS[layout]
        _check(library().hicache_group_plan_load_layers(self.handle, self._kvs(kvs), layout,
                                                        _stream(stream)))

    def load_layer_chained(self, kvs, layer: int, layout=LAYOUT_POOL, stream=None):
        """One layer of every pool in one launch, chained to this plan's
        previous layer on the same stream (nothing else on that stream in
        between); each pool's wait_layer waits for it on the device."""
        if isinstance(layout, str):
            layout = LAYOUTS[layout]
        _check(library().hicache_group_plan_load_layer_chained(self.handle, self._kvs(kvs), layout, layer,
                                                               _stream(stream)))

    def close(self):
        if getattr(self, "handle", None):
            library().hicache_group_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def group_plan(pools, device_pages, host_pages, device_num_pages: int) -> GroupPlan:
    return GroupPlan(pools, device_pages, host_pages, device_num_pages)


class PinnedHost:
    """Pinned host memory from host_alloc, freed when the last reference (the
    pool, or any numpy view of it) goes away."""

    def __init__(self, nbytes: int, thp: bool = False):
        self.nbytes = nbytes
        self.ptr = host_alloc(nbytes, thp)

    def free(self):
        if self.ptr:
            ptr, self.ptr = self.ptr, None
            host_free(ptr)

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


class Pool:
    """A host L2 pool of ``host_num_pages`` pages in one layout.

    If ``host_ptr`` is None the pool allocates its pinned memory with
    host_alloc (``thp`` selects the huge-page path); that memory lives as long
    as the pool or any array returned by host_array()."""

    def __init__(self, num_layers: int, num_buffers: int, page_size: int, row_elems: int,
                 host_num_pages: int, layout="layer_first", elem_bytes: int = 2,
                 host_ptr: int | None = None, host_bytes: int | None = None,
                 launch_ctas: int = 0, thp: bool = False):
        self.desc = _desc(num_layers, num_buffers, page_size, row_elems, host_num_pages, layout,
                          elem_bytes, launch_ctas)
        self.num_layers, self.num_buffers, self.page_size = num_layers, num_buffers, page_size
        self.row_elems, self.host_num_pages, self.elem_bytes = row_elems, host_num_pages, elem_bytes
        self.layout = self.desc.layout
        self.nbytes = num_buffers * num_layers * host_num_pages * page_size * row_elems * elem_bytes
        self._mem = PinnedHost(self.nbytes, thp) if host_ptr is None else None
        self.host_ptr = self._mem.ptr if host_ptr is None else host_ptr
        self.host_bytes = self.nbytes if host_bytes is None else host_bytes
        h = ctypes.c_void_p()
        _check(library().hicache_pool_create(ctypes.byref(self.desc), self.host_ptr,
                                             self.host_bytes, ctypes.byref(h)))
        self.handle = h.value

    def host_array(self, dtype=np.uint16) -> np.ndarray:
        """numpy view of the host pool (no copy); keeps the memory alive."""
        buf = (ctypes.c_uint8 * self.nbytes).from_address(self.host_ptr)
        buf._owner = self._mem
        return np.frombuffer(buf, dtype=np.uint8).view(dtype)

    def _xfer(self, fn, kv: DeviceKV, device_pages, host_pages, layout, stream, *extra):
        dp, hp = _idx(device_pages), _idx(host_pages)
        if dp.size != hp.size:
            raise ValueError("device_pages and host_pages differ in length")
        if isinstance(layout, str):
            layout = LAYOUTS[layout]
        rc = fn(self.handle, kv.ref, _ptr(dp), _ptr(hp), dp.size, layout, *extra, _stream(stream))
        if rc:
            _check(rc)

    def backup(self, kv: DeviceKV, device_pages, host_pages, layout=LAYOUT_POOL, stream=None):
        self._xfer(library().hicache_backup, kv, device_pages, host_pages, layout, stream)

    def load(self, kv: DeviceKV, device_pages, host_pages, layout=LAYOUT_POOL, stream=None):
        self._xfer(library().hicache_load, kv, device_pages, host_pages, layout, stream)

    def load_pipelined(self, kv: DeviceKV, device_pages, host_pages, layout=LAYOUT_POOL, stream=None):
        """Every layer in one launch, each layer marked done on the device as it
        lands (wait_layer then waits for that layer alone)."""
        self._xfer(library().hicache_load_pipelined, kv, device_pages, host_pages, layout, stream)

    def load_layer(self, kv: DeviceKV, device_pages, host_pages, layer: int, layout=LAYOUT_POOL,
                   stream=None):
        self._xfer(library().hicache_load_layer, kv, device_pages, host_pages, layout, stream, layer)

    def backup_load(self, kv: DeviceKV, backup_device_pages, backup_host_pages, load_device_pages,
                    load_host_pages, layout=LAYOUT_POOL, stream=None):
        """A backup and a load in one launch (both directions of the link at once)."""
        bd, bh = _idx(backup_device_pages), _idx(backup_host_pages)
        ld, lh = _idx(load_device_pages), _idx(load_host_pages)
        if bd.size != bh.size or ld.size != lh.size:
            raise ValueError("device and host page lists differ in length")
        if isinstance(layout, str):
            layout = LAYOUTS[layout]
        _check(library().hicache_backup_load(self.handle, kv.ref, _ptr(bd), _ptr(bh), bd.size,
                                             _ptr(ld), _ptr(lh), ld.size, layout, _stream(stream)))

    def page_span(self, host_page: int, buffer: int = -1):
        return page_span(self.desc, host_page, buffer)

    def page_view(self, host_page: int, buffer: int = -1) -> np.ndarray:
        """The bytes of one host page (no copy), ready for an L3 write."""
        off, nb = self.page_span(host_page, buffer)
        return self.host_array(np.uint8)[off:off + nb]

    def pipeline_status(self, layer: int):
        """(counter now, value it will reach) for a layer's pipelined loads."""
        d, t = ctypes.c_uint32(), ctypes.c_uint32()
        _check(library().hicache_pipeline_status(self.handle, layer, ctypes.byref(d), ctypes.byref(t)))
        return d.value, t.value

    def layer_counters(self) -> int:
        """Device address of the pool's per-layer counters (for the other ranks
        of a tensor-parallel load)."""
        out = ctypes.c_void_p()
        _check(library().hicache_pool_layer_counters(self.handle, ctypes.byref(out)))
        return out.value

    def wait_layer(self, layer: int, compute_stream=None):
        _check(library().hicache_wait_layer(self.handle, layer, _stream(compute_stream)))

    def layer_event(self, layer: int) -> int:
        ev = ctypes.c_void_p()
        _check(library().hicache_layer_event(self.handle, layer, ctypes.byref(ev)))
        return ev.value

    def plan(self, device_pages, host_pages, device_num_pages: int, direction: int) -> "Plan":
        return Plan(self, device_pages, host_pages, device_num_pages, direction)

    def close(self):
        if getattr(self, "handle", None):
            _check(library().hicache_pool_destroy(self.handle))
            self.handle = None
        self._mem = None   # freed once no host_array view is left

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Engine:
    """Submission engine over a pool (hicache_engine_*): queue backups and loads,
    one worker thread launches them in order, fusing adjacent opposite-direction
    requests into one launch."""

    def __init__(self, pool: "Pool"):
        h = ctypes.c_void_p()
        _check(library().hicache_engine_create(pool.handle, ctypes.byref(h)))
        self.handle = h.value
        self.pool = pool
        self._kvs = []

    def submit(self, kv: DeviceKV, device_pages, host_pages, direction: int, layout=LAYOUT_POOL,
               after_stream=None) -> int:
        dp, hp = _idx(device_pages), _idx(host_pages)
        if dp.size != hp.size:
            raise ValueError("device_pages and host_pages differ in length")
        if isinstance(layout, str):
            layout = LAYOUTS[layout]
        t = ctypes.c_uint64()
        _check(library().hicache_engine_submit(self.handle, kv.ref, _ptr(dp), _ptr(hp), dp.size,
                                               direction, layout, 0 if after_stream is None else 1,
                                               _stream(after_stream), ctypes.byref(t)))
        return t.value

    def wait(self, ticket: int, timeout_us: int = -1):
        _check(library().hicache_engine_wait(self.handle, ticket, timeout_us))

    def wait_on_stream(self, ticket: int, stream=None):
        _check(library().hicache_engine_wait_on_stream(self.handle, ticket, _stream(stream)))

    def stats(self):
        a, b = ctypes.c_int64(), ctypes.c_int64()
        _check(library().hicache_engine_stats(self.handle, ctypes.byref(a), ctypes.byref(b)))
        return a.value, b.value

    def close(self):
        if getattr(self, "handle", None):
            h, self.handle = self.handle, None
            _check(library().hicache_engine_destroy(h))

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class PageAllocator:
    """LIFO host-page allocator (hicache_allocator_*)."""

    def __init__(self, num_pages: int):
        h = ctypes.c_void_p()
        _check(library().hicache_allocator_create(num_pages, ctypes.byref(h)))
        self.handle = h.value
        self.num_pages = num_pages

    def alloc(self, n: int) -> np.ndarray:
        out = np.empty(n, np.int64)
        _check(library().hicache_allocator_alloc(self.handle, n, _ptr(out)))
        return out

    def free(self, pages):
        p = _idx(pages)
        _check(library().hicache_allocator_free(self.handle, _ptr(p), p.size))

    @property
    def available(self) -> int:
        r = library().hicache_allocator_available(self.handle)
        if r < 0:
            _check(int(r))
        return int(r)

    def close(self):
        if getattr(self, "handle", None):
            library().hicache_allocator_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Plan:
    """A validated, pre-passed transfer that can be executed many times (e.g.
    once per layer)."""

    def __init__(self, pool: Pool, device_pages, host_pages, device_num_pages: int, direction: int):
        dp, hp = _idx(device_pages), _idx(host_pages)
        if dp.size != hp.size:
            raise ValueError("device_pages and host_pages differ in length")
        h = ctypes.c_void_p()
        _check(library().hicache_plan_create(pool.handle, _ptr(dp), _ptr(hp), dp.size,
                                             device_num_pages, direction, ctypes.byref(h)))
        self.pool = pool
        self.handle = h.value

    def execute(self, kv: DeviceKV, layer: int = -1, layout=LAYOUT_POOL, stream=None):
        if isinstance(layout, str):
            layout = LAYOUTS[layout]
        _check(library().hicache_plan_execute(self.handle, kv.ref, layout, layer,
                                              _stream(stream)))

    def load_layers(self, kv: DeviceKV, layout=LAYOUT_POOL, stream=None):
        """Every layer, layer by layer, each followed by its layer event, replayed
        from a CUDA graph the plan captures on first use."""
        if isinstance(layout, str):
            layout = LAYOUTS[layout]
        _check(library().hicache_plan_load_layers(self.handle, kv.ref, layout,
                                                  _stream(stream)))

    def load_layer(self, kv: DeviceKV, layer: int, layout=LAYOUT_POOL, stream=None):
        """Load one layer of a load plan and record that layer's event."""
        if isinstance(layout, str):
            layout = LAYOUTS[layout]
        _check(library().hicache_plan_load_layer(self.handle, kv.ref, layout, layer,
                                                 _stream(stream)))

    def load_layer_chained(self, kv: DeviceKV, layer: int, layout=LAYOUT_POOL, stream=None):
        """Load one layer, chained to this plan's previous layer on the same
        stream (nothing else may go on that stream in between); the pool's
        wait_layer waits for it on the device."""
        if isinstance(layout, str):
            layout = LAYOUTS[layout]
        _check(library().hicache_plan_load_layer_chained(self.handle, kv.ref, layout, layer,
                                                         _stream(stream)))

    def load_pipelined(self, kv: DeviceKV, layout=LAYOUT_POOL, stream=None):
        if isinstance(layout, str):
            layout = LAYOUTS[layout]
        _check(library().hicache_plan_load_pipelined(self.handle, kv.ref, layout,
                                                     _stream(stream)))

    def info(self):
        n, r = ctypes.c_int64(), ctypes.c_int64()
        _check(library().hicache_plan_info(self.handle, ctypes.byref(n), ctypes.byref(r)))
        return n.value, r.value

    def close(self):
        if getattr(self, "handle", None):
            library().hicache_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
