"""Helpers for the GPU tests: seeded device/host data and oracle comparisons.

Expected values always come from the oracle (``oracle/``) run on host copies of
the same inputs; nothing here computes a layout offset itself."""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
import tiered_kv_cache_gb300 as hc

# HICACHE_SOAK=k runs the randomised corpora over k times their seeds (a soak;
# the default, 1, is the committed corpus)
SOAK = max(1, int(os.environ.get("HICACHE_SOAK", "1")))

NP_DT = {1: np.uint8, 2: np.uint16, 4: np.uint32, 8: np.uint64}
TORCH_DT = {1: torch.uint8, 2: torch.int16, 4: torch.int32, 8: torch.int64}

_orc = None


def orc() -> oracle.Oracle:
    global _orc
    if _orc is None:
        _orc = oracle.Oracle()
    return _orc


def random_device_bufs(B, L, P, R, Dp, es=2, seed=0):
    """B*L device buffers of random bit patterns (every 16-bit pattern, NaNs
    and signed zeros included)."""
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    bufs = []
    for _ in range(B * L):
        x = torch.randint(0, 256, (Dp * P, R * es), dtype=torch.uint8, device="cuda", generator=g)
        bufs.append(x.view(TORCH_DT[es]))
    return bufs


def to_np(bufs, es):
    return [np.ascontiguousarray(b.cpu().numpy().view(NP_DT[es])) for b in bufs]


def sentinel_fill(bufs, value=0x5A):
    for b in bufs:
        b.view(torch.uint8).fill_(value)


def check_backup(pool: hc.Pool, bufs, dp, hp, layout, B, L, P, R, Hp, es, stream=None, kv=None,
                 sentinel=0xC3):
    """Backup on the GPU and with the oracle from the same inputs; compare the
    whole host pool."""
    host = pool.host_array(np.uint8)
    host[:] = sentinel
    kv = kv or hc.DeviceKV(bufs, bufs[0].shape[0] // P)
    pool.backup(kv, dp, hp, layout, stream=stream)
    torch.cuda.synchronize()
    want = np.full(host.size, sentinel, np.uint8).view(NP_DT[es])
    orc().backup(to_np(bufs, es), want, B, L, P, R, Hp, dp, hp, layout)
    got = host.view(NP_DT[es])
    if not np.array_equal(got, want):
        bad = np.flatnonzero(got != want)
        raise AssertionError(f"backup mismatch at {bad.size} elements, first {bad[:8]}")


def check_load(pool: hc.Pool, bufs, dp, hp, layout, B, L, P, R, Hp, es, layer=-1, seed=1,
               stream=None, sentinel=0x5A):
    """Load (all layers or one) on the GPU and with the oracle from the same host
    pool contents; compare every device buffer."""
    host = pool.host_array(np.uint8)
    rng = np.random.default_rng(seed)
    host[:] = rng.integers(0, 256, host.size, dtype=np.uint8)
    sentinel_fill(bufs, sentinel)
    torch.cuda.synchronize()
    kv = hc.DeviceKV(bufs, bufs[0].shape[0] // P)
    if layer < 0:
        pool.load(kv, dp, hp, layout, stream=stream)
    else:
        pool.load_layer(kv, dp, hp, layer, layout, stream=stream)
    torch.cuda.synchronize()
    want = [np.zeros((bufs[0].shape[0], R), NP_DT[es]) for _ in bufs]
    for w in want:
        w.view(np.uint8)[:] = sentinel
    orc().load(want, host.view(NP_DT[es]), B, L, P, R, Hp, dp, hp, layout, layer)
    got = to_np(bufs, es)
    for k in range(B * L):
        if not np.array_equal(got[k], want[k]):
            bad = np.flatnonzero(got[k] != want[k])
            raise AssertionError(f"load mismatch in buffer {k} at {bad.size} elements, first {bad[:8]}")


def sampled_host_check(host_words: np.ndarray, bufs, dp, hp, layout, B, L, P, R, Hp,
                       samples: int, seed: int):
    """Compare `samples` random elements of the host pool with the device
    buffers; the oracle gives each element's host and device offsets."""
    o = orc()
    rng = np.random.default_rng(seed)
    n = len(dp)
    idx = rng.integers(0, n, samples)
    bb = rng.integers(0, B, samples)
    ll = rng.integers(0, L, samples)
    tt = rng.integers(0, P, samples)
    ee = rng.integers(0, R, samples)
    hoff = np.empty(samples, np.int64)
    doff = np.empty(samples, np.int64)
    for s in range(samples):
        i = int(idx[s])
        hoff[s] = o.host_offset(layout, B, L, P, R, Hp, int(bb[s]), int(ll[s]), int(hp[i]), int(tt[s]), int(ee[s]))
        doff[s] = o.dev_offset(P, R, int(dp[i]), int(tt[s]), int(ee[s]))
    got_host = host_words[hoff]
    flat = [b.view(-1) for b in bufs]
    dev_vals = np.empty(samples, host_words.dtype)
    key = bb * L + ll
    for k in np.unique(key):
        sel = np.flatnonzero(key == k)
        t = torch.from_numpy(doff[sel]).to("cuda")
        dev_vals[sel] = flat[int(k)].index_select(0, t).cpu().numpy().view(host_words.dtype)
    return np.array_equal(got_host, dev_vals)


_libcuda = None


def stream_wait_event(stream, event_handle: int):
    """Make `stream` wait for a raw cudaEvent_t (e.g. a pool's layer event)
    through the driver API (a runtime event handle is a driver event)."""
    import ctypes
    global _libcuda
    if _libcuda is None:
        _libcuda = ctypes.CDLL("libcuda.so.1")
        _libcuda.cuStreamWaitEvent.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint]
        _libcuda.cuStreamWaitEvent.restype = ctypes.c_int
    rc = _libcuda.cuStreamWaitEvent(ctypes.c_void_p(int(stream.cuda_stream)), ctypes.c_void_p(event_handle), 0)
    assert rc == 0, f"cuStreamWaitEvent returned {rc}"
