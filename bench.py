"""Benchmark: L1 <-> L2 KV movement GB/s at 32K tokens on GB300.

A step is one pass of the hot path over the Llama-3-8B-shaped workload (32
layers, K and V, 8 KV heads x 128, page 64; 512 pages = 32,768 tokens; device
pages from a fragmented allocator, host pages contiguous), in each host layout
(layer_first, page_first, page_first_direct):
    backup   512 pages L1 -> L2                      (4 GiB)
    load     512 pages L2 -> L1                      (4 GiB)
    bidir    backup of request A while request B loads on a second stream
             (4 GiB each way, two launches)
    fused    the same pair as one launch (hicache_backup_load)
so 72 GiB move per step.  Every transfer is one kernel launch of libhicache.

Reported: whole-step GB/s (`value`), per layout/operation GB/s and their
fraction of the host-link peak measured in the same run (pinned
cudaMemcpyAsync of 1 GiB: H2D, D2H, both at once), the roofline of the
dominant kernel, the device-side HBM fraction, clocks during the timed
region, an end-to-end number through the Python API with host wall-clock,
and the oracle's rate on the host cores (``cpu_baseline``).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]

Under torchrun (N > 1) every rank runs its own replica on its own GPU (the
path has no exchange step); value = bytes of all ranks / max time over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "L1↔L2 KV GB/s (load, backup, bidir) at 32K tokens; % of measured host-link peak"
LAYOUT_NAMES = ["layer_first", "page_first", "page_first_direct"]   # the pages' three layouts
LAYOUT_IDS = {"layer_first": 0, "page_first": 1, "page_first_direct": 2, "page_first_direct_kv": 3}
NOMINAL = {"pcie_gen5_x16_per_dir_gbs": 63.0, "nvlink_c2c_per_dir_gbs": 450.0}
GB = 1e9


def kernel_fingerprint() -> str:
    """sha256 (first 16 hex digits) of the transfer kernels' source with comments
    and blank lines removed: a comment edit keeps recorded counters valid, a code
    change voids them."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in ("hicache_kernels.cu", "hicache_internal.h"):
        with open(os.path.join(ROOT, "tiered_kv_cache_gb300", "csrc", f)) as fh:
            src = fh.read()
        src = re.sub(r"//[^\n]*", "", src)
        for line in src.splitlines():
            line = line.strip()
            if line:
                h.update(line.encode() + b"\n")
    return h.hexdigest()[:16]


def recorded_traffic():
    """Per-page DRAM and C2C bytes of each (layout/op) kernel from the last ncu
    capture, if the kernel source has not changed since."""
    path = os.path.join(ROOT, "profiles", "xfer_kernel_traffic.txt")
    out = {}
    if not os.path.exists(path):
        return out
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if "=" in line:
                k, v = (x.strip() for x in line.split("=", 1))
                out[k] = v
    if out.get("kernel_source_sha256_16") != kernel_fingerprint():
        return {}
    return out


def max_over_ranks(seconds: float, world: int) -> float:
    """The slowest rank's time: every rank replicates the same transfers on its
    own GPU and host link, so the job ends when the last rank does."""
    if world <= 1:
        return seconds
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([seconds], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_rank: float, max_seconds: float, world: int) -> float:
    """Bytes moved by all ranks / the slowest rank's time (weak scaling)."""
    return world * bytes_per_rank / max_seconds / GB


def frac(a, b, nd=3):
    return round(a / b, nd) if b else None


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "MEASURED_PEAKS.json"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        smax = [num(r[2]) for r in rows if num(r[2]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for name, val in zip(names, r[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max((num(r[3]) or 0.0) for r in rows)}


# ---------------------------------------------------------------- workload
def build_workload(device, pages=512, launch_ctas=0, name="llama3_8b_32k"):
    """Two requests A and B of `pages` pages each over the workload's pools:
    llama3_8b_32k -- fragmented device pages (runs of 1-8), contiguous host;
    deep78_32k    -- 78 layers, fully scattered device pages, contiguous host.
    (1024 device and 1024 host pages at 512 pages per transfer; 2x `pages`
    each for a scaled-down case.)"""
    import torch
    import tiered_kv_cache_gb300 as hc
    from tiered_kv_cache_gb300 import workloads as wl

    s, a_dev, b_dev, a_host, b_host = workload_indices(name, pages)
    vals = [v.view(torch.int16) for v in wl.kv_values(s, device=device)]
    pool = hc.Pool(s.num_layers, s.num_buffers, s.page_size, s.row_elems, s.host_pages, "layer_first",
                   launch_ctas=launch_ctas)
    kv = hc.DeviceKV(vals, s.device_pages)
    return dict(shape=s, vals=vals, kv=kv, pool=pool, a_dev=a_dev, b_dev=b_dev, a_host=a_host,
                b_host=b_host, bytes_per_xfer=pages * s.page_bytes, pages=pages)


def link_peaks(torch, nbytes=1 << 30, reps=5, hc=None):
    """Pinned cudaMemcpyAsync of 1 GiB: H2D, D2H, and both at once."""
    host_a = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    host_b = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    dev_a = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    dev_b = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()

    def timed(fn):
        best = float("inf")
        for _ in range(reps):
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(s1)
            s2.wait_event(e0)
            fn()
            done = torch.cuda.Event()
            done.record(s2)
            s1.wait_event(done)
            e1.record(s1)
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1) / 1e3)
        return best

    def h2d():
        with torch.cuda.stream(s1):
            dev_a.copy_(host_a, non_blocking=True)

    def d2h():
        with torch.cuda.stream(s1):
            host_b.copy_(dev_b, non_blocking=True)

    def both():
        with torch.cuda.stream(s1):
            dev_a.copy_(host_a, non_blocking=True)
        with torch.cuda.stream(s2):
            host_b.copy_(dev_b, non_blocking=True)

    t_h2d, t_d2h, t_bi = timed(h2d), timed(d2h), timed(both)
    res = {"h2d_gbs": nbytes / t_h2d / GB, "d2h_gbs": nbytes / t_d2h / GB,
           "bidir_gbs": 2 * nbytes / t_bi / GB, "bytes": nbytes, "how": "pinned cudaMemcpyAsync, best of 5"}
    dev_d = torch.empty(nbytes, dtype=torch.uint8, device="cuda")

    def d2d():
        with torch.cuda.stream(s1):
            dev_d.copy_(dev_a)

    t_dd = timed(d2d)
    res["d2d_gbs"] = 2 * nbytes / t_dd / GB      # bytes read + written
    res["d2d_how"] = "device-to-device copy of 1 GiB on the same stream, bytes read + written, best of 5"
    if hc is not None:
        res["zero_copy_kernel"] = link_probe_kernel(torch, hc, timed, s1, s2, host_a, host_b, dev_a, dev_b,
                                                    nbytes)
    res["host_dram"] = host_copy_rate()
    del host_a, host_b, dev_a, dev_b, dev_d
    return res


def binding_resource(link):
    """What caps the host link, from this run's probes: the copy engines and
    the SM streaming kernel at every grid and depth stop at the same rate, and
    a host source small enough for the host's cache is no faster, so neither
    the engine, the requests in flight nor host DRAM binds."""
    k = link.get("zero_copy_kernel") or {}
    if not k or not link.get("h2d_gbs"):
        return None
    h2d = k["h2d_by_grid_x_vecs_per_thread"]
    d2h = k["d2h_by_grid_x_vecs_per_thread"]
    return {
        "resource": "the GPU's NVLink-C2C link to host memory, at the rate it delivers to this GPU",
        "h2d_gbs": {"copy_engine": round(link["h2d_gbs"], 1), "sm_kernel_min": min(h2d.values()),
                    "sm_kernel_max": max(h2d.values()), "sm_kernel_32mib_cached_source": k["h2d_32mib_source_gbs"]},
        "d2h_gbs": {"copy_engine": round(link["d2h_gbs"], 1), "sm_kernel_min": min(d2h.values()),
                    "sm_kernel_max": max(d2h.values())},
        "host_dram_copy_gbs": (link.get("host_dram") or {}).get("copy_gbs_read_plus_write"),
        "sm_kernel_grids": "38-608 CTAs x 4 or 8 16-byte vectors in flight per thread",
        "ncu_c2c_fraction": "of ncu's nominal C2C capacity (about 320 GB/s per direction), protocol bytes "
                            "included: a load fills 66% of RX, a backup 75% of TX, the fused pair 79% "
                            "each way; one direction alone leaves raw capacity unused, so for loads the host "
                            "side's read-return rate binds",
        "nominal": "900 GB/s two-way NVLink-C2C per Grace, which serves two GPUs: 450 two-way, 225 per "
                   "direction per GPU (a reading of the superchip figure)",
    }


def link_probe_kernel(torch, hc, timed, s1, s2, host_a, host_b, dev_a, dev_b, nbytes):
    """The same 1 GiB moves by the library's plain streaming-copy kernel (SM
    loads and stores to mapped pinned memory, no index decode), over a sweep of
    grids and bytes in flight; and a load whose 32 MiB host source is read 32
    times over, so that it can sit in the host's last-level cache instead of
    its DRAM."""
    grids = (38, 76, 152, 304, 608)
    h2d, d2h = {}, {}
    for unroll in (4, 8):
        for g in grids:
            t = timed(lambda: hc.stream_copy(dev_a.data_ptr(), host_a.data_ptr(), nbytes, g, unroll, s1))
            h2d[f"{g}x{unroll}"] = round(nbytes / t / GB, 1)
            t = timed(lambda: hc.stream_copy(host_b.data_ptr(), dev_b.data_ptr(), nbytes, g, unroll, s1))
            d2h[f"{g}x{unroll}"] = round(nbytes / t / GB, 1)

    def both():
        hc.stream_copy(dev_a.data_ptr(), host_a.data_ptr(), nbytes, 152, 4, s1)
        hc.stream_copy(host_b.data_ptr(), dev_b.data_ptr(), nbytes, 95, 4, s2)
    t_bi = timed(both)
    small = 32 << 20

    def cached():
        for k in range(nbytes // small):
            hc.stream_copy(dev_a.data_ptr() + k * small, host_a.data_ptr(), small, 152, 4, s1)
    t_c = timed(cached)
    return {"h2d_gbs": max(h2d.values()), "d2h_gbs": max(d2h.values()),
            "bidir_gbs": round(2 * nbytes / t_bi / GB, 1),
            "h2d_32mib_source_gbs": round(nbytes / t_c / GB, 1),
            "h2d_by_grid_x_vecs_per_thread": h2d, "d2h_by_grid_x_vecs_per_thread": d2h,
            "how": "hicache_stream_copy of 1 GiB, best of 5 per setting; bidir = 152-CTA load and 95-CTA "
                   "backup on two streams; the 32 MiB source case copies one 32 MiB host range into 32 "
                   "device ranges"}


def host_copy_rate(nbytes=1 << 30, reps=3):
    """The host's own memory bandwidth: numpy copies of 1 GiB split over every
    core (bytes read + written)."""
    import threading
    n = os.cpu_count() or 1
    a = np.ones(nbytes, np.uint8)
    b = np.zeros(nbytes, np.uint8)
    parts = [(nbytes * k // n, nbytes * (k + 1) // n) for k in range(n)]
    best = float("inf")
    for _ in range(reps):
        ts = [threading.Thread(target=np.copyto, args=(b[x:y], a[x:y])) for x, y in parts]
        t0 = time.perf_counter()
        for t in ts:
            t.start()
        for t in ts:
            t.join()
        best = min(best, time.perf_counter() - t0)
    return {"copy_gbs_read_plus_write": round(2 * nbytes / best / GB, 1), "threads": n,
            "how": "numpy copy of 1 GiB split over every core, best of 3"}


def run_step(torch, w, s1, s2, ev=None):
    """One step; if `ev` is a list, (name, start, end) event triples are appended."""
    pool, kv = w["pool"], w["kv"]
    for lay in LAYOUT_NAMES:
        lid = LAYOUT_IDS[lay]

        def mark():
            e = torch.cuda.Event(enable_timing=True)
            e.record(s1)
            return e
        e0 = mark() if ev is not None else None
        pool.backup(kv, w["a_dev"], w["a_host"], lid, stream=s1)
        e1 = mark() if ev is not None else None
        pool.load(kv, w["a_dev"], w["a_host"], lid, stream=s1)
        e2 = mark() if ev is not None else None
        if ev is None:
            e2 = torch.cuda.Event()
            e2.record(s1)
        s2.wait_event(e2)
        pool.backup(kv, w["a_dev"], w["a_host"], lid, stream=s1)
        pool.load(kv, w["b_dev"], w["b_host"], lid, stream=s2)
        j = torch.cuda.Event(enable_timing=ev is not None)
        j.record(s2)
        s1.wait_event(j)
        e3 = mark() if ev is not None else None
        pool.backup_load(kv, w["a_dev"], w["a_host"], w["b_dev"], w["b_host"], lid, stream=s1)
        e4 = mark() if ev is not None else None
        if ev is not None:
            ev += [(f"{lay}/backup", e0, e1), (f"{lay}/load", e1, e2), (f"{lay}/bidir", e2, e3),
                   (f"{lay}/bidir_fused", e3, e4)]


def _oracle_rate(shape, pages, seconds, threads=1, layouts=(0, 1, 2)):
    """GB/s of the oracle (single-threaded C, as written) doing backup + load of
    `pages` pages of `shape` per layout, on host arrays.  With threads > 1 the
    pairs are split into `threads` disjoint groups, each handled by one oracle
    call on its own thread (ctypes drops the GIL during the call)."""
    import threading
    import oracle
    from tiered_kv_cache_gb300 import workloads as wl
    o = oracle.Oracle()
    rng = np.random.default_rng(0)
    Dp = Hp = pages * 2
    B, L, P, R = shape.num_buffers, shape.num_layers, shape.page_size, shape.row_elems
    dev = [rng.integers(0, 65535, (Dp * P, R), dtype=np.uint16) for _ in range(B * L)]
    host = np.zeros(B * L * Hp * P * R, np.uint16)
    dp = wl.fragmented_pages(rng, Dp, pages)
    hp = np.arange(pages)
    groups = [(dp[k::threads], hp[k::threads]) for k in range(threads)]

    def run(fn):
        if threads == 1:
            fn(dp, hp)
            return
        ts = [threading.Thread(target=fn, args=g) for g in groups]
        for t in ts:
            t.start()
        for t in ts:
            t.join()

    moved, ops = 0, 0
    t0 = time.perf_counter()
    while True:
        for lid in layouts:
            run(lambda d, h: o.backup(dev, host, B, L, P, R, Hp, d, h, lid))
            run(lambda d, h: o.load(dev, host, B, L, P, R, Hp, d, h, lid))
            moved += 2 * pages * shape.page_bytes
            ops += 2
        el = time.perf_counter() - t0
        if el >= seconds or ops >= 60:
            break
    return moved / el / GB, ops, el


def cpu_baseline(seconds_target=10.0, pages=24):
    """The oracle on the host cores, on bounded samples of the workloads: the
    headline is one core on the Llama-3-8B shape; the deep-78 and MLA shapes
    and an all-cores run of the same loop split over the pairs are reported
    beside it."""
    from tiered_kv_cache_gb300 import workloads as wl
    s = wl.LLAMA3_8B
    v, ops, el = _oracle_rate(s, pages, seconds_target)
    ncores = os.cpu_count() or 1
    va, opsa, ela = _oracle_rate(s, 8 * ncores, 4.0, threads=ncores)
    vd, _, eld = _oracle_rate(wl.DEEP_STRESS, 8, 3.0)
    vm, _, elm = _oracle_rate(wl.MLA_LATENT, 32, 3.0, layouts=(1,))
    return {"value": v, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{ops} transfers of {pages} pages ({pages * s.page_bytes / 2**20:.0f} MiB each) of the "
                      f"llama3_8b shape, backup+load in all three layouts, host arrays, {el:.1f} s",
            "all_cores": {"value": round(va, 2), "cores": ncores,
                          "sample": f"{opsa} transfers of {8 * ncores} pages split over {ncores} threads, "
                                    f"{ela:.1f} s"},
            "deep78_1core": {"value": round(vd, 3), "sample": f"8-page transfers, all layouts, {eld:.1f} s"},
            "mla61_1core": {"value": round(vm, 3), "sample": f"32-page transfers, page_first, {elm:.1f} s"}}


def step_config(args, npages, bpx):
    """The `config` of a step line: the same for both arms."""
    step_bytes = len(LAYOUT_NAMES) * 6 * bpx
    return {"workload": (f"llama3_8b_{npages * 64 // 1024}k: 32 layers, K+V, 8 kv heads x 128, "
                         f"bf16, page 64, {npages} pages = {npages * 64} tokens per transfer, "
                         "fragmented device pages, contiguous host pages")
            if args.workload == "llama3_8b_32k" else
            (f"deep78_{npages * 64 // 1024}k: 78 layers, K+V, 8 kv heads x 128, bf16, page 64, "
             f"{npages} pages per transfer, fully scattered device pages, contiguous host pages"),
            "step": f"per layout ({', '.join(LAYOUT_NAMES)}): backup, load, "
                    "concurrent backup+load of two requests on two streams, and the same pair "
                    f"as one fused launch; {step_bytes / 2**30:.0f} GiB per step",
            "l2": f"inputs larger than L2 ({bpx / 2**20:.0f} MiB per transfer)",
            "launch_ctas": args.ctas or "auto"}


def workload_indices(name, pages):
    """Shape and page indices of requests A and B of a step workload (the
    same draws build_workload makes)."""
    import dataclasses
    from tiered_kv_cache_gb300 import workloads as wl
    s = wl.LLAMA3_8B if name == "llama3_8b_32k" else wl.DEEP_STRESS
    if pages != 512:
        s = dataclasses.replace(s, device_pages=2 * pages, host_pages=2 * pages)
    if name == "llama3_8b_32k":
        a_dev = wl.llama_transfer(s, pages).device_pages
        b_dev = wl.fragmented_pages(wl.index_rng(s.seed + 1), s.device_pages, pages, exclude=a_dev)
    else:
        a, b = wl.deep_bidir_transfers(s, pages)
        a_dev, b_dev = a.device_pages, b.device_pages
    return s, a_dev, b_dev, wl.contiguous_pages(pages, 0), wl.contiguous_pages(pages, pages)


def reference_arm(args):
    """`--impl reference`: the oracle (single-threaded C, as written) on one
    host core, on the same workload as the step: the same pools, pages and
    layouts, at full transfer size.  One oracle transfer of a full request
    takes seconds, so a reference step is ONE of the step's transfers, taken in
    the step's order (per layout: backup A, load A, backup A with load B,
    fused backup A + load B), and GB/s = bytes moved / time."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    s, a_dev, b_dev, a_host, b_host = workload_indices(args.workload, args.pages)
    o = oracle.Oracle()
    B, L, P, R, Dp, Hp = s.num_buffers, s.num_layers, s.page_size, s.row_elems, s.device_pages, s.host_pages
    block = np.random.default_rng(0).integers(0, 1 << 16, 1 << 20, dtype=np.uint16)

    def filled(n):
        a = np.empty(n, np.uint16)
        for off in range(0, n, block.size):
            m = min(block.size, n - off)
            a[off:off + m] = block[:m]
        return a
    dev = [filled(Dp * P * R).reshape(Dp * P, R) for _ in range(B * L)]
    host = filled(B * L * Hp * P * R)
    ops = []
    for lay in LAYOUT_NAMES:
        lid = LAYOUT_IDS[lay]
        ops += [(o.backup, a_dev, a_host, lid), (o.load, a_dev, a_host, lid),
                (o.backup, a_dev, a_host, lid), (o.load, b_dev, b_host, lid),
                (o.backup, a_dev, a_host, lid), (o.load, b_dev, b_host, lid)]
    bpx = args.pages * s.page_bytes
    k = 0

    def step():
        nonlocal k
        fn, d, h, lid = ops[k % len(ops)]
        k += 1
        fn(dev, host, B, L, P, R, Hp, d, h, lid)
        return bpx

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    moved = sum(step() for _ in range(args.steps))
    el = time.perf_counter() - t0
    v = moved / el / GB
    sample = (f"each step one of the GPU step's {len(ops)} transfers of {args.pages} pages "
              f"({bpx / 2**30:.3g} GiB), in the step's order; {args.steps} steps after {args.warmup} "
              f"warm-up steps; host arrays; {el:.1f} s timed")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": step_config(args, args.pages, bpx),
        "cpu_baseline": {"value": v, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def _elapsed(torch, e0, e1):
    return e0.elapsed_time(e1) / 1e3


def breakdown_from_events(ev, bpx, link, stat="mean"):
    """Per-layout, per-operation GB/s (from the mean launch time, or the
    median with stat="median") and their fraction of the in-run link peak,
    from (name, start, end) event triples."""
    per = {}
    for name, a, b in ev:
        per.setdefault(name, []).append(a.elapsed_time(b) / 1e3)
    avg = statistics.median if stat == "median" else statistics.mean
    breakdown = {}
    for lay in LAYOUT_NAMES:
        bk = bpx / avg(per[f"{lay}/backup"]) / GB
        ld = bpx / avg(per[f"{lay}/load"]) / GB
        bi = 2 * bpx / avg(per[f"{lay}/bidir"]) / GB
        bf = 2 * bpx / avg(per[f"{lay}/bidir_fused"]) / GB
        breakdown[lay] = {
            "backup_gbs": round(bk, 1), "load_gbs": round(ld, 1),
            "bidir_streams_gbs": round(bi, 1), "bidir_fused_gbs": round(bf, 1),
            "backup_frac_of_link": frac(bk, link["d2h_gbs"]),
            "load_frac_of_link": frac(ld, link["h2d_gbs"]),
            "bidir_streams_frac_of_link": frac(bi, link["bidir_gbs"]),
            "bidir_fused_frac_of_link": frac(bf, link["bidir_gbs"]),
            # per-op launch times (GB/s above are from the `stat` of these); `slow`
            # counts the steps more than 15% above the fastest (on a shared host,
            # windows of host-memory contention slow the two-direction steps)
            "ms": {op: {"mean": round(statistics.mean(per[f"{lay}/{op}"]) * 1e3, 3),
                        "median": round(statistics.median(per[f"{lay}/{op}"]) * 1e3, 3),
                        "min": round(min(per[f"{lay}/{op}"]) * 1e3, 3), "n": len(per[f"{lay}/{op}"]),
                        "slow": sum(1 for t in per[f"{lay}/{op}"] if t > 1.15 * min(per[f"{lay}/{op}"]))}
                   for op in ("backup", "load", "bidir", "bidir_fused")},
        }
    return per, breakdown


def bench_deep78(torch, hc, args, link, steps=20):
    """The deep-model segment-count stress: 78 layers, K+V, 512 fully scattered
    device pages per request (39,936 page x layer segments per buffer under
    page_first_direct), the same four operations per layout as the headline
    step, timed with events over `steps` steps after one warm-up step.  GB/s
    come from the median launch time, with the mean and the minimum beside it
    in `ms`: on some shared hosts a disturbance every ~0.5 s halves both
    directions of a two-direction transfer for a few tens of ms (one-direction
    transfers are untouched), and it can fall on the same operation of
    several steps in a row."""
    w = build_workload("cuda", 512, args.ctas, "deep78_32k")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    run_step(torch, w, s1, s2)
    torch.cuda.synchronize()
    ev = []
    for _ in range(steps):
        run_step(torch, w, s1, s2, ev)
    torch.cuda.synchronize()
    s = w["shape"]
    seg = {lay: hc.segment_count(s.num_layers, s.num_buffers, s.page_size, s.row_elems, s.host_pages,
                                 LAYOUT_IDS[lay], w["a_dev"], w["a_host"]) // s.num_buffers
           for lay in LAYOUT_NAMES}
    _, br = breakdown_from_events(ev, w["bytes_per_xfer"], link, stat="median")
    w["pool"].close()
    del w
    torch.cuda.empty_cache()
    return {"bytes_per_transfer": 512 * s.page_bytes, "segments_per_buffer": seg, "steps": steps,
            "gbs_from": "median launch time", "breakdown": br}


def bench_host_shuffled(torch, hc, args, link, reps=5):
    """The Llama-3-8B transfer of the headline with the host pages shuffled
    (a random permutation sample of the host pool instead of a contiguous
    range): backup and load of 512 pages per layout, event-timed, median of
    `reps` after one warm-up call."""
    from tiered_kv_cache_gb300 import workloads as wl
    s = wl.LLAMA3_8B
    t = wl.llama_transfer(s, 512, shuffled_host=True)
    vals = [v.view(torch.int16) for v in wl.kv_values(s, device="cuda")]
    kv = hc.DeviceKV(vals, s.device_pages)
    pool = hc.Pool(s.num_layers, s.num_buffers, s.page_size, s.row_elems, s.host_pages, "layer_first",
                   launch_ctas=args.ctas)
    st = torch.cuda.Stream()
    bpx = 512 * s.page_bytes
    out = {}
    for lay in LAYOUT_NAMES:
        lid = LAYOUT_IDS[lay]
        res = {}
        for op, fn in (("backup", pool.backup), ("load", pool.load)):
            fn(kv, t.device_pages, t.host_pages, lid, stream=st)
            times = []
            for _ in range(reps):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(st)
                fn(kv, t.device_pages, t.host_pages, lid, stream=st)
                e1.record(st)
                torch.cuda.synchronize()
                times.append(_elapsed(torch, e0, e1))
            gbs = bpx / statistics.median(times) / GB
            res[f"{op}_gbs"] = round(gbs, 1)
            res[f"{op}_min_ms"] = round(min(times) * 1e3, 3)
            res[f"{op}_frac_of_link"] = frac(gbs, link["d2h_gbs"] if op == "backup" else link["h2d_gbs"])
        out[lay] = res
    pool.close()
    del vals, kv
    torch.cuda.empty_cache()
    return out


def bench_extras(torch, hc, args, link):
    """The other workload shapes, measured after the headline step of the
    default run so that one bench line carries them all."""
    import types
    out = {}
    t0 = time.perf_counter()
    out["llama3_8b_32k_host_shuffled"] = bench_host_shuffled(torch, hc, args, link)
    out["llama3_8b_32k_host_shuffled"]["wall_s"] = round(time.perf_counter() - t0, 1)
    t0 = time.perf_counter()
    out["deep78_32k"] = bench_deep78(torch, hc, args, link)
    out["deep78_32k"]["wall_s"] = round(time.perf_counter() - t0, 1)
    t0 = time.perf_counter()
    mla_args = types.SimpleNamespace(ctas=args.ctas, tokens="4096,16384,65536", steps=min(args.steps, 10),
                                     warmup=3)
    res, launches = bench_mla_overlap(torch, hc, mla_args)
    out["mla61"] = {"results": res, "gpu_launches": launches, "wall_s": round(time.perf_counter() - t0, 1),
                    "how": "61 per-layer loads with an event each (per_layer), the same replayed from a "
                           "plan's graph (graph), one chained call per layer (chained: attention behind "
                           "the layer's counter; chained_events: behind the layer's CUDA event), one "
                           "pipelined launch (pipelined), one all-layer launch; alone and overlapped with "
                           "a stand-in attention on a second stream; overlap efficiency = (load + compute "
                           "- overlapped) / min(load, compute)"}
    torch.cuda.empty_cache()
    t0 = time.perf_counter()
    out["small_mix"] = bench_small_mix(torch, hc, args, link)
    out["small_mix"]["wall_s"] = round(time.perf_counter() - t0, 1)
    torch.cuda.empty_cache()
    # the row-size x page-size stress (fully scattered pages, about 1 GiB per call)
    t0 = time.perf_counter()
    rows = bench_shapes(torch, hc, args)
    for r in rows:
        for k in [k for k in r if k.endswith("_gbs")]:
            peak = link["d2h_gbs"] if k.startswith("backup") else link["h2d_gbs"]
            r[k.replace("_gbs", "_frac_of_link")] = frac(r[k], peak)
    out["shapes"] = {"rows": rows, "wall_s": round(time.perf_counter() - t0, 1)}
    torch.cuda.empty_cache()
    # the buffer group (MLA latent + indexer key + scales) and the tensor-parallel
    # load with stand-in ranks
    small_args = types.SimpleNamespace(ctas=args.ctas, steps=min(args.steps, 5), warmup=3)
    t0 = time.perf_counter()
    res, launches = bench_nsa_group(torch, hc, small_args)
    out["nsa_group"] = {"results": res, "gpu_launches": launches, "wall_s": round(time.perf_counter() - t0, 1)}
    torch.cuda.empty_cache()
    t0 = time.perf_counter()
    out["tp_mla61"] = {"results": bench_tp_mla(torch, hc, small_args),
                       "how": "tp stand-in ranks on one GPU (pools over one host memory); host_read_gbs is "
                              "the group's, over the one host link",
                       "wall_s": round(time.perf_counter() - t0, 1)}
    torch.cuda.empty_cache()
    return out


def bench_mla_overlap(torch, hc, args):
    """MLA latent (61 layers, kv_dim 576, page 64), page_first host pool:
    per-layer loads on a transfer stream, each recording its layer event; a
    stand-in attention kernel per layer on a compute stream that waits on that
    event.  Reports (a) the 61 per-layer loads alone, (b) the compute alone,
    (c) both overlapped, and the overlap efficiency (a + b - c) / min(a, b)."""
    from tiered_kv_cache_gb300 import workloads as wl
    s = wl.MLA_LATENT
    vals = [v.view(torch.int16) for v in wl.kv_values(s, device="cuda")]
    kv = hc.DeviceKV(vals, s.device_pages)
    pool = hc.Pool(s.num_layers, s.num_buffers, s.page_size, s.row_elems, s.host_pages, "page_first",
                   launch_ctas=args.ctas)
    L = s.num_layers
    sums = torch.zeros(L, dtype=torch.int64, device="cuda")
    out = {}
    launches0 = hc.launch_count()
    sizes = [int(t) for t in args.tokens.split(",")] if args.tokens else [4096, 16384, 65536]
    for tokens, prio in [(t, 0) for t in sizes] + [(t, -1) for t in sizes if not args.tokens]:
        # prio -1: the transfer stream outranks the compute stream, so the block
        # scheduler places the transfer's CTAs first as compute CTAs retire
        xfer = torch.cuda.Stream(priority=prio)
        xfer2 = torch.cuda.Stream(priority=prio)
        comp = torch.cuda.Stream()
        t = wl.mla_transfer(s, tokens)
        n = len(t.device_pages)
        plan = pool.plan(t.device_pages, t.host_pages, s.device_pages, hc.LOAD)
        nbytes = n * s.page_bytes

        def timed(fn, reps=args.steps):
            best = []
            for _ in range(max(args.warmup, 3)):
                fn()
            torch.cuda.synchronize()
            for _ in range(reps):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(xfer)
                comp.wait_event(e0)
                xfer2.wait_event(e0)
                fn()
                for other in (comp, xfer2):
                    j = torch.cuda.Event()
                    j.record(other)
                    xfer.wait_event(j)
                e1.record(xfer)
                torch.cuda.synchronize()
                best.append(_elapsed(torch, e0, e1))
            return statistics.median(best)

        def loads():
            for layer in range(L):
                plan.execute(kv, layer=layer, stream=xfer)

        def loads_two_streams():
            # consecutive layers on alternating streams: the start of layer l+1
            # overlaps the tail of layer l
            for layer in range(L):
                plan.execute(kv, layer=layer, stream=xfer if layer % 2 == 0 else xfer2)

        def overlapped_two_streams(reps):
            for layer in range(L):
                plan.execute(kv, layer=layer, stream=xfer if layer % 2 == 0 else xfer2)
                pool.wait_layer(layer, comp)
                hc.layer_checksum(kv, pool, t.device_pages, layer, sums.data_ptr() + 8 * layer, reps=reps,
                                  stream=comp)

        def one_load():
            plan.execute(kv, layer=-1, stream=xfer)

        def computes(reps):
            for layer in range(L):
                hc.layer_checksum(kv, pool, t.device_pages, layer, sums.data_ptr() + 8 * layer, reps=reps,
                                  stream=comp)

        def overlapped(reps):
            for layer in range(L):
                plan.execute(kv, layer=layer, stream=xfer)
                pool.wait_layer(layer, comp)
                hc.layer_checksum(kv, pool, t.device_pages, layer, sums.data_ptr() + 8 * layer, reps=reps,
                                  stream=comp)

        def pipelined():
            plan.load_pipelined(kv, stream=xfer)

        def loads_graph():
            plan.load_layers(kv, stream=xfer)

        def loads_chained():
            for layer in range(L):
                plan.load_layer_chained(kv, layer, stream=xfer)

        def overlapped_chained(reps):
            for layer in range(L):
                plan.load_layer_chained(kv, layer, stream=xfer)
                pool.wait_layer(layer, comp)
                hc.layer_checksum(kv, pool, t.device_pages, layer, sums.data_ptr() + 8 * layer, reps=reps,
                                  stream=comp)

        def overlapped_chained_events(reps):
            # the pages' own form: one call per layer, attention behind that layer's CUDA event
            for layer in range(L):
                plan.load_layer_chained(kv, layer, stream=xfer)
                _stream_wait_raw_event(comp, pool.layer_event(layer))
                hc.layer_checksum(kv, pool, t.device_pages, layer, sums.data_ptr() + 8 * layer, reps=reps,
                                  stream=comp)

        def overlapped_graph(reps):
            plan.load_layers(kv, stream=xfer)
            for layer in range(L):
                pool.wait_layer(layer, comp)
                hc.layer_checksum(kv, pool, t.device_pages, layer, sums.data_ptr() + 8 * layer, reps=reps,
                                  stream=comp)

        def overlapped_pipelined(reps):
            plan.load_pipelined(kv, stream=xfer)
            for layer in range(L):
                pool.wait_layer(layer, comp)
                hc.layer_checksum(kv, pool, t.device_pages, layer, sums.data_ptr() + 8 * layer, reps=reps,
                                  stream=comp)

        a = timed(loads)
        whole = timed(one_load)
        ap = timed(pipelined)
        c1 = timed(lambda: computes(1))
        reps = max(1, int(round(a / c1)))          # stand-in attention about as long as the loads
        b = timed(lambda: computes(reps))
        c = timed(lambda: overlapped(reps))
        cp = timed(lambda: overlapped_pipelined(reps))
        a2 = timed(loads_two_streams)
        c2 = timed(lambda: overlapped_two_streams(reps))
        ag = timed(loads_graph)
        cg = timed(lambda: overlapped_graph(reps))
        ach = timed(loads_chained)
        cch = timed(lambda: overlapped_chained(reps))
        cce = timed(lambda: overlapped_chained_events(reps))
        out[f"{tokens // 1024}k" + ("_xfer_high_priority" if prio else "")] = {
            "pages": n, "bytes": nbytes,
            "per_layer_loads_ms": round(a * 1e3, 3), "per_layer_load_gbs": round(nbytes / a / GB, 1),
            "one_launch_load_ms": round(whole * 1e3, 3), "one_launch_load_gbs": round(nbytes / whole / GB, 1),
            "compute_ms": round(b * 1e3, 3), "compute_reps": reps,
            "overlapped_ms": round(c * 1e3, 3),
            "overlap_efficiency": round((a + b - c) / min(a, b), 3),
            "pipelined_load_ms": round(ap * 1e3, 3), "pipelined_load_gbs": round(nbytes / ap / GB, 1),
            "overlapped_pipelined_ms": round(cp * 1e3, 3),
            "overlap_efficiency_pipelined": round((ap + b - cp) / min(ap, b), 3),
            "per_layer_loads_2streams_ms": round(a2 * 1e3, 3),
            "per_layer_load_2streams_gbs": round(nbytes / a2 / GB, 1),
            "overlapped_2streams_ms": round(c2 * 1e3, 3),
            "overlap_efficiency_2streams": round((a2 + b - c2) / min(a2, b), 3),
            "per_layer_graph_ms": round(ag * 1e3, 3), "per_layer_graph_gbs": round(nbytes / ag / GB, 1),
            "overlapped_graph_ms": round(cg * 1e3, 3),
            "overlap_efficiency_graph": round((ag + b - cg) / min(ag, b), 3),
            "per_layer_chained_ms": round(ach * 1e3, 3),
            "per_layer_chained_gbs": round(nbytes / ach / GB, 1),
            "overlapped_chained_ms": round(cch * 1e3, 3),
            "overlap_efficiency_chained": round((ach + b - cch) / min(ach, b), 3),
            "overlapped_chained_events_ms": round(cce * 1e3, 3),
            "overlap_efficiency_chained_events": round((ach + b - cce) / min(ach, b), 3),
        }
        plan.close()
    launches = hc.launch_count() - launches0
    pool.close()
    return out, launches


_libcuda = None


def _stream_wait_raw_event(stream, event_handle: int):
    """Make a torch stream wait for a raw cudaEvent_t (a pool's layer event)
    through the driver API (a runtime event handle is a driver event)."""
    import ctypes
    global _libcuda
    if _libcuda is None:
        _libcuda = ctypes.CDLL("libcuda.so.1")
        _libcuda.cuStreamWaitEvent.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint]
        _libcuda.cuStreamWaitEvent.restype = ctypes.c_int
    rc = _libcuda.cuStreamWaitEvent(ctypes.c_void_p(int(stream.cuda_stream)), ctypes.c_void_p(event_handle), 0)
    if rc != 0:
        raise RuntimeError(f"cuStreamWaitEvent returned {rc}")


def bench_tp_mla(torch, hc, args):
    """The tensor-parallel load of the MLA latent (61 layers, 576 bf16, page 64,
    page_first) with tp ranks stood in for by tp pools on this one GPU over the
    same host memory, each rank's launch on its own stream: every rank reads
    1/tp of the pages and stores them into all tp ranks' buffers.  On one GPU
    all ranks share one host link, so the whole group moves the request's bytes
    over it once; the rates show what the fan-out stores cost the host reads
    (compare tp = 1, a plain pipelined load)."""
    from tiered_kv_cache_gb300 import workloads as wl
    s = wl.MLA_LATENT
    B, L, P, R, Dp, Hp = s.num_buffers, s.num_layers, s.page_size, s.row_elems, s.device_pages, s.host_pages
    mem = hc.PinnedHost(B * L * Hp * P * R * 2)
    out = {}
    for tp in (1, 2, 4, 8):
        pools = [hc.Pool(L, B, P, R, Hp, "page_first", host_ptr=mem.ptr, host_bytes=mem.nbytes,
                         launch_ctas=args.ctas) for _ in range(tp)]
        bufs = [[torch.empty((Dp * P, R), dtype=torch.int16, device="cuda") for _ in range(L)] for _ in range(tp)]
        kvs = [hc.DeviceKV(b, Dp) for b in bufs]
        counters = [p.layer_counters() for p in pools]
        streams = [torch.cuda.Stream() for _ in range(tp)]
        gate = torch.cuda.Stream()
        for tokens in (4096, 16384, 65536):
            t = wl.mla_transfer(s, tokens)
            nbytes = len(t.device_pages) * s.page_bytes

            def once(plain=False):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                torch.cuda.synchronize()
                torch.cuda._sleep(2_000_000)               # host enqueues every rank before the GPU starts
                e0.record()
                for st in streams:
                    st.wait_event(e0)
                for r, pool in enumerate(pools):
                    if plain:                              # the same bytes as one plain pipelined load
                        pool.load_pipelined(kvs[r], t.device_pages, t.host_pages, stream=streams[r])
                    else:
                        hc.tp_load_pipelined(pool, kvs, counters, r, t.device_pages, t.host_pages,
                                             stream=streams[r])
                for st in streams:
                    j = torch.cuda.Event()
                    j.record(st)
                    torch.cuda.current_stream().wait_event(j)
                e1.record()
                torch.cuda.synchronize()
                return e0.elapsed_time(e1) / 1e3
            for _ in range(3):
                once()
            ts = [once() for _ in range(max(3, min(args.steps, 10)))]
            el = statistics.median(ts)
            out[f"tp{tp}/{tokens // 1024}k"] = {
                "ms": round(el * 1e3, 3), "host_read_gbs": round(nbytes / el / GB, 1),
                "device_write_gbs": round(tp * nbytes / el / GB, 1),
                "host_bytes_per_rank": nbytes // tp}
            if tp == 1:
                # the plain pipelined load of the same pages, timed the same way (two
                # cross-stream hops around the launch), for comparison with tp = 1
                for _ in range(3):
                    once(plain=True)
                el = statistics.median([once(plain=True) for _ in range(max(3, min(args.steps, 10)))])
                out[f"pipelined/{tokens // 1024}k"] = {"ms": round(el * 1e3, 3),
                                                       "host_read_gbs": round(nbytes / el / GB, 1)}
        for p in pools:
            p.close()
        del bufs, kvs
        torch.cuda.empty_cache()
    mem.free()
    return out


def bench_nsa_group(torch, hc, args):
    """A buffer group: an MLA latent (576 bf16) beside an fp8 indexer key (128)
    and its fp32 scales (4 per row), 61 layers, page 64, three page_first pools
    carved from one pinned allocation.  Loads of 4K / 16K / 64K tokens, every
    layer and layer by layer: one launch per pool vs one group launch, the
    pipelined group load (every layer of every pool in one launch, each
    pool's layers signalled as they land), and a group plan's per-layer
    launches replayed from one CUDA graph (its first, capturing call is a
    warm-up), and one chained call per layer (each layer's group launch
    starting as the previous layer's drains).  Each
    variant is enqueued behind a sleep kernel on a gate stream, so the device
    time excludes the host's enqueue cost, which is reported beside it."""
    from tiered_kv_cache_gb300 import workloads as wl
    s = wl.MLA_LATENT
    L, P, Dp, Hp = s.num_layers, s.page_size, s.device_pages, s.host_pages
    kinds = [(576, 2), (128, 1), (4, 4)]
    sizes = [L * Hp * P * R * es for R, es in kinds]
    mem = hc.PinnedHost(sum(sizes))
    pools, kvs, keep, off = [], [], [], 0
    g = torch.Generator(device="cuda")
    g.manual_seed(s.seed)
    for (R, es), nbytes in zip(kinds, sizes):
        pools.append(hc.Pool(L, 1, P, R, Hp, "page_first", elem_bytes=es, host_ptr=mem.ptr + off,
                             host_bytes=nbytes, launch_ctas=args.ctas))
        bufs = [torch.randint(0, 256, (Dp * P, R * es), dtype=torch.uint8, device="cuda", generator=g)
                for _ in range(L)]
        keep.append(bufs)
        kvs.append(hc.DeviceKV(bufs, Dp))
        off += nbytes
    page_bytes = sum(L * P * R * es for R, es in kinds)
    gate, stream = torch.cuda.Stream(), torch.cuda.Stream()
    launches0 = hc.launch_count()

    def gated(fn):
        dev, host = [], []
        for it in range(max(args.warmup, 3) + args.steps):
            torch.cuda.synchronize()
            with torch.cuda.stream(gate):
                torch.cuda._sleep(int(4e7))        # ~20 ms: longer than any enqueue below
            e0 = torch.cuda.Event(enable_timing=True)
            e0.record(gate)
            stream.wait_event(e0)
            h0 = time.perf_counter()
            fn()
            h1 = time.perf_counter()
            e1 = torch.cuda.Event(enable_timing=True)
            e1.record(stream)
            torch.cuda.synchronize()
            if it >= max(args.warmup, 3):
                dev.append(_elapsed(torch, e0, e1))
                host.append(h1 - h0)
        return statistics.median(dev), statistics.median(host)

    out = {}
    for tokens in (4096, 16384, 65536):
        t = wl.mla_transfer(s, tokens)
        dp, hp = t.device_pages, t.host_pages
        nbytes = len(dp) * page_bytes
        variants = {
            "per_layer_per_pool": lambda: [pool.load_layer(kv, dp, hp, layer, stream=stream)
                                           for layer in range(L) for pool, kv in zip(pools, kvs)],
            "per_layer_group": lambda: [hc.group_transfer(pools, kvs, dp, hp, hc.LOAD, layer=layer,
                                                          stream=stream) for layer in range(L)],
            "all_layers_per_pool": lambda: [pool.load(kv, dp, hp, stream=stream) for pool, kv in zip(pools, kvs)],
            "all_layers_group": lambda: hc.group_transfer(pools, kvs, dp, hp, hc.LOAD, stream=stream),
            "pipelined_group": lambda: hc.group_load_pipelined(pools, kvs, dp, hp, stream=stream),
            "per_layer_group_graph": lambda: plan.load_layers(kvs, stream=stream),
            "per_layer_group_chained": lambda: [plan.load_layer_chained(kvs, layer, stream=stream)
                                                for layer in range(L)],
        }
        plan = hc.group_plan(pools, dp, hp, Dp)
        r = {"pages": len(dp), "bytes": nbytes}
        for name, fn in variants.items():
            d, h = gated(fn)
            r[name] = {"device_ms": round(d * 1e3, 3), "gbs": round(nbytes / d / GB, 1),
                       "host_enqueue_ms": round(h * 1e3, 3)}
        plan.close()
        out[f"{tokens // 1024}k"] = r
    launches = hc.launch_count() - launches0
    for pool in pools:
        pool.close()
    del keep
    return out, launches


def bench_shapes(torch, hc, args):
    """Row size x page size sweep: about 1 GiB per call of fully scattered
    device pages (a permutation) and contiguous host pages, 8 layers, K+V, one
    byte per element, load and backup in layer_first and page_first.  Short
    rows at small page sizes give many short runs: the case where tiles span
    runs and the host pre-pass is linear in the pages."""
    st = torch.cuda.Stream()

    def timed(fn, n=5):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        out = []
        for _ in range(n):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(st)
            fn()
            e1.record(st)
            torch.cuda.synchronize()
            out.append(_elapsed(torch, e0, e1))
        return statistics.median(out)

    L, B = 8, 2
    res = []
    for row_bytes in (256, 1152, 2048):
        for P in (1, 16, 64):
            page_bytes = B * L * P * row_bytes
            n = (1 << 30) // page_bytes
            bufs = [torch.empty((n * P, row_bytes), dtype=torch.uint8, device="cuda") for _ in range(B * L)]
            kv = hc.DeviceKV(bufs, n)
            rng = np.random.default_rng(0)
            dp, hp = rng.permutation(n), np.arange(n)
            r = {"row_bytes": row_bytes, "page_size": P, "pages": n}
            for lay, name in ((0, "layer_first"), (1, "page_first")):
                with hc.Pool(L, B, P, row_bytes, n, lay, elem_bytes=1, launch_ctas=args.ctas) as pool:
                    nb = n * page_bytes
                    r[f"load_{name}_gbs"] = round(nb / timed(lambda: pool.load(kv, dp, hp, stream=st)) / GB, 1)
                    r[f"backup_{name}_gbs"] = round(nb / timed(lambda: pool.backup(kv, dp, hp, stream=st)) / GB, 1)
            res.append(r)
            del bufs, kv
            torch.cuda.empty_cache()
    return res


def bench_small_mix(torch, hc, args, link=None):
    """10,000 seeded requests, 1-256 pages log-uniform, 30% backup / 70% load,
    random pages, layer_first.  Per-call latency = host wall clock from the API
    call until the stream is idle; aggregate GB/s without per-call waits, on one
    stream and through the submission engine.  With the link peaks given, the
    one-stream ceiling is each direction's bytes at its own peak, one after the
    other: total / (backup bytes / D2H peak + load bytes / H2D peak)."""
    from tiered_kv_cache_gb300 import workloads as wl
    s = wl.SMALL_MIX
    vals = [v.view(torch.int16) for v in wl.kv_values(s, device="cuda")]
    kv = hc.DeviceKV(vals, s.device_pages)
    pool = hc.Pool(s.num_layers, s.num_buffers, s.page_size, s.row_elems, s.host_pages, "layer_first",
                   launch_ctas=args.ctas)
    reqs = wl.small_mix_requests(s)
    st = torch.cuda.Stream()
    handle = st.cuda_stream

    def call(r):
        if r.direction == "backup":
            pool.backup(kv, r.device_pages, r.host_pages, stream=handle)
        else:
            pool.load(kv, r.device_pages, r.host_pages, stream=handle)

    for r in reqs[:200]:
        call(r)
    hc.wait(handle)
    lat, submit = [], []
    launches0 = hc.launch_count()
    for r in reqs:
        t0 = time.perf_counter()
        call(r)
        t1 = time.perf_counter()
        hc.wait(handle)
        t2 = time.perf_counter()
        submit.append(t1 - t0)
        lat.append(t2 - t0)
    per_call_launches = (hc.launch_count() - launches0) / len(reqs)
    total = sum(len(r.device_pages) for r in reqs) * s.page_bytes
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    e0.record(st)
    for r in reqs:
        call(r)
    e1.record(st)
    hc.wait(handle)
    wall = time.perf_counter() - t0
    dev = _elapsed(torch, e0, e1)
    # the same requests through the submission engine: its worker fuses a backup
    # and a load that commute into one launch, on the engine's own stream
    with hc.Engine(pool) as eng:
        l0, f0 = eng.stats()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        last = 0
        for r in reqs:
            last = eng.submit(kv, r.device_pages, r.host_pages,
                              hc.BACKUP if r.direction == "backup" else hc.LOAD)
        eng.wait(last)
        wall_engine = time.perf_counter() - t0
        l1, f1 = eng.stats()
    lat_us = np.array(lat) * 1e6
    sub_us = np.array(submit) * 1e6
    sizes = np.array([len(r.device_pages) for r in reqs])

    def pct(a, q):
        return round(float(np.percentile(a, q)), 1)
    by_size = {}
    for lo, hi in ((1, 4), (5, 64), (65, 256)):
        m = (sizes >= lo) & (sizes <= hi)
        by_size[f"{lo}-{hi}_pages"] = {"calls": int(m.sum()), "p50_us": pct(lat_us[m], 50),
                                       "p99_us": pct(lat_us[m], 99)}
    out = {"requests": len(reqs), "bytes": total,
           "latency_p50_us": pct(lat_us, 50), "latency_p99_us": pct(lat_us, 99),
           "submit_p50_us": pct(sub_us, 50), "submit_p99_us": pct(sub_us, 99),
           "latency_by_size": by_size, "launches_per_call": per_call_launches,
           "aggregate_gbs_device": round(total / dev / GB, 1),
           "aggregate_gbs_wall": round(total / wall / GB, 1),
           "aggregate_gbs_engine_wall": round(total / wall_engine / GB, 1),
           "engine_launches": l1 - l0, "engine_fused_launches": f1 - f0}
    if link and link.get("h2d_gbs") and link.get("d2h_gbs"):
        back = sum(len(r.device_pages) for r in reqs if r.direction == "backup") * s.page_bytes
        ceiling = total / (back / (link["d2h_gbs"] * GB) + (total - back) / (link["h2d_gbs"] * GB)) / GB
        out["one_stream_ceiling_gbs"] = round(ceiling, 1)
        out["aggregate_device_frac_of_ceiling"] = frac(total / dev / GB, ceiling)
    pool.close()
    return out


def bench_host_alloc(torch, hc, args):
    """Host pool allocation, plain cudaHostAlloc vs mmap + MADV_HUGEPAGE +
    cudaHostRegister, at two pool sizes: time to allocate and pin, and the
    backup / load rate of 512 Llama-3-8B pages whose host pages are scattered
    over the whole pool (the case where host address translation is stressed)."""
    from tiered_kv_cache_gb300 import workloads as wl
    s = wl.LLAMA3_8B
    vals = [v.view(torch.int16) for v in wl.kv_values(s, device="cuda")]
    kv = hc.DeviceKV(vals, s.device_pages)
    st = torch.cuda.Stream()
    rng = np.random.default_rng(9)
    dp = wl.fragmented_pages(rng, s.device_pages, 512)
    out = {}
    for gib in (16, 64):
        hp_pages = gib * 2**30 // s.page_bytes
        hp = np.sort(rng.choice(hp_pages, 512, replace=False))
        for thp in (False, True):
            t0 = time.perf_counter()
            mem = hc.PinnedHost(hp_pages * s.page_bytes, thp=thp)
            t_alloc = time.perf_counter() - t0
            pool = hc.Pool(s.num_layers, s.num_buffers, s.page_size, s.row_elems, hp_pages, "layer_first",
                           host_ptr=mem.ptr, host_bytes=mem.nbytes, launch_ctas=args.ctas)
            rates = {}
            for name, fn in (("backup", pool.backup), ("load", pool.load)):
                for lay in (0, 2):
                    for _ in range(2):
                        fn(kv, dp, hp, lay, stream=st)
                    ts = []
                    for _ in range(max(3, args.steps)):
                        e0 = torch.cuda.Event(enable_timing=True)
                        e1 = torch.cuda.Event(enable_timing=True)
                        e0.record(st)
                        fn(kv, dp, hp, lay, stream=st)
                        e1.record(st)
                        st.synchronize()
                        ts.append(_elapsed(torch, e0, e1))
                    rates[f"{name}_{'lf' if lay == 0 else 'pfd'}_gbs"] = round(
                        512 * s.page_bytes / statistics.median(ts) / GB, 1)
            pool.close()
            t0 = time.perf_counter()
            mem.free()
            t_free = time.perf_counter() - t0
            out[f"{gib}GiB_{'thp_mmap_register' if thp else 'cudaHostAlloc'}"] = {
                "alloc_pin_s": round(t_alloc, 2), "alloc_pin_gbs": round(gib * 2**30 / t_alloc / GB, 1),
                "free_s": round(t_free, 2), **rates}
    return out


def bench_engine_bidir(torch, hc, args):
    """The pages' submitter design: a backup thread and a load thread, each
    moving 512-page requests (Llama-3-8B shape) back to back.  (a) each thread
    calls the library directly on its own stream; (b) both submit to one
    engine, which fuses adjacent backup/load pairs.  Host wall clock from the
    first submission to the last completion."""
    import threading
    w = build_workload("cuda", 512, args.ctas)
    pool, kv = w["pool"], w["kv"]
    reps = max(6, args.steps)
    bpx = w["bytes_per_xfer"]
    out = {}

    def run_direct():
        sb, sl = torch.cuda.Stream(), torch.cuda.Stream()

        def backups():
            for _ in range(reps):
                pool.backup(kv, w["a_dev"], w["a_host"], stream=sb)
            hc.wait(sb)

        def loads():
            for _ in range(reps):
                pool.load(kv, w["b_dev"], w["b_host"], stream=sl)
            hc.wait(sl)
        ts = [threading.Thread(target=backups), threading.Thread(target=loads)]
        t0 = time.perf_counter()
        for t in ts:
            t.start()
        for t in ts:
            t.join()
        return time.perf_counter() - t0

    def run_engine(eng):
        last = {}

        def submit(name, direction, dev, host):
            for _ in range(reps):
                last[name] = eng.submit(kv, dev, host, direction)
        ts = [threading.Thread(target=submit, args=("b", hc.BACKUP, w["a_dev"], w["a_host"])),
              threading.Thread(target=submit, args=("l", hc.LOAD, w["b_dev"], w["b_host"]))]
        t0 = time.perf_counter()
        for t in ts:
            t.start()
        for t in ts:
            t.join()
        for t in last.values():
            eng.wait(t)
        return time.perf_counter() - t0

    run_direct()
    direct = min(run_direct() for _ in range(3))
    with hc.Engine(pool) as eng:
        run_engine(eng)
        l0, f0 = eng.stats()
        eng_t = min(run_engine(eng) for _ in range(3))
        l1, f1 = eng.stats()
    moved = 2 * reps * bpx
    out["direct_two_streams_gbs"] = round(moved / direct / GB, 1)
    out["engine_gbs"] = round(moved / eng_t / GB, 1)
    out["engine_fused_fraction"] = round((f1 - f0) / max(1, l1 - l0), 3)
    out["requests_per_thread"] = reps
    pool.close()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ctas", type=int, default=0, help="CTAs per transfer launch (0 = automatic)")
    ap.add_argument("--pages", type=int, default=512,
                    help="pages per transfer (512 = the 32K-token workload; smaller for profiling)")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the other workload shapes that the default run measures after the step")
    ap.add_argument("--no-link-probe", action="store_true",
                    help="skip the cudaMemcpyAsync host-link probe (profiling runs)")
    ap.add_argument("--workload", default="llama3_8b_32k",
                    choices=["llama3_8b_32k", "deep78_32k", "mla61_overlap", "small_mix", "host_alloc",
                             "engine_bidir", "nsa_group", "shapes", "tp_mla61"],
                    help="llama3_8b_32k is the headline step; the others measure the remaining "
                         "workload shapes")
    ap.add_argument("--tokens", default="",
                    help="mla61_overlap only: comma-separated load sizes in tokens (default 4096,16384,65536 "
                         "and the same with a high-priority transfer stream)")
    ap.add_argument("--layouts", default="pages",
                    help="'pages' (layer_first, page_first, page_first_direct) or 'all' (adds "
                         "page_first_direct_kv)")
    args = ap.parse_args()
    if args.layouts == "all":
        LAYOUT_NAMES.append("page_first_direct_kv")
    if args.impl == "reference":
        return reference_arm(args)

    import torch
    import tiered_kv_cache_gb300 as hc
    from tiered_kv_cache_gb300 import build as hc_build

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    hc_build.build()
    peaks, peaks_src = measured_peaks()

    if args.no_link_probe:
        link = {"h2d_gbs": None, "d2h_gbs": None, "bidir_gbs": None, "how": "skipped"}
    else:
        link = link_peaks(torch, hc=hc)
    if args.workload in ("mla61_overlap", "small_mix", "host_alloc", "engine_bidir", "nsa_group", "shapes",
                         "tp_mla61"):
        t0 = time.perf_counter()
        if args.workload == "tp_mla61":
            res = bench_tp_mla(torch, hc, args)
            launches = None
            value = res["tp8/64k"]["host_read_gbs"]
            what = {"workload": "tp_mla61: tensor-parallel load of the MLA latent (61 layers, 576 bf16, page "
                                "64, page_first), tp = 1/2/4/8 ranks stood in for by pools on one GPU over one "
                                "host memory; each rank reads 1/tp of the pages and stores them into every "
                                "rank's buffers; 4K/16K/64K tokens",
                    "value": "host-read GB/s of the whole group at tp = 8, 64K tokens (one GPU: the ranks "
                             "share one host link)"}
        elif args.workload == "shapes":
            res = bench_shapes(torch, hc, args)
            launches = None
            value = next(r["load_layer_first_gbs"] for r in res if r["row_bytes"] == 1152 and r["page_size"] == 1)
            what = {"workload": "shapes: rows of 256 / 1152 / 2048 bytes x page sizes 1 / 16 / 64, 8 layers, "
                                "K+V, about 1 GiB per call of fully scattered device pages, contiguous host",
                    "value": "load GB/s, layer_first, 1152-byte rows, page size 1"}
        elif args.workload == "nsa_group":
            res, launches = bench_nsa_group(torch, hc, args)
            value = res["4k"]["per_layer_group"]["gbs"]
            what = {"workload": "nsa_group: 61 layers, page 64, page_first; an MLA latent (576 bf16), an fp8 "
                                "indexer key (128) and fp32 scales (4) as three pools of one pinned "
                                "allocation; 4K/16K/64K-token loads, per layer and every layer, one launch "
                                "per pool vs one group launch; device time behind a gate stream",
                    "value": "GB/s of the 61 per-layer group loads at 4K tokens"}
        elif args.workload == "engine_bidir":
            res = bench_engine_bidir(torch, hc, args)
            launches = None
            value = res["engine_gbs"]
            what = {"workload": "engine_bidir: a backup thread and a load thread, 512-page Llama-3-8B requests "
                                "back to back, direct on two streams vs one submission engine",
                    "value": "GB/s through the engine, both directions"}
        elif args.workload == "host_alloc":
            res = bench_host_alloc(torch, hc, args)
            launches = None
            value = res["64GiB_cudaHostAlloc"]["load_lf_gbs"]
            what = {"workload": "host pool allocation: cudaHostAlloc vs mmap+MADV_HUGEPAGE+cudaHostRegister, "
                                "16 and 64 GiB pools; 512 Llama-3-8B pages scattered over the pool",
                    "value": "load GB/s, layer_first, 64 GiB cudaHostAlloc pool"}
        elif args.workload == "mla61_overlap":
            res, launches = bench_mla_overlap(torch, hc, args)
            value = (res.get("64k") or next(iter(res.values())))["per_layer_load_gbs"]
            what = {"workload": "mla61: 61 layers, one latent buffer, kv_dim 576, bf16, page 64, "
                                "page_first host pool; 4K/16K/64K-token per-layer loads with an "
                                "event per layer and a stand-in attention kernel on a second stream",
                    "value": "GB/s of the 61 per-layer loads at 64K tokens"}
        else:
            res = bench_small_mix(torch, hc, args, link)
            launches = int(res["launches_per_call"] * res["requests"])
            value = res["aggregate_gbs_device"]
            what = {"workload": "small_mix: 32 layers, K+V, 8 kv heads x 128, page 16, 10,000 requests "
                                "of 1-256 pages (log-uniform), 30% backup, layer_first",
                    "value": "aggregate GB/s without per-call waits"}
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
                              "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
                              "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                              "config": what, "results": res, "gpu_launches": launches,
                              "link_peak": link, "wall_s": round(time.perf_counter() - t0, 1)}),
                  flush=True)
        return
    w = build_workload("cuda", args.pages, args.ctas, args.workload)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(max(args.warmup, 3)):
        run_step(torch, w, s1, s2)
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    # ---- timed region (device clock) --------------------------------------
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier()
    launches0 = hc.launch_count()
    ev = []
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(s1)
    for _ in range(args.steps):
        run_step(torch, w, s1, s2, ev)
    t_end.record(s1)
    barrier()
    launches = hc.launch_count() - launches0
    clk = clocks.stop()
    elapsed = max_over_ranks(t_start.elapsed_time(t_end) / 1e3, world)
    bpx = w["bytes_per_xfer"]
    step_bytes = len(LAYOUT_NAMES) * 6 * bpx
    npages = w["pages"]
    value = whole_job_gbs(args.steps * step_bytes, elapsed, world)

    per, breakdown = breakdown_from_events(ev, bpx, link)
    # dominant single-direction kernel: the largest total time
    singles = {k: sum(v) for k, v in per.items() if "bidir" not in k}
    dom = max(singles, key=singles.get)
    dom_avg = statistics.mean(per[dom])
    achieved = bpx / dom_avg / GB
    dom_peak = link["d2h_gbs"] if dom.endswith("backup") else link["h2d_gbs"]
    rec = recorded_traffic()
    traffic = rec.get(f"{dom} dram_bytes_per_page")
    link_traffic = rec.get(f"{dom} c2c_bytes_per_page")
    roofline = {"bound": "host_link", "kernel": f"xfer_kernel ({dom})", "achieved": round(achieved, 1),
                "peak": round(dom_peak, 1) if dom_peak else None, "unit": "GB/s",
                "frac": frac(achieved, dom_peak),
                "traffic": int(traffic) * npages if traffic else None,
                "traffic_c2c": int(link_traffic) * npages if link_traffic else None,
                "traffic_source": "ncu dram__bytes_read+write (and ctc__*_bytes_data_user) of a 64-page "
                                  "capture, scaled per page; null when that kernel was not captured or "
                                  "its source changed since" ,
                "peak_source": "in-run pinned cudaMemcpyAsync of 1 GiB, same direction (no host-link "
                               "figure in MEASURED_PEAKS.json)",
                "binding_resource": binding_resource(link),
                "bytes_per_launch": bpx, "avg_launch_ms": round(dom_avg * 1e3, 3)}
    # device side of the same kernel: the payload crosses HBM once
    hbm_peak = float(peaks.get("hbm_gbs", 6800.0))
    roofline_hbm = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                    "frac": round(achieved / hbm_peak, 4),
                    "peak_source": f"{peaks_src} hbm_gbs (of measured)" if peaks_src != "fallback" else "fallback"}

    # ---- end to end through the public API, host wall clock -----------------
    torch.cuda.synchronize()
    e2e_steps = max(2, args.steps // 2)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        run_step(torch, w, s1, s2)
        hc.wait(s1)
    e2e_t = time.perf_counter() - t0
    e2e = {"value": round(world * e2e_steps * step_bytes / e2e_t / GB, 1), "unit": "GB/s",
           "h2d_bytes_per_step": len(LAYOUT_NAMES) * 3 * bpx + len(LAYOUT_NAMES) * 6 * npages * 16,
           "d2h_bytes_per_step": len(LAYOUT_NAMES) * 3 * bpx,
           "how": "host wall clock around the Python API calls (validation, pre-pass, launch) and a "
                  "host wait on the stream each step; host-index bytes counted as H2D"}

    out = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": round(elapsed / args.steps * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": step_config(args, npages, bpx),
        "roofline": roofline,
        "roofline_hbm": roofline_hbm,
        "link_peak": {**{k: round(v, 1) if isinstance(v, float) else v for k, v in link.items()}, **NOMINAL},
        "breakdown": breakdown,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clk,
    }
    w["pool"].close()
    del w
    torch.cuda.empty_cache()
    # the other workload shapes, on the single-GPU run only (under torchrun every
    # rank would pin its own copy of the larger pools at the same time)
    if not args.no_extras and world == 1 and args.workload == "llama3_8b_32k" and args.pages == 512:
        out["workloads"] = bench_extras(torch, hc, args, link)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline()
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
