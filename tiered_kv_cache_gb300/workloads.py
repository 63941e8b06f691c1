"""Seeded synthetic workloads for the L1 <-> L2 KV movement.

This module only draws random numbers: page-index patterns, request mixes and KV
values.  It holds none of the copy's arithmetic (no offsets, no layouts), so the
tests, the benchmark and the CPU oracle can all take their inputs from here
without sharing any part of the method.

The five shapes stand in for the pages' workloads (GLM5-class 78-layer MLA
models, 24K-64K token prefixes, multi-turn agent traffic): the datasets and
model weights themselves are not available, so values are random bf16 and
indices follow the allocator patterns described with each workload.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


@dataclass(frozen=True)
class KVShape:
    name: str
    num_layers: int          # L
    num_buffers: int         # B: 2 = K,V ; 1 = MLA latent
    row_elems: int           # R: kv heads * head_dim, or kv_dim
    page_size: int           # P
    device_pages: int        # Dp
    host_pages: int          # Hp
    elem_bytes: int = 2      # bf16
    value_dist: str = "normal"   # "normal" or "uniform" (uniform[-1, 1])
    seed: int = 0

    @property
    def row_bytes(self) -> int:
        return self.row_elems * self.elem_bytes

    @property
    def page_bytes(self) -> int:
        """Bytes of one page across every buffer and layer (one direction)."""
        return self.num_buffers * self.num_layers * self.page_size * self.row_bytes

    def page_layer_bytes(self) -> int:
        return self.num_buffers * self.page_size * self.row_bytes

    def host_pool_bytes(self) -> int:
        return self.host_pages * self.page_bytes

    def device_buffer_elems(self) -> int:
        return self.device_pages * self.page_size * self.row_elems


TINY_GQA = KVShape("tiny_gqa", num_layers=2, num_buffers=2, row_elems=2 * 64, page_size=16,
                   device_pages=64, host_pages=128, value_dist="uniform", seed=1)
LLAMA3_8B = KVShape("llama3_8b_32k", num_layers=32, num_buffers=2, row_elems=8 * 128,
                    page_size=64, device_pages=1024, host_pages=1024, seed=2)
DEEP_STRESS = KVShape("deep78_32k", num_layers=78, num_buffers=2, row_elems=8 * 128,
                      page_size=64, device_pages=1024, host_pages=1024, seed=3)
MLA_LATENT = KVShape("mla61", num_layers=61, num_buffers=1, row_elems=512 + 64,
                     page_size=64, device_pages=1024, host_pages=2048, seed=4)
SMALL_MIX = KVShape("small_mix", num_layers=32, num_buffers=2, row_elems=8 * 128,
                    page_size=16, device_pages=2048, host_pages=4096, seed=5)

SHAPES = {s.name: s for s in (TINY_GQA, LLAMA3_8B, DEEP_STRESS, MLA_LATENT, SMALL_MIX)}


def index_rng(seed: int) -> np.random.Generator:
    """Generator for page indices: seed + 100, so values and indices never share
    a stream."""
    return np.random.default_rng(seed + 100)


def distinct_pages(rng: np.random.Generator, pool_pages: int, n: int) -> np.ndarray:
    """n distinct pages drawn uniformly from [0, pool_pages)."""
    return rng.choice(pool_pages, size=n, replace=False).astype(np.int64)


def scattered_pages(rng: np.random.Generator, pool_pages: int, n: int) -> np.ndarray:
    """Fully scattered: the first n of a random permutation of the pool."""
    return rng.permutation(pool_pages)[:n].astype(np.int64)


def fragmented_pages(rng: np.random.Generator, pool_pages: int, n: int,
                     max_run: int = 8, exclude: np.ndarray | None = None) -> np.ndarray:
    """Pages from a fragmented allocator: [0, pool_pages) is cut into chunks of
    random length 1..max_run, the chunks are shuffled, and pages are taken chunk
    by chunk until n pages are collected (the last chunk is cut short).  Pages in
    ``exclude`` are dropped first, which keeps two requests disjoint."""
    keep = np.ones(pool_pages, dtype=bool)
    if exclude is not None and len(exclude):
        keep[np.asarray(exclude, dtype=np.int64)] = False
    chunks = []
    start = 0
    while start < pool_pages:
        ln = int(rng.integers(1, max_run + 1))
        chunks.append(np.arange(start, min(start + ln, pool_pages)))
        start += ln
    order = rng.permutation(len(chunks))
    out = []
    total = 0
    for k in order:
        c = chunks[k][keep[chunks[k]]]
        if total + len(c) > n:
            c = c[: n - total]
        out.append(c)
        total += len(c)
        if total >= n:
            break
    res = np.concatenate(out).astype(np.int64) if out else np.zeros(0, np.int64)
    if len(res) < n:
        raise ValueError("pool too small for the requested pages")
    return res


def contiguous_pages(n: int, start: int = 0) -> np.ndarray:
    return np.arange(start, start + n, dtype=np.int64)


@dataclass
class Request:
    direction: str            # "backup" or "load"
    device_pages: np.ndarray
    host_pages: np.ndarray


def small_mix_requests(shape: KVShape = SMALL_MIX, count: int = 10_000,
                       max_pages: int = 256, backup_frac: float = 0.3,
                       seed: int | None = None) -> list[Request]:
    """Multi-turn mix: sizes log-uniform over [1, max_pages] pages
    (n = min(max_pages, floor(exp(u ln(max_pages+1)))), u ~ U[0,1)), each a
    backup with probability backup_frac, else a load, with random distinct pages
    on both sides."""
    rng = index_rng(shape.seed if seed is None else seed)
    reqs = []
    for _ in range(count):
        u = rng.random()
        n = int(min(max_pages, np.floor(np.exp(u * np.log(max_pages + 1)))))
        n = max(n, 1)
        direction = "backup" if rng.random() < backup_frac else "load"
        dp = distinct_pages(rng, shape.device_pages, n)
        hp = distinct_pages(rng, shape.host_pages, n)
        reqs.append(Request(direction, dp, hp))
    return reqs


def kv_values(shape: KVShape, device: str = "cpu", num_pages: int | None = None):
    """B*L bf16 tensors of shape (pages*P, R), buffer-major (K layers then V
    layers), drawn from torch's generator seeded with the workload's seed:
    normal(0, 1) or uniform[-1, 1]."""
    import torch

    pages = shape.device_pages if num_pages is None else num_pages
    g = torch.Generator(device=device)
    g.manual_seed(shape.seed)
    rows = pages * shape.page_size
    bufs = []
    for _ in range(shape.num_buffers * shape.num_layers):
        if shape.value_dist == "uniform":
            x = torch.rand((rows, shape.row_elems), generator=g, device=device,
                           dtype=torch.float32).mul_(2).sub_(1).to(torch.bfloat16)
        else:
            x = torch.randn((rows, shape.row_elems), generator=g, device=device,
                            dtype=torch.bfloat16)
        bufs.append(x)
    return bufs


@dataclass
class Transfer:
    """One transfer of a workload: device pages paired with host pages."""
    device_pages: np.ndarray
    host_pages: np.ndarray
    extra: dict = field(default_factory=dict)


def llama_transfer(shape: KVShape = LLAMA3_8B, n: int = 512, shuffled_host: bool = False,
                   seed: int | None = None) -> Transfer:
    rng = index_rng(shape.seed if seed is None else seed)
    dp = fragmented_pages(rng, shape.device_pages, n)
    hp = scattered_pages(rng, shape.host_pages, n) if shuffled_host else contiguous_pages(n)
    return Transfer(dp, hp)


def deep_bidir_transfers(shape: KVShape = DEEP_STRESS, n: int = 512,
                         seed: int | None = None) -> tuple[Transfer, Transfer]:
    """Request A (backed up) and request B (loaded) of equal size: fully
    scattered, disjoint device pages; contiguous, disjoint host pages."""
    rng = index_rng(shape.seed if seed is None else seed)
    perm = rng.permutation(shape.device_pages).astype(np.int64)
    a = Transfer(perm[:n], contiguous_pages(n, 0))
    b = Transfer(perm[n:2 * n], contiguous_pages(n, n))
    return a, b


def mla_transfer(shape: KVShape = MLA_LATENT, tokens: int = 16384,
                 seed: int | None = None) -> Transfer:
    n = tokens // shape.page_size
    rng = index_rng(shape.seed if seed is None else seed)
    dp = fragmented_pages(rng, shape.device_pages, n)
    return Transfer(dp, contiguous_pages(n))
