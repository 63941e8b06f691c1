// hicache_kernels.cu -- sm_103a transfer kernels for the L1 <-> L2 KV movement.
//
// One tile mover serves backup (device -> host) and load (host -> device) for
// the four host layouts, for every layer at once or for one layer, in every
// kernel here: one direction, both directions fused, a pipelined load that
// signals each layer as it lands, and the same for a group of pools:
//
//   * The pre-pass (host side) sorts the index pairs by host page and merges
//     pages that are consecutive on BOTH sides into runs.  The run table and
//     the B*L device-buffer pointers travel in the kernel parameters, so a
//     call of up to 1536 runs (more with fewer buffers) is exactly one launch
//     and no descriptor or per-segment submission ever reaches the GPU.  (The
//     pages trace the cost of page_first_direct to one DMA descriptor per
//     page x layer segment: "Tuning SGLang HiCache L2 on Kunlunxin P800/P900",
//     sections 2.1 and 2.3; "Baidu's KVCache Overhaul", section "DMA Segment
//     Explosion & Batched Gather/Scatter".  Here every segment boundary is just
//     address arithmetic inside a warp.)
//   * The work is cut into "units" that are contiguous on the HOST side:
//       layer_first, any layer count      unit = (buffer, layer, run)
//       page_first(_direct), all layers   unit = (buffer, run): all layers of
//                                         the run's pages are one host range
//       page_first(_direct), one layer    unit = (buffer, run), host strided
//       page_first_direct_kv, all layers  unit = run: every buffer and layer of
//                                         the run's pages is one host range
//     The units of one outer index (a buffer, a buffer-layer, or everything)
//     lie end to end in one vector range, cut into tiles of 16 KiB (1024
//     vectors of 16 bytes); a tile spans several units where runs are short,
//     so short runs still fill whole tiles.  CTAs take tiles in host-address
//     order (grid-stride), so the host link sees long sequential streams of
//     whole 128-byte lines in every layout.
//   * Each thread of a tile moves 4 independent 16-byte vectors: 4 loads in
//     flight before the first store.  The device-side address of every vector
//     is decoded on the fly (a multiply-high division per dimension), which
//     performs the layout transpose without a shared-memory pass: rows are
//     >= 16 bytes, so each warp's device accesses stay whole 32-byte sectors,
//     and the host side is touched strictly in order.
//
//   * The launches of one call (a run table larger than one parameter block,
//     or the layers of a per-layer graph) overlap: each after the first is a
//     programmatic dependent launch that starts once every CTA of the one
//     before it is on its last tile, so the link does not idle between them.
//
// No tensor cores: nothing here is a contraction.  No TMA multicast, no
// cross-CTA waits, no spin loops: a kernel always runs to completion.  The one
// wait is griddepcontrol.wait at the end of a programmatically launched
// kernel, for the launch before it, which was already running and waits on
// nothing later.

#include <cuda_runtime.h>

#include <mutex>
#include <type_traits>

#include "hicache_internal.h"

namespace hicache {
namespace {

// Streaming (evict-first) 16-byte accesses: every byte is touched once.
__device__ __forceinline__ uint4 ld_stream(const uint4 *p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(uint4 *p, const uint4 &v) { __stcs(p, v); }

// Programmatic dependent launch.  Each CTA allows the next launch on the
// stream on reaching its last tile.  Consecutive launches of one call (a run
// table larger than one parameter block, or one layer after another in a
// per-layer graph) move disjoint destinations, so the next starts work while
// this one drains.  A launch started that way finishes only after the one
// before it has (the wait at the end of the kernel), so whatever follows the
// call on the stream still sees every launch of it complete.  The first
// launch of a one-layer load is programmatic as well, behind work it may
// depend on: it waits for that work before touching memory (wait_previous),
// which keeps plain stream order and hides only the launch itself.  The waits
// are no-ops for a kernel launched plainly.
__device__ __forceinline__ void allow_next_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void finish_after_previous_launch() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

#ifndef HICACHE_CHECKED
#define HICACHE_CHECKED 0
#endif

// Bounds-checked builds: the first failed check (bit 63 set, the check's kind
// in bits 60-62, the offending value in bits 0-59) and the number of failed
// checks, since the host last cleared them.
__device__ unsigned long long g_check_words[2];

__device__ __forceinline__ void report_check(int32_t kind, int64_t value) {
  const unsigned long long code = (1ull << 63) | (static_cast<unsigned long long>(kind & 7) << 60) |
                                  (static_cast<unsigned long long>(value) & ((1ull << 60) - 1));
  atomicCAS(&g_check_words[0], 0ull, code);
  atomicAdd(&g_check_words[1], 1ull);
}

// Address of vector w of the current unit.  `dev` and `host` receive vector
// pointers; b, l, run describe the unit (l is ignored where the unit spans all
// layers).  Each layout gives the device buffer index, the vector offset in
// that buffer and the vector offset in the host pool; a bounds-checked build
// checks the three against their extents and gives null pointers (and records
// the failure) instead of an address outside them.
template <int LAYOUT, bool ALL>
__device__ __forceinline__ void map_vector(const XferHeader &h, uint4 *const *bufs, int b, int l,
                                           const Run &r, uint32_t w, uint4 *&dev, uint4 *&host) {
  int64_t bi, doff, hoff;
  if (LAYOUT == kLayerFirst) {
    // host (B, L, size, R): unit (b, l, run) is contiguous on both sides
    bi = b * h.L + l;
    doff = int64_t(r.d0) * h.PV + w;
    hoff = (int64_t(b * h.L + l) * h.Hp + r.h0) * h.PV + w;
  } else if (LAYOUT == kPageFirstDirect && ALL) {
    // host (B, Hp, L, P, R): the unit is [page j][layer ll][token, elem]
    const uint32_t j = fast_div(w, h.fd_LPV);
    const uint32_t rem = w - j * h.LPV;
    const uint32_t ll = fast_div(rem, h.fd_PV);
    const uint32_t q = rem - ll * h.PV;
    bi = b * h.L + int32_t(ll);
    doff = int64_t(r.d0 + int32_t(j)) * h.PV + q;
    hoff = (int64_t(b) * h.Hp + r.h0) * h.LPV + w;
  } else if (LAYOUT == kPageFirst && ALL) {
    // host (B, size, L, R): the unit is [token][layer ll][elem]
    const uint32_t tok = fast_div(w, h.fd_LV);
    const uint32_t rem = w - tok * h.LV;
    const uint32_t ll = fast_div(rem, h.fd_V);
    const uint32_t v = rem - ll * h.V;
    bi = b * h.L + int32_t(ll);
    doff = (int64_t(r.d0) * h.P + tok) * h.V + v;
    hoff = (int64_t(b) * h.Hp + r.h0) * h.P * h.LV + w;
  } else if (LAYOUT == kPageFirstDirectKV && ALL) {
    // host (Hp, B, L, P, R): the unit is the whole run, every buffer:
    // [page j][buffer bb][layer ll][token, elem]
    const uint32_t j = fast_div(w, h.fd_BLPV);
    uint32_t rem = w - j * h.BLPV;
    const uint32_t bb = fast_div(rem, h.fd_LPV);
    rem -= bb * h.LPV;
    const uint32_t ll = fast_div(rem, h.fd_PV);
    const uint32_t q = rem - ll * h.PV;
    bi = int32_t(bb) * h.L + int32_t(ll);
    doff = int64_t(r.d0 + int32_t(j)) * h.PV + q;
    hoff = int64_t(r.h0) * h.BLPV + w;
  } else if (LAYOUT == kPageFirstDirect) {
    // one layer: device contiguous over the run, host one P*R block per page
    const uint32_t j = fast_div(w, h.fd_PV);
    const uint32_t q = w - j * h.PV;
    bi = b * h.L + l;
    doff = int64_t(r.d0) * h.PV + w;
    hoff = ((int64_t(b) * h.Hp + r.h0 + j) * h.L + l) * h.PV + q;
  } else if (LAYOUT == kPageFirstDirectKV) {
    // one layer: device contiguous over the run, host one P*R block per page
    const uint32_t j = fast_div(w, h.fd_PV);
    const uint32_t q = w - j * h.PV;
    bi = b * h.L + l;
    doff = int64_t(r.d0) * h.PV + w;
    hoff = ((int64_t(r.h0 + int32_t(j)) * h.B + b) * h.L + l) * h.PV + q;
  } else {
    // page_first, one layer: device contiguous over the run, host one row per token
    const uint32_t tok = fast_div(w, h.fd_V);
    const uint32_t v = w - tok * h.V;
    bi = b * h.L + l;
    doff = int64_t(r.d0) * h.PV + w;
    hoff = (((int64_t(b) * h.Hp + r.h0) * h.P + tok) * h.L + l) * h.V + v;
  }
#if HICACHE_CHECKED
  const int32_t kind = check_vector(bi, h.num_bufs, doff, int64_t(h.Dp) * h.PV, hoff, h.host_vecs);
  if (kind != kCheckOk) {
    report_check(kind, kind == kCheckBuffer ? bi : kind == kCheckDevice ? doff : hoff);
    dev = host = nullptr;
    return;
  }
#endif
  dev = bufs[bi] + doff;
  host = static_cast<uint4 *>(h.host) + hoff;
}

// The run holding vector w of an outer unit: the last run with vec0 <= w.
__device__ __forceinline__ int find_run(const Run *runs, int n_runs, uint32_t w) {
  int lo = 0, hi = n_runs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (uint32_t(runs[mid].vec0) <= w) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Move tile `g` of one job: 1024 consecutive vectors (16 KiB) of one outer
// unit's vector range, 4 per thread, all loads issued before the first store.
// The runs of an outer lie end to end in that range, so a tile may span
// several short runs and every tile but an outer's last is full.
//
// The run table sits in the kernel parameters, where loads from different
// addresses within a warp are served one address at a time.  So each warp
// finds the run of its first vector (the same address in every lane) and each
// lane then steps forward from it to its own run: no step where runs are
// longer than a warp's span, one or two where they are a few rows long.
//
// FANOUT (loads of one layer only): every vector is stored to the same place
// in `fan` sets of device buffers, bufs[r * nb + i] for r < fan -- the ranks of
// a tensor-parallel group that each hold the whole replicated latent.  One
// layer's tile lies in one buffer, so only that buffer's base changes per rank.
// With pub.count > 0, thread 0 also publishes the CTA's previous layer between
// this tile's loads and its stores (see tp_pipelined_load_kernel).
struct TpPublish {
  unsigned int *const *counters;   // each rank's per-layer counters
  int32_t layer;
  uint32_t count;                  // 0: nothing to publish
};

template <int LAYOUT, bool ALL, bool TO_HOST, bool FANOUT = false>
__device__ __forceinline__ void move_tile(const XferHeader &h, const Job &job, const Run *runs,
                                          uint4 *const *bufs, int32_t g, int layer, int fan = 1,
                                          int nb = 0, TpPublish pub = {nullptr, 0, 0}) {
  const int32_t outer = g / job.tiles_per_outer;
  const int32_t inner = g - outer * job.tiles_per_outer;
  int b, l;
  if (LAYOUT == kLayerFirst && ALL) {
    b = outer / h.L;
    l = outer - b * h.L;
  } else {
    b = outer;
    l = layer;
  }
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t warp0 = uint32_t(inner) * kTileVecs + (threadIdx.x - lane);  // the warp's first vector
  int rb = 0;                      // the run of the warp's first vector at step k (warp-uniform)
  uint32_t rb_end = 0;

  uint4 v[kUnroll];
  uint4 *dst[kUnroll];
#pragma unroll
  for (int k = 0; k < kUnroll; ++k) {
    const uint32_t base = warp0 + k * kThreads;
    const uint32_t w = base + lane;
    dst[k] = nullptr;
    if (job.run_vecs != 0) {                               // runs of one length: no search
      if (w < job.vecs_per_outer) {
        const uint32_t r = fast_div(w, job.fd_run);
#if HICACHE_CHECKED
        if (r >= uint32_t(job.n_runs)) {
          report_check(kCheckRun, r);
          continue;
        }
#endif
        const Run cur = runs[r];
        uint4 *dev, *host;
        map_vector<LAYOUT, ALL>(h, bufs, b, l, cur, w - r * job.run_vecs, dev, host);
#if HICACHE_CHECKED
        if (dev == nullptr) continue;
#endif
        if (TO_HOST) {
          v[k] = ld_stream(dev);
          dst[k] = host;
        } else {
          v[k] = ld_stream(host);
          dst[k] = dev;
        }
      }
    } else if (base < job.vecs_per_outer) {                // warp-uniform
      if (k == 0 || base >= rb_end) {
        rb = find_run(runs, job.n_runs, base);
        rb_end = uint32_t(runs[rb].vec0) + uint32_t(runs[rb].len) * h.unit_per_page;
      }
      if (w < job.vecs_per_outer) {
        int r = rb;
        uint32_t end = rb_end;
        while (w >= end) {                                 // runs shorter than the warp's span
          ++r;
#if HICACHE_CHECKED
          if (r >= job.n_runs) break;
#endif
          end = uint32_t(runs[r].vec0) + uint32_t(runs[r].len) * h.unit_per_page;
        }
#if HICACHE_CHECKED
        if (r >= job.n_runs) {
          report_check(kCheckRun, r);
          continue;
        }
#endif
        const Run cur = runs[r];
        uint4 *dev, *host;
        map_vector<LAYOUT, ALL>(h, bufs, b, l, cur, w - uint32_t(cur.vec0), dev, host);
#if HICACHE_CHECKED
        if (dev == nullptr) continue;
#endif
        if (TO_HOST) {
          v[k] = ld_stream(dev);
          dst[k] = host;
        } else {
          v[k] = ld_stream(host);
          dst[k] = dev;
        }
      }
    }
  }
  if constexpr (FANOUT) {
    static_assert(!ALL && !TO_HOST, "fan-out is for loads of one layer");
    if (pub.count != 0 && threadIdx.x == 0) {
      // Every thread's stores of the published layer came before the barrier
      // that ended the CTA's previous tile, and that barrier comes before this
      // point, so thread 0's system-wide fence (cumulative) makes the whole
      // CTA's stores of that layer visible to every GPU before the counts.
      // Here the fence waits while this tile's loads are in flight anyway.
      __threadfence_system();
      for (int r = 0; r < fan; ++r) atomicAdd_system(&pub.counters[r][pub.layer], pub.count);
    }
    const int idx = b * h.L + l;
    uint4 *const base0 = bufs[idx];
    for (int r = 0; r < fan; ++r) {
      uint4 *const base = bufs[r * nb + idx];
#pragma unroll
      for (int k = 0; k < kUnroll; ++k)
        if (dst[k] != nullptr) st_stream(base + (dst[k] - base0), v[k]);
    }
    return;
  }
#pragma unroll
  for (int k = 0; k < kUnroll; ++k)
    if (dst[k] != nullptr) st_stream(dst[k], v[k]);
}

template <class Params>
__device__ __forceinline__ const Run *job_runs(const Params &p, int j) {
  return reinterpret_cast<const Run *>(&p.blob[p.h.job[j].runs_word]);
}

template <class Params>
__device__ __forceinline__ void load_buffer_table(const Params &p, uint4 **s_bufs) {
  for (int i = threadIdx.x; i < p.h.num_bufs; i += kThreads)
    s_bufs[i] = reinterpret_cast<uint4 *>(p.blob[i]);
  __syncthreads();
}

// One direction: CTAs take tiles grid-stride in host-address order.
template <int LAYOUT, bool ALL, bool TO_HOST, class Params>
__global__ void __launch_bounds__(kThreads) xfer_kernel(const __grid_constant__ Params p) {
  __shared__ uint4 *s_bufs[kMaxBufs];
  load_buffer_table(p, s_bufs);
  if (p.h.wait_previous) finish_after_previous_launch();
  const Job &job = p.h.job[0];
  const Run *runs = job_runs(p, 0);
  for (int32_t g = blockIdx.x; g < job.total_tiles; g += gridDim.x) {
    if (g + int32_t(gridDim.x) >= job.total_tiles) allow_next_launch();
    move_tile<LAYOUT, ALL, TO_HOST>(p.h, job, runs, s_bufs, g, p.h.layer);
  }
  if (p.h.signal != nullptr) {
    // The barrier orders the CTA's stores before thread 0's fence, which is
    // cumulative: one fence covers the whole CTA before it counts itself done.
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      atomicAdd(p.h.signal, 1u);
    }
  }
  finish_after_previous_launch();
}

// Both directions in one launch: job 0 is a backup, job 1 a load, every layer.
// Each CTA alternates a backup tile and a load tile, so the two directions of
// the host link advance together and neither finishes early, leaving the
// other to run alone; once one job runs out the CTA finishes the other.
template <int LAYOUT, class Params>
__global__ void __launch_bounds__(kThreads) bidir_kernel(const __grid_constant__ Params p) {
  __shared__ uint4 *s_bufs[kMaxBufs];
  load_buffer_table(p, s_bufs);
  if (p.h.wait_previous) finish_after_previous_launch();
  const Job &jb = p.h.job[0];
  const Job &jl = p.h.job[1];
  const Run *rb = job_runs(p, 0);
  const Run *rl = job_runs(p, 1);
  int32_t ib = blockIdx.x, il = blockIdx.x;
  bool backup_turn = true;
  while (ib < jb.total_tiles || il < jl.total_tiles) {
    const bool do_backup = il >= jl.total_tiles || (backup_turn && ib < jb.total_tiles);
    const bool last = (do_backup ? ib + int32_t(gridDim.x) : ib) >= jb.total_tiles &&
                      (do_backup ? il : il + int32_t(gridDim.x)) >= jl.total_tiles;
    if (last) allow_next_launch();
    if (do_backup) {
      move_tile<LAYOUT, true, true>(p.h, jb, rb, s_bufs, ib, 0);
      ib += gridDim.x;
    } else {
      move_tile<LAYOUT, true, false>(p.h, jl, rl, s_bufs, il, 0);
      il += gridDim.x;
    }
    backup_turn = !backup_turn;
  }
  finish_after_previous_launch();
}

// Several pools in one launch (a buffer group): job j owns the tiles
// [tile_start[j], tile_start[j + 1]) and moves them with its own pool's shape,
// host alias, run table and buffer pointers.  The tiles of all jobs are one
// grid-stride range, so the group costs one launch and one ramp whatever the
// number of pools.
template <int LAYOUT, bool ALL, bool TO_HOST, class Params>
__global__ void __launch_bounds__(kThreads) group_kernel(const __grid_constant__ Params p) {
  __shared__ uint4 *s_bufs[kMaxBufs];
  for (int i = threadIdx.x; i < p.g.num_bufs; i += kThreads)
    s_bufs[i] = reinterpret_cast<uint4 *>(p.blob[i]);
  __syncthreads();
  if (p.g.h[0].wait_previous) finish_after_previous_launch();
  const int32_t total = p.g.tile_start[p.g.njobs];
  for (int32_t g = blockIdx.x; g < total; g += gridDim.x) {
    if (g + int32_t(gridDim.x) >= total) allow_next_launch();
    int j = 0;
    while (j + 1 < p.g.njobs && g >= p.g.tile_start[j + 1]) ++j;
    const XferHeader &h = p.g.h[j];
    const Run *runs = reinterpret_cast<const Run *>(&p.blob[h.job[0].runs_word]);
    move_tile<LAYOUT, ALL, TO_HOST>(h, h.job[0], runs, s_bufs + p.g.bufs_word[j], g - p.g.tile_start[j],
                                    h.layer);
  }
  if (p.g.signal[0] != nullptr) {
    __syncthreads();                                    // as in xfer_kernel: one cumulative fence
    if (threadIdx.x == 0) {
      __threadfence();
      for (int j = 0; j < p.g.njobs; ++j) atomicAdd(p.g.signal[j], 1u);
    }
  }
  finish_after_previous_launch();
}

// Every layer of a load in one launch, layer by layer: tile g of the launch
// is tile (g mod T) of layer g / T, where T = the tiles of one layer.  After
// each tile the CTA adds one to its layer's counter, behind a fence, so a
// layer's counter grows by T once the whole layer has landed; a compute stream
// waits for that with a stream memory wait instead of a per-layer launch and
// event.
//
// CTAs take tiles from a counter (sched[0]) rather than by grid stride.  The
// CTAs do not all move at the same rate over the host link, and with a fixed
// share each a layer is only complete when its slowest CTA gets there: the
// fast CTAs run layers ahead while the early layers finish late and the last
// ones all at once.  Taken from a counter, the tiles in flight are always the
// next ones in order, so layer l lands at about (l + 1) / L of the load.
// sched[1] counts the CTAs that are done; the last one puts both words back
// to zero for the next launch on the same scheduler words.
// End of a CTA of a counter-scheduled launch: count it out; the last one out
// puts the two scheduler words back to zero for the next launch.
__device__ __forceinline__ void release_schedule(unsigned int *sched) {
  if (threadIdx.x == 0) {
    __threadfence();                                    // this CTA's last take before its exit count
    if (atomicAdd(&sched[1], 1u) == gridDim.x - 1) {
      __threadfence();                                  // every CTA's takes before the reset
      atomicExch(&sched[0], 0u);
      atomicExch(&sched[1], 0u);
    }
  }
}

template <int LAYOUT, class Params>
__global__ void __launch_bounds__(kThreads)
    pipelined_load_kernel(const __grid_constant__ Params p, unsigned int *layer_done,
                          unsigned int *sched) {
  __shared__ uint4 *s_bufs[kMaxBufs];
  __shared__ int32_t s_next;
  load_buffer_table(p, s_bufs);
  const Job &job = p.h.job[0];
  const Run *runs = job_runs(p, 0);
  const int32_t per_layer = job.total_tiles;            // tiles of one layer
  const int32_t total = per_layer * p.h.L;
  if (threadIdx.x == 0) s_next = int32_t(atomicAdd(&sched[0], 1u));
  __syncthreads();
  for (int32_t g = s_next; g < total; g = s_next) {
    const int32_t layer = g / per_layer;
    move_tile<LAYOUT, false, false>(p.h, job, runs, s_bufs, g - layer * per_layer, layer);
    __threadfence();                                    // this thread's stores, device-wide
    __syncthreads();                                    // every thread is past its fence and has read s_next
    if (threadIdx.x == 0) {
      atomicAdd(&layer_done[layer], 1u);
      s_next = int32_t(atomicAdd(&sched[0], 1u));
    }
    __syncthreads();
  }
  release_schedule(sched);
}

// The share of one rank of a tensor-parallel group in a load of a replicated
// latent ("Baidu's KVCache Overhaul", section "MLA-class cache optimization":
// each GPU reads only its part of the pages over the host link, and the parts
// are spread to every GPU over NVLink, layer by layer, alongside the loads).
// Like pipelined_load_kernel -- every layer in one launch, in layer order,
// tiles taken from a counter -- except that each vector read from the host is
// stored into every rank's buffers (the blob holds f.tp sets of num_bufs
// pointers, rank-major; a peer's buffers are reached over NVLink), and each
// finished tile adds one to that layer's counter of every rank, behind a
// system-wide fence, so a rank's counter of layer l reaches the tiles of all
// ranks' shares once every share of that layer has landed in its buffers.
// No CTA waits for another rank: a launch only stores and counts.
template <int LAYOUT, class Params>
__global__ void __launch_bounds__(kThreads)
    tp_pipelined_load_kernel(const __grid_constant__ Params p, const __grid_constant__ TpFanout f,
                             unsigned int *sched) {
  __shared__ uint4 *s_bufs[kMaxTpBufs];
  __shared__ int32_t s_next;
  const int nb = p.h.num_bufs;
  for (int i = threadIdx.x; i < f.tp * nb; i += kThreads) s_bufs[i] = reinterpret_cast<uint4 *>(p.blob[i]);
  const Job &job = p.h.job[0];
  const Run *runs = job_runs(p, 0);
  const int32_t per_layer = job.total_tiles;            // tiles of one layer
  const int32_t total = per_layer * p.h.L;
  if (threadIdx.x == 0) s_next = int32_t(atomicAdd(&sched[0], 1u));
  __syncthreads();
  // A system-wide fence per tile would hold the loads back (a tile's stores
  // must reach every GPU before the next tile starts), so the CTA holds the
  // count of its finished tiles of one layer and fences and counts them once,
  // when its next tile is in another layer or it has none left.  Tiles come
  // in layer order, so that is as soon as its last tile of the layer is done.
  // All CTAs cross a layer at about the same time; a fence between tiles
  // would stall them all at once and leave the link idle at every layer (a
  // fixed ~2.5 us a layer), so it is taken inside the next tile, after that
  // tile's loads are issued (move_tile's `pub`), and only the CTA's last
  // layer is published after its last tile.  Both follow a barrier that
  // every thread reached after its stores of the published layer (the pattern
  // of a cooperative grid barrier: one cumulative fence by thread 0).
  int32_t held_layer = 0;                               // CTA-uniform, as g is
  uint32_t held = 0;
  for (int32_t g = s_next;; g = s_next) {
    const bool done = g >= total;
    const int32_t layer = done ? -1 : g / per_layer;
    TpPublish pub{f.counters, held_layer, 0};
    if (held != 0 && layer != held_layer) {
      if (done) {
        if (threadIdx.x == 0) {
          __threadfence_system();
          for (int r = 0; r < f.tp; ++r) atomicAdd_system(&f.counters[r][held_layer], held);
        }
      } else {
        pub.count = held;
      }
      held = 0;
    }
    if (done) break;
    move_tile<LAYOUT, false, false, true>(p.h, job, runs, s_bufs, g - layer * per_layer, layer, f.tp, nb,
                                          pub);
    held_layer = layer;
    ++held;
    __syncthreads();                                    // every thread has read s_next
    if (threadIdx.x == 0) s_next = int32_t(atomicAdd(&sched[0], 1u));
    __syncthreads();
  }
  release_schedule(sched);
}

// Every layer of several pools in one launch (a pipelined buffer group): tile
// g is in layer g / T, where T = the tiles of one layer over all pools, and
// within that layer pool j owns [tile_start[j], tile_start[j + 1]).  After each
// tile the CTA adds one to that pool's counter of that layer, so each pool's
// counters behave as those of its own pipelined load; tiles come from the
// counter sched[0], as in pipelined_load_kernel, so all pools' tiles of layer l
// land before those of layer l + 1.
template <int LAYOUT, class Params>
__global__ void __launch_bounds__(kThreads)
    pipelined_group_kernel(const __grid_constant__ Params p) {
  __shared__ uint4 *s_bufs[kMaxBufs];
  __shared__ int32_t s_next;
  for (int i = threadIdx.x; i < p.g.num_bufs; i += kThreads)
    s_bufs[i] = reinterpret_cast<uint4 *>(p.blob[i]);
  const int32_t per_layer = p.g.tile_start[p.g.njobs];   // tiles of one layer, every pool
  const int32_t total = per_layer * p.g.h[0].L;
  unsigned int *const sched = p.g.sched;
  if (threadIdx.x == 0) s_next = int32_t(atomicAdd(&sched[0], 1u));
  __syncthreads();
  for (int32_t g = s_next; g < total; g = s_next) {
    const int32_t layer = g / per_layer;
    const int32_t r = g - layer * per_layer;
    int j = 0;
    while (j + 1 < p.g.njobs && r >= p.g.tile_start[j + 1]) ++j;
    const XferHeader &h = p.g.h[j];
    const Run *runs = reinterpret_cast<const Run *>(&p.blob[h.job[0].runs_word]);
    move_tile<LAYOUT, false, false>(h, h.job[0], runs, s_bufs + p.g.bufs_word[j], r - p.g.tile_start[j],
                                    layer);
    __threadfence();                                    // this thread's stores, device-wide
    __syncthreads();                                    // every thread is past its fence and has read s_next
    if (threadIdx.x == 0) {
      atomicAdd(&p.g.layer_done[j][layer], 1u);
      s_next = int32_t(atomicAdd(&sched[0], 1u));
    }
    __syncthreads();
  }
  release_schedule(sched);
}

// Stand-in for attention on one layer: read every vector of the given pages of
// the layer's buffers `reps` times and add up their 32-bit words.
__global__ void __launch_bounds__(kThreads) checksum_kernel(const __grid_constant__ ChecksumParams p) {
  const uint32_t per_buf = uint32_t(p.n) * p.PV;
  const uint64_t total = uint64_t(per_buf) * p.B;
  unsigned long long acc = 0;
  for (int rep = 0; rep < p.reps; ++rep) {
    for (uint64_t i = uint64_t(blockIdx.x) * kThreads + threadIdx.x; i < total;
         i += uint64_t(gridDim.x) * kThreads) {
      const uint32_t b = uint32_t(i / per_buf);
      const uint32_t w = uint32_t(i - uint64_t(b) * per_buf);
      const uint32_t j = w / p.PV;
      const uint32_t q = w - j * p.PV;
      const uint4 x = __ldcg(static_cast<const uint4 *>(p.bufs[b]) + int64_t(p.pages[j]) * p.PV + q);
      acc += (unsigned long long)x.x + x.y + x.z + x.w;
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_down_sync(0xffffffffu, acc, off);
  if ((threadIdx.x & 31) == 0 && acc != 0) atomicAdd(p.out, acc);
}

// Roofline probe: a plain streaming copy of nvec 16-byte vectors, with no
// index decode.  Each CTA moves tiles of kThreads * UNROLL consecutive vectors,
// UNROLL loads in flight per thread before the first store, CTAs grid-stride in
// address order: the transfer kernels' access pattern on both sides, without
// their address arithmetic.
template <int UNROLL>
__global__ void __launch_bounds__(kThreads)
    stream_copy_kernel(uint4 *__restrict__ dst, const uint4 *__restrict__ src, uint64_t nvec) {
  const uint64_t tile = uint64_t(kThreads) * UNROLL;
  for (uint64_t t = uint64_t(blockIdx.x) * tile; t < nvec; t += uint64_t(gridDim.x) * tile) {
    uint4 v[UNROLL];
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) {
      const uint64_t i = t + uint64_t(k) * kThreads + threadIdx.x;
      if (i < nvec) v[k] = ld_stream(src + i);
    }
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) {
      const uint64_t i = t + uint64_t(k) * kThreads + threadIdx.x;
      if (i < nvec) st_stream(dst + i, v[k]);
    }
  }
}

template <class Params>
const Params &params_for(const XferLaunch &x, Params &small) {
  small.h = x.params->h;
  for (int i = 0; i < x.words; ++i) small.blob[i] = x.params->blob[i];
  return small;
}

// Launch with programmatic stream serialization: the kernel may begin once
// every CTA of the kernel before it on the stream has signalled
// griddepcontrol.launch_dependents (or exited).
template <class Params, class Launch>
cudaError_t launch_programmatic(void (*kernel)(Params), const Launch &x, const Params &p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(x.grid));
  cfg.blockDim = dim3(unsigned(kThreads));
  cfg.dynamicSmemBytes = 0;
  cfg.stream = static_cast<cudaStream_t>(x.stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

template <int LAYOUT, bool ALL, bool TO_HOST>
cudaError_t launch_one(const XferLaunch &x) {
  const cudaStream_t st = static_cast<cudaStream_t>(x.stream);
  const bool pdl = x.pdl;
  if (x.words <= kBlobWordsSmall) {
    XferParamsSmall small;
    if (pdl) return launch_programmatic(&xfer_kernel<LAYOUT, ALL, TO_HOST, XferParamsSmall>, x, params_for(x, small));
    xfer_kernel<LAYOUT, ALL, TO_HOST><<<x.grid, kThreads, 0, st>>>(params_for(x, small));
  } else {
    if (pdl) return launch_programmatic(&xfer_kernel<LAYOUT, ALL, TO_HOST, XferParams>, x, *x.params);
    xfer_kernel<LAYOUT, ALL, TO_HOST><<<x.grid, kThreads, 0, st>>>(*x.params);
  }
  return cudaGetLastError();
}

template <int LAYOUT>
cudaError_t launch_layout(const XferLaunch &x) {
  if (x.bidir) {
    const cudaStream_t st = static_cast<cudaStream_t>(x.stream);
    if (x.words <= kBlobWordsSmall) {
      XferParamsSmall small;
      if (x.pdl) return launch_programmatic(&bidir_kernel<LAYOUT, XferParamsSmall>, x, params_for(x, small));
      bidir_kernel<LAYOUT><<<x.grid, kThreads, 0, st>>>(params_for(x, small));
    } else {
      if (x.pdl) return launch_programmatic(&bidir_kernel<LAYOUT, XferParams>, x, *x.params);
      bidir_kernel<LAYOUT><<<x.grid, kThreads, 0, st>>>(*x.params);
    }
    return cudaGetLastError();
  }
  if (x.all_layers)
    return x.to_host ? launch_one<LAYOUT, true, true>(x) : launch_one<LAYOUT, true, false>(x);
  return x.to_host ? launch_one<LAYOUT, false, true>(x) : launch_one<LAYOUT, false, false>(x);
}

template <int LAYOUT>
cudaError_t launch_pipelined_layout(const XferLaunch &x, unsigned int *layer_done, unsigned int *sched) {
  const cudaStream_t st = static_cast<cudaStream_t>(x.stream);
  if (x.words <= kBlobWordsSmall) {
    XferParamsSmall small;
    pipelined_load_kernel<LAYOUT><<<x.grid, kThreads, 0, st>>>(params_for(x, small), layer_done, sched);
  } else {
    pipelined_load_kernel<LAYOUT><<<x.grid, kThreads, 0, st>>>(*x.params, layer_done, sched);
  }
  return cudaGetLastError();
}

template <int LAYOUT>
cudaError_t launch_tp_layout(const XferLaunch &x, const TpFanout &f, unsigned int *sched) {
  const cudaStream_t st = static_cast<cudaStream_t>(x.stream);
  if (x.words <= kBlobWordsSmall) {
    XferParamsSmall small;
    tp_pipelined_load_kernel<LAYOUT><<<x.grid, kThreads, 0, st>>>(params_for(x, small), f, sched);
  } else {
    tp_pipelined_load_kernel<LAYOUT><<<x.grid, kThreads, 0, st>>>(*x.params, f, sched);
  }
  return cudaGetLastError();
}

}  // namespace

int launch_tp_pipelined_load(const XferLaunch &x, const TpFanout &f, unsigned int *sched) {
  switch (x.layout) {
    case kLayerFirst: return int(launch_tp_layout<kLayerFirst>(x, f, sched));
    case kPageFirst: return int(launch_tp_layout<kPageFirst>(x, f, sched));
    case kPageFirstDirect: return int(launch_tp_layout<kPageFirstDirect>(x, f, sched));
    case kPageFirstDirectKV: return int(launch_tp_layout<kPageFirstDirectKV>(x, f, sched));
    default: return int(cudaErrorInvalidValue);
  }
}

int launch_pipelined_load(const XferLaunch &x, unsigned int *layer_done, unsigned int *sched) {
  switch (x.layout) {
    case kLayerFirst: return int(launch_pipelined_layout<kLayerFirst>(x, layer_done, sched));
    case kPageFirst: return int(launch_pipelined_layout<kPageFirst>(x, layer_done, sched));
    case kPageFirstDirect: return int(launch_pipelined_layout<kPageFirstDirect>(x, layer_done, sched));
    case kPageFirstDirectKV: return int(launch_pipelined_layout<kPageFirstDirectKV>(x, layer_done, sched));
    default: return int(cudaErrorInvalidValue);
  }
}

// Per-layer counters and scheduler words for pipelined loads made without any
// allocation (hicache_load_pipelined_noalloc): a fixed array in the library's
// own device memory, loaded with the module on every GPU that uses the library
// and kept until the process exits.  Every such call on a device shares the
// layer counters; the counts only ever grow (the host keeps the matching
// targets), so nothing needs clearing between calls -- the array starts at
// zero when the module loads.  The scheduler words come in kNoAllocSchedSlots
// pairs that calls take in turn; each launch leaves its pair at zero.
static __device__ __align__(256) unsigned int
    g_noalloc_counters[kNoAllocMaxLayers + 2 * kNoAllocSchedSlots];

int noalloc_layer_counters(unsigned int **out) {
  // The array's name is only a stand-in in host code: the kernel needs its
  // device address, looked up once per device with that device current.
  static std::mutex mu;
  static unsigned int *addr[kNoAllocMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return int(e);
  if (dev < 0 || dev >= kNoAllocMaxDevices) return int(cudaErrorInvalidDevice);
  std::lock_guard<std::mutex> g(mu);
  if (!addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_counters);
    if (e != cudaSuccess) return int(e);
    addr[dev] = static_cast<unsigned int *>(p);
  }
  *out = addr[dev];
  return 0;
}

namespace {

template <int LAYOUT, bool ALL, bool TO_HOST>
cudaError_t launch_group_one(const GroupLaunch &x) {
  const cudaStream_t st = static_cast<cudaStream_t>(x.stream);
  if (x.words <= kGroupBlobWordsSmall) {
    GroupParamsSmall small;
    small.g = x.params->g;
    for (int i = 0; i < x.words; ++i) small.blob[i] = x.params->blob[i];
    if (x.pdl) return launch_programmatic(&group_kernel<LAYOUT, ALL, TO_HOST, GroupParamsSmall>, x, small);
    group_kernel<LAYOUT, ALL, TO_HOST><<<x.grid, kThreads, 0, st>>>(small);
  } else {
    if (x.pdl) return launch_programmatic(&group_kernel<LAYOUT, ALL, TO_HOST, GroupParams>, x, *x.params);
    group_kernel<LAYOUT, ALL, TO_HOST><<<x.grid, kThreads, 0, st>>>(*x.params);
  }
  return cudaGetLastError();
}

template <int LAYOUT>
cudaError_t launch_group_layout(const GroupLaunch &x) {
  if (x.all_layers)
    return x.to_host ? launch_group_one<LAYOUT, true, true>(x) : launch_group_one<LAYOUT, true, false>(x);
  return x.to_host ? launch_group_one<LAYOUT, false, true>(x) : launch_group_one<LAYOUT, false, false>(x);
}

}  // namespace

int launch_pipelined_group(const GroupLaunch &x) {
  const cudaStream_t st = static_cast<cudaStream_t>(x.stream);
  auto go = [&](auto layout_tag) -> cudaError_t {
    constexpr int LAYOUT = decltype(layout_tag)::value;
    if (x.words <= kGroupBlobWordsSmall) {
      GroupParamsSmall small;
      small.g = x.params->g;
      for (int i = 0; i < x.words; ++i) small.blob[i] = x.params->blob[i];
      pipelined_group_kernel<LAYOUT><<<x.grid, kThreads, 0, st>>>(small);
    } else {
      pipelined_group_kernel<LAYOUT><<<x.grid, kThreads, 0, st>>>(*x.params);
    }
    return cudaGetLastError();
  };
  switch (x.layout) {
    case kLayerFirst: return int(go(std::integral_constant<int, kLayerFirst>()));
    case kPageFirst: return int(go(std::integral_constant<int, kPageFirst>()));
    case kPageFirstDirect: return int(go(std::integral_constant<int, kPageFirstDirect>()));
    case kPageFirstDirectKV: return int(go(std::integral_constant<int, kPageFirstDirectKV>()));
    default: return int(cudaErrorInvalidValue);
  }
}

int launch_group(const GroupLaunch &x) {
  switch (x.layout) {
    case kLayerFirst: return int(launch_group_layout<kLayerFirst>(x));
    case kPageFirst: return int(launch_group_layout<kPageFirst>(x));
    case kPageFirstDirect: return int(launch_group_layout<kPageFirstDirect>(x));
    case kPageFirstDirectKV: return int(launch_group_layout<kPageFirstDirectKV>(x));
    default: return int(cudaErrorInvalidValue);
  }
}

int launch_xfer(const XferLaunch &x) {
  switch (x.layout) {
    case kLayerFirst: return int(launch_layout<kLayerFirst>(x));
    case kPageFirst: return int(launch_layout<kPageFirst>(x));
    case kPageFirstDirect: return int(launch_layout<kPageFirstDirect>(x));
    case kPageFirstDirectKV: return int(launch_layout<kPageFirstDirectKV>(x));
    default: return int(cudaErrorInvalidValue);
  }
}

int launch_stream_copy(void *dst, const void *src, uint64_t nvec, int grid, int unroll, void *stream) {
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint4 *d = static_cast<uint4 *>(dst);
  const uint4 *s = static_cast<const uint4 *>(src);
  if (unroll == 8)
    stream_copy_kernel<8><<<grid, kThreads, 0, st>>>(d, s, nvec);
  else if (unroll == 4)
    stream_copy_kernel<4><<<grid, kThreads, 0, st>>>(d, s, nvec);
  else
    return int(cudaErrorInvalidValue);
  return int(cudaGetLastError());
}

int checked_build() { return HICACHE_CHECKED; }

int check_status(unsigned long long *first, unsigned long long *count, bool clear) {
  unsigned long long w[2] = {0, 0};
  cudaError_t e = cudaMemcpyFromSymbol(w, g_check_words, sizeof w);
  if (e == cudaSuccess && clear) {
    const unsigned long long z[2] = {0, 0};
    e = cudaMemcpyToSymbol(g_check_words, z, sizeof z);
  }
  *first = w[0];
  *count = w[1];
  return int(e);
}

int launch_checksum(const ChecksumParams &p, int grid, void *stream) {
  checksum_kernel<<<grid, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(p);
  return int(cudaGetLastError());
}

}  // namespace hicache
