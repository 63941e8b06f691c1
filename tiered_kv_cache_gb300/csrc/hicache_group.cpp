// hicache_group.cpp -- buffer groups: up to HICACHE_MAX_GROUP pools (buffer
// kinds with different rows) moved by one index set in one launch per chunk,
// all layers, one layer, or pipelined with per-layer counters for every pool;
// and group plans, whose per-layer loads replay from one CUDA graph.

#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <mutex>
#include <new>
#include <utility>
#include <vector>

#include "hicache.h"
#include "hicache_host.h"
#include "hicache_internal.h"

namespace hicache {

// Enqueue validated runs for every pool of a group, one launch per chunk of
// runs that fits the parameters of all of them.  pdl_first: the first launch
// may start while the kernel before it on the stream drains; that kernel must
// be a one-layer group load of another layer.
// signal (one-layer loads): every CTA of every launch adds one to each pool's
// counter of that layer once its last tile has landed; *signalled grows by
// the CTAs launched.
int enqueue_group(hicache_pool *const *pools, const hicache_device_kv *kvs, int32_t np,
                  const std::vector<RunRec> &runs, int32_t layout, int32_t layer, bool to_host,
                  void *stream, bool pdl_first = false, bool signal = false, int64_t *signalled = nullptr) {
  if (runs.empty()) return HICACHE_OK;
  const bool all = layer < 0;
  thread_local hicache::GroupParams params;
  hicache::GroupHeader &g = params.g;
  g.njobs = np;
  for (int32_t j = 0; j < hicache::kMaxGroup; ++j)
    g.signal[j] = signal && !all && j < np ? pools[j]->layer_done + layer : nullptr;
  int32_t word = 0;
  int64_t outers[hicache::kMaxGroup], upp[hicache::kMaxGroup];
  for (int32_t j = 0; j < np; ++j) {
    const Shape &s = pools[j]->shape;
    const bool lf_all = (layout == HICACHE_LAYER_FIRST) && all;
    const bool kv_all = (layout == HICACHE_PAGE_FIRST_DIRECT_KV) && all;
    outers[j] = lf_all ? s.B * s.L : (kv_all ? 1 : s.B);
    upp[j] = !all || layout == HICACHE_LAYER_FIRST ? s.PV : (kv_all ? s.BLPV : s.LPV);
    fill_shape(pools[j], upp[j], all ? 0 : layer, kvs[j].device_num_pages, g.h[j]);
    g.bufs_word[j] = word;
    for (int64_t i = 0; i < s.B * s.L; ++i)
      params.blob[word++] = uint64_t(reinterpret_cast<uintptr_t>(kvs[j].buf_ptrs[i]));
  }
  g.num_bufs = word;
  const int64_t capacity = (hicache::kGroupBlobWords - word) / (2 * np);  // runs per launch
  const hicache_pool *p0 = pools[0];
  size_t next = 0;
  while (next < runs.size()) {
    // the most runs every job's table and tile budget can take
    int64_t c = capacity;
    for (int32_t j = 0; j < np; ++j) {
      hicache::Run *table = reinterpret_cast<hicache::Run *>(&params.blob[word]);
      const int32_t cj = fill_runs(runs, next, upp[j], outers[j], c, g.h[j].job[0], table, word, np);
      if (cj < 0) return set_error(HICACHE_ERR_INVALID_ARG, "transfer too large for one launch");
      c = std::min<int64_t>(c, cj);
    }
    int64_t tiles = 0;
    for (int32_t j = 0; j < np; ++j) {
      const int32_t w = word + int32_t(2 * c) * j;
      hicache::Run *table = reinterpret_cast<hicache::Run *>(&params.blob[w]);
      fill_runs(runs, next, upp[j], outers[j], c, g.h[j].job[0], table, w, np);
      g.tile_start[j] = int32_t(tiles);
      tiles += g.h[j].job[0].total_tiles;
    }
    g.tile_start[np] = int32_t(tiles);
    hicache::GroupLaunch x;
    x.params = &params;
    x.words = word + int32_t(2 * c) * np;
    x.layout = layout;
    x.all_layers = all;
    x.to_host = to_host;
    x.grid = int(std::min<int64_t>(tiles, to_host ? p0->backup_ctas : all ? p0->ctas : p0->layer_ctas));
    x.stream = stream;
    x.pdl = next > 0 || !all;          // as enqueue
    g.h[0].wait_previous = next == 0 && !all && !pdl_first ? 1 : 0;
    const int e = hicache::launch_group(x);
    if (e != 0) return cuda_error(cudaError_t(e), "group transfer kernel launch");
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (signalled && g.signal[0]) *signalled += x.grid;
    next += size_t(c);
  }
  return HICACHE_OK;
}

// Enqueue validated load runs for every pool of a group as pipelined launches:
// every layer of every pool, layer by layer, one counter per pool and layer.
// The caller holds every pool's signal lock.
int enqueue_group_pipelined(hicache_pool *const *pools, const hicache_device_kv *kvs, int32_t np,
                            const std::vector<RunRec> &runs, int32_t layout, void *stream) {
  const int64_t L = pools[0]->shape.L;
  thread_local hicache::GroupParams params;
  hicache::GroupHeader &g = params.g;
  g.njobs = np;
  for (int32_t j = 0; j < hicache::kMaxGroup; ++j) g.signal[j] = nullptr;
  int32_t word = 0;
  for (int32_t j = 0; j < np; ++j) {
    const Shape &s = pools[j]->shape;
    fill_shape(pools[j], s.PV, 0, kvs[j].device_num_pages, g.h[j]);
    g.bufs_word[j] = word;
    for (int64_t i = 0; i < s.B * s.L; ++i)
      params.blob[word++] = uint64_t(reinterpret_cast<uintptr_t>(kvs[j].buf_ptrs[i]));
    g.layer_done[j] = pools[j]->layer_done;
  }
  for (int32_t j = np; j < hicache::kMaxGroup; ++j) g.layer_done[j] = nullptr;
  g.sched = pools[0]->layer_done + L;       // pool 0's scheduler words
  g.num_bufs = word;
  const int64_t capacity = (hicache::kGroupBlobWords - word) / (2 * np);
  size_t next = 0;
  while (next < runs.size()) {
    // one layer's units of pool j are (buffer, run); the launch covers L layers
    int64_t c = capacity;
    for (int32_t j = 0; j < np; ++j) {
      const Shape &s = pools[j]->shape;
      hicache::Run *table = reinterpret_cast<hicache::Run *>(&params.blob[word]);
      const int32_t cj = fill_runs(runs, next, s.PV, s.B, c, g.h[j].job[0], table, word, np * L);
      if (cj < 0) return set_error(HICACHE_ERR_INVALID_ARG, "transfer too large for one launch");
      c = std::min<int64_t>(c, cj);
    }
    int64_t tiles = 0;
    for (int32_t j = 0; j < np; ++j) {
      const Shape &s = pools[j]->shape;
      const int32_t w = word + int32_t(2 * c) * j;
      fill_runs(runs, next, s.PV, s.B, c, g.h[j].job[0], reinterpret_cast<hicache::Run *>(&params.blob[w]), w,
                np * L);
      g.tile_start[j] = int32_t(tiles);
      tiles += g.h[j].job[0].total_tiles;
    }
    g.tile_start[np] = int32_t(tiles);
    hicache::GroupLaunch x;
    x.params = &params;
    x.words = word + int32_t(2 * c) * np;
    x.layout = layout;
    x.all_layers = false;
    x.to_host = false;
    x.grid = int(std::min<int64_t>(tiles * L, pools[0]->layer_ctas));
    x.stream = stream;
    const int e = hicache::launch_pipelined_group(x);
    if (e != 0) return cuda_error(cudaError_t(e), "pipelined group kernel launch");
    g_launches.fetch_add(1, std::memory_order_relaxed);
    for (int32_t j = 0; j < np; ++j)
      for (int64_t l = 0; l < L; ++l) {
        pools[j]->layer_target[size_t(l)] += uint32_t(g.h[j].job[0].total_tiles);
        pools[j]->layer_signal[size_t(l)] = 1;
      }
    next += size_t(c);
  }
  return HICACHE_OK;
}

// The checks every group call shares: 1..HICACHE_MAX_GROUP distinct pools on
// one device with equal layers and page size; with kvs, also the same resolved
// layout, valid device KV for each (at least min_pages pages), at most
// kMaxBufs buffers and no buffer named twice.  Returns the resolved layout
// (with kvs) and the bounds the pre-pass must apply to every pool (Dp only
// with kvs).
int check_group(hicache_pool *const *pools, const hicache_device_kv *kvs, int32_t npools, int32_t layout,
                int32_t *lay, int64_t *Hp, int64_t *Dp, int64_t *max_run, bool with_kvs = true,
                int64_t min_pages = 0) {
  if (!pools || (with_kvs && !kvs)) return set_error(HICACHE_ERR_INVALID_ARG, "pools or kvs is NULL");
  if (npools < 1 || npools > HICACHE_MAX_GROUP)
    return set_error(HICACHE_ERR_INVALID_ARG, "npools = %d outside [1, %d]", npools, HICACHE_MAX_GROUP);
  for (int32_t i = 0; i < npools; ++i)
    if (!pools[i]) return set_error(HICACHE_ERR_INVALID_ARG, "pool %d is NULL", i);
  const hicache_pool *p0 = pools[0];
  int rc = HICACHE_OK;
  if (with_kvs && (rc = resolve_layout(layout, p0->shape.layout, lay))) return rc;
  *Hp = INT64_MAX;
  *Dp = INT64_MAX;
  *max_run = INT64_MAX;
  int64_t bufs = 0;
  std::vector<uintptr_t> ptrs;
  for (int32_t i = 0; i < npools; ++i) {
    const hicache_pool *p = pools[i];
    for (int32_t k = 0; k < i; ++k)
      if (pools[k] == p) return set_error(HICACHE_ERR_INVALID_ARG, "pool %d appears twice in the group", i);
    if (p->device != p0->device)
      return set_error(HICACHE_ERR_INVALID_ARG, "pool %d is on device %d, pool 0 on %d", i, p->device,
                       p0->device);
    if (p->shape.L != p0->shape.L || p->shape.P != p0->shape.P)
      return set_error(HICACHE_ERR_INVALID_ARG,
                       "pool %d has %lld layers of %lld-token pages; pool 0 has %lld of %lld", i,
                       (long long)p->shape.L, (long long)p->shape.P, (long long)p0->shape.L,
                       (long long)p0->shape.P);
    *Hp = std::min(*Hp, p->shape.Hp);
    *max_run = std::min(*max_run, max_run_pages(p->shape));
    if (!with_kvs) continue;
    int32_t li = 0;
    if ((rc = resolve_layout(layout, p->shape.layout, &li))) return rc;
    if (li != *lay)
      return set_error(HICACHE_ERR_INVALID_ARG, "pool %d resolves to layout %d, pool 0 to %d", i, li, *lay);
    if ((rc = check_kv(p, &kvs[i], min_pages))) return rc;
    *Dp = std::min(*Dp, kvs[i].device_num_pages);
    bufs += p->shape.B * p->shape.L;
    for (int64_t b = 0; b < p->shape.B * p->shape.L; ++b)
      ptrs.push_back(reinterpret_cast<uintptr_t>(kvs[i].buf_ptrs[b]));
  }
  if (bufs > hicache::kMaxBufs)
    return set_error(HICACHE_ERR_INVALID_ARG, "the group has %lld device buffers; at most %d", (long long)bufs,
                     hicache::kMaxBufs);
  std::sort(ptrs.begin(), ptrs.end());
  if (std::adjacent_find(ptrs.begin(), ptrs.end()) != ptrs.end())
    return set_error(HICACHE_ERR_INVALID_ARG, "a device buffer is named twice in the group");
  return HICACHE_OK;
}

}  // namespace hicache

using namespace hicache;

extern "C" {

int hicache_group_transfer(hicache_pool *const *pools, const hicache_device_kv *kvs, int32_t npools,
                           const int64_t *device_pages, const int64_t *host_pages, int64_t n,
                           int32_t layout, int32_t layer_id, int32_t direction, void *stream) {
  clear_error();
  int32_t lay = 0;
  int64_t Hp = 0, Dp = 0, max_run = 0;
  int rc = check_group(pools, kvs, npools, layout, &lay, &Hp, &Dp, &max_run);
  if (rc) return rc;
  if (direction != HICACHE_DIR_BACKUP && direction != HICACHE_DIR_LOAD)
    return set_error(HICACHE_ERR_INVALID_ARG, "direction %d is neither backup nor load", direction);
  if (layer_id >= pools[0]->shape.L)
    return set_error(HICACHE_ERR_INVALID_ARG, "layer_id %d outside [0, %lld)", layer_id,
                     (long long)pools[0]->shape.L);
  if (layer_id >= 0 && direction != HICACHE_DIR_LOAD)
    return set_error(HICACHE_ERR_INVALID_ARG, "a per-layer transfer must be a load");
  thread_local std::vector<RunRec> runs;
  if ((rc = prepass(Hp, Dp, device_pages, host_pages, n, direction, max_run, &runs))) return rc;
  if ((rc = check_device(pools[0]))) return rc;
  if ((rc = enqueue_group(pools, kvs, npools, runs, lay, layer_id, direction == HICACHE_DIR_BACKUP, stream)))
    return rc;
  if (layer_id >= 0) {
    for (int32_t i = 0; i < npools; ++i) {
      hicache_pool *p = pools[i];
      const cudaError_t e = cudaEventRecord(p->events[size_t(layer_id)], static_cast<cudaStream_t>(stream));
      if (e != cudaSuccess) return cuda_error(e, "cudaEventRecord(layer event)");
      std::lock_guard<std::mutex> g(p->signal_mu);
      p->layer_signal[size_t(layer_id)] = 0;
    }
  } else if (direction == HICACHE_DIR_LOAD && n > 0) {
    for (int32_t i = 0; i < npools; ++i)
      if ((rc = mark_all_layer_load(pools[i], stream))) return rc;
  }
  return HICACHE_OK;
}

int hicache_group_load_pipelined(hicache_pool *const *pools, const hicache_device_kv *kvs, int32_t npools,
                                 const int64_t *device_pages, const int64_t *host_pages, int64_t n,
                                 int32_t layout, void *stream) {
  clear_error();
  int32_t lay = 0;
  int64_t Hp = 0, Dp = 0, max_run = 0;
  int rc = check_group(pools, kvs, npools, layout, &lay, &Hp, &Dp, &max_run);
  if (rc) return rc;
  thread_local std::vector<RunRec> runs;
  if ((rc = prepass(Hp, Dp, device_pages, host_pages, n, HICACHE_DIR_LOAD, max_run, &runs))) return rc;
  if ((rc = check_device(pools[0]))) return rc;
  if ((rc = refuse_capture(stream))) return rc;
  if (!wait_value32())
    return set_error(HICACHE_ERR_CUDA, "the driver offers no cuStreamWaitValue32: no pipelined loads");
  // every pool's signal lock, in address order (the pools are distinct)
  std::vector<hicache_pool *> order(pools, pools + npools);
  std::sort(order.begin(), order.end());
  std::vector<std::unique_lock<std::mutex>> locks;
  for (hicache_pool *p : order) locks.emplace_back(p->signal_mu);
  for (int32_t i = 0; i < npools; ++i)
    if ((rc = check_counted_stream(pools[i], stream))) return rc;
  for (int32_t i = 0; i < npools; ++i) claim_counted_stream(pools[i], stream);
  if ((rc = enqueue_group_pipelined(pools, kvs, npools, runs, lay, stream))) return rc;
  for (int32_t i = 0; i < npools; ++i) {
    hicache_pool *p = pools[i];
    // (the layer events are recorded when asked for: hicache_layer_event)
    const cudaError_t e = cudaEventRecord(p->pipeline_last, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_error(e, "cudaEventRecord(pipelined load)");
    p->chain_open = false;
  }
  return HICACHE_OK;
}


}  // extern "C"

// ---- group plans -----------------------------------------------------------------

struct hicache_group_plan {
  std::vector<hicache_pool *> pools;
  int64_t n = 0;
  int64_t device_num_pages = 0;
  int64_t Hp = 0;
  std::vector<hicache::RunRec> runs;
  // hicache_group_plan_load_layers: the per-layer group launches and every
  // pool's layer events, captured once per device buffers and layout
  std::mutex graph_mu;
  cudaGraphExec_t graph = nullptr;
  std::vector<void *> graph_bufs;        // every pool's buffer pointers, pool by pool
  std::vector<int64_t> graph_pages;      // every pool's device_num_pages
  int32_t graph_layout = -1;
  int64_t graph_launches = 0;
  // hicache_group_plan_load_layer_chained: the stream and layer of the last
  // chained call, and the buffers found disjoint
  std::mutex chain_mu;
  void *chain_stream = nullptr;
  int32_t chain_layer = -1;
  std::vector<void *> chain_bufs;
  std::vector<int64_t> chain_pages;
};

namespace {

// The checks of a group plan's call: the plan's pools with these kvs and
// layout, and kvs holding at least the plan's device pages.
int check_plan_call(const hicache_group_plan *plan, const hicache_device_kv *kvs, int32_t layout,
                    int32_t *lay) {
  if (!plan) return set_error(HICACHE_ERR_INVALID_ARG, "plan is NULL");
  int64_t Hp = 0, Dp = 0, max_run = 0;
  int rc = check_group(plan->pools.data(), kvs, int32_t(plan->pools.size()), layout, lay, &Hp, &Dp, &max_run,
                       true, plan->device_num_pages);
  if (rc) return rc;
  return check_device(plan->pools[0]);
}

}  // namespace

extern "C" {

int hicache_group_plan_create(hicache_pool *const *pools, int32_t npools, const int64_t *device_pages,
                              const int64_t *host_pages, int64_t n, int64_t device_num_pages,
                              hicache_group_plan **out) {
  clear_error();
  if (!out) return set_error(HICACHE_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  int32_t lay = 0;
  int64_t Hp = 0, Dp = 0, max_run = 0;
  int rc = check_group(pools, nullptr, npools, HICACHE_LAYOUT_POOL, &lay, &Hp, &Dp, &max_run, false);
  if (rc) return rc;
  std::vector<RunRec> runs;
  if ((rc = prepass(Hp, device_num_pages, device_pages, host_pages, n, HICACHE_DIR_LOAD, max_run, &runs)))
    return rc;
  hicache_group_plan *p = new (std::nothrow) hicache_group_plan();
  if (!p) return set_error(HICACHE_ERR_NOMEM, "out of host memory");
  p->pools.assign(pools, pools + npools);
  p->n = n;
  p->device_num_pages = device_num_pages;
  p->Hp = Hp;
  p->runs = std::move(runs);
  *out = p;
  return HICACHE_OK;
}

int hicache_group_plan_execute(const hicache_group_plan *plan, const hicache_device_kv *kvs, int32_t layout,
                               int32_t layer_id, void *stream) {
  clear_error();
  int32_t lay = 0;
  int rc = check_plan_call(plan, kvs, layout, &lay);
  if (rc) return rc;
  hicache_pool *const *pools = plan->pools.data();
  const int32_t np = int32_t(plan->pools.size());
  if (layer_id >= pools[0]->shape.L)
    return set_error(HICACHE_ERR_INVALID_ARG, "layer_id %d outside [0, %lld)", layer_id,
                     (long long)pools[0]->shape.L);
  if ((rc = enqueue_group(pools, kvs, np, plan->runs, lay, layer_id < 0 ? -1 : layer_id, false, stream)))
    return rc;
  if (layer_id >= 0) {
    for (int32_t i = 0; i < np; ++i) {
      hicache_pool *p = pools[i];
      const cudaError_t e = cudaEventRecord(p->events[size_t(layer_id)], static_cast<cudaStream_t>(stream));
      if (e != cudaSuccess) return cuda_error(e, "cudaEventRecord(layer event)");
      std::lock_guard<std::mutex> g(p->signal_mu);
      p->layer_signal[size_t(layer_id)] = 0;
    }
  } else if (!plan->runs.empty()) {
    for (int32_t i = 0; i < np; ++i)
      if ((rc = mark_all_layer_load(pools[i], stream))) return rc;
  }
  return HICACHE_OK;
}

int hicache_group_plan_load_layer_chained(hicache_group_plan *plan, const hicache_device_kv *kvs,
                                          int32_t layout, int32_t layer_id, void *stream) {
  clear_error();
  int32_t lay = 0;
  int rc = check_plan_call(plan, kvs, layout, &lay);
  if (rc) return rc;
  hicache_pool *const *pools = plan->pools.data();
  const int32_t np = int32_t(plan->pools.size());
  const int64_t L = pools[0]->shape.L;
  if (layer_id < 0 || layer_id >= L)
    return set_error(HICACHE_ERR_INVALID_ARG, "layer_id %d outside [0, %lld)", layer_id, (long long)L);
  if ((rc = refuse_capture(stream))) return rc;
  if (!wait_value32())
    return set_error(HICACHE_ERR_CUDA, "the driver offers no cuStreamWaitValue32: no chained loads");
  std::lock_guard<std::mutex> g(plan->chain_mu);
  std::vector<void *> bufs;
  std::vector<int64_t> pages;
  for (int32_t i = 0; i < np; ++i) {
    bufs.insert(bufs.end(), kvs[i].buf_ptrs, kvs[i].buf_ptrs + pools[i]->shape.B * L);
    pages.push_back(kvs[i].device_num_pages);
  }
  if (plan->chain_bufs != bufs || plan->chain_pages != pages) {
    // consecutive layers' launches overlap: no two buffers of the group may share bytes
    std::vector<std::pair<uintptr_t, uint64_t>> spans;
    for (int32_t i = 0; i < np; ++i) {
      const Shape &s = pools[i]->shape;
      const uint64_t bytes = uint64_t(kvs[i].device_num_pages) * uint64_t(s.PV) * 16u;
      for (int64_t b = 0; b < s.B * s.L; ++b)
        spans.emplace_back(reinterpret_cast<uintptr_t>(kvs[i].buf_ptrs[b]), bytes);
    }
    if ((rc = check_disjoint(spans))) return rc;
    plan->chain_bufs = bufs;
    plan->chain_pages = pages;
    plan->chain_layer = -1;
  }
  const bool chained = plan->chain_layer >= 0 && plan->chain_stream == stream &&
                       layer_id == plan->chain_layer + 1;
  // every pool's signal lock, in address order (the pools are distinct); the
  // pools' counted loads share their counters: one stream at a time
  std::vector<hicache_pool *> order(pools, pools + np);
  std::sort(order.begin(), order.end());
  std::vector<std::unique_lock<std::mutex>> locks;
  for (hicache_pool *p : order) locks.emplace_back(p->signal_mu);
  for (int32_t i = 0; i < np; ++i)
    if ((rc = check_counted_stream(pools[i], stream))) return rc;
  for (int32_t i = 0; i < np; ++i) claim_counted_stream(pools[i], stream);
  int64_t signalled = 0;
  rc = enqueue_group(pools, kvs, np, plan->runs, lay, layer_id, false, stream, chained, true, &signalled);
  plan->chain_stream = stream;
  plan->chain_layer = rc == HICACHE_OK && layer_id + 1 < L ? layer_id : -1;
  for (int32_t i = 0; i < np; ++i) {
    pools[i]->layer_target[size_t(layer_id)] += uint32_t(signalled);
    pools[i]->layer_signal[size_t(layer_id)] = 1;
    pools[i]->chain_open = true;
  }
  if (rc != HICACHE_OK) return rc;
  if (layer_id + 1 == L) {
    for (int32_t i = 0; i < np; ++i) {
      const cudaError_t e = cudaEventRecord(pools[i]->pipeline_last, static_cast<cudaStream_t>(stream));
      if (e != cudaSuccess) return cuda_error(e, "cudaEventRecord(chained load)");
      pools[i]->chain_open = false;
    }
  }
  return HICACHE_OK;
}

int hicache_group_plan_load_layers(hicache_group_plan *plan, const hicache_device_kv *kvs, int32_t layout,
                                   void *stream) {
  clear_error();
  int32_t lay = 0;
  int rc = check_plan_call(plan, kvs, layout, &lay);
  if (rc) return rc;
  hicache_pool *const *pools = plan->pools.data();
  const int32_t np = int32_t(plan->pools.size());
  const int64_t L = pools[0]->shape.L;
  std::lock_guard<std::mutex> g(plan->graph_mu);
  std::vector<void *> bufs;
  std::vector<int64_t> pages;
  for (int32_t i = 0; i < np; ++i) {
    bufs.insert(bufs.end(), kvs[i].buf_ptrs, kvs[i].buf_ptrs + pools[i]->shape.B * L);
    pages.push_back(kvs[i].device_num_pages);
  }
  if (!plan->graph || plan->graph_bufs != bufs || plan->graph_pages != pages || plan->graph_layout != lay) {
    std::vector<std::pair<uintptr_t, uint64_t>> spans;
    for (int32_t i = 0; i < np; ++i) {
      const Shape &s = pools[i]->shape;
      const uint64_t bytes = uint64_t(kvs[i].device_num_pages) * uint64_t(s.PV) * 16u;
      for (int64_t b = 0; b < s.B * s.L; ++b)
        spans.emplace_back(reinterpret_cast<uintptr_t>(kvs[i].buf_ptrs[b]), bytes);
    }
    if ((rc = check_disjoint(spans))) return rc;
    if (plan->graph) {
      cudaGraphExecDestroy(plan->graph);
      plan->graph = nullptr;
    }
    int64_t launches = 0;
    rc = capture_layer_graph(
        pools, np, L,
        [&](int64_t l, void *cap) {
          return enqueue_group(pools, kvs, np, plan->runs, lay, int32_t(l), false, cap, l > 0);
        },
        &plan->graph, &launches);
    if (rc != HICACHE_OK) return rc;
    plan->graph_bufs = bufs;
    plan->graph_pages = pages;
    plan->graph_layout = lay;
    plan->graph_launches = launches;
  }
  return launch_layer_graph(plan->graph, plan->graph_launches, pools, np, stream);
}

int hicache_group_plan_destroy(hicache_group_plan *plan) {
  if (plan && plan->graph) cudaGraphExecDestroy(plan->graph);
  delete plan;
  return HICACHE_OK;
}

}  // extern "C"
