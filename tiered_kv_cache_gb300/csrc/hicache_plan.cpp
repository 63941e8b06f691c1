// hicache_plan.cpp -- plans: an index set validated and reduced to runs once,
// then executed many times (all layers, one layer, pipelined, or every layer's
// launch replayed from one CUDA graph).

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <functional>
#include <mutex>
#include <new>
#include <utility>
#include <vector>

#include "hicache.h"
#include "hicache_host.h"
#include "hicache_internal.h"

using namespace hicache;

struct hicache_plan {
  hicache_pool *pool = nullptr;
  int32_t direction = 0;
  int64_t n = 0;
  int64_t device_num_pages = 0;
  std::vector<hicache::RunRec> runs;
  // hicache_plan_load_layers: the per-layer launches and layer events of one
  // device KV and layout, captured once as a CUDA graph and replayed
  std::mutex graph_mu;
  cudaGraphExec_t graph = nullptr;
  std::vector<void *> graph_bufs;     // the key: buffer pointers, page count, layout
  int64_t graph_pages = 0;
  int32_t graph_layout = -1;
  int64_t graph_launches = 0;         // kernel launches one replay makes
  // hicache_plan_load_layer_chained: the stream and layer of the last chained
  // call, and the device KV whose buffers were found disjoint
  std::mutex chain_mu;
  void *chain_stream = nullptr;
  int32_t chain_layer = -1;
  std::vector<void *> chain_bufs;
  int64_t chain_pages = 0;
};

namespace hicache {

int check_disjoint(std::vector<std::pair<uintptr_t, uint64_t>> spans) {
  std::sort(spans.begin(), spans.end());
  for (size_t i = 1; i < spans.size(); ++i)
    if (spans[i].first - spans[i - 1].first < spans[i - 1].second)
      return set_error(HICACHE_ERR_INVALID_ARG,
                       "device buffers overlap: each of the %zu buffers needs its own bytes", spans.size());
  return HICACHE_OK;
}

int capture_layer_graph(hicache_pool *const *pools, int32_t np, int64_t L,
                        const std::function<int(int64_t, void *)> &enqueue_layer, cudaGraphExec_t *out,
                        int64_t *launches) {
  // Capture the L layers' launches on a private stream, one after another.
  // Each layer's events are recorded (as external event nodes) on a side
  // branch that forks off after that layer's launches, so the kernel chain
  // itself has no node between consecutive launches.  Every kernel after the
  // first is a programmatic dependent launch: it may start as the previous
  // kernel moves its last tiles (the layers write different buffers and only
  // read the host pool) and ends after it.  A layer's event nodes follow that
  // layer's last kernel and the event nodes before them, so event l means
  // layers 0..l have landed.
  *out = nullptr;
  *launches = 0;
  cudaStream_t cap = nullptr, side = nullptr;
  std::vector<cudaEvent_t> forks(size_t(L) + 1, nullptr);
  cudaError_t e = cudaStreamCreateWithFlags(&cap, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&side, cudaStreamNonBlocking);
  for (auto &f : forks)
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&f, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaStreamBeginCapture(cap, cudaStreamCaptureModeThreadLocal);
  auto release = [&] {
    for (auto f : forks)
      if (f) cudaEventDestroy(f);
    if (side) cudaStreamDestroy(side);
    if (cap) cudaStreamDestroy(cap);
  };
  if (e != cudaSuccess) {
    release();
    return cuda_error(e, "setting up the layer-load capture");
  }
  int rc = HICACHE_OK;
  const int64_t before = g_launches.load();
  for (int64_t l = 0; l < L && rc == HICACHE_OK; ++l) {
    rc = enqueue_layer(l, cap);
    if (rc != HICACHE_OK) break;
    e = cudaEventRecord(forks[size_t(l)], cap);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(side, forks[size_t(l)], 0);
    for (int32_t i = 0; i < np && e == cudaSuccess; ++i)
      e = cudaEventRecordWithFlags(pools[i]->events[size_t(l)], side, cudaEventRecordExternal);
    if (e != cudaSuccess) rc = cuda_error(e, "capturing the layer events");
  }
  if (rc == HICACHE_OK) {                // join the side branch back
    e = cudaEventRecord(forks[size_t(L)], side);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cap, forks[size_t(L)], 0);
    if (e != cudaSuccess) rc = cuda_error(e, "joining the capture");
  }
  const int64_t captured = g_launches.load() - before;
  g_launches.fetch_sub(captured);        // counted when replayed
  cudaGraph_t graph = nullptr;
  e = cudaStreamEndCapture(cap, &graph);
  release();
  if (rc == HICACHE_OK && e != cudaSuccess) rc = cuda_error(e, "cudaStreamEndCapture");
  if (rc == HICACHE_OK) {
    e = cudaGraphInstantiate(out, graph, 0);
    if (e != cudaSuccess) {
      *out = nullptr;
      rc = cuda_error(e, "cudaGraphInstantiate");
    }
  }
  if (graph) cudaGraphDestroy(graph);
  if (rc == HICACHE_OK) *launches = captured;
  return rc;
}

int launch_layer_graph(cudaGraphExec_t graph, int64_t launches, hicache_pool *const *pools, int32_t np,
                       void *stream) {
  const cudaError_t e = cudaGraphLaunch(graph, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_error(e, "cudaGraphLaunch");
  g_launches.fetch_add(launches, std::memory_order_relaxed);
  for (int32_t i = 0; i < np; ++i) {     // hicache_wait_layer uses the events
    std::lock_guard<std::mutex> g(pools[i]->signal_mu);
    for (auto &sig : pools[i]->layer_signal) sig = 0;
  }
  return HICACHE_OK;
}

}  // namespace hicache

extern "C" {

int hicache_plan_create(hicache_pool *pool, const int64_t *device_pages, const int64_t *host_pages,
                        int64_t n, int64_t device_num_pages, int32_t direction,
                        hicache_plan **out) {
  clear_error();
  if (!pool || !out) return set_error(HICACHE_ERR_INVALID_ARG, "pool or out is NULL");
  *out = nullptr;
  std::vector<RunRec> runs;
  int rc = prepass(pool->shape.Hp, device_num_pages, device_pages, host_pages, n, direction,
                   max_run_pages(pool->shape), &runs);
  if (rc) return rc;
  hicache_plan *p = new (std::nothrow) hicache_plan();
  if (!p) return set_error(HICACHE_ERR_NOMEM, "out of host memory");
  p->pool = pool;
  p->direction = direction;
  p->n = n;
  p->device_num_pages = device_num_pages;
  p->runs = std::move(runs);
  *out = p;
  return HICACHE_OK;
}

int hicache_plan_execute(const hicache_plan *plan, const hicache_device_kv *kv, int32_t layout,
                         int32_t layer_id, void *stream) {
  clear_error();
  if (!plan) return set_error(HICACHE_ERR_INVALID_ARG, "plan is NULL");
  hicache_pool *pool = plan->pool;
  int32_t lay = 0;
  int rc = resolve_layout(layout, pool->shape.layout, &lay);
  if (rc) return rc;
  if (layer_id >= pool->shape.L)
    return set_error(HICACHE_ERR_INVALID_ARG, "layer_id %d outside [0, %lld)", layer_id,
                     (long long)pool->shape.L);
  if (layer_id >= 0 && plan->direction != HICACHE_DIR_LOAD)
    return set_error(HICACHE_ERR_INVALID_ARG, "a per-layer transfer must be a load");
  if ((rc = check_kv(pool, kv, plan->device_num_pages))) return rc;
  if ((rc = enqueue(pool, kv, plan->runs, nullptr, lay, layer_id < 0 ? -1 : layer_id,
                    plan->direction == HICACHE_DIR_BACKUP, stream)))
    return rc;
  if (layer_id >= 0) {
    const cudaError_t e =
        cudaEventRecord(pool->events[size_t(layer_id)], static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_error(e, "cudaEventRecord(layer event)");
    std::lock_guard<std::mutex> g(pool->signal_mu);
    pool->layer_signal[size_t(layer_id)] = 0;
  } else if (plan->direction == HICACHE_DIR_LOAD && plan->n > 0) {
    return mark_all_layer_load(pool, stream);
  }
  return HICACHE_OK;
}

int hicache_plan_load_layer(const hicache_plan *plan, const hicache_device_kv *kv, int32_t layout,
                            int32_t layer_id, void *stream) {
  clear_error();
  if (layer_id < 0) return set_error(HICACHE_ERR_INVALID_ARG, "layer_id %d is negative", layer_id);
  return hicache_plan_execute(plan, kv, layout, layer_id, stream);
}

int hicache_plan_load_layer_chained(hicache_plan *plan, const hicache_device_kv *kv, int32_t layout,
                                    int32_t layer_id, void *stream) {
  clear_error();
  if (!plan) return set_error(HICACHE_ERR_INVALID_ARG, "plan is NULL");
  if (plan->direction != HICACHE_DIR_LOAD)
    return set_error(HICACHE_ERR_INVALID_ARG, "a per-layer transfer must be a load");
  hicache_pool *pool = plan->pool;
  const Shape &s = pool->shape;
  if (layer_id < 0 || layer_id >= s.L)
    return set_error(HICACHE_ERR_INVALID_ARG, "layer_id %d outside [0, %lld)", layer_id, (long long)s.L);
  int32_t lay = 0;
  int rc = resolve_layout(layout, s.layout, &lay);
  if (rc) return rc;
  if ((rc = check_kv(pool, kv, plan->device_num_pages))) return rc;
  if ((rc = check_device(pool))) return rc;
  if ((rc = refuse_capture(stream))) return rc;
  if (!wait_value32())
    return set_error(HICACHE_ERR_CUDA, "the driver offers no cuStreamWaitValue32: no chained loads");
  std::lock_guard<std::mutex> g(plan->chain_mu);
  // consecutive layers' kernels overlap, so no two buffers may share bytes
  // (checked once per set of buffers)
  const std::vector<void *> bufs(kv->buf_ptrs, kv->buf_ptrs + s.B * s.L);
  if (plan->chain_bufs != bufs || plan->chain_pages != kv->device_num_pages) {
    std::vector<std::pair<uintptr_t, uint64_t>> spans;
    const uint64_t buf_bytes = uint64_t(kv->device_num_pages) * uint64_t(s.PV) * 16u;
    for (void *b : bufs) spans.emplace_back(reinterpret_cast<uintptr_t>(b), buf_bytes);
    if ((rc = check_disjoint(spans))) return rc;
    plan->chain_bufs = bufs;
    plan->chain_pages = kv->device_num_pages;
    plan->chain_layer = -1;
  }
  // the call continues a chain when it loads the layer after the plan's
  // previous chained call, on the same stream: its kernel then starts as that
  // layer's kernel drains, with nothing in between on the stream
  const bool chained = plan->chain_layer >= 0 && plan->chain_stream == stream &&
                       layer_id == plan->chain_layer + 1;
  // the pool's counted loads share its counters: one stream at a time
  std::lock_guard<std::mutex> gs(pool->signal_mu);
  if ((rc = check_counted_stream(pool, stream))) return rc;
  claim_counted_stream(pool, stream);
  int64_t signalled = 0;
  rc = enqueue(pool, kv, plan->runs, nullptr, lay, layer_id, false, stream, chained,
               pool->layer_done + layer_id, &signalled);
  plan->chain_stream = stream;
  plan->chain_layer = rc == HICACHE_OK && layer_id + 1 < s.L ? layer_id : -1;
  // the launches that went out count towards the layer, even if a later one failed
  pool->layer_target[size_t(layer_id)] += uint32_t(signalled);
  pool->layer_signal[size_t(layer_id)] = 1;
  pool->chain_open = true;
  if (rc != HICACHE_OK) return rc;
  if (layer_id + 1 == s.L) {
    // the pool's counted-load event, behind the last layer's kernel, closes the chain
    const cudaError_t e = cudaEventRecord(pool->pipeline_last, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_error(e, "cudaEventRecord(chained load)");
    pool->chain_open = false;
  }
  return HICACHE_OK;
}

int hicache_plan_load_pipelined(const hicache_plan *plan, const hicache_device_kv *kv, int32_t layout,
                                void *stream) {
  clear_error();
  if (!plan) return set_error(HICACHE_ERR_INVALID_ARG, "plan is NULL");
  if (plan->direction != HICACHE_DIR_LOAD)
    return set_error(HICACHE_ERR_INVALID_ARG, "a pipelined transfer must be a load");
  int32_t lay = 0;
  int rc = resolve_layout(layout, plan->pool->shape.layout, &lay);
  if (rc) return rc;
  if ((rc = check_kv(plan->pool, kv, plan->device_num_pages))) return rc;
  return enqueue_pipelined(plan->pool, kv, plan->runs, lay, stream);
}

int hicache_plan_info(const hicache_plan *plan, int64_t *num_pages, int64_t *num_runs) {
  clear_error();
  if (!plan) return set_error(HICACHE_ERR_INVALID_ARG, "plan is NULL");
  if (num_pages) *num_pages = plan->n;
  if (num_runs) *num_runs = int64_t(plan->runs.size());
  return HICACHE_OK;
}

int hicache_plan_load_layers(hicache_plan *plan, const hicache_device_kv *kv, int32_t layout, void *stream) {
  clear_error();
  if (!plan) return set_error(HICACHE_ERR_INVALID_ARG, "plan is NULL");
  if (plan->direction != HICACHE_DIR_LOAD)
    return set_error(HICACHE_ERR_INVALID_ARG, "a per-layer transfer must be a load");
  hicache_pool *pool = plan->pool;
  const Shape &s = pool->shape;
  int32_t lay = 0;
  int rc = resolve_layout(layout, s.layout, &lay);
  if (rc) return rc;
  if ((rc = check_kv(pool, kv, plan->device_num_pages))) return rc;
  if ((rc = check_device(pool))) return rc;
  std::lock_guard<std::mutex> g(plan->graph_mu);
  const std::vector<void *> bufs(kv->buf_ptrs, kv->buf_ptrs + s.B * s.L);
  if (!plan->graph || plan->graph_bufs != bufs || plan->graph_pages != kv->device_num_pages ||
      plan->graph_layout != lay) {
    std::vector<std::pair<uintptr_t, uint64_t>> spans;
    const uint64_t buf_bytes = uint64_t(kv->device_num_pages) * uint64_t(s.PV) * 16u;
    for (void *b : bufs) spans.emplace_back(reinterpret_cast<uintptr_t>(b), buf_bytes);
    if ((rc = check_disjoint(spans))) return rc;
    if (plan->graph) {
      cudaGraphExecDestroy(plan->graph);
      plan->graph = nullptr;
    }
    int64_t launches = 0;
    rc = capture_layer_graph(
        &pool, 1, s.L,
        [&](int64_t l, void *cap) { return enqueue(pool, kv, plan->runs, nullptr, lay, int32_t(l), false, cap, l > 0); },
        &plan->graph, &launches);
    if (rc != HICACHE_OK) return rc;
    plan->graph_bufs = bufs;
    plan->graph_pages = kv->device_num_pages;
    plan->graph_layout = lay;
    plan->graph_launches = launches;
  }
  return launch_layer_graph(plan->graph, plan->graph_launches, &pool, 1, stream);
}

int hicache_plan_destroy(hicache_plan *plan) {
  if (plan && plan->graph) cudaGraphExecDestroy(plan->graph);
  delete plan;
  return HICACHE_OK;
}

}  // extern "C"
