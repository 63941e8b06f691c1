// hicache_pipeline.cpp -- pipelined loads: every layer in one launch, each
// layer counted on the device as it lands, and the per-layer waits that let
// compute start on a layer before the rest of the load is in (through the
// layer's counter, or its event for per-layer launches).

#include <cuda.h>  // driver types for the stream memory wait (fetched at run time)
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "hicache.h"
#include "hicache_host.h"
#include "hicache_internal.h"

namespace hicache {

// cuStreamWaitValue32 from the driver, fetched through the runtime (no link
// against the driver library); nullptr if the driver does not offer it.
WaitValue32Fn wait_value32() {
  static WaitValue32Fn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuStreamWaitValue32", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<WaitValue32Fn>(p);
  });
  return fn;
}

// Pipelined loads raise each layer's target on the host when the call is
// enqueued, while the device counters rise each time the kernel runs.  A call
// captured into a graph would raise the targets once however often the graph
// is replayed (and never catch up if it is not launched), so hicache_wait_layer
// would pass too early or wait forever.  They refuse a capturing stream.
int refuse_capture(void *stream) {
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  const cudaError_t e = cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &st);
  if (e != cudaSuccess) return cuda_error(e, "cudaStreamIsCapturing");
  if (st != cudaStreamCaptureStatusNone)
    return set_error(HICACHE_ERR_INVALID_ARG,
                     "pipelined loads cannot be captured: their per-layer targets are kept on the host");
  return HICACHE_OK;
}

int check_counted_stream(hicache_pool *pool, void *stream) {
  if (!pool->pipeline_stream_set || pool->pipeline_stream == stream) return HICACHE_OK;
  if (pool->chain_open)
    return set_error(HICACHE_ERR_INVALID_ARG,
                     "a chained per-layer load of this pool on another stream has not reached its last layer");
  if (cudaEventQuery(pool->pipeline_last) != cudaSuccess) {
    (void)cudaGetLastError();
    return set_error(HICACHE_ERR_INVALID_ARG,
                     "a pipelined load of this pool is still running on another stream");
  }
  return HICACHE_OK;
}

void claim_counted_stream(hicache_pool *pool, void *stream) {
  pool->pipeline_stream_set = true;
  pool->pipeline_stream = stream;
}

int enqueue_pipelined(hicache_pool *pool, const hicache_device_kv *kv, const std::vector<RunRec> &runs,
                      int32_t layout, void *stream) {
  if (int rc = check_device(pool)) return rc;
  if (int rc = refuse_capture(stream)) return rc;
  if (!wait_value32())
    return set_error(HICACHE_ERR_CUDA, "the driver offers no cuStreamWaitValue32: no pipelined loads");
  std::lock_guard<std::mutex> g(pool->signal_mu);
  // the counts stay in order while counted loads follow one another on one
  // stream; another stream is fine once the earlier ones have finished
  if (int rc = check_counted_stream(pool, stream)) return rc;
  claim_counted_stream(pool, stream);
  const Shape &s = pool->shape;
  const int32_t nb = int32_t(s.B * s.L);
  thread_local hicache::XferParams params;
  fill_header(pool, kv, params, s.PV, 0);
  size_t next = 0;
  while (next < runs.size()) {
    // one layer's units are (buffer, run); the launch covers L layers of them
    const int32_t c = fill_job(runs, next, s.PV, s.B, (hicache::kBlobWords - nb) / 2, params, nb, 0, s.L);
    if (c < 0) return set_error(HICACHE_ERR_INVALID_ARG, "transfer too large for one launch");
    hicache::XferLaunch x;
    x.params = &params;
    x.words = nb + 2 * c;
    x.layout = layout;
    x.all_layers = false;
    x.to_host = false;
    x.bidir = false;
    x.grid = int(std::min<int64_t>(int64_t(params.h.job[0].total_tiles) * s.L, pool->layer_ctas));
    x.stream = stream;
    const int e = hicache::launch_pipelined_load(x, pool->layer_done, pool->layer_done + s.L);
    if (e != 0) return cuda_error(cudaError_t(e), "pipelined load kernel launch");
    g_launches.fetch_add(1, std::memory_order_relaxed);
    for (int64_t l = 0; l < s.L; ++l) {
      pool->layer_target[size_t(l)] += uint32_t(params.h.job[0].total_tiles);
      pool->layer_signal[size_t(l)] = 1;
    }
    next += size_t(c);
  }
  // (the layer events are recorded when asked for: hicache_layer_event)
  const cudaError_t e = cudaEventRecord(pool->pipeline_last, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_error(e, "cudaEventRecord(pipelined load)");
  pool->chain_open = false;            // the event covers any chain before it on this stream
  return HICACHE_OK;
}

// ---- allocation-free pipelined load ---------------------------------------------
namespace {
// The value the library's static counters reach once every allocation-free
// pipelined load enqueued so far on a device has landed, per device and layer.
std::mutex g_noalloc_mu;
uint32_t g_noalloc_target[hicache::kNoAllocMaxDevices][hicache::kNoAllocMaxLayers];
uint32_t g_noalloc_slot[hicache::kNoAllocMaxDevices];  // next scheduler pair, per device
}  // namespace

int record_counted_layer_event(hicache_pool *pool, int64_t layer) {
  if (!pool->event_stream) {
    const cudaError_t e = cudaStreamCreateWithFlags(&pool->event_stream, cudaStreamNonBlocking);
    if (e != cudaSuccess) {
      pool->event_stream = nullptr;
      return cuda_error(e, "cudaStreamCreateWithFlags(event stream)");
    }
  }
  const bool noalloc = pool->layer_signal[size_t(layer)] == 2;
  unsigned int *counter = (noalloc ? pool->noalloc_done : pool->layer_done) + layer;
  const uint32_t target = noalloc ? pool->noalloc_target[size_t(layer)] : pool->layer_target[size_t(layer)];
  const CUresult r = wait_value32()(static_cast<CUstream>(pool->event_stream),
                                    reinterpret_cast<CUdeviceptr>(counter), target, CU_STREAM_WAIT_VALUE_GEQ);
  if (r != CUDA_SUCCESS) return set_error(HICACHE_ERR_CUDA, "cuStreamWaitValue32 failed (%d)", int(r));
  const cudaError_t e = cudaEventRecord(pool->events[size_t(layer)], pool->event_stream);
  if (e != cudaSuccess) return cuda_error(e, "cudaEventRecord(layer event)");
  return HICACHE_OK;
}

}  // namespace hicache

using namespace hicache;

extern "C" {

int hicache_load_pipelined(hicache_pool *pool, const hicache_device_kv *kv, const int64_t *device_pages,
                           const int64_t *host_pages, int64_t n, int32_t layout, void *stream) {
  clear_error();
  if (!pool) return set_error(HICACHE_ERR_INVALID_ARG, "pool is NULL");
  int32_t lay = 0;
  int rc = resolve_layout(layout, pool->shape.layout, &lay);
  if (rc) return rc;
  if ((rc = check_kv(pool, kv, 0))) return rc;
  thread_local std::vector<RunRec> runs;
  if ((rc = prepass(pool->shape.Hp, kv->device_num_pages, device_pages, host_pages, n, HICACHE_DIR_LOAD,
                    max_run_pages(pool->shape), &runs)))
    return rc;
  return enqueue_pipelined(pool, kv, runs, lay, stream);
}

int hicache_pipeline_status(hicache_pool *pool, int32_t layer, uint32_t *done, uint32_t *target) {
  clear_error();
  if (!pool || !done || !target) return set_error(HICACHE_ERR_INVALID_ARG, "NULL argument");
  if (layer < 0 || layer >= pool->shape.L)
    return set_error(HICACHE_ERR_INVALID_ARG, "layer %d outside [0, %lld)", layer, (long long)pool->shape.L);
  unsigned int v = 0;
  const cudaError_t e = cudaMemcpy(&v, pool->layer_done + layer, sizeof v, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_error(e, "cudaMemcpy(layer counter)");
  std::lock_guard<std::mutex> g(pool->signal_mu);
  *done = v;
  *target = pool->layer_target[size_t(layer)];
  return HICACHE_OK;
}

int hicache_load_pipelined_noalloc(hicache_pool *pool, const hicache_device_kv *kv,
                                   const int64_t *device_pages, const int64_t *host_pages, int64_t n,
                                   int32_t layout, void *stream) {
  clear_error();
  if (!pool) return set_error(HICACHE_ERR_INVALID_ARG, "pool is NULL");
  const Shape &s = pool->shape;
  if (s.L > hicache::kNoAllocMaxLayers)
    return set_error(HICACHE_ERR_INVALID_ARG,
                     "the allocation-free pipelined load takes at most %d layers; this pool has %lld",
                     hicache::kNoAllocMaxLayers, (long long)s.L);
  int32_t lay = 0;
  int rc = resolve_layout(layout, s.layout, &lay);
  if (rc) return rc;
  if ((rc = check_kv(pool, kv, 0))) return rc;
  thread_local std::vector<RunRec> runs;
  if ((rc = prepass(s.Hp, kv->device_num_pages, device_pages, host_pages, n, HICACHE_DIR_LOAD,
                    max_run_pages(s), &runs)))
    return rc;
  if ((rc = check_device(pool))) return rc;
  if ((rc = refuse_capture(stream))) return rc;
  if (!wait_value32())
    return set_error(HICACHE_ERR_CUDA, "the driver offers no cuStreamWaitValue32: no pipelined loads");
  unsigned int *counters = nullptr;
  const int ce = hicache::noalloc_layer_counters(&counters);
  if (ce != 0) return cuda_error(cudaError_t(ce), "address of the static layer counters");
  const int32_t nb = int32_t(s.B * s.L);
  thread_local hicache::XferParams params;
  fill_header(pool, kv, params, s.PV, 0);
  std::lock_guard<std::mutex> gg(g_noalloc_mu);
  std::lock_guard<std::mutex> g(pool->signal_mu);
  uint32_t *target = g_noalloc_target[pool->device];
  pool->noalloc_done = counters;
  if (pool->noalloc_target.size() != size_t(s.L)) pool->noalloc_target.assign(size_t(s.L), 0);
  size_t next = 0;
  while (next < runs.size()) {
    const int32_t c = fill_job(runs, next, s.PV, s.B, (hicache::kBlobWords - nb) / 2, params, nb, 0, s.L);
    if (c < 0) return set_error(HICACHE_ERR_INVALID_ARG, "transfer too large for one launch");
    hicache::XferLaunch x;
    x.params = &params;
    x.words = nb + 2 * c;
    x.layout = lay;
    x.all_layers = false;
    x.to_host = false;
    x.bidir = false;
    x.grid = int(std::min<int64_t>(int64_t(params.h.job[0].total_tiles) * s.L, pool->layer_ctas));
    x.stream = stream;
    unsigned int *sched = counters + hicache::kNoAllocMaxLayers +
                          2 * (g_noalloc_slot[pool->device]++ % hicache::kNoAllocSchedSlots);
    const int e = hicache::launch_pipelined_load(x, counters, sched);
    if (e != 0) return cuda_error(cudaError_t(e), "pipelined load kernel launch");
    g_launches.fetch_add(1, std::memory_order_relaxed);
    // the targets follow every launch that went out, so that a launch error
    // later in a split call leaves waits that cover the launches before it
    for (int64_t l = 0; l < s.L; ++l) {
      target[l] += uint32_t(params.h.job[0].total_tiles);
      pool->noalloc_target[size_t(l)] = target[l];
      pool->layer_signal[size_t(l)] = 2;
    }
    next += size_t(c);
  }
  for (int64_t l = 0; l < s.L; ++l) {
    const cudaError_t e = cudaEventRecord(pool->events[size_t(l)], static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_error(e, "cudaEventRecord(layer event)");
  }
  return HICACHE_OK;
}

int hicache_wait_layer(hicache_pool *pool, int32_t layer, void *compute_stream) {
  clear_error();
  if (!pool) return set_error(HICACHE_ERR_INVALID_ARG, "pool is NULL");
  if (layer < 0 || layer >= pool->shape.L)
    return set_error(HICACHE_ERR_INVALID_ARG, "layer %d outside [0, %lld)", layer,
                     (long long)pool->shape.L);
  std::lock_guard<std::mutex> g(pool->signal_mu);
  const uint8_t sig = pool->layer_signal[size_t(layer)];
  cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
  if (sig == 1 || sig == 2) {
    const cudaError_t ce = cudaStreamIsCapturing(static_cast<cudaStream_t>(compute_stream), &capture);
    if (ce != cudaSuccess) return cuda_error(ce, "cudaStreamIsCapturing");
  }
  if ((sig == 1 || sig == 2) && capture == cudaStreamCaptureStatusNone) {
    // A load signalled on the device: the stream memory wait goes on the
    // pool's event stream and the compute stream waits for the event it
    // records.  A kernel queued right behind a stream memory wait starts
    // late; behind an event wait it does not (61 layers at 4K tokens:
    // attention done 1.41-1.45 ms after the first call, against 1.61-1.66).
    int rc = check_device(pool);
    if (rc) return rc;
    if ((rc = record_counted_layer_event(pool, layer))) return rc;
    const cudaError_t e =
        cudaStreamWaitEvent(static_cast<cudaStream_t>(compute_stream), pool->events[size_t(layer)], 0);
    if (e != cudaSuccess) return cuda_error(e, "cudaStreamWaitEvent");
    return HICACHE_OK;
  }
  // a capturing compute stream takes the stream memory wait itself
  if (pool->layer_signal[size_t(layer)] == 2) {
    // the last load of this layer was an allocation-free pipelined load
    const CUresult r = wait_value32()(static_cast<CUstream>(compute_stream),
                                      reinterpret_cast<CUdeviceptr>(pool->noalloc_done + layer),
                                      pool->noalloc_target[size_t(layer)], CU_STREAM_WAIT_VALUE_GEQ);
    if (r != CUDA_SUCCESS)
      return set_error(HICACHE_ERR_CUDA, "cuStreamWaitValue32 failed (%d)", int(r));
    return HICACHE_OK;
  }
  if (pool->layer_signal[size_t(layer)] == 1) {
    // the last load of this layer was pipelined: wait for its counter
    const CUresult r = wait_value32()(static_cast<CUstream>(compute_stream),
                                      reinterpret_cast<CUdeviceptr>(pool->layer_done + layer),
                                      pool->layer_target[size_t(layer)], CU_STREAM_WAIT_VALUE_GEQ);
    if (r != CUDA_SUCCESS)
      return set_error(HICACHE_ERR_CUDA, "cuStreamWaitValue32 failed (%d)", int(r));
    return HICACHE_OK;
  }
  // signal 3: the last load of this layer loaded every layer
  const cudaEvent_t ev = pool->layer_signal[size_t(layer)] == 3 ? pool->load_all : pool->events[size_t(layer)];
  const cudaError_t e = cudaStreamWaitEvent(static_cast<cudaStream_t>(compute_stream), ev, 0);
  if (e != cudaSuccess) return cuda_error(e, "cudaStreamWaitEvent");
  return HICACHE_OK;
}

}  // extern "C"
