// hicache_api.cpp -- host side of libhicache: errors, pinned host memory,
// pools, the launch of validated runs, backup / load / per-layer load / fused
// backup + load, layer events, bounded stream waits and the stand-in compute.
// The other host files: hicache_index.cpp (validation and the pre-pass),
// hicache_pipeline.cpp (pipelined loads and per-layer waits), hicache_plan.cpp
// (plans), hicache_group.cpp (buffer groups), hicache_engine.cpp (submission
// engine), hicache_alloc.cpp (host-page allocator).
//
// Every transfer call validates everything BEFORE it enqueues anything, so a
// call that fails has no effect.  Kernels are launched through
// hicache::launch_xfer (hicache_kernels.cu).

#include "hicache.h"

#include <cuda_runtime.h>
#include <sys/mman.h>
#include <unistd.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <climits>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <string>
#include <thread>
#include <unordered_map>
#include <vector>

#include "hicache_host.h"
#include "hicache_internal.h"

namespace hicache {

thread_local std::string g_last_error;
std::atomic<int64_t> g_launches{0};

int set_error(int code, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int cuda_error(cudaError_t e, const char *what) {
  return set_error(HICACHE_ERR_CUDA, "%s: %s (%d)", what, cudaGetErrorString(e), int(e));
}

// ---- pinned host allocations -------------------------------------------------
struct HostAlloc {
  size_t bytes;   // mapped length (THP allocations are rounded up to 2 MiB)
  bool thp;
};
std::mutex g_alloc_mu;
std::unordered_map<void *, HostAlloc> g_allocs;

void clear_error() { g_last_error.clear(); }

int set_error_text(int code, const char *msg) {
  g_last_error.clear();
  return set_error(code, "%s", msg);
}

int check_kv(const hicache_pool *pool, const hicache_device_kv *kv, int64_t min_pages) {
  if (!kv || !kv->buf_ptrs) return set_error(HICACHE_ERR_INVALID_ARG, "device KV is NULL");
  if (kv->device_num_pages < 1 || kv->device_num_pages >= INT32_MAX)
    return set_error(HICACHE_ERR_INVALID_ARG, "device_num_pages = %lld must be in [1, 2^31)",
                     (long long)kv->device_num_pages);
  if (kv->device_num_pages < min_pages)
    return set_error(HICACHE_ERR_INVALID_ARG, "device_num_pages = %lld is below the plan's %lld",
                     (long long)kv->device_num_pages, (long long)min_pages);
  const int64_t nb = pool->shape.B * pool->shape.L;
  for (int64_t i = 0; i < nb; ++i) {
    const void *p = kv->buf_ptrs[i];
    if (!p) return set_error(HICACHE_ERR_INVALID_ARG, "device buffer %lld is NULL", (long long)i);
    if (reinterpret_cast<uintptr_t>(p) % 16 != 0)
      return set_error(HICACHE_ERR_ALIGNMENT, "device buffer %lld is not 16-byte aligned",
                       (long long)i);
  }
  return HICACHE_OK;
}

// Copy runs[next..] into a job's run table (at blob word `word`): at most
// max_runs runs, fewer than 2^31 - 1024 vectors per outer unit (the kernels'
// 32-bit vector offsets), and kMaxTiles / launch_factor tiles (so the 32-bit
// tile index never overflows).  Returns the number of runs taken, or -1 if even
// one run is too large -- which the run cap of the pre-pass rules out.
int32_t fill_runs(const std::vector<RunRec> &runs, size_t next, int64_t upp, int64_t outers,
                  int64_t max_runs, hicache::Job &job, hicache::Run *table, int32_t word,
                  int64_t launch_factor) {
  int64_t vecs = 0;
  int32_t count = 0;
  bool uniform = true;
  while (next + size_t(count) < runs.size() && count < max_runs) {
    const RunRec &r = runs[next + size_t(count)];
    if (r.len != runs[next].len) uniform = false;
    const int64_t nv = vecs + r.len * upp;
    const int64_t tiles = (nv + hicache::kTileVecs - 1) / hicache::kTileVecs;
    if (nv > kMaxOuterVecs || tiles * outers * launch_factor > kMaxTiles) {
      if (count == 0) return -1;
      break;
    }
    table[count] = hicache::Run{int32_t(r.h0), int32_t(r.d0), int32_t(r.len), int32_t(vecs)};
    vecs = nv;
    ++count;
  }
  job.n_runs = count;
  job.runs_word = word;
  job.vecs_per_outer = uint32_t(vecs);
  // runs of one length: the kernel finds a vector's run by one division
  job.run_vecs = uniform && count > 0 ? uint32_t(runs[next].len * upp) : 0u;
  job.fd_run = hicache::make_fastdiv(job.run_vecs ? job.run_vecs : 1u);
  job.tiles_per_outer = int32_t((vecs + hicache::kTileVecs - 1) / hicache::kTileVecs);
  job.total_tiles = int32_t(job.tiles_per_outer * outers);
  return count;
}

int32_t fill_job(const std::vector<RunRec> &runs, size_t next, int64_t upp, int64_t outers,
                 int64_t max_runs, hicache::XferParams &params, int32_t word, int j,
                 int64_t launch_factor) {
  return fill_runs(runs, next, upp, outers, max_runs, params.h.job[j],
                   reinterpret_cast<hicache::Run *>(&params.blob[word]), word, launch_factor);
}

// A pool's shape, host alias and dividers, as one launch header.
void fill_shape(const hicache_pool *pool, int64_t upp, int32_t layer, int64_t device_pages,
                hicache::XferHeader &h) {
  const Shape &s = pool->shape;
  const int32_t nb = int32_t(s.B * s.L);
  h.host = pool->host_dev;
  h.L = int32_t(s.L);
  h.P = int32_t(s.P);
  h.V = int32_t(s.V);
  h.num_bufs = nb;
  h.B = int32_t(s.B);
  h.layer = layer;
  h.Hp = int32_t(s.Hp);
  h.unit_per_page = uint32_t(upp);
  h.PV = uint32_t(s.PV);
  h.LV = uint32_t(s.L * s.V);
  h.LPV = uint32_t(s.LPV);
  h.BLPV = uint32_t(s.BLPV);
  h.fd_BLPV = hicache::make_fastdiv(uint32_t(s.BLPV));
  h.fd_V = hicache::make_fastdiv(uint32_t(s.V));
  h.fd_PV = hicache::make_fastdiv(uint32_t(s.PV));
  h.fd_LV = hicache::make_fastdiv(uint32_t(s.L * s.V));
  h.fd_LPV = hicache::make_fastdiv(uint32_t(s.LPV));
  h.job[1] = hicache::Job{0, nb, 0, 0, 0u, 0u, hicache::make_fastdiv(1u)};
  h.wait_previous = 0;
  h.Dp = int32_t(device_pages);
  h.host_vecs = s.B * s.Hp * s.LPV;
  h.signal = nullptr;
}

// Header fields shared by every launch of a pool, and its buffer pointers.
void fill_header(const hicache_pool *pool, const hicache_device_kv *kv, hicache::XferParams &params,
                 int64_t upp, int32_t layer) {
  fill_shape(pool, upp, layer, kv->device_num_pages, params.h);
  const int32_t nb = int32_t(pool->shape.B * pool->shape.L);
  for (int32_t i = 0; i < nb; ++i)
    params.blob[i] = uint64_t(reinterpret_cast<uintptr_t>(kv->buf_ptrs[i]));
}

int check_device(const hicache_pool *pool) {
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess || cur != pool->device)
    return set_error(HICACHE_ERR_INVALID_ARG, "the calling thread's device (%d) is not the pool's (%d)",
                     cur, pool->device);
  return HICACHE_OK;
}

// Enqueue validated runs.  One direction: `runs` moves towards the host if
// to_host; layer < 0 means every layer.  Both directions (`load_runs` not
// NULL): `runs` is a backup and `load_runs` a load, every layer, one kernel
// per chunk so the two directions share every CTA.
int enqueue(const hicache_pool *pool, const hicache_device_kv *kv, const std::vector<RunRec> &runs,
            const std::vector<RunRec> *load_runs, int32_t layout, int32_t layer, bool to_host,
            void *stream, bool pdl_first, unsigned int *signal, int64_t *signalled,
            const std::function<bool()> *more) {
  const bool bidir = load_runs != nullptr;
  bool produced = more == nullptr;        // every run is already in `runs`
  if (!produced && bidir) return set_error(HICACHE_ERR_INVALID_ARG, "runs produced during a fused call");
  const Shape &s = pool->shape;
  const bool all = layer < 0;
  const int32_t nb = int32_t(s.B * s.L);
  // units: (buffer, layer, run) for layer_first with every layer; (run) for
  // page_first_direct_kv with every layer; (buffer, run) otherwise
  const bool lf_all = (layout == HICACHE_LAYER_FIRST) && all;
  const bool kv_all = (layout == HICACHE_PAGE_FIRST_DIRECT_KV) && all;
  const int64_t outers = lf_all ? s.B * s.L : (kv_all ? 1 : s.B);
  const int64_t upp = !all || layout == HICACHE_LAYER_FIRST ? s.PV : (kv_all ? s.BLPV : s.LPV);
  const int64_t capacity = (hicache::kBlobWords - nb) / 2;  // runs per launch

  size_t next0 = 0, next1 = 0;
  // runs still coming in: launch a chunk only once more runs than one launch
  // takes are in, so that the last run, which may still grow, stays behind
  const auto top_up = [&]() {
    while (!produced && runs.size() - next0 <= size_t(capacity)) produced = (*more)();
  };
  top_up();
  if (runs.empty() && (!bidir || load_runs->empty())) return HICACHE_OK;
  if (int rc = check_device(pool)) return rc;

  thread_local hicache::XferParams params;
  hicache::XferHeader &h = params.h;
  fill_header(pool, kv, params, upp, all ? 0 : layer);
  if (!bidir) h.signal = signal;

  const size_t n1 = bidir ? load_runs->size() : 0;
  while (next0 < runs.size() || next1 < n1) {
    const bool more0 = next0 < runs.size(), more1 = next1 < n1;
    const int64_t cap0 = more1 ? capacity / 2 : capacity;
    const int32_t c0 = fill_job(runs, next0, upp, outers, more0 ? cap0 : 0, params, nb, 0);
    if (c0 < 0) return set_error(HICACHE_ERR_INVALID_ARG, "transfer too large for one launch");
    int32_t c1 = 0;
    if (bidir) {
      c1 = fill_job(*load_runs, next1, upp, outers, more1 ? capacity - c0 : 0, params, nb + 2 * c0, 1);
      if (c1 < 0) return set_error(HICACHE_ERR_INVALID_ARG, "transfer too large for one launch");
    }
    hicache::XferLaunch x;
    x.params = &params;
    x.words = nb + 2 * (c0 + c1);
    x.layout = layout;
    x.all_layers = all;
    x.to_host = to_host;
    x.bidir = bidir;
    const int64_t tiles = int64_t(h.job[0].total_tiles) + (bidir ? h.job[1].total_tiles : 0);
    const int64_t ctas = bidir     ? pool->fused_ctas
                         : to_host ? pool->backup_ctas
                         : all     ? pool->ctas
                                   : pool->layer_ctas;
    x.grid = int(std::min<int64_t>(tiles, ctas));
    x.stream = stream;
    // The launches of one call move disjoint destinations: each after the
    // first is programmatic and starts work as the one before it drains.  The
    // first launch of a one-layer load is programmatic too: it follows work
    // it may depend on and waits for it before touching memory, unless the
    // caller knows that work is a one-layer load of another layer
    // (pdl_first); that hides the launch of a short per-layer kernel.  The
    // first launch of any other call is plain (it runs long enough that its
    // launch does not show, and a plain launch places its CTAs on an idle GPU).
    const bool first = next0 == 0 && next1 == 0;
    x.pdl = !first || !all;
    h.wait_previous = first && !all && !pdl_first ? 1 : 0;
    const int e = hicache::launch_xfer(x);
    if (e != 0) return cuda_error(cudaError_t(e), "transfer kernel launch");
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (signalled && h.signal) *signalled += x.grid;
    next0 += size_t(c0);
    next1 += size_t(c1);
    top_up();
  }
  return HICACHE_OK;
}

int transfer(hicache_pool *pool, const hicache_device_kv *kv, const int64_t *dev,
             const int64_t *host, int64_t n, int32_t layout, int32_t layer, int32_t direction,
             void *stream) {
  g_last_error.clear();
  if (!pool) return set_error(HICACHE_ERR_INVALID_ARG, "pool is NULL");
  int32_t lay = 0;
  int rc = resolve_layout(layout, pool->shape.layout, &lay);
  if (rc) return rc;
  if (layer >= pool->shape.L)
    return set_error(HICACHE_ERR_INVALID_ARG, "layer_id %d outside [0, %lld)", layer,
                     (long long)pool->shape.L);
  if ((rc = check_kv(pool, kv, 0))) return rc;
  thread_local std::vector<RunRec> runs;
  const int64_t max_run = max_run_pages(pool->shape);
  bool sorted = true;
  if ((rc = validate_pairs(pool->shape.Hp, kv->device_num_pages, dev, host, n, direction, &sorted))) return rc;
  if (sorted && n > kStreamPairs) {
    // Pairs already in host order (the usual case: a request's host pages
    // come from the allocator in order): the whole call is validated, so the
    // runs are built a chunk at a time and each launch goes out as soon as its
    // runs are final, while the host works on the next chunk.
    runs.clear();
    int64_t done = 0;
    const std::function<bool()> more = [&]() {
      const int64_t stop = std::min(n, done + kStreamPairs);
      append_runs(dev, host, done, stop, max_run, &runs);
      done = stop;
      return done == n;
    };
    rc = enqueue(pool, kv, runs, nullptr, lay, layer, direction == HICACHE_DIR_BACKUP, stream, false, nullptr,
                 nullptr, &more);
  } else {
    build_runs(kv->device_num_pages, dev, host, n, sorted, max_run, &runs);
    rc = enqueue(pool, kv, runs, nullptr, lay, layer, direction == HICACHE_DIR_BACKUP, stream);
  }
  if (rc) return rc;
  if (layer >= 0) {
    const cudaError_t e = cudaEventRecord(pool->events[size_t(layer)], static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_error(e, "cudaEventRecord(layer event)");
    std::lock_guard<std::mutex> g(pool->signal_mu);
    pool->layer_signal[size_t(layer)] = 0;
  } else if (direction == HICACHE_DIR_LOAD && n > 0) {
    return mark_all_layer_load(pool, stream);
  }
  return HICACHE_OK;
}

int mark_all_layer_load(hicache_pool *pool, void *stream) {
  // a load captured into a CUDA graph is not enqueued until the graph runs
  cudaStreamCaptureStatus status = cudaStreamCaptureStatusNone;
  const cudaError_t ce = cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &status);
  if (ce != cudaSuccess) return cuda_error(ce, "cudaStreamIsCapturing");
  if (status != cudaStreamCaptureStatusNone) return HICACHE_OK;
  const cudaError_t e = cudaEventRecord(pool->load_all, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_error(e, "cudaEventRecord(load of every layer)");
  std::lock_guard<std::mutex> g(pool->signal_mu);
  for (auto &sig : pool->layer_signal) sig = 3;
  return HICACHE_OK;
}

}  // namespace hicache

using namespace hicache;

extern "C" {

int32_t hicache_version(void) { return 100; }

const char *hicache_last_error(void) { return g_last_error.c_str(); }

int64_t hicache_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int hicache_host_alloc(size_t bytes, int32_t flags, void **out) {
  g_last_error.clear();
  if (!out || bytes == 0) return set_error(HICACHE_ERR_INVALID_ARG, "bytes must be > 0 and out non-NULL");
  if (flags & ~int32_t(HICACHE_HOST_THP)) return set_error(HICACHE_ERR_INVALID_ARG, "unknown flags");
  *out = nullptr;
  void *p = nullptr;
  size_t mapped = bytes;
  const bool thp = (flags & HICACHE_HOST_THP) != 0;
  if (thp) {
    const size_t huge = size_t(2) << 20;
    mapped = (bytes + huge - 1) / huge * huge;
    p = mmap(nullptr, mapped, PROT_READ | PROT_WRITE, MAP_PRIVATE | MAP_ANONYMOUS, -1, 0);
    if (p == MAP_FAILED) return set_error(HICACHE_ERR_NOMEM, "mmap of %zu bytes failed", mapped);
    // huge pages must be requested before the pages are locked
    (void)madvise(p, mapped, MADV_HUGEPAGE);
    const cudaError_t e =
        cudaHostRegister(p, mapped, cudaHostRegisterMapped | cudaHostRegisterPortable);
    if (e != cudaSuccess) {
      munmap(p, mapped);
      return cuda_error(e, "cudaHostRegister");
    }
  } else {
    const cudaError_t e = cudaHostAlloc(&p, bytes, cudaHostAllocMapped | cudaHostAllocPortable);
    if (e != cudaSuccess) return cuda_error(e, "cudaHostAlloc");
  }
  {
    std::lock_guard<std::mutex> g(g_alloc_mu);
    g_allocs[p] = HostAlloc{mapped, thp};
  }
  *out = p;
  return HICACHE_OK;
}

int hicache_host_free(void *ptr) {
  g_last_error.clear();
  if (!ptr) return HICACHE_OK;
  HostAlloc a;
  {
    std::lock_guard<std::mutex> g(g_alloc_mu);
    auto it = g_allocs.find(ptr);
    if (it == g_allocs.end())
      return set_error(HICACHE_ERR_INVALID_ARG, "pointer was not allocated by hicache_host_alloc");
    a = it->second;
    g_allocs.erase(it);
  }
  if (a.thp) {
    const cudaError_t e = cudaHostUnregister(ptr);
    munmap(ptr, a.bytes);
    if (e != cudaSuccess) return cuda_error(e, "cudaHostUnregister");
  } else {
    const cudaError_t e = cudaFreeHost(ptr);
    if (e != cudaSuccess) return cuda_error(e, "cudaFreeHost");
  }
  return HICACHE_OK;
}

int hicache_pool_create(const hicache_pool_desc *desc, void *host_pool, size_t host_bytes,
                        hicache_pool **out) {
  g_last_error.clear();
  if (!out) return set_error(HICACHE_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  Shape s{};
  int rc = check_desc(desc, &s, true);
  if (rc) return rc;
  if (!host_pool) return set_error(HICACHE_ERR_INVALID_ARG, "host pool pointer is NULL");
  if (reinterpret_cast<uintptr_t>(host_pool) % 16 != 0)
    return set_error(HICACHE_ERR_ALIGNMENT, "host pool is not 16-byte aligned");
  const int64_t need = s.B * s.Hp * s.LPV * 16;
  if (int64_t(host_bytes) < need)
    return set_error(HICACHE_ERR_INVALID_ARG, "host pool of %zu bytes is below the %lld needed",
                     host_bytes, (long long)need);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
  cudaPointerAttributes attr;
  e = cudaPointerGetAttributes(&attr, host_pool);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return set_error(HICACHE_ERR_NOT_PINNED, "host pool is not CUDA host memory: %s",
                     cudaGetErrorString(e));
  }
  if (attr.type != cudaMemoryTypeHost || attr.devicePointer == nullptr)
    return set_error(HICACHE_ERR_NOT_PINNED, "host pool is not page-locked, device-mapped memory");
  // the whole range must be one pinned allocation: check its last byte as well
  cudaPointerAttributes attr_end;
  e = cudaPointerGetAttributes(&attr_end, static_cast<char *>(host_pool) + need - 1);
  if (e != cudaSuccess || attr_end.type != cudaMemoryTypeHost) {
    (void)cudaGetLastError();
    return set_error(HICACHE_ERR_NOT_PINNED, "host pool is not pinned up to its last byte");
  }
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_error(e, "cudaDeviceGetAttribute");

  hicache_pool *p = new (std::nothrow) hicache_pool();
  if (!p) return set_error(HICACHE_ERR_NOMEM, "out of host memory");
  p->desc = *desc;
  p->shape = s;
  p->host = host_pool;
  p->host_dev = attr.devicePointer;
  p->host_bytes = host_bytes;
  p->device = dev;
  p->ctas = desc->launch_ctas > 0 ? desc->launch_ctas : sms * hicache::kDefaultLoadCtasPerSm;
  p->layer_ctas = desc->launch_ctas > 0 ? desc->launch_ctas : std::max(1, sms * hicache::kDefaultLayerCtasPer2Sm / 2);
  p->fused_ctas = desc->launch_ctas > 0 ? 2 * desc->launch_ctas : sms * hicache::kDefaultFusedCtasPerSm;
  p->backup_ctas = desc->launch_ctas > 0
                       ? desc->launch_ctas
                       : std::max(1, sms * hicache::kDefaultBackupCtasPer8Sm / 8);
  p->events.resize(size_t(s.L), nullptr);
  for (auto &ev : p->events) {
    e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
    if (e != cudaSuccess) {
      hicache_pool_destroy(p);
      return cuda_error(e, "cudaEventCreateWithFlags");
    }
  }
  e = cudaEventCreateWithFlags(&p->pipeline_last, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->load_all, cudaEventDisableTiming);
  if (e != cudaSuccess) {
    hicache_pool_destroy(p);
    return cuda_error(e, "cudaEventCreateWithFlags");
  }
  p->layer_target.assign(size_t(s.L), 0);
  p->layer_signal.assign(size_t(s.L), 0);
  // L layer counters, then the two scheduler words of the pipelined kernel
  e = cudaMalloc(reinterpret_cast<void **>(&p->layer_done), size_t(s.L + 2) * sizeof(unsigned int));
  if (e == cudaSuccess) e = cudaMemset(p->layer_done, 0, size_t(s.L + 2) * sizeof(unsigned int));
  if (e != cudaSuccess) {
    hicache_pool_destroy(p);
    return cuda_error(e, "per-layer counters");
  }
  *out = p;
  return HICACHE_OK;
}

int hicache_pool_destroy(hicache_pool *pool) {
  if (!pool) return HICACHE_OK;
  // pipelined loads count into the pool's device words: let the last one end
  // (they all follow one another on one stream) before the words are freed.
  // A chain of per-layer calls left open has no event behind its last kernel,
  // so then the whole device is waited for.
  if (pool->chain_open) (void)cudaDeviceSynchronize();
  else if (pool->pipeline_stream_set && pool->pipeline_last) (void)cudaEventSynchronize(pool->pipeline_last);
  if (pool->event_stream) {
    // its waits read the counters freed below; every one is met once the
    // loads above are done
    (void)cudaStreamSynchronize(pool->event_stream);
    (void)cudaStreamDestroy(pool->event_stream);
  }
  for (auto ev : pool->events)
    if (ev) cudaEventDestroy(ev);
  if (pool->layer_done) cudaFree(pool->layer_done);
  if (pool->pipeline_last) cudaEventDestroy(pool->pipeline_last);
  if (pool->load_all) cudaEventDestroy(pool->load_all);
  delete pool;
  return HICACHE_OK;
}

int hicache_backup(hicache_pool *pool, const hicache_device_kv *kv, const int64_t *device_pages,
                   const int64_t *host_pages, int64_t n, int32_t layout, void *stream) {
  return transfer(pool, kv, device_pages, host_pages, n, layout, -1, HICACHE_DIR_BACKUP, stream);
}

int hicache_load(hicache_pool *pool, const hicache_device_kv *kv, const int64_t *device_pages,
                 const int64_t *host_pages, int64_t n, int32_t layout, void *stream) {
  return transfer(pool, kv, device_pages, host_pages, n, layout, -1, HICACHE_DIR_LOAD, stream);
}

int hicache_load_layer(hicache_pool *pool, const hicache_device_kv *kv,
                       const int64_t *device_pages, const int64_t *host_pages, int64_t n,
                       int32_t layout, int32_t layer_id, void *stream) {
  if (layer_id < 0) {
    g_last_error.clear();
    return set_error(HICACHE_ERR_INVALID_ARG, "layer_id %d is negative", layer_id);
  }
  return transfer(pool, kv, device_pages, host_pages, n, layout, layer_id, HICACHE_DIR_LOAD, stream);
}

int hicache_backup_load(hicache_pool *pool, const hicache_device_kv *kv,
                        const int64_t *backup_device_pages, const int64_t *backup_host_pages,
                        int64_t n_backup, const int64_t *load_device_pages,
                        const int64_t *load_host_pages, int64_t n_load, int32_t layout,
                        void *stream) {
  g_last_error.clear();
  if (!pool) return set_error(HICACHE_ERR_INVALID_ARG, "pool is NULL");
  int32_t lay = 0;
  int rc = resolve_layout(layout, pool->shape.layout, &lay);
  if (rc) return rc;
  if ((rc = check_kv(pool, kv, 0))) return rc;
  thread_local std::vector<RunRec> brun, lrun;
  if ((rc = prepass(pool->shape.Hp, kv->device_num_pages, backup_device_pages, backup_host_pages,
                    n_backup, HICACHE_DIR_BACKUP, max_run_pages(pool->shape), &brun)))
    return rc;
  if ((rc = prepass(pool->shape.Hp, kv->device_num_pages, load_device_pages, load_host_pages, n_load,
                    HICACHE_DIR_LOAD, max_run_pages(pool->shape), &lrun)))
    return rc;
  if (n_backup > 0 && n_load > 0) {
    // the result must not depend on the order of the two directions
    int64_t page = 0;
    if (intersects(std::vector<int64_t>(backup_device_pages, backup_device_pages + n_backup),
                   std::vector<int64_t>(load_device_pages, load_device_pages + n_load), &page))
      return set_error(HICACHE_ERR_INVALID_ARG,
                       "device page %lld is read by the backup and written by the load",
                       (long long)page);
    if (intersects(std::vector<int64_t>(backup_host_pages, backup_host_pages + n_backup),
                   std::vector<int64_t>(load_host_pages, load_host_pages + n_load), &page))
      return set_error(HICACHE_ERR_INVALID_ARG,
                       "host page %lld is written by the backup and read by the load",
                       (long long)page);
  }
  if (lrun.empty()) return enqueue(pool, kv, brun, nullptr, lay, -1, true, stream);
  rc = brun.empty() ? enqueue(pool, kv, lrun, nullptr, lay, -1, false, stream)
                    : enqueue(pool, kv, brun, &lrun, lay, -1, true, stream);
  if (rc) return rc;
  return mark_all_layer_load(pool, stream);
}

int hicache_layer_event(hicache_pool *pool, int32_t layer, void **event_out) {
  g_last_error.clear();
  if (!pool || !event_out) return set_error(HICACHE_ERR_INVALID_ARG, "pool or event_out is NULL");
  if (layer < 0 || layer >= pool->shape.L)
    return set_error(HICACHE_ERR_INVALID_ARG, "layer %d outside [0, %lld)", layer,
                     (long long)pool->shape.L);
  std::lock_guard<std::mutex> g(pool->signal_mu);
  const uint8_t sig = pool->layer_signal[size_t(layer)];
  if (sig == 1 || sig == 2) {
    // the layer's last load is signalled on the device: record its event now,
    // behind a wait for that load's count of the layer
    int rc = check_device(pool);
    if (rc) return rc;
    if ((rc = record_counted_layer_event(pool, layer))) return rc;
  }
  *event_out = sig == 3 ? pool->load_all : pool->events[size_t(layer)];
  return HICACHE_OK;
}

int hicache_wait(void *stream, int64_t timeout_us) {
  g_last_error.clear();
  const auto start = std::chrono::steady_clock::now();
  for (;;) {
    const cudaError_t e = cudaStreamQuery(static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) return HICACHE_OK;
    if (e != cudaErrorNotReady) return cuda_error(e, "cudaStreamQuery");
    const int64_t waited = std::chrono::duration_cast<std::chrono::microseconds>(
                               std::chrono::steady_clock::now() - start)
                               .count();
    if (timeout_us >= 0 && waited >= timeout_us)
      return set_error(HICACHE_ERR_TIMEOUT, "stream still busy after %lld us", (long long)waited);
    // Poll back to back for the first 500 us (small transfers finish within
    // tens of microseconds and a sleep overshoots by the timer slack), then
    // sleep 50 us between polls.
    if (waited < 500) {
      std::this_thread::yield();
    } else {
      int64_t nap = 50;
      if (timeout_us >= 0) nap = std::min<int64_t>(nap, std::max<int64_t>(1, timeout_us - waited));
      std::this_thread::sleep_for(std::chrono::microseconds(nap));
    }
  }
}

// The device address of [p, p + bytes): device memory as it is, pinned host
// memory through its device alias; anything else (pageable memory, a range
// that leaves its allocation) is refused before any launch.
static int device_range(const void *p, size_t bytes, const char *what, void **out) {
  cudaPointerAttributes a, b;
  cudaError_t e = cudaPointerGetAttributes(&a, p);
  if (e == cudaSuccess) e = cudaPointerGetAttributes(&b, static_cast<const char *>(p) + bytes - 1);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return set_error(HICACHE_ERR_NOT_PINNED, "%s is not CUDA memory", what);
  }
  const bool ok_a = a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged ||
                    (a.type == cudaMemoryTypeHost && a.devicePointer != nullptr);
  if (!ok_a || b.type != a.type || b.devicePointer == nullptr)
    return set_error(HICACHE_ERR_NOT_PINNED, "%s is not device memory or pinned, device-mapped host memory "
                     "up to its last byte", what);
  int dev = -1;
  if (a.type == cudaMemoryTypeDevice && (cudaGetDevice(&dev) != cudaSuccess || dev != a.device))
    return set_error(HICACHE_ERR_INVALID_ARG, "%s is on device %d, not the current device", what, a.device);
  *out = a.devicePointer;
  return HICACHE_OK;
}

int hicache_stream_copy(void *dst, const void *src, size_t bytes, int32_t grid, int32_t vecs_per_thread,
                        void *stream) {
  g_last_error.clear();
  if (bytes == 0) return HICACHE_OK;
  if (!dst || !src) return set_error(HICACHE_ERR_INVALID_ARG, "dst or src is NULL");
  if (reinterpret_cast<uintptr_t>(dst) % 16 || reinterpret_cast<uintptr_t>(src) % 16 || bytes % 16)
    return set_error(HICACHE_ERR_ALIGNMENT, "dst, src and bytes must be multiples of 16 bytes");
  if (vecs_per_thread == 0) vecs_per_thread = 4;
  if (vecs_per_thread != 4 && vecs_per_thread != 8)
    return set_error(HICACHE_ERR_INVALID_ARG, "vecs_per_thread must be 4 or 8");
  const char *d = static_cast<const char *>(dst);
  const char *s = static_cast<const char *>(src);
  if (d < s + bytes && s < d + bytes) return set_error(HICACHE_ERR_INVALID_ARG, "dst and src overlap");
  void *dd = nullptr, *sd = nullptr;
  if (int rc = device_range(dst, bytes, "dst", &dd)) return rc;
  if (int rc = device_range(src, bytes, "src", &sd)) return rc;
  if (grid == 0) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_error(e, "cudaDeviceGetAttribute");
    grid = sms;
  }
  if (grid < 1 || grid > 65536) return set_error(HICACHE_ERR_INVALID_ARG, "grid %d outside [1, 65536]", grid);
  const int e = hicache::launch_stream_copy(dd, sd, uint64_t(bytes / 16), grid, vecs_per_thread, stream);
  if (e != 0) return cuda_error(cudaError_t(e), "stream copy kernel launch");
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return HICACHE_OK;
}

int32_t hicache_checked_build(void) { return int32_t(hicache::checked_build()); }

int hicache_check_status(uint64_t *first, uint64_t *count, int32_t clear) {
  g_last_error.clear();
  if (!first || !count) return set_error(HICACHE_ERR_INVALID_ARG, "first or count is NULL");
  unsigned long long f = 0, c = 0;
  const int e = hicache::check_status(&f, &c, clear != 0);
  if (e != 0) return cuda_error(cudaError_t(e), "reading the bounds-check words");
  *first = f;
  *count = c;
  return HICACHE_OK;
}

int hicache_layer_checksum(const hicache_device_kv *kv, const hicache_pool_desc *desc,
                           const int64_t *device_pages, int64_t n, int32_t layer_id,
                           int32_t reps, uint64_t *out_sum_dev, void *stream) {
  g_last_error.clear();
  Shape s{};
  int rc = check_desc(desc, &s, true);
  if (rc) return rc;
  if (!kv || !kv->buf_ptrs || !out_sum_dev)
    return set_error(HICACHE_ERR_INVALID_ARG, "kv or out_sum_dev is NULL");
  if (layer_id < 0 || layer_id >= s.L)
    return set_error(HICACHE_ERR_INVALID_ARG, "layer_id %d outside [0, %lld)", layer_id,
                     (long long)s.L);
  if (s.B > 8) return set_error(HICACHE_ERR_INVALID_ARG, "at most 8 buffers");
  if (reps < 1 || n < 0) return set_error(HICACHE_ERR_INVALID_ARG, "reps must be >= 1, n >= 0");
  if (n > 0 && !device_pages) return set_error(HICACHE_ERR_INVALID_ARG, "device_pages is NULL");
  if (int64_t(n) * s.PV >= INT32_MAX) return set_error(HICACHE_ERR_INVALID_ARG, "too many pages");
  for (int64_t i = 0; i < n; ++i)
    if (device_pages[i] < 0 || device_pages[i] >= kv->device_num_pages)
      return set_error(HICACHE_ERR_INDEX_RANGE, "device_pages[%lld] out of range", (long long)i);
  thread_local hicache::ChecksumParams p;
  for (int64_t b = 0; b < s.B; ++b) {
    p.bufs[b] = kv->buf_ptrs[b * s.L + layer_id];
    if (!p.bufs[b] || reinterpret_cast<uintptr_t>(p.bufs[b]) % 16)
      return set_error(HICACHE_ERR_ALIGNMENT, "buffer NULL or not 16-byte aligned");
  }
  p.B = int32_t(s.B);
  p.reps = reps;
  p.PV = uint32_t(s.PV);
  p.out = reinterpret_cast<unsigned long long *>(out_sum_dev);
  for (int64_t first = 0; first < n; first += hicache::kChecksumMaxPages) {
    const int64_t cnt = std::min<int64_t>(hicache::kChecksumMaxPages, n - first);
    p.n = int32_t(cnt);
    for (int64_t i = 0; i < cnt; ++i) p.pages[i] = int32_t(device_pages[first + i]);
    const int64_t vecs = cnt * s.PV * s.B;
    const int grid = int(std::max<int64_t>(1, std::min<int64_t>(1024, (vecs + hicache::kThreads - 1) / hicache::kThreads)));
    const int e = hicache::launch_checksum(p, grid, stream);
    if (e != 0) return cuda_error(cudaError_t(e), "checksum kernel launch");
    g_launches.fetch_add(1, std::memory_order_relaxed);
  }
  return HICACHE_OK;
}

}  // extern "C"
