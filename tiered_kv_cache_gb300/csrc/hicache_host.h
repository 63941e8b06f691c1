// hicache_host.h -- host-side internals shared by the host files of the
// library (API, index pre-pass, pipelined loads, plans, groups, engine).  Not
// part of the public ABI.
#pragma once

#include <cuda.h>  // driver types for the stream memory wait (fetched at run time)
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cstdint>
#include <functional>
#include <mutex>
#include <utility>
#include <vector>

#include "hicache.h"
#include "hicache_internal.h"

namespace hicache {

// A validated pool shape, in elements and 16-byte vectors.
struct Shape {
  int64_t L, B, P, R, es, Hp;
  int64_t row_bytes, V, PV, LPV, BLPV;
  int32_t layout;
};

// Last-error text of the calling thread.
int set_error(int code, const char *fmt, ...);
int cuda_error(cudaError_t e, const char *what);
void clear_error();

// Kernel launches made by the library (hicache_launch_count).
extern std::atomic<int64_t> g_launches;

// Launch limits: tiles per launch (32-bit tile index) and vectors per outer
// unit (32-bit vector offsets inside a unit, with a tile of headroom).
constexpr int64_t kMaxTiles = int64_t(1) << 30;
constexpr int64_t kMaxOuterVecs = INT32_MAX - kTileVecs;

// hicache_index.cpp: validation and the pre-pass.
int check_desc(const hicache_pool_desc *d, Shape *s, bool need_alignment);
int resolve_layout(int32_t layout, int32_t pool_layout, int32_t *out);
// Validate n pairs and reduce them to runs (sorted by host page).
int prepass(int64_t Hp, int64_t Dp, const int64_t *dev, const int64_t *host, int64_t n,
            int32_t direction, int64_t max_run, std::vector<RunRec> *runs);
int64_t max_run_pages(const Shape &s);
// The checks of prepass alone (ranges, repeated destinations), and whether the
// pairs already come sorted by (host page, device page).
int validate_pairs(int64_t Hp, int64_t Dp, const int64_t *dev, const int64_t *host, int64_t n,
                   int32_t direction, bool *sorted);
// The runs of n pairs that validate_pairs accepted (sorted: as it reported).
void build_runs(int64_t Dp, const int64_t *dev, const int64_t *host, int64_t n, bool sorted, int64_t max_run,
                std::vector<RunRec> *runs);
// Append the runs of sorted pairs [begin, end) to *runs, continuing its last run.
void append_runs(const int64_t *dev, const int64_t *host, int64_t begin, int64_t end, int64_t max_run,
                 std::vector<RunRec> *runs);
bool intersects(std::vector<int64_t> a, std::vector<int64_t> b, int64_t *common);

// cuStreamWaitValue32 from the driver (hicache_pipeline.cpp); nullptr if the
// driver does not offer it.
using WaitValue32Fn = CUresult (*)(CUstream, CUdeviceptr, cuuint32_t, unsigned int);
WaitValue32Fn wait_value32();
// Record `layer`'s event on the pool's event stream behind a wait for the
// counter of the layer's last load (signal 1 or 2) to reach its current
// target.  The caller holds pool->signal_mu, on the pool's device.
int record_counted_layer_event(hicache_pool *pool, int64_t layer);
// After a load of every layer was enqueued on `stream`: record the pool's
// load_all event there and make it every layer's last load (signal 3).
int mark_all_layer_load(hicache_pool *pool, void *stream);

}  // namespace hicache

struct hicache_pool {
  hicache_pool_desc desc;
  hicache::Shape shape;
  void *host = nullptr;       // host pointer of the pool
  void *host_dev = nullptr;   // device-visible alias
  size_t host_bytes = 0;
  int device = 0;
  int ctas = 0;         // grid of a load of every layer
  int layer_ctas = 0;   // grid of a per-layer or pipelined load
  int backup_ctas = 0;  // grid of a backup
  int fused_ctas = 0;   // grid of a fused backup + load
  std::vector<cudaEvent_t> events;  // one per layer

  // Per-layer completion of pipelined loads (hicache_load_pipelined): device
  // counters that the kernel raises as layers land, the value each must reach
  // for the last pipelined load, which signal hicache_wait_layer should use
  // for each layer (0: the layer event, 1: the counter, 2: the allocation-free
  // load's counter, 3: load_all, after a load of every layer), and the one
  // stream all pipelined loads of the pool go on (which keeps the counts in
  // order).
  unsigned int *layer_done = nullptr;
  std::mutex signal_mu;
  std::vector<uint32_t> layer_target;
  std::vector<uint8_t> layer_signal;
  bool pipeline_stream_set = false;
  void *pipeline_stream = nullptr;
  cudaEvent_t pipeline_last = nullptr;  // recorded after each pipelined load
  // a chained per-layer load on pipeline_stream has not reached its last
  // layer (no pipeline_last recorded behind it yet)
  bool chain_open = false;
  // Where hicache_layer_event records the event of a load signalled on the
  // device: a stream of the pool's own that first waits for the layer's
  // counter to reach its target (made on first use, drained and destroyed
  // with the pool).
  cudaStream_t event_stream = nullptr;
  // Recorded behind every load of every layer (hicache_load, a fused backup
  // and load, a plan's or group's load of every layer, an engine load); signal
  // 3 sends hicache_wait_layer and hicache_layer_event of every layer to it.
  cudaEvent_t load_all = nullptr;
  // Allocation-free pipelined loads (signal 2): the library's static counters
  // on this device and, per layer, the value the last such load brings them to.
  unsigned int *noalloc_done = nullptr;
  std::vector<uint32_t> noalloc_target;
};

namespace hicache {

// hicache_api.cpp: launch helpers.
int check_kv(const hicache_pool *pool, const hicache_device_kv *kv, int64_t min_pages);
// The calling thread's device must be the pool's.
int check_device(const hicache_pool *pool);
// Copy runs[next..] into a job's run table at blob word `word` (at most
// max_runs runs, within the launch limits for `launch_factor` repeats of the
// job's tiles); returns the runs taken, or -1 if even one run is too large.
int32_t fill_runs(const std::vector<RunRec> &runs, size_t next, int64_t upp, int64_t outers,
                  int64_t max_runs, Job &job, Run *table, int32_t word, int64_t launch_factor);
int32_t fill_job(const std::vector<RunRec> &runs, size_t next, int64_t upp, int64_t outers,
                 int64_t max_runs, XferParams &params, int32_t word, int j, int64_t launch_factor = 1);
// A pool's shape, host alias and dividers, as one launch header (device_pages:
// the pages of each device buffer, for bounds-checked builds).
void fill_shape(const hicache_pool *pool, int64_t upp, int32_t layer, int64_t device_pages, XferHeader &h);
// fill_shape plus the device buffer pointers at the start of the blob.
void fill_header(const hicache_pool *pool, const hicache_device_kv *kv, XferParams &params, int64_t upp,
                 int32_t layer);
// Enqueue validated runs (see hicache_api.cpp).  A call split over several
// launches has each launch after the first start programmatically behind the
// one before it.  pdl_first: the first launch too, behind the kernel before it
// on the stream, which must be a one-layer load of another layer.  signal (one
// direction only): every CTA of every launch adds one to *signal once its
// last tile has landed; *signalled grows by the CTAs launched.
// more (one direction only): runs still coming in; each call appends the next
// ones to `runs` (the same vector) and returns true once all are in.  Chunks
// go out as their runs become final, so the host's work on later runs
// overlaps the launches of the earlier ones.
int enqueue(const hicache_pool *pool, const hicache_device_kv *kv, const std::vector<RunRec> &runs,
            const std::vector<RunRec> *load_runs, int32_t layout, int32_t layer, bool to_host,
            void *stream, bool pdl_first = false, unsigned int *signal = nullptr,
            int64_t *signalled = nullptr, const std::function<bool()> *more = nullptr);
// Pairs a call must have before its runs are built in chunks during the launches.
constexpr int64_t kStreamPairs = 4096;
// Enqueue validated load runs as pipelined launches (every layer, layer by
// layer, per-layer counters) and update the pool's per-layer signals
// (hicache_pipeline.cpp).
int enqueue_pipelined(hicache_pool *pool, const hicache_device_kv *kv, const std::vector<RunRec> &runs,
                      int32_t layout, void *stream);
// INVALID_ARG if `stream` is capturing (pipelined loads keep their per-layer
// targets on the host, raised at enqueue time), CUDA if that cannot be told.
int refuse_capture(void *stream);
// Counted loads of a pool -- pipelined, tensor-parallel, chained per-layer --
// add into the same per-layer counters, which cannot tell two loads apart, so
// they go on one stream, or on another only once the earlier ones have
// finished: the pool's last counted-load event has fired and no chain is
// left open.  check_counted_stream: INVALID_ARG otherwise (no side effect);
// claim_counted_stream: make `stream` the pool's counted-load stream.  Both
// with pool->signal_mu held.
int check_counted_stream(hicache_pool *pool, void *stream);
void claim_counted_stream(hicache_pool *pool, void *stream);

// hicache_plan.cpp: per-layer graphs.
// INVALID_ARG unless the (address, bytes) spans are pairwise disjoint.
int check_disjoint(std::vector<std::pair<uintptr_t, uint64_t>> spans);
// Capture L layers into an executable graph: enqueue_layer(l, stream) enqueues
// layer l's launches (every launch after the very first programmatic), and
// each pool's event of layer l is recorded after them; *launches = the kernel
// launches of one replay.
int capture_layer_graph(hicache_pool *const *pools, int32_t np, int64_t L,
                        const std::function<int(int64_t, void *)> &enqueue_layer, cudaGraphExec_t *out,
                        int64_t *launches);
// Replay such a graph on `stream`; the pools' per-layer waits use the events.
int launch_layer_graph(cudaGraphExec_t graph, int64_t launches, hicache_pool *const *pools, int32_t np,
                       void *stream);

}  // namespace hicache
