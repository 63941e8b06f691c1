// hicache_tp.cpp -- the tensor-parallel load of a replicated latent pool.
//
// "Baidu's KVCache Overhaul", section "MLA-class cache optimization": with MLA
// (and the CSA/HCA caches of the same page) every rank of a tensor-parallel
// group holds the same latent KV, so instead of each GPU reading every page
// over its host link, each reads only its 1/tp part and the parts are spread
// over NVLink, the host reads and the NVLink traffic running side by side,
// layer by layer.  Here each rank's launch reads its share of the pages from
// the host pool and stores every vector into the same device page of every
// rank's buffers (the NVLink scatter, fused into the load), counting each
// finished tile into every rank's per-layer counter.  A rank's
// hicache_wait_layer then waits for the tiles of ALL ranks' shares of a layer.

#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "hicache.h"
#include "hicache_host.h"
#include "hicache_internal.h"

namespace hicache {
namespace {

// The pair range [first, first + count) of rank `rank` out of n pairs split
// into tp contiguous parts in the caller's order: rank r takes the pairs
// [floor(n r / tp), floor(n (r + 1) / tp)), so part sizes differ by one at most.
// (floor(n r / tp) = (n / tp) r + floor((n mod tp) r / tp), with no overflow.)
void share_of(int64_t n, int32_t tp, int32_t rank, int64_t *first, int64_t *count) {
  const int64_t a = n / tp * rank + (n % tp) * rank / tp;
  const int64_t b = n / tp * (rank + 1) + (n % tp) * (rank + 1) / tp;
  *first = a;
  *count = b - a;
}

// Tiles per layer of the launches that move `runs` as one rank's share (the
// same split into launches as the rank's own call makes).
int64_t share_tiles(const hicache_pool *pool, const std::vector<RunRec> &runs, int32_t words0) {
  const Shape &s = pool->shape;
  thread_local XferParams scratch;
  int64_t tiles = 0;
  size_t next = 0;
  while (next < runs.size()) {
    const int32_t c = fill_job(runs, next, s.PV, s.B, (kBlobWords - words0) / 2, scratch, words0, 0, s.L);
    if (c < 0) return -1;
    tiles += scratch.h.job[0].total_tiles;
    next += size_t(c);
  }
  return tiles;
}

}  // namespace
}  // namespace hicache

using namespace hicache;

extern "C" {

int hicache_tp_share(int64_t n, int32_t tp, int32_t rank, int64_t *first, int64_t *count) {
  clear_error();
  if (!first || !count) return set_error(HICACHE_ERR_INVALID_ARG, "first or count is NULL");
  if (n < 0 || n >= (int64_t(1) << 40)) return set_error(HICACHE_ERR_INVALID_ARG, "n = %lld", (long long)n);
  if (tp < 1 || tp > kMaxTp) return set_error(HICACHE_ERR_INVALID_ARG, "tp = %d outside [1, %d]", tp, kMaxTp);
  if (rank < 0 || rank >= tp) return set_error(HICACHE_ERR_INVALID_ARG, "rank %d outside [0, %d)", rank, tp);
  share_of(n, tp, rank, first, count);
  return HICACHE_OK;
}

int hicache_pool_layer_counters(hicache_pool *pool, void **counters_out) {
  clear_error();
  if (!pool || !counters_out) return set_error(HICACHE_ERR_INVALID_ARG, "pool or counters_out is NULL");
  *counters_out = pool->layer_done;
  return HICACHE_OK;
}

int hicache_tp_load_pipelined(hicache_pool *pool, const hicache_device_kv *rank_kvs,
                              void *const *rank_counters, int32_t tp, int32_t rank,
                              const int64_t *device_pages, const int64_t *host_pages, int64_t n,
                              int32_t layout, void *stream) {
  clear_error();
  if (!pool || !rank_kvs || !rank_counters)
    return set_error(HICACHE_ERR_INVALID_ARG, "pool, rank_kvs or rank_counters is NULL");
  if (tp < 1 || tp > kMaxTp) return set_error(HICACHE_ERR_INVALID_ARG, "tp = %d outside [1, %d]", tp, kMaxTp);
  if (rank < 0 || rank >= tp) return set_error(HICACHE_ERR_INVALID_ARG, "rank %d outside [0, %d)", rank, tp);
  const Shape &s = pool->shape;
  const int32_t nb = int32_t(s.B * s.L);
  if (int64_t(tp) * nb > kMaxTpBufs)
    return set_error(HICACHE_ERR_INVALID_ARG, "tp x buffers x layers = %lld exceeds %d",
                     (long long)(int64_t(tp) * nb), kMaxTpBufs);
  int32_t lay = 0;
  int rc = resolve_layout(layout, s.layout, &lay);
  if (rc) return rc;
  const int64_t Dp = rank_kvs[0].device_num_pages;
  for (int32_t r = 0; r < tp; ++r) {
    if ((rc = check_kv(pool, &rank_kvs[r], 0))) return rc;
    if (rank_kvs[r].device_num_pages != Dp)
      return set_error(HICACHE_ERR_INVALID_ARG, "rank %d holds %lld device pages, rank 0 %lld", r,
                       (long long)rank_kvs[r].device_num_pages, (long long)Dp);
    if (!rank_counters[r] || reinterpret_cast<uintptr_t>(rank_counters[r]) % 4)
      return set_error(HICACHE_ERR_ALIGNMENT, "counters of rank %d are NULL or not 4-byte aligned", r);
  }
  // every rank validates the whole request, so all ranks accept or refuse it alike
  thread_local std::vector<RunRec> runs;
  if ((rc = prepass(s.Hp, Dp, device_pages, host_pages, n, HICACHE_DIR_LOAD, max_run_pages(s), &runs)))
    return rc;
  // each rank's share, and the tiles per layer it adds to every rank's counters
  const int32_t words0 = tp * nb;
  int64_t all_tiles = 0;
  std::vector<RunRec> own;
  for (int32_t r = 0; r < tp; ++r) {
    int64_t first = 0, count = 0;
    share_of(n, tp, r, &first, &count);
    std::vector<RunRec> &dst = r == rank ? own : runs;
    if ((rc = prepass(s.Hp, Dp, count ? device_pages + first : nullptr, count ? host_pages + first : nullptr,
                      count, HICACHE_DIR_LOAD, max_run_pages(s), &dst)))
      return rc;
    const int64_t t = share_tiles(pool, dst, words0);
    if (t < 0) return set_error(HICACHE_ERR_INVALID_ARG, "transfer too large for one launch");
    all_tiles += t;
  }
  if (all_tiles >= (int64_t(1) << 31))
    return set_error(HICACHE_ERR_INVALID_ARG, "%lld tiles per layer: too many for the 32-bit counters",
                     (long long)all_tiles);
  if ((rc = check_device(pool))) return rc;
  if ((rc = refuse_capture(stream))) return rc;
  if (!wait_value32())
    return set_error(HICACHE_ERR_CUDA, "the driver offers no cuStreamWaitValue32: no pipelined loads");
  std::lock_guard<std::mutex> g(pool->signal_mu);
  if ((rc = check_counted_stream(pool, stream))) return rc;
  claim_counted_stream(pool, stream);
  // this rank waits for every other rank's tiles, whatever happens to its own launches
  const int64_t others = all_tiles - share_tiles(pool, own, words0);
  for (int64_t l = 0; l < s.L; ++l) {
    pool->layer_target[size_t(l)] += uint32_t(others);
    pool->layer_signal[size_t(l)] = 1;
  }
  thread_local XferParams params;
  fill_shape(pool, s.PV, 0, Dp, params.h);
  for (int32_t r = 0; r < tp; ++r)
    for (int32_t i = 0; i < nb; ++i)
      params.blob[r * nb + i] = uint64_t(reinterpret_cast<uintptr_t>(rank_kvs[r].buf_ptrs[i]));
  TpFanout f{};
  f.tp = tp;
  for (int32_t r = 0; r < tp; ++r) f.counters[r] = static_cast<unsigned int *>(rank_counters[r]);
  size_t next = 0;
  while (next < own.size()) {
    const int32_t c = fill_job(own, next, s.PV, s.B, (kBlobWords - words0) / 2, params, words0, 0, s.L);
    if (c < 0) return set_error(HICACHE_ERR_INVALID_ARG, "transfer too large for one launch");
    XferLaunch x;
    x.params = &params;
    x.words = words0 + 2 * c;
    x.layout = lay;
    x.all_layers = false;
    x.to_host = false;
    x.bidir = false;
    x.grid = int(std::min<int64_t>(int64_t(params.h.job[0].total_tiles) * s.L, pool->layer_ctas));
    x.stream = stream;
    const int e = launch_tp_pipelined_load(x, f, pool->layer_done + s.L);
    if (e != 0) return cuda_error(cudaError_t(e), "tensor-parallel load kernel launch");
    g_launches.fetch_add(1, std::memory_order_relaxed);
    for (int64_t l = 0; l < s.L; ++l) pool->layer_target[size_t(l)] += uint32_t(params.h.job[0].total_tiles);
    next += size_t(c);
  }
  // (the layer events are recorded when asked for: hicache_layer_event)
  const cudaError_t e = cudaEventRecord(pool->pipeline_last, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_error(e, "cudaEventRecord(pipelined load)");
  pool->chain_open = false;
  return HICACHE_OK;
}

}  // extern "C"
