// hicache_api.cpp -- host side of libhicache: argument validation, the index
// sort / run-length pre-pass, pools, plans, per-layer events and launches.
//
// Every transfer call validates everything BEFORE it enqueues anything, so a
// call that fails has no effect.  Kernels are launched through
// hicache::launch_xfer (hicache_kernels.cu).

#include "hicache.h"

#include <cuda.h>  // driver types for the stream memory wait (fetched at run time)
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

// ---- shape checks ------------------------------------------------------------

int check_desc(const hicache_pool_desc *d, Shape *s, bool need_alignment) {
  if (!d) return set_error(HICACHE_ERR_INVALID_ARG, "pool descriptor is NULL");
  if (d->num_layers < 1 || d->num_buffers < 1 || d->page_size < 1 || d->elem_bytes < 1 ||
      d->row_elems < 1 || d->host_num_pages < 1)
    return set_error(HICACHE_ERR_INVALID_ARG,
                     "pool descriptor sizes must be >= 1 (layers %d, buffers %d, page_size %d, "
                     "elem_bytes %d, row_elems %lld, host pages %lld)",
                     d->num_layers, d->num_buffers, d->page_size, d->elem_bytes,
                     (long long)d->row_elems, (long long)d->host_num_pages);
  if (int64_t(d->num_layers) * d->num_buffers > hicache::kMaxBufs)
    return set_error(HICACHE_ERR_INVALID_ARG, "num_buffers * num_layers = %lld exceeds %d",
                     (long long)d->num_layers * d->num_buffers, hicache::kMaxBufs);
  if (d->layout < HICACHE_LAYER_FIRST || d->layout > HICACHE_PAGE_FIRST_DIRECT_KV)
    return set_error(HICACHE_ERR_INVALID_ARG, "unknown pool layout %d", d->layout);
  if (d->launch_ctas < 0 || d->flags != 0 || d->reserved != 0)
    return set_error(HICACHE_ERR_INVALID_ARG, "launch_ctas must be >= 0; flags and reserved must be 0");
  if (d->host_num_pages >= INT32_MAX)
    return set_error(HICACHE_ERR_INVALID_ARG, "host_num_pages must be < 2^31");
  s->L = d->num_layers;
  s->B = d->num_buffers;
  s->P = d->page_size;
  s->R = d->row_elems;
  s->es = d->elem_bytes;
  s->Hp = d->host_num_pages;
  s->layout = d->layout;
  if (s->R > (int64_t(1) << 40) / s->es)
    return set_error(HICACHE_ERR_INVALID_ARG, "row of %lld elements is too large", (long long)s->R);
  s->row_bytes = s->R * s->es;
  s->V = s->row_bytes / 16;
  s->PV = s->P * s->V;
  s->LPV = s->L * s->PV;
  s->BLPV = s->B * s->LPV;
  if (need_alignment) {
    if (s->row_bytes % 16 != 0)
      return set_error(HICACHE_ERR_ALIGNMENT, "row of %lld bytes is not a multiple of 16",
                       (long long)s->row_bytes);
    if (s->BLPV > INT32_MAX - hicache::kTileVecs)
      return set_error(HICACHE_ERR_INVALID_ARG,
                       "one page of every buffer and layer (%lld x 16 bytes) must be < 32 GiB - 16 KiB",
                       (long long)s->BLPV);
  }
  return HICACHE_OK;
}

int resolve_layout(int32_t layout, int32_t pool_layout, int32_t *out) {
  if (layout == HICACHE_LAYOUT_POOL) layout = pool_layout;
  if (layout < HICACHE_LAYER_FIRST || layout > HICACHE_PAGE_FIRST_DIRECT_KV)
    return set_error(HICACHE_ERR_INVALID_ARG, "unknown layout %d", layout);
  *out = layout;
  return HICACHE_OK;
}

// ---- the pre-pass ------------------------------------------------------------
struct Pair {
  int64_t h, d;
};
inline bool pair_less(const Pair &a, const Pair &b) {
  return a.h < b.h || (a.h == b.h && a.d < b.d);
}

int bit_length(uint64_t v) {
  int b = 0;
  while (v) {
    ++b;
    v >>= 1;
  }
  return b;
}

// Sort pairs by (host page, device page).  Large sets go through an LSD radix
// sort on the key h * 2^dbits + d (11-bit digits, only as many passes as the
// largest key needs): a few linear passes where a comparison sort spends
// ~n log n compares, which for the tens of thousands of one-token pages of a
// long prefix was most of the host's cost of a call.
void sort_pairs(std::vector<Pair> &pairs, int64_t Dp) {
  const size_t n = pairs.size();
  if (n < 2048) {
    std::sort(pairs.begin(), pairs.end(), pair_less);
    return;
  }
  const int dbits = bit_length(uint64_t(Dp - 1));
  uint64_t max_key = 0;
  thread_local std::vector<uint64_t> tls_keys, tls_tmp;
  std::vector<uint64_t> &keys = tls_keys, &tmp = tls_tmp;
  keys.resize(n);
  tmp.resize(n);
  for (size_t i = 0; i < n; ++i) {
    keys[i] = (uint64_t(pairs[i].h) << dbits) | uint64_t(pairs[i].d);
    max_key = std::max(max_key, keys[i]);
  }
  constexpr int kDigit = 11;
  constexpr size_t kBuckets = size_t(1) << kDigit;
  const int bits = bit_length(max_key);
  for (int shift = 0; shift < bits; shift += kDigit) {
    size_t count[kBuckets + 1] = {};
    for (size_t i = 0; i < n; ++i) ++count[((keys[i] >> shift) & (kBuckets - 1)) + 1];
    for (size_t b = 1; b <= kBuckets; ++b) count[b] += count[b - 1];
    for (size_t i = 0; i < n; ++i) tmp[count[(keys[i] >> shift) & (kBuckets - 1)]++] = keys[i];
    keys.swap(tmp);
  }
  const uint64_t dmask = (uint64_t(1) << dbits) - 1;
  for (size_t i = 0; i < n; ++i) pairs[i] = Pair{int64_t(keys[i] >> dbits), int64_t(keys[i] & dmask)};
}

// Whether a load names a destination page twice.  For device pools of up to
// 2^27 pages, one bit per page in a per-thread bitmap, cleared again for just
// the pages set; beyond that, a sort.
bool first_repeated(const int64_t *dev, int64_t n, int64_t Dp, int64_t *repeated) {
  if (Dp <= (int64_t(1) << 27)) {
    thread_local std::vector<uint64_t> tls_bits;
    std::vector<uint64_t> &vbits = tls_bits;
    if (vbits.size() < size_t((Dp + 63) / 64)) vbits.resize(size_t((Dp + 63) / 64), 0);
    uint64_t *const bits = vbits.data();
    int64_t i = 0;
    bool dup = false;
    for (; i < n; ++i) {
      const uint64_t bit = uint64_t(1) << (dev[i] & 63);
      uint64_t &w = bits[size_t(dev[i] >> 6)];
      if (w & bit) {
        dup = true;
        *repeated = dev[i];
        break;
      }
      w |= bit;
    }
    for (int64_t k = 0; k < i; ++k) bits[size_t(dev[k] >> 6)] = 0;
    return dup;
  }
  thread_local std::vector<int64_t> ds;
  ds.assign(dev, dev + n);
  std::sort(ds.begin(), ds.end());
  for (int64_t i = 1; i < n; ++i)
    if (ds[size_t(i)] == ds[size_t(i - 1)]) {
      *repeated = ds[size_t(i)];
      return true;
    }
  return false;
}

// Validate n index pairs and reduce them to runs: pairs sorted by (host page,
// device page), merged while both pages step by one (at most max_run pages per
// run).  On error the last-error text is set and *runs holds no usable table.
int prepass(int64_t Hp, int64_t Dp, const int64_t *dev, const int64_t *host, int64_t n,
            int32_t direction, int64_t max_run, std::vector<RunRec> *runs) {
  if (n < 0) return set_error(HICACHE_ERR_INVALID_ARG, "n = %lld is negative", (long long)n);
  if (direction != HICACHE_DIR_BACKUP && direction != HICACHE_DIR_LOAD)
    return set_error(HICACHE_ERR_INVALID_ARG, "unknown direction %d", direction);
  if (Dp < 1 || Dp >= INT32_MAX)
    return set_error(HICACHE_ERR_INVALID_ARG, "device_num_pages = %lld must be in [1, 2^31)",
                     (long long)Dp);
  runs->clear();
  if (n == 0) return HICACHE_OK;
  if (!dev || !host) return set_error(HICACHE_ERR_INVALID_ARG, "index array is NULL");
  // one lookup of the per-thread buffer: in a shared library every access to
  // a thread_local can be a call, too slow inside a per-page loop
  thread_local std::vector<Pair> tls_pairs;
  std::vector<Pair> &pairs = tls_pairs;
  pairs.resize(size_t(n));
  bool sorted = true;
  for (int64_t i = 0; i < n; ++i) {
    const int64_t d = dev[i], h = host[i];
    if (d < 0 || d >= Dp)
      return set_error(HICACHE_ERR_INDEX_RANGE, "device_pages[%lld] = %lld outside [0, %lld)",
                       (long long)i, (long long)d, (long long)Dp);
    if (h < 0 || h >= Hp)
      return set_error(HICACHE_ERR_INDEX_RANGE, "host_pages[%lld] = %lld outside [0, %lld)",
                       (long long)i, (long long)h, (long long)Hp);
    pairs[size_t(i)] = Pair{h, d};
    if (i > 0 && pair_less(pairs[size_t(i)], pairs[size_t(i - 1)])) sorted = false;
  }
  if (!sorted) sort_pairs(pairs, Dp);
  if (direction == HICACHE_DIR_BACKUP) {
    for (int64_t i = 1; i < n; ++i)
      if (pairs[size_t(i)].h == pairs[size_t(i - 1)].h)
        return set_error(HICACHE_ERR_DUPLICATE_INDEX,
                         "host page %lld is a backup destination twice",
                         (long long)pairs[size_t(i)].h);
  } else if (n <= 32) {
    for (int64_t i = 0; i < n; ++i)
      for (int64_t k = i + 1; k < n; ++k)
        if (dev[i] == dev[k])
          return set_error(HICACHE_ERR_DUPLICATE_INDEX,
                           "device page %lld is a load destination twice", (long long)dev[i]);
  } else {
    int64_t page = 0;
    if (first_repeated(dev, n, Dp, &page))
      return set_error(HICACHE_ERR_DUPLICATE_INDEX, "device page %lld is a load destination twice",
                       (long long)page);
  }
  for (int64_t i = 0; i < n; ++i) {
    const Pair &p = pairs[size_t(i)];
    if (!runs->empty()) {
      RunRec &r = runs->back();
      if (p.h == r.h0 + r.len && p.d == r.d0 + r.len && r.len < max_run) {
        ++r.len;
        continue;
      }
    }
    runs->push_back(RunRec{p.h, p.d, 1});
  }
  return HICACHE_OK;
}

constexpr int64_t kMaxTiles = int64_t(1) << 30;
constexpr int64_t kMaxOuterVecs = INT32_MAX - hicache::kTileVecs;

// Runs are capped so that a unit (at most every buffer and layer of a run)
// stays below 2^31 - 1024 vectors: the kernels index units with 32-bit offsets.
int64_t max_run_pages(const Shape &s) { return std::max<int64_t>(1, kMaxOuterVecs / s.BLPV); }

void clear_error() { g_last_error.clear(); }

}  // namespace hicache

int hicache::set_error_text(int code, const char *msg) {
  g_last_error.clear();
  return set_error(code, "%s", msg);
}

// ---- pool and plan objects -----------------------------------------------------
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
};

namespace hicache {

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
  while (next + size_t(count) < runs.size() && count < max_runs) {
    const RunRec &r = runs[next + size_t(count)];
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
  job.pad = 0;
  job.tiles_per_outer = int32_t((vecs + hicache::kTileVecs - 1) / hicache::kTileVecs);
  job.total_tiles = int32_t(job.tiles_per_outer * outers);
  return count;
}

int32_t fill_job(const std::vector<RunRec> &runs, size_t next, int64_t upp, int64_t outers,
                 int64_t max_runs, hicache::XferParams &params, int32_t word, int j,
                 int64_t launch_factor = 1) {
  return fill_runs(runs, next, upp, outers, max_runs, params.h.job[j],
                   reinterpret_cast<hicache::Run *>(&params.blob[word]), word, launch_factor);
}

// A pool's shape, host alias and dividers, as one launch header.
void fill_shape(const hicache_pool *pool, int64_t upp, int32_t layer, hicache::XferHeader &h) {
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
  h.job[1] = hicache::Job{0, nb, 0, 0};
}

// Header fields shared by every launch of a pool, and its buffer pointers.
void fill_header(const hicache_pool *pool, const hicache_device_kv *kv, hicache::XferParams &params,
                 int64_t upp, int32_t layer) {
  fill_shape(pool, upp, layer, params.h);
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
            void *stream) {
  const bool bidir = load_runs != nullptr;
  if (runs.empty() && (!bidir || load_runs->empty())) return HICACHE_OK;
  if (int rc = check_device(pool)) return rc;
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

  thread_local hicache::XferParams params;
  hicache::XferHeader &h = params.h;
  fill_header(pool, kv, params, upp, all ? 0 : layer);

  size_t next0 = 0, next1 = 0;
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
    // a fused launch carries both directions: one load share of CTAs for each
    const int64_t ctas = bidir ? 2 * int64_t(pool->ctas) : to_host ? pool->backup_ctas : pool->ctas;
    x.grid = int(std::min<int64_t>(tiles, ctas));
    x.stream = stream;
    const int e = hicache::launch_xfer(x);
    if (e != 0) return cuda_error(cudaError_t(e), "transfer kernel launch");
    g_launches.fetch_add(1, std::memory_order_relaxed);
    next0 += size_t(c0);
    next1 += size_t(c1);
  }
  return HICACHE_OK;
}

using WaitValue32Fn = CUresult (*)(CUstream, CUdeviceptr, cuuint32_t, unsigned int);

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

int enqueue_pipelined(hicache_pool *pool, const hicache_device_kv *kv, const std::vector<RunRec> &runs,
                      int32_t layout, void *stream) {
  if (int rc = check_device(pool)) return rc;
  if (!wait_value32())
    return set_error(HICACHE_ERR_CUDA, "the driver offers no cuStreamWaitValue32: no pipelined loads");
  std::lock_guard<std::mutex> g(pool->signal_mu);
  // the counts stay in order while pipelined loads follow one another on one
  // stream; another stream is fine once the earlier ones have finished
  if (pool->pipeline_stream_set && pool->pipeline_stream != stream &&
      cudaEventQuery(pool->pipeline_last) != cudaSuccess) {
    (void)cudaGetLastError();
    return set_error(HICACHE_ERR_INVALID_ARG,
                     "a pipelined load of this pool is still running on another stream");
  }
  pool->pipeline_stream_set = true;
  pool->pipeline_stream = stream;
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
    x.grid = int(std::min<int64_t>(int64_t(params.h.job[0].total_tiles) * s.L, pool->ctas));
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
  // the layer events also fire, once the whole load is in
  for (int64_t l = 0; l < s.L; ++l) {
    const cudaError_t e = cudaEventRecord(pool->events[size_t(l)], static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_error(e, "cudaEventRecord(layer event)");
  }
  const cudaError_t e = cudaEventRecord(pool->pipeline_last, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_error(e, "cudaEventRecord(pipelined load)");
  return HICACHE_OK;
}

// Sorted-merge test: do two page sets share a page?
bool intersects(std::vector<int64_t> a, std::vector<int64_t> b, int64_t *common) {
  std::sort(a.begin(), a.end());
  std::sort(b.begin(), b.end());
  size_t i = 0, k = 0;
  while (i < a.size() && k < b.size()) {
    if (a[i] == b[k]) {
      *common = a[i];
      return true;
    }
    if (a[i] < b[k]) ++i; else ++k;
  }
  return false;
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
  if ((rc = prepass(pool->shape.Hp, kv->device_num_pages, dev, host, n, direction,
                    max_run_pages(pool->shape), &runs)))
    return rc;
  if ((rc = enqueue(pool, kv, runs, nullptr, lay, layer, direction == HICACHE_DIR_BACKUP, stream)))
    return rc;
  if (layer >= 0) {
    const cudaError_t e = cudaEventRecord(pool->events[size_t(layer)], static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_error(e, "cudaEventRecord(layer event)");
    std::lock_guard<std::mutex> g(pool->signal_mu);
    pool->layer_signal[size_t(layer)] = 0;
  }
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
  p->ctas = desc->launch_ctas > 0 ? desc->launch_ctas : sms * hicache::kDefaultCtasPerSm;
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
  // (they all follow one another on one stream) before the words are freed
  if (pool->pipeline_stream_set && pool->pipeline_last) (void)cudaEventSynchronize(pool->pipeline_last);
  for (auto ev : pool->events)
    if (ev) cudaEventDestroy(ev);
  if (pool->layer_done) cudaFree(pool->layer_done);
  if (pool->pipeline_last) cudaEventDestroy(pool->pipeline_last);
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
  if (brun.empty()) return enqueue(pool, kv, lrun, nullptr, lay, -1, false, stream);
  return enqueue(pool, kv, brun, &lrun, lay, -1, true, stream);
}

// ---- buffer groups ------------------------------------------------------------
namespace hicache {

// Enqueue validated runs for every pool of a group, one launch per chunk of
// runs that fits the parameters of all of them.
int enqueue_group(hicache_pool *const *pools, const hicache_device_kv *kvs, int32_t np,
                  const std::vector<RunRec> &runs, int32_t layout, int32_t layer, bool to_host,
                  void *stream) {
  if (runs.empty()) return HICACHE_OK;
  const bool all = layer < 0;
  thread_local hicache::GroupParams params;
  hicache::GroupHeader &g = params.g;
  g.njobs = np;
  int32_t word = 0;
  int64_t outers[hicache::kMaxGroup], upp[hicache::kMaxGroup];
  for (int32_t j = 0; j < np; ++j) {
    const Shape &s = pools[j]->shape;
    const bool lf_all = (layout == HICACHE_LAYER_FIRST) && all;
    const bool kv_all = (layout == HICACHE_PAGE_FIRST_DIRECT_KV) && all;
    outers[j] = lf_all ? s.B * s.L : (kv_all ? 1 : s.B);
    upp[j] = !all || layout == HICACHE_LAYER_FIRST ? s.PV : (kv_all ? s.BLPV : s.LPV);
    fill_shape(pools[j], upp[j], all ? 0 : layer, g.h[j]);
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
    x.grid = int(std::min<int64_t>(tiles, to_host ? p0->backup_ctas : p0->ctas));
    x.stream = stream;
    const int e = hicache::launch_group(x);
    if (e != 0) return cuda_error(cudaError_t(e), "group transfer kernel launch");
    g_launches.fetch_add(1, std::memory_order_relaxed);
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
  int32_t word = 0;
  for (int32_t j = 0; j < np; ++j) {
    const Shape &s = pools[j]->shape;
    fill_shape(pools[j], s.PV, 0, g.h[j]);
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
    x.grid = int(std::min<int64_t>(tiles * L, pools[0]->ctas));
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

}  // namespace hicache

namespace hicache {

// The checks every group call shares: 1..HICACHE_MAX_GROUP distinct pools on
// one device with equal layers, page size and resolved layout, valid device KV
// for each, at most kMaxBufs buffers, no buffer named twice.  Returns the
// resolved layout and the bounds the pre-pass must apply to every pool.
int check_group(hicache_pool *const *pools, const hicache_device_kv *kvs, int32_t npools, int32_t layout,
                int32_t *lay, int64_t *Hp, int64_t *Dp, int64_t *max_run) {
  if (!pools || !kvs) return set_error(HICACHE_ERR_INVALID_ARG, "pools or kvs is NULL");
  if (npools < 1 || npools > HICACHE_MAX_GROUP)
    return set_error(HICACHE_ERR_INVALID_ARG, "npools = %d outside [1, %d]", npools, HICACHE_MAX_GROUP);
  for (int32_t i = 0; i < npools; ++i)
    if (!pools[i]) return set_error(HICACHE_ERR_INVALID_ARG, "pool %d is NULL", i);
  const hicache_pool *p0 = pools[0];
  int rc = resolve_layout(layout, p0->shape.layout, lay);
  if (rc) return rc;
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
    int32_t li = 0;
    if ((rc = resolve_layout(layout, p->shape.layout, &li))) return rc;
    if (li != *lay)
      return set_error(HICACHE_ERR_INVALID_ARG, "pool %d resolves to layout %d, pool 0 to %d", i, li, *lay);
    if ((rc = check_kv(p, &kvs[i], 0))) return rc;
    *Hp = std::min(*Hp, p->shape.Hp);
    *Dp = std::min(*Dp, kvs[i].device_num_pages);
    *max_run = std::min(*max_run, max_run_pages(p->shape));
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

int hicache_group_transfer(hicache_pool *const *pools, const hicache_device_kv *kvs, int32_t npools,
                           const int64_t *device_pages, const int64_t *host_pages, int64_t n,
                           int32_t layout, int32_t layer_id, int32_t direction, void *stream) {
  g_last_error.clear();
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
  }
  return HICACHE_OK;
}

int hicache_group_load_pipelined(hicache_pool *const *pools, const hicache_device_kv *kvs, int32_t npools,
                                 const int64_t *device_pages, const int64_t *host_pages, int64_t n,
                                 int32_t layout, void *stream) {
  g_last_error.clear();
  int32_t lay = 0;
  int64_t Hp = 0, Dp = 0, max_run = 0;
  int rc = check_group(pools, kvs, npools, layout, &lay, &Hp, &Dp, &max_run);
  if (rc) return rc;
  thread_local std::vector<RunRec> runs;
  if ((rc = prepass(Hp, Dp, device_pages, host_pages, n, HICACHE_DIR_LOAD, max_run, &runs))) return rc;
  if ((rc = check_device(pools[0]))) return rc;
  if (!wait_value32())
    return set_error(HICACHE_ERR_CUDA, "the driver offers no cuStreamWaitValue32: no pipelined loads");
  // every pool's signal lock, in address order (the pools are distinct)
  std::vector<hicache_pool *> order(pools, pools + npools);
  std::sort(order.begin(), order.end());
  std::vector<std::unique_lock<std::mutex>> locks;
  for (hicache_pool *p : order) locks.emplace_back(p->signal_mu);
  for (int32_t i = 0; i < npools; ++i) {
    hicache_pool *p = pools[i];
    if (p->pipeline_stream_set && p->pipeline_stream != stream &&
        cudaEventQuery(p->pipeline_last) != cudaSuccess) {
      (void)cudaGetLastError();
      return set_error(HICACHE_ERR_INVALID_ARG,
                       "a pipelined load of pool %d is still running on another stream", i);
    }
  }
  for (int32_t i = 0; i < npools; ++i) {
    pools[i]->pipeline_stream_set = true;
    pools[i]->pipeline_stream = stream;
  }
  if ((rc = enqueue_group_pipelined(pools, kvs, npools, runs, lay, stream))) return rc;
  for (int32_t i = 0; i < npools; ++i) {
    hicache_pool *p = pools[i];
    for (int64_t l = 0; l < p->shape.L; ++l) {
      const cudaError_t e = cudaEventRecord(p->events[size_t(l)], static_cast<cudaStream_t>(stream));
      if (e != cudaSuccess) return cuda_error(e, "cudaEventRecord(layer event)");
    }
    const cudaError_t e = cudaEventRecord(p->pipeline_last, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_error(e, "cudaEventRecord(pipelined load)");
  }
  return HICACHE_OK;
}

int hicache_plan_create(hicache_pool *pool, const int64_t *device_pages, const int64_t *host_pages,
                        int64_t n, int64_t device_num_pages, int32_t direction,
                        hicache_plan **out) {
  g_last_error.clear();
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
  g_last_error.clear();
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
  }
  return HICACHE_OK;
}

int hicache_plan_load_layer(const hicache_plan *plan, const hicache_device_kv *kv, int32_t layout,
                            int32_t layer_id, void *stream) {
  g_last_error.clear();
  if (layer_id < 0) return set_error(HICACHE_ERR_INVALID_ARG, "layer_id %d is negative", layer_id);
  return hicache_plan_execute(plan, kv, layout, layer_id, stream);
}

int hicache_load_pipelined(hicache_pool *pool, const hicache_device_kv *kv, const int64_t *device_pages,
                           const int64_t *host_pages, int64_t n, int32_t layout, void *stream) {
  g_last_error.clear();
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
  g_last_error.clear();
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

int hicache_plan_load_pipelined(const hicache_plan *plan, const hicache_device_kv *kv, int32_t layout,
                                void *stream) {
  g_last_error.clear();
  if (!plan) return set_error(HICACHE_ERR_INVALID_ARG, "plan is NULL");
  if (plan->direction != HICACHE_DIR_LOAD)
    return set_error(HICACHE_ERR_INVALID_ARG, "a pipelined transfer must be a load");
  int32_t lay = 0;
  int rc = resolve_layout(layout, plan->pool->shape.layout, &lay);
  if (rc) return rc;
  if ((rc = check_kv(plan->pool, kv, plan->device_num_pages))) return rc;
  return enqueue_pipelined(plan->pool, kv, plan->runs, lay, stream);
}

// ---- allocation-free pipelined load ---------------------------------------------
namespace {
// The value the library's static counters reach once every allocation-free
// pipelined load enqueued so far on a device has landed, per device and layer.
std::mutex g_noalloc_mu;
uint32_t g_noalloc_target[hicache::kNoAllocMaxDevices][hicache::kNoAllocMaxLayers];
uint32_t g_noalloc_slot[hicache::kNoAllocMaxDevices];  // next scheduler pair, per device
}  // namespace

int hicache_load_pipelined_noalloc(hicache_pool *pool, const hicache_device_kv *kv,
                                   const int64_t *device_pages, const int64_t *host_pages, int64_t n,
                                   int32_t layout, void *stream) {
  g_last_error.clear();
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
    x.grid = int(std::min<int64_t>(int64_t(params.h.job[0].total_tiles) * s.L, pool->ctas));
    x.stream = stream;
    unsigned int *sched = counters + hicache::kNoAllocMaxLayers +
                          2 * (g_noalloc_slot[pool->device]++ % hicache::kNoAllocSchedSlots);
    const int e = hicache::launch_pipelined_load(x, counters, sched);
    if (e != 0) return cuda_error(cudaError_t(e), "pipelined load kernel launch");
    g_launches.fetch_add(1, std::memory_order_relaxed);
    for (int64_t l = 0; l < s.L; ++l) target[l] += uint32_t(params.h.job[0].total_tiles);
    next += size_t(c);
  }
  pool->noalloc_done = counters;
  if (pool->noalloc_target.size() != size_t(s.L)) pool->noalloc_target.assign(size_t(s.L), 0);
  for (int64_t l = 0; l < s.L; ++l) {
    pool->noalloc_target[size_t(l)] = target[l];
    pool->layer_signal[size_t(l)] = 2;
  }
  for (int64_t l = 0; l < s.L; ++l) {
    const cudaError_t e = cudaEventRecord(pool->events[size_t(l)], static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_error(e, "cudaEventRecord(layer event)");
  }
  return HICACHE_OK;
}

int hicache_plan_info(const hicache_plan *plan, int64_t *num_pages, int64_t *num_runs) {
  g_last_error.clear();
  if (!plan) return set_error(HICACHE_ERR_INVALID_ARG, "plan is NULL");
  if (num_pages) *num_pages = plan->n;
  if (num_runs) *num_runs = int64_t(plan->runs.size());
  return HICACHE_OK;
}

int hicache_plan_load_layers(hicache_plan *plan, const hicache_device_kv *kv, int32_t layout, void *stream) {
  g_last_error.clear();
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
    if (plan->graph) {
      cudaGraphExecDestroy(plan->graph);
      plan->graph = nullptr;
    }
    // Capture the L per-layer launches on a private stream, the kernels one
    // after another.  Each layer's event is recorded (as an external event
    // node) on a side branch that forks off after that layer's kernel, so the
    // kernel chain itself has no node between consecutive launches.
    cudaStream_t cap = nullptr, side = nullptr;
    std::vector<cudaEvent_t> forks(size_t(s.L) + 1, nullptr);
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
    const int64_t before = g_launches.load();
    for (int64_t l = 0; l < s.L && rc == HICACHE_OK; ++l) {
      rc = enqueue(pool, kv, plan->runs, nullptr, lay, int32_t(l), false, cap);
      if (rc != HICACHE_OK) break;
      e = cudaEventRecord(forks[size_t(l)], cap);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(side, forks[size_t(l)], 0);
      if (e == cudaSuccess) e = cudaEventRecordWithFlags(pool->events[size_t(l)], side, cudaEventRecordExternal);
      if (e != cudaSuccess) rc = cuda_error(e, "capturing the layer event");
    }
    if (rc == HICACHE_OK) {                // join the side branch back
      e = cudaEventRecord(forks[size_t(s.L)], side);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(cap, forks[size_t(s.L)], 0);
      if (e != cudaSuccess) rc = cuda_error(e, "joining the capture");
    }
    const int64_t captured = g_launches.load() - before;
    g_launches.fetch_sub(captured);      // counted when replayed
    cudaGraph_t graph = nullptr;
    e = cudaStreamEndCapture(cap, &graph);
    release();
    if (rc == HICACHE_OK && e != cudaSuccess) rc = cuda_error(e, "cudaStreamEndCapture");
    if (rc == HICACHE_OK) {
      e = cudaGraphInstantiate(&plan->graph, graph, 0);
      if (e != cudaSuccess) {
        plan->graph = nullptr;
        rc = cuda_error(e, "cudaGraphInstantiate");
      }
    }
    if (graph) cudaGraphDestroy(graph);
    if (rc != HICACHE_OK) return rc;
    plan->graph_bufs = bufs;
    plan->graph_pages = kv->device_num_pages;
    plan->graph_layout = lay;
    plan->graph_launches = captured;
  }
  const cudaError_t e = cudaGraphLaunch(plan->graph, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_error(e, "cudaGraphLaunch");
  g_launches.fetch_add(plan->graph_launches, std::memory_order_relaxed);
  std::lock_guard<std::mutex> gs(pool->signal_mu);
  for (int64_t l = 0; l < s.L; ++l) pool->layer_signal[size_t(l)] = 0;
  return HICACHE_OK;
}

int hicache_plan_destroy(hicache_plan *plan) {
  if (plan && plan->graph) cudaGraphExecDestroy(plan->graph);
  delete plan;
  return HICACHE_OK;
}

int hicache_layer_event(hicache_pool *pool, int32_t layer, void **event_out) {
  g_last_error.clear();
  if (!pool || !event_out) return set_error(HICACHE_ERR_INVALID_ARG, "pool or event_out is NULL");
  if (layer < 0 || layer >= pool->shape.L)
    return set_error(HICACHE_ERR_INVALID_ARG, "layer %d outside [0, %lld)", layer,
                     (long long)pool->shape.L);
  *event_out = pool->events[size_t(layer)];
  return HICACHE_OK;
}

int hicache_wait_layer(hicache_pool *pool, int32_t layer, void *compute_stream) {
  g_last_error.clear();
  if (!pool) return set_error(HICACHE_ERR_INVALID_ARG, "pool is NULL");
  if (layer < 0 || layer >= pool->shape.L)
    return set_error(HICACHE_ERR_INVALID_ARG, "layer %d outside [0, %lld)", layer,
                     (long long)pool->shape.L);
  std::lock_guard<std::mutex> g(pool->signal_mu);
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
  const cudaError_t e = cudaStreamWaitEvent(static_cast<cudaStream_t>(compute_stream),
                                            pool->events[size_t(layer)], 0);
  if (e != cudaSuccess) return cuda_error(e, "cudaStreamWaitEvent");
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

int hicache_prepass(int64_t host_num_pages, int64_t device_num_pages, const int64_t *device_pages,
                    const int64_t *host_pages, int64_t n, int32_t direction, int64_t *num_runs,
                    int64_t *runs_out, int64_t runs_capacity) {
  g_last_error.clear();
  if (!num_runs) return set_error(HICACHE_ERR_INVALID_ARG, "num_runs is NULL");
  if (host_num_pages < 1 || host_num_pages >= INT32_MAX)
    return set_error(HICACHE_ERR_INVALID_ARG, "host_num_pages must be in [1, 2^31)");
  thread_local std::vector<RunRec> tls_runs;
  std::vector<RunRec> &runs = tls_runs;
  const int rc = prepass(host_num_pages, device_num_pages, device_pages, host_pages, n, direction,
                         INT32_MAX, &runs);
  if (rc) return rc;
  *num_runs = int64_t(runs.size());
  if (runs_out && runs_capacity >= int64_t(runs.size())) {
    for (size_t i = 0; i < runs.size(); ++i) {
      runs_out[3 * i] = runs[i].h0;
      runs_out[3 * i + 1] = runs[i].d0;
      runs_out[3 * i + 2] = runs[i].len;
    }
  }
  return HICACHE_OK;
}

int64_t hicache_segment_count(const hicache_pool_desc *desc, const int64_t *device_pages,
                              const int64_t *host_pages, int64_t n, int32_t layout,
                              int32_t layer_id) {
  g_last_error.clear();
  Shape s{};
  int rc = check_desc(desc, &s, false);
  if (rc) return rc;
  int32_t lay = 0;
  if ((rc = resolve_layout(layout, s.layout, &lay))) return rc;
  if (layer_id >= s.L)
    return set_error(HICACHE_ERR_INVALID_ARG, "layer_id %d outside [0, %lld)", layer_id,
                     (long long)s.L);
  if (n < 0) return set_error(HICACHE_ERR_INVALID_ARG, "n is negative");
  if (n == 0) return 0;
  if (!device_pages || !host_pages) return set_error(HICACHE_ERR_INVALID_ARG, "index array is NULL");
  // runs over the set of pairs; repeated sources are fine for a count
  std::vector<Pair> pairs(static_cast<size_t>(n));
  for (int64_t i = 0; i < n; ++i) {
    if (device_pages[i] < 0 || host_pages[i] < 0 || host_pages[i] >= s.Hp)
      return set_error(HICACHE_ERR_INDEX_RANGE, "page index out of range at %lld", (long long)i);
    pairs[size_t(i)] = Pair{host_pages[i], device_pages[i]};
  }
  std::sort(pairs.begin(), pairs.end(), pair_less);
  int64_t nruns = 0;
  for (int64_t i = 0; i < n; ++i) {
    const bool cont = i > 0 && pairs[size_t(i)].h == pairs[size_t(i - 1)].h + 1 &&
                      pairs[size_t(i)].d == pairs[size_t(i - 1)].d + 1;
    if (!cont) ++nruns;
  }
  const int64_t layers = layer_id < 0 ? s.L : 1;
  // with one layer in the pool, every layout stores a buffer's pages back to
  // back, except page_first_direct_kv, which interleaves the buffers of a page
  if (lay == HICACHE_LAYER_FIRST || (s.L == 1 && (lay != HICACHE_PAGE_FIRST_DIRECT_KV || s.B == 1)))
    return s.B * layers * nruns;
  // one segment per (buffer, layer, page): the same layer of the next page is
  // (buffers x) L*P rows further on the host
  if (lay == HICACHE_PAGE_FIRST_DIRECT || lay == HICACHE_PAGE_FIRST_DIRECT_KV) return s.B * layers * n;
  return s.B * layers * n * s.P;  // page_first: one row per (buffer, layer, token)
}

int hicache_page_span(const hicache_pool_desc *desc, int64_t host_page, int32_t buffer,
                      int64_t *offset_bytes, int64_t *nbytes) {
  g_last_error.clear();
  Shape s{};
  int rc = check_desc(desc, &s, false);
  if (rc) return rc;
  if (!offset_bytes || !nbytes) return set_error(HICACHE_ERR_INVALID_ARG, "output pointer is NULL");
  if (host_page < 0 || host_page >= s.Hp)
    return set_error(HICACHE_ERR_INDEX_RANGE, "host page %lld outside [0, %lld)", (long long)host_page,
                     (long long)s.Hp);
  if (buffer < -1 || buffer >= s.B)
    return set_error(HICACHE_ERR_INVALID_ARG, "buffer %d outside [-1, %lld)", buffer, (long long)s.B);
  const int64_t page_buf_bytes = s.L * s.P * s.R * s.es;  // one buffer's share of a page
  switch (s.layout) {
    case HICACHE_PAGE_FIRST:
    case HICACHE_PAGE_FIRST_DIRECT:
      if (buffer < 0 && s.B > 1)
        return set_error(HICACHE_ERR_INVALID_ARG,
                         "with %lld buffers a page is one span per buffer: name the buffer",
                         (long long)s.B);
      *offset_bytes = ((buffer < 0 ? 0 : buffer) * s.Hp + host_page) * page_buf_bytes;
      *nbytes = page_buf_bytes;
      return HICACHE_OK;
    case HICACHE_PAGE_FIRST_DIRECT_KV:
      if (buffer < 0) {
        *offset_bytes = host_page * s.B * page_buf_bytes;
        *nbytes = s.B * page_buf_bytes;
      } else {
        *offset_bytes = (host_page * s.B + buffer) * page_buf_bytes;
        *nbytes = page_buf_bytes;
      }
      return HICACHE_OK;
    default:
      if (s.L == 1 && (buffer >= 0 || s.B == 1)) {
        *offset_bytes = ((buffer < 0 ? 0 : buffer) * s.Hp + host_page) * page_buf_bytes;
        *nbytes = page_buf_bytes;
        return HICACHE_OK;
      }
      return set_error(HICACHE_ERR_INVALID_ARG,
                       "a layer_first page is one span per layer, not one contiguous span");
  }
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
