// hicache_index.cpp -- host-only argument validation and the index pre-pass:
// pool-shape and layout checks, the sort of (host page, device page) pairs and
// their merge into runs, and the host-only calls built on them (the pre-pass
// itself, segment counts and page spans).  Nothing here touches a GPU.

#include <unistd.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <condition_variable>
#include <cstdint>
#include <cstdlib>
#include <functional>
#include <mutex>
#include <thread>
#include <vector>

#include "hicache.h"
#include "hicache_host.h"
#include "hicache_internal.h"

namespace hicache {

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

// ---- validation ----------------------------------------------------------------
//
// One pass over the pairs that only notes whether anything is wrong: ranges,
// order, and repeated destinations.  It is all a large call costs the host
// before its first launch, so it has no early exit; the exact first error is
// looked for only when something was wrong.

struct Scan {
  bool bad = false;       // a page out of range
  bool in_order = true;   // (host page, device page) never decreases
  bool strict = true;     // the destination page always increases
  uint64_t dup = 0;       // nonzero: a destination page met twice in the bitmap
};

// Pairs [lo, hi).  BACKUP: the destination is the host page.  BITS: note each
// destination page below `bound` in `bits`, one bit per page.
template <bool BACKUP, bool BITS>
Scan scan_pairs(const int64_t *dev, const int64_t *host, int64_t lo, int64_t hi, int64_t Hp, int64_t Dp,
                uint64_t bound, uint64_t *bits) {
  Scan r;
  bool bad = false, in_order = true, strict = true;
  uint64_t dup = 0;
  for (int64_t i = lo; i < hi; ++i) {
    const int64_t d = dev[i], h = host[i];
    bad |= uint64_t(d) >= uint64_t(Dp) || uint64_t(h) >= uint64_t(Hp);
    if (i > lo) {
      in_order &= !(h < host[i - 1] || (h == host[i - 1] && d < dev[i - 1]));
      strict &= BACKUP ? h > host[i - 1] : d > dev[i - 1];
    }
    if (BITS) {
      const uint64_t x = uint64_t(BACKUP ? h : d);
      if (x < bound) {
        uint64_t &w = bits[x >> 6];
        const uint64_t bit = uint64_t(1) << (x & 63);
        dup |= w & bit;
        w |= bit;
      }
    }
  }
  r.bad = bad;
  r.in_order = in_order;
  r.strict = strict;
  r.dup = dup;
  return r;
}

// Worker threads for the validation of large calls.  A call of at least
// kParallelPairs pairs splits its pass over up to kValidateParts threads: the
// calling thread and the workers scan chunks of the pairs, each thread into a
// bitmap of its own, and the caller then merges the bitmaps (a page set in
// two of them is a repeated destination).  The pool is made on first
// use in each process (threads do not survive fork(), so a child makes its
// own) and is never destroyed: its workers sleep on it between calls until
// the process exits, and the library is linked so that it is never unloaded.
// One call at a time uses it; a call that finds it busy scans on its own.
// HICACHE_VALIDATE_THREADS=1 (read once) keeps every pass on the calling
// thread; 2 to 4 sets the number of parts.
constexpr int64_t kParallelPairs = 49152;
constexpr int kValidateParts = 4;
constexpr int64_t kValidateChunks = 32;

class Workers {
 public:
  static Workers *get() {
    static std::mutex mu;
    static Workers *pool = nullptr;
    static pid_t owner = 0;
    std::lock_guard<std::mutex> g(mu);
    if (pool && owner == getpid()) return pool->workers_ ? pool : nullptr;
    pool = new Workers;  // never deleted (see above); an old pool of a parent process is left alone
    owner = getpid();
    int parts = kValidateParts;
    const unsigned hw = std::thread::hardware_concurrency();
    if (hw < 2 * kValidateParts) parts = hw >= 4 ? 2 : 1;
    if (const char *env = std::getenv("HICACHE_VALIDATE_THREADS"))
      parts = std::max(1, std::min(kValidateParts, std::atoi(env)));
    for (int k = 1; k < parts; ++k) {
      try {
        std::thread(&Workers::loop, pool, k).detach();
      } catch (...) {
        break;
      }
      ++pool->workers_;
    }
    return pool->workers_ ? pool : nullptr;
  }

  int parts() const { return workers_ + 1; }
  std::mutex &job() { return job_; }
  // the bitmap of part k >= 1 (guarded by job())
  std::vector<uint64_t> &bits(int k) { return bits_[k]; }

  // Run fn(0) on the calling thread and fn(k) for 0 < k < n on the workers;
  // return once all have returned.  The caller holds job().
  void run(int n, const std::function<void(int)> &fn) {
    {
      std::lock_guard<std::mutex> g(m_);
      fn_ = &fn;
      n_ = n;
      pending_ = n - 1;
      ++gen_;
    }
    wake_.notify_all();
    fn(0);
    std::unique_lock<std::mutex> g(m_);
    done_.wait(g, [&] { return pending_ == 0; });
  }

 private:
  void loop(int k) {
    uint64_t seen = 0;
    std::unique_lock<std::mutex> g(m_);
    for (;;) {
      wake_.wait(g, [&] { return gen_ != seen; });
      seen = gen_;
      if (k >= n_) continue;
      const std::function<void(int)> *fn = fn_;
      g.unlock();
      (*fn)(k);
      g.lock();
      if (--pending_ == 0) done_.notify_one();
    }
  }

  std::mutex job_, m_;
  std::condition_variable wake_, done_;
  uint64_t gen_ = 0;
  int n_ = 0, pending_ = 0, workers_ = 0;
  const std::function<void(int)> *fn_ = nullptr;
  std::vector<uint64_t> bits_[kValidateParts];
};

// Scan pairs [0, n) in parts on the workers when the call is large enough and
// the pool is free; otherwise in one part here.  `bits0` is the calling
// thread's bitmap (BITS); every bitmap is left cleared.
template <bool BACKUP, bool BITS>
Scan scan_all(const int64_t *dev, const int64_t *host, int64_t n, int64_t Hp, int64_t Dp, uint64_t bound,
              uint64_t *bits0, size_t words) {
  Workers *w = n >= kParallelPairs ? Workers::get() : nullptr;
  std::unique_lock<std::mutex> j;
  int parts = 1;
  if (w) {
    parts = w->parts();
    // merging the bitmaps costs words x parts; keep that below one step per pair
    while (BITS && parts > 1 && uint64_t(words) * uint64_t(parts) > uint64_t(n)) --parts;
    if (parts > 1) j = std::unique_lock<std::mutex>(w->job(), std::try_to_lock);
    if (!j.owns_lock()) parts = 1;
  }
  if (parts == 1) {
    Scan r = scan_pairs<BACKUP, BITS>(dev, host, 0, n, Hp, Dp, bound, bits0);
    if (BITS) {
      if (words <= size_t(2 * n)) {
        std::fill(bits0, bits0 + words, uint64_t(0));
      } else {
        const int64_t *dst = BACKUP ? host : dev;
        for (int64_t k = 0; k < n; ++k)
          if (uint64_t(dst[k]) < bound) bits0[size_t(dst[k] >> 6)] = 0;
      }
    }
    return r;
  }
  uint64_t *bits[kValidateParts] = {bits0};
  for (int k = 1; k < parts; ++k) {
    std::vector<uint64_t> &v = w->bits(k);
    if (BITS && v.size() < words) v.resize(words, 0);
    bits[k] = v.data();
  }
  // The pairs go out in kValidateChunks contiguous chunks, each thread taking
  // the next free one: the caller starts at once, the workers as they wake.
  Scan rs[kValidateParts];
  std::atomic<int64_t> next{0};
  const std::function<void(int)> part = [&](int k) {
    Scan acc;
    for (int64_t c; (c = next.fetch_add(1, std::memory_order_relaxed)) < kValidateChunks;) {
      const Scan t = scan_pairs<BACKUP, BITS>(dev, host, n * c / kValidateChunks, n * (c + 1) / kValidateChunks,
                                              Hp, Dp, bound, bits[k]);
      acc.bad |= t.bad;
      acc.in_order &= t.in_order;
      acc.strict &= t.strict;
      acc.dup |= t.dup;
    }
    rs[k] = acc;
  };
  w->run(parts, part);
  Scan r;
  for (int k = 0; k < parts; ++k) {
    r.bad |= rs[k].bad;
    r.in_order &= rs[k].in_order;
    r.strict &= rs[k].strict;
    r.dup |= rs[k].dup;
  }
  for (int64_t c = 1; c < kValidateChunks; ++c) {  // the pair before each chunk's first
    const int64_t i = n * c / kValidateChunks;
    r.in_order &= !(host[i] < host[i - 1] || (host[i] == host[i - 1] && dev[i] < dev[i - 1]));
    r.strict &= BACKUP ? host[i] > host[i - 1] : dev[i] > dev[i - 1];
  }
  if (BITS) {
    uint64_t dup = 0;
    for (size_t x = 0; x < words; ++x) {
      uint64_t acc = 0;
      for (int k = 0; k < parts; ++k) {
        dup |= acc & bits[k][x];
        acc |= bits[k][x];
        bits[k][x] = 0;
      }
    }
    r.dup |= dup;
  }
  return r;
}

// Check n index pairs without reducing them: both pages in range, no
// destination named twice (host pages of a backup, device pages of a load),
// and whether the pairs already come in (host page, device page) order.
int validate_pairs(int64_t Hp, int64_t Dp, const int64_t *dev, const int64_t *host, int64_t n,
                   int32_t direction, bool *sorted) {
  if (n < 0) return set_error(HICACHE_ERR_INVALID_ARG, "n = %lld is negative", (long long)n);
  if (direction != HICACHE_DIR_BACKUP && direction != HICACHE_DIR_LOAD)
    return set_error(HICACHE_ERR_INVALID_ARG, "unknown direction %d", direction);
  if (Dp < 1 || Dp >= INT32_MAX)
    return set_error(HICACHE_ERR_INVALID_ARG, "device_num_pages = %lld must be in [1, 2^31)",
                     (long long)Dp);
  *sorted = true;
  if (n == 0) return HICACHE_OK;
  if (!dev || !host) return set_error(HICACHE_ERR_INVALID_ARG, "index array is NULL");
  const bool backup = direction == HICACHE_DIR_BACKUP;
  const int64_t *dst = backup ? host : dev;
  const int64_t bound = backup ? Hp : Dp;
  // A backup whose host pages strictly increase (the usual order) names no
  // host page twice, so it needs no bitmap; other backups are checked
  // afterwards.  A load notes its device pages in a bitmap of one bit per
  // page (pools of up to 2^27 pages).
  const bool bitmap = !backup && n > 32 && bound <= (int64_t(1) << 27);
  Scan r;
  if (backup) {
    r = scan_all<true, false>(dev, host, n, Hp, Dp, uint64_t(bound), nullptr, 0);
  } else if (bitmap) {
    thread_local std::vector<uint64_t> tls_bits;
    std::vector<uint64_t> &vbits = tls_bits;
    const size_t words = size_t((bound + 63) / 64);
    if (vbits.size() < words) vbits.resize(words, 0);
    r = scan_all<false, true>(dev, host, n, Hp, Dp, uint64_t(bound), vbits.data(), words);
  } else {
    r = scan_all<false, false>(dev, host, n, Hp, Dp, uint64_t(bound), nullptr, 0);
  }
  if (r.bad) {
    for (int64_t i = 0; i < n; ++i) {
      if (dev[i] < 0 || dev[i] >= Dp)
        return set_error(HICACHE_ERR_INDEX_RANGE, "device_pages[%lld] = %lld outside [0, %lld)", (long long)i,
                         (long long)dev[i], (long long)Dp);
      if (host[i] < 0 || host[i] >= Hp)
        return set_error(HICACHE_ERR_INDEX_RANGE, "host_pages[%lld] = %lld outside [0, %lld)", (long long)i,
                         (long long)host[i], (long long)Hp);
    }
  }
  *sorted = r.in_order;
  int64_t page = 0;
  bool repeated = false;
  if (r.strict) {
    // strictly increasing destinations: none repeats
  } else if (bitmap) {
    if (r.dup) repeated = first_repeated(dst, n, bound, &page);
  } else if (n <= 32) {
    for (int64_t a = 0; a < n && !repeated; ++a)
      for (int64_t b = a + 1; b < n; ++b)
        if (dst[a] == dst[b]) {
          repeated = true;
          page = dst[a];
          break;
        }
  } else {
    repeated = first_repeated(dst, n, bound, &page);
  }
  if (repeated)
    return set_error(HICACHE_ERR_DUPLICATE_INDEX, "%s page %lld is a %s destination twice",
                     backup ? "host" : "device", (long long)page, backup ? "backup" : "load");
  return HICACHE_OK;
}

// Append the runs of pairs [begin, end) of a sequence sorted by (host page,
// device page) to *runs, continuing its last run where both pages step by one
// (at most max_run pages per run).
void append_runs(const int64_t *dev, const int64_t *host, int64_t begin, int64_t end, int64_t max_run,
                 std::vector<RunRec> *runs) {
  for (int64_t i = begin; i < end; ++i) {
    const int64_t h = host[i], d = dev[i];
    if (!runs->empty()) {
      RunRec &r = runs->back();
      if (h == r.h0 + r.len && d == r.d0 + r.len && r.len < max_run) {
        ++r.len;
        continue;
      }
    }
    runs->push_back(RunRec{h, d, 1});
  }
}

// Validate n index pairs and reduce them to runs: pairs sorted by (host page,
// device page), merged while both pages step by one (at most max_run pages per
// run).  On error the last-error text is set and *runs holds no usable table.
int prepass(int64_t Hp, int64_t Dp, const int64_t *dev, const int64_t *host, int64_t n,
            int32_t direction, int64_t max_run, std::vector<RunRec> *runs) {
  runs->clear();
  bool sorted = true;
  if (int rc = validate_pairs(Hp, Dp, dev, host, n, direction, &sorted)) return rc;
  build_runs(Dp, dev, host, n, sorted, max_run, runs);
  return HICACHE_OK;
}

// The runs of n validated pairs (sorted: they already come in host order).
void build_runs(int64_t Dp, const int64_t *dev, const int64_t *host, int64_t n, bool sorted, int64_t max_run,
                std::vector<RunRec> *runs) {
  runs->clear();
  if (n == 0) return;
  if (sorted) {
    append_runs(dev, host, 0, n, max_run, runs);
    return;
  }
  // one lookup of the per-thread buffer: in a shared library every access to
  // a thread_local can be a call, too slow inside a per-page loop
  thread_local std::vector<Pair> tls_pairs;
  std::vector<Pair> &pairs = tls_pairs;
  pairs.resize(size_t(n));
  for (int64_t i = 0; i < n; ++i) pairs[size_t(i)] = Pair{host[i], dev[i]};
  sort_pairs(pairs, Dp);
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
}

// Runs are capped so that a unit (at most every buffer and layer of a run)
// stays below 2^31 - 1024 vectors: the kernels index units with 32-bit offsets.
int64_t max_run_pages(const Shape &s) { return std::max<int64_t>(1, kMaxOuterVecs / s.BLPV); }

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

}  // namespace hicache

using namespace hicache;

extern "C" {

int hicache_prepass(int64_t host_num_pages, int64_t device_num_pages, const int64_t *device_pages,
                    const int64_t *host_pages, int64_t n, int32_t direction, int64_t *num_runs,
                    int64_t *runs_out, int64_t runs_capacity) {
  clear_error();
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
  clear_error();
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
  clear_error();
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

}  // extern "C"
