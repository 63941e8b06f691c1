// hicache_alloc.cpp -- host-page allocator for the L2 pool: a LIFO free list of
// page runs.
//
// "Tuning SGLang HiCache L2 on Kunlunxin P800/P900", section 2.4, and "Baidu's
// KVCache Overhaul", section "LIFO slot allocation": a FIFO free list pushes
// freed slots to the tail and scans the whole pool, scattering writes; a LIFO
// list hands back the most recently freed slots first, which keeps writes on a
// small set of hot pages (no change to what is cached, only to where).
//
// Here the free list is a stack of runs [start, start + len).  alloc(n) pops
// runs from the top and takes pages from the front of each run, so a request
// is served by as few, as long, ascending runs as the top of the stack allows
// (fewer runs = fewer segments for the transfer pre-pass).  free() sorts the
// pages, merges them into runs and pushes those on top, so they are the next
// ones handed out.  A bitmap rejects double frees and frees of pages that were
// never handed out; every error leaves the allocator unchanged.

#include <algorithm>
#include <climits>
#include <cstdint>
#include <mutex>
#include <new>
#include <vector>

#include "hicache.h"
#include "hicache_internal.h"

using hicache::set_error_text;

namespace {
struct Span {
  int64_t start, len;
};
}  // namespace

struct hicache_page_allocator {
  int64_t num_pages = 0;
  int64_t available = 0;
  std::vector<Span> stack;          // top = back()
  std::vector<uint64_t> allocated;  // one bit per page
  std::mutex mu;

  bool is_allocated(int64_t p) const { return (allocated[size_t(p >> 6)] >> (p & 63)) & 1u; }
  void set(int64_t p, bool v) {
    uint64_t &w = allocated[size_t(p >> 6)];
    const uint64_t bit = uint64_t(1) << (p & 63);
    w = v ? (w | bit) : (w & ~bit);
  }
};

extern "C" {

int hicache_allocator_create(int64_t num_pages, hicache_page_allocator **out) {
  if (!out || num_pages < 1 || num_pages >= INT32_MAX)
    return set_error_text(HICACHE_ERR_INVALID_ARG, "num_pages must be in [1, 2^31) and out non-NULL");
  hicache_page_allocator *a = new (std::nothrow) hicache_page_allocator();
  if (!a) return set_error_text(HICACHE_ERR_NOMEM, "out of host memory");
  a->num_pages = num_pages;
  a->available = num_pages;
  a->stack.push_back(Span{0, num_pages});
  a->allocated.assign(size_t((num_pages + 63) / 64), 0);
  *out = a;
  return HICACHE_OK;
}

int hicache_allocator_destroy(hicache_page_allocator *a) {
  delete a;
  return HICACHE_OK;
}

int64_t hicache_allocator_available(hicache_page_allocator *a) {
  if (!a) return set_error_text(HICACHE_ERR_INVALID_ARG, "allocator is NULL");
  std::lock_guard<std::mutex> g(a->mu);
  return a->available;
}

int hicache_allocator_alloc(hicache_page_allocator *a, int64_t n, int64_t *pages_out) {
  if (!a || n < 0 || (n > 0 && !pages_out))
    return set_error_text(HICACHE_ERR_INVALID_ARG, "bad allocator, count or output array");
  std::lock_guard<std::mutex> g(a->mu);
  if (n > a->available) return set_error_text(HICACHE_ERR_NOMEM, "not enough free host pages");
  int64_t k = 0;
  while (k < n) {
    Span &top = a->stack.back();
    const int64_t take = std::min(top.len, n - k);
    for (int64_t i = 0; i < take; ++i) {
      pages_out[k + i] = top.start + i;
      a->set(top.start + i, true);
    }
    k += take;
    top.start += take;
    top.len -= take;
    if (top.len == 0) a->stack.pop_back();
  }
  a->available -= n;
  return HICACHE_OK;
}

int hicache_allocator_free(hicache_page_allocator *a, const int64_t *pages, int64_t n) {
  if (!a || n < 0 || (n > 0 && !pages))
    return set_error_text(HICACHE_ERR_INVALID_ARG, "bad allocator, count or page array");
  std::lock_guard<std::mutex> g(a->mu);
  std::vector<int64_t> p(pages, pages + n);
  std::sort(p.begin(), p.end());
  for (int64_t i = 0; i < n; ++i) {
    if (p[size_t(i)] < 0 || p[size_t(i)] >= a->num_pages)
      return set_error_text(HICACHE_ERR_INDEX_RANGE, "freed page outside the pool");
    if ((i > 0 && p[size_t(i)] == p[size_t(i - 1)]) || !a->is_allocated(p[size_t(i)]))
      return set_error_text(HICACHE_ERR_DUPLICATE_INDEX, "page freed twice or never handed out");
  }
  // runs pushed highest first, so the lowest freed run ends on top
  std::vector<Span> runs;
  for (int64_t i = 0; i < n; ++i) {
    a->set(p[size_t(i)], false);
    if (!runs.empty() && runs.back().start + runs.back().len == p[size_t(i)])
      ++runs.back().len;
    else
      runs.push_back(Span{p[size_t(i)], 1});
  }
  for (auto it = runs.rbegin(); it != runs.rend(); ++it) a->stack.push_back(*it);
  a->available += n;
  return HICACHE_OK;
}

}  // extern "C"
