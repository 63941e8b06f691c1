/*
 * hicache_oracle.c -- CPU oracle for the L1 <-> L2 KV page movement of a tiered
 * prefix-KV cache (HiCache: GPU HBM is L1, pinned host DRAM is L2).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU-baseline
 * leg of the benchmark load this code.  The product path (the CUDA library under
 * tiered_kv_cache_gb300/) never links, imports or calls it, and this file shares
 * no code, header or helper with it.
 *
 * The oracle is the plain definition of the copy, one element at a time, in the
 * order the definition is stated.  It is deliberately slow and single-threaded.
 *
 * Sources (page title, section):
 *  [T21] "Tuning SGLang HiCache L2 on Kunlunxin P800/P900: Layout, DMA, NUMA and
 *        TP-Shared KV", section 2.1 "Layout choice: page_first_direct to layer_first":
 *        - the device side keeps one buffer per layer ("different layers are
 *          different buffers");
 *        - page_first_direct dims are (page_num, layer_num, page_size, 1, kv_dim),
 *          page outermost;
 *        - layer_first dims are (layer, size, 1, kv_dim);
 *        - segment count: page_num x layer_num for page_first_direct; about
 *          layer_num ("78 contiguous copies") for layer_first with contiguous pages.
 *  [B-L2] "Baidu's KVCache Overhaul: 36% TTFT Cut via Hit-Rate & Multi-Chip
 *        Tuning", sections "L2 Layout Choice: Layer-First vs Page-First Direct"
 *        (L1 is fixed layer-first, contiguous per layer) and "DMA Segment
 *        Explosion & Batched Gather/Scatter" (write-back gathers all layers of a
 *        page, load scatters back; the content moved does not depend on layout).
 *  [H-DT] "HiCache 시스템 설계와 최적화" (HiCache system design and optimisation),
 *        section "데이터 전송 최적화" (data-transfer optimisation): under page_first
 *        all KV of one page is contiguous and an L2 -> GPU copy goes at the
 *        granularity of one token per layer; page_first_direct groups all tokens
 *        of one layer inside a page.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - indices are PAGE indices; device token slot of (page d, token t) is d*P + t;
 *  - page_first dims are (size, layer, 1, kv_dim): token-major, then layer
 *    (the "one token per layer" granularity of [H-DT]);
 *  - separate K and V (MHA/GQA) add a leading buffer dim B in front of the
 *    printed per-buffer dims (K sub-pool, then V sub-pool); MLA has B = 1;
 *  - the i-th device page pairs with the i-th host page; elements are copied as
 *    raw bytes (no dtype conversion, NaN payloads and signed zeros survive);
 *  - a load_layer call moves every buffer of that one layer;
 *  - page_first_direct_kv (an L3-ready variant): dims (page_num, B, layer_num,
 *    page_size, 1, kv_dim), so that ALL the KV of one page -- K and V, every
 *    layer -- is one contiguous block that can go to L3 as a single object.
 *    [B-L2] "L2 Layout Choice": L3 needs page-first, contiguous per page, for
 *    large sequential I/O and zero-copy; "DMA Segment Explosion & Batched
 *    Gather/Scatter": write-back gathers all layers into a contiguous page.
 *    [H-DT] "배치 지향 데이터 구성": all KV of a page in contiguous memory,
 *    handed to L3 as a single object without copies.
 *
 * Notation (matches the pages' dims):
 *   B  buffers (2 = K,V ; 1 = MLA latent)      L  layers (layer_num)
 *   P  page_size (tokens per page)              R  kv_dim elements per token row
 *   Hp host pool pages (page_num)               S  = Hp*P host pool tokens ("size")
 *   es element size in bytes
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_LAYER_FIRST 0
#define ORACLE_PAGE_FIRST 1
#define ORACLE_PAGE_FIRST_DIRECT 2
#define ORACLE_PAGE_FIRST_DIRECT_KV 3

/* Offset, in elements, of element (b, l, h, t, e) inside the host pool.
 * Returns -1 for an unknown layout. */
int64_t oracle_host_elem_offset(int32_t layout, int64_t B, int64_t L, int64_t P,
                                int64_t R, int64_t Hp, int64_t b, int64_t l,
                                int64_t h, int64_t t, int64_t e) {
  const int64_t S = Hp * P;   /* "size": tokens in the host pool, per buffer */
  switch (layout) {
    case ORACLE_LAYER_FIRST:
      /* dims (B, layer, size, 1, kv_dim)                                  [T21] */
      return (((b * L + l) * S) + h * P + t) * R + e;
    case ORACLE_PAGE_FIRST:
      /* dims (B, size, layer, 1, kv_dim): one token holds every layer  [H-DT] */
      return (((b * S) + h * P + t) * L + l) * R + e;
    case ORACLE_PAGE_FIRST_DIRECT:
      /* dims (B, page_num, layer_num, page_size, 1, kv_dim)               [T21] */
      return ((((b * Hp + h) * L + l) * P) + t) * R + e;
    case ORACLE_PAGE_FIRST_DIRECT_KV:
      /* dims (page_num, B, layer_num, page_size, 1, kv_dim)        [B-L2][H-DT] */
      return ((((h * B + b) * L + l) * P) + t) * R + e;
    default:
      return -1;
  }
}

/* Offset, in elements, of element (t, e) of device page d inside the device
 * buffer of (b, l): a layer-first buffer whose rows are token slots.  [T21][B-L2] */
int64_t oracle_dev_elem_offset(int64_t P, int64_t R, int64_t d, int64_t t, int64_t e) {
  return (d * P + t) * R + e;
}

static void copy_elem(uint8_t *dst, const uint8_t *src, int64_t es) {
  int64_t k;
  for (k = 0; k < es; ++k) dst[k] = src[k];
}

static int check_dims(int64_t B, int64_t L, int64_t P, int64_t R, int64_t Hp,
                      int64_t es, int32_t layout) {
  if (B <= 0 || L <= 0 || P <= 0 || R <= 0 || Hp <= 0 || es <= 0) return -1;
  if (layout < ORACLE_LAYER_FIRST || layout > ORACLE_PAGE_FIRST_DIRECT_KV) return -1;
  return 0;
}

/* Backup (L1 -> L2 write-back): for every pair i, every buffer b, every layer l,
 * token t and element e,
 *     host[host_off(b, l, h_i, t, e)] = dev[b][l][dev_off(d_i, t, e)].
 * dev_bufs holds B*L pointers, buffer-major (b*L + l).  Returns 0, or -1 on bad
 * arguments (nothing is written then). */
int oracle_backup(const void *const *dev_bufs, void *host, int64_t B, int64_t L,
                  int64_t P, int64_t R, int64_t Hp, int64_t es,
                  const int64_t *dev_pages, const int64_t *host_pages, int64_t n,
                  int32_t layout) {
  int64_t i, b, l, t, e;
  if (check_dims(B, L, P, R, Hp, es, layout) != 0) return -1;
  for (i = 0; i < n; ++i)
    if (host_pages[i] < 0 || host_pages[i] >= Hp || dev_pages[i] < 0) return -1;
  for (i = 0; i < n; ++i) {
    const int64_t d = dev_pages[i], h = host_pages[i];
    for (b = 0; b < B; ++b)
      for (l = 0; l < L; ++l) {
        const uint8_t *src = (const uint8_t *)dev_bufs[b * L + l];
        for (t = 0; t < P; ++t)
          for (e = 0; e < R; ++e) {
            const int64_t ho = oracle_host_elem_offset(layout, B, L, P, R, Hp, b, l, h, t, e);
            const int64_t dv = oracle_dev_elem_offset(P, R, d, t, e);
            copy_elem((uint8_t *)host + ho * es, src + dv * es, es);
          }
      }
  }
  return 0;
}

/* Load (L2 -> L1): the inverse assignment,
 *     dev[b][l][dev_off(d_i, t, e)] = host[host_off(b, l, h_i, t, e)],
 * over every layer (layer < 0) or over the one layer `layer` (the per-layer load
 * that lets attention on layer l overlap the load of layer l+1). */
int oracle_load(void *const *dev_bufs, const void *host, int64_t B, int64_t L,
                int64_t P, int64_t R, int64_t Hp, int64_t es,
                const int64_t *dev_pages, const int64_t *host_pages, int64_t n,
                int32_t layout, int32_t layer) {
  int64_t i, b, l, t, e, l_begin = 0, l_end = L;
  if (check_dims(B, L, P, R, Hp, es, layout) != 0) return -1;
  if (layer >= L) return -1;
  if (layer >= 0) { l_begin = layer; l_end = layer + 1; }
  for (i = 0; i < n; ++i)
    if (host_pages[i] < 0 || host_pages[i] >= Hp || dev_pages[i] < 0) return -1;
  for (i = 0; i < n; ++i) {
    const int64_t d = dev_pages[i], h = host_pages[i];
    for (b = 0; b < B; ++b)
      for (l = l_begin; l < l_end; ++l) {
        uint8_t *dst = (uint8_t *)dev_bufs[b * L + l];
        for (t = 0; t < P; ++t)
          for (e = 0; e < R; ++e) {
            const int64_t ho = oracle_host_elem_offset(layout, B, L, P, R, Hp, b, l, h, t, e);
            const int64_t dv = oracle_dev_elem_offset(P, R, d, t, e);
            copy_elem(dst + dv * es, (const uint8_t *)host + ho * es, es);
          }
      }
  }
  return 0;
}

/* ---- segment count ------------------------------------------------------
 * A segment is a maximal byte range that is contiguous on BOTH sides of the
 * copy: one DMA descriptor in the pages' terms.  [T21 2.1][B-L2 "DMA Segment
 * Explosion"].  Counted by brute force over token rows: a row (b, l, pair i,
 * token t) is always contiguous on both sides (R elements).  Rows are visited
 * buffer (b, l) by buffer, pairs in ascending (host page, device page) order,
 * tokens ascending -- a fixed order, so that the count depends on the set of
 * pairs and not on the order of the arguments -- and a new segment starts at
 * every row that does not continue the previous one on both the device side
 * (same buffer, next slot) and the host side (next R elements).  layer < 0
 * counts every layer; otherwise only that layer. */

static const int64_t *g_host_keys, *g_dev_keys;  /* qsort has no context argument */
static int cmp_by_host_then_dev(const void *a, const void *b) {
  const int64_t ia = *(const int64_t *)a, ib = *(const int64_t *)b;
  if (g_host_keys[ia] != g_host_keys[ib]) return g_host_keys[ia] < g_host_keys[ib] ? -1 : 1;
  if (g_dev_keys[ia] != g_dev_keys[ib]) return g_dev_keys[ia] < g_dev_keys[ib] ? -1 : 1;
  return (ia > ib) - (ia < ib);
}

int64_t oracle_segment_count(int64_t B, int64_t L, int64_t P, int64_t R, int64_t Hp,
                             const int64_t *dev_pages, const int64_t *host_pages,
                             int64_t n, int32_t layout, int32_t layer) {
  int64_t *order, i, b, l, t, count = 0, l_begin = 0, l_end = L;
  if (check_dims(B, L, P, R, Hp, 1, layout) != 0) return -1;
  if (n <= 0) return 0;
  if (layer >= L) return -1;
  if (layer >= 0) { l_begin = layer; l_end = layer + 1; }
  order = (int64_t *)malloc((size_t)n * sizeof(int64_t));
  if (!order) return -1;
  for (i = 0; i < n; ++i) order[i] = i;
  g_host_keys = host_pages;
  g_dev_keys = dev_pages;
  qsort(order, (size_t)n, sizeof(int64_t), cmp_by_host_then_dev);
  for (b = 0; b < B; ++b)
    for (l = l_begin; l < l_end; ++l) {
      int have_prev = 0;
      int64_t prev_slot = 0, prev_host = 0;
      for (i = 0; i < n; ++i) {
        const int64_t d = dev_pages[order[i]], h = host_pages[order[i]];
        for (t = 0; t < P; ++t) {
          const int64_t slot = d * P + t;
          const int64_t host = oracle_host_elem_offset(layout, B, L, P, R, Hp, b, l, h, t, 0);
          if (!(have_prev && slot == prev_slot + 1 && host == prev_host + R)) ++count;
          have_prev = 1;
          prev_slot = slot;
          prev_host = host;
        }
      }
    }
  free(order);
  return count;
}
