/* A plain C caller of libhicache: a pool on huge-page pinned memory, a backup,
 * per-layer loads into fresh device pages with a compute stream waiting on the
 * layer events, a fused backup + load, a buffer group (a second pool with
 * 32-byte fp32 rows) backed up and then loaded back by one pipelined launch
 * and by a group plan's graph replay, and the error path.  Every element is checked against a position pattern
 * (round trip = identity).  Prints "ok". */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "hicache.h"

#define CHECK(x)                                                                  \
  do {                                                                            \
    int rc_ = (x);                                                                \
    if (rc_ != 0) {                                                               \
      fprintf(stderr, "%s:%d: %s -> %d (%s)\n", __FILE__, __LINE__, #x, rc_,      \
              hicache_last_error());                                              \
      return 1;                                                                   \
    }                                                                             \
  } while (0)

enum { L = 4, B = 2, P = 16, NB = B * L, N = 8 };
static const int64_t R = 128, Hp = 40, Dp = 48;

static uint16_t pattern(int k, int64_t row, int64_t e) {
  return (uint16_t)(k * 7919 + row * 131 + e * 3 + 1);
}

int main(void) {
  const size_t es = 2;
  const size_t host_bytes = (size_t)(B * L * Hp * P * R) * es;
  const size_t buf_bytes = (size_t)(Dp * P * R) * es;
  hicache_pool_desc d;
  memset(&d, 0, sizeof d);
  d.num_layers = L;
  d.num_buffers = B;
  d.page_size = P;
  d.elem_bytes = 2;
  d.row_elems = R;
  d.host_num_pages = Hp;
  d.layout = HICACHE_PAGE_FIRST;
  void *host = NULL;
  CHECK(hicache_host_alloc(host_bytes, HICACHE_HOST_THP, &host));
  hicache_pool *pool = NULL;
  CHECK(hicache_pool_create(&d, host, host_bytes, &pool));

  void *bufs[NB];
  uint16_t *h = (uint16_t *)malloc(buf_bytes);
  for (int k = 0; k < NB; ++k) {
    if (cudaMalloc(&bufs[k], buf_bytes) != cudaSuccess) return 2;
    for (int64_t row = 0; row < Dp * P; ++row)
      for (int64_t e = 0; e < R; ++e) h[row * R + e] = pattern(k, row, e);
    if (cudaMemcpy(bufs[k], h, buf_bytes, cudaMemcpyHostToDevice) != cudaSuccess) return 2;
  }
  hicache_device_kv kv = {bufs, Dp};
  const int64_t src[N] = {3, 4, 5, 17, 30, 31, 9, 40};
  const int64_t hp[N] = {0, 1, 2, 10, 11, 12, 39, 20};
  const int64_t dst[N] = {41, 42, 43, 1, 2, 22, 23, 47};

  cudaStream_t xfer, comp;
  cudaStreamCreateWithFlags(&xfer, cudaStreamNonBlocking);
  cudaStreamCreateWithFlags(&comp, cudaStreamNonBlocking);
  CHECK(hicache_backup(pool, &kv, src, hp, N, HICACHE_LAYOUT_POOL, xfer));
  for (int l = 0; l < L; ++l) {
    CHECK(hicache_load_layer(pool, &kv, dst, hp, N, HICACHE_LAYOUT_POOL, l, xfer));
    CHECK(hicache_wait_layer(pool, l, comp));
  }
  CHECK(hicache_wait(comp, -1));
  CHECK(hicache_wait(xfer, 5 * 1000 * 1000));

  for (int k = 0; k < NB; ++k) {
    if (cudaMemcpy(h, bufs[k], buf_bytes, cudaMemcpyDeviceToHost) != cudaSuccess) return 2;
    for (int i = 0; i < N; ++i)
      for (int64_t t = 0; t < P; ++t)
        for (int64_t e = 0; e < R; ++e) {
          const uint16_t want = pattern(k, src[i] * P + t, e);
          const uint16_t got = h[(dst[i] * P + t) * R + e];
          if (got != want) {
            fprintf(stderr, "buffer %d page %lld token %lld elem %lld: %u != %u\n", k,
                    (long long)dst[i], (long long)t, (long long)e, got, want);
            return 3;
          }
        }
  }

  /* fused: back up pages dst (now copies of src) to new host pages while
   * loading host pages hp into other device pages */
  const int64_t hp2[N] = {30, 31, 32, 33, 34, 35, 36, 37};
  const int64_t dst2[N] = {10, 11, 12, 13, 14, 15, 16, 18};
  CHECK(hicache_backup_load(pool, &kv, dst, hp2, N, dst2, hp, N, HICACHE_LAYOUT_POOL, xfer));
  CHECK(hicache_wait(xfer, -1));
  for (int k = 0; k < NB; ++k) {
    if (cudaMemcpy(h, bufs[k], buf_bytes, cudaMemcpyDeviceToHost) != cudaSuccess) return 2;
    for (int i = 0; i < N; ++i)
      for (int64_t t = 0; t < P; ++t)
        for (int64_t e = 0; e < R; ++e)
          if (h[(dst2[i] * P + t) * R + e] != pattern(k, src[i] * P + t, e)) return 4;
  }

  /* a buffer group: the K,V pool beside a pool of fp32 rows (8 per token) that
   * shares its page numbering; one launch backs up both, one pipelined launch
   * loads both back into other device pages */
  enum { R2 = 8 };
  hicache_pool_desc d2 = d;
  d2.num_buffers = 1;
  d2.elem_bytes = 4;
  d2.row_elems = R2;
  const size_t host2_bytes = (size_t)(L * Hp * P * R2) * 4;
  const size_t buf2_bytes = (size_t)(Dp * P * R2) * 4;
  void *host2 = NULL;
  CHECK(hicache_host_alloc(host2_bytes, 0, &host2));
  hicache_pool *pool2 = NULL;
  CHECK(hicache_pool_create(&d2, host2, host2_bytes, &pool2));
  void *bufs2[L];
  uint32_t *h2 = (uint32_t *)malloc(buf2_bytes);
  for (int l = 0; l < L; ++l) {
    if (cudaMalloc(&bufs2[l], buf2_bytes) != cudaSuccess) return 2;
    for (int64_t row = 0; row < Dp * P; ++row)
      for (int64_t e = 0; e < R2; ++e) h2[row * R2 + e] = 0x9E3779B9u * (uint32_t)(l + 1) + (uint32_t)(row * R2 + e);
    if (cudaMemcpy(bufs2[l], h2, buf2_bytes, cudaMemcpyHostToDevice) != cudaSuccess) return 2;
  }
  hicache_device_kv kv2 = {bufs2, Dp};
  hicache_pool *group[2] = {pool, pool2};
  const hicache_device_kv kvs[2] = {kv, kv2};
  const int64_t hp3[N] = {21, 22, 23, 24, 25, 26, 27, 28};
  const int64_t dst3[N] = {19, 20, 21, 24, 25, 26, 27, 28};
  CHECK(hicache_group_transfer(group, kvs, 2, src, hp3, N, HICACHE_LAYOUT_POOL, -1, HICACHE_DIR_BACKUP, xfer));
  CHECK(hicache_group_load_pipelined(group, kvs, 2, dst3, hp3, N, HICACHE_LAYOUT_POOL, xfer));
  for (int l = 0; l < L; ++l) {
    CHECK(hicache_wait_layer(pool, l, comp));
    CHECK(hicache_wait_layer(pool2, l, comp));
  }
  /* the same host pages once more through a group plan: layer by layer,
   * replayed from one CUDA graph, each layer's event in both pools */
  const int64_t dst4[N] = {0, 1, 2, 6, 7, 8, 10, 11};
  hicache_group_plan *gplan = NULL;
  CHECK(hicache_group_plan_create(group, 2, dst4, hp3, N, Dp, &gplan));
  CHECK(hicache_group_plan_load_layers(gplan, kvs, HICACHE_LAYOUT_POOL, xfer));
  for (int l = 0; l < L; ++l) {
    CHECK(hicache_wait_layer(pool, l, comp));
    CHECK(hicache_wait_layer(pool2, l, comp));
  }
  CHECK(hicache_wait(comp, -1));
  CHECK(hicache_wait(xfer, -1));
  CHECK(hicache_group_plan_destroy(gplan));
  const int64_t *dsts[2] = {dst3, dst4};
  for (int v = 0; v < 2; ++v) {
    for (int k = 0; k < NB; ++k) {
      if (cudaMemcpy(h, bufs[k], buf_bytes, cudaMemcpyDeviceToHost) != cudaSuccess) return 2;
      for (int i = 0; i < N; ++i)
        for (int64_t t = 0; t < P; ++t)
          for (int64_t e = 0; e < R; ++e)
            if (h[(dsts[v][i] * P + t) * R + e] != pattern(k, src[i] * P + t, e)) return 6;
    }
    for (int l = 0; l < L; ++l) {
      if (cudaMemcpy(h2, bufs2[l], buf2_bytes, cudaMemcpyDeviceToHost) != cudaSuccess) return 2;
      for (int i = 0; i < N; ++i)
        for (int64_t t = 0; t < P; ++t)
          for (int64_t e = 0; e < R2; ++e) {
            const uint32_t want = 0x9E3779B9u * (uint32_t)(l + 1) + (uint32_t)((src[i] * P + t) * R2 + e);
            if (h2[(dsts[v][i] * P + t) * R2 + e] != want) return 7;
          }
    }
  }
  CHECK(hicache_pool_destroy(pool2));
  CHECK(hicache_host_free(host2));
  for (int l = 0; l < L; ++l) cudaFree(bufs2[l]);
  free(h2);

  /* the same host pages once more, one chained per-layer call per layer
   * (each layer waited for on the device), then as a one-rank tensor-parallel
   * load, each into other device pages */
  const int64_t dst5[N] = {29, 30, 31, 32, 33, 34, 35, 36};
  const int64_t dst6[N] = {37, 38, 39, 40, 44, 45, 46, 3};
  hicache_plan *plan = NULL;
  CHECK(hicache_plan_create(pool, dst5, hp, N, Dp, HICACHE_DIR_LOAD, &plan));
  for (int l = 0; l < L; ++l) {
    CHECK(hicache_plan_load_layer_chained(plan, &kv, HICACHE_LAYOUT_POOL, l, xfer));
    CHECK(hicache_wait_layer(pool, l, comp));
    void *ev = NULL;                       /* or its CUDA event, recorded on request */
    CHECK(hicache_layer_event(pool, l, &ev));
    if (!ev || cudaStreamWaitEvent(comp, (cudaEvent_t)ev, 0) != cudaSuccess) return 12;
  }
  int64_t first = -1, count = -1;
  CHECK(hicache_tp_share(N, 1, 0, &first, &count));
  if (first != 0 || count != N) return 8;
  void *counters = NULL;
  CHECK(hicache_pool_layer_counters(pool, &counters));
  CHECK(hicache_tp_load_pipelined(pool, &kv, (void *const *)&counters, 1, 0, dst6, hp, N, HICACHE_LAYOUT_POOL,
                                  xfer));
  for (int l = 0; l < L; ++l) CHECK(hicache_wait_layer(pool, l, comp));
  CHECK(hicache_wait(comp, -1));
  CHECK(hicache_wait(xfer, -1));
  CHECK(hicache_plan_destroy(plan));
  const int64_t *dsts2[2] = {dst5, dst6};
  for (int v = 0; v < 2; ++v)
    for (int k = 0; k < NB; ++k) {
      if (cudaMemcpy(h, bufs[k], buf_bytes, cudaMemcpyDeviceToHost) != cudaSuccess) return 2;
      for (int i = 0; i < N; ++i)
        for (int64_t t = 0; t < P; ++t)
          for (int64_t e = 0; e < R; ++e)
            if (h[(dsts2[v][i] * P + t) * R + e] != pattern(k, src[i] * P + t, e)) return 9;
    }

  /* the roofline probe's streaming copy: one device buffer into another */
  CHECK(hicache_stream_copy(bufs[1], bufs[0], buf_bytes, 0, 4, xfer));
  CHECK(hicache_wait(xfer, -1));
  if (cudaMemcpy(h, bufs[1], buf_bytes, cudaMemcpyDeviceToHost) != cudaSuccess) return 2;
  uint16_t *h0 = (uint16_t *)malloc(buf_bytes);
  if (cudaMemcpy(h0, bufs[0], buf_bytes, cudaMemcpyDeviceToHost) != cudaSuccess) return 2;
  if (memcmp(h, h0, buf_bytes) != 0) return 10;
  free(h0);

  /* the plain build reports no failed bounds check (and says it is plain) */
  uint64_t cfirst = 1, ccount = 1;
  CHECK(hicache_check_status(&cfirst, &ccount, 0));
  if (cfirst != 0 || ccount != 0) return 11;

  /* errors enqueue nothing and explain themselves */
  const int64_t bad[1] = {Dp};
  const int64_t okh[1] = {0};
  const int64_t before = hicache_launch_count();
  if (hicache_load(pool, &kv, bad, okh, 1, HICACHE_LAYOUT_POOL, xfer) != HICACHE_ERR_INDEX_RANGE) return 5;
  if (strlen(hicache_last_error()) == 0) return 5;
  if (hicache_launch_count() != before) return 5;

  CHECK(hicache_pool_destroy(pool));
  CHECK(hicache_host_free(host));
  for (int k = 0; k < NB; ++k) cudaFree(bufs[k]);
  free(h);
  printf("ok\n");
  return 0;
}
