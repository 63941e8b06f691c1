/*
 * hicache.h -- C ABI of libhicache: paged KV movement between GPU HBM (L1) and
 * pinned host DRAM (L2) for a tiered prefix-KV cache, on GB300 (sm_103a).
 *
 * The two operations come from the pages' description of HiCache:
 *   - backup (write-back, L1 -> L2): gather every layer of the given device pages
 *     into the given host pages.  "Tuning SGLang HiCache L2 on Kunlunxin
 *     P800/P900", sections 2.1-2.2 (transfer_kv_all_layer, a D2H backup
 *     submitted on its own stream by a backup thread);
 *   - load (L2 -> L1): scatter host pages back into device pages, either all
 *     layers at once or one layer per call (transfer_kv_per_layer) so that
 *     attention on layer i overlaps the load of layer i+1.  Same page, section 2.1;
 *     "HiCache 시스템 설계와 최적화", section "CPU→GPU 전송 최적화" (layer overlap:
 *     layer N computes while layer N+1 loads); "Rethinking the SGLang HiCache
 *     Boundary", section "Why compute, H2D, and D2H should stay in one GPU
 *     execution domain" (an H2D stream, a KV_READY event, the compute stream
 *     waiting on it).
 *
 * Memory layouts.  The device pool is layer-first: for each buffer b (K then V
 * for MHA/GQA; one latent buffer for MLA) and layer l, one caller-owned device
 * allocation of (device_num_pages * page_size) rows of row_elems elements; the
 * row of token t of device page d is row d*page_size + t ("different layers are
 * different buffers", Tuning ... section 2.1).  The host pool is one pinned
 * allocation in one of three layouts, each with a leading buffer dim:
 *   HICACHE_LAYER_FIRST        (B, layer, size, kv_dim)               [Tuning ... 2.1]
 *   HICACHE_PAGE_FIRST         (B, size, layer, kv_dim)               [HiCache 설계, 데이터 전송 최적화]
 *   HICACHE_PAGE_FIRST_DIRECT  (B, page_num, layer_num, page_size, kv_dim) [Tuning ... 2.1]
 * and one L3-ready variant without the leading buffer dim:
 *   HICACHE_PAGE_FIRST_DIRECT_KV (page_num, B, layer_num, page_size, kv_dim): all KV of
 *   a page -- K and V, every layer -- in one block, the single object per page that
 *   L3 wants ("Baidu's KVCache Overhaul", sections "L2 Layout Choice" and "DMA
 *   Segment Explosion & Batched Gather/Scatter"; "HiCache 시스템 설계와 최적화",
 *   section "데이터 전송 최적화": a page's KV contiguous and handed to L3 zero-copy)
 * where size = host_num_pages * page_size.  Indices are page indices (int64);
 * the i-th device page pairs with the i-th host page.  Bytes are copied as-is:
 * no dtype conversion, elem_bytes only sizes the rows.
 *
 * Conventions for every call below.
 *   - Streams and events are CUDA handles (cudaStream_t / cudaEvent_t) passed
 *     as void*; NULL is the legacy default stream.
 *   - Index arrays are HOST memory, read during the call only: the caller may
 *     free or reuse them as soon as the call returns.
 *   - Transfers only enqueue work on the given stream and return; ordering
 *     against the caller's compute is the caller's (record an event before a
 *     backup; use hicache_wait_layer for loads).
 *   - Every argument is validated BEFORE anything is enqueued: a call that
 *     returns a validation error has enqueued nothing.  (A CUDA error while
 *     launching the second or later launch of a call split over several
 *     launches leaves the earlier ones enqueued.)  n == 0 is valid and launches
 *     no kernel (hicache_load_layer still records its layer event).
 *   - The validation of a call of 49,152 pairs or more is split over up to
 *     four host threads: the caller's and up to three worker threads of the
 *     library, started on its first such call in each process, asleep between
 *     calls and never ended before the process ends (the library is therefore
 *     never unloaded: dlclose leaves it mapped).  A call made while another
 *     thread's call holds them validates on the calling thread alone.  The
 *     environment variable HICACHE_VALIDATE_THREADS, read once, caps the
 *     threads (1: the calling thread only).  Results and error reports are
 *     the same either way.
 *   - Transfers must be called with the pool's device current.
 *   - Return value: HICACHE_OK (0) or a negative hicache_status; the text of
 *     the last error of the calling thread is in hicache_last_error().
 *   - Thread safety: a pool may be used from several host threads at once
 *     (e.g. a backup thread and a load thread), each on its own stream.
 *   - Launches overlap where they can.  A call split over several launches
 *     (more page runs than one launch's parameters hold) and the layers of a
 *     per-layer graph replay start each launch as the one before it drains;
 *     the call still completes, for whatever follows it on the stream, only
 *     once every launch of it has.  A one-layer load is launched early behind
 *     the work before it and waits for that work before touching memory.  A kernel of the caller's that is launched
 *     programmatically (programmatic stream serialization) right behind a
 *     transfer may likewise start while the transfer's last tiles move: as
 *     for any programmatic launch, it must call cudaGridDependencySynchronize
 *     before it reads what the transfer wrote.
 */
#ifndef HICACHE_H_
#define HICACHE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  HICACHE_OK = 0,
  HICACHE_ERR_INVALID_ARG = -1,     /* null pointer, bad size, bad layout/layer/direction */
  HICACHE_ERR_INDEX_RANGE = -2,     /* a page index outside its pool */
  HICACHE_ERR_DUPLICATE_INDEX = -3, /* a destination page named twice in one call */
  HICACHE_ERR_ALIGNMENT = -4,       /* pointer or row size not a multiple of 16 bytes */
  HICACHE_ERR_NOT_PINNED = -5,      /* host pool not page-locked / not device-mapped */
  HICACHE_ERR_CUDA = -6,            /* a CUDA runtime call failed (text in last_error) */
  HICACHE_ERR_TIMEOUT = -7,         /* hicache_wait ran out of time */
  HICACHE_ERR_NOMEM = -8            /* host allocation failed */
} hicache_status;

typedef enum {
  HICACHE_LAYOUT_POOL = -1,         /* the pool's own layout (desc.layout) */
  HICACHE_LAYER_FIRST = 0,
  HICACHE_PAGE_FIRST = 1,
  HICACHE_PAGE_FIRST_DIRECT = 2,
  HICACHE_PAGE_FIRST_DIRECT_KV = 3  /* page_first_direct with the buffer dim inside the page */
} hicache_layout;

typedef enum {
  HICACHE_DIR_BACKUP = 0,           /* device -> host (L1 -> L2) */
  HICACHE_DIR_LOAD = 1              /* host -> device (L2 -> L1) */
} hicache_direction;

/* Host allocation flags for hicache_host_alloc. */
#define HICACHE_HOST_THP 0x1        /* anonymous mmap + madvise(MADV_HUGEPAGE) before
                                       page-locking ("Tuning ... section 2.4": huge pages
                                       cut translation entries ~512x; madvise must come
                                       before registration) */

typedef struct {
  int32_t num_layers;       /* L >= 1 */
  int32_t num_buffers;      /* B: 2 = K,V (MHA/GQA), 1 = MLA latent; B*L <= 512 */
  int32_t page_size;        /* P >= 1 tokens per page */
  int32_t elem_bytes;       /* bytes per element (2 for bf16) */
  int64_t row_elems;        /* R: kv_heads*head_dim, or kv_dim (e.g. 576) */
  int64_t host_num_pages;   /* Hp: pages in the host pool */
  int32_t layout;           /* hicache_layout of the host pool (not POOL) */
  int32_t launch_ctas;      /* CTAs of a transfer launch (a fused backup+load
                               gets twice as many); 0 = the defaults: one per
                               SM for a load of every layer, one per two SMs
                               for a per-layer or pipelined load, five per
                               eight SMs for a backup, two per SM for a fused
                               backup+load */
  int32_t flags;            /* must be 0 */
  int32_t reserved;         /* must be 0 */
} hicache_pool_desc;

/* Borrowed device KV, passed to each call.  buf_ptrs: host array of B*L device
 * pointers, buffer-major (K layer 0..L-1, then V layer 0..L-1); each points to
 * device_num_pages*page_size rows of row_elems elements, contiguous, 16-byte
 * aligned.  The library does not keep the pointers after the call returns. */
typedef struct {
  void *const *buf_ptrs;
  int64_t device_num_pages;
} hicache_device_kv;

typedef struct hicache_pool hicache_pool; /* opaque */
typedef struct hicache_plan hicache_plan; /* opaque: a validated, pre-passed index set */

/* ---- version / diagnostics ------------------------------------------------ */

/* Library version as 10000*major + 100*minor + patch. */
int32_t hicache_version(void);

/* Text of the calling thread's most recent error ("" if none).  The pointer
 * stays valid until the thread's next hicache call. */
const char *hicache_last_error(void);

/* Number of kernels the library has launched in this process (all threads). */
int64_t hicache_launch_count(void);

/* ---- pinned host memory --------------------------------------------------- */

/* Allocate `bytes` of page-locked host memory that the current device can
 * address, for use as a host pool.  flags: HICACHE_HOST_THP or 0 (plain
 * cudaHostAlloc).  *out receives the host pointer; free with hicache_host_free.
 * Errors: INVALID_ARG (bytes == 0, out NULL), NOMEM, CUDA. */
int hicache_host_alloc(size_t bytes, int32_t flags, void **out);
int hicache_host_free(void *ptr);

/* ---- pool ----------------------------------------------------------------- */

/* Create a pool over a caller-owned pinned host buffer of host_bytes bytes
 * (borrowed: it must outlive the pool).  The buffer must be page-locked and
 * mapped for the current device (hicache_host_alloc, cudaHostAlloc, or a
 * torch pin_memory tensor), 16-byte aligned, and at least
 * B*L*host_num_pages*page_size*row_elems*elem_bytes bytes.  The pool binds to
 * the current device and creates one CUDA event per layer (timing disabled).
 * Errors: INVALID_ARG, ALIGNMENT (row bytes or pointer not 16-byte multiples),
 * NOT_PINNED, CUDA. */
int hicache_pool_create(const hicache_pool_desc *desc, void *host_pool, size_t host_bytes,
                        hicache_pool **out);
/* Destroys the pool's events and the pool.  Transfers already enqueued still
 * run; the host buffer must stay allocated until they finish.  The pool's
 * pipelined, tensor-parallel and chained per-layer loads count into device
 * words the pool owns, so this first waits on the host for the last of them to
 * finish (for a chain of per-layer calls left before its last layer, for the
 * whole device).  In a tensor-parallel group the other ranks' loads count into
 * this pool too: every rank's pool must outlive the group's loads.  Plans and
 * engines of the pool
 * must be destroyed first, and no other thread may be inside a call on the
 * pool meanwhile. */
int hicache_pool_destroy(hicache_pool *pool);

/* ---- transfers -------------------------------------------------------------
 * device_pages / host_pages: n page indices each (host memory).  Validation:
 * 0 <= device_pages[i] < kv->device_num_pages, 0 <= host_pages[i] <
 * host_num_pages (INDEX_RANGE); a backup may not name a host page twice and a
 * load may not name a device page twice (DUPLICATE_INDEX: the result would
 * depend on execution order); a source page may repeat.
 * Each call enqueues ceil(runs / ((3584 - B*L) / 2)) kernel launches, at most
 * ceil(runs / 1536), where runs is the number of maximal page runs contiguous
 * on both sides (a run is also cut before its pages, counting every buffer
 * and layer, reach 32 GiB); calls of up to 1536 pages are exactly one launch. */

/* L1 -> L2: every layer and buffer of the given device pages into the given
 * host pages. */
int hicache_backup(hicache_pool *pool, const hicache_device_kv *kv, const int64_t *device_pages,
                   const int64_t *host_pages, int64_t n, int32_t layout, void *stream);

/* L2 -> L1: every layer and buffer of the given host pages into the given
 * device pages. */
int hicache_load(hicache_pool *pool, const hicache_device_kv *kv, const int64_t *device_pages,
                 const int64_t *host_pages, int64_t n, int32_t layout, void *stream);

/* L2 -> L1 for one layer (every buffer of layer_id), then records the pool's
 * event for that layer on `stream`.  To load every layer of one set of pages
 * this way, a plan's hicache_plan_load_layers does the same with one graph
 * launch and overlaps consecutive layers (about 209 against 184 GB/s for
 * 4K-token MLA loads on GB300).  The load is launched programmatically: it
 * waits for the work before it on the stream before touching memory, and
 * only its launch overlaps that work's end. */
int hicache_load_layer(hicache_pool *pool, const hicache_device_kv *kv,
                       const int64_t *device_pages, const int64_t *host_pages, int64_t n,
                       int32_t layout, int32_t layer_id, void *stream);

/* Both directions in one launch: a backup of n_backup pages and a load of
 * n_load pages, every layer.  Every CTA alternates a backup tile and a load
 * tile, so both directions of the host link stay busy until both finish (two
 * launches on two streams let one direction finish early and the other run
 * alone).  The concurrent backup of one request and load of another is the
 * pages' bidirectional transfer ("Tuning ... section 2.1": layer_first +
 * bidirectional async; "Baidu's KVCache Overhaul", section "Bidirectional
 * Async Transfer"), here fused into one submission.  Validation is that of
 * hicache_backup for the first set and hicache_load for the second, plus:
 * no device page may be both read by the backup and written by the load, and
 * no host page both written by the backup and read by the load (INVALID_ARG),
 * so the result does not depend on how the two interleave.  Either count may
 * be 0 (then this is a plain backup or load). */
int hicache_backup_load(hicache_pool *pool, const hicache_device_kv *kv,
                        const int64_t *backup_device_pages, const int64_t *backup_host_pages,
                        int64_t n_backup, const int64_t *load_device_pages,
                        const int64_t *load_host_pages, int64_t n_load, int32_t layout,
                        void *stream);

/* L2 -> L1, every layer in ONE launch that moves the layers in order and marks
 * each layer done on the device as it lands: after this call,
 * hicache_wait_layer(pool, l, stream) makes `stream` wait for layer l alone
 * (a stream memory wait on a per-layer counter, cuStreamWaitValue32), so
 * attention on layer l can start while later layers still load -- the
 * per-layer overlap of "HiCache 시스템 설계와 최적화", section "CPU→GPU 전송
 * 최적화", without a launch and an event per layer (hicache_layer_event
 * gives a layer's event when asked for).  Checks as hicache_load.  A
 * pipelined load may only go on another stream than the pool's previous one
 * once that one's counted loads (pipelined, tensor-parallel, chained per-layer)
 * have finished (INVALID_ARG otherwise): the per-layer counts must rise in
 * load order.  A stream that is being captured
 * into a CUDA graph is refused (INVALID_ARG, nothing enqueued): the value each
 * layer's counter must reach is raised on the host when the call is enqueued,
 * so a graph replayed twice, or never, would leave hicache_wait_layer passing
 * early or waiting forever.  If a call split over several launches fails on a
 * launch after the first, the launches before it stay enqueued and
 * hicache_wait_layer waits for them.  CUDA if the driver offers no stream
 * memory wait. */
int hicache_load_pipelined(hicache_pool *pool, const hicache_device_kv *kv,
                           const int64_t *device_pages, const int64_t *host_pages, int64_t n,
                           int32_t layout, void *stream);

/* Diagnostic: the value of layer `layer`'s counter now (*done; reads device
 * memory, synchronously on the legacy stream) and the value the pipelined loads
 * enqueued so far will bring it to (*target). */
int hicache_pipeline_status(hicache_pool *pool, int32_t layer, uint32_t *done, uint32_t *target);

/* ---- plans: pre-pass once, execute many times -------------------------------
 * A plan holds the validated, sorted, run-merged index set of one transfer, so
 * that the L per-layer loads of one request pay for validation and the pre-pass
 * once (the prepare-ahead idea of "Rethinking the SGLang HiCache Boundary",
 * section "PrepareBatch / ExecuteBatch").  device_num_pages bounds the device
 * indices.  A plan is immutable and may be executed from several threads; it
 * refers to its pool, so it must be destroyed before the pool. */
int hicache_plan_create(hicache_pool *pool, const int64_t *device_pages, const int64_t *host_pages,
                        int64_t n, int64_t device_num_pages, int32_t direction,
                        hicache_plan **out);
/* Execute a plan: every layer (layer_id < 0) or one layer (a load plan only;
 * records that layer's event).  kv->device_num_pages must be >= the plan's. */
int hicache_plan_execute(const hicache_plan *plan, const hicache_device_kv *kv, int32_t layout,
                         int32_t layer_id, void *stream);
/* Load one layer of a load plan and record that layer's event: the per-layer
 * load of the pages ("Why compute, H2D, and D2H should stay in one GPU
 * execution domain"), with the index pre-pass done once at plan creation.
 * Same as hicache_plan_execute with layer_id >= 0, except that a negative
 * layer_id is INVALID_ARG here.  Errors: INVALID_ARG (NULL plan, backup plan,
 * layer_id outside [0, num_layers), bad layout or kv), CUDA; on error nothing
 * is enqueued. */
int hicache_plan_load_layer(const hicache_plan *plan, const hicache_device_kv *kv, int32_t layout,
                            int32_t layer_id, void *stream);
/* One layer of a load plan, as hicache_plan_load_layer, chained to the plan's
 * previous layer: the per-layer load of "Why compute, H2D, and D2H should stay
 * in one GPU execution domain" ("Rethinking the SGLang HiCache Boundary"),
 * one call per layer as the layers are needed, without the gap between
 * per-layer kernels.  A call for layer l continues a chain when the plan's
 * previous chained call loaded layer l - 1 on the same stream; its kernel is
 * then a programmatic dependent launch that starts moving data while layer
 * l - 1's kernel drains its last tiles.  The caller guarantees that nothing
 * else is enqueued on that stream between the calls of a chain (compute goes
 * on another stream); any other call -- layer 0, a layer out of order,
 * another stream -- waits for all earlier work on the stream like a plain
 * call.  Layers overlap, so no two device buffers may share bytes (checked
 * once per set of buffers: INVALID_ARG).
 *   - Each layer is signalled on the device, not by an event recorded between
 *     kernels (which would stop them overlapping): every CTA counts itself into
 *     the layer's pool counter once its tiles have landed, and
 *     hicache_wait_layer(pool, l, stream) waits for that count, and
 *     hicache_layer_event(pool, l) gives an event that fires once it is in.
 *   - A capturing stream is refused (INVALID_ARG): the count each layer must
 *     reach is raised on the host when the call is enqueued.
 *   - Calls of one plan's chain come from one thread, in layer order.
 *   - Consecutive layers overlap only if the call for layer l + 1 arrives
 *     before layer l's kernel has ended; a caller that does per-layer host
 *     work between the calls (e.g. enqueueing attention) may lose that, and
 *     is better served by hicache_plan_load_layers or
 *     hicache_plan_load_pipelined, which enqueue every layer at once.
 *   - The pool's counters are shared with its pipelined and tensor-parallel
 *     loads, and counts from two loads cannot be told apart: all of them go
 *     on one stream, or on another only once the earlier ones have finished.
 *     A chain stopped before its last layer counts as unfinished (it has no
 *     event behind it): a counted load on another stream is then refused
 *     (INVALID_ARG) until a counted load on the chain's stream closes it.
 * Errors: INVALID_ARG (NULL plan, backup plan, layer_id outside [0,
 * num_layers), bad layout or kv, overlapping buffers, capturing stream,
 * another stream while a counted load is unfinished), CUDA; on a refused
 * call nothing is enqueued. */
int hicache_plan_load_layer_chained(hicache_plan *plan, const hicache_device_kv *kv, int32_t layout,
                                    int32_t layer_id, void *stream);
/* hicache_load_pipelined without any allocation.  The pages have no
 * counterpart to this entry point: it serves callers that cannot allocate
 * device memory when they load -- for example an engine whose device memory is
 * all handed out by its own allocator, or a code path that must not call
 * cudaMalloc.  hicache_load_pipelined keeps its per-layer counters in memory
 * the pool allocated; this one keeps them in a fixed array inside the library
 * (256 layers at most; 1.5 KiB with the kernel's tile-scheduling words, which
 * calls take in turn from 64 pairs), which every GPU that loads the library holds
 * until the process exits, so the call itself allocates nothing: no cudaMalloc,
 * no cudaFree, no allocating library routine.  Inputs and outputs are the
 * caller's, as for hicache_load_pipelined, and hicache_wait_layer waits for
 * each layer the same way.
 *   - More than 256 layers: INVALID_ARG, nothing enqueued.
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *     A capturing stream is refused, as for hicache_load_pipelined.
 *   - The address and the counts belong to the device's context: after a
 *     cudaDeviceReset in the same process the counts start again from zero
 *     while the library's targets keep their values, so do not use this entry
 *     point on a device after resetting it.
 *   - Every call on a device shares the array and leaves its counts there;
 *     the library tracks the values they reach, so nothing needs clearing
 *     between calls.  Calls whose loads overlap on the GPU (e.g. on two
 *     streams at once, from any pool) race on the counts: issue them one
 *     after another.
 * Other errors as hicache_load_pipelined. */
int hicache_load_pipelined_noalloc(hicache_pool *pool, const hicache_device_kv *kv,
                                   const int64_t *device_pages, const int64_t *host_pages, int64_t n,
                                   int32_t layout, void *stream);
/* hicache_load_pipelined for a load plan. */
int hicache_plan_load_pipelined(const hicache_plan *plan, const hicache_device_kv *kv, int32_t layout,
                                void *stream);
/* Every layer of a load plan, layer by layer, as hicache_plan_load_layer for
 * l = 0..L-1 (L per-layer launches, each followed by that layer's event), from
 * one CUDA graph: the first call for a given device KV and layout captures the
 * launches and event records into a graph that the plan keeps, and every call
 * replays it with one graph launch.  This cuts the host's per-layer launch cost
 * and the gaps between the per-layer kernels (the per-layer load of "Why
 * compute, H2D, and D2H should stay in one GPU execution domain", "Rethinking
 * the SGLang HiCache Boundary"): each layer's kernel after the first is a
 * programmatic dependent launch that may start while the previous layer's
 * kernel moves its last tiles, so no two device buffers may overlap (as for
 * every all-layer call; checked here).  The event of layer l fires once layers
 * 0..l have all landed.  A call with other buffer pointers, page count or
 * layout re-captures.  Errors: INVALID_ARG (NULL plan, backup plan, bad layout
 * or kv, overlapping buffers), CUDA; on error nothing is enqueued.  Destroying the plan
 * while a replay is still running is allowed: CUDA frees the graph once the
 * replay ends. */
int hicache_plan_load_layers(hicache_plan *plan, const hicache_device_kv *kv, int32_t layout, void *stream);
/* Number of pages and of merged runs in a plan. */
int hicache_plan_info(const hicache_plan *plan, int64_t *num_pages, int64_t *num_runs);
int hicache_plan_destroy(hicache_plan *plan);

/* ---- buffer groups: several buffer kinds, one launch -------------------------
 * Models whose layers keep more than one kind of KV row hold one pool per
 * kind, each with its own row size and element size: the MLA and NSA models
 * of "Tuning SGLang HiCache L2 on Kunlunxin P800/P900" (section 2.7) and the
 * MLA-class CSA/HCA caches of "Baidu's KVCache Overhaul" (section
 * "Optimization Techniques"), e.g. a 576-element bf16 latent beside a
 * sparse-attention indexer key of 128 fp8 and its fp32 scales.  Those pools share the page
 * numbering: page p of the request is page p in every pool.  This call moves
 * the same page pairs for all of them in ONE kernel launch (the run table is
 * worked out once; every pool gets its own tile range and shape constants),
 * where separate calls would launch once per pool.
 *   pools[i], kvs[i]: pool i and its device buffers, i < npools, 1 <= npools
 *     <= HICACHE_MAX_GROUP.  All pools on one device, with equal num_layers
 *     and page_size and the same resolved layout; the sum of B*L over the
 *     pools <= 512.
 *   device_pages / host_pages / n: as hicache_backup and hicache_load; every
 *     index must be inside every pool (and every kvs[i]).
 *   direction: HICACHE_DIR_BACKUP or HICACHE_DIR_LOAD.
 *   layer_id: < 0 moves every layer; >= 0 moves that layer only (a load only)
 *     and records that layer's event in every pool, as hicache_load_layer.
 * Errors as hicache_backup / hicache_load, plus INVALID_ARG for a mismatch
 * between the pools; on error nothing is enqueued.  A call whose run table
 * does not fit one launch is split into several, as the single-pool calls. */
#define HICACHE_MAX_GROUP 4
int hicache_group_transfer(hicache_pool *const *pools, const hicache_device_kv *kvs, int32_t npools,
                           const int64_t *device_pages, const int64_t *host_pages, int64_t n,
                           int32_t layout, int32_t layer_id, int32_t direction, void *stream);

/* hicache_load_pipelined for a buffer group: every layer of every pool in ONE
 * launch, layer by layer (all pools' tiles of layer l before any of layer
 * l + 1), each pool's layers marked done on the device as they land, so that
 * hicache_wait_layer(pools[i], l, stream) waits for pool i's layer l alone.
 * Arguments and checks as hicache_group_transfer with a load of every layer;
 * every pool follows the stream rule of hicache_load_pipelined (INVALID_ARG
 * while one of them has a pipelined load still running on another stream);
 * CUDA if the driver offers no stream memory wait. */
int hicache_group_load_pipelined(hicache_pool *const *pools, const hicache_device_kv *kvs, int32_t npools,
                                 const int64_t *device_pages, const int64_t *host_pages, int64_t n,
                                 int32_t layout, void *stream);

/* A load plan for a buffer group: the page pairs validated and reduced to runs
 * once, as hicache_plan_create, for pools that share the page numbering; then
 * loaded many times, every layer at once or layer by layer.
 *   pools / npools: as hicache_group_transfer (1..HICACHE_MAX_GROUP distinct
 *     pools on one device with equal num_layers and page_size).  The plan keeps
 *     the pool pointers: the pools must outlive it.
 *   device_pages / host_pages / n / device_num_pages: as hicache_plan_create
 *     with HICACHE_DIR_LOAD; every host page must be inside every pool.
 * Errors: INVALID_ARG (bad pools or sizes, NULL out), INDEX_RANGE,
 * DUPLICATE_INDEX (a device page twice), NOMEM. */
typedef struct hicache_group_plan hicache_group_plan;
int hicache_group_plan_create(hicache_pool *const *pools, int32_t npools, const int64_t *device_pages,
                              const int64_t *host_pages, int64_t n, int64_t device_num_pages,
                              hicache_group_plan **out);
/* hicache_group_transfer (a load) of a group plan: every layer (layer_id < 0)
 * in one launch, or one layer, recording that layer's event in every pool.
 * kvs[i] belongs to the plan's pool i and holds at least the plan's
 * device_num_pages.  Errors as hicache_group_transfer. */
int hicache_group_plan_execute(const hicache_group_plan *plan, const hicache_device_kv *kvs, int32_t layout,
                               int32_t layer_id, void *stream);
/* hicache_plan_load_layers for a buffer group: every layer, layer by layer,
 * one group launch per layer followed by that layer's event in every pool,
 * captured into a CUDA graph on the first call for a set of device buffers and
 * a layout and replayed with one graph launch afterwards.  As for a single
 * pool, each layer's launch may start while the previous one drains, so no two
 * device buffers of the group may overlap (checked); the event of layer l in
 * any pool fires once layers 0..l of every pool have landed.  Errors as
 * hicache_group_plan_execute, plus INVALID_ARG for overlapping buffers and
 * CUDA; on error nothing is enqueued.  Destroying the plan while a replay runs
 * is allowed. */
int hicache_group_plan_load_layers(hicache_group_plan *plan, const hicache_device_kv *kvs, int32_t layout,
                                   void *stream);
/* hicache_plan_load_layer_chained for a buffer group: one group launch for
 * layer layer_id of every pool, chained to the plan's previous chained call
 * when that loaded layer_id - 1 on the same stream (nothing else enqueued on
 * the stream in between), and every CTA counted into each pool's counter of
 * the layer, so hicache_wait_layer on any pool of the group waits for that
 * pool's layer on the device (and hicache_layer_event gives an event that
 * fires once that count is in).  No two device buffers of the group may
 * overlap; a capturing stream is refused.  Errors as
 * hicache_group_plan_execute, plus INVALID_ARG for layer_id outside [0,
 * num_layers), overlapping buffers or a capturing stream; on a refused call
 * nothing is enqueued. */
int hicache_group_plan_load_layer_chained(hicache_group_plan *plan, const hicache_device_kv *kvs,
                                          int32_t layout, int32_t layer_id, void *stream);
int hicache_group_plan_destroy(hicache_group_plan *plan);

/* ---- per-layer events (KV_READY) ---------------------------------------------- */

/* The last load of a layer, for this call and hicache_wait_layer, is the last
 * call enqueued before it that loaded the layer: one layer or every layer
 * (hicache_load, hicache_backup_load, a plan's or a group's load of every
 * layer), n > 0.  Loads queued through the submission engine are not among
 * them (wait for those through the engine), nor is a load of every layer
 * captured into a CUDA graph.
 *
 * The pool-owned event of the last load of `layer` (*event_out is a
 * cudaEvent_t; do not destroy it): it fires once that load has moved the
 * layer.  Where that load is signalled on the device (pipelined,
 * allocation-free pipelined, tensor-parallel and chained per-layer loads),
 * this call records the event, on a stream of the pool's own that waits for
 * the load's count of the layer; the pool's device must be current.  After a
 * load of every layer it is the pool's event recorded behind that load (one
 * event for all layers); otherwise the event the load recorded on its stream.
 * Errors: INVALID_ARG, CUDA. */
int hicache_layer_event(hicache_pool *pool, int32_t layer, void **event_out);
/* Make `compute_stream` wait (on the device; the host does not block) for the
 * last load of `layer` enqueued before this call: its layer event (the whole
 * load's, for a load of every layer), or, if that load is signalled on the
 * device (pipelined, allocation-free pipelined, tensor-parallel, chained
 * per-layer), that layer's count: the wait for the count goes on the pool's
 * own stream, and compute_stream waits for the event recorded behind it (as
 * hicache_layer_event), so that the kernel enqueued next on compute_stream
 * does not start late behind a stream memory wait.  A compute stream that is
 * being captured waits for the count itself (cuStreamWaitValue32).  For a
 * load signalled on the device the pool's device must be current. */
int hicache_wait_layer(hicache_pool *pool, int32_t layer, void *compute_stream);

/* Block the calling host thread until all work on `stream` is done, for at
 * most timeout_us microseconds (< 0 = no limit).  Polls back to back for the
 * first 500 us, then every 50 us.  Returns OK, TIMEOUT (work still pending;
 * nothing is cancelled) or CUDA. */
int hicache_wait(void *stream, int64_t timeout_us);

/* ---- host-only helpers (no CUDA call; usable without a GPU) ------------------ */

/* Validate a transfer and run the pre-pass without a pool: the checks that a
 * transfer call makes on its indices.  direction: hicache_direction.  On OK,
 * *num_runs receives the number of maximal runs (pairs sorted by host page,
 * merged while device and host page both step by one), and if runs_out is not
 * NULL and runs_capacity >= *num_runs, runs_out receives 3 int64 per run:
 * first host page, first device page, page count. */
int hicache_prepass(int64_t host_num_pages, int64_t device_num_pages, const int64_t *device_pages,
                    const int64_t *host_pages, int64_t n, int32_t direction, int64_t *num_runs,
                    int64_t *runs_out, int64_t runs_capacity);

/* Number of byte ranges contiguous on both sides that the transfer consists of
 * (the DMA-descriptor count of a copy engine; "Tuning ... section 2.1": 39,936
 * for page_first_direct vs 78 for layer_first at 512 pages x 78 layers, per
 * buffer), for every layer (layer_id < 0) or one layer.  Returns the count, or
 * a negative hicache_status. */
int64_t hicache_segment_count(const hicache_pool_desc *desc, const int64_t *device_pages,
                              const int64_t *host_pages, int64_t n, int32_t layout,
                              int32_t layer_id);

/* Byte range of one host page inside the host pool, for handing a page to L3
 * storage without a copy (the pages' zero-copy L2 -> L3 path: "HiCache 시스템 설계와
 * 최적화", section "데이터 전송 최적화" -- memory address and size passed directly).
 * page_first / page_first_direct: the page of buffer `buffer` (0..B-1; -1 allowed
 * when B == 1).  page_first_direct_kv: buffer -1 = the whole page, every buffer;
 * 0..B-1 = that buffer's part.  layer_first keeps a page in L separate spans
 * (INVALID_ARG), unless the pool has one layer.  Host-only: no CUDA call.
 * Errors: INVALID_ARG, INDEX_RANGE. */
int hicache_page_span(const hicache_pool_desc *desc, int64_t host_page, int32_t buffer,
                      int64_t *offset_bytes, int64_t *nbytes);

/* ---- submission engine ---------------------------------------------------------
 * Callers queue backups and loads (every layer); one worker thread launches
 * them in submission order on the engine's own stream.  This is the pages'
 * pair of submitter threads with request queues ("Tuning ... section 2.2";
 * "Baidu's KVCache Overhaul", section "Bidirectional Async Transfer"), with one
 * change for GB300: when the request at the head of the queue and the first
 * request of the other direction among the next 8 use the same device buffers
 * and commute (neither writes a page the other touches, nor one touched by the
 * requests the second would move ahead of), the worker sends them as one fused
 * launch (hicache_backup_load), which keeps both directions of the host link busy.
 * The result is always that of running the requests one by one in submission
 * order.  Validation and the pre-pass run in the submitting thread; a refused
 * request is never queued.  An engine must be destroyed before its pool. */
typedef struct hicache_engine hicache_engine; /* opaque */
/* Starts the worker thread and creates the engine's stream on the pool's device. */
int hicache_engine_create(hicache_pool *pool, hicache_engine **out);
/* Launches whatever is still queued, waits for the engine's stream, stops the
 * worker and frees the engine.  No other thread may be inside a call on the
 * engine (submit, wait, wait_on_stream, stats) meanwhile or afterwards. */
int hicache_engine_destroy(hicache_engine *engine);
/* Queue a backup (direction HICACHE_DIR_BACKUP) or load of every layer of n
 * pages, with the checks of hicache_backup / hicache_load.  If
 * after_stream_valid is non-zero, the transfer starts only after the work
 * already enqueued on after_stream (e.g. the compute that wrote the KV a
 * backup reads); the dependency is recorded on after_stream during this call.
 * kv's buffer table is copied.  *ticket receives the request's id (a request
 * paired ahead of earlier ones may finish before them).  After a launch failure
 * the engine refuses new requests (CUDA).  hicache_wait_layer and
 * hicache_layer_event do not see queued loads: wait for them through the
 * engine. */
int hicache_engine_submit(hicache_engine *engine, const hicache_device_kv *kv,
                          const int64_t *device_pages, const int64_t *host_pages, int64_t n,
                          int32_t direction, int32_t layout, int32_t after_stream_valid,
                          void *after_stream, uint64_t *ticket);
/* Block until the transfer of `ticket` has finished on the GPU, for at most
 * timeout_us (< 0: no limit).  Returns OK, TIMEOUT, INVALID_ARG (unknown
 * ticket) or the engine's launch error. */
int hicache_engine_wait(hicache_engine *engine, uint64_t ticket, int64_t timeout_us);
/* Make `stream` wait on the device for the transfer of `ticket` (e.g. compute
 * that reads loaded KV).  Blocks the host only until the worker has launched
 * the ticket. */
int hicache_engine_wait_on_stream(hicache_engine *engine, uint64_t ticket, void *stream);
/* Launches made so far, and how many of them carried a backup and a load. */
int hicache_engine_stats(hicache_engine *engine, int64_t *launches, int64_t *fused_launches);

/* ---- host-page allocator (LIFO free list of page runs) ------------------------
 * Hands out host pages of an L2 pool.  "Tuning ... section 2.4" and "Baidu's
 * KVCache Overhaul", section "LIFO slot allocation": the most recently freed
 * pages are handed out first, so writes stay on a small set of hot pages.  The
 * free list is a stack of runs; alloc takes pages from the front of the top
 * runs (ascending, as few runs as possible); free pushes the freed pages,
 * merged into runs, on top.  Host-only, thread-safe.  Every error leaves the
 * allocator unchanged. */
typedef struct hicache_page_allocator hicache_page_allocator; /* opaque */
/* num_pages in [1, 2^31).  Errors: INVALID_ARG, NOMEM. */
int hicache_allocator_create(int64_t num_pages, hicache_page_allocator **out);
int hicache_allocator_destroy(hicache_page_allocator *alloc);
/* Writes n page indices to pages_out.  NOMEM if fewer than n pages are free. */
int hicache_allocator_alloc(hicache_page_allocator *alloc, int64_t n, int64_t *pages_out);
/* Returns n pages.  INDEX_RANGE for a page outside the pool, DUPLICATE_INDEX
 * for a page named twice or not currently handed out. */
int hicache_allocator_free(hicache_page_allocator *alloc, const int64_t *pages, int64_t n);
/* Free pages, or a negative hicache_status. */
int64_t hicache_allocator_available(hicache_page_allocator *alloc);

/* ---- measurement helper ------------------------------------------------------ */

/* A stand-in for attention on one layer: reads the given pages of every buffer
 * of `layer` `reps` times and adds every 32-bit word it reads into *out_sum_dev
 * (a device uint64, mod 2^64; reps times the one-pass sum).  Used to show that a
 * compute stream that waited on a layer event sees that layer loaded, and to
 * measure compute/transfer overlap.  desc gives the shape (its host_num_pages
 * and layout are not used); device_pages are host memory, n <= any size (one
 * launch per 6144 pages).  Errors: INVALID_ARG, INDEX_RANGE, ALIGNMENT, CUDA. */
int hicache_layer_checksum(const hicache_device_kv *kv, const hicache_pool_desc *desc,
                           const int64_t *device_pages, int64_t n, int32_t layer_id,
                           int32_t reps, uint64_t *out_sum_dev, void *stream);

/* ---- tensor-parallel load of a replicated latent ---------------------------------
 * "Baidu's KVCache Overhaul", section "MLA-class cache optimization": with MLA
 * latents (and the CSA/HCA caches named there) every rank of a tensor-parallel
 * group of tp GPUs holds the same KV, so each GPU reads only its part of the
 * pages over its host link and the parts reach every GPU over NVLink, the host
 * reads and the NVLink traffic running side by side, layer by layer.
 *
 * hicache_tp_share: the pairs [*first, *first + *count) of rank `rank` when n
 * pairs are split into tp contiguous parts in the caller's order:
 * [floor(n*rank/tp), floor(n*(rank+1)/tp)).  1 <= tp <= 16, 0 <= rank < tp,
 * 0 <= n < 2^40.  Host-only.  Errors: INVALID_ARG.
 * The backup of a replicated latent splits the same way and needs no
 * exchange: rank r calls hicache_backup for its own pairs, from its own
 * replica into the host memory the ranks share (or one rank backs up them
 * all), so each rank's host link carries 1/tp of the bytes. */
int hicache_tp_share(int64_t n, int32_t tp, int32_t rank, int64_t *first, int64_t *count);
/* The device address of the pool's num_layers per-layer counters (uint32, in
 * device memory the pool owns), which hicache_tp_load_pipelined of any rank
 * raises.  Export it to the other ranks of the group (e.g. with
 * cudaIpcGetMemHandle on the allocation) so that their loads can count into
 * it.  Errors: INVALID_ARG. */
int hicache_pool_layer_counters(hicache_pool *pool, void **counters_out);
/* This rank's part of a tensor-parallel load: the pairs of hicache_tp_share(n,
 * tp, rank) are read from `pool`'s host memory (the group's replicated latent,
 * e.g. one host buffer the ranks share) and every vector is stored into the
 * same device page of each rank's buffers, rank_kvs[0..tp) (rank_kvs[rank] is
 * this rank's own; the others are peers' buffers mapped into this GPU's
 * address space with peer access enabled), layer by layer in one launch like
 * hicache_load_pipelined.  Every finished tile of layer l adds one to word l
 * of every rank's counters, rank_counters[0..tp) (hicache_pool_layer_counters
 * of each rank, device-addressable from here), behind a system-wide fence; a
 * CTA adds its tiles of a layer at once, when it moves past that layer.  This
 * pool's per-layer targets rise by the tiles of ALL ranks' parts, so once
 * every rank of the group has made the same call, hicache_wait_layer(pool, l,
 * stream) waits until every part of layer l has landed in this rank's
 * buffers.
 *   - Every rank validates the whole request (range, duplicate device pages)
 *     and accepts or refuses it alike; each rank's buffers hold the same
 *     device_num_pages; tp * num_buffers * num_layers <= 1024.
 *   - The ranks must make the same calls in the same order, and a rank must
 *     not start the next tensor-parallel load of a pool until every rank's
 *     waits for the previous one are satisfied: the counters add up tiles
 *     from every rank and cannot tell two loads apart.
 *   - No kernel waits for another rank; a rank that never makes its call
 *     leaves the other ranks' waits unsatisfied.
 *   - Stream rules and errors as hicache_load_pipelined (a capturing stream is
 *     refused); on a refused call nothing is enqueued and no target changes.
 * One GPU can stand in for the group: tp pools on the same device, each with
 * its own device KV, all over the same host memory. */
int hicache_tp_load_pipelined(hicache_pool *pool, const hicache_device_kv *rank_kvs,
                              void *const *rank_counters, int32_t tp, int32_t rank,
                              const int64_t *device_pages, const int64_t *host_pages, int64_t n,
                              int32_t layout, void *stream);

/* ---- bounds-checked builds ----------------------------------------------------------
 * libhicache_checked.so is this library built with HICACHE_CHECKED=1: every
 * transfer kernel checks each decoded vector before it touches memory -- the
 * device buffer index against B*L, the offset in the device buffer against
 * device_num_pages * page_size * row, the offset in the host pool against the
 * pool, the run index against the run table -- and instead of an access
 * outside them it skips the access and records the failure in a device word
 * (no trap, no fault).  With the host's validation in front, no check should
 * ever fail; the checked build is the device-side evidence of that.
 * hicache_checked_build: 1 for the checked build, 0 otherwise.
 * hicache_check_status: the first failed check since the last clear (0 if
 * none; else bit 63 set, the check in bits 60-62 -- 1 buffer index, 2 device
 * offset, 3 host offset, 4 run index -- and the offending value in bits 0-59)
 * and the number of failed checks, of the current device; clears both if
 * `clear`.  Reads device memory synchronously (call it once the transfers are
 * done); always 0 and 0 in the plain build.  Errors: INVALID_ARG, CUDA. */
int32_t hicache_checked_build(void);
int hicache_check_status(uint64_t *first, uint64_t *count, int32_t clear);

/* ---- roofline probe -----------------------------------------------------------
 * A plain streaming copy of `bytes` from src to dst with no index decode: each
 * CTA of `grid` (0 = one per SM) moves tiles of 256 threads x vecs_per_thread
 * (4 or 8; 0 = 4) consecutive 16-byte vectors, all loads of a tile in flight
 * before its stores, CTAs in address order -- the transfer kernels' access
 * pattern without their address arithmetic.  It is the zero-copy counterpart
 * of the copy-engine baseline (cudaMemcpyAsync) that "HiCache 시스템 설계와
 * 최적화", section "CPU→GPU 전송 최적화", measures its GPU I/O kernels against,
 * and serves to tell which resource caps the host link.  dst and src are
 * device memory of the current device or pinned, device-mapped host memory
 * (each checked up to its last byte with cudaPointerGetAttributes; host
 * memory is addressed through its device alias), 16-byte aligned, not
 * overlapping; bytes a multiple of 16 (0: nothing enqueued).  Enqueues one
 * launch on `stream`.  Errors: INVALID_ARG, ALIGNMENT, NOT_PINNED (pageable
 * or unknown memory), CUDA; on error nothing is enqueued. */
int hicache_stream_copy(void *dst, const void *src, size_t bytes, int32_t grid, int32_t vecs_per_thread,
                        void *stream);

#ifdef __cplusplus
}
#endif

#endif /* HICACHE_H_ */
