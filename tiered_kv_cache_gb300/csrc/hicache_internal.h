// hicache_internal.h -- types shared by the host files (hicache_*.cpp) and the
// transfer kernels (hicache_kernels.cu).  Not part of the public ABI.
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define HC_HD __host__ __device__ __forceinline__
#else
#define HC_HD inline
#endif

namespace hicache {

// ---- launch geometry ------------------------------------------------------
constexpr int kThreads = 256;                    // threads per CTA
#ifndef HICACHE_UNROLL
#define HICACHE_UNROLL 4
#endif
constexpr int kUnroll = HICACHE_UNROLL;          // 16-byte vectors in flight per thread
constexpr int kTileVecs = kThreads * kUnroll;    // vectors per tile (16 KiB at unroll 4)
constexpr int kMaxBufs = 512;                    // B * L device buffers per call
constexpr int kBlobWords = 3584;                 // 28 KiB of kernel parameters: buffer
                                                 // pointers, then the run table
constexpr int kBlobWordsSmall = 480;             // the same in under 4 KiB, for calls
                                                 // whose table fits (cheaper to launch)
// One CTA per SM for a load of every layer: 16 KiB in flight per CTA saturates
// the host link, and holds the link's share against a backup running at the
// same time on another stream.
constexpr int kDefaultLoadCtasPerSm = 1;
// One CTA per two SMs for per-layer and pipelined loads, whose purpose is to
// overlap compute: half the grid still saturates the link (1.2 MiB in flight
// against the ~0.4 MiB its rate times its latency asks for) and leaves more of
// the GPU to that compute.  At one CTA per SM the compute held the transfer's
// CTAs back, and a 4K-token MLA load plus per-layer attention took 15% longer.
constexpr int kDefaultLayerCtasPer2Sm = 1;
// A fused backup + load alternates the directions in every CTA: two per SM.
constexpr int kDefaultFusedCtasPerSm = 2;
// A backup saturates the link with far fewer CTAs: its host writes are posted,
// so it needs no round trip per tile.  With a whole SM's share it also takes
// more than its half of the link from a load running at the same time on
// another stream, and the pair finishes late.  Five CTAs per eight SMs keeps a
// backup alone at the link's rate and lets the two directions finish together.
constexpr int kDefaultBackupCtasPer8Sm = 5;

// ---- division by a run-time constant ---------------------------------------
// q = floor(n / d) for 0 <= n < 2^31 by one multiply-high, an add and a shift:
// the round-up method of Granlund & Montgomery, "Division by invariant integers
// using multiplication" (PLDI 1994): with s = ceil(log2 d) and
// m = floor(2^32 (2^s - d) / d) + 1, floor(n / d) = (mulhi(m, n) + n) >> s.
// (mulhi(m, n) <= n, so the sum fits 32 bits while n < 2^31.)
struct FastDiv {
  uint32_t d;
  uint32_t m;
  uint32_t s;
};

inline FastDiv make_fastdiv(uint32_t d) {
  FastDiv f{d, 1u, 0u};
  uint32_t s = 0;
  while ((uint64_t(1) << s) < d) ++s;
  f.s = s;
  f.m = uint32_t(((uint64_t(1) << 32) * ((uint64_t(1) << s) - d)) / d + 1);
  return f;
}

HC_HD uint32_t fast_div(uint32_t n, const FastDiv &f) {
#if defined(__CUDA_ARCH__)
  const uint32_t hi = __umulhi(n, f.m);
#else
  const uint32_t hi = uint32_t((uint64_t(n) * f.m) >> 32);
#endif
  return (hi + n) >> f.s;
}

// ---- run table -------------------------------------------------------------
// A run: `len` pages whose host pages h0.. and device pages d0.. both step by
// one.  vec0 = vectors of the runs before it within one "outer" unit: the runs
// of an outer are laid end to end in one vector range, which tiles cut in
// 1024-vector pieces whatever the run boundaries.
struct Run {
  int32_t h0;
  int32_t d0;
  int32_t len;
  int32_t vec0;
};

// Host-side run record (before tiling).
struct RunRec {
  int64_t h0;
  int64_t d0;
  int64_t len;
};

enum Layout : int32_t { kLayerFirst = 0, kPageFirst = 1, kPageFirstDirect = 2, kPageFirstDirectKV = 3 };

// One direction of a launch: its run table and tile counts.
struct Job {
  int32_t n_runs;
  int32_t runs_word;          // first word of the job's run table in XferParams::blob
  int32_t tiles_per_outer;    // tiles of one outer unit (a buffer, or a buffer-layer)
  int32_t total_tiles;
  uint32_t vecs_per_outer;    // vectors of one outer unit: every run end to end (< 2^31)
  uint32_t run_vecs;          // nonzero when every run of the job has the same length:
                              // the vectors of one run, so that vector w of an outer
                              // unit is in run w / run_vecs (fd_run) without a search
  FastDiv fd_run;
};

// Everything a transfer launch needs, in vectors of 16 bytes.
struct XferHeader {
  void *host;                 // device-visible alias of the host pool
  int32_t L, P, V, num_bufs;  // layers, page size, vectors per row, B*L
  int32_t B;                  // buffers
  int32_t layer;              // the layer of a single-layer transfer
  int32_t Hp;                 // host pool pages
  uint32_t unit_per_page;     // vectors one page contributes to a unit
  uint32_t PV, LV, LPV, BLPV; // P*V, L*V, L*P*V, B*L*P*V
  FastDiv fd_V, fd_PV, fd_LV, fd_LPV, fd_BLPV;
  Job job[2];                 // [0]: the transfer (the backup of a bidirectional
                              // launch); [1]: the load of a bidirectional launch
  int32_t wait_previous;      // nonzero: the launch was started early behind work
                              // it may depend on; it waits for that work to finish
                              // before it touches memory
  int32_t Dp;                 // device pages per buffer (bounds-checked builds)
  int64_t host_vecs;          // vectors of the whole host pool (bounds-checked builds)
  unsigned int *signal;       // if not null, every CTA of a one-direction launch adds
                              // one here once its last tile has landed
};

// ---- bounds-checked builds (HICACHE_CHECKED) -------------------------------
// A build with HICACHE_CHECKED=1 checks every decoded vector against the
// extents before touching it: the buffer index within [0, num_bufs), the
// vector offset within the device buffer [0, Dp * P * V), the vector offset
// within the host pool [0, host_vecs), and the run index within the run
// table.  A failed check skips the access and is recorded in a device word
// (hicache_check_status); nothing traps.  The predicate, shared by the kernels
// and a host-side test: 0 if the vector is inside every extent, else the kind
// of the first failed check.
enum CheckKind : int32_t { kCheckOk = 0, kCheckBuffer = 1, kCheckDevice = 2, kCheckHost = 3, kCheckRun = 4 };
HC_HD int32_t check_vector(int64_t bi, int64_t num_bufs, int64_t doff, int64_t dev_vecs, int64_t hoff,
                           int64_t host_vecs) {
  if (bi < 0 || bi >= num_bufs) return kCheckBuffer;
  if (doff < 0 || doff >= dev_vecs) return kCheckDevice;
  if (hoff < 0 || hoff >= host_vecs) return kCheckHost;
  return kCheckOk;
}

template <int WORDS>
struct XferParamsT {
  XferHeader h;
  // blob[0 .. num_bufs): device buffer pointers (buffer-major b*L + l);
  // then the run tables of the jobs (two words per Run).
  uint64_t blob[WORDS];
};
using XferParams = XferParamsT<kBlobWords>;
using XferParamsSmall = XferParamsT<kBlobWordsSmall>;
static_assert(sizeof(XferParams) <= 32764, "kernel parameter limit");
static_assert(sizeof(XferParamsSmall) <= 4096, "small parameter block");

// Stand-in compute: pages are passed in the parameters.
constexpr int kChecksumMaxPages = 6144;
struct ChecksumParams {
  void *bufs[8];              // the B buffers of one layer
  int32_t B, n, reps, pad;
  uint32_t PV;                // vectors per page of one buffer
  unsigned long long *out;
  int32_t pages[kChecksumMaxPages];
};
static_assert(sizeof(ChecksumParams) <= 32764, "kernel parameter limit");

// ---- buffer groups ---------------------------------------------------------
// One launch for several pools that share the page numbering but not the row
// shape (hicache_group_transfer): job j is pool j, with its own header (shape,
// host alias, dividers; its run table in h[j].job[0]) and the tiles
// [tile_start[j], tile_start[j + 1]) of the launch.  The blob holds every
// job's buffer pointers (job j's from word bufs_word[j]), then the run tables.
constexpr int kMaxGroup = 4;
struct GroupHeader {
  int32_t njobs;
  int32_t num_bufs;                   // buffer pointers of all jobs
  int32_t tile_start[kMaxGroup + 1];
  int32_t bufs_word[kMaxGroup];
  XferHeader h[kMaxGroup];
  // pipelined groups only: job j's layer counters and the launch's two
  // scheduler words (as launch_pipelined_load)
  unsigned int *layer_done[kMaxGroup];
  unsigned int *sched;
  // one-layer group loads only: if signal[0] is not null, every CTA adds one to
  // signal[j] for each job j once its last tile has landed
  unsigned int *signal[kMaxGroup];
};
template <int WORDS>
struct GroupParamsT {
  GroupHeader g;
  uint64_t blob[WORDS];
};
constexpr int kGroupBlobWords = int((32764 - sizeof(GroupHeader)) / 8);
constexpr int kGroupBlobWordsSmall = int((4096 - sizeof(GroupHeader)) / 8);
using GroupParams = GroupParamsT<kGroupBlobWords>;
using GroupParamsSmall = GroupParamsT<kGroupBlobWordsSmall>;
static_assert(sizeof(GroupParams) <= 32764, "kernel parameter limit");
static_assert(sizeof(GroupParamsSmall) <= 4096, "small parameter block");
static_assert(kGroupBlobWordsSmall >= 64, "room for a small group's tables");

// Launch entry points (hicache_kernels.cu).  Return a cudaError_t value.
struct XferLaunch {
  XferParams *params;         // filled header + blob
  int words;                  // blob words in use (selects the small parameter block)
  int layout;
  bool all_layers;
  bool to_host;
  bool bidir;                 // job[0] backup and job[1] load, all layers, one launch
  int grid;
  void *stream;
  // Programmatic dependent launch: the kernel may start while the kernel
  // before it on the stream moves its last tiles, and finishes after it.  The
  // kernel before it must be a transfer kernel whose destinations are disjoint
  // from this one's (an earlier launch of the same call, or another layer).
  bool pdl = false;
};
int launch_xfer(const XferLaunch &x);
struct GroupLaunch {
  GroupParams *params;        // filled header + blob
  int words;                  // blob words in use (selects the small parameter block)
  int layout;
  bool all_layers;
  bool to_host;
  int grid;
  void *stream;
  bool pdl = false;           // as XferLaunch::pdl (group_kernel only)
};
int launch_group(const GroupLaunch &x);
// Every layer of every pool of a group, layer by layer, in one launch:
// g.layer_done[j][l] grows by pool j's tiles of one layer once pool j's layer
// l has landed.
int launch_pipelined_group(const GroupLaunch &x);
// Every layer of a load, layer by layer, in one launch; layer_done[l] grows by
// job[0].total_tiles (the tiles of one layer) once layer l has landed.
// sched: two device words, zero at launch, that the launch leaves at zero (its
// tile counter and exit count); launches that may overlap on the GPU need
// their own.
int launch_pipelined_load(const XferLaunch &x, unsigned int *layer_done, unsigned int *sched);
// A rank's share of a tensor-parallel load of a replicated latent: every
// vector goes to the same place in each of `tp` ranks' buffers (the launch's
// blob holds tp * num_bufs pointers, rank-major, then the run table), and each
// finished tile of layer l adds one to counters[r][l] for every rank r.
constexpr int kMaxTp = 16;
constexpr int kMaxTpBufs = 1024;   // tp * B * L device buffer pointers
struct TpFanout {
  int32_t tp;
  int32_t pad;
  unsigned int *counters[kMaxTp];
};
int launch_tp_pipelined_load(const XferLaunch &x, const TpFanout &f, unsigned int *sched);
// Counters of allocation-free pipelined loads: a static device array of
// kNoAllocMaxLayers layer counters followed by kNoAllocSchedSlots scheduler
// pairs; *out receives its device address on the current device (looked up
// once per device).  Returns a cudaError_t value.
constexpr int kNoAllocMaxLayers = 256;
constexpr int kNoAllocSchedSlots = 64;
constexpr int kNoAllocMaxDevices = 64;
int noalloc_layer_counters(unsigned int **out);
// Record `msg` as the calling thread's last error and return `code` (hicache_api.cpp).
int set_error_text(int code, const char *msg);
int launch_checksum(const ChecksumParams &p, int grid, void *stream);
// 1 in a bounds-checked build (HICACHE_CHECKED), else 0.
int checked_build();
// The bounds-check words of the current device (first failure, count),
// cleared afterwards if `clear`; returns a cudaError_t value.
int check_status(unsigned long long *first, unsigned long long *count, bool clear);
// Roofline probe: copy nvec 16-byte vectors from src to dst (both
// device-addressable), `unroll` (4 or 8) vectors in flight per thread.
int launch_stream_copy(void *dst, const void *src, uint64_t nvec, int grid, int unroll, void *stream);

}  // namespace hicache
