// hicache_engine.cpp -- a submission engine over one pool: callers queue
// backups and loads; one worker thread launches them, in submission order, on
// the engine's own stream.
//
// The pages move transfer submission off the scheduler thread: a backup thread
// and a load thread consume queues and submit on private streams ("Tuning
// SGLang HiCache L2 on Kunlunxin P800/P900", section 2.2; "Baidu's KVCache
// Overhaul", section "Bidirectional Async Transfer").  On GB300 two launches of
// opposite directions on two streams reach about 0.95 of what the host link
// carries both ways, while one launch carrying both reaches 1.00; so here one
// worker owns the link: when the request at the head of the queue and the one
// right behind it go in opposite directions, use the same device buffers and
// touch no page that the other writes, they go out as one fused launch.  The
// worker also looks a few requests further for the partner, and lets it move
// ahead of same-direction requests only where the two commute, so the outcome
// is always that of submission order.  Everything else goes out alone, in order.
//
// Requests are validated, and pre-passed, in the submitting thread: a bad
// request is refused at submit and never queued.  Completion is tracked per
// launch with one event; launches finish in launch order (one stream), and a
// ticket moved ahead by pairing finishes before the tickets it overtook.

#include <algorithm>
#include <chrono>
#include <condition_variable>
#include <cstring>
#include <deque>
#include <mutex>
#include <new>
#include <set>
#include <string>
#include <thread>
#include <vector>

#include "hicache_host.h"

using hicache::RunRec;

namespace {

struct Request {
  uint64_t ticket = 0;
  int32_t direction = 0;
  int32_t layout = 0;
  std::vector<void *> bufs;           // copy of the caller's buffer table
  int64_t device_num_pages = 0;
  std::vector<RunRec> runs;
  std::vector<int64_t> dev, host;     // the pages, for hazard checks
  cudaEvent_t after = nullptr;        // recorded on the caller's stream, or null
};

struct Launched {
  uint64_t t0, t1;   // the tickets of the launch (t1 = 0: a single request)
  cudaEvent_t done;
  int waiters;     // threads polling `done` right now: the event is not reused meanwhile
  bool finished;   // `done` has been seen complete
};

// Launches kept unfinished on the engine stream at once: one running and one
// queued behind it.  Requests submitted meanwhile wait in the queue, where a
// backup and a load can meet and leave as one fused launch.  A request with
// no partner, and fewer than kLookahead requests behind it, is held while any
// launch is unfinished: launched early it would only queue behind that launch,
// and held it can still meet a partner.
constexpr size_t kDepth = 2;

void poll_until_done(cudaEvent_t ev) {
  const auto start = std::chrono::steady_clock::now();
  while (cudaEventQuery(ev) == cudaErrorNotReady) {
    const auto us = std::chrono::duration_cast<std::chrono::microseconds>(
                        std::chrono::steady_clock::now() - start)
                        .count();
    if (us < 500) std::this_thread::yield();
    else std::this_thread::sleep_for(std::chrono::microseconds(50));
  }
}

// Requests of opposite directions commute when the load writes no device
// page the backup reads and the backup writes no host page the load reads
// (checked on page numbers alone, which is conservative when the two use
// different device buffers).
bool commute(const Request &a, const Request &b) {
  int64_t page = 0;
  return !hicache::intersects(a.dev, b.dev, &page) && !hicache::intersects(a.host, b.host, &page);
}

bool fusable(const Request &a, const Request &b) {
  if (a.direction == b.direction || a.layout != b.layout) return false;
  if (a.device_num_pages != b.device_num_pages || a.bufs != b.bufs) return false;
  if (a.runs.empty() || b.runs.empty()) return false;
  return commute(a, b);
}

// How far behind the head the worker looks for a partner of the other direction.
constexpr size_t kLookahead = 8;

}  // namespace

struct hicache_engine {
  hicache_pool *pool = nullptr;
  cudaStream_t stream = nullptr;
  std::thread worker;
  std::mutex mu;
  std::condition_variable cv_work, cv_launched;
  std::deque<Request> queue;
  std::deque<Launched> inflight;      // launched and not yet retired, in launch order
  std::vector<cudaEvent_t> spare;     // events ready for reuse
  uint64_t next_ticket = 1;
  uint64_t launched_prefix = 0;       // every ticket <= this is launched
  std::set<uint64_t> launched_ahead;  // launched tickets above the prefix
  bool stop = false;
  int error = 0;
  std::string error_text;
  int64_t launches = 0, fused = 0;

  // Under mu.  Mark launches whose event has fired (they finish in order);
  // returns the number still unfinished.
  size_t refresh() {
    size_t unfinished = 0;
    for (auto &l : inflight) {
      if (!l.finished) {
        if (unfinished == 0 && cudaEventQuery(l.done) == cudaSuccess)
          l.finished = true;
        else
          ++unfinished;
      }
    }
    return unfinished;
  }

  // Under mu.
  bool is_launched(uint64_t t) const { return t <= launched_prefix || launched_ahead.count(t) != 0; }
  void mark_launched(uint64_t t) {
    launched_ahead.insert(t);
    while (launched_ahead.count(launched_prefix + 1)) launched_ahead.erase(++launched_prefix);
  }
  // Under mu.  The unretired launch holding ticket t, or nullptr (retired =
  // finished: launches are retired only once their event has fired).
  Launched *find(uint64_t t) {
    for (auto &l : inflight)
      if (l.t0 == t || l.t1 == t) return &l;
    return nullptr;
  }

  // Under mu.  An event for a new launch or dependency: a finished, unwatched
  // launch's event if there is one, else a spare, else a new one.
  cudaEvent_t take_event() {
    refresh();
    while (!inflight.empty() && inflight.front().finished && inflight.front().waiters == 0) {
      spare.push_back(inflight.front().done);
      inflight.pop_front();
    }
    if (!spare.empty()) {
      cudaEvent_t e = spare.back();
      spare.pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return nullptr;
    return e;
  }

  void run() {
    cudaSetDevice(pool->device);
    for (;;) {
      std::unique_lock<std::mutex> lk(mu);
      cv_work.wait(lk, [&] { return stop || !queue.empty(); });
      if (queue.empty()) return;
      // pace the launches by the GPU: wait while kDepth launches are unfinished
      while (refresh() >= kDepth) {
        cudaEvent_t oldest = nullptr;
        for (auto &l : inflight)
          if (!l.finished) {
            oldest = l.done;
            l.waiters++;
            break;
          }
        lk.unlock();
        poll_until_done(oldest);
        lk.lock();
        for (auto &l : inflight)  // our waiter count kept this entry (and its event) alive
          if (l.done == oldest) {
            l.waiters--;
            break;
          }
      }
      // the first request of the other direction among the kLookahead behind
      // the head; it may move ahead of the same-direction requests before it
      // only if it commutes with each of them
      size_t partner = 0;  // its index in the queue (0: none)
      for (size_t i = 1; i < queue.size() && i <= kLookahead; ++i) {
        if (queue[i].direction == queue.front().direction) continue;
        bool ok = fusable(queue.front(), queue[i]);
        for (size_t k = 1; ok && k < i; ++k) ok = commute(queue[k], queue[i]);
        if (ok) partner = i;
        break;
      }
      if (partner == 0 && !stop && queue.size() <= kLookahead && refresh() > 0) {
        // no partner yet, room behind the head for one to arrive, and the link
        // busy: a request launched now would only wait behind the running
        // launch on the engine stream, so hold it until that launch ends or
        // another request arrives.  (With the window full, a later arrival
        // could not pair with the head anyway.)
        const size_t seen = queue.size();
        cv_work.wait_for(lk, std::chrono::microseconds(10),
                         [&] { return stop || queue.size() != seen; });
        continue;
      }
      const bool pair = partner != 0;
      Request b;
      if (pair) {
        b = std::move(queue[partner]);
        queue.erase(queue.begin() + std::ptrdiff_t(partner));
      }
      Request a = std::move(queue.front());
      queue.pop_front();
      cudaEvent_t done = take_event();
      lk.unlock();

      int rc = HICACHE_OK;
      std::string text;
      if (!done) rc = hicache::set_error(HICACHE_ERR_CUDA, "cudaEventCreate failed");
      for (Request *r : {&a, pair ? &b : nullptr}) {
        if (rc == HICACHE_OK && r && r->after && cudaStreamWaitEvent(stream, r->after, 0) != cudaSuccess)
          rc = hicache::set_error(HICACHE_ERR_CUDA, "cudaStreamWaitEvent failed");
      }
      if (rc == HICACHE_OK) {
        const hicache_device_kv kv{a.bufs.data(), a.device_num_pages};
        if (pair) {
          const Request &bk = a.direction == HICACHE_DIR_BACKUP ? a : b;
          const Request &ld = a.direction == HICACHE_DIR_BACKUP ? b : a;
          rc = hicache::enqueue(pool, &kv, bk.runs, &ld.runs, a.layout, -1, true, stream);
        } else {
          rc = hicache::enqueue(pool, &kv, a.runs, nullptr, a.layout, -1,
                                a.direction == HICACHE_DIR_BACKUP, stream);
        }
      }
      if (rc == HICACHE_OK && cudaEventRecord(done, stream) != cudaSuccess)
        rc = hicache::set_error(HICACHE_ERR_CUDA, "cudaEventRecord failed");
      if (rc != HICACHE_OK) text = hicache_last_error();

      lk.lock();
      for (Request *r : {&a, pair ? &b : nullptr})
        if (r && r->after) spare.push_back(r->after);
      if (rc == HICACHE_OK) {
        inflight.push_back(Launched{a.ticket, pair ? b.ticket : 0, done, 0, false});
        ++launches;
        if (pair) ++fused;
      } else {
        if (done) spare.push_back(done);
        if (!error) {
          error = rc;
          error_text = text;
        }
      }
      mark_launched(a.ticket);
      if (pair) mark_launched(b.ticket);
      lk.unlock();
      cv_launched.notify_all();
    }
  }
};

extern "C" {

int hicache_engine_create(hicache_pool *pool, hicache_engine **out) {
  hicache::clear_error();
  if (!pool || !out) return hicache::set_error(HICACHE_ERR_INVALID_ARG, "pool or out is NULL");
  *out = nullptr;
  hicache_engine *e = new (std::nothrow) hicache_engine();
  if (!e) return hicache::set_error(HICACHE_ERR_NOMEM, "out of host memory");
  e->pool = pool;
  int prev = 0;
  cudaGetDevice(&prev);
  cudaSetDevice(pool->device);
  const cudaError_t ce = cudaStreamCreateWithFlags(&e->stream, cudaStreamNonBlocking);
  cudaSetDevice(prev);
  if (ce != cudaSuccess) {
    delete e;
    return hicache::cuda_error(ce, "cudaStreamCreateWithFlags");
  }
  try {
    e->worker = std::thread([e] { e->run(); });
  } catch (...) {
    cudaStreamDestroy(e->stream);
    delete e;
    return hicache::set_error(HICACHE_ERR_NOMEM, "could not start the engine thread");
  }
  *out = e;
  return HICACHE_OK;
}

int hicache_engine_destroy(hicache_engine *e) {
  hicache::clear_error();
  if (!e) return HICACHE_OK;
  {
    std::lock_guard<std::mutex> g(e->mu);
    e->stop = true;
  }
  e->cv_work.notify_all();
  e->worker.join();
  const cudaError_t ce = cudaStreamSynchronize(e->stream);
  for (auto &l : e->inflight) cudaEventDestroy(l.done);
  for (auto ev : e->spare) cudaEventDestroy(ev);
  cudaStreamDestroy(e->stream);
  delete e;
  if (ce != cudaSuccess) return hicache::cuda_error(ce, "cudaStreamSynchronize");
  return HICACHE_OK;
}

int hicache_engine_submit(hicache_engine *e, const hicache_device_kv *kv, const int64_t *device_pages,
                          const int64_t *host_pages, int64_t n, int32_t direction, int32_t layout,
                          int32_t after_stream_valid, void *after_stream, uint64_t *ticket) {
  hicache::clear_error();
  if (!e || !ticket) return hicache::set_error(HICACHE_ERR_INVALID_ARG, "engine or ticket is NULL");
  hicache_pool *pool = e->pool;
  int32_t lay = 0;
  int rc = hicache::resolve_layout(layout, pool->shape.layout, &lay);
  if (rc) return rc;
  if ((rc = hicache::check_kv(pool, kv, 0))) return rc;
  Request r;
  if ((rc = hicache::prepass(pool->shape.Hp, kv->device_num_pages, device_pages, host_pages, n,
                             direction, hicache::max_run_pages(pool->shape), &r.runs)))
    return rc;
  r.direction = direction;
  r.layout = lay;
  r.bufs.assign(kv->buf_ptrs, kv->buf_ptrs + pool->shape.B * pool->shape.L);
  r.device_num_pages = kv->device_num_pages;
  if (n > 0) {
    r.dev.assign(device_pages, device_pages + n);
    r.host.assign(host_pages, host_pages + n);
  }
  {
    std::lock_guard<std::mutex> g(e->mu);
    if (e->error) return hicache::set_error(e->error, "engine stopped after an error: %s", e->error_text.c_str());
    if (after_stream_valid) {
      r.after = e->take_event();
      if (!r.after) return hicache::set_error(HICACHE_ERR_CUDA, "cudaEventCreate failed");
      const cudaError_t ce = cudaEventRecord(r.after, static_cast<cudaStream_t>(after_stream));
      if (ce != cudaSuccess) {
        e->spare.push_back(r.after);
        return hicache::cuda_error(ce, "cudaEventRecord(after_stream)");
      }
    }
    r.ticket = e->next_ticket++;
    *ticket = r.ticket;
    e->queue.push_back(std::move(r));
  }
  e->cv_work.notify_one();
  return HICACHE_OK;
}

int hicache_engine_wait(hicache_engine *e, uint64_t ticket, int64_t timeout_us) {
  hicache::clear_error();
  if (!e) return hicache::set_error(HICACHE_ERR_INVALID_ARG, "engine is NULL");
  const auto start = std::chrono::steady_clock::now();
  auto waited_us = [&] {
    return std::chrono::duration_cast<std::chrono::microseconds>(std::chrono::steady_clock::now() - start)
        .count();
  };
  std::unique_lock<std::mutex> lk(e->mu);
  if (ticket == 0 || ticket >= e->next_ticket)
    return hicache::set_error(HICACHE_ERR_INVALID_ARG, "unknown ticket %llu", (unsigned long long)ticket);
  while (!e->is_launched(ticket)) {
    if (timeout_us >= 0) {
      const int64_t left = timeout_us - waited_us();
      if (left <= 0) return hicache::set_error(HICACHE_ERR_TIMEOUT, "ticket not launched yet");
      e->cv_launched.wait_for(lk, std::chrono::microseconds(left));
    } else {
      e->cv_launched.wait(lk);
    }
  }
  if (e->error) return hicache::set_error(e->error, "engine error: %s", e->error_text.c_str());
  Launched *l = e->find(ticket);
  if (!l || l->finished) return HICACHE_OK;
  l->waiters++;  // keeps the entry (and its event) from being retired
  cudaEvent_t ev = l->done;
  lk.unlock();
  int rc = HICACHE_OK;
  for (;;) {
    const cudaError_t q = cudaEventQuery(ev);
    if (q == cudaSuccess) break;
    if (q != cudaErrorNotReady) {
      rc = hicache::cuda_error(q, "cudaEventQuery");
      break;
    }
    const int64_t w = waited_us();
    if (timeout_us >= 0 && w >= timeout_us) {
      rc = hicache::set_error(HICACHE_ERR_TIMEOUT, "transfer still running after %lld us", (long long)w);
      break;
    }
    if (w < 500) std::this_thread::yield();
    else std::this_thread::sleep_for(std::chrono::microseconds(50));
  }
  lk.lock();
  l = e->find(ticket);  // still there: its waiter count was held
  if (l) {
    l->waiters--;
    if (rc == HICACHE_OK) l->finished = true;
  }
  return rc;
}

int hicache_engine_wait_on_stream(hicache_engine *e, uint64_t ticket, void *stream) {
  hicache::clear_error();
  if (!e) return hicache::set_error(HICACHE_ERR_INVALID_ARG, "engine is NULL");
  std::unique_lock<std::mutex> lk(e->mu);
  if (ticket == 0 || ticket >= e->next_ticket)
    return hicache::set_error(HICACHE_ERR_INVALID_ARG, "unknown ticket %llu", (unsigned long long)ticket);
  e->cv_launched.wait(lk, [&] { return e->is_launched(ticket); });
  if (e->error) return hicache::set_error(e->error, "engine error: %s", e->error_text.c_str());
  Launched *l = e->find(ticket);
  if (!l || l->finished) return HICACHE_OK;
  // under the lock: the event cannot be reused before the wait is enqueued
  const cudaError_t ce = cudaStreamWaitEvent(static_cast<cudaStream_t>(stream), l->done, 0);
  if (ce != cudaSuccess) return hicache::cuda_error(ce, "cudaStreamWaitEvent");
  return HICACHE_OK;
}

int hicache_engine_stats(hicache_engine *e, int64_t *launches, int64_t *fused_launches) {
  hicache::clear_error();
  if (!e) return hicache::set_error(HICACHE_ERR_INVALID_ARG, "engine is NULL");
  std::lock_guard<std::mutex> g(e->mu);
  if (launches) *launches = e->launches;
  if (fused_launches) *fused_launches = e->fused;
  return HICACHE_OK;
}

}  // extern "C"
