// Partial residency: a library-owned pool of expert records on the device,
// filled from the caller's host copy of every record.
//
// Horizon RunMap report, "Partial-residency contract", steps 1-7, as this
// driver keeps them:
//  1-2. a forward plans its routed experts in transactions (groups computed
//       together, at most num_slots of them); a group whose experts are all
//       resident reads the published rows as they are;
//  3. a miss is copied into a row that is not published (a spare row, or
//       the row of an evicted expert once every kernel reading it has
//       retired), through a bounded ring of pinned staging buffers when the
//       host copy is pageable (copied from directly when it is page-locked);
//  4. a staging buffer is refilled only after the event of its previous
//       transfer has completed;
//  5. the group's mapping (expert -> row) is published, as a new generation,
//       only after its copies have completed (the table upload waits on
//       their event on the forward's stream), and atomically (each
//       transaction reads its own table);
//  6. a row that leaves the published set is overwritten only after the
//       kernels of every transaction that read it (their event) are done;
//  7. eviction only drops the mapping: nothing is ever copied back to the
//       host and the host copy is never written.
// A transaction that fails before publication leaves the previous generation
// authoritative (its rows return to the spares, contents untrusted); a
// failure after publication faults the cache: every later forward fails
// until the handle is destroyed. Capacity is fixed at create (num_slots +
// spare_slots rows, staging_records buffers); too little fails create.
// The policies that pick victims live in expert_cache.cpp.
//
// One forward: routing runs on the caller's stream; the expert counts come
// back to the host (the only device -> host copy and the only
// synchronisation); then, transaction by transaction, the copies go to the
// side stream and the expert kernels to the caller's stream. With spare rows
// the next transaction's copies stream while the current one computes.
#include <algorithm>
#include <condition_variable>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <string>
#include <thread>
#include <vector>

#include "expert_cache.h"
#include "layer_internal.h"
#include "residency.h"

namespace moe {

namespace {
thread_local const char* g_res_err = "";
thread_local char g_res_msg[256];
}

struct Residency {
  ExpertCache cache;
  int num_slots = 0, rows = 0, n_records = 0, E = 0;
  size_t rb = 0;
  const uint8_t* host = nullptr;
  bool host_pinned = false;           // page-locked host copy: copied from directly
  uint8_t* pool = nullptr;            // rows x rb
  cudaStream_t side = nullptr;
  int max_txn = 0;
  int tbl_ints = 0;
  std::vector<cudaEvent_t> ev_done;   // per transaction index: its kernels done (caller's stream)
  std::vector<cudaEvent_t> ev_ready;  // per transaction index: its copies done (side stream)
  std::vector<int> row_reader;        // per row: transaction index whose kernels last read it, -1 none
  // pinned staging ring (pageable host copy)
  int n_staging = 0;
  std::vector<uint8_t*> staging;
  std::vector<cudaEvent_t> ev_staging;
  std::vector<char> staging_used;
  int staging_next = 0;
  int32_t* h_counts = nullptr;
  int32_t* h_tbl = nullptr;
  int32_t* d_tbl = nullptr;
  int inject = 0;  // host-side fault injection (one-shot): 1 before publication, 2 after, 3 in a prefetch
  bool faulted = false;
  CodeMaps maps = {};  // tensor maps of the pool (tensor-core path)
  bool maps_tried = false;
  // prefetch (moe-stream, "Findings"): the guess is routed on the side
  // stream once its input is ready (ev_x) and its counts read back (ev_guess);
  // a worker thread plans it and issues its copies, complete at ev_pref; a
  // forward that reads a row the prefetch filled waits on ev_pref first
  cudaEvent_t ev_x = nullptr, ev_guess = nullptr, ev_pref = nullptr;
  std::vector<char> row_prefetched;
  int32_t* h_guess = nullptr;
  uint64_t prefetch_calls = 0;
  bool guess_enqueued = false;  // a guess's routing is on the side stream (caller's thread only)
  int device = 0;
  std::thread worker;
  std::mutex mu;
  std::condition_variable cv;
  bool stop = false, pending = false;  // under mu
  int pending_T = 0;
  moe_layer* pending_L = nullptr;
  moe_status_t async_st = MOE_OK;  // failure of the last background planning, reported once
  std::string async_msg;
  uint64_t waves = 0, h2d_bytes = 0, staged = 0;
  Residency(int n, int cap, int spares, CachePolicy p) : cache(n, cap, spares, p) {}
};

const char* residency_last_error() { return g_res_err; }

void residency_destroy(Residency* r) {
  if (!r) return;
  if (r->worker.joinable()) {
    {
      std::lock_guard<std::mutex> lk(r->mu);
      r->stop = true;
    }
    r->cv.notify_all();
    r->worker.join();
  }
  if (r->side) cudaStreamSynchronize(r->side);
  for (cudaEvent_t e : r->ev_done)
    if (e) cudaEventDestroy(e);
  for (cudaEvent_t e : r->ev_ready)
    if (e) cudaEventDestroy(e);
  for (cudaEvent_t e : r->ev_staging)
    if (e) cudaEventDestroy(e);
  if (r->ev_x) cudaEventDestroy(r->ev_x);
  if (r->ev_guess) cudaEventDestroy(r->ev_guess);
  if (r->ev_pref) cudaEventDestroy(r->ev_pref);
  if (r->h_guess) cudaFreeHost(r->h_guess);
  for (uint8_t* p : r->staging)
    if (p) cudaFreeHost(p);
  if (r->side) cudaStreamDestroy(r->side);
  if (r->pool) cudaFree(r->pool);
  if (r->d_tbl) cudaFree(r->d_tbl);
  if (r->h_tbl) cudaFreeHost(r->h_tbl);
  if (r->h_counts) cudaFreeHost(r->h_counts);
  delete r;
}

moe_status_t residency_create(const moe_layer_config_t& cfg, size_t record_bytes, int n_records,
                              const void* host_backing, Residency** out) {
  *out = nullptr;
  const int spares = cfg.spare_slots;
  Residency* r = new (std::nothrow) Residency(n_records, cfg.num_slots, spares, (CachePolicy)cfg.cache_policy);
  if (!r) {
    g_res_err = "host allocation failed";
    return MOE_ERR_OOM;
  }
  r->num_slots = cfg.num_slots;
  r->rows = cfg.num_slots + spares;
  r->n_records = n_records;
  r->E = cfg.num_experts;
  r->rb = record_bytes;
  r->host = static_cast<const uint8_t*>(host_backing);
  r->max_txn = (n_records + cfg.num_slots - 1) / cfg.num_slots + 1;
  r->tbl_ints = (int)((4 * (size_t)n_records + 1 + 63) / 64 * 64);
  r->row_reader.assign(r->rows, -1);
  r->row_prefetched.assign(r->rows, 0);
  const char* inj = getenv("MOE_FAULT_INJECT");
  if (inj && strcmp(inj, "h2d_fail") == 0) r->inject = 1;
  if (inj && strcmp(inj, "after_publish") == 0) r->inject = 2;
  if (inj && strcmp(inj, "prefetch_fail") == 0) r->inject = 3;

  moe_status_t st = MOE_OK;
  cudaError_t e = cudaMalloc(&r->pool, (size_t)r->rows * record_bytes);
  if (e != cudaSuccess) {
    g_res_err = "slot pool allocation failed";
    st = MOE_ERR_OOM;
  }
  if (st == MOE_OK) {
    cudaPointerAttributes pa = {};
    r->host_pinned = cudaPointerGetAttributes(&pa, host_backing) == cudaSuccess && pa.type == cudaMemoryTypeHost;
    cudaGetLastError();
    if (!r->host_pinned) {
      // pageable host copy: a bounded ring of pinned staging buffers
      r->n_staging = cfg.staging_records > 0 ? cfg.staging_records : 4;
      r->staging.assign(r->n_staging, nullptr);
      r->ev_staging.assign(r->n_staging, nullptr);
      r->staging_used.assign(r->n_staging, 0);
      for (int i = 0; i < r->n_staging && st == MOE_OK; ++i) {
        if (cudaHostAlloc(reinterpret_cast<void**>(&r->staging[i]), record_bytes, cudaHostAllocDefault) != cudaSuccess) {
          g_res_err = "pinned staging allocation failed";
          st = MOE_ERR_OOM;
        } else if (cudaEventCreateWithFlags(&r->ev_staging[i], cudaEventDisableTiming) != cudaSuccess) {
          g_res_err = "event creation failed";
          st = MOE_ERR_CUDA;
        }
      }
    }
  }
  if (st == MOE_OK && cudaStreamCreateWithFlags(&r->side, cudaStreamNonBlocking) != cudaSuccess) {
    g_res_err = "side stream creation failed";
    st = MOE_ERR_CUDA;
  }
  if (st == MOE_OK && cudaGetDevice(&r->device) != cudaSuccess) {
    g_res_err = "no current device";
    st = MOE_ERR_CUDA;
  }
  if (st == MOE_OK && (cudaEventCreateWithFlags(&r->ev_x, cudaEventDisableTiming) != cudaSuccess ||
                       cudaEventCreateWithFlags(&r->ev_guess, cudaEventDisableTiming) != cudaSuccess ||
                       cudaEventCreateWithFlags(&r->ev_pref, cudaEventDisableTiming) != cudaSuccess)) {
    g_res_err = "event creation failed";
    st = MOE_ERR_CUDA;
  }
  if (st == MOE_OK) {
    r->ev_done.assign(r->max_txn, nullptr);
    r->ev_ready.assign(r->max_txn, nullptr);
    for (int i = 0; i < r->max_txn && st == MOE_OK; ++i) {
      if (cudaEventCreateWithFlags(&r->ev_done[i], cudaEventDisableTiming) != cudaSuccess ||
          cudaEventCreateWithFlags(&r->ev_ready[i], cudaEventDisableTiming) != cudaSuccess) {
        g_res_err = "event creation failed";
        st = MOE_ERR_CUDA;
      }
    }
  }
  if (st == MOE_OK) {
    const size_t tb = (size_t)r->max_txn * r->tbl_ints * sizeof(int32_t);
    if (cudaHostAlloc(&r->h_counts, (size_t)cfg.num_experts * sizeof(int32_t), cudaHostAllocDefault) != cudaSuccess ||
        cudaHostAlloc(&r->h_guess, (size_t)cfg.num_experts * sizeof(int32_t), cudaHostAllocDefault) != cudaSuccess ||
        cudaHostAlloc(&r->h_tbl, tb, cudaHostAllocDefault) != cudaSuccess ||
        cudaMalloc(&r->d_tbl, tb) != cudaSuccess) {
      g_res_err = "residency table allocation failed";
      st = MOE_ERR_OOM;
    }
  }
  if (st != MOE_OK) {
    cudaGetLastError();
    residency_destroy(r);
    return st;
  }
  *out = r;
  return MOE_OK;
}

namespace {

// Copies record `expert` into pool row `row` on the side stream, once the
// kernels that last read that row (their transaction's event) are done:
// directly from a page-locked host copy, else through the next staging
// buffer (refilled on the host after its previous transfer completed).
cudaError_t transport(Residency* r, int expert, int row) {
  cudaError_t e = cudaSuccess;
  if (r->row_reader[row] >= 0) e = cudaStreamWaitEvent(r->side, r->ev_done[r->row_reader[row]], 0);
  if (e != cudaSuccess) return e;
  uint8_t* dst = r->pool + (size_t)row * r->rb;
  const uint8_t* src = r->host + (size_t)expert * r->rb;
  if (r->host_pinned) return cudaMemcpyAsync(dst, src, r->rb, cudaMemcpyHostToDevice, r->side);
  const int si = r->staging_next;
  r->staging_next = (si + 1) % r->n_staging;
  if (r->staging_used[si]) {
    e = cudaEventSynchronize(r->ev_staging[si]);
    if (e != cudaSuccess) return e;
  }
  memcpy(r->staging[si], src, r->rb);
  e = cudaMemcpyAsync(dst, r->staging[si], r->rb, cudaMemcpyHostToDevice, r->side);
  if (e == cudaSuccess) e = cudaEventRecord(r->ev_staging[si], r->side);
  r->staging_used[si] = 1;
  r->staged += 1;
  return e;
}

// Waits until no prefetch is being planned on the worker thread.
void join_prefetch(Residency* r) {
  std::unique_lock<std::mutex> lk(r->mu);
  r->cv.wait(lk, [&] { return !r->pending; });
}

}  // namespace

moe_status_t residency_forward(Residency* r, moe_layer* L, const __half* x, int T, __half* out, cudaStream_t s) {
  const moe_layer_config_t& c = L->cfg;
  const int E = c.num_experts, k = c.top_k;
  if (r->faulted)
    return set_error(MOE_ERR_CUDA, "the expert cache is faulted (a failure after publication); destroy the handle");
  if (!r->maps_tried) {
    r->maps_tried = true;
    encode_pool_maps(L, r->pool, r->rows, &r->maps);
  }
  // demanded experts: the only device -> host copy of the forward
  cudaError_t e = cudaMemcpyAsync(r->h_counts, L->counts, (size_t)E * sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return set_error(MOE_ERR_CUDA, "expert counts device->host: %s", cudaGetErrorString(e));
  std::vector<int> demanded;
  std::vector<int> start(E + 1, 0);
  int run = 0;
  for (int i = 0; i < E; ++i) {
    start[i] = run;
    run += r->h_counts[i];
    if (r->h_counts[i] > 0) demanded.push_back(i);
  }
  if (run != T * k) return set_error(MOE_ERR_INTERNAL, "expert counts sum to %d, expected %d", run, T * k);
  if (c.has_shared_expert) demanded.push_back(E);
  // a prefetch planned on the worker thread finishes before this forward
  // plans; its failure (its transaction aborted, the cache consistent) is
  // reported here, once
  join_prefetch(r);
  if (r->async_st != MOE_OK) {
    const moe_status_t ast = r->async_st;
    r->async_st = MOE_OK;
    return set_error(ast, "prefetch: %s", r->async_msg.c_str());
  }

  // every access is counted (ascending id): a hit is an expert published
  // when the forward starts
  for (int ex : demanded) r->cache.touch(ex, r->cache.row_of(ex) >= 0);
  const int n = r->n_records;
  std::vector<int> remaining = demanded;
  for (int ti = 0; !remaining.empty(); ++ti) {
    if (ti >= r->max_txn) return set_error(MOE_ERR_INTERNAL, "too many transactions in one forward");
    const ExpertCache::Txn t = r->cache.next(remaining, ti == 0);
    if (t.experts.empty()) return set_error(MOE_ERR_INTERNAL, "empty transaction");
    // the transaction's table: expert -> row, and its segment list
    int32_t* tbl = r->h_tbl + (size_t)ti * r->tbl_ints;
    int32_t* e2s = tbl;
    int32_t* nseg = tbl + n;
    int32_t* sexp = nseg + 1;
    int32_t* sstart = sexp + n;
    int32_t* scount = sstart + n;
    std::fill(e2s, e2s + n, -1);
    *nseg = (int32_t)t.experts.size();
    // segments in ascending expert id (the order the kernels expect)
    std::vector<int> ord(t.experts.size());
    for (size_t j = 0; j < ord.size(); ++j) ord[j] = (int)j;
    std::sort(ord.begin(), ord.end(), [&](int a, int b) { return t.experts[a] < t.experts[b]; });
    for (size_t q = 0; q < ord.size(); ++q) {
      const int j = ord[q], ex = t.experts[j];
      e2s[ex] = t.rows[j];
      sexp[q] = ex;
      sstart[q] = ex < E ? start[ex] : T * k;
      scount[q] = ex < E ? r->h_counts[ex] : T;
    }
    if (!t.loads.empty()) {
      if (r->inject == 1 && ti >= 1) {
        // injected failure before publication: the previous generation
        // stays authoritative
        r->inject = 0;
        r->cache.abort(t);
        return set_error(MOE_ERR_CUDA, "injected host->device copy failure before publication (transaction %d)", ti);
      }
      for (size_t j = 0; j < t.loads.size() && e == cudaSuccess; ++j) e = transport(r, t.loads[j].first, t.loads[j].second);
      if (e == cudaSuccess) e = cudaEventRecord(r->ev_ready[ti], r->side);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(s, r->ev_ready[ti], 0);
      if (e != cudaSuccess) {
        r->cache.abort(t);
        return set_error(MOE_ERR_CUDA, "expert copy host->device: %s", cudaGetErrorString(e));
      }
    }
    // rows a prefetch filled are read only after its copies completed
    bool reads_prefetched = false;
    for (int row : t.rows) reads_prefetched = reads_prefetched || r->row_prefetched[row];
    if (reads_prefetched) {
      e = cudaStreamWaitEvent(s, r->ev_pref, 0);
      if (e != cudaSuccess) {
        r->cache.abort(t);
        return set_error(MOE_ERR_CUDA, "prefetch dependency: %s", cudaGetErrorString(e));
      }
      std::fill(r->row_prefetched.begin(), r->row_prefetched.end(), 0);
    }
    // publication on the forward's stream, after the copies completed
    int32_t* dtbl = r->d_tbl + (size_t)ti * r->tbl_ints;
    e = cudaMemcpyAsync(dtbl, tbl, (size_t)r->tbl_ints * sizeof(int32_t), cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) {
      r->cache.abort(t);
      return set_error(MOE_ERR_CUDA, "transaction table host->device: %s", cudaGetErrorString(e));
    }
    r->cache.publish(t);
    if (r->inject == 2 && !t.loads.empty()) {
      r->inject = 0;
      r->faulted = true;
      return set_error(MOE_ERR_CUDA, "injected failure after publication: the expert cache is faulted");
    }
    const SegPtrs seg = {dtbl + n, dtbl + n + 1, dtbl + 2 * n + 1, dtbl + 3 * n + 1};
    moe_status_t st = enqueue_experts(L, x, T, s, r->pool, dtbl, r->rows, seg, (int)t.experts.size(), &r->maps);
    if (st != MOE_OK) {
      r->faulted = true;  // published, kernels not enqueued: the state is ambiguous
      return st;
    }
    e = cudaEventRecord(r->ev_done[ti], s);
    if (e != cudaSuccess) {
      r->faulted = true;
      return set_error(MOE_ERR_CUDA, "transaction event: %s", cudaGetErrorString(e));
    }
    for (int row : t.rows) r->row_reader[row] = ti;
    r->waves += 1;
    r->h2d_bytes += (uint64_t)t.loads.size() * r->rb;
    std::vector<int> rest;
    for (int ex : remaining)
      if (std::find(t.experts.begin(), t.experts.end(), ex) == t.experts.end()) rest.push_back(ex);
    remaining.swap(rest);
  }
  return enqueue_combine(L, x, T, out, s);
}

cudaStream_t residency_side(Residency* r) { return r->side; }
cudaEvent_t residency_input_event(Residency* r) { return r->ev_x; }

namespace {

// The guess's planning (worker thread): wait for its expert counts, pick
// the guessed experts, copy the missing ones into the pool on the side
// stream, publish them in the host model.
moe_status_t plan_prefetch(Residency* r, moe_layer* L, int T) {
  const moe_layer_config_t& c = L->cfg;
  const int E = c.num_experts, k = c.top_k;
  cudaError_t e = cudaEventSynchronize(r->ev_guess);
  if (e != cudaSuccess) return set_error(MOE_ERR_CUDA, "guess routing: %s", cudaGetErrorString(e));
  // the guessed experts: the shared one (demanded by every forward), then the
  // routed ones by count (ties to the lower id), as many as fit
  std::vector<int> order;
  int run = 0;
  for (int i = 0; i < E; ++i) {
    run += r->h_guess[i];
    if (r->h_guess[i] > 0) order.push_back(i);
  }
  if (run != T * k) return set_error(MOE_ERR_INTERNAL, "guess counts sum to %d, expected %d", run, T * k);
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return r->h_guess[a] > r->h_guess[b]; });
  std::vector<int> guessed;
  if (c.has_shared_expert) guessed.push_back(E);
  for (int ex : order)
    if ((int)guessed.size() < r->num_slots) guessed.push_back(ex);
  const ExpertCache::Txn t = r->cache.plan_prefetch(guessed);
  if (t.loads.empty()) return MOE_OK;
  if (r->inject == 3) {
    // injected failure before publication: the previous generation stays
    r->inject = 0;
    r->cache.abort(t);
    return set_error(MOE_ERR_CUDA, "injected prefetch copy failure before publication");
  }
  for (size_t j = 0; j < t.loads.size() && e == cudaSuccess; ++j) e = transport(r, t.loads[j].first, t.loads[j].second);
  if (e == cudaSuccess) e = cudaEventRecord(r->ev_pref, r->side);
  if (e != cudaSuccess) {
    r->cache.abort(t);
    return set_error(MOE_ERR_CUDA, "prefetch copy host->device: %s", cudaGetErrorString(e));
  }
  // published in the host model now; a forward reading these rows waits on
  // ev_pref before its table (the device-side publication) is uploaded
  r->cache.publish(t, true);
  for (const auto& l : t.loads) r->row_prefetched[l.second] = 1;
  r->h2d_bytes += (uint64_t)t.loads.size() * r->rb;
  return MOE_OK;
}

void worker_main(Residency* r) {
  cudaSetDevice(r->device);
  std::unique_lock<std::mutex> lk(r->mu);
  for (;;) {
    r->cv.wait(lk, [&] { return r->stop || r->pending; });
    if (r->pending) {
      lk.unlock();
      const moe_status_t st = plan_prefetch(r, r->pending_L, r->pending_T);
      lk.lock();
      if (st != MOE_OK) {
        r->async_st = st;
        r->async_msg = moe_layer_last_error(nullptr);
      }
      r->pending = false;
      r->cv.notify_all();
      continue;
    }
    return;
  }
}

}  // namespace

cudaError_t residency_before_route(Residency* r, cudaStream_t s) {
  if (!r->guess_enqueued) return cudaSuccess;
  r->guess_enqueued = false;
  return cudaStreamWaitEvent(s, r->ev_guess, 0);
}

moe_status_t residency_prefetch(Residency* r, moe_layer* L, int T) {
  const int E = L->cfg.num_experts;
  join_prefetch(r);
  if (r->faulted)
    return set_error(MOE_ERR_CUDA, "the expert cache is faulted (a failure after publication); destroy the handle");
  // the guess's expert counts come back on the side stream; the worker
  // thread plans the copies once they are there
  cudaError_t e = cudaMemcpyAsync(r->h_guess, L->counts, (size_t)E * sizeof(int32_t), cudaMemcpyDeviceToHost, r->side);
  if (e == cudaSuccess) e = cudaEventRecord(r->ev_guess, r->side);
  if (e != cudaSuccess) return set_error(MOE_ERR_CUDA, "guess counts device->host: %s", cudaGetErrorString(e));
  r->guess_enqueued = true;
  r->prefetch_calls += 1;
  {
    std::lock_guard<std::mutex> lk(r->mu);
    r->pending = true;
    r->pending_T = T;
    r->pending_L = L;
    if (!r->worker.joinable()) r->worker = std::thread(worker_main, r);
  }
  r->cv.notify_all();
  return MOE_OK;
}

void residency_fill_stats(Residency* r, moe_layer_stats_t* st) {
  join_prefetch(r);
  st->expert_hits = r->cache.hits;
  st->expert_misses = r->cache.misses;
  st->h2d_bytes = r->h2d_bytes;
  st->waves = r->waves;
  st->d2h_expert_bytes = 0;
  st->generations = r->cache.generation();
  st->evictions = r->cache.evictions;
  st->staged_copies = r->staged;
  st->faulted = r->faulted ? 1 : 0;
  st->prefetch_calls = r->prefetch_calls;
  st->prefetched = r->cache.prefetched;
  st->prefetch_used = r->cache.prefetch_used;
}

}  // namespace moe
