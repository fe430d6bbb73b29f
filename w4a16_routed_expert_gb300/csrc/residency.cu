// Partial residency: a library-owned pool of num_slots expert records on the
// device, filled from the caller's host copy of every record.
//
// Horizon RunMap report, "Partial-residency contract": the host copy is the
// authority and is never written; misses move compact records host -> device
// through page-locked memory, a copy is used only after its transfer has
// completed (an event), eviction simply discards device copies, a failure
// before use leaves the previous mapping authoritative, and too little
// capacity fails at create. F51 Nitro-MoE, "Layer 1 - expert persistence
// cache": a fixed slot pool per layer addressed through expert_to_slot.
//
// One forward: routing runs on the caller's stream; the expert counts come
// back to the host (the only device -> host copy, and the only
// synchronisation); the slot planner splits the demanded experts into waves
// of at most num_slots experts (hits first). For each wave the side stream
// waits until the previous wave's kernels are done with the slots it
// overwrites, copies the wave's misses, and records an event the caller's
// stream waits on before running the wave's expert kernels. Every wave has
// its own events and its own segment table, so nothing is reused before it
// has retired; the next forward's synchronisation retires them all.
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "layer_internal.h"
#include "residency.h"
#include "slot_planner.h"

namespace moe {

namespace {
thread_local const char* g_res_err = "";
thread_local char g_res_msg[256];
}

struct Residency {
  SlotPlanner planner;
  int num_slots = 0, n_records = 0, E = 0;
  size_t rb = 0;
  const uint8_t* host = nullptr;
  bool registered_here = false;
  uint8_t* pool = nullptr;
  cudaStream_t side = nullptr;
  int max_waves = 0;
  int tbl_ints = 0;
  std::vector<cudaEvent_t> ev_free, ev_ready;
  int32_t* h_counts = nullptr;
  int32_t* h_tbl = nullptr;
  int32_t* d_tbl = nullptr;
  int inject_h2d_fail = 0;  // one-shot host-side fault injection
  CodeMaps maps = {};       // tensor maps of the pool (tensor-core path)
  bool maps_tried = false;
  uint64_t hits = 0, misses = 0, h2d_bytes = 0, waves = 0;
  Residency(int n, int s) : planner(n, s) {}
};

const char* residency_last_error() { return g_res_err; }

void residency_destroy(Residency* r) {
  if (!r) return;
  if (r->side) cudaStreamSynchronize(r->side);
  for (cudaEvent_t e : r->ev_free)
    if (e) cudaEventDestroy(e);
  for (cudaEvent_t e : r->ev_ready)
    if (e) cudaEventDestroy(e);
  if (r->side) cudaStreamDestroy(r->side);
  if (r->pool) cudaFree(r->pool);
  if (r->d_tbl) cudaFree(r->d_tbl);
  if (r->h_tbl) cudaFreeHost(r->h_tbl);
  if (r->h_counts) cudaFreeHost(r->h_counts);
  if (r->registered_here) cudaHostUnregister(const_cast<uint8_t*>(r->host));
  delete r;
}

moe_status_t residency_create(const moe_layer_config_t& cfg, size_t record_bytes, int n_records,
                              const void* host_backing, Residency** out) {
  *out = nullptr;
  Residency* r = new (std::nothrow) Residency(n_records, cfg.num_slots);
  if (!r) {
    g_res_err = "host allocation failed";
    return MOE_ERR_OOM;
  }
  r->num_slots = cfg.num_slots;
  r->n_records = n_records;
  r->E = cfg.num_experts;
  r->rb = record_bytes;
  r->host = static_cast<const uint8_t*>(host_backing);
  r->max_waves = (n_records + cfg.num_slots - 1) / cfg.num_slots + 1;
  r->tbl_ints = (int)((4 * (size_t)n_records + 1 + 63) / 64 * 64);
  const char* inj = getenv("MOE_FAULT_INJECT");
  r->inject_h2d_fail = (inj && strcmp(inj, "h2d_fail") == 0) ? 1 : 0;

  moe_status_t st = MOE_OK;
  cudaError_t e = cudaMalloc(&r->pool, (size_t)cfg.num_slots * record_bytes);
  if (e != cudaSuccess) {
    g_res_err = "slot pool allocation failed";
    st = MOE_ERR_OOM;
  }
  if (st == MOE_OK) {
    // already page-locked (cudaHostAlloc or registered by the caller): use as is
    cudaPointerAttributes pa = {};
    const bool pinned = cudaPointerGetAttributes(&pa, host_backing) == cudaSuccess && pa.type == cudaMemoryTypeHost;
    cudaGetLastError();
    if (!pinned) {
      int ro = 0;
      int dev = 0;
      cudaGetDevice(&dev);
      cudaDeviceGetAttribute(&ro, cudaDevAttrHostRegisterReadOnlySupported, dev);
      const unsigned flags = ro ? cudaHostRegisterReadOnly : cudaHostRegisterDefault;
      e = cudaHostRegister(const_cast<void*>(host_backing), (size_t)n_records * record_bytes, flags);
      if (e == cudaSuccess) {
        r->registered_here = true;
      } else if (e == cudaErrorHostMemoryAlreadyRegistered) {
        cudaGetLastError();
      } else {
        cudaGetLastError();
        snprintf(g_res_msg, sizeof(g_res_msg), "registering the host backing failed: %s", cudaGetErrorString(e));
        g_res_err = g_res_msg;
        st = MOE_ERR_CUDA;
      }
    }
  }
  if (st == MOE_OK && cudaStreamCreateWithFlags(&r->side, cudaStreamNonBlocking) != cudaSuccess) {
    g_res_err = "side stream creation failed";
    st = MOE_ERR_CUDA;
  }
  if (st == MOE_OK) {
    r->ev_free.assign(r->max_waves, nullptr);
    r->ev_ready.assign(r->max_waves, nullptr);
    for (int i = 0; i < r->max_waves && st == MOE_OK; ++i) {
      if (cudaEventCreateWithFlags(&r->ev_free[i], cudaEventDisableTiming) != cudaSuccess ||
          cudaEventCreateWithFlags(&r->ev_ready[i], cudaEventDisableTiming) != cudaSuccess) {
        g_res_err = "event creation failed";
        st = MOE_ERR_CUDA;
      }
    }
  }
  if (st == MOE_OK) {
    const size_t tb = (size_t)r->max_waves * r->tbl_ints * sizeof(int32_t);
    if (cudaHostAlloc(&r->h_counts, (size_t)cfg.num_experts * sizeof(int32_t), cudaHostAllocDefault) != cudaSuccess ||
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

moe_status_t residency_forward(Residency* r, moe_layer* L, const __half* x, int T, __half* out, cudaStream_t s) {
  const moe_layer_config_t& c = L->cfg;
  const int E = c.num_experts, k = c.top_k;
  if (!r->maps_tried) {
    r->maps_tried = true;
    encode_pool_maps(L, r->pool, r->num_slots, &r->maps);
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

  const std::vector<SlotPlanner::Wave> waves = r->planner.plan(demanded);
  if ((int)waves.size() > r->max_waves) return set_error(MOE_ERR_INTERNAL, "planner produced too many waves");
  const int n = r->n_records;
  for (size_t wi = 0; wi < waves.size(); ++wi) {
    const SlotPlanner::Wave& w = waves[wi];
    int32_t* tbl = r->h_tbl + wi * r->tbl_ints;
    int32_t* e2s = tbl;
    int32_t* nseg = tbl + n;
    int32_t* sexp = nseg + 1;
    int32_t* sstart = sexp + n;
    int32_t* scount = sstart + n;
    std::fill(e2s, e2s + n, -1);
    *nseg = (int32_t)w.experts.size();
    for (size_t j = 0; j < w.experts.size(); ++j) {
      const int ex = w.experts[j];
      e2s[ex] = w.slots[j];
      sexp[j] = ex;
      sstart[j] = ex < E ? start[ex] : T * k;
      scount[j] = ex < E ? r->h_counts[ex] : T;
    }
    if (!w.loads.empty()) {
      if (r->inject_h2d_fail && wi == 1) {
        // injected failure before this wave's copies: nothing of this wave
        // is published; earlier waves stay committed
        r->inject_h2d_fail = 0;
        return set_error(MOE_ERR_CUDA, "injected host->device copy failure (wave %zu)", wi);
      }
      e = cudaEventRecord(r->ev_free[wi], s);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(r->side, r->ev_free[wi], 0);
      for (size_t j = 0; j < w.loads.size() && e == cudaSuccess; ++j) {
        const int ex = w.loads[j].first, slot = w.loads[j].second;
        e = cudaMemcpyAsync(r->pool + (size_t)slot * r->rb, r->host + (size_t)ex * r->rb, r->rb,
                            cudaMemcpyHostToDevice, r->side);
      }
      if (e == cudaSuccess) e = cudaEventRecord(r->ev_ready[wi], r->side);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(s, r->ev_ready[wi], 0);
      if (e != cudaSuccess) {
        // the slots this wave was filling can no longer be trusted
        for (const auto& ld : w.loads) r->planner.invalidate(ld.second);
        return set_error(MOE_ERR_CUDA, "expert copy host->device: %s", cudaGetErrorString(e));
      }
    }
    int32_t* dtbl = r->d_tbl + wi * r->tbl_ints;
    e = cudaMemcpyAsync(dtbl, tbl, (size_t)r->tbl_ints * sizeof(int32_t), cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return set_error(MOE_ERR_CUDA, "wave table host->device: %s", cudaGetErrorString(e));
    const SegPtrs seg = {dtbl + n, dtbl + n + 1, dtbl + 2 * n + 1, dtbl + 3 * n + 1};
    moe_status_t st = enqueue_experts(L, x, T, s, r->pool, dtbl, r->num_slots, seg, (int)w.experts.size(), &r->maps);
    if (st != MOE_OK) return st;
    r->planner.commit(w);
    r->hits += w.experts.size() - w.loads.size();
    r->misses += w.loads.size();
    r->h2d_bytes += (uint64_t)w.loads.size() * r->rb;
    r->waves += 1;
  }
  return enqueue_combine(L, x, T, out, s);
}

void residency_fill_stats(const Residency* r, moe_layer_stats_t* st) {
  st->expert_hits = r->hits;
  st->expert_misses = r->misses;
  st->h2d_bytes = r->h2d_bytes;
  st->waves = r->waves;
  st->d2h_expert_bytes = 0;
}

}  // namespace moe
