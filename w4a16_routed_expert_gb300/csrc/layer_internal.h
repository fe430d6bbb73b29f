// Internal definition of the layer handle, shared by the runtime
// (moe_layer.cu) and the partial-residency driver (residency.cu).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "kernels.h"
#include "moe_layer.h"

namespace moe {
struct Residency;
}

inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// A stage-timing event: inside a stream capture it becomes an external
// event node of the graph (so replays record it); outside, a plain record.
inline void prof_record(cudaEvent_t ev, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal);
  else
    cudaEventRecord(ev, s);
}

struct Layout {
  size_t off[9];   // gate_q, up_q, down_q, gate_s, up_s, down_s (, gate_z, up_z, down_z)
  size_t size[9];
  size_t record;
  size_t payload;
  bool zp = false;
};

// The canonical record: each section on a 256-byte boundary; with zero
// points, one byte per group of each matrix in three sections after the
// scales.
inline bool record_layout(int H, int I, int G, bool zp, Layout* L) {
  if (H <= 0 || I <= 0 || G <= 0 || (H % 2) || (I % 2)) return false;
  const size_t gh = (size_t)(H + G - 1) / G, gi = (size_t)(I + G - 1) / G;
  const size_t sizes[9] = {(size_t)I * H / 2, (size_t)I * H / 2, (size_t)H * I / 2,
                           2 * (size_t)I * gh,  2 * (size_t)I * gh,  2 * (size_t)H * gi,
                           (size_t)I * gh,      (size_t)I * gh,      (size_t)H * gi};
  const int n = zp ? 9 : 6;
  size_t cur = 0, payload = 0;
  for (int i = 0; i < 9; ++i) {
    L->off[i] = 0;
    L->size[i] = 0;
  }
  for (int i = 0; i < n; ++i) {
    cur = align256(cur);
    L->off[i] = cur;
    L->size[i] = sizes[i];
    cur += sizes[i];
    payload += sizes[i];
  }
  L->record = align256(cur);
  L->payload = payload;
  L->zp = zp;
  return true;
}

struct moe_layer {
  moe_layer_config_t cfg;
  moe_layer_weights_t w;
  int device = 0;
  int num_sms = 0;
  Layout lay;
  int n_records = 0;
  bool pdl = true;
  bool decode_pdl = false;  // the cooperative decode launch also takes programmatic serialisation
  // workspace (one allocation)
  void* ws = nullptr;
  float* logits = nullptr;
  float* logit_part = nullptr;
  __half* xs = nullptr;          // [P][H] tokens in expert-sorted order (GEMM path)
  int32_t* ids = nullptr;
  float* wts = nullptr;
  int32_t* chunk_hist = nullptr;
  int32_t* chunk_base = nullptr;
  int32_t* counts = nullptr;
  int32_t* offsets = nullptr;
  int32_t* perm = nullptr;
  int32_t* inv_perm = nullptr;
  int32_t* seg_expert = nullptr;
  int32_t* seg_start = nullptr;
  int32_t* seg_count = nullptr;
  int32_t* num_seg = nullptr;
  uint32_t* ticket = nullptr;
  uint32_t* err = nullptr;
  __half* hbuf = nullptr;
  float* ypart = nullptr;
  __half* x_stage = nullptr;
  __half* out_stage = nullptr;
  int32_t* ids_stage = nullptr;
  float* w_stage = nullptr;
  int last_T = 0;
  bool variant = false;          // zero points, G = 32 or a gated shared expert: the multi-kernel path only
  bool decode1 = true;           // batch-1 decode kernel (full residency, T == 1)
  bool megakernel = true;        // single-launch decode (full residency)
  int megakernel_max_tokens = 4;  // largest T it takes (<= 16); measured faster than the multi-kernel path up to 4
  bool last_single = false;      // the last profiled forward was one launch
  unsigned long long* trace = nullptr;  // per-CTA phase stamps of the single-launch decode (MOE_TRACE=1)
  unsigned long long* gemm_stats = nullptr;  // GEMM wait counters (MOE_GEMM_STATS=1): [2][CTAs][kGemmStats]
  uint32_t* ctr = nullptr;       // megakernel counters (zero between launches)
  uint32_t* ctr1 = nullptr;      // batch-1 decode epoch counters (zero at create)
  // prefill (tensor-core) path
  int gemm_min_tokens = 48;  // tensor-core GEMM from this T (below it the grouped GEMV is faster)
  bool gemm_ok = false;         // shapes suit the GEMM (H, I multiples of 64)
  moe::CodeMaps pool_maps = {};  // code sections of the caller's pool (full residency)
  moe::TcGemvPlan dec_pg = {}, dec_pd = {};  // GEMV work items: gate/up, down
  CUtensorMap h_map = {};        // h workspace rows
  CUtensorMap xs_map = {};       // tokens in expert-sorted order (xs)
  bool profiling = false;
  cudaEvent_t ev[5] = {};
  moe::Residency* res = nullptr;  // partial residency state
  moe_layer_stats_t stats = {};
};


namespace moe {

// Device pointers of an expert-segment list (see RouteArgs).
struct SegPtrs {
  const int32_t* num_seg;
  const int32_t* seg_expert;
  const int32_t* seg_start;
  const int32_t* seg_count;
};

// Enqueue gate/up + down over the given segments (no combine).
moe_status_t enqueue_experts(moe_layer* L, const __half* x, int T, cudaStream_t s, const uint8_t* pool,
                             const int32_t* e2s, int num_slots, const SegPtrs& seg, int max_seg,
                             const CodeMaps* maps);
// Encode the three code-section tensor maps of a slot pool.
bool encode_pool_maps(const moe_layer* L, const uint8_t* pool, int num_slots, CodeMaps* maps);
// Single-launch decode; MOE_ERR_UNSUPPORTED when no variant fits the shapes.
moe_status_t enqueue_decode(moe_layer* L, const __half* x, int T, __half* out, int32_t* ids_user, float* w_user,
                            cudaStream_t s);
// Batch-1 decode (T == 1); MOE_ERR_UNSUPPORTED when a CTA's share does not
// fit its shared memory.
moe_status_t enqueue_decode1(moe_layer* L, const __half* x, __half* out, int32_t* ids_user, float* w_user,
                             cudaStream_t s);
// Enqueue the weighted combine of the expert outputs into out.
moe_status_t enqueue_combine(moe_layer* L, const __half* x, int T, __half* out, cudaStream_t s);
// Arguments of the batch-1 kernel for one layer (the single-layer launch and
// the stack kernel).
void fill_decode1_args(moe_layer* L, const __half* x, __half* out, int32_t* ids_user, float* w_user,
                       Decode1Args* a);
// Record the calling thread's error message; returns st.
moe_status_t set_error(moe_status_t st, const char* fmt, ...);

}  // namespace moe
