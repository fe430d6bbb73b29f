// Runtime behind the C ABI declared in include/moe_layer.h: validates the
// configuration, owns the workspace, and enqueues the layer's kernels on the
// caller's stream (routing -> gate/up+SwiGLU -> down -> weighted combine).
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <string>
#include <map>
#include <utility>

#include "layer_internal.h"
#include "residency.h"

namespace {

thread_local std::string g_last_error;
constexpr int kTraceCtas = 1024;  // CTAs the phase-trace buffer holds stamps for
constexpr int kInPlaceHostMaxT = 16;  // forward_host reads / writes mapped host buffers in place up to this T

// Device address of a page-locked, mapped host buffer (nullptr for any
// other memory).
void* mapped_device_ptr(const void* p) {
  cudaPointerAttributes a = {};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

moe_status_t fail(moe_status_t st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

moe_status_t cuda_fail(cudaError_t e, const char* what) {
  return fail(MOE_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

}  // namespace

namespace {

moe_status_t validate(const moe_layer_config_t* c, const moe_layer_weights_t* w) {
  if (!c || !w) return fail(MOE_ERR_INVALID_ARG, "config and weights must not be NULL");
  if (c->hidden < 128 || c->hidden > 4096 || c->hidden % 32)
    return fail(MOE_ERR_UNSUPPORTED, "hidden=%d: supported 128..4096, multiple of 32", c->hidden);
  if (c->intermediate < 128 || c->intermediate > 4096 || c->intermediate % 32)
    return fail(MOE_ERR_UNSUPPORTED, "intermediate=%d: supported 128..4096, multiple of 32", c->intermediate);
  if (c->group_size != 32 && c->group_size != 64 && c->group_size != 128)
    return fail(MOE_ERR_UNSUPPORTED, "group_size=%d: supported 32, 64 or 128", c->group_size);
  if (c->zero_points != 0 && c->zero_points != 1) return fail(MOE_ERR_INVALID_ARG, "zero_points must be 0 or 1");
  if (w && w->shared_gate && !c->has_shared_expert)
    return fail(MOE_ERR_INVALID_ARG, "shared_gate needs has_shared_expert = 1");
  if (c->num_experts < 1 || c->num_experts > 1024)
    return fail(MOE_ERR_INVALID_ARG, "num_experts=%d out of 1..1024", c->num_experts);
  if (c->top_k < 1 || c->top_k > 32 || c->top_k > c->num_experts)
    return fail(MOE_ERR_INVALID_ARG, "top_k=%d out of 1..min(32, E)", c->top_k);
  if (c->max_tokens < 1 || c->max_tokens > (1 << 20))
    return fail(MOE_ERR_INVALID_ARG, "max_tokens=%d out of 1..2^20", c->max_tokens);
  if ((long long)c->max_tokens * (c->top_k + 1) > (1LL << 30))
    return fail(MOE_ERR_INVALID_ARG, "max_tokens * (top_k + 1) too large");
  if (c->renormalize != 0 && c->renormalize != 1) return fail(MOE_ERR_INVALID_ARG, "renormalize must be 0 or 1");
  if (c->has_shared_expert != 0 && c->has_shared_expert != 1)
    return fail(MOE_ERR_INVALID_ARG, "has_shared_expert must be 0 or 1");
  if (c->add_residual != 0 && c->add_residual != 1) return fail(MOE_ERR_INVALID_ARG, "add_residual must be 0 or 1");
  if (!w->router_w) return fail(MOE_ERR_INVALID_ARG, "router_w must not be NULL");
  const int n_records = c->num_experts + c->has_shared_expert;
  if (c->residency == MOE_RESIDENCY_FULL) {
    if (!w->slot_pool || !w->expert_to_slot)
      return fail(MOE_ERR_INVALID_ARG, "full residency needs slot_pool and expert_to_slot");
    if (w->host_backing) return fail(MOE_ERR_INVALID_ARG, "full residency takes no host_backing");
    if (c->num_slots < 1) return fail(MOE_ERR_INVALID_ARG, "num_slots=%d", c->num_slots);
    if (reinterpret_cast<uintptr_t>(w->slot_pool) % 256)
      return fail(MOE_ERR_INVALID_ARG, "slot_pool must be 256-byte aligned");
  } else if (c->residency == MOE_RESIDENCY_PARTIAL) {
    if (w->slot_pool || w->expert_to_slot)
      return fail(MOE_ERR_INVALID_ARG, "partial residency owns its pool: slot_pool/expert_to_slot must be NULL");
    if (!w->host_backing) return fail(MOE_ERR_INVALID_ARG, "partial residency needs host_backing");
    if (c->num_slots < 1 || c->num_slots > n_records)
      return fail(MOE_ERR_INVALID_ARG, "num_slots=%d out of 1..%d", c->num_slots, n_records);
    if (c->num_slots < c->top_k + c->has_shared_expert)
      return fail(MOE_ERR_CAPACITY, "num_slots=%d cannot hold one token's %d experts", c->num_slots,
                  c->top_k + c->has_shared_expert);
    if (c->spare_slots < 0 || c->spare_slots > n_records)
      return fail(MOE_ERR_INVALID_ARG, "spare_slots=%d out of 0..%d", c->spare_slots, n_records);
    if (c->staging_records < 0 || c->staging_records > 64)
      return fail(MOE_ERR_INVALID_ARG, "staging_records=%d out of 0..64", c->staging_records);
    if (c->cache_policy < MOE_POLICY_LRU || c->cache_policy > MOE_POLICY_LRU_FREQ)
      return fail(MOE_ERR_INVALID_ARG, "cache_policy=%d unknown", c->cache_policy);
  } else {
    return fail(MOE_ERR_INVALID_ARG, "residency=%d unknown", c->residency);
  }
  return MOE_OK;
}

template <typename T>
T* carve(char*& p, size_t count) {
  T* r = reinterpret_cast<T*>(p);
  p += align256(count * sizeof(T));
  return r;
}

size_t workspace_bytes(const moe_layer_config_t& c) {
  const size_t T = c.max_tokens, k = c.top_k, E = c.num_experts, H = c.hidden, I = c.intermediate;
  const size_t nchunks = (T + moe::kRouteChunkTokens - 1) / moe::kRouteChunkTokens;
  const size_t P = T * k + T;  // sorted positions incl. the shared segment
  size_t b = 0;
  b += align256(moe::kRouterSplitMax * T * E * 4);  // logits (partial planes on the large path)
  b += align256(std::min<size_t>(T, moe::kSmallRouteMaxT) * E * 16 * 4);  // logit partials
  b += 2 * align256(T * k * 4);         // ids, wts
  b += 2 * align256(nchunks * E * 4);   // chunk_hist, chunk_base
  b += align256(E * 4);                 // counts
  b += align256((E + 1) * 4);           // offsets
  b += 2 * align256(T * k * 4);         // perm, inv_perm
  b += 3 * align256((E + 1) * 4);       // segments
  b += 4 * align256(4);                 // num_seg, ticket, err, pad
  b += align256(P * I * 2);             // h
  b += align256(P * H * 4);             // ypart
  if (H % 64 == 0 && I % 64 == 0) b += align256(P * H * 2);  // tokens in sorted order (GEMM path)
  b += 2 * align256(T * H * 2);         // x/out staging
  b += align256(T * k * 4) * 2;         // ids/w staging
  b += align256(2048 * 4);              // megakernel counters
  b += align256(64 * 4);                // batch-1 decode epoch counters
  b += align256(kTraceCtas * moe::kTraceStamps * 8);  // phase trace
  b += align256(2 * 1024 * moe::kGemmStats * 8);  // GEMM wait counters (two launches)
  return b;
}

}  // namespace

extern "C" {

int32_t moe_abi_version(void) { return MOE_ABI_VERSION; }

size_t moe_record_bytes(int32_t hidden, int32_t intermediate, int32_t group_size) {
  return moe_record_bytes_zp(hidden, intermediate, group_size, 0);
}

size_t moe_record_bytes_zp(int32_t hidden, int32_t intermediate, int32_t group_size, int32_t zero_points) {
  Layout L;
  if ((zero_points != 0 && zero_points != 1) || !record_layout(hidden, intermediate, group_size, zero_points != 0, &L))
    return 0;
  return L.record;
}

moe_status_t moe_record_section(int32_t hidden, int32_t intermediate, int32_t group_size, int32_t section,
                                size_t* offset, size_t* bytes) {
  Layout L;
  if (!record_layout(hidden, intermediate, group_size, true, &L)) return fail(MOE_ERR_INVALID_ARG, "invalid shape");
  if (section < 0 || section > 8) return fail(MOE_ERR_INVALID_ARG, "section %d out of 0..8", section);
  if (offset) *offset = L.off[section];
  if (bytes) *bytes = L.size[section];
  return MOE_OK;
}

const char* moe_layer_last_error(const moe_layer_t* layer) {
  (void)layer;
  return g_last_error.c_str();
}

moe_status_t moe_layer_create(const moe_layer_config_t* config, const moe_layer_weights_t* weights,
                              moe_layer_t** out) {
  if (!out) return fail(MOE_ERR_INVALID_ARG, "out must not be NULL");
  *out = nullptr;
  moe_status_t st = validate(config, weights);
  if (st != MOE_OK) return st;
  moe_layer* L = new (std::nothrow) moe_layer();
  if (!L) return fail(MOE_ERR_OOM, "host allocation failed");
  L->cfg = *config;
  L->w = *weights;
  record_layout(config->hidden, config->intermediate, config->group_size, config->zero_points != 0, &L->lay);
  L->variant = config->zero_points != 0 || config->group_size == 32 || weights->shared_gate != nullptr;
  L->n_records = config->num_experts + config->has_shared_expert;
  const char* pdl_env = getenv("MOE_PDL");
  L->pdl = !(pdl_env && pdl_env[0] == '0');
  const char* d1_env = getenv("MOE_DECODE1");
  L->decode1 = !(d1_env && d1_env[0] == '0');
  const char* mk_env = getenv("MOE_MEGAKERNEL");
  L->megakernel = !(mk_env && mk_env[0] == '0');
  if (const char* mt = getenv("MOE_MEGAKERNEL_MAX_T"))
    L->megakernel_max_tokens = std::max(1, std::min(moe::kSmallRouteMaxT, atoi(mt)));
  // probed here, at create time, so that no capture sees a rejected launch
  L->decode_pdl = L->pdl && moe::decode_pdl_supported();
  cudaError_t e = cudaGetDevice(&L->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&L->num_sms, cudaDevAttrMultiProcessorCount, L->device);
  if (e != cudaSuccess) {
    delete L;
    return cuda_fail(e, "device query");
  }
  const size_t wsb = workspace_bytes(L->cfg);
  e = cudaMalloc(&L->ws, wsb);
  if (e != cudaSuccess) {
    delete L;
    cudaGetLastError();
    return fail(MOE_ERR_OOM, "workspace allocation of %zu bytes failed: %s", wsb, cudaGetErrorString(e));
  }
  {
    const size_t T = L->cfg.max_tokens, k = L->cfg.top_k, E = L->cfg.num_experts;
    const size_t H = L->cfg.hidden, I = L->cfg.intermediate;
    const size_t nchunks = (T + moe::kRouteChunkTokens - 1) / moe::kRouteChunkTokens;
    const size_t P = T * k + T;
    char* p = static_cast<char*>(L->ws);
    L->logits = carve<float>(p, moe::kRouterSplitMax * T * E);
    L->logit_part = carve<float>(p, std::min<size_t>(T, moe::kSmallRouteMaxT) * E * 16);
    L->ids = carve<int32_t>(p, T * k);
    L->wts = carve<float>(p, T * k);
    L->chunk_hist = carve<int32_t>(p, nchunks * E);
    L->chunk_base = carve<int32_t>(p, nchunks * E);
    L->counts = carve<int32_t>(p, E);
    L->offsets = carve<int32_t>(p, E + 1);
    L->perm = carve<int32_t>(p, T * k);
    L->inv_perm = carve<int32_t>(p, T * k);
    L->seg_expert = carve<int32_t>(p, E + 1);
    L->seg_start = carve<int32_t>(p, E + 1);
    L->seg_count = carve<int32_t>(p, E + 1);
    L->num_seg = carve<int32_t>(p, 1);
    L->ticket = carve<uint32_t>(p, 1);
    L->err = carve<uint32_t>(p, 1);
    carve<uint32_t>(p, 1);
    L->hbuf = carve<__half>(p, P * I);
    L->ypart = carve<float>(p, P * H);
    if (H % 64 == 0 && I % 64 == 0) L->xs = carve<__half>(p, P * H);
    L->x_stage = carve<__half>(p, T * H);
    L->out_stage = carve<__half>(p, T * H);
    L->ids_stage = carve<int32_t>(p, T * k);
    L->w_stage = carve<float>(p, T * k);
    L->ctr = carve<uint32_t>(p, 2048);
    L->ctr1 = carve<uint32_t>(p, 64);
    unsigned long long* tr = carve<unsigned long long>(p, 1024 * moe::kTraceStamps);
    const char* tr_env = getenv("MOE_TRACE");
    if (tr_env && tr_env[0] == '1') L->trace = tr;
    unsigned long long* gs = carve<unsigned long long>(p, 2 * 1024 * moe::kGemmStats);
    const char* gs_env = getenv("MOE_GEMM_STATS");
    if (gs_env && gs_env[0] == '1') L->gemm_stats = gs;
  }
  // zero the small control words (ticket, error word, segment count)
  e = cudaMemset(L->num_seg, 0, 4 * 256);
  if (e == cudaSuccess) e = cudaMemset(L->ctr, 0, 2048 * 4);
  if (e == cudaSuccess) e = cudaMemset(L->ctr1, 0, 64 * 4);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    cudaFree(L->ws);
    delete L;
    return cuda_fail(e, "workspace init");
  }
  {
    const char* gm = getenv("MOE_GEMM_MIN_TOKENS");
    if (gm) L->gemm_min_tokens = atoi(gm);
    const int H = config->hidden, I = config->intermediate;
    const size_t P = (size_t)config->max_tokens * (config->top_k + 1);
    L->gemm_ok = (H % 64 == 0) && (I % 64 == 0) && P < (1u << 31) && L->xs &&
                 moe::encode_rows_map(&L->h_map, L->hbuf, I, (int)P, moe::gemm_tile_n()) &&
                 moe::encode_rows_map(&L->xs_map, L->xs, H, (int)P, moe::gemm_tile_n());
    // GEMV work items of about 64 KB of codes for both matrices' passes:
    // two quantisation groups per consumer warp amortise the per-item work
    // (MOE_GEMV_ITEM_BYTES overrides, for tuning)
    int item_bytes = 65536;
    if (const char* ib = getenv("MOE_GEMV_ITEM_BYTES")) item_bytes = std::max(4096, std::min(131072, atoi(ib)));
    L->dec_pg = moe::plan_tcgemv(I, H, config->group_size, true, item_bytes, config->zero_points != 0);
    L->dec_pd = moe::plan_tcgemv(H, I, config->group_size, false, item_bytes, config->zero_points != 0);
    if (config->residency == MOE_RESIDENCY_FULL) {
      const uint8_t* pool = static_cast<const uint8_t*>(weights->slot_pool);
      moe::encode_pool_maps(L, pool, config->num_slots, &L->pool_maps);
    }
  }
  if (config->residency == MOE_RESIDENCY_PARTIAL) {
    st = moe::residency_create(L->cfg, L->lay.record, L->n_records, weights->host_backing, &L->res);
    if (st != MOE_OK) {
      cudaFree(L->ws);
      delete L;
      return fail(st, "%s", moe::residency_last_error());
    }
  }
  *out = L;
  return MOE_OK;
}

moe_status_t moe_layer_destroy(moe_layer_t* layer) {
  if (!layer) return MOE_OK;
  for (cudaEvent_t& ev : layer->ev)
    if (ev) cudaEventDestroy(ev);
  if (layer->res) moe::residency_destroy(layer->res);
  if (layer->ws) cudaFree(layer->ws);
  delete layer;
  return MOE_OK;
}

}  // extern "C"

namespace {

}  // namespace

namespace moe {

moe_status_t set_error(moe_status_t st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

// Gate/up + SwiGLU and down over the experts of the given segment list;
// pool/e2s/num_slots select the record table.
bool encode_pool_maps(const moe_layer* L, const uint8_t* pool, int num_slots, CodeMaps* maps) {
  const int H = L->cfg.hidden, I = L->cfg.intermediate;
  const size_t rec = L->lay.record;
  // GEMM: gate/up tiles take 64 rows of each matrix, down tiles 128 rows
  maps->valid = L->gemm_ok && encode_codes_map(&maps->gate, pool + L->lay.off[0], H, I, num_slots, rec, 64) &&
                encode_codes_map(&maps->up, pool + L->lay.off[1], H, I, num_slots, rec, 64) &&
                encode_codes_map(&maps->down, pool + L->lay.off[2], I, H, num_slots, rec, 128);
  // GEMV: one box row per item row
  maps->tvalid = encode_tcgemv_map(&maps->tgate, pool + L->lay.off[0], H, I, num_slots, rec, L->dec_pg.rb) &&
                 encode_tcgemv_map(&maps->tup, pool + L->lay.off[1], H, I, num_slots, rec, L->dec_pg.rb) &&
                 encode_tcgemv_map(&maps->tdown, pool + L->lay.off[2], I, H, num_slots, rec, L->dec_pd.rb);
  return maps->valid || maps->tvalid;
}

namespace {

// Tensor-core path: gate/up + SwiGLU GEMM, then the down GEMM.
moe_status_t enqueue_gemm(moe_layer* L, const __half* x, int T, cudaStream_t s, const uint8_t* pool,
                          const int32_t* e2s, int num_slots, const SegPtrs& seg, const CodeMaps* maps) {
  const moe_layer_config_t& c = L->cfg;
  const int H = c.hidden, I = c.intermediate, k = c.top_k, G = c.group_size;
  // the tokens in expert-sorted order, so that every token tile is one 2-D box
  const int rows = T * k + (c.has_shared_expert ? T : 0);
  cudaError_t e = launch_gather_rows(x, L->xs, L->perm, T * k, k, rows, H, L->num_sms * 4, s, L->pdl);
  if (e != cudaSuccess) return cuda_fail(e, "token gather launch");
  GemmArgs ga = {};
  ga.pool = pool;
  ga.record_bytes = (long long)L->lay.record;
  ga.expert_to_slot = e2s;
  ga.num_slots = num_slots;
  ga.s_off0 = L->lay.off[3];
  ga.s_off1 = L->lay.off[4];
  ga.N = I;
  ga.K = H;
  ga.G = G;
  ga.ng = (H + G - 1) / G;
  ga.zp = L->lay.zp ? 1 : 0;
  ga.z_off0 = L->lay.off[6];
  ga.z_off1 = L->lay.off[7];
  ga.num_seg = seg.num_seg;
  ga.seg_expert = seg.seg_expert;
  ga.seg_start = seg.seg_start;
  ga.seg_count = seg.seg_count;
  ga.perm = L->perm;
  ga.Tk = T * k;
  ga.k = k;
  ga.h_out = L->hbuf;
  ga.y_out = nullptr;
  ga.err = L->err;
  ga.stats = L->gemm_stats;
  e = launch_gemm(true, maps->gate, maps->up, L->xs_map, ga, L->num_sms, s, L->pdl);
  if (e != cudaSuccess) return cuda_fail(e, "gate/up GEMM launch");
  if (L->profiling) prof_record(L->ev[2], s);
  GemmArgs gb = ga;
  gb.s_off0 = L->lay.off[5];
  gb.s_off1 = L->lay.off[5];
  gb.z_off0 = L->lay.off[8];
  gb.z_off1 = L->lay.off[8];
  gb.N = H;
  gb.K = I;
  gb.ng = (I + G - 1) / G;
  gb.h_out = nullptr;
  gb.y_out = L->ypart;
  gb.stats = L->gemm_stats ? L->gemm_stats + (size_t)L->num_sms * kGemmStats : nullptr;
  e = launch_gemm(false, maps->down, maps->down, L->h_map, gb, L->num_sms, s, L->pdl);
  if (e != cudaSuccess) return cuda_fail(e, "down GEMM launch");
  if (L->profiling) prof_record(L->ev[3], s);
  return MOE_OK;
}

}  // namespace

moe_status_t enqueue_experts(moe_layer* L, const __half* x, int T, cudaStream_t s, const uint8_t* pool,
                             const int32_t* e2s, int num_slots, const SegPtrs& seg, int max_seg,
                             const CodeMaps* maps) {
  const moe_layer_config_t& c = L->cfg;
  const int H = c.hidden, I = c.intermediate, k = c.top_k, G = c.group_size;
  if (L->gemm_ok && maps && maps->valid && T >= L->gemm_min_tokens)
    return enqueue_gemm(L, x, T, s, pool, e2s, num_slots, seg, maps);

  if (!maps || !maps->tvalid) return fail(MOE_ERR_UNSUPPORTED, "no GEMV tensor maps for this pool");
  const TcGemvPlan& pg = L->dec_pg;
  const TcGemvPlan& pd = L->dec_pd;
  TcGemvLaunch p = {};
  TcGemvArgs& a = p.a;
  a.pool = pool;
  a.record_bytes = (long long)L->lay.record;
  a.expert_to_slot = e2s;
  a.num_slots = num_slots;
  a.s_off0 = L->lay.off[3];
  a.s_off1 = L->lay.off[4];
  a.N = I;
  a.K = H;
  a.G = G;
  a.ng = (H + G - 1) / G;
  a.rb = pg.rb;
  a.rt = pg.rt;
  a.kparts = pg.kparts;
  a.lkparts = pg.lkparts;
  a.nbox = pg.nbox;
  a.code_mat_bytes = pg.code_mat_bytes;
  a.sstride = pg.sstride;
  a.zp = L->lay.zp ? 1 : 0;
  a.z_off0 = L->lay.off[6];
  a.z_off1 = L->lay.off[7];
  a.zstride = pg.zstride;
  a.seg_expert = seg.seg_expert;
  a.seg_start = seg.seg_start;
  a.seg_count = seg.seg_count;
  a.act = x;
  a.act_gather = 1;
  a.perm = L->perm;
  a.Tk = T * k;
  a.k = k;
  a.h_out = L->hbuf;
  a.y_out = nullptr;
  a.err = L->err;
  p.m0 = maps->tgate;
  p.m1 = maps->tup;
  p.num_seg = seg.num_seg;
  p.slot_bytes = pg.slot_bytes;
  // token columns: a segment holds at most T tokens
  p.ns = T <= 2 ? 2 : (T <= 4 ? 4 : 8);
  p.bs_chunks = ((H / 32) + 1) & ~1;
  p.cs_groups = a.ng;
  p.stages = 0;
  {
    const size_t fixed = tcgemv_smem_bytes(p);
    if (fixed + 2 * (size_t)p.slot_bytes > kSmemBudget) return fail(MOE_ERR_UNSUPPORTED, "GEMV item too large");
    p.stages = (int)std::min<size_t>(kDecodeMaxStages, (kSmemBudget - fixed) / p.slot_bytes);
  }
  const int nrb_g = (I + pg.rb - 1) / pg.rb;
  const int grid_g = std::max(1, std::min(L->num_sms, max_seg * nrb_g));
  cudaError_t e = launch_tcgemv(p, true, grid_g, s, L->pdl);
  if (e != cudaSuccess) return cuda_fail(e, "gate/up launch");
  if (L->profiling) prof_record(L->ev[2], s);

  TcGemvLaunch q = p;
  TcGemvArgs& b = q.a;
  b.s_off0 = L->lay.off[5];
  b.s_off1 = 0;
  b.N = H;
  b.K = I;
  b.ng = (I + G - 1) / G;
  b.rb = pd.rb;
  b.rt = pd.rt;
  b.kparts = pd.kparts;
  b.lkparts = pd.lkparts;
  b.nbox = pd.nbox;
  b.code_mat_bytes = pd.code_mat_bytes;
  b.sstride = pd.sstride;
  b.z_off0 = L->lay.off[8];
  b.z_off1 = 0;
  b.zstride = pd.zstride;
  b.act = L->hbuf;
  b.act_gather = 0;
  b.h_out = nullptr;
  b.y_out = L->ypart;
  q.m0 = maps->tdown;
  q.m1 = maps->tdown;
  q.slot_bytes = pd.slot_bytes;
  q.bs_chunks = ((I / 32) + 1) & ~1;
  q.cs_groups = b.ng;
  q.stages = 0;
  {
    const size_t fixed = tcgemv_smem_bytes(q);
    if (fixed + 2 * (size_t)q.slot_bytes > kSmemBudget) return fail(MOE_ERR_UNSUPPORTED, "GEMV item too large");
    q.stages = (int)std::min<size_t>(kDecodeMaxStages, (kSmemBudget - fixed) / q.slot_bytes);
  }
  const int nrb_d = (H + pd.rb - 1) / pd.rb;
  const int grid_d = std::max(1, std::min(L->num_sms, max_seg * nrb_d));
  e = launch_tcgemv(q, false, grid_d, s, L->pdl);
  if (e != cudaSuccess) return cuda_fail(e, "down launch");
  if (L->profiling) prof_record(L->ev[3], s);
  return MOE_OK;
}

// Single-launch decode (routing, experts, combine) for T <= kSmallRouteMaxT.
// Returns MOE_ERR_UNSUPPORTED (without launching) when the shapes have no
// megakernel variant, so the caller takes the multi-kernel path.
moe_status_t enqueue_decode(moe_layer* L, const __half* x, int T, __half* out, int32_t* ids_user, float* w_user,
                            cudaStream_t s) {
  const moe_layer_config_t& c = L->cfg;
  const int H = c.hidden, I = c.intermediate, E = c.num_experts, k = c.top_k, G = c.group_size;
  const TcGemvPlan& pg = L->dec_pg;
  const TcGemvPlan& pd = L->dec_pd;
  if (!L->pool_maps.tvalid || (H + pd.rb - 1) / pd.rb > 2048 - 2 - (E + 1)) return MOE_ERR_UNSUPPORTED;
  DecodeArgs a = {};
  RouteArgs& r = a.r;
  r.x = x;
  r.wr = L->w.router_w;
  r.bias = L->w.router_bias;
  r.T = T;
  r.H = H;
  r.E = E;
  r.k = k;
  r.renorm = c.renormalize;
  r.has_shared = c.has_shared_expert;
  r.logits = L->logits;
  r.logit_part = L->logit_part;
  r.ids = L->ids;
  r.w = L->wts;
  r.ids_user = ids_user;
  r.w_user = w_user;
  r.counts = L->counts;
  r.offsets = L->offsets;
  r.perm = L->perm;
  r.inv_perm = L->inv_perm;
  r.seg_expert = L->seg_expert;
  r.seg_start = L->seg_start;
  r.seg_count = L->seg_count;
  r.num_seg = L->num_seg;
  r.err = L->err;
  TcGemvArgs& g = a.g;
  g.pool = static_cast<const uint8_t*>(L->w.slot_pool);
  g.record_bytes = (long long)L->lay.record;
  g.expert_to_slot = L->w.expert_to_slot;
  g.num_slots = c.num_slots;
  g.s_off0 = L->lay.off[3];
  g.s_off1 = L->lay.off[4];
  g.N = I;
  g.K = H;
  g.G = G;
  g.ng = (H + G - 1) / G;
  g.rb = pg.rb;
  g.rt = pg.rt;
  g.kparts = pg.kparts;
  g.lkparts = pg.lkparts;
  g.nbox = pg.nbox;
  g.code_mat_bytes = pg.code_mat_bytes;
  g.sstride = pg.sstride;
  g.act = x;
  g.act_gather = 1;
  g.Tk = T * k;
  g.k = k;
  g.h_out = L->hbuf;
  g.err = L->err;
  TcGemvArgs& d = a.d;
  d = g;
  d.s_off0 = L->lay.off[5];
  d.s_off1 = 0;
  d.N = H;
  d.K = I;
  d.ng = (I + G - 1) / G;
  d.rb = pd.rb;
  d.rt = pd.rt;
  d.kparts = pd.kparts;
  d.lkparts = pd.lkparts;
  d.nbox = pd.nbox;
  d.code_mat_bytes = pd.code_mat_bytes;
  d.sstride = pd.sstride;
  d.act = L->hbuf;
  d.act_gather = 0;
  d.h_out = nullptr;
  d.y_out = L->ypart;
  a.tm_gate = L->pool_maps.tgate;
  a.tm_up = L->pool_maps.tup;
  a.tm_down = L->pool_maps.tdown;
  a.out = out;
  a.x_res = c.add_residual ? x : nullptr;
  a.has_shared = c.has_shared_expert;
  a.ctr = L->ctr;
  a.trace = L->trace;
  a.slot_bytes = std::max(pg.slot_bytes, pd.slot_bytes);
  // token columns per tile: the segment of an expert holds at most T tokens
  a.ns = T <= 2 ? 2 : (T <= 4 ? 4 : 8);
  const int kmax = std::max(H, I);
  a.bs_chunks = ((kmax / 32) + 1) & ~1;
  a.cs_groups = (kmax + G - 1) / G;
  const size_t fixed = decode_smem_bytes(a, 0);
  if (fixed + 2 * (size_t)a.slot_bytes > kSmemBudget) return MOE_ERR_UNSUPPORTED;
  a.stages = (int)std::min<size_t>(kDecodeMaxStages, (kSmemBudget - fixed) / a.slot_bytes);
  if (L->profiling) prof_record(L->ev[0], s);
  if (L->trace) cudaMemsetAsync(L->trace, 0, (size_t)L->num_sms * moe::kTraceStamps * 8, s);
  cudaError_t e = launch_decode(a, L->num_sms, s, L->pdl && L->decode_pdl);
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  if (L->profiling) prof_record(L->ev[4], s);
  L->last_single = true;
  return MOE_OK;
}

void fill_decode1_args(moe_layer* L, const __half* x, __half* out, int32_t* ids_user, float* w_user,
                       Decode1Args* ap) {
  const moe_layer_config_t& c = L->cfg;
  const int H = c.hidden, I = c.intermediate, E = c.num_experts, k = c.top_k;
  const int grid = L->num_sms;
  Decode1Args& a = *ap;
  a = Decode1Args{};
  RouteArgs& r = a.r;
  r.x = x;
  r.wr = L->w.router_w;
  r.bias = L->w.router_bias;
  r.T = 1;
  r.H = H;
  r.E = E;
  r.k = k;
  r.renorm = c.renormalize;
  r.has_shared = c.has_shared_expert;
  r.logits = L->logits;
  r.ids = L->ids;
  r.w = L->wts;
  r.ids_user = ids_user;
  r.w_user = w_user;
  r.counts = L->counts;
  r.offsets = L->offsets;
  r.perm = L->perm;
  r.inv_perm = L->inv_perm;
  r.seg_expert = L->seg_expert;
  r.seg_start = L->seg_start;
  r.seg_count = L->seg_count;
  r.num_seg = L->num_seg;
  r.err = L->err;
  a.pool = static_cast<const uint8_t*>(L->w.slot_pool);
  a.record_bytes = (long long)L->lay.record;
  a.expert_to_slot = L->w.expert_to_slot;
  a.num_slots = c.num_slots;
  for (int i = 0; i < 3; ++i) {
    a.off_q[i] = (long long)L->lay.off[i];
    a.off_s[i] = (long long)L->lay.off[3 + i];
  }
  a.I = I;
  a.G = c.group_size;
  a.h = L->hbuf;
  a.out = out;
  a.x_res = c.add_residual ? x : nullptr;
  a.ctr = L->ctr1;
  a.ctr_mod = (uint32_t)grid * 1024u;
  a.trace = L->trace;
  a.nseg_max = k + c.has_shared_expert;
  a.max_units_g = decode1_max_tiles(a.nseg_max, I, grid);
  a.max_units_d = (H / 16 + grid - 1) / grid;
  a.max_rows_rt = (E + grid - 1) / grid;
}

moe_status_t enqueue_decode1(moe_layer* L, const __half* x, __half* out, int32_t* ids_user, float* w_user,
                             cudaStream_t s) {
  const int grid = L->num_sms;
  if (grid < 1) return MOE_ERR_UNSUPPORTED;
  Decode1Args a;
  fill_decode1_args(L, x, out, ids_user, w_user, &a);
  if (decode1_smem_bytes(a) == 0) return MOE_ERR_UNSUPPORTED;
  if (L->profiling) prof_record(L->ev[0], s);
  // (every CTA rewrites its stamps on every launch: no clearing launch)
  cudaError_t e = launch_decode1(a, grid, s, L->pdl && L->decode_pdl);
  if (e != cudaSuccess) return cuda_fail(e, "batch-1 decode launch");
  if (L->profiling) prof_record(L->ev[4], s);
  L->last_single = true;
  return MOE_OK;
}

moe_status_t enqueue_combine(moe_layer* L, const __half* x, int T, __half* out, cudaStream_t s) {
  const moe_layer_config_t& c = L->cfg;
  CombineArgs ca = {};
  ca.ypart = L->ypart;
  ca.w = L->wts;
  ca.x = c.add_residual ? x : nullptr;
  ca.out = out;
  ca.T = T;
  ca.H = c.hidden;
  ca.k = c.top_k;
  ca.has_shared = c.has_shared_expert;
  ca.gate = L->w.shared_gate;
  ca.xin = x;
  cudaError_t e = launch_combine(ca, s, L->pdl);
  if (e != cudaSuccess) return cuda_fail(e, "combine launch");
  if (L->profiling) prof_record(L->ev[4], s);
  return MOE_OK;
}

}  // namespace moe

namespace {

moe_status_t enqueue_route(moe_layer* L, const __half* x, int T, int32_t* ids_user, float* w_user,
                           cudaStream_t s) {
  const moe_layer_config_t& c = L->cfg;
  moe::RouteArgs ra = {};
  ra.x = x;
  ra.wr = L->w.router_w;
  ra.bias = L->w.router_bias;
  ra.T = T;
  ra.H = c.hidden;
  ra.E = c.num_experts;
  ra.k = c.top_k;
  ra.renorm = c.renormalize;
  ra.has_shared = c.has_shared_expert;
  ra.logits = L->logits;
  ra.ids = L->ids;
  ra.w = L->wts;
  ra.ids_user = ids_user;
  ra.w_user = w_user;
  ra.chunk_hist = L->chunk_hist;
  ra.chunk_base = L->chunk_base;
  ra.counts = L->counts;
  ra.offsets = L->offsets;
  ra.perm = L->perm;
  ra.inv_perm = L->inv_perm;
  ra.seg_expert = L->seg_expert;
  ra.seg_start = L->seg_start;
  ra.seg_count = L->seg_count;
  ra.num_seg = L->num_seg;
  ra.ticket = L->ticket;
  ra.err = L->err;
  const bool small = T <= moe::kSmallRouteMaxT && (size_t)T * c.hidden * 2 <= 200 * 1024;
  ra.trace = small ? L->trace : nullptr;
  // (tracing only: the routing CTAs that do not finish leave their finish
  // stamps at zero)
  if (ra.trace) cudaMemsetAsync(L->trace, 0, (size_t)std::min(c.num_experts, kTraceCtas) * moe::kTraceStamps * 8, s);
  if (!small) ra.nsplit = moe::router_split(T, c.num_experts, c.hidden, L->num_sms);
  if (L->profiling) prof_record(L->ev[0], s);
  L->last_single = false;
  cudaError_t e = small ? moe::launch_route_small(ra, s, L->pdl) : moe::launch_route_large(ra, s, L->pdl);
  if (e != cudaSuccess) return cuda_fail(e, "routing launch");
  if (L->profiling) prof_record(L->ev[1], s);
  return MOE_OK;
}

}  // namespace

extern "C" {

moe_status_t moe_layer_forward(moe_layer_t* layer, const void* x, int32_t T, void* out, int32_t* topk_ids,
                               float* topk_w, void* stream) {
  if (!layer) return fail(MOE_ERR_INVALID_ARG, "layer must not be NULL");
  if (T < 0 || T > layer->cfg.max_tokens)
    return fail(MOE_ERR_INVALID_ARG, "T=%d out of 0..max_tokens=%d", T, layer->cfg.max_tokens);
  if (T == 0) return MOE_OK;
  if (!x || !out) return fail(MOE_ERR_INVALID_ARG, "x and out must not be NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const __half* xh = static_cast<const __half*>(x);
  __half* oh = static_cast<__half*>(out);
  // programmatic dependent launch only on explicitly created streams
  const bool pdl_saved = layer->pdl;
  if (s == nullptr) layer->pdl = false;
  // the single-launch decode kernels take the base format only (zero point
  // 8, G of 64 or 128, an ungated shared expert); variants use the
  // multi-kernel path
  if (layer->cfg.residency == MOE_RESIDENCY_FULL && layer->decode1 && !layer->variant && T == 1) {
    moe_status_t sd = moe::enqueue_decode1(layer, xh, oh, topk_ids, topk_w, s);
    if (sd != MOE_ERR_UNSUPPORTED) {
      layer->pdl = pdl_saved;
      if (sd != MOE_OK) return sd;
      layer->last_T = T;
      layer->stats.forward_calls += 1;
      layer->stats.tokens += (uint64_t)T;
      return MOE_OK;
    }
  }
  if (layer->cfg.residency == MOE_RESIDENCY_FULL && layer->megakernel && !layer->variant &&
      T <= layer->megakernel_max_tokens) {
    moe_status_t sd = moe::enqueue_decode(layer, xh, T, oh, topk_ids, topk_w, s);
    if (sd != MOE_ERR_UNSUPPORTED) {
      layer->pdl = pdl_saved;
      if (sd != MOE_OK) return sd;
      layer->last_T = T;
      layer->stats.forward_calls += 1;
      layer->stats.tokens += (uint64_t)T;
      return MOE_OK;
    }
  }
  if (layer->res) {
    const cudaError_t e = moe::residency_before_route(layer->res, s);
    if (e != cudaSuccess) {
      layer->pdl = pdl_saved;
      return cuda_fail(e, "ordering after a prefetch guess");
    }
  }
  moe_status_t st = enqueue_route(layer, xh, T, topk_ids, topk_w, s);
  if (st != MOE_OK) {
    layer->pdl = pdl_saved;
    return st;
  }
  if (layer->cfg.residency == MOE_RESIDENCY_FULL) {
    const moe::SegPtrs seg = {layer->num_seg, layer->seg_expert, layer->seg_start, layer->seg_count};
    const int max_seg = std::min(layer->cfg.num_experts, T * layer->cfg.top_k) + layer->cfg.has_shared_expert;
    st = moe::enqueue_experts(layer, xh, T, s, static_cast<const uint8_t*>(layer->w.slot_pool),
                              layer->w.expert_to_slot, layer->cfg.num_slots, seg, max_seg, &layer->pool_maps);
    if (st == MOE_OK) st = moe::enqueue_combine(layer, xh, T, oh, s);
  } else {
    st = moe::residency_forward(layer->res, layer, xh, T, oh, s);
  }
  layer->pdl = pdl_saved;
  if (st != MOE_OK) return st;
  layer->last_T = T;
  layer->stats.forward_calls += 1;
  layer->stats.tokens += (uint64_t)T;
  return MOE_OK;
}

moe_status_t moe_layer_prefetch(moe_layer_t* layer, const void* x, int32_t T, void* stream) {
  if (!layer) return fail(MOE_ERR_INVALID_ARG, "layer must not be NULL");
  if (T < 0 || T > layer->cfg.max_tokens)
    return fail(MOE_ERR_INVALID_ARG, "T=%d out of 0..max_tokens=%d", T, layer->cfg.max_tokens);
  if (layer->cfg.residency == MOE_RESIDENCY_FULL || T == 0) return MOE_OK;
  if (!x) return fail(MOE_ERR_INVALID_ARG, "x must not be NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaStream_t side = moe::residency_side(layer->res);
  cudaEvent_t ready = moe::residency_input_event(layer->res);
  cudaError_t e = cudaEventRecord(ready, s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(side, ready, 0);
  if (e != cudaSuccess) return cuda_fail(e, "prefetch input dependency");
  // the guess is routed like a forward's tokens, without profiling events
  // and without a programmatic dependency on the side stream's last copy
  const bool pdl_saved = layer->pdl, prof_saved = layer->profiling;
  layer->pdl = false;
  layer->profiling = false;
  moe_status_t st = enqueue_route(layer, static_cast<const __half*>(x), T, nullptr, nullptr, side);
  layer->pdl = pdl_saved;
  layer->profiling = prof_saved;
  if (st != MOE_OK) return st;
  return moe::residency_prefetch(layer->res, layer, T);
}

moe_status_t moe_layer_forward_host(moe_layer_t* layer, const void* x_host, int32_t T, void* out_host,
                                    int32_t* topk_ids_host, float* topk_w_host, void* stream) {
  if (!layer) return fail(MOE_ERR_INVALID_ARG, "layer must not be NULL");
  if (T < 0 || T > layer->cfg.max_tokens)
    return fail(MOE_ERR_INVALID_ARG, "T=%d out of 0..max_tokens=%d", T, layer->cfg.max_tokens);
  if (T == 0) return MOE_OK;
  if (!x_host || !out_host) return fail(MOE_ERR_INVALID_ARG, "x_host and out_host must not be NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (T <= kInPlaceHostMaxT) {
    // page-locked host buffers with a device address (mapped): the kernels
    // read x and write the results in place over the host link, no staging
    // copies; any other buffer takes the staging path below
    const void* xd = mapped_device_ptr(x_host);
    void* od = mapped_device_ptr(out_host);
    void* idd = topk_ids_host ? mapped_device_ptr(topk_ids_host) : nullptr;
    void* wd = topk_w_host ? mapped_device_ptr(topk_w_host) : nullptr;
    if (xd && od && (!topk_ids_host || idd) && (!topk_w_host || wd))
      return moe_layer_forward(layer, xd, T, od, static_cast<int32_t*>(idd), static_cast<float*>(wd), stream);
  }
  const size_t xb = (size_t)T * layer->cfg.hidden * 2, kb = (size_t)T * layer->cfg.top_k * 4;
  cudaError_t e = cudaMemcpyAsync(layer->x_stage, x_host, xb, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(e, "x host->device");
  moe_status_t st = moe_layer_forward(layer, layer->x_stage, T, layer->out_stage,
                                      topk_ids_host ? layer->ids_stage : nullptr,
                                      topk_w_host ? layer->w_stage : nullptr, stream);
  if (st != MOE_OK) return st;
  e = cudaMemcpyAsync(out_host, layer->out_stage, xb, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess && topk_ids_host)
    e = cudaMemcpyAsync(topk_ids_host, layer->ids_stage, kb, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess && topk_w_host) e = cudaMemcpyAsync(topk_w_host, layer->w_stage, kb, cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return cuda_fail(e, "result device->host");
  return MOE_OK;
}

moe_status_t moe_layer_routing(const moe_layer_t* layer, int32_t* counts, int32_t* offsets, int32_t* perm,
                               int32_t* inv_perm, void* stream) {
  if (!layer) return fail(MOE_ERR_INVALID_ARG, "layer must not be NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t E = layer->cfg.num_experts, n = (size_t)layer->last_T * layer->cfg.top_k;
  cudaError_t e = cudaSuccess;
  if (counts) e = cudaMemcpyAsync(counts, layer->counts, E * 4, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess && offsets) e = cudaMemcpyAsync(offsets, layer->offsets, (E + 1) * 4, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess && perm && n) e = cudaMemcpyAsync(perm, layer->perm, n * 4, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess && inv_perm && n)
    e = cudaMemcpyAsync(inv_perm, layer->inv_perm, n * 4, cudaMemcpyDeviceToDevice, s);
  if (e != cudaSuccess) return cuda_fail(e, "routing copy");
  return MOE_OK;
}

moe_status_t moe_layer_sync(moe_layer_t* layer, void* stream) {
  if (!layer) return fail(MOE_ERR_INVALID_ARG, "layer must not be NULL");
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  uint32_t word = 0;
  e = cudaMemcpy(&word, layer->err, 4, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "error word read");
  if (word != 0u) {
    cudaMemset(layer->err, 0, 4);
    cudaDeviceSynchronize();
    if (word == 1) return fail(MOE_ERR_TIMEOUT, "a device-side wait gave up (error word %u)", word);
    return fail(MOE_ERR_INTERNAL, "device-side check failed (error word %u)", word);
  }
  return MOE_OK;
}

moe_status_t moe_layer_set_profiling(moe_layer_t* layer, int32_t enable) {
  if (!layer) return fail(MOE_ERR_INVALID_ARG, "layer must not be NULL");
  if (enable && !layer->ev[0]) {
    for (cudaEvent_t& ev : layer->ev) {
      cudaError_t e = cudaEventCreate(&ev);
      if (e != cudaSuccess) return cuda_fail(e, "event create");
    }
  }
  layer->profiling = enable != 0;
  return MOE_OK;
}

moe_status_t moe_layer_get_profile(moe_layer_t* layer, moe_layer_profile_t* p) {
  if (!layer || !p) return fail(MOE_ERR_INVALID_ARG, "layer and profile must not be NULL");
  if (!layer->ev[0]) return fail(MOE_ERR_INVALID_ARG, "profiling was never enabled");
  cudaError_t e = cudaEventSynchronize(layer->ev[4]);
  float ms[4] = {0, 0, 0, 0}, tot = 0;
  if (!layer->last_single)
    for (int i = 0; i < 4 && e == cudaSuccess; ++i) e = cudaEventElapsedTime(&ms[i], layer->ev[i], layer->ev[i + 1]);
  if (e == cudaSuccess) e = cudaEventElapsedTime(&tot, layer->ev[0], layer->ev[4]);
  int32_t nseg = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&nseg, layer->num_seg, 4, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "profile read");
  p->route_ms = ms[0];
  p->gate_up_ms = ms[1];
  p->down_ms = ms[2];
  p->combine_ms = ms[3];
  p->total_ms = tot;
  p->active_experts = nseg - layer->cfg.has_shared_expert;
  p->tokens = layer->last_T;
  p->single_launch = layer->last_single ? 1 : 0;
  return MOE_OK;
}

moe_status_t moe_layer_get_trace(moe_layer_t* layer, uint64_t* stamps, int32_t max_stamps, int32_t* n_stamps) {
  if (!layer || !stamps || !n_stamps) return fail(MOE_ERR_INVALID_ARG, "layer, stamps and n_stamps must not be NULL");
  if (!layer->trace) return fail(MOE_ERR_INVALID_ARG, "tracing is off (set MOE_TRACE=1 before create)");
  const int n = std::min(max_stamps, kTraceCtas * moe::kTraceStamps);
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(stamps, layer->trace, (size_t)n * 8, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "trace read");
  *n_stamps = n;
  return MOE_OK;
}

moe_status_t moe_layer_get_gemm_stats(moe_layer_t* layer, uint64_t* values, int32_t max_values, int32_t* n_values) {
  if (!layer || !values || !n_values) return fail(MOE_ERR_INVALID_ARG, "layer, values and n_values must not be NULL");
  if (!layer->gemm_stats) return fail(MOE_ERR_INVALID_ARG, "GEMM counters are off (set MOE_GEMM_STATS=1 before create)");
  const int n = std::min(max_values, 2 * layer->num_sms * moe::kGemmStats);
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(values, layer->gemm_stats, (size_t)n * 8, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "GEMM counter read");
  *n_values = n;
  return MOE_OK;
}

moe_status_t moe_layer_get_stats(const moe_layer_t* layer, moe_layer_stats_t* stats) {
  if (!layer || !stats) return fail(MOE_ERR_INVALID_ARG, "layer and stats must not be NULL");
  *stats = layer->stats;
  if (layer->res) moe::residency_fill_stats(layer->res, stats);
  return MOE_OK;
}

}  // extern "C"

// ---------------------------------------------------------------- internal
namespace moe {

cudaError_t ensure_smem_ptr(const void* kern, size_t bytes) {
  // The attribute applies to the device current when it is set, so the
  // record is kept per (device, kernel): a process that uses several GPUs
  // opts every one of them in.
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, size_t> set_bytes;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_pair(dev, kern);
  auto it = set_bytes.find(key);
  if (it != set_bytes.end() && it->second >= bytes) return cudaSuccess;
  if (bytes <= 48 * 1024 && it == set_bytes.end()) {
    set_bytes[key] = 48 * 1024;
    return cudaSuccess;
  }
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) set_bytes[key] = bytes;
  return e;
}

}  // namespace moe
