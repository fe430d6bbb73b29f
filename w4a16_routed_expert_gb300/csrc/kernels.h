// Internal launch interface between the runtime (moe_layer.cu) and the
// kernel files. Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace moe {

// Tokens per routing chunk of the multi-CTA routing path.
constexpr int kRouteChunkTokens = 32;
// Largest T handled by the fused single-launch routing kernel.
constexpr int kSmallRouteMaxT = 16;

// Routing workspace and outputs (all device pointers).
struct RouteArgs {
  const __half* x;      // [T][H]
  const float* wr;      // [E][H]
  const float* bias;    // [E] or nullptr
  int T, H, E, k;
  int renorm;
  int has_shared;
  float* logits;        // [T][E]
  int32_t* ids;         // [T][k] workspace copy
  float* w;             // [T][k] workspace copy
  int32_t* ids_user;    // [T][k] or nullptr
  float* w_user;        // [T][k] or nullptr
  int32_t* chunk_hist;  // [nchunks][E]
  int32_t* chunk_base;  // [nchunks][E]
  int32_t* counts;      // [E]
  int32_t* offsets;     // [E+1]
  int32_t* perm;        // [T*k]
  int32_t* inv_perm;    // [T*k]
  int32_t* seg_expert;  // [E+1]
  int32_t* seg_start;   // [E+1]
  int32_t* seg_count;   // [E+1]
  int32_t* num_seg;     // [1]
  uint32_t* ticket;     // [1], zero between launches
  uint32_t* err;        // [1]
};

// Grouped W4A16 GEMV over expert segments (decode regime).
struct GemvArgs {
  const uint8_t* pool;          // slot pool base
  long long record_bytes;
  const int32_t* expert_to_slot;
  int num_slots;
  long long q_off0, q_off1;     // code sections (gate, up) or (down, -)
  long long s_off0, s_off1;     // scale sections
  int N;                        // output rows per matrix
  int K;                        // reduction length
  int G;                        // group size
  int ng;                       // ceil(K / G)
  int lpr;                      // lanes per row (power of two, 4..32)
  int rb;                       // rows per work item (multiple of 8)
  const int32_t* num_seg;
  const int32_t* seg_expert;
  const int32_t* seg_start;
  const int32_t* seg_count;
  const __half* act;            // gate/up: x [T][K]; down: h [P][K]
  int act_gather;               // 1: row of sorted position p is x[perm[p] / k] (p < Tk) or x[p - Tk]
  const int32_t* perm;
  int Tk;                       // T * k
  int k;
  __half* h_out;                // DUAL: [P][N] FP16 at sorted positions
  float* y_out;                 // single: [Tk + T][N] FP32 at flat index f = perm[p] (p < Tk) or p
  int stages;
  uint32_t stage_bytes;
  uint32_t* err;
};

// Grouped W4A16 GEMM over expert segments (prefill regime, tensor cores).
struct GemmArgs {
  const uint8_t* pool;
  long long record_bytes;
  const int32_t* expert_to_slot;
  int num_slots;
  long long s_off0, s_off1;     // scale sections (gate, up) or (down, -)
  int N, K, G, ng;
  const int32_t* num_seg;
  const int32_t* seg_expert;
  const int32_t* seg_start;
  const int32_t* seg_count;
  const int32_t* perm;
  int Tk;
  int k;
  __half* h_out;                // DUAL: [P][N]
  float* y_out;                 // single: [Tk + T][N]
  uint32_t* err;
};

// Whole-layer decode megakernel (T <= kSmallRouteMaxT, full residency).
struct DecodeArgs {
  RouteArgs r;           // routing inputs and global outputs
  GemvArgs g;            // gate/up items (segment pointers are replaced in-kernel)
  GemvArgs d;            // down items
  __half* out;           // [T][H]
  const __half* x_res;   // residual input or nullptr
  int has_shared;
  uint32_t* ctr;         // zeroed counters: logits_done, final ticket, done_gu[E+1], done_dn[]
  int stages;
  uint32_t slot_bytes;   // ring slot size (max of the two item layouts)
};

// Tensor maps of the three code sections of a slot pool.
struct CodeMaps {
  CUtensorMap gate, up, down;
  bool valid;
};

struct CombineArgs {
  const float* ypart;   // [Tk + T][H]
  const float* w;       // [T][k]
  const __half* x;      // residual input or nullptr
  __half* out;          // [T][H]
  int T, H, k, has_shared;
};

// Launch shape of one grouped-GEMV launch, chosen on the host.
struct GemvPlan {
  int lpr;              // lanes per row
  int kch;              // 16-byte code chunks per lane per row
  int nt;               // token tile (activations held in registers)
  int rb;               // rows per work item
  uint32_t stage_bytes; // shared-memory bytes per pipeline stage
  int stages;           // pipeline depth
};

// Raise a kernel's dynamic shared-memory limit once per kernel (not per
// launch, so launches can be captured into CUDA graphs without attribute
// calls). Defined in moe_layer.cu.
cudaError_t ensure_smem_ptr(const void* kern, size_t bytes);
template <typename... KArgs>
cudaError_t ensure_smem(void (*kern)(KArgs...), size_t bytes) {
  return ensure_smem_ptr(reinterpret_cast<const void*>(kern), bytes);
}

// Launch with the programmatic-dependent-launch attribute when pdl is set.
template <typename... KArgs, typename... Args>
cudaError_t launch_ex(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                      Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

cudaError_t launch_route_small(const RouteArgs& a, cudaStream_t s, bool pdl);
cudaError_t launch_route_large(const RouteArgs& a, cudaStream_t s, bool pdl);
GemvPlan plan_gemv(int N, int K, int G, bool dual, int T);
bool gemv_plan_supported(const GemvPlan& p);
cudaError_t launch_gemv(const GemvArgs& a, bool dual, const GemvPlan& p, int grid, cudaStream_t s, bool pdl);
int gemv_kch(int K, int lpr);
int gemv_lanes_per_row(int K);
size_t gemv_smem_bytes(int stages, uint32_t stage_bytes);
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s, bool pdl);
size_t decode_smem_bytes(int stages, uint32_t slot_bytes);
bool decode_supported(int kg, int ntg, int kd, int ntd);
cudaError_t launch_decode(const DecodeArgs& a, int kg, int ntg, int kd, int ntd, int grid, cudaStream_t s);
cudaError_t launch_gemm(bool dual, const CUtensorMap& codes0, const CUtensorMap& codes1, const CUtensorMap& act,
                        const GemmArgs& a, int grid, cudaStream_t s, bool pdl);
size_t gemm_smem_bytes(bool dual);
bool encode_codes_map(CUtensorMap* tm, const void* pool_section, int K, int N, int num_slots, size_t record_bytes,
                      int box_rows);
bool encode_rows_map(CUtensorMap* tm, const void* base, int cols, int rows, int box_rows);
int gemm_tile_n();
int gemm_tile_k();

}  // namespace moe
