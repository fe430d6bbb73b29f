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
// Most K parts the large-batch router logits are split into (partial-logit
// planes in the logits workspace).
constexpr int kRouterSplitMax = 8;

// Routing workspace and outputs (all device pointers).
// global-timer stamps per CTA written by the traced single-launch decode:
// kTracePhases phase stamps, then two per work item (landed, computed) for
// the first kTraceItems items of consumer warp 0
constexpr int kTracePhases = 16;
constexpr int kTraceItems = 8;
constexpr int kTraceStamps = kTracePhases + 2 * kTraceItems;

struct RouteArgs {
  const __half* x;      // [T][H]
  const float* wr;      // [E][H]
  const float* bias;    // [E] or nullptr
  int T, H, E, k;
  int renorm;
  int has_shared;
  float* logits;        // [T][E], or [nsplit][T][E] partial planes (large path)
  int nsplit;           // large path: planes in logits, summed in order plus the bias; 0: final logits
  float* logit_part;    // [T][E][16] partial logits (single-launch decode), or nullptr
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
  unsigned long long* trace;  // nullable: per-CTA phase stamps of the small-batch routing kernel
};

// Grouped W4A16 GEMM over expert segments (prefill regime, tensor cores).
struct GemmArgs {
  const uint8_t* pool;
  long long record_bytes;
  const int32_t* expert_to_slot;
  int num_slots;
  long long s_off0, s_off1;     // scale sections (gate, up) or (down, -)
  int N, K, G, ng;
  int zp;                       // 1: zero-point sections (one byte per group)
  long long z_off0, z_off1;     // zero-point sections (gate, up) or (down, -)
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
  unsigned long long* stats;    // nullable: [gridDim][kGemmStats] cycles spent waiting, per role
};
// GEMM wait counters per CTA: producer (codes stage free, token stage free),
// MMA (accumulator free, A stage full), dequantiser warp 0 (token stage
// landed, codes landed, A stage free), epilogue warp 0 (accumulator full),
// and the CTA's total cycles.
constexpr int kGemmStats = 9;

// Whole-layer decode megakernel (T <= kSmallRouteMaxT, full residency).
// Tensor-core grouped GEMV over expert segments (decode regime): items of
// rb rows (rt = rb / 16 row tiles) of one or two matrices, codes in 128-byte
// swizzled TMA boxes.
struct TcGemvArgs {
  const uint8_t* pool;          // slot pool base (scale sections are read from it)
  long long record_bytes;
  const int32_t* expert_to_slot;
  int num_slots;
  long long s_off0, s_off1;     // scale sections (gate, up) or (down, -)
  int N;                        // output rows per matrix
  int K;                        // reduction length (multiple of 32)
  int G;                        // group size (multiple of 32)
  int ng;                       // ceil(K / G)
  int rb;                       // rows per work item (multiple of 16)
  int rt;                       // rb / 16 (1, 2, 4 or 8)
  int kparts;                   // consumer warps per row tile (consumer warps / rt), a power of two
  int lkparts;                  // log2(kparts)
  int nbox;                     // ceil(K / 256) code boxes per matrix row
  uint32_t code_mat_bytes;      // nbox * 128 * rb
  uint32_t sstride;             // scale bytes per matrix in a slot (16-byte multiple)
  int zp;                       // 1: zero-point sections (one code per group, one byte each)
  long long z_off0, z_off1;     // zero-point sections (gate, up) or (down, -)
  uint32_t zstride;             // zero-point bytes per matrix in a slot (16-byte multiple)
  const int32_t* seg_expert;
  const int32_t* seg_start;
  const int32_t* seg_count;
  const __half* act;            // gate/up: x [T][K]; down: h [P][K]
  int act_gather;               // 1: row of sorted position p is x[perm[p] / k] (p < Tk) or x[p - Tk]
  const int32_t* perm;
  int Tk;
  int k;
  __half* h_out;                // gate/up: [P][N] FP16 at sorted positions
  float* y_out;                 // down: [Tk + T][N] FP32 at flat index
  uint32_t* err;
};

struct TcGemvPlan {
  int rb, rt, kparts, lkparts, nbox;
  uint32_t code_mat_bytes, sstride, zstride, slot_bytes;  // slot_bytes: multiple of 1024
};
// Items of about item_bytes code bytes with rb a power-of-two multiple of 16
// and rb / 16 <= 8. Requires K % 32 == 0, G % 32 == 0, N % 16 == 0. A slot
// holds the codes, the scale rows and (zp) the zero-point rows.
TcGemvPlan plan_tcgemv(int N, int K, int G, bool dual, int item_bytes, bool zp);
// 3-D map {K / 2 bytes, N rows, slots} of one code section, 128-byte boxes of
// box_rows rows, 128-byte swizzle.
bool encode_tcgemv_map(CUtensorMap* tm, const void* pool_section, int K, int N, int num_slots, size_t record_bytes,
                       int box_rows);

// Kernel parameters of the multi-kernel tensor-core GEMV.
struct TcGemvLaunch {
  TcGemvArgs a;
  CUtensorMap m0, m1;           // code maps (gate, up) or (down, down)
  const int32_t* num_seg;       // segment count (device)
  int stages;
  uint32_t slot_bytes;
  int ns, bs_chunks, cs_groups;
};
size_t tcgemv_smem_bytes(const TcGemvLaunch& p);
cudaError_t launch_tcgemv(const TcGemvLaunch& p, bool dual, int grid, cudaStream_t s, bool pdl);

struct DecodeArgs {
  RouteArgs r;           // routing inputs and global outputs
  TcGemvArgs g;          // gate/up items (segment pointers are replaced in-kernel)
  TcGemvArgs d;          // down items
  CUtensorMap tm_gate, tm_up, tm_down;  // code maps (kernel parameter space)
  __half* out;           // [T][H]
  const __half* x_res;   // residual input or nullptr
  int has_shared;
  uint32_t* ctr;         // zeroed counters: logits_done, final ticket, done_gu[E+1], done_dn[]
  int stages;
  uint32_t slot_bytes;   // ring slot size (max of the two item layouts, multiple of 1024)
  int ns;                // token columns kept per tile (2, 4 or 8)
  int bs_chunks;         // chunks (padded) the B buffer holds: max over gate/up and down K
  int cs_groups;         // groups the constant buffer holds
  unsigned long long* trace;  // nullable: [gridDim][kTraceStamps] global-timer stamps
};

// Tensor maps of the three code sections of a slot pool: GEMM tiles, and
// the GEMV's 128-byte swizzled boxes.
struct CodeMaps {
  CUtensorMap gate, up, down;
  bool valid;
  CUtensorMap tgate, tup, tdown;
  bool tvalid;
};

struct CombineArgs {
  const float* ypart;   // [Tk + T][H]
  const float* w;       // [T][k]
  const __half* x;      // residual input or nullptr
  __half* out;          // [T][H]
  int T, H, k, has_shared;
  const float* gate;    // shared expert gate vector [H] (weight sigmoid(x . gate)) or nullptr (weight 1)
  const __half* xin;    // the layer input [T][H] (for the gate)
};

// Launch shape of one grouped-GEMV launch, chosen on the host.

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
// K parts of the large-batch router logits for this shape (1..kRouterSplitMax)
int router_split(int T, int E, int H, int num_sms);
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s, bool pdl);
constexpr int kDecodeMaxStages = 8;  // ring stages of the single-launch decode
// dynamic shared memory the ring kernels size themselves to: the 227 KB
// per-block limit less room for static shared memory and the per-block
// reservation
constexpr size_t kSmemBudget = 227 * 1024 - 2048;
size_t decode_smem_bytes(const DecodeArgs& a, int stages);
cudaError_t launch_decode(const DecodeArgs& a, int grid, cudaStream_t s, bool pdl);
// whether the decode launch may add programmatic stream serialisation to its
// cooperative launch on this device (probed once, outside any capture)
bool decode_pdl_supported();

// Batch-1 whole-layer decode (T == 1, fully resident table): every CTA's
// share of the selected experts' bytes fits its shared memory, so all of it
// is requested at once. Work comes in units of 16 rows: gate/up units of
// the (selected expert, intermediate row) space and down units of the output
// rows. ctr[0] (logits published) and ctr[1] (gate/up done) are epoch
// counters that every CTA increments exactly once per launch, wrapping at
// ctr_mod (a multiple of the grid); they start at zero.
struct Decode1Args {
  RouteArgs r;                  // T == 1; logits [E]; routing outputs published by CTA 0
  const uint8_t* pool;          // slot pool base
  long long record_bytes;
  const int32_t* expert_to_slot;
  int num_slots;
  long long off_q[3];           // code sections: gate, up, down
  long long off_s[3];           // scale sections: gate, up, down
  int I;                        // intermediate
  int G;                        // group size
  __half* h;                    // [nseg][I] SwiGLU activations, by sorted position
  __half* out;                  // [H]
  const __half* x_res;          // residual input or nullptr
  uint32_t* ctr;
  uint32_t ctr_mod;
  unsigned long long* trace;    // nullable: [gridDim][kTraceStamps]
  int nseg_max;                 // k + has_shared
  int max_units_g;              // most gate/up tiles of a CTA (decode1_max_tiles)
  int max_units_d;              // ceil(H / 16 / grid)
  int max_rows_rt;              // router rows per CTA: ceil(E / grid)
  // stacked layers in one launch (k_decode1_stack), 0 / nullptr otherwise:
  int stack;                    // 1: this layer runs inside the stack kernel
  const float* wr_next;         // next layer's router [E][H], nullptr at the last layer
  float* part_in;               // [grid][E] partial logits of this layer, one row per CTA
  float* part_out;              // [grid][E] partial logits of the next layer
};
// Layers of one stack launch: x of layer l + 1 is the out of layer l; every
// layer has the same shape.
constexpr int kD1MaxLayers = 48;
struct Decode1Stack {
  Decode1Args layer[kD1MaxLayers];
  int n_layers;
  int trace_layer;  // the layer whose phases are stamped (when trace is set)
};
// Most gate/up tiles (16 rows, 8 at an expert's end) any CTA of the grid
// gets when nseg experts' I rows are split in 8-row granules.
int decode1_max_tiles(int nseg, int I, int grid);
// Dynamic shared memory of k_decode1 for these arguments (0: does not fit).
size_t decode1_smem_bytes(const Decode1Args& a);
cudaError_t launch_decode1(const Decode1Args& a, int grid, cudaStream_t s, bool pdl);
cudaError_t launch_decode1_stack(const Decode1Stack& st, int grid, cudaStream_t s, bool pdl);
cudaError_t launch_gemm(bool dual, const CUtensorMap& codes0, const CUtensorMap& codes1, const CUtensorMap& act,
                        const GemmArgs& a, int grid, cudaStream_t s, bool pdl);
size_t gemm_smem_bytes(bool dual);
bool encode_codes_map(CUtensorMap* tm, const void* pool_section, int K, int N, int num_slots, size_t record_bytes,
                      int box_rows);
bool encode_rows_map(CUtensorMap* tm, const void* base, int cols, int rows, int box_rows);
// xs[pos] = x[perm[pos] / k] (pos < Tk) or x[pos - Tk], rows positions of H halves
cudaError_t launch_gather_rows(const __half* x, __half* xs, const int32_t* perm, int Tk, int k, int rows, int H,
                               int grid, cudaStream_t s, bool pdl);
int gemm_tile_n();
int gemm_tile_k();

}  // namespace moe
