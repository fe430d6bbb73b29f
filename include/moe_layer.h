/*
 * moe_layer.h — C ABI of the GB300 (sm_103a) W4A16 routed-expert MoE layer.
 *
 * The layer (Horizon RunMap report, "The complete execution path", steps 1-3;
 * "Architecture invariants"): routed experts are stored compact as INT4
 * qpacked codes with FP16 group scales and executed with FP16 activations
 * (W4A16). For T tokens x[T][H] the layer computes
 *
 *   logits  L[t][e] = sum_h x[t][h] * Wr[e][h] (+ bias[e])        FP32
 *   p[t]    = softmax over all E experts of L[t]                  FP32
 *   ids[t]  = the top_k experts of L[t], ties to the lower id,
 *             in rank order (descending logit, then ascending id);
 *             a NaN logit ranks below every number (inputs with NaN or
 *             Inf give a well-defined selection, never a stalled launch)
 *   w[t][j] = p[t][ids[t][j]]  (divided by sum_j p[t][ids[t][j]] when
 *             renormalising)
 *   y_e(x)  = Wd_e (silu(Wg_e x) * (Wu_e x)),  silu(z) = z / (1 + e^-z),
 *             W = (q - 8) * s dequantised from expert e's record
 *   out[t]  = sum_j w[t][j] * y_{ids[t][j]}(x[t])  (+ y_shared(x[t]))
 *
 * with an optional always-on shared expert (F51 Nitro-MoE, "The thesis": the
 * documented model routes each token to ten experts and also runs one shared
 * expert) applied to every token with weight 1.
 *
 * Expert records (canonical format, one contiguous record per expert so a
 * single copy moves everything an expert needs — moe-stream, "Method"):
 *   gate_q | up_q | down_q | gate_s | up_s | down_s
 * codes row-major with K contiguous, two codes per byte (low nibble = even k),
 * gate/up [I][H], down [H][I]; FP16 scales [N][ceil(K/G)], one per G codes
 * along K; w = (q - 8) * s. Each section starts on a 256-byte boundary and
 * the record size is a multiple of 256 bytes (moe_record_bytes).
 *
 * Records are addressed through expert_to_slot (F51 Nitro-MoE, "Layer 1 -
 * expert persistence cache": an expert_to_slot map over a fixed pool of GPU
 * slots), so a fully resident table and a partially resident slot pool run
 * the same kernels.
 *
 * Conventions
 *  - Every call returns a moe_status_t; nothing aborts and no C++ exception
 *    crosses the ABI. moe_layer_last_error() describes the last failure of
 *    the calling thread.
 *  - The pages publish no interface (Horizon RunMap report, "Scope of the
 *    published results": the runtime source stays private). Each entry point
 *    below cites the passage that defines the operation it performs.
 *  - Device pointers passed in are borrowed: the caller owns them and they
 *    must stay valid until moe_layer_destroy.
 *  - moe_layer_forward is asynchronous on the given CUDA stream (NULL = the
 *    legacy default stream). Its outputs, including ids and weights, are
 *    valid only once that stream has been synchronised.
 *  - One forward at a time per handle: two forwards of one handle that
 *    overlap on the GPU share its workspace and race.
 *  - Kernels never trap. A device-side wait that runs out of time (a
 *    bounded spin of about two seconds) records an error word in the
 *    workspace; moe_layer_sync reports it as MOE_ERR_TIMEOUT.
 *  - The library never writes host_backing and never copies an expert
 *    record from the device to the host.
 */
#ifndef MOE_LAYER_H
#define MOE_LAYER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 3

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* a NULL handle/pointer, a size out of range, T > max_tokens */
  MOE_ERR_OOM = 2,         /* a device or pinned allocation failed in create */
  MOE_ERR_CUDA = 3,        /* a CUDA runtime call failed (message has the CUDA error) */
  MOE_ERR_UNSUPPORTED = 4, /* a shape or mode this build does not run (e.g. H % 32 != 0) */
  MOE_ERR_CAPACITY = 5,    /* partial residency: not enough slots for one expert group */
  MOE_ERR_TIMEOUT = 6,     /* a device-side bounded wait gave up (reported by moe_layer_sync) */
  MOE_ERR_INTERNAL = 7     /* an internal consistency check failed */
} moe_status_t;

typedef enum {
  MOE_RESIDENCY_FULL = 0,   /* every record resident in a caller-owned device pool */
  MOE_RESIDENCY_PARTIAL = 1 /* library-owned pool of num_slots records filled from pinned host backing */
} moe_residency_t;

typedef struct {
  int32_t hidden;            /* H, multiple of 32 */
  int32_t intermediate;      /* I, multiple of 32 */
  int32_t num_experts;       /* E routed experts, 1..1024 */
  int32_t top_k;             /* k, 1..min(E, 32) */
  int32_t group_size;        /* G, 32, 64 or 128 (codes per FP16 scale along K) */
  int32_t renormalize;       /* 0: w = softmax over all E; 1: w renormalised over the top k */
  int32_t has_shared_expert; /* 1: record index E is a shared expert run on every token, weight 1 */
  int32_t max_tokens;        /* upper bound of T; workspace is sized for it at create */
  int32_t num_slots;         /* FULL: records in slot_pool; PARTIAL: slots of the library's pool */
  int32_t residency;         /* moe_residency_t */
  int32_t add_residual;      /* 1: out = fp16(x + fp16(layer(x))) (residual stream of stacked layers) */
  /* PARTIAL residency only (ignored in FULL):
   * spare_slots      unpublished rows beyond the num_slots published ones:
   *                  misses are copied into them while earlier kernels still
   *                  read the published rows (0: misses reuse evicted rows
   *                  once their readers have retired);
   * staging_records  pinned staging buffers (one record each) a pageable
   *                  host_backing is copied through (0: 4); a page-locked
   *                  host_backing is copied from directly;
   * cache_policy     moe_cache_policy_t: which published expert is evicted. */
  int32_t spare_slots;
  int32_t staging_records;
  int32_t cache_policy;
  /* 1: asymmetric quantisation, w = (q - z) * s with one zero code z (0..15)
   * per group, one byte each, in three record sections after the scales
   * (moe_record_bytes_zp, moe_record_section 6..8); 0: z = 8. */
  int32_t zero_points;
} moe_layer_config_t;

typedef enum {
  MOE_POLICY_LRU = 0,     /* least recently used */
  MOE_POLICY_LFU = 1,     /* least frequently used (every access counted) */
  MOE_POLICY_LRU_FREQ = 2 /* lowest freq * 1000 - age; frequencies x0.75 every 2 x num_slots misses */
} moe_cache_policy_t;

typedef struct {
  const float* router_w;         /* device, FP32 [E][H] row-major */
  const float* router_bias;      /* device, FP32 [E] added to the logits, or NULL */
  const void* slot_pool;         /* FULL: device, num_slots * moe_record_bytes bytes, 256-byte aligned.
                                    PARTIAL: must be NULL (the library allocates the pool). */
  const int32_t* expert_to_slot; /* FULL: device int32 [E (+1 if shared)], values in [0, num_slots).
                                    PARTIAL: must be NULL (the library owns the map). */
  const void* host_backing;      /* PARTIAL: host memory, [E (+1)] records back to back, registered
                                    (pinned) by the library for the handle's lifetime and never
                                    written. FULL: must be NULL. */
  const float* shared_gate;      /* device FP32 [H]: the shared expert's output is weighted per token
                                    by sigmoid(x . shared_gate); NULL: weight 1. Needs a shared
                                    expert. */
} moe_layer_weights_t;

typedef struct moe_layer moe_layer_t;

typedef struct {
  uint64_t forward_calls;    /* forwards run (T > 0) */
  uint64_t tokens;           /* tokens processed */
  uint64_t expert_hits;      /* PARTIAL: demanded experts found resident */
  uint64_t expert_misses;    /* PARTIAL: demanded experts not resident when their forward started */
  uint64_t h2d_bytes;        /* PARTIAL: expert bytes copied host -> device (forwards and prefetches) */
  uint64_t d2h_expert_bytes; /* expert bytes copied device -> host: 0 by construction */
  uint64_t waves;            /* PARTIAL: expert-compute waves (transactions: one routed group each) */
  uint64_t generations;      /* PARTIAL: cache generations published (a group with misses publishes one) */
  uint64_t evictions;        /* PARTIAL: experts dropped from the published set */
  uint64_t staged_copies;    /* PARTIAL: records copied through the pinned staging buffers */
  int32_t faulted;           /* PARTIAL: 1 once a failure after publication has faulted the cache */
  int32_t reserved;
  uint64_t prefetch_calls;   /* PARTIAL: moe_layer_prefetch calls that planned a guess */
  uint64_t prefetched;       /* PARTIAL: experts a prefetch copied in */
  uint64_t prefetch_used;    /* PARTIAL: of those, demanded by a later forward while resident (once each) */
} moe_layer_stats_t;

typedef struct {
  float route_ms;         /* routing kernels (logits, top-k, permutation) */
  float gate_up_ms;       /* gate/up + SwiGLU expert kernel */
  float down_ms;          /* down-projection expert kernel */
  float combine_ms;       /* weighted combine */
  float total_ms;         /* whole forward */
  int32_t active_experts; /* distinct routed experts selected (E_u) */
  int32_t tokens;         /* T of the profiled forward */
  int32_t single_launch;  /* 1: the forward ran as one kernel (stage times are 0, total_ms is the kernel) */
} moe_layer_profile_t;

/* ABI version of the loaded library (MOE_ABI_VERSION of its build). */
int32_t moe_abi_version(void);

/* Padded size in bytes of one canonical expert record; 0 for an invalid shape. */
size_t moe_record_bytes(int32_t hidden, int32_t intermediate, int32_t group_size);

/* Padded size of one record with (zero_points = 1) or without zero-point
 * sections; 0 for an invalid shape. */
size_t moe_record_bytes_zp(int32_t hidden, int32_t intermediate, int32_t group_size, int32_t zero_points);

/* Byte offset and size of section `section` (0 gate_q, 1 up_q, 2 down_q,
 * 3 gate_s, 4 up_s, 5 down_s, and in a record with zero points 6 gate_z,
 * 7 up_z, 8 down_z) inside one record. */
moe_status_t moe_record_section(int32_t hidden, int32_t intermediate, int32_t group_size,
                                int32_t section, size_t* offset, size_t* bytes);

/* Horizon RunMap report, "The complete execution path", step 1 (the routed
 * experts loaded once as compact INT4 + FP16-scale tensors into the pool the
 * kernels read) and F51 Nitro-MoE, "Layer 1 - expert persistence cache" (a
 * fixed pool of slots addressed through expert_to_slot).
 * Validates the configuration, records the borrowed pointers and allocates
 * the workspace for max_tokens tokens on the current CUDA device. Fails with
 * INVALID_ARG / UNSUPPORTED / OOM / CAPACITY; *out is NULL on failure. No
 * allocation happens in moe_layer_forward afterwards. */
moe_status_t moe_layer_create(const moe_layer_config_t* config, const moe_layer_weights_t* weights,
                              moe_layer_t** out);

/* Horizon RunMap report, "The complete execution path", steps 2-3 (routing
 * selects each token's experts, the custom kernels run them on FP16
 * activations) and moe-stream, "Method" (top-8 of 64 experts per token).
 * One forward of T tokens on `stream` (a cudaStream_t, NULL = default).
 *   x        device FP16 [T][H], read only
 *   out      device FP16 [T][H]; must not overlap x
 *   topk_ids device int32 [T][k] or NULL; rank order
 *   topk_w   device FP32 [T][k] or NULL
 * T = 0 returns MOE_OK without launching. T > max_tokens -> INVALID_ARG.
 * FULL residency: enqueues kernels only, no synchronisation and no
 * allocation. PARTIAL residency: synchronises the stream once to read the
 * demanded expert set, copies missing records into the pool on a side
 * stream and runs the experts in waves (not capturable in a CUDA graph). */
moe_status_t moe_layer_forward(moe_layer_t* layer, const void* x, int32_t T, void* out,
                               int32_t* topk_ids, float* topk_w, void* stream);

/* Same computation for callers whose tokens live in host memory (x host
 * FP16 [T][H]; out, ids, weights host buffers; ids, weights may be NULL).
 * Up to 16 tokens, when every buffer given is page-locked and mapped into
 * the device's address space (cudaHostAlloc / pinned torch tensors on this
 * platform), the kernels read x and write the results in place over the
 * host link, with no staging copies. Otherwise x is copied to a device
 * staging buffer, the forward runs, and out / ids / weights are copied back.
 * Asynchronous on `stream`; synchronise it before reading the results. */
moe_status_t moe_layer_forward_host(moe_layer_t* layer, const void* x_host, int32_t T, void* out_host,
                                    int32_t* topk_ids_host, float* topk_w_host, void* stream);

/* Copies the routing of the last forward (or prefetch guess) on this handle into device buffers
 * (any may be NULL): counts int32 [E], offsets int32 [E+1] (exclusive prefix
 * sum of counts), perm int32 [T*k] (flat index t*k+j at each sorted position,
 * ascending flat index inside an expert), inv_perm int32 [T*k]. Asynchronous
 * on `stream`. */
moe_status_t moe_layer_routing(const moe_layer_t* layer, int32_t* counts, int32_t* offsets, int32_t* perm,
                               int32_t* inv_perm, void* stream);

/* Synchronises `stream` and reports (then clears) a device-side error word:
 * MOE_ERR_TIMEOUT if a bounded wait gave up, MOE_ERR_CUDA on a CUDA error. */
moe_status_t moe_layer_sync(moe_layer_t* layer, void* stream);

/* Tracing: when enabled, each forward records CUDA events between its
 * stages on the forward's stream (also inside a captured CUDA graph).
 * moe_layer_get_profile waits for the last forward's events and reports the
 * stage times and the number of distinct experts it selected. */
moe_status_t moe_layer_set_profiling(moe_layer_t* layer, int32_t enable);
moe_status_t moe_layer_get_profile(moe_layer_t* layer, moe_layer_profile_t* profile);

/* Tracing of the single-launch decode kernels: when the handle was created
 * with the environment variable MOE_TRACE=1, every CTA of those kernels
 * writes 32 global-timer stamps (ns) per forward (0 where not reached).
 * Batch-1 kernel (one token): 0 entry, 1 past the dependency on the previous
 * launch, 2 own logits published, 3 all logits seen, 4 per-group candidates
 * ranked, 5 selection done, 6 gate/up copies issued, 7 routing weights done,
 * 8 down copies issued, 9..12 gate/up tiles 0..3 landed, 13..16 tiles 0..3
 * computed (consumer warp 0), 17 the CTA's h written, 18 every CTA's h
 * seen, 19 / 21 down inputs staged by consumer warp 0 / the last consumer
 * warp, 20 / 22 their down work done, 23 all down partials done, 24 output
 * rows written, 25 exit. Stack kernel (moe_stack_forward at one token):
 * the same stamps for one layer (the second of the stack, the first if it
 * is alone), in the first layer's buffer; 0 is that layer's entry (the
 * end of the layer before), 2 the partial logits and the input loaded.
 * Small-batch routing kernel of the multi-kernel path (one CTA per
 * expert): 0 entry, 1 past the dependency, 2 the expert's logit partials
 * done, 4 its ticket taken, and in the CTA that finishes the routing 3
 * top-k done, 5 routing done. Small-batch decode kernel (2..16 tokens): 0 entry, 1 own
 * logit partials written, 2 all partials seen, 3 top-k done, 4 routing
 * done, 5 first gate/up item started, 6 last gate/up item done, 7 first down
 * item started, 8 consumers done, 9 finisher done, 10 all warps done, 11
 * exit, 12 first down wait entered, 13 its counter seen, 14 its activations
 * staged; then for the CTA's first 8 work items, item i's bytes landed
 * (16 + 2i) and item i computed (17 + 2i), as seen by consumer warp 0.
 * Synchronises the device and copies min(max_stamps, 32 * 1024) stamps
 * (32 per CTA for CTAs 0..1023, CTA-major; CTAs the last launch did not
 * have keep older stamps) into host memory; *n_stamps receives the count. */
moe_status_t moe_layer_get_trace(moe_layer_t* layer, uint64_t* stamps, int32_t max_stamps, int32_t* n_stamps);

/* Wait counters of the tensor-core GEMM path: when the handle was created
 * with MOE_GEMM_STATS=1, each CTA of the last gate/up and down GEMM records
 * 9 cycle counts: producer waiting for a free code stage and a free token
 * stage; MMA thread waiting for a free accumulator and a full A stage;
 * dequantiser warp 0 waiting for a landed token stage, for codes and for a
 * free A stage; epilogue warp 0 waiting for an accumulator; the CTA's
 * total. Layout
 * [launch (gate/up, down)][CTA][9]. Synchronises the device and copies
 * min(max_values, 2 * 9 * CTAs) counts; *n_values receives the count. */
moe_status_t moe_layer_get_gemm_stats(moe_layer_t* layer, uint64_t* values, int32_t max_values, int32_t* n_values);

/* Copies the handle's counters into *stats. */
moe_status_t moe_layer_get_stats(const moe_layer_t* layer, moe_layer_stats_t* stats);

/* Horizon RunMap report, "Partial-residency contract": the pool and its
 * host registration end with the handle.
 * Frees the workspace (and, in PARTIAL mode, the pool and the host
 * registration). NULL is accepted and returns MOE_OK. Call after the last
 * forward has completed. */
moe_status_t moe_layer_destroy(moe_layer_t* layer);

/* Stacked layers: the residual stream of a decoder's MoE layers, the layer
 * of Horizon RunMap report, "The complete execution path", steps 2-3, run
 * once per layer. A stack borrows n_layers (>= 1) layer handles that map
 * H -> H (they must outlive it) and runs x_{l+1} = layer_l(x_l) for
 * l = 0..n_layers-1 on one stream, each layer with its own configuration
 * (add_residual included); out = x_{n_layers}.
 *   x       device FP16 [T][H], read only
 *   out     device FP16 [T][H]; must overlap neither x nor states
 *   states  device FP16 [n_layers - 1][T][H] receiving x_1 .. x_{n_layers-1}
 *           (the inputs of layers 1.., e.g. for checking each layer), or NULL
 * T <= the smallest max_tokens of the layers. One token over fully
 * resident layers of one shape (H, I, E <= 128, k, G, shared expert) runs as
 * a single cooperative launch (moe_stack_single_launch reports it; set
 * MOE_STACK1=0 before create to turn it off): one grid-wide step per layer
 * boundary instead of a launch. There each layer's router logits are summed
 * from per-CTA partials over the rows of its input in a fixed order (not
 * the order of a layer's own forward), so its FP32 logits may differ from
 * that forward's in the last bits; results are repeatable bit for bit.
 * Otherwise the layers' own forwards run one after another. Routing of the
 * last stack forward is read per layer with moe_layer_routing; every layer's
 * forward counters advance. Asynchronous; no allocation after create;
 * graph-capturable when every layer's forward is. moe_stack_sync reports
 * device-side failures (MOE_ERR_TIMEOUT) of the stack kernel and of every
 * layer. */
typedef struct moe_stack moe_stack_t;
moe_status_t moe_stack_create(moe_layer_t* const* layers, int32_t n_layers, moe_stack_t** out);
moe_status_t moe_stack_forward(moe_stack_t* stack, const void* x, int32_t T, void* out, void* states,
                               void* stream);
moe_status_t moe_stack_sync(moe_stack_t* stack, void* stream);
int32_t moe_stack_single_launch(const moe_stack_t* stack);
/* NULL is accepted. Call after the last forward has completed. */
moe_status_t moe_stack_destroy(moe_stack_t* stack);

/* moe-stream, "Findings" (prefetching: the next layer's router, run early on
 * the current state, guesses that layer's experts; most guesses are used).
 * Routes the guess input x (device FP16 [T][H], e.g. the previous layer's
 * input while that layer runs) with this handle's router on the handle's
 * side stream once x is ready on `stream`, and returns without waiting. A
 * thread the handle owns waits for the guess's expert counts and copies the
 * guessed experts that are not resident into the pool on the side stream:
 * the shared expert, then routed experts by guessed count (ties to the lower
 * id), at most num_slots in all; resident ones stay; victims follow the
 * cache policy and are overwritten only after their readers retire. The
 * guess is published in the cache; a later forward that reads a row it
 * filled waits (on the forward's stream) for its copies before using it.
 * Results of later forwards are identical with or without prefetches. The
 * handle's next forward orders its routing after the guess's (they share
 * the handle's routing buffers) and waits for the thread's planning before
 * its own; a failure of that planning (its copies aborted, the previous
 * generation kept) is returned once, by that forward, as MOE_ERR_CUDA.
 * Call it after the forward that precedes the guessed one has been enqueued
 * on `stream`. FULL residency: returns MOE_OK and does nothing. T = 0:
 * MOE_OK. T > max_tokens -> INVALID_ARG; a faulted cache -> MOE_ERR_CUDA. */
moe_status_t moe_layer_prefetch(moe_layer_t* layer, const void* x, int32_t T, void* stream);

/* Routing without any device allocation, for callers that must not allocate
 * device memory (a host runtime that owns every device byte and forbids
 * allocation after start-up, a fixed-arena process, a plug-in handed only
 * input and output buffers). The pages describe no such entry point; it is
 * this library's addition. It runs the small-batch routing kernel (FP32
 * logits, softmax over all E, top-k with ties to the lower id, weights) with
 * its scratch in a static device array of 192 KiB that every GPU loading the
 * library keeps until exit.
 *   x          device FP16 [T][H]; router_w device FP32 [E][H];
 *   router_bias device FP32 [E] or NULL; renormalize 0 or 1
 *   topk_ids   device int32 [T][k] (rank order); topk_w device FP32 [T][k]
 * Limits: 0 <= T <= 16, 1 <= E <= 1024, 1 <= k <= min(32, E), H a multiple
 * of 32 in 128..4096; anything else returns MOE_ERR_INVALID_ARG with a
 * message. The first call on a device (with that device current) looks up
 * the scratch array's address and caches it with the id of the device's
 * current context: make that first call before any stream capture. After a
 * device reset the context id changes and the next call looks the address
 * up again. All calls share the array and it keeps the last call's
 * contents; calls that overlap on the GPU race. Asynchronous on `stream`;
 * results are valid once it is synchronised. Calls no allocating routine. */
moe_status_t moe_route_topk_static(const void* x, int32_t T, int32_t H, const float* router_w,
                                   const float* router_bias, int32_t E, int32_t k, int32_t renormalize,
                                   int32_t* topk_ids, float* topk_w, void* stream);

/* Message of the calling thread's last failed call ("" if none). The pointer
 * stays valid until the thread's next call into the library. `layer` may be
 * NULL: the message is kept per thread, not per handle, because a create
 * that fails has no handle to attach it to. */
const char* moe_layer_last_error(const moe_layer_t* layer);

#ifdef __cplusplus
}
#endif

#endif /* MOE_LAYER_H */
