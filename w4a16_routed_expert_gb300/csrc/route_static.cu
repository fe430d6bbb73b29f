// Router entry point that allocates nothing: the small-batch routing kernel
// (logits, softmax, top-k, routing weights) run with its scratch in a
// file-scope device array instead of a handle's workspace.
//
// Some callers cannot allocate device memory at all: a host runtime that
// plans every device byte itself and forbids allocation once it has started,
// a fixed-arena or safety-certified process, or a plug-in that is only ever
// handed input and output buffers. They can still route tokens through this
// entry point; they pass the inputs and the ids / weights outputs, and the
// library uses the static array below for everything else.
//
// Every GPU that loads the library holds this array until the process exits.
// All calls on a device share it and it keeps the last call's contents: calls
// that overlap on the GPU (different streams, or threads without ordering)
// race on it. Set-up: the first call on a device, with that device current,
// looks up the array's device address (cudaGetSymbolAddress) and caches it
// together with the unique id of the device's current context; make that
// first call before any stream capture. A device reset (cudaDeviceReset)
// ends the context and the array may come back at another address: a call
// that finds a different context id looks the address up again.
#include <mutex>

#include "layer_internal.h"

namespace moe {
namespace {

constexpr size_t kStaticScratchBytes = 192 * 1024;
constexpr int kStaticMaxT = kSmallRouteMaxT;  // 16 tokens
constexpr int kStaticMaxE = 1024;
constexpr int kStaticMaxK = 32;
constexpr int kMaxDevices = 64;

// The routing scratch (logits, workspace ids / weights, counts, offsets,
// permutation, segment list, ticket, error word), 256-byte aligned.
static __device__ __align__(256) unsigned char g_route_scratch[kStaticScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};

// Unique id of the calling thread's current context (0 if unavailable), via
// the driver entry points (no link-time dependence on the driver library).
unsigned long long current_context_id() {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static bool looked_up = false;
  if (!looked_up) {
    looked_up = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(p);
    cudaGetLastError();
  }
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current && get_id && get_current(&ctx) == CUDA_SUCCESS && ctx && get_id(ctx, &id) == CUDA_SUCCESS) return id;
  return 0;
}

moe_status_t fail_static(moe_status_t st, const char* msg) { return set_error(st, "%s", msg); }

size_t a256(size_t v) { return (v + 255) & ~size_t(255); }

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_route_topk_static(const void* x, int32_t T, int32_t H, const float* router_w,
                                              const float* router_bias, int32_t E, int32_t k, int32_t renormalize,
                                              int32_t* topk_ids, float* topk_w, void* stream) {
  using namespace moe;
  if (T == 0) return MOE_OK;
  if (!x || !router_w || !topk_ids || !topk_w)
    return fail_static(MOE_ERR_INVALID_ARG, "x, router_w, topk_ids and topk_w must not be NULL");
  if (T < 0 || T > kStaticMaxT)
    return fail_static(MOE_ERR_INVALID_ARG, "moe_route_topk_static: T must be in 0..16");
  if (E < 1 || E > kStaticMaxE) return fail_static(MOE_ERR_INVALID_ARG, "moe_route_topk_static: E must be in 1..1024");
  if (k < 1 || k > kStaticMaxK || k > E)
    return fail_static(MOE_ERR_INVALID_ARG, "moe_route_topk_static: k must be in 1..min(32, E)");
  if (H < 128 || H > 4096 || H % 32)
    return fail_static(MOE_ERR_INVALID_ARG, "moe_route_topk_static: H must be a multiple of 32 in 128..4096");
  if (renormalize != 0 && renormalize != 1)
    return fail_static(MOE_ERR_INVALID_ARG, "moe_route_topk_static: renormalize must be 0 or 1");

  // carve the static scratch; the sizes above bound it by construction
  const size_t tk = (size_t)T * k;
  size_t off[12];
  size_t cur = 0;
  const size_t sizes[12] = {(size_t)T * E * 4, tk * 4, tk * 4, (size_t)E * 4, (size_t)(E + 1) * 4, tk * 4, tk * 4,
                            (size_t)(E + 1) * 4, (size_t)(E + 1) * 4, (size_t)(E + 1) * 4, 4, 8};
  for (int i = 0; i < 12; ++i) {
    off[i] = cur;
    cur += a256(sizes[i]);
  }
  if (cur > kStaticScratchBytes)
    return fail_static(MOE_ERR_INVALID_ARG, "moe_route_topk_static: T * E exceeds the static scratch");

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return fail_static(MOE_ERR_CUDA, "moe_route_topk_static: no current CUDA device");
  unsigned char* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    const unsigned long long ctx = current_context_id();
    if (!g_scratch_addr[dev] || ctx != g_scratch_ctx[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_route_scratch);
      if (e != cudaSuccess || !p) {
        cudaGetLastError();
        return fail_static(MOE_ERR_CUDA, "moe_route_topk_static: cudaGetSymbolAddress of the scratch failed");
      }
      g_scratch_addr[dev] = p;
      // the lookup made the device's primary context current if it was not
      g_scratch_ctx[dev] = current_context_id();
    }
    base = static_cast<unsigned char*>(g_scratch_addr[dev]);
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  RouteArgs a = {};
  a.x = static_cast<const __half*>(x);
  a.wr = router_w;
  a.bias = router_bias;
  a.T = T;
  a.H = H;
  a.E = E;
  a.k = k;
  a.renorm = renormalize;
  a.has_shared = 0;
  a.logits = reinterpret_cast<float*>(base + off[0]);
  a.ids = reinterpret_cast<int32_t*>(base + off[1]);
  a.w = reinterpret_cast<float*>(base + off[2]);
  a.ids_user = topk_ids;
  a.w_user = topk_w;
  a.counts = reinterpret_cast<int32_t*>(base + off[3]);
  a.offsets = reinterpret_cast<int32_t*>(base + off[4]);
  a.perm = reinterpret_cast<int32_t*>(base + off[5]);
  a.inv_perm = reinterpret_cast<int32_t*>(base + off[6]);
  a.seg_expert = reinterpret_cast<int32_t*>(base + off[7]);
  a.seg_start = reinterpret_cast<int32_t*>(base + off[8]);
  a.seg_count = reinterpret_cast<int32_t*>(base + off[9]);
  a.num_seg = reinterpret_cast<int32_t*>(base + off[10]);
  a.ticket = reinterpret_cast<uint32_t*>(base + off[11]);
  a.err = a.ticket + 1;
  a.chunk_hist = nullptr;
  a.chunk_base = nullptr;
  // the last-CTA ticket must start at zero on every call
  e = cudaMemsetAsync(a.ticket, 0, 8, s);
  if (e == cudaSuccess) e = launch_route_small(a, s, false);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return set_error(MOE_ERR_CUDA, "moe_route_topk_static: launch failed: %s", cudaGetErrorString(e));
  }
  return MOE_OK;
}
