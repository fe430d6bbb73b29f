// Stacked layers: x_{l+1} = layer_l(x_l) over borrowed layer handles on one
// stream. A batch-1 forward over fully resident layers of one shape runs as
// one cooperative launch of the stack kernel (decode1.cu): no launch and no
// separate input hand-off between layers. Anything else runs the layers'
// own forwards one after another through two library-owned buffers.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "layer_internal.h"

struct moe_stack {
  std::vector<moe_layer*> layers;
  int H = 0, E = 0, max_tokens = 0, grid = 0;
  bool single_launch = false;     // batch-1 forwards run as one stack-kernel launch
  uint32_t* ctr = nullptr;        // stack kernel epoch counters (zero at create)
  uint32_t* err = nullptr;        // stack kernel error word
  float* parts = nullptr;         // [2][grid][E] partial logits
  __half* xs = nullptr;           // [2][max_tokens][H] inputs of layers 1..n-1
  moe::Decode1Stack* args = nullptr;
};

namespace {

moe_status_t cuda_err(cudaError_t e, const char* what) {
  cudaGetLastError();
  return moe::set_error(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

void free_stack(moe_stack* st) {
  if (!st) return;
  if (st->ctr) cudaFree(st->ctr);
  if (st->err) cudaFree(st->err);
  if (st->parts) cudaFree(st->parts);
  if (st->xs) cudaFree(st->xs);
  delete st->args;
  delete st;
}

// Batch-1 single-launch eligibility: every layer fully resident in the base
// format, with the batch-1 kernel enabled, and of the first layer's shape; the stack layout
// fits in shared memory; the partial logits of E experts are summed by the
// stack kernel (E <= 128).
bool stack_kernel_fits(const moe_stack* st) {
  const char* env = getenv("MOE_STACK1");
  if (env && strcmp(env, "0") == 0) return false;
  const int n = (int)st->layers.size();
  if (n > moe::kD1MaxLayers) return false;
  const moe_layer* L0 = st->layers[0];
  const moe_layer_config_t& c0 = L0->cfg;
  if (c0.num_experts > 128 || L0->num_sms < 1) return false;
  for (const moe_layer* L : st->layers) {
    const moe_layer_config_t& c = L->cfg;
    if (c.residency != MOE_RESIDENCY_FULL || !L->decode1 || L->variant || L->num_sms != L0->num_sms ||
        L->device != L0->device ||
        c.hidden != c0.hidden || c.intermediate != c0.intermediate || c.num_experts != c0.num_experts ||
        c.top_k != c0.top_k || c.group_size != c0.group_size || c.has_shared_expert != c0.has_shared_expert)
      return false;
  }
  moe::Decode1Args a;
  moe::fill_decode1_args(st->layers[0], nullptr, nullptr, nullptr, nullptr, &a);
  a.stack = 1;
  return moe::decode1_smem_bytes(a) != 0;
}

}  // namespace

extern "C" {

moe_status_t moe_stack_create(moe_layer_t* const* layers, int32_t n_layers, moe_stack_t** out) {
  if (!out) return moe::set_error(MOE_ERR_INVALID_ARG, "out must not be NULL");
  *out = nullptr;
  if (!layers || n_layers < 1) return moe::set_error(MOE_ERR_INVALID_ARG, "need at least one layer");
  moe_stack* st = new (std::nothrow) moe_stack();
  if (!st) return moe::set_error(MOE_ERR_OOM, "host allocation failed");
  for (int l = 0; l < n_layers; ++l) {
    if (!layers[l]) {
      free_stack(st);
      return moe::set_error(MOE_ERR_INVALID_ARG, "layer %d is NULL", l);
    }
    st->layers.push_back(layers[l]);
  }
  st->H = layers[0]->cfg.hidden;
  st->E = layers[0]->cfg.num_experts;
  st->max_tokens = layers[0]->cfg.max_tokens;
  for (moe_layer* L : st->layers) {
    if (L->cfg.hidden != st->H) {
      free_stack(st);
      return moe::set_error(MOE_ERR_INVALID_ARG, "every layer of a stack maps H=%d to H (a layer has H=%d)", st->H,
                            L->cfg.hidden);
    }
    st->max_tokens = L->cfg.max_tokens < st->max_tokens ? L->cfg.max_tokens : st->max_tokens;
  }
  st->single_launch = stack_kernel_fits(st);
  st->grid = layers[0]->num_sms;
  cudaError_t e = cudaMalloc(&st->xs, 2 * (size_t)st->max_tokens * st->H * sizeof(__half));
  if (e == cudaSuccess) e = cudaMalloc(&st->err, 64);
  if (e == cudaSuccess) e = cudaMemset(st->err, 0, 64);
  if (e == cudaSuccess && st->single_launch) {
    e = cudaMalloc(&st->ctr, 64);
    if (e == cudaSuccess) e = cudaMemset(st->ctr, 0, 64);
    if (e == cudaSuccess) e = cudaMalloc(&st->parts, 2 * (size_t)st->grid * st->E * sizeof(float));
    if (e == cudaSuccess) {
      st->args = new (std::nothrow) moe::Decode1Stack();
      if (!st->args) e = cudaErrorMemoryAllocation;
    }
  }
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    free_stack(st);
    cudaGetLastError();
    return moe::set_error(MOE_ERR_OOM, "stack workspace: %s", cudaGetErrorString(e));
  }
  *out = st;
  return MOE_OK;
}

moe_status_t moe_stack_forward(moe_stack_t* st, const void* x, int32_t T, void* out, void* states, void* stream) {
  if (!st) return moe::set_error(MOE_ERR_INVALID_ARG, "stack must not be NULL");
  if (T < 0 || T > st->max_tokens)
    return moe::set_error(MOE_ERR_INVALID_ARG, "T=%d out of 0..max_tokens=%d", T, st->max_tokens);
  if (T == 0) return MOE_OK;
  if (!x || !out) return moe::set_error(MOE_ERR_INVALID_ARG, "x and out must not be NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int n = (int)st->layers.size();
  const size_t plane = (size_t)T * st->H;
  // input of layer l (l >= 1) and output of layer l (l < n - 1)
  auto buf = [&](int l) -> __half* {
    return states ? static_cast<__half*>(states) + (size_t)l * plane : st->xs + (size_t)(l % 2) * plane;
  };
  auto x_of = [&](int l) -> const __half* { return l == 0 ? static_cast<const __half*>(x) : buf(l - 1); };
  auto out_of = [&](int l) -> __half* { return l == n - 1 ? static_cast<__half*>(out) : buf(l); };
  if (T == 1 && st->single_launch) {
    moe::Decode1Stack& a = *st->args;
    const size_t pl = (size_t)st->grid * st->E;
    for (int l = 0; l < n; ++l) {
      moe::Decode1Args& d = a.layer[l];
      moe::fill_decode1_args(st->layers[l], x_of(l), out_of(l), nullptr, nullptr, &d);
      d.stack = 1;
      d.wr_next = l + 1 < n ? st->layers[l + 1]->w.router_w : nullptr;
      d.part_in = st->parts + (size_t)(l % 2) * pl;
      d.part_out = st->parts + (size_t)((l + 1) % 2) * pl;
      d.ctr = st->ctr;
      d.ctr_mod = (uint32_t)st->grid * 1024u;
      d.r.err = st->err;
      d.trace = st->layers[0]->trace;
    }
    a.n_layers = n;
    a.trace_layer = n > 1 ? 1 : 0;
    const moe_layer* L0 = st->layers[0];
    const cudaError_t e = moe::launch_decode1_stack(a, st->grid, s, s != nullptr && L0->pdl && L0->decode_pdl);
    if (e != cudaSuccess) return cuda_err(e, "stack decode launch");
    for (moe_layer* L : st->layers) {
      L->last_T = 1;
      L->last_single = true;
      L->stats.forward_calls += 1;
      L->stats.tokens += 1;
    }
    return MOE_OK;
  }
  for (int l = 0; l < n; ++l) {
    const moe_status_t r = moe_layer_forward(st->layers[l], x_of(l), T, out_of(l), nullptr, nullptr, stream);
    if (r != MOE_OK) return r;
  }
  return MOE_OK;
}

moe_status_t moe_stack_sync(moe_stack_t* st, void* stream) {
  if (!st) return moe::set_error(MOE_ERR_INVALID_ARG, "stack must not be NULL");
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_err(e, "stream synchronize");
  uint32_t word = 0;
  e = cudaMemcpy(&word, st->err, 4, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_err(e, "error word read");
  if (word != 0u) {
    cudaMemset(st->err, 0, 4);
    cudaDeviceSynchronize();
    if (word == 1) return moe::set_error(MOE_ERR_TIMEOUT, "a device-side wait gave up (error word %u)", word);
    return moe::set_error(MOE_ERR_INTERNAL, "device-side check failed (error word %u)", word);
  }
  for (moe_layer* L : st->layers) {
    const moe_status_t r = moe_layer_sync(L, stream);
    if (r != MOE_OK) return r;
  }
  return MOE_OK;
}

int32_t moe_stack_single_launch(const moe_stack_t* st) { return st && st->single_launch ? 1 : 0; }

moe_status_t moe_stack_destroy(moe_stack_t* st) {
  free_stack(st);
  return MOE_OK;
}

}  // extern "C"
