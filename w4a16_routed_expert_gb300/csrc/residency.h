// Partial residency (library-owned slot pool filled from pinned host backing).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "moe_layer.h"

struct moe_layer;

namespace moe {

struct Residency;

moe_status_t residency_create(const moe_layer_config_t& cfg, size_t record_bytes, int n_records,
                              const void* host_backing, Residency** out);
void residency_destroy(Residency* r);
const char* residency_last_error();
moe_status_t residency_forward(Residency* r, moe_layer* L, const __half* x, int T, __half* out, cudaStream_t s);
void residency_fill_stats(Residency* r, moe_layer_stats_t* st);
// Prefetch: the side stream the guess is routed on, the event the caller
// records once the guess input is ready, and the read-back of the guess's
// expert counts (its routing already enqueued on the side stream) handed to
// the handle's worker thread, which plans the copies. A forward's routing
// is ordered after an enqueued guess's routing (they share the handle's
// routing buffers) by residency_before_route on the forward's stream.
cudaStream_t residency_side(Residency* r);
cudaEvent_t residency_input_event(Residency* r);
moe_status_t residency_prefetch(Residency* r, moe_layer* L, int T);
cudaError_t residency_before_route(Residency* r, cudaStream_t s);

}  // namespace moe
