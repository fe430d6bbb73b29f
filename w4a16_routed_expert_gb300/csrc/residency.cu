// Partial residency: placeholder until the slot pool lands.
#include "residency.h"

namespace moe {

struct Residency {
  int unused;
};

moe_status_t residency_create(const moe_layer_config_t&, size_t, int, const void*, Residency** out) {
  *out = nullptr;
  return MOE_ERR_UNSUPPORTED;
}
void residency_destroy(Residency* r) { delete r; }
const char* residency_last_error() { return "partial residency is not built yet"; }
moe_status_t residency_forward(Residency*, moe_layer*, const __half*, int, __half*, cudaStream_t) {
  return MOE_ERR_UNSUPPORTED;
}
void residency_fill_stats(const Residency*, moe_layer_stats_t*) {}

}  // namespace moe
