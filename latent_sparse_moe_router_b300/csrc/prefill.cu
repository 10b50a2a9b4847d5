// Prefill path (T > 16): not built yet in this revision; forward returns UNSUPPORTED.
#include "prefill.cuh"

namespace edge0 {

size_t prefill_workspace_bytes(const edge0_moe_desc&, int) { return 0; }
void prefill_workspace_carve(const edge0_moe_desc&, int max_tokens, char*, PrefillWorkspace* pf) {
  pf->max_tokens = max_tokens;
}
cudaError_t prefill_init(const edge0_moe_desc&, PrefillWorkspace*, int) { return cudaSuccess; }
edge0_status prefill_forward(const edge0_moe_desc&, PrefillWorkspace*, int, const __nv_bfloat16*,
                             __nv_bfloat16*, int, cudaStream_t) {
  return EDGE0_ERR_UNSUPPORTED;
}
const void* prefill_debug_tensor(const PrefillWorkspace*, int, const edge0_moe_desc&, int, size_t*) {
  return nullptr;
}
__nv_bfloat16* prefill_stack_scratch(PrefillWorkspace*) { return nullptr; }
void prefill_destroy(PrefillWorkspace*) {}

}  // namespace edge0
