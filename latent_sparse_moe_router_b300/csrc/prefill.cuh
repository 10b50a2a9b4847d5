// Prefill path (T > 16) of the latent-MoE layer.
#pragma once

#include "../../include/edge0_moe.h"
#include "common.cuh"

namespace edge0 {

struct PrefillWorkspace {
  int max_tokens = 0;
  // routing outputs (owned by the handle's common workspace)
  int* idx = nullptr; float* w = nullptr; int* counts = nullptr; int* offsets = nullptr;
  int* perm = nullptr; int* pos = nullptr;
  int* err = nullptr;
  void* scratch = nullptr;
};

size_t prefill_workspace_bytes(const edge0_moe_desc& d, int max_tokens);
void prefill_workspace_carve(const edge0_moe_desc& d, int max_tokens, char* base, PrefillWorkspace* pf);
cudaError_t prefill_init(const edge0_moe_desc& d, PrefillWorkspace* pf, int num_sms);
edge0_status prefill_forward(const edge0_moe_desc& d, PrefillWorkspace* pf, int num_sms,
                             const __nv_bfloat16* x, __nv_bfloat16* y, int T, cudaStream_t s);
const void* prefill_debug_tensor(const PrefillWorkspace* pf, int what, const edge0_moe_desc& d, int T,
                                 size_t* bytes);
__nv_bfloat16* prefill_stack_scratch(PrefillWorkspace* pf);
void prefill_destroy(PrefillWorkspace* pf);

}  // namespace edge0
