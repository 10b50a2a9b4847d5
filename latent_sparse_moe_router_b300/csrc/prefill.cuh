// Prefill path (T > 16) of the latent-MoE layer: dense tensor-core GEMMs for the
// latent and router projections and for U, routing and permutation kernels, and
// grouped NVFP4 tensor-core GEMMs for the experts.
#pragma once

#include "../../include/edge0_moe.h"
#include "grouped.cuh"

namespace edge0 {

struct PrefillWorkspace {
  int max_tokens = 0;
  // routing outputs (owned by the handle's common workspace)
  int* idx = nullptr; float* w = nullptr; int* counts = nullptr; int* offsets = nullptr;
  int* perm = nullptr; int* pos = nullptr;
  int* err = nullptr;
  const float* rd = nullptr;        // folded router R D, fp32 [E][hidden] (handle-owned)
  float dnorm = 0.f;                // max_r sum_h |D[r][h]|
  // prefill buffers (carved from the handle's workspace)
  __nv_bfloat16* rdcat = nullptr;   // [2E][hidden]: rows 2e, 2e+1 = bf16 high / low parts of R D row e
  __half* zh = nullptr;             // [T][G latent]  z * 2^-e_t in f16 (e_t: exponent of the bound
                                    //               dnorm * max|x_t| of |z_t|, so |z * 2^-e_t| < 1)
  float* zsc = nullptr;             // [T] 2^-e_t
  float* zinv = nullptr;            // [T] 2^e_t
  float* pos_inv = nullptr;         // [T K + T] 2^e_t of the token at each grouped position
  float* logits = nullptr;          // [T][E]
  int* chunk_cnt = nullptr;         // [T/64][E] per-chunk expert counts, then per-chunk bases
  int* tprefix = nullptr;           // [E+2] token-tile prefix of the expert groups (+ shared)
  __half* zg = nullptr;             // [T K][latent] zh rows in expert-grouped order
  __nv_bfloat16* hb = nullptr;      // [T K + T][ffn] SwiGLU activations (routed, then shared)
  __nv_bfloat16* ob = nullptr;      // [T K + T][latent] expert outputs (routed, then shared)
  __nv_bfloat16* cb = nullptr;      // [T][G latent] combined latent (G latent groups)
  __nv_bfloat16* scratch = nullptr; // [T][hidden] layer output for stacked calls
  float* upart = nullptr;           // [splits][min(T, 768)][hidden] fp32 partial sums of a K-split U GEMM
  int* abort = nullptr;             // per-forward abort word of the bounded waits
  // stage timing (profiling): events[0] before the first kernel, events[i + 1]
  // after stage i
  bool profile = false;
  bool timed = false;               // the last forward recorded the events
  cudaEvent_t events[11] = {};
  // tensor maps fixed for the handle's lifetime
  CUtensorMap m_D, m_rdcat, m_U, m_cb;
  GgMaps maps1, maps2;
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
cudaError_t prefill_profile(PrefillWorkspace* pf, bool enable);
edge0_status prefill_stage_times(PrefillWorkspace* pf, float* ms, int max, int* n_out);

}  // namespace edge0
