// Decode path (T <= 16) of the latent-MoE layer: one persistent cooperative kernel.
//
// The layer ("Edge0-145B · Q3_K" model card, section "Architecture"; "Edge0-145B
// hardware requirements", section "Edge0-145B latent MoE architecture"):
//   z = D x;  l = R z + b;  top-k + renormalised softmax;  o_e = W_d (silu(W_g z) * W_up z);
//   c = o_shared + sum_k w_k o_k;  y = U c.
// At T <= 16 every step is a GEMV bound by HBM bandwidth, and each step needs all
// of the previous one (z before the router, the routing before the routed
// experts, every h before the down projection, all of c before U).  So one CTA
// per SM runs five phases separated by software grid barriers:
//   P0  z = D x            (D rows of this CTA; L2 prefetch of R, U, shared record)
//   P1  logits = R z + b;  shared expert gate/up -> h_shared
//   P2  top-k + weights + permutation (redundantly per CTA, in shared memory);
//       routed gate/up -> h (rows of the union of selected experts);
//       L2 prefetch of the selected experts' down matrices
//   P3  down projections of every used expert for this CTA's latent rows; combine -> c
//   P4  y = U c
// Each CTA stages its slab of weights in shared memory with bulk copies
// (cp.async.bulk, completion on mbarriers) and dequantises NVFP4 in registers.
// A stack of layers (residual + RMSNorm between them) runs in the same launch.
#pragma once

#include "common.cuh"

namespace edge0 {

constexpr int kDecThreads = 512;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kMaxTopK = 16;
constexpr int kDecodeMaxT = 16;
constexpr int kMaxBatches = 8;  // mbarriers per round

// One layer's weights as the decode kernel sees them.
struct LayerW {
  const __nv_bfloat16* D;   // [L][H]
  const __nv_bfloat16* U;   // [H][L]
  const __nv_bfloat16* R;   // [E][L]
  const float* bias;        // [E] or null
  const uint8_t* experts;   // E records
  const uint8_t* shared;    // 1 record
  unsigned long long stride;
};

struct DecodeArgs {
  const LayerW* layers;     // device array [n_layers]
  int n_layers;
  float eps;                // RMSNorm epsilon between layers
  const __nv_bfloat16* x;   // [T][H]
  __nv_bfloat16* y;         // [T][H]
  int T;
  int H, L, E, K, F;
  // workspace
  float* z;                 // [T][L]
  float* logits;            // [T][E]
  float* h;                 // [T*K + T][F]  routed slots, then the shared slot of each token
  unsigned int* hmax;       // [T*K + T]     max |h| per slot (float bits)
  float* c;                 // [T][L]
  __nv_bfloat16* ybuf;      // [2][T][H] layer outputs inside a stack
  __nv_bfloat16* xbuf;      // [T][H]    normalised input of the current layer (debug)
  int* idx; float* w; int* counts; int* offsets; int* perm; int* pos;  // last layer's routing
  __nv_bfloat16* trace_x;   // optional [n_layers][T][H]: input of every layer
  __nv_bfloat16* trace_y;   // optional [n_layers][T][H]: output of every layer
  GridBarrier* bar;
  int* err;
  // shared-memory plan (bytes from the dynamic base)
  int off_act, act_bytes;   // x bf16 / z fp32 / c fp32 / h f16 (P3, together with zh)
  int off_zh;               // zh f16 [T][L] (directly after act)
  int off_slab, slab_bytes; // staged weights
  int off_res, res_rows;    // gate/up dot results: 2 x res_rows x TB fp32
};

// Shared tables at the start of dynamic shared memory.
struct alignas(16) DecTables {
  uint64_t mbar[kMaxBatches];
  int idx[kDecodeMaxT * kMaxTopK];
  float w[kDecodeMaxT * kMaxTopK];
  int perm[kDecodeMaxT * kMaxTopK];     // grouped position -> slot
  int posn[kDecodeMaxT * kMaxTopK];     // slot -> grouped position
  int gexp[kDecodeMaxT * kMaxTopK];     // distinct experts, ascending
  int goff[kDecodeMaxT * kMaxTopK + 1]; // group g = perm[goff[g] .. goff[g+1])
  int nu;                                // number of distinct experts
  int mb_phase;                          // parity bits of mbar[] (uniform)
  int stuck;                             // bit b: a wait on mbar[b] ran out
  int round_nb;                          // batches of the current round
  float zsc[kDecodeMaxT], zinv[kDecodeMaxT];
  float hsc[kDecodeMaxT * (kMaxTopK + 1)], hinv[kDecodeMaxT * (kMaxTopK + 1)];
  float red[kDecWarps * kDecodeMaxT];
  float inv_rms[kDecodeMaxT];
  // per-round task tables
  int task_row[512];                     // generic per-round row descriptors
  int task_aux[512];
  unsigned int task_off[512];
  unsigned int task_off2[512];
};

size_t decode_tables_bytes();

}  // namespace edge0
