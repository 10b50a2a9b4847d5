// Decode path (T <= 16) of the latent-MoE layer: one persistent cooperative kernel.
//
// The layer ("Edge0-145B · Q3_K" model card, section "Architecture"; "Edge0-145B
// hardware requirements", section "Edge0-145B latent MoE architecture"):
//   z = D x;  l = R z + b;  top-k + renormalised softmax;  o_e = W_d (silu(W_g z) * W_up z);
//   c = o_shared + sum_k w_k o_k;  y = U c.
// At T <= 16 every step is a matrix-vector product bound by HBM bandwidth and each
// step needs all of the previous one.  One CTA per SM runs four phases separated by
// software grid barriers (the minimum for this dependency chain):
//   P0  z = D x and l = (R D) x + b     R D is folded once, in fp32, when the handle
//                                        is created, so the router needs no phase of its own
//   P1  top-k + weights + permutation   redundantly per CTA, in shared memory
//       gate/up -> h                    rows of the union of the selected experts and
//                                        of the shared expert (staged during P0)
//   P2  down projections + combine -> c (the down rows are fetched during P1)
//   P3  y = U c                          (U rows: the end of the ring stream)
// Every product runs on m16n8k16 mma.sync with the tokens on N.  The expert rows move
// through a ring of shared-memory slots: each slot is one bulk-copied unit of work
// (8 gate/up row pairs in P1, a few experts' down rows and their h rows in P2, U rows
// for P3), the
// warp that finishes the last part of a unit refills its slot with the unit S places
// further on, and units of P1 and P2 form one stream, so that the first down units are
// in flight before P1 ends.  A stack of layers (residual + RMSNorm between them) runs
// in the same launch, each layer prefetching the next one's D and R D into L2.
#pragma once

#include "common.cuh"

namespace edge0 {

constexpr int kDecThreads = 512;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kMaxTopK = 16;
constexpr int kDecodeMaxT = 16;
constexpr int kMaxSlots = kDecodeMaxT * (kMaxTopK + 1);
constexpr int kNumMbar = 20;
constexpr int kTopkCand = 64;   // candidates per warp of the top-k (shared memory)
// mbarrier roles
constexpr int kMbRing = 0;       // 0..11: ring slots (P1 gate/up units, P2 down units)
constexpr int kRingMax = 12;
constexpr int kMbShared = 12;    // shared-expert gate/up rows (P0 -> P1)
constexpr int kMbP0 = 13;        // 13..16: P0 row tiles
constexpr int kP0Tiles = 4;
constexpr int kMbScale = 18;     // fp32 scales of the selected records (P1 -> P1, P2)
constexpr int kScaleWarp = 2;    // the warp that copies them (one arrival per lane)
constexpr int kPartCap = 24;     // P1 partial-sum entries (ring slots x parts of a unit)
constexpr int kPadElems = 32;    // row padding (16-bit elements) of x, zh and c in shared memory
constexpr int kConvPieces = 4;   // 16-byte pieces of an h row per lane in the down phase: F <= 1024

// Row pitches (bytes) of rows staged in shared memory: the padding puts rows g and
// g + 1 of an MMA fragment load in different bank groups.
__host__ __device__ constexpr int pitch_bf16_row(int K) { return K * 2 + 64; }
__host__ __device__ constexpr int pitch_f32_row(int K) { return K * 4 + 16; }
__host__ __device__ constexpr int pitch_gu_row(int L) { return 9 * L / 8 + 16; }

// Phase stamps of a profiled launch, per layer (ns of %globaltimer): CTA 0's time at
// each point, and the latest (max) / earliest (stored as ~t, max) phase end over all
// CTAs before each grid barrier.
enum DecStamp {
  kStP0Start = 0,    // CTA 0, start of P0 (after the kernel's set-up)
  kStP0EndMax, kStP0EndMin, kStBar1,        // P0 end over CTAs; CTA 0 after barrier 1
  kStRouted,                                // CTA 0, routing done (before the expert copies)
  kStP1EndMax, kStP1EndMin, kStBar2,
  kStP2EndMax, kStP2EndMin, kStBar3,
  kStP3EndMax, kStP3EndMin, kStBar4,        // barrier 4: stacks only
  kStRouteLoaded,                           // CTA 0: logits and zh in shared memory
  kStTopk,                                  // CTA 0: top-k and weights done
  kStP1Issued,                              // CTA 0: first gate/up units issued
  kStP2Staged,                              // CTA 0: h rows of the first down units requested
  kStP2Tasks,                               // CTA 0: all down units done
  kStampSlots = 24
};

// One layer's weights as the decode kernel sees them.
struct LayerW {
  const __nv_bfloat16* D;   // [L][H]
  const __nv_bfloat16* U;   // [H][L]
  const float* RD;          // [E][H] fp32: router folded with D (R D)
  const float* bias;        // [E] or null
  const uint8_t* experts;   // E records
  const uint8_t* shared;    // 1 record
  unsigned long long stride;
  float dnorm;              // max_r sum_h |D[r][h]|: bounds |z| / max|x|
  // residency tiering (all null when the layer's records are all in device memory):
  // record e is at rec_table[e], in device memory when resident[e] != 0, else in
  // host memory mapped into the device address space
  const uint8_t* const* rec_table;
  const uint8_t* resident;
  uint8_t* staging;         // device, >= T K records at `stride`: this forward's misses
  unsigned int* use;        // [E] selections per expert (the residency policy reads them)
  unsigned long long* tier_stats;  // [0] forwards, [1] misses, [2] bytes read from host memory
};

struct DecodeArgs {
  LayerW l0;                // the first layer (kernel parameter: no load before P0)
  const LayerW* layers;     // device array [n_layers]
  int n_layers;
  float eps;                // RMSNorm epsilon between layers
  int final_norm;           // 1: y = RMSNorm(x_last + y_last) (stack output)
  const __nv_bfloat16* x;   // [T][H]
  __nv_bfloat16* y;         // [T][H]
  int T;
  int H, L, E, K, F;
  // workspace
  float* z;                 // [T][L]
  __half* zh;               // [T][L] f16 copy of z * 2^-e_t (the experts' input)
  float* logits;            // [T][E]
  __nv_bfloat16* h;         // [T*K + T][F]  SwiGLU output: grouped positions, then the shared slot of each token
  float* c;                 // [T][L]
  __nv_bfloat16* ybuf;      // [2][T][H] layer outputs inside a stack
  __nv_bfloat16* xbuf;      // [2][T][H] normalised layer inputs inside a stack
  int* idx; float* w; int* counts; int* offsets; int* perm; int* pos;  // last layer's routing
  __nv_bfloat16* trace_x;   // optional [n_layers][T][H]: input of every layer
  __nv_bfloat16* trace_y;   // optional [n_layers][T][H]: output of every layer
  int* trace_idx;           // optional [n_layers][T][K]: experts each layer picked, in rank order
  const float* dnorm_dev;   // optional: device copy of the first layer's dnorm (used in place of l0.dnorm)
  unsigned long long* stamps; // optional [n_layers][kStampSlots] %globaltimer phase stamps (zeroed before launch)
  GridBarrier* bar;
  int* err;
  // shared-memory plan (bytes from the 128-aligned dynamic base)
  int off_sh, sh_bytes;     // shared-expert gate/up rows of this CTA (pitch pitch_gu_row)
  int off_a, a_bytes;       // phase-local arrays: x (P0), zh + partial sums (P1),
                            // per-slot down outputs (P2), c in bf16 (P3)
  int off_ring, ring_bytes; // staged weights: P0 rows, the P1/P2 ring; the logits during
                            // routing; per-warp partial sums (P0, P3)
  int ring_slots, slot_bytes;
};

// Tables at the start of dynamic shared memory.
struct alignas(16) DecTables {
  uint64_t mbar[kNumMbar];
  int idx[kDecodeMaxT * kMaxTopK];
  float w[kDecodeMaxT * kMaxTopK];
  int perm[kDecodeMaxT * kMaxTopK];     // grouped position -> slot
  int posn[kDecodeMaxT * kMaxTopK];     // slot -> grouped position
  short tokp[kDecodeMaxT * kMaxTopK];   // grouped position -> token
  int gexp[kDecodeMaxT * kMaxTopK];     // distinct experts, ascending
  const uint8_t* gptr[kDecodeMaxT * kMaxTopK];  // record of each distinct expert for this forward
  int gmiss[kDecodeMaxT * kMaxTopK];    // tiering: staging index of a non-resident expert, else -1
  int mgrp[kDecodeMaxT * kMaxTopK];     // tiering: group of staging record m
  int n_miss;                            // tiering: non-resident experts of this forward
  int goff[kDecodeMaxT * kMaxTopK + 1]; // group g = perm[goff[g] .. goff[g+1])
  int nu;                                // number of distinct experts
  int stuck;                             // bit b: a wait on mbar[b] ran out
  int pair_ctr[2];                       // next (unit, part) of P1 / P2
  int ring_cnt[kRingMax];                // parts of units finished on each slot (this phase)
  int ring_gen[kRingMax];                // units finished on each slot (this layer)
  int p2_ready;                          // the P2 unit table is built
  int n2;                                // P2 units of this CTA
  int p2_gmax;                           // the most groups in one P2 unit
  float zsc[kDecodeMaxT], zinv[kDecodeMaxT];
  float4 gsc[kDecodeMaxT * kMaxTopK + 1];  // (gate, up, down, -) fp32 scales of group j:
                                         // j = 0 the shared expert, j >= 1 expert gexp[j - 1]
  float red[kDecWarps * kDecodeMaxT];
  float inv_rms[kDecodeMaxT];
  // P2 units: unit k takes the slots q in [p2_qa[k], p2_qa[k + 1]) of the order
  // (shared slots of tokens 0..T-1, then grouped positions), groups [p2_ja[k], p2_jb[k])
  short p2_qa[kMaxSlots + 1];
  short p2_ja[kMaxSlots];
  short p2_jb[kMaxSlots];
};

size_t decode_tables_bytes();

}  // namespace edge0
