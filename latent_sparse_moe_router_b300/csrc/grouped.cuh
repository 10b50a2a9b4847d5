// Grouped NVFP4 x bf16 GEMMs of the routed and shared experts (prefill path).
//
// The experts of the latent-MoE layer run l -> 640 -> l as SwiGLU FFNs on NVFP4
// weights ("Edge0-145B · Q3_K" model card, section "Architecture"; NVFP4 per
// "Edge0-145B en local", introduction).  Tokens are grouped by expert (positions
// p of the permutation); a work tile is (group g, token tile nt, weight tile mt),
// and a cluster of two CTAs on two SMs (a pair) runs the weight tiles 2u, 2u + 1 of
// one token tile of up to 256 rows as tcgen05.mma.cta_group::2 with the tokens on
// the MMA's M side (128 rows per CTA, so each TMEM lane is one token) and the
// weights on its N side (256: the two CTAs' dequantised tiles of 128 rows):
//   MODE 1 (gate/up): weight tile = 64 gate rows + 64 up rows (f0 = 64 mt), token
//     rows = z * 2^-e_t in f16 of the group, K = l; f16 operands; epilogue
//     h = silu(g_gate 2^e_t gate) * (g_up 2^e_t up), stored bf16 to H[p][f].
//   MODE 2 (down):    weight tile = 128 latent rows (r0 = 128 mt, 64 row pairs),
//     token rows = rows of H, K = F; epilogue o = g_down * acc, stored bf16 to O[p][r].
// Persistent pairs (one CTA per SM) walk the pair tiles in index order with a
// stride of the number of pairs, pair tile = (token tile, weight-tile pair u) with
// u fastest, so the pairs working at one time share a few token tiles through L2.
// CTA r of a pair owns weight tile 2u + r (it dequantises those 128 rows: columns
// 128 r .. 128 r + 127 of the MMA's N) and token rows 128 r .. 128 r + 127 of the
// tile (its accumulator lanes).  Warp roles in both CTAs:
//   warp 0 (one lane): TMA producer of the tile's E4M3 scales (double-buffered)
//     and raw NVFP4 codes (4 KB per 64-wide k-step, 6-deep ring);
//   warp 18 (one lane): TMA producer of this CTA's 128 token rows (64-row boxes,
//     128-byte swizzle; boxes wholly past the tile's rows skipped), into the stages
//     the MMA releases; completion on rank 0's barrier;
//   warp 1 (one lane, rank 0 only): tcgen05.mma.cta_group::2, M=256 (tokens),
//     N=256 (weights), K=16, into one of two TMEM accumulators of 256 columns in
//     each CTA; commits arrive in both CTAs;
//   warps 2-9: dequantisation, two threads per weight row, exact: mode 1 E2M1 -> f16
//     by cvt times the E4M3 scale in one f16x2 multiply; mode 2 the same f16
//     moved to the bf16 exponent range with shift/mask and multiplied by the
//     block scale * 2^112 in bf16x2; into 128-byte-swizzled tiles; each warp
//     then arrives on rank 0's stage barrier;
//   warps 10-17: epilogue of the previous accumulator (TMEM lane = token; two warps
//     per TMEM lane quarter, one per half of the 256 weight columns; each warp's 32
//     token rows staged in a padded buffer and stored as whole 16-byte pieces of
//     their output rows) while the next tile's main loop runs; each warp then arrives
//     on rank 0's accumulator barrier.
#pragma once

#include "pair.cuh"

namespace edge0 {

constexpr int kGgThreads = 608;  // 19 warps
constexpr int kGgDqWarp0 = 2;     // dequantisation warps 2..9
constexpr int kGgDqThreads = 256;
constexpr int kGgDqWarps = 8;
constexpr int kGgEpWarp0 = 10;    // epilogue warps 10..17
constexpr int kGgEpThreads = 256;
constexpr int kGgBWarp = 18;      // B-tile producer
constexpr int kGgBN = 256;        // token tile
constexpr int kGgSA = 4;          // A (dequantised weight) stages
constexpr int kGgSB = 4;          // B (token row) stages
constexpr int kGgR = 6;           // raw code stages

struct GgSmem {
  static constexpr int kA = 128 * 64 * 2;        // 16 KB
  static constexpr int kB = kGgBN / 2 * 64 * 2;  // 16 KB: this CTA's half of the token rows
  static constexpr int kRaw = 128 * 32;          // 4 KB
  static constexpr int kSc = 16384;              // scales of one tile (<= 128 rows x 128 B)
  static constexpr int kEpiPitch = 80;           // bytes per token row of an epilogue warp's staging
  static constexpr int kEpi = 8 * 32 * kEpiPitch;  // 8 epilogue warps x 32 token rows
  static constexpr int offA = 0;
  static constexpr int offB = offA + kGgSA * kA;
  static constexpr int offRaw = offB + kGgSB * kB;
  static constexpr int offSc = offRaw + kGgR * kRaw;
  static constexpr int offEpi = offSc + 2 * kSc;
  static constexpr int offBar = offEpi + kEpi;
  static constexpr int kBytes = offBar + 1024 + 1024;  // barriers + alignment slack
};

struct GgParams {
  int mode;                 // 1 gate/up, 2 down
  int T, TK, L, F, E;
  int mtiles;               // weight tiles per group (F/64 or L/128; even)
  const int* counts;        // [E]   tokens per routed expert
  const int* offsets;       // [E+1] first position of each routed expert
  const int* tprefix;       // [E+2] first token tile of each group (group E = shared)
  const uint8_t* experts;   // records (for the fp32 per-matrix scales)
  unsigned long long stride;
  const uint8_t* shared;
  __nv_bfloat16* out;       // H [TK+T][F] (mode 1) or O [TK+T][L] (mode 2)
  int out_ld;
  const float* pos_inv;     // mode 1: [TK+T] inverse scale of the f16 z row at each position
  int* err;
  int* abort;               // set when any wait gives up; every CTA then winds down
};

struct GgMaps {
  CUtensorMap a_codes;      // routed records: 3-D (bytes of a row, rows, expert)
  CUtensorMap a_scales;
  CUtensorMap s_codes;      // shared record: 2-D
  CUtensorMap s_scales;
  CUtensorMap b_routed;     // mode 1: gathered z rows [TK][L]; mode 2: H [TK+T][F]
  CUtensorMap b_shared;     // mode 1: z rows [T][L]; mode 2: H again (shared rows from TK)
};

}  // namespace edge0
