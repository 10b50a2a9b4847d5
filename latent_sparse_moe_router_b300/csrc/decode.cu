// Decode path (T <= 16): persistent cooperative kernel, one CTA per SM.
// Phase structure and data flow are described in decode.cuh.
#include "decode.cuh"

#include <math.h>

namespace edge0 {

size_t decode_tables_bytes() { return (sizeof(DecTables) + 127) & ~size_t(127); }

namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float silu_f(float v) { return v / (1.0f + expf(-v)); }

// ------------------------------------------------------------------ mbarrier bookkeeping
struct Ctx {
  DecTables* tb;
  int* err;
  uint32_t mbp;  // parity bits of tb->mbar (identical in every thread)
};

// Wait for the current phase of mbarrier b (idempotent until the phase is released).
__device__ __forceinline__ void wait_mb(Ctx& cx, int b) {
  if (!mbar_wait(&cx.tb->mbar[b], (cx.mbp >> b) & 1u, cx.err)) atomicOr(&cx.tb->stuck, 1 << b);
}
// Release the barriers in `mask` after their use (all threads, uniformly).
__device__ __forceinline__ void release_mb(Ctx& cx, uint32_t mask) { cx.mbp ^= mask; }

// ------------------------------------------------------------------ dot products
template <int TB>
__device__ __forceinline__ void group_reduce(float* acc, int nl) {
#pragma unroll
  for (int i = 0; i < TB; ++i)
    for (int o = nl >> 1; o > 0; o >>= 1) acc[i] += __shfl_xor_sync(kFull, acc[i], o);
}

// 8 consecutive activation values of row t as fp32 (bf16 or fp32 storage).
template <bool ACT_F32>
__device__ __forceinline__ void act8(const void* act, int K, int t, int c, float* af) {
  if (ACT_F32) {
    const float4* ap = reinterpret_cast<const float4*>(static_cast<const float*>(act) + size_t(t) * K);
    const float4 a0 = ap[2 * c], a1 = ap[2 * c + 1];
    af[0] = a0.x; af[1] = a0.y; af[2] = a0.z; af[3] = a0.w;
    af[4] = a1.x; af[5] = a1.y; af[6] = a1.z; af[7] = a1.w;
  } else {
    const uint4 av = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(act) + size_t(t) * K)[c];
    af[0] = bf16_lo(av.x); af[1] = bf16_hi(av.x); af[2] = bf16_lo(av.y); af[3] = bf16_hi(av.y);
    af[4] = bf16_lo(av.z); af[5] = bf16_hi(av.z); af[6] = bf16_lo(av.w); af[7] = bf16_hi(av.w);
  }
}

// acc[t] += W_row . act[t] over K; weights bf16 (W_F32 = false) or fp32, in shared
// memory; lanes l, l+nl, ... of an aligned group of nl lanes, 8 elements per step.
template <int TB, bool W_F32, bool ACT_F32>
__device__ __forceinline__ void row_dot(const uint8_t* wrow, int K, const void* act, int T, int l,
                                        int nl, float* acc) {
  for (int c = l; c < K / 8; c += nl) {
    float wf[8];
    if (W_F32) {
      const float4* wp = reinterpret_cast<const float4*>(wrow);
      const float4 w0 = wp[2 * c], w1 = wp[2 * c + 1];
      wf[0] = w0.x; wf[1] = w0.y; wf[2] = w0.z; wf[3] = w0.w;
      wf[4] = w1.x; wf[5] = w1.y; wf[6] = w1.z; wf[7] = w1.w;
    } else {
      const uint4 wv = reinterpret_cast<const uint4*>(wrow)[c];
      wf[0] = bf16_lo(wv.x); wf[1] = bf16_hi(wv.x); wf[2] = bf16_lo(wv.y); wf[3] = bf16_hi(wv.y);
      wf[4] = bf16_lo(wv.z); wf[5] = bf16_hi(wv.z); wf[6] = bf16_lo(wv.w); wf[7] = bf16_hi(wv.w);
    }
#pragma unroll
    for (int t = 0; t < TB; ++t) {
      if (t < T) {
        float af[8];
        act8<ACT_F32>(act, K, t, c, af);
        float s0 = wf[0] * af[0], s1 = wf[1] * af[1];
#pragma unroll
        for (int i = 2; i < 8; i += 2) {
          s0 = fmaf(wf[i], af[i], s0);
          s1 = fmaf(wf[i + 1], af[i + 1], s1);
        }
        acc[t] += s0 + s1;
      }
    }
  }
}

// acc[i] += sum_k e2m1(code[k]) * e4m3(scale[k/16]) * act_i[k] for n activation
// rows (f16, pre-scaled).  Lane l of a group of nl lanes takes blocks l, l+nl, ...
// Products of one 16-block are summed in f16x2 (two chains of 4 per half); the
// block sum is scaled and accumulated in fp32.  With TB == 1 the single activation
// row is used unconditionally (callers pass a valid row when n == 0).
template <int TB>
__device__ __forceinline__ void fp4_dot(const uint8_t* codes, const uint8_t* scales, int nblk,
                                        const __half* const* arow, int n, int l, int nl,
                                        float* acc) {
#pragma unroll 2
  for (int b = l; b < nblk; b += nl) {
    const uint2 cw = reinterpret_cast<const uint2*>(codes)[b];
    const float s = e4m3_to_f32(scales[b]);
    __half2 wv[8];
    wv[0] = u32_as_h2(e2m1x2_to_h2(cw.x & 0xFF));
    wv[1] = u32_as_h2(e2m1x2_to_h2((cw.x >> 8) & 0xFF));
    wv[2] = u32_as_h2(e2m1x2_to_h2((cw.x >> 16) & 0xFF));
    wv[3] = u32_as_h2(e2m1x2_to_h2(cw.x >> 24));
    wv[4] = u32_as_h2(e2m1x2_to_h2(cw.y & 0xFF));
    wv[5] = u32_as_h2(e2m1x2_to_h2((cw.y >> 8) & 0xFF));
    wv[6] = u32_as_h2(e2m1x2_to_h2((cw.y >> 16) & 0xFF));
    wv[7] = u32_as_h2(e2m1x2_to_h2(cw.y >> 24));
#pragma unroll
    for (int i = 0; i < TB; ++i) {
      if (TB == 1 || i < n) {
        const uint4* ap = reinterpret_cast<const uint4*>(arow[i] + b * 16);
        const uint4 a0 = ap[0], a1 = ap[1];
        __half2 p = __hmul2(wv[0], u32_as_h2(a0.x));
        __half2 q = __hmul2(wv[4], u32_as_h2(a1.x));
        p = __hfma2(wv[1], u32_as_h2(a0.y), p);
        q = __hfma2(wv[5], u32_as_h2(a1.y), q);
        p = __hfma2(wv[2], u32_as_h2(a0.z), p);
        q = __hfma2(wv[6], u32_as_h2(a1.z), q);
        p = __hfma2(wv[3], u32_as_h2(a0.w), p);
        q = __hfma2(wv[7], u32_as_h2(a1.w), q);
        const float2 f = __half22float2(p);
        const float2 g = __half22float2(q);
        acc[i] = fmaf(s, (f.x + f.y) + (g.x + g.y), acc[i]);
      }
    }
  }
}

// ------------------------------------------------------------------ dense rows (bf16 / fp32)
// Up to two row ranges of row-major matrices, staged in the dynamic region by bulk
// copies (<= kMbRounds batches per round) and reduced by one half-warp per row:
// out_fn(m, t, row, value) with m the matrix index.
struct RowSet {
  const uint8_t* base;   // matrix m, row-major
  int r0, r1;            // rows of this CTA
  int row_bytes;         // K * element size
  int f32;               // 1: fp32 weights, 0: bf16
};

// Rows of a round [from, from + n) of the concatenated row list: set-0 rows first.
struct RoundRows {
  int c0;      // rows of set 0 in the round
  int rb0, rb1;
  int from, n, nb;
  __device__ __forceinline__ uint32_t offset(int i) const {
    return i < c0 ? uint32_t(i) * rb0 : uint32_t(c0) * rb0 + uint32_t(i - c0) * rb1;
  }
  __device__ __forceinline__ int batch(int i) const {
    int b = 0;
    while (i >= n * (b + 1) / nb) ++b;
    return b;
  }
};

__device__ __forceinline__ RoundRows round_rows(const RowSet* rs, int nset, int from, int n) {
  RoundRows rr;
  const int n0 = rs[0].r1 - rs[0].r0;
  rr.c0 = max(0, min(from + n, n0) - from);
  rr.rb0 = rs[0].row_bytes;
  rr.rb1 = nset > 1 ? rs[1].row_bytes : rs[0].row_bytes;
  rr.from = from;
  rr.n = n;
  rr.nb = min(kMbRounds, n);
  return rr;
}

// Lanes of warp 0: bulk copies of a round, lane b one batch (<= 2 copies: one
// per set piece).  Call from all 32 lanes of warp 0.
__device__ void stage_rows(Ctx& cx, const RowSet* rs, int nset, int from, int n, uint8_t* dst) {
  const RoundRows rr = round_rows(rs, nset, from, n);
  const int n0 = rs[0].r1 - rs[0].r0;
  const int b = threadIdx.x & 31;
  if (b < rr.nb) {
    const int i0 = n * b / rr.nb, i1 = n * (b + 1) / rr.nb;
    mbar_arrive_expect_tx(&cx.tb->mbar[kMbRound + b], rr.offset(i1) - rr.offset(i0));
    // set 0 piece [i0, min(i1, c0)), set 1 piece [max(i0, c0), i1)
    if (i0 < rr.c0) {
      const int ie = min(i1, rr.c0);
      const int row = rs[0].r0 + from + i0;
      bulk_g2s(dst + rr.offset(i0), rs[0].base + size_t(row) * rr.rb0, uint32_t(ie - i0) * rr.rb0,
               &cx.tb->mbar[kMbRound + b]);
    }
    if (i1 > rr.c0) {
      const int ia = max(i0, rr.c0);
      const int row = rs[1].r0 + (from + ia - n0);
      bulk_g2s(dst + rr.offset(ia), rs[1].base + size_t(row) * rr.rb1, uint32_t(i1 - ia) * rr.rb1,
               &cx.tb->mbar[kMbRound + b]);
    }
  }
}

__device__ __forceinline__ int dense_cap(const RowSet* rs, int nset, int dyn_bytes) {
  int maxrb = 0;
  for (int m = 0; m < nset; ++m) maxrb = max(maxrb, rs[m].row_bytes);
  return min(512, dyn_bytes / maxrb);
}

// Rows of the sets, round by round, one warp per row; out_fn(m, t, row, v).
// With `prestaged`, warp 0 already ran stage_rows for the first round
// (rows [0, min(cap, total))) before the CTA's last __syncthreads.
template <int TB, bool ACT_F32, class OutFn>
__device__ void dense_rows(Ctx& cx, const RowSet* rs, int nset, const void* act, int K, int T,
                           uint8_t* dyn, int dyn_bytes, bool prestaged, OutFn out_fn) {
  const int wv = threadIdx.x >> 5, wl = threadIdx.x & 31;
  int total = 0;
  for (int m = 0; m < nset; ++m) total += rs[m].r1 - rs[m].r0;
  const int n0 = rs[0].r1 - rs[0].r0;
  const int cap = dense_cap(rs, nset, dyn_bytes);
  if (cap < 1) {   // not even one row fits (the host rejects such shapes): stop, do not spin
    if (threadIdx.x == 0 && total > 0) atomicOr(cx.err, kErrTimeout);
    return;
  }
  for (int from = 0; from < total; from += cap) {
    const int n = min(cap, total - from);
    if (!(prestaged && from == 0)) {
      if (threadIdx.x < 32) stage_rows(cx, rs, nset, from, n, dyn);
    }
    const RoundRows rr = round_rows(rs, nset, from, n);
    for (int i = wv; i < n; i += kDecWarps) {
      const int m = i >= rr.c0 ? 1 : 0;
      wait_mb(cx, kMbRound + rr.batch(i));
      float acc[TB];
#pragma unroll
      for (int t = 0; t < TB; ++t) acc[t] = 0.f;
      const uint8_t* wrow = dyn + rr.offset(i);
      if (rs[m].f32) row_dot<TB, true, ACT_F32>(wrow, K, act, T, wl, 32, acc);
      else row_dot<TB, false, ACT_F32>(wrow, K, act, T, wl, 32, acc);
      group_reduce<TB>(acc, 32);
      if (wl == 0) {
        const int q = from + i;
        const int row = q < n0 ? rs[0].r0 + q : rs[1].r0 + (q - n0);
#pragma unroll
        for (int t = 0; t < TB; ++t)
          if (t < T) out_fn(m, t, row, acc[t]);
      }
    }
    for (int b = 0; b < rr.nb; ++b) wait_mb(cx, kMbRound + b);
    __syncthreads();
    release_mb(cx, (1u << rr.nb) - 1u);
  }
}

// ------------------------------------------------------------------ top-k (tree of warp sorts)
// The k largest of E logits by (value descending, index ascending).  Chunks of 32
// experts are sorted across the lanes of a warp (bitonic network over shuffles);
// sorted top-16 lists are then merged pairwise (bitonic merge) level by level.
struct Cand {
  float v;
  int i;
};

__device__ __forceinline__ bool cand_first(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// Top-k of one token's E logits (E a multiple of 32, in shared memory) by one warp,
// ranked by (value descending, index ascending); a NaN logit ranks as -inf.
// tau, the K-th largest of the 32 lane maxima (lane l sees logits l, l + 32, ...),
// is reached by K distinct logits, so every logit of the top K is >= tau: only
// the candidates >= tau (few for any spread-out row) are ranked, each by counting
// the candidates that beat it.  More than kTopkCap candidates (ties, -inf rows)
// take K rounds of a warp-wide selection instead.  Writes idx[0..K) in rank order
// and w[0..K) = exp(l_k - l_0) / sum_j exp(l_j - l_0).
constexpr int kTopkCap = kTopkCand;

__device__ __forceinline__ float logit_at(const float* row, int i) {
  const float v = row[i];
  return v != v ? -INFINITY : v;
}

// Any E (a multiple of 32): the logits stay in shared memory.
__device__ void warp_topk_any(const float* row, int E, int K, Cand* cand, int* idx, float* w) {
  const int lane = threadIdx.x & 31, nj = E >> 5;
  float m = -INFINITY;
  for (int j = 0; j < nj; ++j) m = fmaxf(m, logit_at(row, j * 32 + lane));
  float s = m;
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const float o = __shfl_xor_sync(kFull, s, j);
      const bool keep_max = ((lane & j) == 0) == ((lane & k) == 0 || k == 32);
      s = keep_max ? fmaxf(s, o) : fminf(s, o);
    }
  }
  const float tau = __shfl_sync(kFull, s, K - 1);
  int cnt = 0;
  for (int j = 0; j < nj; ++j) cnt += logit_at(row, j * 32 + lane) >= tau;
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += t;
  }
  const int total = __shfl_sync(kFull, incl, 31);
  if (total <= kTopkCap) {
    int at = incl - cnt;
    for (int j = 0; j < nj; ++j) {
      const float v = logit_at(row, j * 32 + lane);
      if (v >= tau) cand[at++] = Cand{v, j * 32 + lane};
    }
    __syncwarp();
    for (int i = lane; i < total; i += 32) {
      const Cand c = cand[i];
      int r = 0;
      for (int q = 0; q < total; ++q) {
        const Cand o = cand[q];
        r += cand_first(o.v, o.i, c.v, c.i);
      }
      if (r < K) idx[r] = c.i;
    }
  } else {
    for (int r = 0; r < K; ++r) {
      // K rounds of a warp-wide selection among the logits not yet chosen
      float bv = -INFINITY;
      int bi = 0x7fffffff;
      for (int j = 0; j < nj; ++j) {
        const int i = j * 32 + lane;
        const float v = logit_at(row, i);
        bool taken = false;
        for (int q = 0; q < r; ++q) taken |= idx[q] == i;
        if (!taken && cand_first(v, i, bv, bi)) { bv = v; bi = i; }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(kFull, bv, o);
        const int oi = __shfl_xor_sync(kFull, bi, o);
        if (cand_first(ov, oi, bv, bi)) { bv = ov; bi = oi; }
      }
      if (lane == 0) idx[r] = bi;
      __syncwarp();
    }
  }
  __syncwarp();
  const float vk = lane < K ? logit_at(row, idx[lane]) : 0.f;
  const float top0 = __shfl_sync(kFull, vk, 0);
  const float ev = lane < K ? expf(vk - top0) : 0.f;
  float den = ev;
  for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(kFull, den, o);
  if (lane < K) w[lane] = ev / den;
}

// NJ = E / 32 logits per lane, held in registers (one load each, issued together).
template <int NJ>
__device__ void warp_topk_reg(const float* row, int K, Cand* cand, int* idx, float* w) {
  const int lane = threadIdx.x & 31;
  float v[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) v[j] = logit_at(row, j * 32 + lane);
  float m = v[0];
#pragma unroll
  for (int j = 1; j < NJ; ++j) m = fmaxf(m, v[j]);
  // the 32 lane maxima sorted descending across the warp (bitonic network)
  float s = m;
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const float o = __shfl_xor_sync(kFull, s, j);
      const bool keep_max = ((lane & j) == 0) == ((lane & k) == 0 || k == 32);
      s = keep_max ? fmaxf(s, o) : fminf(s, o);
    }
  }
  const float tau = __shfl_sync(kFull, s, K - 1);
  int cnt = 0;
#pragma unroll
  for (int j = 0; j < NJ; ++j) cnt += v[j] >= tau;
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += t;
  }
  const int total = __shfl_sync(kFull, incl, 31);
  if (total <= kTopkCap) {
    int at = incl - cnt;
#pragma unroll
    for (int j = 0; j < NJ; ++j)
      if (v[j] >= tau) cand[at++] = Cand{v[j], j * 32 + lane};
    __syncwarp();
    for (int i = lane; i < total; i += 32) {
      const Cand c = cand[i];
      int r = 0;
      for (int q = 0; q < total; ++q) {
        const Cand o = cand[q];
        r += cand_first(o.v, o.i, c.v, c.i);
      }
      if (r < K) idx[r] = c.i;
    }
  } else {
    uint32_t taken = 0;   // bit j: logit j * 32 + lane already chosen
    for (int r = 0; r < K; ++r) {
      float bv = -INFINITY;
      int bi = 0x7fffffff;
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        const int i = j * 32 + lane;
        if (!((taken >> j) & 1u) && cand_first(v[j], i, bv, bi)) { bv = v[j]; bi = i; }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(kFull, bv, o);
        const int oi = __shfl_xor_sync(kFull, bi, o);
        if (cand_first(ov, oi, bv, bi)) { bv = ov; bi = oi; }
      }
      if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
      if (lane == 0) idx[r] = bi;
    }
  }
  __syncwarp();
  const float vk = lane < K ? logit_at(row, idx[lane]) : 0.f;
  const float top0 = __shfl_sync(kFull, vk, 0);
  const float ev = lane < K ? expf(vk - top0) : 0.f;
  float den = ev;
  for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(kFull, den, o);
  if (lane < K) w[lane] = ev / den;
}

__device__ void warp_topk(const float* row, int E, int K, Cand* cand, int* idx, float* w) {
  switch (E >> 5) {
    case 1: warp_topk_reg<1>(row, K, cand, idx, w); break;
    case 2: warp_topk_reg<2>(row, K, cand, idx, w); break;
    case 4: warp_topk_reg<4>(row, K, cand, idx, w); break;
    case 8: warp_topk_reg<8>(row, K, cand, idx, w); break;
    case 16: warp_topk_reg<16>(row, K, cand, idx, w); break;
    case 32: warp_topk_reg<32>(row, K, cand, idx, w); break;
    default: warp_topk_any(row, E, K, cand, idx, w);
  }
}

// power-of-two scale that brings max |v| into [0.5, 1)
__device__ __forceinline__ void pow2_scale(float maxabs, float* sc, float* inv) {
  int e = 0;
  if (maxabs > 0.f && isfinite(maxabs)) frexpf(maxabs, &e);
  *sc = ldexpf(1.0f, -e);
  *inv = ldexpf(1.0f, e);
}

// x_out = bf16(v / sqrt(mean(v^2) + eps)), v = x + y, for T rows of H (all threads of
// the CTA), in the library's one summation order (group_sumsq per 16-byte group, the
// group sums of a row added by lane l = g mod 32 in order, then the xor tree), which
// edge0_residual_rmsnorm's kernel shares.  Every thread's first loads are issued
// before `hook()` runs (once per thread); the group sums go to `part` [T][H/8].
template <class Hook>
__device__ void residual_norm(DecTables* tb, const __nv_bfloat16* xp, const __nv_bfloat16* yp,
                              __nv_bfloat16* xs, float* part, int T, int H, float eps, Hook hook) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ng = T * H / 8, gpr = H / 8;
  const uint4* xv = reinterpret_cast<const uint4*>(xp);
  const uint4* yv = reinterpret_cast<const uint4*>(yp);
  bool hooked = false;
  for (int g0 = tid; g0 < ng || !hooked; g0 += 4 * kDecThreads) {
    uint4 ga[4], gb[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int g = g0 + j * kDecThreads;
      ga[j] = g < ng ? xv[g] : make_uint4(0u, 0u, 0u, 0u);
      gb[j] = g < ng ? yv[g] : make_uint4(0u, 0u, 0u, 0u);
    }
    if (!hooked) { hook(); hooked = true; }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int g = g0 + j * kDecThreads;
      if (g < ng) part[g] = group_sumsq(ga[j], gb[j]);
    }
  }
  __syncthreads();
  if (warp < T) {
    float sum = 0.f;
    for (int g = lane; g < gpr; g += 32) sum += part[size_t(warp) * gpr + g];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(kFull, sum, o);
    if (lane == 0) tb->inv_rms[warp] = 1.0f / sqrtf(sum / float(H) + eps);
  }
  __syncthreads();
  // 16-byte groups, four per thread in flight together
  for (int g0 = tid; g0 < ng; g0 += 4 * kDecThreads) {
    uint4 ga[4], gb[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int g = g0 + j * kDecThreads;
      ga[j] = g < ng ? xv[g] : make_uint4(0u, 0u, 0u, 0u);
      gb[j] = g < ng ? yv[g] : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int g = g0 + j * kDecThreads;
      if (g < ng) {
        const float inv = tb->inv_rms[g / gpr];
        const uint32_t aa[4] = {ga[j].x, ga[j].y, ga[j].z, ga[j].w}, bb[4] = {gb[j].x, gb[j].y, gb[j].z, gb[j].w};
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float v0 = __uint_as_float(aa[i] << 16) + __uint_as_float(bb[i] << 16);
          const float v1 = __uint_as_float(aa[i] & 0xFFFF0000u) + __uint_as_float(bb[i] & 0xFFFF0000u);
          const __nv_bfloat162 r = __floats2bfloat162_rn(v0 * inv, v1 * inv);
          o[i] = *reinterpret_cast<const uint32_t*>(&r);
        }
        reinterpret_cast<uint4*>(xs)[g] = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
  }
  __syncthreads();
}

// SwiGLU of one gate/up row pair by one warp: lanes 0-15 reduce the gate row,
// lanes 16-31 the up row, for n activation rows; h_fn(i, h) per activation i.
template <int TB, class HFn>
__device__ __forceinline__ void gateup_row(const uint8_t* gc, const uint8_t* gs, const uint8_t* uc,
                                           const uint8_t* us, int L, const __half* const* arow, int n,
                                           float gg, float gu, const float* ainv, HFn h_fn) {
  const int lane = threadIdx.x & 31, hl = lane & 15;
  const bool up = lane >= 16;
  float acc[TB];
#pragma unroll
  for (int i = 0; i < TB; ++i) acc[i] = 0.f;
  fp4_dot<TB>(up ? uc : gc, up ? us : gs, L / 16, arow, n, hl, 16, acc);
  group_reduce<TB>(acc, 16);
#pragma unroll
  for (int i = 0; i < TB; ++i) {
    const float other = __shfl_xor_sync(kFull, acc[i], 16);
    if (i < n && lane == i) {
      // lane i < 16 holds the gate sum in acc[i] and the up sum in `other`
      const float gv = gg * acc[i] * ainv[i];
      const float uv = gu * other * ainv[i];
      h_fn(i, silu_f(gv) * uv);
    }
  }
}

// ------------------------------------------------------------------ NVFP4 x f16 on mma.sync
// An expert dot product over K runs as m16n8k16 MMAs: A = 16 weight rows (NVFP4
// decoded in registers, times the E4M3 block scale, exact in f16), B = up to 8
// activation rows (f16), fp32 accumulators.  A dot product does not depend on the
// order of its K terms, so K is taken in 32-column chunks with both operands read in
// one fixed permutation: thread c of a quad holds the fragment columns 2c, 2c + 1,
// 2c + 8, 2c + 9 of two MMAs, which are mapped to the chunk's physical columns
// 8c .. 8c + 7 (first MMA 8c .. 8c + 3, second 8c + 4 .. 8c + 7).  The thread then
// reads one 32-bit code word (8 codes, one 16-block scale) per A row and one 16-byte
// activation vector per B row, instead of scattered bytes.
struct MmaRows {
  const uint8_t* code[2];   // A rows g and g + 8: code bytes of the row (K / 2)
  const uint8_t* scale[2];  // their E4M3 scales (K / 16)
};

// acc[t] += A (rows g, g + 8) x B tile t over 32-column chunks [s0, s1).
template <int NT>
__device__ __forceinline__ void fp4_mma_chunks(const MmaRows& ar, const __half* const* brow, const bool* bval,
                                               int s0, int s1, float (*acc)[4]) {
  const int c = threadIdx.x & 3;
  const uint8_t* ca = ar.code[0] + 4 * c;
  const uint8_t* cb = ar.code[1] + 4 * c;
  const uint8_t* sa = ar.scale[0] + (c >> 1);
  const uint8_t* sb = ar.scale[1] + (c >> 1);
#pragma unroll 2
  for (int s = s0; s < s1; ++s) {
    const uint32_t wa = *reinterpret_cast<const uint32_t*>(ca + 16 * s);
    const uint32_t wb = *reinterpret_cast<const uint32_t*>(cb + 16 * s);
    const uint32_t ka = scale_f16x2(sa[2 * s]), kb = scale_f16x2(sb[2 * s]);
    uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
    e2m1x8_to_h2x4(wa, a0, a1, a2, a3);
    e2m1x8_to_h2x4(wb, b0, b1, b2, b3);
    a0 = hmul2_u32(a0, ka); a1 = hmul2_u32(a1, ka); a2 = hmul2_u32(a2, ka); a3 = hmul2_u32(a3, ka);
    b0 = hmul2_u32(b0, kb); b1 = hmul2_u32(b1, kb); b2 = hmul2_u32(b2, kb); b3 = hmul2_u32(b3, kb);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      uint4 z = make_uint4(0u, 0u, 0u, 0u);
      if (bval[t]) z = *reinterpret_cast<const uint4*>(brow[t] + 32 * s + 8 * c);
      mma16816(acc[t], a0, b0, a1, b1, z.x, z.y);
      mma16816(acc[t], a2, b2, a3, b3, z.z, z.w);
    }
  }
}

// The same with bf16 operands (the down projection: B = SwiGLU activations in bf16).
// NVFP4 -> f16 by cvt, then to the bf16 exponent range and times the block scale
// (exact: E2M1 x E4M3 has at most 5 significant bits).
template <int NT>
__device__ __forceinline__ void fp4_mma_chunks_bf16(const MmaRows& ar, const __nv_bfloat16* const* brow,
                                                    const bool* bval, int s0, int s1, float (*acc)[4]) {
  const int c = threadIdx.x & 3;
  const uint8_t* ca = ar.code[0] + 4 * c;
  const uint8_t* cb = ar.code[1] + 4 * c;
  const uint8_t* sa = ar.scale[0] + (c >> 1);
  const uint8_t* sb = ar.scale[1] + (c >> 1);
#pragma unroll 2
  for (int s = s0; s < s1; ++s) {
    const uint32_t wa = *reinterpret_cast<const uint32_t*>(ca + 16 * s);
    const uint32_t wb = *reinterpret_cast<const uint32_t*>(cb + 16 * s);
    const uint32_t ka = scale_bf16x2(sa[2 * s]), kb = scale_bf16x2(sb[2 * s]);
    uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
    e2m1x8_to_h2x4(wa, a0, a1, a2, a3);
    e2m1x8_to_h2x4(wb, b0, b1, b2, b3);
    a0 = h2_to_bf2_scaled(a0, ka); a1 = h2_to_bf2_scaled(a1, ka);
    a2 = h2_to_bf2_scaled(a2, ka); a3 = h2_to_bf2_scaled(a3, ka);
    b0 = h2_to_bf2_scaled(b0, kb); b1 = h2_to_bf2_scaled(b1, kb);
    b2 = h2_to_bf2_scaled(b2, kb); b3 = h2_to_bf2_scaled(b3, kb);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      uint4 z = make_uint4(0u, 0u, 0u, 0u);
      if (bval[t]) z = *reinterpret_cast<const uint4*>(brow[t] + 32 * s + 8 * c);
      mma16816_bf16(acc[t], a0, b0, a1, b1, z.x, z.y);
      mma16816_bf16(acc[t], a2, b2, a3, b3, z.z, z.w);
    }
  }
}

// Split of a task's chunks over ks warps (at most 16 warp tasks in all, ks <= kmax):
// the partial accumulators of part p go to part_buf[(task * ks + p) * 32 + lane]
// and are summed in part order afterwards.
__device__ __forceinline__ int mma_ksplit(int ntask, int kmax) {
  int ks = ntask >= 9 ? 1 : ntask >= 5 ? 2 : ntask >= 3 ? 4 : 8;
  return ks < kmax ? ks : kmax;
}

}  // namespace

// ------------------------------------------------------------------ the kernel
template <int TB>
__global__ void __launch_bounds__(kDecThreads, 1) moe_decode_kernel(const __grid_constant__ DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t dsm[];
  DecTables* tb = reinterpret_cast<DecTables*>(dsm);
  Ctx cx{tb, a.err, 0u};
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, bid = blockIdx.x;
  const int T = a.T, H = a.H, L = a.L, E = a.E, K = a.K, F = a.F;
  const int TK = T * K, nslot = TK + T;
  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(dsm + a.off_xs);
  float* act = reinterpret_cast<float*>(dsm + a.off_act);
  __half* zh = reinterpret_cast<__half*>(dsm + a.off_zh);
  uint8_t* shr = dsm + a.off_sh;
  uint8_t* dyn = dsm + a.off_dyn;
  // record layout: GU block of F rows (gate codes | up codes | gate scales | up
  // scales, 9L/8 bytes), D block of L/2 row pairs (codes 2p | codes 2p+1 |
  // scales 2p | scales 2p+1, 9F/8 bytes), then the three fp32 scales
  const int gu_row = 9 * L / 8, d_pair = 9 * F / 8;
  const size_t rec_dblk = size_t(F) * gu_row;
  const size_t rec_body = rec_dblk + size_t(L / 2) * d_pair;
  const int cofs_up = L / 2, sofs_g = L, sofs_u = L + L / 16;   // offsets inside a GU row
  // this CTA's row ranges (latent rows in whole pairs)
  const int r0 = 2 * int(long(bid) * (L / 2) / G), r1 = 2 * int(long(bid + 1) * (L / 2) / G);
  const int e0 = int(long(bid) * E / G), e1 = int(long(bid + 1) * E / G);      // router rows
  const int f0 = int(long(bid) * F / G), f1 = int(long(bid + 1) * F / G);      // shared rows
  const int j0 = int(long(bid) * H / G), j1 = int(long(bid + 1) * H / G);      // hidden rows
  const int nr = r1 - r0, nsr = f1 - f0;

  // launched as a programmatic dependent of the preceding kernel on the stream: its
  // results (this launch's input, the workspace) are complete from here on
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // a launch after one whose wait ran out finds the grid barrier mid-round (reset
  // by edge0_moe_get_error): it does no work and leaves the error word set
  if (ld_relaxed_u32(&a.bar->abort)) {
    if (tid == 0) atomicOr(a.err, kErrTimeout);
    return;
  }
  if (tid == 0) {
    for (int b = 0; b < kNumMbar; ++b) mbar_init(&tb->mbar[b], b == kMbScale ? kScaleWarps : 1);
    fence_mbar_init();
    tb->stuck = 0;
  }
  __syncthreads();

  // profiling stamps (no-ops unless the launch carries a stamp buffer)
  auto stamp0 = [&](int li, int slot) {
    if (a.stamps && bid == 0 && tid == 0) a.stamps[li * kStampSlots + slot] = globaltimer_ns();
  };
  auto stamp_end = [&](int li, int slot) {   // slot: the max slot; slot + 1 the min slot
    if (a.stamps) {                          // uniform: the whole CTA is done with the phase
      __syncthreads();
      if (tid == 0) {
        const unsigned long long t = globaltimer_ns();
        atomicMax(&a.stamps[li * kStampSlots + slot], t);
        atomicMax(&a.stamps[li * kStampSlots + slot + 1], ~t);
      }
    }
  };
  LayerW lw = a.l0;
  for (int li = 0; li < a.n_layers; ++li) {
    const bool last = (li == a.n_layers - 1);
    stamp0(li, kStP0Start);
    __nv_bfloat16* xcur = a.xbuf + size_t(li & 1) * T * H;
    // ================================================================ P0: z = D x, l = (R D) x + b
    {
      // the shared expert's fp32 scales: loaded now, stored at the end of the phase
      float2 sh_gu = make_float2(0.f, 0.f);
      float sh_d = 0.f;
      if (tid == 32) {
        const float* gs = reinterpret_cast<const float*>(lw.shared + rec_body);
        sh_gu = *reinterpret_cast<const float2*>(gs);
        sh_d = gs[2];
      }
      // router rows first: they are the longer ones (fp32) and feed the routing
      RowSet rs[2] = {{reinterpret_cast<const uint8_t*>(lw.RD), e0, e1, H * 4, 1},
                      {reinterpret_cast<const uint8_t*>(lw.D), r0, r1, H * 2, 0}};
      // this CTA's router bias entries, in flight while x is read
      const int ne = e1 - e0;
      const int bj = tid - (kDecThreads - 32);          // lanes of the last warp
      const float bv = (bj >= 0 && bj < ne && lw.bias) ? lw.bias[e0 + bj] : 0.f;
      // the weight rows and the shared-expert rows (P1) go out right after x's loads,
      // so that those few loads are not queued behind the bulk copies
      auto stage = [&]() {
        if (warp == 0 && nr + (e1 - e0) > 0)
          stage_rows(cx, rs, 2, 0, min(dense_cap(rs, 2, a.dyn_bytes), (e1 - e0) + nr), dyn);
        if (tid == 32 && nsr > 0) {
          mbar_arrive_expect_tx(&tb->mbar[kMbShared], uint32_t(nsr) * gu_row);
          bulk_g2s(shr, lw.shared + size_t(f0) * gu_row, uint32_t(nsr) * gu_row, &tb->mbar[kMbShared]);
        }
      };
      if (li == 0) {
        for (int i = tid; i < T * H / 8; i += kDecThreads)
          cp_async16(reinterpret_cast<uint4*>(xs) + i, reinterpret_cast<const uint4*>(a.x) + i);
        cp_async_commit();
        stage();
        cp_async_wait_all();
        __syncthreads();
      } else {
        // x_l = bf16(RMSNorm(x_{l-1} + y_{l-1})), computed by every CTA
        residual_norm(tb, a.xbuf + size_t((li - 1) & 1) * T * H, a.ybuf + size_t((li - 1) & 1) * T * H,
                      xs, reinterpret_cast<float*>(xs + size_t(T) * H), T, H, a.eps, stage);
      }
      if (bid == 0) {
        for (int i = tid; i < T * H / 8; i += kDecThreads)
          reinterpret_cast<uint4*>(xcur)[i] = reinterpret_cast<const uint4*>(xs)[i];
        if (a.trace_x)
          for (int i = tid; i < T * H / 8; i += kDecThreads)
            reinterpret_cast<uint4*>(a.trace_x + size_t(li) * T * H)[i] = reinterpret_cast<const uint4*>(xs)[i];
      }
      if (bj >= 0 && bj < ne) tb->w[bj] = bv;       // read after the barriers below
      // per-token power-of-two scale of z for its f16 copy, from the bound
      // |z_r| <= max_r sum_h |D_rh| * max_h |x_h|, identical in every CTA
      for (int t = 0; t < T; ++t) {
        float m = 0.f;
        for (int k = tid; k < H; k += kDecThreads) m = fmaxf(m, fabsf(__bfloat162float(xs[size_t(t) * H + k])));
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
        if (lane == 0) tb->red[warp * kDecodeMaxT + t] = m;
      }
      __syncthreads();
      if (tid < T) {
        float m = 0.f;
        for (int wv = 0; wv < kDecWarps; ++wv) m = fmaxf(m, tb->red[wv * kDecodeMaxT + tid]);
        const float dn = (li == 0 && a.dnorm_dev) ? *a.dnorm_dev : lw.dnorm;
        pow2_scale(m * dn, &tb->zsc[tid], &tb->zinv[tid]);
      }
      __syncthreads();
      float* z = a.z;
      __half* zg = a.zh;
      float* logits = a.logits;
      const float* zsc = tb->zsc;
      const float* rbias = tb->w;
      dense_rows<TB, false>(cx, rs, 2, xs, H, T, dyn, a.dyn_bytes, true, [&](int m, int t, int row, float v) {
        if (m == 1) {
          z[size_t(t) * L + row] = v;
          zg[size_t(t) * L + row] = __float2half_rn(v * zsc[t]);
        } else {
          logits[size_t(t) * E + row] = v + (ne <= 32 ? rbias[row - e0] : (lw.bias ? lw.bias[row] : 0.f));
        }
      });
      if (tid == 32) tb->gsc[0] = make_float4(sh_gu.x, sh_gu.y, sh_d, 0.f);
    }
    stamp_end(li, kStP0EndMax);
    if (!grid_sync(a.bar, a.err)) return;
    stamp0(li, kStBar1);
    // ================================================================ P1: routing, gate/up -> h
    {
      if (tid == 0) tb->task_ctr = 0;
      // the experts' f16 input zh, and the logits rows [T][E] into act
      for (int i = tid; i < T * L / 8; i += kDecThreads)
        cp_async16(reinterpret_cast<uint4*>(zh) + i, reinterpret_cast<const uint4*>(a.zh) + i);
      cp_async_commit();
      float* lg = act;
      for (int i = tid; i < T * E / 4; i += kDecThreads)
        reinterpret_cast<float4*>(lg)[i] = reinterpret_cast<const float4*>(a.logits)[i];
      // U rows of this CTA into L2 for P3 (routing-independent), after the logits loads
      if (tid == 0 && j1 > j0) l2_prefetch_share(lw.U + size_t(j0) * L, size_t(j1 - j0) * L * 2, 0, 1);
      cp_async_wait_all();
      __syncthreads();
      stamp0(li, kStRouteLoaded);
      // top-k + weights: one warp per token
      Cand* cbuf = reinterpret_cast<Cand*>(lg + size_t(T) * E) + warp * kTopkCap;
      for (int t = warp; t < T; t += kDecWarps) warp_topk(lg + size_t(t) * E, E, K, cbuf, tb->idx + t * K, tb->w + t * K);
      __syncthreads();
      stamp0(li, kStTopk);
      // permutation: stable order by (expert, slot)
      for (int s = tid; s < TK; s += kDecThreads) {
        const int key = tb->idx[s];
        int r = 0;
        for (int u = 0; u < TK; ++u) {
          const int k2 = tb->idx[u];
          r += (k2 < key) || (k2 == key && u < s);
        }
        tb->posn[s] = r;
        tb->perm[r] = s;
      }
      __syncthreads();
      if (warp == 0) {
        int base = 0;
        for (int p0 = 0; p0 < TK; p0 += 32) {
          const int p = p0 + lane;
          const bool start = p < TK && (p == 0 || tb->idx[tb->perm[p]] != tb->idx[tb->perm[p - 1]]);
          const unsigned bal = __ballot_sync(kFull, start);
          if (start) {
            const int gi = base + __popc(bal & ((1u << lane) - 1u));
            tb->gexp[gi] = tb->idx[tb->perm[p]];
            tb->goff[gi] = p;
          }
          base += __popc(bal);
        }
        if (lane == 0) { tb->nu = base; tb->goff[base] = TK; }
      }
      __syncthreads();
      stamp0(li, kStRouted);
      const int nu = tb->nu;
      // the record of every distinct expert: its place in the layer's array, or with
      // residency tiering its device slot or, for an expert not resident, a staging
      // record that all CTAs first fill from host memory (one more grid barrier)
      if (!lw.rec_table) {
        for (int g = tid; g < nu; g += kDecThreads) tb->gptr[g] = lw.experts + size_t(tb->gexp[g]) * lw.stride;
        __syncthreads();
      } else {
        if (warp == 0) {
          int base = 0;
          for (int g0 = 0; g0 < nu; g0 += 32) {
            const int g = g0 + lane;
            const bool miss = g < nu && !lw.resident[tb->gexp[g]];
            const unsigned bal = __ballot_sync(kFull, miss);
            const int m = base + __popc(bal & ((1u << lane) - 1u));
            if (g < nu) tb->gmiss[g] = miss ? m : -1;
            if (miss) tb->mgrp[m] = g;
            base += __popc(bal);
          }
          if (lane == 0) tb->n_miss = base;
        }
        __syncthreads();
        const int n_miss = tb->n_miss;
        if (n_miss > 0) {
          // records [0, n_miss) of the staging area from host memory, 16 bytes per
          // thread-step over the whole grid (plain loads through the device mapping)
          const size_t per = lw.stride / 16, total = size_t(n_miss) * per;
          for (size_t i = size_t(bid) * kDecThreads + tid; i < total; i += size_t(G) * kDecThreads) {
            const int m = int(i / per);
            const uint4* src = reinterpret_cast<const uint4*>(lw.rec_table[tb->gexp[tb->mgrp[m]]]) + (i - size_t(m) * per);
            reinterpret_cast<uint4*>(lw.staging)[i] = *src;
          }
          asm volatile("fence.proxy.async.global;" ::: "memory");
          if (!grid_sync(a.bar, a.err)) return;
          asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        for (int g = tid; g < nu; g += kDecThreads)
          tb->gptr[g] = tb->gmiss[g] >= 0 ? lw.staging + size_t(tb->gmiss[g]) * lw.stride : lw.rec_table[tb->gexp[g]];
        if (bid == 0) {
          for (int g = tid; g < nu; g += kDecThreads) atomicAdd(&lw.use[tb->gexp[g]], unsigned(tb->goff[g + 1] - tb->goff[g]));
          if (tid == 0) {
            atomicAdd(&lw.tier_stats[0], 1ull);
            atomicAdd(&lw.tier_stats[1], (unsigned long long)n_miss);
            atomicAdd(&lw.tier_stats[2], (unsigned long long)n_miss * lw.stride);
          }
        }
        __syncthreads();
      }
      // routed gate/up rows: q in [q0, q1) of nu * F (group-major), in whole tasks of 8
      const long ntq = long(nu) * (F / 8);
      const int q0 = 8 * int(ntq * bid / G), q1 = 8 * int(ntq * (bid + 1) / G);
      const int per_row = gu_row;
      // stage P2's down rows now when the whole P1 slab and the down slab both fit
      const int ngr = nu + 1;                          // routed groups + the shared expert
      const int down_grp = (nr / 2) * d_pair;
      const int down_bytes = ngr * down_grp;
      const int gu_bytes = (q1 - q0) * per_row;
      const int hrows_bytes = nslot * F * 2;
      const int ob_bytes = (nslot * nr * 4 + 127) & ~127;
      const int gu_alloc = (gu_bytes + 1023) & ~1023;
      const bool stage_down = nr > 0 && (q1 - q0) <= 256 &&
                              gu_alloc + down_bytes + hrows_bytes + ob_bytes <= a.dyn_bytes;
      if (tid == 0) {
        tb->down_staged = stage_down ? 1 : 0;
        tb->down_off = gu_alloc;
      }
      // the routing tables for the caller (trace, and the last layer's copy read by
      // edge0_moe_debug_routing), written after the expert copies are issued and
      // spread over the CTAs: each writes a slice
      auto publish_routing = [&]() {
        const int s0 = int(long(TK) * bid / G), s1 = int(long(TK) * (bid + 1) / G);
        if (a.trace_idx)
          for (int s = s0 + tid; s < s1; s += kDecThreads) a.trace_idx[size_t(li) * TK + s] = tb->idx[s];
        if (!last) return;
        for (int s = s0 + tid; s < s1; s += kDecThreads) {
          a.idx[s] = tb->idx[s]; a.w[s] = tb->w[s]; a.perm[s] = tb->perm[s]; a.pos[s] = tb->posn[s];
        }
        const int ea = int(long(E + 1) * bid / G), eb = int(long(E + 1) * (bid + 1) / G);
        for (int e = ea + tid; e < eb; e += kDecThreads) {
          int off = TK, cnt = 0;
          for (int g = 0; g < nu; ++g) {
            if (tb->gexp[g] >= e) { off = tb->goff[g]; if (tb->gexp[g] == e) cnt = tb->goff[g + 1] - tb->goff[g]; break; }
          }
          a.offsets[e] = off;
          if (e < E) a.counts[e] = cnt;
        }
      };
      // fp32 scales of the selected records, one per lane of warps 8..15: the loads
      // stay in flight across the next barrier; stored and announced on kMbScale after it
      float3 rsc = make_float3(0.f, 0.f, 0.f);
      const int sj = tid - kScaleWarp0 * 32;            // routed group of this lane
      if (sj >= 0 && sj < nu) {
        const float* gs = reinterpret_cast<const float*>(tb->gptr[sj] + rec_body);
        const float2 gu = *reinterpret_cast<const float2*>(gs);
        rsc = make_float3(gu.x, gu.y, gs[2]);
      }
      auto publish_scales = [&]() {
        if (warp >= kScaleWarp0 && warp < kScaleWarp0 + kScaleWarps) {
          if (sj < nu) tb->gsc[sj + 1] = make_float4(rsc.x, rsc.y, rsc.z, 0.f);
          __syncwarp();
          if (lane == 0) mbar_arrive(&tb->mbar[kMbScale]);
        }
      };
      const float sgg = tb->gsc[0].x, sgu = tb->gsc[0].y;
      const int* goff = tb->goff;
      const int* perm = tb->perm;
      constexpr int NT = TB > 8 ? 2 : 1;                // 8-token MMA tiles
      const int nst = (nsr + 7) / 8;                    // shared-expert tasks (8 row pairs each)
      const int nch = L / 32;                           // 32-column chunks of a gate/up row
      float4* part_buf = reinterpret_cast<float4*>(act);  // [warp task][lane][NT] partial sums
      int qa = q0;
      bool first_round = true;
      while (qa < q1 || first_round) {
        int nrow = 0, TPB = 1, nb = 0;
        if (qa < q1) {
          // with the down rows staged behind it, every round stays inside gu_alloc
          const int cap = min(256, (stage_down ? gu_alloc : a.dyn_bytes) / per_row) & ~7;
          if (cap < 8) {   // not even one 8-row task fits (the host rejects such shapes): stop, do not spin
            if (tid == 0) atomicOr(a.err, kErrTimeout);
            break;
          }
          nrow = min(cap, q1 - qa);                     // whole tasks: q0, q1 are multiples of 8
          const int nt = nrow / 8;
          TPB = (nt + kMbRounds - 1) / kMbRounds;       // tasks per batch, one lane of warp 0 each
          nb = (nt + TPB - 1) / TPB;
          if (warp == 0 && lane < nb) {
            const int s0 = qa + lane * TPB * 8, s1 = min(s0 + TPB * 8, qa + nrow);
            const int b = lane;
            mbar_arrive_expect_tx(&tb->mbar[kMbRound + b], uint32_t(s1 - s0) * per_row);
            uint32_t off = uint32_t(s0 - qa) * per_row;
            for (int q = s0; q < s1;) {
              // rows of one expert are one byte range of its GU block
              const int g = q / F, fa = q % F;
              const int n = min(s1, (g + 1) * F) - q;
              const uint8_t* rec = tb->gptr[g];
              bulk_g2s(dyn + off, rec + size_t(fa) * gu_row, uint32_t(n) * gu_row, &tb->mbar[kMbRound + b]);
              off += uint32_t(n) * gu_row;
              q += n;
            }
          }
        }
        if (first_round && stage_down && warp == 1) {
          // down rows [r0, r1) of every used expert (shared first), for P2, issued right
          // behind the gate/up rows (staging means one round, so the regions are disjoint):
          // the batch leader arms the barrier, then one lane per expert issues its copy
          uint8_t* dd = dyn + gu_alloc;
          const int per_b = (ngr + kMbDownN - 1) / kMbDownN;
          for (int gbase = 0; gbase < ngr; gbase += 32) {
            const int gi = gbase + lane;
            if (gi < ngr && gi % per_b == 0) {
              const int n_in = min(per_b, ngr - gi);
              mbar_arrive_expect_tx(&tb->mbar[kMbDown + gi / per_b], uint32_t(n_in) * down_grp);
            }
            __syncwarp();
            if (gi < ngr) {
              // this CTA's row pairs of one expert's D block: one byte range
              const uint8_t* rec = (gi == 0) ? lw.shared : tb->gptr[gi - 1];
              bulk_g2s(dd + size_t(gi) * down_grp, rec + rec_dblk + size_t(r0 / 2) * d_pair,
                       uint32_t(down_grp), &tb->mbar[kMbDown + gi / per_b]);
            }
          }
        }
        __syncthreads();
        if (first_round) stamp0(li, kStP1Issued);
        if (first_round) publish_scales();
        if (first_round) publish_routing();
        // tasks of 8 row pairs: A rows 0-7 the gate rows, 8-15 the up rows of the same
        // f, so that each thread holds gate and up of (f, token) for the SwiGLU
        const int ntr = nrow / 8;
        const int ntask = ntr + (first_round ? nst : 0);
        const int ks = mma_ksplit(ntask, 8);
        const int g8 = lane >> 2, c4 = lane & 3;
        // task i: routed (i < ntr: rows qa + 8 i ..) or shared (task i - ntr)
        auto task_info = [&](int i, MmaRows& ar, const __half** brow, bool* bval, int& grp, int& fbase,
                             int& ns) {
          if (i < ntr) {
            const int q = qa + 8 * i;
            grp = q / F;
            fbase = q % F;
            ns = goff[grp + 1] - goff[grp];
            const uint8_t* row = dyn + size_t(8 * i + g8) * gu_row;
            ar.code[0] = row; ar.code[1] = row + cofs_up;
            ar.scale[0] = row + sofs_g; ar.scale[1] = row + sofs_u;
#pragma unroll
            for (int t = 0; t < NT; ++t) {
              const int n = 8 * t + g8;
              bval[t] = n < ns;
              brow[t] = zh + size_t(n < ns ? perm[goff[grp] + n] / K : 0) * L;
            }
          } else {
            const int si = i - ntr;
            grp = -1;
            fbase = f0 + 8 * si;
            ns = T;
            const int r = 8 * si + g8;
            const uint8_t* row = shr + size_t(r < nsr ? r : 0) * gu_row;
            ar.code[0] = row; ar.code[1] = row + cofs_up;
            ar.scale[0] = row + sofs_g; ar.scale[1] = row + sofs_u;
#pragma unroll
            for (int t = 0; t < NT; ++t) {
              const int n = 8 * t + g8;
              bval[t] = n < T;
              brow[t] = zh + size_t(n < T ? n : 0) * L;
            }
          }
        };
        // SwiGLU of a finished task: thread (g8, c4) holds gate / up of row f = fbase + g8
        // for the group's activation rows n = 8 t + 2 c4 + j
        auto finish = [&](int i, float (*acc)[4]) {
          MmaRows ar;
          const __half* brow[NT];
          bool bval[NT];
          int grp, fbase, ns;
          task_info(i, ar, brow, bval, grp, fbase, ns);
          const int f = fbase + g8;
          if (grp < 0 && 8 * (i - ntr) + g8 >= nsr) return;
          const float gg = grp < 0 ? sgg : tb->gsc[grp + 1].x, gu = grp < 0 ? sgu : tb->gsc[grp + 1].y;
#pragma unroll
          for (int t = 0; t < NT; ++t) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const int n = 8 * t + 2 * c4 + j;
              if (n < ns) {
                const int slot = grp < 0 ? TK + n : perm[goff[grp] + n];
                const float zi = tb->zinv[grp < 0 ? n : slot / K];
                a.h[size_t(slot) * F + f] = __float2bfloat16_rn(silu_f(gg * acc[t][j] * zi) * (gu * acc[t][2 + j] * zi));
              }
            }
          }
        };
        for (int wt = warp; wt < ntask * ks; wt += kDecWarps) {
          const int i = wt / ks, part = wt - i * ks;
          MmaRows ar;
          const __half* brow[NT];
          bool bval[NT];
          int grp, fbase, ns;
          task_info(i, ar, brow, bval, grp, fbase, ns);
          if (i < ntr) {
            wait_mb(cx, kMbRound + i / TPB);
            wait_mb(cx, kMbScale);
          } else {
            wait_mb(cx, kMbShared);
          }
          float acc[NT][4];
#pragma unroll
          for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
          fp4_mma_chunks<NT>(ar, brow, bval, nch * part / ks, nch * (part + 1) / ks, acc);
          if (ks == 1) {
            finish(i, acc);
          } else {
#pragma unroll
            for (int t = 0; t < NT; ++t)
              part_buf[(size_t(wt) * 32 + lane) * NT + t] = make_float4(acc[t][0], acc[t][1], acc[t][2], acc[t][3]);
          }
        }
        if (ks > 1) {
          __syncthreads();
          for (int i = warp; i < ntask; i += kDecWarps) {
            float acc[NT][4];
#pragma unroll
            for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
            for (int p = 0; p < ks; ++p) {
#pragma unroll
              for (int t = 0; t < NT; ++t) {
                const float4 v = part_buf[(size_t(i * ks + p) * 32 + lane) * NT + t];
                acc[t][0] += v.x; acc[t][1] += v.y; acc[t][2] += v.z; acc[t][3] += v.w;
              }
            }
            finish(i, acc);
          }
        }
        for (int b = 0; b < nb; ++b) wait_mb(cx, kMbRound + b);
        if (first_round && nsr > 0) wait_mb(cx, kMbShared);
        __syncthreads();
        release_mb(cx, (1u << nb) - 1u);
        if (first_round && nsr > 0) release_mb(cx, 1u << kMbShared);
        qa += nrow;
        first_round = false;
      }
      if (tid == 0 && li + 1 < a.n_layers) {
        // next layer's D and R D into L2 while this layer finishes
        const LayerW nx = a.layers[li + 1];
        l2_prefetch_share(nx.D, size_t(L) * H * 2, bid, G);
        l2_prefetch_share(nx.RD, size_t(E) * H * 4, bid, G);
      }
    }
    stamp_end(li, kStP1EndMax);
    if (!grid_sync(a.bar, a.err)) return;
    stamp0(li, kStBar2);
    // ================================================================ P2: down + combine -> c
    LayerW nxt = lw;
    if (li + 1 < a.n_layers) nxt = a.layers[li + 1];
    {
      const int nu = tb->nu;
      const bool down_staged = tb->down_staged != 0;
      const int ngr = nu + 1;
      const int down_grp = (nr / 2) * d_pair;
      const int per_b = (ngr + kMbDownN - 1) / kMbDownN;
      const int n_down_b = (ngr + per_b - 1) / per_b;
      // stage P3's U rows (L2-resident by now) where P1's gate/up slab was
      const int nur = j1 - j0;
      const int u_bytes = nur * L * 2;
      const bool stage_u = down_staged && u_bytes <= tb->down_off;
      if (tid == 0) tb->u_staged = stage_u ? 1 : 0;
      // the U copies go out first: P3 waits on them, and issued later they arrive late
      bool u_issued = false;
      auto issue_u = [&]() {
        if (tid == 0 && stage_u && nur > 0) {
          const int nc = (u_bytes + 16383) / 16384;
          mbar_arrive_expect_tx(&tb->mbar[kMbU], uint32_t(u_bytes));
          for (int c = 0; c < nc; ++c) {
            const int ra = nur * c / nc, rb = nur * (c + 1) / nc;
            if (rb > ra)
              bulk_g2s(dyn + size_t(ra) * L * 2, lw.U + size_t(j0 + ra) * L, uint32_t(rb - ra) * L * 2,
                       &tb->mbar[kMbU]);
          }
        }
        u_issued = true;
      };
      issue_u();
      // region for h rows and per-slot outputs: after the staged down rows, or the
      // whole dynamic region when the down rows go in rounds
      uint8_t* region;
      int region_bytes;
      if (down_staged) {
        region = dyn + tb->down_off + ngr * down_grp;
        region_bytes = a.dyn_bytes - (tb->down_off + ngr * down_grp);
      } else {
        region = dyn;
        region_bytes = a.dyn_bytes;
      }
      float* ob = reinterpret_cast<float*>(region);
      const int ob_bytes = (nslot * nr * 4 + 127) & ~127;
      constexpr int NTD = TB > 8 ? 2 : 1;             // 8-token MMA tiles
      const int hrow = F * 2;
      wait_mb(cx, kMbScale);
      // Slots in one order q: q < T the shared expert's slot of token q (slot TK + q),
      // q >= T grouped position q - T (slot perm[q - T]).  Group j covers
      // [qlo(j), qhi(j)): j = 0 the shared expert, j >= 1 routed expert gexp[j - 1].
      // A round takes slots [qa, qb); its first and last group may be partial, so a
      // group whose h rows exceed the region is split over rounds.
      auto qlo = [&](int j) { return j == 0 ? 0 : T + tb->goff[j - 1]; };
      auto qhi = [&](int j) { return j == 0 ? T : T + tb->goff[j]; };
      int qa = 0, ja = 0;
      while (nr > 0 && qa < nslot) {
        while (qhi(ja) <= qa) ++ja;                 // the group holding slot qa
        int qb = qa, ng = 0;
        {
          const int wb = down_staged ? 0 : down_grp;
          int bytes = ob_bytes;
          for (int j = ja; j < ngr && ng < 512 && ng < (down_staged ? 512 : kMbRounds * 64); ++j) {
            const int want = qhi(j) - qb;
            const int room = (region_bytes - bytes - wb) / hrow;
            if (room <= 0) break;
            const int take = min(want, room);
            bytes += wb + take * hrow;
            qb += take;
            ++ng;
            if (take < want) break;
          }
        }
        if (ng == 0) {  // the region holds less than one h row and one down block: stop, do not spin
          if (tid == 0) atomicOr(a.err, kErrTimeout);
          break;
        }
        const int nq = qb - qa;
        const int nb = down_staged ? 0 : min(kMbRounds, ng);
        uint8_t* wbase = down_staged ? dyn + tb->down_off : region + ob_bytes + nq * hrow;
        if (tid == 0 && !down_staged) {
          for (int b = 0; b < nb; ++b) {
            const int ga = ng * b / nb, gb = ng * (b + 1) / nb;
            mbar_arrive_expect_tx(&tb->mbar[kMbRound + b], uint32_t(gb - ga) * down_grp);
            for (int jj = ga; jj < gb; ++jj) {
              const int j = ja + jj;
              const uint8_t* rec = (j == 0) ? lw.shared : tb->gptr[j - 1];
              bulk_g2s(wbase + size_t(jj) * down_grp, rec + rec_dblk + size_t(r0 / 2) * d_pair,
                       uint32_t(down_grp), &tb->mbar[kMbRound + b]);
              tb->task_aux[jj] = b;
            }
          }
        }
        // h rows of the round's slots (bf16, row i = slot q = qa + i), copied as they are
        __nv_bfloat16* hs = reinterpret_cast<__nv_bfloat16*>(region + ob_bytes);
        {
          const int cpr = F / 8;                   // 16-byte pieces per row
          for (int i = tid; i < nq * cpr; i += kDecThreads) {
            const int r = i / cpr, k = i - r * cpr;
            const int q = qa + r;
            const int slot = (q < T) ? TK + q : tb->perm[q - T];
            cp_async16(reinterpret_cast<uint4*>(hs + size_t(r) * F) + k,
                       reinterpret_cast<const uint4*>(a.h + size_t(slot) * F) + k);
          }
          cp_async_commit();
          cp_async_wait_all();
        }
        __syncthreads();
        if (qa == 0) stamp0(li, kStP2Staged);
        // tasks (group, 16-row tile of this CTA's latent rows): MMAs over the F columns,
        // A = the down rows (rho = tile row), B = the group's h rows of this round
        const int g8 = lane >> 2, c4 = lane & 3;
        const int rt = (nr + 15) / 16;
        const int ntask2 = ng * rt;
        const int ks2 = mma_ksplit(ntask2, 4);
        const int nchd = F / 32;
        float4* part_buf = reinterpret_cast<float4*>(act);
        auto dtask = [&](int i, MmaRows& ar, const __nv_bfloat16** brow, bool* bval, int& j, int& qs, int& ns,
                         int& rbase) {
          const int jj = i / rt;
          rbase = 16 * (i - jj * rt);
          j = ja + jj;
          qs = max(qa, qlo(j));
          ns = min(qb, qhi(j)) - qs;
          const uint8_t* gbase = wbase + size_t(down_staged ? j : jj) * down_grp;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            int rho = rbase + g8 + 8 * h;
            if (rho >= nr) rho = 0;
            const uint8_t* pr = gbase + size_t(rho / 2) * d_pair;
            ar.code[h] = pr + (rho & 1) * (F / 2);
            ar.scale[h] = pr + F + (rho & 1) * (F / 16);
          }
#pragma unroll
          for (int t = 0; t < NTD; ++t) {
            const int n = 8 * t + g8;
            bval[t] = n < ns;
            brow[t] = hs + size_t(qs - qa + (n < ns ? n : 0)) * F;
          }
        };
        auto dfinish = [&](int i, float (*acc)[4]) {
          MmaRows ar;
          const __nv_bfloat16* brow[NTD];
          bool bval[NTD];
          int j, qs, ns, rbase;
          dtask(i, ar, brow, bval, j, qs, ns, rbase);
          const float gd = tb->gsc[j].z;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int rho = rbase + g8 + 8 * h;
            if (rho >= nr) continue;
#pragma unroll
            for (int t = 0; t < NTD; ++t) {
#pragma unroll
              for (int jx = 0; jx < 2; ++jx) {
                const int n = 8 * t + 2 * c4 + jx;
                if (n < ns) {
                  const int q = qs + n;
                  const int slot = (q < T) ? TK + q : tb->perm[q - T];
                  ob[size_t(slot) * nr + rho] = gd * acc[t][2 * h + jx];
                }
              }
            }
          }
        };
        for (int wt = warp; wt < ntask2 * ks2; wt += kDecWarps) {
          const int i = wt / ks2, part = wt - i * ks2;
          MmaRows ar;
          const __nv_bfloat16* brow[NTD];
          bool bval[NTD];
          int j, qs, ns, rbase;
          dtask(i, ar, brow, bval, j, qs, ns, rbase);
          if (down_staged) wait_mb(cx, kMbDown + j / per_b);
          else wait_mb(cx, kMbRound + tb->task_aux[i / rt]);
          float acc[NTD][4];
#pragma unroll
          for (int t = 0; t < NTD; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
          fp4_mma_chunks_bf16<NTD>(ar, brow, bval, nchd * part / ks2, nchd * (part + 1) / ks2, acc);
          if (ks2 == 1) {
            dfinish(i, acc);
          } else {
#pragma unroll
            for (int t = 0; t < NTD; ++t)
              part_buf[(size_t(wt) * 32 + lane) * NTD + t] = make_float4(acc[t][0], acc[t][1], acc[t][2], acc[t][3]);
          }
        }
        if (ks2 > 1) {
          __syncthreads();
          for (int i = warp; i < ntask2; i += kDecWarps) {
            float acc[NTD][4];
#pragma unroll
            for (int t = 0; t < NTD; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
            for (int pp = 0; pp < ks2; ++pp) {
#pragma unroll
              for (int t = 0; t < NTD; ++t) {
                const float4 v = part_buf[(size_t(i * ks2 + pp) * 32 + lane) * NTD + t];
                acc[t][0] += v.x; acc[t][1] += v.y; acc[t][2] += v.z; acc[t][3] += v.w;
              }
            }
            dfinish(i, acc);
          }
        }
        if (!down_staged) {
          for (int b = 0; b < nb; ++b) wait_mb(cx, kMbRound + b);
        }
        __syncthreads();
        if (!down_staged) release_mb(cx, (1u << nb) - 1u);
        qa = qb;
      }
      stamp0(li, kStP2Tasks);
      if (!u_issued) issue_u();
      if (down_staged) {
        for (int b = 0; b < n_down_b; ++b) wait_mb(cx, kMbDown + b);
        __syncthreads();
        release_mb(cx, ((1u << n_down_b) - 1u) << kMbDown);
      }
      // combine: c[t][r] = o_shared + sum_j w[t][j] o[t*K + j], j ascending
      for (int p = tid; p < T * nr; p += kDecThreads) {
        const int t = p / nr, r = p % nr;
        float cv = ob[size_t(TK + t) * nr + r];
        for (int j = 0; j < K; ++j) cv = fmaf(tb->w[t * K + j], ob[size_t(t * K + j) * nr + r], cv);
        a.c[size_t(t) * L + r0 + r] = cv;
      }
      release_mb(cx, 1u << kMbScale);
    }
    stamp_end(li, kStP2EndMax);
    if (!grid_sync(a.bar, a.err)) return;
    stamp0(li, kStBar3);
    // ================================================================ P3: y = U c
    // the next kernel on the stream may be scheduled from here (it waits for this
    // grid's completion before reading anything)
    if (last) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    {
      for (int i = tid; i < T * L / 4; i += kDecThreads)
        reinterpret_cast<float4*>(act)[i] = reinterpret_cast<const float4*>(a.c)[i];
      __syncthreads();
      __nv_bfloat16* yo = (last && !a.final_norm) ? a.y : a.ybuf + size_t(li & 1) * T * H;
      __nv_bfloat16* ty = a.trace_y ? a.trace_y + size_t(li) * T * H : nullptr;
      auto emit = [&](int t, int j, float v) {
        const __nv_bfloat16 b = __float2bfloat16_rn(v);
        yo[size_t(t) * H + j] = b;
        if (ty) ty[size_t(t) * H + j] = b;
      };
      const int nur = j1 - j0;
      if (tb->u_staged) {
        if (nur > 0) wait_mb(cx, kMbU);
        const int hw = tid >> 4, hl = tid & 15;
        for (int base = (hw & ~1); base < nur; base += kDecThreads / 16) {
          const int i = base + (hw & 1);
          const bool valid = i < nur;
          float acc[TB];
#pragma unroll
          for (int t = 0; t < TB; ++t) acc[t] = 0.f;
          if (valid) row_dot<TB, false, true>(dyn + size_t(i) * L * 2, L, act, T, hl, 16, acc);
          group_reduce<TB>(acc, 16);
          if (valid && hl == 0) {
#pragma unroll
            for (int t = 0; t < TB; ++t)
              if (t < T) emit(t, j0 + i, acc[t]);
          }
        }
        __syncthreads();
        if (nur > 0) release_mb(cx, 1u << kMbU);
      } else {
        RowSet rs[1] = {{reinterpret_cast<const uint8_t*>(lw.U), j0, j1, L * 2, 0}};
        dense_rows<TB, true>(cx, rs, 1, act, L, T, dyn, a.dyn_bytes, false,
                             [&](int, int t, int j, float v) { emit(t, j, v); });
      }
    }
    stamp_end(li, kStP3EndMax);
    if (!last || a.final_norm) {
      if (!grid_sync(a.bar, a.err)) return;
      stamp0(li, kStBar4);
    }
    if (last && a.final_norm) {
      // stack output: RMSNorm(x_last + y_last); every CTA normalises, each writes its slice
      residual_norm(tb, xcur, a.ybuf + size_t(li & 1) * T * H, xs, reinterpret_cast<float*>(xs + size_t(T) * H), T,
                    H, a.eps, [] {});
      const int n8 = T * H / 8;
      const int i0 = int(long(bid) * n8 / G), i1 = int(long(bid + 1) * n8 / G);
      for (int i = i0 + tid; i < i1; i += kDecThreads)
        reinterpret_cast<uint4*>(a.y)[i] = reinterpret_cast<const uint4*>(xs)[i];
    }
    lw = nxt;
  }
  // a wait that ran out may leave a copy in flight: wait for it once more (bounded)
  __syncthreads();
  if (tid == 0 && tb->stuck) {
    for (int b = 0; b < kNumMbar; ++b)
      if ((tb->stuck >> b) & 1) mbar_wait(&tb->mbar[b], (cx.mbp >> b) & 1u, a.err);
  }
}

// ------------------------------------------------------------------ host side
template <int TB>
static cudaError_t launch_tb(const DecodeArgs& a, int grid, int smem, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeCooperative;
  at[0].val.cooperative = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  // programmatic serialization lets the launch overlap the tail of the preceding
  // kernel; where the runtime refuses it with a cooperative launch, launch without
  static int pdl = 1;
  cfg.numAttrs = pdl ? 2 : 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, moe_decode_kernel<TB>, a);
  if (e != cudaSuccess && pdl) {
    cudaGetLastError();
    pdl = 0;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, moe_decode_kernel<TB>, a);
  }
  return e;
}

template <int TB>
static cudaError_t prepare_tb(int smem) {
  return cudaFuncSetAttribute(moe_decode_kernel<TB>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

template <int TB>
static cudaError_t occupancy_tb(int smem, int* blocks) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, moe_decode_kernel<TB>, kDecThreads, smem);
}

int decode_bucket(int T) { return T <= 1 ? 1 : T <= 2 ? 2 : T <= 4 ? 4 : T <= 8 ? 8 : 16; }

cudaError_t decode_prepare(int smem) {
  cudaError_t e;
  if ((e = prepare_tb<1>(smem)) != cudaSuccess) return e;
  if ((e = prepare_tb<2>(smem)) != cudaSuccess) return e;
  if ((e = prepare_tb<4>(smem)) != cudaSuccess) return e;
  if ((e = prepare_tb<8>(smem)) != cudaSuccess) return e;
  return prepare_tb<16>(smem);
}

cudaError_t decode_occupancy(int smem, int* blocks) {
  int b1 = 0, b16 = 0;
  cudaError_t e;
  if ((e = occupancy_tb<1>(smem, &b1)) != cudaSuccess) return e;
  if ((e = occupancy_tb<16>(smem, &b16)) != cudaSuccess) return e;
  *blocks = b1 < b16 ? b1 : b16;
  return cudaSuccess;
}

cudaError_t decode_launch(const DecodeArgs& a, int grid, int smem, cudaStream_t s) {
  switch (decode_bucket(a.T)) {
    case 1: return launch_tb<1>(a, grid, smem, s);
    case 2: return launch_tb<2>(a, grid, smem, s);
    case 4: return launch_tb<4>(a, grid, smem, s);
    case 8: return launch_tb<8>(a, grid, smem, s);
    default: return launch_tb<16>(a, grid, smem, s);
  }
}

}  // namespace edge0
