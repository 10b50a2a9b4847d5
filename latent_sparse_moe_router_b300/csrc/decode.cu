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
  if (!mbar_wait_sleep(&cx.tb->mbar[b], (cx.mbp >> b) & 1u, cx.err)) atomicOr(&cx.tb->stuck, 1 << b);
}
// Release the barriers in `mask` after their use (all threads, uniformly).
__device__ __forceinline__ void release_mb(Ctx& cx, uint32_t mask) { cx.mbp ^= mask; }

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
// The candidates >= tau are compacted by ballots (in j-major order; their order does not
// matter); up to 32 of them are ranked across the lanes by shuffles, lane l holding
// candidate l, and the weights computed in place (the largest logit, top0, is the first
// of the sorted lane maxima).
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
  const float top0 = __shfl_sync(kFull, s, 0);
  const unsigned below = (1u << lane) - 1u;
  int total = 0;
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const bool p = v[j] >= tau;
    const unsigned bal = __ballot_sync(kFull, p);
    const int at = total + __popc(bal & below);
    if (p && at < kTopkCap) cand[at] = Cand{v[j], j * 32 + lane};
    total += __popc(bal);
  }
  __syncwarp();
  if (total <= 32) {
    const Cand c = lane < total ? cand[lane] : Cand{-INFINITY, 0x7fffffff};
    int r = 0;
#pragma unroll 4
    for (int q = 0; q < total; ++q) {
      const float ov = __shfl_sync(kFull, c.v, q);
      const int oi = __shfl_sync(kFull, c.i, q);
      r += cand_first(ov, oi, c.v, c.i);
    }
    const bool top = lane < total && r < K;
    const float ev = top ? expf(c.v - top0) : 0.f;
    float den = ev;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(kFull, den, o);
    if (top) {
      idx[r] = c.i;
      w[r] = ev / den;
    }
    __syncwarp();
    return;
  }
  if (total <= kTopkCap) {
    for (int i = lane; i < total; i += 32) {
      const Cand c = cand[i];
      int r = 0;
#pragma unroll 8
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
  const float t0 = __shfl_sync(kFull, vk, 0);
  const float ev = lane < K ? expf(vk - t0) : 0.f;
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

// x_out = bf16(v / sqrt(mean(v^2) + eps)), v = x + y, for T rows of H into xs (row pitch
// xpitch elements), in the library's one summation order (group_sumsq per 16-byte group,
// the group sums of a row added by lane l = g mod 32 in order, then the xor tree), which
// edge0_residual_rmsnorm's kernel shares: warp t (T <= 16 warps) sums row t.  Every
// warp calls `hook()` once, the warps holding a row right after their first loads.
template <class Hook>
__device__ void residual_norm(DecTables* tb, const __nv_bfloat16* xp, const __nv_bfloat16* yp,
                              __nv_bfloat16* xs, int xpitch, int T, int H, float eps, Hook hook) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gpr = H / 8;
  if (warp < T) {
    const uint4* xv = reinterpret_cast<const uint4*>(xp + size_t(warp) * H);
    const uint4* yv = reinterpret_cast<const uint4*>(yp + size_t(warp) * H);
    float sum = 0.f;
    bool hooked = false;
    for (int g0 = lane; g0 < gpr || !hooked; g0 += 4 * 32) {
      uint4 ga[4], gb[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int g = g0 + 32 * j;
        ga[j] = g < gpr ? xv[g] : make_uint4(0u, 0u, 0u, 0u);
        gb[j] = g < gpr ? yv[g] : make_uint4(0u, 0u, 0u, 0u);
      }
      if (!hooked) { hook(); hooked = true; }
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (g0 + 32 * j < gpr) sum += group_sumsq(ga[j], gb[j]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(kFull, sum, o);
    if (lane == 0) tb->inv_rms[warp] = 1.0f / sqrtf(sum / float(H) + eps);
  } else {
    hook();
  }
  __syncthreads();
  // 16-byte groups, four per thread in flight together
  const int ng = T * gpr;
  const uint4* xv = reinterpret_cast<const uint4*>(xp);
  const uint4* yv = reinterpret_cast<const uint4*>(yp);
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
        const int t = g / gpr;
        const float inv = tb->inv_rms[t];
        const uint32_t aa[4] = {ga[j].x, ga[j].y, ga[j].z, ga[j].w}, bb[4] = {gb[j].x, gb[j].y, gb[j].z, gb[j].w};
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float v0 = __uint_as_float(aa[i] << 16) + __uint_as_float(bb[i] << 16);
          const float v1 = __uint_as_float(aa[i] & 0xFFFF0000u) + __uint_as_float(bb[i] & 0xFFFF0000u);
          const __nv_bfloat162 r = __floats2bfloat162_rn(v0 * inv, v1 * inv);
          o[i] = *reinterpret_cast<const uint32_t*>(&r);
        }
        *reinterpret_cast<uint4*>(xs + size_t(t) * xpitch + 8 * (g - t * gpr)) = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
  }
  __syncthreads();
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

// acc[t] += A (rows g, g + 8) x B tile t over 32-column chunks [s0, s1).  The operands
// of chunk s + 1 are loaded while chunk s is decoded, and the chunk's two MMAs feed two
// accumulator chains that meet at the end.
template <int NT>
__device__ __forceinline__ void fp4_mma_chunks(const MmaRows& ar, const __half* const* brow, const bool* bval,
                                               int s0, int s1, float (*acc)[4]) {
  if (s0 >= s1) return;
  const int c = threadIdx.x & 3;
  const uint8_t* ca = ar.code[0] + 4 * c;
  const uint8_t* cb = ar.code[1] + 4 * c;
  const uint8_t* sa = ar.scale[0] + (c >> 1);
  const uint8_t* sb = ar.scale[1] + (c >> 1);
  float acc2[NT][4];
#pragma unroll
  for (int t = 0; t < NT; ++t) acc2[t][0] = acc2[t][1] = acc2[t][2] = acc2[t][3] = 0.f;
  uint32_t wa = *reinterpret_cast<const uint32_t*>(ca + 16 * s0);
  uint32_t wb = *reinterpret_cast<const uint32_t*>(cb + 16 * s0);
  uint32_t xa = sa[2 * s0], xb = sb[2 * s0];
  uint4 z[NT];
#pragma unroll
  for (int t = 0; t < NT; ++t)
    z[t] = bval[t] ? *reinterpret_cast<const uint4*>(brow[t] + 32 * s0 + 8 * c) : make_uint4(0u, 0u, 0u, 0u);
  for (int s = s0; s < s1; ++s) {
    const uint32_t cwa = wa, cwb = wb, cxa = xa, cxb = xb;
    uint4 cz[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) cz[t] = z[t];
    if (s + 1 < s1) {
      wa = *reinterpret_cast<const uint32_t*>(ca + 16 * (s + 1));
      wb = *reinterpret_cast<const uint32_t*>(cb + 16 * (s + 1));
      xa = sa[2 * (s + 1)];
      xb = sb[2 * (s + 1)];
#pragma unroll
      for (int t = 0; t < NT; ++t)
        if (bval[t]) z[t] = *reinterpret_cast<const uint4*>(brow[t] + 32 * (s + 1) + 8 * c);
    }
    const uint32_t ka = scale_f16x2(cxa), kb = scale_f16x2(cxb);
    uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
    e2m1x8_to_h2x4(cwa, a0, a1, a2, a3);
    e2m1x8_to_h2x4(cwb, b0, b1, b2, b3);
    a0 = hmul2_u32(a0, ka); a1 = hmul2_u32(a1, ka); a2 = hmul2_u32(a2, ka); a3 = hmul2_u32(a3, ka);
    b0 = hmul2_u32(b0, kb); b1 = hmul2_u32(b1, kb); b2 = hmul2_u32(b2, kb); b3 = hmul2_u32(b3, kb);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      mma16816(acc[t], a0, b0, a1, b1, cz[t].x, cz[t].y);
      mma16816(acc2[t], a2, b2, a3, b3, cz[t].z, cz[t].w);
    }
  }
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    acc[t][0] += acc2[t][0]; acc[t][1] += acc2[t][1]; acc[t][2] += acc2[t][2]; acc[t][3] += acc2[t][3];
  }
}

// The same scheme for bf16 weight rows held in shared memory (D, U): ra and rb are A
// rows g and g + 8, one 16-byte load each per 32-column chunk.
template <int NT>
__device__ __forceinline__ void bf16_mma_chunks(const __nv_bfloat16* ra, const __nv_bfloat16* rb,
                                                const __nv_bfloat16* const* brow, const bool* bval, int s0, int s1,
                                                float (*acc)[4]) {
  const int c = threadIdx.x & 3;
#pragma unroll 2
  for (int s = s0; s < s1; ++s) {
    const uint4 u = *reinterpret_cast<const uint4*>(ra + 32 * s + 8 * c);
    const uint4 v = *reinterpret_cast<const uint4*>(rb + 32 * s + 8 * c);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      uint4 z = make_uint4(0u, 0u, 0u, 0u);
      if (bval[t]) z = *reinterpret_cast<const uint4*>(brow[t] + 32 * s + 8 * c);
      mma16816_bf16(acc[t], u.x, v.x, u.y, v.y, z.x, z.y);
      mma16816_bf16(acc[t], u.z, v.z, u.w, v.w, z.z, z.w);
    }
  }
}

// An fp32 value as the sum of two bf16 terms: hi = bf16(v), lo = bf16(v - hi); the
// remainder is below 2^-17 |v|.  Two values at once, packed as bf16x2 (first low).
__device__ __forceinline__ void split_bf16x2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  const __nv_bfloat162 l = __floats2bfloat162_rn(a - __low2float(h), b - __high2float(h));
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// fp32 weight rows (the folded router R D): A row g holds the high bf16 term of row r and
// A row g + 8 its low term, so that output row g plus output row g + 8 is the dot
// product with the fp32 row (each bf16 x bf16 product exact in the fp32 accumulator).
template <int NT>
__device__ __forceinline__ void f32_split_mma_chunks(const float* r, const __nv_bfloat16* const* brow,
                                                     const bool* bval, int s0, int s1, float (*acc)[4]) {
  const int c = threadIdx.x & 3;
#pragma unroll 2
  for (int s = s0; s < s1; ++s) {
    const float4 p = *reinterpret_cast<const float4*>(r + 32 * s + 8 * c);
    const float4 q = *reinterpret_cast<const float4*>(r + 32 * s + 8 * c + 4);
    uint32_t h0, l0, h1, l1, h2, l2, h3, l3;
    split_bf16x2(p.x, p.y, h0, l0);
    split_bf16x2(p.z, p.w, h1, l1);
    split_bf16x2(q.x, q.y, h2, l2);
    split_bf16x2(q.z, q.w, h3, l3);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      uint4 z = make_uint4(0u, 0u, 0u, 0u);
      if (bval[t]) z = *reinterpret_cast<const uint4*>(brow[t] + 32 * s + 8 * c);
      mma16816_bf16(acc[t], h0, l0, h1, l1, z.x, z.y);
      mma16816_bf16(acc[t], h2, l2, h3, l3, z.z, z.w);
    }
  }
}

// Partial sums of a CTA's warps (fragment layout: [warp][lane][NT] float4), reduced by
// warp w over the warps w * n .. w * n + n - 1 in that order.
template <int NT>
__device__ __forceinline__ void partial_store(float4* part, float (*acc)[4]) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int t = 0; t < NT; ++t)
    part[(size_t(warp) * 32 + lane) * NT + t] = make_float4(acc[t][0], acc[t][1], acc[t][2], acc[t][3]);
}

template <int NT>
__device__ __forceinline__ void partial_sum(const float4* part, int first, int n, float (*acc)[4]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
  for (int p = 0; p < n; ++p) {
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const float4 v = part[(size_t(first + p) * 32 + lane) * NT + t];
      acc[t][0] += v.x; acc[t][1] += v.y; acc[t][2] += v.z; acc[t][3] += v.w;
    }
  }
}

// A CTA that gives up (a grid barrier or a wait ran out) lets its own bulk copies land
// before it exits: 50 us of %globaltimer.
__device__ __forceinline__ void drain_copies() {
  if (threadIdx.x == 0) {
    const unsigned long long t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 50000ull) {
    }
  }
}

}  // namespace

// ------------------------------------------------------------------ the kernel
template <int NT>
__global__ void __launch_bounds__(kDecThreads, 1) moe_decode_kernel(const __grid_constant__ DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t dsm[];
  DecTables* tb = reinterpret_cast<DecTables*>(dsm);
  Ctx cx{tb, a.err, 0u};
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g8 = lane >> 2, c4 = lane & 3;
  const int G = gridDim.x, bid = blockIdx.x;
  const int T = a.T, H = a.H, L = a.L, E = a.E, K = a.K, F = a.F;
  const int TK = T * K, nslot = TK + T;
  uint8_t* shr = dsm + a.off_sh;                                 // shared-expert gate/up rows
  uint8_t* areg = dsm + a.off_a;                                 // phase-local arrays
  uint8_t* ring = dsm + a.off_ring;                              // staged weights
  const int xp = H + kPadElems, zp = L + kPadElems;              // row pitches (elements)
  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(areg);    // P0: x [T][xp]
  __half* zs = reinterpret_cast<__half*>(areg);                  // P1: zh [T][zp]
  float4* part1 = reinterpret_cast<float4*>(areg + ((size_t(T) * zp * 2 + 127) & ~size_t(127)));
  float* ob = reinterpret_cast<float*>(areg);                    // P2: down outputs [half][slot][nr]
  __nv_bfloat16* cs = reinterpret_cast<__nv_bfloat16*>(areg);    // P3: c [T][zp] in bf16
  float4* partw = reinterpret_cast<float4*>(ring);               // P0 / P3: per-warp partial sums
  // record layout: GU block of F rows (gate codes | up codes | gate scales | up
  // scales, 9L/8 bytes), D block of L/2 row pairs (codes 2p | codes 2p+1 |
  // scales 2p | scales 2p+1, 9F/8 bytes), then the three fp32 scales
  const int gu_row = 9 * L / 8, d_pair = 9 * F / 8, gu_pitch = pitch_gu_row(L);
  const size_t rec_dblk = size_t(F) * gu_row;
  const size_t rec_body = rec_dblk + size_t(L / 2) * d_pair;
  const int cofs_up = L / 2, sofs_g = L, sofs_u = L + L / 16;   // offsets inside a GU row
  // this CTA's row ranges (latent rows in whole pairs)
  // (32-bit: every product below is under 2^31 for the shapes the host accepts)
  const int r0 = 2 * (bid * (L / 2) / G), r1 = 2 * ((bid + 1) * (L / 2) / G);
  const int e0 = bid * E / G, e1 = (bid + 1) * E / G;                          // router rows
  const int f0 = bid * F / G, f1 = (bid + 1) * F / G;                          // shared rows
  const int j0 = bid * H / G, j1 = (bid + 1) * H / G;                          // hidden rows
  const int nr = r1 - r0, nsr = f1 - f0, ne = e1 - e0, nur = j1 - j0;
  // the ring: S slots of SB bytes; a unit is split into ks parts (P1: K ranges)
  const int S = a.ring_slots, SB = a.slot_bytes;
  const int ks = (kDecWarps + S - 1) / S;
  const int nst = (nsr + 7) / 8;                                 // shared-expert gate/up units
  const int down_grp = (nr / 2) * d_pair, hrow = F * 2;

  if (tid == 0) {
    // ring slots complete on two arrivals (a unit's copies may be issued in two parts)
    for (int b = 0; b < kNumMbar; ++b)
      mbar_init(&tb->mbar[b], b < kMbRing + kRingMax ? 2 : (b == kMbScale ? 32 : 1));
    fence_mbar_init();
    tb->stuck = 0;
  }
  __syncthreads();
  // P0's rows: router tiles of 8 fp32 rows (high / low bf16 terms in A rows g / g + 8),
  // D tiles of 16 bf16 rows; every row bulk-copied to its padded place in the ring area
  const int nrt = (ne + 7) / 8, ndt = (nr + 15) / 16, ntile = nrt + ndt;
  const int pf = pitch_f32_row(H), pb = pitch_bf16_row(H);
  uint8_t* rows_d = ring + size_t(ne) * pf;
  auto issue_d_rows = [&](const LayerW& w) {           // warp 0
    if (lane < ndt) mbar_arrive_expect_tx(&tb->mbar[kMbP0 + nrt + lane], uint32_t(min(16, nr - 16 * lane)) * H * 2);
    __syncwarp();
    for (int r = lane; r < nr; r += 32)
      bulk_g2s(rows_d + size_t(r) * pb, w.D + size_t(r0 + r) * H, uint32_t(H) * 2, &tb->mbar[kMbP0 + nrt + r / 16]);
  };
  auto issue_rd_rows = [&](const LayerW& w) {          // warp 0
    if (lane < nrt) mbar_arrive_expect_tx(&tb->mbar[kMbP0 + lane], uint32_t(min(8, ne - 8 * lane)) * H * 4);
    __syncwarp();
    for (int i = lane; i < ne; i += 32)
      bulk_g2s(ring + size_t(i) * pf, w.RD + size_t(e0 + i) * H, uint32_t(H) * 4, &tb->mbar[kMbP0 + i / 8]);
  };
  auto issue_shared_rows = [&](const LayerW& w) {      // warp 1
    if (nsr <= 0) return;
    if (lane == 0) mbar_arrive_expect_tx(&tb->mbar[kMbShared], uint32_t(nsr) * gu_row);
    __syncwarp();
    if (lane < nsr)
      bulk_g2s(shr + size_t(lane) * gu_pitch, w.shared + size_t(f0 + lane) * gu_row, uint32_t(gu_row),
               &tb->mbar[kMbShared]);
  };
  // the first layer's D rows and shared-expert rows are weights no kernel writes: their
  // copies go out before the wait on the preceding kernel (R D may come from it)
  if (warp == 0) issue_d_rows(a.l0);
  if (warp == 1) issue_shared_rows(a.l0);

  // launched as a programmatic dependent of the preceding kernel on the stream: its
  // results (this launch's input, the workspace) are complete from here on
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // a launch after one whose wait ran out finds the grid barrier mid-round (reset
  // by edge0_moe_get_error): it does no work and leaves the error word set
  if (ld_relaxed_u32(&a.bar->abort)) {
    if (tid == 0) atomicOr(a.err, kErrTimeout);
    drain_copies();
    return;
  }

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
  // Ring unit u lives in slot u % S.  Before waiting for its copy, a warp waits until
  // the slot has finished the u / S units before it (the warp refilling a slot bumps
  // its generation after issuing the copy), so the slot's mbarrier is then in the
  // phase of unit u.  Units u < nst (the shared expert's rows, staged in P0) occupy a
  // slot position but no copy.
  auto ring_wait = [&](int u) {
    const int s = u % S, need = u / S;
    if (lane == 0) {
      volatile int* gp = &tb->ring_gen[s];
      if (*gp < need) {
        const unsigned long long t0 = globaltimer_ns();
        while (*gp < need) {
          __nanosleep(64);                                   // leave the issue slots to the working warps
          if (globaltimer_ns() - t0 > kWaitLimitNs) {
            atomicOr(a.err, kErrTimeout);
            break;
          }
        }
      }
    }
    __syncwarp();
    const int csh = s < nst ? 1 : 0;                           // copy-less units on slot s (nst <= S)
    const uint32_t par = ((cx.mbp >> (kMbRing + s)) ^ uint32_t(need - csh)) & 1u;
    if (!mbar_wait_sleep(&tb->mbar[kMbRing + s], par, a.err)) atomicOr(&tb->stuck, 1 << (kMbRing + s));
  };
  // One part of unit u done: true for the warp that finished the unit's last part
  // (parts counted per slot and phase; `kp` parts per unit).
  auto part_done = [&](int u, int kp) -> bool {
    if (kp == 1) return true;
    __syncwarp();
    int old = 0;
    if (lane == 0) {
      __threadfence_block();
      old = atomicAdd(&tb->ring_cnt[u % S], 1);
    }
    old = __shfl_sync(kFull, old, 0);
    if ((old + 1) % kp != 0) return false;
    __threadfence_block();
    return true;
  };
  auto slot_ptr = [&](int u) { return ring + size_t(u % S) * SB; };
  auto slot_bar = [&](int u) { return &tb->mbar[kMbRing + u % S]; };

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
      // this CTA's router bias entries, in flight while x is read
      const int bj = tid - (kDecThreads - 32);          // lanes of the last warp
      const float bv = (bj >= 0 && bj < ne && lw.bias) ? lw.bias[e0 + bj] : 0.f;
      // the weight rows go out right after x's loads (layer 0: the router rows only)
      auto stage = [&]() {
        if (warp == 0) {
          issue_rd_rows(lw);
          if (li > 0) issue_d_rows(lw);
        }
        if (warp == 1 && li > 0) issue_shared_rows(lw);
      };
      const int h8 = H / 8;
      if (li == 0) {
        for (int i = tid; i < T * h8; i += kDecThreads) {
          const int t = i / h8;
          cp_async16(xs + size_t(t) * xp + 8 * (i - t * h8), reinterpret_cast<const uint4*>(a.x) + i);
        }
        cp_async_commit();
        stage();
        cp_async_wait_all();
        __syncthreads();
      } else {
        // x_l = bf16(RMSNorm(x_{l-1} + y_{l-1})), computed by every CTA
        residual_norm(tb, a.xbuf + size_t((li - 1) & 1) * T * H, a.ybuf + size_t((li - 1) & 1) * T * H, xs, xp, T,
                      H, a.eps, stage);
      }
      if (bid == 0) {
        for (int i = tid; i < T * h8; i += kDecThreads) {
          const int t = i / h8;
          const uint4 v = *reinterpret_cast<const uint4*>(xs + size_t(t) * xp + 8 * (i - t * h8));
          reinterpret_cast<uint4*>(xcur)[i] = v;
          if (a.trace_x) reinterpret_cast<uint4*>(a.trace_x + size_t(li) * T * H)[i] = v;
        }
      }
      if (bj >= 0 && bj < ne) tb->w[bj] = bv;       // read after the barriers below
      // per-token power-of-two scale of z for its f16 copy, from the bound
      // |z_r| <= max_r sum_h |D_rh| * max_h |x_h|, identical in every CTA
      for (int t = 0; t < T; ++t) {
        float m = 0.f;
        for (int k = tid; k < H; k += kDecThreads) m = fmaxf(m, fabsf(__bfloat162float(xs[size_t(t) * xp + k])));
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
      // the MMAs: the warps split each tile's K range evenly
      const int wpt = ntile > 0 ? kDecWarps / ntile : kDecWarps;
      const int tile = warp / wpt, part = warp - tile * wpt;
      float acc[NT][4];
#pragma unroll
      for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
      if (tile < ntile) {
        wait_mb(cx, kMbP0 + tile);
        const __nv_bfloat16* brow[NT];
        bool bval[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const int n = 8 * t + g8;
          bval[t] = n < T;
          brow[t] = xs + size_t(n < T ? n : 0) * xp;
        }
        const int nch = H / 32, s0 = nch * part / wpt, s1 = nch * (part + 1) / wpt;
        if (tile < nrt) {
          int rr = 8 * tile + g8;
          if (rr >= ne) rr = 8 * tile;
          f32_split_mma_chunks<NT>(reinterpret_cast<const float*>(ring + size_t(rr) * pf), brow, bval, s0, s1, acc);
        } else {
          const int rbase = 16 * (tile - nrt);
          int ra = rbase + g8, rb = rbase + g8 + 8;
          if (ra >= nr) ra = rbase;
          if (rb >= nr) rb = rbase;
          bf16_mma_chunks<NT>(reinterpret_cast<const __nv_bfloat16*>(rows_d + size_t(ra) * pb),
                              reinterpret_cast<const __nv_bfloat16*>(rows_d + size_t(rb) * pb), brow, bval, s0, s1,
                              acc);
        }
      }
      __syncthreads();                 // every tile's rows are read: the partial sums overwrite them
      partial_store<NT>(partw, acc);
      __syncthreads();
      if (warp < ntile) {
        partial_sum<NT>(partw, warp * wpt, wpt, acc);
        if (warp < nrt) {
          const int rr = 8 * warp + g8;
          if (rr < ne) {
            const int row = e0 + rr;
            const float bias = ne <= 32 ? tb->w[rr] : (lw.bias ? lw.bias[row] : 0.f);
#pragma unroll
            for (int t = 0; t < NT; ++t)
#pragma unroll
              for (int j = 0; j < 2; ++j) {
                const int n = 8 * t + 2 * c4 + j;
                if (n < T) a.logits[size_t(n) * E + row] = (acc[t][j] + acc[t][2 + j]) + bias;
              }
          }
        } else {
          const int rbase = 16 * (warp - nrt);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int rho = rbase + g8 + 8 * hh;
            if (rho >= nr) continue;
            const int row = r0 + rho;
#pragma unroll
            for (int t = 0; t < NT; ++t)
#pragma unroll
              for (int j = 0; j < 2; ++j) {
                const int n = 8 * t + 2 * c4 + j;
                if (n < T) {
                  const float v = acc[t][2 * hh + j];
                  a.z[size_t(n) * L + row] = v;
                  a.zh[size_t(n) * L + row] = __float2half_rn(v * tb->zsc[n]);
                }
              }
          }
        }
      }
      if (ntile > 0) release_mb(cx, ((1u << ntile) - 1u) << kMbP0);
      if (tid == 32) tb->gsc[0] = make_float4(sh_gu.x, sh_gu.y, sh_d, 0.f);
    }
    stamp_end(li, kStP0EndMax);
    if (!grid_sync(a.bar, a.err)) { drain_copies(); return; }
    stamp0(li, kStBar1);
    // ================================================================ P1: routing, gate/up -> h
    int nu = 0, n1 = 0;
    {
      // the experts' f16 input zh (padded rows), and the logits rows [T][E] into the ring area
      const int l8 = L / 8;
      for (int i = tid; i < T * l8; i += kDecThreads) {
        const int t = i / l8;
        cp_async16(zs + size_t(t) * zp + 8 * (i - t * l8), reinterpret_cast<const uint4*>(a.zh) + i);
      }
      cp_async_commit();
      float* lg = reinterpret_cast<float*>(ring);
      for (int i = tid; i < T * E / 4; i += kDecThreads)
        reinterpret_cast<float4*>(lg)[i] = reinterpret_cast<const float4*>(a.logits)[i];
      // U rows of this CTA into L2 for P3 (routing-independent), after the logits loads
      if (tid == 0 && nur > 0) l2_prefetch_share(lw.U + size_t(j0) * L, size_t(nur) * L * 2, 0, 1);
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
#pragma unroll 8
        for (int u = 0; u < TK; ++u) {
          const int k2 = tb->idx[u];
          r += (k2 < key) || (k2 == key && u < s);
        }
        tb->posn[s] = r;
        tb->perm[r] = s;
        tb->tokp[r] = short(s / K);
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
      nu = tb->nu;
      // the record of every distinct expert: its place in the layer's array, or with
      // residency tiering its device slot or, for an expert not resident, a staging
      // record that all CTAs first fill from host memory (one more grid barrier)
      if (!lw.rec_table) {
        for (int g = tid; g < nu; g += kDecThreads) tb->gptr[g] = lw.experts + size_t(tb->gexp[g]) * lw.stride;
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
          if (!grid_sync(a.bar, a.err)) { drain_copies(); return; }
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
      }
      if (tid < kRingMax) { tb->ring_cnt[tid] = 0; tb->ring_gen[tid] = 0; }
      if (tid == 0) { tb->pair_ctr[0] = 0; tb->pair_ctr[1] = 0; tb->p2_ready = 0; tb->n2 = 0; }
      __syncthreads();
    }
    // routed gate/up rows: q in [q0, q1) of nu * F (group-major), in units of 8 rows;
    // the stream: units [0, nst) the shared expert's rows, [nst, n1) the routed rows,
    // [n1, n1 + n2) the down units of P2
    const int ngr = nu + 1;                             // groups: the shared expert, then the routed experts
    const int ntq = nu * (F / 8);
    const int q0 = 8 * (ntq * bid / G), q1 = 8 * (ntq * (bid + 1) / G);
    n1 = nst + (q1 - q0) / 8;
    // P2 slots in one order q: q < T the shared expert's slot of token q, q >= T grouped
    // position q - T; group j covers [qlo(j), qhi(j)) (j = 0 the shared expert)
    auto qlo = [&](int j) { return j == 0 ? 0 : T + tb->goff[j - 1]; };
    auto qhi = [&](int j) { return j == 0 ? T : T + tb->goff[j]; };
    auto p2_rec = [&](int j) -> const uint8_t* { return j == 0 ? lw.shared : tb->gptr[j - 1]; };
    // unit u >= nst: 8 gate/up row pairs of one expert, as two copies of 4 rows, the
    // second 16 bytes further on (rows r and r + 4 then fall in different banks)
    auto issue_p1 = [&](int u) {
      const int q = q0 + 8 * (u - nst), g = q / F, fa = q - g * F;
      const uint8_t* src = tb->gptr[g] + size_t(fa) * gu_row;
      uint8_t* dst = slot_ptr(u);
      uint64_t* bar = slot_bar(u);
      mbar_arrive_expect_tx(bar, 8u * uint32_t(gu_row));
      bulk_g2s(dst, src, 4u * uint32_t(gu_row), bar);
      bulk_g2s(dst + size_t(4) * gu_row + 16, src + size_t(4) * gu_row, 4u * uint32_t(gu_row), bar);
      mbar_arrive(bar);
    };
    auto issue_p2_down = [&](int u) {                   // first part of a down unit: the groups' down rows
      const int k = u - n1, ja = tb->p2_ja[k], jb = tb->p2_jb[k];
      uint8_t* dst = slot_ptr(u);
      uint64_t* bar = slot_bar(u);
      mbar_arrive_expect_tx(bar, uint32_t(jb - ja) * uint32_t(down_grp));
      for (int j = ja; j < jb; ++j)
        bulk_g2s(dst + size_t(j - ja) * down_grp, p2_rec(j) + rec_dblk + size_t(r0 / 2) * d_pair, uint32_t(down_grp),
                 bar);
    };
    auto issue_p2_h = [&](int u) {                      // second part: the h rows of its slots (after P1)
      const int k = u - n1, qa = tb->p2_qa[k], qb = tb->p2_qa[k + 1];
      uint8_t* dst = slot_ptr(u) + size_t(tb->p2_jb[k] - tb->p2_ja[k]) * down_grp;
      uint64_t* bar = slot_bar(u);
      mbar_arrive_expect_tx(bar, uint32_t(qb - qa) * uint32_t(hrow));
      const int sb = min(qb, T);                        // shared slots: h rows TK + q
      if (sb > qa) bulk_g2s(dst, a.h + size_t(TK + qa) * F, uint32_t(sb - qa) * hrow, bar);
      const int ra = max(qa, T);                        // grouped positions: h rows q - T
      if (qb > ra) bulk_g2s(dst + size_t(ra - qa) * hrow, a.h + size_t(ra - T) * F, uint32_t(qb - ra) * hrow, bar);
    };
    // the stream ends with the U rows of P3: nU pieces of up to rpp contiguous rows,
    // each one copy into a slot, issued as the last down units free their slots
    const int rpp = max(1, SB / (L * 2)), nU = (nur + rpp - 1) / rpp;
    auto issue_u = [&](int v, int n2) {
      const int i = v - (n1 + n2), ra = i * rpp, rb = min(nur, ra + rpp);
      uint64_t* bar = slot_bar(v);
      mbar_arrive_expect_tx(bar, uint32_t(rb - ra) * L * 2);
      bulk_g2s(slot_ptr(v), lw.U + size_t(j0 + ra) * L, uint32_t(rb - ra) * L * 2, bar);
      mbar_arrive(bar);
    };
    // P2 units: consecutive slots q packed into a slot's bytes (down rows of each group
    // touched, then the h rows); a group too large for one unit continues in the next
    auto build_p2 = [&]() {
      int k = 0;
      if (nr > 0) {
        int qa = 0, j = 0;
        while (qa < nslot && k < kMaxSlots) {
          while (qhi(j) <= qa) ++j;
          int bytes = 0, qb = qa, jj = j;
          for (; jj < ngr; ++jj) {
            const int want = qhi(jj) - qb;
            const int room = (SB - bytes - down_grp) / hrow;
            if (room <= 0) break;
            const int take = min(want, room);
            bytes += down_grp + take * hrow;
            qb += take;
            if (take < want) { ++jj; break; }
          }
          tb->p2_qa[k] = short(qa);
          tb->p2_ja[k] = short(j);
          tb->p2_jb[k] = short(jj);
          ++k;
          qa = qb;
        }
      }
      int gmax = 1;
      for (int i = 0; i < k; ++i) gmax = max(gmax, tb->p2_jb[i] - tb->p2_ja[i]);
      tb->p2_qa[k] = short(nslot);
      tb->n2 = k;
      tb->p2_gmax = gmax;
      __threadfence_block();
      *reinterpret_cast<volatile int*>(&tb->p2_ready) = 1;
    };
    // a down unit may be issued once the table exists (built by warp 1 at the start of P1)
    auto p2_table = [&]() -> int {
      volatile int* rp = &tb->p2_ready;
      if (!*rp) {
        const unsigned long long t0 = globaltimer_ns();
        while (!*rp) {
          __nanosleep(64);
          if (globaltimer_ns() - t0 > kWaitLimitNs) {
            atomicOr(a.err, kErrTimeout);
            return 0;
          }
        }
      }
      __threadfence_block();
      return tb->n2;
    };
    // warp-wide refills (every lane calls): lane 0 arms the slot's barrier and the copies
    // go out from different lanes, which the copy engine accepts faster than from one
    auto refill_p1 = [&](int v) {
      const int q = q0 + 8 * (v - nst), g = q / F, fa = q - g * F;
      uint64_t* bar = slot_bar(v);
      if (lane == 0) mbar_arrive_expect_tx(bar, 8u * uint32_t(gu_row));
      __syncwarp();
      if (lane < 2)
        bulk_g2s(slot_ptr(v) + size_t(lane) * (4 * gu_row + 16), tb->gptr[g] + size_t(fa + 4 * lane) * gu_row,
                 4u * uint32_t(gu_row), bar);
      if (lane == 0) mbar_arrive(bar);
    };
    auto refill_p2 = [&](int v, bool with_h) {
      const int k = v - n1, ja = tb->p2_ja[k], jb = tb->p2_jb[k];
      uint8_t* dst = slot_ptr(v);
      uint64_t* bar = slot_bar(v);
      if (lane == 0) mbar_arrive_expect_tx(bar, uint32_t(jb - ja) * uint32_t(down_grp));
      __syncwarp();
      for (int j = ja + lane; j < jb; j += 32)
        bulk_g2s(dst + size_t(j - ja) * down_grp, p2_rec(j) + rec_dblk + size_t(r0 / 2) * d_pair, uint32_t(down_grp),
                 bar);
      if (!with_h) return;
      const int qa = tb->p2_qa[k], qb = tb->p2_qa[k + 1];
      uint8_t* hd = dst + size_t(jb - ja) * down_grp;
      if (lane == 0) mbar_arrive_expect_tx(bar, uint32_t(qb - qa) * uint32_t(hrow));
      __syncwarp();
      const int sb = min(qb, T), ra = max(qa, T);
      if (lane == 1 && sb > qa) bulk_g2s(hd, a.h + size_t(TK + qa) * F, uint32_t(sb - qa) * hrow, bar);
      if (lane == 2 && qb > ra) bulk_g2s(hd + size_t(ra - qa) * hrow, a.h + size_t(ra - T) * F, uint32_t(qb - ra) * hrow, bar);
    };
    auto refill_u = [&](int v, int n2) {
      if (lane == 0) issue_u(v, n2);
    };
    {
      // the first units of the ring, and the fp32 scales of the selected records (16
      // bytes from each record's scale block: gate, up, down and the record's padding);
      // the routing tables for the caller are written while they are in flight
      if (warp == 0) {
        const int u = nst + lane;
        if (lane < S && u < n1) issue_p1(u);
      }
      if (warp == kScaleWarp) {                          // async copies: they complete on kMbScale
        for (int g = lane; g < nu; g += 32) cp_async16(&tb->gsc[g + 1], tb->gptr[g] + rec_body);
        asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(&tb->mbar[kMbScale]))
                     : "memory");
      }
      stamp0(li, kStP1Issued);
      // the routing tables for the caller (trace, and the last layer's copy read by
      // edge0_moe_debug_routing), each CTA a slice
      {
        const int s0 = TK * bid / G, s1 = TK * (bid + 1) / G;
        if (a.trace_idx)
          for (int s = s0 + tid; s < s1; s += kDecThreads) a.trace_idx[size_t(li) * TK + s] = tb->idx[s];
        if (last) {
          for (int s = s0 + tid; s < s1; s += kDecThreads) {
            a.idx[s] = tb->idx[s]; a.w[s] = tb->w[s]; a.perm[s] = tb->perm[s]; a.pos[s] = tb->posn[s];
          }
          const int ea = (E + 1) * bid / G, eb = (E + 1) * (bid + 1) / G;
          for (int e = ea + tid; e < eb; e += kDecThreads) {
            int off = TK, cnt = 0;
            for (int g = 0; g < nu; ++g) {
              if (tb->gexp[g] >= e) { off = tb->goff[g]; if (tb->gexp[g] == e) cnt = tb->goff[g + 1] - tb->goff[g]; break; }
            }
            a.offsets[e] = off;
            if (e < E) a.counts[e] = cnt;
          }
        }
      }
      if (warp == 1) {
        if (lane == 0) {
          build_p2();
          const int n2 = tb->n2;
          for (int u = n1; u < min(S + nst, n1 + n2); ++u) issue_p2_down(u);
          for (int u = n1 + n2; u < min(S + nst, n1 + n2 + nU); ++u) issue_u(u, n2);
        }
        __syncwarp();
      }
      // the gate/up units, part by part (a part: a range of K), in stream order
      const float sgg = tb->gsc[0].x, sgu = tb->gsc[0].y;
      const int nch = L / 32;
      const int np1 = n1 * ks;
      for (;;) {
        int pi = 0;
        if (lane == 0) pi = atomicAdd(&tb->pair_ctr[0], 1);
        pi = __shfl_sync(kFull, pi, 0);
        if (pi >= np1) break;
        const int u = pi / ks, part = pi - u * ks;
        // A rows 0-7 the gate rows, 8-15 the up rows of the same 8 f, so that each thread
        // holds gate and up of (f, token) for the SwiGLU
        MmaRows ar;
        const __half* brow[NT];
        bool bval[NT];
        int grp, fbase, ns;
        const uint8_t* row;
        if (u < nst) {                                   // the shared expert's rows f0 + 8u ..
          grp = -1;
          fbase = f0 + 8 * u;
          ns = T;
          const int r = 8 * u + g8;
          row = shr + size_t(r < nsr ? r : 0) * gu_pitch;
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            const int n = 8 * t + g8;
            bval[t] = n < T;
            brow[t] = zs + size_t(n < T ? n : 0) * zp;
          }
          wait_mb(cx, kMbShared);
        } else {
          const int q = q0 + 8 * (u - nst);
          grp = q / F;
          fbase = q - grp * F;
          ns = tb->goff[grp + 1] - tb->goff[grp];
          row = slot_ptr(u) + size_t(g8) * gu_row + (g8 >= 4 ? 16 : 0);
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            const int n = 8 * t + g8;
            bval[t] = n < ns;
            brow[t] = zs + size_t(n < ns ? tb->tokp[tb->goff[grp] + n] : 0) * zp;
          }
          ring_wait(u);
        }
        ar.code[0] = row; ar.code[1] = row + cofs_up;
        ar.scale[0] = row + sofs_g; ar.scale[1] = row + sofs_u;
        float acc[NT][4];
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
        // a group of at most 8 tokens needs one token tile
        if (NT == 1 || ns <= 8) fp4_mma_chunks<1>(ar, brow, bval, nch * part / ks, nch * (part + 1) / ks, acc);
        else fp4_mma_chunks<NT>(ar, brow, bval, nch * part / ks, nch * (part + 1) / ks, acc);
        if (ks > 1) {
          // partial sums of the unit's parts, added in part order by the last one
          float4* pb = part1 + (size_t((u % S) * ks + part) * 32 + lane) * NT;
#pragma unroll
          for (int t = 0; t < NT; ++t) pb[t] = make_float4(acc[t][0], acc[t][1], acc[t][2], acc[t][3]);
          if (!part_done(u, ks)) continue;
        }
        // every part has read the slot: refill it with the unit S places on (a down
        // unit: its first part); the slot's unit count moves on once the partial sums
        // are read too (the next unit on the slot writes them)
        {
          const int v = u + S;
          if (u >= nst) {
            if (v < n1) {
              refill_p1(v);
            } else {
              const int n2v = p2_table();
              if (v < n1 + n2v) refill_p2(v, false);
              else if (v < n1 + n2v + nU) refill_u(v, n2v);
            }
          }
        }
        if (ks > 1) partial_sum<NT>(part1, (u % S) * ks, ks, acc);
        __syncwarp();
        if (lane == 0) atomicAdd(&tb->ring_gen[u % S], 1);
        // SwiGLU: thread (g8, c4) holds gate / up of row f = fbase + g8 for the tokens
        // n = 8 t + 2 c4 + j; h in grouped order (the shared slots after them)
        if (grp >= 0) wait_mb(cx, kMbScale);
        const float gg = grp < 0 ? sgg : tb->gsc[grp + 1].x, gu = grp < 0 ? sgu : tb->gsc[grp + 1].y;
        if (grp >= 0 || 8 * u + g8 < nsr) {
          const int f = fbase + g8;
#pragma unroll
          for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const int n = 8 * t + 2 * c4 + j;
              if (n < ns) {
                const int hr = grp < 0 ? TK + n : tb->goff[grp] + n;
                const float zi = tb->zinv[grp < 0 ? n : tb->tokp[tb->goff[grp] + n]];
                a.h[size_t(hr) * F + f] = __float2bfloat16_rn(silu_f(gg * acc[t][j] * zi) * (gu * acc[t][2 + j] * zi));
              }
            }
        }
        __syncwarp();
      }
      __syncthreads();
      if (nsr > 0) release_mb(cx, 1u << kMbShared);
      if (tid < kRingMax) tb->ring_cnt[tid] = 0;          // parts are counted per phase
      if (tid == 0 && li + 1 < a.n_layers) {
        // next layer's D and R D into L2 while this layer finishes
        const LayerW nx = a.layers[li + 1];
        l2_prefetch_share(nx.D, size_t(L) * H * 2, bid, G);
        l2_prefetch_share(nx.RD, size_t(E) * H * 4, bid, G);
      }
    }
    stamp_end(li, kStP1EndMax);
    // h is written with generic stores and read by other CTAs' bulk copies
    asm volatile("fence.proxy.async.global;" ::: "memory");
    if (!grid_sync(a.bar, a.err)) { drain_copies(); return; }
    asm volatile("fence.proxy.async.global;" ::: "memory");
    stamp0(li, kStBar2);
    // ================================================================ P2: down + combine -> c
    LayerW nxt = lw;
    if (li + 1 < a.n_layers) nxt = a.layers[li + 1];
    {
      const int n2 = tb->n2;
      // the h rows of the units whose down rows were issued during P1
      // (units [n1, n1 + S): issued by the initial window or by a gate/up unit's refill)
      if (warp == 0 && lane < min(S, n2)) issue_p2_h(n1 + lane);
      stamp0(li, kStP2Staged);
      wait_mb(cx, kMbScale);
      // units of one or more groups; in the 16-token bucket each group's F columns are
      // split in two halves (more, shorter items for the warps; below it a group is one
      // item), and part p of a unit takes the items p, p + ks2, ... (ks2: the most items
      // in a unit, at most 8): every 16-row tile, A = the down rows (rho =
      // tile row), B = the half's h columns, first turned in place from bf16 into f16
      // times 2^-e_r (e_r from the max |h| of row r's half: exact for every element above
      // 2^-24 of it), so the down products run on the f16 path; each half writes its own
      // outputs, added in a fixed order by the combine
      constexpr int NH = NT == 2 ? 2 : 1;              // halves of F per group
      const int ks2 = min(8, NH * tb->p2_gmax);
      const int nchd = F / 32, f8 = F / 8, hch = nchd / NH;
      const int np2 = n2 * ks2;
      for (;;) {
        int pi = 0;
        if (lane == 0) pi = atomicAdd(&tb->pair_ctr[1], 1);
        pi = __shfl_sync(kFull, pi, 0);
        if (pi >= np2) break;
        const int k = pi / ks2, part = pi - k * ks2, u = n1 + k;
        ring_wait(u);
        const int qa = tb->p2_qa[k], qb = tb->p2_qa[k + 1], ja = tb->p2_ja[k], jb = tb->p2_jb[k];
        uint8_t* sbase = slot_ptr(u);
        uint8_t* hbase = sbase + size_t(jb - ja) * down_grp;
        for (int it = part; it < NH * (jb - ja); it += ks2) {
          const int jj = it / NH, half = it - jj * NH, j = ja + jj;
          const int qs = max(qa, qlo(j)), ns = min(qb, qhi(j)) - qs;
          const int x0 = half * hch * 4, x1 = half == NH - 1 ? f8 : (half + 1) * hch * 4;  // 16-byte pieces of a row
          float* obh = ob + size_t(half) * nslot * nr;
          float inv_row = 1.f;                          // lane r < ns: 2^e_r of row r
          for (int r = 0; r < ns; ++r) {
            uint4* rp = reinterpret_cast<uint4*>(hbase + size_t(qs - qa + r) * hrow);
            // the half's 16-byte pieces of the row, up to kConvPieces per lane in registers
            uint4 v[kConvPieces];
            float m = 0.f;
#pragma unroll
            for (int i = 0; i < kConvPieces; ++i) {
              const int ix = x0 + lane + 32 * i;
              v[i] = ix < x1 ? rp[ix] : make_uint4(0u, 0u, 0u, 0u);
              const float m01 = fmaxf(fmaxf(fabsf(bf16_lo(v[i].x)), fabsf(bf16_hi(v[i].x))),
                                      fmaxf(fabsf(bf16_lo(v[i].y)), fabsf(bf16_hi(v[i].y))));
              const float m23 = fmaxf(fmaxf(fabsf(bf16_lo(v[i].z)), fabsf(bf16_hi(v[i].z))),
                                      fmaxf(fabsf(bf16_lo(v[i].w)), fabsf(bf16_hi(v[i].w))));
              m = fmaxf(m, fmaxf(m01, m23));
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
            // sc = 2^-e with m * sc in [0.5, 1), from m's exponent field; sc = 1 for a zero
            // or subnormal max (the row then rounds to f16 zeros)
            const int ex = int((__float_as_uint(m) >> 23) & 0xFFu);
            float sc = 1.f, inv = 1.f;
            if (ex > 0 && ex < 253) {
              sc = __uint_as_float(uint32_t(253 - ex) << 23);
              inv = __uint_as_float(uint32_t(ex + 1) << 23);
            } else if (ex >= 253) {
              pow2_scale(m, &sc, &inv);
            }
            if (lane == r) inv_row = inv;
#pragma unroll
            for (int i = 0; i < kConvPieces; ++i) {
              const int ix = x0 + lane + 32 * i;
              if (ix < x1) {
                const uint32_t w4[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
                uint32_t o4[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const __half2 hv = __floats2half2_rn(bf16_lo(w4[e]) * sc, bf16_hi(w4[e]) * sc);
                  o4[e] = *reinterpret_cast<const uint32_t*>(&hv);
                }
                rp[ix] = make_uint4(o4[0], o4[1], o4[2], o4[3]);
              }
            }
          }
          __syncwarp();
          const float gd = tb->gsc[j].z;
          for (int rbase = 0; rbase < nr; rbase += 16) {
            MmaRows ar;
            const __half* brow[NT];
            bool bval[NT];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              int rho = rbase + g8 + 8 * hh;
              if (rho >= nr) rho = 0;
              const uint8_t* pr = sbase + size_t(jj) * down_grp + size_t(rho / 2) * d_pair;
              ar.code[hh] = pr + (rho & 1) * (F / 2);
              ar.scale[hh] = pr + F + (rho & 1) * (F / 16);
            }
#pragma unroll
            for (int t = 0; t < NT; ++t) {
              const int n = 8 * t + g8;
              bval[t] = n < ns;
              brow[t] = reinterpret_cast<const __half*>(hbase + size_t(qs - qa + (n < ns ? n : 0)) * hrow);
            }
            float acc[NT][4];
#pragma unroll
            for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
            const int c0 = half * hch, c1 = half == NH - 1 ? nchd : (half + 1) * hch;
            if (NT == 1 || ns <= 8) fp4_mma_chunks<1>(ar, brow, bval, c0, c1, acc);
            else fp4_mma_chunks<NT>(ar, brow, bval, c0, c1, acc);
#pragma unroll
            for (int t = 0; t < NT; ++t)
#pragma unroll
              for (int jx = 0; jx < 2; ++jx) {
                const int n = 8 * t + 2 * c4 + jx;
                const float inv_n = __shfl_sync(kFull, inv_row, n & 31);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                  const int rho = rbase + g8 + 8 * hh;
                  if (rho < nr && n < ns) {
                    const int q = qs + n;
                    const int slot = (q < T) ? TK + q : tb->perm[q - T];
                    obh[size_t(slot) * nr + rho] = gd * (acc[t][2 * hh + jx] * inv_n);
                  }
                }
              }
          }
        }
        if (!part_done(u, ks2)) continue;
        {
          const int v = u + S;
          if (v >= n1 + n2) {
            if (v < n1 + n2 + nU) refill_u(v, n2);
          } else {
            refill_p2(v, true);
          }
        }
        __syncwarp();
        if (lane == 0) atomicAdd(&tb->ring_gen[u % S], 1);
        __syncwarp();
      }
      __syncthreads();
      stamp0(li, kStP2Tasks);
      // combine: c[t][r] = o_shared + sum_k w[t][k] o[t*K + k], k ascending, each o the
      // sum of its halves of F (16-token bucket)
      const float* ob1 = ob + size_t(nslot) * nr;
      for (int p = tid; p < T * nr; p += kDecThreads) {
        const int t = p / nr, r = p % nr;
        const size_t sh = size_t(TK + t) * nr + r;
        float cv = NT == 2 ? ob[sh] + ob1[sh] : ob[sh];
        for (int j = 0; j < K; ++j) {
          const size_t o = size_t(t * K + j) * nr + r;
          cv = fmaf(tb->w[t * K + j], NT == 2 ? ob[o] + ob1[o] : ob[o], cv);
        }
        a.c[size_t(t) * L + r0 + r] = cv;
      }
      release_mb(cx, 1u << kMbScale);
    }
    stamp_end(li, kStP2EndMax);
    if (!grid_sync(a.bar, a.err)) { drain_copies(); return; }
    stamp0(li, kStBar3);
    // ================================================================ P3: y = U c
    // the next kernel on the stream may be scheduled from here (it waits for this
    // grid's completion before reading anything)
    if (last) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    {
      // U rows: the last nU units of the ring stream (each MMA warp waits for the pieces
      // holding its tile's rows)
      const int n2 = tb->n2, ubase = n1 + n2;
      const int nut = (nur + 15) / 16, wpt = nut > 0 ? kDecWarps / nut : kDecWarps;
      const int tile = warp / wpt, part = warp - tile * wpt;
      const int nchl = L / 32, s0 = nchl * part / wpt, s1 = nchl * (part + 1) / wpt;
      const bool mma_warp = tile < nut;
      auto u_row = [&](int r) {
        return reinterpret_cast<const __nv_bfloat16*>(slot_ptr(ubase + r / rpp) + size_t(r % rpp) * L * 2);
      };
      // c (all CTAs' rows) into shared memory in bf16, padded rows
      const int l8 = L / 8;
      for (int i = tid; i < T * l8; i += kDecThreads) {
        const int t = i / l8;
        const float4 p = reinterpret_cast<const float4*>(a.c)[2 * i];
        const float4 q = reinterpret_cast<const float4*>(a.c)[2 * i + 1];
        const __nv_bfloat162 b0 = __floats2bfloat162_rn(p.x, p.y), b1 = __floats2bfloat162_rn(p.z, p.w);
        const __nv_bfloat162 b2 = __floats2bfloat162_rn(q.x, q.y), b3 = __floats2bfloat162_rn(q.z, q.w);
        *reinterpret_cast<uint4*>(cs + size_t(t) * zp + 8 * (i - t * l8)) =
            make_uint4(*reinterpret_cast<const uint32_t*>(&b0), *reinterpret_cast<const uint32_t*>(&b1),
                       *reinterpret_cast<const uint32_t*>(&b2), *reinterpret_cast<const uint32_t*>(&b3));
      }
      __syncthreads();
      __nv_bfloat16* yo = (last && !a.final_norm) ? a.y : a.ybuf + size_t(li & 1) * T * H;
      __nv_bfloat16* ty = a.trace_y ? a.trace_y + size_t(li) * T * H : nullptr;
      float acc[NT][4];
#pragma unroll
      for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
      if (mma_warp) {
        const __nv_bfloat16* brow[NT];
        bool bval[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const int n = 8 * t + g8;
          bval[t] = n < T;
          brow[t] = cs + size_t(n < T ? n : 0) * zp;
        }
        const int ra0 = 16 * tile, ra1 = min(nur, ra0 + 16);
        for (int pc = ra0 / rpp; pc <= (ra1 - 1) / rpp; ++pc) ring_wait(ubase + pc);
        int ra = ra0 + g8, rb = ra0 + g8 + 8;
        if (ra >= nur) ra = ra0;
        if (rb >= nur) rb = ra0;
        bf16_mma_chunks<NT>(u_row(ra), u_row(rb), brow, bval, s0, s1, acc);
      }
      __syncthreads();                 // the U rows are read: the partial sums overwrite them
      partial_store<NT>(partw, acc);
      __syncthreads();
      if (warp < nut) {
        partial_sum<NT>(partw, warp * wpt, wpt, acc);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int rho = 16 * warp + g8 + 8 * hh;
          if (rho >= nur) continue;
#pragma unroll
          for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int jx = 0; jx < 2; ++jx) {
              const int n = 8 * t + 2 * c4 + jx;
              if (n < T) {
                const __nv_bfloat16 b = __float2bfloat16_rn(acc[t][2 * hh + jx]);
                yo[size_t(n) * H + j0 + rho] = b;
                if (ty) ty[size_t(n) * H + j0 + rho] = b;
              }
            }
        }
      }
    }
    // every ring slot's copies of this layer have been waited for: advance its parity by
    // the number of copies it took (its units, less the copy-less shared unit; nst <= S)
    {
      const int n_all = n1 + tb->n2 + nU, q = n_all / S, r = n_all - q * S;
      uint32_t flip = 0;
      for (int s = 0; s < S; ++s) flip |= uint32_t((q + (s < r) - (s < nst)) & 1) << (kMbRing + s);
      release_mb(cx, flip);
    }
    stamp_end(li, kStP3EndMax);
    if (!last || a.final_norm) {
      if (!grid_sync(a.bar, a.err)) { drain_copies(); return; }
      stamp0(li, kStBar4);
    }
    if (last && a.final_norm) {
      // stack output: RMSNorm(x_last + y_last); every CTA normalises, each writes its slice
      residual_norm(tb, xcur, a.ybuf + size_t(li & 1) * T * H, xs, xp, T, H, a.eps, [] {});
      const int h8 = H / 8, n8 = T * h8;
      const int i0 = bid * n8 / G, i1 = (bid + 1) * n8 / G;
      for (int i = i0 + tid; i < i1; i += kDecThreads) {
        const int t = i / h8;
        reinterpret_cast<uint4*>(a.y)[i] = *reinterpret_cast<const uint4*>(xs + size_t(t) * xp + 8 * (i - t * h8));
      }
    }
    lw = nxt;
  }
  // a wait that ran out may leave a copy in flight: let it land before exiting
  __syncthreads();
  if (tb->stuck) drain_copies();
}

// ------------------------------------------------------------------ host side
template <int NT>
static cudaError_t launch_nt(const DecodeArgs& a, int grid, int smem, cudaStream_t s) {
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
  cudaError_t e = cudaLaunchKernelEx(&cfg, moe_decode_kernel<NT>, a);
  if (e != cudaSuccess && pdl) {
    cudaGetLastError();
    pdl = 0;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, moe_decode_kernel<NT>, a);
  }
  return e;
}

int decode_bucket(int T) { return T <= 1 ? 1 : T <= 2 ? 2 : T <= 4 ? 4 : T <= 8 ? 8 : 16; }

cudaError_t decode_prepare(int smem) {
  cudaError_t e = cudaFuncSetAttribute(moe_decode_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(moe_decode_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

cudaError_t decode_occupancy(int smem, int* blocks) {
  int b1 = 0, b2 = 0;
  cudaError_t e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b1, moe_decode_kernel<1>, kDecThreads, smem)) != cudaSuccess)
    return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b2, moe_decode_kernel<2>, kDecThreads, smem)) != cudaSuccess)
    return e;
  *blocks = b1 < b2 ? b1 : b2;
  return cudaSuccess;
}

cudaError_t decode_launch(const DecodeArgs& a, int grid, int smem, cudaStream_t s) {
  return a.T > 8 ? launch_nt<2>(a, grid, smem, s) : launch_nt<1>(a, grid, smem, s);
}

}  // namespace edge0
