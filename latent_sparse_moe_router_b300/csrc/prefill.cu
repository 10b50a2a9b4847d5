// Prefill path (T > 16) of the latent-MoE layer.
//
// The layer ("Edge0-145B · Q3_K" model card, section "Architecture"): z = D x,
// router logits R z + b, top-k experts with renormalised softmax weights, the
// k routed SwiGLU experts plus the shared expert on z, their weighted sum c,
// y = U c.  At prefill sizes every step but routing is a contraction, so:
//   0. per-token power-of-two scale 2^-e_t with |z_t| * 2^-e_t < 1, from the bound
//      |z_t| <= max_r sum_h |D_rh| * max_h |x_t,h|;
//   1. one tcgen05 GEMM  x [T][H] x [D ; RDcat]^T -> z * 2^-e_t in f16 [T][L] and
//      logits fp32 [T][E]  (RDcat: the router folded into D once, R D in fp32, split
//      into bf16 high and low rows so the tensor cores keep ~16 mantissa bits);
//   2. top-k + softmax per token, expert histogram per 64-token chunk;
//   3. per-expert scan over the chunks, expert offsets and token-tile prefix;
//   4. deterministic scatter: slot s = t K + k goes to position
//      offsets[e] + (number of earlier slots of expert e), i.e. ordered by (t, k);
//   5. gather of the z rows in that order (and of their scales);
//   6. grouped NVFP4 GEMM gate/up + SwiGLU -> H bf16 (routed groups and the shared
//      expert as group E; f16 operands, the token scale undone in the epilogue);
//   7. grouped NVFP4 GEMM down -> O bf16;
//   8. combine c[t] = O[shared t] + sum_k w[t,k] O[pos[t,k]] in fixed k order;
//   9. tcgen05 GEMM  c x U^T -> y bf16 (round to nearest even).
// Grouped latent projections (G D/U pairs, a group label per expert): step 1's D is
// the G stacked D_g (z is [T][G l]), the router fold uses each expert's own D_g,
// step 5 gathers the latent of each expert's group, the shared expert reads its
// group's latent, step 8 adds each expert into its group's block of c [T][G l], and
// step 9 contracts over all G l columns (U [H][G l]): y = sum_g U_g c_g.
#include <algorithm>

#include "gemm_pair.cuh"
#include "grouped_kernel.cuh"
#include "prefill.cuh"
#include "tmap.cuh"

namespace edge0 {

namespace {

constexpr int kChunk = 64;          // tokens per routing chunk
constexpr int kPfBox = 128, kPfStages = 6;   // CTA-pair GEMM: 128-row B halves, 6 stages
// U GEMM split along K when its output tiles would leave most SM pairs idle (few tokens):
// at most kUSplits partial sums, for up to kUSplitTokens tokens
constexpr int kUSplits = 8, kUSplitTokens = 768;
// up to this many tokens the dense GEMMs put the weights on the MMA's M side and the
// tokens on N (rounded up to 16) instead of padding the tokens to 256 rows
constexpr int kSwapTokens = 64;
constexpr int kSwapStages = 10;     // their stages are 20 KB (16 KB of weights + <= 4 KB of tokens)

size_t pf_align(size_t v) { return (v + 1023) & ~size_t(1023); }

int pf_groups(const edge0_moe_desc& d) { return d.n_groups > 1 ? d.n_groups : 1; }

bool prefill_shapes_ok(const edge0_moe_desc& d) {
  return d.latent <= 2048 && d.ffn <= 2048 && d.n_experts <= 1024 && d.hidden % 64 == 0 &&
         size_t(pf_groups(d)) * d.latent <= 16384;
}

// ------------------------------------------------------------------ kernels
__global__ void split_rd_kernel(const float* __restrict__ rd, __nv_bfloat16* __restrict__ rdcat, int E, int H) {
  const size_t n = size_t(E) * H;
  for (size_t i = blockIdx.x * size_t(blockDim.x) + threadIdx.x; i < n; i += size_t(gridDim.x) * blockDim.x) {
    const size_t e = i / H, h = i % H;
    const float v = rd[i];
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
    rdcat[(2 * e) * H + h] = hi;
    rdcat[(2 * e + 1) * H + h] = lo;
  }
}

// Epilogue of x [D ; RDcat]^T: latent columns -> z * 2^-e_t in f16, router column
// pairs (high, low) -> logits fp32 (+ bias).
struct EpiXZ {
  __half* zh;
  const float* zsc;
  float* logits;
  const float* bias;
  int L, E;
  __device__ __forceinline__ void operator()(int row, int col0, const float* v) const {
    if (col0 < L) {
      const float sc = zsc[row];
      uint4* dst = reinterpret_cast<uint4*>(zh + size_t(row) * L + col0);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t u[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const __half2 b = __floats2half2_rn(v[8 * q + 2 * i] * sc, v[8 * q + 2 * i + 1] * sc);
          u[i] = *reinterpret_cast<const uint32_t*>(&b);
        }
        dst[q] = make_uint4(u[0], u[1], u[2], u[3]);
      }
    } else {
      const int e0 = (col0 - L) >> 1;
      if (e0 >= E) return;
      float4* dst = reinterpret_cast<float4*>(logits + size_t(row) * E + e0);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int j = 4 * q + i;
          o[i] = (v[2 * j] + v[2 * j + 1]) + (bias ? bias[e0 + j] : 0.f);
        }
        dst[q] = make_float4(o[0], o[1], o[2], o[3]);
      }
    }
  }
  // one value of output (row, col); the 32 lanes of a warp hold 32 consecutive columns
  // (L is a multiple of 32, so a warp is on one side of it; router columns 2e, 2e + 1
  // are lanes of the same warp)
  __device__ __forceinline__ void swapped(int row, int col, float v) const {
    if (col < L) {
      zh[size_t(row) * L + col] = __float2half_rn(v * zsc[row]);
    } else {
      const float lo = __shfl_down_sync(0xFFFFFFFFu, v, 1);
      const int e = (col - L) >> 1;
      if (!(col & 1) && e < E) logits[size_t(row) * E + e] = (v + lo) + (bias ? bias[e] : 0.f);
    }
  }
};

// fp32 partial sums of a K-split GEMM: row r + s M of split s lands in part[s][r][..].
struct EpiStoreF32 {
  float* part;
  int ldc;
  __device__ __forceinline__ void operator()(int row, int col0, const float* v) const {
    float* dst = part + size_t(row) * ldc + col0;
    if (col0 + 32 <= ldc) {
#pragma unroll
      for (int q = 0; q < 8; ++q)
        reinterpret_cast<float4*>(dst)[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    } else {
      for (int i = 0; i < 32; ++i)
        if (col0 + i < ldc) dst[i] = v[i];
    }
  }
  __device__ __forceinline__ void swapped(int row, int col, float v) const {
    if (col < ldc) part[size_t(row) * ldc + col] = v;
  }
};

// y = bf16(sum over s = 0 .. S-1 of part[s]) element by element, in s order.
__global__ void splitk_reduce_bf16_kernel(const float* __restrict__ part, int S, int MN, __nv_bfloat16* __restrict__ y) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < MN / 4; i += gridDim.x * blockDim.x) {
    float4 a = reinterpret_cast<const float4*>(part)[i];
    for (int sp = 1; sp < S; ++sp) {
      const float4 b = reinterpret_cast<const float4*>(part + size_t(sp) * MN)[i];
      a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
    }
    const __nv_bfloat162 lo = __floats2bfloat162_rn(a.x, a.y), hi = __floats2bfloat162_rn(a.z, a.w);
    reinterpret_cast<uint2*>(y)[i] = make_uint2(*reinterpret_cast<const uint32_t*>(&lo),
                                                *reinterpret_cast<const uint32_t*>(&hi));
  }
}

struct EpiStoreBF16 {
  __nv_bfloat16* C;
  int ldc, N;
  __device__ __forceinline__ void operator()(int row, int col0, const float* v) const {
    __nv_bfloat16* dst = C + size_t(row) * ldc + col0;
    if (col0 + 32 <= N) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t u[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const __nv_bfloat162 b = __floats2bfloat162_rn(v[8 * q + 2 * i], v[8 * q + 2 * i + 1]);
          u[i] = *reinterpret_cast<const uint32_t*>(&b);
        }
        reinterpret_cast<uint4*>(dst)[q] = make_uint4(u[0], u[1], u[2], u[3]);
      }
    } else {
      for (int i = 0; i < 32; ++i)
        if (col0 + i < N) dst[i] = __float2bfloat16_rn(v[i]);
    }
  }
  __device__ __forceinline__ void swapped(int row, int col, float v) const {
    if (col < N) C[size_t(row) * ldc + col] = __float2bfloat16_rn(v);
  }
};

// (value, index) order of the router: larger logit first, equal logits by lower index.
__device__ __forceinline__ bool pf_better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// Top-k + softmax weights per token (one warp per token, 8 warps, 64 tokens per
// block = one chunk) and the chunk's expert histogram.
__global__ void __launch_bounds__(256) topk_hist_kernel(const float* __restrict__ logits, int T, int E, int K,
                                                        int* __restrict__ idx, float* __restrict__ w,
                                                        int* __restrict__ chunk_cnt) {
  extern __shared__ float pf_sm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* buf = pf_sm + warp * E;
  int* hist = reinterpret_cast<int*>(pf_sm + 8 * E);
  for (int i = threadIdx.x; i < E; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int nj = E / 32;
  for (int tt = warp; tt < kChunk; tt += 8) {
    const int t = blockIdx.x * kChunk + tt;
    if (t >= T) break;
    const float* row = logits + size_t(t) * E;
    for (int i = lane; i < E; i += 32) {
      const float v = row[i];
      buf[i] = (v != v) ? -INFINITY : v;   // a NaN logit ranks last
    }
    __syncwarp();
    uint32_t taken = 0;
    float myv = 0.f;
    int myi = 0;
    for (int r = 0; r < K; ++r) {
      float bv = -INFINITY;
      int bi = 0x7FFFFFFF;
      for (int j = 0; j < nj; ++j) {
        if ((taken >> j) & 1u) continue;
        const int i = j * 32 + lane;
        const float v = buf[i];
        if (pf_better(v, i, bv, bi)) { bv = v; bi = i; }
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
        const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
        if (pf_better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
      }
      if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
      if (lane == r) { myv = bv; myi = bi; }
    }
    const float m = __shfl_sync(0xFFFFFFFFu, myv, 0);
    const float ex = lane < K ? expf(myv - m) : 0.f;
    float sum = ex;
#pragma unroll
    for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
    if (lane < K) {
      idx[size_t(t) * K + lane] = myi;
      w[size_t(t) * K + lane] = ex / sum;
      atomicAdd(&hist[myi], 1);
    }
    __syncwarp();
  }
  __syncthreads();
  for (int i = threadIdx.x; i < E; i += blockDim.x) chunk_cnt[size_t(blockIdx.x) * E + i] = hist[i];
}

// The same for E = 32 NJ with each lane's NJ logits in registers (no shared-memory
// pass per selection round): one warp per token, 16 warps of 4 tokens per block
// of 64 tokens.
template <int NJ>
__global__ void __launch_bounds__(512) topk_hist_reg_kernel(const float* __restrict__ logits, int T, int K,
                                                            int* __restrict__ idx, float* __restrict__ w,
                                                            int* __restrict__ chunk_cnt) {
  constexpr int E = NJ * 32;
  __shared__ int hist[E];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < E; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  for (int tt = warp; tt < kChunk; tt += 16) {
    const int t = blockIdx.x * kChunk + tt;
    if (t >= T) break;
    const float* row = logits + size_t(t) * E;
    float v[NJ];
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const float x = row[j * 32 + lane];
      v[j] = (x != x) ? -INFINITY : x;   // a NaN logit ranks last
    }
    uint32_t taken = 0;
    float myv = 0.f;
    int myi = 0;
    for (int r = 0; r < K; ++r) {
      float bv = -INFINITY;
      int bi = 0x7FFFFFFF;
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        const int i = j * 32 + lane;
        if (!((taken >> j) & 1u) && pf_better(v[j], i, bv, bi)) { bv = v[j]; bi = i; }
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
        const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
        if (pf_better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
      }
      if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
      if (lane == r) { myv = bv; myi = bi; }
    }
    const float m = __shfl_sync(0xFFFFFFFFu, myv, 0);
    const float ex = lane < K ? expf(myv - m) : 0.f;
    float sum = ex;
#pragma unroll
    for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
    if (lane < K) {
      idx[size_t(t) * K + lane] = myi;
      w[size_t(t) * K + lane] = ex / sum;
      atomicAdd(&hist[myi], 1);
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < E; i += blockDim.x) chunk_cnt[size_t(blockIdx.x) * E + i] = hist[i];
}

cudaError_t launch_topk_hist(const float* logits, int T, int E, int K, int* idx, float* w, int* chunk_cnt,
                             cudaStream_t s) {
  const int nch = (T + kChunk - 1) / kChunk;
  switch (E / 32) {
    case 2: topk_hist_reg_kernel<2><<<nch, 512, 0, s>>>(logits, T, K, idx, w, chunk_cnt); break;
    case 4: topk_hist_reg_kernel<4><<<nch, 512, 0, s>>>(logits, T, K, idx, w, chunk_cnt); break;
    case 8: topk_hist_reg_kernel<8><<<nch, 512, 0, s>>>(logits, T, K, idx, w, chunk_cnt); break;
    case 16: topk_hist_reg_kernel<16><<<nch, 512, 0, s>>>(logits, T, K, idx, w, chunk_cnt); break;
    default: topk_hist_kernel<<<nch, 256, (8 * E + E) * 4, s>>>(logits, T, E, K, idx, w, chunk_cnt);
  }
  return cudaGetLastError();
}

// Per expert: total count, and the chunk counts replaced by their exclusive
// prefix over the chunks.  Block = 32 experts x 32 chunk slices.
__global__ void __launch_bounds__(1024) scan_chunks_kernel(int* __restrict__ chunk_cnt, int nch, int E,
                                                           int* __restrict__ counts) {
  __shared__ int part[32][33];
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int e = blockIdx.x * 32 + tx;
  const int per = (nch + 31) / 32, c0 = ty * per, c1 = min(nch, c0 + per);
  int s = 0;
  for (int c = c0; c < c1; ++c) s += chunk_cnt[size_t(c) * E + e];
  part[ty][tx] = s;
  __syncthreads();
  if (ty == 0) {
    int run = 0;
    for (int k = 0; k < 32; ++k) {
      const int v = part[k][tx];
      part[k][tx] = run;
      run += v;
    }
    counts[e] = run;
  }
  __syncthreads();
  int run = part[ty][tx];
  for (int c = c0; c < c1; ++c) {
    const int v = chunk_cnt[size_t(c) * E + e];
    chunk_cnt[size_t(c) * E + e] = run;
    run += v;
  }
}

// Expert offsets (exclusive scan of the counts) and the token-tile prefix of the
// groups: tprefix[e] = sum over e' < e of ceil(count / 256), tprefix[E+1] adds the
// shared expert's ceil(T / 256).  One block of 1024 threads (E <= 1024).
__global__ void __launch_bounds__(1024) offsets_kernel(const int* __restrict__ counts, int E, int T,
                                                       int* __restrict__ offsets, int* __restrict__ tprefix) {
  __shared__ int wa[32], wb[32];
  const int e = threadIdx.x, lane = e & 31, warp = e >> 5;
  const int c = e < E ? counts[e] : 0;
  const int nt = (c + kGgBN - 1) / kGgBN;
  int a = c, b = nt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int ta = __shfl_up_sync(0xFFFFFFFFu, a, o), tb = __shfl_up_sync(0xFFFFFFFFu, b, o);
    if (lane >= o) { a += ta; b += tb; }
  }
  if (lane == 31) { wa[warp] = a; wb[warp] = b; }
  __syncthreads();
  if (warp == 0) {
    int x = wa[lane], y = wb[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int tx = __shfl_up_sync(0xFFFFFFFFu, x, o), ty = __shfl_up_sync(0xFFFFFFFFu, y, o);
      if (lane >= o) { x += tx; y += ty; }
    }
    wa[lane] = x;
    wb[lane] = y;
  }
  __syncthreads();
  const int ex_a = (warp ? wa[warp - 1] : 0) + a - c, ex_b = (warp ? wb[warp - 1] : 0) + b - nt;
  if (e < E) { offsets[e] = ex_a; tprefix[e] = ex_b; }
  if (e == E - 1) {
    offsets[E] = ex_a + c;
    tprefix[E] = ex_b + nt;
    tprefix[E + 1] = ex_b + nt + (T + kGgBN - 1) / kGgBN;
  }
}

// Slot s = t K + k of expert e goes to position offsets[e] + chunk base of e +
// rank among the chunk's earlier slots of e (slots in increasing s): the order
// (t, k) inside each expert group, independent of scheduling.  One warp per chunk.
__global__ void __launch_bounds__(256) scatter_kernel(const int* __restrict__ idx, const int* __restrict__ chunk_base,
                                                      const int* __restrict__ offsets, int T, int K, int E, int nch,
                                                      int* __restrict__ perm, int* __restrict__ pos) {
  extern __shared__ int pf_run[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x * 8 + warp;
  if (c >= nch) return;
  int* run = pf_run + warp * E;
  for (int i = lane; i < E; i += 32) run[i] = offsets[i] + chunk_base[size_t(c) * E + i];
  __syncwarp();
  const uint32_t lt = (1u << lane) - 1u;
  const int s0 = c * kChunk * K, s1 = min(T, (c + 1) * kChunk) * K;
  for (int b = s0; b < s1; b += 32) {
    const int s = b + lane;
    const bool act = s < s1;
    const uint32_t am = __ballot_sync(0xFFFFFFFFu, act);
    if (act) {
      const int e = idx[s];
      const uint32_t m = __match_any_sync(am, e);
      const int p = run[e] + __popc(m & lt);
      perm[p] = s;
      pos[s] = p;
      __syncwarp(am);
      if ((m & lt) == 0) run[e] += __popc(m);
    }
    __syncwarp();
  }
}

// Per-token scale: e_t = exponent of dnorm * max_h |x_t,h| (frexp: the bound lies in
// [2^(e-1), 2^e)), zsc = 2^-e_t, zinv = 2^e_t; the shared expert's positions
// TK + t take zinv too.  One warp per token.
__global__ void __launch_bounds__(256) token_scale_kernel(const __nv_bfloat16* __restrict__ x, int T, int H,
                                                          float dnorm, int TK, float* __restrict__ zsc,
                                                          float* __restrict__ zinv, float* __restrict__ pos_inv) {
  const int lane = threadIdx.x & 31, t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  const uint4* xv = reinterpret_cast<const uint4*>(x + size_t(t) * H);
  uint32_t m = 0;   // max |x| as bits (non-negative floats order as integers)
  for (int g = lane; g < H / 8; g += 32) {
    const uint4 a = xv[g];
    const uint32_t aa[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) m = max(m, max((aa[i] << 16) & 0x7FFF0000u, aa[i] & 0x7FFF0000u));
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if (lane == 0) {
    const float bound = __uint_as_float(m) * dnorm;
    int e = 0;
    if (bound > 0.f && isfinite(bound)) frexpf(bound, &e);
    zsc[t] = ldexpf(1.0f, -e);
    zinv[t] = ldexpf(1.0f, e);
    pos_inv[TK + t] = ldexpf(1.0f, e);
  }
}

// zg[p] = the latent of token perm[p] / K (with grouped projections: of the group
// labels[e] of its expert e = idx[perm[p]], columns labels[e] L .. of a row of ld
// elements; labels = null: one group, ld = L) and its scale: one warp per row,
// 16-byte copies.
__global__ void __launch_bounds__(256) gather_rows_kernel(const __half* __restrict__ zh,
                                                          const float* __restrict__ zinv,
                                                          const int* __restrict__ perm, int TK, int K, int L,
                                                          const int* __restrict__ idx,
                                                          const int* __restrict__ labels, int ld,
                                                          __half* __restrict__ zg, float* __restrict__ pos_inv) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n16 = L / 8;
  for (int p = blockIdx.x * 8 + warp; p < TK; p += gridDim.x * 8) {
    const int s = perm[p], t = s / K;
    const size_t col = labels ? size_t(labels[idx[s]]) * L : 0;
    const uint4* src = reinterpret_cast<const uint4*>(zh + size_t(t) * ld + col);
    uint4* dst = reinterpret_cast<uint4*>(zg + size_t(p) * L);
    for (int i = lane; i < n16; i += 32) dst[i] = src[i];
    if (lane == 0) pos_inv[p] = zinv[t];
  }
}

// c[t] = O[TK + t] + sum_k w[t,k] O[pos[t,k]]  (fp32, k in rank order) -> bf16.
// Block = one token, thread = 8 latent columns.
__global__ void combine_kernel(const __nv_bfloat16* __restrict__ ob, const int* __restrict__ pos,
                               const float* __restrict__ w, int T, int K, int L, __nv_bfloat16* __restrict__ cb) {
  const int t = blockIdx.x, j = threadIdx.x * 8;
  if (j >= L) return;
  const size_t TK = size_t(T) * K;
  float acc[8];
  {
    const uint4 u = *reinterpret_cast<const uint4*>(ob + (TK + t) * L + j);
    const uint32_t uu[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) { acc[2 * i] = bf16_lo(uu[i]); acc[2 * i + 1] = bf16_hi(uu[i]); }
  }
  for (int k = 0; k < K; ++k) {
    const int p = pos[size_t(t) * K + k];
    const float wk = w[size_t(t) * K + k];
    const uint4 u = *reinterpret_cast<const uint4*>(ob + size_t(p) * L + j);
    const uint32_t uu[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[2 * i] = fmaf(wk, bf16_lo(uu[i]), acc[2 * i]);
      acc[2 * i + 1] = fmaf(wk, bf16_hi(uu[i]), acc[2 * i + 1]);
    }
  }
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
    o[i] = *reinterpret_cast<const uint32_t*>(&b);
  }
  *reinterpret_cast<uint4*>(cb + size_t(t) * L + j) = make_uint4(o[0], o[1], o[2], o[3]);
}

// Grouped projections: c[t][g L + j] = [g = gs] O[TK + t][j] + sum over k with
// labels[idx[t,k]] = g of w[t,k] O[pos[t,k]][j]  (fp32, k in rank order) -> bf16;
// a group nobody used gets zeros.  Block (t, y) = token t, columns from 2048 y in
// steps of 2048 gridDim.y; thread = 8 columns at a time.
__global__ void __launch_bounds__(256) combine_grouped_kernel(const __nv_bfloat16* __restrict__ ob,
                                                              const int* __restrict__ pos,
                                                              const float* __restrict__ w,
                                                              const int* __restrict__ idx,
                                                              const int* __restrict__ labels, int gs, int T,
                                                              int K, int L, int G,
                                                              __nv_bfloat16* __restrict__ cb) {
  const int t = blockIdx.x, GL = G * L;
  const size_t TK = size_t(T) * K;
  for (int col = (blockIdx.y * blockDim.x + threadIdx.x) * 8; col < GL; col += gridDim.y * blockDim.x * 8) {
    const int g = col / L, j = col - g * L;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (g == gs) {
      const uint4 u = *reinterpret_cast<const uint4*>(ob + (TK + t) * L + j);
      const uint32_t uu[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) { acc[2 * i] = bf16_lo(uu[i]); acc[2 * i + 1] = bf16_hi(uu[i]); }
    }
    for (int k = 0; k < K; ++k) {
      if (labels[idx[size_t(t) * K + k]] != g) continue;
      const int p = pos[size_t(t) * K + k];
      const float wk = w[size_t(t) * K + k];
      const uint4 u = *reinterpret_cast<const uint4*>(ob + size_t(p) * L + j);
      const uint32_t uu[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] = fmaf(wk, bf16_lo(uu[i]), acc[2 * i]);
        acc[2 * i + 1] = fmaf(wk, bf16_hi(uu[i]), acc[2 * i + 1]);
      }
    }
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
      o[i] = *reinterpret_cast<const uint32_t*>(&b);
    }
    *reinterpret_cast<uint4*>(cb + size_t(t) * GL + col) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

cudaError_t launch_grouped(const GgMaps& maps, const GgParams& p, int num_sms, cudaStream_t s) {
  static int max_pairs = 0;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kGgThreads);
  cfg.dynamicSmemBytes = GgSmem::kBytes;
  cfg.stream = s;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  if (max_pairs == 0) {
    cudaError_t e =
        cudaFuncSetAttribute(grouped_nvfp4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, GgSmem::kBytes);
    cfg.gridDim = dim3(2 * (num_sms / 2));
    int clusters = 0;
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveClusters(&clusters, grouped_nvfp4_kernel, &cfg);
    if (e != cudaSuccess) return e;
    if (clusters < 1) return cudaErrorInvalidConfiguration;
    max_pairs = clusters;
  }
  // persistent: every resident pair walks the pair tiles (their count is read on the device)
  cfg.gridDim = dim3(2 * max_pairs);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, grouped_nvfp4_kernel, maps, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

// ------------------------------------------------------------------ workspace
size_t prefill_workspace_bytes(const edge0_moe_desc& d, int max_tokens) {
  // one group: T <= 16 runs the decode kernel; grouped layers run these kernels at every T
  if ((max_tokens <= 16 && pf_groups(d) == 1) || max_tokens < 1 || !prefill_shapes_ok(d)) return 0;
  const size_t T = max_tokens, H = d.hidden, L = d.latent, E = d.n_experts, K = d.top_k, F = d.ffn;
  const size_t GL = size_t(pf_groups(d)) * L;
  const size_t nch = (T + kChunk - 1) / kChunk;
  size_t n = 0;
  n += pf_align(2 * E * H * 2);               // rdcat
  n += pf_align(T * GL * 2);                  // zh
  n += pf_align(T * 4) * 2;                   // zsc, zinv
  n += pf_align((T * K + T) * 4);             // pos_inv
  n += pf_align(T * E * 4);                   // logits
  n += pf_align(nch * E * 4);                 // chunk_cnt
  n += pf_align((E + 2) * 4);                 // tprefix
  n += pf_align(T * K * L * 2);               // zg
  n += pf_align((T * K + T) * F * 2);         // hb
  n += pf_align((T * K + T) * L * 2);         // ob
  n += pf_align(T * GL * 2);                  // cb
  n += pf_align(T * H * 2);                   // scratch
  n += pf_align(size_t(kUSplits) * std::min<size_t>(T, kUSplitTokens) * H * 4);   // U partial sums
  n += pf_align(4);                           // abort
  return n;
}

void prefill_workspace_carve(const edge0_moe_desc& d, int max_tokens, char* base, PrefillWorkspace* pf) {
  pf->max_tokens = max_tokens;
  if (prefill_workspace_bytes(d, max_tokens) == 0) return;
  const size_t T = max_tokens, H = d.hidden, L = d.latent, E = d.n_experts, K = d.top_k, F = d.ffn;
  const size_t GL = size_t(pf_groups(d)) * L;
  const size_t nch = (T + kChunk - 1) / kChunk;
  size_t o = 0;
  auto take = [&](size_t bytes) { char* p = base + o; o += pf_align(bytes); return p; };
  pf->rdcat = reinterpret_cast<__nv_bfloat16*>(take(2 * E * H * 2));
  pf->zh = reinterpret_cast<__half*>(take(T * GL * 2));
  pf->zsc = reinterpret_cast<float*>(take(T * 4));
  pf->zinv = reinterpret_cast<float*>(take(T * 4));
  pf->pos_inv = reinterpret_cast<float*>(take((T * K + T) * 4));
  pf->logits = reinterpret_cast<float*>(take(T * E * 4));
  pf->chunk_cnt = reinterpret_cast<int*>(take(nch * E * 4));
  pf->tprefix = reinterpret_cast<int*>(take((E + 2) * 4));
  pf->zg = reinterpret_cast<__half*>(take(T * K * L * 2));
  pf->hb = reinterpret_cast<__nv_bfloat16*>(take((T * K + T) * F * 2));
  pf->ob = reinterpret_cast<__nv_bfloat16*>(take((T * K + T) * L * 2));
  pf->cb = reinterpret_cast<__nv_bfloat16*>(take(T * GL * 2));
  pf->scratch = reinterpret_cast<__nv_bfloat16*>(take(T * H * 2));
  pf->upart = reinterpret_cast<float*>(take(size_t(kUSplits) * std::min<size_t>(T, kUSplitTokens) * H * 4));
  pf->abort = reinterpret_cast<int*>(take(4));
}

cudaError_t prefill_init(const edge0_moe_desc& d, PrefillWorkspace* pf, int num_sms) {
  if (!pf->rdcat) return cudaSuccess;
  const int H = d.hidden, L = d.latent, E = d.n_experts, K = d.top_k, F = d.ffn;
  const int G = pf_groups(d), GL = G * L, gs = G > 1 ? d.shared_group : 0;
  const size_t T = pf->max_tokens, TK = T * K;
  split_rd_kernel<<<num_sms * 4, 256>>>(pf->rd, pf->rdcat, E, H);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const auto SW = CU_TENSOR_MAP_SWIZZLE_128B, NS = CU_TENSOR_MAP_SWIZZLE_NONE;
  const uint8_t* ex = static_cast<const uint8_t*>(d.experts);
  const uint8_t* sh = static_cast<const uint8_t*>(d.shared_expert);
  const uint64_t gu_row = 9ull * L / 8, d_pair = 9ull * F / 8, d_block = uint64_t(F) * gu_row;
  bool ok = true;
  // dense GEMM operands
  ok &= make_tmap_2d(&pf->m_D, d.D, BF, 2, GL, H, uint64_t(H) * 2, 64, kPfBox, SW);
  ok &= make_tmap_2d(&pf->m_rdcat, pf->rdcat, BF, 2, 2ull * E, H, uint64_t(H) * 2, 64, kPfBox, SW);
  ok &= make_tmap_2d(&pf->m_U, d.U, BF, 2, H, GL, uint64_t(GL) * 2, 64, kPfBox, SW);
  ok &= make_tmap_2d(&pf->m_cb, pf->cb, BF, 2, T, GL, uint64_t(GL) * 2, 64, 128, SW);
  // gate/up: records' GU blocks [E][F rows][9L/8 bytes]
  ok &= make_tmap_3d(&pf->maps1.a_codes, ex, U8, gu_row, F, E, gu_row, d.expert_stride, 32, 64, 1, NS);
  ok &= make_tmap_3d(&pf->maps1.a_scales, ex, U8, gu_row, F, E, gu_row, d.expert_stride, L / 16, 64, 1, NS);
  ok &= make_tmap_2d(&pf->maps1.s_codes, sh, U8, 1, F, gu_row, gu_row, 32, 64, NS);
  ok &= make_tmap_2d(&pf->maps1.s_scales, sh, U8, 1, F, gu_row, gu_row, L / 16, 64, NS);
  const auto F16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  ok &= make_tmap_2d(&pf->maps1.b_routed, pf->zg, F16, 2, TK, L, uint64_t(L) * 2, 64, kGgBBox, SW);
  ok &= make_tmap_2d(&pf->maps1.b_shared, pf->zh + size_t(gs) * L, F16, 2, T, L, uint64_t(GL) * 2, 64, kGgBBox,
                     SW);
  // down: records' D blocks [E][L/2 row pairs][9F/8 bytes]
  ok &= make_tmap_3d(&pf->maps2.a_codes, ex + d_block, U8, d_pair, L / 2, E, d_pair, d.expert_stride, 32, 64, 1, NS);
  ok &= make_tmap_3d(&pf->maps2.a_scales, ex + d_block, U8, d_pair, L / 2, E, d_pair, d.expert_stride, F / 8, 64, 1,
                     NS);
  ok &= make_tmap_2d(&pf->maps2.s_codes, sh + d_block, U8, 1, L / 2, d_pair, d_pair, 32, 64, NS);
  ok &= make_tmap_2d(&pf->maps2.s_scales, sh + d_block, U8, 1, L / 2, d_pair, d_pair, F / 8, 64, NS);
  ok &= make_tmap_2d(&pf->maps2.b_routed, pf->hb, BF, 2, TK + T, F, uint64_t(F) * 2, 64, kGgBBox, SW);
  pf->maps2.b_shared = pf->maps2.b_routed;
  return ok ? cudaSuccess : cudaErrorInvalidValue;
}

edge0_status prefill_forward(const edge0_moe_desc& d, PrefillWorkspace* pf, int num_sms, const __nv_bfloat16* x,
                             __nv_bfloat16* y, int T, cudaStream_t s) {
  if (!pf->rdcat) return EDGE0_ERR_UNSUPPORTED;
  if (T > pf->max_tokens) return EDGE0_ERR_INVALID_ARG;
  const int H = d.hidden, L = d.latent, E = d.n_experts, K = d.top_k, F = d.ffn;
  const int G = pf_groups(d), GL = G * L;
  const int TK = T * K, nch = (T + kChunk - 1) / kChunk;
  CUtensorMap mx;
  if (!make_tmap_2d(&mx, x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, T, H, uint64_t(H) * 2, 64, 128,
                    CU_TENSOR_MAP_SWIZZLE_128B))
    return EDGE0_ERR_CUDA;
  cudaError_t e = cudaMemsetAsync(pf->abort, 0, sizeof(int), s);
  pf->timed = false;
  int stage = 0;
  auto mark = [&]() {
    if (pf->profile && e == cudaSuccess) e = cudaEventRecord(pf->events[stage++], s);
  };
  mark();
  // 0. token scales
  if (e == cudaSuccess) {
    token_scale_kernel<<<(T + 7) / 8, 256, 0, s>>>(x, T, H, pf->dnorm, TK, pf->zsc, pf->zinv, pf->pos_inv);
    e = cudaGetLastError();
  }
  // 1. x -> z (f16, scaled), logits
  const bool swap = T <= kSwapTokens;
  const uint32_t nb2 = uint32_t(((T + 15) & ~15) / 2);   // token rows per CTA with swapped roles
  if (e == cudaSuccess) {
    const EpiXZ epi{pf->zh, pf->zsc, pf->logits, d.router_bias, GL, E};
    if (swap) {
      CUtensorMap mxs;
      if (!make_tmap_2d(&mxs, x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, T, H, uint64_t(H) * 2, 64, nb2,
                        CU_TENSOR_MAP_SWIZZLE_128B))
        return EDGE0_ERR_CUDA;
      e = launch_gemm_pair<kSwapStages, EpiXZ, true>(mxs, pf->m_D, pf->m_rdcat, T, GL + 2 * E, H, GL, pf->err,
                                                   pf->abort, epi, s);
    } else {
      e = launch_gemm_pair<kPfStages>(mx, pf->m_D, pf->m_rdcat, T, GL + 2 * E, H, GL, pf->err, pf->abort, epi, s);
    }
  }
  mark();
  // 2-4. routing and permutation
  if (e == cudaSuccess) {
    e = launch_topk_hist(pf->logits, T, E, K, pf->idx, pf->w, pf->chunk_cnt, s);
  }
  mark();
  if (e == cudaSuccess) {
    scan_chunks_kernel<<<E / 32, dim3(32, 32), 0, s>>>(pf->chunk_cnt, nch, E, pf->counts);
    e = cudaGetLastError();
  }
  mark();
  if (e == cudaSuccess) {
    offsets_kernel<<<1, 1024, 0, s>>>(pf->counts, E, T, pf->offsets, pf->tprefix);
    e = cudaGetLastError();
  }
  mark();
  if (e == cudaSuccess) {
    scatter_kernel<<<(nch + 7) / 8, 256, 8 * E * 4, s>>>(pf->idx, pf->chunk_cnt, pf->offsets, T, K, E, nch, pf->perm,
                                                         pf->pos);
    e = cudaGetLastError();
  }
  mark();
  // 5. grouped z rows
  if (e == cudaSuccess) {
    const int blocks = std::min((TK + 7) / 8, num_sms * 16);
    gather_rows_kernel<<<blocks, 256, 0, s>>>(pf->zh, pf->zinv, pf->perm, TK, K, L, pf->idx,
                                              G > 1 ? d.expert_group : nullptr, GL, pf->zg, pf->pos_inv);
    e = cudaGetLastError();
  }
  mark();
  // 6-7. experts
  GgParams gp;
  gp.T = T; gp.TK = TK; gp.L = L; gp.F = F; gp.E = E;
  gp.counts = pf->counts; gp.offsets = pf->offsets; gp.tprefix = pf->tprefix;
  gp.experts = static_cast<const uint8_t*>(d.experts);
  gp.stride = d.expert_stride;
  gp.shared = static_cast<const uint8_t*>(d.shared_expert);
  gp.err = pf->err;
  gp.abort = pf->abort;
  if (e == cudaSuccess) {
    gp.mode = 1; gp.mtiles = F / 64; gp.out = pf->hb; gp.out_ld = F; gp.pos_inv = pf->pos_inv;
    e = launch_grouped(pf->maps1, gp, num_sms, s);
  }
  mark();
  if (e == cudaSuccess) {
    gp.mode = 2; gp.mtiles = L / 128; gp.out = pf->ob; gp.out_ld = L; gp.pos_inv = nullptr;
    e = launch_grouped(pf->maps2, gp, num_sms, s);
  }
  mark();
  // 8. combine
  if (e == cudaSuccess) {
    if (G == 1) {
      combine_kernel<<<T, (L / 8 + 31) / 32 * 32, 0, s>>>(pf->ob, pf->pos, pf->w, T, K, L, pf->cb);
    } else {
      // enough blocks for the SMs when there are few tokens, one per token otherwise
      const int gy = std::max(1, std::min((GL + 2047) / 2048, (8 * num_sms + T - 1) / T));
      combine_grouped_kernel<<<dim3(T, gy), 256, 0, s>>>(pf->ob, pf->pos, pf->w, pf->idx, d.expert_group,
                                                         d.shared_group, T, K, L, G, pf->cb);
    }
    e = cudaGetLastError();
  }
  mark();
  // 9. y = c U^T; with few output tiles, split along K (partial sums, then their sum
  // in split order) so that the SM pairs stream U together
  if (e == cudaSuccess) {
    const int pairs = num_sms / 2, tiles = ((T + 255) / 256) * ((H + 255) / 256);
    const int ksp = T <= kUSplitTokens && 2 * tiles <= pairs ? std::min({kUSplits, pairs / tiles, GL / 128}) : 1;
    CUtensorMap mcs;                          // c rows, boxes of nb2 rows (swapped roles)
    if (swap && !make_tmap_2d(&mcs, pf->cb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, T, GL, uint64_t(GL) * 2, 64, nb2,
                              CU_TENSOR_MAP_SWIZZLE_128B))
      return EDGE0_ERR_CUDA;
    if (ksp > 1) {
      if (swap)
        e = launch_gemm_pair<kSwapStages, EpiStoreF32, true>(mcs, pf->m_U, pf->m_U, T, H, GL, 1 << 30, pf->err,
                                                           pf->abort, EpiStoreF32{pf->upart, H}, s, ksp);
      else
        e = launch_gemm_pair<kPfStages>(pf->m_cb, pf->m_U, pf->m_U, T, H, GL, 1 << 30, pf->err, pf->abort,
                                        EpiStoreF32{pf->upart, H}, s, ksp);
      if (e == cudaSuccess) {
        splitk_reduce_bf16_kernel<<<std::min((T * H / 4 + 255) / 256, num_sms * 4), 256, 0, s>>>(pf->upart, ksp,
                                                                                                 T * H, y);
        e = cudaGetLastError();
      }
    } else if (swap) {
      e = launch_gemm_pair<kSwapStages, EpiStoreBF16, true>(mcs, pf->m_U, pf->m_U, T, H, GL, 1 << 30, pf->err,
                                                          pf->abort, EpiStoreBF16{y, H, H}, s);
    } else {
      e = launch_gemm_pair<kPfStages>(pf->m_cb, pf->m_U, pf->m_U, T, H, GL, 1 << 30, pf->err, pf->abort,
                                      EpiStoreBF16{y, H, H}, s);
    }
  }
  mark();
  if (pf->profile && e == cudaSuccess) pf->timed = (stage == 11);
  return e == cudaSuccess ? EDGE0_OK : EDGE0_ERR_CUDA;
}

const void* prefill_debug_tensor(const PrefillWorkspace* pf, int what, const edge0_moe_desc& d, int T,
                                 size_t* bytes) {
  if (!pf->rdcat) return nullptr;
  const size_t GL = size_t(pf_groups(d)) * d.latent;
  if (what == 0) { *bytes = size_t(T) * GL * 2; return pf->zh; }
  if (what == 1) { *bytes = size_t(T) * d.n_experts * 4; return pf->logits; }
  if (what == 2) { *bytes = size_t(T) * GL * 2; return pf->cb; }
  const size_t rows = size_t(T) * d.top_k + T;
  if (what == 3) { *bytes = rows * d.ffn * 2; return pf->hb; }
  if (what == 4) { *bytes = rows * d.latent * 2; return pf->ob; }
  return nullptr;
}

__nv_bfloat16* prefill_stack_scratch(PrefillWorkspace* pf) { return pf->scratch; }

cudaError_t prefill_profile(PrefillWorkspace* pf, bool enable) {
  if (enable && !pf->events[0]) {
    for (auto& ev : pf->events) {
      const cudaError_t e = cudaEventCreate(&ev);
      if (e != cudaSuccess) return e;
    }
  }
  pf->profile = enable;
  pf->timed = false;
  return cudaSuccess;
}

edge0_status prefill_stage_times(PrefillWorkspace* pf, float* ms, int max, int* n_out) {
  if (!pf->timed) return EDGE0_ERR_UNSUPPORTED;
  if (cudaEventSynchronize(pf->events[10]) != cudaSuccess) return EDGE0_ERR_CUDA;
  const int n = max < 10 ? max : 10;
  for (int i = 0; i < n; ++i)
    if (cudaEventElapsedTime(&ms[i], pf->events[i], pf->events[i + 1]) != cudaSuccess) return EDGE0_ERR_CUDA;
  if (n_out) *n_out = n;
  return EDGE0_OK;
}

void prefill_destroy(PrefillWorkspace* pf) {
  for (auto& ev : pf->events)
    if (ev) cudaEventDestroy(ev);
}

}  // namespace edge0
