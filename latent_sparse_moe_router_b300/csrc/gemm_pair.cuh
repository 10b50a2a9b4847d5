// Dense bf16 GEMM on a CTA pair (2-SM tcgen05), C = A * B^T.
//
//   A [M][K] bf16 row-major (K-major), B [N][K] bf16 row-major (K-major),
//   fp32 accumulation in TMEM, results handed to an epilogue functor.
// A cluster of two CTAs computes 256 x 256 output tiles: CTA r (rank in the pair)
// stages rows m0 + 128 r .. + 127 of A and rows n0 + 128 r .. + 127 of B (128 x 64,
// 128-byte swizzle) per 64-wide k-step, so each SM moves half the B tile a
// single-CTA 128 x 256 tile would need through its shared memory and from L2.
// Persistent: the pairs walk the tiles (i -> split = i % k_splits, and with
// j = i / k_splits, m = j / n_tiles, n = j % n_tiles) with a stride of the number of
// pairs; a tile of split s covers k-steps [s nk / k_splits, (s + 1) nk / k_splits) and
// hands its rows to the epilogue as row + s M (k_splits = 1: the whole K, row).
// Warp roles in both CTAs:
//   warp 0 (one lane): TMA producer; both CTAs' copies complete on rank 0's `full`
//     barrier (two arrivals with their byte counts);
//   warp 1 (one lane, rank 0 only): tcgen05.mma.cta_group::2 (M=256, N=256, K=16,
//     four per k-step) into one of two TMEM accumulators of 256 columns; its commits
//     arrive on `empty` / `acc_full` in both CTAs;
//   warps 2-5: epilogue of the CTA's 128 accumulator rows (tcgen05.ld, thread = row,
//     32 columns per load), overlapping the next tile's main loop; each warp then
//     arrives on rank 0's `acc_empty` (eight arrivals).
// Every wait is bounded; both CTAs run the same tile sequence and reach the
// collective TMEM allocation and release.
//
// SWAP (few rows of A, M <= 64): the roles turn around so that the tensor cores do not
// compute 256 padded rows.  The MMA's M side takes 256 rows of B (CTA r: rows
// n0 + 128 r ..), its N side A's rows rounded up to NB, a multiple of 16 (CTA r: A rows
// r NB/2 .. r NB/2 + NB/2 - 1, the A map's box NB/2 rows high), so the accumulator is
// [B row][A row]: epilogue thread = one output column, and the epilogue's
// swapped(row, col, v) takes one value of one output row at a time (all 32 lanes of a
// warp call it together, for 32 consecutive columns).
#pragma once

#include "pair.cuh"

namespace edge0 {

constexpr int kGemmPairThreads = 192;

// Named barrier `id` over n threads that also returns whether pred held in all of them.
__device__ __forceinline__ bool gemm_named_and(int id, int n, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
      " barrier.cta.red.and.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r) : "r"(uint32_t(pred)), "r"(id), "r"(n) : "memory");
  return r != 0;
}

template <int STAGES, bool SWAP = false>
struct GemmPairSmem {
  static constexpr int kA = 128 * 64 * 2;   // one A stage (bytes; with SWAP: B's 128 rows)
  // one B stage (this CTA's half; with SWAP: A's NB/2 <= 32 rows)
  static constexpr int kB = SWAP ? 32 * 64 * 2 : 128 * 64 * 2;
  static constexpr int kStage = kA + kB;
  // barriers and tmem slot, alignment, and 16 KB of slack past the last stage
  static constexpr int kBytes = STAGES * kStage + 1024 + 1024 + 16384;
};

// Epilogue interface: operator()(int row, int col0, const float* v32) for the 32
// consecutive columns col0 .. col0+31 of one row (plus s M for split s of a K-split
// launch); rows >= M are not passed.
// Output columns [0, n_split) multiply B's rows, columns from n_split on multiply
// B2's rows (n_split a multiple of 256; pass B2 = B for one matrix).
template <int STAGES, class Epi, bool SWAP>
__global__ void __launch_bounds__(kGemmPairThreads, 1)
gemm_pair_bf16_tn_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                         const __grid_constant__ CUtensorMap tmB2, int M, int N, int K, int n_split,
                         int k_splits, int* err, int* abort, Epi epi) {
  using S = GemmPairSmem<STAGES, SWAP>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * S::kStage);   // rank 0: 2 arrivals + bytes
  uint64_t* empty = full + STAGES;         // both: MMA commit
  uint64_t* acc_full = empty + STAGES;     // [2] both: MMA commit
  uint64_t* acc_empty = acc_full + 2;      // [2] rank 0: one arrival per epilogue warp of the pair
  uint64_t* mma_done = acc_empty + 2;      // rank 0
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  int* s_bad = reinterpret_cast<int*>(tmem_slot + 2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int nk = K / 64;
  const int n_tiles = (N + 255) / 256;
  const int m_tiles = SWAP ? 1 : (M + 255) / 256;
  const int NB = SWAP ? (M + 15) & ~15 : 256;     // the MMA's N
  const int total = m_tiles * n_tiles * k_splits;
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  if (pair >= total) return;   // both CTAs of the pair leave together

  if (threadIdx.x == 0) {
    *s_bad = 0;
    for (int s = 0; s < STAGES; ++s) { mbar_init(&full[s], 2); mbar_init(&empty[s], 1); }
    for (int b = 0; b < 2; ++b) { mbar_init(&acc_full[b], 1); mbar_init(&acc_empty[b], 8); }
    mbar_init(mma_done, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (warp == 1) { tmem_alloc_pair(tmem_slot, 512); tmem_relinquish_pair(); }
  tc_fence_before();
  // both CTAs' barriers exist and the pair's TMEM is allocated before anyone signals
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmB);
      prefetch_tmap(&tmB2);
      const uint32_t full0 = mapa_shared(smem_u32(full), 0);
      int it = 0;
      for (int tile = pair; ok && tile < total; tile += npairs) {
        const int ks = tile % k_splits, mn = tile / k_splits;
        const int m0 = (mn / n_tiles) * 256, n0 = (mn % n_tiles) * 256;
        const int ya = m0 + 128 * int(rank), yb = n0 + 128 * int(rank);
        const int kb1 = (ks + 1) * nk / k_splits;
        for (int kb = ks * nk / k_splits; kb < kb1; ++kb, ++it) {
          const int s = it % STAGES;
          if (!mbar_wait_abort(&empty[s], ((it / STAGES) & 1) ^ 1, err, abort)) { ok = false; break; }
          uint8_t* sa = smem + s * S::kStage;
          const uint32_t fb = full0 + uint32_t(s) * 8u;
          if constexpr (SWAP) {
            // M side: B's (or B2's) 128 rows of this CTA; N side: A's NB / 2 rows
            mbar_arrive_expect_tx_cl(fb, S::kA + uint32_t(NB / 2) * 128u);
            if (n0 < n_split) tma_load_2d_pair(sa, &tmB, kb * 64, yb, fb);
            else tma_load_2d_pair(sa, &tmB2, kb * 64, yb - n_split, fb);
            tma_load_2d_pair(sa + S::kA, &tmA, kb * 64, (NB / 2) * int(rank), fb);
          } else {
            mbar_arrive_expect_tx_cl(fb, S::kStage);
            tma_load_2d_pair(sa, &tmA, kb * 64, ya, fb);
            // columns [0, n_split) come from B's rows, later columns from B2's rows
            if (n0 < n_split) tma_load_2d_pair(sa + S::kA, &tmB, kb * 64, yb, fb);
            else tma_load_2d_pair(sa + S::kA, &tmB2, kb * 64, yb - n_split, fb);
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      const uint32_t idesc = idesc_bf16_f32(256, NB);
      int it = 0, ti = 0;
      for (int tile = pair; ok && tile < total; tile += npairs, ++ti) {
        const int ab = ti & 1;
        if (!mbar_wait_cl_abort(&acc_empty[ab], ((ti >> 1) & 1) ^ 1, err, abort)) { ok = false; break; }
        tc_fence_after();
        const uint32_t acc = tmem + ab * 256;
        const int ks = tile % k_splits, kb0 = ks * nk / k_splits, kb1 = (ks + 1) * nk / k_splits;
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const int s = it % STAGES;
          // the stage's bytes were written by bulk copies: the barrier's completion orders
          // them before the MMA, no cluster-scope acquire is needed
          if (!mbar_wait_abort(&full[s], (it / STAGES) & 1, err, abort)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + s * S::kStage);
          const uint32_t sb = sa + S::kA;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_pair_f16(acc, sw128_desc(sa + k * 32), sw128_desc(sb + k * 32), idesc, kb != kb0 || k != 0);
          mma_pair_commit_both(&empty[s]);
        }
        if (!ok) break;
        mma_pair_commit_both(&acc_full[ab]);
      }
      // every MMA issued has finished, and both CTAs' epilogues have released the
      // last two accumulators (their arrivals land here), before this CTA winds down
      mma_pair_commit(mma_done);
      mbar_wait_abort(mma_done, 0, err, nullptr);
      for (int j = ti - 2; ok && j < ti; ++j)
        if (j >= 0 && !mbar_wait_cl_abort(&acc_empty[j & 1], (j >> 1) & 1, err, abort)) ok = false;
    }
  } else {
    // epilogue: warp q = warp % 4 reads TMEM lanes 32q .. 32q + 31 (this CTA's rows)
    const int q = warp & 3;
    const uint32_t acc_empty0 = mapa_shared(smem_u32(acc_empty), 0);
    int ti = 0;
    for (int tile = pair; ok && tile < total; tile += npairs, ++ti) {
      const int ks = tile % k_splits, mn = tile / k_splits;
      const int m0 = (mn / n_tiles) * 256, n0 = (mn % n_tiles) * 256;
      const int ab = ti & 1;
      ok = mbar_wait_abort(&acc_full[ab], (ti >> 1) & 1, err, abort);
      if (!gemm_named_and(1, 128, ok)) { ok = false; break; }
      tc_fence_after();
      if constexpr (SWAP) {
        // thread = output column n0 + 128 rank + 32 q + lane; accumulator column = A row
        const int col = n0 + 128 * int(rank) + q * 32 + lane;
#pragma unroll 1
        for (int c = 0; c * 32 < M; ++c) {
          uint32_t r[32];
          tmem_ld32(tmem + (uint32_t(q * 32) << 16) + ab * 256 + c * 32, r);
          tmem_ld_wait();
          const int nr = min(32, M - 32 * c);
          for (int j = 0; j < nr; ++j) epi.swapped(32 * c + j + ks * M, col, __uint_as_float(r[j]));
        }
      } else {
        const int row = m0 + 128 * int(rank) + q * 32 + lane;
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          uint32_t r[32];
          tmem_ld32(tmem + (uint32_t(q * 32) << 16) + ab * 256 + c * 32, r);
          tmem_ld_wait();
          if (row < M) epi(row + ks * M, n0 + c * 32, reinterpret_cast<const float*>(r));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cl(acc_empty0 + uint32_t(ab) * 8u);
    }
  }
  if (!ok) *s_bad = 1;
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  // after a wait gave up, bulk copies issued by this CTA may still be landing:
  // give them a bounded time before the shared memory is released
  if (*s_bad && threadIdx.x == 0) {
    const unsigned long long t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 50000ull) {}
  }
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem, 512);
}

// Launch of one GEMM on CTA pairs: min(tiles, resident pairs) clusters of two.
// A's, B's and B2's maps have 64 x 128 boxes (128-byte swizzle); with SWAP, A's box is
// 64 x NB/2 (NB = M rounded up to 16) and M <= 64.  K a multiple of 64,
// 1 <= k_splits <= K / 64.
template <int STAGES, class Epi, bool SWAP = false>
cudaError_t launch_gemm_pair(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tb2, int M, int N,
                             int K, int n_split, int* err, int* abort, const Epi& epi, cudaStream_t s,
                             int k_splits = 1) {
  using Sm = GemmPairSmem<STAGES, SWAP>;
  auto kern = gemm_pair_bf16_tn_kernel<STAGES, Epi, SWAP>;
  static int max_pairs = 0;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kGemmPairThreads);
  cfg.dynamicSmemBytes = Sm::kBytes;
  cfg.stream = s;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  if (max_pairs == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Sm::kBytes);
    int dev = 0, sms = 0;
    if (e == cudaSuccess) e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cfg.gridDim = dim3(2 * (sms / 2));
    int clusters = 0;
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
    if (e != cudaSuccess) return e;
    if (clusters < 1) return cudaErrorInvalidConfiguration;
    max_pairs = clusters;
  }
  if (k_splits < 1 || k_splits > K / 64 || (SWAP && M > 64)) return cudaErrorInvalidValue;
  const long tiles = long(SWAP ? 1 : (M + 255) / 256) * ((N + 255) / 256) * k_splits;
  const int pairs = int(tiles < max_pairs ? tiles : max_pairs);
  if (pairs <= 0) return cudaSuccess;
  cfg.gridDim = dim3(2 * pairs);
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, ta, tb, tb2, M, N, K, n_split, k_splits, err, abort, epi);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace edge0
