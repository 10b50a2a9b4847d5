// Dense bf16 GEMM on the 5th-generation tensor cores (tcgen05), C = A * B^T.
//
//   A [M][K] bf16 row-major (K-major), B [N][K] bf16 row-major (K-major),
//   fp32 accumulation in TMEM, results handed to an epilogue functor.
// One CTA computes a 128 x BN tile: warp 0 (one lane) streams 128x64 A and BNx64
// B tiles with TMA (128-byte swizzle) through a STAGES-deep mbarrier ring, warp 1
// (one lane) issues tcgen05.mma (M=128, N=BN, K=16, four per 64-wide k-step) into
// a TMEM accumulator, warp 2 owns the TMEM allocation, and after the last k-step
// all four warps read the accumulator with tcgen05.ld (thread = row, 32 columns
// per load) and call the epilogue.
// Used for the layer's dense projections: x -> [z | router logits] (B = D and the
// folded router R D split in two bf16 halves) and c -> y (B = U).
#pragma once

#include "tc.cuh"

namespace edge0 {

constexpr int kGemmThreads = 128;

template <int BN, int STAGES>
struct GemmSmem {
  static constexpr int kA = 128 * 64 * 2;   // one A stage (bytes)
  static constexpr int kB = BN * 64 * 2;    // one B stage
  static constexpr int kStage = kA + kB;
  static constexpr int kBars = 2 * STAGES + 1;
  static constexpr int kBytes = STAGES * kStage + 1024 /*barriers, tmem slot*/ + 1024 /*alignment*/;
};

// Epilogue interface: operator()(int row, int col0, const float* v32) for the 32
// consecutive columns col0 .. col0+31 of one row; rows >= M are not passed.
// Output columns [0, n_split) multiply B's rows, columns from n_split on multiply
// B2's rows (n_split a multiple of the tile width; pass B2 = B for one matrix).
template <int BN, int STAGES, class Epi>
__global__ void __launch_bounds__(kGemmThreads, 1)
gemm_bf16_tn_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmB2, int M, int K, int n_split, int* err, int* abort,
                    Epi epi) {
  using S = GemmSmem<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * S::kStage);
  uint64_t* empty = full + STAGES;
  uint64_t* accf = empty + STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accf + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.y * 128, n0 = blockIdx.x * BN;
  const int nk = K / 64;
  __shared__ int s_bad;

  // a wait of another launch or CTA that ran out: leave before touching anything
  if (threadIdx.x == 0) s_bad = (abort && ld_relaxed_s32(abort)) ? 2 : 0;
  __syncthreads();
  if (s_bad) return;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    mbar_init(accf, 1);
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(n0 < n_split ? &tmB : &tmB2);
  }
  if (warp == 2) { tmem_alloc(tmem_slot, BN); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // TMA producer
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % STAGES;
      const uint32_t ph = (kb / STAGES) & 1;
      if (!mbar_wait_abort(&empty[s], ph ^ 1, err, abort)) { s_bad = 1; break; }
      uint8_t* sa = smem + s * S::kStage;
      mbar_arrive_expect_tx(&full[s], S::kStage);
      tma_load_2d(sa, &tmA, kb * 64, m0, &full[s]);
      // columns [0, n_split) come from B's rows, later columns from B2's rows
      if (n0 < n_split) tma_load_2d(sa + S::kA, &tmB, kb * 64, n0, &full[s]);
      else tma_load_2d(sa + S::kA, &tmB2, kb * 64, n0 - n_split, &full[s]);
    }
  } else if (warp == 1 && lane == 0) {
    // MMA issuer
    constexpr uint32_t idesc = idesc_bf16_f32(128, BN);
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % STAGES;
      const uint32_t ph = (kb / STAGES) & 1;
      if (!mbar_wait_abort(&full[s], ph, err, abort)) { s_bad = 1; break; }
      tc_fence_after();
      const uint32_t sa = smem_u32(smem + s * S::kStage);
      const uint32_t sb = sa + S::kA;
#pragma unroll
      for (int k = 0; k < 4; ++k)
        mma_bf16(tmem, sw128_desc(sa + k * 32), sw128_desc(sb + k * 32), idesc, (kb | k) != 0);
      mma_commit(&empty[s]);
    }
    mma_commit(accf);
  }
  // epilogue: every warp reads its 32 TMEM lanes.  The issuer always commits
  // accf, so this wait ends once every MMA issued has finished (time limit only).
  __syncwarp();
  const bool acc_ok = mbar_wait_abort(accf, 0, err, nullptr);
  tc_fence_after();
  const int row = m0 + warp * 32 + lane;
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    uint32_t r[32];
    tmem_ld32(tmem + (uint32_t(warp * 32) << 16) + c * 32, r);
    tmem_ld_wait();
    if (row < M && acc_ok) epi(row, n0 + c * 32, reinterpret_cast<const float*>(r));
  }
  tc_fence_before();
  __syncthreads();
  // after a wait gave up, bulk copies issued by this CTA may still be landing:
  // give them a bounded time before the shared memory is released
  if (s_bad && threadIdx.x == 0) {
    const unsigned long long t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 50000ull) {}
  }
  __syncthreads();
  if (warp == 2) tmem_dealloc(tmem, BN);
}

// Launch of one GEMM: grid (ceil(N / BN), ceil(M / 128)); A's map has a 64 x 128
// box, B's and B2's 64 x BN boxes (128-byte swizzle).  K a multiple of 64.
template <int BN, int STAGES, class Epi>
cudaError_t launch_gemm_tn(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tb2, int M, int N, int K,
                           int n_split, int* err, int* abort, const Epi& epi, cudaStream_t s) {
  using Sm = GemmSmem<BN, STAGES>;
  static bool attr = false;
  if (!attr) {
    const cudaError_t e = cudaFuncSetAttribute(gemm_bf16_tn_kernel<BN, STAGES, Epi>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, Sm::kBytes);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  const dim3 grid((N + BN - 1) / BN, (M + 127) / 128);
  gemm_bf16_tn_kernel<BN, STAGES, Epi><<<grid, kGemmThreads, Sm::kBytes, s>>>(ta, tb, tb2, M, K, n_split, err, abort,
                                                                               epi);
  return cudaGetLastError();
}

}  // namespace edge0
