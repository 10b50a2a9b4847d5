// Dense bf16 GEMM on the 5th-generation tensor cores (tcgen05), C = A * B^T.
//
//   A [M][K] bf16 row-major (K-major), B [N][K] bf16 row-major (K-major),
//   fp32 accumulation in TMEM, results handed to an epilogue functor.
// Persistent: one CTA per SM walks the 128 x BN output tiles (tile index i ->
// m = i / n_tiles, n = i % n_tiles, so concurrent CTAs share A rows in L2) with a
// stride of the grid.  Warp roles:
//   warp 0 (one lane): TMA producer of 128x64 A and BNx64 B tiles (128-byte
//     swizzle) through a STAGES-deep mbarrier ring;
//   warp 1 (one lane): tcgen05.mma (M=128, N=BN, K=16, four per 64-wide k-step)
//     into one of two TMEM accumulators of BN columns;
//   warps 2-5: epilogue of the previous accumulator (tcgen05.ld, thread = row, 32
//     columns per load) while the next tile's main loop runs.
// Used for the layer's dense projections: x -> [z | router logits] (B = D and the
// folded router R D split in two bf16 halves) and c -> y (B = U).
#pragma once

#include "tc.cuh"

namespace edge0 {

constexpr int kGemmThreads = 192;

template <int BN, int STAGES>
struct GemmSmem {
  static constexpr int kA = 128 * 64 * 2;   // one A stage (bytes)
  static constexpr int kB = BN * 64 * 2;    // one B stage
  static constexpr int kStage = kA + kB;
  static constexpr int kBytes = STAGES * kStage + 1024 /*barriers, tmem slot*/ + 1024 /*alignment*/;
};

__device__ __forceinline__ bool gemm_named_and(int id, int n, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
      " barrier.cta.red.and.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r) : "r"(uint32_t(pred)), "r"(id), "r"(n) : "memory");
  return r != 0;
}

// Epilogue interface: operator()(int row, int col0, const float* v32) for the 32
// consecutive columns col0 .. col0+31 of one row; rows >= M are not passed.
// Output columns [0, n_split) multiply B's rows, columns from n_split on multiply
// B2's rows (n_split a multiple of the tile width; pass B2 = B for one matrix).
template <int BN, int STAGES, class Epi>
__global__ void __launch_bounds__(kGemmThreads, 1)
gemm_bf16_tn_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmB2, int M, int N, int K, int n_split, int* err, int* abort,
                    Epi epi) {
  using S = GemmSmem<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * S::kStage);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;     // [2] MMA commit
  uint64_t* acc_empty = acc_full + 2;      // [2] one arrival per epilogue warp
  uint64_t* mma_done = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  int* s_bad = reinterpret_cast<int*>(tmem_slot + 2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = K / 64;
  const int n_tiles = (N + BN - 1) / BN;
  const int total = ((M + 127) / 128) * n_tiles;

  // a wait of another launch or CTA that ran out: leave before touching anything
  if (threadIdx.x == 0) {
    *s_bad = (abort && ld_relaxed_s32(abort)) ? 2 : 0;
    for (int s = 0; s < STAGES; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    for (int b = 0; b < 2; ++b) { mbar_init(&acc_full[b], 1); mbar_init(&acc_empty[b], 4); }
    mbar_init(mma_done, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (*s_bad || blockIdx.x >= total) return;
  if (warp == 1) { tmem_alloc(tmem_slot, 2 * BN); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmB);
      prefetch_tmap(&tmB2);
      int it = 0;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        const int m0 = (tile / n_tiles) * 128, n0 = (tile % n_tiles) * BN;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % STAGES;
          if (!mbar_wait_abort(&empty[s], ((it / STAGES) & 1) ^ 1, err, abort)) { ok = false; break; }
          uint8_t* sa = smem + s * S::kStage;
          mbar_arrive_expect_tx(&full[s], S::kStage);
          tma_load_2d(sa, &tmA, kb * 64, m0, &full[s]);
          // columns [0, n_split) come from B's rows, later columns from B2's rows
          if (n0 < n_split) tma_load_2d(sa + S::kA, &tmB, kb * 64, n0, &full[s]);
          else tma_load_2d(sa + S::kA, &tmB2, kb * 64, n0 - n_split, &full[s]);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, BN);
      int it = 0, ti = 0;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x, ++ti) {
        const int ab = ti & 1;
        if (!mbar_wait_abort(&acc_empty[ab], ((ti >> 1) & 1) ^ 1, err, abort)) { ok = false; break; }
        tc_fence_after();
        const uint32_t acc = tmem + ab * BN;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % STAGES;
          if (!mbar_wait_abort(&full[s], (it / STAGES) & 1, err, abort)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + s * S::kStage);
          const uint32_t sb = sa + S::kA;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_bf16(acc, sw128_desc(sa + k * 32), sw128_desc(sb + k * 32), idesc, (kb | k) != 0);
          mma_commit(&empty[s]);
        }
        if (!ok) break;
        mma_commit(&acc_full[ab]);
      }
      // every MMA issued has finished before the accumulators are released
      mma_commit(mma_done);
      mbar_wait_abort(mma_done, 0, err, nullptr);
    }
  } else {
    // epilogue: warp q = warp % 4 reads TMEM lanes 32q .. 32q + 31 (output rows)
    const int q = warp & 3;
    int ti = 0;
    for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x, ++ti) {
      const int m0 = (tile / n_tiles) * 128, n0 = (tile % n_tiles) * BN;
      const int ab = ti & 1;
      ok = mbar_wait_abort(&acc_full[ab], (ti >> 1) & 1, err, abort);
      if (!gemm_named_and(1, 128, ok)) { ok = false; break; }
      tc_fence_after();
      const int row = m0 + q * 32 + lane;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tmem + (uint32_t(q * 32) << 16) + ab * BN + c * 32, r);
        tmem_ld_wait();
        if (row < M) epi(row, n0 + c * 32, reinterpret_cast<const float*>(r));
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[ab]);
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
  if (warp == 1) tmem_dealloc(tmem, 2 * BN);
}

// Launch of one GEMM: a persistent grid of min(tiles, SMs) CTAs; A's map has a
// 64 x 128 box, B's and B2's 64 x BN boxes (128-byte swizzle).  K a multiple of 64.
template <int BN, int STAGES, class Epi>
cudaError_t launch_gemm_tn(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tb2, int M, int N, int K,
                           int n_split, int* err, int* abort, const Epi& epi, cudaStream_t s) {
  using Sm = GemmSmem<BN, STAGES>;
  static bool attr = false;
  static int sms = 0;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(gemm_bf16_tn_kernel<BN, STAGES, Epi>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Sm::kBytes);
    int dev = 0;
    if (e == cudaSuccess) e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  const long tiles = long((M + 127) / 128) * ((N + BN - 1) / BN);
  const int grid = int(tiles < sms ? tiles : sms);
  if (grid <= 0) return cudaSuccess;
  gemm_bf16_tn_kernel<BN, STAGES, Epi><<<grid, kGemmThreads, Sm::kBytes, s>>>(ta, tb, tb2, M, N, K, n_split, err,
                                                                               abort, epi);
  return cudaGetLastError();
}

}  // namespace edge0
