// Plain dense bf16 GEMM entry point (C fp32 = A B^T) on the CTA-pair tcgen05 kernel of gemm_pair.cuh.
#include "../../include/edge0_moe.h"
#include "gemm_pair.cuh"
#include "tmap.cuh"

namespace edge0 {
namespace {

struct EpiStoreF32 {
  float* C;
  int ldc, N;
  __device__ __forceinline__ void operator()(int row, int col0, const float* v) const {
    float* dst = C + size_t(row) * ldc + col0;
    if (col0 + 32 <= N && (ldc & 3) == 0) {
#pragma unroll
      for (int i = 0; i < 32; i += 4)
        *reinterpret_cast<float4*>(dst + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
    } else {
      for (int i = 0; i < 32; ++i)
        if (col0 + i < N) dst[i] = v[i];
    }
  }
};

constexpr int kStages = 6;

}  // namespace

}  // namespace edge0

using namespace edge0;

extern "C" edge0_status edge0_gemm_bf16_tn(const void* A, const void* B, float* C, int M, int N, int K,
                                           int* err, edge0_stream_t stream) {
  if (M < 0 || N < 0 || K < 0) return EDGE0_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return EDGE0_OK;
  if (!A || !B || !C || K == 0 || K % 64 || (reinterpret_cast<uintptr_t>(A) & 15) ||
      (reinterpret_cast<uintptr_t>(B) & 15) || (reinterpret_cast<uintptr_t>(C) & 15))
    return EDGE0_ERR_INVALID_ARG;
  CUtensorMap ta, tb;
  if (!make_tmap_2d(&ta, A, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, M, K, uint64_t(K) * 2, 64, 128,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d(&tb, B, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, N, K, uint64_t(K) * 2, 64, 128,
                    CU_TENSOR_MAP_SWIZZLE_128B))
    return EDGE0_ERR_CUDA;
  EpiStoreF32 epi{C, N, N};
  return launch_gemm_pair<kStages>(ta, tb, tb, M, N, K, 1 << 30, err, nullptr, epi, (cudaStream_t)stream) ==
                 cudaSuccess
             ? EDGE0_OK
             : EDGE0_ERR_CUDA;
}
