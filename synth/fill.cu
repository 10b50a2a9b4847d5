// Device-side fill of seeded NVFP4 expert bytes (input generation only).
//
// Writes the same bytes as synth.expert_bytes (SplitMix64 counter streams,
// E4M3 round-to-nearest-even of u * 0.008 + 0.002) for a range of experts,
// in the per-expert logical layout: codes [n][3FL/2], scales [n][3FL/16],
// globals [n][3].  Holds none of the layer's arithmetic.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ uint64_t splitmix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ uint64_t stream_key(uint64_t seed, uint64_t layer, uint64_t expert, uint64_t kind) {
  uint64_t k = splitmix64(seed);
  k = splitmix64(k ^ layer);
  k = splitmix64(k ^ expert);
  return splitmix64(k ^ kind);
}

// positive finite double -> E4M3FN byte, round to nearest even, saturating at 448
__device__ __forceinline__ uint8_t e4m3_byte(double v) {
  if (!(v > 0.0)) return 0;
  if (v >= 448.0) return 0x7E;
  if (v < 0.015625) return (uint8_t)rint(__dmul_rn(v, 512.0));
  int ex;
  const double fr = frexp(v, &ex);
  int e = ex - 1;
  double mant = rint(__dmul_rn(__dsub_rn(__dmul_rn(2.0, fr), 1.0), 8.0));
  if (mant == 8.0) { mant = 0.0; e += 1; }
  int code = ((e + 7) << 3) + (int)mant;
  return (uint8_t)(code > 0x7E ? 0x7E : code);
}

__global__ void fill_kernel(uint64_t seed, int layer, int expert0, int n_codes, int n_scales,
                            uint8_t* codes, uint8_t* scales, float* globals) {
  const int e = blockIdx.y;
  const uint64_t expert = (uint64_t)(expert0 + e);
  const uint64_t kc = stream_key(seed, (uint64_t)layer, expert, 1);
  const uint64_t ks = stream_key(seed, (uint64_t)layer, expert, 2);
  uint64_t* cw = reinterpret_cast<uint64_t*>(codes + (size_t)e * n_codes);
  uint8_t* sc = scales + (size_t)e * n_scales;
  const int nw = n_codes / 8;
  const int stride = gridDim.x * blockDim.x;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < nw + n_scales; i += stride) {
    if (i < nw) {
      cw[i] = splitmix64(kc + (uint64_t)i);   // little-endian bytes, as on the host
    } else {
      const int j = i - nw;
      const uint64_t h = splitmix64(ks + (uint64_t)j);
      const double u = (double)(h >> 11) * 1.1102230246251565e-16;   // 2^-53, exact
      const double v = __dadd_rn(__dmul_rn(u, 0.008), 0.002);
      sc[j] = e4m3_byte(v);
    }
  }
  if (blockIdx.x == 0 && threadIdx.x < 3) globals[(size_t)e * 3 + threadIdx.x] = 1.0f;
}

}  // namespace

extern "C" int synth_fill_experts(unsigned long long seed, int layer, int expert0, int n_experts,
                                  int latent, int ffn, void* codes, void* scales, void* globals,
                                  void* stream) {
  if (n_experts <= 0) return 0;
  const int n_codes = 3 * ffn * latent / 2, n_scales = 3 * ffn * latent / 16;
  if (n_codes % 8) return 1;
  fill_kernel<<<dim3(128, n_experts), 256, 0, (cudaStream_t)stream>>>(
      seed, layer, expert0, n_codes, n_scales, (uint8_t*)codes, (uint8_t*)scales, (float*)globals);
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}
