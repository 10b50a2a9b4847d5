// C ABI of the latent-MoE layer library (declared in include/edge0_moe.h).
#include "../../include/edge0_moe.h"

#include <cuda_runtime.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "decode.cuh"
#include "prefill.cuh"

namespace edge0 {
int decode_bucket(int T);
cudaError_t decode_prepare(int smem);
cudaError_t decode_occupancy(int smem, int* blocks);
cudaError_t decode_launch(const DecodeArgs& a, int grid, int smem, cudaStream_t s);
}  // namespace edge0

using namespace edge0;

namespace {

constexpr int kStackMax = 64;
constexpr int kMaxGroups = 16;     // latent groups (D/U pairs) per layer

struct Handle {
  edge0_moe_desc d;
  int device = 0;
  int num_sms = 0;
  int smem_total = 0;         // dynamic shared memory of the decode kernel
  int dec_max_t = 0;          // decode workspace tokens
  char* ws = nullptr;         // one allocation for the whole workspace
  size_t ws_bytes = 0;
  float* z = nullptr; float* logits = nullptr; float* h = nullptr;
  float* c = nullptr;
  __nv_bfloat16* ybuf = nullptr; __nv_bfloat16* xbuf = nullptr;
  int* idx = nullptr; float* w = nullptr; int* counts = nullptr; int* offsets = nullptr;
  int* perm = nullptr; int* pos = nullptr;
  GridBarrier* bar = nullptr; int* err = nullptr;
  float* rd = nullptr;        // R D, fp32 [n_experts][hidden] (grouped: row e = R_e D_(g(e)))
  int groups = 1;             // latent groups G (d.n_groups normalised to >= 1)
  int* labels = nullptr;      // G > 1: device copy of the experts' group labels (d.expert_group points here)
  float dnorm = 0.f;          // max_r sum_h |D[r][h]|
  __half* zh = nullptr;       // f16 copy of z for the decode experts
  LayerW* d_layer = nullptr;  // this layer (1 entry)
  LayerW* d_stack = nullptr;  // kStackMax entries for stack calls
  PrefillWorkspace pf;        // prefill path buffers (T > 16)
  std::vector<LayerW> stack_tab;  // the layer table last uploaded to d_stack
  int last_T = 0;
  int last_path = 0;          // 0 none, 1 decode, 2 prefill
  // residency tiering of the routed records (decode forwards; off by default)
  bool tiered = false;
  const uint8_t* host_records = nullptr;  // the caller's host records (pinned)
  const uint8_t* host_dev = nullptr;      // their device alias (mapped host memory)
  int n_slots = 0;
  uint8_t* slots = nullptr;               // device [n_slots][stride]
  uint8_t* staging = nullptr;             // device [kDecodeMaxT * top_k][stride]
  char* tier_ws = nullptr;                // device: table, resident flags, use counts, stats
  const uint8_t** d_table = nullptr;      // [E] record of each expert
  uint8_t* d_resident = nullptr;          // [E]
  unsigned int* d_use = nullptr;          // [E]
  unsigned long long* d_stats = nullptr;  // [3]
  std::vector<int> slot_expert;           // [n_slots] expert in each slot, -1 empty
  // decode phase profiling (off by default)
  bool dec_profile = false;
  unsigned long long* stamps = nullptr;   // [kStackMax][kStampSlots], own allocation
  int stamped_layers = 0;                 // layers of the last profiled decode launch
};

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool shapes_ok(int latent, int ffn) {
  return latent > 0 && ffn > 0 && latent % 256 == 0 && ffn % 128 == 0;
}

// Source byte offset, in the per-matrix arrays, of the 16-byte chunk at byte `o`
// of a record body (see the record layout in edge0_moe.h).  Sets *from_scales.
__host__ __device__ inline size_t record_src(size_t o, size_t L, size_t F, bool* from_scales) {
  const size_t gu_row = 9 * L / 8, d_pair = 9 * F / 8;
  if (o < F * gu_row) {
    const size_t f = o / gu_row, w = o % gu_row;
    if (w < L / 2) { *from_scales = false; return f * (L / 2) + w; }
    if (w < L) { *from_scales = false; return F * (L / 2) + f * (L / 2) + (w - L / 2); }
    if (w < L + L / 16) { *from_scales = true; return f * (L / 16) + (w - L); }
    *from_scales = true;
    return F * (L / 16) + f * (L / 16) + (w - L - L / 16);
  }
  const size_t od = o - F * gu_row, pr = od / d_pair, w = od % d_pair;
  if (w < F) { *from_scales = false; return F * L + pr * F + w; }
  *from_scales = true;
  return 2 * F * (L / 16) + pr * (F / 8) + (w - F);
}

// Shared-memory plan of the decode kernel for a bucket of TB tokens: the tables, the
// shared expert's gate/up rows, the phase-local arrays, then the ring area (to the end).
void decode_plan(const Handle* hd, int TB, DecodeArgs& a) {
  const int H = hd->d.hidden, L = hd->d.latent, F = hd->d.ffn, K = hd->d.top_k, G = hd->num_sms;
  const int NT = TB > 8 ? 2 : 1;
  size_t off = decode_tables_bytes();
  const int shared_rows = (F + G - 1) / G;
  a.off_sh = (int)off;
  a.sh_bytes = (int)align_up((size_t)shared_rows * pitch_gu_row(L), 128);
  off += a.sh_bytes;
  // x [T][H + pad] (P0); zh [T][L + pad] and the partial sums (P1); the per-slot down
  // outputs of both halves of F (P2); c [T][L + pad] (P3)
  const int nr_max = 2 * ((L / 2 + G - 1) / G);
  const size_t xs = size_t(TB) * (H + kPadElems) * 2;
  const size_t zs = align_up(size_t(TB) * (L + kPadElems) * 2, 128);
  const size_t p1 = zs + size_t(kPartCap) * 32 * NT * 16;
  const size_t p2 = 2 * size_t(TB) * (K + 1) * nr_max * 4;        // two halves of F
  size_t ar = xs > p1 ? xs : p1;
  if (p2 > ar) ar = p2;
  a.off_a = (int)off;
  a.a_bytes = (int)align_up(ar, 128);
  off = align_up(off + a.a_bytes, 1024);
  a.off_ring = (int)off;
  a.ring_bytes = hd->smem_total > (int)off ? (int)((hd->smem_total - off) & ~size_t(127)) : 0;
  const int unit1 = (int)align_up(size_t(8) * pitch_gu_row(L), 128);
  int S = a.ring_bytes / unit1;
  if (S > kRingMax) S = kRingMax;
  a.ring_slots = S;
  a.slot_bytes = S > 0 ? (a.ring_bytes / S) & ~127 : 0;
}

// Every decode bucket's plan holds what each phase stages: at least two ring slots, the
// P0 rows of a CTA, the logits and top-k candidates, a P2 unit of one expert's down
// rows and one h row, and the U rows of P3 in at most one piece per slot.
bool decode_fits(const Handle* hd) {
  const int H = hd->d.hidden, L = hd->d.latent, E = hd->d.n_experts, F = hd->d.ffn, G = hd->num_sms;
  const int ne = (E + G - 1) / G, nr = 2 * ((L / 2 + G - 1) / G), nsr = (F + G - 1) / G, nur = (H + G - 1) / G;
  if ((ne + 7) / 8 + (nr + 15) / 16 > kP0Tiles || ne + nr > 32 || nsr > 32 || (nur + 15) / 16 > kDecWarps) return false;
  if (F / 8 > 32 * kConvPieces) return false;                           // h rows held in registers
  for (int TB = 1; TB <= kDecodeMaxT; TB *= 2) {
    DecodeArgs a;
    decode_plan(hd, TB, a);
    const int NT = TB > 8 ? 2 : 1;
    const size_t ring = (size_t)a.ring_bytes;
    if (a.ring_slots < 2 || (nsr + 7) / 8 > a.ring_slots) return false;
    if (size_t(ne) * pitch_f32_row(H) + size_t(nr) * pitch_bf16_row(H) > ring) return false;
    if (size_t(kDecWarps) * 32 * NT * 16 > ring) return false;
    if (size_t(TB) * E * 4 + size_t(kDecWarps) * kTopkCand * 8 > ring) return false;
    if (size_t(nr / 2) * (9 * F / 8) + size_t(F) * 2 > (size_t)a.slot_bytes) return false;
    const int rpp = std::max(1, a.slot_bytes / (L * 2));
    if ((nur + rpp - 1) / rpp > a.ring_slots) return false;           // the U pieces of P3
  }
  return true;
}

edge0_status cuda_status(cudaError_t e) { return e == cudaSuccess ? EDGE0_OK : EDGE0_ERR_CUDA; }

LayerW layer_of(const Handle* hd) {
  LayerW l;
  l.D = static_cast<const __nv_bfloat16*>(hd->d.D);
  l.U = static_cast<const __nv_bfloat16*>(hd->d.U);
  l.RD = hd->rd;
  l.bias = hd->d.router_bias;
  l.experts = static_cast<const uint8_t*>(hd->d.experts);
  l.shared = static_cast<const uint8_t*>(hd->d.shared_expert);
  l.stride = hd->d.expert_stride;
  l.dnorm = hd->dnorm;
  l.rec_table = hd->tiered ? hd->d_table : nullptr;
  l.resident = hd->tiered ? hd->d_resident : nullptr;
  l.staging = hd->tiered ? hd->staging : nullptr;
  l.use = hd->tiered ? hd->d_use : nullptr;
  l.tier_stats = hd->tiered ? hd->d_stats : nullptr;
  return l;
}

void fill_decode_args(const Handle* hd, DecodeArgs& a, const void* x, void* y, int T) {
  memset(&a, 0, sizeof(a));
  a.l0 = layer_of(hd);
  a.layers = hd->d_layer;
  a.n_layers = 1;
  a.eps = 1e-6f;
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.y = static_cast<__nv_bfloat16*>(y);
  a.T = T;
  a.H = hd->d.hidden; a.L = hd->d.latent; a.E = hd->d.n_experts; a.K = hd->d.top_k; a.F = hd->d.ffn;
  a.z = hd->z; a.zh = hd->zh; a.logits = hd->logits; a.h = reinterpret_cast<__nv_bfloat16*>(hd->h); a.c = hd->c;
  a.ybuf = hd->ybuf; a.xbuf = hd->xbuf;
  a.idx = hd->idx; a.w = hd->w; a.counts = hd->counts; a.offsets = hd->offsets;
  a.perm = hd->perm; a.pos = hd->pos;
  a.bar = hd->bar; a.err = hd->err;
  decode_plan(hd, decode_bucket(T), a);
}

// ------------------------------------------------------------------ small kernels
__global__ void pack_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales,
                            const float* __restrict__ globals, int L, int F, int n_codes, int n_scales,
                            uint8_t* __restrict__ records, size_t stride) {
  const int e = blockIdx.y;
  uint8_t* rec = records + size_t(e) * stride;
  const uint8_t* ce = codes + size_t(e) * n_codes;
  const uint8_t* se = scales + size_t(e) * n_scales;
  const int nchunk = (n_codes + n_scales) / 16;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < nchunk; i += gridDim.x * blockDim.x) {
    bool sc = false;
    const size_t src = record_src(size_t(i) * 16, L, F, &sc);
    reinterpret_cast<uint4*>(rec)[i] = *reinterpret_cast<const uint4*>((sc ? se : ce) + src);
  }
  if (blockIdx.x == 0 && threadIdx.x < 3) {
    reinterpret_cast<float*>(rec + n_codes + n_scales)[threadIdx.x] = globals[size_t(e) * 3 + threadIdx.x];
  }
}

// RD[e][h] = sum_l R[e][l] * D[l][h] in fp32 (the router folded with the
// down-projection, so decode computes the logits from x directly).  32x32 output
// tiles, K staged through shared memory in fixed order.  With grouped projections
// (labels non-null) D is D_g and only the rows of the experts labelled g are written.
__global__ void fold_router_kernel(const __nv_bfloat16* __restrict__ R, const __nv_bfloat16* __restrict__ D,
                                   float* __restrict__ RD, int E, int L, int H, const int* __restrict__ labels,
                                   int g) {
  __shared__ float rs[32][33];
  __shared__ float ds[32][33];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;   // 32 x 8 threads
  const int e0 = blockIdx.y * 32, h0 = blockIdx.x * 32;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int l0 = 0; l0 < L; l0 += 32) {
    for (int i = ty; i < 32; i += 8) {
      rs[i][tx] = (e0 + i < E) ? __bfloat162float(R[size_t(e0 + i) * L + l0 + tx]) : 0.f;
      ds[i][tx] = (h0 + tx < H) ? __bfloat162float(D[size_t(l0 + i) * H + h0 + tx]) : 0.f;
    }
    __syncthreads();
    for (int k = 0; k < 32; ++k) {
      const float dv = ds[k][tx];
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[j] = fmaf(rs[ty + 8 * j][k], dv, acc[j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int e = e0 + ty + 8 * j;
    if (e < E && h0 + tx < H && (!labels || labels[e] == g)) RD[size_t(e) * H + h0 + tx] = acc[j];
  }
}

// *out = max_r sum_h |D[r][h]|: one warp per row (lane-strided sums, then an xor
// tree: a fixed order per row); the maximum is taken with an integer atomicMax on
// the bits of the non-negative sums, which is exact in any order.  *out must be 0.
__global__ void row_l1_max_kernel(const __nv_bfloat16* __restrict__ D, int rows, int cols, float* out) {
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  float m = 0.f;
  for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows; r += warps) {
    float s = 0.f;
    for (int c = lane; c < cols; c += 32) s += fabsf(__bfloat162float(D[size_t(r) * cols + c]));
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    m = fmaxf(m, s);
  }
  if (lane == 0 && m > 0.f) atomicMax(reinterpret_cast<int*>(out), __float_as_int(m));
}

// E4M3FN round-to-nearest-even of a non-negative double, saturating at 448.
__device__ uint32_t e4m3_rne(double x) {
  if (!(x > 0.0)) return 0u;
  if (x >= 448.0) return 0x7Eu;
  if (x < 0.015625) {                       // below 2^-6: subnormal grid m * 2^-9
    return (uint32_t)rint(x * 512.0);       // m = 8 lands on 0x08 = 2^-6
  }
  int ex;
  const double fr = frexp(x, &ex);          // x = fr * 2^ex, fr in [0.5, 1)
  int e = ex - 1;
  double mant = rint((2.0 * fr - 1.0) * 8.0);
  if (mant == 8.0) { mant = 0.0; e += 1; }
  uint32_t code = (uint32_t)((e + 7) << 3) + (uint32_t)mant;
  return code > 0x7Eu ? 0x7Eu : code;
}

__device__ double e4m3_value_d(uint32_t b) {
  const int e = (b >> 3) & 15, m = b & 7;
  return e == 0 ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
}

// Nearest E2M1 magnitude code (0..7) of |r|, ties to the even code.
__device__ uint32_t e2m1_mag_rne(double a) {
  if (a <= 0.25) return 0;
  if (a < 0.75) return 1;
  if (a <= 1.25) return 2;
  if (a < 1.75) return 3;
  if (a <= 2.5) return 4;
  if (a < 3.5) return 5;
  if (a <= 5.0) return 6;
  return 7;
}

// One thread per 16-element block.
__global__ void quantize_kernel(const float* __restrict__ w, int rows, int K, float g,
                                uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
  const long nblk = long(rows) * (K / 16);
  for (long bi = blockIdx.x * long(blockDim.x) + threadIdx.x; bi < nblk; bi += long(gridDim.x) * blockDim.x) {
    const long r = bi / (K / 16), b = bi % (K / 16);
    const float* src = w + r * K + b * 16;
    double amax = 0.0;
    for (int i = 0; i < 16; ++i) amax = fmax(amax, fabs((double)src[i]));
    const double gd = (double)g;
    const uint32_t sb = e4m3_rne(amax / (6.0 * gd));
    const double denom = e4m3_value_d(sb) * gd;
    uint8_t* cdst = codes + r * (K / 2) + b * 8;
    for (int i = 0; i < 16; i += 2) {
      uint32_t cc[2];
      for (int j = 0; j < 2; ++j) {
        const double rv = denom > 0.0 ? (double)src[i + j] / denom : 0.0;
        const uint32_t m = e2m1_mag_rne(fabs(rv));
        cc[j] = m | ((rv < 0.0 && m > 0) ? 8u : 0u);
      }
      cdst[i / 2] = (uint8_t)(cc[0] | (cc[1] << 4));
    }
    scales[r * (K / 16) + b] = (uint8_t)sb;
  }
}

// out[t] = bf16(v / sqrt(mean(v^2) + eps)), v = x[t] + y[t]; one block per token.
// Launched with the decode kernel's block size and summation order, so a stack run
// as separate layer calls reproduces the fused stack bit for bit.
// out = bf16((x + y) / sqrt(mean((x + y)^2) + eps)): one warp per token row.
__global__ void __launch_bounds__(256) residual_rmsnorm_kernel(const __nv_bfloat16* x, const __nv_bfloat16* y,
                                                               __nv_bfloat16* out, int T, int hidden, float eps) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  const size_t base = size_t(t) * hidden;
  const float inv = 1.0f / sqrtf(row_sumsq_warp(x + base, y + base, hidden, lane) / float(hidden) + eps);
  const uint4* xv = reinterpret_cast<const uint4*>(x + base);
  const uint4* yv = reinterpret_cast<const uint4*>(y + base);
  uint4* ov = reinterpret_cast<uint4*>(out + base);
  for (int g = lane; g < hidden / 8; g += 32) {
    const uint4 a = xv[g], b = yv[g];
    const uint32_t aa[4] = {a.x, a.y, a.z, a.w}, bb[4] = {b.x, b.y, b.z, b.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float v0 = __uint_as_float(aa[i] << 16) + __uint_as_float(bb[i] << 16);
      const float v1 = __uint_as_float(aa[i] & 0xFFFF0000u) + __uint_as_float(bb[i] & 0xFFFF0000u);
      const __nv_bfloat162 r = __floats2bfloat162_rn(v0 * inv, v1 * inv);
      o[i] = *reinterpret_cast<const uint32_t*>(&r);
    }
    ov[g] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

edge0_status launch_status() { return cuda_status(cudaGetLastError()); }

// A profiled decode launch carries the handle's zeroed stamp buffer.
cudaError_t attach_stamps(Handle* hd, DecodeArgs& a, int n_layers, cudaStream_t s) {
  if (!hd->dec_profile) return cudaSuccess;
  a.stamps = hd->stamps;
  hd->stamped_layers = n_layers;
  return cudaMemsetAsync(hd->stamps, 0, sizeof(unsigned long long) * kStampSlots * n_layers, s);
}

// One mbarrier that nothing arrives at, waited on with the library's bounded wait.
__global__ void wait_probe_kernel(int* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait_abort(&bar, 0, err, nullptr);
}

}  // namespace

extern "C" {

size_t edge0_expert_record_bytes(int latent, int ffn) {
  if (!shapes_ok(latent, ffn)) return 0;
  return size_t(3) * latent * ffn / 2 + size_t(3) * latent * ffn / 16 + 12;
}

size_t edge0_expert_record_stride(int latent, int ffn) {
  const size_t b = edge0_expert_record_bytes(latent, ffn);
  return b ? align_up(b, 256) : 0;
}

edge0_status edge0_pack_expert_host(const uint8_t* codes, const uint8_t* scales, const float* globals,
                                    int latent, int ffn, void* record_out) {
  if (!codes || !scales || !globals || !record_out || !shapes_ok(latent, ffn)) return EDGE0_ERR_INVALID_ARG;
  const size_t nc = size_t(3) * latent * ffn / 2, ns = size_t(3) * latent * ffn / 16;
  uint8_t* r = static_cast<uint8_t*>(record_out);
  for (size_t o = 0; o < nc + ns; o += 16) {
    bool sc = false;
    const size_t src = record_src(o, size_t(latent), size_t(ffn), &sc);
    memcpy(r + o, (sc ? scales : codes) + src, 16);
  }
  memcpy(r + nc + ns, globals, 12);
  return EDGE0_OK;
}

edge0_status edge0_pack_experts(const uint8_t* codes, const uint8_t* scales, const float* globals,
                                int n_experts, int latent, int ffn, void* records, size_t stride,
                                edge0_stream_t stream) {
  if (!codes || !scales || !globals || !records || n_experts < 0 || !shapes_ok(latent, ffn))
    return EDGE0_ERR_INVALID_ARG;
  if (stride < edge0_expert_record_bytes(latent, ffn) || stride % 16 || !aligned(records, 256) ||
      !aligned(codes, 16) || !aligned(scales, 16) || !aligned(globals, 4))
    return EDGE0_ERR_INVALID_ARG;
  if (n_experts == 0) return EDGE0_OK;
  const int nc = 3 * latent * ffn / 2, ns = 3 * latent * ffn / 16;
  if (n_experts > 65535) return EDGE0_ERR_UNSUPPORTED;
  pack_kernel<<<dim3(64, n_experts), 256, 0, (cudaStream_t)stream>>>(
      codes, scales, globals, latent, ffn, nc, ns, static_cast<uint8_t*>(records), stride);
  return launch_status();
}

edge0_status edge0_quantize_nvfp4(const float* w, int rows, int K, float g, uint8_t* codes,
                                  uint8_t* scales, edge0_stream_t stream) {
  if (!w || !codes || !scales || rows < 0 || K <= 0 || K % 16 || !(g > 0.f) || !isfinite(g))
    return EDGE0_ERR_INVALID_ARG;
  if (rows == 0) return EDGE0_OK;
  const long nblk = long(rows) * (K / 16);
  const int blocks = (int)((nblk + 255) / 256 < 4096 ? (nblk + 255) / 256 : 4096);
  quantize_kernel<<<blocks, 256, 0, (cudaStream_t)stream>>>(w, rows, K, g, codes, scales);
  return launch_status();
}

edge0_status edge0_moe_create(const edge0_moe_desc* desc, void** handle_out) {
  if (!handle_out) return EDGE0_ERR_INVALID_ARG;
  *handle_out = nullptr;
  if (!desc) return EDGE0_ERR_INVALID_ARG;
  const edge0_moe_desc& d = *desc;
  if (d.hidden <= 0 || d.hidden % 64 || !shapes_ok(d.latent, d.ffn) || d.top_k < 1 ||
      d.top_k > kMaxTopK || d.n_experts < d.top_k || d.n_experts > 1024 || d.n_experts % 32 ||
      d.max_tokens < 0)
    return EDGE0_ERR_INVALID_ARG;
  if (!d.D || !d.U || !d.router || !d.experts || !d.shared_expert) return EDGE0_ERR_INVALID_ARG;
  if (!aligned(d.D, 16) || !aligned(d.U, 16) || !aligned(d.router, 16) ||
      !aligned(d.experts, 256) || !aligned(d.shared_expert, 256) ||
      (d.router_bias && !aligned(d.router_bias, 4)))
    return EDGE0_ERR_INVALID_ARG;
  if (d.expert_stride < edge0_expert_record_bytes(d.latent, d.ffn) || d.expert_stride % 256)
    return EDGE0_ERR_INVALID_ARG;
  // grouped latent projections: G D/U pairs, a group label per routed expert
  const int G = d.n_groups > 1 ? d.n_groups : 1;
  std::vector<int> labels;
  if (d.n_groups < 0 || d.n_groups > kMaxGroups) return EDGE0_ERR_INVALID_ARG;
  if (G > 1) {
    if (size_t(G) * d.latent > 16384 || d.latent > 2048 || !d.expert_group || !aligned(d.expert_group, 4) ||
        d.shared_group < 0 || d.shared_group >= G)
      return EDGE0_ERR_INVALID_ARG;
    labels.resize(d.n_experts);
    if (cudaMemcpy(labels.data(), d.expert_group, sizeof(int) * d.n_experts, cudaMemcpyDeviceToHost) !=
        cudaSuccess) {
      cudaGetLastError();
      return EDGE0_ERR_INVALID_ARG;
    }
    for (int v : labels)
      if (v < 0 || v >= G) return EDGE0_ERR_INVALID_ARG;
  }

  Handle* hd = new Handle();
  hd->d = d;
  hd->d.n_groups = G;
  hd->d.shared_group = G > 1 ? d.shared_group : 0;
  hd->d.expert_group = nullptr;
  hd->groups = G;
  cudaError_t ce = cudaGetDevice(&hd->device);
  cudaDeviceProp prop;
  if (ce == cudaSuccess) ce = cudaGetDeviceProperties(&prop, hd->device);
  if (ce != cudaSuccess) { delete hd; return EDGE0_ERR_CUDA; }
  if (prop.major < 10 || !prop.cooperativeLaunch) { delete hd; return EDGE0_ERR_UNSUPPORTED; }
  hd->num_sms = prop.multiProcessorCount;
  hd->smem_total = (int)prop.sharedMemPerBlockOptin - 1024;
  if (G == 1) {                     // the decode kernel serves one latent group
    if (!decode_fits(hd)) { delete hd; return EDGE0_ERR_UNSUPPORTED; }
    if ((ce = decode_prepare(hd->smem_total)) != cudaSuccess) { delete hd; return EDGE0_ERR_CUDA; }
    int occ = 0;
    if ((ce = decode_occupancy(hd->smem_total, &occ)) != cudaSuccess || occ < 1) {
      delete hd;
      return ce != cudaSuccess ? EDGE0_ERR_CUDA : EDGE0_ERR_UNSUPPORTED;
    }
  }

  // workspace
  const int H = d.hidden, L = d.latent, E = d.n_experts, K = d.top_k, F = d.ffn;
  const int TD = kDecodeMaxT;
  hd->dec_max_t = TD;
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes, 256); return o; };
  const size_t o_z = take(size_t(TD) * L * 4), o_lg = take(size_t(TD) * E * 4);
  const size_t o_zh = take(size_t(TD) * L * 2), o_dn = take(sizeof(float));
  const size_t o_h = take(size_t(TD * K + TD) * F * 4);
  const size_t o_c = take(size_t(TD) * L * 4);
  const size_t o_y = take(size_t(2) * TD * H * 2), o_x = take(size_t(2) * TD * H * 2);
  const int TKmax = (d.max_tokens > TD ? d.max_tokens : TD) * K;
  const size_t o_idx = take(size_t(TKmax) * 4), o_w = take(size_t(TKmax) * 4);
  const size_t o_cnt = take(size_t(E) * 4), o_off = take(size_t(E + 1) * 4);
  const size_t o_perm = take(size_t(TKmax) * 4), o_pos = take(size_t(TKmax) * 4);
  const size_t o_bar = take(sizeof(GridBarrier)), o_err = take(sizeof(int));
  const size_t o_lw = take(sizeof(LayerW)), o_st = take(sizeof(LayerW) * kStackMax);
  const size_t o_rd = take(size_t(E) * H * 4);
  const size_t o_lab = take(size_t(E) * 4);
  // grouped layers run the prefill kernels at every T (at least the decode sizes)
  const int pf_tokens = G > 1 ? std::max(d.max_tokens, TD) : d.max_tokens;
  const size_t pf_bytes = prefill_workspace_bytes(hd->d, pf_tokens);
  if (G > 1 && pf_bytes == 0) { delete hd; return EDGE0_ERR_UNSUPPORTED; }
  const size_t o_pf = take(pf_bytes);
  hd->ws_bytes = off;
  if (cudaMalloc(&hd->ws, hd->ws_bytes) != cudaSuccess) {
    cudaGetLastError();
    delete hd;
    return EDGE0_ERR_OOM;
  }
  char* b = hd->ws;
  hd->z = (float*)(b + o_z); hd->logits = (float*)(b + o_lg); hd->h = (float*)(b + o_h);
  hd->zh = (__half*)(b + o_zh);
  float* d_dnorm = (float*)(b + o_dn);
  hd->c = (float*)(b + o_c);
  hd->ybuf = (__nv_bfloat16*)(b + o_y); hd->xbuf = (__nv_bfloat16*)(b + o_x);
  hd->idx = (int*)(b + o_idx); hd->w = (float*)(b + o_w); hd->counts = (int*)(b + o_cnt);
  hd->offsets = (int*)(b + o_off); hd->perm = (int*)(b + o_perm); hd->pos = (int*)(b + o_pos);
  hd->bar = (GridBarrier*)(b + o_bar); hd->err = (int*)(b + o_err);
  hd->d_layer = (LayerW*)(b + o_lw); hd->d_stack = (LayerW*)(b + o_st);
  hd->rd = (float*)(b + o_rd);
  if (G > 1) {
    hd->labels = (int*)(b + o_lab);
    hd->d.expert_group = hd->labels;
  }
  prefill_workspace_carve(hd->d, pf_tokens, b + o_pf, &hd->pf);
  hd->pf.idx = hd->idx; hd->pf.w = hd->w; hd->pf.counts = hd->counts; hd->pf.offsets = hd->offsets;
  hd->pf.perm = hd->perm; hd->pf.pos = hd->pos;
  hd->pf.err = hd->err;
  hd->pf.rd = hd->rd;
  ce = cudaMemset(hd->ws, 0, o_lw);
  if (ce == cudaSuccess && G > 1)
    ce = cudaMemcpy(hd->labels, labels.data(), sizeof(int) * E, cudaMemcpyHostToDevice);
  if (ce == cudaSuccess) {
    row_l1_max_kernel<<<(G * L + 7) / 8, 256>>>(static_cast<const __nv_bfloat16*>(d.D), G * L, H, d_dnorm);
    ce = cudaGetLastError();
  }
  if (ce == cudaSuccess) ce = cudaMemcpy(&hd->dnorm, d_dnorm, sizeof(float), cudaMemcpyDeviceToHost);
  hd->pf.dnorm = hd->dnorm;
  const LayerW lw = layer_of(hd);
  for (int g = 0; g < G && ce == cudaSuccess; ++g) {   // grouped: row e folds with D_(g(e))
    fold_router_kernel<<<dim3((H + 31) / 32, (E + 31) / 32), 256>>>(
        static_cast<const __nv_bfloat16*>(d.router), static_cast<const __nv_bfloat16*>(d.D) + size_t(g) * L * H,
        hd->rd, E, L, H, hd->labels, g);
    ce = cudaGetLastError();
  }
  if (ce == cudaSuccess) ce = cudaMemcpy(hd->d_layer, &lw, sizeof(lw), cudaMemcpyHostToDevice);
  if (ce == cudaSuccess) ce = prefill_init(hd->d, &hd->pf, hd->num_sms);
  // the fold and the initialisation above ran on the legacy stream: finish them
  // before the handle is used from any stream
  if (ce == cudaSuccess) ce = cudaDeviceSynchronize();
  if (ce != cudaSuccess) {
    cudaFree(hd->ws);
    delete hd;
    return EDGE0_ERR_CUDA;
  }
  *handle_out = hd;
  return EDGE0_OK;
}

edge0_status edge0_moe_forward(void* handle, const void* x, void* y, int T, edge0_stream_t stream) {
  Handle* hd = static_cast<Handle*>(handle);
  if (!hd || T < 0) return EDGE0_ERR_INVALID_ARG;
  if (T == 0) return EDGE0_OK;
  if (!x || !y || !aligned(x, 16) || !aligned(y, 16) || T > (hd->d.max_tokens > kDecodeMaxT ? hd->d.max_tokens : kDecodeMaxT))
    return EDGE0_ERR_INVALID_ARG;
  if (T > hd->d.max_tokens && T > kDecodeMaxT) return EDGE0_ERR_INVALID_ARG;
  const size_t xy = size_t(T) * hd->d.hidden * 2;
  const char* xc = static_cast<const char*>(x);
  const char* yc = static_cast<const char*>(y);
  if (xc < yc + xy && yc < xc + xy) return EDGE0_ERR_INVALID_ARG;
  if (T <= kDecodeMaxT && hd->groups == 1) {
    DecodeArgs a;
    fill_decode_args(hd, a, x, y, T);
    if (attach_stamps(hd, a, 1, (cudaStream_t)stream) != cudaSuccess) return EDGE0_ERR_CUDA;
    const cudaError_t e = decode_launch(a, hd->num_sms, hd->smem_total, (cudaStream_t)stream);
    if (e != cudaSuccess) return EDGE0_ERR_CUDA;
    hd->last_T = T;
    hd->last_path = 1;
    return EDGE0_OK;
  }
  if (T > hd->pf.max_tokens) return EDGE0_ERR_INVALID_ARG;
  if (hd->tiered) return EDGE0_ERR_UNSUPPORTED;   // prefill reads every record from device memory
  const edge0_status st = prefill_forward(hd->d, &hd->pf, hd->num_sms,
                                          static_cast<const __nv_bfloat16*>(x),
                                          static_cast<__nv_bfloat16*>(y), T, (cudaStream_t)stream);
  if (st == EDGE0_OK) { hd->last_T = T; hd->last_path = 2; }
  return st;
}

edge0_status edge0_moe_debug_routing(void* handle, int* idx, float* w, int* counts, int* offsets,
                                     int* perm, int* pos, edge0_stream_t stream) {
  Handle* hd = static_cast<Handle*>(handle);
  if (!hd) return EDGE0_ERR_INVALID_ARG;
  if (!hd->last_path) return EDGE0_ERR_UNSUPPORTED;
  const size_t tk = size_t(hd->last_T) * hd->d.top_k;
  const int E = hd->d.n_experts;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaSuccess;
  if (idx && e == cudaSuccess) e = cudaMemcpyAsync(idx, hd->idx, tk * 4, cudaMemcpyDeviceToDevice, s);
  if (w && e == cudaSuccess) e = cudaMemcpyAsync(w, hd->w, tk * 4, cudaMemcpyDeviceToDevice, s);
  if (counts && e == cudaSuccess) e = cudaMemcpyAsync(counts, hd->counts, size_t(E) * 4, cudaMemcpyDeviceToDevice, s);
  if (offsets && e == cudaSuccess) e = cudaMemcpyAsync(offsets, hd->offsets, size_t(E + 1) * 4, cudaMemcpyDeviceToDevice, s);
  if (perm && e == cudaSuccess) e = cudaMemcpyAsync(perm, hd->perm, tk * 4, cudaMemcpyDeviceToDevice, s);
  if (pos && e == cudaSuccess) e = cudaMemcpyAsync(pos, hd->pos, tk * 4, cudaMemcpyDeviceToDevice, s);
  return cuda_status(e);
}

edge0_status edge0_moe_debug_tensor(void* handle, int what, void* dst, size_t bytes, edge0_stream_t stream) {
  Handle* hd = static_cast<Handle*>(handle);
  if (!hd || !dst) return EDGE0_ERR_INVALID_ARG;
  if (!hd->last_path) return EDGE0_ERR_UNSUPPORTED;
  const size_t T = hd->last_T;
  const void* src = nullptr;
  size_t n = 0;
  if (hd->last_path == 1) {
    if (what == 0) { src = hd->z; n = T * hd->d.latent * 4; }
    else if (what == 1) { src = hd->logits; n = T * hd->d.n_experts * 4; }
    else if (what == 2) { src = hd->c; n = T * hd->d.latent * 4; }
  } else {
    src = prefill_debug_tensor(&hd->pf, what, hd->d, (int)T, &n);
  }
  if (!src) return what >= 0 && what <= 4 ? EDGE0_ERR_UNSUPPORTED : EDGE0_ERR_INVALID_ARG;
  if (bytes < n) return EDGE0_ERR_INVALID_ARG;
  return cuda_status(cudaMemcpyAsync(dst, src, n, cudaMemcpyDeviceToDevice, (cudaStream_t)stream));
}

edge0_status edge0_residual_rmsnorm(const void* x, const void* y, void* out, int T, int hidden, float eps,
                                    edge0_stream_t stream) {
  if (T < 0 || hidden <= 0 || hidden % 8 || !(eps >= 0.f)) return EDGE0_ERR_INVALID_ARG;
  if (T == 0) return EDGE0_OK;
  if (!x || !y || !out) return EDGE0_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(y, 16) || !aligned(out, 16)) return EDGE0_ERR_INVALID_ARG;
  residual_rmsnorm_kernel<<<(T + 7) / 8, 256, 0, (cudaStream_t)stream>>>(
      static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(y),
      static_cast<__nv_bfloat16*>(out), T, hidden, eps);
  return launch_status();
}

static bool same_layers(const std::vector<LayerW>& a, const std::vector<LayerW>& b) {
  if (a.size() != b.size()) return false;
  for (size_t i = 0; i < a.size(); ++i)
    if (a[i].D != b[i].D || a[i].U != b[i].U || a[i].RD != b[i].RD || a[i].bias != b[i].bias ||
        a[i].experts != b[i].experts || a[i].shared != b[i].shared || a[i].stride != b[i].stride ||
        a[i].dnorm != b[i].dnorm || a[i].rec_table != b[i].rec_table || a[i].resident != b[i].resident ||
        a[i].staging != b[i].staging || a[i].use != b[i].use || a[i].tier_stats != b[i].tier_stats)
      return false;
  return true;
}

static edge0_status stack_impl(void* const* handles, int n_layers, const void* x, void* y, int T, float eps,
                               void* trace_x, void* trace_y, int* trace_idx, edge0_stream_t stream) {
  if (!handles || n_layers < 1 || T < 0 || !(eps >= 0.f)) return EDGE0_ERR_INVALID_ARG;
  if (T == 0) return EDGE0_OK;
  Handle* h0 = static_cast<Handle*>(handles[0]);
  if (!h0 || !x || !y || !aligned(x, 16) || !aligned(y, 16)) return EDGE0_ERR_INVALID_ARG;
  for (int i = 0; i < n_layers; ++i) {
    const Handle* hi = static_cast<const Handle*>(handles[i]);
    if (!hi || hi->d.hidden != h0->d.hidden || hi->d.latent != h0->d.latent ||
        hi->d.n_experts != h0->d.n_experts || hi->d.top_k != h0->d.top_k || hi->d.ffn != h0->d.ffn ||
        hi->groups != h0->groups || hi->device != h0->device)
      return EDGE0_ERR_INVALID_ARG;
  }
  if (T > kDecodeMaxT || n_layers > kStackMax || h0->groups > 1) {
    if (trace_x || trace_y || trace_idx) return EDGE0_ERR_UNSUPPORTED;
    for (int i = 0; i < n_layers; ++i)
      if (static_cast<const Handle*>(handles[i])->tiered) return EDGE0_ERR_UNSUPPORTED;
    // chain: layer forward into the prefill scratch of handle 0, then the residual norm
    if (T > h0->pf.max_tokens) return EDGE0_ERR_INVALID_ARG;
    __nv_bfloat16* tmp = prefill_stack_scratch(&h0->pf);
    if (!tmp) return EDGE0_ERR_UNSUPPORTED;
    const void* cur = x;
    for (int i = 0; i < n_layers; ++i) {
      edge0_status st = edge0_moe_forward(handles[i], cur, tmp, T, stream);
      if (st != EDGE0_OK) return st;
      st = edge0_residual_rmsnorm(cur, tmp, y, T, h0->d.hidden, eps, stream);
      if (st != EDGE0_OK) return st;
      cur = y;
    }
    return EDGE0_OK;
  }
  std::vector<LayerW> lws(n_layers);
  for (int i = 0; i < n_layers; ++i) lws[i] = layer_of(static_cast<const Handle*>(handles[i]));
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaSuccess;
  // the device layer table is uploaded only when the list of layers changes, so a
  // call captured into a CUDA graph refers to device data alone
  if (!same_layers(h0->stack_tab, lws)) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) return EDGE0_ERR_CUDA;
    if (cs != cudaStreamCaptureStatusNone) return EDGE0_ERR_UNSUPPORTED;
    // pageable source: the copy is staged before the call returns
    e = cudaMemcpyAsync(h0->d_stack, lws.data(), sizeof(LayerW) * n_layers, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return EDGE0_ERR_CUDA;
    h0->stack_tab = lws;
  }
  DecodeArgs a;
  fill_decode_args(h0, a, x, y, T);
  a.layers = h0->d_stack;
  a.n_layers = n_layers;
  a.eps = eps;
  a.final_norm = 1;
  a.trace_x = static_cast<__nv_bfloat16*>(trace_x);
  a.trace_y = static_cast<__nv_bfloat16*>(trace_y);
  a.trace_idx = trace_idx;
  if (attach_stamps(h0, a, n_layers, s) != cudaSuccess) return EDGE0_ERR_CUDA;
  e = decode_launch(a, h0->num_sms, h0->smem_total, s);
  if (e != cudaSuccess) return EDGE0_ERR_CUDA;
  h0->last_T = T;
  h0->last_path = 1;
  return EDGE0_OK;
}

edge0_status edge0_moe_stack_forward(void* const* handles, int n_layers, const void* x, void* y, int T,
                                     float eps, edge0_stream_t stream) {
  return stack_impl(handles, n_layers, x, y, T, eps, nullptr, nullptr, nullptr, stream);
}

edge0_status edge0_moe_stack_forward_trace(void* const* handles, int n_layers, const void* x, void* y,
                                           int T, float eps, void* trace_x, void* trace_y, int* trace_idx,
                                           edge0_stream_t stream) {
  return stack_impl(handles, n_layers, x, y, T, eps, trace_x, trace_y, trace_idx, stream);
}

edge0_status edge0_moe_debug_wait_probe(void* handle, edge0_stream_t stream) {
  Handle* hd = static_cast<Handle*>(handle);
  if (!hd) return EDGE0_ERR_INVALID_ARG;
  wait_probe_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(hd->err);
  return launch_status();
}

edge0_status edge0_moe_profile_stages(void* handle, int enable) {
  Handle* hd = static_cast<Handle*>(handle);
  if (!hd) return EDGE0_ERR_INVALID_ARG;
  return cuda_status(prefill_profile(&hd->pf, enable != 0));
}

edge0_status edge0_moe_stage_times(void* handle, float* ms, int max, int* n_out) {
  Handle* hd = static_cast<Handle*>(handle);
  if (!hd || !ms || max < 0) return EDGE0_ERR_INVALID_ARG;
  if (hd->last_path != 2) return EDGE0_ERR_UNSUPPORTED;
  return prefill_stage_times(&hd->pf, ms, max, n_out);
}

edge0_status edge0_moe_profile_decode(void* handle, int enable) {
  Handle* hd = static_cast<Handle*>(handle);
  if (!hd) return EDGE0_ERR_INVALID_ARG;
  if (enable && !hd->stamps) {
    if (cudaMalloc(&hd->stamps, sizeof(unsigned long long) * kStampSlots * kStackMax) != cudaSuccess) {
      cudaGetLastError();
      return EDGE0_ERR_OOM;
    }
  }
  hd->dec_profile = enable != 0;
  hd->stamped_layers = 0;
  return EDGE0_OK;
}

edge0_status edge0_moe_decode_phase_times(void* handle, float* us, int max, int* n_out) {
  Handle* hd = static_cast<Handle*>(handle);
  if (!hd || !us || max < 0) return EDGE0_ERR_INVALID_ARG;
  if (!hd->stamps || hd->stamped_layers < 1) return EDGE0_ERR_UNSUPPORTED;
  unsigned long long st[kStampSlots * kStackMax];
  const int nl = hd->stamped_layers;
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpy(st, hd->stamps, sizeof(unsigned long long) * kStampSlots * nl, cudaMemcpyDeviceToHost) != cudaSuccess)
    return EDGE0_ERR_CUDA;
  int n = 0;
  for (int l = 0; l < nl; ++l) {
    const unsigned long long* t = st + l * kStampSlots;
    auto d = [](unsigned long long a, unsigned long long b) { return b >= a ? float(b - a) * 1e-3f : 0.f; };
    const unsigned long long e0 = ~t[kStP0EndMin], e1 = ~t[kStP1EndMin], e2 = ~t[kStP2EndMin], e3 = ~t[kStP3EndMin];
    const float v[EDGE0_DECODE_PHASES] = {
        d(t[kStP0Start], t[kStP0EndMax]), d(e0, t[kStP0EndMax]), d(t[kStP0EndMax], t[kStBar1]),
        d(t[kStBar1], t[kStRouted]), d(t[kStRouted], t[kStP1EndMax]), d(e1, t[kStP1EndMax]),
        d(t[kStP1EndMax], t[kStBar2]), d(t[kStBar2], t[kStP2EndMax]), d(e2, t[kStP2EndMax]),
        d(t[kStP2EndMax], t[kStBar3]), d(t[kStBar3], t[kStP3EndMax]), d(e3, t[kStP3EndMax]),
        t[kStBar4] ? d(t[kStP3EndMax], t[kStBar4]) : 0.f,
        d(t[kStP0Start], t[kStBar4] ? t[kStBar4] : t[kStP3EndMax]),
        d(t[kStBar1], t[kStRouteLoaded]), d(t[kStRouteLoaded], t[kStTopk]), d(t[kStRouted], t[kStP1Issued]),
        d(t[kStBar2], t[kStP2Staged]), d(t[kStP2Staged], t[kStP2Tasks])};
    for (int i = 0; i < EDGE0_DECODE_PHASES && n < max; ++i) us[n++] = v[i];
  }
  if (n_out) *n_out = n;
  return EDGE0_OK;
}

edge0_status edge0_moe_get_error(void* handle) {
  Handle* hd = static_cast<Handle*>(handle);
  if (!hd) return EDGE0_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return EDGE0_ERR_CUDA;
  int err = 0;
  if (cudaMemcpy(&err, hd->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return EDGE0_ERR_CUDA;
  if (err) {
    // clear the word and reset the grid barrier an aborted launch may have left behind
    if (cudaMemset(hd->err, 0, sizeof(int)) != cudaSuccess ||
        cudaMemset(hd->bar, 0, sizeof(GridBarrier)) != cudaSuccess)
      return EDGE0_ERR_CUDA;
    return EDGE0_ERR_TIMEOUT;
  }
  return EDGE0_OK;
}

// ------------------------------------------------------------------ residency tiering
int edge0_tier_plan(const unsigned int* use, int n_experts, int n_slots, const int* cur, int* next) {
  if (!use || !cur || !next || n_experts < 0 || n_slots < 0 || n_slots > n_experts) return -1;
  // the n_slots most-used experts (ties: lower index first); an expert not used at all
  // is not promoted, so a slot it would take keeps its current expert
  std::vector<int> order(n_experts);
  for (int e = 0; e < n_experts; ++e) order[e] = e;
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return use[a] > use[b]; });
  std::vector<char> want(n_experts, 0), placed(n_experts, 0);
  int n_want = 0;
  for (int i = 0; i < n_slots && i < n_experts && use[order[i]] > 0; ++i) { want[order[i]] = 1; ++n_want; }
  // experts already in a slot and still wanted stay where they are
  for (int s = 0; s < n_slots; ++s) {
    const int e = cur[s];
    next[s] = (e >= 0 && e < n_experts && want[e] && !placed[e]) ? e : -1;
    if (next[s] >= 0) placed[next[s]] = 1;
  }
  // the other wanted experts take the freed slots in rank order; slots left over keep
  // their current expert if it is not placed elsewhere
  int i = 0, changed = 0;
  for (int s = 0; s < n_slots; ++s) {
    if (next[s] >= 0) continue;
    while (i < n_experts && !(want[order[i]] && !placed[order[i]])) ++i;
    if (i < n_experts) {
      next[s] = order[i];
      placed[order[i]] = 1;
    } else {
      const int e = cur[s];
      next[s] = (e >= 0 && e < n_experts && !placed[e]) ? e : -1;
      if (next[s] >= 0) placed[next[s]] = 1;
    }
  }
  for (int s = 0; s < n_slots; ++s) changed += next[s] != cur[s];
  (void)n_want;
  return changed;
}

static edge0_status tier_upload(Handle* hd, cudaStream_t s) {
  const int E = hd->d.n_experts;
  const size_t stride = hd->d.expert_stride;
  std::vector<const uint8_t*> table(E);
  std::vector<uint8_t> res(E, 0);
  for (int e = 0; e < E; ++e) table[e] = hd->host_dev + size_t(e) * stride;
  for (int k = 0; k < hd->n_slots; ++k) {
    const int e = hd->slot_expert[k];
    if (e >= 0) { table[e] = hd->slots + size_t(k) * stride; res[e] = 1; }
  }
  // pageable sources: staged before the calls return, stream-ordered on the device
  if (cudaMemcpyAsync(hd->d_table, table.data(), sizeof(void*) * E, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(hd->d_resident, res.data(), E, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return EDGE0_ERR_CUDA;
  return cudaStreamSynchronize(s) == cudaSuccess ? EDGE0_OK : EDGE0_ERR_CUDA;
}

edge0_status edge0_moe_tier_attach(void* handle, const void* host_records, int n_slots, edge0_stream_t stream) {
  Handle* hd = static_cast<Handle*>(handle);
  if (!hd || !host_records || n_slots < 0 || n_slots > hd->d.n_experts) return EDGE0_ERR_INVALID_ARG;
  if (hd->tiered) return EDGE0_ERR_UNSUPPORTED;
  if (hd->d.max_tokens > kDecodeMaxT || hd->groups > 1) return EDGE0_ERR_UNSUPPORTED;   // decode forwards only
  void* dev = nullptr;
  if (cudaHostGetDevicePointer(&dev, const_cast<void*>(host_records), 0) != cudaSuccess || !dev) {
    cudaGetLastError();
    return EDGE0_ERR_INVALID_ARG;                    // not pinned host memory mapped for the device
  }
  if (!aligned(dev, 256)) return EDGE0_ERR_INVALID_ARG;
  const int E = hd->d.n_experts;
  const size_t stride = hd->d.expert_stride;
  const size_t o_tab = 0, o_res = align_up(sizeof(void*) * E, 256), o_use = o_res + align_up(E, 256);
  const size_t o_st = o_use + align_up(sizeof(unsigned int) * E, 256), ws = o_st + 256;
  uint8_t* slots = nullptr;
  uint8_t* staging = nullptr;
  char* tws = nullptr;
  if ((n_slots > 0 && cudaMalloc(&slots, size_t(n_slots) * stride) != cudaSuccess) ||
      cudaMalloc(&staging, size_t(kDecodeMaxT) * hd->d.top_k * stride) != cudaSuccess ||
      cudaMalloc(&tws, ws) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(slots); cudaFree(staging); cudaFree(tws);
    return EDGE0_ERR_OOM;
  }
  hd->host_records = static_cast<const uint8_t*>(host_records);
  hd->host_dev = static_cast<const uint8_t*>(dev);
  hd->n_slots = n_slots;
  hd->slots = slots;
  hd->staging = staging;
  hd->tier_ws = tws;
  hd->d_table = reinterpret_cast<const uint8_t**>(tws + o_tab);
  hd->d_resident = reinterpret_cast<uint8_t*>(tws + o_res);
  hd->d_use = reinterpret_cast<unsigned int*>(tws + o_use);
  hd->d_stats = reinterpret_cast<unsigned long long*>(tws + o_st);
  hd->slot_expert.assign(n_slots, -1);
  hd->tiered = true;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemsetAsync(hd->d_use, 0, sizeof(unsigned int) * E, s) != cudaSuccess ||
      cudaMemsetAsync(hd->d_stats, 0, 256, s) != cudaSuccess)
    return EDGE0_ERR_CUDA;
  return tier_upload(hd, s);
}

edge0_status edge0_moe_tier_place(void* handle, const int* slot_expert, edge0_stream_t stream) {
  Handle* hd = static_cast<Handle*>(handle);
  if (!hd || !slot_expert) return EDGE0_ERR_INVALID_ARG;
  if (!hd->tiered) return EDGE0_ERR_UNSUPPORTED;
  const int E = hd->d.n_experts;
  std::vector<char> seen(E, 0);
  for (int k = 0; k < hd->n_slots; ++k) {
    const int e = slot_expert[k];
    if (e < -1 || e >= E || (e >= 0 && seen[e])) return EDGE0_ERR_INVALID_ARG;
    if (e >= 0) seen[e] = 1;
  }
  cudaStream_t s = (cudaStream_t)stream;
  const size_t stride = hd->d.expert_stride;
  // the table first points every leaving expert back at host memory, then the slots
  // are refilled (stream order: forwards already enqueued finish with the old slots)
  std::vector<int> cur = hd->slot_expert;
  for (int k = 0; k < hd->n_slots; ++k)
    if (cur[k] != slot_expert[k]) hd->slot_expert[k] = -1;
  edge0_status st = tier_upload(hd, s);
  if (st != EDGE0_OK) return st;
  for (int k = 0; k < hd->n_slots; ++k) {
    const int e = slot_expert[k];
    if (e >= 0 && cur[k] != e &&
        cudaMemcpyAsync(hd->slots + size_t(k) * stride, hd->host_records + size_t(e) * stride, stride,
                        cudaMemcpyHostToDevice, s) != cudaSuccess)
      return EDGE0_ERR_CUDA;
    hd->slot_expert[k] = e;
  }
  return tier_upload(hd, s);
}

edge0_status edge0_moe_tier_rebalance(void* handle, edge0_stream_t stream) {
  Handle* hd = static_cast<Handle*>(handle);
  if (!hd) return EDGE0_ERR_INVALID_ARG;
  if (!hd->tiered) return EDGE0_ERR_UNSUPPORTED;
  const int E = hd->d.n_experts;
  cudaStream_t s = (cudaStream_t)stream;
  std::vector<unsigned int> use(E);
  if (cudaMemcpyAsync(use.data(), hd->d_use, sizeof(unsigned int) * E, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return EDGE0_ERR_CUDA;
  std::vector<int> next(hd->n_slots);
  if (edge0_tier_plan(use.data(), E, hd->n_slots, hd->slot_expert.data(), next.data()) < 0) return EDGE0_ERR_CUDA;
  const edge0_status st = edge0_moe_tier_place(handle, next.data(), stream);
  if (st != EDGE0_OK) return st;
  return cuda_status(cudaMemsetAsync(hd->d_use, 0, sizeof(unsigned int) * E, s));
}

edge0_status edge0_moe_tier_stats(void* handle, unsigned long long* out) {
  Handle* hd = static_cast<Handle*>(handle);
  if (!hd || !out) return EDGE0_ERR_INVALID_ARG;
  if (!hd->tiered) return EDGE0_ERR_UNSUPPORTED;
  unsigned long long st[3];
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpy(st, hd->d_stats, sizeof(st), cudaMemcpyDeviceToHost) != cudaSuccess)
    return EDGE0_ERR_CUDA;
  int resident = 0;
  for (int e : hd->slot_expert) resident += e >= 0;
  out[0] = st[0]; out[1] = st[1]; out[2] = st[2]; out[3] = (unsigned long long)resident;
  return EDGE0_OK;
}

edge0_status edge0_moe_tier_detach(void* handle) {
  Handle* hd = static_cast<Handle*>(handle);
  if (!hd) return EDGE0_ERR_INVALID_ARG;
  if (!hd->tiered) return EDGE0_OK;
  if (cudaDeviceSynchronize() != cudaSuccess) return EDGE0_ERR_CUDA;
  cudaFree(hd->slots);
  cudaFree(hd->staging);
  cudaFree(hd->tier_ws);
  hd->tiered = false;
  hd->slots = hd->staging = nullptr;
  hd->tier_ws = nullptr;
  hd->d_table = nullptr; hd->d_resident = nullptr; hd->d_use = nullptr; hd->d_stats = nullptr;
  hd->slot_expert.clear();
  hd->n_slots = 0;
  return EDGE0_OK;
}

const char* edge0_status_string(edge0_status s) {
  switch (s) {
    case EDGE0_OK: return "ok";
    case EDGE0_ERR_INVALID_ARG: return "invalid argument";
    case EDGE0_ERR_UNSUPPORTED: return "unsupported";
    case EDGE0_ERR_CUDA: return "CUDA error";
    case EDGE0_ERR_OOM: return "out of device memory";
    case EDGE0_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

void edge0_moe_destroy(void* handle) {
  Handle* hd = static_cast<Handle*>(handle);
  if (!hd) return;
  cudaDeviceSynchronize();
  prefill_destroy(&hd->pf);
  if (hd->stamps) cudaFree(hd->stamps);
  if (hd->tiered) {
    cudaFree(hd->slots);
    cudaFree(hd->staging);
    cudaFree(hd->tier_ws);
  }
  cudaFree(hd->ws);
  delete hd;
}

}  // extern "C"

// ------------------------------------------------------------------ forward without allocation
// Some callers cannot call cudaMalloc: code that runs under a fixed device-memory
// budget handed out by another allocator, plug-ins living inside a host program
// that owns every allocation, or real-time loops where an allocation (and the
// device synchronisation it can trigger) is not allowed.  For them the decode
// forward can run with its scratch in this file's static device array instead of
// a handle's workspace.  Every GPU that loads the library holds the array until
// the process exits.  All calls share it, so calls that overlap on the GPU (two
// streams, two host threads) race and must be serialised by the caller.
namespace {

// Limits of the static scratch (the layer shapes it can hold).
constexpr int kNaMaxT = kDecodeMaxT;       // 16 tokens
constexpr int kNaMaxH = 3072, kNaMaxL = 2048, kNaMaxE = 512, kNaMaxK = kMaxTopK, kNaMaxF = 1024;

constexpr size_t na_align(size_t v) { return (v + 255) / 256 * 256; }
constexpr size_t kNaRD = 0;                                                  // fp32 [E][H]
constexpr size_t kNaZ = kNaRD + na_align(size_t(kNaMaxE) * kNaMaxH * 4);     // fp32 [T][L]
constexpr size_t kNaZh = kNaZ + na_align(size_t(kNaMaxT) * kNaMaxL * 4);     // f16 [T][L]
constexpr size_t kNaLg = kNaZh + na_align(size_t(kNaMaxT) * kNaMaxL * 2);    // fp32 [T][E]
constexpr size_t kNaH = kNaLg + na_align(size_t(kNaMaxT) * kNaMaxE * 4);     // fp32 [T*K+T][F]
constexpr size_t kNaC = kNaH + na_align(size_t(kNaMaxT) * (kNaMaxK + 1) * kNaMaxF * 4);
constexpr size_t kNaYb = kNaC + na_align(size_t(kNaMaxT) * kNaMaxL * 4);     // bf16 [2][T][H]
constexpr size_t kNaXb = kNaYb + na_align(size_t(2) * kNaMaxT * kNaMaxH * 2);
constexpr size_t kNaRt = kNaXb + na_align(size_t(2) * kNaMaxT * kNaMaxH * 2); // idx w perm pos
constexpr size_t kNaCnt = kNaRt + na_align(size_t(4) * kNaMaxT * kNaMaxK * 4);
constexpr size_t kNaOff = kNaCnt + na_align(size_t(kNaMaxE) * 4);
constexpr size_t kNaBar = kNaOff + na_align(size_t(kNaMaxE + 1) * 4);        // barrier, error word, dnorm
constexpr size_t kNaBytes = kNaBar + 256;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNaBytes];

struct NoAllocDevice {
  bool ready = false;
  unsigned char* scratch = nullptr;   // device address of g_noalloc_scratch on this device
  int num_sms = 0;
  int smem_total = 0;
};
constexpr int kNaMaxDevices = 64;
NoAllocDevice g_na_dev[kNaMaxDevices];
std::mutex g_na_mutex;

// Once per device, with that device current: the array's device address and the
// decode kernel's launch limits.
edge0_status noalloc_setup(int dev, NoAllocDevice** out) {
  if (dev < 0 || dev >= kNaMaxDevices) return EDGE0_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_na_mutex);
  NoAllocDevice& d = g_na_dev[dev];
  if (!d.ready) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return EDGE0_ERR_CUDA;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return EDGE0_ERR_CUDA;
    if (prop.major < 10 || !prop.cooperativeLaunch) return EDGE0_ERR_UNSUPPORTED;
    const int smem = (int)prop.sharedMemPerBlockOptin - 1024;
    int occ = 0;
    if (decode_prepare(smem) != cudaSuccess || decode_occupancy(smem, &occ) != cudaSuccess) return EDGE0_ERR_CUDA;
    if (occ < 1) return EDGE0_ERR_UNSUPPORTED;
    d.scratch = static_cast<unsigned char*>(p);
    d.num_sms = prop.multiProcessorCount;
    d.smem_total = smem;
    d.ready = true;
  }
  *out = &d;
  return EDGE0_OK;
}

}  // namespace

extern "C" edge0_status edge0_moe_forward_noalloc(const edge0_moe_desc* desc, const void* x, void* y, int T,
                                                  int* status_out, edge0_stream_t stream) {
  if (!desc || T < 0) return EDGE0_ERR_INVALID_ARG;
  const edge0_moe_desc& d = *desc;
  if (d.hidden <= 0 || d.hidden % 64 || !shapes_ok(d.latent, d.ffn) || d.top_k < 1 || d.top_k > kMaxTopK ||
      d.n_experts < d.top_k || d.n_experts % 32)
    return EDGE0_ERR_INVALID_ARG;
  if (!d.D || !d.U || !d.router || !d.experts || !d.shared_expert || !aligned(d.D, 16) || !aligned(d.U, 16) ||
      !aligned(d.router, 16) || !aligned(d.experts, 256) || !aligned(d.shared_expert, 256) ||
      (d.router_bias && !aligned(d.router_bias, 4)) ||
      d.expert_stride < edge0_expert_record_bytes(d.latent, d.ffn) || d.expert_stride % 256)
    return EDGE0_ERR_INVALID_ARG;
  // sizes beyond what the static scratch holds; grouped projections run on handles only
  if (T > kNaMaxT || d.hidden > kNaMaxH || d.latent > kNaMaxL || d.n_experts > kNaMaxE || d.ffn > kNaMaxF ||
      d.n_groups > 1)
    return EDGE0_ERR_UNSUPPORTED;
  if (T == 0) return EDGE0_OK;
  if (!x || !y || !aligned(x, 16) || !aligned(y, 16)) return EDGE0_ERR_INVALID_ARG;
  const size_t xy = size_t(T) * d.hidden * 2;
  const char* xc = static_cast<const char*>(x);
  const char* yc = static_cast<const char*>(y);
  if (xc < yc + xy && yc < xc + xy) return EDGE0_ERR_INVALID_ARG;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return EDGE0_ERR_CUDA;
  NoAllocDevice* nd = nullptr;
  const edge0_status st = noalloc_setup(dev, &nd);
  if (st != EDGE0_OK) return st;
  unsigned char* s = nd->scratch;
  cudaStream_t cs = (cudaStream_t)stream;

  // a handle-shaped view of the static scratch (nothing is allocated)
  Handle view;
  view.d = d;
  view.device = dev;
  view.num_sms = nd->num_sms;
  view.smem_total = nd->smem_total;
  view.rd = reinterpret_cast<float*>(s + kNaRD);
  view.z = reinterpret_cast<float*>(s + kNaZ);
  view.zh = reinterpret_cast<__half*>(s + kNaZh);
  view.logits = reinterpret_cast<float*>(s + kNaLg);
  view.h = reinterpret_cast<float*>(s + kNaH);
  view.c = reinterpret_cast<float*>(s + kNaC);
  view.ybuf = reinterpret_cast<__nv_bfloat16*>(s + kNaYb);
  view.xbuf = reinterpret_cast<__nv_bfloat16*>(s + kNaXb);
  const int tk = kNaMaxT * kNaMaxK;
  view.idx = reinterpret_cast<int*>(s + kNaRt);
  view.w = reinterpret_cast<float*>(s + kNaRt) + tk;
  view.perm = reinterpret_cast<int*>(s + kNaRt) + 2 * tk;
  view.pos = reinterpret_cast<int*>(s + kNaRt) + 3 * tk;
  view.counts = reinterpret_cast<int*>(s + kNaCnt);
  view.offsets = reinterpret_cast<int*>(s + kNaOff);
  view.bar = reinterpret_cast<GridBarrier*>(s + kNaBar);
  view.err = reinterpret_cast<int*>(s + kNaBar + 128);
  // the decode kernel's shared-memory plan must fit this device (as create checks)
  if (!decode_fits(&view)) return EDGE0_ERR_UNSUPPORTED;
  // the array keeps the previous call's contents: the barrier, the error word and
  // the |z| bound's maximum must start at zero
  if (cudaMemsetAsync(s + kNaBar, 0, 256, cs) != cudaSuccess) return EDGE0_ERR_CUDA;
  float* dnorm_dev = reinterpret_cast<float*>(s + kNaBar + 192);
  // R D and the bound max_r sum_h |D_rh| for this layer, into the scratch (the
  // kernel scales z per token by a power of two from that bound, as on a handle)
  const int H = d.hidden, L = d.latent, E = d.n_experts;
  fold_router_kernel<<<dim3((H + 31) / 32, (E + 31) / 32), 256, 0, cs>>>(
      static_cast<const __nv_bfloat16*>(d.router), static_cast<const __nv_bfloat16*>(d.D), view.rd, E, L, H,
      nullptr, 0);
  row_l1_max_kernel<<<(L + 7) / 8, 256, 0, cs>>>(static_cast<const __nv_bfloat16*>(d.D), L, H, dnorm_dev);
  if (cudaGetLastError() != cudaSuccess) return EDGE0_ERR_CUDA;
  DecodeArgs a;
  fill_decode_args(&view, a, x, y, T);
  a.layers = nullptr;              // one layer: the kernel reads only a.l0
  a.dnorm_dev = dnorm_dev;
  if (decode_launch(a, nd->num_sms, nd->smem_total, cs) != cudaSuccess) return EDGE0_ERR_CUDA;
  if (status_out &&
      cudaMemcpyAsync(status_out, view.err, sizeof(int), cudaMemcpyDeviceToDevice, cs) != cudaSuccess)
    return EDGE0_ERR_CUDA;
  return EDGE0_OK;
}
