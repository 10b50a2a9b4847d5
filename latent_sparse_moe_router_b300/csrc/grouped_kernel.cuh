// The grouped NVFP4 GEMM kernel (types and tiling in grouped.cuh).  Included by
// one translation unit only.
#pragma once

#include "grouped.cuh"

namespace edge0 {

__device__ __forceinline__ float silu_gg(float v) { return v / (1.0f + expf(-v)); }

// Two E2M1 codes (one byte) times a block scale, as bf16x2 (exact).  sc2 holds the
// scale times 2^112 in both bf16 halves: the f16 -> bf16 move below leaves the
// value 2^-112 too small (exponent field kept, mantissa truncated to the 7 bits
// bf16 has, which the E2M1 values never use).
__device__ __forceinline__ uint32_t dq_pair(uint32_t byte, uint32_t sc2) {
  const uint32_t h = e2m1x2_to_h2(byte);
  const uint32_t t = ((h >> 3) & 0x0FFF0FFFu) | (h & 0x80008000u);
  __nv_bfloat162 r = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&t),
                             *reinterpret_cast<const __nv_bfloat162*>(&sc2));
  return *reinterpret_cast<uint32_t*>(&r);
}

// bf16x2 (both halves) of an E4M3 scale times 2^112.
__device__ __forceinline__ uint32_t scale_bf16x2(uint32_t e4m3) {
  const float s = e4m3_to_f32(e4m3) * 5.192296858534828e33f;  // 2^112
  __nv_bfloat162 r = __floats2bfloat162_rn(s, s);
  return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Barrier `id` over n threads that also returns whether pred held in all of them.
__device__ __forceinline__ bool named_and(int id, int n, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
      " barrier.cta.red.and.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r) : "r"(uint32_t(pred)), "r"(id), "r"(n) : "memory");
  return r != 0;
}

__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__global__ void __launch_bounds__(kGgThreads, 1)
grouped_nvfp4_kernel(const __grid_constant__ GgMaps maps, const __grid_constant__ GgParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + GgSmem::offBar);
  uint64_t* a_full = bars;                 // [S] 128 dequant arrivals
  uint64_t* b_full = a_full + kGgS;        // [S] TMA bytes
  uint64_t* ab_empty = b_full + kGgS;      // [S] MMA commit
  uint64_t* raw_full = ab_empty + kGgS;    // [R] TMA bytes
  uint64_t* raw_empty = raw_full + kGgR;   // [R] 128 dequant arrivals
  uint64_t* sc_full = raw_empty + kGgR;    // TMA bytes
  uint64_t* accf = sc_full + 1;            // MMA commit
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accf + 1);
  int* tile_info = reinterpret_cast<int*>(tmem_slot + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- which tile: token tile tt = b / mtiles of group g (binary search over the
  // token-tile prefix), weight tile mt = b % mtiles; consecutive CTAs share tt
  __shared__ int s_bad;
  if (threadIdx.x == 0) {
    const int tt = blockIdx.x / p.mtiles;
    int g = -1;
    if (!(p.abort && ld_relaxed_s32(p.abort)) && tt < p.tprefix[p.E + 1]) {
      int lo = 0, hi = p.E + 1;            // tprefix[lo] <= tt < tprefix[hi]
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (p.tprefix[mid] <= tt) lo = mid; else hi = mid;
      }
      g = lo;
      tile_info[1] = tt - p.tprefix[lo];
      tile_info[2] = blockIdx.x % p.mtiles;
    }
    tile_info[0] = g;
    s_bad = 0;
  }
  __syncthreads();
  const int g = tile_info[0];
  if (g < 0) return;
  const int nt = tile_info[1], mt = tile_info[2];
  const bool shared = (g == p.E);
  const int n_g = shared ? p.T : p.counts[g];
  const int row0 = nt * kGgBN;                                   // first token of the tile in the group
  const int n_rows = min(kGgBN, n_g - row0);
  const int out0 = (shared ? p.TK : p.offsets[g]) + row0;        // position of the tile's first token
  const int pos0 = (shared && p.mode == 1) ? row0 : out0;        // its B row
  const int K = p.mode == 1 ? p.L : p.F;
  const int nk = K / 64;
  const int n_mma = (n_rows + 15) & ~15;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGgS; ++s) { mbar_init(&a_full[s], 128); mbar_init(&b_full[s], 1); mbar_init(&ab_empty[s], 1); }
    for (int s = 0; s < kGgR; ++s) { mbar_init(&raw_full[s], 1); mbar_init(&raw_empty[s], 128); }
    mbar_init(sc_full, 1);
    mbar_init(accf, 1);
    fence_mbar_init();
  }
  if (warp == 5) { tmem_alloc(tmem_slot, 256); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const CUtensorMap* mcodes = shared ? &maps.s_codes : &maps.a_codes;
  const CUtensorMap* mscales = shared ? &maps.s_scales : &maps.a_scales;
  const CUtensorMap* mb = (shared && p.mode == 1) ? &maps.b_shared : &maps.b_routed;

  bool ok = true;   // this thread's waits all succeeded
  if (warp == 4) {
    if (lane == 0) {
      // ---- producer: scales once, then raw codes (R ring) and B tiles (S ring)
      const int scb = p.mode == 1 ? 2 * 64 * (p.L / 16) : 64 * (p.F / 8);
      mbar_arrive_expect_tx(sc_full, scb);
      uint8_t* sc = smem + GgSmem::offSc;
      if (p.mode == 1) {
        const int f0 = mt * 64;
        if (shared) {
          tma_load_2d(sc, mscales, p.L, f0, sc_full);
          tma_load_2d(sc + 64 * (p.L / 16), mscales, p.L + p.L / 16, f0, sc_full);
        } else {
          tma_load_3d(sc, mscales, p.L, f0, g, sc_full);
          tma_load_3d(sc + 64 * (p.L / 16), mscales, p.L + p.L / 16, f0, g, sc_full);
        }
      } else {
        const int q0 = mt * 64;   // first row pair
        if (shared) tma_load_2d(sc, mscales, p.F, q0, sc_full);
        else tma_load_3d(sc, mscales, p.F, q0, g, sc_full);
      }
      for (int kb = 0; kb < nk; ++kb) {
        const int r = kb % kGgR;
        if (!mbar_wait_abort(&raw_empty[r], ((kb / kGgR) & 1) ^ 1, p.err, p.abort)) { s_bad = 1; break; }
        mbar_arrive_expect_tx(&raw_full[r], GgSmem::kRaw);
        uint8_t* raw = smem + GgSmem::offRaw + r * GgSmem::kRaw;
        // first half: gate rows (mode 1) / even latent rows (mode 2); second half:
        // up rows / odd latent rows
        const int x0 = kb * 32, x1 = (p.mode == 1 ? p.L / 2 : p.F / 2) + kb * 32;
        const int y = mt * 64;
        if (shared) {
          tma_load_2d(raw, mcodes, x0, y, &raw_full[r]);
          tma_load_2d(raw + 2048, mcodes, x1, y, &raw_full[r]);
        } else {
          tma_load_3d(raw, mcodes, x0, y, g, &raw_full[r]);
          tma_load_3d(raw + 2048, mcodes, x1, y, g, &raw_full[r]);
        }
        const int s = kb % kGgS;
        if (!mbar_wait_abort(&ab_empty[s], ((kb / kGgS) & 1) ^ 1, p.err, p.abort)) { s_bad = 1; break; }
        mbar_arrive_expect_tx(&b_full[s], GgSmem::kB);
        tma_load_2d(smem + GgSmem::offB + s * GgSmem::kB, mb, kb * 64, pos0, &b_full[s]);
      }
    }
  } else if (warp == 5) {
    if (lane == 0) {
      // ---- MMA issuer
      const uint32_t idesc = idesc_bf16_f32(128, n_mma);
      for (int kb = 0; kb < nk; ++kb) {
        const int s = kb % kGgS;
        const uint32_t ph = (kb / kGgS) & 1;
        if (!mbar_wait_abort(&a_full[s], ph, p.err, p.abort) || !mbar_wait_abort(&b_full[s], ph, p.err, p.abort)) {
          s_bad = 1;
          break;
        }
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + GgSmem::offA + s * GgSmem::kA);
        const uint32_t sb = smem_u32(smem + GgSmem::offB + s * GgSmem::kB);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16(tmem, sw128_desc(sa + k * 32), sw128_desc(sb + k * 32), idesc, (kb | k) != 0);
        mma_commit(&ab_empty[s]);
      }
      mma_commit(accf);
    }
  } else {
    // ---- dequant: thread r owns A row r
    const int r = threadIdx.x;
    const uint8_t* sc = smem + GgSmem::offSc;
    // this row's scales: mode 1 rows 0-63 gate, 64-127 up; mode 2 rows r = 2q + h
    const uint8_t* my_sc = p.mode == 1 ? sc + r * (p.L / 16) : sc + (r >> 1) * (p.F / 8) + (r & 1) * (p.F / 16);
    const int raw_off = p.mode == 1 ? r * 32 : (r & 1) * 2048 + (r >> 1) * 32;
    ok = mbar_wait_abort(sc_full, 0, p.err, p.abort);
    for (int kb = 0; ok && kb < nk; ++kb) {
      const int rr = kb % kGgR, s = kb % kGgS;
      if (!mbar_wait_abort(&raw_full[rr], (kb / kGgR) & 1, p.err, p.abort)) { ok = false; break; }
      const uint8_t* raw = smem + GgSmem::offRaw + rr * GgSmem::kRaw + raw_off;
      const uint4 c0 = reinterpret_cast<const uint4*>(raw)[0];
      const uint4 c1 = reinterpret_cast<const uint4*>(raw)[1];
      const uint32_t s4 = *reinterpret_cast<const uint32_t*>(my_sc + kb * 4);
      mbar_arrive(&raw_empty[rr]);
      if (!mbar_wait_abort(&ab_empty[s], ((kb / kGgS) & 1) ^ 1, p.err, p.abort)) { ok = false; break; }
      uint8_t* arow = smem + GgSmem::offA + s * GgSmem::kA + r * 128;
      const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint32_t sc2 = scale_bf16x2((s4 >> (8 * (c >> 1))) & 0xFF);
        uint4 o;
        o.x = dq_pair(cw[c] & 0xFF, sc2);
        o.y = dq_pair((cw[c] >> 8) & 0xFF, sc2);
        o.z = dq_pair((cw[c] >> 16) & 0xFF, sc2);
        o.w = dq_pair(cw[c] >> 24, sc2);
        *reinterpret_cast<uint4*>(arow + ((c ^ (r & 7)) << 4)) = o;
      }
      fence_async_smem();
      mbar_arrive(&a_full[s]);
    }
    if (!ok) s_bad = 1;
  }

  // ---- epilogue (warps 0-3).  The issuer always commits accf, so this wait ends
  // once every MMA it issued has finished (time limit only); the 128 threads then
  // agree, in one barrier, whether all of them got that far.
  bool acc_ok = false;
  if (warp < 4) acc_ok = mbar_wait_abort(accf, 0, p.err, nullptr);
  if (warp < 4 && named_and(1, 128, ok && acc_ok && !s_bad)) {
    tc_fence_after();
    // the stages are free now: reuse the A ring as transpose buffers
    float* ubuf = reinterpret_cast<float*>(smem + GgSmem::offA);             // [64][33] fp32
    __nv_bfloat16* tbuf = reinterpret_cast<__nv_bfloat16*>(smem + GgSmem::offA + 16384);  // [32][136]
    const uint8_t* rec = shared ? p.shared : p.experts + size_t(g) * p.stride;
    const float* gl = reinterpret_cast<const float*>(rec + size_t(27) * p.F * p.L / 16);
    const uint32_t lane_base = uint32_t(warp * 32) << 16;
    for (int c = 0; c * 32 < n_rows; ++c) {
      uint32_t v[32];
      tmem_ld32(tmem + lane_base + c * 32, v);
      tmem_ld_wait();
      if (p.mode == 1) {
        // lanes 64-127 (warps 2, 3) hold up rows: hand them to the gate warps
        if (warp >= 2) {
          const int fl = (warp - 2) * 32 + lane;
#pragma unroll
          for (int j = 0; j < 32; ++j) ubuf[fl * 33 + j] = __uint_as_float(v[j]);
        }
        named_sync(1, 128);
        if (warp < 2) {
          const int fl = warp * 32 + lane;
          const float gg = gl[0], gu = gl[1];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float h = silu_gg(gg * __uint_as_float(v[j])) * (gu * ubuf[fl * 33 + j]);
            tbuf[j * 136 + fl] = __float2bfloat16_rn(h);
          }
        }
        named_sync(1, 128);
        // 32 token rows x 64 f (128 B): 4 threads per row, 32 B each
        const int tr = threadIdx.x >> 2, part = threadIdx.x & 3;
        if (c * 32 + tr < n_rows) {
          const uint4* src = reinterpret_cast<const uint4*>(tbuf + tr * 136 + part * 16);
          uint4* dst = reinterpret_cast<uint4*>(p.out + size_t(out0 + c * 32 + tr) * p.out_ld + mt * 64 + part * 16);
          dst[0] = src[0];
          dst[1] = src[1];
        }
        named_sync(1, 128);
      } else {
        const float gd = gl[2];
        const int rl = warp * 32 + lane;   // latent row in the tile
#pragma unroll
        for (int j = 0; j < 32; ++j) tbuf[j * 136 + rl] = __float2bfloat16_rn(gd * __uint_as_float(v[j]));
        named_sync(1, 128);
        // 32 token rows x 128 latent rows (256 B): 4 threads per row, 64 B each
        const int tr = threadIdx.x >> 2, part = threadIdx.x & 3;
        if (c * 32 + tr < n_rows) {
          const uint4* src = reinterpret_cast<const uint4*>(tbuf + tr * 136 + part * 32);
          uint4* dst = reinterpret_cast<uint4*>(p.out + size_t(out0 + c * 32 + tr) * p.out_ld + mt * 128 + part * 32);
#pragma unroll
          for (int q = 0; q < 4; ++q) dst[q] = src[q];
        }
        named_sync(1, 128);
      }
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  // after a wait gave up, bulk copies issued by this CTA may still be landing:
  // give them a bounded time before the shared memory is released
  if (s_bad && threadIdx.x == 0) {
    const unsigned long long t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 50000ull) {}
  }
  __syncthreads();
  if (warp == 5) tmem_dealloc(tmem, 256);
}

}  // namespace edge0
