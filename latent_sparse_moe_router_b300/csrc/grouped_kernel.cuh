// The grouped NVFP4 GEMM kernel (types, tiling and warp roles in grouped.cuh).
// Included by one translation unit only.
#pragma once

#include "grouped.cuh"

namespace edge0 {

constexpr int kGgBBox = 64;       // rows of one B box (TMA)

// silu(v) = v / (1 + e^-v) with the hardware exponential and the fast division (the
// result is rounded to bf16, far coarser than their error); v -> -inf gives -0.
__device__ __forceinline__ float silu_gg(float v) { return __fdividef(v, 1.0f + __expf(-v)); }

// f16x2 holding E2M1 values -> bf16x2 times a block scale, exact.  sc2 holds the
// scale times 2^112 in both bf16 halves: moving the f16 bits right by 3 puts the
// exponent field in bf16 position (the value becomes 2^-112 too small) and drops
// three mantissa bits the E2M1 values never use; the sign bits are kept as they are.
__device__ __forceinline__ uint32_t h2_to_bf2_scaled(uint32_t h, uint32_t sc2) {
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

struct GgTile {
  int g, mt, n_rows, n_mma, pos0, out0;
  bool shared;
};

// CTA `rank`'s part of pair tile `tile`: token tile tt = tile / (mtiles / 2) of
// group g (binary search over the token-tile prefix), weight tile
// mt = 2 (tile % (mtiles / 2)) + rank.
__device__ __forceinline__ GgTile gg_tile(const GgParams& p, int tile, int rank) {
  GgTile t;
  const int mp = p.mtiles >> 1;
  const int tt = tile / mp;
  t.mt = 2 * (tile % mp) + rank;
  int lo = 0, hi = p.E + 1;            // tprefix[lo] <= tt < tprefix[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(&p.tprefix[mid]) <= tt) lo = mid; else hi = mid;
  }
  t.g = lo;
  t.shared = (lo == p.E);
  const int row0 = (tt - __ldg(&p.tprefix[lo])) * kGgBN;
  const int n_g = t.shared ? p.T : __ldg(&p.counts[lo]);
  t.n_rows = min(kGgBN, n_g - row0);
  t.n_mma = (t.n_rows + 15) & ~15;
  t.out0 = (t.shared ? p.TK : __ldg(&p.offsets[lo])) + row0;
  t.pos0 = (t.shared && p.mode == 1) ? row0 : t.out0;
  return t;
}

__global__ void __launch_bounds__(kGgThreads, 1)
grouped_nvfp4_kernel(const __grid_constant__ GgMaps maps, const __grid_constant__ GgParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + GgSmem::offBar);
  uint64_t* a_full = bars;                 // [SA] one arrival per dequant warp
  uint64_t* a_empty = a_full + kGgSA;      // [SA] MMA commit
  uint64_t* b_full = a_empty + kGgSA;      // [SB] TMA bytes
  uint64_t* b_empty = b_full + kGgSB;      // [SB] MMA commit
  uint64_t* raw_full = b_empty + kGgSB;    // [R] TMA bytes
  uint64_t* raw_empty = raw_full + kGgR;   // [R] one arrival per dequant warp
  uint64_t* sc_full = raw_empty + kGgR;    // [2] TMA bytes
  uint64_t* sc_empty = sc_full + 2;        // [2] one arrival per dequant warp
  uint64_t* acc_full = sc_empty + 2;       // [2] MMA commit
  uint64_t* acc_empty = acc_full + 2;      // [2] one arrival per epilogue warp
  uint64_t* mma_done = acc_empty + 2;      // final MMA commit
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  int* s_flags = reinterpret_cast<int*>(tmem_slot + 2);   // [0] total tiles, [1] bad
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = int(cluster_ctarank());
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    // the pair-tile count both CTAs read from the same word, so that they agree
    s_flags[0] = p.tprefix[p.E + 1] * (p.mtiles >> 1);
    s_flags[1] = 0;
    // consumer barriers take one arrival per warp (lane 0 after a __syncwarp); the
    // stage and accumulator barriers of rank 0 count both CTAs' warps
    for (int s = 0; s < kGgSA; ++s) { mbar_init(&a_full[s], 2 * kGgDqWarps); mbar_init(&a_empty[s], 1); }
    for (int s = 0; s < kGgSB; ++s) { mbar_init(&b_full[s], 2); mbar_init(&b_empty[s], 1); }
    for (int s = 0; s < kGgR; ++s) { mbar_init(&raw_full[s], 1); mbar_init(&raw_empty[s], kGgDqWarps); }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sc_full[b], 1); mbar_init(&sc_empty[b], kGgDqWarps);
      mbar_init(&acc_full[b], 1); mbar_init(&acc_empty[b], 2 * (kGgEpThreads / 32));
    }
    mbar_init(mma_done, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const int total = s_flags[0];
  if (pair >= total) return;   // both CTAs of the pair leave together
  if (warp == 1) { tmem_alloc_pair(tmem_slot, 512); tmem_relinquish_pair(); }
  tc_fence_before();
  // both CTAs' barriers exist and the pair's TMEM is allocated before anyone signals
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int K = p.mode == 1 ? p.L : p.F;
  const int nk = K / 64;
  bool ok = true;   // this thread's waits all succeeded

  if (warp == 0) {
    if (lane == 0) {
      // ---- scale and raw-code producer
      const int scb = p.mode == 1 ? 2 * 64 * (p.L / 16) : 64 * (p.F / 8);
      int it = 0, ti = 0;
      for (int tile = pair; ok && tile < total; tile += npairs, ++ti) {
        const GgTile t = gg_tile(p, tile, rank);
        const CUtensorMap* mcodes = t.shared ? &maps.s_codes : &maps.a_codes;
        const CUtensorMap* mscales = t.shared ? &maps.s_scales : &maps.a_scales;
        const int sb = ti & 1;
        if (!mbar_wait_abort(&sc_empty[sb], ((ti >> 1) & 1) ^ 1, p.err, p.abort)) { ok = false; break; }
        mbar_arrive_expect_tx(&sc_full[sb], scb);
        uint8_t* sc = smem + GgSmem::offSc + sb * GgSmem::kSc;
        const int y = t.mt * 64;   // first gate/up row, or first down row pair
        if (p.mode == 1) {
          if (t.shared) {
            tma_load_2d(sc, mscales, p.L, y, &sc_full[sb]);
            tma_load_2d(sc + 64 * (p.L / 16), mscales, p.L + p.L / 16, y, &sc_full[sb]);
          } else {
            tma_load_3d(sc, mscales, p.L, y, t.g, &sc_full[sb]);
            tma_load_3d(sc + 64 * (p.L / 16), mscales, p.L + p.L / 16, y, t.g, &sc_full[sb]);
          }
        } else {
          if (t.shared) tma_load_2d(sc, mscales, p.F, y, &sc_full[sb]);
          else tma_load_3d(sc, mscales, p.F, y, t.g, &sc_full[sb]);
        }
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int r = it % kGgR;
          if (!mbar_wait_abort(&raw_empty[r], ((it / kGgR) & 1) ^ 1, p.err, p.abort)) { ok = false; break; }
          mbar_arrive_expect_tx(&raw_full[r], GgSmem::kRaw);
          uint8_t* raw = smem + GgSmem::offRaw + r * GgSmem::kRaw;
          // first half: gate rows (mode 1) / even latent rows (mode 2); second
          // half: up rows / odd latent rows
          const int x0 = kb * 32, x1 = (p.mode == 1 ? p.L / 2 : p.F / 2) + kb * 32;
          if (t.shared) {
            tma_load_2d(raw, mcodes, x0, y, &raw_full[r]);
            tma_load_2d(raw + 2048, mcodes, x1, y, &raw_full[r]);
          } else {
            tma_load_3d(raw, mcodes, x0, y, t.g, &raw_full[r]);
            tma_load_3d(raw + 2048, mcodes, x1, y, t.g, &raw_full[r]);
          }
        }
      }
    }
  } else if (warp == kGgBWarp) {
    if (lane == 0) {
      // ---- B producer: this CTA's half of the tile's token rows (MMA columns
      // rank * N/2 ..), one k-slice per stage, completing on rank 0's barrier
      const uint32_t bfull0 = mapa_shared(smem_u32(b_full), 0);
      int it = 0;
      for (int tile = pair; ok && tile < total; tile += npairs) {
        const GgTile t = gg_tile(p, tile, rank);
        const CUtensorMap* mb = (t.shared && p.mode == 1) ? &maps.b_shared : &maps.b_routed;
        const int half = t.n_mma >> 1;
        const int row0 = t.pos0 + rank * half;
        const int nbox = (half + kGgBBox - 1) / kGgBBox;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % kGgSB;
          if (!mbar_wait_abort(&b_empty[s], ((it / kGgSB) & 1) ^ 1, p.err, p.abort)) { ok = false; break; }
          const uint32_t fb = bfull0 + uint32_t(s) * 8u;
          mbar_arrive_expect_tx_cl(fb, nbox * kGgBBox * 128);
          uint8_t* bs = smem + GgSmem::offB + s * GgSmem::kB;
          for (int bx = 0; bx < nbox; ++bx)
            tma_load_2d_pair(bs + bx * kGgBBox * 128, mb, kb * 64, row0 + bx * kGgBBox, fb);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---- MMA issuer (rank 0 of the pair)
      int it = 0, ti = 0;
      for (int tile = pair; ok && tile < total; tile += npairs, ++ti) {
        const GgTile t = gg_tile(p, tile, 0);
        const uint32_t idesc = p.mode == 1 ? idesc_f16_f32(256, t.n_mma) : idesc_bf16_f32(256, t.n_mma);
        const int ab = ti & 1;
        if (!mbar_wait_abort(&acc_empty[ab], ((ti >> 1) & 1) ^ 1, p.err, p.abort)) { ok = false; break; }
        tc_fence_after();
        const uint32_t acc = tmem + ab * 256;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int sa_i = it % kGgSA, sb_i = it % kGgSB;
          if (!mbar_wait_abort(&a_full[sa_i], (it / kGgSA) & 1, p.err, p.abort) ||
              !mbar_wait_abort(&b_full[sb_i], (it / kGgSB) & 1, p.err, p.abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + GgSmem::offA + sa_i * GgSmem::kA);
          const uint32_t sbb = smem_u32(smem + GgSmem::offB + sb_i * GgSmem::kB);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_pair_f16(acc, sw128_desc(sa + k * 32), sw128_desc(sbb + k * 32), idesc, (kb | k) != 0);
          mma_pair_commit_both(&a_empty[sa_i]);
          mma_pair_commit_both(&b_empty[sb_i]);
        }
        if (!ok) break;
        mma_pair_commit_both(&acc_full[ab]);
      }
      // every MMA issued has finished, and both CTAs' epilogues have released the
      // last two accumulators (their arrivals land here), before this CTA winds down
      mma_pair_commit(mma_done);
      mbar_wait_abort(mma_done, 0, p.err, nullptr);
      for (int j = ti - 2; ok && j < ti; ++j)
        if (j >= 0 && !mbar_wait_abort(&acc_empty[j & 1], (j >> 1) & 1, p.err, p.abort)) ok = false;
    }
  } else if (warp < kGgEpWarp0) {
    // ---- dequantisation: thread pair (r, hh) owns A row r, elements 32 hh .. 32 hh + 31.
    // A rows come in pairs 2i, 2i+1: mode 1 gate and up row f0 + i (so the epilogue
    // finds both in neighbouring lanes), mode 2 latent rows 2(q0 + i) and 2(q0 + i) + 1.
    // Raw codes: first 2 KB the 64 even-row slices, then the 64 odd-row slices.
    const int td = threadIdx.x - kGgDqWarp0 * 32;
    const int r = td >> 1, hh = td & 1;
    const int raw_off = (r & 1) * 2048 + (r >> 1) * 32 + hh * 16;
    const int sc_off = (p.mode == 1 ? (r & 1) * 64 * (p.L / 16) + (r >> 1) * (p.L / 16)
                                    : (r >> 1) * (p.F / 8) + (r & 1) * (p.F / 16)) + hh * 2;
    const uint32_t afull0 = mapa_shared(smem_u32(a_full), 0);
    int it = 0, ti = 0;
    for (int tile = pair; ok && tile < total; tile += npairs, ++ti) {
      const int sb = ti & 1;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait_abort(&sc_full[sb], (ti >> 1) & 1, p.err, p.abort))) { ok = false; break; }
      const uint8_t* my_sc = smem + GgSmem::offSc + sb * GgSmem::kSc + sc_off;
      for (int kb = 0; kb < nk; ++kb, ++it) {
        const int rr = it % kGgR, s = it % kGgSA;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait_abort(&raw_full[rr], (it / kGgR) & 1, p.err, p.abort))) { ok = false; break; }
        const uint4 cw4 = *reinterpret_cast<const uint4*>(smem + GgSmem::offRaw + rr * GgSmem::kRaw + raw_off);
        const uint32_t s2 = *reinterpret_cast<const uint16_t*>(my_sc + kb * 4);
        // dequantise into registers first: only the stores wait for the stage
        const uint32_t cw[4] = {cw4.x, cw4.y, cw4.z, cw4.w};
        uint4 o[4];
        if (p.mode == 1) {
          const uint32_t sc0 = scale_f16x2(s2 & 0xFF), sc1 = scale_f16x2(s2 >> 8);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            // 16-byte chunk c = 4 hh + j of the row: elements 8c .. 8c + 7, block c / 2
            const uint32_t sc2 = j < 2 ? sc0 : sc1;
            uint32_t h0, h1, h2, h3;
            e2m1x8_to_h2x4(cw[j], h0, h1, h2, h3);
            o[j] = make_uint4(hmul2_u32(h0, sc2), hmul2_u32(h1, sc2), hmul2_u32(h2, sc2), hmul2_u32(h3, sc2));
          }
        } else {
          const uint32_t sc0 = scale_bf16x2(s2 & 0xFF), sc1 = scale_bf16x2(s2 >> 8);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t sc2 = j < 2 ? sc0 : sc1;
            uint32_t h0, h1, h2, h3;
            e2m1x8_to_h2x4(cw[j], h0, h1, h2, h3);
            o[j].x = h2_to_bf2_scaled(h0, sc2);
            o[j].y = h2_to_bf2_scaled(h1, sc2);
            o[j].z = h2_to_bf2_scaled(h2, sc2);
            o[j].w = h2_to_bf2_scaled(h3, sc2);
          }
        }
        // the raw stage is released only once every lane's codes and scales have been
        // consumed into registers (the arithmetic above depends on both loads): a
        // release straight after the loads let the next TMA fill overwrite the first
        // half of the stage while a lane's read was still outstanding
        __syncwarp();
        if (lane == 0) mbar_arrive(&raw_empty[rr]);
        if (!__all_sync(0xFFFFFFFFu, mbar_wait_abort(&a_empty[s], ((it / kGgSA) & 1) ^ 1, p.err, p.abort))) { ok = false; break; }
        uint8_t* arow = smem + GgSmem::offA + s * GgSmem::kA + r * 128;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int c = 4 * hh + j;
          *reinterpret_cast<uint4*>(arow + ((c ^ (r & 7)) << 4)) = o[j];
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(afull0 + uint32_t(s) * 8u);
      }
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(&sc_empty[sb]);
    }
  } else {
    // ---- epilogue: warp q = warp % 4 reads TMEM lanes 32q .. 32q + 31 (A rows), and
    // half ch of every 32-column chunk (columns 16 ch .. 16 ch + 15).  Neighbouring
    // lanes hold the row pair (2i, 2i+1); after one shuffle per column pair the even
    // lane finishes the half's first 8 token columns, the odd lane the last 8.
    const int q = warp & 3;
    const int te = threadIdx.x - kGgEpWarp0 * 32;   // 0..255
    const int ch = te >> 7;
    const int odd = lane & 1, pr = q * 16 + (lane >> 1);   // row pair in the tile
    // mode 1: [32 tokens][72] bf16 (64 f used); mode 2: [32 tokens][68] u32 (64 latent pairs used)
    __nv_bfloat16* hbuf = reinterpret_cast<__nv_bfloat16*>(smem + GgSmem::offEpi);
    uint32_t* obuf = reinterpret_cast<uint32_t*>(smem + GgSmem::offEpi);
    float* zbuf = reinterpret_cast<float*>(smem + GgSmem::offEpi + GgSmem::kEpiT);   // [256] token scales
    const uint32_t accempty0 = mapa_shared(smem_u32(acc_empty), 0);
    int ti = 0;
    for (int tile = pair; ok && tile < total; tile += npairs, ++ti) {
      const GgTile t = gg_tile(p, tile, rank);
      const int ab = ti & 1;
      // the tile's global reads go out before the accumulator wait: the record's fp32
      // scales, and (mode 1) one column's token scale per thread into the shared table
      // (the previous tile's last named barrier has passed: no thread still reads it)
      const uint8_t* rec = t.shared ? p.shared : p.experts + size_t(t.g) * p.stride;
      const float* gl = reinterpret_cast<const float*>(rec + size_t(27) * p.F * p.L / 16);
      const float g0 = p.mode == 1 ? gl[0] : gl[2], g1 = gl[1];
      if (p.mode == 1) zbuf[te] = te < t.n_rows ? __ldg(&p.pos_inv[t.out0 + te]) : 1.0f;
      // uniform across the epilogue warps: all agree the accumulator is complete (this
      // barrier also publishes the token-scale table)
      ok = mbar_wait_abort(&acc_full[ab], (ti >> 1) & 1, p.err, p.abort);
      if (!named_and(1, kGgEpThreads, ok)) { ok = false; break; }
      tc_fence_after();
      const uint32_t tbase = tmem + (uint32_t(q * 32) << 16) + ab * 256 + ch * 16;
      const int tr = te >> 3, part = te & 7;
      for (int c = 0; c * 32 < t.n_rows; ++c) {
        uint32_t v[16];
        tmem_ld16(tbase + c * 32, v);
        tmem_ld_wait();
        const int col0 = ch * 16 + odd * 8;   // first token column this lane finishes
        if (p.mode == 1) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint32_t va = v[j], vb = v[8 + j];
            const float x = __uint_as_float(__shfl_xor_sync(0xFFFFFFFFu, odd ? va : vb, 1));
            const float gate = odd ? x : __uint_as_float(va);
            const float up = odd ? __uint_as_float(vb) : x;
            // undo the token's power-of-two scale of z (exact)
            const float zi = zbuf[c * 32 + col0 + j];
            hbuf[(col0 + j) * 72 + pr] = __float2bfloat16_rn(silu_gg(g0 * zi * gate) * (g1 * zi * up));
          }
          named_sync(1, kGgEpThreads);
          // 32 token rows x 64 f (128 B): 8 threads per row, 16 B each
          if (c * 32 + tr < t.n_rows) {
            const uint4* src = reinterpret_cast<const uint4*>(hbuf + tr * 72 + part * 8);
            uint4* dst = reinterpret_cast<uint4*>(p.out + size_t(t.out0 + c * 32 + tr) * p.out_ld + t.mt * 64 + part * 8);
            dst[0] = src[0];
          }
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint32_t va = v[j], vb = v[8 + j];
            const float x = __uint_as_float(__shfl_xor_sync(0xFFFFFFFFu, odd ? va : vb, 1));
            const float lo = odd ? x : __uint_as_float(va);            // latent row 2i
            const float hi = odd ? __uint_as_float(vb) : x;            // latent row 2i + 1
            const __nv_bfloat162 b = __floats2bfloat162_rn(g0 * lo, g0 * hi);
            obuf[(col0 + j) * 68 + pr] = *reinterpret_cast<const uint32_t*>(&b);
          }
          named_sync(1, kGgEpThreads);
          // 32 token rows x 128 latent rows (256 B): 8 threads per row, 32 B each
          if (c * 32 + tr < t.n_rows) {
            const uint4* src = reinterpret_cast<const uint4*>(obuf + tr * 68 + part * 8);
            uint4* dst =
                reinterpret_cast<uint4*>(p.out + size_t(t.out0 + c * 32 + tr) * p.out_ld + t.mt * 128 + part * 16);
            dst[0] = src[0];
            dst[1] = src[1];
          }
        }
        named_sync(1, kGgEpThreads);
      }
      // the accumulator's TMEM columns are free for the tile after next
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(accempty0 + uint32_t(ab) * 8u);
    }
  }
  if (!ok) s_flags[1] = 1;
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  // after a wait gave up, bulk copies issued by this CTA may still be landing:
  // give them a bounded time before the shared memory is released
  if (s_flags[1] && threadIdx.x == 0) {
    const unsigned long long t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 50000ull) {}
  }
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem, 512);
}

}  // namespace edge0
