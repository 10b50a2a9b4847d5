// The grouped NVFP4 GEMM kernel (types, tiling and warp roles in grouped.cuh).
// Included by one translation unit only.
#pragma once

#include "grouped.cuh"

namespace edge0 {

constexpr int kGgBBox = 64;       // rows of one B box (TMA)

// silu(v) = v / (1 + e^-v) with the hardware exponential and the fast division (the
// result is rounded to bf16, far coarser than their error); v -> -inf gives -0.
__device__ __forceinline__ float silu_gg(float v) { return __fdividef(v, 1.0f + __expf(-v)); }

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
      // ---- token producer: this CTA's 128 token rows of the tile (MMA rows 128 rank ..,
      // the M side), one k-slice per stage, completing on rank 0's barrier.  Boxes
      // wholly past the tile's rows are not loaded: those accumulator rows are never read
      const uint32_t bfull0 = mapa_shared(smem_u32(b_full), 0);
      int it = 0;
      for (int tile = pair; ok && tile < total; tile += npairs) {
        const GgTile t = gg_tile(p, tile, rank);
        const CUtensorMap* mb = (t.shared && p.mode == 1) ? &maps.b_shared : &maps.b_routed;
        const int mine = min(128, max(0, t.n_rows - 128 * rank));
        const int row0 = t.pos0 + rank * 128;
        const int nbox = (mine + kGgBBox - 1) / kGgBBox;
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
        // M = 256 token rows (128 per CTA), N = 256 weight rows (the two CTAs' tiles)
        const uint32_t idesc = p.mode == 1 ? idesc_f16_f32(256, 256) : idesc_bf16_f32(256, 256);
        (void)t;
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
            mma_pair_f16(acc, sw128_desc(sbb + k * 32), sw128_desc(sa + k * 32), idesc, (kb | k) != 0);
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
    // ---- epilogue: TMEM lane = token row 128 rank + lane of the pair tile.  Warp q =
    // warp % 4 reads lanes 32q .. 32q + 31, and half ch of the 256 columns: the weight
    // rows of CTA ch's tile (mode 1: columns 2i, 2i + 1 = gate, up of f = 64 mt + i;
    // mode 2: column i = latent row 128 mt + i), 32 columns per TMEM load.  Each
    // thread then stores its token's values as whole 16-byte pieces of its output row.
    const int q = warp & 3;
    const int ch = (warp - kGgEpWarp0) >> 2;
    const uint32_t accempty0 = mapa_shared(smem_u32(acc_empty), 0);
    int ti = 0;
    for (int tile = pair; ok && tile < total; tile += npairs, ++ti) {
      const GgTile t = gg_tile(p, tile, rank);
      const int ab = ti & 1;
      const int tok = 128 * rank + 32 * q + lane;
      const bool valid = tok < t.n_rows;
      const int mtc = t.mt - rank + ch;           // the weight tile whose columns this half holds
      // the tile's global reads go out before the accumulator wait: the record's fp32
      // scales (of CTA ch's expert: the pair shares the group) and this token's scale
      const uint8_t* rec = t.shared ? p.shared : p.experts + size_t(t.g) * p.stride;
      const float* gl = reinterpret_cast<const float*>(rec + size_t(27) * p.F * p.L / 16);
      const float g0 = p.mode == 1 ? gl[0] : gl[2], g1 = gl[1];
      const float zi = (p.mode == 1 && valid) ? __ldg(&p.pos_inv[t.out0 + tok]) : 1.0f;
      // uniform across the epilogue warps: all agree the accumulator is complete
      ok = mbar_wait_abort(&acc_full[ab], (ti >> 1) & 1, p.err, p.abort);
      if (!named_and(1, kGgEpThreads, ok)) { ok = false; break; }
      tc_fence_after();
      const uint32_t tbase = tmem + (uint32_t(q * 32) << 16) + ab * 256 + ch * 128;
      // this warp's 32 token rows go through a padded staging buffer (one row per
      // thread, written conflict-free), then out as row-contiguous 16-byte pieces
      uint8_t* stg = smem + GgSmem::offEpi + (warp - kGgEpWarp0) * 32 * GgSmem::kEpiPitch;
      const int tok0 = 128 * rank + 32 * q;          // the warp's first token row
      const int nvalid = min(32, max(0, t.n_rows - tok0));
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld32(tbase + c * 32, v);
        tmem_ld_wait();
        uint4* my = reinterpret_cast<uint4*>(stg + lane * GgSmem::kEpiPitch);
        if (p.mode == 1) {
          // 16 f values: f = 64 mtc + 16 c + i, gate in column 2i, up in 2i + 1
          uint32_t o[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float h0 = silu_gg(g0 * zi * __uint_as_float(v[4 * i])) * (g1 * zi * __uint_as_float(v[4 * i + 1]));
            const float h1 =
                silu_gg(g0 * zi * __uint_as_float(v[4 * i + 2])) * (g1 * zi * __uint_as_float(v[4 * i + 3]));
            const __nv_bfloat162 b = __floats2bfloat162_rn(h0, h1);
            o[i] = *reinterpret_cast<const uint32_t*>(&b);
          }
          my[0] = make_uint4(o[0], o[1], o[2], o[3]);
          my[1] = make_uint4(o[4], o[5], o[6], o[7]);
          __syncwarp();
          // 32 rows x 32 bytes: two threads per row
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int i = lane + 32 * k, r = i >> 1, pc = i & 1;
            if (r < nvalid) {
              const uint4 val = *reinterpret_cast<const uint4*>(stg + r * GgSmem::kEpiPitch + pc * 16);
              *reinterpret_cast<uint4*>(p.out + size_t(t.out0 + tok0 + r) * p.out_ld + 64 * mtc + 16 * c + 8 * pc) = val;
            }
          }
        } else {
          // 32 latent rows 128 mtc + 32 c + j
          uint32_t o[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const __nv_bfloat162 b =
                __floats2bfloat162_rn(g0 * __uint_as_float(v[2 * i]), g0 * __uint_as_float(v[2 * i + 1]));
            o[i] = *reinterpret_cast<const uint32_t*>(&b);
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) my[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
          __syncwarp();
          // 32 rows x 64 bytes: four threads per row
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int i = lane + 32 * k, r = i >> 2, pc = i & 3;
            if (r < nvalid) {
              const uint4 val = *reinterpret_cast<const uint4*>(stg + r * GgSmem::kEpiPitch + pc * 16);
              *reinterpret_cast<uint4*>(p.out + size_t(t.out0 + tok0 + r) * p.out_ld + 128 * mtc + 32 * c + 8 * pc) = val;
            }
          }
        }
        __syncwarp();   // the staging rows are rewritten by the next chunk
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
