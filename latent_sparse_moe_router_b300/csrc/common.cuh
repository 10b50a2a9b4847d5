// Shared device helpers for the latent-MoE kernels (sm_103a): bulk-copy / mbarrier
// wrappers, bounded waits, a software grid barrier, and NVFP4 element decoding.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace edge0 {

// Device error word bits (the handle's error word).
constexpr int kErrTimeout = 1;

// Limit of every device-side spin wait, in nanoseconds of %globaltimer.
constexpr unsigned long long kWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Arrive once and add `bytes` to the expected transaction count of the current phase.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
               ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.  Returns false
// (after recording a timeout in *err) if the limit ran out.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicOr(err, kErrTimeout);
      return false;
    }
  }
  return true;
}

// The same wait with the thread suspended in the barrier between polls (up to
// `sleep_ns` each; it resumes when the phase completes), so that waiting warps leave
// the issue slots to the working ones.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t sleep_ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity), "r"(sleep_ns) : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* bar, uint32_t parity, int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait_sleep(bar, parity, 1000u)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicOr(err, kErrTimeout);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ int ld_relaxed_s32(const int* p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Bounded wait for grids of many CTAs.  Gives up at once when *abort (if given)
// is non-zero, so that one CTA's timeout ends the waits of every other CTA
// within microseconds; on running out of time it ORs kErrTimeout into *err (if
// given) and sets *abort.  Returns false if it gave up.
__device__ __forceinline__ bool mbar_wait_abort(uint64_t* bar, uint32_t parity, int* err, int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  unsigned int spins = 0;
  while (!mbar_try_wait(bar, parity)) {
    if ((++spins & 63u) == 0) {
      if (abort && ld_relaxed_s32(abort)) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        if (err) atomicOr(err, kErrTimeout);
        if (abort) atomicExch(abort, 1);
        return false;
      }
    }
  }
  return true;
}

// ---------------------------------------------------------------- bulk copies
// Global -> shared bulk copy (TMA, non-tensor), completion counted on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
// 16 bytes global -> shared without a register round trip (completion: cp_async_wait_all).
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

// Same, with an L2 eviction-priority policy (from createpolicy).
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;"
      ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Bulk prefetch of a global range into L2 (16-byte aligned, multiple of 16 bytes).
__device__ __forceinline__ void l2_prefetch(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Prefetch [base, base+bytes) into L2, the part this CTA owns when the range is
// split evenly over `parts` CTAs in 16-byte granules; pieces of at most 64 KB.
__device__ __forceinline__ void l2_prefetch_share(const void* base, size_t bytes, int part,
                                                  int parts) {
  const size_t gran = bytes / 16;
  size_t a = gran * part / parts * 16, b = gran * (part + 1) / parts * 16;
  if (part == parts - 1) b = bytes & ~size_t(15);
  const char* p = static_cast<const char*>(base);
  while (a < b) {
    uint32_t n = static_cast<uint32_t>((b - a) > 65536 ? 65536 : (b - a));
    l2_prefetch(p + a, n);
    a += n;
  }
}

// ---------------------------------------------------------------- grid barrier
// Ticket barrier over all CTAs of a co-resident (cooperative) grid.  Every
// barrier adds exactly gridDim.x to `ticket`; a CTA's arrival returns its ticket
// and it waits until the counter reaches the end of that round.  The counter
// never resets between launches (it stays a multiple of the grid size), so
// nothing needs clearing before a launch.  An aborted launch leaves it in the
// middle of a round: the host must zero the struct before the next launch.
struct GridBarrier {
  unsigned long long ticket;
  unsigned int abort;
  unsigned int pad[13];
};

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned int ld_relaxed_u32(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// All threads of every CTA call this.  Returns false if the barrier was
// aborted (some CTA's wait ran out); the error word then holds kErrTimeout.
__device__ __forceinline__ bool grid_sync(GridBarrier* bar, int* err) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    unsigned long long tk;
    // acquire-release: the CTA that arrives last sees every other arrival in the
    // value it gets back and needs no further load; the others poll with acquire
    // loads, the one that sees the round complete ordering this CTA after every
    // other CTA's release (its arrival); the __syncthreads below passes that on
    asm volatile("atom.add.acq_rel.gpu.global.u64 %0, [%1], 1;" : "=l"(tk) : "l"(&bar->ticket) : "memory");
    const unsigned long long target = (tk / gridDim.x + 1) * gridDim.x;
    if (tk + 1 != target && ld_acquire_u64(&bar->ticket) < target) {
      const unsigned long long t0 = globaltimer_ns();
      unsigned int spins = 0;
      while (ld_acquire_u64(&bar->ticket) < target) {
        if ((++spins & 31u) == 0) {
          if (ld_relaxed_u32(&bar->abort)) { ok = 0; break; }
          if (globaltimer_ns() - t0 > kWaitLimitNs) {
            atomicOr(err, kErrTimeout);
            atomicExch(&bar->abort, 1u);
            ok = 0;
            break;
          }
        }
      }
    }
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

// ---------------------------------------------------------------- residual RMSNorm
// The library's one summation order for sum((x + y)^2) over a token row (bf16 inputs,
// fp32 sums), shared by the stacked decode kernel and the standalone kernel:
//   group_sumsq: the 8 squares of one 16-byte group, fmaf in element order from 0;
//   the group sums of a row are added by lane l = g mod 32 in increasing g;
//   the 32 lane sums meet in an xor tree.  H % 8 == 0.
__device__ __forceinline__ float group_sumsq(uint4 a, uint4 b) {
  const uint32_t aa[4] = {a.x, a.y, a.z, a.w}, bb[4] = {b.x, b.y, b.z, b.w};
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float v0 = __uint_as_float(aa[i] << 16) + __uint_as_float(bb[i] << 16);
    const float v1 = __uint_as_float(aa[i] & 0xFFFF0000u) + __uint_as_float(bb[i] & 0xFFFF0000u);
    s = fmaf(v0, v0, s);
    s = fmaf(v1, v1, s);
  }
  return s;
}

// One row by one warp (loads of four groups in flight together).
__device__ __forceinline__ float row_sumsq_warp(const __nv_bfloat16* x, const __nv_bfloat16* y, int H, int lane) {
  float s = 0.f;
  const uint4* xv = reinterpret_cast<const uint4*>(x);
  const uint4* yv = reinterpret_cast<const uint4*>(y);
  const int ng = H / 8;
  for (int g0 = lane; g0 < ng; g0 += 4 * 32) {
    uint4 a[4], b[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int g = g0 + 32 * j;
      a[j] = g < ng ? xv[g] : make_uint4(0u, 0u, 0u, 0u);
      b[j] = g < ng ? yv[g] : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (g0 + 32 * j < ng) s += group_sumsq(a[j], b[j]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return s;
}

// ---------------------------------------------------------------- NVFP4 decode
// Two E2M1 codes (one byte, low nibble first) -> half2 (x = low, y = high).
__device__ __forceinline__ uint32_t e2m1x2_to_h2(uint32_t byte) {
  uint32_t r;
  asm("{\n .reg .b8 b;\n cvt.u8.u32 b, %1;\n cvt.rn.f16x2.e2m1x2 %0, b;\n}\n"
      : "=r"(r) : "r"(byte));
  return r;
}

// E4M3FN byte -> float (exact).
__device__ __forceinline__ float e4m3_to_f32(uint32_t byte) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<unsigned short>(byte & 0xFF)));
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFF)));
}

// Four E2M1 pairs (one 32-bit word, byte i = elements 2i, 2i+1, low nibble first)
// -> four f16x2.
__device__ __forceinline__ void e2m1x8_to_h2x4(uint32_t w, uint32_t& h0, uint32_t& h1, uint32_t& h2,
                                               uint32_t& h3) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}\n"
      : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3) : "r"(w));
}

// f16x2 (both halves) of an E4M3 scale (exact).
__device__ __forceinline__ uint32_t scale_f16x2(uint32_t e4m3) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(static_cast<unsigned short>(e4m3 | (e4m3 << 8))));
  return r;
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

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

// D += A B (m16n8k16, f16 inputs, fp32 accumulate), warp-wide.  Fragments per
// thread (g = lane / 4, c = lane % 4): a0 (row g, k 2c, 2c+1), a1 (row g + 8, same
// k), a2 (row g, k 2c + 8, 2c + 9), a3 (row g + 8, same); b0 (k 2c, 2c+1, column g),
// b1 (k 2c + 8, 2c + 9, column g); d0, d1 (row g, columns 2c, 2c + 1), d2, d3 (row
// g + 8, same columns).  The lower-indexed element of a pair sits in the low half.
__device__ __forceinline__ void mma16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The same MMA with bf16 inputs.
__device__ __forceinline__ void mma16816_bf16(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ __half2 u32_as_h2(uint32_t v) {
  return *reinterpret_cast<__half2*>(&v);
}

}  // namespace edge0
