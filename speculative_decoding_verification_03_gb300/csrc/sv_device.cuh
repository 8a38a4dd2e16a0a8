// Device building blocks for the sm_103a kernels: Philox4x32-10, mbarrier
// and bulk-copy (TMA, non-tensor) wrappers written as inline PTX, bounded
// waits, and small numeric helpers.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "specverify.h"

namespace sv {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr double kLn2d = 0.6931471805599453094;
constexpr double kLog2ed = 1.4426950408889634074;

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As
// Easy as 1, 2, 3", SC'11).  Each round multiplies counter words 0 and 2 by
// the two round constants, mixes the high halves with words 1 and 3 and the
// key, and the key advances by the two Weyl increments between rounds.
// ---------------------------------------------------------------------------
struct U32x4 {
  uint32_t w[4];
};

__device__ __forceinline__ U32x4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                               uint32_t k0, uint32_t k1) {
  constexpr uint32_t kMulA = 0xD2511F53u, kMulB = 0xCD9E8D57u;
  constexpr uint32_t kWeylA = 0x9E3779B9u, kWeylB = 0xBB67AE85u;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t hiA = __umulhi(kMulA, c0), loA = kMulA * c0;
    const uint32_t hiB = __umulhi(kMulB, c2), loB = kMulB * c2;
    const uint32_t n0 = hiB ^ c1 ^ k0;
    const uint32_t n2 = hiA ^ c3 ^ k1;
    c0 = n0;
    c1 = loB;
    c2 = n2;
    c3 = loA;
    k0 += kWeylA;
    k1 += kWeylB;
  }
  U32x4 out;
  out.w[0] = c0;
  out.w[1] = c1;
  out.w[2] = c2;
  out.w[3] = c3;
  return out;
}

// Uniform for (seed, sequence b, position pos): word `draw` of the block with
// counter (b, pos, 0, 0); the top 24 bits scaled by 2^-24 (exact in fp32).
// Draw 0 = acceptance, draw 1 = residual/bonus sampling.
__device__ __forceinline__ float uniform24f(uint64_t seed, uint32_t b, uint32_t pos, int draw) {
  const U32x4 r = philox4x32_10(b, pos, 0u, 0u, (uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32));
  return (float)(r.w[draw & 3] >> 8) * (1.0f / 16777216.0f);
}

// ---------------------------------------------------------------------------
// Timers and bounded waits.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait with a suspend-time hint: a warp whose phase is not complete
// sleeps in hardware (up to hint_ns) instead of spinning on issue slots.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Wait until the phase with the given parity of `bar` has completed, for at
// most limit_ns.  On time-out (or when another thread of the CTA already
// gave up) the CTA-wide abort flag is set, the status word gets
// SV_FLAG_TIMEOUT and false is returned.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                                  uint32_t* status, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if (*abort_flag) return false;
    if (global_ns() - t0 > limit_ns) {
      *abort_flag = 1;
      atomicOr(status, SV_FLAG_TIMEOUT);
      return false;
    }
  }
}

// GPU-scope relaxed store / acquire load of a 32-bit queue entry.
__device__ __forceinline__ void st_relaxed_gpu(int* p, int v) {
  asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// 1-D bulk copy global -> shared (TMA engine, no tensor map), completing on
// `bar` with `bytes` of transaction count.  Both addresses 16-byte aligned,
// bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// An L2 policy that marks the lines a copy brings in as the first to evict:
// for streams read once (or re-read only long after), so that they do not
// push out of L2 what is re-read soon.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// bulk_g2s with an L2 cache policy for the lines it reads
__device__ __forceinline__ void bulk_g2s_hint(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar,
                                              uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
          "r"(smem_addr(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
      : "memory");
}

// ---------------------------------------------------------------------------
// Numerics.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Kahan's compensated addition s += v: cmp holds the low-order part that the
// previous addition lost (the sum is s - cmp), so a thread's sum of many
// positive terms keeps fp32 precision however long the row (terms below half
// an ulp of a plain running sum would be rounded away one by one).
__device__ __forceinline__ void kahan_add(float &s, float &cmp, float v) {
  const float y = __fsub_rn(v, cmp);
  const float t = __fadd_rn(s, y);
  cmp = __fsub_rn(__fsub_rn(t, s), y);
  s = t;
}

// bf16 pair packed in a 32-bit word -> two fp32 values (exact widening).
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Element-wise max of two packed bf16 pairs (NaN-ignoring).
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Warp max in one instruction (redux.sync on f32, NaN inputs ignored as by
// fmaxf; -0 and +0 compare equal).
__device__ __forceinline__ float warp_max(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ int warp_min_i(int v) { return __reduce_min_sync(0xffffffffu, v); }

}  // namespace sv
