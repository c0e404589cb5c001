// Shared-memory pipeline helpers of the expert kernels (sm_103a): mbarrier
// waits with a time limit, 1-D bulk copies (cp.async.bulk, the TMA engine)
// into shared memory, and the dequantize + mma.sync work of one 64-byte
// chunk of two fragment rows.
#pragma once
#include "common.cuh"
#include "kernels.h"

namespace musemoe {

constexpr unsigned long long kWaitLimitNs = 200ull * 1000 * 1000;

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;\n" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, int count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes)
               : "memory");
}
// One bounded sleep on the mbarrier phase: the thread is woken when the phase
// completes, or after about kSuspendNs.
constexpr uint32_t kSuspendNs = 20000;
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t phase) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(phase), "r"(kSuspendNs)
      : "memory");
  return ok != 0;
}
// Whether the mbarrier phase has completed (never blocks).
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t phase) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(phase)
      : "memory");
  return ok != 0;
}
// Waits for the mbarrier phase to complete, at most `limit_ns`.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t phase,
                                          unsigned long long limit_ns) {
  if (mbar_try_wait(bar, phase)) return true;
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(bar, phase))
    if (globaltimer() - t0 > limit_ns) return false;
  return true;
}
// 1-D bulk copy global -> shared, completion counted on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// L2 cache policy for data read once: evicted before normal-priority lines.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(pol));
  return pol;
}
// 1-D bulk copy global -> shared with an L2 cache policy.
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;\n" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(pol)
      : "memory");
}
// The mma work of one 64-byte chunk of the fragment rows g (codes L, scales
// sl) and g + 8 (codes H, scales sh) against the n-tiles' B fragments, which
// `bfrag(nt, j)` returns: for FP4 the uint2 of k-step j (0..7), for BF16 the
// uint2 of k-step j (0..1), for FP8 the uint4 of both k-steps (j unused).
template <int Q, int NT, typename BFrag>
__device__ __forceinline__ void chunk_mma(float (&acc)[NT][4], const uint4& L, const uint4& H,
                                          uint2 sl, uint2 sh, int ntile_act, BFrag&& bfrag) {
  if constexpr (Q == kFP8) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      if (nt >= ntile_act) break;
      const uint4 bv = bfrag(nt, 0);
      mma_e4m3_16832(acc[nt], L.x, H.x, L.y, H.y, bv.x, bv.y);
      mma_e4m3_16832(acc[nt], L.z, H.z, L.w, H.w, bv.z, bv.w);
    }
  } else if constexpr (Q == kBF16) {
    // bf16 codes as stored (the pack transposes a chunk's 4-byte words so
    // that L / H are rows g / g + 8 at k 2q, 2q + 8 of k-step 0, then k-step 1)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      if (nt >= ntile_act) break;
      const uint2 b0 = bfrag(nt, 0), b1 = bfrag(nt, 1);
      mma_bf16_16816(acc[nt], L.x, H.x, L.y, H.y, b0.x, b0.y);
      mma_bf16_16816(acc[nt], L.z, H.z, L.w, H.w, b1.x, b1.y);
    }
  } else if constexpr (Q == kMXFP4) {
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const float fl = ue8m0_byte_to_f32(sl.x, b);
      const float fh = ue8m0_byte_to_f32(sh.x, b);
      uint32_t a00, a02, a10, a12, a01, a03, a11, a13;
      e2m1x8_to_f16x2x4(word_of(L, b), a00, a02, a10, a12);
      e2m1x8_to_f16x2x4(word_of(H, b), a01, a03, a11, a13);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        if (nt >= ntile_act) break;
        const uint2 b0 = bfrag(nt, 2 * b), b1 = bfrag(nt, 2 * b + 1);
        float t[4];
        mma_f16_16816_zc(t, a00, a01, a02, a03, b0.x, b0.y);
        mma_f16_16816(t, a10, a11, a12, a13, b1.x, b1.y);
        acc[nt][0] = fmaf(t[0], fl, acc[nt][0]);
        acc[nt][1] = fmaf(t[1], fl, acc[nt][1]);
        acc[nt][2] = fmaf(t[2], fh, acc[nt][2]);
        acc[nt][3] = fmaf(t[3], fh, acc[nt][3]);
      }
    }
  } else {  // NVFP4: one e4m3 scale per k-step
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t slw = (j < 4 ? sl.x : sl.y) >> (8 * (j & 3));
      const uint32_t shw = (j < 4 ? sh.x : sh.y) >> (8 * (j & 3));
      const uint32_t sfl = e4m3x2_to_f16x2(slw & 0xFFu);
      const uint32_t sfh = e4m3x2_to_f16x2(shw & 0xFFu);
      const uint32_t sl2 = __byte_perm(sfl, sfl, 0x1010);  // broadcast low half
      const uint32_t sh2 = __byte_perm(sfh, sfh, 0x1010);
      uint32_t l0, l1, l2, l3, h0, h1, h2, h3;
      e2m1x8_to_f16x2x4(word_of(L, j >> 1), l0, l1, l2, l3);
      e2m1x8_to_f16x2x4(word_of(H, j >> 1), h0, h1, h2, h3);
      const uint32_t a0 = hmul2((j & 1) ? l2 : l0, sl2);
      const uint32_t a1 = hmul2((j & 1) ? h2 : h0, sh2);
      const uint32_t a2 = hmul2((j & 1) ? l3 : l1, sl2);
      const uint32_t a3 = hmul2((j & 1) ? h3 : h1, sh2);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        if (nt >= ntile_act) break;
        const uint2 bv = bfrag(nt, j);
        mma_f16_16816(acc[nt], a0, a1, a2, a3, bv.x, bv.y);
      }
    }
  }
}

// Waits for the mbarrier phase, at most `limit_ns`; gives up early when
// another warp of the CTA has aborted. False when it did not complete.
__device__ __forceinline__ bool mbar_wait_or_abort(uint32_t bar, uint32_t phase,
                                                   volatile int* abort_flag) {
  if (mbar_try_wait(bar, phase)) return true;
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(bar, phase)) {
    if (*abort_flag) return false;
    if (globaltimer() - t0 > kWaitLimitNs) return false;
  }
  return true;
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}

}  // namespace musemoe
