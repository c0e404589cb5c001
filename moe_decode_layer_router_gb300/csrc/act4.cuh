// FP4 rounding shared by the online weight rounding and the W4A4 expert
// inputs.
//
// MXFP4 (OCP MX; page "vllm.models.muse_spark.amd.muse_moe_runner": the
// online rounding of BF16 experts and the Quark w_mxfp4_a_mxfp4 scheme with
// dynamic MXFP4 activations): per 32 consecutive elements the scale is
// 2^(floor(log2 amax) - 2), its exponent clamped to [-126, 127], 2^0 for an
// all-zero block.
// NVFP4 (providers page, ExpertsInput: e2m1 codes with one e4m3 block scale
// per 16 and no global scale): the scale is the e4m3 value nearest
// fp32(amax / 6), ties to even, saturating at 448.
// Each element then takes the e2m1 magnitude nearest |v| / scale (the
// quotient exact for MXFP4, an IEEE fp32 quotient for NVFP4), ties to the
// even code, saturating at 6, with the sign bit of v; an NVFP4 block whose
// scale is 0 takes magnitude 0.
#pragma once
#include "common.cuh"

namespace musemoe {

// round to nearest on {0, .5, 1, 1.5, 2, 3, 4, 6}, ties to the even code
// (the weight rounding's form, one element at a time)
__device__ __forceinline__ uint32_t e2m1_nearest(float a) {
  return a <= 0.25f ? 0u
       : a < 0.75f  ? 1u
       : a <= 1.25f ? 2u
       : a < 1.75f  ? 3u
       : a <= 2.5f  ? 4u
       : a < 3.5f   ? 5u
       : a <= 5.0f  ? 6u
                    : 7u;
}

// floor(log2(m)) of a finite positive fp32 (subnormals included)
__device__ __forceinline__ int floor_log2_f32(float m) {
  const uint32_t b = __float_as_uint(m);
  const int ef = (int)(b >> 23);
  return ef > 0 ? ef - 127 : (31 - __clz((int)b)) - 149;
}

// MXFP4 scale exponent of a block with amax m (m a bf16 value, so the
// exponent stays within [-126, 125] and 2^-e is a normal fp32)
__device__ __forceinline__ int mx_scale_exp(float m) {
  const int e = m > 0.f ? floor_log2_f32(m) - 2 : 0;
  return min(max(e, -126), 127);
}

// NVFP4 block scale code (e4m3) of a block with amax m
__device__ __forceinline__ uint32_t nv_scale_code(float m) {
  return f32x2_to_e4m3x2(__fdiv_rn(m, 6.0f), 0.f) & 0xFFu;
}

__device__ __forceinline__ float e4m3_to_f32(uint32_t code) {
  const uint32_t h2 = e4m3x2_to_f16x2(code);
  return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

// One block's scale in the form the element rounding wants.
struct Fp4Scale {
  float scale;  // the block scale (2^e or the e4m3 value)
  float inv;    // MXFP4: 2^-e (exact); NVFP4: unused
};

// mode 1: MXFP4, mode 2: NVFP4
__device__ __forceinline__ Fp4Scale fp4_block_scale(float amax, int mode) {
  Fp4Scale s;
  if (mode == 1) {
    const int e = mx_scale_exp(amax);
    s.scale = __int_as_float((e + 127) << 23);
    s.inv = __int_as_float((127 - e) << 23);
  } else {
    s.scale = e4m3_to_f32(nv_scale_code(amax));
    s.inv = 0.f;
  }
  return s;
}

// Two non-negative fp32 -> two e2m1 magnitude codes, `lo` in the low nibble:
// the hardware conversion rounds to nearest, ties to the even code, and
// saturates at 6, the rule above.
__device__ __forceinline__ uint32_t f32x2_to_e2m1x2(float lo, float hi) {
  uint16_t r;
  asm("{\n .reg .b8 b;\n cvt.rn.satfinite.e2m1x2.f32 b, %1, %2;\n cvt.u16.u8 %0, b;\n}\n"
      : "=h"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// The codes of v0, v1 in a block with scale s as one byte (v0 in the low
// nibble, sign in bit 3 of each nibble): the magnitudes of |v| / s (an exact
// product for MXFP4, an IEEE fp32 quotient for NVFP4) from the hardware
// conversion, the sign bits of v set explicitly.
__device__ __forceinline__ uint32_t fp4_code2(float v0, float v1, const Fp4Scale& s, int mode) {
  float a0 = 0.f, a1 = 0.f;
  if (mode == 1) {
    a0 = fabsf(v0) * s.inv;
    a1 = fabsf(v1) * s.inv;
  } else if (s.scale > 0.f) {
    a0 = __fdiv_rn(fabsf(v0), s.scale);
    a1 = __fdiv_rn(fabsf(v1), s.scale);
  }
  return (f32x2_to_e2m1x2(a0, a1) & 0x77u) | ((__float_as_uint(v0) >> 31) << 3) |
         ((__float_as_uint(v1) >> 31) << 7);
}

// the values of a byte of two codes (exact in fp32)
__device__ __forceinline__ void fp4_value2(uint32_t byte, const Fp4Scale& s, float& r0, float& r1) {
  const uint32_t h2 = e2m1x2_to_f16x2(byte);
  r0 = __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu))) * s.scale;
  r1 = __half2float(__ushort_as_half((unsigned short)(h2 >> 16))) * s.scale;
}

}  // namespace musemoe
