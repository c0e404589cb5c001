// Online rounding of BF16 expert weights to MXFP4 on load (page
// "vllm.models.muse_spark.amd.muse_moe_runner", _quantize_experts_to_mxfp4;
// every decoder layer but the first and the last, _online_mxfp4_applies).
//
// The page names OCP MXFP4 and a library routine but prints no formula; the
// plain OCP MX reading: per block of 32 consecutive elements of a row, the
// shared scale is 2^(floor(log2(amax)) - 2) (2 = the largest e2m1 exponent,
// so amax / scale lies in [4, 8)), its exponent clamped to [-126, 127] (the
// UE8M0 codes 1..254 the kernel layout accepts), 2^0 for an all-zero block;
// each element becomes the e2m1 magnitude nearest |v| / scale, ties to the
// even code, saturating at 6, with the sign bit of v. Inputs are finite.
//
// Each lane rounds 8 consecutive elements (one 16-byte load); the 4 lanes of
// a block take its amax with two shuffles on the bf16 magnitude bits, which
// order like unsigned integers, so the scale needs no floating point.
//
// Also here: the NVFP4 expert input of the W4A4 form (codes and e4m3 block
// scales, the rule in act4.cuh).
#include "act4.cuh"
#include "kernels.h"

namespace musemoe {

constexpr int kQuantThreads = 256;

// The 8 elements of one lane: amax over its block's 4 lanes, scale, codes.
__device__ __forceinline__ void quant8(const uint4& v, long long i, bool ok, int lane,
                                       uint8_t* codes, uint8_t* scales) {
  const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
  uint32_t m = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) m = max(m, max(wd[j] & 0x7FFFu, (wd[j] >> 16) & 0x7FFFu));
  m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
  m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
  // floor(log2(amax)) from the bits: normal exponent field - 127, or the top
  // mantissa bit of a subnormal (value mantissa * 2^-133)
  const int ef = (int)(m >> 7);
  const int fl = ef > 0 ? ef - 127 : (31 - __clz((int)m)) - 133;
  int e = m == 0 ? 0 : fl - 2;
  e = min(max(e, -126), 127);
  const float inv = __int_as_float((127 - e) << 23);  // 2^-e (e <= 125 for finite bf16)
  uint32_t packed = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t h = (j & 1) ? (wd[j >> 1] >> 16) : (wd[j >> 1] & 0xFFFFu);
    const float a = fabsf(__uint_as_float(h << 16)) * inv;  // exact: a power of two
    const uint32_t c = e2m1_nearest(a) | ((h >> 15) << 3);
    packed |= c << (4 * j);
  }
  if (ok) {
    reinterpret_cast<uint32_t*>(codes)[i] = packed;
    if ((lane & 3) == 0) scales[i >> 2] = (uint8_t)(e + 127);
  }
}

__global__ void __launch_bounds__(kQuantThreads) k_quant_mxfp4(const uint16_t* w, uint8_t* codes,
                                                              uint8_t* scales, long long n8) {
  const int lane = threadIdx.x & 31;
  const long long stride = (long long)gridDim.x * kQuantThreads;
  // the warp walks together (its shuffles need every lane); n8 is a
  // multiple of 4, so a block's 4 lanes are all in range or all out
  for (long long base = (long long)blockIdx.x * kQuantThreads + (threadIdx.x & ~31); base < n8;
       base += stride) {
    const long long i = base + lane;
    const uint4 v = i < n8 ? __ldg(reinterpret_cast<const uint4*>(w) + i) : make_uint4(0, 0, 0, 0);
    quant8(v, i, i < n8, lane, codes, scales);
  }
}

cudaError_t launch_quant_mxfp4(const uint16_t* w, uint8_t* codes, uint8_t* scales,
                               long long elements, int sms, cudaStream_t s) {
  const long long n8 = elements / 8;
  long long grid = (n8 + kQuantThreads - 1) / kQuantThreads;
  grid = grid < (long long)sms * 16 ? grid : (long long)sms * 16;
  if (grid < 1) grid = 1;
  k_quant_mxfp4<<<(unsigned)grid, kQuantThreads, 0, s>>>(w, codes, scales, n8);
  return cudaGetLastError();
}

// The NVFP4 expert input (providers page, ExpertsInput): bf16 activations
// [rows, cols] -> e2m1 codes [rows, cols/2] (element 2j in the low nibble of
// byte j) and one e4m3 block scale per 16 elements [rows, cols/16]. Each
// lane rounds 8 consecutive elements (one 16-byte load); the 2 lanes of a
// block take its amax with one shuffle.
__global__ void __launch_bounds__(kQuantThreads) k_quant_act_nvfp4(const uint16_t* x, uint8_t* codes,
                                                                  uint8_t* scales, long long n8) {
  const int lane = threadIdx.x & 31;
  const long long stride = (long long)gridDim.x * kQuantThreads;
  // n8 is even, so the 2 lanes of a block are both in range or both out
  for (long long base = (long long)blockIdx.x * kQuantThreads + (threadIdx.x & ~31); base < n8;
       base += stride) {
    const long long i = base + lane;
    const uint4 v = i < n8 ? __ldg(reinterpret_cast<const uint4*>(x) + i) : make_uint4(0, 0, 0, 0);
    const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
    float f[8];
    float m = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      f[j] = bf16_bits_to_f32((j & 1) ? (wd[j >> 1] >> 16) : (wd[j >> 1] & 0xFFFFu));
      m = fmaxf(m, fabsf(f[j]));
    }
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    const uint32_t sc = nv_scale_code(m);
    Fp4Scale s;
    s.scale = e4m3_to_f32(sc);
    s.inv = 0.f;
    uint32_t packed = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) packed |= fp4_code2(f[2 * j], f[2 * j + 1], s, 2) << (8 * j);
    if (i < n8) {
      reinterpret_cast<uint32_t*>(codes)[i] = packed;
      if ((lane & 1) == 0) scales[i >> 1] = (uint8_t)sc;
    }
  }
}

cudaError_t launch_quant_act_nvfp4(const uint16_t* x, uint8_t* codes, uint8_t* scales,
                                   long long elements, int sms, cudaStream_t s) {
  const long long n8 = elements / 8;
  long long grid = (n8 + kQuantThreads - 1) / kQuantThreads;
  grid = grid < (long long)sms * 16 ? grid : (long long)sms * 16;
  if (grid < 1) grid = 1;
  k_quant_act_nvfp4<<<(unsigned)grid, kQuantThreads, 0, s>>>(x, codes, scales, n8);
  return cudaGetLastError();
}

}  // namespace musemoe
