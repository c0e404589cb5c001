// Tail of the expert phase: the FP8 per-route requantization of the bf16
// activation between w13 and w2, and the per-route post-expert norm, router
// weighting and sum over the k routes of each token.
#include <algorithm>

#include "act4.cuh"
#include "common.cuh"
#include "kernels.h"
#include "pipeline.cuh"

namespace musemoe {

// ---- health self-test -----------------------------------------------------
// The library's two bounded waits, each on something nothing completes: an
// mbarrier phase (as a stage whose copies never land) and a flag (as a split
// tile's owner waiting for a partial that never comes). Each gives up after
// kWaitLimitNs and records the timeout in the health word, as a forward
// would; no copy is in flight, so the CTA leaves cleanly.
__global__ void k_wait_selftest(int32_t* health, const int32_t* never) {
  __shared__ __align__(8) unsigned long long bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x != 0) return;
  if (!mbar_wait_or_abort(smem_u32(&bar), 0u, &abort_flag)) atomicOr(health, kHealthTimeout);
  int v = 0;
  const unsigned long long t0 = globaltimer();
  do {
    __nanosleep(256);
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];\n" : "=r"(v) : "l"(never) : "memory");
  } while (v == 0 && globaltimer() - t0 <= kWaitLimitNs);
  if (v == 0) atomicOr(health, kHealthTimeout);
}

cudaError_t launch_wait_selftest(int32_t* health, const int32_t* never, cudaStream_t s) {
  k_wait_selftest<<<1, 32, 0, s>>>(health, never);
  return cudaGetLastError();
}

// ---- FP8: per-route dynamic quantization of the bf16 activation ------------
__global__ void __launch_bounds__(256) k_act_quant(ActQuantParams p) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (r >= p.routes) return;
  const uint16_t* a = p.act + (size_t)r * p.I;
  float amax = 0.f;
  for (int i = lane * 2; i < p.I; i += 64) {
    const uint32_t v = __ldcg(reinterpret_cast<const unsigned int*>(a + i));
    amax = fmaxf(amax, fmaxf(fabsf(bf16_bits_to_f32(v & 0xFFFFu)), fabsf(bf16_bits_to_f32(v >> 16))));
  }
  amax = warp_max(amax);
  const float s = amax / 448.0f;
  for (int i = lane * 2; i < p.I; i += 64) {
    const uint32_t v = __ldcg(reinterpret_cast<const unsigned int*>(a + i));
    const float x0 = bf16_bits_to_f32(v & 0xFFFFu), x1 = bf16_bits_to_f32(v >> 16);
    const uint16_t qv = f32x2_to_e4m3x2(s > 0.f ? x0 / s : 0.f, s > 0.f ? x1 / s : 0.f);
    reinterpret_cast<uint16_t*>(p.q + (size_t)r * p.I)[i / 2] = qv;
  }
  if (lane == 0) p.scale[r] = s;
}

// ---- W4A4: per-route FP4 rounding of the bf16 activation ------------------
// (page "vllm.models.muse_spark.amd.muse_moe_runner": the Quark
// w_mxfp4_a_mxfp4 scheme rounds the expert inputs to MXFP4 dynamically;
// providers page, ExpertsInput: the NVFP4 form). One warp per 256 elements
// of a route (I is a multiple of 128, so a warp's span is whole blocks); a
// lane rounds 8 consecutive elements (one 16-byte load), so a block is 4
// (MXFP4) or 2 (NVFP4) neighbouring lanes, the first of which stores the
// block's scale. Output: w2's operand, e2m1 codes [routes, I / 2] (the lower
// element of a pair in the low nibble) and one scale byte per block
// [routes, I / blk] (UE8M0 / e4m3); a value that is not finite raises
// kHealthActRange.
constexpr int kActSpan = 256;

template <int MODE>  // 1 MXFP4, 2 NVFP4
__global__ void __launch_bounds__(256) k_act_fp4(ActQuantParams p) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int spans = (p.I + kActSpan - 1) / kActSpan;
  const int wid = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (wid >= p.routes * spans) return;  // the whole warp
  const int r = wid / spans;
  const int i = (wid - r * spans) * kActSpan + lane * 8;
  const bool ok = i < p.I;
  const uint4 v = ok ? __ldcg(reinterpret_cast<const uint4*>(p.act + (size_t)r * p.I + i))
                     : make_uint4(0, 0, 0, 0);
  const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
  float x[8];
  float m = 0.f;
  int bad = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    x[j] = bf16_bits_to_f32((j & 1) ? (wd[j >> 1] >> 16) : (wd[j >> 1] & 0xFFFFu));
    m = fmaxf(m, fabsf(x[j]));
    bad |= !(fabsf(x[j]) <= 3.40282347e38f);  // NaN or infinite (above FLT_MAX)
  }
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
  if (MODE == 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
  const Fp4Scale sc = fp4_block_scale(m, MODE);
  uint32_t codes = 0;
#pragma unroll
  for (int c = 0; c < 4; ++c) codes |= fp4_code2(x[2 * c], x[2 * c + 1], sc, MODE) << (8 * c);
  if (ok) {
    reinterpret_cast<uint32_t*>(p.q + (size_t)r * (p.I >> 1))[i >> 3] = codes;
    constexpr int kSh = MODE == 1 ? 5 : 4;  // log2 of the elements per block
    if ((i & ((1 << kSh) - 1)) == 0)
      p.sf[(size_t)r * (p.I >> kSh) + (i >> kSh)] =
          (uint8_t)(MODE == 1 ? (uint32_t)(mx_scale_exp(m) + 127) : nv_scale_code(m));
  }
  if (bad) atomicOr(p.health, kHealthActRange);
}

cudaError_t launch_act_quant(const ActQuantParams& p, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = p.mode ? dim3((p.routes * ((p.I + kActSpan - 1) / kActSpan) + 7) / 8)
                       : dim3((p.routes + 7) / 8);
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (p.mode == 1) return cudaLaunchKernelEx(&cfg, k_act_fp4<1>, p);
  if (p.mode == 2) return cudaLaunchKernelEx(&cfg, k_act_fp4<2>, p);
  return cudaLaunchKernelEx(&cfg, k_act_quant, p);
}

// ---- tail: post-expert norm of each route, router weight, sum over k ------
// (page "vllm.models.muse_spark.amd.muse_moe_runner",
// MuseSparkTopKWeightAndReduce.apply: norm to fp32, times topk_weights, sum
// over k; moe_out stored as bf16.)
constexpr int kFinalizeThreads = 512;
constexpr int kFinalizeUnroll = 8;

// One CTA per token. All k route rows are read with every load of a round in
// flight and kept in shared memory when they fit (`stash`), so the rows
// leave HBM/L2 once.
__global__ void __launch_bounds__(kFinalizeThreads) k_finalize(FinalizeParams p) {
  pdl_launch_dependents();
  pdl_wait();
  extern __shared__ __align__(16) float4 fsm4[];
  __shared__ float part[kFinalizeUnroll * 2][kFinalizeThreads / 32];
  __shared__ float rstd[256], wt[256];
  __shared__ int loc[256];  // the route contributes (always, unless expert parallel)
  const int t = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int NW = kFinalizeThreads / 32;
  const int P4 = p.P / 4;
  const bool stash = p.stash != 0;
  const float4* y4 = reinterpret_cast<const float4*>(p.y) + (size_t)t * p.k * P4;
  for (int j = threadIdx.x; j < p.k; j += kFinalizeThreads) {
    wt[j] = __ldcg(p.weights + (size_t)t * p.k + j);
    int l = 1;
    if (p.part) {  // expert parallel: another rank holds this route's expert
      const int e = __ldcg(p.ids + (size_t)t * p.k + j);
      l = (e >= p.ep_first && e < p.ep_first + p.ep_count);
    }
    loc[j] = l;
  }
  __syncthreads();
  // sums of squares, kFinalizeUnroll routes per round, all their loads in flight
  for (int j0 = 0; j0 < p.k; j0 += kFinalizeUnroll) {
    float ss[kFinalizeUnroll];
#pragma unroll
    for (int u = 0; u < kFinalizeUnroll; ++u) ss[u] = 0.f;
    for (int i0 = 0; i0 < P4; i0 += kFinalizeThreads) {
      const int i = i0 + threadIdx.x;
      float4 v[kFinalizeUnroll];
#pragma unroll
      for (int u = 0; u < kFinalizeUnroll; ++u)
        v[u] = (j0 + u < p.k && i < P4 && loc[j0 + u]) ? __ldcg(y4 + (size_t)(j0 + u) * P4 + i)
                                                        : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int u = 0; u < kFinalizeUnroll; ++u) {
        ss[u] += v[u].x * v[u].x + v[u].y * v[u].y + v[u].z * v[u].z + v[u].w * v[u].w;
        if (stash && j0 + u < p.k && i < P4) fsm4[(size_t)(j0 + u) * P4 + i] = v[u];
      }
    }
#pragma unroll
    for (int u = 0; u < kFinalizeUnroll; ++u) {
      const float w = warp_sum(ss[u]);
      if (lane == 0) part[u][warp] = w;
    }
    __syncthreads();
    if (threadIdx.x < kFinalizeUnroll && j0 + threadIdx.x < p.k) {
      float a = 0.f;
      for (int w = 0; w < NW; ++w) a += part[threadIdx.x][w];
      rstd[j0 + threadIdx.x] = 1.0f / sqrtf(a / (float)p.P + p.eps);
    }
    __syncthreads();
  }
  for (int i = threadIdx.x; i < P4; i += kFinalizeThreads) {
    const uint2 wpb = *reinterpret_cast<const uint2*>(p.w_post_norm + 4 * i);
    const float w0 = bf16_bits_to_f32(wpb.x & 0xFFFFu), w1 = bf16_bits_to_f32(wpb.x >> 16);
    const float w2 = bf16_bits_to_f32(wpb.y & 0xFFFFu), w3 = bf16_bits_to_f32(wpb.y >> 16);
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll 8
    for (int j = 0; j < p.k; ++j) {
      if (!loc[j]) continue;  // (expert parallel) its y row was never written
      const float4 v = stash ? fsm4[(size_t)j * P4 + i] : __ldcg(y4 + (size_t)j * P4 + i);
      const float r = rstd[j], c = wt[j];
      a0 = fmaf(c, (v.x * r) * w0, a0);
      a1 = fmaf(c, (v.y * r) * w1, a1);
      a2 = fmaf(c, (v.z * r) * w2, a2);
      a3 = fmaf(c, (v.w * r) * w3, a3);
    }
    if (p.part) {
      reinterpret_cast<float4*>(p.part + (size_t)t * p.P)[i] = make_float4(a0, a1, a2, a3);
      continue;
    }
    uint2 o;
    o.x = (uint32_t)f32_to_bf16_bits(a0) | ((uint32_t)f32_to_bf16_bits(a1) << 16);
    o.y = (uint32_t)f32_to_bf16_bits(a2) | ((uint32_t)f32_to_bf16_bits(a3) << 16);
    reinterpret_cast<uint2*>(p.moe_out + (size_t)t * p.P)[i] = o;
  }
}

// fp32 -> bf16, four per thread (the summed expert-parallel moe_out)
__global__ void __launch_bounds__(256) k_round_bf16(const float4* src, uint2* dst, long long n4) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
       i += (long long)gridDim.x * blockDim.x) {
    const float4 v = __ldcg(src + i);
    dst[i] = make_uint2((uint32_t)f32_to_bf16_bits(v.x) | ((uint32_t)f32_to_bf16_bits(v.y) << 16),
                        (uint32_t)f32_to_bf16_bits(v.z) | ((uint32_t)f32_to_bf16_bits(v.w) << 16));
  }
}

cudaError_t launch_round_bf16(const float* src, uint16_t* dst, long long n, cudaStream_t s) {
  const long long n4 = n / 4;
  const unsigned grid = (unsigned)std::min<long long>((n4 + 255) / 256, 1024);
  k_round_bf16<<<grid, 256, 0, s>>>(reinterpret_cast<const float4*>(src),
                                    reinterpret_cast<uint2*>(dst), n4);
  return cudaGetLastError();
}

cudaError_t launch_finalize(const FinalizeParams& p, cudaStream_t s, bool pdl) {
  FinalizeParams q = p;
  const size_t stash = (size_t)p.k * p.P * sizeof(float);
  q.stash = stash <= 160 * 1024;
  const size_t smem = q.stash ? stash : 0;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k_finalize, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.rows);
  cfg.blockDim = dim3(kFinalizeThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_finalize, q);
}

}  // namespace musemoe
