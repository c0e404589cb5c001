// FFN boundary (page "vllm.models.muse_spark.nvidia.specialized_decode.runtime.
// providers", BoundaryProvider docstring): post_ffn_norm of the unpooler
// output, gated add into the fp32 residual stream in place, and the next
// pre-norm into bf16 out. One CTA per row; the unpooler's K-split partial
// sums are added here in a fixed order.
// Gated add: stream += gate * post_ffn_norm(u), one scalar gate per layer
// (the decoder page names add_ffn alpha/beta but prints no formula; this is
// the plain reading with alpha = 1, beta = gate).
#include "common.cuh"
#include "kernels.h"

namespace musemoe {

constexpr int kBoundaryThreads = 512;

__global__ void __launch_bounds__(kBoundaryThreads) k_boundary(BoundaryParams p) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ float scratch[32];
  extern __shared__ float buf[];  // [H]
  const int t = blockIdx.x;
  float ss = 0.f;
  for (int i = threadIdx.x; i < p.H; i += kBoundaryThreads) {
    float u = 0.f;
    for (int ks = 0; ks < p.ks; ++ks) u += __ldcg(p.part + ((size_t)ks * p.rows + t) * p.H + i);
    buf[i] = u;
    if (p.u_tap) p.u_tap[(size_t)t * p.H + i] = u;
    ss += u * u;
  }
  ss = block_sum(ss, scratch);
  const float rstd = 1.0f / sqrtf(ss / (float)p.H + p.eps);
  const float gate = __ldg(p.gate);
  float* srow = p.stream + (size_t)t * p.H;
  float ss2 = 0.f;
  for (int i = threadIdx.x; i < p.H; i += kBoundaryThreads) {
    const float add = (buf[i] * rstd) * bf16_bits_to_f32(p.w_ffn_norm[i]);
    const float s = fmaf(gate, add, srow[i]);
    srow[i] = s;
    buf[i] = s;
    ss2 += s * s;
  }
  ss2 = block_sum(ss2, scratch);
  const float rstd2 = 1.0f / sqrtf(ss2 / (float)p.H + p.eps);
  for (int i = threadIdx.x; i < p.H; i += kBoundaryThreads)
    p.out[(size_t)t * p.H + i] =
        f32_to_bf16_bits((buf[i] * rstd2) * bf16_bits_to_f32(p.w_next_norm[i]));
}

cudaError_t launch_boundary(const BoundaryParams& p, cudaStream_t s, bool pdl) {
  const size_t smem = (size_t)p.H * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k_boundary, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.rows);
  cfg.blockDim = dim3(kBoundaryThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_boundary, p);
}

}  // namespace musemoe
