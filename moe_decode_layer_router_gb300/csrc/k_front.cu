// Front of the block: the fp32 router GEMV and the bf16 pooler GEMV in one
// launch (the two read the same input and are independent), and the same
// bf16 GEMV for the unpooler.
//
// Router: fp32 weight [E, H] times the bf16 input (page
// "vllm.models.muse_spark.nvidia.specialized_decode.runtime.providers",
// MoEProvider docstring: the router is an fp32 linear layer from [b, H] to
// one logit per expert), fp32 FFMA so the logits keep fp32 products.
// Pooler [P, H] / unpooler [H, P]: bf16 weights streamed once from HBM with
// 128-bit loads straight into mma.sync fragments (weight rows = M, tokens =
// N), fp32 accumulation.
// Both split K across CTAs and write fp32 partial sums; the consumer adds
// them in a fixed order, so results do not depend on scheduling.
#include "common.cuh"
#include "kernels.h"

namespace musemoe {

constexpr int kFrontThreads = 128;  // 4 warps
constexpr int kRouterRowsPerCta = 16;
constexpr int kGemvRowsPerCta = 64;

// True in every thread of the CTA that finishes the last of `splits` CTAs
// sharing `ticket`; that CTA resets the ticket. No thread waits on another CTA.
__device__ __forceinline__ bool last_of_tile(int32_t* ticket, int splits) {
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int prev = atomicAdd(ticket, 1);
    s_last = (prev == splits - 1);
    if (s_last) *ticket = 0;
  }
  __syncthreads();
  if (s_last) __threadfence();
  return s_last;
}

// Sum of `splits` partials spaced `stride` floats apart, in a fixed order,
// with up to 8 loads in flight.
__device__ __forceinline__ float sum_splits(const float* p, size_t stride, int splits) {
  float v = 0.f;
  int s = 0;
  for (; s + 8 <= splits; s += 8) {
    float a[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = __ldcg(p + (size_t)(s + i) * stride);
#pragma unroll
    for (int i = 0; i < 8; ++i) v += a[i];
  }
  float a[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) a[i] = (s + i < splits) ? __ldcg(p + (size_t)(s + i) * stride) : 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) v += a[i];
  return v;
}

__device__ __forceinline__ void router_cta(const FrontParams& p, int task) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int EB = (p.E + kRouterRowsPerCta - 1) / kRouterRowsPerCta;
  const int eb = task % EB;
  const int rest = task / EB;
  const int ks = rest % p.ks_r;
  const int tb = rest / p.ks_r;
  const int K4 = p.K / 4;  // float4 columns
  const int per = (K4 + p.ks_r - 1) / p.ks_r;
  const int c0 = ks * per, c1 = min(K4, c0 + per);
  const int e0 = eb * kRouterRowsPerCta + warp * 4;
  const int t0 = tb * 8;
  float acc[4][8];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int t = 0; t < 8; ++t) acc[r][t] = 0.f;
  for (int c = c0 + lane; c < c1; c += 32) {
    float4 wv[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int e = min(e0 + r, p.E - 1);
      wv[r] = __ldg(reinterpret_cast<const float4*>(p.w_router + (size_t)e * p.K) + c);
    }
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      if (t0 + t < p.rows) {
        const uint2 xv = *reinterpret_cast<const uint2*>(p.x + (size_t)(t0 + t) * p.K + 4 * c);
        const float x0 = bf16_bits_to_f32(xv.x & 0xFFFFu), x1 = bf16_bits_to_f32(xv.x >> 16);
        const float x2 = bf16_bits_to_f32(xv.y & 0xFFFFu), x3 = bf16_bits_to_f32(xv.y >> 16);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          float a = acc[r][t];
          a = fmaf(wv[r].x, x0, a);
          a = fmaf(wv[r].y, x1, a);
          a = fmaf(wv[r].z, x2, a);
          a = fmaf(wv[r].w, x3, a);
          acc[r][t] = a;
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const float v = warp_sum(acc[r][t]);
      if (lane == 0 && e0 + r < p.E && t0 + t < p.rows)
        p.logit_part[((size_t)ks * p.rows + t0 + t) * p.E + e0 + r] = v;
    }
  // the last split of this (expert block, token block) adds the partials
  if (!last_of_tile(p.router_tickets + eb + EB * tb, p.ks_r)) return;
  const int ntok = min(8, p.rows - t0);
  for (int idx = threadIdx.x; idx < kRouterRowsPerCta * ntok; idx += kFrontThreads) {
    const int e = eb * kRouterRowsPerCta + idx % kRouterRowsPerCta;
    const int t = t0 + idx / kRouterRowsPerCta;
    if (e >= p.E) continue;
    p.logits[(size_t)t * p.E + e] =
        sum_splits(p.logit_part + (size_t)t * p.E + e, (size_t)p.rows * p.E, p.ks_r);
  }
}

template <int NT>
__device__ __forceinline__ void gemv_cta(const FrontParams& p, int task) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, q = lane & 3;
  const int RB = p.M / kGemvRowsPerCta;
  const int rb = task % RB;
  const int rest = task / RB;
  const int ks = rest % p.ks;
  const int tb = rest / p.ks;
  const int KC = p.K / 32;
  const int c0 = ks * p.kchunks_per_split, c1 = min(KC, c0 + p.kchunks_per_split);
  const int row_lo = rb * kGemvRowsPerCta + warp * 16 + g;
  const uint16_t* a_lo = p.w + (size_t)row_lo * p.K + q * 8;
  const uint16_t* a_hi = a_lo + (size_t)8 * p.K;
  const int tok0 = tb * 8 * NT;
  const uint16_t* bptr[NT];
  bool bval[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int n = tok0 + nt * 8 + g;
    bval[nt] = n < p.rows;
    bptr[nt] = p.x + (size_t)(bval[nt] ? n : 0) * p.K + q * 8;
  }
  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[nt][i] = 0.f;

  constexpr int U = 4;
  int c = c0;
  for (; c + U <= c1; c += U) {
    uint4 lo[U], hi[U], bv[U][NT];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      lo[u] = ld_stream_v4(a_lo + (size_t)(c + u) * 32);
      hi[u] = ld_stream_v4(a_hi + (size_t)(c + u) * 32);
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        bv[u][nt] = bval[nt] ? ld_act_v4(bptr[nt] + (size_t)(c + u) * 32) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int u = 0; u < U; ++u) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        if (tok0 + nt * 8 >= p.rows) break;
        mma_bf16_16816(acc[nt], lo[u].x, hi[u].x, lo[u].y, hi[u].y, bv[u][nt].x, bv[u][nt].y);
        mma_bf16_16816(acc[nt], lo[u].z, hi[u].z, lo[u].w, hi[u].w, bv[u][nt].z, bv[u][nt].w);
      }
    }
  }
  for (; c < c1; ++c) {
    const uint4 lo = ld_stream_v4(a_lo + (size_t)c * 32);
    const uint4 hi = ld_stream_v4(a_hi + (size_t)c * 32);
    uint4 bv[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
      bv[nt] = bval[nt] ? ld_act_v4(bptr[nt] + (size_t)c * 32) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      if (tok0 + nt * 8 >= p.rows) break;
      mma_bf16_16816(acc[nt], lo.x, hi.x, lo.y, hi.y, bv[nt].x, bv[nt].y);
      mma_bf16_16816(acc[nt], lo.z, hi.z, lo.w, hi.w, bv[nt].z, bv[nt].w);
    }
  }
  // D fragment: c0/c1 = (row g, tokens 2q, 2q+1), c2/c3 = (row g+8, same tokens)
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int n0 = tok0 + nt * 8 + 2 * q;
    float* base = p.part + (size_t)ks * p.rows * p.M;
    if (n0 < p.rows) {
      base[(size_t)n0 * p.M + row_lo] = acc[nt][0];
      base[(size_t)n0 * p.M + row_lo + 8] = acc[nt][2];
    }
    if (n0 + 1 < p.rows) {
      base[(size_t)(n0 + 1) * p.M + row_lo] = acc[nt][1];
      base[(size_t)(n0 + 1) * p.M + row_lo + 8] = acc[nt][3];
    }
  }
  // the last split of this (row block, token block) adds the partials
  if (!last_of_tile(p.tickets + rb + RB * tb, p.ks)) return;
  const int ntok = min(8 * NT, p.rows - tok0);
  for (int idx = threadIdx.x; idx < kGemvRowsPerCta * ntok; idx += kFrontThreads) {
    const int row = rb * kGemvRowsPerCta + idx % kGemvRowsPerCta;
    const int t = tok0 + idx / kGemvRowsPerCta;
    p.y[(size_t)t * p.M + row] = sum_splits(p.part + (size_t)t * p.M + row, (size_t)p.rows * p.M, p.ks);
  }
}

template <int NT>
__global__ void __launch_bounds__(kFrontThreads) k_front(FrontParams p) {
  pdl_launch_dependents();
  pdl_wait();  // x may be the previous kernel's output
  const int b = blockIdx.x;
  if (b < p.router_ctas)
    router_cta(p, b);
  else
    gemv_cta<NT>(p, b - p.router_ctas);
}

int front_ctas(const FrontParams& p) {
  const int gemv = (p.M / kGemvRowsPerCta) * p.ks * p.token_blocks;
  return p.router_ctas + gemv;
}

cudaError_t launch_front(const FrontParams& p, int nt, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(front_ctas(p));
  cfg.blockDim = dim3(kFrontThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  switch (nt) {
    case 1: return cudaLaunchKernelEx(&cfg, k_front<1>, p);
    case 2: return cudaLaunchKernelEx(&cfg, k_front<2>, p);
    case 4: return cudaLaunchKernelEx(&cfg, k_front<4>, p);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace musemoe
