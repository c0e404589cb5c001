// Routed experts: grouped GEMV/GEMM over the selected experts only.
//
// Work item = (token group of one expert, tile of weight rows). A CTA of 8
// warps splits the item's reduction dimension K across its warps and sums
// the 8 partial tiles in shared memory (fixed order: deterministic). CTAs
// take contiguous runs of items, so a CTA mostly stays on one expert group.
//
// Weights are streamed once from HBM with 128-bit loads straight into
// mma.sync fragments. Each thread's 16 bytes of a row cover:
//  * FP4 (kernel layout, see musemoe_pack_experts): 8 k-steps of m16n8k16;
//    k-step j of the 64-byte group holds elements 16j..16j+15 and thread q
//    owns 16j+4q..16j+4q+3, so one k-step never crosses a scale block. The
//    e2m1 pairs become f16 pairs with one cvt (exact). MXFP4 scales (UE8M0,
//    per 32) multiply the fp32 partial of each pair of k-steps; NVFP4 scales
//    (e4m3, per 16) multiply the f16 operand (e2m1 * e4m3 is exact in f16) and
//    the fp32 global scale multiplies the result.
//  * FP8: 2 k-steps of m16n8k32 e4m3 x e4m3; the per-row weight scale and the
//    per-row activation scale multiply the fp32 result.
// Activations (the N side, tokens) come from L1/L2: h or act rows in f16
// (FP4) or e4m3 (FP8).
//
// w13 (role 0): rows = 8 gate rows i..i+7 and the matching 8 up rows I+i..,
// so one thread holds gate and up of the same (i, token) and applies
// SiLU(gate) * up in registers; the activation is stored as bf16 (the MoE
// activations are bf16: page "vllm.models.muse_spark.amd.mono",
// maybe_attach_mono), converted to f16 for the FP4 w2 operand.
// w2 (role 1): 16 * RT rows of [P, I]; one unweighted fp32 output per route
// (page "vllm.models.muse_spark.amd.muse_moe_runner", MuseSparkAiterExperts:
// unit router weights; the weighting comes after the post-expert norm).
#include "common.cuh"
#include "kernels.h"

namespace musemoe {

constexpr int kExpertThreads = 256;
constexpr int kExpertWarps = kExpertThreads / 32;
constexpr int kChunkBytes = 64;  // bytes of one weight row per thread-quad
constexpr int kCMax = 2;         // chunks loaded ahead per warp

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;\n" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

template <int Q, int ROLE, int NT, int RT>
__global__ void __launch_bounds__(kExpertThreads) k_expert(ExpertParams p) {
  pdl_launch_dependents();
  pdl_wait();
  extern __shared__ __align__(16) float4 red[];  // [warps][RT][NT][32]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, q = lane & 3;
  const int n_groups = __ldcg(p.counters + kNumGroups);
  const int tiles = (ROLE == 0) ? p.I / 8 : p.N / (16 * RT);
  const int n_items = n_groups * tiles;
  const int i0 = (int)((long long)n_items * blockIdx.x / gridDim.x);
  const int i1 = (int)((long long)n_items * (blockIdx.x + 1) / gridDim.x);
  const int rowbytes = (Q == kFP8) ? p.K : p.K / 2;
  const int NC = rowbytes / kChunkBytes;
  const int kel = (Q == kFP8) ? 1 : 2;  // bytes per activation element
  const int nc_w = warp < NC ? (NC - warp + kExpertWarps - 1) / kExpertWarps : 0;

  for (int item = i0; item < i1; ++item) {
    const int grp = item / tiles, tile = item % tiles;
    const int4 gd = __ldcg(reinterpret_cast<const int4*>(p.groups) + grp);
    const int e = gd.x, rbase = gd.y, ntok = gd.z;
    const int ntile_act = (ntok + 7) >> 3;

    // activation row of this lane's B column in every n-tile
    const uint8_t* brow[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int n = nt * 8 + g;
      brow[nt] = nullptr;
      if (n < ntok) {
        const int r = __ldcg(p.route_list + rbase + n);
        const int br = p.b_by_token ? r / p.k : r;
        brow[nt] = p.b + (size_t)br * p.K * kel;
      }
    }
    // weight rows of this lane
    const uint8_t* wlo[RT];
    const uint8_t* whi[RT];
    int rlo[RT];
#pragma unroll
    for (int rt = 0; rt < RT; ++rt) {
      int lo, hi;
      if (ROLE == 0) {
        lo = tile * 8 + g;
        hi = p.I + tile * 8 + g;
      } else {
        lo = tile * 16 * RT + rt * 16 + g;
        hi = lo + 8;
      }
      rlo[rt] = lo;
      wlo[rt] = p.w + ((size_t)e * p.N + lo) * rowbytes + q * 16;
      whi[rt] = p.w + ((size_t)e * p.N + hi) * rowbytes + q * 16;
    }
    const size_t srow = (Q == kMXFP4) ? p.K / 32 : (Q == kNVFP4) ? p.K / 16 : 0;
    const uint8_t* sb = reinterpret_cast<const uint8_t*>(p.scale);

    float acc[RT][NT][4];
#pragma unroll
    for (int rt = 0; rt < RT; ++rt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[rt][nt][i] = 0.f;

    for (int cb = 0; cb < nc_w; cb += kCMax) {
      uint4 L[kCMax][RT], H[kCMax][RT];
      uint2 SL[kCMax][RT], SH[kCMax][RT];
#pragma unroll
      for (int u = 0; u < kCMax; ++u) {
        if (cb + u < nc_w) {
          const int c = warp + kExpertWarps * (cb + u);
#pragma unroll
          for (int rt = 0; rt < RT; ++rt) {
            L[u][rt] = ld_stream_v4(wlo[rt] + (size_t)c * kChunkBytes);
            H[u][rt] = ld_stream_v4(whi[rt] + (size_t)c * kChunkBytes);
            if (Q == kMXFP4) {
              const int lo = ROLE == 0 ? rlo[rt] : rlo[rt];
              const int hi = ROLE == 0 ? p.I + rlo[rt] : rlo[rt] + 8;
              SL[u][rt].x = ld_stream_u32(sb + ((size_t)e * p.N + lo) * srow + c * 4);
              SH[u][rt].x = ld_stream_u32(sb + ((size_t)e * p.N + hi) * srow + c * 4);
            } else if (Q == kNVFP4) {
              const int lo = rlo[rt];
              const int hi = ROLE == 0 ? p.I + rlo[rt] : rlo[rt] + 8;
              SL[u][rt] = ld_stream_v2(sb + ((size_t)e * p.N + lo) * srow + c * 8);
              SH[u][rt] = ld_stream_v2(sb + ((size_t)e * p.N + hi) * srow + c * 8);
            }
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kCMax; ++u) {
        if (cb + u >= nc_w) break;
        const int c = warp + kExpertWarps * (cb + u);
#pragma unroll
        for (int rt = 0; rt < RT; ++rt) {
          if (Q == kFP8) {
            // one chunk = 64 K = 2 k-steps of m16n8k32
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              if (nt >= ntile_act) break;
              uint4 bv = make_uint4(0, 0, 0, 0);
              if (brow[nt]) bv = ld_act_v4(brow[nt] + (size_t)c * 64 + q * 16);
              mma_e4m3_16832(acc[rt][nt], L[u][rt].x, H[u][rt].x, L[u][rt].y, H[u][rt].y, bv.x,
                             bv.y);
              mma_e4m3_16832(acc[rt][nt], L[u][rt].z, H[u][rt].z, L[u][rt].w, H[u][rt].w, bv.z,
                             bv.w);
            }
          } else if (Q == kMXFP4) {
            // one chunk = 128 K = 4 scale blocks of 32 = 8 k-steps
#pragma unroll
            for (int b = 0; b < 4; ++b) {
              const float fl = ue8m0_to_f32(SL[u][rt].x >> (8 * b));
              const float fh = ue8m0_to_f32(SH[u][rt].x >> (8 * b));
              const uint32_t wl = word_of(L[u][rt], b), wh = word_of(H[u][rt], b);
              const uint32_t a00 = e2m1x2_to_f16x2(wl), a01 = e2m1x2_to_f16x2(wh);
              const uint32_t a02 = e2m1x2_to_f16x2(wl >> 8), a03 = e2m1x2_to_f16x2(wh >> 8);
              const uint32_t a10 = e2m1x2_to_f16x2(wl >> 16), a11 = e2m1x2_to_f16x2(wh >> 16);
              const uint32_t a12 = e2m1x2_to_f16x2(wl >> 24), a13 = e2m1x2_to_f16x2(wh >> 24);
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) {
                if (nt >= ntile_act) break;
                uint2 b0 = make_uint2(0, 0), b1 = make_uint2(0, 0);
                if (brow[nt]) {
                  const uint8_t* bp = brow[nt] + ((size_t)c * 128 + 32 * b + 4 * q) * 2;
                  b0 = ld_act_v2(bp);
                  b1 = ld_act_v2(bp + 32);
                }
                float t[4] = {0.f, 0.f, 0.f, 0.f};
                mma_f16_16816(t, a00, a01, a02, a03, b0.x, b0.y);
                mma_f16_16816(t, a10, a11, a12, a13, b1.x, b1.y);
                acc[rt][nt][0] = fmaf(t[0], fl, acc[rt][nt][0]);
                acc[rt][nt][1] = fmaf(t[1], fl, acc[rt][nt][1]);
                acc[rt][nt][2] = fmaf(t[2], fh, acc[rt][nt][2]);
                acc[rt][nt][3] = fmaf(t[3], fh, acc[rt][nt][3]);
              }
            }
          } else {  // NVFP4: one chunk = 8 k-steps, one e4m3 scale per k-step
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const uint32_t slw = (j < 4 ? SL[u][rt].x : SL[u][rt].y) >> (8 * (j & 3));
              const uint32_t shw = (j < 4 ? SH[u][rt].x : SH[u][rt].y) >> (8 * (j & 3));
              const uint32_t sfl = e4m3x2_to_f16x2(slw & 0xFFu);
              const uint32_t sfh = e4m3x2_to_f16x2(shw & 0xFFu);
              const uint32_t sl2 = __byte_perm(sfl, sfl, 0x1010);  // broadcast low half
              const uint32_t sh2 = __byte_perm(sfh, sfh, 0x1010);
              const uint32_t wl = word_of(L[u][rt], j >> 1) >> (16 * (j & 1));
              const uint32_t wh = word_of(H[u][rt], j >> 1) >> (16 * (j & 1));
              const uint32_t a0 = hmul2(e2m1x2_to_f16x2(wl), sl2);
              const uint32_t a1 = hmul2(e2m1x2_to_f16x2(wh), sh2);
              const uint32_t a2 = hmul2(e2m1x2_to_f16x2(wl >> 8), sl2);
              const uint32_t a3 = hmul2(e2m1x2_to_f16x2(wh >> 8), sh2);
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) {
                if (nt >= ntile_act) break;
                uint2 bv = make_uint2(0, 0);
                if (brow[nt]) bv = ld_act_v2(brow[nt] + ((size_t)c * 128 + 16 * j + 4 * q) * 2);
                mma_f16_16816(acc[rt][nt], a0, a1, a2, a3, bv.x, bv.y);
              }
            }
          }
        }
      }
    }

    // ---- reduce the 8 K-slices -------------------------------------------
#pragma unroll
    for (int rt = 0; rt < RT; ++rt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        if (nt < ntile_act)
          red[((warp * RT + rt) * NT + nt) * 32 + lane] =
              make_float4(acc[rt][nt][0], acc[rt][nt][1], acc[rt][nt][2], acc[rt][nt][3]);
    __syncthreads();
    const int slots = RT * NT * 32;
    for (int s = threadIdx.x; s < slots; s += kExpertThreads) {
      const int ln = s & 31, nt = (s >> 5) % NT, rt = s / (32 * NT);
      if (nt >= ntile_act) continue;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int w = 0; w < kExpertWarps; ++w) {
        const float4 x = red[((w * RT + rt) * NT + nt) * 32 + ln];
        v.x += x.x;
        v.y += x.y;
        v.z += x.z;
        v.w += x.w;
      }
      const int ge = ln >> 2, qe = ln & 3;
      const int n0 = nt * 8 + 2 * qe;
      float gsc = 1.f;
      if (Q == kNVFP4) gsc = __ldg(p.gscale + e);
      if (ROLE == 0) {
        const int i = tile * 8 + ge;
        float sg = gsc, su = gsc;
        if (Q == kFP8) {
          const float* ws = reinterpret_cast<const float*>(p.scale);
          sg = __ldg(ws + (size_t)e * p.N + i);
          su = __ldg(ws + (size_t)e * p.N + p.I + i);
        }
        const float gate[2] = {v.x * sg, v.y * sg};
        const float up[2] = {v.z * su, v.w * su};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int n = n0 + h;
          if (n >= ntok) continue;
          const int r = __ldcg(p.route_list + rbase + n);
          float gt = gate[h], ut = up[h];
          if (Q == kFP8) {
            const float bs = __ldcg(p.b_scale + r / p.k);
            gt *= bs;
            ut *= bs;
          }
          const float a = round_bf16(silu(gt) * ut);
          if (Q == kFP8) {
            reinterpret_cast<uint16_t*>(p.out)[(size_t)r * p.I + i] = f32_to_bf16_bits(a);
          } else {
            reinterpret_cast<__half*>(p.out)[(size_t)r * p.I + i] = __float2half_rn(a);
            if (!(fabsf(a) <= 65504.f)) atomicOr(p.health, kHealthActRange);
          }
        }
      } else {
        const int plo = tile * 16 * RT + rt * 16 + ge, phi = plo + 8;
        float sl = gsc, sh = gsc;
        if (Q == kFP8) {
          const float* ws = reinterpret_cast<const float*>(p.scale);
          sl = __ldg(ws + (size_t)e * p.N + plo);
          sh = __ldg(ws + (size_t)e * p.N + phi);
        }
        const float lo[2] = {v.x * sl, v.y * sl};
        const float hi[2] = {v.z * sh, v.w * sh};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int n = n0 + h;
          if (n >= ntok) continue;
          const int r = __ldcg(p.route_list + rbase + n);
          const float bs = (Q == kFP8) ? __ldcg(p.b_scale + r) : 1.f;
          float* y = reinterpret_cast<float*>(p.out) + (size_t)r * p.P;
          y[plo] = lo[h] * bs;
          y[phi] = hi[h] * bs;
        }
      }
    }
    __syncthreads();
  }
}

template <int Q, int ROLE, int NT, int RT>
static cudaError_t launch_expert_t(const ExpertParams& p, cudaStream_t s, bool pdl) {
  const size_t smem = (size_t)kExpertWarps * RT * NT * 32 * sizeof(float4);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k_expert<Q, ROLE, NT, RT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(kExpertThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_expert<Q, ROLE, NT, RT>, p);
}

template <int Q, int ROLE>
static cudaError_t launch_expert_q(const ExpertParams& p, int nt, cudaStream_t s, bool pdl) {
  // w2 takes two 16-row tiles per item while the token tile is small
  switch (nt) {
    case 1: return launch_expert_t<Q, ROLE, 1, ROLE == 1 ? 2 : 1>(p, s, pdl);
    case 2: return launch_expert_t<Q, ROLE, 2, ROLE == 1 ? 2 : 1>(p, s, pdl);
    case 4: return launch_expert_t<Q, ROLE, 4, 1>(p, s, pdl);
    case 8: return launch_expert_t<Q, ROLE, 8, 1>(p, s, pdl);
    default: return cudaErrorInvalidValue;
  }
}

int expert_rows_per_tile(int role, int nt) { return role == 1 && nt <= 2 ? 32 : 16; }

cudaError_t launch_expert(const ExpertParams& p, int nt, cudaStream_t s, bool pdl) {
  switch (p.quant * 2 + p.role) {
    case 0: return launch_expert_q<kMXFP4, 0>(p, nt, s, pdl);
    case 1: return launch_expert_q<kMXFP4, 1>(p, nt, s, pdl);
    case 2: return launch_expert_q<kNVFP4, 0>(p, nt, s, pdl);
    case 3: return launch_expert_q<kNVFP4, 1>(p, nt, s, pdl);
    case 4: return launch_expert_q<kFP8, 0>(p, nt, s, pdl);
    case 5: return launch_expert_q<kFP8, 1>(p, nt, s, pdl);
    default: return cudaErrorInvalidValue;
  }
}

template <int Q, int ROLE, int NT, int RT>
static int occ_t() {
  int n = 0;
  const size_t smem = (size_t)kExpertWarps * RT * NT * 32 * sizeof(float4);
  if (smem > 48 * 1024)
    cudaFuncSetAttribute(k_expert<Q, ROLE, NT, RT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem);
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_expert<Q, ROLE, NT, RT>, kExpertThreads,
                                                    smem) != cudaSuccess)
    return 1;
  return n > 0 ? n : 1;
}
template <int Q, int ROLE>
static int occ_q(int nt) {
  switch (nt) {
    case 1: return occ_t<Q, ROLE, 1, ROLE == 1 ? 2 : 1>();
    case 2: return occ_t<Q, ROLE, 2, ROLE == 1 ? 2 : 1>();
    case 4: return occ_t<Q, ROLE, 4, 1>();
    default: return occ_t<Q, ROLE, 8, 1>();
  }
}
int expert_ctas_per_sm(int quant, int role, int nt) {
  switch (quant * 2 + role) {
    case 0: return occ_q<kMXFP4, 0>(nt);
    case 1: return occ_q<kMXFP4, 1>(nt);
    case 2: return occ_q<kNVFP4, 0>(nt);
    case 3: return occ_q<kNVFP4, 1>(nt);
    case 4: return occ_q<kFP8, 0>(nt);
    default: return occ_q<kFP8, 1>(nt);
  }
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

cudaError_t launch_act_quant(const ActQuantParams& p, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((p.routes + 7) / 8);
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_act_quant, p);
}

// ---- tail: post-expert norm of each route, router weight, sum over k ------
// (page "vllm.models.muse_spark.amd.muse_moe_runner",
// MuseSparkTopKWeightAndReduce.apply: norm to fp32, times topk_weights, sum
// over k; moe_out stored as bf16.)
__global__ void __launch_bounds__(256) k_finalize(FinalizeParams p) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ float scratch[32];
  extern __shared__ float rstd[];
  const int t = blockIdx.x;
  for (int j = 0; j < p.k; ++j) {
    const float* y = p.y + ((size_t)t * p.k + j) * p.P;
    float ss = 0.f;
    for (int i = threadIdx.x; i < p.P; i += blockDim.x) {
      const float v = __ldcg(y + i);
      ss += v * v;
    }
    ss = block_sum(ss, scratch);
    if (threadIdx.x == 0) rstd[j] = 1.0f / sqrtf(ss / (float)p.P + p.eps);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < p.P; i += blockDim.x) {
    const float wp = bf16_bits_to_f32(p.w_post_norm[i]);
    float acc = 0.f;
    for (int j = 0; j < p.k; ++j) {
      const float v = __ldcg(p.y + ((size_t)t * p.k + j) * p.P + i);
      const float n = (v * rstd[j]) * wp;
      acc = fmaf(__ldcg(p.weights + (size_t)t * p.k + j), n, acc);
    }
    p.moe_out[(size_t)t * p.P + i] = f32_to_bf16_bits(acc);
  }
}

cudaError_t launch_finalize(const FinalizeParams& p, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.rows);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = (size_t)p.k * sizeof(float);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_finalize, p);
}

// ---- weight re-layout: plain FP4 rows -> kernel layout ---------------------
// Within every 64-byte group: byte 8j + 2q + b -> byte 16q + 2j + b.
__global__ void k_pack_fp4(const uint8_t* src, uint8_t* dst, size_t groups) {
  const size_t gi = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (gi >= groups) return;
  const uint4* s4 = reinterpret_cast<const uint4*>(src + gi * 64);
  uint32_t in[16];
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const uint4 x = s4[v];
    in[4 * v] = x.x;
    in[4 * v + 1] = x.y;
    in[4 * v + 2] = x.z;
    in[4 * v + 3] = x.w;
  }
  uint32_t out[16];
#pragma unroll
  for (int w = 0; w < 16; ++w) {
    uint32_t o = 0;
#pragma unroll
    for (int bb = 0; bb < 4; ++bb) {
      const int dpos = 4 * w + bb;               // = 16q + 2j + b
      const int qq = dpos >> 4, j = (dpos >> 1) & 7, b = dpos & 1;
      const int spos = 8 * j + 2 * qq + b;
      const uint32_t byte = (in[spos >> 2] >> (8 * (spos & 3))) & 0xFFu;
      o |= byte << (8 * bb);
    }
    out[w] = o;
  }
  uint4* d4 = reinterpret_cast<uint4*>(dst + gi * 64);
#pragma unroll
  for (int v = 0; v < 4; ++v)
    d4[v] = make_uint4(out[4 * v], out[4 * v + 1], out[4 * v + 2], out[4 * v + 3]);
}

cudaError_t launch_pack_fp4(const uint8_t* src, uint8_t* dst, size_t bytes, cudaStream_t s) {
  const size_t groups = bytes / 64;
  if (groups == 0) return cudaSuccess;
  k_pack_fp4<<<(unsigned)((groups + 255) / 256), 256, 0, s>>>(src, dst, groups);
  return cudaGetLastError();
}

}  // namespace musemoe
