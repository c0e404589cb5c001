// Front of the block and the unpooler: dense bf16 GEMVs Y = X W^T with the
// weight tile streamed in by the tensor memory accelerator, and the fp32
// router GEMV.
//
// Router: fp32 weight [E, H] times the bf16 input (page
// "vllm.models.muse_spark.nvidia.specialized_decode.runtime.providers",
// MoEProvider docstring: the router is an fp32 linear layer from [b, H] to
// one logit per expert), fp32 FFMA so the logits keep fp32 products. It is
// its own launch, just before the pooler's.
//
// Pooler [P, H] / unpooler [H, P] (bf16, row-major as the caller holds
// them): one CTA per 16-row tile (and token block) holds the tile's whole
// reduction length in shared memory. Weights never depend on the previous
// kernel, so thread 0 issues every [16 rows x 64] box of the tile (2-D
// tensor copies, 128-byte swizzle, one mbarrier per box) before the kernel
// waits for its predecessor; the copies overlap the predecessor's tail. The
// 8 warps then split K, read conflict-free A fragments with ldmatrix, take
// the activation fragments (at most 8 NT tokens) from L1/L2, accumulate
// with mma.sync (bf16 in, fp32 out) and add their 8 partials in a fixed
// order in shared memory. Rows and tokens past the end are never stored.
// For the pooler, the CTA that stores a token block's last tile applies the
// pre-expert norm to the block's rows (no separate launch, no waiting).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "pipeline.cuh"
#include "route_dev.cuh"

namespace musemoe {

constexpr int kGWarps = 8;
constexpr int kGThreads = kGWarps * 32;
constexpr int kGTileRows = 16;                 // weight rows per CTA
constexpr int kGBoxK = 64;                     // elements per box row (128 B)
constexpr int kGBoxBytes = kGTileRows * 128;   // one [16 x 64] bf16 box
constexpr int kGMaxK = 5632;                   // reduction length held in shared memory

__host__ __device__ constexpr int g_red_bytes(int nt) { return kGWarps * nt * 32 * 16; }
// boxes (64-element chunks of the reduction) per warp
__host__ __device__ constexpr int g_chunks_per_warp(int K) { return (K / kGBoxK + kGWarps - 1) / kGWarps; }
constexpr int kGXRing = 4;          // activation boxes in flight per warp (one token tile)
constexpr int kGXBox = 8 * 128;     // one [8 tokens x 64] bf16 box
__host__ __device__ constexpr size_t g_smem_bytes(int K, int nt) {
  return (size_t)kGWarps * g_chunks_per_warp(K) * kGBoxBytes +
         (nt == 1 ? (size_t)kGWarps * kGXRing * kGXBox : 0) + g_red_bytes(nt) + 1024;
}

// 16-byte asynchronous copy global -> shared (L2 only), and its groups.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// Byte offset of 16-byte unit u of row r in a box of 128-byte rows written
// with the 128-byte swizzle (the box starts on a 1024-byte boundary).
__device__ __forceinline__ uint32_t swz(int r, int u) { return r * 128 + ((u ^ (r & 7)) << 4); }

// Router CTA: expert e = blockIdx % E for tokens [8 tb, 8 tb + 8). Thread 0
// copies the tokens' input rows into shared memory (1-D bulk copies, one
// mbarrier); meanwhile every thread loads its float4 columns t, t + 256, ...
// of the expert's fp32 weight row (at most kRouterCols). Then each thread
// accumulates its columns for every token, and the CTA adds its threads'
// sums (warp shuffles, then the 8 warps in order).
constexpr int kRouterCols = 8;   // float4 columns per thread: K <= 8192
constexpr int kRouterCols4 = 5;  // with four experts per CTA: K <= 5120
static_assert(kGThreads == kRouteThreads, "the route tail runs the route kernel's block code");

// Route tail of a router CTA (forward chain): after its logits, the CTA that
// stores the last expert of an 8-token block (atomic ticket, no waiting)
// routes the block's rows, one warp per row; the block that finishes last
// builds the permute (a single block does it at once, from the ids it keeps
// in shared memory). The routing needs nothing else, so it completes with
// the router's launch.
template <int EPL>
__device__ __noinline__ void router_route_tail(const FrontParams& p, int tb, int t0, int ntok,
                                               const float* bias_s, uint8_t* smem, int ctas_per_block) {
  __shared__ float s_w[kGWarps][256];
  __shared__ int top[kGWarps][256];
  __shared__ int last_s;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const RouteParams& rp = p.route;
  __syncthreads();  // orders the CTA's logits stores before thread 0's fence and ticket
  if (tid == 0) {
    __threadfence();
    last_s = atomicAdd(p.route_ticket + tb, 1) == ctas_per_block - 1;
    if (last_s) {
      // the fence orders the other CTAs' logits (released before their
      // tickets) before this CTA's reads; the reset after it (for the next
      // launch) leaves the fence no store of its own to wait for
      __threadfence();
      p.route_ticket[tb] = 0;
    }
  }
  __syncthreads();
  if (!last_s) return;
  const int nblk = (rp.rows + 7) / 8;
  const int rt = rp.rows * rp.k;
  int16_t* ids_s = reinterpret_cast<int16_t*>(smem);  // the input rows' staging, done with
  unsigned char* work = smem + (((size_t)rt * 2 + 15) & ~(size_t)15);
  if (nblk == 1) {
    // one token block: its rows' ids stay in shared memory for the permute
    if (warp < ntok) route_row_warp<EPL>(rp, t0 + warp, lane, s_w[warp], top[warp], ids_s, bias_s);
    __syncthreads();
    if (rt <= kRouteThreads && rp.E <= kRouteThreads) permute_small(rp, ids_s);
    else permute(rp, ids_s, work);
    return;
  }
  if (warp < ntok) route_row_warp<EPL>(rp, t0 + warp, lane, s_w[warp], top[warp], nullptr, bias_s);
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    last_s = atomicAdd(p.route_done, 1) == nblk - 1;
    if (last_s) {
      __threadfence();
      *p.route_done = 0;  // for the next launch
    }
  }
  __syncthreads();
  if (!last_s) return;
  for (int i = tid; i < rt; i += kGThreads) ids_s[i] = (int16_t)__ldcg(rp.ids + i);
  __syncthreads();
  if (rt <= kRouteThreads && rp.E <= kRouteThreads) permute_small(rp, ids_s);
  else permute(rp, ids_s, work);
}

// EG experts per CTA (EG > 1 for more than 8 rows: the 8 tokens' rows in
// shared memory serve EG weight rows, EG times fewer input-row copies), at
// most NCOL float4 weight columns per thread and expert.
template <int EPL, int EG, int NCOL>
__device__ __forceinline__ void router_cta(const FrontParams& p, int task, uint8_t* smem) {
  __shared__ float red[kGWarps][8 * EG];
  __shared__ __align__(8) unsigned long long xbar;
  __shared__ int abort_flag;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ng = p.E / EG;  // CTAs per token block
  const int e0 = (task % ng) * EG, t0 = (task / ng) * 8;
  const int ntok = min(8, p.rows - t0);
  const int K4 = p.K / 4;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&xbar), 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();
  // the weight row (and, for the route tail, the selection bias) does not
  // depend on the previous kernel
  __shared__ float bias_s[256];
  if (p.route_tail)
    for (int i = threadIdx.x; i < p.E; i += kGThreads) bias_s[i] = __ldg(p.route.expert_bias + i);
  float4 wv[EG][NCOL];
#pragma unroll
  for (int g = 0; g < EG; ++g) {
    const float4* wr = reinterpret_cast<const float4*>(p.w_router + (size_t)(e0 + g) * p.K);
#pragma unroll
    for (int u = 0; u < NCOL; ++u) {
      const int c = threadIdx.x + u * kGThreads;
      wv[g][u] = c < K4 ? __ldg(wr + c) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  pdl_wait();  // x may be the previous kernel's output
  // dependents launch only now: the pooler two launches on reads x without
  // a wait of its own
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    mbar_expect_tx(smem_u32(&xbar), (uint32_t)(ntok * p.K * 2));
    for (int t = 0; t < ntok; ++t)
      bulk_g2s(smem_u32(smem) + t * p.K * 2, p.x + (size_t)(t0 + t) * p.K, p.K * 2, smem_u32(&xbar));
  }
  float acc[EG][8];
#pragma unroll
  for (int g = 0; g < EG; ++g)
#pragma unroll
    for (int t = 0; t < 8; ++t) acc[g][t] = 0.f;
  const bool ok = mbar_wait_or_abort(smem_u32(&xbar), 0u, &abort_flag);
  if (ok) {
    const uint16_t* xs = reinterpret_cast<const uint16_t*>(smem);
#pragma unroll
    for (int u = 0; u < NCOL; ++u) {
      const int c = threadIdx.x + u * kGThreads;
      if (c >= K4) break;
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        if (t >= ntok) break;
        const uint2 xv = *reinterpret_cast<const uint2*>(xs + t * p.K + 4 * c);
        const float x0 = bf16_bits_to_f32(xv.x & 0xFFFFu), x1 = bf16_bits_to_f32(xv.x >> 16);
        const float x2 = bf16_bits_to_f32(xv.y & 0xFFFFu), x3 = bf16_bits_to_f32(xv.y >> 16);
#pragma unroll
        for (int g = 0; g < EG; ++g) {
          float a = acc[g][t];
          a = fmaf(wv[g][u].x, x0, a);
          a = fmaf(wv[g][u].y, x1, a);
          a = fmaf(wv[g][u].z, x2, a);
          a = fmaf(wv[g][u].w, x3, a);
          acc[g][t] = a;
        }
      }
    }
  } else if (!abort_flag) {
    abort_flag = 1;
    if (p.health) atomicOr(p.health, kHealthTimeout);
  }
#pragma unroll
  for (int g = 0; g < EG; ++g)
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const float v = warp_sum(acc[g][t]);
      if (lane == 0) red[warp][g * 8 + t] = v;
    }
  __syncthreads();
  if (threadIdx.x < 8 * EG) {
    const int g = threadIdx.x >> 3, t = threadIdx.x & 7;
    if (t < ntok) {
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < kGWarps; ++w) v += red[w][threadIdx.x];
      p.logits[(size_t)(t0 + t) * p.E + e0 + g] = v;
    }
  }
  // the copies must have landed before the CTA leaves (after a timeout)
  if (threadIdx.x == 0 && !ok) {
    const unsigned long long tw0 = globaltimer();
    while (!mbar_try_wait(smem_u32(&xbar), 0u))
      if (globaltimer() - tw0 > kWaitLimitNs) break;
  }
  if (p.route_tail) router_route_tail<EPL>(p, task / ng, t0, ntok, bias_s, smem, ng);
}

// Pre-expert RMSNorm (page "vllm.models.muse_spark.nvidia.specialized_decode.
// runtime.providers", MoEProvider docstring) of the pooled rows [t0, t1) of
// y, one warp per row: the bf16 h, and the expert operand, h in f16 (exact
// for |h| in [2^-14, 65504]) or, for FP8 W8A8, e4m3 codes with the per-row
// dynamic scale amax / 448. A row of at most kNV * 128 elements is held in
// registers (its loads and its norm weights' issued together); a longer one
// is read from L2 once per pass.
constexpr int kNV = 16;
// W4A4 writes h only: the forward rounds it to FP4 next (k_act_fp4, many
// warps per row) and a value that is not finite raises kHealthHRange here.
__device__ __forceinline__ void norm_rows(const FrontParams& p, int t0, int t1) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n4 = p.M / 4;
  const uint2* wsrc = reinterpret_cast<const uint2*>(p.w_pre_norm);
  int bad = 0;
  for (int t = t0 + warp; t < t1; t += kGWarps) {
    const float4* src = reinterpret_cast<const float4*>(p.y + (size_t)t * p.M);
    uint2* hdst = reinterpret_cast<uint2*>(p.h + (size_t)t * p.M);
    // float4 i of the row: its loads, and the bf16 h, (x * rstd) * w rounded
    auto load = [&](int i, float4& v, uint2& wb) {
      v = i < n4 ? __ldcg(src + i) : make_float4(0.f, 0.f, 0.f, 0.f);
      wb = (i < n4 && p.pre_norm) ? __ldg(wsrc + i) : make_uint2(0u, 0u);
    };
    // (x * rstd) * w rounded to bf16, one conversion per pair: the packed
    // bits in hbits, the values in hb
    auto h4 = [&](const float4& x, const uint2& wb, float rstd, float (&hb)[4], uint32_t (&hbits)[2]) {
      const float xv[4] = {x.x, x.y, x.z, x.w};
      const float wv[4] = {bf16_bits_to_f32(wb.x & 0xFFFFu), bf16_bits_to_f32(wb.x >> 16),
                           bf16_bits_to_f32(wb.y & 0xFFFFu), bf16_bits_to_f32(wb.y >> 16)};
      float v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = p.pre_norm ? (xv[j] * rstd) * wv[j] : xv[j];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const __nv_bfloat162 b2 = __floats2bfloat162_rn(v[2 * c], v[2 * c + 1]);
        hbits[c] = *reinterpret_cast<const uint32_t*>(&b2);
        hb[2 * c] = __uint_as_float(hbits[c] << 16);
        hb[2 * c + 1] = __uint_as_float(hbits[c] & 0xFFFF0000u);
      }
    };
    // stores h (and the f16 operand) of float4 i; returns its amax
    auto put = [&](int i, const float (&hb)[4], const uint32_t (&hbits)[2]) -> float {
      float am = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) am = fmaxf(am, fabsf(hb[c]));
      hdst[i] = make_uint2(hbits[0], hbits[1]);
      if (p.act4) {
#pragma unroll
        for (int c = 0; c < 4; ++c) bad |= !(fabsf(hb[c]) <= 3.40282347e38f);  // NaN or infinite
      } else if (p.quant == kMXFP4 || p.quant == kNVFP4) {  // the f16 operand (BF16 and FP8 have their own)
#pragma unroll
        for (int c = 0; c < 4; ++c) bad |= !(fabsf(hb[c]) <= 65504.f);  // NaN too
        uint32_t opbits[2];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const __half2 h2 = __floats2half2_rn(hb[2 * c], hb[2 * c + 1]);
          opbits[c] = *reinterpret_cast<const uint32_t*>(&h2);
        }
        reinterpret_cast<uint2*>(p.h_op + (size_t)t * p.M * 2)[i] = make_uint2(opbits[0], opbits[1]);
      }
      return am;
    };
    auto put_q = [&](int i, const float (&hb)[4], float sc) {
      uint16_t q[2];
#pragma unroll
      for (int c = 0; c < 2; ++c)
        q[c] = f32x2_to_e4m3x2(sc > 0.f ? hb[2 * c] / sc : 0.f, sc > 0.f ? hb[2 * c + 1] / sc : 0.f);
      reinterpret_cast<uint32_t*>(p.h_op + (size_t)t * p.M)[i] = (uint32_t)q[0] | ((uint32_t)q[1] << 16);
    };
    float ss = 0.f, amax = 0.f;
    if (n4 <= kNV * 32) {
      float4 v[kNV];
      uint2 wb[kNV];
#pragma unroll
      for (int j = 0; j < kNV; ++j) load(j * 32 + lane, v[j], wb[j]);
#pragma unroll
      for (int j = 0; j < kNV; ++j) ss += v[j].x * v[j].x + v[j].y * v[j].y + v[j].z * v[j].z + v[j].w * v[j].w;
      ss = warp_sum(ss);
      const float rstd = p.pre_norm ? 1.0f / sqrtf(ss / (float)p.M + p.norm_eps) : 1.0f;
#pragma unroll
      for (int j = 0; j < kNV; ++j) {
        const int i = j * 32 + lane;
        if (i < n4) {
          float hb[4];
          uint32_t hbits[2];
          h4(v[j], wb[j], rstd, hb, hbits);
          amax = fmaxf(amax, put(i, hb, hbits));
        }
      }
      if (p.quant == kFP8) {
        amax = warp_max(amax);
        const float sc = amax / 448.0f;
#pragma unroll
        for (int j = 0; j < kNV; ++j) {
          const int i = j * 32 + lane;
          if (i < n4) {
            float hb[4];
            uint32_t hbits[2];
            h4(v[j], wb[j], rstd, hb, hbits);
            put_q(i, hb, sc);
          }
        }
        if (lane == 0) p.h_scale[t] = sc;
      }
    } else {
      constexpr int kB = 4;  // float4s per lane in flight
      for (int base = 0; base < n4; base += kB * 32) {
        float4 v[kB];
#pragma unroll
        for (int j = 0; j < kB; ++j) {
          const int i = base + j * 32 + lane;
          v[j] = i < n4 ? __ldcg(src + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int j = 0; j < kB; ++j) ss += v[j].x * v[j].x + v[j].y * v[j].y + v[j].z * v[j].z + v[j].w * v[j].w;
      }
      ss = warp_sum(ss);
      const float rstd = p.pre_norm ? 1.0f / sqrtf(ss / (float)p.M + p.norm_eps) : 1.0f;
      for (int pass = 0; pass < (p.quant == kFP8 ? 2 : 1); ++pass) {
        const float sc = pass ? warp_max(amax) / 448.0f : 0.f;
        for (int base = 0; base < n4; base += kB * 32) {
          float4 v[kB];
          uint2 wb[kB];
#pragma unroll
          for (int j = 0; j < kB; ++j) load(base + j * 32 + lane, v[j], wb[j]);
#pragma unroll
          for (int j = 0; j < kB; ++j) {
            const int i = base + j * 32 + lane;
            if (i >= n4) break;
            float hb[4];
            uint32_t hbits[2];
            h4(v[j], wb[j], rstd, hb, hbits);
            if (pass == 0) amax = fmaxf(amax, put(i, hb, hbits));
            else put_q(i, hb, sc);
          }
        }
        if (pass == 1 && lane == 0) p.h_scale[t] = sc;
      }
    }
  }
  if (bad) atomicOr(p.health, kHealthHRange);
}

// NT = 1: every warp streams its activation boxes ([8 tokens x 64], 16-byte
// asynchronous copies to the 128-byte-swizzled addresses, issued right after
// the wait for the previous kernel) through a ring of kGXRing shared-memory
// slots and reads its B fragments with ldmatrix. NT > 1: the fragments of the next box load from L1/L2 while the
// current one runs.
template <int NT, bool POOL>
__device__ __forceinline__ void gemv_cta(const CUtensorMap* tw, const FrontParams& p,
                                         uint8_t* smem_raw) {
  __shared__ __align__(8) unsigned long long warp_b[kGWarps];
  __shared__ int abort_flag;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, q = lane & 3;
  const int tiles = (p.M + kGTileRows - 1) / kGTileRows;
  const int tile = blockIdx.x % tiles, tbk = blockIdx.x / tiles;
  const int nbox = p.K / kGBoxK, nch = g_chunks_per_warp(p.K);
  // 1024-byte aligned tile (the 128-byte swizzle repeats every 1024 bytes)
  const uint32_t wt = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t xring = wt + kGWarps * nch * kGBoxBytes + warp * kGXRing * kGXBox;
  float4* red = reinterpret_cast<float4*>(smem_raw + (wt - smem_u32(smem_raw)) +
                                          (size_t)kGWarps * nch * kGBoxBytes +
                                          (NT == 1 ? (size_t)kGWarps * kGXRing * kGXBox : 0));

  if (threadIdx.x == 0) {
    for (int w = 0; w < kGWarps; ++w) mbar_init(smem_u32(&warp_b[w]), 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();
  if (POOL && blockIdx.x == 0 && threadIdx.x == 32) {
    // the norm weights, read by the last CTA of each token block, into L2
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(p.w_pre_norm),
                 "r"((uint32_t)(p.M * 2))
                 : "memory");
  }
  if (threadIdx.x == 0) {
    // the weight tile does not depend on the previous kernel: load it now,
    // one copy per warp of its nch chunks x 16 rows x 64 (past the end of
    // the reduction the copy engine fills zeros; those chunks are skipped)
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(tw)) : "memory");
    for (int w = 0; w < kGWarps; ++w) {
      if (w * nch >= nbox) break;
      mbar_expect_tx(smem_u32(&warp_b[w]), (uint32_t)(nch * kGBoxBytes));
      tma_load_3d(wt + w * nch * kGBoxBytes, tw, 0, tile * kGTileRows, w * nch, smem_u32(&warp_b[w]));
    }
  }
  if constexpr (!POOL) {
    pdl_wait();  // x is the previous kernel's output
    pdl_launch_dependents();
  }
  // The pooler reads x without waiting: x is the router's input, final
  // before this launch starts (the router signals its dependents only after
  // its own wait for the kernel that writes x). It waits for the route
  // kernel before it exits.

  const int a_row = (lane & 7) + ((lane >> 3) & 1) * 8, a_u = lane >> 4;
  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[nt][i] = 0.f;
  const int b0 = warp * nch, b1 = min(b0 + nch, nbox), nb = max(0, b1 - b0);
  bool ok = true;
  if constexpr (NT == 1) {
    // box b0 + i into slot i % kGXRing: lane l copies the 16-byte units l and
    // l + 32 (token row u / 8, unit u % 8); rows past the last token repeat it
    auto issue_x = [&](int i) {
      if (i < nb) {
        const uint32_t slot = xring + (i % kGXRing) * kGXBox;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int pc = lane + 32 * h, r = pc >> 3, u = pc & 7;
          const uint16_t* src = p.x + (size_t)min(tbk * 8 + r, p.rows - 1) * p.K + (b0 + i) * kGBoxK + u * 8;
          cp_async16(slot + swz(r, u), src);
        }
      }
      cp_async_commit();
    };
#pragma unroll
    for (int i = 0; i < kGXRing; ++i) issue_x(i);
    if (nb > 0)
      ok = __all_sync(0xffffffffu, mbar_wait_or_abort(smem_u32(&warp_b[warp]), 0u, &abort_flag));
    const int b_row = lane & 7, b_u = lane >> 3;
    for (int i = 0; i < nb && ok; ++i) {
      cp_async_wait<kGXRing - 1>();  // box i has landed
      __syncwarp();
      const uint32_t box = wt + (b0 + i) * kGBoxBytes, xs = xring + (i % kGXRing) * kGXBox;
#pragma unroll
      for (int s2 = 0; s2 < 2; ++s2) {
        uint32_t bf[4];
        ldsm_x4(xs + swz(b_row, 4 * s2 + b_u), bf[0], bf[1], bf[2], bf[3]);
#pragma unroll
        for (int s1 = 0; s1 < 2; ++s1) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4(box + swz(a_row, 2 * (2 * s2 + s1) + a_u), a0, a1, a2, a3);
          mma_bf16_16816(acc[0], a0, a1, a2, a3, bf[2 * s1], bf[2 * s1 + 1]);
        }
      }
      __syncwarp();
      issue_x(i + kGXRing);  // the slot just read
    }
    cp_async_wait<0>();
  } else {
    // activation rows of this lane's tokens (lanes past the last token read
    // the last token's row; their results are never stored)
    const uint16_t* xr[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
      xr[nt] = p.x + (size_t)min(tbk * 8 * NT + nt * 8 + g, p.rows - 1) * p.K + 2 * q;
    // B fragments of box b's 4 k-steps: k 2q, 2q+1 and 2q+8, 2q+9 of token g
    auto load_b = [&](uint32_t (&f)[NT][4][2], int b) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int s4 = 0; s4 < 4; ++s4) {
          const uint16_t* xp = xr[nt] + b * kGBoxK + s4 * 16;
          f[nt][s4][0] = *reinterpret_cast<const uint32_t*>(xp);
          f[nt][s4][1] = *reinterpret_cast<const uint32_t*>(xp + 8);
        }
    };
    auto box_mma = [&](int b, const uint32_t (&f)[NT][4][2]) {
      const uint32_t box = wt + b * kGBoxBytes;
#pragma unroll
      for (int s4 = 0; s4 < 4; ++s4) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(box + swz(a_row, 2 * s4 + a_u), a0, a1, a2, a3);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(acc[nt], a0, a1, a2, a3, f[nt][s4][0], f[nt][s4][1]);
      }
    };
    uint32_t bf[2][NT][4][2];
    if (nb > 0) {
      load_b(bf[0], b0);
      ok = __all_sync(0xffffffffu, mbar_wait_or_abort(smem_u32(&warp_b[warp]), 0u, &abort_flag));
    }
    for (int b = b0; b < b1 && ok; b += 2) {
      if (b + 1 < b1) load_b(bf[1], b + 1);
      box_mma(b, bf[0]);
      if (b + 1 >= b1) break;
      if (b + 2 < b1) load_b(bf[0], b + 2);
      box_mma(b + 1, bf[1]);
    }
  }
  if (!ok && lane == 0 && !abort_flag) {
    abort_flag = 1;
    atomicOr(p.health, kHealthTimeout);
  }
  // the 8 warps' partial tiles, added in warp order
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
    red[(warp * NT + nt) * 32 + lane] = make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]);
  __syncthreads();
  if (warp < NT) {
    const int nt = warp;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kGWarps; ++w) {
      const float4 x = red[(w * NT + nt) * 32 + lane];
      v.x += x.x;
      v.y += x.y;
      v.z += x.z;
      v.w += x.w;
    }
    const int r_lo = tile * kGTileRows + g, r_hi = r_lo + 8;
    const float lo[2] = {v.x, v.y}, hi[2] = {v.z, v.w};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int t = tbk * 8 * NT + nt * 8 + 2 * q + h;
      if (t >= p.rows) continue;
      if (r_lo < p.M) p.y[(size_t)t * p.M + r_lo] = lo[h];
      if (r_hi < p.M) p.y[(size_t)t * p.M + r_hi] = hi[h];
    }
  }
  if (threadIdx.x == 0 && abort_flag) {
    for (int w = 0; w < kGWarps && w * nch < nbox; ++w) {
      const unsigned long long t0 = globaltimer();
      while (!mbar_try_wait(smem_u32(&warp_b[w]), 0u))
        if (globaltimer() - t0 > kWaitLimitNs) break;
    }
  }
  if (POOL && !p.norm_in_tail) {
    // the norm is the next launch; this one completes only after the router
    pdl_wait();
    pdl_launch_dependents();
  } else if constexpr (POOL) {
    // the CTA that stores a token block's last tile (atomic ticket, no
    // waiting) normalizes the block's rows: the barrier orders the CTA's y
    // stores before thread 0's fence and ticket; the last CTA's thread 0
    // fences after the ticket (before its reset for the next launch, so the
    // fence has no store of its own to wait for), and the barrier orders
    // its reads after that
    __shared__ int last;
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      last = (atomicAdd(p.norm_ticket + tbk, 1) == tiles - 1);
      if (last) {
        __threadfence();
        p.norm_ticket[tbk] = 0;
      }
    }
    __syncthreads();
    // The expert kernel after this one reads the routing before its own
    // wait: dependents launch only once the router (which routes in its
    // tail) has completed. In the CTA that applies the norm only warp 0
    // waits and signals (then normalizes its rows): the norm reads nothing
    // the router writes, and the expert kernel's weight copies overlap it.
    if (!last || warp == 0) {
      pdl_wait();
      pdl_launch_dependents();
    }
    if (last) norm_rows(p, tbk * 8 * NT, min(p.rows, (tbk + 1) * 8 * NT));
  }
}

template <int NT, bool POOL>
__global__ void __launch_bounds__(kGThreads)
    k_gemv(const __grid_constant__ CUtensorMap tw, FrontParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  gemv_cta<NT, POOL>(&tw, p, smem);
}

// The pre-expert norm of eight rows per CTA (the pooler ran as a dense
// tensor-core GEMM): the expert kernel launched next reads the routing
// before its own wait, so this kernel lets it launch only after its own wait
// (the pooler, and the router before it, have completed).
__global__ void __launch_bounds__(kGThreads) k_pool_norm(FrontParams p) {
  pdl_wait();
  pdl_launch_dependents();
  const int t0 = blockIdx.x * kGWarps;
  norm_rows(p, t0, min(p.rows, t0 + kGWarps));
}

template <int EPL, int EG, int NCOL>
__global__ void __launch_bounds__(kGThreads) k_router(FrontParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  router_cta<EPL, EG, NCOL>(p, blockIdx.x, smem);
}

// ---- host ------------------------------------------------------------------
namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

// 3-D bf16 view of a row-major [rows, K] tensor: (64 elements of a chunk,
// row, chunk), strides K * 2 bytes for a row and 128 bytes for a chunk; box
// (64, 16 rows, nch chunks) lands as nch [16 x 64] boxes, 128-byte swizzle;
// zero fill out of bounds.
cudaError_t make_map(CUtensorMap* m, const void* base, uint64_t K, uint64_t rows, uint32_t nch) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {(cuuint64_t)kGBoxK, rows, K / kGBoxK};
  const cuuint64_t strides[2] = {K * 2, (cuuint64_t)kGBoxK * 2};
  const cuuint32_t box[3] = {(cuuint32_t)kGBoxK, (cuuint32_t)kGTileRows, nch};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int NT, bool POOL>
cudaError_t launch_t(const FrontParams& p, cudaStream_t s, bool pdl) {
  CUtensorMap tw{};
  cudaError_t e = make_map(&tw, p.w, (uint64_t)p.K, (uint64_t)p.M, (uint32_t)g_chunks_per_warp(p.K));
  if (e != cudaSuccess) return e;
  const size_t smem = g_smem_bytes(p.K, NT);
  e = cudaFuncSetAttribute(k_gemv<NT, POOL>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.gemv_ctas);
  cfg.blockDim = dim3(kGThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_gemv<NT, POOL>, tw, p);
}
}  // namespace

int front_gemv_ctas(int M, int rows, int nt) {
  return ((M + kGTileRows - 1) / kGTileRows) * ((rows + 8 * nt - 1) / (8 * nt));
}
int front_max_k() { return kGMaxK; }

cudaError_t launch_pool_norm(const FrontParams& p, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((p.rows + kGWarps - 1) / kGWarps);
  cfg.blockDim = dim3(kGThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_pool_norm, p);
}

cudaError_t launch_front(const FrontParams& p, int nt, cudaStream_t s, bool pdl) {
  if (p.gemv_ctas == 0) return cudaSuccess;
  switch (nt) {
    case 1: return p.h ? launch_t<1, true>(p, s, pdl) : launch_t<1, false>(p, s, pdl);
    case 2: return p.h ? launch_t<2, true>(p, s, pdl) : launch_t<2, false>(p, s, pdl);
    case 4: return p.h ? launch_t<4, true>(p, s, pdl) : launch_t<4, false>(p, s, pdl);
    default: return cudaErrorInvalidValue;
  }
}

template <int EPL, int EG, int NCOL>
static cudaError_t launch_router_t(const FrontParams& p, cudaStream_t s, bool pdl) {
  size_t smem = (size_t)8 * p.K * 2;  // the 8 tokens' input rows
  if (p.route_tail) {
    // the route tail reuses it for the permute: ids, ranks, per-chunk histograms
    const size_t rt = (size_t)p.route.rows * p.route.k, nch = (rt + 31) / 32;
    const size_t need = ((rt * 2 + 15) & ~(size_t)15) + ((rt + 15) & ~(size_t)15) + nch * p.E * 2;
    smem = std::max(smem, (need + 15) & ~(size_t)15);
  }
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k_router<EPL, EG, NCOL>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.router_ctas / EG);
  cfg.blockDim = dim3(kGThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_router<EPL, EG, NCOL>, p);
}

template <int EG, int NCOL>
static cudaError_t launch_router_g(const FrontParams& p, cudaStream_t s, bool pdl) {
  if (p.E <= 32) return launch_router_t<1, EG, NCOL>(p, s, pdl);
  if (p.E <= 64) return launch_router_t<2, EG, NCOL>(p, s, pdl);
  if (p.E <= 128) return launch_router_t<4, EG, NCOL>(p, s, pdl);
  return launch_router_t<8, EG, NCOL>(p, s, pdl);
}

cudaError_t launch_router(const FrontParams& p, cudaStream_t s, bool pdl) {
  if (p.router_ctas == 0) return cudaSuccess;
  if (p.K / 4 > kRouterCols * kGThreads) return cudaErrorInvalidValue;
  // more than 8 rows: four experts per CTA where their weight columns fit the
  // registers (K <= 5 * 4 * 256) and the experts divide evenly
  if (p.rows > 8 && p.E % 4 == 0 && p.K / 4 <= kRouterCols4 * kGThreads)
    return launch_router_g<4, kRouterCols4>(p, s, pdl);
  return launch_router_g<1, kRouterCols>(p, s, pdl);
}

}  // namespace musemoe
