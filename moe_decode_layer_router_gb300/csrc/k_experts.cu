// Routed experts: grouped GEMV/GEMM over the selected experts only.
//
// Work item = (token group of one expert, tile of weight rows). Each CTA
// walks a contiguous run of items; its thread 0 streams the items' weight
// codes and block scales into a ring of shared-memory stages with 1-D bulk
// copies (cp.async.bulk, completion counted on one mbarrier per stage), a few
// items ahead of the 8 consumer warps. Every wait is bounded: past the limit
// the CTA raises a health bit and leaves. The consumer warps split the
// item's reduction dimension K (chunk c goes to warp c % 8) and sum their 8
// partial tiles in shared memory in a fixed order (deterministic).
//
// Kernel weight layout (written by musemoe_pack_experts): rows in groups of
// 8, each group stored chunk by chunk, [E][N/8][NC][8 rows][64 B] for codes
// and [E][N/8][NC][8 rows][SB B] for MXFP4 (SB = 4) / NVFP4 (SB = 8) scales,
// so an item is one or two contiguous blocks and the 8 rows of a chunk are
// 512 contiguous bytes (conflict-free 128-bit shared loads). Thread (g, q)
// of a warp reads 16 bytes of row g and of row g + 8:
//  * FP4: 8 k-steps of m16n8k16; within the 64-byte chunk, k-step j holds
//    elements 16j..16j+15 and thread q owns 16j+4q..16j+4q+3, so one k-step
//    never crosses a scale block. The e2m1 pairs become f16 pairs with one
//    cvt (exact). MXFP4 scales (UE8M0, per 32) multiply the fp32 partial of
//    each pair of k-steps; NVFP4 scales (e4m3, per 16) multiply the f16
//    operand (e2m1 * e4m3 is exact in f16) and the fp32 global scale
//    multiplies the result.
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

constexpr int kComputeWarps = 8;
constexpr int kExpertWarps = kComputeWarps;          // warps sharing one item's K
constexpr int kExpertThreads = (kComputeWarps + 2) * 32;  // + producer + epilogue
constexpr int kChunkBytes = 64;      // bytes of one weight row per thread-quad
constexpr int kGroupChunk = 8 * 64;  // bytes of one chunk of a row group
constexpr int kStageBudget = 64 * 1024;  // three CTAs per SM
constexpr int kMetaGroups = 8;  // token groups whose metadata a CTA keeps in shared memory
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

// Geometry of one work item's weights in a stage.
struct StageGeo {
  int NC;            // 64-byte chunks per row
  int code_group;    // code bytes of one row group (NC * 512)
  int scale_group;   // scale bytes of one row group
  int groups;        // row groups per item
  int stage_bytes;   // codes then scales, rounded up to 128
};

template <int Q, int ROLE, int RT>
__host__ __device__ __forceinline__ StageGeo stage_geo(int K) {
  StageGeo g;
  const int rowbytes = (Q == kFP8) ? K : K / 2;
  g.NC = rowbytes / kChunkBytes;
  g.code_group = g.NC * kGroupChunk;
  g.scale_group = (Q == kMXFP4) ? g.NC * 32 : (Q == kNVFP4) ? g.NC * 64 : 0;
  g.groups = (ROLE == 0) ? 2 : 2 * RT;
  g.stage_bytes = (g.groups * (g.code_group + g.scale_group) + 127) & ~127;
  return g;
}

// Thread 0: start the copies of item `item` into stage buffer `dst`.
template <int Q, int ROLE, int RT>
__device__ __forceinline__ void issue_item(const ExpertParams& p, const StageGeo& G, int e,
                                           int tile, uint32_t dst, uint32_t bar) {
  const int NG = p.N / 8;  // row groups per expert
  const uint8_t* sb = reinterpret_cast<const uint8_t*>(p.scale);
  mbar_expect_tx(bar, G.groups * (G.code_group + G.scale_group));
  if (ROLE == 0) {
    const int rg[2] = {tile, p.I / 8 + tile};  // gate rows, up rows
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const size_t gi = (size_t)e * NG + rg[h];
      bulk_g2s(dst + h * G.code_group, p.w + gi * G.code_group, G.code_group, bar);
      if (G.scale_group)
        bulk_g2s(dst + 2 * G.code_group + h * G.scale_group, sb + gi * G.scale_group,
                 G.scale_group, bar);
    }
  } else {
    const size_t gi = (size_t)e * NG + (size_t)tile * 2 * RT;
    bulk_g2s(dst, p.w + gi * G.code_group, G.groups * G.code_group, bar);
    if (G.scale_group)
      bulk_g2s(dst + G.groups * G.code_group, sb + gi * G.scale_group,
               G.groups * G.scale_group, bar);
  }
}

// The mma work of one 64-byte chunk of the fragment rows g (codes L, scales
// sl) and g + 8 (codes H, scales sh) against the n-tiles' B fragments, which
// `bfrag(nt, j)` returns: for FP4 the uint2 of k-step j (0..7), for FP8 the
// uint4 of both k-steps (j unused).
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

// Warp roles: warps 0..7 compute (each owns the chunks c with c % 8 == warp),
// warp 8 produces (its lane 0 issues the bulk copies), warp 9 finishes items
// (sums the 8 partial tiles, applies scales / SiLU * up, stores). Hand-offs:
// full[s] (copies landed), empty[s] (8 compute warps done with stage s),
// ready[r] / freed[r] for the two partial-tile buffers.
// BC: a compute warp keeps the B fragments of its (at most CPW) chunks in
// registers while consecutive items stay on one token group.
template <int Q, int ROLE, int NT, int RT, bool BC, int CPW>
__global__ void __launch_bounds__(kExpertThreads, (NT <= 2 && ROLE == 0 ? 3 : 1)) k_expert(ExpertParams p) {
  pdl_launch_dependents();
  pdl_wait();
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) unsigned long long full_b[8], empty_b[8], ready_b[2], freed_b[2];
  __shared__ int abort_flag;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, q = lane & 3;
  const StageGeo G = stage_geo<Q, ROLE, RT>(p.K);
  const int S = p.stages;
  constexpr int kSlots = RT * NT * 32;  // float4 slots of one warp's partial tile
  float4* red = reinterpret_cast<float4*>(smem + (size_t)S * G.stage_bytes);  // [2][8][slots]
  const int n_groups = __ldcg(p.counters + kNumGroups);
  const int tiles = (ROLE == 0) ? p.I / 8 : p.N / (16 * RT);
  const int n_items = n_groups * tiles;
  const int i0 = (int)((long long)n_items * blockIdx.x / gridDim.x);
  const int i1 = (int)((long long)n_items * (blockIdx.x + 1) / gridDim.x);
  const int mine = i1 - i0;
  const int kel = (Q == kFP8) ? 1 : 2;  // bytes per activation element
  const uint32_t stage0 = smem_u32(smem);

  // metadata of the token groups this CTA's items touch (the first
  // kMetaGroups of them; items of later groups read it from global memory)
  __shared__ int4 meta_g[kMetaGroups];
  __shared__ int meta_r[kMetaGroups][8 * NT];
  const int g_first = mine > 0 ? i0 / tiles : 0;
  const int g_count = mine > 0 ? min(kMetaGroups, (i1 - 1) / tiles - g_first + 1) : 0;
  for (int i = threadIdx.x; i < g_count; i += kExpertThreads)
    meta_g[i] = __ldcg(reinterpret_cast<const int4*>(p.groups) + g_first + i);
  if (threadIdx.x == 0) {
    for (int st = 0; st < S; ++st) {
      mbar_init(smem_u32(&full_b[st]), 1);
      mbar_init(smem_u32(&empty_b[st]), kComputeWarps);
    }
    for (int r = 0; r < 2; ++r) {
      mbar_init(smem_u32(&ready_b[r]), kComputeWarps);
      mbar_init(smem_u32(&freed_b[r]), 1);
    }
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();
  for (int i = threadIdx.x; i < g_count * 8 * NT; i += kExpertThreads) {
    const int gi = i / (8 * NT), n = i % (8 * NT);
    if (n < meta_g[gi].z) meta_r[gi][n] = __ldcg(p.route_list + meta_g[gi].y + n);
  }
  __syncthreads();  // the last CTA-wide barrier
  auto group_of = [&](int grp) -> int4 {
    const int gi = grp - g_first;
    return gi < kMetaGroups ? meta_g[gi] : __ldcg(reinterpret_cast<const int4*>(p.groups) + grp);
  };
  auto route_of = [&](int grp, int rbase, int n) -> int {
    const int gi = grp - g_first;
    return gi < kMetaGroups ? meta_r[gi][n] : __ldcg(p.route_list + rbase + n);
  };
  auto fail = [&]() {
    abort_flag = 1;
    atomicOr(p.health, kHealthTimeout);
  };

  if (warp == kComputeWarps) {
    // ---------------- producer ----------------
    if (lane == 0) {
      for (int n = 0; n < mine; ++n) {
        const int st = n % S, use = n / S;
        if (use > 0 && !mbar_wait_or_abort(smem_u32(&empty_b[st]), (uint32_t)(use - 1) & 1u,
                                           &abort_flag)) {
          if (!abort_flag) fail();
          break;
        }
        if (use > 0) asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
        const int it = i0 + n;
        issue_item<Q, ROLE, RT>(p, G, group_of(it / tiles).x, it % tiles,
                                stage0 + st * G.stage_bytes, smem_u32(&full_b[st]));
      }
      // the copies still in flight must land before the CTA leaves
      for (int st = 0; st < S && st < mine; ++st) {
        const int last = st + ((mine - 1 - st) / S) * S;  // last item issued into stage st
        const unsigned long long t0 = globaltimer();
        while (!mbar_try_wait(smem_u32(&full_b[st]), (uint32_t)(last / S) & 1u))
          if (globaltimer() - t0 > kWaitLimitNs) break;
      }
    }
    return;
  }

  if (warp == kComputeWarps + 1) {
    // ---------------- epilogue ----------------
    for (int n = 0; n < mine; ++n) {
      const int r = n & 1;
      const bool ok = __all_sync(0xffffffffu, mbar_wait_or_abort(smem_u32(&ready_b[r]),
                                                                (uint32_t)(n >> 1) & 1u, &abort_flag));
      if (!ok) {
        if (lane == 0 && !abort_flag) fail();
        break;
      }
      const int item = i0 + n;
      const int grp = item / tiles, tile = item % tiles;
      const int4 gd = group_of(grp);
      const int e = gd.x, rbase = gd.y, ntok = gd.z;
      const int ntile_act = (ntok + 7) >> 3;
      const float4* rb = red + (size_t)r * kComputeWarps * kSlots;
      for (int sl = lane; sl < kSlots; sl += 32) {
        const int ln = sl & 31, nt = (sl >> 5) % NT, rt = sl / (32 * NT);
        if (nt >= ntile_act) continue;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kComputeWarps; ++w) {
          const float4 x = rb[w * kSlots + sl];
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
            const int nn = n0 + h;
            if (nn >= ntok) continue;
            const int ro = route_of(grp, rbase, nn);
            float gt = gate[h], ut = up[h];
            if (Q == kFP8) {
              const float bs = __ldcg(p.b_scale + ro / p.k);
              gt *= bs;
              ut *= bs;
            }
            const float a = round_bf16(silu(gt) * ut);
            if (Q == kFP8) {
              reinterpret_cast<uint16_t*>(p.out)[(size_t)ro * p.I + i] = f32_to_bf16_bits(a);
            } else {
              reinterpret_cast<__half*>(p.out)[(size_t)ro * p.I + i] = __float2half_rn(a);
              if (!(fabsf(a) <= 65504.f)) atomicOr(p.health, kHealthActRange);
            }
          }
        } else {
          const int plo = tile * 16 * RT + rt * 16 + ge, phi = plo + 8;
          float sl2 = gsc, sh2 = gsc;
          if (Q == kFP8) {
            const float* ws = reinterpret_cast<const float*>(p.scale);
            sl2 = __ldg(ws + (size_t)e * p.N + plo);
            sh2 = __ldg(ws + (size_t)e * p.N + phi);
          }
          const float lo[2] = {v.x * sl2, v.y * sl2};
          const float hi[2] = {v.z * sh2, v.w * sh2};
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int nn = n0 + h;
            if (nn >= ntok) continue;
            const int ro = route_of(grp, rbase, nn);
            const float bs = (Q == kFP8) ? __ldcg(p.b_scale + ro) : 1.f;
            float* y = reinterpret_cast<float*>(p.out) + (size_t)ro * p.P;
            y[plo] = lo[h] * bs;
            y[phi] = hi[h] * bs;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&freed_b[r]));
    }
    return;
  }

  // ---------------- compute warps ----------------
  int cached_grp = -1;
  uint2 bcache4[BC && Q != kFP8 ? CPW : 1][BC && Q != kFP8 ? NT : 1][8];
  uint4 bcache8[BC && Q == kFP8 ? CPW : 1][BC && Q == kFP8 ? NT : 1];
  (void)bcache4;
  (void)bcache8;
  for (int n = 0; n < mine; ++n) {
    const int item = i0 + n;
    const int st = n % S;
    const uint32_t phase = (uint32_t)(n / S) & 1u;
    const int grp = item / tiles;
    const int4 gd = group_of(grp);
    const int rbase = gd.y, ntok = gd.z;
    const int ntile_act = (ntok + 7) >> 3;
    const uint8_t* brow[NT];
    if (!BC || grp != cached_grp) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int nn = nt * 8 + g;
        brow[nt] = nullptr;
        if (nn < ntok) {
          const int ro = route_of(grp, rbase, nn);
          const int br = p.b_by_token ? ro / p.k : ro;
          brow[nt] = p.b + (size_t)br * p.K * kel;
        }
      }
    }
    if constexpr (BC) {
      if (grp != cached_grp) {  // fetch this warp's B fragments of the new group
        cached_grp = grp;
#pragma unroll
        for (int u = 0; u < CPW; ++u) {
          const int c = warp + kComputeWarps * u;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const bool v = c < G.NC && brow[nt] != nullptr;
            if constexpr (Q == kFP8) {
              bcache8[u][nt] = v ? ld_act_v4(brow[nt] + (size_t)c * 64 + q * 16) : make_uint4(0, 0, 0, 0);
            } else {
#pragma unroll
              for (int j = 0; j < 8; ++j)
                bcache4[u][nt][j] =
                    v ? ld_act_v2(brow[nt] + ((size_t)c * 128 + 16 * j + 4 * q) * 2) : make_uint2(0, 0);
            }
          }
        }
      }
    }
    if (!__all_sync(0xffffffffu, mbar_wait_or_abort(smem_u32(&full_b[st]), phase, &abort_flag))) {
      if (lane == 0 && !abort_flag) fail();
      break;
    }
    const uint8_t* stg = smem + (size_t)st * G.stage_bytes;

    float acc[RT][NT][4];
#pragma unroll
    for (int rt = 0; rt < RT; ++rt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[rt][nt][i] = 0.f;

    // fragment rows g (lo) and g + 8 (hi) of row tile rt: their row groups
    auto chunk = [&](int c, int rt, auto&& bfrag) {
      const int glo = (ROLE == 0) ? 0 : 2 * rt, ghi = (ROLE == 0) ? 1 : 2 * rt + 1;
      const uint4 L = *reinterpret_cast<const uint4*>(stg + glo * G.code_group + c * kGroupChunk +
                                                      g * 64 + q * 16);
      const uint4 Hh = *reinterpret_cast<const uint4*>(stg + ghi * G.code_group + c * kGroupChunk +
                                                       g * 64 + q * 16);
      const uint8_t* sc = stg + G.groups * G.code_group;
      uint2 sl = make_uint2(0, 0), sh = make_uint2(0, 0);
      if (Q == kMXFP4) {
        sl.x = *reinterpret_cast<const uint32_t*>(sc + glo * G.scale_group + c * 32 + g * 4);
        sh.x = *reinterpret_cast<const uint32_t*>(sc + ghi * G.scale_group + c * 32 + g * 4);
      } else if (Q == kNVFP4) {
        sl = *reinterpret_cast<const uint2*>(sc + glo * G.scale_group + c * 64 + g * 8);
        sh = *reinterpret_cast<const uint2*>(sc + ghi * G.scale_group + c * 64 + g * 8);
      }
      chunk_mma<Q, NT>(acc[rt], L, Hh, sl, sh, ntile_act, bfrag);
    };
    if constexpr (BC) {
#pragma unroll
      for (int u = 0; u < CPW; ++u) {
        const int c = warp + kComputeWarps * u;
        if (c >= G.NC) break;
#pragma unroll
        for (int rt = 0; rt < RT; ++rt) {
          if constexpr (Q == kFP8)
            chunk(c, rt, [&](int nt, int) { return bcache8[u][nt]; });
          else
            chunk(c, rt, [&](int nt, int j) { return bcache4[u][nt][j]; });
        }
      }
    } else {
      for (int c = warp; c < G.NC; c += kComputeWarps) {
#pragma unroll
        for (int rt = 0; rt < RT; ++rt) {
          if constexpr (Q == kFP8)
            chunk(c, rt, [&](int nt, int) {
              return brow[nt] ? ld_act_v4(brow[nt] + (size_t)c * 64 + q * 16) : make_uint4(0, 0, 0, 0);
            });
          else
            chunk(c, rt, [&](int nt, int j) {
              return brow[nt] ? ld_act_v2(brow[nt] + ((size_t)c * 128 + 16 * j + 4 * q) * 2)
                              : make_uint2(0, 0);
            });
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty_b[st]));  // stage st may be refilled

    // hand the partial tile to the epilogue warp
    const int r = n & 1;
    if (n >= 2 && !__all_sync(0xffffffffu,
                              mbar_wait_or_abort(smem_u32(&freed_b[r]),
                                                 (uint32_t)((n >> 1) - 1) & 1u, &abort_flag))) {
      if (lane == 0 && !abort_flag) fail();
      break;
    }
    float4* mine_red = red + ((size_t)r * kComputeWarps + warp) * kSlots;
#pragma unroll
    for (int rt = 0; rt < RT; ++rt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        if (nt < ntile_act)
          mine_red[(rt * NT + nt) * 32 + lane] =
              make_float4(acc[rt][nt][0], acc[rt][nt][1], acc[rt][nt][2], acc[rt][nt][3]);
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&ready_b[r]));
  }
}

template <int Q, int ROLE, int NT, int RT>
static void expert_smem_t(int K, int* stages, size_t* smem) {
  const StageGeo G = stage_geo<Q, ROLE, RT>(K);
  const size_t red = (size_t)2 * kComputeWarps * RT * NT * 32 * sizeof(float4);
  int S = (int)((kStageBudget > (int)red ? kStageBudget - (int)red : 0) / G.stage_bytes);
  S = S < 2 ? 2 : (S > 8 ? 8 : S);
  *stages = S;
  *smem = (size_t)S * G.stage_bytes + red;
}

using ExpertKernel = void (*)(ExpertParams);

// The instantiation for reduction length K: B fragments cached in registers
// when the token tile is small and the warp's chunks fit the cache.
template <int Q, int ROLE, int NT, int RT>
static ExpertKernel expert_kernel(int K) {
  constexpr int CPW = (Q == kFP8) ? 4 : 2;
  const int NC = stage_geo<Q, ROLE, RT>(K).NC;
  if constexpr (NT <= 2) {
    if (NC <= kExpertWarps * CPW) return k_expert<Q, ROLE, NT, RT, true, CPW>;
  }
  return k_expert<Q, ROLE, NT, RT, false, CPW>;
}

template <int Q, int ROLE, int NT, int RT>
static cudaError_t launch_expert_t(const ExpertParams& p, cudaStream_t s, bool pdl) {
  int S;
  size_t smem;
  expert_smem_t<Q, ROLE, NT, RT>(p.K, &S, &smem);
  const ExpertKernel kern = expert_kernel<Q, ROLE, NT, RT>(p.K);
  if (smem > 48 * 1024) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  ExpertParams q = p;
  q.stages = S;
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
  return cudaLaunchKernelEx(&cfg, kern, q);
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
static int occ_t(int K) {
  int n = 0, S;
  size_t smem;
  expert_smem_t<Q, ROLE, NT, RT>(K, &S, &smem);
  const ExpertKernel kern = expert_kernel<Q, ROLE, NT, RT>(K);
  if (smem > 48 * 1024)
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kExpertThreads, smem) != cudaSuccess)
    return 1;
  return n > 0 ? n : 1;
}
template <int Q, int ROLE>
static int occ_q(int nt, int K) {
  switch (nt) {
    case 1: return occ_t<Q, ROLE, 1, ROLE == 1 ? 2 : 1>(K);
    case 2: return occ_t<Q, ROLE, 2, ROLE == 1 ? 2 : 1>(K);
    case 4: return occ_t<Q, ROLE, 4, 1>(K);
    default: return occ_t<Q, ROLE, 8, 1>(K);
  }
}
int expert_ctas_per_sm(int quant, int role, int nt, int K) {
  switch (quant * 2 + role) {
    case 0: return occ_q<kMXFP4, 0>(nt, K);
    case 1: return occ_q<kMXFP4, 1>(nt, K);
    case 2: return occ_q<kNVFP4, 0>(nt, K);
    case 3: return occ_q<kNVFP4, 1>(nt, K);
    case 4: return occ_q<kFP8, 0>(nt, K);
    default: return occ_q<kFP8, 1>(nt, K);
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
  const int t = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int NW = kFinalizeThreads / 32;
  const int P4 = p.P / 4;
  const bool stash = p.stash != 0;
  const float4* y4 = reinterpret_cast<const float4*>(p.y) + (size_t)t * p.k * P4;
  for (int j = threadIdx.x; j < p.k; j += kFinalizeThreads) wt[j] = __ldcg(p.weights + (size_t)t * p.k + j);
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
        v[u] = (j0 + u < p.k && i < P4) ? __ldcg(y4 + (size_t)(j0 + u) * P4 + i)
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
      const float4 v = stash ? fsm4[(size_t)j * P4 + i] : __ldcg(y4 + (size_t)j * P4 + i);
      const float r = rstd[j], c = wt[j];
      a0 = fmaf(c, (v.x * r) * w0, a0);
      a1 = fmaf(c, (v.y * r) * w1, a1);
      a2 = fmaf(c, (v.z * r) * w2, a2);
      a3 = fmaf(c, (v.w * r) * w3, a3);
    }
    uint2 o;
    o.x = (uint32_t)f32_to_bf16_bits(a0) | ((uint32_t)f32_to_bf16_bits(a1) << 16);
    o.y = (uint32_t)f32_to_bf16_bits(a2) | ((uint32_t)f32_to_bf16_bits(a3) << 16);
    reinterpret_cast<uint2*>(p.moe_out + (size_t)t * p.P)[i] = o;
  }
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

// ---- weight re-layout: plain rows -> kernel layout --------------------------
// One CTA per group of 8 consecutive rows: the group's bytes are read into
// shared memory, then written back interleaved, so src may equal dst.
// Kernel layout of a [rows, row_bytes] tensor whose row is cut into `nc`
// chunks of `cb` bytes: [rows / 8][nc][8][cb]. With `permute_fp4`, the 64
// bytes of each chunk are also reordered (byte 8j + 2q + b -> 16q + 2j + b).
// Raises *bad when a byte of [p, p + n) is 0x00 or 0xFF (UE8M0 codes the
// kernels do not take).
__global__ void k_check_ue8m0(const uint8_t* p, size_t n, int* bad) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x)
    if (p[i] == 0x00 || p[i] == 0xFF) *bad = 1;
}

cudaError_t check_ue8m0(const uint8_t* p, size_t n, int* bad_dev, cudaStream_t s) {
  k_check_ue8m0<<<1024, 256, 0, s>>>(p, n, bad_dev);
  return cudaGetLastError();
}

__global__ void k_pack_rows(const uint8_t* src, uint8_t* dst, int row_bytes, int cb,
                            int permute_fp4) {
  extern __shared__ __align__(16) uint8_t blk[];
  const size_t base = (size_t)blockIdx.x * 8 * row_bytes;
  const int nbytes = 8 * row_bytes;
  for (int i = threadIdx.x * 4; i < nbytes; i += blockDim.x * 4)
    *reinterpret_cast<uint32_t*>(blk + i) = *reinterpret_cast<const uint32_t*>(src + base + i);
  __syncthreads();
  const int nc = row_bytes / cb;
  for (int o = threadIdx.x; o < nbytes; o += blockDim.x) {
    const int c = o / (8 * cb), r = (o / cb) % 8;
    int b = o % cb;
    if (permute_fp4) {  // o's byte within the chunk is 16q + 2j + bb
      const int qq = b >> 4, j = (b >> 1) & 7, bb = b & 1;
      b = 8 * j + 2 * qq + bb;
    }
    dst[base + o] = blk[r * row_bytes + c * cb + b];
    (void)nc;
  }
}

cudaError_t launch_pack_rows(const uint8_t* src, uint8_t* dst, size_t rows, int row_bytes, int cb,
                             bool permute_fp4, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  const size_t smem = (size_t)8 * row_bytes;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k_pack_rows, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  k_pack_rows<<<(unsigned)(rows / 8), 256, smem, s>>>(src, dst, row_bytes, cb, permute_fp4 ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace musemoe
