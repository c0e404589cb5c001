// Routed experts: grouped GEMV / GEMM over the selected experts only, in
// Stream-K form. Every compute warp owns 16 weight rows of a tile for the
// whole reduction K, so the dot products, the SiLU * up of w13 and the stores
// all stay in the warp's registers.
//
// Tiles: w13 (role 0) takes 64 i per CTA tile, warp w the 8 gate rows
// i0 + 8w .. +7 and the matching 8 up rows I + i0 + 8w .. (the two halves of
// the fused matrix are gate then up); thread (g, q) then holds gate and up of
// the same (i, token) in its accumulator fragment. w2 (role 1) takes 128 P
// rows per CTA tile, 16 per warp. The w13 activation is stored as bf16 (the
// MoE activations are bf16: page "vllm.models.muse_spark.amd.mono",
// maybe_attach_mono), as f16 for the FP4 w2 operand; w2 writes one
// unweighted fp32 row per route (page "vllm.models.muse_spark.amd.
// muse_moe_runner", MuseSparkAiterExperts: unit router weights, the
// weighting comes after the post-expert norm).
//
// Work units = (token group, tile, K-slice of 4 64-byte chunks), numbered in
// that order; CTA c runs units [U c / G, U (c + 1) / G) of the U units, so
// every CTA streams the same number of weight bytes. A tile whose slices
// span several CTAs leaves one fp32 partial per CTA and warp; the CTA that
// holds the tile's last unit owns it: each of its warps waits (bounded) until
// the tile's other CTAs have signalled their partials through the tile's
// ticket, then adds the partials in CTA order, so results do not depend on
// scheduling.
//
// Data movement: a producer lane streams each unit into a ring of shared
// memory stages with 1-D bulk copies (cp.async.bulk), completion counted on
// one mbarrier per stage: the unit's codes and block scales are two
// contiguous blocks each in the kernel layout ([E][N/64][slice][8 groups]
// [chunks][8 rows][64 B]); the group's activation rows of the slice (up to
// 8 per token tile) come along (padded rows, conflict-free fragment reads).
// The 8 compute warps release a
// stage through a second mbarrier. Every wait is bounded: past the limit the
// CTA raises a health bit and leaves.
//
// Fragments (m16n8k16 f16 for FP4, m16n8k32 e4m3 for FP8): thread (g, q)
// reads 16 bytes of fragment rows g and g + 8 per 64-byte chunk. FP4: 8
// k-steps, k-step j holding chunk elements 16j..16j+15 with thread q owning
// 16j+4q..+3 (the pack reorders each chunk's bytes for this), e2m1 pairs
// converted to f16 with one cvt (exact); MXFP4 scales (UE8M0 per 32)
// multiply the fp32 partial of each pair of k-steps, NVFP4 scales (e4m3 per
// 16) the f16 operand (exact), the fp32 global scale the result. FP8: 2
// k-steps; the per-row weight scale and per-row activation scale multiply
// the fp32 result.
#include "pipeline.cuh"

namespace musemoe {

constexpr int kXWarps = 8;                      // compute warps
constexpr int kXThreads = (kXWarps + 1) * 32;   // + producer warp
constexpr int kXMeta = 8;                       // token groups cached in shared memory
constexpr int kXSmemBudget = 112 * 1024;        // two CTAs per SM
constexpr int kXCodeBlock = 8 * kSliceChunks * 512;  // codes of one row tile's slice (16 KB)

struct XGeo {
  int NC;           // 64-byte chunks per weight row
  int KS;           // K-slices per tile
  int tiles;        // CTA tiles per token group
  int SB;           // scale bytes per row and chunk (MX 4, NV 8, FP8 0)
  int cbB;          // activation bytes of one chunk (FP4 128 f16, FP8 64 e4m3)
  int RS;           // stride of an activation row in the stage
  int scale_off;    // stage: codes [2][8][slots][8][64] | scales [2][8][slots][8][SB] | B [8][RS]
  int b_off;
  int stage_bytes;
};

template <int Q, int ROLE, int NT>
__host__ __device__ __forceinline__ XGeo x_geo(int K, int N) {
  XGeo g;
  const int rowbytes = (Q == kFP8) ? K : (Q == kBF16) ? 2 * K : K / 2;
  g.NC = rowbytes / 64;
  g.KS = (g.NC + kSliceChunks - 1) / kSliceChunks;
  g.tiles = (ROLE == 0) ? (N / 2) / 64 : N / 128;
  g.SB = (Q == kMXFP4) ? 4 : (Q == kNVFP4) ? 8 : 0;
  g.cbB = (Q == kFP8 || Q == kBF16) ? 64 : 256;  // activation bytes of one 64-byte code chunk
  g.RS = kSliceChunks * g.cbB + 32;
  g.scale_off = 2 * kXCodeBlock;
  g.b_off = g.scale_off + 2 * 8 * kSliceChunks * 8 * g.SB;
  g.stage_bytes = (g.b_off + 8 * NT * g.RS + 127) & ~127;
  return g;
}

// Index of the CTA whose unit range holds unit u (units [U c / G, U (c+1) / G)).
__device__ __forceinline__ int x_cta_of(long long u, long long U, int G) {
  return (int)(((u + 1) * G - 1) / U);
}
__device__ __forceinline__ long long x_start(int c, long long U, int G) { return U * c / G; }

// Two CTAs per SM where the accumulators fit the register share; one for the
// widest token tiles.
template <int Q, int NT>
constexpr int x_min_blocks() {
  return NT >= 4 ? 1 : 2;
}

template <int Q, int ROLE, int NT>
__global__ void __launch_bounds__(kXThreads, x_min_blocks<Q, NT>()) k_expert(ExpertParams p) {
  // The groups, route lists and counters below are the route kernel's
  // output, complete before this launch starts: the kernel launched between
  // the two (the pooler, or w13 for w2) signals its dependents only after it
  // has waited for its own predecessor. What the previous kernel writes (the
  // activations) is read only after pdl_wait: by the producer before its
  // activation copies, by the compute warps before anything else.
  pdl_launch_dependents();
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) unsigned long long full_b[8], empty_b[8];
  __shared__ int abort_flag;
  __shared__ int4 meta_g[kXMeta];
  __shared__ int meta_r[kXMeta][8 * NT];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, q = lane & 3;
  const XGeo G = x_geo<Q, ROLE, NT>(p.K, p.N);
  const int S = p.stages;
  const int n_groups = __ldcg(p.counters + kNumGroups);
  const long long per_group = (long long)G.tiles * G.KS;
  const long long U = (long long)n_groups * per_group;
  // CTAs beyond the unit count get no work; the partition uses the others,
  // so that every CTA of a tile's contributor range holds units of it
  const int GE = (int)min((long long)gridDim.x, U);
  const long long u0 = blockIdx.x < GE ? x_start(blockIdx.x, U, GE) : 0;
  const long long u1 = blockIdx.x < GE ? x_start(blockIdx.x + 1, U, GE) : 0;
  const int kel = (Q == kFP8) ? 1 : 2;  // bytes per activation element
  const uint32_t stage0 = smem_u32(smem);
  // Processing order of the CTA's units: its whole tiles [b0, b1), then the
  // units [b1, u1) of the tile it shares with the next CTA (it holds that
  // tile's first units and only leaves a partial), then the units [u0, b0)
  // of the tile it shares with the previous CTA (it holds that tile's last
  // unit: it waits for the other partials and finishes the tile). A range
  // inside one tile is a single leave-a-partial part. Only owners wait, and
  // an owner's part comes after everything the CTA's own partials need, so
  // no wait depends on a waiting CTA.
  // (unit indices fit in 32 bits: groups x tiles x slices)
  const int U0 = (int)u0, U1 = (int)u1, KS = G.KS, PG = (int)per_group;
  int b0 = (U0 + KS - 1) / KS * KS, b1 = U1 / KS * KS;
  if (b0 > b1) b0 = b1 = U0;  // inside one tile: [u0, u1) is the "next-CTA" part
  const int nM = b1 - b0, nE = U1 - b1;
  const int count = U1 - U0;
  // walks the units in processing order: unit index, its group, tile and
  // slice, and the bounds of its part; divisions only where a part starts
  struct Walk {
    int u, grp, tile, slice, lo, hi, part, left;
  };
  auto walk_begin = [&](Walk& w) {
    w.part = -1;
    w.left = 0;
  };
  // the three parts as (first unit, end) in processing order: [b0, b1),
  // [b1, U1), [U0, b0) (selects, not an indexed array: no local memory)
  auto part_lo = [&](int i) { return i == 0 ? b0 : (i == 1 ? b1 : U0); };
  auto part_hi = [&](int i) { return i == 0 ? b1 : (i == 1 ? U1 : b0); };
  auto walk_next = [&](Walk& w) {
    if (w.left == 0) {
      do {
        ++w.part;
      } while (w.part < 3 && part_hi(w.part) <= part_lo(w.part));
      w.lo = part_lo(w.part);
      w.hi = part_hi(w.part);
      w.left = w.hi - w.lo;
      w.u = w.lo;
      w.grp = w.u / PG;
      const int rem = w.u - w.grp * PG;
      w.tile = rem / KS;
      w.slice = rem - w.tile * KS;
    } else {
      ++w.u;
      if (++w.slice == KS) {
        w.slice = 0;
        if (++w.tile == G.tiles) {
          w.tile = 0;
          ++w.grp;
        }
      }
    }
    --w.left;
  };
  (void)nM;
  (void)nE;

  const int g_first = (u1 > u0) ? (int)(u0 / per_group) : 0;
  const int g_count = (u1 > u0) ? min(kXMeta, (int)((u1 - 1) / per_group) - g_first + 1) : 0;
  for (int i = threadIdx.x; i < g_count; i += kXThreads)
    meta_g[i] = __ldcg(reinterpret_cast<const int4*>(p.groups) + g_first + i);
  if (threadIdx.x == 0) {
    for (int st = 0; st < S; ++st) {
      mbar_init(smem_u32(&full_b[st]), 1);
      mbar_init(smem_u32(&empty_b[st]), kXWarps);
    }
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();
  for (int i = threadIdx.x; i < g_count * 8 * NT; i += kXThreads) {
    const int gi = i / (8 * NT), n = i % (8 * NT);
    if (n < meta_g[gi].z) meta_r[gi][n] = __ldcg(p.route_list + meta_g[gi].y + n);
  }
  __syncthreads();  // the last CTA-wide barrier
  auto group_of = [&](int grp) -> int4 {
    const int gi = grp - g_first;
    int4 r;
    if (gi < kXMeta) r = meta_g[gi];
    else r = __ldcg(reinterpret_cast<const int4*>(p.groups) + grp);
    return r;
  };
  auto route_of = [&](int grp, int rbase, int n) -> int {
    const int gi = grp - g_first;
    int r;
    if (gi < kXMeta) r = meta_r[gi][n];
    else r = __ldcg(p.route_list + rbase + n);
    return r;
  };
  auto b_row = [&](int ro) -> const uint8_t* {  // activation row of route ro
    return p.b + (size_t)(p.b_by_token ? ro / p.k : ro) * p.K * kel;
  };
  auto fail = [&]() {
    abort_flag = 1;
    atomicOr(p.health, kHealthTimeout);
  };

  if (warp == kXWarps) {
    // ---------------- producer ----------------
    if (lane == 0) {
      const int NRT = p.N / 64;  // row tiles per expert
      const size_t tile_codes = (size_t)G.NC * 4096, tile_scales = (size_t)G.NC * 64 * G.SB;
      const uint8_t* sb = reinterpret_cast<const uint8_t*>(p.scale);
      int n = 0;
      Walk wk;
      walk_begin(wk);
      int gcur = -1;
      int4 gd = make_int4(0, 0, 0, 0);
      // the weights are read once: their lines leave L2 first
      const uint64_t pol_first = l2_policy_evict_first();
      // the weight tiles and block scales of a unit into stage st
      auto issue_w = [&](int st, int e_id, int tile, int slice, int nc) {
        const uint32_t dst = stage0 + st * G.stage_bytes;
        const uint32_t bar = smem_u32(&full_b[st]);
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
          const int rt = (ROLE == 0) ? (blk == 0 ? tile : p.I / 64 + tile) : 2 * tile + blk;
          const size_t ti = (size_t)e_id * NRT + rt;
          bulk_g2s_hint(dst + blk * kXCodeBlock,
                        p.w + ti * tile_codes + (size_t)slice * kSliceChunks * 4096, nc * 4096, bar,
                        pol_first);
          if (G.SB)
            bulk_g2s_hint(dst + G.scale_off + blk * 8 * kSliceChunks * 8 * G.SB,
                          sb + ti * tile_scales + (size_t)slice * kSliceChunks * 64 * G.SB,
                          nc * 64 * G.SB, bar, pol_first);
        }
      };
      // the activation rows of a unit (its group's tokens) into stage st
      auto issue_b = [&](int st, int grp, const int4& g4, int slice, int nc) {
        const uint32_t dst = stage0 + st * G.stage_bytes;
        const uint32_t bar = smem_u32(&full_b[st]);
        for (int t = 0; t < g4.z; ++t)
          bulk_g2s(dst + G.b_off + t * G.RS,
                   b_row(route_of(grp, g4.y, t)) + (size_t)slice * kSliceChunks * G.cbB, nc * G.cbB,
                   bar);
      };
      // The first S units' weights go out before the wait for the previous
      // kernel (they depend only on the routing); their activation rows
      // after it.
      const int n_early = min(S, count);
      bool waited = false;
      // after the wait: the activation rows of the early units, found by a
      // second walk over them
      auto issue_early_b = [&]() {
        Walk w2;
        walk_begin(w2);
        int gc = -1;
        int4 g4 = make_int4(0, 0, 0, 0);
        for (int m = 0; m < n_early; ++m) {
          walk_next(w2);
          if (w2.grp != gc) {
            gc = w2.grp;
            g4 = group_of(gc);
          }
          issue_b(m, gc, g4, w2.slice, min(kSliceChunks, G.NC - w2.slice * kSliceChunks));
        }
      };
      int st = -1, use = 0;  // stage of unit n and how often it was filled before
      for (; n < count; ++n) {
        walk_next(wk);
        const int grp = wk.grp, tile = wk.tile, slice = wk.slice;
        if (grp != gcur) {
          gd = group_of(grp);
          gcur = grp;
        }
        if (++st == S) {
          st = 0;
          ++use;
        }
        if (n == n_early && !waited) {
          pdl_wait();
          waited = true;
          issue_early_b();
        }
        if (use > 0 && !mbar_wait_or_abort(smem_u32(&empty_b[st]), (uint32_t)(use - 1) & 1u,
                                           &abort_flag)) {
          if (!abort_flag) fail();
          break;
        }
        if (use > 0) asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
        const int nc = min(kSliceChunks, G.NC - slice * kSliceChunks);
        uint32_t bytes = 2u * nc * (4096 + 64 * G.SB);
        bytes += (uint32_t)(gd.z * nc * G.cbB);
        mbar_expect_tx(smem_u32(&full_b[st]), bytes);
        issue_w(st, gd.x, tile, slice, nc);
        if (n >= n_early) issue_b(st, grp, gd, slice, nc);
      }
      if (!waited && n == n_early) {
        // every unit was early (count <= S)
        pdl_wait();
        waited = true;
        issue_early_b();
      }
      // the copies still in flight must land before the CTA leaves
      const int issued = n;
      for (int st = 0; st < S && st < issued; ++st) {
        const int last = st + ((issued - 1 - st) / S) * S;  // last unit issued into stage st
        const unsigned long long t0 = globaltimer();
        while (!mbar_try_wait(smem_u32(&full_b[st]), (uint32_t)(last / S) & 1u))
          if (globaltimer() - t0 > kWaitLimitNs) break;
      }
    }
    return;
  }

  // ---------------- compute warps ----------------
  pdl_wait();  // the activations, partial slots and outputs of the previous kernel
  int grp = 0, tile = 0, slice = 0;
  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[nt][i] = 0.f;
  int ntok = 0, rbase = 0, e = 0, ntile_act = 0;
  bool fresh = true;  // the next unit starts a tile (or this CTA's range)
  // the warp's two fragment row groups in the stage: (code block, group)
  const int blk_lo = (ROLE == 0) ? 0 : warp / 4, blk_hi = (ROLE == 0) ? 1 : warp / 4;
  const int gi_lo = (ROLE == 0) ? warp : 2 * (warp % 4), gi_hi = (ROLE == 0) ? warp : 2 * (warp % 4) + 1;

  // the epilogue of one finished tile: scales, SiLU * up (w13), stores
  auto finish = [&](const float (&v)[NT][4]) {
    float gsc = 1.f;
    if (Q == kNVFP4) gsc = __ldg(p.gscale + e);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      if (nt >= ntile_act) break;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int nn = nt * 8 + 2 * q + h;
        if (nn >= ntok) continue;
        const int ro = route_of(grp, rbase, nn);
        if (ROLE == 0) {
          const int i = tile * 64 + warp * 8 + g;
          float sg = gsc, su = gsc;
          if (Q == kFP8) {
            const float* ws = reinterpret_cast<const float*>(p.scale);
            const float bs = __ldcg(p.b_scale + ro / p.k);
            sg = __ldg(ws + (size_t)e * p.N + i) * bs;
            su = __ldg(ws + (size_t)e * p.N + p.I + i) * bs;
          }
          const float a = round_bf16(silu(v[nt][h] * sg) * (v[nt][2 + h] * su));
          if (Q == kFP8 || Q == kBF16 || p.act_bf16) {
            reinterpret_cast<uint16_t*>(p.out)[(size_t)ro * p.I + i] = f32_to_bf16_bits(a);
          } else {
            reinterpret_cast<__half*>(p.out)[(size_t)ro * p.I + i] = __float2half_rn(a);
            if (!(fabsf(a) <= 65504.f)) atomicOr(p.health, kHealthActRange);
          }
        } else {
          const int plo = tile * 128 + warp * 16 + g, phi = plo + 8;
          float sl2 = gsc, sh2 = gsc;
          if (Q == kFP8) {
            const float* ws = reinterpret_cast<const float*>(p.scale);
            const float bs = __ldcg(p.b_scale + ro);
            sl2 = __ldg(ws + (size_t)e * p.N + plo) * bs;
            sh2 = __ldg(ws + (size_t)e * p.N + phi) * bs;
          }
          float* y = reinterpret_cast<float*>(p.out) + (size_t)ro * p.P;
          y[plo] = v[nt][h] * sl2;
          y[phi] = v[nt][2 + h] * sh2;
        }
      }
    }
  };

  Walk wk;
  walk_begin(wk);
  int st = -1;          // stage of unit n
  uint32_t phase = 0u;  // parity of the stage's fill: (n / S) & 1
  for (int n = 0; n < count; ++n) {
    walk_next(wk);
    const int u = wk.u;
    grp = wk.grp;
    tile = wk.tile;
    slice = wk.slice;
    if (++st == S) {
      st = 0;
      phase ^= 1u;
    }
    if (fresh) {
      const int4 gd = group_of(grp);
      e = gd.x;
      rbase = gd.y;
      ntok = gd.z;
      ntile_act = (ntok + 7) >> 3;
      fresh = false;
    }
    const int c0 = slice * kSliceChunks;
    const int nc = min(kSliceChunks, G.NC - c0);
    const uint8_t* stg = smem + (size_t)st * G.stage_bytes;
    // A fragments (rows g and g + 8 of the warp's two row groups) and block
    // scales of chunk c of the stage
    auto load_a = [&](int c, uint4& L, uint4& Hh, uint2& sl, uint2& sh) {
      const int lo = gi_lo * nc + c, hi = gi_hi * nc + c;
      // FP8 blocks are stored 64-byte swizzled (unit q of row g at q ^ ((g >> 1) & 3))
      const int qs = (Q == kFP8) ? (q ^ ((g >> 1) & 3)) : q;
      L = *reinterpret_cast<const uint4*>(stg + blk_lo * kXCodeBlock + lo * 512 + g * 64 + qs * 16);
      Hh = *reinterpret_cast<const uint4*>(stg + blk_hi * kXCodeBlock + hi * 512 + g * 64 + qs * 16);
      sl = make_uint2(0, 0);
      sh = make_uint2(0, 0);
      const uint8_t* sc = stg + G.scale_off;
      if constexpr (Q == kMXFP4) {
        sl.x = *reinterpret_cast<const uint32_t*>(sc + blk_lo * 8 * kSliceChunks * 32 + lo * 32 + g * 4);
        sh.x = *reinterpret_cast<const uint32_t*>(sc + blk_hi * 8 * kSliceChunks * 32 + hi * 32 + g * 4);
      } else if constexpr (Q == kNVFP4) {
        sl = *reinterpret_cast<const uint2*>(sc + blk_lo * 8 * kSliceChunks * 64 + lo * 64 + g * 8);
        sh = *reinterpret_cast<const uint2*>(sc + blk_hi * 8 * kSliceChunks * 64 + hi * 64 + g * 8);
      }
    };
    const bool ok = __all_sync(0xffffffffu, mbar_wait_or_abort(smem_u32(&full_b[st]),
                                                               phase, &abort_flag));
    if (!ok) {
      if (lane == 0 && !abort_flag) fail();
      break;
    }
    if constexpr (NT == 1) {
      // one token tile: B fragments from the stage's activation rows, the
      // next chunk's read while the current one runs (two register buffers).
      // FP4: k-step j of chunk c is 4 f16 at element 128 c + 16 j + 4 q;
      // FP8: both k-steps of chunk c are 16 e4m3 at byte 64 c + 16 q;
      // BF16: k-step j of chunk c is the bf16 pairs at elements 32 c + 16 j
      // + 2 q and + 8 (the natural mma order).
      const uint8_t* bp =
          stg + G.b_off + min(g, ntok - 1) * G.RS + q * (Q == kFP8 ? 16 : Q == kBF16 ? 4 : 8);
      uint2 b4[2][8];
      uint4 b8[2];
      auto ldb = [&](int buf, int c) {
        if constexpr (Q == kFP8) {
          b8[buf] = *reinterpret_cast<const uint4*>(bp + c * 64);
        } else if constexpr (Q == kBF16) {
          const uint8_t* cp = bp + c * 64;
          b4[buf][0] = make_uint2(*reinterpret_cast<const uint32_t*>(cp),
                                  *reinterpret_cast<const uint32_t*>(cp + 16));
          b4[buf][1] = make_uint2(*reinterpret_cast<const uint32_t*>(cp + 32),
                                  *reinterpret_cast<const uint32_t*>(cp + 48));
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) b4[buf][j] = *reinterpret_cast<const uint2*>(bp + c * 256 + j * 32);
        }
      };
      ldb(0, 0);
      if (nc == kSliceChunks) {
#pragma unroll
        for (int c = 0; c < kSliceChunks; ++c) {
          if (c + 1 < kSliceChunks) ldb((c + 1) & 1, c + 1);
          uint4 L, Hh;
          uint2 sl, sh;
          load_a(c, L, Hh, sl, sh);
          if constexpr (Q == kFP8)
            chunk_mma<Q, 1>(acc, L, Hh, sl, sh, 1, [&](int, int) { return b8[c & 1]; });
          else
            chunk_mma<Q, 1>(acc, L, Hh, sl, sh, 1, [&](int, int j) { return b4[c & 1][j]; });
        }
      } else {
        // a ragged last slice (reduction length not a multiple of 4 chunks)
        for (int c = 0; c < nc; ++c) {
          if (c > 0) ldb(0, c);
          uint4 L, Hh;
          uint2 sl, sh;
          load_a(c, L, Hh, sl, sh);
          if constexpr (Q == kFP8)
            chunk_mma<Q, 1>(acc, L, Hh, sl, sh, 1, [&](int, int) { return b8[0]; });
          else
            chunk_mma<Q, 1>(acc, L, Hh, sl, sh, 1, [&](int, int j) { return b4[0][j]; });
        }
      }
    } else {
      // several token tiles: the B fragments of tile nt from the stage's
      // activation rows 8 nt + g, at the offsets of the one-tile case; lanes
      // past the group's last token read that token's row (their results
      // are never stored), so every fragment read is of a row this unit
      // copied
      const uint8_t* bpn[NT];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        bpn[nt] = stg + G.b_off + min(nt * 8 + g, ntok - 1) * G.RS +
                  q * (Q == kFP8 ? 16 : Q == kBF16 ? 4 : 8);
#pragma unroll
      for (int c = 0; c < kSliceChunks; ++c) {
        if (c >= nc) break;
        uint4 L, Hh;
        uint2 sl, sh;
        load_a(c, L, Hh, sl, sh);
        if constexpr (Q == kFP8)
          chunk_mma<Q, NT>(acc, L, Hh, sl, sh, ntile_act, [&](int nt, int) {
            return *reinterpret_cast<const uint4*>(bpn[nt] + c * 64);
          });
        else if constexpr (Q == kBF16)
          chunk_mma<Q, NT>(acc, L, Hh, sl, sh, ntile_act, [&](int nt, int j) {
            const uint8_t* e0 = bpn[nt] + c * 64 + 32 * j;
            return make_uint2(*reinterpret_cast<const uint32_t*>(e0),
                              *reinterpret_cast<const uint32_t*>(e0 + 16));
          });
        else
          chunk_mma<Q, NT>(acc, L, Hh, sl, sh, ntile_act, [&](int nt, int j) {
            return *reinterpret_cast<const uint2*>(bpn[nt] + c * 256 + j * 32);
          });
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty_b[st]));  // stage st may be refilled

    const bool tile_end = (slice == G.KS - 1);
    if (tile_end || u + 1 == wk.hi) {
      const int tb = u - slice;  // first unit of the tile
      if (tile_end && tb >= wk.lo) {
        finish(acc);
      } else {
        // the tile spans several CTAs; the one holding its last unit (tile_end)
        // owns it. A CTA without the last unit stores its partial and signals
        // (no fence, no wait); the owner waits for the others' signals and
        // adds all partials in CTA order.
        const int c_first = x_cta_of(tb, U, GE);
        const int c_last = x_cta_of(tb + G.KS - 1, U, GE);
        const int slot_sz = kXWarps * NT * 32;
        auto slot_of = [&](int c) -> size_t {
          const int which = (x_start(c, U, GE) >= tb) ? 0 : 1;
          return ((size_t)c * 2 + which) * slot_sz + (size_t)warp * NT * 32;
        };
        float4* part = reinterpret_cast<float4*>(p.part);
        int32_t* flag = p.tickets + ((size_t)grp * G.tiles + tile) * kXWarps + warp;
        if (!tile_end) {
          const size_t mine = slot_of(blockIdx.x);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            if (nt < ntile_act)
              part[mine + nt * 32 + lane] = make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]);
          __syncwarp();  // orders the lanes' stores before lane 0's release
          if (lane == 0) asm volatile("red.release.gpu.global.add.s32 [%0], 1;\n" ::"l"(flag) : "memory");
        } else {
          int got = 1;
          if (lane == 0) {
            const int want = c_last - c_first;
            int v = 0;
            asm volatile("ld.acquire.gpu.global.s32 %0, [%1];\n" : "=r"(v) : "l"(flag) : "memory");
            if (v < want) {
              const unsigned long long t0 = globaltimer();
              do {
                __nanosleep(256);
                asm volatile("ld.acquire.gpu.global.s32 %0, [%1];\n" : "=r"(v) : "l"(flag) : "memory");
              } while (v < want && globaltimer() - t0 <= kWaitLimitNs && !abort_flag);
            }
            got = (v >= want);
            if (got) *flag = 0;  // ready for the next launch
          }
          got = __shfl_sync(0xffffffffu, got, 0);
          __syncwarp();
          if (!got) {
            if (lane == 0 && !abort_flag) fail();
            break;
          }
          float v[NT][4];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) v[nt][i] = 0.f;
          for (int c = c_first; c < c_last; ++c) {
            const size_t sc = slot_of(c);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              if (nt >= ntile_act) break;
              const float4 x = __ldcg(part + sc + nt * 32 + lane);
              v[nt][0] += x.x;
              v[nt][1] += x.y;
              v[nt][2] += x.z;
              v[nt][3] += x.w;
            }
          }
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) v[nt][i] += acc[nt][i];
          finish(v);
        }
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[nt][i] = 0.f;
      fresh = true;
    }
  }
}

template <int Q, int ROLE, int NT>
static void x_smem(int K, int N, int* stages, size_t* smem) {
  const XGeo G = x_geo<Q, ROLE, NT>(K, N);
  int S = kXSmemBudget / G.stage_bytes;
  S = S < 2 ? 2 : (S > 8 ? 8 : S);
  *stages = S;
  *smem = (size_t)S * G.stage_bytes;
}

template <int Q, int ROLE, int NT>
static cudaError_t launch_x_t(const ExpertParams& p, cudaStream_t s, bool pdl) {
  int S;
  size_t smem;
  x_smem<Q, ROLE, NT>(p.K, p.N, &S, &smem);
  auto kern = k_expert<Q, ROLE, NT>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  ExpertParams q = p;
  q.stages = S;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(kXThreads);
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
static cudaError_t launch_x_q(const ExpertParams& p, int nt, cudaStream_t s, bool pdl) {
  switch (nt) {
    case 1: return launch_x_t<Q, ROLE, 1>(p, s, pdl);
    case 2: return launch_x_t<Q, ROLE, 2>(p, s, pdl);
    case 4: return launch_x_t<Q, ROLE, 4>(p, s, pdl);
    case 8: return launch_x_t<Q, ROLE, 8>(p, s, pdl);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_expert(const ExpertParams& p, int nt, cudaStream_t s, bool pdl) {
  switch (p.quant * 2 + p.role) {
    case 0: return launch_x_q<kMXFP4, 0>(p, nt, s, pdl);
    case 1: return launch_x_q<kMXFP4, 1>(p, nt, s, pdl);
    case 2: return launch_x_q<kNVFP4, 0>(p, nt, s, pdl);
    case 3: return launch_x_q<kNVFP4, 1>(p, nt, s, pdl);
    case 4: return launch_x_q<kFP8, 0>(p, nt, s, pdl);
    case 5: return launch_x_q<kFP8, 1>(p, nt, s, pdl);
    case 6: return launch_x_q<kBF16, 0>(p, nt, s, pdl);
    case 7: return launch_x_q<kBF16, 1>(p, nt, s, pdl);
    default: return cudaErrorInvalidValue;
  }
}

template <int Q, int ROLE, int NT>
static int x_occ_t(int K, int N) {
  int n = 0, S;
  size_t smem;
  x_smem<Q, ROLE, NT>(K, N, &S, &smem);
  auto kern = k_expert<Q, ROLE, NT>;
  if (smem > 48 * 1024)
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kXThreads, smem) != cudaSuccess)
    return 1;
  return n > 0 ? n : 1;
}
template <int Q, int ROLE>
static int x_occ_q(int nt, int K, int N) {
  switch (nt) {
    case 1: return x_occ_t<Q, ROLE, 1>(K, N);
    case 2: return x_occ_t<Q, ROLE, 2>(K, N);
    case 4: return x_occ_t<Q, ROLE, 4>(K, N);
    default: return x_occ_t<Q, ROLE, 8>(K, N);
  }
}
int expert_ctas_per_sm(int quant, int role, int nt, int K, int N) {
  switch (quant * 2 + role) {
    case 0: return x_occ_q<kMXFP4, 0>(nt, K, N);
    case 1: return x_occ_q<kMXFP4, 1>(nt, K, N);
    case 2: return x_occ_q<kNVFP4, 0>(nt, K, N);
    case 3: return x_occ_q<kNVFP4, 1>(nt, K, N);
    case 4: return x_occ_q<kFP8, 0>(nt, K, N);
    case 5: return x_occ_q<kFP8, 1>(nt, K, N);
    case 6: return x_occ_q<kBF16, 0>(nt, K, N);
    default: return x_occ_q<kBF16, 1>(nt, K, N);
  }
}

// Bytes of the partial-sum slots a launch may use, and tickets per matrix.
size_t expert_part_bytes(int grid, int nt) {
  return (size_t)grid * 2 * kXWarps * nt * 32 * sizeof(float4);
}
size_t expert_tickets(int max_groups, int quant, int role, int K, int N) {
  (void)quant;
  (void)K;
  const int tiles = (role == 0) ? (N / 2) / 64 : N / 128;
  return (size_t)max_groups * tiles * kXWarps;
}

}  // namespace musemoe
