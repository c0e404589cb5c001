// Routed experts on the fifth-generation tensor cores (tcgen05), for the
// buckets where an expert's token group makes the expert work a dense
// contraction (up to 64 tokens per group). Same contract as k_expert (the
// same work units, the same outputs, the same split-tile partial sums), so
// the forward picks either kernel per call.
//
// One CTA per SM (persistent), Stream-K over units = (token group, tile of
// 128 weight rows, K-slice of 4 64-byte chunks). The MMA is
// D[128 weight rows x N tokens] += A[128 x K] * B[N x K]^T with N the group's
// tokens rounded up to 16, fp32 accumulation in tensor memory (four
// accumulators of 64 columns, so the epilogue of a tile overlaps the MMAs of
// the next ones; FP4 adds four 64-column A slots).
//
// w13 (role 0): a tile is 64 gate rows and the matching 64 up rows,
// interleaved by 8-row groups in A (group 2j gate rows i0 + 8j.., group
// 2j + 1 the up rows I + i0 + 8j..), so that the thread holding gate row i
// and the thread holding up row i are lanes l and l ^ 8 of one warp: the
// SiLU(gate) * up epilogue pairs them with one shuffle. w2 (role 1): 128
// consecutive P rows.
//
// Operands (K-major, canonical shared-memory layouts):
// * FP8 W8A8 (kind::f8f6f4, e4m3 x e4m3): A straight from the bulk-copied
//   weight stage (the pack stores each [8 rows][64 B] block 64-byte
//   swizzled), B the tokens' e4m3 rows of the slice, 64-byte swizzled. The
//   per-row weight scale and the per-row activation scale multiply the fp32
//   result.
// * MXFP4 / NVFP4 (kind::f16, f16 x f16): dequantizing warps convert each
//   64-byte chunk of codes to f16 (one cvt per e2m1 pair, exact) times its
//   block scale (UE8M0 2^(s-127) as an f16 power of two, exact for s in
//   104..140; e4m3 exact) and store it into an A slot in tensor memory
//   (tcgen05.st: row m in lane m, f16 pairs in K order), so the dequantized
//   operand never crosses shared memory; B the tokens' f16 rows of the
//   chunk (shared memory, 128-byte swizzle). The NVFP4 global scale
//   multiplies the fp32 result.
//   The W4A4 forms run here too: their f16 operands hold FP4-rounded values.
//
// Warp roles: epilogue (4 warps, one per tensor-memory lane quarter),
// dequantizers (FP4 only, 8 warps), a producer lane (bulk copies of the
// weights), an MMA lane (issues the MMAs and commits them to the mbarriers
// that free the stages), B loaders (2 warps FP4, 4 FP8: 16-byte cp.async gathers of the
// token rows, completion signalled by the copy engine on the slot's
// mbarrier). Every wait is bounded: past the limit the CTA raises the
// health word, lets its copies and MMAs finish and frees its tensor memory.
#include "pipeline.cuh"
#include "tc.cuh"

namespace musemoe {

namespace {

constexpr int kTM = 128;         // weight rows per tile (MMA M)
constexpr int kTN = 64;          // tokens per group at most (MMA N, padded to 16)
constexpr int kTAcc = 64;        // tensor-memory columns of one accumulator
constexpr int kTEpi = 4;         // epilogue warps
constexpr int kTDq = 8;          // dequantizing warps (FP4)
constexpr int kTMeta = 4;        // token groups cached in shared memory
constexpr int kTBSlot = 16384;   // one B piece (64 tokens x 256 B)
constexpr int kTAOff = 4 * 64;   // tensor-memory column of the first A slot (FP4), after 4 accumulators
constexpr int kTCodeBlock = 8 * kSliceChunks * 512;  // codes of one 64-row block's slice
constexpr int kTSmemMax = 227 * 1024;  // dynamic + static shared memory of a CTA
constexpr int kTReserve = 3 * 1024;    // alignment slack (1024) + static shared memory (< 2048)

// forms of the kernel beyond the weight formats: W4A4 on the FP4 tensor cores
constexpr int kA4MX = 4, kA4NV = 5;

template <int Q>
struct TcCfg {
  static constexpr bool fp4 = (Q == kMXFP4 || Q == kNVFP4);  // FP4 weights dequantized to f16
  static constexpr bool a4 = (Q == kA4MX || Q == kA4NV);     // W4A4, block-scaled FP4 MMA
  static constexpr int apc = Q == kA4NV ? 2 : 1;  // W4A4: scale atoms per 64-byte code chunk
  static constexpr int sf_bytes = a4 ? kSliceChunks * apc * 512 : 0;  // an operand's atoms per slice
  static constexpr int loaders = fp4 ? 2 : 4;  // B loader warps
  static constexpr int sfw = a4 ? 1 : 0;       // W4A4: the scale-atom copy warp
  static constexpr int warps = kTEpi + (fp4 ? kTDq : 0) + 2 + loaders + sfw;
  static constexpr int w_dq0 = kTEpi;                       // first dequant warp
  static constexpr int w_prod = kTEpi + (fp4 ? kTDq : 0);   // producer warp
  static constexpr int w_mma = w_prod + 1;
  static constexpr int w_load0 = w_prod + 2;
  static constexpr int w_sf = w_load0 + loaders;
  static constexpr int threads = warps * 32;
  static constexpr int SB = (Q == kMXFP4) ? 4 : (Q == kNVFP4) ? 8 : 0;  // scale bytes / row / chunk
  static constexpr int scale_block = 8 * kSliceChunks * 8 * SB;        // scales of one block's slice
  // a weight stage: the unit's codes, their scales (FP4) or scale atoms (W4A4)
  static constexpr int stage_bytes = 2 * kTCodeBlock + 2 * scale_block + sf_bytes;
  // a B slot: the tokens' rows of a piece (+ W4A4: their scale atoms)
  static constexpr int bslot = kTBSlot + sf_bytes;
  // weight stages: FP4 next to four chunk slots; FP8 / W4A4 one B slot per
  // stage; kTReserve is left for the 1024-byte alignment and the static
  // shared memory (barriers, token-group cache)
  static constexpr int stages =
      fp4 ? ((kTSmemMax - kTReserve - 4 * bslot) / stage_bytes > 4
                 ? 4
                 : (kTSmemMax - kTReserve - 4 * bslot) / stage_bytes)
          : ((kTSmemMax - kTReserve) / (stage_bytes + bslot) > 4
                 ? 4
                 : (kTSmemMax - kTReserve) / (stage_bytes + bslot));
  static constexpr int n_b = fp4 ? 4 : stages;  // B slots (FP8 / W4A4: a unit's B rows ride in its stage)
  static constexpr int n_a = fp4 ? 4 : 0;       // A slots (tensor memory, 64 columns each)
  // accumulators (64 columns each): four, so that the epilogue may lag three
  // tiles (FP4: next to four 64-column A slots, the whole tensor memory)
  static constexpr int n_acc = 4;
  static constexpr int tmem_cols = (fp4 || a4) ? 512 : 256;
  // W4A4: the scale atoms of stage st in tensor memory, A then B, 4 columns each
  static constexpr int sf_cols = a4 ? 2 * kSliceChunks * apc * 4 : 0;
};

template <int Q>
__host__ __device__ constexpr int tc_stages() {
  return TcCfg<Q>::stages;
}
template <int Q>
__host__ __device__ constexpr int tc_smem_bytes() {
  return 1024 + tc_stages<Q>() * TcCfg<Q>::stage_bytes + TcCfg<Q>::n_b * TcCfg<Q>::bslot;
}
static_assert(tc_stages<kMXFP4>() >= 2 && tc_stages<kNVFP4>() >= 2 && tc_stages<kFP8>() >= 2 &&
                  tc_stages<kA4MX>() >= 2 && tc_stages<kA4NV>() >= 2,
              "at least two weight stages");
static_assert(tc_stages<kFP8>() == 4, "FP8: four stages");
static_assert(tc_smem_bytes<kMXFP4>() + kTReserve - 1024 <= kTSmemMax &&
                  tc_smem_bytes<kNVFP4>() + kTReserve - 1024 <= kTSmemMax &&
                  tc_smem_bytes<kFP8>() + kTReserve - 1024 <= kTSmemMax &&
                  tc_smem_bytes<kA4MX>() + kTReserve - 1024 <= kTSmemMax &&
                  tc_smem_bytes<kA4NV>() + kTReserve - 1024 <= kTSmemMax,
              "dynamic + static shared memory within a CTA's maximum");
static_assert(TcCfg<kNVFP4>::n_acc * kTAcc + TcCfg<kNVFP4>::n_a * 64 <= 512 && kTAOff == 4 * kTAcc,
              "FP4 tensor memory: accumulators, then the A slots");
static_assert(TcCfg<kFP8>::n_acc * kTAcc <= TcCfg<kFP8>::tmem_cols, "FP8 tensor memory");
static_assert(TcCfg<kA4NV>::n_acc * kTAcc + tc_stages<kA4NV>() * TcCfg<kA4NV>::sf_cols <= 512 &&
                  TcCfg<kA4MX>::n_acc * kTAcc + tc_stages<kA4MX>() * TcCfg<kA4MX>::sf_cols <= 512,
              "W4A4 tensor memory: accumulators and scale atoms");

// CTA c runs units [U c / G, U (c + 1) / G); the CTA holding unit u:
__device__ __forceinline__ int tc_cta_of(long long u, long long U, int G) {
  return (int)(((u + 1) * G - 1) / U);
}
__device__ __forceinline__ long long tc_start(int c, long long U, int G) { return U * c / G; }

// A CTA's unit range in processing order: its whole tiles [b0, b1), then the
// units [b1, U1) of the tile it shares with the next CTA (it leaves a
// partial and signals, never waits), then the units [U0, b0) of the tile it
// shares with the previous CTA (it owns that tile: it waits for the other
// partials and finishes it). A range inside one tile is a single
// leave-a-partial part. No owner wait can depend on a waiting CTA.
struct SKRange {
  int U0, U1, b0, b1, KS, PG, tiles;
  __device__ void init(long long u0, long long u1, int ks, int tl) {
    U0 = (int)u0;
    U1 = (int)u1;
    KS = ks;
    tiles = tl;
    PG = ks * tl;
    b0 = (U0 + KS - 1) / KS * KS;
    b1 = U1 / KS * KS;
    if (b0 > b1) b0 = b1 = U0;
  }
  __device__ int lo(int i) const { return i == 0 ? b0 : (i == 1 ? b1 : U0); }
  __device__ int hi(int i) const { return i == 0 ? b1 : (i == 1 ? U1 : b0); }
  __device__ int count() const { return U1 - U0; }
};
struct SKWalk {
  int u, grp, tile, slice, lo, hi, part, left;
  __device__ void begin() {
    part = -1;
    left = 0;
  }
  __device__ void next(const SKRange& R) {
    if (left == 0) {
      do {
        ++part;
      } while (part < 3 && R.hi(part) <= R.lo(part));
      lo = R.lo(part);
      hi = R.hi(part);
      left = hi - lo;
      u = lo;
      grp = u / R.PG;
      const int rem = u - grp * R.PG;
      tile = rem / R.KS;
      slice = rem - tile * R.KS;
    } else {
      ++u;
      if (++slice == R.KS) {
        slice = 0;
        if (++tile == R.tiles) {
          tile = 0;
          ++grp;
        }
      }
    }
    --left;
  }
  // the unit closes an accumulator: its tile ends, or its part does
  __device__ bool closes(const SKRange& R) const { return slice == R.KS - 1 || u + 1 == hi; }
};

// UE8M0 code -> f16 bits of 2^(s - 127) when exact products with e2m1 stay in
// the f16 range (s in 104..140); 0 flags a scale outside it.
__device__ __forceinline__ uint32_t ue8m0_to_f16_bits(uint32_t s) {
  const int t = (int)s - 127;
  if (t < -23 || t > 13) return 0u;
  return t >= -14 ? (uint32_t)((t + 15) << 10) : (1u << (t + 24));
}

}  // namespace

// Optional phase timeline (compile with -DMUSEMOE_TIMELINE; off in the
// library build): %globaltimer stamps of each role's waits in four CTAs
// (the first two, the middle one, the last one), the event kind in the low
// 4 bits, w13 in the first half of each role's events and w2 in the second,
// read back with musemoe_tc_timeline_read.
#ifdef MUSEMOE_TIMELINE
constexpr int kTlCtas = 4, kTlRoles = 5, kTlEvents = 1024;
__device__ unsigned long long g_tc_tl[kTlCtas][kTlRoles][kTlEvents];
__device__ __forceinline__ int tl_cta() {
  const int b = blockIdx.x, g = gridDim.x;
  return b == 0 ? 0 : b == 1 ? 1 : b == g / 2 ? 2 : b == g - 1 ? 3 : -1;
}
#define TL(role, cnt, kind)                                                               \
  do {                                                                                    \
    const int tl_c = tl_cta();                                                            \
    if (tl_c >= 0 && (cnt) < kTlEvents / 2)                                               \
      g_tc_tl[tl_c][role][ROLE * (kTlEvents / 2) + (cnt)++] =                             \
          (globaltimer() & ~15ull) | (unsigned long long)(kind);                           \
  } while (0)
#else
#define TL(role, cnt, kind) \
  do {                      \
  } while (0)
#endif

template <int Q, int ROLE>
__global__ void __launch_bounds__(TcCfg<Q>::threads, 1) k_expert_tc(ExpertParams p) {
  using C = TcCfg<Q>;
  pdl_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  // FP8: stage st holds a unit's weights (producer) and its B rows
  // (loaders): full_b[st] counts both, empty_b[st] is the MMA's commit.
  // FP4: stage st holds a unit's codes (producer -> dequantizers); chunk slot
  // cs holds a chunk's A (tensor memory, dequantizers) and B rows (shared
  // memory, loaders): cfull[cs] counts both, cempty[cs] is the MMA's commit.
  __shared__ __align__(8) unsigned long long full_b[4], empty_b[4];
  __shared__ __align__(8) unsigned long long cfull[4], cempty[4];
  __shared__ __align__(8) unsigned long long accfull[4], accempty[4], drain_b;
  __shared__ __align__(8) unsigned long long sffull[4];  // W4A4: a stage's scale atoms in tensor memory
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ int4 meta_g[kTMeta];
  __shared__ int meta_r[kTMeta][kTN];
  static_assert(sizeof(meta_g) + sizeof(meta_r) + 16 * 8 + 64 <= kTReserve - 1024,
                "static shared memory within the reserve");

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kNA = C::n_a > 0 ? C::n_a : 1;  // A slots (FP4; 1 keeps the other forms' dead code defined)
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* const sbase = smem_raw + (base - smem_u32(smem_raw));
  constexpr int S = tc_stages<Q>();
  const uint32_t st0 = base;
  const uint32_t b0s = base + S * C::stage_bytes;

  // geometry: weight rows of N, reduction K
  const int rowbytes = (Q == kFP8) ? p.K : p.K / 2;
  const int NC = rowbytes / 64;
  const int KS = (NC + kSliceChunks - 1) / kSliceChunks;
  const int tiles = (ROLE == 0) ? p.I / 64 : p.N / 128;
  const int n_groups = __ldcg(p.counters + kNumGroups);
  const long long U = (long long)n_groups * tiles * KS;
  const int GE = (int)min((long long)gridDim.x, U);
  const long long u0 = blockIdx.x < GE ? tc_start(blockIdx.x, U, GE) : 0;
  const long long u1 = blockIdx.x < GE ? tc_start(blockIdx.x + 1, U, GE) : 0;
  SKRange R;
  R.init(u0, u1, KS, tiles);
  const int count = R.count();
  const int kel = (Q == kFP8) ? 1 : 2;  // bytes per activation element

  // token groups of the range (cached) and their routes
  const int PG = R.PG;
  const int g_first = count > 0 ? (int)(u0 / PG) : 0;
  const int g_count = count > 0 ? min(kTMeta, (int)((u1 - 1) / PG) - g_first + 1) : 0;
  for (int i = tid; i < g_count; i += blockDim.x)
    meta_g[i] = __ldcg(reinterpret_cast<const int4*>(p.groups) + g_first + i);
  if (tid == 0) {
    for (int i = 0; i < 4; ++i) {
      mbar_init(smem_u32(&sffull[i]), 1);
      mbar_init(smem_u32(&full_b[i]), C::fp4 ? 1 : 1 + C::loaders * 32);
      mbar_init(smem_u32(&empty_b[i]), C::fp4 ? kTDq : 1);
      mbar_init(smem_u32(&cfull[i]), kTDq + C::loaders * 32);
      mbar_init(smem_u32(&cempty[i]), 1);
    }
    for (int i = 0; i < C::n_acc; ++i) {
      mbar_init(smem_u32(&accfull[i]), 1);
      mbar_init(smem_u32(&accempty[i]), kTEpi);
    }
    mbar_init(smem_u32(&drain_b), 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == 0) {
    tc::tmem_alloc(smem_u32(&tmem_slot), C::tmem_cols);
    tc::tmem_relinquish();
  }
  __syncthreads();
  for (int i = tid; i < g_count * kTN; i += blockDim.x) {
    const int gi = i / kTN, n = i % kTN;
    if (n < meta_g[gi].z) meta_r[gi][n] = __ldcg(p.route_list + meta_g[gi].y + n);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_slot;

  auto group_of = [&](int grp) -> int4 {
    const int gi = grp - g_first;
    return gi < kTMeta ? meta_g[gi] : __ldcg(reinterpret_cast<const int4*>(p.groups) + grp);
  };
  auto route_of = [&](int grp, int rbase, int n) -> int {
    const int gi = grp - g_first;
    return gi < kTMeta ? meta_r[gi][n] : __ldcg(p.route_list + rbase + n);
  };
  auto fail = [&]() {
    if (atomicExch(&abort_flag, 1) == 0) atomicOr(p.health, kHealthTimeout);
  };
  auto wait = [&](unsigned long long* bar, uint32_t phase) -> bool {
    return mbar_wait_or_abort(smem_u32(bar), phase, &abort_flag);
  };

  if (warp == C::w_prod) {
    // ---------------- producer: the weight codes and scales ----------------
    if (lane == 0) {
      [[maybe_unused]] int tlc = 0;
      TL(0, tlc, 0);
      const int NRT = p.N / 64;
      const size_t tile_codes = (size_t)NC * 4096, tile_scales = (size_t)NC * 64 * C::SB;
      const uint8_t* sb = reinterpret_cast<const uint8_t*>(p.scale);
      const uint64_t pol = l2_policy_evict_first();
      SKWalk wk;
      wk.begin();
      int gcur = -1, e = 0;
      int issued = 0;
      for (int n = 0; n < count; ++n) {
        wk.next(R);
        if (wk.grp != gcur) {
          gcur = wk.grp;
          e = group_of(gcur).x;
        }
        const int st = n % S, use = n / S;
        if (use > 0 && !wait(&empty_b[st], (uint32_t)(use - 1) & 1u)) {
          fail();
          break;
        }
        if (use > 0) asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
        TL(0, tlc, 1);
        const int nc = min(kSliceChunks, NC - wk.slice * kSliceChunks);
        const uint32_t bar = smem_u32(&full_b[st]);
        mbar_expect_tx(bar, 2u * nc * (4096 + 64 * C::SB) + (C::a4 ? (uint32_t)(nc * C::apc * 512) : 0u));
        const uint32_t dst = st0 + st * C::stage_bytes;
        for (int blk = 0; blk < 2; ++blk) {
          const int rt = (ROLE == 0) ? (blk == 0 ? wk.tile : p.I / 64 + wk.tile) : 2 * wk.tile + blk;
          const size_t ti = (size_t)e * NRT + rt;
          const uint8_t* src = p.w + ti * tile_codes + (size_t)wk.slice * kSliceChunks * 4096;
          if (!C::fp4 && ROLE == 0) {
            // 8-row groups interleaved: group g of the gate block -> A group
            // 2g, of the up block -> 2g + 1
            for (int g8 = 0; g8 < 8; ++g8)
              bulk_g2s_hint(dst + (2 * g8 + blk) * nc * 512, src + g8 * nc * 512, nc * 512, bar, pol);
          } else {
            bulk_g2s_hint(dst + blk * 8 * nc * 512, src, nc * 4096, bar, pol);
          }
          if (C::SB)
            bulk_g2s_hint(dst + 2 * kTCodeBlock + blk * C::scale_block,
                          sb + ti * tile_scales + (size_t)wk.slice * kSliceChunks * 64 * C::SB,
                          nc * 64 * C::SB, bar, pol);
        }
        if (C::a4) {
          // W4A4: the slice's weight scale atoms ([tiles][slice][atom][512] per expert)
          const size_t tile_atoms = (size_t)NC * C::apc * 512;
          bulk_g2s_hint(dst + 2 * kTCodeBlock,
                        sb + ((size_t)e * tiles + wk.tile) * tile_atoms + (size_t)wk.slice * C::sf_bytes,
                        nc * C::apc * 512, bar, pol);
        }
        issued = n + 1;
        TL(0, tlc, 2);
      }
      // every copy issued must land before the CTA leaves
      for (int st = 0; st < S && st < issued; ++st) {
        const int last = st + ((issued - 1 - st) / S) * S;
        const unsigned long long t0 = globaltimer();
        while (!mbar_try_wait(smem_u32(&full_b[st]), (uint32_t)(last / S) & 1u))
          if (globaltimer() - t0 > kWaitLimitNs) break;
      }
    }
  } else if (C::a4 && warp == C::w_sf) {
    // ---------------- W4A4: scale atoms -> tensor memory ----------------
    // Once a unit's stage has landed (which also means that the MMAs of the
    // stage's previous unit, the last readers of its tensor-memory columns,
    // have completed), one lane copies the unit's A and B scale atoms into
    // the stage's columns and commits the copies to sffull[stage].
    if (lane == 0) {
      SKWalk wk;
      wk.begin();
      int issued = 0;
      for (int n = 0; n < count; ++n) {
        wk.next(R);
        const int st = n % S;
        if (!wait(&full_b[st], (uint32_t)(n / S) & 1u)) {
          fail();
          break;
        }
        tc::fence_after_sync();
        const int nc = min(kSliceChunks, NC - wk.slice * kSliceChunks);
        const uint32_t sfa_t = tmem + C::n_acc * kTAcc + st * C::sf_cols;
        const uint32_t sfb_t = sfa_t + C::sf_cols / 2;
        const uint32_t sa = st0 + st * C::stage_bytes + 2 * kTCodeBlock;
        const uint32_t sbb = b0s + st * C::bslot + kTBSlot;
        for (int a = 0; a < nc * C::apc; ++a) {
          tc::cp_scale_atom(sfa_t + 4 * a, sa + 512 * a);
          tc::cp_scale_atom(sfb_t + 4 * a, sbb + 512 * a);
        }
        tc::commit(smem_u32(&sffull[st]));
        issued = n + 1;
      }
      // the copies must land before the tensor memory is freed
      for (int st = 0; st < S && st < issued; ++st) {
        const int last = st + ((issued - 1 - st) / S) * S;
        const unsigned long long t0 = globaltimer();
        while (!mbar_try_wait(smem_u32(&sffull[st]), (uint32_t)(last / S) & 1u))
          if (globaltimer() - t0 > kWaitLimitNs) break;
      }
    }
  } else if (warp >= C::w_load0) {
    // ---------------- B loaders: the tokens' rows of each piece ----------------
    // Thread lt copies 16-byte unit uu = lt % 16 of the rows r0, r0 + RSTEP,
    // ... of every piece; the rows' byte offsets are looked up once per token
    // group, so a piece is a run of independent cp.async.
    pdl_wait();  // the activations are the previous kernel's output
    const int lt = tid - C::w_load0 * 32;
    constexpr int LT = C::loaders * 32;
    constexpr int RSTEP = LT / 16;
    constexpr int RPT = kTN / RSTEP;  // rows per thread
    constexpr int kLag = 1;           // copy groups left in flight when a piece is released
    const int uu = lt & 15, r0 = lt >> 4;
    const size_t rowB = C::a4 ? (size_t)p.K / 2 : (size_t)p.K * kel;
    const int sf_row = p.K / (Q == kA4NV ? 16 : 32);  // W4A4: scale bytes of a B row
    uint32_t roff[RPT];
    uint32_t rsf[C::a4 ? RPT : 1];
    int nrow = 0;
    [[maybe_unused]] int tlc = 0;
    if (lt == 0) TL(3, tlc, 0);
    SKWalk wk;
    wk.begin();
    int gcur = -1;
    int piece = 0, released = 0;  // pieces issued / released to the MMA side
    bool ok = true;
    for (int n = 0; n < count && ok; ++n) {
      wk.next(R);
      if (wk.grp != gcur) {
        gcur = wk.grp;
        const int4 gd = group_of(gcur);
        nrow = 0;
#pragma unroll
        for (int m = 0; m < RPT; ++m) {
          const int tn = r0 + RSTEP * m;
          roff[m] = 0;
          if (tn < gd.z) {
            const int ro = route_of(gcur, gd.y, tn);
            const int brow = p.b_by_token ? ro / p.k : ro;
            roff[m] = (uint32_t)((size_t)brow * rowB);
            if constexpr (C::a4) rsf[m] = (uint32_t)brow * (uint32_t)sf_row;
            nrow = m + 1;
          }
        }
      }
      const int nc = min(kSliceChunks, NC - wk.slice * kSliceChunks);
      const int pieces = C::fp4 ? nc : 1;
      for (int c = 0; c < pieces; ++c, ++piece) {
        const int bs = piece % C::n_b, use = piece / C::n_b;
        unsigned long long* const eb = C::fp4 ? &cempty[bs] : &empty_b[bs];
        if (use > 0) {
          const uint32_t ph = (uint32_t)(use - 1) & 1u;
          if (!__all_sync(0xffffffffu, mbar_test(smem_u32(eb), ph))) {
            // the slot is still in use: release the pending pieces before
            // blocking on it, so that no finished piece waits behind it
            if (piece > released) {
              asm volatile("cp.async.wait_all;\n" ::: "memory");
              tc::fence_proxy_async_smem();
              for (; released < piece; ++released)
                mbar_arrive(smem_u32(C::fp4 ? &cfull[released % C::n_b] : &full_b[released % C::n_b]));
            }
            if (!__all_sync(0xffffffffu, wait(eb, ph))) {
              if (lane == 0) fail();
              ok = false;
              break;
            }
          }
        }
        if (lt == 0) TL(3, tlc, 1);
        const uint32_t dst = b0s + bs * C::bslot;
        if constexpr (C::fp4) {
          // f16 chunk slice * 4 + c of each row: 256 B = 16 units, 128-byte swizzle
          const uint8_t* src = p.b + (size_t)(wk.slice * kSliceChunks + c) * 256 + uu * 16;
          const uint32_t d0 = dst + (uu >> 3) * 8192;
#pragma unroll
          for (int m = 0; m < RPT; ++m)
            if (m < nrow)
              asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(
                               d0 + tc::sw128_off(r0 + RSTEP * m, uu & 7)),
                           "l"(src + roff[m]));
        } else {
          // e4m3 slice: nc chunks of 64 B, 64-byte swizzle [N/8][nc][8][64]
          const int cc = uu >> 2, u4 = uu & 3;
          if (cc < nc) {
            const uint8_t* src = p.b + (size_t)(wk.slice * kSliceChunks + cc) * 64 + u4 * 16;
#pragma unroll
            for (int m = 0; m < RPT; ++m)
              if (m < nrow)
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(
                                 dst + cc * 512 + tc::sw64_off(r0 + RSTEP * m, u4, nc * 512)),
                             "l"(src + roff[m]));
          }
          if constexpr (C::a4) {
            // the rows' scale atoms: atom uu of the slice holds blocks 4 uu .. 4 uu + 3,
            // token n's four bytes at (n % 32) * 16 + (n / 32) * 4
            if (uu < nc * C::apc) {
              const uint8_t* ssrc = p.b_sf + (size_t)(wk.slice * kSliceChunks * C::apc + uu) * 4;
              const uint32_t sdst = dst + kTBSlot + uu * 512;
#pragma unroll
              for (int m = 0; m < RPT; ++m)
                if (m < nrow) {
                  const int tn = r0 + RSTEP * m;
                  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(
                                   sdst + (tn & 31) * 16 + (tn >> 5) * 4),
                               "l"(ssrc + rsf[m]));
                }
            }
          }
        }
        // one copy group per piece; the pieces issued kLag pieces earlier
        // or before have landed once all but the newest kLag groups have:
        // the thread makes its rows visible to the tensor core (async proxy)
        // and arrives on those pieces' slots, so the MMA side needs no
        // proxy fence
        asm volatile("cp.async.commit_group;\n" ::: "memory");
        if (piece - kLag >= released) {
          asm volatile("cp.async.wait_group %0;\n" ::"n"(kLag) : "memory");
          tc::fence_proxy_async_smem();
          for (; released <= piece - kLag; ++released)
            mbar_arrive(smem_u32(C::fp4 ? &cfull[released % C::n_b] : &full_b[released % C::n_b]));
        }
        if (lt == 0) TL(3, tlc, 2);
      }
    }
    // the pieces still in flight: land, publish, arrive (nothing in flight at exit)
    asm volatile("cp.async.wait_all;\n" ::: "memory");
    tc::fence_proxy_async_smem();
    for (; released < piece; ++released)
      mbar_arrive(smem_u32(C::fp4 ? &cfull[released % C::n_b] : &full_b[released % C::n_b]));
  } else if (warp == C::w_mma) {
    // ---------------- MMA issue (one lane) ----------------
    if (lane == 0) {
      [[maybe_unused]] int tlc = 0;
      TL(1, tlc, 0);
      SKWalk wk;
      wk.begin();
      int gcur = -1;
      uint32_t idesc = 0, idesc_hi = 0;  // W4A4 MXFP4: the second step of an atom (scale-ID 2)
      int piece = 0, achunk = 0, acc = 0, acc_use = 0;
      bool fresh = true, ok = true;
      for (int n = 0; n < count && ok; ++n) {
        wk.next(R);
        if (wk.grp != gcur) {
          gcur = wk.grp;
          const int nt = group_of(gcur).z;
          const int npad = (nt + 15) & ~15;
          if constexpr (C::a4) {
            idesc = tc::instr_desc_fp4(kTM, npad, Q == kA4MX ? 1u : 0u, 0u);
            idesc_hi = tc::instr_desc_fp4(kTM, npad, 1u, 2u);
          } else {
            idesc = (Q == kFP8) ? tc::instr_desc(tc::kE4M3, tc::kE4M3, kTM, npad)
                                : tc::instr_desc(tc::kF16, tc::kF16, kTM, npad);
          }
        }
        if (fresh) {
          // the accumulator must have been drained by the epilogue
          if (acc_use >= C::n_acc && !wait(&accempty[acc], (uint32_t)(acc_use / C::n_acc - 1) & 1u)) {
            fail();
            break;
          }
          tc::fence_after_sync();
          TL(1, tlc, 1);
        }
        const uint32_t d_tmem = tmem + acc * kTAcc;
        const int nc = min(kSliceChunks, NC - wk.slice * kSliceChunks);
        if constexpr (!C::fp4) {
          const int st = n % S;
          const int bs = st;  // the unit's B rows ride in its stage
          if (!wait(&full_b[st], (uint32_t)(n / S) & 1u)) {
            fail();
            break;
          }
          TL(1, tlc, 3);
          tc::fence_after_sync();
          // descriptors of the unit's first k-step; k-step (c, h) starts
          // c * 512 + h * 32 bytes further (the start-address field counts 16 B)
          const uint64_t da0 = tc::smem_desc(st0 + st * C::stage_bytes, 16, nc * 512, tc::kSw64);
          const uint64_t db0 = tc::smem_desc(b0s + bs * C::bslot, 16, nc * 512, tc::kSw64);
          if constexpr (C::a4) {
            // the unit's scale atoms, copied into this stage's tensor-memory
            // columns (A then B) by the scale warp
            if (!wait(&sffull[st], (uint32_t)(n / S) & 1u)) {
              fail();
              break;
            }
            tc::fence_after_sync();
            const uint32_t sfa_t = tmem + C::n_acc * kTAcc + st * C::sf_cols;
            const uint32_t sfb_t = sfa_t + C::sf_cols / 2;
#pragma unroll
            for (int c = 0; c < kSliceChunks; ++c)
#pragma unroll
              for (int h = 0; h < 2; ++h)
                if (c < nc) {
                  const uint32_t acc_in = (fresh && c == 0 && h == 0) ? 0u : 1u;
                  if constexpr (Q == kA4NV) {
                    const int atom = 2 * c + h;  // four blocks of 16 per 64-element step
                    tc::mma_nvf4(d_tmem, da0 + (uint64_t)(c * 32 + h * 2), db0 + (uint64_t)(c * 32 + h * 2),
                                 idesc, sfa_t + 4 * atom, sfb_t + 4 * atom, acc_in);
                  } else {
                    // the chunk's atom holds both steps: scale-ID 0, then 2
                    tc::mma_mxf4(d_tmem, da0 + (uint64_t)(c * 32 + h * 2), db0 + (uint64_t)(c * 32 + h * 2),
                                 h ? idesc_hi : idesc, sfa_t + 4 * c, sfb_t + 4 * c, acc_in);
                  }
                }
          } else {
#pragma unroll
            for (int c = 0; c < kSliceChunks; ++c)
#pragma unroll
              for (int h = 0; h < 2; ++h)
                if (c < nc)
                  tc::mma_f8f6f4(d_tmem, da0 + (uint64_t)(c * 32 + h * 2), db0 + (uint64_t)(c * 32 + h * 2),
                                 idesc, (fresh && c == 0 && h == 0) ? 0u : 1u);
          }
          tc::commit(smem_u32(&empty_b[st]));
          TL(1, tlc, 4);
          ++piece;
        } else {
          for (int c = 0; c < nc; ++c, ++piece, ++achunk) {
            const int as = achunk % kNA, bs = as;  // A and B of a chunk share its slot
            if (!wait(&cfull[as], (uint32_t)(achunk / kNA) & 1u)) {
              fail();
              ok = false;
              break;
            }
            TL(1, tlc, 3);
            tc::fence_after_sync();
            const uint32_t a_t = tmem + kTAOff + as * kTAcc;
            // k-step j: A columns 8j.., B bytes (j / 4) * 8192 + (j % 4) * 32
            // (the descriptor's start-address field counts 16 B)
            const uint64_t db0 = tc::smem_desc(b0s + bs * C::bslot, 16, 1024, tc::kSw128);
            const uint32_t acc0 = (fresh && c == 0) ? 0u : 1u;
#pragma unroll
            for (int j = 0; j < 8; ++j)
              tc::mma_f16_ta(d_tmem, a_t + 8 * j, db0 + (uint64_t)((j >> 2) * 512 + (j & 3) * 2), idesc,
                             j == 0 ? acc0 : 1u);
            tc::commit(smem_u32(&cempty[as]));
            TL(1, tlc, 4);
          }
          if (!ok) break;
        }
        fresh = false;
        if (wk.closes(R)) {
          tc::commit(smem_u32(&accfull[acc]));
          acc = acc + 1 == C::n_acc ? 0 : acc + 1;
          ++acc_use;
          fresh = true;
        }
      }
      // every MMA issued must complete before the tensor memory is freed
      tc::commit(smem_u32(&drain_b));
      const unsigned long long t0 = globaltimer();
      while (!mbar_try_wait(smem_u32(&drain_b), 0u))
        if (globaltimer() - t0 > kWaitLimitNs) break;
    }
  } else if (C::fp4 && warp >= C::w_dq0 && warp < C::w_dq0 + kTDq) {
    // ---------------- dequantizers (FP4): codes -> f16 A in tensor memory ----------------
    // Warp w writes tensor-memory lanes 32 (w % 4) .. + 31 (A rows), and the
    // half w / 4 of each chunk's 128 K elements: 32 columns of f16 pairs.
    const int dw = warp - C::w_dq0;
    const int r = (warp & 3) * 32 + lane;  // A row = tensor-memory lane
    const int hh = dw >> 2;                // elements 64 hh .. 64 hh + 63 of the chunk
    const uint32_t t_lane = (uint32_t)((warp & 3) * 32) << 16;
    // source row of A row r: w13 interleaves gate / up by 8-row groups
    const int ga = r >> 3;
    const int blk = (ROLE == 0) ? (ga & 1) : (ga >> 3);
    const int sg = (ROLE == 0) ? (ga >> 1) : (ga & 7);  // 8-row group within the block
    const int sr = r & 7;
    SKWalk wk;
    wk.begin();
    int achunk = 0;
    [[maybe_unused]] int tlc = 0;
    bool ok = true;
    const bool tl0 = (dw == 0 && lane == 0);
    if (tl0) TL(2, tlc, 0);
    for (int n = 0; n < count && ok; ++n) {
      wk.next(R);
      const int st = n % S;
      if (!__all_sync(0xffffffffu, wait(&full_b[st], (uint32_t)(n / S) & 1u))) {
        if (lane == 0) fail();
        break;
      }
      if (tl0) TL(2, tlc, 1);
      const int nc = min(kSliceChunks, NC - wk.slice * kSliceChunks);
      const uint8_t* stg = sbase + st * C::stage_bytes;
      for (int c = 0; c < nc; ++c, ++achunk) {
        const int as = achunk % kNA, use = achunk / kNA;
        if (use > 0 && !__all_sync(0xffffffffu, wait(&cempty[as], (uint32_t)(use - 1) & 1u))) {
          if (lane == 0) fail();
          ok = false;
          break;
        }
        tc::fence_after_sync();
        if (tl0) TL(2, tlc, 2);
        // codes of the row's chunk in the pack's byte order: unit q, bytes
        // 2j, 2j + 1 = elements 16j + 4q .. + 3. k-steps j = 4hh .. 4hh + 3
        // are words 2hh, 2hh + 1 of every unit
        const uint8_t* crow = stg + blk * 8 * nc * 512 + (sg * nc + c) * 512 + sr * 64 + hh * 8;
        uint2 cw[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) cw[q] = *reinterpret_cast<const uint2*>(crow + 16 * q);
        const uint8_t* srow = stg + 2 * kTCodeBlock + blk * C::scale_block +
                              (sg * nc + c) * 8 * C::SB + sr * C::SB;
        uint32_t s2[4];  // block scale of k-step 4hh + jj as f16x2
        if constexpr (Q == kMXFP4) {
          const uint32_t sw = *reinterpret_cast<const uint32_t*>(srow);
#pragma unroll
          for (int b = 0; b < 2; ++b) {  // k-steps 4hh + 2b, + 1 share a UE8M0 scale
            const uint32_t f = ue8m0_to_f16_bits((sw >> (8 * (2 * hh + b))) & 0xFFu);
            if (f == 0u) atomicOr(p.health, kHealthWRange);
            s2[2 * b] = s2[2 * b + 1] = f | (f << 16);
          }
        } else {
          const uint32_t sw = *(reinterpret_cast<const uint32_t*>(srow) + hh);
#pragma unroll
          for (int b = 0; b < 2; ++b) {
            const uint32_t f = e4m3x2_to_f16x2((sw >> (16 * b)) & 0xFFFFu);
            s2[2 * b] = __byte_perm(f, f, 0x1010);
            s2[2 * b + 1] = __byte_perm(f, f, 0x3232);
          }
        }
        // column 8 jj + 2q + e (jj = j - 4hh) holds elements 16j + 4q + 2e, + 1
        uint32_t v[32];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
#pragma unroll
          for (int wd = 0; wd < 2; ++wd) {  // word wd: k-steps 2wd (bytes 0, 1), 2wd + 1 (bytes 2, 3)
            uint32_t a0, a1, a2, a3;
            e2m1x8_to_f16x2x4(wd == 0 ? cw[q].x : cw[q].y, a0, a1, a2, a3);
            v[8 * (2 * wd) + 2 * q] = hmul2(a0, s2[2 * wd]);
            v[8 * (2 * wd) + 2 * q + 1] = hmul2(a1, s2[2 * wd]);
            v[8 * (2 * wd + 1) + 2 * q] = hmul2(a2, s2[2 * wd + 1]);
            v[8 * (2 * wd + 1) + 2 * q + 1] = hmul2(a3, s2[2 * wd + 1]);
          }
        }
        const uint32_t ta = tmem + kTAOff + as * kTAcc + hh * 32 + t_lane;
        tc::st_32x32b_x16(ta, *reinterpret_cast<const uint32_t(*)[16]>(&v[0]));
        tc::st_32x32b_x16(ta + 16, *reinterpret_cast<const uint32_t(*)[16]>(&v[16]));
        tc::wait_st();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&cfull[as]));
        if (tl0) TL(2, tlc, 3);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty_b[st]));  // the codes of the unit are used
    }
  } else if (warp < kTEpi) {
    // ---------------- epilogue: tensor memory -> outputs ----------------
    pdl_wait();  // the activation scales, and the outputs' previous readers
    const int row = warp * 32 + lane;  // tensor-memory lane = A row
    const uint32_t t_row = (uint32_t)(warp * 32) << 16;
    [[maybe_unused]] int tlc = 0;
    if (tid == 0) TL(4, tlc, 0);
    SKWalk wk;
    wk.begin();
    int acc = 0, acc_use = 0, gcur = -1;
    int4 gd = make_int4(0, 0, 0, 0);
    float4* part = reinterpret_cast<float4*>(p.part);
    const int slot_f4 = kTM * kTAcc / 4;  // float4 per partial slot
    for (int n = 0; n < count; ++n) {
      wk.next(R);
      if (!wk.closes(R)) continue;
      if (wk.grp != gcur) {
        gcur = wk.grp;
        gd = group_of(gcur);
      }
      const int e = gd.x, ntok = gd.z;
      // the tile's weight-row scales, loaded ahead of the accumulator wait
      // so that their latency hides behind it: w13 gate / up row scales
      // (sg, su), w2 the row's scale (sg); NVFP4 the expert's global scale
      float sg = 1.f, su = 1.f;
      if (Q == kNVFP4 || Q == kA4NV) sg = su = __ldg(p.gscale + e);
      if (Q == kFP8) {
        const float* ws = reinterpret_cast<const float*>(p.scale);
        if (ROLE == 0) {
          const int i = wk.tile * 64 + (row >> 4) * 8 + (row & 7);
          sg = __ldg(ws + (size_t)e * p.N + i);
          su = __ldg(ws + (size_t)e * p.N + p.I + i);
        } else {
          sg = __ldg(ws + (size_t)e * p.N + wk.tile * 128 + row);
        }
      }
      if (!__all_sync(0xffffffffu, wait(&accfull[acc], (uint32_t)(acc_use / C::n_acc) & 1u))) {
        if (lane == 0) fail();
        break;
      }
      if (tid == 0) TL(4, tlc, 1);
      tc::fence_after_sync();
      const int ncol = (ntok + 15) >> 4;  // 16-column chunks holding tokens
      const int tb = wk.u - wk.slice;     // the tile's first unit
      const bool tile_end = (wk.slice == KS - 1);
      const uint32_t tsrc = tmem + acc * kTAcc + t_row;
      int mode = (tile_end && tb >= wk.lo) ? 0 : (!tile_end ? 1 : 2);  // finish, leave, own
      const int c_first = tc_cta_of(tb, U, GE), c_last = tc_cta_of(tb + KS - 1, U, GE);
      auto slot_of = [&](int c) -> int {
        const int which = (tc_start(c, U, GE) >= tb) ? 0 : 1;
        return (c * 2 + which) * slot_f4;
      };
      int32_t* flag = p.tickets + ((size_t)gcur * tiles + wk.tile) * 8 + warp;
      bool good = true;
      if (mode == 2) {
        // wait (bounded) until the tile's other CTAs have signalled
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
        good = __shfl_sync(0xffffffffu, got, 0) != 0;
        if (!good && lane == 0) fail();
      }
      bool released = false;
      for (int cc = 0; cc < ncol && good; ++cc) {
        float v[16];
        tc::ld_32x32b_x16(tsrc + cc * 16, v);
        tc::wait_ld();
        if (cc == ncol - 1) {
          // the accumulator is in registers: the MMA lane may reuse it
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&accempty[acc]));
          released = true;
        }
        if (mode == 1) {
          float4* dst = part + slot_of(blockIdx.x) + (cc * kTM + row) * 4;
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
          continue;
        }
        if (mode == 2) {
          // the other CTAs' partials, summed in CTA order; two contributors'
          // loads are in flight together
          float s[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) s[i] = 0.f;
          int c = c_first;
          for (; c < c_last; c += 2) {
            const bool two = c + 1 < c_last;
            const float4* s0 = part + slot_of(c) + (cc * kTM + row) * 4;
            const float4* s1 = part + slot_of(two ? c + 1 : c) + (cc * kTM + row) * 4;
            float4 x0[4], x1[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) x0[i] = __ldcg(s0 + i);
#pragma unroll
            for (int i = 0; i < 4; ++i) x1[i] = two ? __ldcg(s1 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              s[4 * i] += x0[i].x;
              s[4 * i + 1] += x0[i].y;
              s[4 * i + 2] += x0[i].z;
              s[4 * i + 3] += x0[i].w;
            }
            if (two) {
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                s[4 * i] += x1[i].x;
                s[4 * i + 1] += x1[i].y;
                s[4 * i + 2] += x1[i].z;
                s[4 * i + 3] += x1[i].w;
              }
            }
          }
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = s[i] + v[i];
        }
        if (ROLE == 0) {
          // lanes l (gate) and l ^ 8 (up) hold the same i: the gate lane
          // finishes columns 0..7 of the chunk, the up lane 8..15
          const bool is_gate = ((row >> 3) & 1) == 0;
          const int i = wk.tile * 64 + (row >> 4) * 8 + (row & 7);
          float g8[8], u8[8];
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            const float send = is_gate ? v[8 + t] : v[t];
            const float recv = __shfl_xor_sync(0xffffffffu, send, 8);
            g8[t] = is_gate ? v[t] : recv;
            u8[t] = is_gate ? recv : v[8 + t];
          }
          // the chunk's routes (and FP8 activation scales), all loads in
          // flight together ahead of the stores
          int ro8[8];
          float bs8[8];
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            const int nn = cc * 16 + (is_gate ? 0 : 8) + t;
            ro8[t] = nn < ntok ? route_of(gcur, gd.y, nn) : -1;
          }
#pragma unroll
          for (int t = 0; t < 8; ++t)
            bs8[t] = (Q == kFP8 && ro8[t] >= 0) ? __ldcg(p.b_scale + ro8[t] / p.k) : 1.f;
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            const int ro = ro8[t];
            if (ro < 0) break;
            float gs = sg, us = su;
            if (Q == kFP8) {
              gs *= bs8[t];
              us *= bs8[t];
            }
            const float a = round_bf16(silu(g8[t] * gs) * (u8[t] * us));
            if (Q == kFP8 || p.act_bf16) {
              reinterpret_cast<uint16_t*>(p.out)[(size_t)ro * p.I + i] = f32_to_bf16_bits(a);
            } else {
              reinterpret_cast<__half*>(p.out)[(size_t)ro * p.I + i] = __float2half_rn(a);
              if (!(fabsf(a) <= 65504.f)) atomicOr(p.health, kHealthActRange);
            }
          }
        } else {
          const int pr = wk.tile * 128 + row;
          const float sc = sg;
          int ro16[16];
          float bs16[16];
#pragma unroll
          for (int t = 0; t < 16; ++t) ro16[t] = cc * 16 + t < ntok ? route_of(gcur, gd.y, cc * 16 + t) : -1;
#pragma unroll
          for (int t = 0; t < 16; ++t) bs16[t] = (Q == kFP8 && ro16[t] >= 0) ? __ldcg(p.b_scale + ro16[t]) : 1.f;
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            const int ro = ro16[t];
            if (ro < 0) break;
            float s = sc;
            if (Q == kFP8) s *= bs16[t];
            reinterpret_cast<float*>(p.out)[(size_t)ro * p.P + pr] = v[t] * s;
          }
        }
      }
      if (mode == 1) {
        __syncwarp();  // orders the lanes' partial stores before lane 0's release
        if (lane == 0) asm volatile("red.release.gpu.global.add.s32 [%0], 1;\n" ::"l"(flag) : "memory");
      }
      if (!released) {
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&accempty[acc]));
      }
      if (tid == 0) TL(4, tlc, 2 + mode);
      acc = acc + 1 == C::n_acc ? 0 : acc + 1;
      ++acc_use;
      if (!good) break;
    }
  }

  // every role is done: the MMAs have completed (drained), the tensor memory
  // loads are waited for; free the tensor memory
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tmem, C::tmem_cols);
}

template <int Q, int ROLE>
static cudaError_t launch_tc_t(const ExpertParams& p, cudaStream_t s, bool pdl) {
  constexpr int smem = tc_smem_bytes<Q>();
  auto kern = k_expert_tc<Q, ROLE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(TcCfg<Q>::threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

cudaError_t launch_expert_tc(const ExpertParams& p, cudaStream_t s, bool pdl) {
  if (p.act4) {
    if (p.quant != (p.act4 == 2 ? kNVFP4 : kMXFP4) || !p.b_sf) return cudaErrorInvalidValue;
    switch ((p.act4 == 2 ? 2 : 0) + p.role) {
      case 0: return launch_tc_t<kA4MX, 0>(p, s, pdl);
      case 1: return launch_tc_t<kA4MX, 1>(p, s, pdl);
      case 2: return launch_tc_t<kA4NV, 0>(p, s, pdl);
      case 3: return launch_tc_t<kA4NV, 1>(p, s, pdl);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (p.quant * 2 + p.role) {
    case 0: return launch_tc_t<kMXFP4, 0>(p, s, pdl);
    case 1: return launch_tc_t<kMXFP4, 1>(p, s, pdl);
    case 2: return launch_tc_t<kNVFP4, 0>(p, s, pdl);
    case 3: return launch_tc_t<kNVFP4, 1>(p, s, pdl);
    case 4: return launch_tc_t<kFP8, 0>(p, s, pdl);
    case 5: return launch_tc_t<kFP8, 1>(p, s, pdl);
    default: return cudaErrorInvalidValue;
  }
}

#ifdef MUSEMOE_TIMELINE
extern "C" int musemoe_tc_timeline_read(void* host, int reset) {
  if (host && cudaMemcpyFromSymbol(host, g_tc_tl, sizeof(g_tc_tl)) != cudaSuccess) return 1;
  if (reset) {
    void* d = nullptr;
    if (cudaGetSymbolAddress(&d, g_tc_tl) != cudaSuccess) return 2;
    if (cudaMemset(d, 0, sizeof(g_tc_tl)) != cudaSuccess) return 3;
  }
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : 4;
}
#endif

size_t expert_tc_part_bytes(int grid) { return (size_t)grid * 2 * kTM * kTAcc * sizeof(float); }
int expert_tc_group_tokens() { return kTN; }

}  // namespace musemoe
