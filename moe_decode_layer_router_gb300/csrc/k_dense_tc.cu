// Dense bf16 GEMM Y[rows, M] = X[rows, K] W[M, K]^T on the fifth-generation
// tensor cores (tcgen05, kind::f16 with bf16 operands, fp32 accumulation in
// tensor memory), for the pooler (H -> P) and the unpooler (P -> H) of the
// larger buckets, where the token count makes them dense contractions (page
// "vllm.models.muse_spark.nvidia.specialized_decode.runtime.providers",
// MoEProvider: the pooler GEMM and the unpooler GEMM of the routed MoE).
//
// One CTA per SM (persistent), Stream-K over units = (token block of up to
// 256 rows, tile of 128 weight rows, 64-element K block). The MMA is
// D[128 weight rows x N tokens] += W_tile[128 x 64] X_block[N x 64]^T with N
// the block's rows rounded up to 16. A producer lane loads both operands
// with 2-D tensor copies (128-byte swizzle: the canonical K-major layout the
// MMA reads); an MMA lane issues 4 MMAs per unit; 4 epilogue warps read the
// accumulators (two, so a tile's epilogue overlaps the next tile's MMAs) and
// store Y, or a partial sum when the tile's K blocks span several CTAs; the
// contributors of a split tile then share its final sums (below), each
// adding all partials in CTA order, so results do not depend on scheduling.
// Rows past the end are zero-filled by the tensor copy and never stored.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "pipeline.cuh"
#include "tc.cuh"

namespace musemoe {

namespace {

constexpr int kDM = 128;                       // weight rows per tile
constexpr int kDK = 64;                        // K elements per unit (128 B)
constexpr int kDN = 256;                       // tokens per block at most
constexpr int kDStages = 4;
constexpr int kDStageA = kDM * 128;            // 16 KB
constexpr int kDStageB = kDN * 128;            // 32 KB
constexpr int kDStage = kDStageA + kDStageB;   // 48 KB
constexpr int kDSmem = 1024 + kDStages * kDStage;
constexpr int kDEpi = 4;
constexpr int kDThreads = (kDEpi + 2) * 32;    // epilogue, producer, MMA
constexpr int kDTmemCols = 512;                // two accumulators of up to 256 columns

__device__ __forceinline__ int d_cta_of(long long u, long long U, int G) {
  return (int)(((u + 1) * G - 1) / U);
}
__device__ __forceinline__ long long d_start(int c, long long U, int G) { return U * c / G; }

struct DRange {
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
};
// units in processing order: whole tiles, then the leading part (leave a
// partial), then the trailing part (own the tile): no wait depends on a
// waiting CTA
struct DWalk {
  int u, blk, tile, kb, lo, hi, part, left;
  __device__ void begin() {
    part = -1;
    left = 0;
  }
  __device__ void next(const DRange& R) {
    if (left == 0) {
      do {
        ++part;
      } while (part < 3 && R.hi(part) <= R.lo(part));
      lo = R.lo(part);
      hi = R.hi(part);
      left = hi - lo;
      u = lo;
      blk = u / R.PG;
      const int rem = u - blk * R.PG;
      tile = rem / R.KS;
      kb = rem - tile * R.KS;
    } else {
      ++u;
      if (++kb == R.KS) {
        kb = 0;
        if (++tile == R.tiles) {
          tile = 0;
          ++blk;
        }
      }
    }
    --left;
  }
  __device__ bool closes(const DRange& R) const { return kb == R.KS - 1 || u + 1 == hi; }
};

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%2, %3}], [%4], %5;\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(pol)
      : "memory");
}

}  // namespace

// Optional phase timeline (compile with -DMUSEMOE_TIMELINE): stamps of the
// producer (0), MMA (1) and epilogue warp 0 (2) in CTAs 0, 1, G/2, G-1; the
// event kind in the low 4 bits; read with musemoe_dense_timeline_read.
#ifdef MUSEMOE_TIMELINE
constexpr int kDTlEvents = 512;
__device__ unsigned long long g_dense_tl[4][3][kDTlEvents];
__device__ __forceinline__ int dtl_cta() {
  const int b = blockIdx.x, g = gridDim.x;
  return b == 0 ? 0 : b == 1 ? 1 : b == g / 2 ? 2 : b == g - 1 ? 3 : -1;
}
#define DTL(role, cnt, kind)                                                                   \
  do {                                                                                         \
    const int tl_c = dtl_cta();                                                                \
    if (tl_c >= 0 && (cnt) < kDTlEvents)                                                       \
      g_dense_tl[tl_c][role][(cnt)++] = (globaltimer() & ~15ull) | (unsigned long long)(kind); \
  } while (0)
extern "C" int musemoe_dense_timeline_read(void* host, int reset) {
  if (host && cudaMemcpyFromSymbol(host, g_dense_tl, sizeof(g_dense_tl)) != cudaSuccess) return 1;
  if (reset) {
    void* d = nullptr;
    if (cudaGetSymbolAddress(&d, g_dense_tl) != cudaSuccess) return 2;
    if (cudaMemset(d, 0, sizeof(g_dense_tl)) != cudaSuccess) return 3;
  }
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : 4;
}
#else
#define DTL(role, cnt, kind) \
  do {                       \
  } while (0)
#endif

__global__ void __launch_bounds__(kDThreads, 1)
    k_dense_tc(const __grid_constant__ CUtensorMap tw, const __grid_constant__ CUtensorMap tx,
               DenseParams p) {
  pdl_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) unsigned long long full_b[kDStages], empty_b[kDStages];
  __shared__ __align__(8) unsigned long long accfull[2], accempty[2], drain_b;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;

  const int tiles = (p.M + kDM - 1) / kDM;
  const int KS = p.K / kDK;
  const int blocks = (p.rows + kDN - 1) / kDN;
  const long long U = (long long)blocks * tiles * KS;
  const int GE = (int)min((long long)gridDim.x, U);
  const long long u0 = blockIdx.x < GE ? d_start(blockIdx.x, U, GE) : 0;
  const long long u1 = blockIdx.x < GE ? d_start(blockIdx.x + 1, U, GE) : 0;
  DRange R;
  R.init(u0, u1, KS, tiles);
  const int count = R.U1 - R.U0;

  if (tid == 0) {
    for (int i = 0; i < kDStages; ++i) {
      mbar_init(smem_u32(&full_b[i]), 1);
      mbar_init(smem_u32(&empty_b[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&accfull[i]), 1);
      mbar_init(smem_u32(&accempty[i]), kDEpi);
    }
    mbar_init(smem_u32(&drain_b), 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == 0) {
    tc::tmem_alloc(smem_u32(&tmem_slot), kDTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_slot;
  auto fail = [&]() {
    if (atomicExch(&abort_flag, 1) == 0) atomicOr(p.health, kHealthTimeout);
  };
  auto wait = [&](unsigned long long* bar, uint32_t phase) -> bool {
    return mbar_wait_or_abort(smem_u32(bar), phase, &abort_flag);
  };
  auto rows_of = [&](int blk) { return min(kDN, p.rows - blk * kDN); };
  const int box_rows = min(kDN, (p.rows + 15) & ~15);  // rows of the token tensor copy

  if (warp == kDEpi) {
    // ---------------- producer: weight tile and token rows of each unit ----------------
    if (lane == 0) {
      int tlc = 0;
      DTL(0, tlc, 0);
      const uint64_t pol_w = l2_policy_evict_first();
      uint64_t pol_x;
      asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;\n" : "=l"(pol_x));
      DWalk wk;
      wk.begin();
      int issued = 0;
      bool waited = false;
      for (int n = 0; n < count; ++n) {
        wk.next(R);
        const int st = n % kDStages, use = n / kDStages;
        if (use > 0 && !wait(&empty_b[st], (uint32_t)(use - 1) & 1u)) {
          fail();
          break;
        }
        const uint32_t bar = smem_u32(&full_b[st]);
        const uint32_t dst = base + st * kDStage;
        mbar_expect_tx(bar, kDStageA + box_rows * 128);  // the copy writes the whole box
        // the weights never depend on the previous kernel; the token rows do
        tma_load_2d(dst, &tw, wk.kb * kDK, wk.tile * kDM, bar, pol_w);
        if (!waited) {
          pdl_wait();
          waited = true;
        }
        tma_load_2d(dst + kDStageA, &tx, wk.kb * kDK, wk.blk * kDN, bar, pol_x);
        issued = n + 1;
        DTL(0, tlc, 1);
      }
      for (int st = 0; st < kDStages && st < issued; ++st) {
        const int last = st + ((issued - 1 - st) / kDStages) * kDStages;
        const unsigned long long t0 = globaltimer();
        while (!mbar_try_wait(smem_u32(&full_b[st]), (uint32_t)(last / kDStages) & 1u))
          if (globaltimer() - t0 > kWaitLimitNs) break;
      }
    }
  } else if (warp == kDEpi + 1) {
    // ---------------- MMA issue (one lane) ----------------
    if (lane == 0) {
      int tlc = 0;
      DTL(1, tlc, 0);
      DWalk wk;
      wk.begin();
      int acc = 0, acc_use = 0;
      bool fresh = true;
      for (int n = 0; n < count; ++n) {
        wk.next(R);
        if (fresh) {
          if (acc_use > 1 && !wait(&accempty[acc], (uint32_t)((acc_use >> 1) - 1) & 1u)) {
            fail();
            break;
          }
          tc::fence_after_sync();
        }
        const int st = n % kDStages;
        if (!wait(&full_b[st], (uint32_t)(n / kDStages) & 1u)) {
          fail();
          break;
        }
        DTL(1, tlc, 1);
        tc::fence_after_sync();
        const int npad = (rows_of(wk.blk) + 15) & ~15;
        const uint32_t idesc = tc::instr_desc(tc::kBF16, tc::kBF16, kDM, npad);
        const uint64_t da = tc::smem_desc(base + st * kDStage, 16, 1024, tc::kSw128);
        const uint64_t db = tc::smem_desc(base + st * kDStage + kDStageA, 16, 1024, tc::kSw128);
        const uint32_t d_tmem = tmem + acc * kDN;
#pragma unroll
        for (int j = 0; j < 4; ++j)  // K = 16 per MMA: 32 bytes further in the 128-byte rows
          tc::mma_f16(d_tmem, da + (uint64_t)(2 * j), db + (uint64_t)(2 * j), idesc,
                      (fresh && j == 0) ? 0u : 1u);
        tc::commit(smem_u32(&empty_b[st]));
        fresh = false;
        if (wk.closes(R)) {
          tc::commit(smem_u32(&accfull[acc]));
          acc ^= 1;
          ++acc_use;
          fresh = true;
        }
      }
      tc::commit(smem_u32(&drain_b));
      const unsigned long long t0 = globaltimer();
      while (!mbar_try_wait(smem_u32(&drain_b), 0u))
        if (globaltimer() - t0 > kWaitLimitNs) break;
    }
  } else {
    // ---------------- epilogue (warps 0..3): tensor memory -> Y ----------------
    // A tile finished inside this CTA is stored directly. A tile whose K
    // blocks span several CTAs: every contributor stores its partial and
    // signals the tile's ticket as soon as its part closes; only after all of
    // its own parts does it wait for the tile's other contributors, then sums
    // its share of the tile's 16-column chunks (chunk cc goes to contributor
    // cc mod n) over all partials in CTA order. Every signal comes before
    // every wait, so no wait depends on a waiting CTA; the sums do not
    // depend on scheduling.
    pdl_wait();  // Y's previous readers are done
    const int row = warp * 32 + lane;  // weight row within the tile
    const uint32_t t_row = (uint32_t)(warp * 32) << 16;
    int tlc = 0;
    if (tid == 0) DTL(2, tlc, 0);
    DWalk wk;
    wk.begin();
    int acc = 0, acc_use = 0;
    float4* part = reinterpret_cast<float4*>(p.part);
    const int slot_f4 = kDM * kDN / 4;
    auto slot_of = [&](int c, int tb) -> int {
      const int which = (d_start(c, U, GE) >= tb) ? 0 : 1;  // the CTA's first or last tile
      return (c * 2 + which) * slot_f4;
    };
    int nsplit = 0;
    int sp_blk[2] = {0, 0}, sp_tile[2] = {0, 0}, sp_tb[2] = {0, 0};
    bool good = true;
    for (int n = 0; n < count && good; ++n) {
      wk.next(R);
      if (!wk.closes(R)) continue;
      if (!__all_sync(0xffffffffu, wait(&accfull[acc], (uint32_t)(acc_use >> 1) & 1u))) {
        if (lane == 0) fail();
        good = false;
        break;
      }
      if (tid == 0) DTL(2, tlc, 1);
      tc::fence_after_sync();
      const int nr = rows_of(wk.blk);
      const int ncol = (nr + 15) >> 4;
      const int tb = wk.u - wk.kb;
      const bool whole = (wk.kb == KS - 1) && tb >= wk.lo;
      const uint32_t tsrc = tmem + acc * kDN + t_row;
      const int m = wk.tile * kDM + row;
      // 32 columns (two 16-column chunks) per tensor-memory load and wait
      for (int c2 = 0; c2 < ncol; c2 += 2) {
        float v2[32];
        tc::ld_32x32b_x32(tsrc + c2 * 16, v2);
        tc::wait_ld();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int cc = c2 + h;
          if (cc >= ncol) break;
          const float* v = v2 + 16 * h;
          if (!whole) {
            float4* dst = part + slot_of(blockIdx.x, tb) + (cc * kDM + row) * 4;
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
          } else if (m < p.M) {
#pragma unroll
            for (int t = 0; t < 16; ++t) {
              const int tok = cc * 16 + t;
              if (tok < nr) p.y[(size_t)(wk.blk * kDN + tok) * p.M + m] = v[t];
            }
          }
        }
      }
      if (!whole) {
        __syncwarp();  // orders the lanes' partial stores before lane 0's release
        int32_t* flag = p.tickets + (((size_t)wk.blk * tiles + wk.tile) * kDEpi + warp) * 2;
        if (lane == 0) asm volatile("red.release.gpu.global.add.s32 [%0], 1;\n" ::"l"(flag) : "memory");
        sp_blk[nsplit] = wk.blk;
        sp_tile[nsplit] = wk.tile;
        sp_tb[nsplit] = tb;
        ++nsplit;
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&accempty[acc]));
      if (tid == 0) DTL(2, tlc, 3 + (whole ? 0 : 1));
      acc ^= 1;
      ++acc_use;
    }
    // the split tiles' sums: this CTA's share of each
    for (int k = 0; k < nsplit && good; ++k) {
      const int blk = sp_blk[k], tile = sp_tile[k], tb = sp_tb[k];
      const int c_first = d_cta_of(tb, U, GE), c_last = d_cta_of(tb + KS - 1, U, GE);
      const int ncon = c_last - c_first + 1;  // contributors, this CTA among them
      int32_t* flag = p.tickets + (((size_t)blk * tiles + tile) * kDEpi + warp) * 2;
      int got = 1;
      if (lane == 0) {
        int v = 0;
        asm volatile("ld.acquire.gpu.global.s32 %0, [%1];\n" : "=r"(v) : "l"(flag) : "memory");
        if (v < ncon) {
          const unsigned long long t0 = globaltimer();
          do {
            __nanosleep(128);
            asm volatile("ld.acquire.gpu.global.s32 %0, [%1];\n" : "=r"(v) : "l"(flag) : "memory");
          } while (v < ncon && globaltimer() - t0 <= kWaitLimitNs && !abort_flag);
        }
        got = (v >= ncon);
      }
      if (!__shfl_sync(0xffffffffu, got, 0)) {
        if (lane == 0) fail();
        good = false;
        break;
      }
      if (tid == 0) DTL(2, tlc, 2);
      const int nr = rows_of(blk);
      const int ncol = (nr + 15) >> 4;
      const int m = tile * kDM + row;
      for (int cc = (int)blockIdx.x - c_first; cc < ncol; cc += ncon) {
        float s[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) s[i] = 0.f;
        int c = c_first;
        // four contributors' loads in flight at a time, added in CTA order
        for (; c + 4 <= c_last + 1; c += 4) {
          float4 x[4][4];
#pragma unroll
          for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int i = 0; i < 4; ++i) x[a][i] = __ldcg(part + slot_of(c + a, tb) + (cc * kDM + row) * 4 + i);
#pragma unroll
          for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              s[4 * i] += x[a][i].x;
              s[4 * i + 1] += x[a][i].y;
              s[4 * i + 2] += x[a][i].z;
              s[4 * i + 3] += x[a][i].w;
            }
        }
        for (; c <= c_last; ++c)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float4 x = __ldcg(part + slot_of(c, tb) + (cc * kDM + row) * 4 + i);
            s[4 * i] += x.x;
            s[4 * i + 1] += x.y;
            s[4 * i + 2] += x.z;
            s[4 * i + 3] += x.w;
          }
        if (m < p.M) {
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            const int tok = cc * 16 + t;
            if (tok < nr) p.y[(size_t)(blk * kDN + tok) * p.M + m] = s[t];
          }
        }
      }
      // the last contributor done with the tile zeroes its tickets for the next launch
      __syncwarp();
      if (lane == 0) {
        int d = 0;
        asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;\n" : "=r"(d) : "l"(flag + 1) : "memory");
        if (d == ncon - 1) {
          flag[0] = 0;
          flag[1] = 0;
        }
      }
      if (tid == 0) DTL(2, tlc, 5);
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tmem, kDTmemCols);
}

// ---- host --------------------------------------------------------------------
namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_enc = nullptr;
std::once_flag g_enc_once;

// 2-D bf16 view of a row-major [rows, K] tensor, box (64 elements, box_rows),
// 128-byte swizzle, zero fill past the end.
cudaError_t map_2d(CUtensorMap* m, const void* base, uint64_t K, uint64_t rows, uint32_t box_rows) {
  std::call_once(g_enc_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {K, rows};
  const cuuint64_t strides[1] = {K * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kDK, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                           strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}
}  // namespace

cudaError_t launch_dense_tc(const DenseParams& p, cudaStream_t s, bool pdl) {
  if (p.K % kDK || p.rows < 1) return cudaErrorInvalidValue;
  CUtensorMap tw{}, tx{};
  const int box_rows = std::min(kDN, (p.rows + 15) & ~15);
  cudaError_t e = map_2d(&tw, p.w, (uint64_t)p.K, (uint64_t)p.M, kDM);
  if (e == cudaSuccess) e = map_2d(&tx, p.x, (uint64_t)p.K, (uint64_t)p.rows, (uint32_t)box_rows);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k_dense_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, kDSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(kDThreads);
  cfg.dynamicSmemBytes = kDSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_dense_tc, tw, tx, p);
}

size_t dense_tc_part_bytes(int grid) { return (size_t)grid * 2 * kDM * kDN * sizeof(float); }
size_t dense_tc_tickets(int rows, int M) {
  return (size_t)((rows + kDN - 1) / kDN) * ((M + kDM - 1) / kDM) * kDEpi * 2;
}

}  // namespace musemoe
