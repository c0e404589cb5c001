// Dense bf16 GEMM Y[rows, M] = X[rows, K] W[M, K]^T on the fifth-generation
// tensor cores (tcgen05, kind::f16 with bf16 operands, fp32 accumulation in
// tensor memory), for the pooler (H -> P) and the unpooler (P -> H) of the
// larger buckets, where the token count makes them dense contractions (page
// "vllm.models.muse_spark.nvidia.specialized_decode.runtime.providers",
// MoEProvider: the pooler GEMM and the unpooler GEMM of the routed MoE).
//
// Split K across a thread-block cluster: one cluster per work item (a tile of
// 128 weight rows x a token block of up to 256 rows), its C CTAs each
// accumulate a disjoint range of the 64-element K blocks. C is the largest
// size (at most 8, at most the K blocks, at most the SMs' share per item) at
// which all the items' clusters are resident at once, so the launch is one
// wave. The MMA is D[128 weight rows x N tokens] +=
// W_tile[128 x 64] X_block[N x 64]^T with N the block's rows rounded up to
// 16. A producer lane loads both operands with 2-D tensor copies (128-byte
// swizzle: the canonical K-major layout the MMA reads) into a 4-stage ring;
// an MMA lane issues 4 MMAs per K block into one tensor-memory accumulator.
// The partial sums never leave the cluster: after a cluster barrier (every
// CTA's MMAs done, its stages free) the 4 epilogue warps write each row of
// their accumulator into the stage memory of the row's owner (rank r owns
// rows [ceil(128 r / C), ceil(128 (r + 1) / C))) through distributed shared
// memory; after a second barrier each owner adds the C slots of its rows in
// rank order and stores Y (8 rows x 4 tokens per warp step), so results do
// not depend on scheduling. Rows past the end are zero-filled by the tensor
// copy and never stored. The weight copies never wait for the previous
// kernel; the token rows' copies do unless x_ready (the pooler's input, final
// before the router launches), and every thread waits before it stores Y, so
// the launch completes only after its predecessor.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
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
constexpr int kDTmemCols = kDN;                // one accumulator of up to 256 columns
constexpr int kDMaxCluster = 8;
// A slot row (one output row's N fp32) is N + 4 floats apart from the next:
// the 32 lanes of a warp, one row each, then store to distinct banks, and
// the summing threads (8 rows x 4 tokens per warp) load from distinct banks.
constexpr int kDSlotPad = 4;
// the exchange slots (C of them, each the owner's rows x N fp32) fit the stages
constexpr bool dense_slots_fit() {
  for (int c = 1; c <= kDMaxCluster; ++c)
    if (c * ((kDM + c - 1) / c) * (kDN + kDSlotPad) * 4 > kDStages * kDStage) return false;
  return true;
}
static_assert(dense_slots_fit(), "exchange slots within the stage memory");

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;\n" : "=r"(r));
  return r;
}
// every thread of every CTA of the cluster: release its earlier memory
// operations, then acquire the others'
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
// the shared::cluster address of a shared::cta address in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t peer_addr(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "f"(a), "f"(b), "f"(c),
               "f"(d)
               : "memory");
}
// first row of the tile that rank r of C owns (ceil(128 r / C))
__device__ __forceinline__ int own_first(int r, int C) { return (r * kDM + C - 1) / C; }

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
  __shared__ __align__(8) unsigned long long accfull, drain_b;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;

  const int C = (int)cluster_size(), r = (int)cluster_rank();
  const int tiles = (p.M + kDM - 1) / kDM;
  const int item = blockIdx.x / C;  // one (token block, tile) per cluster
  const int tile = item % tiles, blk = item / tiles;
  const int KS = p.K / kDK;
  const int k0 = r * KS / C, nk = (r + 1) * KS / C - k0;  // this CTA's K blocks
  const int nr = min(kDN, p.rows - blk * kDN);             // the block's rows
  const int npad = (nr + 15) & ~15;
  const int box_rows = min(kDN, (p.rows + 15) & ~15);      // rows of the token tensor copy

  if (tid == 0) {
    for (int i = 0; i < kDStages; ++i) {
      mbar_init(smem_u32(&full_b[i]), 1);
      mbar_init(smem_u32(&empty_b[i]), 1);
    }
    mbar_init(smem_u32(&accfull), 1);
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

  bool have = false;  // epilogue: the accumulator holds this CTA's partial
  if (warp == kDEpi) {
    // ---------------- producer: weight tile and token rows of each K block ----------------
    if (lane == 0) {
      [[maybe_unused]] int tlc = 0;
      DTL(0, tlc, 0);
      const uint64_t pol_w = l2_policy_evict_first();
      uint64_t pol_x;
      asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;\n" : "=l"(pol_x));
      int issued = 0;
      bool waited = false;
      for (int n = 0; n < nk; ++n) {
        const int st = n % kDStages, use = n / kDStages;
        if (use > 0 && !wait(&empty_b[st], (uint32_t)(use - 1) & 1u)) {
          fail();
          break;
        }
        const uint32_t bar = smem_u32(&full_b[st]);
        const uint32_t dst = base + st * kDStage;
        mbar_expect_tx(bar, kDStageA + box_rows * 128);  // the copy writes the whole box
        // the weights never depend on the previous kernel; the token rows
        // do, unless they are final before the launch (x_ready)
        tma_load_2d(dst, &tw, (k0 + n) * kDK, tile * kDM, bar, pol_w);
        if (!waited && !p.x_ready) {
          pdl_wait();
          waited = true;
        }
        tma_load_2d(dst + kDStageA, &tx, (k0 + n) * kDK, blk * kDN, bar, pol_x);
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
      [[maybe_unused]] int tlc = 0;
      DTL(1, tlc, 0);
      const uint32_t idesc = tc::instr_desc(tc::kBF16, tc::kBF16, kDM, npad);
      int n = 0;
      for (; n < nk; ++n) {
        const int st = n % kDStages;
        if (!wait(&full_b[st], (uint32_t)(n / kDStages) & 1u)) {
          fail();
          break;
        }
        DTL(1, tlc, 1);
        tc::fence_after_sync();
        const uint64_t da = tc::smem_desc(base + st * kDStage, 16, 1024, tc::kSw128);
        const uint64_t db = tc::smem_desc(base + st * kDStage + kDStageA, 16, 1024, tc::kSw128);
#pragma unroll
        for (int j = 0; j < 4; ++j)  // K = 16 per MMA: 32 bytes further in the 128-byte rows
          tc::mma_f16(tmem, da + (uint64_t)(2 * j), db + (uint64_t)(2 * j), idesc,
                      (n == 0 && j == 0) ? 0u : 1u);
        tc::commit(smem_u32(&empty_b[st]));
      }
      // the accumulator is complete (or, after a timeout, abandoned)
      tc::commit(smem_u32(n == nk ? &accfull : &drain_b));
      if (n != nk) {
        const unsigned long long t0 = globaltimer();
        while (!mbar_try_wait(smem_u32(&drain_b), 0u))
          if (globaltimer() - t0 > kWaitLimitNs) break;
      }
    }
  } else {
    // ---------------- epilogue (warps 0..3), part 1: the accumulator is complete ----------------
    if (nk > 0) {
      have = __all_sync(0xffffffffu, wait(&accfull, 0u));
      if (!have && lane == 0) fail();
    }
    tc::fence_after_sync();
  }
  [[maybe_unused]] int etl = 0;
  if (tid == 0) DTL(2, etl, 1);

  // every CTA of the cluster has finished its MMAs: its stage memory is free
  // for the exchange (all warps of every CTA reach both barriers on every path)
  __syncwarp();
  cluster_sync();
  if (tid == 0) DTL(2, etl, 5);

  const int R = (kDM + C - 1) / C;  // rows per owner slot
  const int ss = npad + kDSlotPad;    // floats from one slot row to the next
  if (warp < kDEpi) {
    // part 2: each row of this CTA's partial goes to slot r of the row's owner
    const int row = warp * 32 + lane;
    int o = 0;
    while (o + 1 < C && own_first(o + 1, C) <= row) ++o;
    const int lr = row - own_first(o, C);
    const uint32_t slot = peer_addr(base + (uint32_t)(((r * R + lr) * ss) * 4), (uint32_t)o);
    const uint32_t tsrc = tmem + ((uint32_t)(warp * 32) << 16);
    for (int c0 = 0; c0 < npad; c0 += 32) {
      float v[32];
      if (c0 + 16 < npad) {
        tc::ld_32x32b_x32(tsrc + c0, v);
      } else {
        float h[16];
        tc::ld_32x32b_x16(tsrc + c0, h);
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = h[i];
      }
      tc::wait_ld();
      const int nc = min(32, npad - c0);
      if (!have || nk == 0)
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.f;  // no K blocks (or abandoned): contributes zeros
#pragma unroll
      for (int i = 0; i < 32; i += 4)
        if (i < nc) st_cluster_v4(slot + (uint32_t)((c0 + i) * 4), v[i], v[i + 1], v[i + 2], v[i + 3]);
    }
  }
  if (tid == 0) DTL(2, etl, 2);
  tc::fence_before_sync();
  __syncwarp();
  cluster_sync();
  if (tid == 0) DTL(2, etl, 3);

  // Y is stored, and the launch completes, only after the previous kernel
  // (the pooler's: the router, whose routing the expert kernels read before
  // their own wait once this launch and the norm after it are done)
  pdl_wait();
  {
    // part 3: this CTA's rows, the C slots added in rank order, by every warp
    // of the CTA. A warp takes 8 rows x 4 token quads at a time: each lane
    // loads its row's quad from the C slots (16 bytes, distinct banks) and
    // stores 4 tokens; a token's 8 rows m are one 32-byte sector of y.
    const int rf = own_first(r, C), rn = own_first(r + 1, C) - rf;
    const int nq = (nr + 3) >> 2, rb = (rn + 7) >> 3, qb = (nq + 3) >> 2;
    const float* sl = reinterpret_cast<const float*>(smem_raw + (base - smem_u32(smem_raw)));
    for (int b = warp; b < rb * qb; b += kDThreads / 32) {
      const int lr = (b % rb) * 8 + (lane & 7), qd = (b / rb) * 4 + (lane >> 3);
      const int m = tile * kDM + rf + lr;
      if (lr >= rn || qd >= nq || m >= p.M) continue;
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int q = 0; q < kDMaxCluster; ++q) {
        if (q < C) {
          const float4 v = *reinterpret_cast<const float4*>(sl + (q * R + lr) * ss + 4 * qd);
          a.x += v.x;
          a.y += v.y;
          a.z += v.z;
          a.w += v.w;
        }
      }
      float* yo = p.y + (size_t)(blk * kDN + 4 * qd) * p.M + m;
      const int nt = nr - 4 * qd;  // tokens of this quad in the block
      yo[0] = a.x;
      if (nt > 1) yo[p.M] = a.y;
      if (nt > 2) yo[2 * (size_t)p.M] = a.z;
      if (nt > 3) yo[3 * (size_t)p.M] = a.w;
    }
  }
  if (tid == 0) DTL(2, etl, 4);

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

// How many clusters of C CTAs of this kernel (one per SM: its shared
// memory) can be resident at once (a cluster must fit one GPC); asked once
// per size.
int clusters_resident(int C) {
  static int known[kDMaxCluster + 1] = {0};  // 0 unknown, else count + 1
  if (known[C] == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C);
    cfg.blockDim = dim3(kDThreads);
    cfg.dynamicSmemBytes = kDSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    const cudaError_t e = cudaOccupancyMaxActiveClusters(&n, k_dense_tc, &cfg);
    if (e != cudaSuccess) {
      (void)cudaGetLastError();
      n = 0;
    }
    known[C] = n + 1;
  }
  return known[C] - 1;
}

cudaError_t launch_dense_tc(const DenseParams& p, cudaStream_t s, bool pdl) {
  if (p.K % kDK || p.rows < 1 || p.M < 1) return cudaErrorInvalidValue;
  CUtensorMap tw{}, tx{};
  const int box_rows = std::min(kDN, (p.rows + 15) & ~15);
  cudaError_t e = map_2d(&tw, p.w, (uint64_t)p.K, (uint64_t)p.M, kDM);
  if (e == cudaSuccess) e = map_2d(&tx, p.x, (uint64_t)p.K, (uint64_t)p.rows, (uint32_t)box_rows);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k_dense_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, kDSmem);
  if (e != cudaSuccess) return e;
  // one cluster per (token block, tile); as many K-splitting CTAs per
  // cluster as fill the SMs (p.grid), at most 8 and at most the K blocks
  const int items = ((p.rows + kDN - 1) / kDN) * ((p.M + kDM - 1) / kDM);
  // the largest cluster (at most 8 CTAs, at most the K blocks, at most the
  // SMs' share) whose clusters all fit at once: one wave
  int C = std::max(1, std::min(std::min(kDMaxCluster, p.K / kDK), p.grid / items));
  while (C > 1 && clusters_resident(C) < items) --C;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(items * C);
  cfg.blockDim = dim3(kDThreads);
  cfg.dynamicSmemBytes = kDSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, k_dense_tc, tw, tx, p);
}

// the cluster kernel keeps its partial sums on chip: no workspace beyond a
// token (a non-null pointer marks the dense path as available)

}  // namespace musemoe
