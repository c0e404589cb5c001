// Fifth-generation tensor core helpers (tcgen05, sm_103a): tensor memory
// allocation, shared-memory matrix descriptors, the instruction descriptor,
// the MMA issue and its completion, and tensor-memory loads. Inline PTX only.
//
// Conventions used by the kernels here:
// * cta_group::1, M = 128: row m of the accumulator D is tensor-memory lane m
//   and column n is column (base + n), one fp32 per cell. Warp w of a
//   warpgroup reads lanes 32 (w % 4) .. + 31.
// * Both operands K-major: A [M rows][K], B [N rows][K] (D = A B^T), staged
//   in shared memory in one of the canonical layouts below.
#pragma once
#include "common.cuh"

namespace musemoe {
namespace tc {

// ---- tensor memory ---------------------------------------------------------
// Allocates `cols` columns (a power of two, 32..512) for the CTA; one full
// warp executes it. The base address lands in shared memory at `dst_smem`.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t cols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(dst_smem),
               "r"(cols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(cols)
               : "memory");
}
// Orders tcgen05 operations across a thread synchronization (barrier or
// mbarrier): `before` ahead of the sync in the producing thread, `after`
// behind it in the consuming thread.
__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}

// ---- descriptors -------------------------------------------------------------
// Swizzle modes of the shared-memory descriptor (bits 61..63).
enum Swizzle : uint32_t { kSwNone = 0, kSw128 = 2, kSw64 = 4, kSw32 = 6 };

// Shared-memory matrix descriptor: start address, leading-dimension byte
// offset (K-major, no swizzle: the distance between core matrices adjacent
// in K), stride-dimension byte offset (the distance between 8-row groups),
// descriptor version 1 (bit 46), base offset 0 (atoms aligned to their
// size), swizzle mode.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              uint32_t swz) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= (uint64_t)(swz & 7u) << 61;
  return d;
}

// Operand formats of the instruction descriptor (bits 7..9 A, 10..12 B).
enum Fmt : uint32_t { kF16 = 0, kBF16 = 1, kE4M3 = 0 };

// Instruction descriptor of a dense MMA with fp32 accumulation, both
// operands K-major: D type (bits 4..5) = F32, A and B formats, N >> 3 (bits
// 17..22), M >> 4 (bits 24..28).
__host__ __device__ __forceinline__ uint32_t instr_desc(uint32_t afmt, uint32_t bfmt, int M, int N) {
  return (1u << 4) | (afmt << 7) | (bfmt << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// ---- MMA -------------------------------------------------------------------
// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread. accumulate = 0
// overwrites D.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_f8f6f4(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T: A (M rows x K) in tensor memory, row m in
// lane m, two 16-bit elements per 32-bit column in K order.
__device__ __forceinline__ void mma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Block-scaled FP4 MMA (kind::mxf4nvf4): A and B e2m1, two per byte, each
// 64-element K step scaled per block by scale factors in tensor memory
// (`sfa`, `sfb`: the column of the step's scale atom, see cp_scale_atom).
// scale_vec::4X: blocks of 16 with e4m3 scales (NVFP4), the atom's four
// bytes the step's four blocks; scale_vec::2X: blocks of 32 with UE8M0
// scales (MXFP4), an atom holding two steps, selected by the descriptor's
// scale-IDs 0 (bytes 0, 1) and 2 (bytes 2, 3).
__device__ __forceinline__ void mma_nvf4(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], "
      "[%5], p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_mxf4(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], "
      "[%5], p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}
// Instruction descriptor of the block-scaled FP4 MMA, both operands E2M1 (1)
// and K-major: B scale-ID (bits 4..5), A / B formats (7..9, 10..12), N >> 3
// (17..22), scale type (23: e4m3 0, UE8M0 1), M >> 4 (24..28), A scale-ID
// (29..30).
__host__ __device__ __forceinline__ uint32_t instr_desc_fp4(int M, int N, uint32_t ue8m0,
                                                            uint32_t sf_id) {
  return (sf_id << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | (ue8m0 << 23) |
         ((uint32_t)(M >> 4) << 24) | (sf_id << 29);
}
// One scale atom, shared memory -> tensor memory: 32 rows of 16 bytes (row l
// holds the four scale bytes of matrix rows l, l + 32, l + 64, l + 96), copied
// into four columns from `taddr` of lanes l of every lane quarter. Issued by
// the MMA thread; the MMAs it issues afterwards see the copy.
__device__ __forceinline__ void cp_scale_atom(uint32_t taddr, uint32_t smem_addr) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;\n" ::"r"(taddr),
               "l"(smem_desc(smem_addr, 128, 128, kSwNone))
               : "memory");
}

// The mbarrier at `bar` (shared) receives one arrival once every MMA this
// thread issued before has completed.
__device__ __forceinline__ void commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
      : "memory");
}

// ---- tensor memory -> registers ----------------------------------------------
// 16 consecutive fp32 columns of this thread's lane (32x32b shape, x16).
__device__ __forceinline__ void ld_32x32b_x16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
// 32 consecutive fp32 columns of this thread's lane (32x32b shape, x32).
__device__ __forceinline__ void ld_32x32b_x32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}
// registers -> 16 consecutive 32-bit columns of this thread's lane (32x32b, x16)
__device__ __forceinline__ void st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};\n" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}

// Makes this thread's generic-proxy shared-memory writes visible to the
// tensor core (async proxy) reads that follow a synchronization.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

// ---- canonical K-major layouts (byte offset of 16-byte unit u of row r) ------
// 128-byte swizzle: 8-row atoms of 128-byte rows (1024 B), units XOR row % 8.
__host__ __device__ __forceinline__ uint32_t sw128_off(int r, int u) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((u ^ (r & 7)) << 4));
}
// 64-byte swizzle: 8-row atoms of 64-byte rows (512 B), units XOR (row / 2) % 4;
// `group_stride` is the distance between consecutive 8-row atoms.
__host__ __device__ __forceinline__ uint32_t sw64_off(int r, int u, int group_stride) {
  return (uint32_t)((r >> 3) * group_stride + (r & 7) * 64 + ((u ^ ((r >> 1) & 3)) << 4));
}

}  // namespace tc
}  // namespace musemoe
