// Weight re-layout of the expert tensors (plain rows -> kernel layout) and
// the UE8M0 scale check that precedes it.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace musemoe {

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

// One output byte per thread step: output offset o of the kernel layout
// [tiles][slice][8 groups][chunks of the slice][8 rows][cb] takes source
// byte (row, byte) of the plain row-major [rows, row_bytes] tensor. Code
// chunks also reorder their bytes so that a thread's 16 bytes are its mma
// fragments: FP4 (permute 1), output 16q + 2j + b <- chunk byte 8j + 2q + b;
// BF16 (permute 2, 32 values per chunk), a 4 x 4 transpose of 4-byte words,
// output 16q + 4j + b <- chunk byte 16j + 4q + b. FP8 (permute 3): the
// 64-byte swizzle of the tensor cores' shared-memory operands within each
// [8 rows][64 B] block, 16-byte unit u of row r stored at unit
// u ^ ((r >> 1) & 3), so that a bulk copy of a block is a canonical
// 64-byte-swizzled K-major operand.
__global__ void k_pack_tiles(const uint8_t* src, uint8_t* dst, size_t bytes, int row_bytes, int cb,
                             int permute) {
  const int NC = row_bytes / cb;
  const size_t tile_bytes = (size_t)64 * row_bytes;
  const size_t full = (size_t)64 * kSliceChunks * cb;  // a full slice of a tile
  for (size_t o = (size_t)blockIdx.x * blockDim.x + threadIdx.x; o < bytes;
       o += (size_t)gridDim.x * blockDim.x) {
    const size_t t = o / tile_bytes, ot = o % tile_bytes;
    const int s = (int)(ot / full);
    const int rem = (int)(ot - (size_t)s * full);
    const int ncs = min(kSliceChunks, NC - kSliceChunks * s);
    const int gi = rem / (ncs * 8 * cb);
    const int r2 = rem % (ncs * 8 * cb);
    const int c = r2 / (8 * cb), r = (r2 / cb) % 8;
    int b = r2 % cb;
    if (permute == 1) {
      const int qq = b >> 4, j = (b >> 1) & 7, bb = b & 1;
      b = 8 * j + 2 * qq + bb;
    } else if (permute == 2) {
      const int qq = b >> 4, j = (b >> 2) & 3, bb = b & 3;
      b = 16 * j + 4 * qq + bb;
    } else if (permute == 3) {
      b = (((b >> 4) ^ ((r >> 1) & 3)) << 4) | (b & 15);
    }
    dst[o] = src[t * tile_bytes + (size_t)(gi * 8 + r) * row_bytes +
                 (size_t)(kSliceChunks * s + c) * cb + b];
  }
}

cudaError_t launch_pack_tiles(const uint8_t* src, uint8_t* dst, size_t rows, int row_bytes, int cb,
                              int permute, uint8_t* tmp, size_t tmp_bytes, cudaStream_t s) {
  const size_t tile_bytes = (size_t)64 * row_bytes;
  const size_t tiles = rows / 64;
  const bool in_place = (src == dst);
  const size_t batch = in_place ? std::max<size_t>(1, tmp_bytes / tile_bytes) : tiles;
  if (in_place && tmp_bytes < tile_bytes) return cudaErrorInvalidValue;
  for (size_t t0 = 0; t0 < tiles; t0 += batch) {
    const size_t n = std::min(batch, tiles - t0);
    const size_t off = t0 * tile_bytes, bytes = n * tile_bytes;
    const uint8_t* from = src + off;
    if (in_place) {
      cudaError_t e = cudaMemcpyAsync(tmp, src + off, bytes, cudaMemcpyDeviceToDevice, s);
      if (e != cudaSuccess) return e;
      from = tmp;
    }
    const unsigned grid = (unsigned)std::min<size_t>((bytes + 255) / 256, 16384);
    k_pack_tiles<<<grid, 256, 0, s>>>(from, dst + off, bytes, row_bytes, cb, permute);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// ---- W4A4: block scales -> the tensor cores' scale atoms --------------------
// One output byte per thread step of one expert: output offset o of
// [tiles][slice][atoms of the slice][512] is the scale of A-tile row m =
// (b / 16) % 32 + 32 * ((b % 16) / 4) and block j = b % 4 of the atom (b = o %
// 512); the atom's four blocks are blocks 4 * (atom index along K) .. + 3 of
// the row.
__global__ void k_pack_sf_atoms(const uint8_t* src, uint8_t* dst, int N, int I, int nblk, int role,
                                int apc, size_t bytes) {
  const int NC = nblk * (apc == 1 ? 32 : 16) / 128;  // 128-element chunks of a row
  const size_t tile_bytes = (size_t)NC * apc * 512;
  const size_t slice_bytes = (size_t)kSliceChunks * apc * 512;
  for (size_t o = (size_t)blockIdx.x * blockDim.x + threadIdx.x; o < bytes;
       o += (size_t)gridDim.x * blockDim.x) {
    const int t = (int)(o / tile_bytes);
    const size_t ot = o % tile_bytes;
    const int sl = (int)(ot / slice_bytes);
    const int a = (int)((ot % slice_bytes) / 512), b = (int)(ot % 512);
    const int m = b / 16 + 32 * ((b % 16) / 4), j = b % 4;
    int row;
    if (role == 0) {
      const int ga = m >> 3;  // 8-row group of the tile: even gate, odd up
      row = ((ga & 1) ? I : 0) + t * 64 + (ga >> 1) * 8 + (m & 7);
    } else {
      row = t * 128 + m;
    }
    const int blk = 4 * (sl * kSliceChunks * apc + a) + j;
    dst[o] = src[(size_t)row * nblk + blk];
  }
}

cudaError_t launch_pack_sf_atoms(const uint8_t* src, uint8_t* dst, int E, int N, int I, int K,
                                 int role, int nv, uint8_t* tmp, size_t tmp_bytes, cudaStream_t s) {
  const int nblk = K / (nv ? 16 : 32), apc = nv ? 2 : 1;
  const size_t per = (size_t)N * nblk;  // one expert's scale bytes
  if (K % 128 || (role == 0 ? (N != 2 * I || I % 64) : N % 128)) return cudaErrorInvalidValue;
  const bool in_place = (src == dst);
  if (in_place && (!tmp || tmp_bytes < per)) return cudaErrorInvalidValue;
  const unsigned grid = (unsigned)std::min<size_t>((per + 255) / 256, 4096);
  for (int e = 0; e < E; ++e) {
    const uint8_t* from = src + (size_t)e * per;
    if (in_place) {
      cudaError_t err = cudaMemcpyAsync(tmp, from, per, cudaMemcpyDeviceToDevice, s);
      if (err != cudaSuccess) return err;
      from = tmp;
    }
    k_pack_sf_atoms<<<grid, 256, 0, s>>>(from, dst + (size_t)e * per, N, I, nblk, role, apc, per);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

}  // namespace musemoe
