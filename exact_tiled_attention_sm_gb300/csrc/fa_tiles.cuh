// fa_tiles.cuh -- 128-row bf16 tiles in shared memory and the tcgen05 MMA
// sequences over them.
//
// Shared-memory tile layout (what TMA writes with the 128-byte swizzle and a
// 64-column x 128-row box): a [128 rows][D] bf16 tile is D/64 column chunks
// of 16 KiB; in a chunk, row r occupies bytes [128r, 128r + 128) with its
// 16-byte pieces XOR-permuted by (r mod 8).  Every chunk starts on a
// 1024-byte boundary.
//
// Read as an MMA operand, such a tile is
//   K-major  when the reduction runs along its columns (Q or K in S = QK^T),
//   MN-major when the reduction runs along its rows    (V in O += PV).
#pragma once
#include "ptx.cuh"

namespace fa {

constexpr int kChunkBytes = 128 * 128;  // one 64-column chunk of 128 rows

// Shared-memory descriptors of a tile (see sdesc_sw128) read K-major and
// MN-major.  The start-address field is the descriptor's low bits (address
// >> 4), so moving a descriptor by `bytes` within shared memory is adding
// bytes >> 4: the MMA sequences below build one descriptor per tile and step
// it with adds, which keeps the single issuing thread's cost per MMA small.
__device__ __forceinline__ uint64_t kdesc(uint32_t saddr) {
  return sdesc_sw128(saddr, 16, 1024);
}
__device__ __forceinline__ uint64_t mdesc(uint32_t saddr) {
  return sdesc_sw128(saddr, kChunkBytes, 1024);
}
// K-major step kk (16 elements): 32 bytes inside a 128-byte row, a new
// 64-column chunk every 4 steps.
__host__ __device__ constexpr uint32_t kstep(int kk) {
  return (uint32_t)(((kk >> 2) * kChunkBytes + (kk & 3) * 32) >> 4);
}
// MN-major step kk (16 rows of 128 bytes).
__host__ __device__ constexpr uint32_t mstep(int kk) {
  return (uint32_t)((kk * 16 * 128) >> 4);
}

// D(128 x 128) (+)= A B^T with A, B both [128][Dk] K-major tiles (Dk/16 MMAs
// of K = 16).
template <int Dk>
__device__ __forceinline__ void mma_rows_x_rows(uint32_t d_tmem, uint32_t sa,
                                                uint32_t sb, uint32_t idesc) {
  const uint64_t da = kdesc(sa), db = kdesc(sb);
#pragma unroll
  for (int kk = 0; kk < Dk / 16; ++kk)
    umma_ss(d_tmem, da + kstep(kk), db + kstep(kk), idesc, kk > 0 ? 1u : 0u);
}

// D(128 x Dn) (+)= A B with A (128 x 128) in TMEM (bf16 pairs, lanes = rows)
// and B a [128][Dn] tile read MN-major (8 MMAs of K = 16 rows; the Dn/64
// chunks are kChunkBytes apart).
__device__ __forceinline__ void mma_tmem_x_rows(uint32_t d_tmem, uint32_t a_tmem,
                                                uint32_t sb, uint32_t idesc,
                                                bool accumulate) {
  const uint64_t db = mdesc(sb);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    umma_ts(d_tmem, a_tmem + kk * 8, db + mstep(kk), idesc,
            (accumulate || kk > 0) ? 1u : 0u);
}

// As mma_tmem_x_rows, with the A operand's 8 column groups (16 K-rows each)
// split in two halves: groups 0-3 at a_lo + 8*kk, groups 4-7 at
// a_hi + 8*(kk-4).
__device__ __forceinline__ void mma_tmem2_x_rows(uint32_t d_tmem, uint32_t a_lo,
                                                 uint32_t a_hi, uint32_t sb,
                                                 uint32_t idesc, bool accumulate) {
  const uint64_t db = mdesc(sb);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    umma_ts(d_tmem, kk < 4 ? a_lo + kk * 8 : a_hi + (kk - 4) * 8,
            db + mstep(kk), idesc, (accumulate || kk > 0) ? 1u : 0u);
}

// D(128 x Dn) = A B with A^T a [128 (K)][128 (M)] tile read MN-major (its
// two 64-column chunks are the M runs) and B a [128 (K)][Dn] tile read
// MN-major.
__device__ __forceinline__ void mma_colsT_x_rows(uint32_t d_tmem, uint32_t sat,
                                                 uint32_t sb, uint32_t idesc) {
  const uint64_t da = mdesc(sat), db = mdesc(sb);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    umma_ss(d_tmem, da + mstep(kk), db + mstep(kk), idesc, kk > 0 ? 1u : 0u);
}

// 8-bit (E4M3) tiles.  A [128][128] byte tile (d = 128) is one 16 KiB chunk
// of the layout above, byte-for-byte like a 64-column bf16 chunk, and one MMA
// consumes K = 32 elements = 32 bytes: the K-major steps are kstep's, four
// per 128-byte row.
// D(128 x 128) (+)= A B^T with A, B both [128][RowBytes] K-major byte tiles.
template <int RowBytes>
__device__ __forceinline__ void mma_rows_x_rows_f8(uint32_t d_tmem, uint32_t sa,
                                                   uint32_t sb, uint32_t idesc) {
  const uint64_t da = kdesc(sa), db = kdesc(sb);
#pragma unroll
  for (int kk = 0; kk < RowBytes / 32; ++kk)
    umma_ss_f8(d_tmem, da + kstep(kk), db + kstep(kk), idesc, kk > 0 ? 1u : 0u);
}

// MN-major step kk of an 8-bit tile: 32 rows of 128 bytes.
__host__ __device__ constexpr uint32_t mstep_f8(int kk) {
  return (uint32_t)((kk * 32 * 128) >> 4);
}

// D(128 x 128) (+)= A B with A (128 x 128) in TMEM as E4M3 (four per 32-bit
// column, lanes = rows; 8 columns per MMA) and B a [128][128] byte tile read
// MN-major (4 MMAs of K = 32 rows).
__device__ __forceinline__ void mma_tmem_x_rows_f8(uint32_t d_tmem, uint32_t a_tmem,
                                                   uint32_t sb, uint32_t idesc,
                                                   bool accumulate) {
  const uint64_t db = mdesc(sb);
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)
    umma_ts_f8(d_tmem, a_tmem + kk * 8, db + mstep_f8(kk), idesc,
               (accumulate || kk > 0) ? 1u : 0u);
}

// Byte offset of the 16-byte piece `p` (0..15 across a 128-element row) of
// row r in the layout above.
__device__ __forceinline__ uint32_t swz_offset(int r, int p) {
  return (uint32_t)((p >> 3) * kChunkBytes + r * 128 + (((p & 7) ^ (r & 7)) << 4));
}

}  // namespace fa
