// Tile geometry shared by the forward and backward kernels.
//
// Every Q/K/V/O/dO tile is 128 rows x D columns of bf16, loaded by TMA from a
// [B*H, N, D] view of the tensor.  Rows of D <= 64 elements are one swizzle
// atom wide; D = 128 rows are split into two 64-column TMA boxes placed
// 16 KB apart.  The swizzle width equals the row width (32/64/128 bytes), so
// every layout is a canonical tcgen05 operand layout in both K-major and
// MN-major use.
#pragma once
#include "ptx.cuh"

namespace fa2 {

constexpr int kTileRows = 128;

// The descriptor of an operand `off` bytes (a multiple of 16) past the one
// `d` describes: only the start-address field changes, and it stays inside
// its 14 bits for any shared-memory address, so adding to the low word is
// exact.  Written so that the descriptor of the operand's base is built once
// and each K step costs one 32-bit add.
__device__ __forceinline__ uint64_t smem_desc_step(uint64_t d, uint32_t off) {
  const uint32_t lo = static_cast<uint32_t>(d) + (off >> 4);
  return (d & 0xFFFFFFFF00000000ull) | lo;
}  // BLOCK_M = BLOCK_N = 128 query / key rows

template <int D>
struct HeadDim {
  static_assert(D == 16 || D == 32 || D == 64 || D == 128, "head dim must be 16, 32, 64 or 128");
  static constexpr int kBoxCols = D >= 64 ? 64 : D;       // TMA box inner extent, elements
  static constexpr int kNumBoxes = D / kBoxCols;          // boxes per tile
  static constexpr int kRowBytes = kBoxCols * 2;          // 128, 64 or 32 bytes
  static constexpr int kBoxBytes = kTileRows * kRowBytes;  // one [128 x kBoxCols] box
  static constexpr int kTileBytes = kTileRows * D * 2;
  static constexpr int kSBO = 8 * kRowBytes;  // byte stride between 8-row groups
  static constexpr uint32_t kSwizzle = D >= 64 ? kSwizzle128B : (D == 32 ? kSwizzle64B : kSwizzle32B);

  // Operand whose rows are the M (or N) index and whose D columns are the
  // contraction index K ("K-major"), at contraction step kk (16 columns).
  static __device__ __forceinline__ uint64_t kmajor_desc(uint32_t base, int kk) {
    const int k = kk * 16;
    return smem_desc_step(make_smem_desc(base, 16, kSBO, kSwizzle), (k / kBoxCols) * kBoxBytes + (k % kBoxCols) * 2);
  }
  // Operand whose rows are the contraction index K and whose D columns are
  // the M (or N) index ("MN-major"), at contraction step kk (16 rows).
  static __device__ __forceinline__ uint64_t mnmajor_desc(uint32_t base, int kk) {
    return smem_desc_step(make_smem_desc(base, kBoxBytes, kSBO, kSwizzle), kk * 16 * kRowBytes);
  }
};

// Byte offset of 16-byte chunk j of row `row` in a tile with ROW_BYTES-byte
// rows (32, 64 or 128) swizzled the way TMA's 32B/64B/128B swizzle lays it
// out: address bits [4,7) XOR bits [7,10) (masked to the swizzle width).
template <int ROW_BYTES>
__device__ __forceinline__ uint32_t swizzle_offset(uint32_t row, uint32_t j) {
  const uint32_t off = row * ROW_BYTES + j * 16;
  constexpr uint32_t mask = ROW_BYTES == 128 ? 7u : (ROW_BYTES == 64 ? 3u : 1u);
  return off ^ (((off >> 7) & mask) << 4);
}

// 128 x 128 bf16 tile written by threads (P, dS): same layout as HeadDim<128>.
using Square = HeadDim<128>;

// Thread `row` stores 8 consecutive bf16 values (columns 8*c16 .. 8*c16+7)
// of a 128 x 128 tile laid out as Square.
__device__ __forceinline__ void store_square_chunk(uint32_t base, uint32_t row, uint32_t c16, uint32_t w0,
                                                   uint32_t w1, uint32_t w2, uint32_t w3) {
  const uint32_t box = c16 >> 3;
  st_shared_v4(base + box * Square::kBoxBytes + sw128_offset(row, c16 & 7u), w0, w1, w2, w3);
}

}  // namespace fa2
