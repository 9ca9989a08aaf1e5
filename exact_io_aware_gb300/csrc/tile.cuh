// Shared-memory tile layouts of 16-bit operands and their tcgen05 descriptors.
//
// A tile of R rows x C 16-bit elements is brought in by TMA as C / BoxCols boxes, each
// R rows x BoxCols elements, stored back to back.  A box row is RowBytes = 2 * BoxCols bytes
// (32, 64 or 128) and uses the TMA swizzle of the same width, so eight consecutive rows form
// one swizzle atom of 8 * RowBytes bytes.  Boxes must start on 1024-byte boundaries.
//
// The same bytes serve two operand orientations:
//   K-major  — tile rows are the M (or N) index, columns the reduction index K.
//   MN-major — tile rows are the reduction index K, columns the M (or N) index.
// One MMA consumes 16 reduction elements (kind::f16); `kk` below counts those steps.
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace ea {

template <int C>
struct RowLayout {
  static_assert(C % 16 == 0 && C >= 16 && C <= 256, "tile width must be 16..256, step 16");
  static constexpr int kBoxCols = C < 64 ? C : 64;
  static constexpr int kRowBytes = kBoxCols * 2;
  static constexpr int kBoxes = C / kBoxCols;
  static constexpr uint32_t kSwz =
      kRowBytes == 128 ? kSwz128 : (kRowBytes == 64 ? kSwz64 : kSwz32);
  static_assert(C % kBoxCols == 0, "tile width must be a whole number of boxes");
};

template <int R, int C>
struct Tile {
  using L = RowLayout<C>;
  static constexpr int kRows = R;
  static constexpr int kCols = C;
  static constexpr int kBoxBytes = R * L::kRowBytes;
  static constexpr int kBytes = kBoxBytes * L::kBoxes;
  static_assert(R % 8 == 0, "rows must be a multiple of the 8-row swizzle atom");

  // Operand whose rows are M/N and whose columns are the reduction index (K-major).
  __device__ static __forceinline__ uint64_t desc_k(uint32_t base, int kk) {
    const int byte = kk * 32;  // 16 elements of 2 bytes
    const int box = byte / L::kRowBytes;
    const int off = byte % L::kRowBytes;
    return smem_desc(base + box * kBoxBytes + off, 16, 8 * L::kRowBytes, L::kSwz);
  }

  // Operand whose rows are the reduction index and whose columns are M/N (MN-major).
  __device__ static __forceinline__ uint64_t desc_mn(uint32_t base, int kk) {
    return smem_desc(base + kk * 16 * L::kRowBytes, kBoxBytes, 8 * L::kRowBytes, L::kSwz);
  }

  // desc_k(base, kk) - desc_k(base, 0) and desc_mn(base, kk) - desc_mn(base, 0): the kk-th
  // 16-element step only moves the descriptor's start-address field (16-byte units), so a
  // descriptor built once per buffer serves every step by adding these constants.
  __host__ __device__ static constexpr uint64_t k_step(int kk) {
    return static_cast<uint64_t>(((kk * 32) / L::kRowBytes) * kBoxBytes + (kk * 32) % L::kRowBytes) >> 4;
  }
  __host__ __device__ static constexpr uint64_t mn_step(int kk) {
    return static_cast<uint64_t>(kk * 16 * L::kRowBytes) >> 4;
  }

  // Byte offset of element (r, c) inside the swizzled tile (for threads that write operands).
  // The TMA/UMMA swizzle of width RowBytes XORs address bits [4, 4+B) with bits [7, 7+B),
  // B = log2(RowBytes / 16); the tile base is 1024-byte aligned, so offsets suffice.
  __host__ __device__ static constexpr uint32_t offset(int r, int c) {
    const uint32_t a = (c / L::kBoxCols) * kBoxBytes + r * L::kRowBytes + (c % L::kBoxCols) * 2;
    return a ^ (((a >> 7) & (L::kRowBytes / 16 - 1)) << 4);
  }
};

// A float32 tile of R rows x C columns staged for TMA: boxes of R rows x min(C, 32) columns
// (rows of 64 or 128 bytes) with the matching swizzle, stored back to back.
template <int R, int C>
struct F32Tile {
  static constexpr int kBoxCols = C < 32 ? C : 32;
  static constexpr int kRowBytes = kBoxCols * 4;
  static constexpr int kBoxes = C / kBoxCols;
  static constexpr int kBoxBytes = R * kRowBytes;
  static constexpr int kBytes = kBoxBytes * kBoxes;
  static_assert(kRowBytes == 64 || kRowBytes == 128, "fp32 tile rows must be 64 or 128 bytes");
  __host__ __device__ static constexpr uint32_t offset(int r, int c) {
    const uint32_t a = (c / kBoxCols) * kBoxBytes + r * kRowBytes + (c % kBoxCols) * 4;
    return a ^ (((a >> 7) & (kRowBytes / 16 - 1)) << 4);
  }
};

}  // namespace ea
