// Dropout mask of the attention probabilities, replayed identically by every pass.
//
// The pages' base procedure has no dropout and require of a dropout extension that its
// reverse pass reuse the realised mask of the forward ("Exact tiled attention and
// memory-aware differentiation").  The mask here is a pure function of (seed, head, query
// row, key), so each kernel regenerates it where it needs it and no mask is stored.  One
// generator call decides a 4 x 4 patch of (query, key) pairs:
//   words = Philox4x32-10(counter = (i / 4, j / 4, bh, 0), key = (seed_lo, seed_hi))
//   pair (i, j) kept  iff  byte j % 4 of words[i % 4] >= t,  t = floor(p 256 + 1/2) <= 255
// so the drop probability is p' = t / 256 and kept probabilities are scaled by 1 / (1 - p').
// Philox4x32 is the counter-based generator of Salmon, Moraes, Dror and Shaw ("Parallel
// random numbers: as easy as 1, 2, 3", SC 2011): ten rounds of two 32x32->64-bit products
// mixed with the key, the key advanced by fixed odd constants between rounds.
#pragma once
#include <cstdint>

namespace ea {

struct DropoutArgs {
  uint32_t thr4;     // the 8-bit threshold t in each byte: keep a pair iff its byte >= t
  float scale;       // 1 / (1 - t / 256), applied to every kept probability
  uint32_t seed_lo;  // generator key
  uint32_t seed_hi;
};

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
  }
  return c;
}

// 1 in bit 4 b of the result for each byte b of `ge` that is 0xFF (bytes are 0x00 or 0xFF):
// the top bits 7, 15, 23, 31 land on 28 .. 31 of the product (their partial products fall on
// distinct bits, so no carries).
__device__ __forceinline__ uint32_t byte_flags(uint32_t ge) {
  return ((ge & 0x80808080u) * 0x00204081u) >> 28;
}

// Keep bits of the 4 x 4 patch of rows 4 r .. 4 r + 3 and keys 4 g .. 4 g + 3 in head bh:
// bit 4 x + y <-> (row 4 r + x, key 4 g + y).
__device__ __forceinline__ uint32_t keep_patch(const DropoutArgs& dr, uint32_t r, uint32_t g,
                                               uint32_t bh) {
  const uint4 w = philox4x32_10(make_uint4(r, g, bh, 0u), dr.seed_lo, dr.seed_hi);
  return byte_flags(__vcmpgeu4(w.x, dr.thr4)) | (byte_flags(__vcmpgeu4(w.y, dr.thr4)) << 4) |
         (byte_flags(__vcmpgeu4(w.z, dr.thr4)) << 8) | (byte_flags(__vcmpgeu4(w.w, dr.thr4)) << 12);
}

// Keep bit of the single pair (i, j).
__device__ __forceinline__ bool keep1(const DropoutArgs& dr, uint32_t i, uint32_t j, uint32_t bh) {
  return (keep_patch(dr, i >> 2, j >> 2, bh) >> (4u * (i & 3u) + (j & 3u))) & 1u;
}

// a[i] for a lane-dependent i in 0 .. 3, without indexing a register array dynamically.
__device__ __forceinline__ uint32_t pick4(const uint32_t (&a)[4], uint32_t i) {
  const uint32_t lo = (i & 1u) ? a[1] : a[0];
  const uint32_t hi = (i & 1u) ? a[3] : a[2];
  return (i & 2u) ? hi : lo;
}

// Within each aligned group of four lanes (sub = lane % 4): part[s] = w[sub] of lane s.  Round t
// swaps with lane sub ^ t, sending the word that lane wants.
__device__ __forceinline__ void exchange4(const uint32_t (&w)[4], uint32_t (&part)[4]) {
  const uint32_t sub = threadIdx.x & 3u;
  uint32_t recv[4];  // recv[t]: from lane sub ^ t
  recv[0] = pick4(w, sub);
#pragma unroll
  for (uint32_t t = 1; t < 4; ++t) recv[t] = __shfl_xor_sync(0xFFFFFFFFu, pick4(w, sub ^ t), t);
#pragma unroll
  for (uint32_t s = 0; s < 4; ++s) part[s] = pick4(recv, s ^ sub);
}

// Keep bits of one row for two runs of 2 K keys each, drawn by the four lanes of an aligned
// group (lanes 4a .. 4a + 3, holding rows 4 r .. 4 r + 3 in lane order): lanes 0 and 1 of the
// group draw the K patches of keys 4 (g0 + s K) .. + 4 K, lanes 2 and 3 those of keys
// 4 (g1 + (s - 2) K) .., and three exchanges give every lane the K-nibble words of its own row.
// part[s] receives lane s's keys of this lane's row, bit 4 u + y <-> the u-th patch's key y.
// With g1 = g0 + 2 K the four lanes cover one run of 16 K keys.  Warp-collective: every lane
// must call it.
template <int K>
__device__ __forceinline__ void keep_rows(const DropoutArgs& dr, uint32_t r, uint32_t g0,
                                         uint32_t g1, uint32_t bh, uint32_t (&part)[4]) {
  static_assert(4 * K <= 32, "at most 32 keys per lane");
  const uint32_t sub = threadIdx.x & 3u;
  const uint32_t gb = sub < 2u ? g0 + sub * K : g1 + (sub - 2u) * K;
  uint32_t w[4] = {0u, 0u, 0u, 0u};  // w[x]: row 4 r + x over this lane's keys
#pragma unroll 1
  for (int u = 0; u < K; ++u) {
    const uint32_t m = keep_patch(dr, r, gb + u, bh);
#pragma unroll
    for (int x = 0; x < 4; ++x) w[x] |= ((m >> (4 * x)) & 0xFu) << (4 * u);
  }
  exchange4(w, part);
}

// The same for a key-major layout (one key per lane): the four lanes of an aligned group hold
// keys 4 g .. 4 g + 3; lanes 0 and 1 draw the K patches of rows 4 (r0 + s K) .. + 4 K, lanes 2
// and 3 those of rows 4 (r1 + (s - 2) K) .., and part[s] receives this lane's key over lane s's
// rows, bit 4 u + x <-> the u-th patch's row x.
template <int K>
__device__ __forceinline__ void keep_cols(const DropoutArgs& dr, uint32_t r0, uint32_t r1,
                                         uint32_t g, uint32_t bh, uint32_t (&part)[4]) {
  static_assert(4 * K <= 32, "at most 32 rows per lane");
  const uint32_t sub = threadIdx.x & 3u;
  const uint32_t rb = sub < 2u ? r0 + sub * K : r1 + (sub - 2u) * K;
  uint32_t w[4] = {0u, 0u, 0u, 0u};  // w[y]: key 4 g + y over this lane's rows
#pragma unroll 1
  for (int u = 0; u < K; ++u) {
    const uint32_t m = keep_patch(dr, rb + u, g, bh);
    // column y of the patch: bits y, 4 + y, 8 + y, 12 + y -> one nibble (multiply places them on
    // bits 12 .. 15: the partial products fall on distinct bits)
#pragma unroll
    for (int y = 0; y < 4; ++y) w[y] |= ((((m >> y) & 0x1111u) * 0x1248u) >> 12 & 0xFu) << (4 * u);
  }
  exchange4(w, part);
}

}  // namespace ea
