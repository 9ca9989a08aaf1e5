// Dropout mask of the attention probabilities, replayed identically by every pass.
//
// The pages' base procedure has no dropout and require of a dropout extension that its
// reverse pass reuse the realised mask of the forward ("Exact tiled attention and
// memory-aware differentiation").  The mask here is a pure function of (seed, head, query
// row, key), so each kernel regenerates it where it needs it and no mask is stored:
//   words = Philox4x32-10(counter = (i, j / 4, bh, 0), key = (seed_lo, seed_hi))
//   pair (i, j) kept  iff  words[j % 4] >= threshold,  threshold = floor(p 2^32 + 1/2)
// Philox4x32 is the counter-based generator of Salmon, Moraes, Dror and Shaw ("Parallel
// random numbers: as easy as 1, 2, 3", SC 2011): ten rounds of two 32x32->64-bit products
// mixed with the key, the key advanced by fixed odd constants between rounds.
#pragma once
#include <cstdint>

namespace ea {

struct DropoutArgs {
  uint32_t thr;      // keep a pair iff its word >= thr
  float scale;       // 1 / (1 - p), applied to every kept probability
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

// Keep bits of keys 4g .. 4g+3 of query row i in head bh (bit t <-> key 4g + t).
__device__ __forceinline__ uint32_t keep4(const DropoutArgs& dr, uint32_t i, uint32_t g,
                                          uint32_t bh) {
  const uint4 w = philox4x32_10(make_uint4(i, g, bh, 0u), dr.seed_lo, dr.seed_hi);
  return (w.x >= dr.thr ? 1u : 0u) | (w.y >= dr.thr ? 2u : 0u) | (w.z >= dr.thr ? 4u : 0u) |
         (w.w >= dr.thr ? 8u : 0u);
}

// Keep bit of the single pair (i, j).
__device__ __forceinline__ bool keep1(const DropoutArgs& dr, uint32_t i, uint32_t j, uint32_t bh) {
  return (keep4(dr, i, j >> 2, bh) >> (j & 3u)) & 1u;
}

}  // namespace ea
