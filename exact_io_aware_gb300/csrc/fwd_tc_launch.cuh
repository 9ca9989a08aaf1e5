// Host launcher for the tcgen05 forward kernel, instantiated per head dimension in
// fwd_tc_d*.cu so the translation units compile in parallel.
#pragma once
#include <cstdio>

#include "fwd_tc.cuh"
#include "tmap.h"

namespace ea {
namespace fwd {

template <bool kBf16, int D, int DV, int BN, bool kDrop, bool kCap = false>
int run(const AttnArgs& a, cudaStream_t s, std::string& err) {
  using Cfg = Config<D, DV, BN>;
  const int nk = a.nk > 0 ? a.nk : a.n;
  const size_t smem = Cfg::smem_bytes(nk, a.mask_kind);
  if (smem > static_cast<size_t>(kMaxDynSmem)) {
    err = "n too large for the bitmap step table of the forward at this key block (use a "
          "smaller kv_block)";
    return -2;
  }
  const uint64_t heads = static_cast<uint64_t>(a.B) * a.H;
  CUtensorMap tq, tk, tv, to;
  constexpr uint32_t bc = RowLayout<D>::kBoxCols;
  constexpr uint32_t bcv = RowLayout<DV>::kBoxCols;
  if (!encode_tile_map(&tq, a.q, kBf16, heads, a.n, D, kRowsPerTile, bc) ||
      !encode_tile_map(&tk, a.k, kBf16, heads, nk, D, BN, bc) ||
      !encode_tile_map(&tv, a.v, kBf16, heads, nk, DV, BN, bcv) ||
      !encode_tile_map(&to, a.o_out, kBf16, heads, a.n, DV, kRowsPerTile, bcv)) {
    err = "cuTensorMapEncodeTiled rejected a forward tensor map";
    return -5;
  }
  auto kern = fwd_tc_kernel<kBf16, D, DV, BN, kDrop, kCap>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) {
    err = std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e);
    return -5;
  }
  const int nsplit = a.num_splits > 1 ? a.num_splits : 1;
  FwdParams p{a.n, a.c, a.mask_kind, a.mask_bits, a.mask_row_words, a.mask_head_stride_words,
              a.lse, a.status, nsplit, nsplit > 1 ? a.o_part : nullptr,
              nsplit > 1 ? a.lse_part : nullptr, a.drop, nk, nk - a.n,
              a.n >= kRowsPerTile ? kPrefetch : 0};
  p.ring_k = Ring::make(ring_depth(a.ring_stages, 1, Cfg::NSK));
  p.ring_v = Ring::make(ring_depth(a.ring_stages, 1, Cfg::NSV));
  p.rows_cta = a.fwd_rows_cta == kRowsPerTile ? kRowsPerTile : 2 * kRowsPerTile;
  p.next_cta = a.sms;
  dim3 grid((a.n + p.rows_cta - 1) / p.rows_cta, static_cast<unsigned>(heads),
            static_cast<unsigned>(nsplit));
  kern<<<grid, kThreads, smem, s>>>(tq, tk, tv, to, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    err = std::string("forward launch: ") + cudaGetErrorString(e);
    return -5;
  }
  return 0;
}

template <int D, int DV, bool kDrop>
int launch_dd(bool bf16, const AttnArgs& a, cudaStream_t s, std::string& err) {
  const int bn = a.kv_block == 0 ? 128 : a.kv_block;
  if (a.ring_stages != 0) {
    // ring depths from the launch: one instantiation, as a testing aid
    if constexpr (D == 128 && DV == 128 && !kDrop) {
      if (bf16 && bn == 128) return run<true, 128, 128, 128, false, true>(a, s, err);
    }
    err = "a ring-depth cap applies to bf16, d = v = 128, key block 128, without dropout";
    return -2;
  }
  switch (bn) {
    case 32:
      return bf16 ? run<true, D, DV, 32, kDrop>(a, s, err) : run<false, D, DV, 32, kDrop>(a, s, err);
    case 64:
      return bf16 ? run<true, D, DV, 64, kDrop>(a, s, err) : run<false, D, DV, 64, kDrop>(a, s, err);
    case 128:
      return bf16 ? run<true, D, DV, 128, kDrop>(a, s, err) : run<false, D, DV, 128, kDrop>(a, s, err);
    default: err = "kv_block must be 0, 32, 64 or 128"; return -2;
  }
}

// Instantiations with and without dropout for one (key width, value width) pair.
template <int D, int DV = D>
int launch_d(bool bf16, const AttnArgs& a, cudaStream_t s, std::string& err) {
  return a.dropout ? launch_dd<D, DV, true>(bf16, a, s, err) : launch_dd<D, DV, false>(bf16, a, s, err);
}

}  // namespace fwd
}  // namespace ea
