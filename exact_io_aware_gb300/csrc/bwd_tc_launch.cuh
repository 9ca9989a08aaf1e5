// Host launcher for the tcgen05 backward kernel (instantiated per head dimension).
#pragma once
#include "bwd_tc.cuh"
#include "tmap.h"

namespace ea {
namespace bwd {

constexpr int kMaxDynSmem = 227 * 1024 - 1024;

template <bool kBf16, int D>
int run(const AttnArgs& a, float* Dv, float* acc, cudaStream_t s, std::string& err) {
  using Cfg = Config<D>;
  const size_t smem = Cfg::smem_bytes(a.n, a.mask_kind == kMaskBitmap);
  if (smem > static_cast<size_t>(kMaxDynSmem)) {
    err = "n too large for the backward step table";
    return -2;
  }
  const uint64_t heads = static_cast<uint64_t>(a.B) * a.H;
  constexpr uint32_t bc = RowLayout<D>::kBoxCols;
  CUtensorMap tq, tk, tv, tg, tdk, tdv, tdq;
  if (!encode_tile_map(&tq, a.q, kBf16, heads, a.n, D, Cfg::BQ, bc) ||
      !encode_tile_map(&tg, a.d_o, kBf16, heads, a.n, D, Cfg::BQ, bc) ||
      !encode_tile_map(&tk, a.k, kBf16, heads, a.n, D, kKeys, bc) ||
      !encode_tile_map(&tv, a.v, kBf16, heads, a.n, D, kKeys, bc) ||
      !encode_tile_map(&tdk, a.dk, kBf16, heads, a.n, D, kKeys, bc) ||
      !encode_tile_map(&tdv, a.dv, kBf16, heads, a.n, D, kKeys, bc) ||
      !encode_f32_map(&tdq, acc, heads, a.n, D, Cfg::BQ, Cfg::TDQ::kBoxCols)) {
    err = "cuTensorMapEncodeTiled rejected a backward tensor map";
    return -5;
  }
  auto kern = bwd_tc_kernel<kBf16, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) {
    err = std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e);
    return -5;
  }
  BwdParams p{a.n, a.c, a.mask_kind, a.mask_bits, a.mask_row_words, a.mask_head_stride_words,
              a.lse, Dv, acc, a.status};
  dim3 grid((a.n + kKeys - 1) / kKeys, static_cast<unsigned>(heads));
  kern<<<grid, kThreads, smem, s>>>(tq, tk, tv, tg, tdk, tdv, tdq, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    err = std::string("backward launch: ") + cudaGetErrorString(e);
    return -5;
  }
  return 0;
}

}  // namespace bwd
}  // namespace ea
