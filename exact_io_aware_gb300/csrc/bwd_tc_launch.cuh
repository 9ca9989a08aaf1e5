// Host launchers of the tcgen05 backward kernels (dK/dV by key tiles, dQ by query tiles),
// instantiated per head dimension.
#pragma once
#include "bwd_tc.cuh"
#include "dq_tc.cuh"
#include "tmap.h"

namespace ea {
namespace bwd {

constexpr int kMaxDynSmem = 227 * 1024 - 1024;

template <bool kBf16, int D, int DV, bool kDrop, bool kCap = false>
int run(const AttnArgs& a, float* table, cudaStream_t s, std::string& err) {
  using Cfg = Config<D, DV>;
  using QCfg = dq::Config<D, DV>;
  const bool bitmap = a.mask_kind == kMaskBitmap;
  const size_t smem = Cfg::smem_bytes(a.n, bitmap);
  const size_t qsmem = QCfg::smem_bytes(a.n, bitmap);
  if (smem > static_cast<size_t>(kMaxDynSmem) || qsmem > static_cast<size_t>(kMaxDynSmem)) {
    err = "n too large for the backward step tables under a bitmap mask at this head dimension";
    return -2;
  }
  const uint64_t heads = static_cast<uint64_t>(a.B) * a.H;
  constexpr uint32_t bc = RowLayout<D>::kBoxCols;
  constexpr uint32_t bcv = RowLayout<DV>::kBoxCols;
  CUtensorMap tq, tk, tv, tg, tdk, tdv, tdq, to;
  if (!encode_tile_map(&tq, a.q, kBf16, heads, a.n, D, 128, bc) ||
      !encode_tile_map(&tg, a.d_o, kBf16, heads, a.n, DV, 128, bcv) ||
      !encode_tile_map(&tk, a.k, kBf16, heads, a.n, D, 128, bc) ||
      !encode_tile_map(&tv, a.v, kBf16, heads, a.n, DV, 128, bcv) ||
      !encode_tile_map(&tdk, a.dk, kBf16, heads, a.n, D, 128, bc) ||
      !encode_tile_map(&tdv, a.dv, kBf16, heads, a.n, DV, 128, bcv) ||
      !encode_tile_map(&tdq, a.dq, kBf16, heads, a.n, D, 128, bc) ||
      !encode_tile_map(&to, a.o, kBf16, heads, a.n, DV, 128, bcv)) {
    err = "cuTensorMapEncodeTiled rejected a backward tensor map";
    return -5;
  }
  const int n_pad = bwd_pad_rows(a.n);
  float* L2 = table;
  BwdParams p{a.n,  a.c, a.mask_kind, a.mask_bits, a.mask_row_words, a.mask_head_stride_words,
              L2,   L2 + static_cast<size_t>(heads) * n_pad, n_pad, a.lse, a.status};
  p.drop = a.drop;
  p.next_cta = a.sms;
  // the dK/dV kernel issues S_{i+1} before dK_i releases stage i, and the dQ kernel S_{i+1}
  // before dQ_i releases K_i: those rings need two stages; the dQ kernel's V ring stages the
  // tile's dO and O in its last two stages at the start
  p.ring_q = Ring::make(ring_depth(a.ring_stages, 2, Cfg::NS));
  p.ring_k = Ring::make(ring_depth(a.ring_stages, 2, QCfg::NSK));
  p.ring_v = Ring::make(ring_depth(a.ring_stages, 2, QCfg::NSV));
  const dim3 grid((a.n + 127) / 128, static_cast<unsigned>(heads));
  // the dQ kernel writes the row table the dK/dV kernel reads
  auto qkern = dq::dq_tc_kernel<kBf16, D, DV, kDrop, kCap>;
  cudaError_t e = cudaFuncSetAttribute(qkern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(qsmem));
  if (e == cudaSuccess) {
    qkern<<<grid, dq::kThreads, qsmem, s>>>(tk, tv, tdq, tq, tg, to, p);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) {
    err = std::string("dQ launch: ") + cudaGetErrorString(e);
    return -5;
  }
  auto kern = bwd_tc_kernel<kBf16, D, DV, kDrop, kCap>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem));
  if (e == cudaSuccess) {
    kern<<<grid, kThreads, smem, s>>>(tq, tk, tv, tg, tdk, tdv, p);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) {
    err = std::string("dK/dV launch: ") + cudaGetErrorString(e);
    return -5;
  }
  return 0;
}

// Instantiations with and without dropout for one (key width, value width) pair.
template <int D, int DV = D>
int run_d(bool bf16, const AttnArgs& a, float* table, cudaStream_t s, std::string& err) {
  if (a.ring_stages != 0) {
    // ring depths from the launch: one instantiation, as a testing aid
    if constexpr (D == 128 && DV == 128) {
      if (bf16 && !a.dropout) return run<true, 128, 128, false, true>(a, table, s, err);
    }
    err = "a ring-depth cap applies to bf16, d = v = 128, without dropout";
    return -2;
  }
  if (a.dropout)
    return bf16 ? run<true, D, DV, true>(a, table, s, err) : run<false, D, DV, true>(a, table, s, err);
  return bf16 ? run<true, D, DV, false>(a, table, s, err) : run<false, D, DV, false>(a, table, s, err);
}

}  // namespace bwd
}  // namespace ea
