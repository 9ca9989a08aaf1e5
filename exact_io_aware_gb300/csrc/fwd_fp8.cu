// Host launcher of the FP8 (E4M3) forward kernel, d = 64 and 128.
#include <string>

#include "fwd_fp8.cuh"
#include "tmap.h"

namespace ea {
namespace fp8 {

template <int D, bool kBlocks, bool kCap = false>
int run(const AttnArgs& a, const void* vt8, float sq, float sk, float sv, const float* sq_blk,
        const float* sk_blk, const float* sv_blk, cudaStream_t s, std::string& err) {
  using Cfg = Config<D>;
  const size_t smem = Cfg::smem_bytes(a.n, a.mask_kind);
  if (smem > static_cast<size_t>(kMaxDynSmem)) {
    err = "n too large for the bitmap step table of the FP8 forward";
    return -2;
  }
  const uint64_t heads = static_cast<uint64_t>(a.B) * a.H;
  CUtensorMap tq, tk, tv;
  if (!encode_byte_map(&tq, a.q, heads, a.n, D, kRowsPerTile, D) ||
      !encode_byte_map(&tk, a.k, heads, a.n, D, BN, D) ||
      !encode_byte_map(&tv, vt8, heads, D, a.n, D, BN)) {
    err = "cuTensorMapEncodeTiled rejected an FP8 tensor map";
    return -5;
  }
  auto kern = fwd_fp8_kernel<D, kBlocks, kCap>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) {
    err = std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e);
    return -5;
  }
  Params p{a.n,
           a.c * sq * sk * 1.4426950408889634f,
           sv,
           a.mask_kind,
           a.mask_bits,
           a.mask_row_words,
           a.mask_head_stride_words,
           static_cast<__nv_bfloat16*>(a.o_out),
           a.lse,
           a.status,
           sq_blk,
           sk_blk,
           sv_blk};
  p.ring = Ring::make(ring_depth(a.ring_stages, 1, Config<D>::NS));
  dim3 grid((a.n + 2 * kRowsPerTile - 1) / (2 * kRowsPerTile), static_cast<unsigned>(heads));
  kern<<<grid, kThreads, smem, s>>>(tq, tk, tv, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    err = std::string("FP8 forward launch: ") + cudaGetErrorString(e);
    return -5;
  }
  return 0;
}

}  // namespace fp8

int launch_fwd_fp8(const AttnArgs& a, const void* vt8, float sq, float sk, float sv,
                   const float* sq_blk, const float* sk_blk, const float* sv_blk, cudaStream_t s,
                   std::string& err) {
  if (a.ring_stages != 0) {
    // ring depth from the launch: one instantiation, as a testing aid
    if (a.d == 128 && !sk_blk)
      return fp8::run<128, false, true>(a, vt8, sq, sk, sv, sq_blk, sk_blk, sv_blk, s, err);
    err = "a ring-depth cap applies to the FP8 forward with d = 128 and per-tensor scales";
    return -2;
  }
  switch (a.d) {
    case 64:
      return sk_blk ? fp8::run<64, true>(a, vt8, sq, sk, sv, sq_blk, sk_blk, sv_blk, s, err)
                    : fp8::run<64, false>(a, vt8, sq, sk, sv, sq_blk, sk_blk, sv_blk, s, err);
    case 128:
      return sk_blk ? fp8::run<128, true>(a, vt8, sq, sk, sv, sq_blk, sk_blk, sv_blk, s, err)
                    : fp8::run<128, false>(a, vt8, sq, sk, sv, sq_blk, sk_blk, sv_blk, s, err);
    default: err = "the FP8 forward supports d = 64 and 128"; return -2;
  }
}

}  // namespace ea
