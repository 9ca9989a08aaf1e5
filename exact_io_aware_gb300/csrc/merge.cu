// Merge of partial attention results computed over disjoint key sets.
//
// "Exact tiled attention and memory-aware differentiation" merges the stable summaries
// (m, l, z) of two disjoint key sets S, T of one query row as
//     m' = max(m_S, m_T),  l' = e^{m_S - m'} l_S + e^{m_T - m'} l_T,
//     z' = e^{m_S - m'} z_S + e^{m_T - m'} z_T,
// with the empty set's state as the identity, and the same page reads key-sharded attention
// as this merge applied to the shards' summaries.  A partial result in normalised form,
// O_g = z_g / l_g and LSE_g = m_g + ln l_g, is the summary (LSE_g, 1, O_g) of the same key set
// (a summary is unchanged by moving a common factor between m and (l, z)), so folding the
// merge over the parts gives
//     LSE = M + ln sum_g e^{LSE_g - M},   O = sum_g e^{LSE_g - LSE} O_g,   M = max_g LSE_g.
// A part with LSE_g = -inf is the empty state and adds nothing; a row whose parts are all
// empty has no defined output and is written as O = 0, LSE = -inf with the empty-row flag.
//
// Memory-bound: one warp per row reads num_parts float32 rows of d values and writes one row
// in the output type; lanes cover the row with 16-byte loads.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <string>

#include "kernels.h"
#include "status.cuh"

namespace ea {
namespace merge {

constexpr int kWarps = 8;

template <typename T>
__device__ __forceinline__ void store4(T* dst, float4 v);

template <>
__device__ __forceinline__ void store4<float>(float* dst, float4 v) {
  *reinterpret_cast<float4*>(dst) = v;
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* dst, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
  uint2 w;
  w.x = *reinterpret_cast<uint32_t*>(&a);
  w.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(dst) = w;
}
template <>
__device__ __forceinline__ void store4<__half>(__half* dst, float4 v) {
  __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
  uint2 w;
  w.x = *reinterpret_cast<uint32_t*>(&a);
  w.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(dst) = w;
}

template <typename T>
__global__ void __launch_bounds__(kWarps * 32)
    merge_kernel(int parts, int64_t rows, int d, const float* __restrict__ o_part,
                 const float* __restrict__ lse_part, T* __restrict__ o, float* __restrict__ lse,
                 uint32_t* status) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  float mx = -INFINITY;
  for (int g = 0; g < parts; ++g) mx = fmaxf(mx, __ldg(lse_part + g * rows + row));
  if (mx == -INFINITY) {  // every part empty
    for (int c = 4 * lane; c < d; c += 128) store4<T>(o + row * d + c, make_float4(0.f, 0.f, 0.f, 0.f));
    if (lane == 0) {
      lse[row] = -INFINITY;
      raise_empty_row(status);
    }
    return;
  }
  float sum = 0.0f;
  for (int g = 0; g < parts; ++g) sum += expf(__ldg(lse_part + g * rows + row) - mx);
  const float inv = 1.0f / sum;
  for (int c = 4 * lane; c < d; c += 128) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int g = 0; g < parts; ++g) {
      const float w = expf(__ldg(lse_part + g * rows + row) - mx) * inv;
      if (w == 0.0f) continue;  // an empty part (its O_g is zero anyway)
      const float4 x = __ldg(reinterpret_cast<const float4*>(o_part + (g * rows + row) * d + c));
      acc.x = fmaf(w, x.x, acc.x);
      acc.y = fmaf(w, x.y, acc.y);
      acc.z = fmaf(w, x.z, acc.z);
      acc.w = fmaf(w, x.w, acc.w);
    }
    store4<T>(o + row * d + c, acc);
  }
  if (lane == 0) lse[row] = mx + logf(sum);
}

}  // namespace merge

int launch_merge(int dtype_out, int num_parts, int64_t rows, int d, const float* o_part,
                 const float* lse_part, void* o, float* lse, uint32_t* status, cudaStream_t s,
                 std::string& err) {
  const int64_t blocks = (rows + merge::kWarps - 1) / merge::kWarps;
  if (blocks > 0x7FFFFFFF) {
    err = "too many rows for the merge grid";
    return -2;
  }
  dim3 grid(static_cast<unsigned>(blocks));
  dim3 block(merge::kWarps * 32);
  switch (dtype_out) {
    case 0:
      merge::merge_kernel<float><<<grid, block, 0, s>>>(num_parts, rows, d, o_part, lse_part,
                                                        static_cast<float*>(o), lse, status);
      break;
    case 1:
      merge::merge_kernel<__half><<<grid, block, 0, s>>>(num_parts, rows, d, o_part, lse_part,
                                                         static_cast<__half*>(o), lse, status);
      break;
    case 2:
      merge::merge_kernel<__nv_bfloat16><<<grid, block, 0, s>>>(
          num_parts, rows, d, o_part, lse_part, static_cast<__nv_bfloat16*>(o), lse, status);
      break;
    default:
      err = "unknown output dtype";
      return -1;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    err = std::string("merge launch: ") + cudaGetErrorString(e);
    return -5;
  }
  return 0;
}

}  // namespace ea
