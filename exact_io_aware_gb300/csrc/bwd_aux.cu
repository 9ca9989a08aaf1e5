// Backward preprocessing and postprocessing.
//
// Preprocessing computes the per-row term of the reverse procedure of "Exact tiled attention
// and memory-aware differentiation", delta_i = sum_a G_ia Y_ia, from the stored output O and
// the upstream dO (the "D vector" that "Bellek Duvarının Fiziği" notes comes for free from
// O).  For the tensor-core backward it writes a padded per-row table (LSE in log2 units and D)
// that the kernels copy into shared memory in 512-byte bulk transfers.  Postprocessing scales a
// float32 dQ accumulator by c and rounds it to the 16-bit output type.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.h"

namespace ea {
namespace aux {

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__half>(__half x) { return __half2float(x); }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

// One warp per row; rows = B*H*n.  Lanes stride over the d columns.
template <typename T>
__global__ void __launch_bounds__(256) pre_kernel(const T* __restrict__ O, const T* __restrict__ G,
                                                  float* __restrict__ Dv, int64_t rows, int d,
                                                  float4* __restrict__ zero, int64_t zero_vec4) {
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int lane = threadIdx.x & 31;
  for (int64_t r = warp0; r < rows; r += nwarps) {
    float acc = 0.0f;
    const T* o = O + r * d;
    const T* g = G + r * d;
    for (int a = lane; a < d; a += 32) acc = fmaf(to_f(o[a]), to_f(g[a]), acc);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
    if (lane == 0) Dv[r] = acc;
  }
  if (zero) {
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t nth = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t e = tid; e < zero_vec4; e += nth) zero[e] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// Row table of the tensor-core backward, padded to n_pad rows per head: L2 = LSE * log2(e)
// (+inf for rows with no allowed key and rows past n, so that their probabilities are 0) and
// D = rowsum(dO * O) (0 past n).  d/8 lanes cover a row with 16-byte loads (8 elements), a warp
// takes 32/(d/8) rows at once, and each thread keeps two such row groups in flight.
template <typename T>
__global__ void __launch_bounds__(256) pre_rows_kernel(const T* __restrict__ O,
                                                       const T* __restrict__ G,
                                                       const float* __restrict__ lse,
                                                       float* __restrict__ L2,
                                                       float* __restrict__ Dv, int64_t heads, int n,
                                                       int n_pad, int d) {
  constexpr int kGroups = 2;
  const int lpr = d / 8;
  const int rpw = 32 / lpr;
  const int lane = threadIdx.x & 31;
  const int sub = lane / lpr, part = lane % lpr;
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int64_t total = heads * n_pad;
  for (int64_t base = warp0 * rpw; base < total; base += nwarps * rpw * kGroups) {
    int64_t rr[kGroups], bh[kGroups], r[kGroups];
    bool live[kGroups];
    uint4 ov[kGroups], gv[kGroups];
#pragma unroll
    for (int g = 0; g < kGroups; ++g) {
      rr[g] = base + static_cast<int64_t>(g) * nwarps * rpw + sub;
      bh[g] = 0;
      r[g] = 0;
      live[g] = false;
      if (rr[g] < total) {
        bh[g] = rr[g] / n_pad;
        r[g] = rr[g] - bh[g] * n_pad;
        live[g] = r[g] < n;
      }
      ov[g] = gv[g] = make_uint4(0u, 0u, 0u, 0u);
      if (live[g]) {
        const int64_t off = (bh[g] * n + r[g]) * d + 8 * part;
        ov[g] = *reinterpret_cast<const uint4*>(O + off);
        gv[g] = *reinterpret_cast<const uint4*>(G + off);
      }
    }
#pragma unroll
    for (int g = 0; g < kGroups; ++g) {
      const T* o8 = reinterpret_cast<const T*>(&ov[g]);
      const T* g8 = reinterpret_cast<const T*>(&gv[g]);
      float acc = 0.0f;
#pragma unroll
      for (int e = 0; e < 8; ++e) acc = fmaf(to_f(o8[e]), to_f(g8[e]), acc);
      for (int off = lpr / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
      if (rr[g] < total && part == 0) {
        float l2 = INFINITY;
        if (live[g]) {
          const float lv = lse[bh[g] * n + r[g]];
          if (lv != -INFINITY) l2 = lv * 1.4426950408889634f;
        }
        L2[rr[g]] = l2;
        Dv[rr[g]] = live[g] ? acc : 0.0f;
      }
    }
  }
}

template <bool kBf16>
__global__ void __launch_bounds__(256) post_kernel(const float4* __restrict__ acc, uint2* __restrict__ out,
                                                   int64_t nvec4, float c) {
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nth = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t e = tid; e < nvec4; e += nth) {
    const float4 v = acc[e];
    uint2 r;
    if constexpr (kBf16) {
      __nv_bfloat162 a = __floats2bfloat162_rn(c * v.x, c * v.y);
      __nv_bfloat162 b = __floats2bfloat162_rn(c * v.z, c * v.w);
      r.x = *reinterpret_cast<uint32_t*>(&a);
      r.y = *reinterpret_cast<uint32_t*>(&b);
    } else {
      __half2 a = __floats2half2_rn(c * v.x, c * v.y);
      __half2 b = __floats2half2_rn(c * v.z, c * v.w);
      r.x = *reinterpret_cast<uint32_t*>(&a);
      r.y = *reinterpret_cast<uint32_t*>(&b);
    }
    out[e] = r;
  }
}

inline int grid_for(int64_t work, int per_block) {
  int64_t g = (work + per_block - 1) / per_block;
  if (g > 152 * 16) g = 152 * 16;
  return g < 1 ? 1 : static_cast<int>(g);
}

}  // namespace aux

int launch_bwd_pre(int dtype, const AttnArgs& a, float* D, float* zero, size_t zero_elems,
                   cudaStream_t s, std::string& err) {
  const int64_t rows = static_cast<int64_t>(a.B) * a.H * a.n;
  const int grid = aux::grid_for(rows, 8);
  float4* z = reinterpret_cast<float4*>(zero);
  const int64_t zv = static_cast<int64_t>(zero_elems / 4);
  switch (dtype) {
    case 0:
      aux::pre_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float*>(a.o),
                                                  static_cast<const float*>(a.d_o), D, rows, a.d, z, zv);
      break;
    case 1:
      aux::pre_kernel<__half><<<grid, 256, 0, s>>>(static_cast<const __half*>(a.o),
                                                   static_cast<const __half*>(a.d_o), D, rows, a.d, z, zv);
      break;
    default:
      aux::pre_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(
          static_cast<const __nv_bfloat16*>(a.o), static_cast<const __nv_bfloat16*>(a.d_o), D, rows,
          a.d, z, zv);
      break;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    err = std::string("backward preprocessing launch: ") + cudaGetErrorString(e);
    return -5;
  }
  return 0;
}

int launch_bwd_pre_rows(bool bf16, const AttnArgs& a, float* L2, float* Dv, int n_pad,
                        cudaStream_t s, std::string& err) {
  const int64_t heads = static_cast<int64_t>(a.B) * a.H;
  const int rpw = 32 / (a.d / 8);
  const int grid = aux::grid_for(heads * n_pad, 8 * rpw * 2);
  if (bf16)
    aux::pre_rows_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(
        static_cast<const __nv_bfloat16*>(a.o), static_cast<const __nv_bfloat16*>(a.d_o), a.lse, L2,
        Dv, heads, a.n, n_pad, a.d);
  else
    aux::pre_rows_kernel<__half><<<grid, 256, 0, s>>>(static_cast<const __half*>(a.o),
                                                      static_cast<const __half*>(a.d_o), a.lse, L2,
                                                      Dv, heads, a.n, n_pad, a.d);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    err = std::string("backward preprocessing launch: ") + cudaGetErrorString(e);
    return -5;
  }
  return 0;
}

int launch_bwd_post(bool bf16, const AttnArgs& a, const float* acc, cudaStream_t s,
                    std::string& err) {
  const int64_t nvec = static_cast<int64_t>(a.B) * a.H * a.n * a.d / 4;
  const int grid = aux::grid_for(nvec, 256);
  if (bf16)
    aux::post_kernel<true><<<grid, 256, 0, s>>>(reinterpret_cast<const float4*>(acc),
                                                static_cast<uint2*>(a.dq), nvec, a.c);
  else
    aux::post_kernel<false><<<grid, 256, 0, s>>>(reinterpret_cast<const float4*>(acc),
                                                 static_cast<uint2*>(a.dq), nvec, a.c);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    err = std::string("backward postprocessing launch: ") + cudaGetErrorString(e);
    return -5;
  }
  return 0;
}

}  // namespace ea
