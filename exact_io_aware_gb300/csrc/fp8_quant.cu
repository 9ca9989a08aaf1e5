// Block quantization of Q, K and V to E4M3 for the block-scaled FP8 forward, with optional
// incoherent processing of Q and K.
//
// "Bellek Duvarının Fiziği" names the FP8 forward of FlashAttention-3 with per-block scaling
// and incoherent processing (random sign multipliers) as the way its precision loss is kept
// small.  This kernel produces that forward's operands:
//   * a block is 128 consecutive rows of one head of Q, K or V (the last one ragged), with one
//     float32 scale = absmax / 448 (1 for an all-zero block); codes = E4M3(x * (448 / absmax))
//     in float32 with round-to-nearest-even and saturation;
//   * incoherent processing (when signs are given) multiplies the columns of Q and K by the
//     signs and applies the order-d Walsh–Hadamard transform along each row, Q' = (Q ∘ σ) H_d,
//     K' = (K ∘ σ) H_d.  H_d H_dᵀ = d I, so Q' K'ᵀ = d Q Kᵀ: Q's scales carry the factor 1/d;
//   * V is written transposed, vt8 [d][n] per head, the layout the forward's second product
//     reads, with the same per-block scales over 128 keys.
//
// One CTA of 256 threads per (block, head, tensor); blockIdx.z selects Q, K or V.  Rows of Q
// and K: each lane holds 8 consecutive columns of one row (one 16-byte load), D/8 lanes a row;
// the transform's first three stages run inside the lane and the rest across lanes with
// shuffles.  V: each thread holds 8 keys x 8 columns, packs four keys of a column per 32-bit
// word and writes 8-byte runs of the transposed rows, 128 contiguous bytes per column per warp.
// The block stays in registers between the absmax reduction and the conversion, so the input
// is read once.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <string>

#include "kernels.h"
#include "ptx.cuh"

namespace ea {
namespace fp8q {

constexpr int kRows = 128;
constexpr int kThreads = 256;

struct Params {
  int n;
  int nblk;
  const void* x[3];   // q, k, v [heads][n][D] 16-bit
  uint8_t* out[3];    // q8, k8 [heads][n][D]; vt8 [heads][D][n]
  float* scales[3];   // [heads][nblk]
  const int8_t* signs;  // D entries (negative flips the column), or null: no rotation
  float q_mul;        // factor on Q's scales (1/D when rotating, else 1)
};

template <bool kBf16>
__device__ __forceinline__ void load8(const void* base, int64_t elem, float (&x)[8]) {
  const uint4 u = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + elem));
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (kBf16) {
      const __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&w[i]);
      const float2 f = __bfloat1622float2(h);
      x[2 * i] = f.x;
      x[2 * i + 1] = f.y;
    } else {
      const __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
      const float2 f = __half22float2(h);
      x[2 * i] = f.x;
      x[2 * i + 1] = f.y;
    }
  }
}

// Maximum over the CTA of each thread's value (non-negative); every thread gets the result.
__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  const int warp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) red[warp] = v;
  __syncthreads();
  float m = red[0];
#pragma unroll
  for (int w = 1; w < kThreads / 32; ++w) m = fmaxf(m, red[w]);
  return m;
}

template <bool kBf16, int D>
__global__ void __launch_bounds__(kThreads, 3) quant_kernel(Params p) {
  __shared__ float red[kThreads / 32];
  const int blk = blockIdx.x;
  const int bh = blockIdx.y;
  const int which = blockIdx.z;
  const int n = p.n;
  const int row0 = blk * kRows;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const void* src = which == 0 ? p.x[0] : which == 1 ? p.x[1] : p.x[2];
  const int64_t head = static_cast<int64_t>(bh) * n;

  if (which < 2) {
    // ------------------------------------------------------------ rows of Q or K
    constexpr int L = D / 8;         // lanes per row
    constexpr int RW = 32 / L;       // rows per warp per pass
    constexpr int RP = 8 * RW;       // rows per pass of the CTA
    constexpr int IT = kRows / RP;   // passes
    const int sub = lane / L;
    const int cc = lane % L;         // this lane holds columns 8 cc .. 8 cc + 7
    const bool rot = p.signs != nullptr;
    float sg[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) sg[e] = rot && p.signs[cc * 8 + e] < 0 ? -1.0f : 1.0f;
    float x[IT][8];
    float amax = 0.0f;
#pragma unroll
    for (int it = 0; it < IT; ++it) {
      const int row = row0 + it * RP + warp * RW + sub;
      if (row < n) {
        load8<kBf16>(src, (head + row) * D + cc * 8, x[it]);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) x[it][e] = 0.0f;
      }
      if (rot) {
#pragma unroll
        for (int e = 0; e < 8; ++e) x[it][e] *= sg[e];
        // Walsh–Hadamard butterflies (a, b) -> (a + b, a - b) over column pairs h apart:
        // h = 1, 2, 4 inside the lane, h = 8 .. D/2 between lanes (lane bit h/8).
#pragma unroll
        for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            if (e & h) continue;
            const float a = x[it][e], b = x[it][e + h];
            x[it][e] = a + b;
            x[it][e + h] = a - b;
          }
        }
#pragma unroll
        for (int hl = 1; hl < L; hl <<= 1) {
          const bool upper = (cc & hl) != 0;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float o = __shfl_xor_sync(0xFFFFFFFFu, x[it][e], hl);
            x[it][e] = upper ? o - x[it][e] : x[it][e] + o;
          }
        }
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(x[it][e]));
    }
    const float A = block_max(amax, red);
    const float inv = A > 0.0f ? 448.0f / A : 1.0f;
    if (tid == 0)
      (which == 0 ? p.scales[0] : p.scales[1])[static_cast<int64_t>(bh) * p.nblk + blk] =
          (A > 0.0f ? A / 448.0f : 1.0f) * (which == 0 ? p.q_mul : 1.0f);
    uint8_t* dst = which == 0 ? p.out[0] : p.out[1];
#pragma unroll
    for (int it = 0; it < IT; ++it) {
      const int row = row0 + it * RP + warp * RW + sub;
      if (row < n) {
        uint2 w;
        w.x = pack4_e4m3(x[it][0] * inv, x[it][1] * inv, x[it][2] * inv, x[it][3] * inv);
        w.y = pack4_e4m3(x[it][4] * inv, x[it][5] * inv, x[it][6] * inv, x[it][7] * inv);
        *reinterpret_cast<uint2*>(dst + (head + row) * D + cc * 8) = w;
      }
    }
  } else {
    // ------------------------------------------------------------ V, written transposed
    // Thread (cc, kg): columns 8 cc .. 8 cc + 7, keys 8 kg .. 8 kg + 7 of the block; kg runs
    // fastest so that a warp's stores of one column cover 16 key groups = 128 bytes.
    constexpr int NCC = D / 8;
    const int kg = tid % 16;
    const int cc = tid / 16;
    const bool mine = cc < NCC;
    float x[8][8];  // [key][column]
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int key = row0 + kg * 8 + i;
      if (mine && key < n) {
        load8<kBf16>(src, (head + key) * D + cc * 8, x[i]);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) x[i][e] = 0.0f;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(x[i][e]));
    }
    const float A = block_max(amax, red);
    const float inv = A > 0.0f ? 448.0f / A : 1.0f;
    if (tid == 0)
      p.scales[2][static_cast<int64_t>(bh) * p.nblk + blk] = A > 0.0f ? A / 448.0f : 1.0f;
    const int key0 = row0 + kg * 8;
    if (mine && key0 < n) {  // n is a multiple of 8, so the run of 8 keys is whole
      uint8_t* dst = p.out[2] + static_cast<int64_t>(bh) * D * n;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        uint2 w;
        w.x = pack4_e4m3(x[0][e] * inv, x[1][e] * inv, x[2][e] * inv, x[3][e] * inv);
        w.y = pack4_e4m3(x[4][e] * inv, x[5][e] * inv, x[6][e] * inv, x[7][e] * inv);
        *reinterpret_cast<uint2*>(dst + static_cast<int64_t>(cc * 8 + e) * n + key0) = w;
      }
    }
  }
}

template <bool kBf16, int D>
int run(const Params& p, int heads, cudaStream_t s, std::string& err) {
  dim3 grid(p.nblk, heads, 3);
  quant_kernel<kBf16, D><<<grid, kThreads, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    err = std::string("FP8 quantize launch: ") + cudaGetErrorString(e);
    return -5;
  }
  return 0;
}

}  // namespace fp8q

int launch_fp8_quantize(bool bf16, int B, int H, int n, int d, const void* q, const void* k,
                        const void* v, const int8_t* signs, void* q8, void* k8, void* vt8,
                        float* sq, float* sk, float* sv, cudaStream_t s, std::string& err) {
  fp8q::Params p{};
  p.n = n;
  p.nblk = (n + fp8q::kRows - 1) / fp8q::kRows;
  p.x[0] = q;
  p.x[1] = k;
  p.x[2] = v;
  p.out[0] = static_cast<uint8_t*>(q8);
  p.out[1] = static_cast<uint8_t*>(k8);
  p.out[2] = static_cast<uint8_t*>(vt8);
  p.scales[0] = sq;
  p.scales[1] = sk;
  p.scales[2] = sv;
  p.signs = signs;
  p.q_mul = signs ? 1.0f / static_cast<float>(d) : 1.0f;
  const int heads = B * H;
  if (d == 64) return bf16 ? fp8q::run<true, 64>(p, heads, s, err) : fp8q::run<false, 64>(p, heads, s, err);
  if (d == 128) return bf16 ? fp8q::run<true, 128>(p, heads, s, err) : fp8q::run<false, 128>(p, heads, s, err);
  err = "the FP8 quantization supports d = 64 and 128";
  return -2;
}

}  // namespace ea
