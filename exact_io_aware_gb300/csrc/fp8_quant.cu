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
// Persistent CTAs of 256 threads (three per SM) walk the (block, head, tensor) items; each
// thread copies its chunks of the next item into shared memory with cp.async while it
// converts the current one.  Rows of Q and K: each lane holds 8 consecutive columns of one row
// (one 16-byte chunk), D/8 lanes a row; the transform's first three stages run inside the lane
// and the rest across lanes with shuffles.  V: each thread holds 8 keys x 8 columns, packs
// four keys of a column per 32-bit word and writes 8-byte runs of the transposed rows, 128
// contiguous bytes per column per warp.  The block stays in registers between the absmax
// reduction and the conversion, so the input is read once.
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

// Eight 16-bit values of one 16-byte chunk, as floats.
template <bool kBf16>
__device__ __forceinline__ void unpack8(const uint4 u, float (&x)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (kBf16) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
      x[2 * i] = f.x;
      x[2 * i + 1] = f.y;
    } else {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      x[2 * i] = f.x;
      x[2 * i + 1] = f.y;
    }
  }
}

// 16-byte asynchronous copy global -> shared; src_bytes = 0 fills the chunk with zeros.
__device__ __forceinline__ void cp_async16(void* sdst, const void* gsrc, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(sdst)), "l"(gsrc),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

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

constexpr int kChunks = 8;  // 16-byte chunks a thread copies per block (at most)

// One work item: 128-row block `blk` of head `bh` of tensor `which` (0 Q, 1 K, 2 V).
struct Item {
  int which, bh, blk;
};
__device__ __forceinline__ Item item_at(int it, int heads, int nblk) {
  const int per = heads * nblk;
  const int which = it / per;
  const int rem = it - which * per;
  return Item{which, rem / nblk, rem % nblk};
}

// Thread layouts.  Q, K: lane holds columns 8 cc .. of row row0 + c RP + warp RW + sub for
// chunk c.  V: thread (cc, kg) holds columns 8 cc .. of keys row0 + 8 kg + c.
template <int D>
struct Layout {
  static constexpr int L = D / 8;        // lanes per row (Q, K)
  static constexpr int RW = 32 / L;      // rows per warp per pass
  static constexpr int RP = 8 * RW;      // rows per pass of the CTA
  static constexpr int IT = kRows / RP;  // chunks per thread (Q, K)
  static constexpr int NCC = D / 8;      // column chunks of a row (V)
};

// Issues this thread's copies of item `it` into buffer `buf` (zeros past n).
template <int D>
__device__ __forceinline__ void issue(const Params& p, int it, int heads, uint4* buf) {
  using Ly = Layout<D>;
  const Item w = item_at(it, heads, p.nblk);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = p.n;
  const int row0 = w.blk * kRows;
  const int64_t head = static_cast<int64_t>(w.bh) * n;
  const uint16_t* src =
      static_cast<const uint16_t*>(w.which == 0 ? p.x[0] : w.which == 1 ? p.x[1] : p.x[2]);
  if (w.which < 2) {
    const int sub = lane / Ly::L, cc = lane % Ly::L;
#pragma unroll
    for (int c = 0; c < Ly::IT; ++c) {
      const int row = row0 + c * Ly::RP + warp * Ly::RW + sub;
      const bool in = row < n;
      cp_async16(buf + c * kThreads + tid, src + (head + (in ? row : 0)) * D + cc * 8, in ? 16u : 0u);
    }
  } else {
    const int kg = tid % 16, cc = tid / 16;
    if (cc < Ly::NCC) {
#pragma unroll
      for (int c = 0; c < kChunks; ++c) {
        const int key = row0 + kg * 8 + c;
        const bool in = key < n;
        cp_async16(buf + c * kThreads + tid, src + (head + (in ? key : 0)) * D + cc * 8, in ? 16u : 0u);
      }
    }
  }
}

// Persistent CTAs walk the items (block, head, tensor).  Each thread copies the next item's
// chunks into the other buffer with cp.async while it converts the current one, and reads back
// only the chunks it copied itself, so the buffers need no CTA-wide barrier; the absmax
// scratch alternates by item parity so consecutive reductions do not share it.
template <bool kBf16, int D>
__global__ void __launch_bounds__(kThreads, 3) quant_kernel(Params p, int heads, int items) {
  using Ly = Layout<D>;
  extern __shared__ uint4 qbuf[];  // [2][kChunks][kThreads] chunks
  __shared__ float red[2][kThreads / 32];
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int n = p.n;
  int it = blockIdx.x;
  if (it < items) issue<D>(p, it, heads, qbuf);
  cp_async_commit();
  for (int k = 0; it < items; it += gridDim.x, ++k) {
    const int nxt = it + gridDim.x;
    if (nxt < items) issue<D>(p, nxt, heads, qbuf + ((k + 1) & 1) * kChunks * kThreads);
    cp_async_commit();
    cp_async_wait1();  // this item's chunks (this thread's own copies) have landed
    const uint4* buf = qbuf + (k & 1) * kChunks * kThreads;
    const Item w = item_at(it, heads, p.nblk);
    const int row0 = w.blk * kRows;
    const int64_t head = static_cast<int64_t>(w.bh) * n;
    float* rd = red[k & 1];

    if (w.which < 2) {
      // ---------------------------------------------------------- rows of Q or K
      const int sub = lane / Ly::L;
      const int cc = lane % Ly::L;  // this lane holds columns 8 cc .. 8 cc + 7
      const bool rot = p.signs != nullptr;
      float x[Ly::IT][8];
      float amax = 0.0f;
#pragma unroll
      for (int c = 0; c < Ly::IT; ++c) {
        unpack8<kBf16>(buf[c * kThreads + tid], x[c]);
        if (rot) {
#pragma unroll
          for (int e = 0; e < 8; ++e)
            if (p.signs[cc * 8 + e] < 0) x[c][e] = -x[c][e];
          // Walsh–Hadamard butterflies (a, b) -> (a + b, a - b) over column pairs h apart:
          // h = 1, 2, 4 inside the lane, h = 8 .. D/2 between lanes (lane bit h/8).
#pragma unroll
          for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              if (e & h) continue;
              const float a = x[c][e], b = x[c][e + h];
              x[c][e] = a + b;
              x[c][e + h] = a - b;
            }
          }
#pragma unroll
          for (int hl = 1; hl < Ly::L; hl <<= 1) {
            const bool upper = (cc & hl) != 0;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float o = __shfl_xor_sync(0xFFFFFFFFu, x[c][e], hl);
              x[c][e] = upper ? o - x[c][e] : x[c][e] + o;
            }
          }
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(x[c][e]));
      }
      const float A = block_max(amax, rd);
      const float inv = A > 0.0f ? 448.0f / A : 1.0f;
      if (tid == 0)
        (w.which == 0 ? p.scales[0] : p.scales[1])[static_cast<int64_t>(w.bh) * p.nblk + w.blk] =
            (A > 0.0f ? A / 448.0f : 1.0f) * (w.which == 0 ? p.q_mul : 1.0f);
      uint8_t* dst = w.which == 0 ? p.out[0] : p.out[1];
#pragma unroll
      for (int c = 0; c < Ly::IT; ++c) {
        const int row = row0 + c * Ly::RP + warp * Ly::RW + sub;
        if (row < n) {
          uint2 o;
          o.x = pack4_e4m3(x[c][0] * inv, x[c][1] * inv, x[c][2] * inv, x[c][3] * inv);
          o.y = pack4_e4m3(x[c][4] * inv, x[c][5] * inv, x[c][6] * inv, x[c][7] * inv);
          *reinterpret_cast<uint2*>(dst + (head + row) * D + cc * 8) = o;
        }
      }
    } else {
      // ---------------------------------------------------------- V, written transposed
      // Thread (cc, kg): columns 8 cc .. 8 cc + 7, keys 8 kg .. 8 kg + 7 of the block; kg runs
      // fastest so that a warp's stores of one column cover 16 key groups = 128 bytes.
      const int kg = tid % 16;
      const int cc = tid / 16;
      const bool mine = cc < Ly::NCC;
      float x[kChunks][8];  // [key][column]
      float amax = 0.0f;
#pragma unroll
      for (int c = 0; c < kChunks; ++c) {
        if (mine) {
          unpack8<kBf16>(buf[c * kThreads + tid], x[c]);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) x[c][e] = 0.0f;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(x[c][e]));
      }
      const float A = block_max(amax, rd);
      const float inv = A > 0.0f ? 448.0f / A : 1.0f;
      if (tid == 0)
        p.scales[2][static_cast<int64_t>(w.bh) * p.nblk + w.blk] = A > 0.0f ? A / 448.0f : 1.0f;
      const int key0 = row0 + kg * 8;
      if (mine && key0 < n) {  // n is a multiple of 8, so the run of 8 keys is whole
        uint8_t* dst = p.out[2] + static_cast<int64_t>(w.bh) * D * n;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          uint2 o;
          o.x = pack4_e4m3(x[0][e] * inv, x[1][e] * inv, x[2][e] * inv, x[3][e] * inv);
          o.y = pack4_e4m3(x[4][e] * inv, x[5][e] * inv, x[6][e] * inv, x[7][e] * inv);
          *reinterpret_cast<uint2*>(dst + static_cast<int64_t>(cc * 8 + e) * n + key0) = o;
        }
      }
    }
  }
}

inline int sm_count() {
  static int count = [] {
    int dev = 0, c = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || c < 1)
      c = 1;
    return c;
  }();
  return count;
}

template <bool kBf16, int D>
int run(const Params& p, int heads, cudaStream_t s, std::string& err) {
  const int items = 3 * heads * p.nblk;
  const int ctas = items < 3 * sm_count() ? items : 3 * sm_count();
  const size_t smem = 2 * kChunks * kThreads * sizeof(uint4);
  auto kern = quant_kernel<kBf16, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e == cudaSuccess) {
    kern<<<ctas, kThreads, smem, s>>>(p, heads, items);
    e = cudaGetLastError();
  }
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
