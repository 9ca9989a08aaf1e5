// float32 forward and backward on the CUDA cores.
//
// The tensor cores have no float32 multiply (tf32 drops 13 mantissa bits), so the float32 path
// runs the same algorithm with FFMA: the tiled forward procedure and the recomputing reverse
// procedure of "Exact tiled attention and memory-aware differentiation".
//
// Forward: a CTA holds 32 query rows; each warp owns 4 of them.  Key/value blocks of b rows
// (the caller's key-block size) are staged in shared memory; per block every row forms its
// block summary (max, shifted normaliser, shifted value sum) and merges it into its running
// summary.  A block with no allowed key leaves the summary unchanged.  Lanes take keys for the
// scores and output columns for the value sums.
//
// Key split (gridDim.z > 1): CTA z walks only its share of the key blocks and writes its rows'
// normalised partial (O_z, LSE_z) to the split buffers; a merge kernel combines the shares.
//
// Dropout (drop = true): the mask of dropout.cuh is drawn per (query, key) pair; kept
// probabilities enter O and dV scaled by 1/(1-p), the normaliser keeps every probability, and
// dS = P (keep ? dP/(1-p) : 0) - P D.
//
// Backward: two kernels, no atomics.  The dQ kernel walks key blocks past 32 query rows; the
// dK/dV kernel walks query blocks past 32 key rows.  Both recompute s_ij and
// p_ij = exp(s_ij - LSE_i) and use D_i = dO_i . O_i from the preprocessing kernel.
//
// Template parameters D (width of Q and K rows) and DV (width of V, O and dO rows: the value
// width, D unless the values are wider or narrower than the keys).  The launchers in
// simt_f32.cu (DV = D) and simt_f32_vd.cu (DV != D) instantiate them.
#pragma once
#include <cmath>
#include <string>

#include "kernels.h"
#include "status.cuh"

namespace ea {
namespace f32 {

constexpr int kWarps = 8;
constexpr int kRowsPerWarp = 4;
constexpr int kRows = kWarps * kRowsPerWarp;  // 32 rows per CTA

struct Mask {
  int kind;
  int n;  // query rows
  const uint32_t* bits;
  int64_t row_words;
  int64_t head_stride;
  int nk;   // keys
  int off;  // causal: query i sees keys j <= i + off
  __device__ __forceinline__ bool allowed(int bh, int i, int j) const {
    if (j >= nk || i >= n) return false;
    if (kind == kMaskCausal) return j <= i + off;
    if (kind == kMaskBitmap) {
      const uint32_t w = __ldg(bits + bh * head_stride + static_cast<int64_t>(i) * row_words + j / 32);
      return (w >> (j % 32)) & 1u;
    }
    return true;
  }
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// ------------------------------------------------------------------------------- forward
template <int D, int DV, int BN>
__global__ void __launch_bounds__(kWarps * 32) fwd_kernel(const float* __restrict__ Q,
                                                          const float* __restrict__ K,
                                                          const float* __restrict__ V,
                                                          float* __restrict__ O,
                                                          float* __restrict__ lse, float c,
                                                          Mask mk, uint32_t* status,
                                                          DropoutArgs dr, bool drop) {
  extern __shared__ float sm[];
  float* sQ = sm;                       // [kRows][D]
  float* sK = sQ + kRows * D;           // [BN][D + 1]
  float* sV = sK + BN * (D + 1);        // [BN][DV]
  constexpr int NU = (DV + 31) / 32;    // output columns per lane
  constexpr int NJ = BN / 32;           // keys per lane per block
  const int n = mk.n;    // query rows
  const int nk = mk.nk;  // keys
  const int bh = blockIdx.y;
  const int row_base = blockIdx.x * kRows;
  const size_t head = static_cast<size_t>(bh) * n * D;      // Q rows of this head
  const size_t k_head = static_cast<size_t>(bh) * nk * D;   // K rows of this head
  const size_t v_head = static_cast<size_t>(bh) * nk * DV;  // V rows of this head
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool partial_out = gridDim.z > 1;  // O, lse point at the split buffers
  const size_t out_head = (static_cast<size_t>(blockIdx.z) * gridDim.y + bh) * n;

  for (int e = threadIdx.x; e < kRows * D; e += blockDim.x) {
    const int r = e / D, col = e % D;
    sQ[e] = (row_base + r < n) ? Q[head + static_cast<size_t>(row_base + r) * D + col] : 0.0f;
  }
  float m[kRowsPerWarp], l[kRowsPerWarp], z[kRowsPerWarp][NU];
#pragma unroll
  for (int q = 0; q < kRowsPerWarp; ++q) {
    m[q] = -INFINITY;
    l[q] = 0.0f;
#pragma unroll
    for (int u = 0; u < NU; ++u) z[q][u] = 0.0f;
  }
  const int last_row = min(row_base + kRows, n) - 1;
  const int key_end = mk.kind == kMaskCausal ? max(0, min(nk, last_row + mk.off + 1)) : nk;
  const int reach = (key_end + BN - 1) / BN;  // key blocks the rows reach
  const int share = (reach + gridDim.z - 1) / gridDim.z;
  const int kb_lo = min(static_cast<int>(blockIdx.z) * share, reach);
  const int kb_hi = min(kb_lo + share, reach);
  for (int key0 = kb_lo * BN; key0 < kb_hi * BN; key0 += BN) {
    __syncthreads();
    for (int e = threadIdx.x; e < BN * D; e += blockDim.x) {
      const int j = e / D, col = e % D;
      sK[j * (D + 1) + col] = key0 + j < nk ? K[k_head + static_cast<size_t>(key0 + j) * D + col] : 0.0f;
    }
    for (int e = threadIdx.x; e < BN * DV; e += blockDim.x) {
      const int j = e / DV, col = e % DV;
      sV[e] = key0 + j < nk ? V[v_head + static_cast<size_t>(key0 + j) * DV + col] : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < kRowsPerWarp; ++q) {
      const int r = warp * kRowsPerWarp + q;
      const int i = row_base + r;
      float s[NJ];
#pragma unroll
      for (int u = 0; u < NJ; ++u) {
        const int j = u * 32 + lane;
        float acc = 0.0f;
#pragma unroll 8
        for (int col = 0; col < D; ++col) acc = fmaf(sQ[r * D + col], sK[j * (D + 1) + col], acc);
        s[u] = mk.allowed(bh, i, key0 + j) ? c * acc : -INFINITY;
      }
      float bmax = s[0];
#pragma unroll
      for (int u = 1; u < NJ; ++u) bmax = fmaxf(bmax, s[u]);
      bmax = warp_max(bmax);
      if (bmax == -INFINITY) continue;  // J_t ∩ A_i empty: summary unchanged
      const float mn = fmaxf(m[q], bmax);
      const float scale = expf(m[q] - mn);  // 0 when the summary was still empty
      float ps = 0.0f;
#pragma unroll
      for (int u = 0; u < NJ; ++u) {
        s[u] = expf(s[u] - mn);
        ps += s[u];
        if (drop && !keep1(dr, static_cast<uint32_t>(i), static_cast<uint32_t>(key0 + u * 32 + lane),
                           static_cast<uint32_t>(bh)))
          s[u] = 0.0f;  // dropped: out of the value sum, still in the normaliser
      }
      l[q] = l[q] * scale + warp_sum(ps);
      m[q] = mn;
#pragma unroll
      for (int u = 0; u < NU; ++u) z[q][u] *= scale;
#pragma unroll
      for (int u = 0; u < NJ; ++u) {
        for (int jj = 0; jj < 32; ++jj) {
          const float pj = __shfl_sync(0xFFFFFFFFu, s[u], jj);
          const int j = u * 32 + jj;
#pragma unroll
          for (int w = 0; w < NU; ++w) {
            const int col = w * 32 + lane;
            if (col < DV) z[q][w] = fmaf(pj, sV[j * DV + col], z[q][w]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int q = 0; q < kRowsPerWarp; ++q) {
    const int i = row_base + warp * kRowsPerWarp + q;
    if (i >= n) continue;
    const bool empty = !(l[q] > 0.0f);
    const float inv = empty ? 0.0f : (drop ? dr.scale : 1.0f) / l[q];
#pragma unroll
    for (int w = 0; w < NU; ++w) {
      const int col = w * 32 + lane;
      if (col < DV) O[(out_head + i) * DV + col] = z[q][w] * inv;
    }
    if (lane == 0) {
      lse[out_head + i] = empty ? -INFINITY : m[q] + logf(l[q]);
      if (empty && !partial_out) raise_empty_row(status);
    }
  }
}

// ------------------------------------------------------------------------------- dQ
template <int D, int DV>
__global__ void __launch_bounds__(kWarps * 32) dq_kernel(
    const float* __restrict__ Q, const float* __restrict__ K, const float* __restrict__ V,
    const float* __restrict__ dO, const float* __restrict__ lse, const float* __restrict__ Dv,
    float* __restrict__ dQ, float c, Mask mk, DropoutArgs dr, bool drop) {
  constexpr int BN = 64;
  extern __shared__ float sm[];
  float* sQ = sm;                   // [kRows][D]
  float* sG = sQ + kRows * D;       // [kRows][DV]  (dO rows)
  float* sK = sG + kRows * DV;      // [BN][D + 1]
  float* sV = sK + BN * (D + 1);    // [BN][DV + 1]
  constexpr int NU = (D + 31) / 32;
  constexpr int NJ = BN / 32;
  const int n = mk.n;
  const int bh = blockIdx.y;
  const int row_base = blockIdx.x * kRows;
  const size_t head = static_cast<size_t>(bh) * n * D;     // Q, K, dQ rows
  const size_t vhead = static_cast<size_t>(bh) * n * DV;   // V, dO rows
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = threadIdx.x; e < kRows * D; e += blockDim.x) {
    const int r = e / D, col = e % D;
    sQ[e] = row_base + r < n ? Q[head + static_cast<size_t>(row_base + r) * D + col] : 0.0f;
  }
  for (int e = threadIdx.x; e < kRows * DV; e += blockDim.x) {
    const int r = e / DV, col = e % DV;
    sG[e] = row_base + r < n ? dO[vhead + static_cast<size_t>(row_base + r) * DV + col] : 0.0f;
  }
  float acc[kRowsPerWarp][NU];
  float L[kRowsPerWarp], Dd[kRowsPerWarp];
#pragma unroll
  for (int q = 0; q < kRowsPerWarp; ++q) {
    const int i = row_base + warp * kRowsPerWarp + q;
    L[q] = i < n ? lse[static_cast<size_t>(bh) * n + i] : -INFINITY;
    Dd[q] = i < n ? Dv[static_cast<size_t>(bh) * n + i] : 0.0f;
#pragma unroll
    for (int u = 0; u < NU; ++u) acc[q][u] = 0.0f;
  }
  const int last_row = min(row_base + kRows, n) - 1;
  const int key_end = mk.kind == kMaskCausal ? last_row + 1 : n;
  for (int key0 = 0; key0 < key_end; key0 += BN) {
    __syncthreads();
    for (int e = threadIdx.x; e < BN * D; e += blockDim.x) {
      const int j = e / D, col = e % D;
      sK[j * (D + 1) + col] = key0 + j < n ? K[head + static_cast<size_t>(key0 + j) * D + col] : 0.0f;
    }
    for (int e = threadIdx.x; e < BN * DV; e += blockDim.x) {
      const int j = e / DV, col = e % DV;
      sV[j * (DV + 1) + col] = key0 + j < n ? V[vhead + static_cast<size_t>(key0 + j) * DV + col] : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < kRowsPerWarp; ++q) {
      const int r = warp * kRowsPerWarp + q;
      const int i = row_base + r;
      if (L[q] == -INFINITY) continue;
      float ds[NJ];
#pragma unroll
      for (int u = 0; u < NJ; ++u) {
        const int j = u * 32 + lane;
        float sdot = 0.0f, pdot = 0.0f;
#pragma unroll 8
        for (int col = 0; col < D; ++col) sdot = fmaf(sQ[r * D + col], sK[j * (D + 1) + col], sdot);
#pragma unroll 8
        for (int col = 0; col < DV; ++col) pdot = fmaf(sG[r * DV + col], sV[j * (DV + 1) + col], pdot);
        const float pij = mk.allowed(bh, i, key0 + j) ? expf(c * sdot - L[q]) : 0.0f;
        if (drop)
          pdot = keep1(dr, static_cast<uint32_t>(i), static_cast<uint32_t>(key0 + j),
                       static_cast<uint32_t>(bh)) ? pdot * dr.scale : 0.0f;
        ds[u] = pij * (pdot - Dd[q]);
      }
#pragma unroll
      for (int u = 0; u < NJ; ++u) {
        for (int jj = 0; jj < 32; ++jj) {
          const float g = __shfl_sync(0xFFFFFFFFu, ds[u], jj);
          const int j = u * 32 + jj;
#pragma unroll
          for (int w = 0; w < NU; ++w) {
            const int col = w * 32 + lane;
            if (col < D) acc[q][w] = fmaf(g, sK[j * (D + 1) + col], acc[q][w]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int q = 0; q < kRowsPerWarp; ++q) {
    const int i = row_base + warp * kRowsPerWarp + q;
    if (i >= n) continue;
#pragma unroll
    for (int w = 0; w < NU; ++w) {
      const int col = w * 32 + lane;
      if (col < D) dQ[head + static_cast<size_t>(i) * D + col] = c * acc[q][w];
    }
  }
}

// ------------------------------------------------------------------------------- dK, dV
template <int D, int DV>
__global__ void __launch_bounds__(kWarps * 32) dkdv_kernel(
    const float* __restrict__ Q, const float* __restrict__ K, const float* __restrict__ V,
    const float* __restrict__ dO, const float* __restrict__ lse, const float* __restrict__ Dv,
    float* __restrict__ dK, float* __restrict__ dV, float c, Mask mk, DropoutArgs dr, bool drop) {
  constexpr int BM = 64;
  extern __shared__ float sm[];
  float* sK = sm;                   // [kRows][D]   this CTA's key rows
  float* sVr = sK + kRows * D;      // [kRows][DV]  this CTA's value rows
  float* sQ = sVr + kRows * DV;     // [BM][D + 1]
  float* sG = sQ + BM * (D + 1);    // [BM][DV + 1]
  float* sL = sG + BM * (DV + 1);   // [BM]
  float* sD = sL + BM;              // [BM]
  constexpr int NU = (D + 31) / 32;
  constexpr int NUV = (DV + 31) / 32;
  constexpr int NI = BM / 32;
  const int n = mk.n;
  const int bh = blockIdx.y;
  const int key_base = blockIdx.x * kRows;
  const size_t head = static_cast<size_t>(bh) * n * D;     // Q, K, dK rows
  const size_t vhead = static_cast<size_t>(bh) * n * DV;   // V, dO, dV rows
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = threadIdx.x; e < kRows * D; e += blockDim.x) {
    const int r = e / D, col = e % D;
    sK[e] = key_base + r < n ? K[head + static_cast<size_t>(key_base + r) * D + col] : 0.0f;
  }
  for (int e = threadIdx.x; e < kRows * DV; e += blockDim.x) {
    const int r = e / DV, col = e % DV;
    sVr[e] = key_base + r < n ? V[vhead + static_cast<size_t>(key_base + r) * DV + col] : 0.0f;
  }
  float ak[kRowsPerWarp][NU], av[kRowsPerWarp][NUV];
#pragma unroll
  for (int q = 0; q < kRowsPerWarp; ++q) {
#pragma unroll
    for (int u = 0; u < NU; ++u) ak[q][u] = 0.0f;
#pragma unroll
    for (int u = 0; u < NUV; ++u) av[q][u] = 0.0f;
  }
  const int q_start = mk.kind == kMaskCausal ? (key_base / BM) * BM : 0;
  for (int qb = q_start; qb < n; qb += BM) {
    __syncthreads();
    for (int e = threadIdx.x; e < BM * D; e += blockDim.x) {
      const int i = e / D, col = e % D;
      sQ[i * (D + 1) + col] = qb + i < n ? Q[head + static_cast<size_t>(qb + i) * D + col] : 0.0f;
    }
    for (int e = threadIdx.x; e < BM * DV; e += blockDim.x) {
      const int i = e / DV, col = e % DV;
      sG[i * (DV + 1) + col] = qb + i < n ? dO[vhead + static_cast<size_t>(qb + i) * DV + col] : 0.0f;
    }
    for (int i = threadIdx.x; i < BM; i += blockDim.x) {
      const bool in = qb + i < n;
      sL[i] = in ? lse[static_cast<size_t>(bh) * n + qb + i] : -INFINITY;
      sD[i] = in ? Dv[static_cast<size_t>(bh) * n + qb + i] : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < kRowsPerWarp; ++q) {
      const int r = warp * kRowsPerWarp + q;
      const int j = key_base + r;
      float pp[NI], ds[NI];
#pragma unroll
      for (int u = 0; u < NI; ++u) {
        const int i = u * 32 + lane;
        float sdot = 0.0f, pdot = 0.0f;
#pragma unroll 8
        for (int col = 0; col < D; ++col) sdot = fmaf(sQ[i * (D + 1) + col], sK[r * D + col], sdot);
#pragma unroll 8
        for (int col = 0; col < DV; ++col) pdot = fmaf(sG[i * (DV + 1) + col], sVr[r * DV + col], pdot);
        const bool ok = sL[i] != -INFINITY && mk.allowed(bh, qb + i, j);
        const float pij = ok ? expf(c * sdot - sL[i]) : 0.0f;
        pp[u] = pij;
        if (drop) {
          const bool kept = keep1(dr, static_cast<uint32_t>(qb + i), static_cast<uint32_t>(j),
                                  static_cast<uint32_t>(bh));
          pp[u] = kept ? pij * dr.scale : 0.0f;
          pdot = kept ? pdot * dr.scale : 0.0f;
        }
        ds[u] = pij * (pdot - sD[i]);
      }
#pragma unroll
      for (int u = 0; u < NI; ++u) {
        for (int ii = 0; ii < 32; ++ii) {
          const float pv = __shfl_sync(0xFFFFFFFFu, pp[u], ii);
          const float g = __shfl_sync(0xFFFFFFFFu, ds[u], ii);
          const int i = u * 32 + ii;
#pragma unroll
          for (int w = 0; w < NUV; ++w) {
            const int col = w * 32 + lane;
            if (col < DV) av[q][w] = fmaf(pv, sG[i * (DV + 1) + col], av[q][w]);
          }
#pragma unroll
          for (int w = 0; w < NU; ++w) {
            const int col = w * 32 + lane;
            if (col < D) ak[q][w] = fmaf(g, sQ[i * (D + 1) + col], ak[q][w]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int q = 0; q < kRowsPerWarp; ++q) {
    const int j = key_base + warp * kRowsPerWarp + q;
    if (j >= n) continue;
#pragma unroll
    for (int w = 0; w < NU; ++w) {
      const int col = w * 32 + lane;
      if (col < D) dK[head + static_cast<size_t>(j) * D + col] = c * ak[q][w];
    }
#pragma unroll
    for (int w = 0; w < NUV; ++w) {
      const int col = w * 32 + lane;
      if (col < DV) dV[vhead + static_cast<size_t>(j) * DV + col] = av[q][w];
    }
  }
}

template <typename Kern>
int set_smem(Kern k, size_t bytes, std::string& err) {
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(bytes));
  if (e != cudaSuccess) {
    err = std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e);
    return -5;
  }
  return 0;
}

inline Mask make_mask(const AttnArgs& a) {
  const int nk = a.nk > 0 ? a.nk : a.n;
  return Mask{a.mask_kind, a.n, a.mask_bits, a.mask_row_words, a.mask_head_stride_words, nk,
              nk - a.n};
}

template <int D, int DV, int BN>
int fwd_run(const AttnArgs& a, cudaStream_t s, std::string& err) {
  const size_t smem = sizeof(float) * (kRows * D + BN * (D + 1) + BN * DV);
  auto k = fwd_kernel<D, DV, BN>;
  if (int rc = set_smem(k, smem, err)) return rc;
  const bool split = a.num_splits > 1;
  dim3 grid((a.n + kRows - 1) / kRows, a.B * a.H, split ? a.num_splits : 1);
  k<<<grid, kWarps * 32, smem, s>>>(static_cast<const float*>(a.q), static_cast<const float*>(a.k),
                                    static_cast<const float*>(a.v),
                                    split ? a.o_part : static_cast<float*>(a.o_out),
                                    split ? a.lse_part : a.lse, a.c, make_mask(a), a.status,
                                    a.drop, a.dropout);
  return 0;
}

template <int D, int DV = D>
int fwd_d(const AttnArgs& a, cudaStream_t s, std::string& err) {
  const int bn = a.kv_block == 0 ? 64 : a.kv_block;
  switch (bn) {
    case 32: return fwd_run<D, DV, 32>(a, s, err);
    case 64: return fwd_run<D, DV, 64>(a, s, err);
    case 128: return fwd_run<D, DV, 128>(a, s, err);
    default: err = "kv_block must be 0, 32, 64 or 128"; return -2;
  }
}

template <int D, int DV = D>
int bwd_d(const AttnArgs& a, const float* Dv, cudaStream_t s, std::string& err) {
  const size_t smem_q = sizeof(float) * (kRows * (D + DV) + 64 * (D + 1) + 64 * (DV + 1));
  const size_t smem_k = sizeof(float) * (kRows * (D + DV) + 64 * (D + 1) + 64 * (DV + 1) + 2 * 64);
  auto kq = dq_kernel<D, DV>;
  auto kk = dkdv_kernel<D, DV>;
  if (int rc = set_smem(kq, smem_q, err)) return rc;
  if (int rc = set_smem(kk, smem_k, err)) return rc;
  dim3 grid((a.n + kRows - 1) / kRows, a.B * a.H);
  const float* q = static_cast<const float*>(a.q);
  const float* k = static_cast<const float*>(a.k);
  const float* v = static_cast<const float*>(a.v);
  const float* g = static_cast<const float*>(a.d_o);
  kq<<<grid, kWarps * 32, smem_q, s>>>(q, k, v, g, a.lse, Dv, static_cast<float*>(a.dq), a.c,
                                       make_mask(a), a.drop, a.dropout);
  kk<<<grid, kWarps * 32, smem_k, s>>>(q, k, v, g, a.lse, Dv, static_cast<float*>(a.dk),
                                       static_cast<float*>(a.dv), a.c, make_mask(a), a.drop,
                                       a.dropout);
  return 0;
}

}  // namespace f32
}  // namespace ea
