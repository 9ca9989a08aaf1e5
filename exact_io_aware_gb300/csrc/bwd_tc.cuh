// Backward pass, part 1 of 2: dK and dV on the tcgen05 tensor cores (fp16 / bf16).
//
// Follows the reverse procedure of "Exact tiled attention and memory-aware differentiation":
// every score block is recomputed from Q and K, p_ij = exp(s_ij - LSE_i) uses the retained row
// statistic, g_ij = p_ij (dO_i . V_j - D_i) with D_i = dO_i . O_i, and
//   dV_j += p_ij dO_i,   dK_j += c g_ij Q_i.
// The dQ_i += c g_ij K_j part is computed by the query-tile kernel in dq_tc.cuh, which
// recomputes the same p and g; splitting keeps every product 128 x 128 (full tensor-core rate),
// needs no float32 atomics, and leaves tensor memory to the four accumulators below.
// No probability matrix is ever stored.
//
// One CTA owns a tile of 128 keys of one head and walks the 128-query blocks that can reach it
// (all of them, those at or after the diagonal under the causal mask, or the nonempty ones
// under a bitmap).  Per query block:
//   Sᵀ  = K Qᵀ              (tensor memory, one key per lane, 128 query columns)
//   Pᵀ  = exp2(Sᵀ c log2e - LSE log2e)   softmax warps; 16-bit, written over Sᵀ and kept in
//                                         registers for the dS pass
//   dPᵀ = V dOᵀ
//   dSᵀ = Pᵀ (dPᵀ - D)                   softmax warps; 16-bit, written over dPᵀ
//   dV += Pᵀ dO,  dK += dSᵀ Q            (A operand read from tensor memory)
// Roles:
//   warp  0    TMEM allocator and MMA issuer (lowest warp slot: the warp schedulers favour it
//              over the softmax warps it shares a sub-partition with)
//   warps 1-8  softmax: warp w owns TMEM lanes 32 (w % 4).. and, of the block's query
//              columns, the 32-column chunks 64 t + 32 h (h = (w - 1) / 4; P and dS are
//              elementwise, so the warps never meet); P is published in two halves (chunks
//              t = 0, then t = 1); at the end warps 1-4 write dV and warps 5-8 dK
//   warp  9    TMA producer (K, V once; dO, Q, LSE, D per block through an NS-stage ring, dO
//              and Q on barriers of their own)
// Issue order per block i: dV_i (its first four k-steps once P's first half is stored),
// S_{i+1}, dK_i, dP_{i+1}: S_{i+1} follows dV_i, the last reader of P_i, and dP_{i+1} follows
// dK_i, the last reader of dS_i.
// Dropout (kDrop): the mask of dropout.cuh is redrawn for the block's (query, key) pairs; the
// dV operand is P with dropped pairs zeroed (dV is scaled by 1/(1-p) in the epilogue), and
// dS = P (keep ? dP/(1-p) : 0) - P D uses the unzeroed P.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.h"
#include "tile.cuh"

namespace ea {
namespace bwd {

constexpr int kKeys = 128;
constexpr int BQ = 128;  // queries per block
constexpr int kThreads = 320;
constexpr int kSoftmaxWarps = 8;
constexpr int kMmaWarp = 0;
constexpr int kFirstSoftmaxWarp = 1;
constexpr int kProducerWarp = 9;
constexpr uint32_t kSkip = 0, kFull = 1, kPartial = 2;

struct BwdParams {
  int n;
  float c;
  int mask_kind;
  const uint32_t* mask_bits;
  int64_t mask_row_words;
  int64_t mask_head_stride_words;
  // Row table [heads][n_pad] (n_pad = n rounded up to 128), written by the dQ kernel, which
  // runs first, and read by the dK/dV kernel: L2 = LSE * log2(e), +inf where a row has no
  // allowed key or lies past n; Dv = D_i = rowsum(dO_i * O_i), 0 past n.
  float* L2;
  float* Dv;
  int n_pad;
  // the forward's LSE, which the dQ kernel builds the table from (O, dO and Q it reads through
  // their tensor maps)
  const float* lse;
  uint32_t* status;
  DropoutArgs drop;  // read only by the dropout instantiations
  Ring ring_q;          // depth of the dK/dV kernel's (Q, dO, row table) ring
  Ring ring_k, ring_v;  // depths of the dQ kernel's K and V rings
  int next_cta;         // CTAs resident at once (the SM count): the CTA launched that many after
                        // this one has its first tiles requested into L2 (0: none)
};

__host__ __device__ constexpr int pad32(int x) { return x < 32 ? 32 : x; }

// Column (within an S or dP buffer) of the 16-bit pair holding column c (a query of Sᵀ, a key
// of dP).  Each 32-column chunk packs its pairs into the first 16 of its own fp32 columns: a
// softmax warp owns whole chunks, so the two warps sharing a lane quadrant never overwrite
// columns the other still reads.  The 16 columns of one k-step stay 8 adjacent words.
__host__ __device__ constexpr int packed_col(int c) { return (c / 32) * 32 + (c % 32) / 2; }

// D: width of Q, K, dK rows; DV: width of V, dO, dV rows (the value width).
template <int D, int DV>
struct Config {
  using TK = Tile<kKeys, D>;   // K (and dK staging)
  using TV = Tile<kKeys, DV>;  // V (and dV staging)
  using TQ = Tile<BQ, D>;      // Q stages
  using TG = Tile<BQ, DV>;     // dO stages
  // tensor-memory columns: S, dP, dV, dK
  static constexpr int kColS = 0;
  static constexpr int kColDP = BQ;
  static constexpr int kColDV = 2 * BQ;
  static constexpr int kColDK = kColDV + pad32(DV);
  static constexpr int kTmemCols = kColDK + pad32(D);
  static_assert(kTmemCols <= 512, "tensor memory overflow");
  static constexpr int kTmemAlloc = kTmemCols <= 256 ? 256 : 512;
  // shared memory: K, V, then NS stages of (Q, dO, LSE, D), the step table, and (bitmap masks)
  // each stage's allowed-key words
  static constexpr int kBudget = 227 * 1024 - 2048;
  static constexpr int kStage = TQ::kBytes + TG::kBytes + 2 * BQ * 4;
  static constexpr int kMaxStepBytes = 4 * 1024;
  static constexpr int kFixed = TK::kBytes + TV::kBytes;
  static constexpr int kFit = (kBudget - kFixed - kMaxStepBytes - 4 * BQ * 16) / kStage;
  static constexpr int NS = kFit > 4 ? 4 : kFit;
  static_assert(NS >= 2, "need two query stages");
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + TK::kBytes;
  static constexpr int kOffQ = kOffV + TV::kBytes;
  static constexpr int kOffG = kOffQ + NS * TQ::kBytes;
  static constexpr int kOffL = kOffG + NS * TG::kBytes;  // [NS][BQ] LSE (log2 units)
  static constexpr int kOffD = kOffL + NS * BQ * 4;      // [NS][BQ] D
  static constexpr int kOffSteps = kOffD + NS * BQ * 4;
  __host__ __device__ static constexpr int off_bits(int n) {
    return (kOffSteps + 4 * ((n + BQ - 1) / BQ) + 15) / 16 * 16;
  }
  static size_t smem_bytes(int n, bool bitmap) {
    return 1024 + static_cast<size_t>(off_bits(n)) + (bitmap ? NS * BQ * 16 : 0);
  }
};

struct Barriers {
  uint64_t kv_full;
  uint64_t q_full[4], g_full[4], q_empty[4], g_empty[4], ld_full[4];
  uint64_t s_full, p_full[2], dp_full, ds_full;  // p_full[t]: queries 64 t .. 64 t + 63
  uint64_t kv_done;
  uint32_t tmem_base;
  uint32_t nsteps;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ void named_barrier(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// 32 consecutive floats of shared memory (16-byte aligned) with eight 16-byte loads.
__device__ __forceinline__ void load32(const float* src, float (&dst)[32]) {
  const float4* s4 = reinterpret_cast<const float4*>(src);
#pragma unroll
  for (int v = 0; v < 8; ++v) {
    const float4 t = s4[v];
    dst[4 * v] = t.x;
    dst[4 * v + 1] = t.y;
    dst[4 * v + 2] = t.z;
    dst[4 * v + 3] = t.w;
  }
}

template <bool kBf16>
__device__ __forceinline__ void unpack2(uint32_t w, float& lo, float& hi) {
  if constexpr (kBf16) {
    lo = __uint_as_float(w << 16);
    hi = __uint_as_float(w & 0xFFFF0000u);
  } else {
    __half2 h = *reinterpret_cast<__half2*>(&w);
    float2 f = __half22float2(h);
    lo = f.x;
    hi = f.y;
  }
}

// Rounds kW accumulator columns of this thread's TMEM lane (from taddr) times `scale` to 16-bit
// pairs and writes them to row r of the staged tile T from column c_first: up to 64 columns
// are loaded before one wait.  Zeros when `have` is false (no product was accumulated).
template <bool kBf16, class T, int kW>
__device__ __forceinline__ void stage_acc(uint32_t taddr, float scale, uint8_t* stage, int r,
                                          int c_first, bool have) {
  static_assert(kW % 16 == 0, "16-column loads");
  constexpr int kB = kW < 64 ? kW : 64;
#pragma unroll
  for (int c0 = 0; c0 < kW; c0 += kB) {
    uint32_t v[kB];
    if (have) {
#pragma unroll
      for (int c = 0; c < kB; c += 16)
        tmem_ld16(taddr + c0 + c, *reinterpret_cast<uint32_t(*)[16]>(v + c));
      tmem_wait_ld();
    } else {
#pragma unroll
      for (int k = 0; k < kB; ++k) v[k] = 0u;
    }
#pragma unroll
    for (int c = 0; c < kB; c += 8) {
      uint32_t pk[4];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        pk[k] = pack2<kBf16>(scale * __uint_as_float(v[c + 2 * k]), scale * __uint_as_float(v[c + 2 * k + 1]));
      *reinterpret_cast<uint4*>(stage + T::offset(r, c_first + c0 + c)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
  }
}

// kCap: ring depth from the launch (p.ring_q) instead of the compile-time count.
template <bool kBf16, int D, int DV, bool kDrop, bool kCap = false>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
                  const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                  BwdParams p) {
  using C = Config<D, DV>;
  using TK = typename C::TK;
  using TV = typename C::TV;
  using TQ = typename C::TQ;
  using TG = typename C::TG;
  constexpr int NS = C::NS;
  const auto ring_q = ring_of<kCap, NS>(p.ring_q);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sK = smem + C::kOffK;
  uint8_t* sV = smem + C::kOffV;
  uint8_t* sQ = smem + C::kOffQ;
  uint8_t* sG = smem + C::kOffG;
  float* sL = reinterpret_cast<float*>(smem + C::kOffL);
  float* sD = reinterpret_cast<float*>(smem + C::kOffD);
  uint32_t* sBits = reinterpret_cast<uint32_t*>(smem + C::off_bits(p.n));
  uint32_t* steps = reinterpret_cast<uint32_t*>(smem + C::kOffSteps);
  __shared__ Barriers bars;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int n = p.n;
  // heaviest (causal: the first) key tiles first, by groups of heads (work_item)
  const uint32_t wgroup = p.mask_kind == kMaskCausal ? kCausalHeadGroup : 1u;
  uint32_t wrank, whead;
  work_item(blockIdx.y * gridDim.x + blockIdx.x, gridDim.x, gridDim.y, wgroup, wrank, whead);
  const int bh = static_cast<int>(whead);
  const int key0 = static_cast<int>(wrank) * kKeys;
  const int nqb = (n + BQ - 1) / BQ;

  // ---------------------------------------------------------------- prologue
  if (tid == 0) {
    mbar_init(&bars.kv_full, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bars.q_full[s], 1);
      mbar_init(&bars.g_full[s], 1);
      mbar_init(&bars.q_empty[s], 1);
      mbar_init(&bars.g_empty[s], 1);
      mbar_init(&bars.ld_full[s], 32);
    }
    mbar_init(&bars.s_full, 1);
    mbar_init(&bars.p_full[0], kSoftmaxWarps);
    mbar_init(&bars.p_full[1], kSoftmaxWarps);
    mbar_init(&bars.dp_full, 1);
    mbar_init(&bars.ds_full, kSoftmaxWarps);
    mbar_init(&bars.kv_done, 1);
    fence_barrier_init();
  }
  if (warp == kMmaWarp) tmem_alloc(&bars.tmem_base, C::kTmemAlloc);

  // Classify each query block against this key tile: skip / full / partial.  Under no mask
  // or the causal mask the blocks taken are a contiguous run (from the first block holding a
  // row at or past key0 under causal) and each step is classified on the fly; a bitmap mask
  // builds a table of the blocks taken.
  const bool use_table = p.mask_kind == kMaskBitmap;
  const bool causal = p.mask_kind == kMaskCausal;
  const bool key_tail = key0 + kKeys > n;
  const int first_blk = causal ? key0 / BQ : 0;
  if (use_table) {
    for (int i = tid; i < nqb; i += kThreads) steps[i] = 0;
    __syncthreads();
    if (tid < 256) {
      const int nwords = (min(key0 + kKeys, n) - key0 + 31) / 32;
      for (int q0 = 0; q0 < n; q0 += 256) {
        const int q = q0 + tid;
        bool any = false, all = true;
        if (q < n) {
          const uint32_t* row = p.mask_bits + static_cast<int64_t>(bh) * p.mask_head_stride_words +
                                static_cast<int64_t>(q) * p.mask_row_words + key0 / 32;
          for (int w = 0; w < nwords; ++w) {
            const int nk = n - (key0 + 32 * w);
            const uint32_t live = nk >= 32 ? 0xFFFFFFFFu : ((1u << nk) - 1u);
            const uint32_t bits = __ldg(row + w) & live;
            any |= bits != 0;
            all &= bits == live;
          }
        }
        // a warp's 32 rows lie in one query block (BQ is a multiple of 32)
        const bool wany = __any_sync(0xFFFFFFFFu, any);
        const bool wall = __all_sync(0xFFFFFFFFu, all);
        if (lane == 0 && q0 + warp * 32 < n) {
          const uint32_t bits = (wany ? 1u : 0u) | (wall ? 0u : 2u);
          if (bits) atomicOr(&steps[(q0 + warp * 32) / BQ], bits);
        }
      }
    }
    __syncthreads();
    if (warp == 0) {
      // compaction in place, 32 blocks a round: a taken block's entry goes to the count of
      // taken blocks before it, never past its own index
      int ns = 0;
      for (int i0 = 0; i0 < nqb; i0 += 32) {
        const int i = i0 + lane;
        const uint32_t b = i < nqb ? steps[i] : 0u;
        const bool take = (b & 1u) != 0;
        const bool tail = key_tail || (i + 1) * BQ > n;
        const uint32_t cls = ((b & 2u) || tail) ? kPartial : kFull;
        const uint32_t ballot = __ballot_sync(0xFFFFFFFFu, take);
        __syncwarp();
        if (take) steps[ns + __popc(ballot & ((1u << lane) - 1u))] = static_cast<uint32_t>(i) | (cls << 16);
        __syncwarp();
        ns += __popc(ballot);
      }
      if (lane == 0) bars.nsteps = ns;
    }
  } else if (tid == 0) {
    bars.nsteps = nqb - first_blk;
  }
  // Step word: query block | class << 16.
  auto step_at = [&](int i) -> uint32_t {
    if (use_table) return steps[i];
    const int j = first_blk + i;
    const bool all = !causal || j * BQ >= key0 + kKeys - 1;
    const bool tail = key_tail || (j + 1) * BQ > n;
    return static_cast<uint32_t>(j) | ((all && !tail ? kFull : kPartial) << 16);
  };
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const int nsteps = bars.nsteps;
  const uint32_t tmem = bars.tmem_base;

  if (warp == kProducerWarp) {
    // ---------------------------------------------------------------- producer warp
    // Lane 0 issues the TMA loads, including the bulk copies of each block's rows of the row
    // table; for bitmap masks all lanes stage the block's allowed-key words.
    const float* l2_h = p.L2 + static_cast<int64_t>(bh) * p.n_pad;
    const float* d_h = p.Dv + static_cast<int64_t>(bh) * p.n_pad;
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_g);
      // The CTA launched p.next_cta after this one (one per SM, in launch order) finds its K and
      // V tiles and its first query block in L2 instead of waiting on DRAM when it starts.
      if (p.next_cta > 0) {
        const uint32_t nx = gridDim.x, ny = gridDim.y;
        const uint32_t later = blockIdx.y * nx + blockIdx.x + p.next_cta;
        if (later < nx * ny) {
          uint32_t rank_l, head_l;
          work_item(later, nx, ny, wgroup, rank_l, head_l);
          const int key0_l = static_cast<int>(rank_l) * kKeys;
          const int bh_l = static_cast<int>(head_l);
          const int q0_l = p.mask_kind == kMaskCausal ? key0_l : 0;
#pragma unroll
          for (int b = 0; b < TK::L::kBoxes; ++b) tma_prefetch_l2_3d(&tm_k, b * TK::L::kBoxCols, key0_l, bh_l);
#pragma unroll
          for (int b = 0; b < TV::L::kBoxes; ++b) tma_prefetch_l2_3d(&tm_v, b * TV::L::kBoxCols, key0_l, bh_l);
#pragma unroll
          for (int b = 0; b < TQ::L::kBoxes; ++b) tma_prefetch_l2_3d(&tm_q, b * TQ::L::kBoxCols, q0_l, bh_l);
#pragma unroll
          for (int b = 0; b < TG::L::kBoxes; ++b) tma_prefetch_l2_3d(&tm_g, b * TG::L::kBoxCols, q0_l, bh_l);
        }
      }
      mbar_arrive_expect_tx(&bars.kv_full, TK::kBytes + TV::kBytes);
#pragma unroll
      for (int b = 0; b < TK::L::kBoxes; ++b)
        tma_load_3d(sK + b * TK::kBoxBytes, &tm_k, &bars.kv_full, b * TK::L::kBoxCols, key0, bh);
#pragma unroll
      for (int b = 0; b < TV::L::kBoxes; ++b)
        tma_load_3d(sV + b * TV::kBoxBytes, &tm_v, &bars.kv_full, b * TV::L::kBoxCols, key0, bh);
    }
    for (int i = 0; i < nsteps; ++i) {
      const int s = ring_q.stage(i);
      const int q0 = static_cast<int>(step_at(i) & 0xFFFFu) * BQ;
      // dO's stage is free once dV of the step NS before has read it, about a product's time
      // before Q's stage (freed by dK): its load goes first, and Q's (which S waits on) then
      // has the SM's load bandwidth to itself.
      if (!mbar_wait(&bars.g_empty[s], ring_q.parity(i) ^ 1, p.status, 33)) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars.g_full[s], TG::kBytes);
#pragma unroll
        for (int b = 0; b < TG::L::kBoxes; ++b)
          tma_load_3d(sG + s * TG::kBytes + b * TG::kBoxBytes, &tm_g, &bars.g_full[s],
                      b * TG::L::kBoxCols, q0, bh);
      }
      if (!mbar_wait(&bars.q_empty[s], ring_q.parity(i) ^ 1, p.status, 21)) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars.q_full[s], TQ::kBytes);
#pragma unroll
        for (int b = 0; b < TQ::L::kBoxes; ++b)
          tma_load_3d(sQ + s * TQ::kBytes + b * TQ::kBoxBytes, &tm_q, &bars.q_full[s],
                      b * TQ::L::kBoxCols, q0, bh);
      }
      if (lane == 0) {
        // rows q0 .. q0+BQ-1 of the row table (always inside the padded table)
        mbar_expect_tx(&bars.ld_full[s], 2 * BQ * 4);
        bulk_load(sL + s * BQ, l2_h + q0, BQ * 4, &bars.ld_full[s]);
        bulk_load(sD + s * BQ, d_h + q0, BQ * 4, &bars.ld_full[s]);
      }
      if (use_table && ((steps[i] >> 16) & 3u) == kPartial) {
        // words of allowed-key bits for rows q0.. of this block and keys key0..key0+127;
        // rows past n and keys past n read as not allowed
        const uint32_t* bits = p.mask_bits + static_cast<int64_t>(bh) * p.mask_head_stride_words;
        for (int e = lane; e < BQ * 4; e += 32) {
          const int t = e >> 2, w = e & 3;
          const int q = q0 + t, kw = key0 + 32 * w;
          uint32_t word = 0u;
          if (q < n && kw < n) {
            word = __ldg(bits + static_cast<int64_t>(q) * p.mask_row_words + kw / 32);
            const int nk = n - kw;
            if (nk < 32) word &= (1u << nk) - 1u;
          }
          sBits[(s * BQ + t) * 4 + w] = word;
        }
      }
      mbar_arrive(&bars.ld_full[s]);
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA issuer
    // The whole warp runs the loop so that descriptors stay warp-uniform; one elected lane
    // issues.  Operand descriptors are built once per buffer: a 16-element step or a ring
    // stage only adds a constant to the start-address field.
    constexpr uint32_t id_s = idesc_f16(128, BQ, kBf16 ? 1 : 0, 0, 0);  // Sᵀ, dPᵀ
    constexpr uint32_t id_dk = idesc_f16(128, D, kBf16 ? 1 : 0, 0, 1);   // dK
    constexpr uint32_t id_dv = idesc_f16(128, DV, kBf16 ? 1 : 0, 0, 1);  // dV
    constexpr uint64_t kStage = TQ::kBytes >> 4;
    constexpr uint64_t kStageG = TG::kBytes >> 4;
    const uint64_t dk = TK::desc_k(smem_u32(sK), 0), dv = TV::desc_k(smem_u32(sV), 0);
    const uint64_t dq0 = TQ::desc_k(smem_u32(sQ), 0), dg0 = TG::desc_k(smem_u32(sG), 0);
    const uint64_t dqmn0 = TQ::desc_mn(smem_u32(sQ), 0), dgmn0 = TG::desc_mn(smem_u32(sG), 0);
    bool ok = mbar_wait_warp(&bars.kv_full, 0, p.status, 22);
    auto wait_q = [&](int i) -> bool {
      return mbar_wait_warp(&bars.q_full[ring_q.stage(i)], ring_q.parity(i), p.status, 23);
    };
    auto wait_g = [&](int i) -> bool {
      return mbar_wait_warp(&bars.g_full[ring_q.stage(i)], ring_q.parity(i), p.status, 34);
    };
    auto issue_s = [&](int i) {
      const uint64_t dq = dq0 + static_cast<uint64_t>(ring_q.stage(i)) * kStage;
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tmem + C::kColS, dk + TK::k_step(kk), dq + TQ::k_step(kk), id_s, kk > 0 ? 1u : 0u);
        mma_commit(&bars.s_full);
      }
      __syncwarp();
    };
    auto issue_dp = [&](int i) {
      const uint64_t dg = dg0 + static_cast<uint64_t>(ring_q.stage(i)) * kStageG;
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < DV / 16; ++kk)
          mma_ss(tmem + C::kColDP, dv + TV::k_step(kk), dg + TG::k_step(kk), id_s, kk > 0 ? 1u : 0u);
        mma_commit(&bars.dp_full);
      }
      __syncwarp();
    };
    if (ok && nsteps > 0) {
      ok = wait_q(0);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        ok = wait_g(0);
        if (ok) {
          tc_fence_after();
          issue_dp(0);
        }
      }
    }
    for (int i = 0; i < nsteps && ok; ++i) {
      const int s = ring_q.stage(i);
      // dV in two halves of four k-steps, each as soon as its 64 queries of P are stored
      const uint64_t dgmn = dgmn0 + static_cast<uint64_t>(s) * kStageG;
#pragma unroll
      for (int t = 0; t < 2 && ok; ++t) {
        ok = mbar_wait_warp(&bars.p_full[t], i & 1, p.status, 24);
        if (!ok) break;
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int kk = 4 * t; kk < 4 * t + 4; ++kk)
            mma_ts(tmem + C::kColDV, tmem + C::kColS + packed_col(16 * kk), dgmn + TG::mn_step(kk),
                   id_dv, (i > 0 || kk > 0) ? 1u : 0u);
          if (t == 1) mma_commit(&bars.g_empty[s]);
        }
        __syncwarp();
      }
      if (!ok) break;
      const bool more = i + 1 < nsteps;
      if (more) {
        ok = wait_q(i + 1);
        if (!ok) break;
        tc_fence_after();
        issue_s(i + 1);
      }
      ok = mbar_wait_warp(&bars.ds_full, i & 1, p.status, 25);
      if (!ok) break;
      tc_fence_after();
      const uint64_t dqmn = dqmn0 + static_cast<uint64_t>(s) * kStage;
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk)
          mma_ts(tmem + C::kColDK, tmem + C::kColDP + packed_col(16 * kk), dqmn + TQ::mn_step(kk),
                 id_dk, (i > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bars.q_empty[s]);
      }
      __syncwarp();
      if (more) {
        ok = wait_g(i + 1);
        if (!ok) break;
        tc_fence_after();
        issue_dp(i + 1);
      }
    }
    if (elect_one()) mma_commit(&bars.kv_done);
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- softmax: P and dS
    const int quad = warp % 4;
    const int r = quad * 32 + lane;  // key row within the tile = TMEM lane
    const int j = key0 + r;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    // The two warps of a lane quadrant split the query columns in 32-column chunks: chunk t of
    // this warp is [64 t + 32 half, + 32).  Chunk 0 of both warps is queries 0 .. 63, the first
    // four k-steps of dV, which the tensor core starts while the chunks 1 are computed.
    constexpr int kChunks = BQ / 64;
    static_assert(BQ == 128, "two 32-column chunks per warp");
    const int half = (warp - kFirstSoftmaxWarp) / 4;
    auto col0 = [&](int t) { return 64 * t + 32 * half; };
    const float sl2 = p.c * 1.4426950408889634f;
    const uint32_t tS = tmem + C::kColS + lane_off;
    const uint32_t tP = tmem + C::kColDP + lane_off;
    bool ok = true;
    for (int i = 0; i < nsteps && ok; ++i) {
      const uint32_t sw = step_at(i);
      const int q0 = static_cast<int>(sw & 0xFFFFu) * BQ;
      const bool partial = ((sw >> 16) & 3u) == kPartial;
      const int stg = ring_q.stage(i);
      const float* L = sL + stg * BQ;
      const float* Dd = sD + stg * BQ;
      ok = mbar_wait_spin(&bars.ld_full[stg], ring_q.parity(i), p.status, 32);
      if (!ok) break;
      // Dropout: keep bits of this key with the warp's query columns (bit k of word t <->
      // query q0 + col0(t) + k), drawn while the scores are still being computed.  One
      // generator call decides a 4 x 4 patch of (query, key) pairs; the four lanes of a key
      // group (keys 4 g .. 4 g + 3, lanes 4 a .. 4 a + 3) share its calls: lane s draws the
      // patches of queries q0 + col0(s / 2) + 16 (s % 2) .. + 15 and the group exchanges them.
      uint32_t kbits[kDrop ? kChunks : 1];
      if constexpr (kDrop) {
        uint32_t part[4];
        keep_cols<4>(p.drop, static_cast<uint32_t>(q0 + col0(0)) >> 2, static_cast<uint32_t>(q0 + col0(1)) >> 2,
                     static_cast<uint32_t>(j) >> 2, bh, part);
        kbits[0] = part[0] | part[1] << 16;
        kbits[1] = part[2] | part[3] << 16;
      }
      ok = mbar_wait_spin(&bars.s_full, i & 1, p.status, 27);
      if (!ok) break;
      tc_fence_after();
      uint32_t pkeep[kChunks * 16];  // this warp's P pairs, kept for the dS pass
      // both chunks are loaded before one wait: the load latency is paid once
      uint32_t rr[kChunks][32];
#pragma unroll
      for (int t = 0; t < kChunks; ++t) tmem_ld32(tS + col0(t), rr[t]);
      tmem_wait_ld();
#pragma unroll
      for (int t = 0; t < kChunks; ++t) {
        const int c0 = col0(t);
        float pv[32];
        // The block's LSE values are the same for every lane: 16-byte loads take a quarter of
        // the shared-memory cycles of scalar ones, cycles the products' operand reads need.
        float lv[32];
        load32(L + c0, lv);
#pragma unroll
        for (int k = 0; k < 32; ++k) pv[k] = ex2(__uint_as_float(rr[t][k]) * sl2 - lv[k]);
        // Masking is a separate pass over the chunk so the common (full-block) path above
        // stays one compact run of instructions.
        if (partial) {
          if (p.mask_kind == kMaskBitmap) {
            // this warp's 32 keys share one word per query row (staged by the producer)
            const uint32_t* wb = sBits + (stg * BQ + c0) * 4 + quad;
#pragma unroll
            for (int k = 0; k < 32; ++k)
              if (!((wb[4 * k] >> lane) & 1u)) pv[k] = 0.0f;
          } else {
#pragma unroll
            for (int k = 0; k < 32; ++k) {
              const int q = q0 + c0 + k;
              if (q >= n || j >= n || (causal && j > q)) pv[k] = 0.0f;
            }
          }
        }
        uint32_t pk[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          pkeep[16 * t + k] = pack2<kBf16>(pv[2 * k], pv[2 * k + 1]);
          if constexpr (kDrop) {
            const uint32_t kb = kbits[t] >> (2 * k);
            pk[k] = pack2<kBf16>(kb & 1u ? pv[2 * k] : 0.0f, kb & 2u ? pv[2 * k + 1] : 0.0f);
          } else {
            pk[k] = pkeep[16 * t + k];
          }
        }
        tmem_st16(tS + packed_col(c0), pk);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.p_full[t]);
      }

      ok = mbar_wait_spin(&bars.dp_full, i & 1, p.status, 28);
      if (!ok) break;
      tc_fence_after();
      uint32_t dp[kChunks][32];
#pragma unroll
      for (int t = 0; t < kChunks; ++t) tmem_ld32(tP + col0(t), dp[t]);
      tmem_wait_ld();
#pragma unroll
      for (int t = 0; t < kChunks; ++t) {
        const int c0 = col0(t);
        uint32_t pk[16];
        float dv[32];
        load32(Dd + c0, dv);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          float p0, p1;
          unpack2<kBf16>(pkeep[16 * t + k], p0, p1);
          float d0 = __uint_as_float(dp[t][2 * k]);
          float d1 = __uint_as_float(dp[t][2 * k + 1]);
          if constexpr (kDrop) {
            const uint32_t kb = kbits[t] >> (2 * k);
            d0 = kb & 1u ? d0 * p.drop.scale : 0.0f;
            d1 = kb & 2u ? d1 * p.drop.scale : 0.0f;
          }
          const float g0 = p0 * (d0 - dv[2 * k]);
          const float g1 = p1 * (d1 - dv[2 * k + 1]);
          pk[k] = pack2<kBf16>(g0, g1);
        }
        tmem_st16(tP + packed_col(c0), pk);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.ds_full);
    }
    // ---------------------------------------------------------------- epilogue
    // dV = Pᵀ dO (the warps of half 0) and dK = c * (dSᵀ Q) (half 1), rounded and staged in
    // the (now idle) V and K tiles, then stored by TMA.
    if (ok) ok = mbar_wait_spin(&bars.kv_done, 0, p.status, 31);
    tc_fence_after();
    if (ok) {
      if (half == 0)  // dV = (P with dropped pairs zeroed)ᵀ dO / (1-p)
        stage_acc<kBf16, TV, DV>(tmem + C::kColDV + lane_off, kDrop ? p.drop.scale : 1.0f, sV, r, 0,
                                 nsteps > 0);
      else
        stage_acc<kBf16, TK, D>(tmem + C::kColDK + lane_off, p.c, sK, r, 0, nsteps > 0);
    }
    fence_proxy_async_smem();
    named_barrier(2, kSoftmaxWarps * 32);
    if (ok && half == 0 && r == 0) {
#pragma unroll
      for (int b = 0; b < TK::L::kBoxes; ++b)
        tma_store_3d(&tm_dk, sK + b * TK::kBoxBytes, b * TK::L::kBoxCols, key0, bh);
#pragma unroll
      for (int b = 0; b < TV::L::kBoxes; ++b)
        tma_store_3d(&tm_dv, sV + b * TV::kBoxBytes, b * TV::L::kBoxCols, key0, bh);
      tma_store_commit();
      tma_store_wait_all();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemAlloc);
  }
}

}  // namespace bwd
}  // namespace ea
