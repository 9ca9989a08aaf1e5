// Backward pass, part 2 of 2: dQ on the tcgen05 tensor cores (fp16 / bf16).
//
// The query-row side of the reverse procedure of "Exact tiled attention and memory-aware
// differentiation": for each query row i and allowed key j, recompute s_ij from Q and K,
// p_ij = exp(s_ij - LSE_i), g_ij = p_ij (dO_i . V_j - D_i), and accumulate
//   dQ_i += c g_ij K_j.
// (dK and dV come from the key-tile kernel in bwd_tc.cuh, which recomputes the same p and g.)
//
// One CTA owns a tile of 128 query rows of one head and walks the 128-key blocks they reach,
// exactly like the forward; LSE_i and D_i are per-row scalars held by the row's thread.  The
// kernel computes D_i = rowsum(dO_i * O_i) itself (each softmax warp of a row sums half of
// the columns) and writes the row table (LSE_i log2 e and D_i) that the dK/dV kernel, launched
// after it, copies per query block.
// Q and dO are the same for every key block, so the softmax warps write them into tensor
// memory once (the rows they read for D_i anyway, from the tile's Q, dO and O staged in
// shared memory by TMA; 16-bit pairs per column, the A-operand layout), and all three
// products read only their B operand from shared memory.  With both
// operands in shared memory a 128 x 128 x 16 product needs the SM's whole shared-memory
// bandwidth, and the products ran at ~88 instead of ~64 cycles.  Per key block j:
//   S  = Q K_jᵀ           (A = Q in tensor memory; one buffer, free again as soon as the
//                          softmax warps have loaded it)
//   P  = exp2(S c log2e - LSE log2e)     softmax warps, kept in registers
//   dP = dO V_jᵀ          (A = dO in tensor memory; one buffer)
//   dS = P (dP - D)                      softmax warps; 16-bit, written over dP
//   dQ += dS K_j                         (A = dS in tensor memory)
// Dropout (kDrop): dS = P (keep ? dP/(1-p) : 0) - P D with the mask of dropout.cuh redrawn for
// the block's (query, key) pairs; P itself is not masked here (dQ needs only dS).
// Roles (the control warps take the lowest warp slots, which the warp schedulers favour over
// the softmax warps they share a sub-partition with):
//   warp  0    TMEM allocator and MMA issuer
//   warp  1    TMA producer of the K ring (NSK stages); blocks a few steps ahead are
//              requested into L2
//   warp  2    TMA producer of the V ring (NSV stages): the two rings are released by
//              different products (K after dQ, V after dP), so neither waits on the other;
//              it first stages the tile's Q, dO and O (its last two stages hold dO and O
//              until the softmax warps have read them)
//   warps 3-10 softmax: warp w owns TMEM lanes 32 (w % 4).. and half (w - 3) / 4 of the
//              block's key columns (and of Q's and dO's columns when it stages them); each
//              half writes half of dQ's columns at the end
// Issue order per block i: [S_{i+1} once S_i is loaded], dQ_i once dS_i is written, then
// dP_{i+1}, which overwrites dS_i after dQ_i has read it (one thread's MMAs run in issue
// order).  The softmax warps compute P_{i+1} while dQ_i and dP_{i+1} run, and the tensor core
// runs S_{i+2} while they compute dS_{i+1}.  K is held from S_i to dQ_i, across two issue
// rounds, hence its deeper ring.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "bwd_tc.cuh"

namespace ea {
namespace dq {

constexpr int kRows = 128;  // query rows per CTA
constexpr int BN = 128;     // keys per block
constexpr int kThreads = 352;
constexpr int kSoftmaxWarps = 8;
constexpr int kMmaWarp = 0;
constexpr int kKProducerWarp = 1;
constexpr int kVProducerWarp = 2;
constexpr int kFirstSoftmaxWarp = 3;
constexpr int kPrefetch = 4;  // key blocks requested into L2 ahead of the ring loads
using bwd::kFull;
using bwd::kPartial;
using bwd::kSkip;
using bwd::packed_col;
using bwd::pad32;
using bwd::unpack2;

// D: width of Q, K, dQ rows; DV: width of V, dO rows (the value width).
template <int D, int DV>
struct Config {
  using TQ = Tile<kRows, D>;   // dQ staging
  using TK = Tile<BN, D>;      // K stages
  using TV = Tile<BN, DV>;     // V stages
  // tensor-memory columns: S, dP, dQ, then Q and dO (two 16-bit elements a column)
  static constexpr int kColS = 0;
  static constexpr int kColDP = BN;
  static constexpr int kColDQ = 2 * BN;
  static constexpr int kColQ = kColDQ + pad32(D);
  static constexpr int kColG = kColQ + pad32(D / 2);
  static constexpr int kTmemCols = kColG + DV / 2;
  static_assert(kTmemCols <= 512, "tensor memory overflow");
  static constexpr int kTmemAlloc = 512;
  static constexpr int kBudget = 227 * 1024 - 2048;  // dynamic limit less alignment slack
  static constexpr int kFixed = TQ::kBytes;
  static constexpr int kStepReserve = 1024;  // smallest step table kept room for (bitmap masks)
  static constexpr int kAvail = kBudget - kFixed - kStepReserve;
  static constexpr int kPairs = kAvail / (TK::kBytes + TV::kBytes);
  static constexpr int NSV = kPairs > 4 ? 4 : kPairs;
  static constexpr int kKFit = (kAvail - NSV * TV::kBytes) / TK::kBytes;
  static constexpr int NSK = kKFit > 4 ? 4 : kKFit;
  static_assert(NSV >= 2 && NSK >= 2, "need two key and two value stages");
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + TQ::kBytes;
  static constexpr int kOffV = kOffK + NSK * TK::kBytes;
  static constexpr int kOffSteps = kOffV + NSV * TV::kBytes;
  // Only a bitmap mask needs the step table; the walk under the other masks is computed.
  static size_t smem_bytes(int n, bool bitmap) {
    return 1024 + kOffSteps + (bitmap ? 4 * static_cast<size_t>((n + BN - 1) / BN) : 0);
  }
};

struct Barriers {
  uint64_t qg_full;  // Q and dO are in tensor memory (one arrival per softmax warp)
  uint64_t st_full;  // the tile's Q, dO and O have arrived in shared memory (TMA bytes)
  uint64_t st_free;  // the softmax warps have read them (one arrival per softmax warp)
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint64_t s_full, s_free, dp_full, ds_full;
  uint64_t dq_done;
  uint32_t tmem_base;
  uint32_t nsteps;
  float dpart[2][kRows];  // per-row partial sums of dO * O over each half of the columns
};

// Stores n consecutive 32-bit columns of this thread's TMEM lane (n = 4, 8, 16 or 32).
template <int N>
__device__ __forceinline__ void st_cols(uint32_t taddr, const uint32_t (&w)[N]) {
  if constexpr (N == 4) {
    tmem_st4(taddr, w);
  } else if constexpr (N == 8) {
    tmem_st8(taddr, w);
  } else if constexpr (N == 16) {
    tmem_st16(taddr, w);
  } else {
    static_assert(N == 32, "4, 8, 16 or 32 columns");
    tmem_st16(taddr, *reinterpret_cast<const uint32_t(*)[16]>(&w[0]));
    tmem_st16(taddr + 16, *reinterpret_cast<const uint32_t(*)[16]>(&w[16]));
  }
}

// kCap: ring depths from the launch (p.ring_k, p.ring_v) instead of the compile-time counts.
template <bool kBf16, int D, int DV, bool kDrop, bool kCap = false>
__global__ void __launch_bounds__(kThreads, 1)
    dq_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                 const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_q,
                 const __grid_constant__ CUtensorMap tm_g, const __grid_constant__ CUtensorMap tm_o,
                 bwd::BwdParams p) {
  using C = Config<D, DV>;
  using TQ = typename C::TQ;
  using TK = typename C::TK;
  using TV = typename C::TV;
  constexpr int NSK = C::NSK;
  constexpr int NSV = C::NSV;
  const auto ring_k = ring_of<kCap, NSK>(p.ring_k);
  const auto ring_v = ring_of<kCap, NSV>(p.ring_v);
  // stages of the V ring in use; the last two hold the tile's dO and O at the start
  const int nv = kCap ? static_cast<int>(p.ring_v.n) : NSV;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = bwd::align1024(smem_raw);
  uint8_t* sQ = smem + C::kOffQ;
  uint8_t* sK = smem + C::kOffK;
  uint8_t* sV = smem + C::kOffV;
  uint32_t* steps = reinterpret_cast<uint32_t*>(smem + C::kOffSteps);
  __shared__ Barriers bars;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int n = p.n;
  // heaviest (causal) query tiles first, by groups of heads (work_item)
  const uint32_t wgroup = p.mask_kind == kMaskCausal ? kCausalHeadGroup : 1u;
  uint32_t wrank, whead;
  work_item(blockIdx.y * gridDim.x + blockIdx.x, gridDim.x, gridDim.y, wgroup, wrank, whead);
  const int bh = static_cast<int>(whead);
  const int tile = static_cast<int>(gridDim.x - 1 - wrank);
  const int row0 = tile * kRows;
  const int nblk = (n + BN - 1) / BN;

  // ---------------------------------------------------------------- prologue
  if (tid == 0) {
    mbar_init(&bars.qg_full, kSoftmaxWarps);
    mbar_init(&bars.st_full, 1);
    mbar_init(&bars.st_free, kSoftmaxWarps);
    for (int s = 0; s < NSK; ++s) {
      mbar_init(&bars.k_full[s], 1);
      mbar_init(&bars.k_empty[s], 1);
    }
    for (int s = 0; s < NSV; ++s) {
      mbar_init(&bars.v_full[s], 1);
      mbar_init(&bars.v_empty[s], 1);
    }
    mbar_init(&bars.s_full, 1);
    mbar_init(&bars.s_free, kSoftmaxWarps);
    mbar_init(&bars.dp_full, 1);
    mbar_init(&bars.ds_full, kSoftmaxWarps);
    mbar_init(&bars.dq_done, 1);
    fence_barrier_init();
  }
  if (warp == kMmaWarp) tmem_alloc(&bars.tmem_base, C::kTmemAlloc);

  // Walk over key blocks.  Under a bitmap mask every block is classified (skip / full /
  // partial) into a table of the blocks the tile takes; otherwise step i is block i, up to the
  // last block the tile's rows reach, and is classified on the fly.
  const bool use_table = p.mask_kind == kMaskBitmap;
  const bool causal = p.mask_kind == kMaskCausal;
  const int last_row = min(row0 + kRows, n) - 1;
  if (use_table) {
    for (int j = tid; j < nblk; j += kThreads) steps[j] = 0;
    __syncthreads();
    if (tid < kRows) {
      const int row = row0 + tid;
      const bool valid = row < n;
      const uint32_t* rowbits = p.mask_bits + static_cast<int64_t>(bh) * p.mask_head_stride_words +
                                static_cast<int64_t>(valid ? row : 0) * p.mask_row_words;
      for (int j = 0; j < nblk; ++j) {
        bool any = false, all = true;
        if (valid) {
#pragma unroll
          for (int q = 0; q < BN / 32; ++q) {
            const int key0 = j * BN + q * 32;
            if (key0 < n) {
              uint32_t w = __ldg(rowbits + key0 / 32);
              const int nk = n - key0;
              const uint32_t live = nk >= 32 ? 0xFFFFFFFFu : ((1u << nk) - 1u);
              w &= live;
              any |= w != 0;
              all &= w == live;
            }
          }
        }
        const bool wany = __any_sync(0xFFFFFFFFu, any);
        const bool wall = __all_sync(0xFFFFFFFFu, all);
        if (lane == 0) {
          const uint32_t bits = (wany ? 1u : 0u) | (wall ? 0u : 2u);
          if (bits) atomicOr(&steps[j], bits);
        }
      }
    }
    __syncthreads();
    if (tid == 0) {
      int ns = 0;
      for (int j = 0; j < nblk; ++j) {
        const uint32_t b = steps[j];
        if (!(b & 1u)) continue;
        const bool tail = (j + 1) * BN > n || row0 + kRows > n;
        const uint32_t cls = ((b & 2u) || tail) ? kPartial : kFull;
        steps[ns++] = static_cast<uint32_t>(j) | (cls << 16);
      }
      bars.nsteps = ns;
    }
  } else if (tid == 0) {
    bars.nsteps = row0 < n ? (causal ? last_row / BN + 1 : nblk) : 0;
  }
  // Step word: key block j | class << 16.
  auto step_at = [&](int i) -> uint32_t {
    if (use_table) return steps[i];
    const bool tail = (i + 1) * BN > n || row0 + kRows > n;
    const bool full = !tail && (!causal || (i + 1) * BN - 1 <= row0);
    return static_cast<uint32_t>(i) | ((full ? kFull : kPartial) << 16);
  };
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const int nsteps = bars.nsteps;
  const uint32_t tmem = bars.tmem_base;

  auto key0_at = [&](int i) { return static_cast<int>(step_at(i) & 0xFFFFu) * BN; };
  if (warp == kKProducerWarp) {
    // ---------------------------------------------------------------- TMA producer: K
    // The CTA launched p.next_cta after this one (one per SM, in launch order) finds the rows
    // its softmax warps load first (Q, dO, O) and its first key block in L2 when it starts.
    if (lane == 0 && p.next_cta > 0) {
      const uint32_t nx = gridDim.x, ny = gridDim.y;
      const uint32_t later = blockIdx.y * nx + blockIdx.x + p.next_cta;
      if (later < nx * ny) {
        uint32_t rank_l, head_l;
        work_item(later, nx, ny, wgroup, rank_l, head_l);
        const int row0_l = (static_cast<int>(nx) - 1 - static_cast<int>(rank_l)) * kRows;
        const int bh_l = static_cast<int>(head_l);
#pragma unroll
        for (int b = 0; b < TK::L::kBoxes; ++b) tma_prefetch_l2_3d(&tm_q, b * TK::L::kBoxCols, row0_l, bh_l);
#pragma unroll
        for (int b = 0; b < TV::L::kBoxes; ++b) tma_prefetch_l2_3d(&tm_g, b * TV::L::kBoxCols, row0_l, bh_l);
#pragma unroll
        for (int b = 0; b < TV::L::kBoxes; ++b) tma_prefetch_l2_3d(&tm_o, b * TV::L::kBoxCols, row0_l, bh_l);
#pragma unroll
        for (int b = 0; b < TK::L::kBoxes; ++b) tma_prefetch_l2_3d(&tm_k, b * TK::L::kBoxCols, 0, bh_l);
#pragma unroll
        for (int b = 0; b < TV::L::kBoxes; ++b) tma_prefetch_l2_3d(&tm_v, b * TV::L::kBoxCols, 0, bh_l);
      }
    }
    if (lane == 0 && nsteps > 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      for (int i = 0; i < nsteps; ++i) {
        const int s = ring_k.stage(i);
        if (!mbar_wait(&bars.k_empty[s], ring_k.parity(i) ^ 1, p.status, 42)) break;
        mbar_arrive_expect_tx(&bars.k_full[s], TK::kBytes);
#pragma unroll
        for (int b = 0; b < TK::L::kBoxes; ++b)
          tma_load_3d(sK + s * TK::kBytes + b * TK::kBoxBytes, &tm_k, &bars.k_full[s],
                      b * TK::L::kBoxCols, key0_at(i), bh);
        if (i + kPrefetch < nsteps) {
          const int kp = key0_at(i + kPrefetch);
#pragma unroll
          for (int b = 0; b < TK::L::kBoxes; ++b) tma_prefetch_l2_3d(&tm_k, b * TK::L::kBoxCols, kp, bh);
#pragma unroll
          for (int b = 0; b < TV::L::kBoxes; ++b) tma_prefetch_l2_3d(&tm_v, b * TV::L::kBoxCols, kp, bh);
        }
      }
    }
  } else if (warp == kVProducerWarp) {
    // ---------------------------------------------------------------- TMA producer: V
    if (lane == 0) {
      // The tile's Q (into the dQ staging slot), dO and O (into the last two V stages) for the
      // softmax warps, which read their rows from there: one bulk copy each instead of every
      // lane loading its own row.
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_g);
      tma_prefetch_desc(&tm_o);
      mbar_arrive_expect_tx(&bars.st_full, TQ::kBytes + 2 * TV::kBytes);
#pragma unroll
      for (int b = 0; b < TQ::L::kBoxes; ++b)
        tma_load_3d(sQ + b * TQ::kBoxBytes, &tm_q, &bars.st_full, b * TQ::L::kBoxCols, row0, bh);
#pragma unroll
      for (int b = 0; b < TV::L::kBoxes; ++b)
        tma_load_3d(sV + (nv - 1) * TV::kBytes + b * TV::kBoxBytes, &tm_g, &bars.st_full,
                    b * TV::L::kBoxCols, row0, bh);
#pragma unroll
      for (int b = 0; b < TV::L::kBoxes; ++b)
        tma_load_3d(sV + (nv - 2) * TV::kBytes + b * TV::kBoxBytes, &tm_o, &bars.st_full,
                    b * TV::L::kBoxCols, row0, bh);
      for (int i = 0; i < nsteps; ++i) {
        const int s = ring_v.stage(i);
        // the last two stages take their first V block once dO and O have been read
        if (i < nv && s >= nv - 2 && !mbar_wait(&bars.st_free, 0, p.status, 52)) break;
        if (!mbar_wait(&bars.v_empty[s], ring_v.parity(i) ^ 1, p.status, 41)) break;
        mbar_arrive_expect_tx(&bars.v_full[s], TV::kBytes);
#pragma unroll
        for (int b = 0; b < TV::L::kBoxes; ++b)
          tma_load_3d(sV + s * TV::kBytes + b * TV::kBoxBytes, &tm_v, &bars.v_full[s],
                      b * TV::L::kBoxCols, key0_at(i), bh);
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA issuer
    // The whole warp runs the loop so that descriptors stay warp-uniform; one elected lane
    // issues.  Operand descriptors are built once per buffer: a 16-element step or a ring
    // stage only adds a constant to the start-address field.
    constexpr uint32_t id_s = idesc_f16(128, BN, kBf16 ? 1 : 0, 0, 0);  // S, dP
    constexpr uint32_t id_q = idesc_f16(128, D, kBf16 ? 1 : 0, 0, 1);   // dQ
    constexpr uint64_t kStage = TK::kBytes >> 4;
    constexpr uint64_t kStageV = TV::kBytes >> 4;
    const uint64_t dk0 = TK::desc_k(smem_u32(sK), 0), dv0 = TV::desc_k(smem_u32(sV), 0);
    const uint64_t dkmn0 = TK::desc_mn(smem_u32(sK), 0);
    bool ok = nsteps == 0 || mbar_wait_warp(&bars.qg_full, 0, p.status, 43);
    auto issue_s = [&](int i) -> bool {
      const int ks = ring_k.stage(i);
      if (!mbar_wait_warp(&bars.k_full[ks], ring_k.parity(i), p.status, 44)) return false;
      tc_fence_after();
      const uint64_t dk = dk0 + static_cast<uint64_t>(ks) * kStage;
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ts(tmem + C::kColS, tmem + C::kColQ + kk * 8, dk + TK::k_step(kk), id_s, kk > 0 ? 1u : 0u);
        mma_commit(&bars.s_full);
      }
      __syncwarp();
      return true;
    };
    auto issue_dp = [&](int i) -> bool {
      const int vs = ring_v.stage(i);
      if (!mbar_wait_warp(&bars.v_full[vs], ring_v.parity(i), p.status, 45)) return false;
      tc_fence_after();
      const uint64_t dv = dv0 + static_cast<uint64_t>(vs) * kStageV;
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < DV / 16; ++kk)
          mma_ts(tmem + C::kColDP, tmem + C::kColG + kk * 8, dv + TV::k_step(kk), id_s,
                 kk > 0 ? 1u : 0u);
        mma_commit(&bars.dp_full);
        mma_commit(&bars.v_empty[vs]);
      }
      __syncwarp();
      return true;
    };
    if (ok && nsteps > 0) ok = issue_s(0) && issue_dp(0);
    for (int i = 0; i < nsteps && ok; ++i) {
      if (i + 1 < nsteps) {
        // S_{i+1} overwrites S_i: wait until every softmax warp has loaded it
        ok = mbar_wait_warp(&bars.s_free, i & 1, p.status, 50);
        if (!ok) break;
        tc_fence_after();
        ok = issue_s(i + 1);
        if (!ok) break;
      }
      ok = mbar_wait_warp(&bars.ds_full, i & 1, p.status, 46);
      if (!ok) break;
      tc_fence_after();
      const int ks = ring_k.stage(i);
      const uint64_t dkmn = dkmn0 + static_cast<uint64_t>(ks) * kStage;
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_ts(tmem + C::kColDQ, tmem + C::kColDP + packed_col(16 * kk), dkmn + TK::mn_step(kk),
                 id_q, (i > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bars.k_empty[ks]);
      }
      __syncwarp();
      // dP_{i+1} overwrites dS_i, which dQ_i (issued before it) has read
      if (i + 1 < nsteps) {
        ok = issue_dp(i + 1);
        if (!ok) break;
      }
    }
    if (elect_one()) mma_commit(&bars.dq_done);
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- softmax: P and dS
    const int quad = warp % 4;
    const int r = quad * 32 + lane;  // query row within the tile = TMEM lane
    const int row = row0 + r;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    constexpr int kHalf = BN / 2;  // key columns of this warp: [c_lo, c_lo + kHalf)
    const int half = (warp - kFirstSoftmaxWarp) / 4;
    const int c_lo = half * kHalf;
    const float sl2 = p.c * 1.4426950408889634f;
    // D_i: this warp sums dO * O over its half of the value columns.  The same dO words, and
    // this half of the row's Q, go into tensor memory as the A operands of dP and S: memory
    // order puts element 2c in the low half of word c, which is the operand layout (two 16-bit
    // elements a column).  The rows come from the tiles staged in shared memory (16-byte reads;
    // rows past n arrive as zeros).
    float dpar = 0.0f;
    bool ok = mbar_wait_spin(&bars.st_full, 0, p.status, 51);
    {
      constexpr int kGW = DV / 4;  // dO columns of this half
      constexpr int kQW = D / 4;   // Q columns of this half
      uint32_t gcol[kGW], qcol[kQW];
      const uint8_t* sG = sV + (nv - 1) * TV::kBytes;
      const uint8_t* sO = sV + (nv - 2) * TV::kBytes;
#pragma unroll
      for (int v = 0; v < DV / 16; ++v) {
        const int c = half * (DV / 2) + 8 * v;
        const uint4 a = *reinterpret_cast<const uint4*>(sO + TV::offset(r, c));
        const uint4 g = *reinterpret_cast<const uint4*>(sG + TV::offset(r, c));
        const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float a0, a1, g0, g1;
          unpack2<kBf16>(aw[e], a0, a1);
          unpack2<kBf16>(gw[e], g0, g1);
          dpar = fmaf(a0, g0, dpar);
          dpar = fmaf(a1, g1, dpar);
          gcol[4 * v + e] = gw[e];
        }
      }
#pragma unroll
      for (int v = 0; v < D / 16; ++v) {
        const uint4 q = *reinterpret_cast<const uint4*>(sQ + TQ::offset(r, half * (D / 2) + 8 * v));
        qcol[4 * v] = q.x;
        qcol[4 * v + 1] = q.y;
        qcol[4 * v + 2] = q.z;
        qcol[4 * v + 3] = q.w;
      }
      // dO and O are read: their V stages may take V blocks
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.st_free);
      st_cols<kQW>(tmem + lane_off + C::kColQ + half * kQW, qcol);
      st_cols<kGW>(tmem + lane_off + C::kColG + half * kGW, gcol);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.qg_full);
    }
    bars.dpart[half][r] = dpar;
    bwd::named_barrier(3, kSoftmaxWarps * 32);
    const float dd = row < n ? bars.dpart[0][r] + bars.dpart[1][r] : 0.0f;
    // rows past n or with no allowed key carry +inf here, so their probabilities are 0
    float lse_l2 = INFINITY;
    if (row < n) {
      const float lv = __ldg(p.lse + static_cast<int64_t>(bh) * n + row);
      if (lv != -INFINITY) lse_l2 = lv * 1.4426950408889634f;
    }
    if (half == 0) {  // this tile's rows of the table, padded rows included
      p.L2[static_cast<int64_t>(bh) * p.n_pad + row] = lse_l2;
      p.Dv[static_cast<int64_t>(bh) * p.n_pad + row] = dd;
    }
    const uint32_t* rowbits =
        p.mask_kind == kMaskBitmap
            ? p.mask_bits + static_cast<int64_t>(bh) * p.mask_head_stride_words +
                  static_cast<int64_t>(row < n ? row : 0) * p.mask_row_words
            : nullptr;
    for (int i = 0; i < nsteps && ok; ++i) {
      const uint32_t sw = step_at(i);
      const int key0 = static_cast<int>(sw & 0xFFFFu) * BN;
      const bool partial = ((sw >> 16) & 3u) == kPartial;
      uint32_t mword[kHalf / 32];
      if (partial && p.mask_kind == kMaskBitmap) {
#pragma unroll
        for (int q = 0; q < kHalf / 32; ++q) {
          const int kq = key0 + c_lo + q * 32;
          uint32_t w = (row < n && kq < n) ? __ldg(rowbits + kq / 32) : 0u;
          const int nk = n - kq;
          if (nk < 32) w &= nk > 0 ? (1u << nk) - 1u : 0u;
          mword[q] = w;
        }
      }
      ok = mbar_wait_spin(&bars.s_full, i & 1, p.status, 47);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tS = tmem + C::kColS + lane_off;
      const uint32_t tP = tmem + C::kColDP + lane_off;
      uint32_t pkeep[kHalf / 2];  // this warp's P pairs, kept for the dS pass
      // both 32-column chunks are loaded before one wait: the load latency is paid once
      uint32_t rr[kHalf / 32][32];
#pragma unroll
      for (int h = 0; h < kHalf / 32; ++h) tmem_ld32(tS + c_lo + 32 * h, rr[h]);
      tmem_wait_ld();
      // S is in registers: the tensor core may overwrite it with S_{i+1}
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.s_free);
#pragma unroll
      for (int cc = 0; cc < kHalf; cc += 32) {
        const int c0 = c_lo + cc;
        float pv[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) pv[k] = ex2(__uint_as_float(rr[cc / 32][k]) * sl2 - lse_l2);
        if (partial) {
          if (p.mask_kind == kMaskBitmap) {
            const uint32_t w = mword[cc / 32];
#pragma unroll
            for (int k = 0; k < 32; ++k)
              if (!((w >> k) & 1u)) pv[k] = 0.0f;
          } else {
            const bool causal = p.mask_kind == kMaskCausal;
#pragma unroll
            for (int k = 0; k < 32; ++k) {
              const int key = key0 + c0 + k;
              if (key >= n || (causal && key > row)) pv[k] = 0.0f;
            }
          }
        }
#pragma unroll
        for (int k = 0; k < 16; ++k) pkeep[cc / 2 + k] = pack2<kBf16>(pv[2 * k], pv[2 * k + 1]);
      }
      // Dropout: keep bits of this row with the warp's key columns (bit k of word h <-> key
      // key0 + c_lo + 32 h + k), drawn before the wait for dP.
      uint32_t kbits[kDrop ? kHalf / 32 : 1];
      if constexpr (kDrop) {
        // one generator call per 4 x 4 patch: lane s of each group of four (rows 4 r ..) draws
        // the patches of keys key0 + c_lo + 16 s .. + 15
        uint32_t part[4];
        keep_rows<kHalf / 16>(p.drop, static_cast<uint32_t>(row) >> 2,
                              static_cast<uint32_t>(key0 + c_lo) >> 2,
                              (static_cast<uint32_t>(key0 + c_lo) >> 2) + kHalf / 8, bh, part);
#pragma unroll
        for (int h = 0; h < kHalf / 32; ++h) kbits[h] = 0u;
#pragma unroll
        for (int s = 0; s < 4; ++s) kbits[(s * kHalf / 4) / 32] |= part[s] << ((s * kHalf / 4) % 32);
      }
      ok = mbar_wait_spin(&bars.dp_full, i & 1, p.status, 48);
      if (!ok) break;
      tc_fence_after();
      uint32_t dp[kHalf / 32][32];
#pragma unroll
      for (int h = 0; h < kHalf / 32; ++h) tmem_ld32(tP + c_lo + 32 * h, dp[h]);
      tmem_wait_ld();
#pragma unroll
      for (int cc = 0; cc < kHalf; cc += 32) {
        const int c0 = c_lo + cc;
        uint32_t pk[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          float p0, p1;
          unpack2<kBf16>(pkeep[cc / 2 + k], p0, p1);
          float d0 = __uint_as_float(dp[cc / 32][2 * k]);
          float d1 = __uint_as_float(dp[cc / 32][2 * k + 1]);
          if constexpr (kDrop) {
            const uint32_t kb = kbits[cc / 32] >> (2 * k);
            d0 = kb & 1u ? d0 * p.drop.scale : 0.0f;
            d1 = kb & 2u ? d1 * p.drop.scale : 0.0f;
          }
          pk[k] = pack2<kBf16>(p0 * (d0 - dd), p1 * (d1 - dd));
        }
        tmem_st16(tP + packed_col(c0), pk);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.ds_full);
    }
    // ---------------------------------------------------------------- epilogue
    // dQ = c * (dS K) rounded and stored through the (now idle) Q tile: each half of the warps
    // stages half of the columns (half 0 all of them when a half would be narrower than 16).
    constexpr int kSplit = D / 2 >= 16 ? 2 : 1;
    constexpr int kWq = D / kSplit;
    if (ok && nsteps > 0) ok = mbar_wait_spin(&bars.dq_done, 0, p.status, 49);
    tc_fence_after();
    if (ok && half < kSplit)
      bwd::stage_acc<kBf16, TQ, kWq>(tmem + C::kColDQ + lane_off + half * kWq, p.c, sQ, r,
                                     half * kWq, nsteps > 0);
    fence_proxy_async_smem();
    bwd::named_barrier(2, kSoftmaxWarps * 32);
    if (ok && half == 0 && r == 0) {
#pragma unroll
      for (int b = 0; b < TQ::L::kBoxes; ++b)
        tma_store_3d(&tm_dq, sQ + b * TQ::kBoxBytes, b * TQ::L::kBoxCols, row0, bh);
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

}  // namespace dq
}  // namespace ea
