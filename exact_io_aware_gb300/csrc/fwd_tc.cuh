// Forward pass of exact tiled softmax attention on the tcgen05 tensor cores (fp16 / bf16).
//
// Follows the tiled forward procedure of "Exact tiled attention and memory-aware
// differentiation": key blocks J_t are visited in order, blocks with no allowed key are
// skipped, each query row keeps the summary (m, l, z) and merges every new block into it,
// and at the end O_i = z_i / l_i.  Retained statistic: LSE_i = m_i + ln l_i.
//
// One CTA owns two tiles of 128 query rows of one head (256 rows).  Roles:
//   warp  0    MMA issuer for tile 0 (one elected lane); allocates tensor memory
//   warp  1    MMA issuer for tile 1
//   warps 2-5  softmax for tile 0   (thread = query row = TMEM lane of the warp's quadrant)
//   warps 6-9  softmax for tile 1
//   warp  10   TMA producer: Q tiles once, then K and V blocks through two rings (NSK and
//              NSV stages); K runs one block ahead of V, and (full query tiles only) blocks
//              kPrefetch steps ahead are requested into L2 so that the ring loads find them
// Tensor memory: S_t = Q_t K_jᵀ (BN fp32 columns per tile; the 16-bit P_t is written over
// the first BN/2 of them) and O_t, the unnormalised weighted value sum z (DV columns per tile,
// DV the value width).
// Each tile's MMA warp issues, per key block j, PV_{j-1} then S_j for its tile, so the tensor
// core works on one tile while the other tile's softmax runs.  One issuer per tile keeps a
// tile's waits (its softmax, the next K block) off the other tile's issue path: the tensor
// core accepts only a few MMAs ahead, so an issuer spends most of its time blocked in issue.
// The issuers have the lowest warp slots, which the warp schedulers favour over the
// softmax warps they share a sub-partition with.
//
// Query and key lengths may differ (a key/value cache): p.n query rows against p.nk keys, and
// under the causal mask query i sees keys j <= i + p.off (off = nk - n: the queries are the
// last rows of the sequence).  With n = nk this is ordinary causal attention.
//
// Key split (gridDim.z > 1): the pair's key blocks are cut into gridDim.z contiguous shares and
// CTA z walks share z only.  It writes its rows' summary of that share in normalised form,
// O_z = z/l (float32) and LSE_z = m + ln l (-inf for a row with no allowed key in the share),
// which a merge kernel combines by the merge rule of the stable summaries.
//
// Dropout (kDrop): the realised mask of dropout.cuh zeroes dropped probabilities on their way
// into P (the row sum l keeps every probability), and the factor 1/(1-p) is applied to O in
// the epilogue, so the 16-bit P never exceeds the range it has without dropout.
//
// Online softmax (the running-maximum recurrence of "The Arithmetic of Intelligence",
// chapter 12): scores are taken to base 2 with the folded factor c·log2(e) (the exp2
// prescale described in "Bellek Duvarının Fiziği", online softmax section).  The running
// maximum m is raised only when a block's maximum exceeds it by more than kLazy (2^8), and
// then l and z are multiplied by e^{m-m'}; otherwise the stale m is kept and probabilities
// up to 2^8 enter P.  The final z / l and m + log2 l are unchanged by this (a common shift of
// every score cancels in z / l), and 2^8 stays far inside the fp16 range.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.h"
#include "tile.cuh"

namespace ea {
namespace fwd {

constexpr int kRowsPerTile = 128;
constexpr int kThreads = 352;
constexpr int kSoftmaxThreads = 256;
constexpr int kFirstSoftmaxWarp = 2;
constexpr int kProducerWarp = 10;
constexpr float kLazy = 8.0f;  // log2 units
// Of every four exponentials of the softmax loop, kFmaExp are computed on the FMA pipe
// (ex2_fma) and the rest on the MUFU unit.  Measured at B 8, H 16, n 4096, d 128: 0.748 ms with
// none, 0.84 ms with one in four, 1.14 ms with two: the loop is bound by issue and ALU work, not
// by the MUFU unit, so every exponential stays on MUFU.
constexpr int kFmaExp = 0;
constexpr uint32_t kSkip = 0, kFull = 1, kPartial = 2;

// Opt-in dynamic shared memory per CTA on sm_103a (227 KiB) less the kernel's static barrier
// block.
constexpr int kMaxDynSmem = 227 * 1024 - 1024;
// Key blocks requested into L2 ahead of the ring loads when the CTA's query tiles are full
// (compute-bound).  With a few query rows (decoding over a key/value cache) the CTA streams
// K and V at the HBM rate, and the early requests cost re-reads from DRAM (measured: reads
// 1.235x the K/V bytes with them, 1.000x without, and 22 % less time), so the launcher sets
// the distance to 0 there.
constexpr int kPrefetch = 4;

// D: width of Q and K rows; DV: width of V and O rows (the value width v, equal to D unless
// the caller's values are wider or narrower than its keys).
template <int D, int DV, int BN>
struct Config {
  using TQ = Tile<kRowsPerTile, D>;
  using TK = Tile<BN, D>;
  using TV = Tile<BN, DV>;
  using TO = Tile<kRowsPerTile, DV>;  // O staging, in the tile's Q slot
  static constexpr int kQSlot = TQ::kBytes > TO::kBytes ? TQ::kBytes : TO::kBytes;
  static constexpr int kSmemBudget = kMaxDynSmem - 1024;  // minus the 1024-byte alignment slack
  static constexpr int kFixed = 2 * kQSlot;
  static constexpr int kStepReserve = 1024;  // smallest step table kept room for (bitmap masks)
  static constexpr int kAvail = kSmemBudget - kFixed - kStepReserve;
  // V is consumed one step after K, so K takes the odd slot: its loads are the ones a step waits on.
  static constexpr int kPairs = kAvail / (TK::kBytes + TV::kBytes);
  static constexpr int NSV = kPairs > 4 ? 4 : kPairs;
  static constexpr int kKFit = (kAvail - NSV * TV::kBytes) / TK::kBytes;
  static constexpr int NSK = kKFit > 4 ? 4 : kKFit;
  static_assert(NSV >= 2 && NSK >= 2, "need at least two pipeline stages");
  static constexpr int kTmemCols = 2 * BN + 2 * DV;
  static constexpr int kTmemAlloc = kTmemCols <= 32    ? 32
                                    : kTmemCols <= 64  ? 64
                                    : kTmemCols <= 128 ? 128
                                    : kTmemCols <= 256 ? 256
                                                       : 512;
  static_assert(kTmemCols <= 512, "tensor memory overflow");
  // dynamic shared memory layout (offsets from a 1024-aligned base)
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + 2 * kQSlot;
  static constexpr int kOffV = kOffK + NSK * TK::kBytes;
  static constexpr int kOffSteps = kOffV + NSV * TV::kBytes;
  // Only a bitmap mask needs the step table (one word per key block); the walk under the
  // other masks is computed on the fly.
  static size_t smem_bytes(int n, int mask_kind) {
    const size_t nblk = (static_cast<size_t>(n) + BN - 1) / BN;
    return 1024 + kOffSteps + (mask_kind == kMaskBitmap ? 4 * nblk : 0);
  }
};

struct Barriers {
  uint64_t q_full[2];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_done[2];
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint32_t tmem_base;
  uint32_t nsteps;
  uint32_t act;  // bit t: tile t takes part in some step
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ void named_barrier(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Step word of the walk under no mask or the causal mask: key block j, and for each of the two
// query tiles (rows r0 .. r0 + 127 of the pair; rows from n on do not exist) whether it skips
// the block, takes it whole or needs the mask pass (causal diagonal or the ragged key tail).
// Same encoding as the bitmap table: j | cls0 << 16 | cls1 << 18.
__device__ __forceinline__ uint32_t dense_step(int j, int BN, int nblk, int n, int nk, int off,
                                               int pair_row0, bool causal) {
  uint32_t w = static_cast<uint32_t>(j);
  const bool tail_blk = (nk % BN) != 0 && j == nblk - 1;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int r0 = pair_row0 + t * kRowsPerTile;
    if (r0 >= n) continue;
    const int last_row = min(r0 + kRowsPerTile, n) - 1;
    const bool any = !causal || j * BN <= last_row + off;
    const bool all = !causal || (j + 1) * BN - 1 <= r0 + off;
    const uint32_t cls = any ? ((all && !tail_blk) ? kFull : kPartial) : kSkip;
    w |= cls << (16 + 2 * t);
  }
  return w;
}

// kCap: ring depths from the launch (p.ring_k, p.ring_v) instead of the compile-time counts.
template <bool kBf16, int D, int DV, int BN, bool kDrop, bool kCap = false>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                  FwdParams p) {
  using C = Config<D, DV, BN>;
  using TQ = typename C::TQ;
  using TK = typename C::TK;
  using TV = typename C::TV;
  using TO = typename C::TO;
  constexpr int NSK = C::NSK;
  constexpr int NSV = C::NSV;
  const auto ring_k = ring_of<kCap, NSK>(p.ring_k);
  const auto ring_v = ring_of<kCap, NSV>(p.ring_v);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sQ = smem + C::kOffQ;
  uint8_t* sK = smem + C::kOffK;
  uint8_t* sV = smem + C::kOffV;
  uint32_t* steps = reinterpret_cast<uint32_t*>(smem + C::kOffSteps);
  __shared__ Barriers bars;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int n = p.n;    // query rows
  const int nk = p.nk;  // keys
  const int off = p.off;
  const int bh = blockIdx.y;
  const int pair = (gridDim.x - 1 - blockIdx.x);  // heaviest (causal) query tiles first
  // tile t starts at pair_row0 + 128 t; with p.rows_cta = 128 (grids that would fill at most half
  // the multiprocessors) a CTA owns one tile and tile 1 has no rows
  const int pair_row0 = pair * p.rows_cta;
  const int nrow = min(n, pair_row0 + p.rows_cta);  // end of this CTA's rows
  const int nblk = (nk + BN - 1) / BN;
  const int split = blockIdx.z;
  const int nsplit = gridDim.z;
  const bool partial_out = p.o_part != nullptr;

  // ---------------------------------------------------------------- prologue
  if (tid == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars.q_full[t], 1);
      mbar_init(&bars.s_full[t], 1);
      mbar_init(&bars.p_full[t], 4);
      mbar_init(&bars.o_done[t], 1);
    }
    for (int s = 0; s < NSK; ++s) mbar_init(&bars.k_full[s], 1);
    for (int s = 0; s < NSV; ++s) mbar_init(&bars.v_full[s], 1);
  }
  if (warp == 0) tmem_alloc(&bars.tmem_base, C::kTmemAlloc);

  // Walk over key blocks.  Under a bitmap mask every block of this CTA's share is classified
  // for both tiles (skip / full / partial) into a table of the blocks some tile takes;
  // otherwise step i is block j_lo + i, up to the last block of the share.
  const bool use_table = p.mask_kind == kMaskBitmap;
  const bool causal = p.mask_kind == kMaskCausal;
  const int pair_last = nrow - 1;  // last row of the CTA
  const int last_key = pair_last + off;  // causal: the last key the pair's rows see
  const int reach = use_table ? nblk : (causal ? (last_key < 0 ? 0 : last_key / BN + 1) : nblk);
  const int share = (reach + nsplit - 1) / nsplit;
  const int j_lo = min(split * share, reach);
  const int j_hi = min(j_lo + share, reach);
  if (use_table) {
    for (int j = tid; j < nblk; j += kThreads) steps[j] = 0;
    __syncthreads();
    if (tid < kSoftmaxThreads) {
      const int t = tid / kRowsPerTile;
      const int row = pair_row0 + t * kRowsPerTile + (tid % kRowsPerTile);
      const bool valid = row < nrow;
      const uint32_t* rowbits =
          p.mask_bits + static_cast<int64_t>(bh) * p.mask_head_stride_words +
          static_cast<int64_t>(valid ? row : 0) * p.mask_row_words;
      for (int j = j_lo; j < j_hi; ++j) {
        bool any = false, all = true;
        if (valid) {
#pragma unroll
          for (int q = 0; q < BN / 32; ++q) {
            const int key0 = j * BN + q * 32;
            if (key0 < nk) {
              uint32_t w = __ldg(rowbits + key0 / 32);
              const int left = nk - key0;
              const uint32_t live = left >= 32 ? 0xFFFFFFFFu : ((1u << left) - 1u);
              w &= live;
              any |= w != 0;
              all &= w == live;
            }
          }
        }
        const bool wany = __any_sync(0xFFFFFFFFu, any);
        const bool wall = __all_sync(0xFFFFFFFFu, all);
        if (lane == 0) {
          uint32_t bits = (wany ? (1u << t) : 0u) | (wall ? 0u : (4u << t));
          if (bits) atomicOr(&steps[j], bits);
        }
      }
    }
    __syncthreads();
    if (warp == 0) {
      // compaction in place by one warp, 32 blocks a round: a taken block's entry goes to the
      // count of taken blocks before it, never past its own index
      const bool tail = (nk % BN) != 0;
      int ns = 0;
      uint32_t act = 0;
      for (int j0 = j_lo; j0 < j_hi; j0 += 32) {
        const int j = j0 + lane;
        const uint32_t b = j < j_hi ? steps[j] : 0u;
        const bool part_tail = tail && j == nblk - 1;
        const uint32_t cls0 = (b & 1u) ? (((b & 4u) || part_tail) ? kPartial : kFull) : kSkip;
        const uint32_t cls1 = (b & 2u) ? (((b & 8u) || part_tail) ? kPartial : kFull) : kSkip;
        const bool take = (cls0 | cls1) != 0u;
        const uint32_t ballot = __ballot_sync(0xFFFFFFFFu, take);
        __syncwarp();
        if (take)
          steps[ns + __popc(ballot & ((1u << lane) - 1u))] =
              static_cast<uint32_t>(j) | (cls0 << 16) | (cls1 << 18);
        __syncwarp();
        ns += __popc(ballot);
        act |= (cls0 ? 1u : 0u) | (cls1 ? 2u : 0u);
      }
      act = __reduce_or_sync(0xFFFFFFFFu, act);
      if (lane == 0) {
        bars.nsteps = ns;
        bars.act = act;
      }
    }
  } else if (tid == 0) {
    bars.nsteps = j_hi - j_lo;
    // a tile with rows takes every block of the share up to the last one its rows reach
    uint32_t act = 0;
    for (int t = 0; t < 2; ++t) {
      const int r0 = pair_row0 + t * kRowsPerTile;
      if (r0 >= nrow || j_lo >= j_hi) continue;
      const int tile_last_key = min(r0 + kRowsPerTile, nrow) - 1 + off;
      if (causal && tile_last_key < 0) continue;  // no row of the tile sees a key
      const int last_blk = causal ? tile_last_key / BN : nblk - 1;
      if (j_lo <= last_blk) act |= 1u << t;
    }
    bars.act = act;
  }
  if (tid == 0) {
    // A ring stage is free once the MMA warp of every active tile has released it.
    const uint32_t a = bars.act;
    const uint32_t issuers = (a & 1u) + ((a >> 1) & 1u);
    for (int s = 0; s < NSK; ++s) mbar_init(&bars.k_empty[s], issuers ? issuers : 1u);
    for (int s = 0; s < NSV; ++s) mbar_init(&bars.v_empty[s], issuers ? issuers : 1u);
    fence_barrier_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const int nsteps = bars.nsteps;
  const uint32_t tmem = bars.tmem_base;
  const uint32_t act = bars.act;
  // tensor memory: S_t at tmem + t*BN, O_t at tmem + 2*BN + t*DV
  auto step_at = [&](int i) -> uint32_t {
    return use_table ? steps[i] : dense_step(j_lo + i, BN, nblk, nrow, nk, off, pair_row0, causal);
  };

  if (warp == kProducerWarp) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        if (!((act >> t) & 1u)) continue;
        mbar_arrive_expect_tx(&bars.q_full[t], TQ::kBytes);
#pragma unroll
        for (int b = 0; b < TQ::L::kBoxes; ++b)
          tma_load_3d(sQ + t * C::kQSlot + b * TQ::kBoxBytes, &tm_q, &bars.q_full[t],
                      b * TQ::L::kBoxCols, pair_row0 + t * kRowsPerTile, bh);
      }
      // The CTA launched p.next_cta after this one (CTAs start in launch order, one per SM)
      // finds its query tiles in L2: a fresh CTA's first loads come from DRAM at its share of
      // the HBM bandwidth, which would otherwise hold it ~3 us before its first product.
      if (p.next_cta > 0) {
        const uint32_t nx = gridDim.x, ny = gridDim.y;
        const uint32_t later = (blockIdx.z * ny + blockIdx.y) * nx + blockIdx.x + p.next_cta;
        if (later < nx * ny * gridDim.z) {
          const int row_l = (static_cast<int>(nx) - 1 - static_cast<int>(later % nx)) * p.rows_cta;
          const int bh_l = static_cast<int>((later / nx) % ny);
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const int r0 = row_l + t * kRowsPerTile;
            if (r0 >= n || r0 >= row_l + p.rows_cta) continue;
#pragma unroll
            for (int b = 0; b < TQ::L::kBoxes; ++b)
              tma_prefetch_l2_3d(&tm_q, b * TQ::L::kBoxCols, r0, bh_l);
          }
        }
      }
      // Ring loads in the order K_0, K_1, V_0, K_2, V_1, ...: K, which the next step waits
      // on first, stays one block ahead of V.
      auto key0_at = [&](int i) { return static_cast<int>(step_at(i) & 0xFFFFu) * BN; };
      auto load_k = [&](int i) -> bool {
        const int s = ring_k.stage(i);
        if (!mbar_wait(&bars.k_empty[s], ring_k.parity(i) ^ 1, p.status, 1)) return false;
        const int key0 = key0_at(i);
        mbar_arrive_expect_tx(&bars.k_full[s], TK::kBytes);
#pragma unroll
        for (int b = 0; b < TK::L::kBoxes; ++b)
          tma_load_3d(sK + s * TK::kBytes + b * TK::kBoxBytes, &tm_k, &bars.k_full[s],
                      b * TK::L::kBoxCols, key0, bh);
        if (p.prefetch > 0 && i + p.prefetch < nsteps) {
          const int kp = key0_at(i + p.prefetch);
#pragma unroll
          for (int b = 0; b < TK::L::kBoxes; ++b) tma_prefetch_l2_3d(&tm_k, b * TK::L::kBoxCols, kp, bh);
#pragma unroll
          for (int b = 0; b < TV::L::kBoxes; ++b) tma_prefetch_l2_3d(&tm_v, b * TV::L::kBoxCols, kp, bh);
        }
        return true;
      };
      auto load_v = [&](int i) -> bool {
        const int s = ring_v.stage(i);
        if (!mbar_wait(&bars.v_empty[s], ring_v.parity(i) ^ 1, p.status, 2)) return false;
        const int key0 = key0_at(i);
        mbar_arrive_expect_tx(&bars.v_full[s], TV::kBytes);
#pragma unroll
        for (int b = 0; b < TV::L::kBoxes; ++b)
          tma_load_3d(sV + s * TV::kBytes + b * TV::kBoxBytes, &tm_v, &bars.v_full[s],
                      b * TV::L::kBoxCols, key0, bh);
        return true;
      };
      if (nsteps > 0 && load_k(0)) {
        for (int i = 0; i < nsteps; ++i) {
          if (i + 1 < nsteps && !load_k(i + 1)) break;
          if (!load_v(i)) break;
        }
      }
    }
  } else if (warp < kFirstSoftmaxWarp) {
    // ---------------------------------------------------------------- MMA issuer (tile t)
    // Per step i: PV_{i-1} (once this tile's P_{i-1} is in tensor memory), then S_i if the tile
    // takes block i.  PV_{i-1} reads P_{i-1} before S_i overwrites it (one thread's MMAs run in
    // issue order).  Every step releases its K stage and the previous step's V stage, whether
    // or not this tile used them, after waiting for the loads (which keeps each release in the
    // stage's current phase).  The whole warp runs the loop so that descriptors stay
    // warp-uniform; one elected lane issues.  Operand descriptors are built once per buffer: a
    // 16-element step or a ring stage only adds a constant to the start-address field.
    const int t = warp;
    constexpr uint32_t id_s = idesc_f16(128, BN, kBf16 ? 1 : 0, 0, 0);
    constexpr uint32_t id_o = idesc_f16(128, DV, kBf16 ? 1 : 0, 0, 1);
    constexpr uint64_t kStageK = TK::kBytes >> 4;
    constexpr uint64_t kStageV = TV::kBytes >> 4;
    const uint64_t dq = TQ::desc_k(smem_u32(sQ + t * C::kQSlot), 0);
    const uint64_t dk0 = TK::desc_k(smem_u32(sK), 0);
    const uint64_t dv0 = TV::desc_mn(smem_u32(sV), 0);
    const uint32_t tS = tmem + t * BN;
    const uint32_t tO = tmem + 2 * BN + t * DV;
    bool ok = (act >> t) & 1u;
    if (ok) ok = mbar_wait_warp(&bars.q_full[t], 0, p.status, 3);
    bool pend = false;     // this tile took part in the previous step (PV owed)
    bool started = false;  // O_t already holds a partial sum
    uint32_t pph = 0;      // parity of the next p_full[t] phase
    for (int i = 0; i <= nsteps && ok; ++i) {
      const int prev = i - 1;
      if (prev >= 0) {
        ok = mbar_wait_warp(&bars.v_full[ring_v.stage(prev)], ring_v.parity(prev), p.status, 5);
        if (!ok) break;
      }
      const bool cur = i < nsteps && ((step_at(i) >> (16 + 2 * t)) & 3u) != 0;
      const int s = ring_k.stage(i);
      if (i < nsteps) {
        ok = mbar_wait_warp(&bars.k_full[s], ring_k.parity(i), p.status, 6);
        if (!ok) break;
      }
      tc_fence_after();
      if (pend) {
        ok = mbar_wait_warp(&bars.p_full[t], pph, p.status, 4);
        if (!ok) break;
        pph ^= 1u;
        tc_fence_after();
        const uint64_t dv = dv0 + static_cast<uint64_t>(ring_v.stage(prev)) * kStageV;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_ts(tO, tS + kk * 8, dv + TV::mn_step(kk), id_o, (started || kk > 0) ? 1u : 0u);
        }
        __syncwarp();
        started = true;
      }
      if (cur) {
        const uint64_t dk = dk0 + static_cast<uint64_t>(s) * kStageK;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(tS, dq + TQ::k_step(kk), dk + TK::k_step(kk), id_s, kk > 0 ? 1u : 0u);
          mma_commit(&bars.s_full[t]);
        }
        __syncwarp();
      }
      if (elect_one()) {
        if (i < nsteps) mma_commit(&bars.k_empty[s]);
        if (prev >= 0) mma_commit(&bars.v_empty[ring_v.stage(prev)]);
      }
      __syncwarp();
      pend = cur;
    }
    if (ok && elect_one()) mma_commit(&bars.o_done[t]);
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- softmax (tile t)
    const int t = (warp - kFirstSoftmaxWarp) / 4;
    const int quad = warp % 4;  // TMEM lane quadrant this warp may access
    const int r = quad * 32 + lane;
    const int row = pair_row0 + t * kRowsPerTile + r;
    const uint32_t tS = tmem + t * BN;
    const uint32_t tO = tmem + 2 * BN + t * DV;
    const bool active = (act >> t) & 1u;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    // The scale c·log2(e) is folded into the exponent's FFMA, so the raw scores are reduced:
    // their maximum for c > 0, their minimum for c < 0; c = 0 is run as the smallest normal
    // positive scale, which leaves every finite score's exponent at zero (all weights equal).
    const float sl2_raw = p.c * 1.4426950408889634f;
    const float sl2 = sl2_raw == 0.0f ? 1.17549435e-38f : sl2_raw;
    const bool pos = sl2 > 0.0f;
    const float mv = pos ? -INFINITY : INFINITY;  // raw value of a masked score
    float m = -INFINITY;  // running maximum, log2 units (possibly stale by < kLazy)
    float l = 0.0f;       // running normaliser relative to m
    uint32_t s_phase = 0;
    bool first = true;
    bool ok = true;  // false once a bounded wait gave up; an inactive tile skips every step
    const uint32_t* rowbits =
        p.mask_kind == kMaskBitmap
            ? p.mask_bits + static_cast<int64_t>(bh) * p.mask_head_stride_words +
                  static_cast<int64_t>(row < nrow ? row : 0) * p.mask_row_words
            : nullptr;
    for (int i = 0; i < nsteps && ok; ++i) {
      const uint32_t sw = step_at(i);
      const uint32_t cls = (sw >> (16 + 2 * t)) & 3u;
      if (cls == kSkip) continue;
      const int key0 = static_cast<int>(sw & 0xFFFFu) * BN;
      // Dropout: the block's keep bits (bit k of word q <-> key key0 + 32 q + k) are drawn
      // while the scores are still being computed; the exponential loop only tests them.
      uint32_t kbits[kDrop ? BN / 32 : 1];
      if constexpr (kDrop) {
        // rows 4 r .. 4 r + 3 are lanes 4 a .. 4 a + 3 (the warp's rows start at a multiple of
        // 32); lane s of such a group draws the generator calls of keys key0 + s BN / 4 ..
        uint32_t part[4];
        keep_rows<BN / 16>(p.drop, static_cast<uint32_t>(row) >> 2, static_cast<uint32_t>(key0) >> 2,
                           (static_cast<uint32_t>(key0) >> 2) + BN / 8, bh, part);
#pragma unroll
        for (int q = 0; q < BN / 32; ++q) kbits[q] = 0u;
#pragma unroll
        for (int s = 0; s < 4; ++s) kbits[(s * BN / 4) / 32] |= part[s] << ((s * BN / 4) % 32);
      }
      // Masking (partial blocks only): the block's allowed-key words (bit k of word q <-> key
      // key0 + 32 q + k), formed while the scores are still being computed and applied to the
      // scores in registers below.
      uint32_t mw[BN / 32];
      if (__builtin_expect(cls == kPartial, 0)) {
#pragma unroll
        for (int q = 0; q < BN / 32; ++q) {
          const int kq = key0 + q * 32;
          uint32_t w;
          if (p.mask_kind == kMaskBitmap) {
            w = (row < nrow && kq < nk) ? __ldg(rowbits + kq / 32) : 0u;
            const int left = nk - kq;
            if (left < 32) w &= left > 0 ? (1u << left) - 1u : 0u;
          } else {
            // allowed keys kq .. lim: lim = min(row + off, nk - 1) (causal) or nk - 1 (key tail)
            const int lim = p.mask_kind == kMaskCausal ? min(row + off, nk - 1) : nk - 1;
            const int cnt = min(max(lim - kq + 1, 0), 32);
            w = cnt >= 32 ? 0xFFFFFFFFu : ((1u << cnt) - 1u);
          }
          mw[q] = w;
        }
      }
      ok = mbar_wait(&bars.s_full[t], s_phase, p.status, 8);
      if (!ok) break;
      s_phase ^= 1;
      tc_fence_after();
      // All TMEM loads first, one wait: the row's BN raw scores land in registers.
      float sv[BN];
      {
        uint32_t rr[BN];
#pragma unroll
        for (int c0 = 0; c0 < BN; c0 += 32)
          tmem_ld32(tS + lane_off + c0, *reinterpret_cast<uint32_t(*)[32]>(rr + c0));
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < BN; ++k) sv[k] = __uint_as_float(rr[k]);
      }
      // masked entries take the raw value whose scaled image is -inf
      if (__builtin_expect(cls == kPartial, 0)) {
#pragma unroll
        for (int k = 0; k < BN; ++k)
          if (!((mw[k / 32] >> (k % 32)) & 1u)) sv[k] = mv;
      }
      // Row extreme of the raw scores with four independent accumulators (short chains).
      float a0 = mv, a1 = mv, a2 = mv, a3 = mv;
      if (pos) {
#pragma unroll
        for (int k = 0; k < BN; k += 8) {
          a0 = fmax3(a0, sv[k], sv[k + 1]);
          a1 = fmax3(a1, sv[k + 2], sv[k + 3]);
          a2 = fmax3(a2, sv[k + 4], sv[k + 5]);
          a3 = fmax3(a3, sv[k + 6], sv[k + 7]);
        }
        a0 = fmax3(a0, a1, fmaxf(a2, a3));
      } else {
#pragma unroll
        for (int k = 0; k < BN; k += 8) {
          a0 = fmin3(a0, sv[k], sv[k + 1]);
          a1 = fmin3(a1, sv[k + 2], sv[k + 3]);
          a2 = fmin3(a2, sv[k + 4], sv[k + 5]);
          a3 = fmin3(a3, sv[k + 6], sv[k + 7]);
        }
        a0 = fmin3(a0, a1, fminf(a2, a3));
      }
      const float mx = a0 == mv ? -INFINITY : a0 * sl2;  // block maximum, log2 units
      float alpha = 1.0f;
      if (mx > m + kLazy || (m == -INFINITY && mx != -INFINITY)) {
        alpha = ex2(m - mx);  // m = -inf gives 0
        m = mx;
        l *= alpha;
      }
      const float neg_mu = (m == -INFINITY) ? 0.0f : -m;
      const float sc = sl2;
      // z *= alpha: only after the first block, and only if some row of this warp needs it
      // (rare with the lazy threshold, so the loop stays rolled and out of the common path).
      if (__builtin_expect(!first && __any_sync(0xFFFFFFFFu, alpha != 1.0f), 0)) {
#pragma unroll 1
        for (int c0 = 0; c0 < DV; c0 += 16) {
          uint32_t rr[16];
          tmem_ld16(tO + lane_off + c0, rr);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 16; ++k) rr[k] = __float_as_uint(__uint_as_float(rr[k]) * alpha);
          tmem_st16(tO + lane_off + c0, rr);
        }
      }
      first = false;
      float r0 = 0.0f, r1 = 0.0f, r2 = 0.0f, r3 = 0.0f;
#pragma unroll
      for (int c0 = 0; c0 < BN; c0 += 32) {
        uint32_t pk[16];
#pragma unroll
        for (int k = 0; k < 16; k += 2) {
          const float x0 = fmaf(sv[c0 + 2 * k], sc, neg_mu);
          const float x1 = fmaf(sv[c0 + 2 * k + 1], sc, neg_mu);
          const float x2 = fmaf(sv[c0 + 2 * k + 2], sc, neg_mu);
          const float x3 = fmaf(sv[c0 + 2 * k + 3], sc, neg_mu);
          const float p0 = ex2(x0);
          const float p1 = kFmaExp >= 2 ? ex2_fma(x1) : ex2(x1);
          const float p2 = kFmaExp >= 3 ? ex2_fma(x2) : ex2(x2);
          const float p3 = kFmaExp >= 1 ? ex2_fma(x3) : ex2(x3);
          r0 += p0;
          r1 += p1;
          r2 += p2;
          r3 += p3;
          if constexpr (kDrop) {
            const uint32_t kb = kbits[c0 / 32] >> (2 * k);  // keys c0 + 2k .. c0 + 2k + 3
            pk[k] = pack2<kBf16>(kb & 1u ? p0 : 0.0f, kb & 2u ? p1 : 0.0f);
            pk[k + 1] = pack2<kBf16>(kb & 4u ? p2 : 0.0f, kb & 8u ? p3 : 0.0f);
          } else {
            pk[k] = pack2<kBf16>(p0, p1);
            pk[k + 1] = pack2<kBf16>(p2, p3);
          }
        }
        tmem_st16(tS + lane_off + c0 / 2, pk);
      }
      const float rowsum = (r0 + r1) + (r2 + r3);
      l += rowsum;
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.p_full[t]);
    }
    // ---------------------------------------------------------------- epilogue
    if (partial_out) {
      // Key split: this share's normalised partial, float32, one row per thread.  A row with
      // no allowed key in the share gets O_z = 0 and LSE_z = -inf (not an empty row overall).
      if (pair_row0 + t * kRowsPerTile < nrow) {
        if (active && ok) ok = mbar_wait(&bars.o_done[t], 0, p.status, 9);
        tc_fence_after();
        const float inv = l > 0.0f ? (kDrop ? p.drop.scale : 1.0f) / l : 0.0f;
        // The TMEM loads are warp-collective: every lane takes part, rows past n included;
        // only the stores are per row.
        if (ok) {
          const int64_t prow = (static_cast<int64_t>(split) * gridDim.y + bh) * n + row;
          float4* dst = reinterpret_cast<float4*>(p.o_part + prow * DV);
#pragma unroll
          for (int c0 = 0; c0 < DV; c0 += 16) {
            uint32_t rr[16];
            if (active) {
              tmem_ld16(tO + lane_off + c0, rr);
              tmem_wait_ld();
            } else {
#pragma unroll
              for (int k = 0; k < 16; ++k) rr[k] = 0u;
            }
            if (row < nrow) {
#pragma unroll
              for (int k = 0; k < 16; k += 4)
                dst[(c0 + k) / 4] =
                    make_float4(__uint_as_float(rr[k]) * inv, __uint_as_float(rr[k + 1]) * inv,
                                __uint_as_float(rr[k + 2]) * inv, __uint_as_float(rr[k + 3]) * inv);
            }
          }
          if (row < nrow)
            p.lse_part[prow] = l > 0.0f ? (m + __log2f(l)) * 0.6931471805599453f : -INFINITY;
        }
      }
    } else if (pair_row0 + t * kRowsPerTile < nrow) {
      // A tile with rows but no allowed key at all (possible only under a bitmap) writes zeros
      // and -inf, like any other row with an empty allowed set.
      if (active && ok) ok = mbar_wait(&bars.o_done[t], 0, p.status, 9);
      tc_fence_after();
      const float inv = l > 0.0f ? (kDrop ? p.drop.scale : 1.0f) / l : 0.0f;
      uint8_t* stage = sQ + t * C::kQSlot;  // Q_t is dead once every MMA of tile t is done
      if (ok) {
        // up to 64 columns of O loaded before one wait
        constexpr int kB = DV < 64 ? DV : 64;
#pragma unroll
        for (int c0 = 0; c0 < DV; c0 += kB) {
          uint32_t rr[kB];
          if (active) {
#pragma unroll
            for (int c = 0; c < kB; c += 16)
              tmem_ld16(tO + lane_off + c0 + c, *reinterpret_cast<uint32_t(*)[16]>(rr + c));
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int k = 0; k < kB; ++k) rr[k] = 0u;
          }
#pragma unroll
          for (int c = 0; c < kB; c += 8) {
            uint32_t pk[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
              pk[k] = pack2<kBf16>(__uint_as_float(rr[c + 2 * k]) * inv,
                                   __uint_as_float(rr[c + 2 * k + 1]) * inv);
            *reinterpret_cast<uint4*>(stage + TO::offset(r, c0 + c)) =
                make_uint4(pk[0], pk[1], pk[2], pk[3]);
          }
        }
        if (row < nrow) {
          p.lse[static_cast<int64_t>(bh) * n + row] =
              l > 0.0f ? (m + __log2f(l)) * 0.6931471805599453f : -INFINITY;
          if (!(l > 0.0f)) raise_empty_row(p.status);
        }
      }
      fence_proxy_async_smem();
      named_barrier(1 + t, 128);
      if (ok && r == 0) {
#pragma unroll
        for (int b = 0; b < TO::L::kBoxes; ++b)
          tma_store_3d(&tm_o, stage + b * TO::kBoxBytes, b * TO::L::kBoxCols, pair_row0 + t * kRowsPerTile, bh);
        tma_store_commit();
        tma_store_wait_all();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemAlloc);
  }
}

}  // namespace fwd
}  // namespace ea
