// Forward pass of exact tiled softmax attention with FP8 (E4M3) operands on the tcgen05 tensor
// cores (kind::f8f6f4), bf16 output.
//
// The algorithm is the tiled forward of "Exact tiled attention and memory-aware
// differentiation" (key blocks in order, empty blocks skipped, each row's summary (m, l, z)
// merged block by block, O = z / l, LSE = m + ln l).  The inputs are 8-bit with one scale per
// tensor: Q = sq q8, K = sk k8, V = sv v8, and the caller passes V transposed, vt8 [d][n] per
// head, so that both products read K-major operands:
//   S = q8 k8ᵀ (fp32 in TMEM), scores = c sq sk S;
//   P = 2^8 exp(score - m) rounded to E4M3 (m the running maximum, raised only when a block's
//       maximum exceeds it by more than kLazy8 = 0.75 in log2 units, so P <= 2^8.75 < 448, and
//       probabilities down to 2^-14 of the row maximum stay in E4M3's normal range);
//   z += P v8 (fp32 in TMEM);  l += the unrounded 2^8 exp(score - m);
//   O = sv z / l (bf16), LSE = m + ln(l / 2^8).
// The rounding of P to E4M3 is the step that FP8 adds; its effect on O is bounded elementwise
// by sum_j (2^-4 p_ij + 2^-18) |V_j| / l_i (half an E4M3 ulp relative, or half the smallest
// subnormal step).
//
// Block scaling (the FP8 variant the same page names for FlashAttention-3): with one scale per
// 128-row block, sq_I of the query tile and sk_J of key block J make the score factor
// c sq_I sk_J per block (a scalar per row and step); the value scale sv_J of block J enters
// through the probabilities: P'_ij = 2^8 exp(score - m) r_J with r_J = sv_J / max_J sv_J <= 1,
// added to the exponent as log2 r_J, and z is multiplied by max_J sv_J in the epilogue.  The
// row sum takes each block's sum of P' divided by r_J, so l stays the sum of 2^8 exp(score - m).
//
// Layout and roles as the 16-bit kernel: one CTA owns two tiles of 128 query rows of one head;
// warp 0 and 1 issue the MMAs of tile 0 and 1, warps 2-9 are the softmax (one query row per
// lane), warp 10 the TMA producer.  Key blocks of 128; d in {64, 128}; no key split, no dropout.
#pragma once
#include <cuda_bf16.h>

#include "kernels.h"
#include "tile.cuh"

namespace ea {
namespace fp8 {

constexpr int kRowsPerTile = 128;
constexpr int BN = 128;
constexpr int kThreads = 352;
constexpr int kSoftmaxThreads = 256;
constexpr int kFirstSoftmaxWarp = 2;
constexpr int kProducerWarp = 10;
constexpr uint32_t kSkip = 0, kFull = 1, kPartial = 2;
constexpr int kMaxDynSmem = 227 * 1024 - 1024;
// Lazy raise of the running maximum (log2 units): the stale maximum is at most this far below
// the true one, so P = 2^8 2^(s - m) stays at most 2^8.75 = 430.5 < 448 (no saturation), and the
// row maximum's own P is still at least 2^8, which the error bound of the P rounding needs.
constexpr float kLazy8 = 0.75f;
// Of every four exponentials of the softmax loop, kFmaExp are computed on the FMA pipe
// (ex2_fma) and the rest on the MUFU unit.  Measured at B 8, H 16, n 4096, d 128: 0.835 ms with
// none, 0.970 ms with one in four, 1.077 ms with two, so every exponential stays on MUFU.
constexpr int kFmaExp = 0;

struct Params {
  int n;
  float sl2;  // c sq sk log2(e): raw 8-bit score products to base-2 exponents
  float sv;   // value scale
  int mask_kind;
  const uint32_t* mask_bits;
  int64_t mask_row_words;
  int64_t mask_head_stride_words;
  __nv_bfloat16* o;
  float* lse;
  uint32_t* status;
  // Block scales [heads][ceil(n / 128)] (null: one scale per tensor, folded into sl2 and sv).
  // With them sl2 is c log2(e) and sv is unused.
  const float* sq_blk;
  const float* sk_blk;
  const float* sv_blk;
  Ring ring;  // depth of the (K, V) ring
};

// Tiles of 8-bit elements use the 16-bit layouts with half as many columns: a row of C bytes
// is a row of C/2 16-bit elements, and a 32-element K step of an 8-bit product moves the same
// 32 bytes as a 16-element step of a 16-bit one.
template <int D>
struct Config {
  using TQ = Tile<kRowsPerTile, D / 2>;  // q8 tile: 128 rows x D bytes
  using TK = Tile<BN, D / 2>;            // k8 block: 128 keys x D bytes
  using TV = Tile<D, BN / 2>;            // vt8 block: D value columns x 128 keys (bytes)
  static constexpr int kSmemBudget = kMaxDynSmem - 1024;
  static constexpr int kFixed = 2 * TQ::kBytes;
  static constexpr int kStepReserve = 1024;
  static constexpr int kPair = TK::kBytes + TV::kBytes;
  static constexpr int kStages = (kSmemBudget - kFixed - kStepReserve) / kPair;
  static constexpr int NS = kStages > 4 ? 4 : kStages;
  static_assert(NS >= 2, "need two stages");
  static constexpr int kTmemCols = 2 * BN + 2 * D;
  static_assert(kTmemCols <= 512, "tensor memory overflow");
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + 2 * TQ::kBytes;
  static constexpr int kOffV = kOffK + NS * TK::kBytes;
  static constexpr int kOffSteps = kOffV + NS * TV::kBytes;
  static size_t smem_bytes(int n, int mask_kind) {
    const size_t nblk = (static_cast<size_t>(n) + BN - 1) / BN;
    return 1024 + kOffSteps + (mask_kind == kMaskBitmap ? 4 * nblk : 0);
  }
};

struct Barriers {
  uint64_t q_full[2], s_full[2], p_full[2], o_done[2];
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint32_t tmem_base;
  uint32_t nsteps;
  uint32_t act;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Step word of a walk without a table (none / causal): block j and each tile's class.
__device__ __forceinline__ uint32_t dense_step(int j, int nblk, int n, int pair_row0, bool causal) {
  uint32_t w = static_cast<uint32_t>(j);
  const bool tail_blk = (n % BN) != 0 && j == nblk - 1;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int r0 = pair_row0 + t * kRowsPerTile;
    if (r0 >= n) continue;
    const int last_row = min(r0 + kRowsPerTile, n) - 1;
    const bool any = !causal || j * BN <= last_row;
    const bool all = !causal || (j + 1) * BN - 1 <= r0;
    w |= (any ? ((all && !tail_blk) ? kFull : kPartial) : kSkip) << (16 + 2 * t);
  }
  return w;
}

// kCap: ring depth from the launch (p.ring) instead of the compile-time count.
template <int D, bool kBlocks, bool kCap = false>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_fp8_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_vt, Params p) {
  using C = Config<D>;
  using TQ = typename C::TQ;
  using TK = typename C::TK;
  using TV = typename C::TV;
  constexpr int NS = C::NS;
  const auto ring = ring_of<kCap, NS>(p.ring);

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
  const int n = p.n;
  const int bh = blockIdx.y;
  const int pair = gridDim.x - 1 - blockIdx.x;
  const int pair_row0 = pair * 2 * kRowsPerTile;
  const int nblk = (n + BN - 1) / BN;
  const bool use_table = p.mask_kind == kMaskBitmap;
  const bool causal = p.mask_kind == kMaskCausal;

  if (tid == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars.q_full[t], 1);
      mbar_init(&bars.s_full[t], 1);
      mbar_init(&bars.p_full[t], 4);
      mbar_init(&bars.o_done[t], 1);
    }
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bars.k_full[s], 1);
      mbar_init(&bars.v_full[s], 1);
    }
  }
  if (warp == 0) tmem_alloc(&bars.tmem_base, 512);

  // walk over key blocks (as in the 16-bit kernel)
  if (use_table) {
    for (int j = tid; j < nblk; j += kThreads) steps[j] = 0;
    __syncthreads();
    if (tid < kSoftmaxThreads) {
      const int t = tid / kRowsPerTile;
      const int row = pair_row0 + t * kRowsPerTile + (tid % kRowsPerTile);
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
              const int left = n - key0;
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
          const uint32_t bits = (wany ? (1u << t) : 0u) | (wall ? 0u : (4u << t));
          if (bits) atomicOr(&steps[j], bits);
        }
      }
    }
    __syncthreads();
    if (tid == 0) {
      const bool tail = (n % BN) != 0;
      int ns = 0;
      for (int j = 0; j < nblk; ++j) {
        const uint32_t b = steps[j];
        const bool part_tail = tail && j == nblk - 1;
        const uint32_t cls0 = (b & 1u) ? (((b & 4u) || part_tail) ? kPartial : kFull) : kSkip;
        const uint32_t cls1 = (b & 2u) ? (((b & 8u) || part_tail) ? kPartial : kFull) : kSkip;
        if (cls0 | cls1) steps[ns++] = static_cast<uint32_t>(j) | (cls0 << 16) | (cls1 << 18);
      }
      uint32_t act = 0;
      for (int i = 0; i < ns; ++i)
        act |= ((steps[i] >> 16) & 3u ? 1u : 0u) | ((steps[i] >> 18) & 3u ? 2u : 0u);
      bars.nsteps = ns;
      bars.act = act;
    }
  } else if (tid == 0) {
    const int pair_last = min(pair_row0 + 2 * kRowsPerTile, n) - 1;
    bars.nsteps = causal ? pair_last / BN + 1 : nblk;
    bars.act = (pair_row0 < n ? 1u : 0u) | (pair_row0 + kRowsPerTile < n ? 2u : 0u);
  }
  if (tid == 0) {
    const uint32_t a = bars.act;
    const uint32_t issuers = (a & 1u) + ((a >> 1) & 1u);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bars.k_empty[s], issuers ? issuers : 1u);
      mbar_init(&bars.v_empty[s], issuers ? issuers : 1u);
    }
    fence_barrier_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const int nsteps = bars.nsteps;
  const uint32_t tmem = bars.tmem_base;
  const uint32_t act = bars.act;
  auto step_at = [&](int i) -> uint32_t {
    return use_table ? steps[i] : dense_step(i, nblk, n, pair_row0, causal);
  };

  if (warp == kProducerWarp) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_vt);
      for (int t = 0; t < 2; ++t) {
        if (!((act >> t) & 1u)) continue;
        mbar_arrive_expect_tx(&bars.q_full[t], TQ::kBytes);
        tma_load_3d(sQ + t * TQ::kBytes, &tm_q, &bars.q_full[t], 0, pair_row0 + t * kRowsPerTile, bh);
      }
      for (int i = 0; i < nsteps; ++i) {
        const int s = ring.stage(i);
        const uint32_t ph = ring.parity(i) ^ 1;
        const int key0 = static_cast<int>(step_at(i) & 0xFFFFu) * BN;
        if (!mbar_wait(&bars.k_empty[s], ph, p.status, 1)) break;
        mbar_arrive_expect_tx(&bars.k_full[s], TK::kBytes);
        tma_load_3d(sK + s * TK::kBytes, &tm_k, &bars.k_full[s], 0, key0, bh);
        if (!mbar_wait(&bars.v_empty[s], ph, p.status, 2)) break;
        mbar_arrive_expect_tx(&bars.v_full[s], TV::kBytes);
        tma_load_3d(sV + s * TV::kBytes, &tm_vt, &bars.v_full[s], key0, 0, bh);
      }
    }
  } else if (warp < kFirstSoftmaxWarp) {
    // ---------------------------------------------------------------- MMA issuer (tile t)
    const int t = warp;
    constexpr uint32_t id_s = idesc_e4m3(128, BN);
    constexpr uint32_t id_o = idesc_e4m3(128, D);
    const uint64_t dq = TQ::desc_k(smem_u32(sQ + t * TQ::kBytes), 0);
    const uint64_t dk0 = TK::desc_k(smem_u32(sK), 0);
    const uint64_t dv0 = TV::desc_k(smem_u32(sV), 0);
    const uint32_t tS = tmem + t * BN;
    const uint32_t tO = tmem + 2 * BN + t * D;
    bool ok = (act >> t) & 1u;
    if (ok) ok = mbar_wait_warp(&bars.q_full[t], 0, p.status, 3);
    bool pend = false, started = false;
    uint32_t pph = 0;
    for (int i = 0; i <= nsteps && ok; ++i) {
      const int prev = i - 1;
      if (prev >= 0) {
        ok = mbar_wait_warp(&bars.v_full[ring.stage(prev)], ring.parity(prev), p.status, 5);
        if (!ok) break;
      }
      const bool cur = i < nsteps && ((step_at(i) >> (16 + 2 * t)) & 3u) != 0;
      const int s = ring.stage(i);
      if (i < nsteps) {
        ok = mbar_wait_warp(&bars.k_full[s], ring.parity(i), p.status, 6);
        if (!ok) break;
      }
      tc_fence_after();
      if (pend) {
        ok = mbar_wait_warp(&bars.p_full[t], pph, p.status, 4);
        if (!ok) break;
        pph ^= 1u;
        tc_fence_after();
        const uint64_t dv = dv0 + static_cast<uint64_t>(ring.stage(prev)) * (TV::kBytes >> 4);
        if (elect_one()) {
          // z += P vt8ᵀ: A = P in tensor memory (four 8-bit values a column), 32 keys a step
#pragma unroll
          for (int kk = 0; kk < BN / 32; ++kk)
            mma_ts_f8(tO, tS + kk * 8, dv + TV::k_step(kk), id_o, (started || kk > 0) ? 1u : 0u);
        }
        __syncwarp();
        started = true;
      }
      if (cur) {
        const uint64_t dk = dk0 + static_cast<uint64_t>(s) * (TK::kBytes >> 4);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 32; ++kk)
            mma_ss_f8(tS, dq + TQ::k_step(kk), dk + TK::k_step(kk), id_s, kk > 0 ? 1u : 0u);
          mma_commit(&bars.s_full[t]);
        }
        __syncwarp();
      }
      if (elect_one()) {
        if (i < nsteps) mma_commit(&bars.k_empty[s]);
        if (prev >= 0) mma_commit(&bars.v_empty[ring.stage(prev)]);
      }
      __syncwarp();
      pend = cur;
    }
    if (ok && elect_one()) mma_commit(&bars.o_done[t]);
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- softmax (tile t)
    const int t = (warp - kFirstSoftmaxWarp) / 4;
    const int quad = warp % 4;
    const int r = quad * 32 + lane;
    const int row = pair_row0 + t * kRowsPerTile + r;
    const uint32_t tS = tmem + t * BN;
    const uint32_t tO = tmem + 2 * BN + t * D;
    const bool active = (act >> t) & 1u;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const float sl2 = p.sl2 == 0.0f ? 1.17549435e-38f : p.sl2;  // c = 0: all weights equal
    const bool pos = sl2 > 0.0f;
    const float mv = pos ? -INFINITY : INFINITY;
    constexpr bool blocks = kBlocks;
    const int sbase = bh * nblk;  // this head's first block scale
    // largest value-block scale of the head (every lane gets it)
    auto head_vmax = [&]() -> float {
      float mxv = 0.0f;
      for (int jb = lane; jb < nblk; jb += 32) mxv = fmaxf(mxv, __ldg(p.sv_blk + sbase + jb));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mxv = fmaxf(mxv, __shfl_xor_sync(0xFFFFFFFFu, mxv, o));
      return mxv;
    };
    float kq = sl2;  // score factor without the key block's scale
    float l2vmax = 0.0f;
    if (blocks) {
      kq = sl2 * __ldg(p.sq_blk + sbase + min(pair * 2 + t, nblk - 1));
      l2vmax = __log2f(head_vmax());
    }
    float m = -INFINITY;  // running maximum (stale by at most kLazy8), log2 units
    float l = 0.0f;       // running sum of 2^8 exp(score - m)
    uint32_t s_phase = 0;
    bool first = true;
    bool ok = true;
    const uint32_t* rowbits =
        use_table ? p.mask_bits + static_cast<int64_t>(bh) * p.mask_head_stride_words +
                        static_cast<int64_t>(row < n ? row : 0) * p.mask_row_words
                  : nullptr;
    for (int i = 0; i < nsteps && ok; ++i) {
      const uint32_t sw = step_at(i);
      const uint32_t cls = (sw >> (16 + 2 * t)) & 3u;
      if (cls == kSkip) continue;
      const int key0 = static_cast<int>(sw & 0xFFFFu) * BN;
      // this block's score factor kj, log2 r_J and 1 / r_J (loaded before the wait)
      float kj = sl2, lr = 0.0f, inv_r = 1.0f;
      if (blocks) {
        const int jb = static_cast<int>(sw & 0xFFFFu);
        kj = kq * __ldg(p.sk_blk + sbase + jb);
        kj = pos ? fmaxf(kj, 1.17549435e-38f) : fminf(kj, -1.17549435e-38f);
        lr = __log2f(__ldg(p.sv_blk + sbase + jb)) - l2vmax;
        inv_r = ex2(-lr);
      }
      // partial blocks: the allowed-key words (bit k of word q <-> key key0 + 32 q + k), applied
      // to the scores in registers once they are loaded
      uint32_t mw[BN / 32];
      if (cls == kPartial) {
#pragma unroll
        for (int q = 0; q < BN / 32; ++q) {
          const int kq = key0 + q * 32;
          uint32_t w;
          if (use_table) {
            w = (row < n && kq < n) ? __ldg(rowbits + kq / 32) : 0u;
            const int left = n - kq;
            if (left < 32) w &= left > 0 ? (1u << left) - 1u : 0u;
          } else {
            const int lim = causal ? min(row, n - 1) : n - 1;
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
      if (cls == kPartial) {
#pragma unroll
        for (int k = 0; k < BN; ++k)
          if (!((mw[k / 32] >> (k % 32)) & 1u)) sv[k] = mv;
      }
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
      const float mx = a0 == mv ? -INFINITY : a0 * kj;
      float alpha = 1.0f;
      if (mx > m + kLazy8 || (m == -INFINITY && mx != -INFINITY)) {
        alpha = ex2(m - mx);  // m = -inf gives 0
        m = mx;
        l *= alpha;
      }
      if (!first && __any_sync(0xFFFFFFFFu, alpha != 1.0f)) {
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 16) {
          uint32_t rr[16];
          tmem_ld16(tO + lane_off + c0, rr);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 16; ++k) rr[k] = __float_as_uint(__uint_as_float(rr[k]) * alpha);
          tmem_st16(tO + lane_off + c0, rr);
        }
      }
      first = false;
      // P = 2^8 r_J exp2(s kj - m): the +8 in the exponent keeps small probabilities normal in
      // E4M3; r_J (block scales) rides along in the exponent
      const float neg_mu = (m == -INFINITY) ? 0.0f : 8.0f - m + lr;
      float r0 = 0.0f, r1 = 0.0f, r2 = 0.0f, r3 = 0.0f;
#pragma unroll
      for (int c0 = 0; c0 < BN; c0 += 64) {
        uint32_t pk[16];  // 64 keys, four per word
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float x0 = fmaf(sv[c0 + 4 * k], kj, neg_mu);
          const float x1 = fmaf(sv[c0 + 4 * k + 1], kj, neg_mu);
          const float x2 = fmaf(sv[c0 + 4 * k + 2], kj, neg_mu);
          const float x3 = fmaf(sv[c0 + 4 * k + 3], kj, neg_mu);
          const float p0 = ex2(x0);
          const float p1 = kFmaExp >= 2 ? ex2_fma(x1) : ex2(x1);
          const float p2 = kFmaExp >= 3 ? ex2_fma(x2) : ex2(x2);
          const float p3 = kFmaExp >= 1 ? ex2_fma(x3) : ex2(x3);
          r0 += p0;
          r1 += p1;
          r2 += p2;
          r3 += p3;
          pk[k] = pack4_e4m3(p0, p1, p2, p3);
        }
        tmem_st16(tS + lane_off + c0 / 4, pk);
      }
      l += ((r0 + r1) + (r2 + r3)) * inv_r;
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.p_full[t]);
    }
    // ---------------------------------------------------------------- epilogue
    // O = sv z / l in bf16, one row per thread with 16-byte stores; LSE = m + ln(l / 2^8).
    if (pair_row0 + t * kRowsPerTile < n) {
      if (active && ok) ok = mbar_wait(&bars.o_done[t], 0, p.status, 9);
      tc_fence_after();
      const float vmax = blocks ? head_vmax() : p.sv;  // reloaded: not held through the loop
      const float inv = l > 0.0f ? vmax / l : 0.0f;
      if (ok) {
        uint4* dst = reinterpret_cast<uint4*>(p.o + (static_cast<int64_t>(bh) * n + row) * D);
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 16) {
          uint32_t rr[16];
          if (active) {
            tmem_ld16(tO + lane_off + c0, rr);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int k = 0; k < 16; ++k) rr[k] = 0u;
          }
          uint32_t pk[8];
#pragma unroll
          for (int k = 0; k < 8; ++k)
            pk[k] = pack2<true>(__uint_as_float(rr[2 * k]) * inv, __uint_as_float(rr[2 * k + 1]) * inv);
          if (row < n) {
            dst[c0 / 8] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            dst[c0 / 8 + 1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          }
        }
        if (row < n) {
          p.lse[static_cast<int64_t>(bh) * n + row] =
              l > 0.0f ? (m + __log2f(l) - 8.0f) * 0.6931471805599453f : -INFINITY;
          if (!(l > 0.0f)) raise_empty_row(p.status);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace fp8
}  // namespace ea
