/*
 * exactattn — exact tiled softmax attention on NVIDIA GB300 (sm_103a).  C ABI.
 *
 * What is computed.  For every head (b, h) and query row i (0-based), with scale c and the
 * allowed-key set A_i chosen by the mask:
 *
 *     s_ij  = c * sum_r Q[i][r] * K[j][r]            (j in A_i)
 *     LSE_i = m_i + ln( sum_{j in A_i} exp(s_ij - m_i) ),  m_i = max_{j in A_i} s_ij
 *     O_i   = sum_{j in A_i} exp(s_ij - LSE_i) * V_j
 *
 * This is the masked scaled dot-product attention of "Exact tiled attention and
 * memory-aware differentiation" (definition of the stable summary; exactness theorem), with
 * the two retained row statistics (m_i, l_i) kept as the single number LSE_i.  The forward
 * streams key/value blocks past an on-chip tile of query rows and updates the running
 * maximum, normaliser and weighted value sum, rescaling older partial sums by e^(m - m')
 * (same page, tiled forward; "The Arithmetic of Intelligence", chapter 12, streaming
 * softmax).  It never forms the n x n score matrix and writes only O and LSE.
 *
 * The backward recomputes each score and probability block from Q, K and the saved LSE
 * (same page, reverse procedure): with G = dO,
 *     D_i   = sum_a G[i][a] * O[i][a]
 *     p_ij  = exp(s_ij - LSE_i),   g_ij = p_ij * (G_i . V_j - D_i)
 *     dQ_i  = c * sum_j g_ij K_j,  dK_j = c * sum_i g_ij Q_i,  dV_j = sum_i p_ij G_i
 * It never reads a stored probability matrix.
 *
 * Layout.  Q, K, V, O, dO, dQ, dK, dV are contiguous row-major [B][H][n][d] arrays of the
 * call's dtype (value dimension v = d).  LSE is [B][H][n] float32 (natural log).  All device
 * pointers must be 16-byte aligned.  Masks:
 *   ATTN_MASK_NONE    every key is allowed;
 *   ATTN_MASK_CAUSAL  key j is allowed for query i iff j <= i;
 *   ATTN_MASK_BITMAP  caller-owned packed allowed sets: device array of uint32 words, row i of
 *                     head bh starts at word  bh * mask_head_stride_words + i * mask_row_words,
 *                     key j is allowed iff bit (j % 32) of word (j / 32) of that row is set.
 *                     mask_row_words >= ceil(n / 32); mask_head_stride_words = 0 shares one
 *                     bitmap across all heads.  The library only reads it.
 *
 * Precision.  ATTN_F32 runs on the CUDA cores in float32 throughout.  ATTN_F16 / ATTN_BF16
 * run on the tcgen05 tensor cores: the 16-bit inputs are multiplied with float32
 * accumulation, the probabilities are rounded to the input type (nearest-even) before the
 * P*V product, and O, dQ, dK, dV are rounded to the input type at the end.
 *
 * Supported: d in {16, 32, 64, 128}; n >= 1; B * H >= 1; kv_block in {0 (auto), 32, 64, 128}.
 * The key-block size b only changes the order of floating-point accumulation: every b gives
 * the same allowed sets and the same result up to rounding.
 *
 * Ownership and errors.  The caller allocates every buffer (inputs, outputs, LSE, workspace,
 * bitmap).  The library allocates no device memory per call and keeps no state between calls
 * apart from cached function attributes.  Every entry point returns ATTN_OK (0) or a negative
 * error code and never throws; attn_last_error() gives a message for the calling thread's last
 * failure.  Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy default
 * stream).  A row whose allowed set is empty has no defined output (the pages assume every
 * A_i is nonempty): the library writes O_i = 0, LSE_i = -inf, adds no gradient for that row
 * and raises ATTN_WARN_EMPTY_ROW in the device status word.
 */
#ifndef EXACTATTN_H
#define EXACTATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { ATTN_F32 = 0, ATTN_F16 = 1, ATTN_BF16 = 2 } attn_dtype;
typedef enum { ATTN_MASK_NONE = 0, ATTN_MASK_CAUSAL = 1, ATTN_MASK_BITMAP = 2 } attn_mask_kind;

enum {
  ATTN_OK = 0,
  ATTN_WARN_EMPTY_ROW = 1,       /* status only: some row had an empty allowed set */
  ATTN_ERR_INVALID_ARG = -1,     /* null pointer, non-positive size, bad enum */
  ATTN_ERR_UNSUPPORTED = -2,     /* head dim / key block / dtype combination not built */
  ATTN_ERR_ALIGNMENT = -3,       /* a device pointer is not 16-byte aligned */
  ATTN_ERR_WORKSPACE = -4,       /* workspace missing or smaller than attn_bwd_workspace_bytes */
  ATTN_ERR_CUDA = -5,            /* a CUDA runtime/driver call failed (message has details) */
  ATTN_ERR_DEVICE_TIMEOUT = -6   /* a bounded in-kernel wait gave up (see attn_device_status) */
};

/*
 * Forward pass.  Writes o [B][H][n][d] (dtype) and lse [B][H][n] (float32, natural log).
 * Definition: the tiled forward procedure of "Exact tiled attention and memory-aware
 * differentiation"; O_i = z_i / l_i and LSE_i = m_i + ln l_i from the final row summary.
 *   dtype      ATTN_F32 / ATTN_F16 / ATTN_BF16, the type of q, k, v and o
 *   B, H, n, d batch, heads, tokens, head dimension
 *   c          score scale (commonly 1/sqrt(d))
 *   q, k, v    device inputs, [B][H][n][d]
 *   mask_kind  ATTN_MASK_NONE / CAUSAL / BITMAP; the three mask_* words are read only for BITMAP
 *   kv_block   key-block size b (0 = library choice)
 *   o, lse     device outputs
 *   stream     cudaStream_t
 */
int attn_fwd(int dtype, int B, int H, int n, int d, float c,
             const void* q, const void* k, const void* v,
             int mask_kind, const uint32_t* mask_bits, int64_t mask_row_words,
             int64_t mask_head_stride_words, int kv_block,
             void* o, float* lse, void* stream);

/*
 * Forward pass with dropout on the attention probabilities.  The pages' base procedure has no
 * dropout and ask of any dropout extension that its reverse pass replay the realised mask
 * ("Exact tiled attention and memory-aware differentiation", reverse procedure; closing
 * remark).  Here the mask is a pure function of (seed, head, query row, key), so the forward
 * and attn_bwd_dropout draw the same mask and no mask is stored.  One generator call decides a
 * 4 x 4 patch of (query, key) pairs:
 *   words = Philox4x32-10(counter = (floor(i / 4), floor(j / 4), b * H + h, 0),
 *           key = (seed mod 2^32, floor(seed / 2^32)))  (Salmon et al., "Parallel random
 *           numbers: as easy as 1, 2, 3", SC 2011); the pair (i, j) is kept iff byte j mod 4
 *           (least significant first) of words[i mod 4] >= t, t = floor(p_drop 256 + 1/2).
 *   O_i = sum_j P_ij keep_ij V_j / (1 - p'), p' = t / 256, P = softmax as without dropout.
 * The drop probability is thus p_drop rounded to a multiple of 1/256.  LSE is that of the
 * undropped scores (the statistic the backward needs).
 *   p_drop  drop probability, 0 <= p_drop < 1 and t <= 255 (0 gives exactly attn_fwd's result);
 *           ATTN_ERR_INVALID_ARG otherwise
 *   seed    64-bit generator key; the same (seed, p_drop) must be passed to attn_bwd_dropout
 * Other arguments, outputs and errors as for attn_fwd.
 */
int attn_fwd_dropout(int dtype, int B, int H, int n, int d, float c,
                     const void* q, const void* k, const void* v,
                     int mask_kind, const uint32_t* mask_bits, int64_t mask_row_words,
                     int64_t mask_head_stride_words, int kv_block, float p_drop, uint64_t seed,
                     void* o, float* lse, void* stream);

/*
 * Key-split forward: the same O and LSE as attn_fwd, computed as num_splits partial results
 * over disjoint shares of the key blocks and combined by attn_merge's rule.  This is the
 * key-sharded reading of the merge of stable summaries in "Exact tiled attention and
 * memory-aware differentiation": the summary of a union of disjoint key sets is the merge of
 * the sets' summaries, so the shares can run in parallel.  It fills the GPU when B * H * n is
 * small next to the key length (few heads, long rows), where attn_fwd launches too few CTAs.
 *   num_splits  0 = library choice (attn_fwd_split_count), else 1..32; 1 runs attn_fwd
 *   workspace   device buffer of at least attn_fwd_split_workspace_bytes(...) bytes for the
 *               number of splits actually used, 16-byte aligned (ignored when that is 1); it
 *               holds the float32 partial O and LSE of every share and is overwritten
 *   Other arguments, outputs and errors as for attn_fwd.  Two launches on `stream`.
 * Each row's key blocks are cut into num_splits contiguous shares of equal block count (the
 * blocks its rows reach under the causal mask); a row with no allowed key in a share takes
 * that share as the empty summary.  Results agree with attn_fwd up to rounding.
 */
int attn_fwd_split(int dtype, int B, int H, int n, int d, float c,
                   const void* q, const void* k, const void* v,
                   int mask_kind, const uint32_t* mask_bits, int64_t mask_row_words,
                   int64_t mask_head_stride_words, int kv_block, int num_splits,
                   void* o, float* lse, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Forward pass of n_q query rows against n_kv keys: attention over a key/value cache (for
 * instance decoding, n_q small and n_kv long).  q and o are [B][H][n_q][d], k and v
 * [B][H][n_kv][d], lse [B][H][n_q].  The queries are the last n_q positions of the sequence:
 * under ATTN_MASK_CAUSAL query i sees keys j <= i + n_kv - n_q (n_q = n_kv is attn_fwd's causal
 * mask; with n_q > n_kv the first n_q - n_kv rows see no key and are empty rows).  A bitmap has
 * n_q rows of mask_row_words >= ceil(n_kv / 32) words.  The keys are cut into num_splits shares
 * as in attn_fwd_split (0 = attn_fwd_kv_split_count), which is what fills the GPU when n_q is
 * small; workspace as for attn_fwd_split with n = n_q (attn_fwd_split_workspace_bytes).
 * The pages' tiled forward and its merge of stable summaries of disjoint key sets define the
 * result for any query and key counts ("Exact tiled attention and memory-aware
 * differentiation": inputs n queries, keys and values of any length).  Forward only: the
 * backward entry points require n_q = n_kv.  Other arguments and errors as for attn_fwd_split.
 */
int attn_fwd_kv(int dtype, int B, int H, int n_q, int n_kv, int d, float c,
                const void* q, const void* k, const void* v,
                int mask_kind, const uint32_t* mask_bits, int64_t mask_row_words,
                int64_t mask_head_stride_words, int kv_block, int num_splits,
                void* o, float* lse, void* workspace, size_t workspace_bytes, void* stream);

/*
 * FP8 forward: exact tiled attention with E4M3 operands on the tensor cores (kind::f8f6f4),
 * bfloat16 output.  The inputs carry one scale each: Q = q_scale q8, K = k_scale k8 and
 * V = v_scale vt8ᵀ, where
 *   q8, k8  E4M3 [B][H][n][d]
 *   vt8     E4M3 [B][H][d][n]: V transposed (the value columns are rows), so that the P V
 *           product reads a K-major operand
 * The scores are c·q_scale·k_scale·(q8·k8) accumulated in float32.  Each probability enters the
 * P V product as an E4M3 value of 2^8 exp(s - m) (m the running maximum, at most 0.75 log2
 * units below the true one, so the value stays below 448); the row sum
 * keeps the unrounded values.  The output therefore differs from exact attention on the
 * dequantized inputs by at most sum_j (2^-4 P_ij + 2^-18) |V_j| per element (the rounding of P),
 * plus float32 and bfloat16 rounding.  lse is float32, natural log, of the scaled scores.
 *   d: 64 or 128; n: a multiple of 16; masks as for attn_fwd; o: bfloat16 [B][H][n][d].
 * The pages' FP8 forward (FlashAttention-3 on H100, "Bellek Duvarının Fiziği") adds block
 * scaling and incoherent processing: see attn_fp8_quantize and attn_fwd_fp8_blocks.  This
 * entry point takes one scale per tensor.
 */
int attn_fwd_fp8(int B, int H, int n, int d, float c,
                 const void* q8, const void* k8, const void* vt8,
                 float q_scale, float k_scale, float v_scale,
                 int mask_kind, const uint32_t* mask_bits, int64_t mask_row_words,
                 int64_t mask_head_stride_words, void* o, float* lse, void* stream);

/*
 * Block quantization for the FP8 forward, with optional incoherent processing (the FP8 variant
 * of "Bellek Duvarının Fiziği": per-block scales and random sign multipliers).
 *
 * A block is 128 consecutive rows of one (b, h) head of Q, K or V (the last one ragged).  Each
 * block gets one float32 scale, absmax / 448 (1 for an all-zero block), and its codes are
 * E4M3(x * (448 / absmax)) computed in float32, rounded to nearest even and saturated.
 * With signs != NULL, Q and K are first incoherently processed: each row x becomes (x ∘ σ) H_d,
 * σ_a = -1 where signs[a] < 0 else +1, H_d the order-d Walsh–Hadamard matrix (Sylvester's
 * construction, entry (i, j) = (-1)^popcount(i & j)).  H_d H_dᵀ = d I, so the product of the
 * processed Q and K is d Q Kᵀ; the factor 1/d is folded into Q's scales.  V is never rotated.
 *   dtype      ATTN_BF16 or ATTN_F16 (type of q, k, v)
 *   q, k, v    device [B][H][n][d], contiguous, 16-byte aligned
 *   signs      device int8 [d], or NULL for no incoherent processing
 *   q8, k8     device E4M3 [B][H][n][d] (outputs)
 *   vt8        device E4M3 [B][H][d][n] (output): V's codes transposed
 *   q_scales, k_scales, v_scales
 *              device float32 [B][H][ceil(n / 128)] (outputs), 4-byte aligned
 *   d: 64 or 128; n: a multiple of 16.  Asynchronous on `stream`; allocates nothing.
 * Errors: ATTN_ERR_INVALID_ARG (non-positive sizes, null pointers), ATTN_ERR_UNSUPPORTED
 * (dtype, d, n), ATTN_ERR_ALIGNMENT, ATTN_ERR_CUDA (launch).
 */
int attn_fp8_quantize(int dtype, int B, int H, int n, int d,
                      const void* q, const void* k, const void* v, const int8_t* signs,
                      void* q8, void* k8, void* vt8,
                      float* q_scales, float* k_scales, float* v_scales, void* stream);

/*
 * FP8 forward with block scales: as attn_fwd_fp8, but Q, K and V carry one float32 scale per
 * block of 128 rows, [B][H][ceil(n / 128)] device arrays as attn_fp8_quantize writes them:
 * row i of Q is q_scales[i / 128] q8_i, key j is k_scales[j / 128] k8_j, value j is
 * v_scales[j / 128] v8_j.  The score of (i, j) is c·q_scales[i/128]·k_scales[j/128]·(q8_i·k8_j).
 * A value block's scale enters through the probabilities: those of key block J are rounded to
 * E4M3 as 2^8 exp(s - m) r_J, r_J = v_scales[J] / max_J v_scales[J], and the output is
 * multiplied by the largest scale at the end.  The output then differs from exact attention on
 * the dequantized inputs by at most sum_j (2^-4 P_ij + 2^-18 / r_J(j)) |V_j| per element, plus
 * float32 and bfloat16 rounding.  Other arguments, layouts and errors as for attn_fwd_fp8
 * (ATTN_ERR_INVALID_ARG for a null scale pointer, ATTN_ERR_ALIGNMENT for a misaligned one).
 */
int attn_fwd_fp8_blocks(int B, int H, int n, int d, float c,
                        const void* q8, const void* k8, const void* vt8,
                        const float* q_scales, const float* k_scales, const float* v_scales,
                        int mask_kind, const uint32_t* mask_bits, int64_t mask_row_words,
                        int64_t mask_head_stride_words, void* o, float* lse, void* stream);

/* The number of key shares attn_fwd_kv uses when num_splits = 0 on the current device. */
int attn_fwd_kv_split_count(int dtype, int B, int H, int n_q, int n_kv, int d, int kv_block);

/* The number of key shares attn_fwd_split uses when num_splits = 0 on the current device:
 * enough that the forward grid covers every multiprocessor, at most one per key block and
 * at most 32.  0 for non-positive sizes. */
int attn_fwd_split_count(int dtype, int B, int H, int n, int d, int kv_block);

/* Bytes of workspace attn_fwd_split needs with num_splits shares (1..32; 0 bytes for 1):
 * float32 partial outputs [num_splits][B][H][n][d] and LSEs [num_splits][B][H][n], each
 * rounded up to 256 bytes. */
size_t attn_fwd_split_workspace_bytes(int dtype, int B, int H, int n, int d, int num_splits);

/*
 * Merge partial attention results over disjoint key sets into the result over their union
 * (the merge rule of the stable summaries, "Exact tiled attention and memory-aware
 * differentiation"; key-sharded attention combines shards this way).  For each of `rows`
 * rows, with parts g = 0 .. num_parts-1 given in normalised form (O_g, LSE_g):
 *     LSE = M + ln sum_g exp(LSE_g - M),  M = max_g LSE_g
 *     O   = sum_g exp(LSE_g - LSE) O_g
 * A part with LSE_g = -inf is an empty key set and contributes nothing; a row whose parts are
 * all empty is written as O = 0, LSE = -inf and raises ATTN_WARN_EMPTY_ROW.
 *   dtype      type of o (ATTN_F32 / ATTN_F16 / ATTN_BF16)
 *   o_parts    device float32 [num_parts][rows][d], 16-byte aligned; d a multiple of 4
 *   lse_parts  device float32 [num_parts][rows] (natural log)
 *   o, lse     device outputs [rows][d] (dtype) and [rows] (float32)
 * Memory-bound, one launch on `stream`; inputs are only read.
 */
int attn_merge(int dtype, int num_parts, int64_t rows, int d, const float* o_parts,
               const float* lse_parts, void* o, float* lse, void* stream);

/* Bytes of device workspace attn_bwd needs for these sizes: 16-bit types, a per-row table of
 * float32 LSE*log2(e) and D with n rounded up to 128 rows per head; float32, per-row D. */
size_t attn_bwd_workspace_bytes(int dtype, int B, int H, int n, int d);

/*
 * Backward pass (vector-Jacobian product) for upstream d_o = G.  Writes dq, dk, dv
 * [B][H][n][d] (dtype).  Definition: the reverse procedure of "Exact tiled attention and
 * memory-aware differentiation", with the retained statistics given as lse (from attn_fwd on
 * the same q, k, v, c and mask) and delta_i computed from the stored o.
 *   workspace  device buffer of at least attn_bwd_workspace_bytes(...) bytes, 16-byte aligned;
 *              the call overwrites it (its contents on entry do not matter)
 *   Other arguments as for attn_fwd.
 */
int attn_bwd(int dtype, int B, int H, int n, int d, float c,
             const void* q, const void* k, const void* v, const void* o, const float* lse,
             const void* d_o,
             int mask_kind, const uint32_t* mask_bits, int64_t mask_row_words,
             int64_t mask_head_stride_words, int kv_block,
             void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
             void* stream);

/*
 * Backward pass of attn_fwd_dropout, replaying the same mask (same seed and p_drop).  With
 * p' = floor(p_drop 256 + 1/2) / 256 and P~ = P * keep / (1 - p'): dV = P~^T dO;
 * D_i = dO_i . O_i (O the dropped output);  dS_ij = P_ij (keep_ij (dO_i . V_j) / (1 - p') - D_i);
 * dQ = c dS K,  dK = c dS^T Q.
 * Other arguments, outputs, workspace and errors as for attn_bwd.
 */
int attn_bwd_dropout(int dtype, int B, int H, int n, int d, float c,
                     const void* q, const void* k, const void* v, const void* o,
                     const float* lse, const void* d_o,
                     int mask_kind, const uint32_t* mask_bits, int64_t mask_row_words,
                     int64_t mask_head_stride_words, int kv_block, float p_drop, uint64_t seed,
                     void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                     void* stream);

/*
 * Forward and backward with values of their own width v (v_dim): Q, K in R^{n x d} and V in
 * R^{n x v}, the general shape of "Exact tiled attention and memory-aware differentiation"
 * (inputs n, d, v; output Y in R^{n x v}).  Scores and their gradients live in the d-wide
 * space, O, dO and dV in the v-wide one:
 *   q, k, dq, dk   [B][H][n][d]
 *   v, o, d_o, dv  [B][H][n][v_dim]
 * Supported: v_dim = d (the same as attn_fwd_dropout / attn_bwd_dropout), or (d, v_dim) =
 * (64, 128) or (128, 64), in every dtype, with every mask, key block and dropout (p_drop = 0:
 * none; the mask and seed rules of attn_fwd_dropout).  The backward's workspace is
 * attn_bwd_workspace_bytes(dtype, B, H, n, d).  Other arguments, outputs and errors as for
 * attn_fwd_dropout and attn_bwd_dropout; ATTN_ERR_UNSUPPORTED for another (d, v_dim) pair.
 */
int attn_fwd_vdim(int dtype, int B, int H, int n, int d, int v_dim, float c,
                  const void* q, const void* k, const void* v,
                  int mask_kind, const uint32_t* mask_bits, int64_t mask_row_words,
                  int64_t mask_head_stride_words, int kv_block, float p_drop, uint64_t seed,
                  void* o, float* lse, void* stream);

int attn_bwd_vdim(int dtype, int B, int H, int n, int d, int v_dim, float c,
                  const void* q, const void* k, const void* v, const void* o,
                  const float* lse, const void* d_o,
                  int mask_kind, const uint32_t* mask_bits, int64_t mask_row_words,
                  int64_t mask_head_stride_words, int kv_block, float p_drop, uint64_t seed,
                  void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                  void* stream);

/*
 * attn_bwd without a workspace argument, for callers that cannot allocate device memory at
 * the time they call the backward: an engine or framework that owns every device allocation
 * and gives its plugins no allocator, or a system that fixes its memory budget at start-up
 * and allows no cudaMalloc afterwards.  The pages have no counterpart to this entry point; it
 * computes exactly what attn_bwd computes.
 *
 * The float32 scratch (the per-row table of LSE*log2(e) and D that attn_bwd keeps in its
 * workspace) lives in one static device array of
 * ATTN_BWD_NOALLOC_SCRATCH_BYTES (32 MiB) that every GPU which loads this library holds
 * until the process exits.  A problem with attn_bwd_workspace_bytes(...) larger than that
 * is rejected with ATTN_ERR_WORKSPACE (see attn_last_error) before anything runs.  The first
 * call on a device looks up the array's address on that device (cudaGetSymbolAddress); make
 * it before any stream capture there.  The lookup happens once per device per process (safe
 * when several host threads make their first call at once) and is kept, so the entry point
 * must not be used after cudaDeviceReset in the same process.  All calls share the array, which keeps the last
 * call's contents; each call rewrites the table before reading it, but calls that overlap on the
 * GPU (unordered streams) race on it.  No cudaMalloc, cudaFree or allocating library call is
 * made.  Other arguments, outputs and errors as for attn_bwd.
 */
#define ATTN_BWD_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
int attn_bwd_noalloc(int dtype, int B, int H, int n, int d, float c,
                     const void* q, const void* k, const void* v, const void* o,
                     const float* lse, const void* d_o,
                     int mask_kind, const uint32_t* mask_bits, int64_t mask_row_words,
                     int64_t mask_head_stride_words, int kv_block,
                     void* dq, void* dk, void* dv, void* stream);

/*
 * Synchronises `stream`, then reads and clears the device status word of the current device.
 * Returns ATTN_OK, ATTN_WARN_EMPTY_ROW, ATTN_ERR_DEVICE_TIMEOUT (a bounded wait inside a kernel
 * gave up; the kernel freed its resources and returned without finishing) or ATTN_ERR_CUDA.
 */
int attn_device_status(void* stream);

/*
 * Self-test of the failure path (no counterpart on the pages): launches one warp that waits,
 * with the same bounded wait every kernel of the library uses, on a barrier nothing ever
 * completes.  After the wait's limit (2 s) the kernel records a timeout in the device status
 * word and returns, so the next attn_device_status(stream) returns ATTN_ERR_DEVICE_TIMEOUT
 * and the CUDA context stays usable.  Asynchronous on `stream`.
 */
int attn_selftest_wait_timeout(void* stream);

/*
 * Self-test of the exponential the forward kernels can compute on the FMA pipe instead of the
 * MUFU unit (no counterpart on the pages): for the n float32 values x (device pointers),
 * y_fma[i] = 2^x[i] by range reduction to [-1/2, 1/2] and a degree-3 relative-minimax
 * polynomial (relative error below 7.5e-5; 0 for x < -125 and x = -inf), and
 * y_mufu[i] = ex2.approx.ftz(x[i]).  Returns ATTN_ERR_INVALID_ARG for n < 0 or null pointers.
 * Asynchronous on `stream`.
 */
int attn_selftest_exp2(const float* x, float* y_fma, float* y_mufu, int64_t n, void* stream);

/*
 * Testing aid for the kernels' pipelines (no counterpart on the pages): caps the depth of every
 * shared-memory ring (the forward's K and V rings, the backward's query-block and K/V rings)
 * at `stages` for the calls that follow, in every thread of the process; 0 restores the
 * default (as many stages as shared memory holds).  A ring whose schedule needs two stages
 * keeps two.  The depth changes only when a tile is loaded, never the arithmetic or its order,
 * so results are bit for bit the same at every depth.  While a cap is set, only calls with
 * bf16 inputs, d = v = 128, key block 128 (or 0) and no dropout, and the FP8 forward with
 * d = 128 and per-tensor scales, run (one instantiation of each kernel reads its depths at
 * launch; the others keep them constant and cost nothing); other calls return
 * ATTN_ERR_UNSUPPORTED.  Returns ATTN_ERR_INVALID_ARG unless 0 <= stages <= 4.
 */
int attn_debug_set_ring_stages(int stages);

/* Message describing the calling thread's most recent failed call ("" if none). */
const char* attn_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* EXACTATTN_H */
