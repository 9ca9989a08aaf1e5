// Internal interface between the C ABI (api.cu) and the kernel translation units.
#pragma once
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <string>

#include "dropout.cuh"

namespace ea {

enum MaskKind : int { kMaskNone = 0, kMaskCausal = 1, kMaskBitmap = 2 };

// Depth of a shared-memory ring chosen at launch (at most the stage count the kernel's shared
// memory holds): use i of the ring takes stage i mod n in phase parity (i / n) mod 2.  The
// division is a multiply-high by ceil(2^32 / n), exact for every i below 2^31 when n <= 4.
struct Ring {
  uint32_t n;      // stages in use, 1 .. 4
  uint32_t magic;  // ceil(2^32 / n) for n >= 2
  static Ring make(int stages) {
    Ring r{static_cast<uint32_t>(stages), 0u};
    if (stages >= 2) r.magic = static_cast<uint32_t>(((uint64_t(1) << 32) + stages - 1) / stages);
    return r;
  }
#ifdef __CUDACC__
  __device__ __forceinline__ uint32_t div(int i) const {
    return n == 1 ? static_cast<uint32_t>(i) : __umulhi(static_cast<uint32_t>(i), magic);
  }
  __device__ __forceinline__ int stage(int i) const {
    return static_cast<int>(static_cast<uint32_t>(i) - div(i) * n);
  }
  __device__ __forceinline__ uint32_t parity(int i) const { return div(i) & 1u; }
#endif
};

// A ring of N stages fixed at compile time (the production kernels): the same interface as
// Ring with constant divisions.
template <int N>
struct StaticRing {
#ifdef __CUDACC__
  __device__ __forceinline__ static constexpr int stage(int i) { return i % N; }
  __device__ __forceinline__ static constexpr uint32_t parity(int i) { return (i / N) & 1; }
#endif
};

#ifdef __CUDACC__
// The ring a kernel walks: the launch-time depth in the capped instantiations (kCap), else the
// compile-time stage count.
template <bool kCap, int N>
__device__ __forceinline__ auto ring_of(const Ring& r) {
  if constexpr (kCap) {
    return r;
  } else {
    return StaticRing<N>{};
  }
}

// Work item of CTA c in launch order (c = blockIdx.y * nx + blockIdx.x) for a grid of nx items
// per head (rank 0 the heaviest) over ny heads.  Heads are taken in groups of `group`, and
// within a group the items of all its heads go heaviest first: under the causal mask the
// launch then ends on the lightest items of the last group instead of on each head's
// heaviest, which would otherwise start last and hold the tail.  group = 1 is head by head.
__device__ __forceinline__ void work_item(uint32_t c, uint32_t nx, uint32_t ny, uint32_t group,
                                          uint32_t& rank, uint32_t& head) {
  const uint32_t per = group * nx;
  const uint32_t g = c / per;
  const uint32_t h0 = g * group;
  const uint32_t gh = min(group, ny - h0);
  const uint32_t r = c - g * per;
  rank = r / gh;
  head = h0 + r % gh;
}
// Heads per group of the causal work order (16 heads' K, V, Q and dO stay within L2).
constexpr uint32_t kCausalHeadGroup = 16;
#endif

// Stage count of a ring at launch: the caller's cap (0 = none) within [lo, hi].
inline int ring_depth(int cap, int lo, int hi) {
  const int want = cap > 0 ? cap : hi;
  return want < lo ? lo : (want > hi ? hi : want);
}

// Scalar arguments of the forward kernels (tensor maps travel separately).
struct FwdParams {
  int n;    // query rows
  float c;
  int mask_kind;
  const uint32_t* mask_bits;
  int64_t mask_row_words;
  int64_t mask_head_stride_words;
  float* lse;
  uint32_t* status;
  // Key-split forward (gridDim.z = num_splits > 1): CTA z walks only its share of the key
  // blocks and writes the normalised partial O_z (float32, [num_splits][B*H][n][d]) and its
  // LSE_z ([num_splits][B*H][n], -inf where no allowed key fell in the share) instead of o, lse.
  int num_splits;
  float* o_part;
  float* lse_part;
  DropoutArgs drop;  // read only by the dropout instantiations
  int nk;            // keys (n for square attention)
  int off;           // causal offset nk - n: query i sees keys j <= i + off
  int prefetch;      // key blocks requested into L2 ahead of the ring loads (0: none)
  Ring ring_k, ring_v;  // depths of the K and V rings
  int rows_cta;      // query rows per CTA: 256 (two tiles), or 128 when a grid is small
  int next_cta;      // CTAs resident at once (the SM count): the CTA launched that many after
                     // this one has its first tiles requested into L2 (0: none)
};

// Everything a launcher needs; pointers are device pointers.
struct AttnArgs {
  int B, H, n, d;
  int v_dim;  // value width (columns of V, O, dO, dV); d unless the values are wider or narrower
  int nk;  // keys; the forward allows nk != n (queries at the end of the key sequence)
  float c;
  const void* q;
  const void* k;
  const void* v;
  const void* o;   // backward: forward output
  void* o_out;     // forward: output
  float* lse;      // forward: output; backward: input
  const void* d_o;
  void* dq;
  void* dk;
  void* dv;
  int mask_kind;
  const uint32_t* mask_bits;
  int64_t mask_row_words;
  int64_t mask_head_stride_words;
  int kv_block;
  void* workspace;
  size_t workspace_bytes;
  uint32_t* status;
  int num_splits;   // forward: 1, or the number of key shards (partials go to o_part, lse_part)
  float* o_part;
  float* lse_part;
  bool dropout;     // drop probabilities with the mask of dropout.cuh (p > 0)
  DropoutArgs drop;
  int ring_stages;  // cap on the depth of every shared-memory ring (0: as deep as memory allows)
  int fwd_rows_cta;  // forward: query rows per CTA (256, or 128 for grids under half the SMs)
  int sms;           // multiprocessors of the device
};

// Each launcher returns 0 or a negative ATTN_ERR_* code and fills `err` on failure.
int launch_fwd_tc(bool bf16, const AttnArgs& a, cudaStream_t s, std::string& err);
int launch_bwd_tc(bool bf16, const AttnArgs& a, cudaStream_t s, std::string& err);
int launch_fwd_f32(const AttnArgs& a, cudaStream_t s, std::string& err);
int launch_bwd_f32(const AttnArgs& a, cudaStream_t s, std::string& err);

// FP8 forward: a.q, a.k are E4M3 [B*H][n][d], vt8 E4M3 [B*H][d][n] (V transposed), per-tensor
// scales; a.o_out bfloat16.
// sq_blk, sk_blk, sv_blk: per-block scales [heads][ceil(n / 128)], or null for the scalars.
int launch_fwd_fp8(const AttnArgs& a, const void* vt8, float sq, float sk, float sv,
                   const float* sq_blk, const float* sk_blk, const float* sv_blk, cudaStream_t s,
                   std::string& err);

// Block quantization of 16-bit Q, K, V to E4M3 (q8, k8 [heads][n][d], vt8 [heads][d][n]) with
// float32 scales per 128 rows; signs (d entries, or null) turn on incoherent processing.
int launch_fp8_quantize(bool bf16, int B, int H, int n, int d, const void* q, const void* k,
                        const void* v, const int8_t* signs, void* q8, void* k8, void* vt8,
                        float* sq, float* sk, float* sv, cudaStream_t s, std::string& err);

// O = sum_g exp(LSE_g - LSE) O_g, LSE = ln sum_g exp(LSE_g) over num_parts partial results
// (float32 o_part [parts][rows][d], lse_part [parts][rows]); o in the output dtype.
int launch_merge(int dtype_out, int num_parts, int64_t rows, int d, const float* o_part,
                 const float* lse_part, void* o, float* lse, uint32_t* status, cudaStream_t s,
                 std::string& err);

// D_i = sum_a dO[i][a] * O[i][a] for float32 inputs.
int launch_bwd_pre_f32(const AttnArgs& a, float* D, cudaStream_t s, std::string& err);
// Rows per head of the tensor-core backward's row table: n rounded up to 128.
constexpr int bwd_pad_rows(int n) { return (n + 127) / 128 * 128; }

size_t bwd_tc_workspace_bytes(int B, int H, int n, int d);
size_t bwd_f32_workspace_bytes(int B, int H, int n, int d);

// Sets the message attn_last_error() returns on the calling thread.
void set_last_error(const std::string& msg);

}  // namespace ea
