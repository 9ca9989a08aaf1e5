// C ABI of the exact tiled attention library: argument checks, dispatch to the kernels,
// error reporting and the device status word.  See include/exactattn.h for the contract.
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <mutex>
#include <string>

#include "exactattn.h"
#include "kernels.h"
#include "ptx.cuh"

namespace {

thread_local std::string g_last_error;

// Cap on every kernel's shared-memory ring depth (attn_debug_set_ring_stages; 0 = none).
std::atomic<int> g_ring_stages{0};

// One status word per device, in static device memory (no allocation).  Kernels OR flags
// into it; attn_device_status reads and clears it.
__device__ uint32_t g_status_word;

constexpr int kMaxDevices = 64;

// Per-device facts looked up once (std::call_once orders each lookup before every reader, so
// host threads making their first calls at the same time neither race nor repeat it).
struct DeviceInfo {
  std::once_flag status_once, sm_once;
  uint32_t* status = nullptr;
  cudaError_t status_err = cudaSuccess;
  int sms = 0;
};
DeviceInfo g_dev[kMaxDevices];

int fail(int code, const std::string& msg) {
  g_last_error = msg;
  return code;
}

// An NVTX range named after the entry point, open for the length of the host call (the range
// marks the call's argument checks and launches in a timeline; the kernels are asynchronous).
struct CallRange {
  explicit CallRange(const char* name) { nvtxRangePushA(name); }
  ~CallRange() { nvtxRangePop(); }
  CallRange(const CallRange&) = delete;
  CallRange& operator=(const CallRange&) = delete;
};

int status_ptr(uint32_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(ATTN_ERR_UNSUPPORTED, "device ordinal too large");
  // Bind the device's primary context to the calling thread: the tensor-map encoder is a driver
  // call and fails on a thread (an autograd worker, say) whose first CUDA call it would be.
  e = cudaSetDevice(dev);
  if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, std::string("cudaSetDevice: ") + cudaGetErrorString(e));
  DeviceInfo& info = g_dev[dev];
  std::call_once(info.status_once, [&info] {
    void* p = nullptr;
    info.status_err = cudaGetSymbolAddress(&p, g_status_word);
    info.status = info.status_err == cudaSuccess ? static_cast<uint32_t*>(p) : nullptr;
  });
  if (info.status_err != cudaSuccess || !info.status)
    return fail(ATTN_ERR_CUDA, std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(info.status_err));
  *out = info.status;
  return ATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int kMaxSplits = 32;
size_t round256(size_t x) { return (x + 255) / 256 * 256; }

// Streaming multiprocessors of the current device (looked up once per device).
int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  DeviceInfo& info = g_dev[dev];
  std::call_once(info.sm_once, [&info, dev] {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess) info.sms = v;
  });
  return info.sms;
}

// Library choice of the key split (at most one share per key block and at most kMaxSplits).
// With several query tiles per head: no split once the tiles fill the multiprocessors (a split
// adds float32 partials of every row), else enough shares for one full wave.  With a single
// query tile per head (a key/value cache read by a few queries, where the keys are the work):
// the smallest share count whose CTAs cover every multiprocessor and fill the last wave at
// least 90 %, failing that the count with the fullest waves.
int auto_splits(int dtype, int B, int H, int nq, int nk, int kv_block) {
  const int rows_per_cta = dtype == ATTN_F32 ? 32 : 256;
  const int bn = kv_block ? kv_block : (dtype == ATTN_F32 ? 64 : 128);
  const int64_t ctas = static_cast<int64_t>((nq + rows_per_cta - 1) / rows_per_cta) * B * H;
  const int sms = sm_count();
  const int max_s = std::min(kMaxSplits, (nk + bn - 1) / bn);
  if (sms <= 0 || max_s <= 1) return 1;
  if (nq > rows_per_cta) {
    if (ctas >= sms) return 1;
    return static_cast<int>(std::min<int64_t>(max_s, (sms + ctas - 1) / ctas));
  }
  int best = 1;
  double best_fill = 0.0;
  for (int sp = 1; sp <= max_s; ++sp) {
    const int64_t total = ctas * sp;
    const int64_t waves = (total + sms - 1) / sms;
    const double fill = static_cast<double>(total) / static_cast<double>(waves * sms);
    if (total >= sms && fill >= 0.9) return sp;
    if (fill > best_fill + 1e-9) {
      best_fill = fill;
      best = sp;
    }
  }
  return best;
}

size_t split_part_bytes(int B, int H, int n, int d, int splits) {
  return round256(static_cast<size_t>(splits) * B * H * n * d * sizeof(float));
}

size_t split_ws_bytes(int B, int H, int n, int d, int splits) {
  return split_part_bytes(B, H, n, d, splits) +
         round256(static_cast<size_t>(splits) * B * H * n * sizeof(float));
}

// n: query rows; nk: keys (the bitmap's words cover the keys).
int check_common(int dtype, int B, int H, int n, int d, const void* q, const void* k,
                 const void* v, int mask_kind, const uint32_t* bits, int64_t row_words,
                 int64_t head_stride, int kv_block, int nk = -1) {
  if (nk < 0) nk = n;
  if (dtype < ATTN_F32 || dtype > ATTN_BF16) return fail(ATTN_ERR_INVALID_ARG, "unknown dtype");
  if (B < 1 || H < 1 || n < 1) return fail(ATTN_ERR_INVALID_ARG, "B, H and n must be positive");
  if (d != 16 && d != 32 && d != 64 && d != 128)
    return fail(ATTN_ERR_UNSUPPORTED, "head dimension must be 16, 32, 64 or 128");
  if (static_cast<int64_t>(B) * H > 65535)
    return fail(ATTN_ERR_UNSUPPORTED, "B * H must be at most 65535");
  if (kv_block != 0 && kv_block != 32 && kv_block != 64 && kv_block != 128)
    return fail(ATTN_ERR_UNSUPPORTED, "kv_block must be 0, 32, 64 or 128");
  if (!q || !k || !v) return fail(ATTN_ERR_INVALID_ARG, "null input pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v))
    return fail(ATTN_ERR_ALIGNMENT, "q, k and v must be 16-byte aligned");
  if (mask_kind < ATTN_MASK_NONE || mask_kind > ATTN_MASK_BITMAP)
    return fail(ATTN_ERR_INVALID_ARG, "unknown mask kind");
  if (mask_kind == ATTN_MASK_BITMAP) {
    if (!bits) return fail(ATTN_ERR_INVALID_ARG, "bitmap mask without mask_bits");
    if ((reinterpret_cast<uintptr_t>(bits) & 3u) != 0)
      return fail(ATTN_ERR_ALIGNMENT, "mask_bits must be 4-byte aligned");
    if (row_words < (nk + 31) / 32)
      return fail(ATTN_ERR_INVALID_ARG, "mask_row_words < ceil(keys/32)");
    if (head_stride < 0) return fail(ATTN_ERR_INVALID_ARG, "negative mask_head_stride_words");
  }
  return ATTN_OK;
}

ea::AttnArgs make_args(int B, int H, int n, int d, float c, const void* q, const void* k,
                       const void* v, int mask_kind, const uint32_t* bits, int64_t row_words,
                       int64_t head_stride, int kv_block) {
  ea::AttnArgs a{};
  a.B = B;
  a.H = H;
  a.n = n;
  a.d = d;
  a.v_dim = d;
  a.c = c;
  a.q = q;
  a.k = k;
  a.v = v;
  a.mask_kind = mask_kind;
  a.mask_bits = mask_kind == ATTN_MASK_BITMAP ? bits : nullptr;
  a.mask_row_words = row_words;
  a.mask_head_stride_words = head_stride;
  a.kv_block = kv_block;
  a.num_splits = 1;
  a.nk = n;
  a.ring_stages = g_ring_stages.load(std::memory_order_relaxed);
  a.fwd_rows_cta = 256;
  a.sms = sm_count();
  return a;
}

// Value width v of V, O, dO and dV: v = d, or (d, v) one of the pairs with instantiated kernels.
int check_vdim(int d, int v_dim) {
  if (v_dim == d) return ATTN_OK;
  if ((d == 64 && v_dim == 128) || (d == 128 && v_dim == 64)) return ATTN_OK;
  return fail(ATTN_ERR_UNSUPPORTED, "value width v != d is supported for (d, v) = (64, 128) and (128, 64)");
}

// One warp waits, with the library's bounded wait, on an mbarrier that nothing arrives on.
__global__ void selftest_wait_kernel(uint32_t* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    ea::mbar_init(&bar, 1);
    ea::fence_barrier_init();
  }
  __syncwarp();
  ea::mbar_wait(&bar, 0, status, 0x3F);
}

// y_fma[i] = ex2_fma(x[i]) (FMA pipe), y_mufu[i] = ex2.approx.ftz(x[i]) (MUFU unit).
__global__ void selftest_exp2_kernel(const float* x, float* y_fma, float* y_mufu, int64_t n) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    y_fma[i] = ea::ex2_fma(x[i]);
    y_mufu[i] = ea::ex2(x[i]);
  }
}

}  // namespace

void ea::set_last_error(const std::string& msg) { g_last_error = msg; }

extern "C" {

}  // extern "C"

namespace {

// Dropout arguments of a call: p in [0, 1); 8-bit threshold t = floor(p 256 + 1/2) <= 255
// (the drop probability realised is t / 256), scale 256 / (256 - t).
int set_dropout(float p_drop, uint64_t seed, ea::AttnArgs& a) {
  if (!(p_drop >= 0.0f && p_drop < 1.0f))
    return fail(ATTN_ERR_INVALID_ARG, "p_drop must lie in [0, 1)");
  const int t = static_cast<int>(std::floor(static_cast<double>(p_drop) * 256.0 + 0.5));
  if (t > 255) return fail(ATTN_ERR_INVALID_ARG, "p_drop rounds to 1 at the mask's 1/256 resolution");
  a.dropout = p_drop > 0.0f;
  a.drop.thr4 = static_cast<uint32_t>(t) * 0x01010101u;
  a.drop.scale = static_cast<float>(256.0 / (256.0 - t));
  a.drop.seed_lo = static_cast<uint32_t>(seed);
  a.drop.seed_hi = static_cast<uint32_t>(seed >> 32);
  return ATTN_OK;
}

// Every forward entry point: nq query rows against nk keys (nk = nq for square attention),
// optional dropout, and a key split of `splits` shares (1 = one pass straight into o, lse).
int fwd_general(int dtype, int B, int H, int nq, int nk, int d, int v_dim, float c, const void* q,
                const void* k, const void* v, int mask_kind, const uint32_t* mask_bits,
                int64_t mask_row_words, int64_t mask_head_stride_words, int kv_block,
                float p_drop, uint64_t seed, int splits, void* o, float* lse, void* workspace,
                size_t workspace_bytes, void* stream) {
  if (nk < 1) return fail(ATTN_ERR_INVALID_ARG, "the key length must be positive");
  if (int rc = check_common(dtype, B, H, nq, d, q, k, v, mask_kind, mask_bits, mask_row_words,
                            mask_head_stride_words, kv_block, nk))
    return rc;
  if (int rc = check_vdim(d, v_dim)) return rc;
  if (!o || !lse) return fail(ATTN_ERR_INVALID_ARG, "null output pointer");
  if (!aligned16(o)) return fail(ATTN_ERR_ALIGNMENT, "o must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
    return fail(ATTN_ERR_ALIGNMENT, "lse must be 4-byte aligned");
  ea::AttnArgs a = make_args(B, H, nq, d, c, q, k, v, mask_kind, mask_bits, mask_row_words,
                             mask_head_stride_words, kv_block);
  a.nk = nk;
  a.v_dim = v_dim;
  a.o_out = o;
  a.lse = lse;
  if (int rc = set_dropout(p_drop, seed, a)) return rc;
  // One 128-row tile per CTA when two-tile CTAs would fill at most half the multiprocessors:
  // twice the CTAs then run at once, and each finishes its tile sooner than a pair.
  if (splits == 1 && dtype != ATTN_F32) {
    const int64_t ctas = static_cast<int64_t>((nq + 255) / 256) * B * H;
    const int sms = sm_count();
    if (sms > 0 && 2 * ctas <= sms) a.fwd_rows_cta = 128;
  }
  if (splits > 1) {
    const size_t need = split_ws_bytes(B, H, nq, v_dim, splits);
    if (!workspace || workspace_bytes < need)
      return fail(ATTN_ERR_WORKSPACE,
                  "workspace missing or smaller than attn_fwd_split_workspace_bytes");
    if (!aligned16(workspace))
      return fail(ATTN_ERR_ALIGNMENT, "workspace must be 16-byte aligned");
    a.num_splits = splits;
    a.o_part = static_cast<float*>(workspace);
    a.lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                          split_part_bytes(B, H, nq, v_dim, splits));
  }
  if (int rc = status_ptr(&a.status)) return rc;
  if (a.ring_stages != 0 && dtype == ATTN_F32)
    return fail(ATTN_ERR_UNSUPPORTED, "a ring-depth cap applies to the tensor-core kernels");
  std::string err;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int rc = dtype == ATTN_F32 ? ea::launch_fwd_f32(a, s, err)
                             : ea::launch_fwd_tc(dtype == ATTN_BF16, a, s, err);
  if (rc) return fail(rc, err);
  if (splits > 1) {
    rc = ea::launch_merge(dtype, splits, static_cast<int64_t>(B) * H * nq, v_dim, a.o_part,
                          a.lse_part, o, lse, a.status, s, err);
    if (rc) return fail(rc, err);
  }
  return ATTN_OK;
}

}  // namespace

extern "C" {

int attn_fwd(int dtype, int B, int H, int n, int d, float c, const void* q, const void* k,
             const void* v, int mask_kind, const uint32_t* mask_bits, int64_t mask_row_words,
             int64_t mask_head_stride_words, int kv_block, void* o, float* lse, void* stream) {
  CallRange range("attn_fwd");
  return fwd_general(dtype, B, H, n, n, d, d, c, q, k, v, mask_kind, mask_bits, mask_row_words,
                     mask_head_stride_words, kv_block, 0.0f, 0, 1, o, lse, nullptr, 0, stream);
}

int attn_fwd_dropout(int dtype, int B, int H, int n, int d, float c, const void* q, const void* k,
                     const void* v, int mask_kind, const uint32_t* mask_bits,
                     int64_t mask_row_words, int64_t mask_head_stride_words, int kv_block,
                     float p_drop, uint64_t seed, void* o, float* lse, void* stream) {
  CallRange range("attn_fwd_dropout");
  return fwd_general(dtype, B, H, n, n, d, d, c, q, k, v, mask_kind, mask_bits, mask_row_words,
                     mask_head_stride_words, kv_block, p_drop, seed, 1, o, lse, nullptr, 0,
                     stream);
}

int attn_fwd_split_count(int dtype, int B, int H, int n, int d, int kv_block) {
  if (B < 1 || H < 1 || n < 1 || d < 1) return 0;
  return auto_splits(dtype, B, H, n, n, kv_block);
}

int attn_fwd_kv_split_count(int dtype, int B, int H, int n_q, int n_kv, int d, int kv_block) {
  if (B < 1 || H < 1 || n_q < 1 || n_kv < 1 || d < 1) return 0;
  return auto_splits(dtype, B, H, n_q, n_kv, kv_block);
}

size_t attn_fwd_split_workspace_bytes(int dtype, int B, int H, int n, int d, int num_splits) {
  (void)dtype;
  if (B < 1 || H < 1 || n < 1 || d < 1 || num_splits < 1 || num_splits > kMaxSplits) return 0;
  if (num_splits == 1) return 0;
  return split_ws_bytes(B, H, n, d, num_splits);
}

int attn_fwd_split(int dtype, int B, int H, int n, int d, float c, const void* q, const void* k,
                   const void* v, int mask_kind, const uint32_t* mask_bits, int64_t mask_row_words,
                   int64_t mask_head_stride_words, int kv_block, int num_splits, void* o,
                   float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  CallRange range("attn_fwd_split");
  if (num_splits < 0 || num_splits > kMaxSplits)
    return fail(ATTN_ERR_INVALID_ARG, "num_splits must be 0 (library choice) or 1..32");
  if (B < 1 || H < 1 || n < 1) return fail(ATTN_ERR_INVALID_ARG, "B, H and n must be positive");
  const int splits = num_splits ? num_splits : auto_splits(dtype, B, H, n, n, kv_block);
  return fwd_general(dtype, B, H, n, n, d, d, c, q, k, v, mask_kind, mask_bits, mask_row_words,
                     mask_head_stride_words, kv_block, 0.0f, 0, splits, o, lse, workspace,
                     workspace_bytes, stream);
}

int attn_fwd_kv(int dtype, int B, int H, int n_q, int n_kv, int d, float c, const void* q,
                const void* k, const void* v, int mask_kind, const uint32_t* mask_bits,
                int64_t mask_row_words, int64_t mask_head_stride_words, int kv_block,
                int num_splits, void* o, float* lse, void* workspace, size_t workspace_bytes,
                void* stream) {
  CallRange range("attn_fwd_kv");
  if (num_splits < 0 || num_splits > kMaxSplits)
    return fail(ATTN_ERR_INVALID_ARG, "num_splits must be 0 (library choice) or 1..32");
  if (B < 1 || H < 1 || n_q < 1 || n_kv < 1)
    return fail(ATTN_ERR_INVALID_ARG, "B, H, n_q and n_kv must be positive");
  const int splits = num_splits ? num_splits : auto_splits(dtype, B, H, n_q, n_kv, kv_block);
  return fwd_general(dtype, B, H, n_q, n_kv, d, d, c, q, k, v, mask_kind, mask_bits,
                     mask_row_words, mask_head_stride_words, kv_block, 0.0f, 0, splits, o, lse,
                     workspace, workspace_bytes, stream);
}

int attn_fwd_fp8(int B, int H, int n, int d, float c, const void* q8, const void* k8,
                 const void* vt8, float q_scale, float k_scale, float v_scale, int mask_kind,
                 const uint32_t* mask_bits, int64_t mask_row_words,
                 int64_t mask_head_stride_words, void* o, float* lse, void* stream) {
  CallRange range("attn_fwd_fp8");
  if (d != 64 && d != 128) return fail(ATTN_ERR_UNSUPPORTED, "the FP8 forward supports d = 64 and 128");
  if (int rc = check_common(ATTN_BF16, B, H, n, d, q8, k8, vt8, mask_kind, mask_bits,
                            mask_row_words, mask_head_stride_words, 0))
    return rc;
  if (n % 16 != 0) return fail(ATTN_ERR_UNSUPPORTED, "the FP8 forward needs n a multiple of 16");
  if (!(q_scale > 0.0f) || !(k_scale > 0.0f) || !(v_scale > 0.0f) || !std::isfinite(q_scale) ||
      !std::isfinite(k_scale) || !std::isfinite(v_scale))
    return fail(ATTN_ERR_INVALID_ARG, "the FP8 scales must be finite and positive");
  if (!o || !lse) return fail(ATTN_ERR_INVALID_ARG, "null output pointer");
  if (!aligned16(o)) return fail(ATTN_ERR_ALIGNMENT, "o must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
    return fail(ATTN_ERR_ALIGNMENT, "lse must be 4-byte aligned");
  ea::AttnArgs a = make_args(B, H, n, d, c, q8, k8, vt8, mask_kind, mask_bits, mask_row_words,
                             mask_head_stride_words, 0);
  a.o_out = o;
  a.lse = lse;
  if (int rc = status_ptr(&a.status)) return rc;
  std::string err;
  int rc = ea::launch_fwd_fp8(a, vt8, q_scale, k_scale, v_scale, nullptr, nullptr, nullptr,
                              static_cast<cudaStream_t>(stream), err);
  if (rc) return fail(rc, err);
  return ATTN_OK;
}

int attn_fwd_fp8_blocks(int B, int H, int n, int d, float c, const void* q8, const void* k8,
                        const void* vt8, const float* q_scales, const float* k_scales,
                        const float* v_scales, int mask_kind, const uint32_t* mask_bits,
                        int64_t mask_row_words, int64_t mask_head_stride_words, void* o,
                        float* lse, void* stream) {
  CallRange range("attn_fwd_fp8_blocks");
  if (d != 64 && d != 128) return fail(ATTN_ERR_UNSUPPORTED, "the FP8 forward supports d = 64 and 128");
  if (int rc = check_common(ATTN_BF16, B, H, n, d, q8, k8, vt8, mask_kind, mask_bits,
                            mask_row_words, mask_head_stride_words, 0))
    return rc;
  if (n % 16 != 0) return fail(ATTN_ERR_UNSUPPORTED, "the FP8 forward needs n a multiple of 16");
  if (!q_scales || !k_scales || !v_scales) return fail(ATTN_ERR_INVALID_ARG, "null scale pointer");
  if ((reinterpret_cast<uintptr_t>(q_scales) | reinterpret_cast<uintptr_t>(k_scales) |
       reinterpret_cast<uintptr_t>(v_scales)) & 3u)
    return fail(ATTN_ERR_ALIGNMENT, "scales must be 4-byte aligned");
  if (!std::isfinite(c)) return fail(ATTN_ERR_INVALID_ARG, "c must be finite");
  if (!o || !lse) return fail(ATTN_ERR_INVALID_ARG, "null output pointer");
  if (!aligned16(o)) return fail(ATTN_ERR_ALIGNMENT, "o must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
    return fail(ATTN_ERR_ALIGNMENT, "lse must be 4-byte aligned");
  ea::AttnArgs a = make_args(B, H, n, d, c, q8, k8, vt8, mask_kind, mask_bits, mask_row_words,
                             mask_head_stride_words, 0);
  a.o_out = o;
  a.lse = lse;
  if (int rc = status_ptr(&a.status)) return rc;
  std::string err;
  int rc = ea::launch_fwd_fp8(a, vt8, 1.0f, 1.0f, 1.0f, q_scales, k_scales, v_scales,
                              static_cast<cudaStream_t>(stream), err);
  if (rc) return fail(rc, err);
  return ATTN_OK;
}

int attn_fp8_quantize(int dtype, int B, int H, int n, int d, const void* q, const void* k,
                      const void* v, const int8_t* signs, void* q8, void* k8, void* vt8,
                      float* q_scales, float* k_scales, float* v_scales, void* stream) {
  CallRange range("attn_fp8_quantize");
  if (dtype != ATTN_BF16 && dtype != ATTN_F16)
    return fail(ATTN_ERR_UNSUPPORTED, "the FP8 quantization reads bf16 or fp16 inputs");
  if (d != 64 && d != 128) return fail(ATTN_ERR_UNSUPPORTED, "the FP8 quantization supports d = 64 and 128");
  if (B < 1 || H < 1 || n < 1) return fail(ATTN_ERR_INVALID_ARG, "B, H and n must be positive");
  if (n % 16 != 0) return fail(ATTN_ERR_UNSUPPORTED, "the FP8 quantization needs n a multiple of 16");
  if (!q || !k || !v || !q8 || !k8 || !vt8 || !q_scales || !k_scales || !v_scales)
    return fail(ATTN_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(q8) || !aligned16(k8) ||
      !aligned16(vt8))
    return fail(ATTN_ERR_ALIGNMENT, "tensors must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(q_scales) | reinterpret_cast<uintptr_t>(k_scales) |
       reinterpret_cast<uintptr_t>(v_scales)) & 3u)
    return fail(ATTN_ERR_ALIGNMENT, "scales must be 4-byte aligned");
  if (static_cast<int64_t>(B) * H > 65535)
    return fail(ATTN_ERR_UNSUPPORTED, "B * H above 65535");
  std::string err;
  int rc = ea::launch_fp8_quantize(dtype == ATTN_BF16, B, H, n, d, q, k, v, signs, q8, k8, vt8,
                                   q_scales, k_scales, v_scales, static_cast<cudaStream_t>(stream),
                                   err);
  if (rc) return fail(rc, err);
  return ATTN_OK;
}

int attn_merge(int dtype, int num_parts, int64_t rows, int d, const float* o_parts,
               const float* lse_parts, void* o, float* lse, void* stream) {
  CallRange range("attn_merge");
  if (dtype < ATTN_F32 || dtype > ATTN_BF16) return fail(ATTN_ERR_INVALID_ARG, "unknown dtype");
  if (num_parts < 1 || rows < 1 || d < 4)
    return fail(ATTN_ERR_INVALID_ARG, "num_parts and rows must be positive and d >= 4");
  if (d % 4 != 0) return fail(ATTN_ERR_UNSUPPORTED, "d must be a multiple of 4");
  if (!o_parts || !lse_parts || !o || !lse) return fail(ATTN_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(o_parts) || !aligned16(o))
    return fail(ATTN_ERR_ALIGNMENT, "o_parts and o must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(lse_parts) & 3u) != 0 ||
      (reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
    return fail(ATTN_ERR_ALIGNMENT, "lse_parts and lse must be 4-byte aligned");
  uint32_t* st = nullptr;
  if (int rc = status_ptr(&st)) return rc;
  std::string err;
  int rc = ea::launch_merge(dtype, num_parts, rows, d, o_parts, lse_parts, o, lse, st,
                            static_cast<cudaStream_t>(stream), err);
  if (rc) return fail(rc, err);
  return ATTN_OK;
}

size_t attn_bwd_workspace_bytes(int dtype, int B, int H, int n, int d) {
  if (B < 1 || H < 1 || n < 1 || d < 1) return 0;
  return dtype == ATTN_F32 ? ea::bwd_f32_workspace_bytes(B, H, n, d)
                           : ea::bwd_tc_workspace_bytes(B, H, n, d);
}

}  // extern "C"

namespace {

int bwd_impl(int dtype, int B, int H, int n, int d, int v_dim, float c, const void* q, const void* k,
             const void* v, const void* o, const float* lse, const void* d_o, int mask_kind,
             const uint32_t* mask_bits, int64_t mask_row_words, int64_t mask_head_stride_words,
             int kv_block, float p_drop, uint64_t seed, void* dq, void* dk, void* dv,
             void* workspace, size_t workspace_bytes, void* stream) {
  if (int rc = check_common(dtype, B, H, n, d, q, k, v, mask_kind, mask_bits, mask_row_words,
                            mask_head_stride_words, kv_block))
    return rc;
  if (int rc = check_vdim(d, v_dim)) return rc;
  if (!o || !lse || !d_o) return fail(ATTN_ERR_INVALID_ARG, "null o, lse or d_o");
  if (!dq || !dk || !dv) return fail(ATTN_ERR_INVALID_ARG, "null gradient pointer");
  if (!aligned16(o) || !aligned16(d_o) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return fail(ATTN_ERR_ALIGNMENT, "o, d_o, dq, dk and dv must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
    return fail(ATTN_ERR_ALIGNMENT, "lse must be 4-byte aligned");
  const size_t need = attn_bwd_workspace_bytes(dtype, B, H, n, d);
  if (!workspace || workspace_bytes < need)
    return fail(ATTN_ERR_WORKSPACE, "workspace missing or smaller than attn_bwd_workspace_bytes");
  if (!aligned16(workspace)) return fail(ATTN_ERR_ALIGNMENT, "workspace must be 16-byte aligned");
  ea::AttnArgs a = make_args(B, H, n, d, c, q, k, v, mask_kind, mask_bits, mask_row_words,
                             mask_head_stride_words, kv_block);
  a.v_dim = v_dim;
  a.o = o;
  a.lse = const_cast<float*>(lse);
  a.d_o = d_o;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  if (int rc = set_dropout(p_drop, seed, a)) return rc;
  if (int rc = status_ptr(&a.status)) return rc;
  if (a.ring_stages != 0 && dtype == ATTN_F32)
    return fail(ATTN_ERR_UNSUPPORTED, "a ring-depth cap applies to the tensor-core kernels");
  std::string err;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int rc = dtype == ATTN_F32 ? ea::launch_bwd_f32(a, s, err)
                             : ea::launch_bwd_tc(dtype == ATTN_BF16, a, s, err);
  if (rc) return fail(rc, err);
  return ATTN_OK;
}

}  // namespace

extern "C" {

int attn_bwd(int dtype, int B, int H, int n, int d, float c, const void* q, const void* k,
             const void* v, const void* o, const float* lse, const void* d_o, int mask_kind,
             const uint32_t* mask_bits, int64_t mask_row_words, int64_t mask_head_stride_words,
             int kv_block, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
             void* stream) {
  CallRange range("attn_bwd");
  return bwd_impl(dtype, B, H, n, d, d, c, q, k, v, o, lse, d_o, mask_kind, mask_bits,
                  mask_row_words, mask_head_stride_words, kv_block, 0.0f, 0, dq, dk, dv,
                  workspace, workspace_bytes, stream);
}

int attn_bwd_dropout(int dtype, int B, int H, int n, int d, float c, const void* q,
                     const void* k, const void* v, const void* o, const float* lse,
                     const void* d_o, int mask_kind, const uint32_t* mask_bits,
                     int64_t mask_row_words, int64_t mask_head_stride_words, int kv_block,
                     float p_drop, uint64_t seed, void* dq, void* dk, void* dv, void* workspace,
                     size_t workspace_bytes, void* stream) {
  CallRange range("attn_bwd_dropout");
  return bwd_impl(dtype, B, H, n, d, d, c, q, k, v, o, lse, d_o, mask_kind, mask_bits,
                  mask_row_words, mask_head_stride_words, kv_block, p_drop, seed, dq, dk, dv,
                  workspace, workspace_bytes, stream);
}

int attn_fwd_vdim(int dtype, int B, int H, int n, int d, int v_dim, float c, const void* q,
                  const void* k, const void* v, int mask_kind, const uint32_t* mask_bits,
                  int64_t mask_row_words, int64_t mask_head_stride_words, int kv_block,
                  float p_drop, uint64_t seed, void* o, float* lse, void* stream) {
  CallRange range("attn_fwd_vdim");
  return fwd_general(dtype, B, H, n, n, d, v_dim, c, q, k, v, mask_kind, mask_bits,
                     mask_row_words, mask_head_stride_words, kv_block, p_drop, seed, 1, o, lse,
                     nullptr, 0, stream);
}

int attn_bwd_vdim(int dtype, int B, int H, int n, int d, int v_dim, float c, const void* q,
                  const void* k, const void* v, const void* o, const float* lse, const void* d_o,
                  int mask_kind, const uint32_t* mask_bits, int64_t mask_row_words,
                  int64_t mask_head_stride_words, int kv_block, float p_drop, uint64_t seed,
                  void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                  void* stream) {
  CallRange range("attn_bwd_vdim");
  return bwd_impl(dtype, B, H, n, d, v_dim, c, q, k, v, o, lse, d_o, mask_kind, mask_bits,
                  mask_row_words, mask_head_stride_words, kv_block, p_drop, seed, dq, dk, dv,
                  workspace, workspace_bytes, stream);
}

int attn_device_status(void* stream) {
  CallRange range("attn_device_status");
  uint32_t* p = nullptr;
  if (int rc = status_ptr(&p)) return rc;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess)
    return fail(ATTN_ERR_CUDA, std::string("cudaStreamSynchronize: ") + cudaGetErrorString(e));
  uint32_t word = 0;
  e = cudaMemcpy(&word, p, sizeof(word), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(p, 0, sizeof(word));
  if (e != cudaSuccess)
    return fail(ATTN_ERR_CUDA, std::string("status word: ") + cudaGetErrorString(e));
  if (word & 1u) {
    char buf[96];
    snprintf(buf, sizeof(buf), "an in-kernel wait gave up (sites 0x%02x)", (word >> 8) & 0xFFu);
    return fail(ATTN_ERR_DEVICE_TIMEOUT, buf);
  }
  if (word & 2u) return ATTN_WARN_EMPTY_ROW;
  return ATTN_OK;
}

int attn_selftest_wait_timeout(void* stream) {
  CallRange range("attn_selftest_wait_timeout");
  uint32_t* st = nullptr;
  if (int rc = status_ptr(&st)) return rc;
  selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(st);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return fail(ATTN_ERR_CUDA, std::string("self-test launch: ") + cudaGetErrorString(e));
  return ATTN_OK;
}

int attn_selftest_exp2(const float* x, float* y_fma, float* y_mufu, int64_t n, void* stream) {
  CallRange range("attn_selftest_exp2");
  if (n < 0) return fail(ATTN_ERR_INVALID_ARG, "n must be non-negative");
  if (n == 0) return ATTN_OK;
  if (!x || !y_fma || !y_mufu) return fail(ATTN_ERR_INVALID_ARG, "null pointer");
  const int64_t blocks = std::min<int64_t>((n + 255) / 256, 4096);
  selftest_exp2_kernel<<<static_cast<unsigned>(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      x, y_fma, y_mufu, n);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return fail(ATTN_ERR_CUDA, std::string("exp2 self-test launch: ") + cudaGetErrorString(e));
  return ATTN_OK;
}

int attn_debug_set_ring_stages(int stages) {
  if (stages < 0 || stages > 4) return fail(ATTN_ERR_INVALID_ARG, "ring stages must be 0 .. 4");
  g_ring_stages.store(stages, std::memory_order_relaxed);
  return ATTN_OK;
}

const char* attn_last_error(void) { return g_last_error.c_str(); }

}  // extern "C"
