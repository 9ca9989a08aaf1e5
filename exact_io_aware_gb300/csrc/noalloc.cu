// attn_bwd_noalloc: the backward pass without a caller-provided workspace.
//
// Some callers cannot allocate device memory when they call the backward: an engine or
// framework that owns every device allocation and gives its plugins no allocator, or a
// system that fixes its whole memory budget at start-up and forbids cudaMalloc afterwards.
// Such callers can pass inputs and outputs they already own, but not the float32 scratch
// (the per-row table of LSE*log2(e) and D) that attn_bwd expects in `workspace`.  This entry
// point takes that scratch from one file-scope device array instead.
//
// Facts a caller must know:
//  * The array is kScratchBytes (32 MiB) of device memory.  Every GPU on which this library is
//    loaded holds it until the process exits, whether or not this entry point is used.
//  * A call needs attn_bwd_workspace_bytes(dtype, B, H, n, d) <= kScratchBytes; larger
//    problems are rejected with ATTN_ERR_WORKSPACE before anything is launched.
//  * The first call on each device looks up the array's device address with
//    cudaGetSymbolAddress while that device is current; make that first call before any
//    stream capture on the device.  The lookup runs once per device for the life of the
//    process (std::call_once, so host threads making their first calls at the same time are
//    safe) and its result is kept: after cudaDeviceReset the library's module is gone and
//    this entry point must not be used again in that process.
//  * All calls share the one array and it keeps the last call's contents.  Each call rewrites
//    the whole table before reading it, so stale contents never leak into results,
//    but two calls whose work overlaps on the GPU (different streams, no ordering between
//    them) race on the array and give wrong gradients.  Order such calls on one stream.
//  * It calls no cudaMalloc, cudaFree or allocating library routine; everything else behaves
//    as attn_bwd (same arguments, same outputs, same errors).
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <string>

#include "exactattn.h"
#include "kernels.h"

namespace {

constexpr size_t kScratchBytes = ATTN_BWD_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;

// The array's device address on one device, looked up once.  std::call_once orders the
// lookup before every reader, so concurrent first calls from several host threads neither
// race nor look it up twice.
struct DeviceScratch {
  std::once_flag once;
  void* ptr = nullptr;
  cudaError_t err = cudaSuccess;
};
DeviceScratch g_scratch[kMaxDevices];

// Device address of g_bwd_scratch on the current device.
int scratch_ptr(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    ea::set_last_error(std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    return ATTN_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    ea::set_last_error("device ordinal too large");
    return ATTN_ERR_UNSUPPORTED;
  }
  DeviceScratch& s = g_scratch[dev];
  std::call_once(s.once, [&s] {
    void* p = nullptr;
    s.err = cudaGetSymbolAddress(&p, g_bwd_scratch);
    s.ptr = s.err == cudaSuccess ? p : nullptr;
  });
  if (s.err != cudaSuccess || s.ptr == nullptr) {
    ea::set_last_error(std::string("cudaGetSymbolAddress(scratch): ") + cudaGetErrorString(s.err));
    return ATTN_ERR_CUDA;
  }
  *out = s.ptr;
  return ATTN_OK;
}

}  // namespace

extern "C" int attn_bwd_noalloc(int dtype, int B, int H, int n, int d, float c, const void* q,
                                const void* k, const void* v, const void* o, const float* lse,
                                const void* d_o, int mask_kind, const uint32_t* mask_bits,
                                int64_t mask_row_words, int64_t mask_head_stride_words,
                                int kv_block, void* dq, void* dk, void* dv, void* stream) {
  // attn_bwd checks every other argument; only a problem larger than the array is refused here.
  const size_t need = attn_bwd_workspace_bytes(dtype, B, H, n, d);
  if (need > kScratchBytes) {
    ea::set_last_error("attn_bwd_noalloc: the problem needs " + std::to_string(need) +
                       " bytes of scratch, more than the " + std::to_string(kScratchBytes) +
                       " bytes it holds; use attn_bwd with a caller workspace");
    return ATTN_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  if (int rc = scratch_ptr(&scratch)) return rc;
  return attn_bwd(dtype, B, H, n, d, c, q, k, v, o, lse, d_o, mask_kind, mask_bits,
                  mask_row_words, mask_head_stride_words, kv_block, dq, dk, dv, scratch,
                  kScratchBytes, stream);
}
