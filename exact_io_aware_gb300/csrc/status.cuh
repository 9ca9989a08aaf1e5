// Device status word shared by every kernel of the library.
//
// Kernels receive a pointer to one 32-bit word.  Bit 0 records that a bounded wait gave up
// (a producer never arrived); bits 8-15 hold the OR of the wait sites that gave up.  Bit 1
// records that some query row had an empty allowed-key set (no output is defined for such a
// row; the library writes zeros and a -inf row statistic).  The host reads and clears the
// word with attn_device_status().
#pragma once
#include <cstdint>

namespace ea {

enum : uint32_t {
  kStatusTimeout = 1u << 0,
  kStatusEmptyRow = 1u << 1,
};

__device__ __forceinline__ void raise_timeout(uint32_t* status, uint32_t site) {
  atomicOr(status, kStatusTimeout | ((site & 0xFFu) << 8));
}

__device__ __forceinline__ void raise_empty_row(uint32_t* status) {
  atomicOr(status, kStatusEmptyRow);
}

__device__ __forceinline__ bool device_timed_out(const uint32_t* status) {
  return (*reinterpret_cast<const volatile uint32_t*>(status) & kStatusTimeout) != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

}  // namespace ea
