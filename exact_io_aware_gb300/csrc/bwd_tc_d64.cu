// tcgen05 backward kernels (dK/dV and dQ) for head dimension 64.
#include "bwd_tc_launch.cuh"

namespace ea {
int launch_bwd_tc_d64(bool bf16, const AttnArgs& a, float* table, cudaStream_t s, std::string& err) {
  return bf16 ? bwd::run<true, 64>(a, table, s, err) : bwd::run<false, 64>(a, table, s, err);
}
}  // namespace ea
