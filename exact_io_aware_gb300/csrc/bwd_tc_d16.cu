// tcgen05 backward kernels (dK/dV and dQ) for head dimension 16.
#include "bwd_tc_launch.cuh"

namespace ea {
int launch_bwd_tc_d16(bool bf16, const AttnArgs& a, float* table, cudaStream_t s, std::string& err) {
  return bwd::run_d<16>(bf16, a, table, s, err);
}
}  // namespace ea
