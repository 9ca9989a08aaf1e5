// tcgen05 forward kernels for head dimension 32.
#include "fwd_tc_launch.cuh"

namespace ea {
int launch_fwd_tc_d32(bool bf16, const AttnArgs& a, cudaStream_t s, std::string& err) {
  return fwd::launch_d<32>(bf16, a, s, err);
}
}  // namespace ea
