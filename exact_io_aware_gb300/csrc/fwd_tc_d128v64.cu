// tcgen05 forward kernels for keys of width 128 and values of width 64.
#include "fwd_tc_launch.cuh"

namespace ea {
int launch_fwd_tc_d128v64(bool bf16, const AttnArgs& a, cudaStream_t s, std::string& err) {
  return fwd::launch_d<128, 64>(bf16, a, s, err);
}
}  // namespace ea
