// tcgen05 forward kernels for keys of width 64 and values of width 128.
#include "fwd_tc_launch.cuh"

namespace ea {
int launch_fwd_tc_d64v128(bool bf16, const AttnArgs& a, cudaStream_t s, std::string& err) {
  return fwd::launch_d<64, 128>(bf16, a, s, err);
}
}  // namespace ea
