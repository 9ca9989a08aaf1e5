// tcgen05 backward kernels for keys of width 128 and values of width 64.
#include "bwd_tc_launch.cuh"

namespace ea {
int launch_bwd_tc_d128v64(bool bf16, const AttnArgs& a, float* table, cudaStream_t s,
                           std::string& err) {
  return bwd::run_d<128, 64>(bf16, a, table, s, err);
}
}  // namespace ea
