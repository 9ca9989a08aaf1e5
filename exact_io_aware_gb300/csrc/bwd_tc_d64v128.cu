// tcgen05 backward kernels for keys of width 64 and values of width 128.
#include "bwd_tc_launch.cuh"

namespace ea {
int launch_bwd_tc_d64v128(bool bf16, const AttnArgs& a, float* table, cudaStream_t s,
                           std::string& err) {
  return bwd::run_d<64, 128>(bf16, a, table, s, err);
}
}  // namespace ea
