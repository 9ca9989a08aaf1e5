// Head-dimension dispatch of the tcgen05 forward kernels.
#include "kernels.h"

namespace ea {
int launch_fwd_tc_d16(bool bf16, const AttnArgs& a, cudaStream_t s, std::string& err);
int launch_fwd_tc_d32(bool bf16, const AttnArgs& a, cudaStream_t s, std::string& err);
int launch_fwd_tc_d64(bool bf16, const AttnArgs& a, cudaStream_t s, std::string& err);
int launch_fwd_tc_d128(bool bf16, const AttnArgs& a, cudaStream_t s, std::string& err);
int launch_fwd_tc_d64v128(bool bf16, const AttnArgs& a, cudaStream_t s, std::string& err);
int launch_fwd_tc_d128v64(bool bf16, const AttnArgs& a, cudaStream_t s, std::string& err);

int launch_fwd_tc(bool bf16, const AttnArgs& a, cudaStream_t s, std::string& err) {
  if (a.v_dim != a.d) {
    if (a.d == 64 && a.v_dim == 128) return launch_fwd_tc_d64v128(bf16, a, s, err);
    if (a.d == 128 && a.v_dim == 64) return launch_fwd_tc_d128v64(bf16, a, s, err);
    err = "value width v != d is supported for (d, v) = (64, 128) and (128, 64)";
    return -2;
  }
  switch (a.d) {
    case 16: return launch_fwd_tc_d16(bf16, a, s, err);
    case 32: return launch_fwd_tc_d32(bf16, a, s, err);
    case 64: return launch_fwd_tc_d64(bf16, a, s, err);
    case 128: return launch_fwd_tc_d128(bf16, a, s, err);
    default: err = "head dimension must be 16, 32, 64 or 128"; return -2;
  }
}
}  // namespace ea
