// Head-dimension dispatch of the tcgen05 forward kernels.
#include "kernels.h"

namespace ea {
int launch_fwd_tc_d16(bool bf16, const AttnArgs& a, cudaStream_t s, std::string& err);
int launch_fwd_tc_d32(bool bf16, const AttnArgs& a, cudaStream_t s, std::string& err);
int launch_fwd_tc_d64(bool bf16, const AttnArgs& a, cudaStream_t s, std::string& err);
int launch_fwd_tc_d128(bool bf16, const AttnArgs& a, cudaStream_t s, std::string& err);

int launch_fwd_tc(bool bf16, const AttnArgs& a, cudaStream_t s, std::string& err) {
  switch (a.d) {
    case 16: return launch_fwd_tc_d16(bf16, a, s, err);
    case 32: return launch_fwd_tc_d32(bf16, a, s, err);
    case 64: return launch_fwd_tc_d64(bf16, a, s, err);
    case 128: return launch_fwd_tc_d128(bf16, a, s, err);
    default: err = "head dimension must be 16, 32, 64 or 128"; return -2;
  }
}
}  // namespace ea
