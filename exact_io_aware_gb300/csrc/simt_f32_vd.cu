// float32 forward and backward for keys and values of different widths: (d, v) = (64, 128)
// and (128, 64).
#include "simt_f32.cuh"

namespace ea {

int launch_fwd_f32_vd(const AttnArgs& a, cudaStream_t s, std::string& err) {
  if (a.d == 64 && a.v_dim == 128) return f32::fwd_d<64, 128>(a, s, err);
  if (a.d == 128 && a.v_dim == 64) return f32::fwd_d<128, 64>(a, s, err);
  err = "value width v != d is supported for (d, v) = (64, 128) and (128, 64)";
  return -2;
}

int launch_bwd_f32_vd(const AttnArgs& a, const float* Dv, cudaStream_t s, std::string& err) {
  if (a.d == 64 && a.v_dim == 128) return f32::bwd_d<64, 128>(a, Dv, s, err);
  if (a.d == 128 && a.v_dim == 64) return f32::bwd_d<128, 64>(a, Dv, s, err);
  err = "value width v != d is supported for (d, v) = (64, 128) and (128, 64)";
  return -2;
}

}  // namespace ea
