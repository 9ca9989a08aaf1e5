// float32 forward and backward on the CUDA cores: dispatch over the head dimension (keys and
// values of one width; simt_f32_vd.cu holds the pairs of different widths).
#include "simt_f32.cuh"

namespace ea {

int launch_fwd_f32_vd(const AttnArgs& a, cudaStream_t s, std::string& err);
int launch_bwd_f32_vd(const AttnArgs& a, const float* Dv, cudaStream_t s, std::string& err);

int launch_fwd_f32(const AttnArgs& a, cudaStream_t s, std::string& err) {
  int rc;
  if (a.v_dim != a.d) {
    rc = launch_fwd_f32_vd(a, s, err);
  } else {
    switch (a.d) {
      case 16: rc = f32::fwd_d<16>(a, s, err); break;
      case 32: rc = f32::fwd_d<32>(a, s, err); break;
      case 64: rc = f32::fwd_d<64>(a, s, err); break;
      case 128: rc = f32::fwd_d<128>(a, s, err); break;
      default: err = "head dimension must be 16, 32, 64 or 128"; return -2;
    }
  }
  if (rc) return rc;
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    err = std::string("float32 forward launch: ") + cudaGetErrorString(e);
    return -5;
  }
  return 0;
}

size_t bwd_f32_workspace_bytes(int B, int H, int n, int) {
  return (static_cast<size_t>(B) * H * n * sizeof(float) + 255) / 256 * 256;
}

int launch_bwd_f32(const AttnArgs& a, cudaStream_t s, std::string& err) {
  float* Dv = static_cast<float*>(a.workspace);
  if (int rc = launch_bwd_pre_f32(a, Dv, s, err)) return rc;
  int rc;
  if (a.v_dim != a.d) {
    rc = launch_bwd_f32_vd(a, Dv, s, err);
  } else {
    switch (a.d) {
      case 16: rc = f32::bwd_d<16>(a, Dv, s, err); break;
      case 32: rc = f32::bwd_d<32>(a, Dv, s, err); break;
      case 64: rc = f32::bwd_d<64>(a, Dv, s, err); break;
      case 128: rc = f32::bwd_d<128>(a, Dv, s, err); break;
      default: err = "head dimension must be 16, 32, 64 or 128"; return -2;
    }
  }
  if (rc) return rc;
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    err = std::string("float32 backward launch: ") + cudaGetErrorString(e);
    return -5;
  }
  return 0;
}

}  // namespace ea
