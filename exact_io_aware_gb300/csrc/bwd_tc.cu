// tcgen05 backward: preprocessing (D and a cleared dQ accumulator), the main kernel, and the
// dQ postprocessing, all on the caller's stream.
#include "kernels.h"

namespace ea {
int launch_bwd_tc_d16(bool, const AttnArgs&, float*, float*, cudaStream_t, std::string&);
int launch_bwd_tc_d32(bool, const AttnArgs&, float*, float*, cudaStream_t, std::string&);
int launch_bwd_tc_d64(bool, const AttnArgs&, float*, float*, cudaStream_t, std::string&);
int launch_bwd_tc_d128(bool, const AttnArgs&, float*, float*, cudaStream_t, std::string&);

namespace {
size_t align256(size_t x) { return (x + 255) / 256 * 256; }
}  // namespace

// Workspace: D [B*H*n] float32, then the dQ accumulator [B*H*n*d] float32.
size_t bwd_tc_workspace_bytes(int B, int H, int n, int d) {
  const size_t rows = static_cast<size_t>(B) * H * n;
  return align256(rows * 4) + align256(rows * d * 4);
}

int launch_bwd_tc(bool bf16, const AttnArgs& a, cudaStream_t s, std::string& err) {
  const size_t rows = static_cast<size_t>(a.B) * a.H * a.n;
  float* Dv = static_cast<float*>(a.workspace);
  float* acc = reinterpret_cast<float*>(static_cast<char*>(a.workspace) + align256(rows * 4));
  if (int rc = launch_bwd_pre(bf16 ? 2 : 1, a, Dv, acc, rows * a.d, s, err)) return rc;
  int rc;
  switch (a.d) {
    case 16: rc = launch_bwd_tc_d16(bf16, a, Dv, acc, s, err); break;
    case 32: rc = launch_bwd_tc_d32(bf16, a, Dv, acc, s, err); break;
    case 64: rc = launch_bwd_tc_d64(bf16, a, Dv, acc, s, err); break;
    case 128: rc = launch_bwd_tc_d128(bf16, a, Dv, acc, s, err); break;
    default: err = "head dimension must be 16, 32, 64 or 128"; return -2;
  }
  if (rc) return rc;
  return launch_bwd_post(bf16, a, acc, s, err);
}
}  // namespace ea
