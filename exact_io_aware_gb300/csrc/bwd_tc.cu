// tcgen05 backward: D = rowsum(dO * O), then the dK/dV kernel (key tiles) and the dQ kernel
// (query tiles), all on the caller's stream.
#include "kernels.h"

namespace ea {
int launch_bwd_tc_d16(bool, const AttnArgs&, const float*, cudaStream_t, std::string&);
int launch_bwd_tc_d32(bool, const AttnArgs&, const float*, cudaStream_t, std::string&);
int launch_bwd_tc_d64(bool, const AttnArgs&, const float*, cudaStream_t, std::string&);
int launch_bwd_tc_d128(bool, const AttnArgs&, const float*, cudaStream_t, std::string&);

// Workspace: the row table, L2 then D, each [B*H][n_pad] float32 with n_pad = n rounded up to
// 128 (so every 128-row block of it is a whole, 512-byte-aligned bulk copy).
size_t bwd_tc_workspace_bytes(int B, int H, int n, int) {
  const size_t rows = static_cast<size_t>(B) * H * bwd_pad_rows(n);
  return 2 * rows * 4;
}

int launch_bwd_tc(bool bf16, const AttnArgs& a, cudaStream_t s, std::string& err) {
  const int n_pad = bwd_pad_rows(a.n);
  float* L2 = static_cast<float*>(a.workspace);
  float* Dv = L2 + static_cast<size_t>(a.B) * a.H * n_pad;
  if (int rc = launch_bwd_pre_rows(bf16, a, L2, Dv, n_pad, s, err)) return rc;
  switch (a.d) {
    case 16: return launch_bwd_tc_d16(bf16, a, L2, s, err);
    case 32: return launch_bwd_tc_d32(bf16, a, L2, s, err);
    case 64: return launch_bwd_tc_d64(bf16, a, L2, s, err);
    case 128: return launch_bwd_tc_d128(bf16, a, L2, s, err);
    default: err = "head dimension must be 16, 32, 64 or 128"; return -2;
  }
}
}  // namespace ea
