// tcgen05 backward: the dQ kernel (query tiles; it also writes the per-row table of LSE and
// D = rowsum(dO * O)), then the dK/dV kernel (key tiles), both on the caller's stream.
#include "kernels.h"

namespace ea {
int launch_bwd_tc_d16(bool, const AttnArgs&, float*, cudaStream_t, std::string&);
int launch_bwd_tc_d32(bool, const AttnArgs&, float*, cudaStream_t, std::string&);
int launch_bwd_tc_d64(bool, const AttnArgs&, float*, cudaStream_t, std::string&);
int launch_bwd_tc_d128(bool, const AttnArgs&, float*, cudaStream_t, std::string&);
int launch_bwd_tc_d64v128(bool, const AttnArgs&, float*, cudaStream_t, std::string&);
int launch_bwd_tc_d128v64(bool, const AttnArgs&, float*, cudaStream_t, std::string&);

// Workspace: the row table, L2 then D, each [B*H][n_pad] float32 with n_pad = n rounded up to
// 128 (so every 128-row block of it is a whole, 512-byte-aligned bulk copy).
size_t bwd_tc_workspace_bytes(int B, int H, int n, int) {
  const size_t rows = static_cast<size_t>(B) * H * bwd_pad_rows(n);
  return 2 * rows * 4;
}

int launch_bwd_tc(bool bf16, const AttnArgs& a, cudaStream_t s, std::string& err) {
  float* table = static_cast<float*>(a.workspace);
  if (a.v_dim != a.d) {
    if (a.d == 64 && a.v_dim == 128) return launch_bwd_tc_d64v128(bf16, a, table, s, err);
    if (a.d == 128 && a.v_dim == 64) return launch_bwd_tc_d128v64(bf16, a, table, s, err);
    err = "value width v != d is supported for (d, v) = (64, 128) and (128, 64)";
    return -2;
  }
  switch (a.d) {
    case 16: return launch_bwd_tc_d16(bf16, a, table, s, err);
    case 32: return launch_bwd_tc_d32(bf16, a, table, s, err);
    case 64: return launch_bwd_tc_d64(bf16, a, table, s, err);
    case 128: return launch_bwd_tc_d128(bf16, a, table, s, err);
    default: err = "head dimension must be 16, 32, 64 or 128"; return -2;
  }
}
}  // namespace ea
