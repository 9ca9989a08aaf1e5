// Preprocessing of the float32 backward.
//
// Computes the per-row term of the reverse procedure of "Exact tiled attention and
// memory-aware differentiation", delta_i = sum_a G_ia Y_ia, from the stored output O and the
// upstream dO (the "D vector" that "Bellek Duvarının Fiziği" notes comes for free from O).
// The 16-bit tensor-core backward computes the same sums inside its dQ kernel.
#include "kernels.h"

namespace ea {
namespace aux {

// One warp per row; rows = B*H*n.  Lanes stride over the d columns (the value width).
__global__ void __launch_bounds__(256) pre_kernel(const float* __restrict__ O,
                                                  const float* __restrict__ G,
                                                  float* __restrict__ Dv, int64_t rows, int d) {
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int lane = threadIdx.x & 31;
  for (int64_t r = warp0; r < rows; r += nwarps) {
    float acc = 0.0f;
    const float* o = O + r * d;
    const float* g = G + r * d;
    for (int a = lane; a < d; a += 32) acc = fmaf(o[a], g[a], acc);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
    if (lane == 0) Dv[r] = acc;
  }
}

inline int grid_for(int64_t work, int per_block) {
  int64_t g = (work + per_block - 1) / per_block;
  if (g > 152 * 16) g = 152 * 16;
  return g < 1 ? 1 : static_cast<int>(g);
}

}  // namespace aux

int launch_bwd_pre_f32(const AttnArgs& a, float* D, cudaStream_t s, std::string& err) {
  const int64_t rows = static_cast<int64_t>(a.B) * a.H * a.n;
  aux::pre_kernel<<<aux::grid_for(rows, 8), 256, 0, s>>>(
      static_cast<const float*>(a.o), static_cast<const float*>(a.d_o), D, rows, a.v_dim);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    err = std::string("backward preprocessing launch: ") + cudaGetErrorString(e);
    return -5;
  }
  return 0;
}

}  // namespace ea
