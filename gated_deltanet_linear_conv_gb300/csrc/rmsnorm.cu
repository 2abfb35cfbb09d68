// Gated RMSNorm of the mixer output: y = x / sqrt(mean(x^2) + eps) * w * silu(z)
// over each head's Dv vector ("Qwen3.5 Simulation Support Design Document",
// section 2.2 op 6; "Qwen3.5 Dense Model Architecture", section Linear
// Attention, self.norm(core_output, z)).
//
// Memory-bound: dim/4 lanes per row, 4 elements per lane (8-byte bf16 /
// 16-byte fp32 accesses), shuffle reduction of the sum of squares, grid-stride
// over rows with the grid sized to the SM count.

#include "common.cuh"
#include "launch.h"

namespace gdn {
namespace {

template <typename Tx, typename Tz, typename Ty>
__global__ void __launch_bounds__(256)
gated_rmsnorm_kernel(RmsNormArgs p) {
  const int lanes_per_row = p.dim / 4;
  const int rows_per_warp = 32 / lanes_per_row;
  const int lane = threadIdx.x & 31;
  const int sub = lane / lanes_per_row;           // row slot inside the warp
  const int col = (lane % lanes_per_row) * 4;
  float w[4];
  load4(p.w + col, w);
  const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int64_t warp_id = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const float inv_dim = 1.0f / (float)p.dim;
  for (int64_t r0 = warp_id * rows_per_warp; r0 < p.rows; r0 += warps_total * rows_per_warp) {
    const int64_t row = r0 + sub;
    const bool ok = row < p.rows;
    float x[4] = {0.f, 0.f, 0.f, 0.f}, z[4] = {0.f, 0.f, 0.f, 0.f};
    if (ok) {
      load4(static_cast<const Tx*>(p.x) + row * p.dim + col, x);
      load4(static_cast<const Tz*>(p.z) + row * p.dim + col, z);
    }
    float ss = x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3];
    ss = group_sum(ss, lanes_per_row);
    const float inv = 1.0f / sqrtf(ss * inv_dim + p.eps);
    float y[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) y[c] = x[c] * inv * w[c] * siluf_(z[c]);
    if (ok) store4(static_cast<Ty*>(p.y) + row * p.dim + col, y);
  }
}

template <typename Tx, typename Tz>
cudaError_t launch_y(const RmsNormArgs& p, cudaStream_t s, int blocks) {
  if (p.out_bf16) gated_rmsnorm_kernel<Tx, Tz, bf16><<<blocks, 256, 0, s>>>(p);
  else gated_rmsnorm_kernel<Tx, Tz, float><<<blocks, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gated_rmsnorm(const RmsNormArgs& p, cudaStream_t s) {
  if (p.rows == 0) return cudaSuccess;
  const int rows_per_block = 8 * (32 / (p.dim / 4));
  int64_t need = (p.rows + rows_per_block - 1) / rows_per_block;
  const int blocks = (int)std::min<int64_t>(need, 152 * 8);
  if (p.x_bf16) {
    return p.z_bf16 ? launch_y<bf16, bf16>(p, s, blocks) : launch_y<bf16, float>(p, s, blocks);
  }
  return p.z_bf16 ? launch_y<float, bf16>(p, s, blocks) : launch_y<float, float>(p, s, blocks);
}

}  // namespace gdn
