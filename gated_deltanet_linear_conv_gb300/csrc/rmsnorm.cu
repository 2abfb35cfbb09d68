// Gated RMSNorm of the mixer output: y = x / sqrt(mean(x^2) + eps) * w * silu(z)
// over each head's Dv vector ("Qwen3.5 Simulation Support Design Document",
// section 2.2 op 6; "Qwen3.5 Dense Model Architecture", section Linear
// Attention, self.norm(core_output, z)).
//
// Memory-bound: dim/8 lanes per row, 8 elements per lane (16-byte bf16
// accesses), UNROLL row groups per warp iteration with every load issued
// before the first use, shuffle reduction of the sum of squares, grid-stride
// over rows with the grid sized to the SM count.

#include "common.cuh"
#include "launch.h"

namespace gdn {
namespace {

constexpr int UNROLL = 2;

template <typename Tx, typename Tz, typename Ty>
__global__ void __launch_bounds__(256, 3)
gated_rmsnorm_kernel(RmsNormArgs p) {
  const int lanes_per_row = p.dim / 8;
  const int rows_per_step = 32 / lanes_per_row;          // rows per warp per unrolled step
  const int rows_per_iter = rows_per_step * UNROLL;
  const int lane = threadIdx.x & 31;
  const int sub = lane / lanes_per_row;
  const int col = (lane % lanes_per_row) * 8;
  float w[8];
  load8(p.w + col, w);
  const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int64_t warp_id = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const float inv_dim = 1.0f / (float)p.dim;
  const Tx* X = static_cast<const Tx*>(p.x);
  const Tz* Z = static_cast<const Tz*>(p.z);
  Ty* Y = static_cast<Ty*>(p.y);
  for (int64_t r0 = warp_id * rows_per_iter; r0 < p.rows; r0 += warps_total * rows_per_iter) {
    float x[UNROLL][8], z[UNROLL][8];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int64_t row = r0 + u * rows_per_step + sub;
      if (row < p.rows) {
        load8(X + row * p.dim + col, x[u]);
        load8(Z + row * p.dim + col, z[u]);
      } else {
#pragma unroll
        for (int c = 0; c < 8; ++c) { x[u][c] = 0.f; z[u][c] = 0.f; }
      }
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int64_t row = r0 + u * rows_per_step + sub;
      float ss = 0.f;
#pragma unroll
      for (int c = 0; c < 8; ++c) ss = fmaf(x[u][c], x[u][c], ss);
      ss = group_sum(ss, lanes_per_row);
      const float inv = rsqrtf(ss * inv_dim + p.eps);
      float y[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) y[c] = x[u][c] * inv * w[c] * silu_fast(z[u][c]);
      if (row < p.rows) store8(Y + row * p.dim + col, y);
    }
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
  const int rows_per_block = 8 * (32 / (p.dim / 8)) * UNROLL;
  const int64_t need = (p.rows + rows_per_block - 1) / rows_per_block;
  const int blocks = (int)std::min<int64_t>(need, 152 * 8);
  if (p.x_bf16) {
    return p.z_bf16 ? launch_y<bf16, bf16>(p, s, blocks) : launch_y<bf16, float>(p, s, blocks);
  }
  return p.z_bf16 ? launch_y<float, bf16>(p, s, blocks) : launch_y<float, float>(p, s, blocks);
}

}  // namespace gdn
