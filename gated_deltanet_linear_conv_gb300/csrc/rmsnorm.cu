// Gated RMSNorm of the mixer output: y = x / sqrt(mean(x^2) + eps) * w * silu(z)
// over each head's Dv vector ("Qwen3.5 Simulation Support Design Document",
// section 2.2 op 6; "Qwen3.5 Dense Model Architecture", section Linear
// Attention, self.norm(core_output, z)).
//
// Memory-bound: dim/8 lanes per row, 8 elements per lane (16-byte bf16
// accesses), UNROLL row groups per warp iteration whose loads are all issued
// one iteration ahead (the next rows are in flight while these are computed),
// shuffle reduction of the sum of squares, element pairs through the packed
// fp32x2 multiply (each half rounded as the scalar one), grid-stride over rows
// with three resident CTAs per SM.

#include "common.cuh"
#include "launch.h"

namespace gdn {
namespace {

// Eight consecutive elements held as loaded (packed bf16 or fp32) until used,
// so UNROLL rows of x and z fit in flight with few registers.
template <typename T> struct Raw8;
template <> struct Raw8<bf16> {
  uint4 u;
  __device__ __forceinline__ void load(const bf16* p) { u = *reinterpret_cast<const uint4*>(p); }
  __device__ __forceinline__ void zero() { u = make_uint4(0u, 0u, 0u, 0u); }
  __device__ __forceinline__ void get(float (&f)[8]) const {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 v = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
      f[2 * i] = v.x;
      f[2 * i + 1] = v.y;
    }
  }
};
template <> struct Raw8<float> {
  float4 a, b;
  __device__ __forceinline__ void load(const float* p) {
    a = *reinterpret_cast<const float4*>(p);
    b = *reinterpret_cast<const float4*>(p + 4);
  }
  __device__ __forceinline__ void zero() { a = b = make_float4(0.f, 0.f, 0.f, 0.f); }
  __device__ __forceinline__ void get(float (&f)[8]) const {
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  }
};

__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// silu(z) = h + h tanh(h), h = z / 2: the hardware tanh when y is rounded to
// bf16, exact division for fp32.  The tanh's relative error (about 2^-11) gives
// an absolute error of at most about 2^-11 |h|: within half a bf16 ulp of the
// result for z >= -2; for more negative z silu is near zero and the error, still
// far below the bf16 rounding of O(1) values, is no longer small relative to it.
template <typename Ty> __device__ __forceinline__ float gate_silu(float z);
template <> __device__ __forceinline__ float gate_silu<bf16>(float z) {
  const float h = 0.5f * z;
  return fmaf(h, tanh_approx(h), h);
}
template <> __device__ __forceinline__ float gate_silu<float>(float z) { return silu_fast(z); }

template <typename Tx, typename Tz, typename Ty>
__global__ void __launch_bounds__(256, 3)
gated_rmsnorm_kernel(RmsNormArgs p) {
  // rows per warp step: 2 for bf16 x and z, 1 for wider types (with the next step's rows
  // also in flight, this keeps three CTAs per SM: more resident warps beat deeper unrolling)
  constexpr int UNROLL = sizeof(Tx) + sizeof(Tz) == 4 ? 2 : 1;
  const int lanes_per_row = p.dim / 8;
  const int rows_per_step = 32 / lanes_per_row;          // rows per warp per unrolled step
  const int rows_per_iter = rows_per_step * UNROLL;
  const int lane = threadIdx.x & 31;
  const int sub = lane / lanes_per_row;
  const int col = (lane % lanes_per_row) * 8;
  float2 w[4];
  {
    float wf[8];
    load8(p.w + col, wf);
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = make_float2(wf[2 * i], wf[2 * i + 1]);
  }
  const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int64_t warp_id = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t step = warps_total * rows_per_iter;
  const float inv_dim = 1.0f / (float)p.dim;
  const Tx* X = static_cast<const Tx*>(p.x);
  const Tz* Z = static_cast<const Tz*>(p.z);
  Ty* Y = static_cast<Ty*>(p.y);
  auto load = [&](int64_t r0, Raw8<Tx>(&xr)[UNROLL], Raw8<Tz>(&zr)[UNROLL]) {
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int64_t row = r0 + u * rows_per_step + sub;
      if (row < p.rows) {
        xr[u].load(X + row * p.dim + col);
        zr[u].load(Z + row * p.dim + col);
      } else {
        xr[u].zero();
        zr[u].zero();
      }
    }
  };
  int64_t r0 = warp_id * rows_per_iter;
  Raw8<Tx> xr[UNROLL];
  Raw8<Tz> zr[UNROLL];
  load(r0, xr, zr);
  for (; r0 < p.rows; r0 += step) {
    Raw8<Tx> xn[UNROLL];
    Raw8<Tz> zn[UNROLL];
    load(r0 + step, xn, zn);                 // the next rows go in flight first
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int64_t row = r0 + u * rows_per_step + sub;
      float xf[8], zf[8];
      xr[u].get(xf);
      zr[u].get(zf);
      float2 x[4], z[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        x[i] = make_float2(xf[2 * i], xf[2 * i + 1]);
        z[i] = make_float2(zf[2 * i], zf[2 * i + 1]);
      }
      float2 ss2 = __fmul2_rn(x[0], x[0]);
#pragma unroll
      for (int i = 1; i < 4; ++i) ss2 = __ffma2_rn(x[i], x[i], ss2);
      const float ss = group_sum(ss2.x + ss2.y, lanes_per_row);
      const float inv = rsqrtf(ss * inv_dim + p.eps);
      const float2 inv2 = make_float2(inv, inv);
      float y[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 t = __fmul2_rn(__fmul2_rn(x[i], inv2), w[i]);
        y[2 * i] = t.x * gate_silu<Ty>(z[i].x);
        y[2 * i + 1] = t.y * gate_silu<Ty>(z[i].y);
      }
      if (row < p.rows) store8(Y + row * p.dim + col, y);
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      xr[u] = xn[u];
      zr[u] = zn[u];
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
  const int rows_per_block = 8 * (32 / (p.dim / 8)) * 4;
  const int64_t need = (p.rows + rows_per_block - 1) / rows_per_block;
  const int blocks = (int)std::min<int64_t>(need, (int64_t)num_sms() * 3);   // three resident per SM
  if (p.x_bf16) {
    return p.z_bf16 ? launch_y<bf16, bf16>(p, s, blocks) : launch_y<bf16, float>(p, s, blocks);
  }
  return p.z_bf16 ? launch_y<float, bf16>(p, s, blocks) : launch_y<float, float>(p, s, blocks);
}

}  // namespace gdn
