// Shared device helpers of the GB300 Gated DeltaNet library: typed vector
// loads/stores, the elementwise functions of the mixer, warp reductions and
// the sticky device error flag.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

namespace gdn {

// SM count of the current device, read once per device (grids of the
// streaming kernels are sized as a multiple of it).
inline int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
    cached[dev] = n;
  }
  return cached[dev];
}

using bf16 = __nv_bfloat16;

// Device error codes written to the sticky flag (first writer wins).
enum DeviceError : int {
  kDevErrNone = 0,
  kDevErrSeqlens = 1,   // cu_seqlens not monotone / out of [0, total_tokens]
  kDevErrTimeout = 2,   // a bounded wait on an mbarrier ran out
};

__device__ __forceinline__ void raise_error(int* flag, int code) {
  if (flag) atomicCAS(flag, 0, code);
}

// ---- typed loads / stores of 4 consecutive elements (8 B bf16, 16 B f32) ----
__device__ __forceinline__ void load4(const bf16* p, float (&f)[4]) {
  uint2 u = *reinterpret_cast<const uint2*>(p);
  __nv_bfloat162 lo = *reinterpret_cast<__nv_bfloat162*>(&u.x);
  __nv_bfloat162 hi = *reinterpret_cast<__nv_bfloat162*>(&u.y);
  float2 a = __bfloat1622float2(lo), b = __bfloat1622float2(hi);
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
}
__device__ __forceinline__ void load4(const float* p, float (&f)[4]) {
  float4 v = *reinterpret_cast<const float4*>(p);
  f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
}
__device__ __forceinline__ void store4(bf16* p, const float (&f)[4]) {
  __nv_bfloat162 lo = __floats2bfloat162_rn(f[0], f[1]);
  __nv_bfloat162 hi = __floats2bfloat162_rn(f[2], f[3]);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&lo);
  u.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(p) = u;
}
__device__ __forceinline__ void store4(float* p, const float (&f)[4]) {
  *reinterpret_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]);
}

// ---- 8 consecutive elements (16 B bf16, 2 x 16 B f32) ----
__device__ __forceinline__ void load8(const bf16* p, float (&f)[8]) {
  uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
    f[2 * i] = a.x;
    f[2 * i + 1] = a.y;
  }
}
__device__ __forceinline__ void load8(const float* p, float (&f)[8]) {
  float4 a = *reinterpret_cast<const float4*>(p);
  float4 b = *reinterpret_cast<const float4*>(p + 4);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}
__device__ __forceinline__ void store8(bf16* p, const float (&f)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t*>(&h);
  }
  *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}
__device__ __forceinline__ void store8(float* p, const float (&f)[8]) {
  *reinterpret_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]);
  *reinterpret_cast<float4*>(p + 4) = make_float4(f[4], f[5], f[6], f[7]);
}

// x * sigmoid(x) with the fast exponential and divide (a few ulp; for very
// negative x the denominator overflows to inf and the fast divide returns 0).
__device__ __forceinline__ float silu_fast(float x) { return __fdividef(x, 1.0f + __expf(-x)); }

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(bf16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f32<bf16>(float x) { return __float2bfloat16_rn(x); }

// ---- elementwise functions of the mixer (fp32) ----
__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }
__device__ __forceinline__ float siluf_(float x) { return x / (1.0f + expf(-x)); }
// log(1 + e^x) = max(x, 0) + log(1 + e^-|x|), finite for every x.
__device__ __forceinline__ float softplusf_(float x) {
  return fmaxf(x, 0.0f) + log1pf(expf(-fabsf(x)));
}

// ---- reductions ----
// Sum over groups of `width` consecutive lanes (width a power of two <= 32).
__device__ __forceinline__ float group_sum(float v, int width) {
  for (int off = width >> 1; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// Sequence of token `t` in a packed batch: the s with cu[s] <= t < cu[s+1]
// (binary search; cu has num_seqs + 1 entries).  Equal split when cu is NULL.
__device__ __forceinline__ int find_seq(const int32_t* cu, int num_seqs, int total, int t) {
  if (cu == nullptr) {
    int len = total / num_seqs;
    return len > 0 ? min(t / len, num_seqs - 1) : 0;
  }
  int lo = 0, hi = num_seqs - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (__ldg(cu + mid) <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}
__device__ __forceinline__ int seq_start(const int32_t* cu, int num_seqs, int total, int s) {
  if (cu == nullptr) return s * (total / num_seqs);
  return __ldg(cu + s);
}

// Bounds [bos, eos) of sequence s.  Returns false (and leaves the bounds
// empty) when a device-side cu_seqlens is inconsistent for this sequence.
__device__ __forceinline__ bool seq_bounds(const int32_t* cu, int num_seqs, int total, int s,
                                           int& bos, int& eos) {
  if (cu == nullptr) {
    const int len = total / num_seqs;
    bos = s * len;
    eos = bos + len;
    return true;
  }
  bos = __ldg(cu + s);
  eos = __ldg(cu + s + 1);
  const bool ok = bos >= 0 && eos >= bos && eos <= total && (s > 0 || bos == 0) &&
                  (s + 1 < num_seqs || eos == total);
  if (!ok) bos = eos = 0;
  return ok;
}

}  // namespace gdn
