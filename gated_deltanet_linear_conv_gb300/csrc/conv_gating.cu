// Prefill front end of the Gated DeltaNet mixer: depthwise causal conv (K=4)
// with cached left context + SiLU, split into q/k/v heads, L2-norm of q and k,
// q scale, and the gates beta = sigmoid(b), g = -exp(A_log) softplus(a + dt_bias).
// ("Qwen3.5 Dense Model Architecture", section Linear Attention, forward
// listing; "Qwen3.5 Simulation Support Design Document", section 2.2 ops 2-3.)
//
// Memory-bound.  One warp owns a strip of 32*CPL channels (CPL per lane:
// 16-byte accesses) over a block of TB tokens and slides a 4-row window down
// the block; the 3-row left halo is re-read from the previous rows (L2 hits)
// or, for the first 3 tokens of a sequence, from the conv state.  A strip
// never straddles a q/k/v region and holds whole heads, so the per-head
// L2-norm is a shuffle reduction over Dk/CPL lanes.

#include "common.cuh"
#include "launch.h"

namespace gdn {
namespace {

constexpr int WARPS = 8;

template <int CPL> struct Vec;
template <> struct Vec<4> {
  template <typename T> static __device__ __forceinline__ void ld(const T* p, float (&f)[4]) { load4(p, f); }
  template <typename T> static __device__ __forceinline__ void st(T* p, const float (&f)[4]) { store4(p, f); }
};
template <> struct Vec<8> {
  template <typename T> static __device__ __forceinline__ void ld(const T* p, float (&f)[8]) { load8(p, f); }
  template <typename T> static __device__ __forceinline__ void st(T* p, const float (&f)[8]) { store8(p, f); }
};

template <typename Tin, typename Tout, int CPL, int TB>
__global__ void __launch_bounds__(WARPS * 32)
conv_gating_kernel(ConvGatingArgs p) {
  constexpr int STRIP = 32 * CPL;
  const int lane = threadIdx.x & 31;
  const int warp_global = blockIdx.x * WARPS + (threadIdx.x >> 5);
  const int nstrips = p.C / STRIP;
  const int ntb = (p.total + TB - 1) / TB;
  if (warp_global >= nstrips * ntb) return;
  const int strip = warp_global % nstrips;
  const int tb = warp_global / nstrips;
  const int t0 = tb * TB;
  const int t_end = min(t0 + TB, p.total);
  const int c0 = strip * STRIP + lane * CPL;       // first of my CPL channels

  const Tin* x = static_cast<const Tin*>(p.x);
  // rows t0-3 .. t0+TB-1, all loads issued before any use
  float win[TB + 3][CPL];
#pragma unroll
  for (int r = 0; r < TB + 3; ++r) {
    const int t = t0 - 3 + r;
    if (t >= 0 && t < t_end) {
      Vec<CPL>::ld(x + (size_t)t * p.C + c0, win[r]);
    } else {
#pragma unroll
      for (int c = 0; c < CPL; ++c) win[r][c] = 0.f;
    }
  }
  float wt[4][CPL];                              // [tap][channel]
  {
    const Tin* w = static_cast<const Tin*>(p.w) + (size_t)c0 * 4;
#pragma unroll
    for (int c = 0; c < CPL; c += 2) {
      float tmp[8];
      load8(w + c * 4, tmp);                     // taps of channels c and c + 1
#pragma unroll
      for (int j = 0; j < 4; ++j) { wt[j][c] = tmp[j]; wt[j][c + 1] = tmp[4 + j]; }
    }
  }
  float bias[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) bias[c] = 0.f;
  if (p.bias) Vec<CPL>::ld(static_cast<const Tin*>(p.bias) + c0, bias);

  // Tokens of this block in the first 3 positions of their sequence take part
  // of their left context from the conv state (bitmask of those tokens).
  const int kd = p.Nk * p.Dk;
  const int region = c0 < kd ? 0 : (c0 < 2 * kd ? 1 : 2);   // q, k, v
  uint32_t near_start = 0;                                   // bit r: token t0 + r has pos < 3
  {
    int seq = find_seq(p.cu, p.num_seqs, p.total, max(t0 - 3, 0));
    for (int s = seq; s < p.num_seqs; ++s) {
      const int st = seq_start(p.cu, p.num_seqs, p.total, s);
      if (st >= t_end) break;
      for (int r = max(st - t0, 0); r < min(st + 3 - t0, TB); ++r) near_start |= 1u << r;
    }
  }

  const Tin* st_in = static_cast<const Tin*>(p.state_in);
  Tout* qout = static_cast<Tout*>(p.q);
  Tout* kout = static_cast<Tout*>(p.k);
  Tout* vout = static_cast<Tout*>(p.v);
  const int vd = p.Nv * p.Dv;
#pragma unroll
  for (int r = 0; r < TB; ++r) {
    const int t = t0 + r;
    if (t >= t_end) break;
    float y[CPL];
    if (!(near_start >> r & 1u)) {
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        float acc = bias[c];
        acc = fmaf(wt[0][c], win[r][c], acc);
        acc = fmaf(wt[1][c], win[r + 1][c], acc);
        acc = fmaf(wt[2][c], win[r + 2][c], acc);
        acc = fmaf(wt[3][c], win[r + 3][c], acc);
        y[c] = acc;
      }
    } else {
      // first 3 tokens of a sequence: taps before the sequence start read the state
      const int seq = find_seq(p.cu, p.num_seqs, p.total, t);
      const int pos = t - seq_start(p.cu, p.num_seqs, p.total, seq);
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        float acc = bias[c];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float xv = win[r + j][c];
          if (pos + j < 3) {
            const int si = pos + j;
            xv = (st_in != nullptr && si >= 0) ? to_f32(st_in[((size_t)seq * p.C + c0 + c) * 3 + si]) : 0.f;
          }
          acc = fmaf(wt[j][c], xv, acc);
        }
        y[c] = acc;
      }
    }
#pragma unroll
    for (int c = 0; c < CPL; ++c) y[c] = silu_fast(y[c]);
    if (region < 2) {
      float ss = 0.f;
#pragma unroll
      for (int c = 0; c < CPL; ++c) ss = fmaf(y[c], y[c], ss);
      ss = group_sum(ss, p.Dk / CPL);
      float inv = rsqrtf(ss + p.l2_eps);
      if (region == 0) inv *= p.q_scale;
#pragma unroll
      for (int c = 0; c < CPL; ++c) y[c] *= inv;
      Tout* dst = region == 0 ? qout : kout;
      Vec<CPL>::st(dst + (size_t)t * kd + (c0 - region * kd), y);
    } else {
      Vec<CPL>::st(vout + (size_t)t * vd + (c0 - 2 * kd), y);
    }
  }

  // gates: the warps of v strips also produce g and beta of their heads
  if (region == 2) {
    const int hps = STRIP / p.Dv;                      // heads per strip
    const int h0 = (strip * STRIP - 2 * kd) / p.Dv;
    const Tin* a = static_cast<const Tin*>(p.a);
    const Tin* b = static_cast<const Tin*>(p.b);
    for (int idx = lane; idx < TB * hps; idx += 32) {
      const int t = t0 + idx / hps;
      const int h = h0 + idx % hps;
      if (t < t_end) {
        const size_t o = (size_t)t * p.Nv + h;
        const float av = to_f32(a[o]), bv = to_f32(b[o]);
        p.beta[o] = sigmoidf_(bv);
        p.g[o] = -expf(p.A_log[h]) * softplusf_(av + p.dt_bias[h]);
      }
    }
  }
}

// New conv state of each sequence: the last 3 entries of [state_in ; x].
// One thread per (sequence, channel); it reads its old state before writing,
// so state_out may alias state_in.
template <typename Tin>
__global__ void conv_state_kernel(ConvGatingArgs p) {
  const int s = blockIdx.y;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= p.C) return;
  int bos, eos;
  if (!seq_bounds(p.cu, p.num_seqs, p.total, s, bos, eos)) {
    if (c == 0) raise_error(p.err, kDevErrSeqlens);
    return;
  }
  const int L = eos - bos;
  const Tin* x = static_cast<const Tin*>(p.x);
  const Tin* sin = static_cast<const Tin*>(p.state_in);
  Tin* sout = static_cast<Tin*>(p.state_out);
  Tin old[3];
#pragma unroll
  for (int i = 0; i < 3; ++i)
    old[i] = sin ? sin[((size_t)s * p.C + c) * 3 + i] : from_f32<Tin>(0.f);
  Tin nw[3];
#pragma unroll
  for (int i = 0; i < 3; ++i) {
    const int xi = L + i;                     // index into [old(3) ; x(L)]
    nw[i] = xi >= 3 ? x[(size_t)(bos + xi - 3) * p.C + c] : old[xi];
  }
#pragma unroll
  for (int i = 0; i < 3; ++i) sout[((size_t)s * p.C + c) * 3 + i] = nw[i];
}

template <typename Tin, typename Tout, int CPL, int TB>
cudaError_t launch_main(const ConvGatingArgs& p, cudaStream_t s) {
  const int nstrips = p.C / (32 * CPL);
  const long long items = (long long)nstrips * ((p.total + TB - 1) / TB);
  if (items > 0) {
    const int blocks = (int)((items + WARPS - 1) / WARPS);
    conv_gating_kernel<Tin, Tout, CPL, TB><<<blocks, WARPS * 32, 0, s>>>(p);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

template <typename Tin, typename Tout>
cudaError_t launch_typed(const ConvGatingArgs& p, cudaStream_t s) {
  const int kd = p.Nk * p.Dk, vd = p.Nv * p.Dv;
  cudaError_t e;
  // 8 channels per lane when every region holds whole 256-channel strips
  if (kd % 256 == 0 && vd % 256 == 0) e = launch_main<Tin, Tout, 8, 8>(p, s);
  else e = launch_main<Tin, Tout, 4, 16>(p, s);
  if (e != cudaSuccess) return e;
  if (p.state_out != nullptr) {
    dim3 grid((p.C + 255) / 256, p.num_seqs);
    conv_state_kernel<Tin><<<grid, 256, 0, s>>>(p);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_conv_gating(const ConvGatingArgs& p, cudaStream_t s) {
  if (p.in_bf16) {
    return p.out_bf16 ? launch_typed<bf16, bf16>(p, s) : launch_typed<bf16, float>(p, s);
  }
  return p.out_bf16 ? launch_typed<float, bf16>(p, s) : launch_typed<float, float>(p, s);
}

// ---------------------------------------------------------------------------
// gates alone
// ---------------------------------------------------------------------------
namespace {
template <typename Tin>
__global__ void gating_kernel(GatingArgs p) {
  const int64_t n = p.rows * p.Nv;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int h = (int)(i % p.Nv);
    const float av = to_f32(static_cast<const Tin*>(p.a)[i]);
    const float bv = to_f32(static_cast<const Tin*>(p.b)[i]);
    p.beta[i] = sigmoidf_(bv);
    p.g[i] = -expf(p.A_log[h]) * softplusf_(av + p.dt_bias[h]);
  }
}
}  // namespace

cudaError_t launch_gating(const GatingArgs& p, cudaStream_t s) {
  const int64_t n = p.rows * p.Nv;
  if (n == 0) return cudaSuccess;
  const int blocks = (int)std::min<int64_t>((n + 255) / 256, 152 * 16);
  if (p.in_bf16) gating_kernel<bf16><<<blocks, 256, 0, s>>>(p);
  else gating_kernel<float><<<blocks, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace gdn
