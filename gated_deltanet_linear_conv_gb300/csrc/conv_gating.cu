// Prefill front end of the Gated DeltaNet mixer: depthwise causal conv (K=4)
// with cached left context + SiLU, split into q/k/v heads, L2-norm of q and k,
// q scale, and the gates beta = sigmoid(b), g = -exp(A_log) softplus(a + dt_bias).
// ("Qwen3.5 Dense Model Architecture", section Linear Attention, forward
// listing; "Qwen3.5 Simulation Support Design Document", section 2.2 ops 2-3.)
//
// Memory-bound.  One warp owns a strip of 128 channels (4 per lane, 8-byte
// bf16 / 16-byte fp32 loads) over a block of TB tokens; the 3-token left halo
// is read from the previous rows (L2 hits) or, for the first 3 tokens of a
// sequence, from the conv state.  A strip never straddles a q/k/v region and
// holds whole heads, so the per-head L2-norm is a shuffle reduction over
// Dk/4 lanes.

#include "common.cuh"
#include "launch.h"

namespace gdn {
namespace {

constexpr int TB = 16;          // tokens per warp work item
constexpr int WARPS = 8;

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(WARPS * 32)
conv_gating_kernel(ConvGatingArgs p) {
  const int lane = threadIdx.x & 31;
  const int warp_global = blockIdx.x * WARPS + (threadIdx.x >> 5);
  const int nstrips = p.C / 128;
  const int ntb = (p.total + TB - 1) / TB;
  if (warp_global >= nstrips * ntb) return;
  const int strip = warp_global % nstrips;
  const int tb = warp_global / nstrips;
  const int t0 = tb * TB;
  const int t_end = min(t0 + TB, p.total);
  const int c0 = strip * 128 + lane * 4;       // first of my 4 channels

  const Tin* x = static_cast<const Tin*>(p.x);
  const Tin* w = static_cast<const Tin*>(p.w);
  float wt[4][4];                              // [channel][tap]
#pragma unroll
  for (int c = 0; c < 4; ++c) load4(w + (size_t)(c0 + c) * 4, wt[c]);
  float bias[4] = {0.f, 0.f, 0.f, 0.f};
  if (p.bias) load4(static_cast<const Tin*>(p.bias) + c0, bias);

  // rows t0-3 .. t0+TB-1 of my 4 channels
  float win[TB + 3][4];
#pragma unroll
  for (int r = 0; r < TB + 3; ++r) {
    int t = t0 - 3 + r;
    if (t >= 0 && t < t_end) {
      load4(x + (size_t)t * p.C + c0, win[r]);
    } else {
#pragma unroll
      for (int c = 0; c < 4; ++c) win[r][c] = 0.f;
    }
  }

  const int kd = p.Nk * p.Dk;
  const int region = c0 < kd ? 0 : (c0 < 2 * kd ? 1 : 2);   // q, k, v
  const Tin* st_in = static_cast<const Tin*>(p.state_in);

  int seq = find_seq(p.cu, p.num_seqs, p.total, t0);
  int sstart = seq_start(p.cu, p.num_seqs, p.total, seq);
  int snext = seq + 1 < p.num_seqs ? seq_start(p.cu, p.num_seqs, p.total, seq + 1) : p.total;

#pragma unroll
  for (int r = 0; r < TB; ++r) {
    const int t = t0 + r;
    if (t >= t_end) break;
    while (t >= snext && seq + 1 < p.num_seqs) {
      ++seq;
      sstart = snext;
      snext = seq + 1 < p.num_seqs ? seq_start(p.cu, p.num_seqs, p.total, seq + 1) : p.total;
    }
    const int pos = t - sstart;             // position inside the sequence
    float y[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) y[c] = bias[c];
#pragma unroll
    for (int j = 0; j < 4; ++j) {          // tap j reads xpad[pos + j]
      float xv[4];
      if (pos + j >= 3) {
#pragma unroll
        for (int c = 0; c < 4; ++c) xv[c] = win[r + j][c];
      } else {
        const int si = pos + j;            // 0..2, inside the cached context
#pragma unroll
        for (int c = 0; c < 4; ++c)
          xv[c] = (st_in != nullptr && si >= 0)
                      ? to_f32(st_in[((size_t)seq * p.C + c0 + c) * 3 + si]) : 0.f;
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) y[c] = fmaf(wt[c][j], xv[c], y[c]);
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) y[c] = siluf_(y[c]);

    if (region < 2) {
      float ss = y[0] * y[0] + y[1] * y[1] + y[2] * y[2] + y[3] * y[3];
      ss = group_sum(ss, p.Dk / 4);
      float inv = 1.0f / sqrtf(ss + p.l2_eps);
      if (region == 0) inv *= p.q_scale;
#pragma unroll
      for (int c = 0; c < 4; ++c) y[c] *= inv;
      Tout* dst = static_cast<Tout*>(region == 0 ? p.q : p.k);
      store4(dst + (size_t)t * kd + (c0 - region * kd), y);
    } else {
      const int vd = p.Nv * p.Dv;
      store4(static_cast<Tout*>(p.v) + (size_t)t * vd + (c0 - 2 * kd), y);
    }
  }

  // gates: the warps of v strips also produce g and beta of their heads
  if (region == 2) {
    const int hps = 128 / p.Dv;                      // heads per strip
    const int h0 = (strip * 128 - 2 * kd) / p.Dv;
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

template <typename Tin, typename Tout>
cudaError_t launch_typed(const ConvGatingArgs& p, cudaStream_t s) {
  const int nstrips = p.C / 128;
  const long long items = (long long)nstrips * ((p.total + TB - 1) / TB);
  if (items > 0) {
    const int blocks = (int)((items + WARPS - 1) / WARPS);
    conv_gating_kernel<Tin, Tout><<<blocks, WARPS * 32, 0, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
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
