// Decode path of the Gated DeltaNet mixer: the token-by-token gated delta rule
// with the fp32 state read-modify-written in place, standalone and fused with
// the conv-state update, gating and gated RMSNorm.
// ("Qwen3.5 Dense Model Architecture", section Linear Attention, the recurrent
// branch of the forward listing and the state update
// S_t = decay(g_t) S_{t-1} + delta_update(k_t, v_t, beta_t); "Qwen3.5
// Simulation Support Design Document", sections 2.2 op 5, 2.4 and 3.1.3.)
//
// HBM-bound on the state: one CTA streams a [Dk, Dv] fp32 state through
// registers once per step (coalesced 16-byte accesses along Dv), so each step
// reads and writes the state exactly once.  256 threads: thread (rg, cg) holds
// columns 4cg..4cg+3 of rows rg, rg + RG, ...  The reductions S^T k and S^T q
// over Dk go through shared memory.

#include "common.cuh"
#include "launch.h"

namespace gdn {
namespace {

constexpr int NT = 256;

template <int DK, int DV>
struct Layout {
  static constexpr int CG = DV / 4;     // column groups of 4
  static constexpr int RG = NT / CG;    // row groups
  static constexpr int RPT = DK / RG;   // rows per thread
  static_assert(DK % RG == 0, "bad tile");
};

template <int DK, int DV>
struct StepSmem {
  float q[DK];
  float k[DK];
  float v[DV];
  float u[DV];
  float red_k[Layout<DK, DV>::RG][DV];
  float red_q[Layout<DK, DV>::RG][DV];
  float scal[8];     // [0] = k.q, [1] = alpha, [2] = beta, [3..] rms partials
  float o[DV];
};

template <int DK, int DV>
__device__ __forceinline__ void load_state(const float* S, float (&s)[Layout<DK, DV>::RPT][4]) {
  using Ly = Layout<DK, DV>;
  const int cg = threadIdx.x % Ly::CG, rg = threadIdx.x / Ly::CG;
#pragma unroll
  for (int r = 0; r < Ly::RPT; ++r) {
    const int i = rg + Ly::RG * r;
    float4 t = __ldcs(reinterpret_cast<const float4*>(S + (size_t)i * DV + cg * 4));
    s[r][0] = t.x; s[r][1] = t.y; s[r][2] = t.z; s[r][3] = t.w;
  }
}

template <int DK, int DV>
__device__ __forceinline__ void store_state(float* S, const float (&s)[Layout<DK, DV>::RPT][4]) {
  using Ly = Layout<DK, DV>;
  const int cg = threadIdx.x % Ly::CG, rg = threadIdx.x / Ly::CG;
#pragma unroll
  for (int r = 0; r < Ly::RPT; ++r) {
    const int i = rg + Ly::RG * r;
    __stcs(reinterpret_cast<float4*>(S + (size_t)i * DV + cg * 4),
           make_float4(s[r][0], s[r][1], s[r][2], s[r][3]));
  }
}

// One recurrent step on the register-resident state.  Expects sm.q (already
// scaled), sm.k, sm.v, sm.scal[0] = k.q, sm.scal[1] = alpha, sm.scal[2] = beta
// to be visible to all threads.  Leaves o_t in sm.o (valid after the call for
// every thread) and the updated state in s.
template <int DK, int DV>
__device__ __forceinline__ void recurrent_step(StepSmem<DK, DV>& sm,
                                               float (&s)[Layout<DK, DV>::RPT][4]) {
  using Ly = Layout<DK, DV>;
  const int cg = threadIdx.x % Ly::CG, rg = threadIdx.x / Ly::CG;
  float pk[4] = {0.f, 0.f, 0.f, 0.f}, pq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int r = 0; r < Ly::RPT; ++r) {
    const int i = rg + Ly::RG * r;
    const float ki = sm.k[i], qi = sm.q[i];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      pk[c] = fmaf(s[r][c], ki, pk[c]);
      pq[c] = fmaf(s[r][c], qi, pq[c]);
    }
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    sm.red_k[rg][cg * 4 + c] = pk[c];
    sm.red_q[rg][cg * 4 + c] = pq[c];
  }
  __syncthreads();
  const float alpha = sm.scal[1];
  if (threadIdx.x < DV) {
    const int col = threadIdx.x;
    float ks = 0.f, qs = 0.f;
#pragma unroll
    for (int g = 0; g < Ly::RG; ++g) { ks += sm.red_k[g][col]; qs += sm.red_q[g][col]; }
    // u = beta (v - (alpha S)^T k);  o = (alpha S + k u^T)^T q = alpha S^T q + (k.q) u
    const float u = sm.scal[2] * (sm.v[col] - alpha * ks);
    sm.u[col] = u;
    sm.o[col] = fmaf(sm.scal[0], u, alpha * qs);
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < Ly::RPT; ++r) {
    const int i = rg + Ly::RG * r;
    const float ki = sm.k[i];
#pragma unroll
    for (int c = 0; c < 4; ++c) s[r][c] = fmaf(alpha, s[r][c], ki * sm.u[cg * 4 + c]);
  }
}

// k.q over DK, by warp 0, into sm.scal[0].
template <int DK, int DV>
__device__ __forceinline__ void dot_kq(StepSmem<DK, DV>& sm) {
  if (threadIdx.x < 32) {
    float acc = 0.f;
    for (int i = threadIdx.x; i < DK; i += 32) acc = fmaf(sm.k[i], sm.q[i], acc);
    acc = group_sum(acc, 32);
    if (threadIdx.x == 0) sm.scal[0] = acc;
  }
}

// ------------------------------------------------------------ standalone step
template <int DK, int DV, typename Tin, typename Tout>
__global__ void __launch_bounds__(NT, 2)
recurrent_decode_kernel(DecodeArgs p) {
  using Ly = Layout<DK, DV>;
  __shared__ StepSmem<DK, DV> sm;
  const int h = blockIdx.x, s = blockIdx.y;
  const int hk = h / (p.Nv / p.Nk);
  int bos, eos;
  if (!seq_bounds(p.cu, p.num_seqs, p.total, s, bos, eos)) {
    if (threadIdx.x == 0 && h == 0) raise_error(p.err, kDevErrSeqlens);
    return;
  }
  float* S = p.state + ((size_t)s * p.Nv + h) * DK * DV;
  float st[Ly::RPT][4];
  load_state<DK, DV>(S, st);
  const Tin* q = static_cast<const Tin*>(p.q);
  const Tin* k = static_cast<const Tin*>(p.k);
  const Tin* v = static_cast<const Tin*>(p.v);
  for (int t = bos; t < eos; ++t) {
    __syncthreads();                                  // smem reuse across tokens
    for (int i = threadIdx.x; i < DK; i += NT) {
      const size_t off = ((size_t)t * p.Nk + hk) * DK + i;
      sm.q[i] = to_f32(q[off]) * p.scale;
      sm.k[i] = to_f32(k[off]);
    }
    for (int i = threadIdx.x; i < DV; i += NT) sm.v[i] = to_f32(v[((size_t)t * p.Nv + h) * DV + i]);
    if (threadIdx.x == 0) {
      sm.scal[1] = expf(p.g[(size_t)t * p.Nv + h]);
      sm.scal[2] = p.beta[(size_t)t * p.Nv + h];
    }
    __syncthreads();
    dot_kq<DK, DV>(sm);
    recurrent_step<DK, DV>(sm, st);
    if (threadIdx.x < DV)
      static_cast<Tout*>(p.o)[((size_t)t * p.Nv + h) * DV + threadIdx.x] = from_f32<Tout>(sm.o[threadIdx.x]);
    if (p.step_states != nullptr)      // the state after token t (speculative-decode rollback points)
      store_state<DK, DV>(p.step_states + ((size_t)t * p.Nv + h) * DK * DV, st);
  }
  store_state<DK, DV>(S, st);
}

// ------------------------------------------------------------ fused decode
// CTA = (sequence b, key head j); it owns the conv channels of q/k head j and
// of the r = Nv/Nk value heads j*r .. j*r+r-1, so the in-place conv-state
// update has a single reader/writer, then runs the r value heads in turn.
template <int DK, int DV, typename Tin, typename Tout>
__global__ void __launch_bounds__(NT, 2)
decode_fused_kernel(DecodeFusedArgs p) {
  using Ly = Layout<DK, DV>;
  __shared__ StepSmem<DK, DV> sm;
  extern __shared__ float vbuf[];                       // [r][DV] conv'd v
  __shared__ float gates[2][32];
  __shared__ float norms[2];
  const int j = blockIdx.x, b = blockIdx.y;
  const int r = p.Nv / p.Nk;
  const int kd = p.Nk * DK;
  const Tin* x = static_cast<const Tin*>(p.x);
  const Tin* w = static_cast<const Tin*>(p.w);
  const Tin* bias = static_cast<const Tin*>(p.bias);
  Tin* cst = static_cast<Tin*>(p.conv_state);

  // the state of the first value head streams in while the conv runs
  float st[Ly::RPT][4];
  load_state<DK, DV>(p.state + ((size_t)b * p.Nv + j * r) * DK * DV, st);

  // conv-state update + conv + SiLU over this CTA's channels
  const int nch = 2 * DK + r * DV;
  for (int idx = threadIdx.x; idx < nch; idx += NT) {
    int c;
    if (idx < DK) c = j * DK + idx;
    else if (idx < 2 * DK) c = kd + j * DK + (idx - DK);
    else c = 2 * kd + j * r * DV + (idx - 2 * DK);
    float wt[4];
    load4(w + (size_t)c * 4, wt);
    Tin* sp = cst + ((size_t)b * p.C + c) * 3;
    const Tin s0 = sp[0], s1 = sp[1], s2 = sp[2];
    const Tin xn = x[(size_t)b * p.C + c];
    float acc = bias ? to_f32(bias[c]) : 0.f;
    acc = fmaf(wt[0], to_f32(s0), acc);
    acc = fmaf(wt[1], to_f32(s1), acc);
    acc = fmaf(wt[2], to_f32(s2), acc);
    acc = fmaf(wt[3], to_f32(xn), acc);
    sp[0] = s1; sp[1] = s2; sp[2] = xn;
    const float y = siluf_(acc);
    if (idx < DK) sm.q[idx] = y;
    else if (idx < 2 * DK) sm.k[idx - DK] = y;
    else vbuf[idx - 2 * DK] = y;
  }
  if (threadIdx.x < r && threadIdx.x < 32) {
    const int h = j * r + threadIdx.x;
    const size_t o = (size_t)b * p.Nv + h;
    const float av = to_f32(static_cast<const Tin*>(p.a)[o]);
    const float bv = to_f32(static_cast<const Tin*>(p.b)[o]);
    gates[0][threadIdx.x] = expf(-expf(p.A_log[h]) * softplusf_(av + p.dt_bias[h]));  // alpha
    gates[1][threadIdx.x] = sigmoidf_(bv);
  }
  __syncthreads();
  // L2 norms of q (warp 0) and k (warp 1)
  if (threadIdx.x < 64) {
    const float* src = threadIdx.x < 32 ? sm.q : sm.k;
    float acc = 0.f;
    for (int i = threadIdx.x & 31; i < DK; i += 32) acc = fmaf(src[i], src[i], acc);
    acc = group_sum(acc, 32);
    if ((threadIdx.x & 31) == 0) norms[threadIdx.x >> 5] = 1.0f / sqrtf(acc + p.l2_eps);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < DK; i += NT) {
    sm.q[i] *= norms[0] * p.q_scale;
    sm.k[i] *= norms[1];
  }
  __syncthreads();
  dot_kq<DK, DV>(sm);

  for (int hh = 0; hh < r; ++hh) {
    const int h = j * r + hh;
    float* S = p.state + ((size_t)b * p.Nv + h) * DK * DV;
    if (hh > 0) load_state<DK, DV>(S, st);
    for (int i = threadIdx.x; i < DV; i += NT) sm.v[i] = vbuf[hh * DV + i];
    if (threadIdx.x == 0) { sm.scal[1] = gates[0][hh]; sm.scal[2] = gates[1][hh]; }
    __syncthreads();
    recurrent_step<DK, DV>(sm, st);
    store_state<DK, DV>(S, st);
    // gated RMSNorm of o over DV (threads < DV own one column each)
    float ov = 0.f;
    if (threadIdx.x < DV) ov = sm.o[threadIdx.x];
    float ss = group_sum(ov * ov, 32);
    if (threadIdx.x < DV && (threadIdx.x & 31) == 0) sm.scal[3 + (threadIdx.x >> 5)] = ss;
    __syncthreads();
    if (threadIdx.x < DV) {
      float tot = 0.f;
#pragma unroll
      for (int wi = 0; wi < DV / 32; ++wi) tot += sm.scal[3 + wi];
      const float inv = 1.0f / sqrtf(tot / (float)DV + p.norm_eps);
      const size_t off = ((size_t)b * p.Nv + h) * DV + threadIdx.x;
      const float zv = to_f32(static_cast<const Tin*>(p.z)[off]);
      const float yv = ov * inv * p.norm_w[threadIdx.x] * siluf_(zv);
      static_cast<Tout*>(p.y)[off] = from_f32<Tout>(yv);
    }
    __syncthreads();                                   // sm reuse by next head
  }
}

template <int DK, int DV, typename Tin, typename Tout>
cudaError_t launch_dec(const DecodeArgs& p, cudaStream_t s) {
  dim3 grid(p.Nv, p.num_seqs);
  recurrent_decode_kernel<DK, DV, Tin, Tout><<<grid, NT, 0, s>>>(p);
  return cudaGetLastError();
}

template <int DK, int DV, typename Tin, typename Tout>
cudaError_t launch_fused(const DecodeFusedArgs& p, cudaStream_t s) {
  dim3 grid(p.Nk, p.B);
  const size_t dyn = (size_t)(p.Nv / p.Nk) * DV * sizeof(float);
  decode_fused_kernel<DK, DV, Tin, Tout><<<grid, NT, dyn, s>>>(p);
  return cudaGetLastError();
}

template <int DK, int DV>
cudaError_t dispatch_dec(const DecodeArgs& p, cudaStream_t s) {
  if (p.in_bf16) return p.out_bf16 ? launch_dec<DK, DV, bf16, bf16>(p, s) : launch_dec<DK, DV, bf16, float>(p, s);
  return p.out_bf16 ? launch_dec<DK, DV, float, bf16>(p, s) : launch_dec<DK, DV, float, float>(p, s);
}
template <int DK, int DV>
cudaError_t dispatch_fused(const DecodeFusedArgs& p, cudaStream_t s) {
  if (p.in_bf16) return p.out_bf16 ? launch_fused<DK, DV, bf16, bf16>(p, s) : launch_fused<DK, DV, bf16, float>(p, s);
  return p.out_bf16 ? launch_fused<DK, DV, float, bf16>(p, s) : launch_fused<DK, DV, float, float>(p, s);
}

}  // namespace

cudaError_t launch_recurrent_decode(const DecodeArgs& p, cudaStream_t s) {
  if (p.Dk == 128 && p.Dv == 128) return dispatch_dec<128, 128>(p, s);
  if (p.Dk == 64 && p.Dv == 64) return dispatch_dec<64, 64>(p, s);
  if (p.Dk == 128 && p.Dv == 64) return dispatch_dec<128, 64>(p, s);
  return dispatch_dec<64, 128>(p, s);
}

cudaError_t launch_decode_fused(const DecodeFusedArgs& p, cudaStream_t s) {
  if (p.Dk == 128 && p.Dv == 128) return dispatch_fused<128, 128>(p, s);
  if (p.Dk == 64 && p.Dv == 64) return dispatch_fused<64, 64>(p, s);
  if (p.Dk == 128 && p.Dv == 64) return dispatch_fused<128, 64>(p, s);
  return dispatch_fused<64, 128>(p, s);
}

}  // namespace gdn
