// Chunked gated delta rule on CUDA cores in fp32 (the accuracy variant of
// gdn_chunk_prefill).  ("Qwen3.5 Simulation Support Design Document",
// Appendix B: chunk 64, intra-chunk attention + inter-chunk recurrence;
// "Qwen3.5 Dense Model Architecture", section Linear Attention,
// chunk_gated_delta_rule with initial and final state.)
//
// Chunk form, per chunk of L <= 64 tokens with entry state S0, G = cumsum(g):
//   A[r,j] = beta_r exp(G_r - G_j) k_r.k_j                (j < r)
//   (I + A) [U~ | W] = [diag(beta) V | diag(beta exp(G)) K]   (forward substitution)
//   U   = U~ - W S0
//   O   = diag(exp(G)) Q S0 + (M o Q K^T) U,   M[r,j] = exp(G_r - G_j), j <= r
//   S_L = exp(G_L) S0 + (diag(exp(G_L - G)) K)^T U
// Every exponent is <= 0.  Padding rows (beyond L) carry beta = g = 0 and
// zero q/k/v, which leaves the state unchanged.
//
// One CTA per (sequence, value head, 32-column slice of Dv): columns of S,
// U, O are independent, so slices need no communication.

#include "common.cuh"
#include "launch.h"

namespace gdn {
namespace {

constexpr int CT = 64;     // chunk length
constexpr int DVS = 32;    // Dv columns per CTA
constexpr int NT = 256;

template <int DK>
struct SimtSmem {
  static constexpr int QS = DK + 1;              // padded row stride
  static constexpr int PS = CT + 1;
  static constexpr int XS = DVS + DK;
  static constexpr size_t q_off = 0;
  static constexpr size_t k_off = q_off + CT * QS;
  static constexpr size_t v_off = k_off + CT * QS;
  static constexpr size_t s_off = v_off + CT * DVS;
  static constexpr size_t a_off = s_off + DK * DVS;
  static constexpr size_t p_off = a_off + CT * PS;
  static constexpr size_t x_off = p_off + CT * PS;
  static constexpr size_t u_off = x_off + CT * XS;
  static constexpr size_t gv_off = u_off + CT * DVS;   // G, beta, gamma, decay-to-end
  static constexpr size_t total_floats = gv_off + 4 * CT;
  static constexpr size_t bytes = total_floats * sizeof(float);
};

template <int DK, typename Tin, typename Tout>
__global__ void __launch_bounds__(NT, 1)
chunk_simt_kernel(ChunkArgs p) {
  using L = SimtSmem<DK>;
  extern __shared__ float smem[];
  float* Qs = smem + L::q_off;
  float* Ks = smem + L::k_off;
  float* Vs = smem + L::v_off;
  float* Ss = smem + L::s_off;
  float* Am = smem + L::a_off;
  float* Pm = smem + L::p_off;
  float* Xs = smem + L::x_off;
  float* Us = smem + L::u_off;
  float* Gs = smem + L::gv_off;
  float* Bs = Gs + CT;
  float* Gam = Bs + CT;
  float* Dec = Gam + CT;

  const int tid = threadIdx.x;
  const int v0 = blockIdx.x * DVS;
  const int h = blockIdx.y;
  const int s = blockIdx.z;
  const int hk = h / (p.Nv / p.Nk);
  const int Dv = p.Dv;
  int bos, eos;
  if (!seq_bounds(p.cu, p.num_seqs, p.total, s, bos, eos)) {
    if (tid == 0 && blockIdx.x == 0 && h == 0) raise_error(p.err, kDevErrSeqlens);
    return;
  }
  const size_t state_base = ((size_t)s * p.Nv + h) * DK * Dv;
  for (int idx = tid; idx < DK * DVS; idx += NT) {
    const int i = idx / DVS, c = idx % DVS;
    Ss[idx] = p.S0 ? p.S0[state_base + (size_t)i * Dv + v0 + c] : 0.f;
  }
  const Tin* q = static_cast<const Tin*>(p.q);
  const Tin* k = static_cast<const Tin*>(p.k);
  const Tin* v = static_cast<const Tin*>(p.v);
  Tout* o = static_cast<Tout*>(p.o);

  for (int c0 = bos; c0 < eos; c0 += CT) {
    const int len = min(CT, eos - c0);
    __syncthreads();
    // ---- 1. load the chunk
    for (int idx = tid; idx < CT * DK; idx += NT) {
      const int r = idx / DK, i = idx % DK;
      float qv = 0.f, kv = 0.f;
      if (r < len) {
        const size_t off = ((size_t)(c0 + r) * p.Nk + hk) * DK + i;
        qv = to_f32(q[off]) * p.scale;
        kv = to_f32(k[off]);
      }
      Qs[r * L::QS + i] = qv;
      Ks[r * L::QS + i] = kv;
    }
    for (int idx = tid; idx < CT * DVS; idx += NT) {
      const int r = idx / DVS, c = idx % DVS;
      Vs[idx] = r < len ? to_f32(v[((size_t)(c0 + r) * p.Nv + h) * Dv + v0 + c]) : 0.f;
    }
    if (tid < CT) {
      Gs[tid] = tid < len ? p.g[(size_t)(c0 + tid) * p.Nv + h] : 0.f;
      Bs[tid] = tid < len ? p.beta[(size_t)(c0 + tid) * p.Nv + h] : 0.f;
    }
    __syncthreads();
    // ---- 2. G = cumsum(g) (warp 0: lane l scans elements l and l + 32)
    if (tid < 32) {
      float a0 = Gs[tid], a1 = Gs[tid + 32];
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float t0 = __shfl_up_sync(0xffffffffu, a0, off);
        const float t1 = __shfl_up_sync(0xffffffffu, a1, off);
        if (tid >= off) { a0 += t0; a1 += t1; }
      }
      a1 += __shfl_sync(0xffffffffu, a0, 31);
      const float glast = __shfl_sync(0xffffffffu, a1, 31);
      Gs[tid] = a0;
      Gs[tid + 32] = a1;
      Gam[tid] = expf(a0);
      Gam[tid + 32] = expf(a1);
      Dec[tid] = expf(glast - a0);
      Dec[tid + 32] = expf(glast - a1);
    }
    __syncthreads();
    // ---- 3. A (strictly lower, with beta and decay) and P = M o QK^T
    for (int idx = tid; idx < CT * CT; idx += NT) {
      const int r = idx / CT, j = idx % CT;
      float kk = 0.f, qk = 0.f;
      if (j <= r) {
        const float* kr = Ks + r * L::QS;
        const float* qr = Qs + r * L::QS;
        const float* kj = Ks + j * L::QS;
#pragma unroll 8
        for (int i = 0; i < DK; ++i) {
          kk = fmaf(kr[i], kj[i], kk);
          qk = fmaf(qr[i], kj[i], qk);
        }
      }
      const float dec = j <= r ? expf(Gs[r] - Gs[j]) : 0.f;
      Am[r * L::PS + j] = j < r ? Bs[r] * dec * kk : 0.f;
      Pm[r * L::PS + j] = dec * qk;
    }
    __syncthreads();
    // ---- 4. forward substitution, one column of [U~ | W] per thread
    if (tid < L::XS) {
      const int col = tid;
      for (int r = 0; r < CT; ++r) {
        float x = col < DVS ? Bs[r] * Vs[r * DVS + col]
                            : Bs[r] * Gam[r] * Ks[r * L::QS + (col - DVS)];
        const float* ar = Am + r * L::PS;
        for (int j = 0; j < r; ++j) x = fmaf(-ar[j], Xs[j * L::XS + col], x);
        Xs[r * L::XS + col] = x;
      }
    }
    __syncthreads();
    // ---- 5. U = U~ - W S0
    for (int idx = tid; idx < CT * DVS; idx += NT) {
      const int r = idx / DVS, c = idx % DVS;
      const float* wr = Xs + r * L::XS + DVS;
      float acc = Xs[r * L::XS + c];
#pragma unroll 8
      for (int i = 0; i < DK; ++i) acc = fmaf(-wr[i], Ss[i * DVS + c], acc);
      Us[idx] = acc;
    }
    __syncthreads();
    // ---- 6. O = diag(gamma) Q S0 + P U
    for (int idx = tid; idx < CT * DVS; idx += NT) {
      const int r = idx / DVS, c = idx % DVS;
      if (r < len) {
        const float* qr = Qs + r * L::QS;
        float acc = 0.f;
#pragma unroll 8
        for (int i = 0; i < DK; ++i) acc = fmaf(qr[i], Ss[i * DVS + c], acc);
        acc *= Gam[r];
        const float* pr = Pm + r * L::PS;
        for (int j = 0; j <= r; ++j) acc = fmaf(pr[j], Us[j * DVS + c], acc);
        o[((size_t)(c0 + r) * p.Nv + h) * Dv + v0 + c] = from_f32<Tout>(acc);
      }
    }
    // ---- 7. S_L = exp(G_L) S0 + (diag(exp(G_L - G)) K)^T U
    constexpr int PER = DK * DVS / NT;
    float snew[PER];
    const float gl = Gam[CT - 1];
#pragma unroll
    for (int m = 0; m < PER; ++m) {
      const int idx = tid + m * NT;
      const int i = idx / DVS, c = idx % DVS;
      float acc = gl * Ss[idx];
#pragma unroll 8
      for (int r = 0; r < CT; ++r) acc = fmaf(Dec[r] * Ks[r * L::QS + i], Us[r * DVS + c], acc);
      snew[m] = acc;
    }
    __syncthreads();
#pragma unroll
    for (int m = 0; m < PER; ++m) Ss[tid + m * NT] = snew[m];
  }
  __syncthreads();
  if (p.ST) {
    for (int idx = tid; idx < DK * DVS; idx += NT) {
      const int i = idx / DVS, c = idx % DVS;
      p.ST[state_base + (size_t)i * Dv + v0 + c] = Ss[idx];
    }
  }
}

template <int DK, typename Tin, typename Tout>
cudaError_t launch_t(const ChunkArgs& p, cudaStream_t s) {
  const size_t bytes = SimtSmem<DK>::bytes;
  cudaError_t e = cudaFuncSetAttribute(chunk_simt_kernel<DK, Tin, Tout>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  dim3 grid(p.Dv / DVS, p.Nv, p.num_seqs);
  chunk_simt_kernel<DK, Tin, Tout><<<grid, NT, bytes, s>>>(p);
  return cudaGetLastError();
}

template <int DK>
cudaError_t dispatch(const ChunkArgs& p, cudaStream_t s) {
  if (p.in_bf16) return p.out_bf16 ? launch_t<DK, bf16, bf16>(p, s) : launch_t<DK, bf16, float>(p, s);
  return p.out_bf16 ? launch_t<DK, float, bf16>(p, s) : launch_t<DK, float, float>(p, s);
}

}  // namespace

cudaError_t launch_chunk_simt(const ChunkArgs& p, cudaStream_t s) {
  return p.Dk == 128 ? dispatch<128>(p, s) : dispatch<64>(p, s);
}

}  // namespace gdn
