// Chunked gated delta rule on the 5th-generation tensor cores (tcgen05, bf16
// operands, fp32 accumulation in tensor memory), Dk = Dv = 128, chunk 64.
// ("Qwen3.5 Simulation Support Design Document", Appendix B: chunk 64,
// intra-chunk attention + inter-chunk recurrence, and section 2.2 op 4;
// "Qwen3.5 Dense Model Architecture", section Linear Attention:
// chunk_gated_delta_rule with initial and final state.)
//
// Per chunk of L <= 64 tokens with entry state S (fp32, [Dk, Dv], resident in
// tensor memory) and G = cumsum(g), gamma = exp(G):
//   D1   = [Q; K] K^T                             (128 x 64 x 128)
//   P    = M o QK^T,  A = diag(beta) (M' o KK^T)   (M: exp(G_r - G_j), j <= r / j < r)
//   T    = (I + A)^-1                             (fp32, CUDA cores)
//   U~^T = V^T (T diag beta)^T,  W^T = K^T (T diag(beta gamma))^T    (128 x 64 x 64 each)
//   U^T  = U~^T - S^T W^T                         (128 x 64 x 128, negated A operand)
//   O    = diag(gamma) Q S + P U                  (64 x 128 x 128 + 64 x 128 x 64)
//   S   <- gamma_L S + (diag(exp(G_L - G)) K)^T U (128 x 128 x 64, accumulated on the
//          gamma_L-scaled state in tensor memory)
// Padding rows beyond L get beta = g = 0, which makes them exact identities.
//
// One CTA (128 threads) per (sequence, value head).  Thread 0 issues the TMA
// loads and the MMAs; all four warps run the tensor-memory epilogues and the
// triangular inverse.  Every mbarrier wait is bounded; on a timeout the CTA
// raises the device error flag, drains and releases its tensor memory.

#include <cuda.h>

#include "common.cuh"
#include "launch.h"
#include "tc_util.cuh"

namespace gdn {
namespace {

using namespace tc;

constexpr int CT = 64;        // chunk length
constexpr int DK = 128;
constexpr int DV = 128;
constexpr int NT = 128;
constexpr uint32_t WAIT_LIMIT = 1u << 22;
constexpr int FS = 68;        // fp32 matrix row stride (16-byte aligned rows)

// shared memory map (bytes from a 1024-aligned base)
constexpr uint32_t OFF_QK0 = 0;          // [Q box0 | K box0 | Q box1 | K box1], 8 KB each
constexpr uint32_t OFF_QK1 = 32768;
constexpr uint32_t OFF_V = 65536;        // [V box0 | V box1]
constexpr uint32_t OFF_KT = 81920;       // K scaled by exp(G_L - G_j), same layout as the K boxes
constexpr uint32_t OFF_P = 98304;        // P [r][j] K-major
constexpr uint32_t OFF_TB = 106496;      // T diag(beta) [r][j]
constexpr uint32_t OFF_TBG = 114688;     // T diag(beta gamma) [r][j]
constexpr uint32_t OFF_WMN = 122880;     // W as [dk rows][r], MN-major B
constexpr uint32_t OFF_UK = 139264;      // U^T as [dv rows][j], K-major
constexpr uint32_t OFF_SMN = 155648;     // S as [dk rows][dv], two 64-column blocks of 16 KB
constexpr uint32_t OFF_AF = 188416;      // A fp32 [64][FS]
constexpr uint32_t OFF_TF = OFF_AF + 64 * FS * 4;   // T fp32 [64][FS]
constexpr uint32_t OFF_VEC = OFF_TF + 64 * FS * 4;  // G, gamma, beta, dec, beta*gamma (5 x 64 floats)
constexpr uint32_t OFF_BAR = OFF_VEC + 5 * 64 * 4;  // mbarriers + tmem slot
constexpr uint32_t SMEM_BYTES = OFF_BAR + 128 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

// tensor memory columns
constexpr uint32_t TM_D1 = 0, TM_UT = 64, TM_WT = 128, TM_O = 192, TM_S = 320;

struct Bars {
  uint64_t qk[2];
  uint64_t v;
  uint64_t mma;
  uint32_t tslot;
};

// Write 64 bf16 values (v[0..63]) as one 128-byte swizzled row `row` of a
// 64-column block at byte offset `base`.
__device__ __forceinline__ void st_row64(uint8_t* smem, uint32_t base, uint32_t row, const float* v) {
#pragma unroll
  for (int ch = 0; ch < 8; ++ch) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 h = __floats2bfloat162_rn(v[ch * 8 + 2 * i], v[ch * 8 + 2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    const uint32_t off = base + row * 128u + ((((uint32_t)ch ^ (row & 7u)) & 7u) << 4);
    *reinterpret_cast<uint4*>(smem + off) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// Load 64 consecutive tensor-memory columns of this thread's lane.
__device__ __forceinline__ void tm_ld64(uint32_t taddr, float (&v)[64]) {
  float a[32], b[32];
  tmem_ld32(taddr, a);
  tmem_ld32(taddr + 32, b);
  tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 32; ++i) { v[i] = a[i]; v[32 + i] = b[i]; }
}

// Scale every 16-byte chunk of a swizzled bf16 tile: rows of 128 bytes, the
// factor of row r is f[r & 63].  `src` may equal `dst`.
__device__ __forceinline__ void scale_rows(uint8_t* sm, uint32_t src, uint32_t dst, int nbytes, const float* f) {
  for (int off = threadIdx.x * 16; off < nbytes; off += NT * 16) {
    const int row = (off >> 7) & 63;
    uint4 u = *reinterpret_cast<const uint4*>(sm + src + off);
    const float sc = f[row];
    uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 x = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&w[i]));
      __nv_bfloat162 y = __floats2bfloat162_rn(x.x * sc, x.y * sc);
      w[i] = *reinterpret_cast<uint32_t*>(&y);
    }
    *reinterpret_cast<uint4*>(sm + dst + off) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// Block-uniform bounded wait: every thread polls, then the CTA agrees.
__device__ __forceinline__ bool wait_all(uint64_t* bar, uint32_t parity) {
  const bool ok = mbar_wait(bar, parity, WAIT_LIMIT);
  return __syncthreads_and(ok ? 1 : 0) != 0;
}

// C[i][j] (rows i0 + 2*ti + {0,1}, cols j0 + 4*tj + {0..3}) = sum_k X[xr + i][xc + k] * Y[yr + k][yc + j]
// over k < K, for a 32 x 32 output split over 128 threads (16 x 8 tiles of 2 x 4).
__device__ __forceinline__ void gemm32_tile(const float* X, int xr, int xc, const float* Y, int yr, int yc,
                                            int K, float (&acc)[2][4]) {
  const int ti = threadIdx.x >> 3, tj = threadIdx.x & 7;
#pragma unroll
  for (int a = 0; a < 2; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
#pragma unroll 8
  for (int k = 0; k < K; ++k) {
    const float x0 = X[(xr + 2 * ti) * FS + xc + k];
    const float x1 = X[(xr + 2 * ti + 1) * FS + xc + k];
    const float4 y = *reinterpret_cast<const float4*>(Y + (yr + k) * FS + yc + 4 * tj);
    acc[0][0] = fmaf(x0, y.x, acc[0][0]); acc[0][1] = fmaf(x0, y.y, acc[0][1]);
    acc[0][2] = fmaf(x0, y.z, acc[0][2]); acc[0][3] = fmaf(x0, y.w, acc[0][3]);
    acc[1][0] = fmaf(x1, y.x, acc[1][0]); acc[1][1] = fmaf(x1, y.y, acc[1][1]);
    acc[1][2] = fmaf(x1, y.z, acc[1][2]); acc[1][3] = fmaf(x1, y.w, acc[1][3]);
  }
}

// T = (I + A)^-1 for a 64 x 64 strictly lower A (fp32, stride FS); T is fully
// written (zeros above the diagonal).  16 x 16 diagonal blocks by right-looking
// substitution, then the two 16 -> 32 merges and the 32 -> 64 merge, each
// T21 = -T22 A21 T11.
__device__ void invert_unit_lower(const float* AF, float* TF) {
  const int tid = threadIdx.x;
  for (int i = tid * 4; i < 64 * FS; i += NT * 4)
    *reinterpret_cast<float4*>(TF + i) = make_float4(0.f, 0.f, 0.f, 0.f);
  __syncthreads();
  if (tid < 64) {
    const int b16 = (tid >> 4) * 16, cc = tid & 15;
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = (i == cc) ? 1.f : 0.f;
#pragma unroll
    for (int j = 0; j < 15; ++j) {
#pragma unroll
      for (int i = j + 1; i < 16; ++i) x[i] = fmaf(-AF[(b16 + i) * FS + b16 + j], x[j], x[i]);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) TF[(b16 + i) * FS + b16 + cc] = x[i];
  }
  __syncthreads();
  {   // 16 -> 32: pair p = tid / 64 handles block (2p+1, 2p); 2 x 2 outputs per thread
    const int pr = tid >> 6, q = tid & 63, ti = q >> 3, tj = q & 7;
    const int R = (2 * pr + 1) * 16, C = 2 * pr * 16;
    float y[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const float a0 = AF[(R + 2 * ti) * FS + C + k], a1 = AF[(R + 2 * ti + 1) * FS + C + k];
      const float2 t = *reinterpret_cast<const float2*>(TF + (C + k) * FS + C + 2 * tj);
      y[0][0] = fmaf(a0, t.x, y[0][0]); y[0][1] = fmaf(a0, t.y, y[0][1]);
      y[1][0] = fmaf(a1, t.x, y[1][0]); y[1][1] = fmaf(a1, t.y, y[1][1]);
    }
#pragma unroll
    for (int a = 0; a < 2; ++a)
      *reinterpret_cast<float2*>(TF + (R + 2 * ti + a) * FS + C + 2 * tj) = make_float2(y[a][0], y[a][1]);
    __syncthreads();
    float x[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const float t0 = TF[(R + 2 * ti) * FS + R + k], t1 = TF[(R + 2 * ti + 1) * FS + R + k];
      const float2 yy = *reinterpret_cast<const float2*>(TF + (R + k) * FS + C + 2 * tj);
      x[0][0] = fmaf(t0, yy.x, x[0][0]); x[0][1] = fmaf(t0, yy.y, x[0][1]);
      x[1][0] = fmaf(t1, yy.x, x[1][0]); x[1][1] = fmaf(t1, yy.y, x[1][1]);
    }
    __syncthreads();
#pragma unroll
    for (int a = 0; a < 2; ++a)
      *reinterpret_cast<float2*>(TF + (R + 2 * ti + a) * FS + C + 2 * tj) = make_float2(-x[a][0], -x[a][1]);
    __syncthreads();
  }
  {   // 32 -> 64: T[32:64][0:32] = -T[32:64][32:64] (A[32:64][0:32] T[0:32][0:32])
    const int ti = tid >> 3, tj = tid & 7;
    float acc[2][4];
    gemm32_tile(AF, 32, 0, TF, 0, 0, 32, acc);
#pragma unroll
    for (int a = 0; a < 2; ++a)
      *reinterpret_cast<float4*>(TF + (32 + 2 * ti + a) * FS + 4 * tj) =
          make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
    __syncthreads();
    gemm32_tile(TF, 32, 32, TF, 32, 0, 32, acc);
    __syncthreads();
#pragma unroll
    for (int a = 0; a < 2; ++a)
      *reinterpret_cast<float4*>(TF + (32 + 2 * ti + a) * FS + 4 * tj) =
          make_float4(-acc[a][0], -acc[a][1], -acc[a][2], -acc[a][3]);
    __syncthreads();
  }
}

template <typename Tout>
__global__ void __launch_bounds__(NT, 1)
chunk_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                const __grid_constant__ CUtensorMap tmv, ChunkArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* Gs = reinterpret_cast<float*>(sm + OFF_VEC);
  float* Gam = Gs + CT;
  float* Bet = Gam + CT;
  float* Dec = Bet + CT;
  float* BG = Dec + CT;
  float* AF = reinterpret_cast<float*>(sm + OFF_AF);
  float* TF = reinterpret_cast<float*>(sm + OFF_TF);
  Bars* bars = reinterpret_cast<Bars*>(sm + OFF_BAR);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int h = blockIdx.x;
  const int s = blockIdx.y;
  const int hk = h / (p.Nv / p.Nk);
  int bos, eos;
  if (!seq_bounds(p.cu, p.num_seqs, p.total, s, bos, eos)) {
    if (tid == 0 && h == 0) raise_error(p.err, kDevErrSeqlens);
    return;
  }
  const int nchunks = (eos - bos + CT - 1) / CT;

  if (tid == 0) {
    mbar_init(&bars->qk[0], 1);
    mbar_init(&bars->qk[1], 1);
    mbar_init(&bars->v, 1);
    mbar_init(&bars->mma, 1);
    fence_barrier_init();
    prefetch_tmap(&tmq);
    prefetch_tmap(&tmk);
    prefetch_tmap(&tmv);
  }
  if (warp == 0) tmem_alloc(&bars->tslot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = bars->tslot;
  const uint32_t lane_base = tbase + ((uint32_t)(warp * 32) << 16);   // this warp's 32 lanes
  const uint32_t s_base = smem_u32(sm);

  auto issue_qk = [&](int chunk, int stage) {
    const int t = bos + chunk * CT;
    const uint32_t base = (stage ? OFF_QK1 : OFF_QK0);
    uint64_t* bar = &bars->qk[stage];
    mbar_arrive_expect_tx(bar, 4 * 8192);
    tma_load_2d(sm + base, &tmq, bar, hk * DK, t);
    tma_load_2d(sm + base + 8192, &tmk, bar, hk * DK, t);
    tma_load_2d(sm + base + 16384, &tmq, bar, hk * DK + 64, t);
    tma_load_2d(sm + base + 24576, &tmk, bar, hk * DK + 64, t);
  };
  auto issue_v = [&](int chunk) {
    const int t = bos + chunk * CT;
    mbar_arrive_expect_tx(&bars->v, 2 * 8192);
    tma_load_2d(sm + OFF_V, &tmv, &bars->v, h * DV, t);
    tma_load_2d(sm + OFF_V + 8192, &tmv, &bars->v, h * DV + 64, t);
  };
  if (tid == 0 && nchunks > 0) {
    issue_qk(0, 0);
    issue_v(0);
  }

  // initial state -> tensor memory (lane = dk row, 128 columns = dv)
  {
    const int dk = tid;
    const float* src = p.S0 ? p.S0 + (((size_t)s * p.Nv + h) * DK + dk) * DV : nullptr;
#pragma unroll
    for (int c0 = 0; c0 < DV; c0 += 32) {
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        float4 t4 = src ? *reinterpret_cast<const float4*>(src + c0 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        v[i] = t4.x; v[i + 1] = t4.y; v[i + 2] = t4.z; v[i + 3] = t4.w;
      }
      tmem_st32(lane_base + TM_S + c0, v);
    }
    tmem_st_wait();
  }

  uint32_t ph_qk0 = 0u, ph_qk1 = 0u, ph_v = 0u, ph_mma = 0u;
  bool ok = true;
  Tout* o = static_cast<Tout*>(p.o);

  // gates of chunk 0, then always one chunk ahead (threads 0..63 own one token each)
  float g_next = 0.f, b_next = 0.f;
  if (tid < CT && nchunks > 0 && tid < eos - bos) {
    g_next = p.g[(size_t)(bos + tid) * p.Nv + h];
    b_next = p.beta[(size_t)(bos + tid) * p.Nv + h];
  }

  for (int c = 0; c < nchunks && ok; ++c) {
    const int c0 = bos + c * CT;
    const int len = min(CT, eos - c0);
    const int stage = c & 1;
    const uint32_t qk_off = stage ? OFF_QK1 : OFF_QK0;

    // ---- (1) gates of the chunk, cumulative log-decay; prefetch the next chunk's
    if (tid < CT) {
      Gs[tid] = g_next;
      Bet[tid] = b_next;
      g_next = 0.f;
      b_next = 0.f;
      if (c + 1 < nchunks && c0 + CT + tid < eos) {
        g_next = p.g[(size_t)(c0 + CT + tid) * p.Nv + h];
        b_next = p.beta[(size_t)(c0 + CT + tid) * p.Nv + h];
      }
    }
    __syncthreads();
    if (warp == 0) {
      float a0 = Gs[lane], a1 = Gs[lane + 32];
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float t0 = __shfl_up_sync(0xffffffffu, a0, off);
        const float t1 = __shfl_up_sync(0xffffffffu, a1, off);
        if (lane >= off) { a0 += t0; a1 += t1; }
      }
      a1 += __shfl_sync(0xffffffffu, a0, 31);
      const float gl = __shfl_sync(0xffffffffu, a1, 31);
      Gs[lane] = a0;
      Gs[lane + 32] = a1;
      const float e0 = __expf(a0), e1 = __expf(a1);
      Gam[lane] = e0;
      Gam[lane + 32] = e1;
      BG[lane] = Bet[lane] * e0;
      BG[lane + 32] = Bet[lane + 32] * e1;
      Dec[lane] = __expf(gl - a0);
      Dec[lane + 32] = __expf(gl - a1);
    }
    __syncthreads();
    const float gamma_L = Gam[CT - 1];

    // ---- (2) state epilogue: bf16 S -> smem (MMA operand), gamma_L * S -> tensor memory
    {
      const int dk = tid;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float v[64];
        tm_ld64(lane_base + TM_S + half * 64, v);
        st_row64(sm, OFF_SMN + half * 16384, dk, v);
        float a[32], b[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) { a[i] = v[i] * gamma_L; b[i] = v[32 + i] * gamma_L; }
        tmem_st32(lane_base + TM_S + half * 64, a);
        tmem_st32(lane_base + TM_S + half * 64 + 32, b);
      }
      tmem_st_wait();
    }

    // ---- (3) this chunk's q / k tiles
    if (!wait_all(&bars->qk[stage], stage ? ph_qk1 : ph_qk0)) { ok = false; break; }
    if (stage) ph_qk1 ^= 1u; else ph_qk0 ^= 1u;
    if (tid == 0 && c + 1 < nchunks) issue_qk(c + 1, stage ^ 1);

    // ---- (4) D1 = [Q; K] K^T, while K~ = diag(exp(G_L - G)) K is formed
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
      const uint32_t id = idesc_bf16(128, 64, false, false);
      for (int ks = 0; ks < DK / 16; ++ks) {
        const uint64_t ad = sdesc_sw128(s_base + qk_off + kstep_offset(true, ks, 16384), 16, 1024);
        const uint64_t bd = sdesc_sw128(s_base + qk_off + 8192 + kstep_offset(true, ks, 16384), 16, 1024);
        mma_bf16(tbase + TM_D1, ad, bd, id, ks > 0);
      }
      mma_commit(&bars->mma);
    }
    scale_rows(sm, qk_off + 8192, OFF_KT, 8192, Dec);
    scale_rows(sm, qk_off + 24576, OFF_KT + 8192, 8192, Dec);
    if (!wait_all(&bars->mma, ph_mma)) { ok = false; break; }
    ph_mma ^= 1u;
    tc_fence_after();
    // Q is not read raw again: scale it in place to diag(gamma) Q for the output product
    scale_rows(sm, qk_off, qk_off, 8192, Gam);
    scale_rows(sm, qk_off + 16384, qk_off + 16384, 8192, Gam);

    // ---- (5) P (lanes 0-63) and the lower triangle of A (lanes 64-127) from D1
    {
      float v[64];
      tm_ld64(lane_base + TM_D1, v);
      if (tid < CT) {
        const int r = tid;
        const float gr = Gs[r];
#pragma unroll
        for (int jb = 0; jb < 4; ++jb) {
          if (jb * 16 <= r) {
#pragma unroll
            for (int j = jb * 16; j < jb * 16 + 16; ++j) v[j] = j <= r ? __expf(gr - Gs[j]) * v[j] : 0.f;
          } else {
#pragma unroll
            for (int j = jb * 16; j < jb * 16 + 16; ++j) v[j] = 0.f;
          }
        }
        st_row64(sm, OFF_P, r, v);
      } else {
        const int r = tid - CT;
        const float gr = Gs[r], br = Bet[r];
#pragma unroll
        for (int jb = 0; jb < 4; ++jb) {
          if (jb * 16 < r) {
#pragma unroll
            for (int j = jb * 16; j < jb * 16 + 16; ++j)
              if (j < r) AF[r * FS + j] = br * __expf(gr - Gs[j]) * v[j];
          }
        }
      }
    }
    tc_fence_before();
    __syncthreads();

    // ---- (6) T = (I + A)^-1, then T diag(beta) and T diag(beta gamma) as bf16 [r][j] tiles
    invert_unit_lower(AF, TF);
    for (int idx = tid; idx < CT * 8; idx += NT) {
      const int r = idx >> 3, ch = idx & 7;
      const float4 t0 = *reinterpret_cast<const float4*>(TF + r * FS + ch * 8);
      const float4 t1 = *reinterpret_cast<const float4*>(TF + r * FS + ch * 8 + 4);
      const float4 b0 = *reinterpret_cast<const float4*>(Bet + ch * 8);
      const float4 b1 = *reinterpret_cast<const float4*>(Bet + ch * 8 + 4);
      const float4 g0 = *reinterpret_cast<const float4*>(BG + ch * 8);
      const float4 g1 = *reinterpret_cast<const float4*>(BG + ch * 8 + 4);
      const float t[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
      const float bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
      const float bg[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
      uint32_t wa[4], wb[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 ha = __floats2bfloat162_rn(t[2 * i] * bb[2 * i], t[2 * i + 1] * bb[2 * i + 1]);
        __nv_bfloat162 hb = __floats2bfloat162_rn(t[2 * i] * bg[2 * i], t[2 * i + 1] * bg[2 * i + 1]);
        wa[i] = *reinterpret_cast<uint32_t*>(&ha);
        wb[i] = *reinterpret_cast<uint32_t*>(&hb);
      }
      const uint32_t sw = r * 128u + ((((uint32_t)ch ^ (uint32_t)(r & 7)) & 7u) << 4);
      *reinterpret_cast<uint4*>(sm + OFF_TB + sw) = make_uint4(wa[0], wa[1], wa[2], wa[3]);
      *reinterpret_cast<uint4*>(sm + OFF_TBG + sw) = make_uint4(wb[0], wb[1], wb[2], wb[3]);
    }

    // ---- (7) U~^T = V^T (T diag beta)^T, W^T = K^T (T diag(beta gamma))^T
    if (!wait_all(&bars->v, ph_v)) { ok = false; break; }
    ph_v ^= 1u;
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
      const uint32_t id = idesc_bf16(128, 64, true, false);
      for (int ks = 0; ks < CT / 16; ++ks) {
        const uint64_t ad = sdesc_sw128(s_base + OFF_V + ks * 2048, 8192, 1024);
        const uint64_t bd = sdesc_sw128(s_base + OFF_TB + ks * 32, 16, 1024);
        mma_bf16(tbase + TM_UT, ad, bd, id, ks > 0);
      }
      for (int ks = 0; ks < CT / 16; ++ks) {
        const uint64_t ad = sdesc_sw128(s_base + qk_off + 8192 + ks * 2048, 16384, 1024);
        const uint64_t bd = sdesc_sw128(s_base + OFF_TBG + ks * 32, 16, 1024);
        mma_bf16(tbase + TM_WT, ad, bd, id, ks > 0);
      }
      mma_commit(&bars->mma);
    }
    if (!wait_all(&bars->mma, ph_mma)) { ok = false; break; }
    ph_mma ^= 1u;
    tc_fence_after();
    if (tid == 0 && c + 1 < nchunks) issue_v(c + 1);

    // ---- (8) W^T (lane dk, columns r) -> bf16 [dk rows][r] MN-major B
    {
      float v[64];
      tm_ld64(lane_base + TM_WT, v);
      st_row64(sm, OFF_WMN, tid, v);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---- (9) U^T = U~^T - S^T W^T ;  O = (diag(gamma) Q) S
    if (tid == 0) {
      const uint32_t idf = idesc_bf16(128, 64, true, true, true);
      for (int ks = 0; ks < DK / 16; ++ks) {
        const uint64_t ad = sdesc_sw128(s_base + OFF_SMN + ks * 2048, 16384, 1024);
        const uint64_t bd = sdesc_sw128(s_base + OFF_WMN + ks * 2048, 16384, 1024);
        mma_bf16(tbase + TM_UT, ad, bd, idf, 1u);
      }
      const uint32_t ido = idesc_bf16(64, 128, false, true);
      for (int ks = 0; ks < DK / 16; ++ks) {
        const uint64_t ad = sdesc_sw128(s_base + qk_off + kstep_offset(true, ks, 16384), 16, 1024);
        const uint64_t bd = sdesc_sw128(s_base + OFF_SMN + ks * 2048, 16384, 1024);
        mma_bf16(tbase + TM_O, ad, bd, ido, ks > 0);
      }
      mma_commit(&bars->mma);
    }
    if (!wait_all(&bars->mma, ph_mma)) { ok = false; break; }
    ph_mma ^= 1u;
    tc_fence_after();

    // ---- (10) U^T (lane dv, columns j) -> bf16 [dv rows][j] K-major
    {
      float v[64];
      tm_ld64(lane_base + TM_UT, v);
      st_row64(sm, OFF_UK, tid, v);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---- (11) O += P U ;  S += K~^T U
    if (tid == 0) {
      const uint32_t idp = idesc_bf16(64, 128, false, false);
      for (int ks = 0; ks < CT / 16; ++ks) {
        const uint64_t ad = sdesc_sw128(s_base + OFF_P + ks * 32, 16, 1024);
        const uint64_t bd = sdesc_sw128(s_base + OFF_UK + ks * 32, 16, 1024);
        mma_bf16(tbase + TM_O, ad, bd, idp, 1u);
      }
      const uint32_t ids = idesc_bf16(128, 128, true, false);
      for (int ks = 0; ks < CT / 16; ++ks) {
        const uint64_t ad = sdesc_sw128(s_base + OFF_KT + ks * 2048, 8192, 1024);
        const uint64_t bd = sdesc_sw128(s_base + OFF_UK + ks * 32, 16, 1024);
        mma_bf16(tbase + TM_S, ad, bd, ids, 1u);
      }
      mma_commit(&bars->mma);
    }
    if (!wait_all(&bars->mma, ph_mma)) { ok = false; break; }
    ph_mma ^= 1u;
    tc_fence_after();

    // ---- (12) O rows -> o[c0 + r][h][:].  The 64-row accumulator holds row
    // r = 16 * warp + lane in lanes 0-15 of each warp's lane quarter.
    {
      const int r = warp * 16 + lane;
      const bool valid = lane < 16 && r < len;
      Tout* dst = o + ((size_t)(c0 + r) * p.Nv + h) * DV;
#pragma unroll
      for (int c32 = 0; c32 < DV; c32 += 32) {
        float v[32];
        tmem_ld32(lane_base + TM_O + c32, v);
        tmem_ld_wait();
        if (valid) {
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            float w8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) w8[e] = p.scale * v[i + e];
            store8(dst + c32 + i, w8);
          }
        }
      }
    }
    tc_fence_before();
    __syncthreads();
  }

  if (!ok) {
    // a bounded wait ran out: report, let outstanding copies and products land, release TMEM
    if (tid == 0) {
      raise_error(p.err, kDevErrTimeout);
      mbar_wait(&bars->mma, ph_mma, WAIT_LIMIT);
      mbar_wait(&bars->qk[0], ph_qk0, WAIT_LIMIT);
      mbar_wait(&bars->qk[1], ph_qk1, WAIT_LIMIT);
      mbar_wait(&bars->v, ph_v, WAIT_LIMIT);
    }
  } else if (p.ST) {
    tc_fence_after();
    const int dk = tid;
    float* dst = p.ST + (((size_t)s * p.Nv + h) * DK + dk) * DV;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float v[64];
      tm_ld64(lane_base + TM_S + half * 64, v);
#pragma unroll
      for (int i = 0; i < 64; i += 4)
        *reinterpret_cast<float4*>(dst + half * 64 + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, 512);
}

// ---- host: tensor maps and launch
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encoder() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// 2-D bf16 map over a token-major [rows, cols] matrix with a 64 x 64 box, 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* base, int rows, int cols) {
  EncodeTiledFn enc = get_encoder();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, 64};
  cuuint32_t es[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename Tout>
cudaError_t launch_t(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const ChunkArgs& p,
                     cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(chunk_tc_kernel<Tout>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)SMEM_BYTES);
  if (e != cudaSuccess) return e;
  dim3 grid(p.Nv, p.num_seqs);
  chunk_tc_kernel<Tout><<<grid, NT, SMEM_BYTES, s>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace

bool chunk_tc_supported(const ChunkArgs& p) {
  return p.Dk == DK && p.Dv == DV && p.in_bf16 && get_encoder() != nullptr;
}

cudaError_t launch_chunk_tc(const ChunkArgs& p, cudaStream_t s) {
  if (p.total == 0) {
    // no tokens: the final state is the initial state
    if (p.ST && p.ST != p.S0) {
      const size_t bytes = (size_t)p.num_seqs * p.Nv * DK * DV * sizeof(float);
      if (p.S0) return cudaMemcpyAsync(p.ST, p.S0, bytes, cudaMemcpyDeviceToDevice, s);
      return cudaMemsetAsync(p.ST, 0, bytes, s);
    }
    return cudaSuccess;
  }
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, p.q, p.total, p.Nk * DK) || !make_map(&mk, p.k, p.total, p.Nk * DK) ||
      !make_map(&mv, p.v, p.total, p.Nv * DV))
    return cudaErrorInvalidValue;
  return p.out_bf16 ? launch_t<bf16>(mq, mk, mv, p, s) : launch_t<float>(mq, mk, mv, p, s);
}

}  // namespace gdn
