// Chunked gated delta rule on the 5th-generation tensor cores (tcgen05, bf16
// operands, fp32 accumulation in tensor memory), Dk = Dv = 128, chunk 64.
// ("Qwen3.5 Simulation Support Design Document", Appendix B: chunk 64,
// intra-chunk attention + inter-chunk recurrence, and section 2.2 op 4;
// "Qwen3.5 Dense Model Architecture", section Linear Attention:
// chunk_gated_delta_rule with initial and final state.)
//
// Per chunk of L <= 64 tokens with entry state S (fp32, [Dk, Dv], resident in
// tensor memory) and G = cumsum(g), gamma = exp(G):
//   D1  = [Q; K] K^T                              (tensor core, 128 x 64 x 128)
//   P   = M o QK^T,  A = diag(beta) (M' o KK^T)    (M: exp(G_r - G_j), j <= r / j < r)
//   T   = (I + A)^-1                              (fp32, CUDA cores, 16/32/64 blocks)
//   U~^T = V^T (T diag beta)^T,  W^T = K^T (T diag(beta gamma))^T    (128 x 64 x 64 each)
//   U^T  = U~^T - S^T W^T                          (128 x 64 x 128, negated A)
//   SQ   = S^T Q^T,  UP = U^T P^T                  (128 x 64 x 128, 128 x 64 x 64)
//   O^T  = SQ diag(gamma) + UP
//   S   <- gamma_L S + (diag(exp(G_L - G)) K)^T U (128 x 128 x 64, accumulated on the
//          gamma_L-scaled state in tensor memory)
// Every product is M = 128 (Dv or Dk on the tensor-memory lanes).  Padding
// rows beyond L get beta = g = 0, which makes them exact identities.
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

// shared memory map (bytes from a 1024-aligned base)
constexpr uint32_t OFF_QK0 = 0;          // [Q box0 | K box0 | Q box1 | K box1], 8 KB each
constexpr uint32_t OFF_QK1 = 32768;
constexpr uint32_t OFF_V = 65536;        // [V box0 | V box1]
constexpr uint32_t OFF_KT = 81920;       // K scaled by exp(G_L - G_j), same layout as K boxes
constexpr uint32_t OFF_P = 98304;        // P [r][j] K-major
constexpr uint32_t OFF_TB = 106496;      // T diag(beta) [r][j]
constexpr uint32_t OFF_TBG = 114688;     // T diag(beta gamma) [r][j]
constexpr uint32_t OFF_WMN = 122880;     // W as [dk rows][r], MN-major B
constexpr uint32_t OFF_UK = 139264;      // U^T as [dv rows][j], K-major
constexpr uint32_t OFF_SMN = 155648;     // S as [dk rows][dv], two 64-column blocks of 16 KB
constexpr uint32_t OFF_AF = 188416;      // A fp32 [64][65]
constexpr uint32_t OFF_TF = 205056;      // T fp32 [64][65]
constexpr uint32_t OFF_VEC = 221696;     // G, gamma, beta, dec (4 x 64 floats)
constexpr uint32_t OFF_BAR = 222720;     // mbarriers + tmem slot + flags
constexpr uint32_t SMEM_BYTES = 222720 + 128 + 1024;
constexpr int FS = 65;                   // fp32 matrix row stride

// tensor memory columns
constexpr uint32_t TM_D1 = 0, TM_UT = 64, TM_WT = 128, TM_SQ = 192, TM_UP = 256, TM_S = 320;

struct Bars {
  uint64_t qk[2];
  uint64_t v;
  uint64_t mma;
  uint32_t tslot;
  int abort;
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

// Block-uniform bounded wait: every thread polls, then the CTA agrees.
__device__ __forceinline__ bool wait_all(uint64_t* bar, uint32_t parity) {
  const bool ok = mbar_wait(bar, parity, WAIT_LIMIT);
  return __syncthreads_and(ok ? 1 : 0) != 0;
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
  float* AF = reinterpret_cast<float*>(sm + OFF_AF);
  float* TF = reinterpret_cast<float*>(sm + OFF_TF);
  Bars* bars = reinterpret_cast<Bars*>(sm + OFF_BAR);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
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
    bars->abort = 0;
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
  const float* gsrc = p.g;
  const float* bsrc = p.beta;
  Tout* o = static_cast<Tout*>(p.o);

  for (int c = 0; c < nchunks && ok; ++c) {
    const int c0 = bos + c * CT;
    const int len = min(CT, eos - c0);
    const int stage = c & 1;
    const uint32_t qk_off = stage ? OFF_QK1 : OFF_QK0;

    // ---- (1) gates of the chunk, cumulative log-decay
    if (tid < CT) {
      Gs[tid] = tid < len ? gsrc[(size_t)(c0 + tid) * p.Nv + h] : 0.f;
      Bet[tid] = tid < len ? bsrc[(size_t)(c0 + tid) * p.Nv + h] : 0.f;
    }
    __syncthreads();
    if (warp == 0) {
      float a0 = Gs[tid], a1 = Gs[tid + 32];
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float t0 = __shfl_up_sync(0xffffffffu, a0, off);
        const float t1 = __shfl_up_sync(0xffffffffu, a1, off);
        if (tid >= off) { a0 += t0; a1 += t1; }
      }
      a1 += __shfl_sync(0xffffffffu, a0, 31);
      const float gl = __shfl_sync(0xffffffffu, a1, 31);
      Gs[tid] = a0;
      Gs[tid + 32] = a1;
      Gam[tid] = __expf(a0);
      Gam[tid + 32] = __expf(a1);
      Dec[tid] = __expf(gl - a0);
      Dec[tid + 32] = __expf(gl - a1);
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

    // ---- (4) D1 = [Q; K] K^T
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
    // K scaled by exp(G_L - G_j): 2 boxes x 64 rows x 8 chunks of 16 B
    for (int idx = tid; idx < 2 * 64 * 8; idx += NT) {
      const int box = idx >> 9, rem = idx & 511, row = rem >> 3, ch = rem & 7;
      const uint32_t src = qk_off + 8192 + box * 16384 + row * 128 + ch * 16;
      const uint32_t dst = OFF_KT + box * 8192 + row * 128 + ch * 16;
      uint4 u = *reinterpret_cast<const uint4*>(sm + src);
      const float sc = Dec[row];
      uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float2 f = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&w[i]));
        __nv_bfloat162 r = __floats2bfloat162_rn(f.x * sc, f.y * sc);
        w[i] = *reinterpret_cast<uint32_t*>(&r);
      }
      *reinterpret_cast<uint4*>(sm + dst) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    if (!wait_all(&bars->mma, ph_mma)) { ok = false; break; }
    ph_mma ^= 1u;
    tc_fence_after();

    // ---- (5) P (lanes 0-63) and A (lanes 64-127) from D1
    {
      float v[64];
      tm_ld64(lane_base + TM_D1, v);
      if (tid < CT) {
        const int r = tid;
        const float gr = Gs[r];
#pragma unroll
        for (int j = 0; j < CT; ++j) v[j] = j <= r ? __expf(gr - Gs[j]) * v[j] : 0.f;
        st_row64(sm, OFF_P, r, v);
      } else {
        const int r = tid - CT;
        const float gr = Gs[r], br = Bet[r];
#pragma unroll
        for (int j = 0; j < CT; ++j) AF[r * FS + j] = j < r ? br * __expf(gr - Gs[j]) * v[j] : 0.f;
      }
    }
    tc_fence_before();
    __syncthreads();

    // ---- (6) T = (I + A)^-1 in fp32: 16x16 diagonal blocks, then 16->32, then 32->64
    if (tid < CT) {
      const int b16 = (tid >> 4) * 16, cc = tid & 15;
      float x[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float acc = (i == cc) ? 1.f : 0.f;
        if (i > cc) {
#pragma unroll
          for (int j = 0; j < i; ++j)
            if (j >= cc) acc = fmaf(-AF[(b16 + i) * FS + b16 + j], x[j], acc);
        }
        x[i] = acc;
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) TF[(b16 + i) * FS + b16 + cc] = x[i];
    }
    __syncthreads();
    {   // level 1: T[2p+1][2p] = -T[2p+1][2p+1] A[2p+1][2p] T[2p][2p], p = 0, 1
      float y[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int e = tid + m * NT;            // 0..511
        const int pr = e >> 8, i = (e >> 4) & 15, j = e & 15;
        const int R = (2 * pr + 1) * 16, Cc = 2 * pr * 16;
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < 16; ++k) acc = fmaf(AF[(R + i) * FS + Cc + k], TF[(Cc + k) * FS + Cc + j], acc);
        y[m] = acc;
      }
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int e = tid + m * NT;
        const int pr = e >> 8, i = (e >> 4) & 15, j = e & 15;
        TF[((2 * pr + 1) * 16 + i) * FS + 2 * pr * 16 + j] = y[m];
      }
      __syncthreads();
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int e = tid + m * NT;
        const int pr = e >> 8, i = (e >> 4) & 15, j = e & 15;
        const int R = (2 * pr + 1) * 16, Cc = 2 * pr * 16;
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < 16; ++k) acc = fmaf(TF[(R + i) * FS + R + k], TF[(R + k) * FS + Cc + j], acc);
        y[m] = -acc;
      }
      __syncthreads();
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int e = tid + m * NT;
        const int pr = e >> 8, i = (e >> 4) & 15, j = e & 15;
        TF[((2 * pr + 1) * 16 + i) * FS + 2 * pr * 16 + j] = y[m];
      }
      __syncthreads();
    }
    {   // level 2: T[32:64][0:32] = -T[32:64][32:64] A[32:64][0:32] T[0:32][0:32]
      float y[8];
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int e = tid + m * NT;            // 0..1023
        const int i = e >> 5, j = e & 31;
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const float t = (k >= j) ? TF[k * FS + j] : 0.f;
          acc = fmaf(AF[(32 + i) * FS + k], t, acc);
        }
        y[m] = acc;
      }
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int e = tid + m * NT;
        TF[(32 + (e >> 5)) * FS + (e & 31)] = y[m];
      }
      __syncthreads();
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int e = tid + m * NT;
        const int i = e >> 5, j = e & 31;
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const float t = (k <= i) ? TF[(32 + i) * FS + 32 + k] : 0.f;
          acc = fmaf(t, TF[(32 + k) * FS + j], acc);
        }
        y[m] = -acc;
      }
      __syncthreads();
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int e = tid + m * NT;
        TF[(32 + (e >> 5)) * FS + (e & 31)] = y[m];
      }
      __syncthreads();
    }
    // T diag(beta) and T diag(beta gamma) as bf16 [r][j] tiles (lower triangle only)
    for (int idx = tid; idx < CT * 8; idx += NT) {
      const int r = idx >> 3, ch = idx & 7;
      float a[8], b[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int j = ch * 8 + i;
        const float t = j <= r ? TF[r * FS + j] : 0.f;
        a[i] = t * Bet[j];
        b[i] = a[i] * Gam[j];
      }
      const uint32_t sw = r * 128u + ((((uint32_t)ch ^ (uint32_t)(r & 7)) & 7u) << 4);
      uint32_t wa[4], wb[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 ha = __floats2bfloat162_rn(a[2 * i], a[2 * i + 1]);
        __nv_bfloat162 hb = __floats2bfloat162_rn(b[2 * i], b[2 * i + 1]);
        wa[i] = *reinterpret_cast<uint32_t*>(&ha);
        wb[i] = *reinterpret_cast<uint32_t*>(&hb);
      }
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

    // ---- (9) U^T = U~^T - S^T W^T ; SQ = S^T Q^T
    if (tid == 0) {
      const uint32_t idf = idesc_bf16(128, 64, true, true, true);
      for (int ks = 0; ks < DK / 16; ++ks) {
        const uint64_t ad = sdesc_sw128(s_base + OFF_SMN + ks * 2048, 16384, 1024);
        const uint64_t bd = sdesc_sw128(s_base + OFF_WMN + ks * 2048, 16384, 1024);
        mma_bf16(tbase + TM_UT, ad, bd, idf, 1u);
      }
      const uint32_t idq = idesc_bf16(128, 64, true, false);
      for (int ks = 0; ks < DK / 16; ++ks) {
        const uint64_t ad = sdesc_sw128(s_base + OFF_SMN + ks * 2048, 16384, 1024);
        const uint64_t bd = sdesc_sw128(s_base + qk_off + kstep_offset(true, ks, 16384), 16, 1024);
        mma_bf16(tbase + TM_SQ, ad, bd, idq, ks > 0);
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

    // ---- (11) UP = U^T P^T ; S += K~^T U
    if (tid == 0) {
      const uint32_t idp = idesc_bf16(128, 64, false, false);
      for (int ks = 0; ks < CT / 16; ++ks) {
        const uint64_t ad = sdesc_sw128(s_base + OFF_UK + ks * 32, 16, 1024);
        const uint64_t bd = sdesc_sw128(s_base + OFF_P + ks * 32, 16, 1024);
        mma_bf16(tbase + TM_UP, ad, bd, idp, ks > 0);
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

    // ---- (12) O^T = SQ diag(gamma) + UP  -> o[c0 + r][h][dv]
    {
      float sq[64], up[64];
      tm_ld64(lane_base + TM_SQ, sq);
      tm_ld64(lane_base + TM_UP, up);
      const int dv = tid;
      Tout* dst = o + ((size_t)c0 * p.Nv + h) * DV + dv;
#pragma unroll
      for (int r = 0; r < CT; ++r) {
        // q enters P and SQ linearly, so its scale applies to the output once
        if (r < len) dst[(size_t)r * p.Nv * DV] = from_f32<Tout>(p.scale * fmaf(sq[r], Gam[r], up[r]));
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
