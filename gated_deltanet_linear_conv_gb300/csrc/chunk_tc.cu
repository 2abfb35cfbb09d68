// Chunked gated delta rule on the 5th-generation tensor cores (tcgen05, bf16
// operands, fp32 accumulation in tensor memory), Dk = Dv = 128, chunk 64.
// ("Qwen3.5 Simulation Support Design Document", Appendix B: chunk 64,
// intra-chunk attention + inter-chunk recurrence, and section 2.2 op 4;
// "Qwen3.5 Dense Model Architecture", section Linear Attention:
// chunk_gated_delta_rule with initial and final state.)
//
// Per chunk of L <= 64 tokens with entry state S (fp32, [Dk, Dv]) and
// G = cumsum(g), gamma = exp(G):
//   A    = diag(beta) (M' o K K^T)                 M'[r,j] = exp(G_r - G_j), j < r
//   T    = (I + A)^-1
//   U~^T = V^T (T diag beta)^T,  W^T = K^T (T diag(beta gamma))^T
//   U^T  = U~^T - S^T W^T
//   O^T  = S^T (diag(gamma) Q)^T + U^T P^T,  P = M o Q K^T   (M[r,j] = exp(G_r - G_j), j <= r)
//   S   <- gamma_L S + (diag(exp(G_L - G)) K)^T U
// Padding rows beyond L get beta = g = 0, which makes them exact identities.
//
// Two launches:
//  * chunk_solve_kernel, parallel over every (chunk, value head): K K^T on
//    the tensor core, A, and T = (I + A)^-1 in fp32 on CUDA cores; writes
//    T diag(beta) and T diag(beta gamma) as bf16 128-byte-swizzled tiles to
//    the workspace (16 KB per chunk and head).
//  * chunk_scan_kernel, one CTA per (sequence, value head), walks the chunks
//    with the state resident in tensor memory.  Three warpgroups run as a
//    pipeline: PREP (TMA, Q K^T and the T products, P, the scaled Q and K
//    tiles, W) works one chunk ahead of STATE (the S-dependent products and
//    their epilogues), and OUT stores each chunk's output rows.  Every product
//    is an M = 128 tcgen05.mma with Dv or Dk on the tensor-memory lanes.
// Every mbarrier wait is bounded; on a timeout the CTA raises the device
// error flag, lets its outstanding copies and products land, releases its
// tensor memory and exits.

#include <cuda.h>

#include "common.cuh"
#include "launch.h"
#include "tc_util.cuh"
#include "tmap.cuh"

#include <mutex>

namespace gdn {
namespace {

using namespace tc;

constexpr int CT = 64;        // chunk length
constexpr int DK = 128;
constexpr int DV = 128;
constexpr uint32_t WAIT_LIMIT = 1u << 22;
constexpr int FS = 68;        // fp32 matrix row stride (16-byte aligned rows)
constexpr uint32_t TILE_T_BYTES = 16384;   // T diag(beta) | T diag(beta gamma), bf16

// ---------------------------------------------------------------------------
// shared helpers
// ---------------------------------------------------------------------------

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

// Scale the 64 rows of a swizzled 8 KB bf16 box in place: row r times f[r].
__device__ __forceinline__ void scale_box(uint8_t* sm, uint32_t box, const float* f, int t, int nt) {
  for (int off = t * 16; off < 8192; off += nt * 16) {
    const int row = off >> 7;
    uint4 u = *reinterpret_cast<const uint4*>(sm + box + off);
    const float sc = f[row];
    uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 x = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&w[i]));
      __nv_bfloat162 y = __floats2bfloat162_rn(x.x * sc, x.y * sc);
      w[i] = *reinterpret_cast<uint32_t*>(&y);
    }
    *reinterpret_cast<uint4*>(sm + box + off) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// Inclusive prefix sum of g over the chunk by one warp (lane l owns l, l+32);
// writes G, gamma = exp(G) and dec = exp(G_L - G).
__device__ __forceinline__ void chunk_cumsum(float* Gs, float* Gam, float* Dec, int lane) {
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
  Gam[lane] = __expf(a0);
  Gam[lane + 32] = __expf(a1);
  Dec[lane] = __expf(gl - a0);
  Dec[lane + 32] = __expf(gl - a1);
}

// Workspace slot of chunk c of sequence s: floor(bos_s / 64) + s + c.  Slots
// of different sequences never collide and stay below total / 64 + num_seqs.
__device__ __forceinline__ int slot_base(const ChunkArgs& p, int s) {
  return seq_start(p.cu, p.num_seqs, p.total, s) / CT + s;
}

// C[i][j] (rows 2*ti + {0,1}, cols 4*tj + {0..3}) = sum_k X[xr + i][xc + k] * Y[yr + k][yc + j]
// over k < K, a 32 x 32 output split over 128 threads (16 x 8 tiles of 2 x 4).
__device__ __forceinline__ void gemm32_tile(const float* X, int xr, int xc, const float* Y, int yr, int yc,
                                            int K, float (&acc)[2][4], int tid) {
  const int ti = tid >> 3, tj = tid & 7;
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

// T = (I + A)^-1 for a 64 x 64 strictly lower A (fp32, stride FS), by 128
// threads; T is fully written (zeros above the diagonal).  16 x 16 diagonal
// blocks by right-looking substitution, then the two 16 -> 32 merges and the
// 32 -> 64 merge, each T21 = -T22 A21 T11.
__device__ void invert_unit_lower(const float* AF, float* TF, int tid) {
  for (int i = tid * 4; i < 64 * FS; i += 128 * 4)
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
    gemm32_tile(AF, 32, 0, TF, 0, 0, 32, acc, tid);
#pragma unroll
    for (int a = 0; a < 2; ++a)
      *reinterpret_cast<float4*>(TF + (32 + 2 * ti + a) * FS + 4 * tj) =
          make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
    __syncthreads();
    gemm32_tile(TF, 32, 32, TF, 32, 0, 32, acc, tid);
    __syncthreads();
#pragma unroll
    for (int a = 0; a < 2; ++a)
      *reinterpret_cast<float4*>(TF + (32 + 2 * ti + a) * FS + 4 * tj) =
          make_float4(-acc[a][0], -acc[a][1], -acc[a][2], -acc[a][3]);
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// kernel 1: T tiles, parallel over (chunk slot, value head)
// ---------------------------------------------------------------------------
constexpr uint32_t S1_K = 0;                        // K box0 | K box1 (16 KB)
constexpr uint32_t S1_AF = 16384;                   // A fp32 [64][FS]
constexpr uint32_t S1_TF = S1_AF + 64 * FS * 4;     // T fp32 [64][FS]
constexpr uint32_t S1_VEC = S1_TF + 64 * FS * 4;    // G, beta, beta*gamma (3 x 64 floats)
constexpr uint32_t S1_BAR = S1_VEC + 3 * 64 * 4;
constexpr uint32_t S1_SMEM = S1_BAR + 64 + 1024;

__global__ void __launch_bounds__(128)
chunk_solve_kernel(const __grid_constant__ CUtensorMap tmk, ChunkArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* AF = reinterpret_cast<float*>(sm + S1_AF);
  float* TF = reinterpret_cast<float*>(sm + S1_TF);
  float* Gs = reinterpret_cast<float*>(sm + S1_VEC);
  float* Bet = Gs + CT;
  float* BG = Bet + CT;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + S1_BAR);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + S1_BAR + 16);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int slot = blockIdx.x, h = blockIdx.y;
  const int hk = h / (p.Nv / p.Nk);

  // slot -> (sequence, chunk)
  int lo = 0, hi = p.num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (slot_base(p, mid) <= slot) lo = mid; else hi = mid - 1;
  }
  const int s = lo, c = slot - slot_base(p, s);
  int bos, eos;
  if (!seq_bounds(p.cu, p.num_seqs, p.total, s, bos, eos)) return;   // reported by the scan kernel
  if (c < 0 || c * CT >= eos - bos) return;                           // slot not used
  const int c0 = bos + c * CT, len = min(CT, eos - c0);

  if (tid == 0) {
    mbar_init(bar, 1);
    fence_barrier_init();
    mbar_arrive_expect_tx(bar, 16384);
    tma_load_2d(sm + S1_K, &tmk, bar, hk * DK, c0);
    tma_load_2d(sm + S1_K + 8192, &tmk, bar, hk * DK + 64, c0);
  }
  if (warp == 0) tmem_alloc(tslot, 64);
  if (tid < CT) {
    Gs[tid] = tid < len ? p.g[(size_t)(c0 + tid) * p.Nv + h] : 0.f;
    Bet[tid] = tid < len ? p.beta[(size_t)(c0 + tid) * p.Nv + h] : 0.f;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  if (warp == 0) {
    float* Gam = TF;            // scratch for the cumsum helper (TF is rewritten later)
    float* Dec = TF + 64;
    chunk_cumsum(Gs, Gam, Dec, lane);
    BG[lane] = Bet[lane] * Gam[lane];
    BG[lane + 32] = Bet[lane + 32] * Gam[lane + 32];
  }
  const bool loaded = mbar_wait(bar, 0, WAIT_LIMIT);
  if (__syncthreads_and(loaded ? 1 : 0)) {
    tc_fence_after();
    if (tid == 0) {
      // K K^T: 64 x 64 x 128, rows of the result on lanes 16 w + (0..15)
      const uint32_t id = idesc_bf16(64, 64, false, false);
      const uint32_t kb = smem_u32(sm + S1_K);
      for (int ks = 0; ks < DK / 16; ++ks) {
        const uint64_t d = sdesc_sw128(kb + kstep_offset(true, ks, 8192), 16, 1024);
        mma_bf16(tbase, d, d, id, ks > 0);
      }
      mma_commit(bar);
    }
    const bool done = mbar_wait(bar, 1, WAIT_LIMIT);
    if (__syncthreads_and(done ? 1 : 0)) {
      tc_fence_after();
      float v[64];
      tm_ld64(tbase + ((uint32_t)(warp * 32) << 16), v);
      if (lane < 16) {
        const int r = warp * 16 + lane;
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
      tc_fence_before();
      __syncthreads();
      invert_unit_lower(AF, TF, tid);
      uint8_t* dst = static_cast<uint8_t*>(p.workspace) + ((size_t)slot * p.Nv + h) * TILE_T_BYTES;
      for (int idx = tid; idx < CT * 8; idx += 128) {
        const int r = idx >> 3, ch = idx & 7;
        const float4 t0 = *reinterpret_cast<const float4*>(TF + r * FS + ch * 8);
        const float4 t1 = *reinterpret_cast<const float4*>(TF + r * FS + ch * 8 + 4);
        const float t[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
        uint32_t wa[4], wb[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int j = ch * 8 + 2 * i;
          __nv_bfloat162 ha = __floats2bfloat162_rn(t[2 * i] * Bet[j], t[2 * i + 1] * Bet[j + 1]);
          __nv_bfloat162 hb = __floats2bfloat162_rn(t[2 * i] * BG[j], t[2 * i + 1] * BG[j + 1]);
          wa[i] = *reinterpret_cast<uint32_t*>(&ha);
          wb[i] = *reinterpret_cast<uint32_t*>(&hb);
        }
        const uint32_t sw = r * 128u + ((((uint32_t)ch ^ (uint32_t)(r & 7)) & 7u) << 4);
        *reinterpret_cast<uint4*>(dst + sw) = make_uint4(wa[0], wa[1], wa[2], wa[3]);
        *reinterpret_cast<uint4*>(dst + 8192 + sw) = make_uint4(wb[0], wb[1], wb[2], wb[3]);
      }
    } else if (tid == 0) {
      raise_error(p.err, kDevErrTimeout);
    }
  } else if (tid == 0) {
    raise_error(p.err, kDevErrTimeout);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, 64);
}

// ---------------------------------------------------------------------------
// kernel 2: the scan over chunks, three warpgroups
// ---------------------------------------------------------------------------
constexpr int NT2 = 384;
constexpr uint32_t K2_QK = 0;          // 3 stages x [Q box0 | K box0 | Q box1 | K box1] (32 KB)
constexpr uint32_t K2_V = 98304;       // V box0 | V box1 (16 KB)
constexpr uint32_t K2_TB = 114688;     // T diag(beta) | T diag(beta gamma) (16 KB)
constexpr uint32_t K2_P = 131072;      // 2 x P [r][j] (8 KB)
constexpr uint32_t K2_WMN = 147456;    // W as [dk rows][r] (16 KB)
constexpr uint32_t K2_UK = 163840;     // U^T as [dv rows][j] (16 KB)
constexpr uint32_t K2_SMN = 180224;    // S as [dk rows][dv], two 64-column blocks (32 KB)
constexpr uint32_t K2_VEC = 212992;    // 3 stages x (G, gamma, dec) (768 B each)
constexpr uint32_t K2_BAR = K2_VEC + 3 * 768;
constexpr uint32_t K2_SMEM = K2_BAR + 256 + 1024;
static_assert(K2_SMEM <= 232448, "shared memory budget");

// tensor memory columns
constexpr uint32_t TM_D1 = 0, TM_WT = 64, TM_UT = 128, TM_OT = 256, TM_S = 384;

struct ScanBars {
  uint64_t qk[3];   // q/k tiles of a stage landed
  uint64_t vt;      // v and T tiles landed
  uint64_t p;       // PREP products done
  uint64_t pv;      // PREP gates of a chunk written (G, gamma, dec)
  uint64_t sc;      // OUT scaled Q and K of a chunk in place and wrote W
  uint64_t ready[2];// PREP of a chunk done
  uint64_t fg;      // U^T - S^T W^T and S^T Q~^T done
  uint64_t gh[2];   // U^T P^T and the state update done
  uint64_t st[2];   // U^T of a chunk read out of tensor memory
  uint64_t of[2];   // output of a chunk stored
  uint32_t tslot;
  int abort;
};

// Bounded wait that also gives up when another warpgroup aborted.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort) {
  for (uint32_t i = 0; i < WAIT_LIMIT; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 1023u) == 1023u && *abort) return false;
  }
  *abort = 1;
  return false;
}

template <typename Tout>
__global__ void __launch_bounds__(NT2, 1)
chunk_scan_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv, ChunkArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  ScanBars* B = reinterpret_cast<ScanBars*>(sm + K2_BAR);
  volatile int* abort = &B->abort;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int wg = warp >> 2;                   // 0 PREP, 1 STATE, 2 OUT
  const int wt = tid & 127;                   // thread index in the warpgroup = its tensor-memory lane
  const int h = blockIdx.x, s = blockIdx.y;
  const int hk = h / (p.Nv / p.Nk);
  int bos, eos;
  if (!seq_bounds(p.cu, p.num_seqs, p.total, s, bos, eos)) {
    if (tid == 0 && h == 0) raise_error(p.err, kDevErrSeqlens);
    return;
  }
  const int n = (eos - bos + CT - 1) / CT;
  const int slot0 = slot_base(p, s);

  if (tid == 0) {
    for (int i = 0; i < 3; ++i) mbar_init(&B->qk[i], 1);
    mbar_init(&B->vt, 1);
    mbar_init(&B->p, 1);
    mbar_init(&B->pv, 1);
    mbar_init(&B->sc, 1);
    mbar_init(&B->fg, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&B->ready[i], 1);
      mbar_init(&B->gh[i], 1);
      mbar_init(&B->st[i], 1);
      mbar_init(&B->of[i], 1);
    }
    B->abort = 0;
    fence_barrier_init();
    prefetch_tmap(&tmq);
    prefetch_tmap(&tmk);
    prefetch_tmap(&tmv);
  }
  if (warp == 0) tmem_alloc(&B->tslot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = B->tslot;
  const uint32_t lane_base = tbase + ((uint32_t)((warp & 3) * 32) << 16);
  const uint32_t sb = smem_u32(sm);

  auto issue_qk = [&](int c) {
    const int t = bos + c * CT;
    const uint32_t base = K2_QK + (c % 3) * 32768;
    uint64_t* bar = &B->qk[c % 3];
    mbar_arrive_expect_tx(bar, 4 * 8192);
    tma_load_2d(sm + base, &tmq, bar, hk * DK, t);
    tma_load_2d(sm + base + 8192, &tmk, bar, hk * DK, t);
    tma_load_2d(sm + base + 16384, &tmq, bar, hk * DK + 64, t);
    tma_load_2d(sm + base + 24576, &tmk, bar, hk * DK + 64, t);
  };
  auto issue_vt = [&](int c) {
    const int t = bos + c * CT;
    mbar_arrive_expect_tx(&B->vt, 2 * 8192 + TILE_T_BYTES);
    tma_load_2d(sm + K2_V, &tmv, &B->vt, h * DV, t);
    tma_load_2d(sm + K2_V + 8192, &tmv, &B->vt, h * DV + 64, t);
    const uint8_t* src = static_cast<const uint8_t*>(p.workspace) + ((size_t)(slot0 + c) * p.Nv + h) * TILE_T_BYTES;
    bulk_load(sm + K2_TB, src, TILE_T_BYTES, &B->vt);
  };

  if (wg == 0) {
    // ============================== PREP ==============================
    int issued_qk = 0, issued_vt = 0;     // chunks whose loads were issued (thread 0)
    if (wt == 0 && n > 0) {
      issue_qk(0);
      if (n > 1) issue_qk(1);
      issue_vt(0);
      issued_qk = n > 1 ? 2 : 1;
      issued_vt = 1;
    }
    float g_next = 0.f;
    if (wt < CT && n > 0 && wt < eos - bos) g_next = p.g[(size_t)(bos + wt) * p.Nv + h];
    int c = 0;
    bool fail = false;
    for (; c < n; ++c) {
      const int st3 = c % 3, b = c & 1;
      const uint32_t qk = K2_QK + st3 * 32768;
      float* Gs = reinterpret_cast<float*>(sm + K2_VEC + st3 * 768);
      float* Gam = Gs + CT;
      float* Dec = Gam + CT;
      const int c0 = bos + c * CT;
      // gates of this chunk (prefetched one chunk ahead)
      if (wt < CT) {
        Gs[wt] = g_next;
        g_next = 0.f;
        if (c + 1 < n && c0 + CT + wt < eos) g_next = p.g[(size_t)(c0 + CT + wt) * p.Nv + h];
      }
      named_sync(1, 128);
      if (warp == 0) chunk_cumsum(Gs, Gam, Dec, lane);
      bool ok = wait_bar(&B->qk[st3], (c / 3) & 1, abort) && wait_bar(&B->vt, c & 1, abort);
      if (ok && c >= 2) ok = wait_bar(&B->st[b], ((c >> 1) - 1) & 1, abort);   // U~^T buffer free
      if (named_sync_or(1, 128, !ok)) { fail = true; break; }
      tc_fence_after();
      if (wt == 0) {
        mbar_arrive(&B->pv);                  // gates of chunk c are in shared memory
        // D1 = [Q; K] K^T ; U~^T = V^T (T diag beta)^T ; W^T = K^T (T diag(beta gamma))^T
        const uint32_t id1 = idesc_bf16(128, 64, false, false);
        const uint64_t a1 = sdesc_sw128(sb + qk, 16, 1024), b1 = sdesc_sw128(sb + qk + 8192, 16, 1024);
        for (int ks = 0; ks < DK / 16; ++ks) {
          const uint32_t o = kstep_offset(true, ks, 16384) >> 4;
          mma_bf16(tbase + TM_D1, a1 + o, b1 + o, id1, ks > 0);
        }
        const uint32_t id2 = idesc_bf16(128, 64, true, false);
        const uint64_t av = sdesc_sw128(sb + K2_V, 8192, 1024), bt = sdesc_sw128(sb + K2_TB, 16, 1024);
        const uint64_t ak = sdesc_sw128(sb + qk + 8192, 16384, 1024), bg = sdesc_sw128(sb + K2_TB + 8192, 16, 1024);
        for (int ks = 0; ks < CT / 16; ++ks)
          mma_bf16(tbase + TM_UT + b * 64, av + ks * (2048 >> 4), bt + ks * (32 >> 4), id2, ks > 0);
        for (int ks = 0; ks < CT / 16; ++ks)
          mma_bf16(tbase + TM_WT, ak + ks * (2048 >> 4), bg + ks * (32 >> 4), id2, ks > 0);
        mma_commit(&B->p);
      }
      ok = wait_bar(&B->p, c & 1, abort);
      if (ok && c >= 2) ok = wait_bar(&B->gh[b], ((c >> 1) - 1) & 1, abort);   // P[b] free
      if (named_sync_or(1, 128, !ok)) { fail = true; break; }
      tc_fence_after();
      if (wt == 0 && c + 1 < n) { issue_vt(c + 1); issued_vt = c + 2; }
      {
        float v[64];
        tm_ld64(lane_base + TM_D1, v);          // warps 0, 1: rows r = wt of Q K^T
        if (wt < CT) {
          const int r = wt;
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
          st_row64(sm, K2_P + b * 8192, r, v);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      ok = wait_bar(&B->sc, c & 1, abort);      // OUT scaled Q, K and wrote W
      if (named_sync_or(1, 128, !ok)) { fail = true; break; }
      if (wt == 0) {
        mbar_arrive(&B->ready[b]);
        // q/k tiles of chunk c + 2 go to the stage of chunk c - 1 once its last product ran
        if (c + 2 < n) {
          if (c < 1 || wait_bar(&B->gh[(c - 1) & 1], ((c - 1) >> 1) & 1, abort)) {
            issue_qk(c + 2);
            issued_qk = c + 3;
          }
        }
      }
    }
    if (fail && wt == 0) {
      // let the copies and products this warpgroup issued land before the exit
      for (int k = max(c, 0); k < issued_qk; ++k) mbar_wait(&B->qk[k % 3], (k / 3) & 1, WAIT_LIMIT);
      for (int k = max(c, 0); k < issued_vt; ++k) mbar_wait(&B->vt, k & 1, WAIT_LIMIT);
      mbar_wait(&B->p, c & 1, WAIT_LIMIT);
    }
  } else if (wg == 1) {
    // ============================== STATE ==============================
    {
      // initial state -> tensor memory (lane = dk, 128 columns = dv)
      const int dk = wt;
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
    bool fail = false;
    int c = 0;
    for (; c < n; ++c) {
      const int st3 = c % 3, b = c & 1;
      const uint32_t qk = K2_QK + st3 * 32768;
      const float* Gam = reinterpret_cast<const float*>(sm + K2_VEC + st3 * 768) + CT;
      bool ok = wait_bar(&B->ready[b], (c >> 1) & 1, abort);
      if (named_sync_or(2, 128, !ok)) { fail = true; break; }
      tc_fence_after();
      const float gamma_L = Gam[CT - 1];
      // bf16 S -> shared memory (operand), gamma_L S -> tensor memory (accumulator)
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float v[64];
        tm_ld64(lane_base + TM_S + half * 64, v);
        st_row64(sm, K2_SMN + half * 16384, wt, v);
        float a[32], bb[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) { a[i] = v[i] * gamma_L; bb[i] = v[32 + i] * gamma_L; }
        tmem_st32(lane_base + TM_S + half * 64, a);
        tmem_st32(lane_base + TM_S + half * 64 + 32, bb);
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      ok = c < 2 || wait_bar(&B->of[b], ((c >> 1) - 1) & 1, abort);    // O^T buffer free
      if (named_sync_or(2, 128, !ok)) { fail = true; break; }
      tc_fence_after();
      if (wt == 0) {
        // U^T = U~^T - S^T W^T ;  O^T = S^T (diag(gamma) Q)^T
        const uint32_t idf = idesc_bf16(128, 64, true, true, true);
        const uint64_t as = sdesc_sw128(sb + K2_SMN, 16384, 1024), bw = sdesc_sw128(sb + K2_WMN, 16384, 1024);
        for (int ks = 0; ks < DK / 16; ++ks)
          mma_bf16(tbase + TM_UT + b * 64, as + ks * (2048 >> 4), bw + ks * (2048 >> 4), idf, 1u);
        const uint32_t idq = idesc_bf16(128, 64, true, false);
        const uint64_t bq = sdesc_sw128(sb + qk, 16, 1024);
        for (int ks = 0; ks < DK / 16; ++ks)
          mma_bf16(tbase + TM_OT + b * 64, as + ks * (2048 >> 4), bq + (kstep_offset(true, ks, 16384) >> 4), idq,
                   ks > 0);
        mma_commit(&B->fg);
      }
      ok = wait_bar(&B->fg, c & 1, abort);
      if (named_sync_or(2, 128, !ok)) { fail = true; break; }
      tc_fence_after();
      {
        float v[64];
        tm_ld64(lane_base + TM_UT + b * 64, v);   // lane dv holds U[0..63][dv]
        st_row64(sm, K2_UK, wt, v);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      named_sync(2, 128);
      tc_fence_after();
      if (wt == 0) {
        mbar_arrive(&B->st[b]);
        // O^T += U^T P^T ;  S += (diag(exp(G_L - G)) K)^T U
        const uint32_t idp = idesc_bf16(128, 64, false, false);
        const uint64_t au = sdesc_sw128(sb + K2_UK, 16, 1024), bp = sdesc_sw128(sb + K2_P + b * 8192, 16, 1024);
        for (int ks = 0; ks < CT / 16; ++ks)
          mma_bf16(tbase + TM_OT + b * 64, au + ks * (32 >> 4), bp + ks * (32 >> 4), idp, 1u);
        const uint32_t ids = idesc_bf16(128, 128, true, false);
        const uint64_t akt = sdesc_sw128(sb + qk + 8192, 16384, 1024);
        for (int ks = 0; ks < CT / 16; ++ks)
          mma_bf16(tbase + TM_S, akt + ks * (2048 >> 4), au + ks * (32 >> 4), ids, 1u);
        mma_commit(&B->gh[b]);
      }
      ok = wait_bar(&B->gh[b], (c >> 1) & 1, abort);
      if (named_sync_or(2, 128, !ok)) { fail = true; break; }
      tc_fence_after();
    }
    if (fail) {
      if (wt == 0) {
        mbar_wait(&B->fg, c & 1, WAIT_LIMIT);
        mbar_wait(&B->gh[c & 1], (c >> 1) & 1, WAIT_LIMIT);
      }
    } else if (p.ST) {
      const int dk = wt;
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
  } else {
    // ============================== OUT ==============================
    // Per chunk: scale Q by gamma and K by exp(G_L - G) in place once PREP's
    // products have read them raw, write W for STATE, then store the
    // previous chunk's output rows.
    Tout* o = static_cast<Tout*>(p.o);
    const int dv = wt;
    auto store_out = [&](int c) -> bool {
      const int b = c & 1;
      const int c0 = bos + c * CT, len = min(CT, eos - c0);
      const bool ok = wait_bar(&B->gh[b], (c >> 1) & 1, abort);
      if (named_sync_or(3, 128, !ok)) return false;
      tc_fence_after();
      float v[64];
      tm_ld64(lane_base + TM_OT + b * 64, v);   // lane dv holds O[0..63][dv]
      Tout* dst = o + ((size_t)c0 * p.Nv + h) * DV + dv;
#pragma unroll
      for (int r = 0; r < CT; ++r)
        if (r < len) dst[(size_t)r * p.Nv * DV] = from_f32<Tout>(p.scale * v[r]);
      tc_fence_before();
      named_sync(3, 128);
      if (wt == 0) mbar_arrive(&B->of[b]);
      return true;
    };
    bool alive = true;
    for (int c = 0; c < n && alive; ++c) {
      const int st3 = c % 3;
      const uint32_t qk = K2_QK + st3 * 32768;
      const float* Gam = reinterpret_cast<const float*>(sm + K2_VEC + st3 * 768) + CT;
      const float* Dec = Gam + CT;
      bool ok = wait_bar(&B->pv, c & 1, abort) && wait_bar(&B->p, c & 1, abort);
      if (ok && c >= 1) ok = wait_bar(&B->fg, (c - 1) & 1, abort);   // W buffer free
      if (named_sync_or(3, 128, !ok)) break;
      tc_fence_after();
      scale_box(sm, qk, Gam, wt, 128);
      scale_box(sm, qk + 16384, Gam, wt, 128);
      scale_box(sm, qk + 8192, Dec, wt, 128);
      scale_box(sm, qk + 24576, Dec, wt, 128);
      {
        float v[64];
        tm_ld64(lane_base + TM_WT, v);          // lane dk holds W[0..63][dk]
        st_row64(sm, K2_WMN, wt, v);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      named_sync(3, 128);
      if (wt == 0) mbar_arrive(&B->sc);
      if (c >= 1) alive = store_out(c - 1);
    }
    if (alive && n > 0) store_out(n - 1);
  }

  if (*abort && tid == 0) raise_error(p.err, kDevErrTimeout);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, 512);
}

// ---- host: tensor maps and launch
// 2-D bf16 map over a token-major [rows, cols] matrix with a 64 x 64 box, 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* base, int rows, int cols) {
  return make_tmap_2d(map, base, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rows, cols, 64, 64,
                      CU_TENSOR_MAP_SWIZZLE_128B);
}

template <typename Tout>
cudaError_t launch_scan(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const ChunkArgs& p,
                        cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(chunk_scan_kernel<Tout>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)K2_SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid(p.Nv, p.num_seqs);
  chunk_scan_kernel<Tout><<<grid, NT2, K2_SMEM, s>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace

bool chunk_tc_supported(const ChunkArgs& p) {
  return p.Dk == DK && p.Dv == DV && p.in_bf16 && tmap_encoder() != nullptr;
}

size_t chunk_tc_workspace_bytes(int num_seqs, int total, int Nv) {
  return ((size_t)(total / CT) + (size_t)num_seqs) * (size_t)Nv * TILE_T_BYTES;
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
  cudaError_t e = cudaFuncSetAttribute(chunk_solve_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)S1_SMEM);
  if (e != cudaSuccess) return e;
  const int slots = p.total / CT + p.num_seqs;
  dim3 g1(slots, p.Nv);
  chunk_solve_kernel<<<g1, 128, S1_SMEM, s>>>(mk, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return p.out_bf16 ? launch_scan<bf16>(mq, mk, mv, p, s) : launch_scan<float>(mq, mk, mv, p, s);
}

// ---------------------------------------------------------------------------
// Library-owned scratch for callers that cannot allocate device memory.
// A fixed array in the module's device memory replaces the caller-provided
// workspace of gdn_chunk_prefill.  Every device that loads the library holds
// it until the process exits; every call shares it.
// ---------------------------------------------------------------------------
namespace {
__device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];
std::mutex g_static_mu;
void* g_static_ptr[64];
}  // namespace

cudaError_t static_scratch(void** ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (g_static_ptr[dev] == nullptr) {
    // host code sees only a stand-in for the array: ask the runtime for its
    // address on the current device (once per device)
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return e;
    g_static_ptr[dev] = p;
  }
  *ptr = g_static_ptr[dev];
  return cudaSuccess;
}

}  // namespace gdn
