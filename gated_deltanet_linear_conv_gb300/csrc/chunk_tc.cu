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
// Two parts:
//  * the solve, independent per (chunk, value head): K K^T and Q K^T on the
//    tensor core, A and P, T = (I + A)^-1 in fp32 on CUDA cores, and
//    W = T diag(beta gamma) K; it writes one workspace tile per (chunk, head):
//    [-W | diag(gamma) Q], P, the decays, and T diag(beta), as bf16 tiles in
//    the 128-byte-swizzled layout of a TMA load;
//  * the scan, one CTA per (sequence, value head), carries S through the
//    chunks with S^T resident in tensor memory.  PREP (warp 0) forms
//    [U~^T | 0]; STATE (warps 1-4) runs the S-dependent products, whose A
//    operands (bf16 S^T and U^T) it writes back into tensor memory; OUT
//    (warps 5-8) issues the O product and stores the output rows; a LOADER
//    warp (fused launch) brings each chunk's tiles in.  Every product is an
//    M = 128 tcgen05.mma with Dv on the tensor-memory lanes.
// A single sequence runs both parts in one cooperative launch: the scan CTAs
// take the chunks' tiles as soon as solve groups on the other SMs publish
// them.  Packed batches run the solve kernel, then the scan kernel.
// Every mbarrier wait is bounded; on a timeout the CTA raises the device
// error flag, lets its outstanding copies and products land, releases its
// tensor memory and exits.

#include <cuda.h>

#include "common.cuh"
#include "launch.h"
#include "tc_util.cuh"
#include "tmap.cuh"

#include <array>
#include <mutex>

namespace gdn {
namespace {

using namespace tc;

constexpr int CT = 64;        // chunk length
constexpr int DK = 128;
constexpr int DV = 128;
constexpr uint32_t WAIT_LIMIT = 1u << 22;
// workspace per (chunk, value head), written by the solve kernel:
//   [-W dk0-63 | Q~ dk0-63 | -W dk64-127 | Q~ dk64-127]  the N = 128 operand of the S products
//   P, then dec = exp(G_L - G) (64 floats) and gamma_L, then T diag(beta)
// (bf16 tiles in the 128-byte-swizzled layout a TMA load would give).
constexpr uint32_t WS_QW = 0, WS_P = 32768, WS_VEC = 40960, WS_TB = 41472;
constexpr uint32_t TILE_T_BYTES = 49664;

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
  tmem_ld_fence(a);
  tmem_ld_fence(b);
#pragma unroll
  for (int i = 0; i < 32; ++i) { v[i] = a[i]; v[32 + i] = b[i]; }
}

// Inclusive prefix sum of g over the chunk by one warp (lane l owns l, l+32);
// writes G, gamma = exp(G) and dec = exp(G_L - G).
__device__ __forceinline__ void chunk_cumsum(float* Gs, float* Gam, float* Dec, float* Alp, int lane) {
  float a0 = Gs[lane], a1 = Gs[lane + 32];
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float t0 = __shfl_up_sync(0xffffffffu, a0, off);
    const float t1 = __shfl_up_sync(0xffffffffu, a1, off);
    if (lane >= off) { a0 += t0; a1 += t1; }
  }
  a1 += __shfl_sync(0xffffffffu, a0, 31);
  const float gl = __shfl_sync(0xffffffffu, a1, 31);
  // per-token factors e^(G_t - G_(t-1)): their products over t = j+1..r telescope to e^(G_r - G_j)
  const float p0 = __shfl_up_sync(0xffffffffu, a0, 1), p1 = __shfl_up_sync(0xffffffffu, a1, 1);
  const float a0_31 = __shfl_sync(0xffffffffu, a0, 31);
  Gs[lane] = a0;
  Gs[lane + 32] = a1;
  Gam[lane] = __expf(a0);
  Gam[lane + 32] = __expf(a1);
  Dec[lane] = __expf(gl - a0);
  Dec[lane + 32] = __expf(gl - a1);
  Alp[lane] = lane > 0 ? __expf(a0 - p0) : __expf(a0);
  Alp[lane + 32] = __expf(a1 - (lane > 0 ? p1 : a0_31));
}

// Workspace slot of chunk c of sequence s: floor(bos_s / 64) + s + c.  Slots
// of different sequences never collide and stay below total / 64 + num_seqs.
__device__ __forceinline__ int slot_base(const ChunkArgs& p, int s) {
  return seq_start(p.cu, p.num_seqs, p.total, s) / CT + s;
}

// ---------------------------------------------------------------------------
// kernel 1: per (chunk slot, value head), in parallel over all of them
//   D1 = [K; Q] K^T (rows 0-63 K K^T, rows 64-127 Q K^T), A and P from it,
//   T = (I + A)^-1 in fp32 on CUDA cores, W = T diag(beta gamma) K.
//   Writes every workspace tile of the head.
// ---------------------------------------------------------------------------
constexpr int FS = 68;                              // fp32 row stride: 16-byte rows, conflict-free columns
constexpr uint32_t S1_QK = 0;                       // K box0 | Q box0 | K box1 | Q box1 (32 KB)
constexpr uint32_t S1_AT = 32768;                   // A^T fp32 [k][i]; later [T diag(beta gamma)] twice, bf16
constexpr uint32_t S1_TR = S1_AT + 64 * FS * 4;     // T fp32 [i][j]
constexpr uint32_t S1_XS = S1_TR + 64 * FS * 4;     // block-product scratch, fp32 32 x 36
constexpr uint32_t S1_VEC = S1_XS + 32 * 36 * 4;    // G, beta, beta*gamma, gamma, dec, alpha (6 x 64 floats)
constexpr uint32_t S1_BAR = S1_VEC + 6 * 64 * 4;
constexpr uint32_t S1_SMEM = S1_BAR + 64 + 1024;
static_assert(S1_TR % 1024 == 0 && S1_AT % 1024 == 0, "tile alignment");

// One warp's m16n8k8 product on the tensor core through mma.sync, tf32 operands
// (10-bit mantissa, rounded to nearest) and fp32 accumulation: d += a b.
// Fragments (g = lane / 4, t = lane % 4):  a = A[g][t], A[g+8][t], A[g][t+4], A[g+8][t+4];
// b = B[t][g], B[t+4][g];  d = D[g][2t], D[g][2t+1], D[g+8][2t], D[g+8][2t+1].
__device__ __forceinline__ uint32_t tf32_rn(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ void mma_tf32(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One warp: T[R:R+16M][C+8w : C+8w+8] = -T[R:R+16M][R:R+16M] (A[R:R+16M][C:C+16M] T[C:C+16M][C+8w : ...])
// for an M x M block (M = 1: 16 x 16, M = 2: 32 x 32) below the diagonal, w the warp's
// 8-column tile.  The intermediate X (16M x 8) goes through the warp's own scratch XW
// (16M x 8 floats) from accumulator to operand layout.
template <int M>
__device__ __forceinline__ void merge_tile(const float* AT, float* TR, float* XW, int R, int C, int w, int lane) {
  const int g = lane >> 2, t = lane & 3;
  const int n0 = C + 8 * w;
  float x[M][4];
#pragma unroll
  for (int mt = 0; mt < M; ++mt) x[mt][0] = x[mt][1] = x[mt][2] = x[mt][3] = 0.f;
#pragma unroll
  for (int ks = 0; ks < 2 * M; ++ks) {             // X = A21 T11: K = 16 M
    const int k = C + 8 * ks + t;
    const uint32_t b0 = tf32_rn(TR[k * FS + n0 + g]), b1 = tf32_rn(TR[(k + 4) * FS + n0 + g]);
#pragma unroll
    for (int mt = 0; mt < M; ++mt) {
      const int r = R + 16 * mt + g;                // A[r][k] = AT[k][r]
      mma_tf32(x[mt], tf32_rn(AT[k * FS + r]), tf32_rn(AT[k * FS + r + 8]), tf32_rn(AT[(k + 4) * FS + r]),
               tf32_rn(AT[(k + 4) * FS + r + 8]), b0, b1);
    }
  }
#pragma unroll
  for (int mt = 0; mt < M; ++mt) {
    *reinterpret_cast<float2*>(XW + (16 * mt + g) * 8 + 2 * t) = make_float2(x[mt][0], x[mt][1]);
    *reinterpret_cast<float2*>(XW + (16 * mt + g + 8) * 8 + 2 * t) = make_float2(x[mt][2], x[mt][3]);
  }
  __syncwarp();
  float y[M][4];
#pragma unroll
  for (int mt = 0; mt < M; ++mt) y[mt][0] = y[mt][1] = y[mt][2] = y[mt][3] = 0.f;
#pragma unroll
  for (int ks = 0; ks < 2 * M; ++ks) {             // T21 = -T22 X: K = 16 M
    const int k = 8 * ks + t;
    const uint32_t b0 = tf32_rn(XW[k * 8 + g]), b1 = tf32_rn(XW[(k + 4) * 8 + g]);
#pragma unroll
    for (int mt = 0; mt < M; ++mt) {
      const float* tr = TR + (R + 16 * mt + g) * FS + R + k;
      mma_tf32(y[mt], tf32_rn(tr[0]), tf32_rn(tr[8 * FS]), tf32_rn(tr[4]), tf32_rn(tr[8 * FS + 4]), b0, b1);
    }
  }
#pragma unroll
  for (int mt = 0; mt < M; ++mt) {
    *reinterpret_cast<float2*>(TR + (R + 16 * mt + g) * FS + n0 + 2 * t) = make_float2(-y[mt][0], -y[mt][1]);
    *reinterpret_cast<float2*>(TR + (R + 16 * mt + g + 8) * FS + n0 + 2 * t) = make_float2(-y[mt][2], -y[mt][3]);
  }
}

// Write 64 bf16 values (times sc) as swizzled row `row` of a 64-column block in global memory.
__device__ __forceinline__ void st_row64_global(uint8_t* dst, uint32_t row, const float* v, float sc) {
#pragma unroll
  for (int ch = 0; ch < 8; ++ch) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 h = __floats2bfloat162_rn(sc * v[ch * 8 + 2 * i], sc * v[ch * 8 + 2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    const uint32_t off = row * 128u + ((((uint32_t)ch ^ (row & 7u)) & 7u) << 4);
    *reinterpret_cast<uint4*>(dst + off) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// T = (I + A)^-1 for a 64 x 64 strictly lower A given transposed (AT[k][i] =
// A[i][k], stride FS), by 128 threads into TR (row-major, stride FS; TR must
// hold zeros above the diagonal blocks on entry).
//   1. the four 16 x 16 diagonal blocks, one column per thread (64 threads), fp32;
//   2. T[b+1][b] = -T[b+1][b+1] (A[b+1][b] T[b][b]) for the pairs (0,1), (2,3): warp w
//      takes pair w / 2, columns 8 (w % 2) .. + 8 of the block;
//   3. T[32:64][0:32] = -T[32:64][32:64] (A[32:64][0:32] T[0:32][0:32]): warp w takes
//      columns 8w .. 8w + 8.
// The block products of 2 and 3 run on the tensor core (mma.sync, tf32 operands, fp32
// accumulation); T is rounded to bf16 when it is used.  XS is fp32 scratch of 4 KB.
// The 128 threads synchronise on named barrier barid.
__device__ __forceinline__ void invert_unit_lower(const float* AT, float* TR, float* XS, int tid, uint32_t barid) {
  if (tid < 64) {
    const int b = (tid >> 4) * 16, c = tid & 15;
    float2 x[8];                                       // x[i / 2] holds elements i, i + 1
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = make_float2(2 * i == c ? 1.f : 0.f, 2 * i + 1 == c ? 1.f : 0.f);
#pragma unroll
    for (int k = 0; k < 15; ++k) {
      const float xk = (k & 1) ? x[k >> 1].y : x[k >> 1].x;
      const float2 nxk = make_float2(-xk, -xk);
#pragma unroll
      for (int i4 = ((k + 1) >> 2) << 2; i4 < 16; i4 += 4) {
        const float4 a = *reinterpret_cast<const float4*>(AT + (b + k) * FS + b + i4);
#pragma unroll
        for (int hp = 0; hp < 2; ++hp) {             // the pair (i, i + 1), i = i4 + 2 hp
          const int i = i4 + 2 * hp;
          const float2 ap = hp ? make_float2(a.z, a.w) : make_float2(a.x, a.y);
          if (i > k) x[i >> 1] = __ffma2_rn(ap, nxk, x[i >> 1]);
          else if (i + 1 > k) x[i >> 1].y = fmaf(ap.y, -xk, x[i >> 1].y);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      TR[(b + 2 * i) * FS + b + c] = x[i].x;
      TR[(b + 2 * i + 1) * FS + b + c] = x[i].y;
    }
  }
  named_sync(barid, 128);
  const int w = tid >> 5, lane = tid & 31;
  merge_tile<1>(AT, TR, XS + w * 256, 16 * (2 * (w >> 1) + 1), 32 * (w >> 1), w & 1, lane);
  named_sync(barid, 128);
  merge_tile<2>(AT, TR, XS + w * 256, 32, 0, w, lane);
  named_sync(barid, 128);
}

// The scan's waits are bounded in time: each gives up after limit_ns of device
// time (%globaltimer), or at once when another role of the CTA aborted.  An mbarrier
// wait takes its start time on entry; a flag poll reads the timer only every 64th
// poll, the first such read being its start.  A poll cap far above any limit in use
// ends the loop even if the timer were not to advance.  (The mbarrier wait has no
// separate test_wait fast path: the smaller inlined loop measured faster.)
struct WaitCtl {
  volatile int* abort;
  uint64_t limit_ns;
};
constexpr uint32_t POLL_CAP = 1u << 28;

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait (thread 0 of a solve group) until a chunk's flag reached `need`: its
// tiles were published and every scan that reads them released them.
__device__ __forceinline__ bool wait_count(const int* f, int need, uint64_t limit_ns) {
  const uint64_t t0 = global_ns();
  for (uint32_t i = 0; i < POLL_CAP; ++i) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
    if (v >= need) return true;
    if (v < 0 || global_ns() - t0 > limit_ns) break;
    __nanosleep(64);
  }
  return false;
}

// Token range of chunk slot `slot`: false when the slot holds no chunk (past the end
// of its sequence, or a sequence whose bounds are inconsistent: the scan reports that).
__device__ __forceinline__ bool slot_chunk(const ChunkArgs& p, int slot, int& c0, int& len) {
  int lo = 0, hi = p.num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (slot_base(p, mid) <= slot) lo = mid; else hi = mid - 1;
  }
  const int s = lo, c = slot - slot_base(p, s);
  int bos, eos;
  if (!seq_bounds(p.cu, p.num_seqs, p.total, s, bos, eos)) return false;
  if (c < 0 || c * CT >= eos - bos) return false;
  c0 = bos + c * CT;
  len = min(CT, eos - c0);
  return true;
}

// This thread's gate value of an item: g (threads 0-63) or beta (threads 64-127) of
// token c0 + tid % 64 of value head h; 0 past the chunk's end.
__device__ __forceinline__ float solve_gate(const ChunkArgs& p, int tid, int c0, int len, int h) {
  return (tid & 63) < len ? __ldg((tid < CT ? p.g : p.beta) + (size_t)(c0 + (tid & 63)) * p.Nv + h) : 0.f;
}

// The Q and K tiles of an item into the group's QK buffer (thread 0).
__device__ __forceinline__ void solve_load_tiles(uint8_t* sm, uint64_t* bar, const CUtensorMap* tmq,
                                                 const CUtensorMap* tmk, const ChunkArgs& p, int c0, int h) {
  const int hk = h / (p.Nv / p.Nk);
  mbar_arrive_expect_tx(bar, 32768);
  tma_load_2d(sm + S1_QK, tmk, bar, hk * DK, c0);
  tma_load_2d(sm + S1_QK + 8192, tmq, bar, hk * DK, c0);
  tma_load_2d(sm + S1_QK + 16384, tmk, bar, hk * DK + 64, c0);
  tma_load_2d(sm + S1_QK + 24576, tmq, bar, hk * DK + 64, c0);
}

// Loads of the next item that a group issues while it works on the current one.
struct SolveAhead {
  bool tiles;    // its Q, K tiles were issued into the QK buffer (on the group's mbarrier)
  bool gate;     // gb holds this thread's gate value of it
  float gb;
  int slot, c0, len;   // its chunk slot and token range (slot -1: not known yet)
};

// A flag store after solve_item's closing fence: the fence (acq_rel, gpu scope, by the
// storing thread after a barrier of the whole group) and this strong relaxed store form a
// release of every tile store of the group (a release store would fence a second time).
__device__ __forceinline__ void st_flag(int* f, int v) {
  asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(f), "r"(v) : "memory");
}

// Claim the next work item: a relaxed atomic add issued where it stands in the program
// (its result is read only after the current item, so its latency hides under it).
__device__ __forceinline__ int claim_item(int* counter) {
  int v;
  asm volatile("atom.relaxed.gpu.global.add.s32 %0, [%1], 1;" : "=r"(v) : "l"(counter) : "memory");
  return v;
}

// One (chunk slot, value head) by 128 threads (tid 0-127 of a group that
// synchronises on named barrier barid).  sm is the group's 1024-aligned
// shared memory (S1_BYTES), bar an initialised mbarrier whose next phase
// parity is ph & 1 (ph advances by three), tbase 128 allocated tensor-memory
// columns.  The tiles go to workspace tile `tile` (of the item's head) as direct
// 16-byte stores, once `rel` (if given) reached rel_need; when this returns, thread 0
// has fenced them for the group after a barrier (a relaxed flag store of its then publishes them).  `ahead` carries the
// loads this item issues for the next one (nslot < 0: none): its gate values, in
// flight under this item's A and P rows, and its Q, K tiles, issued by thread 0 as
// soon as this item's W product has completed (the last reader of the QK buffer).
// Returns false, with the device error flag raised, on a timeout.
__device__ bool solve_item(uint8_t* sm, int tid, uint32_t barid, uint64_t* bar, uint32_t& ph, uint32_t tbase,
                           const CUtensorMap* tmq, const CUtensorMap* tmk, const ChunkArgs& p, int slot, int h,
                           SolveAhead& ahead, int nslot, int nh, size_t tile, const int* rel, int rel_need,
                           bool publish = true) {
  float* AT = reinterpret_cast<float*>(sm + S1_AT);
  float* TR = reinterpret_cast<float*>(sm + S1_TR);
  float* XS = reinterpret_cast<float*>(sm + S1_XS);
  float* Gs = reinterpret_cast<float*>(sm + S1_VEC);
  float* Bet = Gs + CT;
  float* BG = Bet + CT;
  float* Gam = BG + CT;
  float* Dec = Gam + CT;
  float* Alp = Dec + CT;                 // e^(G_t - G_(t-1))
  const int warp = tid >> 5, lane = tid & 31;
  int c0 = 0, len = 0;
  const bool used = ahead.slot == slot ? (c0 = ahead.c0, len = ahead.len, true) : slot_chunk(p, slot, c0, len);
  int nc0 = 0, nlen = 0;
  const bool nused = nslot >= 0 && slot_chunk(p, nslot, nc0, nlen);
  ahead.slot = nused ? nslot : -1;     // (the next item reuses its range)
  ahead.c0 = nc0;
  ahead.len = nlen;
  if (!used) {                // nothing to solve (tiles are only ever prefetched for used slots)
    ahead.gate = false;
    return true;
  }
  uint8_t* ws = static_cast<uint8_t*>(p.workspace) + (tile * p.Nv + h) * TILE_T_BYTES;
  const uint32_t lane_base = tbase + ((uint32_t)(warp * 32) << 16);
  const uint32_t sb = smem_u32(sm);

  if (tid == 0 && !ahead.tiles) solve_load_tiles(sm, bar, tmq, tmk, p, c0, h);
  ahead.tiles = false;
  // threads 0-63 hold g, threads 64-127 beta (loaded during the item before, else now);
  // the zeroing of T (which starts at zero above its diagonal blocks) runs meanwhile
  const float gb = ahead.gate ? ahead.gb : solve_gate(p, tid, c0, len, h);
  for (int i = tid * 4; i < 64 * FS; i += 128 * 4)
    *reinterpret_cast<float4*>(TR + i) = make_float4(0.f, 0.f, 0.f, 0.f);
  (tid < CT ? Gs : Bet)[tid & 63] = gb;
  named_sync(barid, 128);
  if (warp == 0) {
    chunk_cumsum(Gs, Gam, Dec, Alp, lane);
    BG[lane] = Bet[lane] * Gam[lane];
    BG[lane + 32] = Bet[lane + 32] * Gam[lane + 32];
  }
  bool ok = mbar_wait(bar, ph & 1u, WAIT_LIMIT);
  ph += 1;
  if (!named_sync_or(barid, 128, !ok)) {
    tc_fence_after();
    if (tid == 0) {
      const uint32_t id = idesc_bf16(128, 64, false, false);
      const uint64_t a = sdesc_sw128(sb + S1_QK, 16, 1024);
#pragma unroll
      for (int ks = 0; ks < DK / 16; ++ks) {
        const uint32_t o = ((ks >> 2) * 16384 + (ks & 3) * 32) >> 4;
        mma_bf16(tbase, a + o, a + o, id, ks > 0 ? 1u : 0u);
      }
      mma_commit(bar);
    }
    ok = mbar_wait(bar, ph & 1u, WAIT_LIMIT);
  }
  ph += 1;
  // the next item's gate value, in flight under this item's work
  ahead.gate = nused;
  if (nused) ahead.gb = solve_gate(p, tid, nc0, nlen, nh);
  // a ring position is written only once the chunk that used it before is released
  if (tid == 0 && rel != nullptr && ok && !wait_count(rel, rel_need, p.wait_ns)) ok = false;
  bool done = false;
  if (!named_sync_or(barid, 128, !ok)) {
    tc_fence_after();
    {
      float v[64];
      tm_ld64(lane_base, v);
      // The decay e^(G_r - G_j), j <= r, is a running product of the per-token factors
      // (no exponential per element).
      if (tid < CT) {
        // K K^T is symmetric: this thread's row j of it is column j, and column j of
        // A (A[r][j] = beta_r (k_r . k_j) e^(G_r - G_j), r > j) is row j of A^T
        const int j = tid;
        float cur = 1.f;
#pragma unroll
        for (int rb = 0; rb < 64; rb += 16) {
          float al[16], be[16];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float4 ta = *reinterpret_cast<const float4*>(Alp + rb + 4 * i);
            const float4 tb = *reinterpret_cast<const float4*>(Bet + rb + 4 * i);
            al[4 * i] = ta.x; al[4 * i + 1] = ta.y; al[4 * i + 2] = ta.z; al[4 * i + 3] = ta.w;
            be[4 * i] = tb.x; be[4 * i + 1] = tb.y; be[4 * i + 2] = tb.z; be[4 * i + 3] = tb.w;
          }
#pragma unroll
          for (int r = rb; r < rb + 16; ++r) {
            cur = r > j ? cur * al[r - rb] : cur;
            v[r] = r > j ? be[r - rb] * v[r] * cur : 0.f;
          }
        }
#pragma unroll
        for (int r = 0; r < 64; r += 4)
          *reinterpret_cast<float4*>(AT + j * FS + r) = make_float4(v[r], v[r + 1], v[r + 2], v[r + 3]);
      } else {
        // row r of P = M o Q K^T: (q_r . k_j) e^(G_r - G_j) for j <= r, the product taken from j = r down
        const int r = tid - CT;
        float cur = 1.f;
#pragma unroll
        for (int jb = 48; jb >= 0; jb -= 16) {
          float al[17];                       // alpha[jb + 1 .. jb + 16]
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float4 ta = *reinterpret_cast<const float4*>(Alp + jb + 4 * i);
            al[4 * i] = ta.x; al[4 * i + 1] = ta.y; al[4 * i + 2] = ta.z; al[4 * i + 3] = ta.w;
          }
          al[16] = jb + 16 < 64 ? Alp[jb + 16] : 1.f;
#pragma unroll
          for (int j = jb + 15; j >= jb; --j) {
            cur = j < r ? cur * al[j + 1 - jb] : cur;
            v[j] = j <= r ? v[j] * cur : 0.f;
          }
        }
        st_row64_global(ws + WS_P, r, v, 1.f);
      }
    }
    // diag(gamma) Q -> rows 64-127 of the two [-W; Q~] blocks (same swizzled rows as
    // the TMA tiles), then dec and gamma_L
    {
      uint4 qu[8];
      float f[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {          // every read before the first store
        const int i = tid + 128 * k;
        const uint32_t off = (uint32_t)(i >> 9) * 16384u + (uint32_t)(i & 511) * 16u;
        qu[k] = *reinterpret_cast<const uint4*>(sm + S1_QK + 8192 + off);
        f[k] = Gam[(i & 511) >> 3];
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int i = tid + 128 * k;
        const uint32_t off = (uint32_t)(i >> 9) * 16384u + (uint32_t)(i & 511) * 16u;
        uint32_t w[4] = {qu[k].x, qu[k].y, qu[k].z, qu[k].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 x = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&w[j]));
          __nv_bfloat162 y = __floats2bfloat162_rn(x.x * f[k], x.y * f[k]);
          w[j] = *reinterpret_cast<uint32_t*>(&y);
        }
        *reinterpret_cast<uint4*>(ws + WS_QW + 8192 + off) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    if (tid < CT) reinterpret_cast<float*>(ws + WS_VEC)[tid] = Dec[tid];
    if (tid == 0) reinterpret_cast<float*>(ws + WS_VEC)[CT] = Gam[CT - 1];
    tc_fence_before();
    named_sync(barid, 128);
    invert_unit_lower(AT, TR, XS, tid, barid);
    // A^T is dead: its space becomes the [T diag(beta gamma); T diag(beta gamma)] operand (the
    // rows twice, so that all four warps take a share of W out of tensor memory)
    uint8_t* tbg = sm + S1_AT;
    {
      // thread (r, ch) = (tid / 8 + 16 k, tid % 8): every read of T, beta and beta gamma
      // before the first store (the stores go over the dead A^T)
      const int ch = tid & 7;
      float4 t0[4], t1[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int r = (tid >> 3) + 16 * k;
        t0[k] = *reinterpret_cast<const float4*>(TR + r * FS + ch * 8);
        t1[k] = *reinterpret_cast<const float4*>(TR + r * FS + ch * 8 + 4);
      }
      const float4 be0 = *reinterpret_cast<const float4*>(Bet + ch * 8);
      const float4 be1 = *reinterpret_cast<const float4*>(Bet + ch * 8 + 4);
      const float4 bg0 = *reinterpret_cast<const float4*>(BG + ch * 8);
      const float4 bg1 = *reinterpret_cast<const float4*>(BG + ch * 8 + 4);
      const float be[8] = {be0.x, be0.y, be0.z, be0.w, be1.x, be1.y, be1.z, be1.w};
      const float bgv[8] = {bg0.x, bg0.y, bg0.z, bg0.w, bg1.x, bg1.y, bg1.z, bg1.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int r = (tid >> 3) + 16 * k;
        const float t[8] = {t0[k].x, t0[k].y, t0[k].z, t0[k].w, t1[k].x, t1[k].y, t1[k].z, t1[k].w};
        uint32_t wa[4], wb[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          __nv_bfloat162 ha = __floats2bfloat162_rn(t[2 * i] * be[2 * i], t[2 * i + 1] * be[2 * i + 1]);
          __nv_bfloat162 hb = __floats2bfloat162_rn(t[2 * i] * bgv[2 * i], t[2 * i + 1] * bgv[2 * i + 1]);
          wa[i] = *reinterpret_cast<uint32_t*>(&ha);
          wb[i] = *reinterpret_cast<uint32_t*>(&hb);
        }
        const uint32_t sw = r * 128u + ((((uint32_t)ch ^ (uint32_t)(r & 7)) & 7u) << 4);
        *reinterpret_cast<uint4*>(ws + WS_TB + sw) = make_uint4(wa[0], wa[1], wa[2], wa[3]);
        *reinterpret_cast<uint4*>(tbg + sw) = make_uint4(wb[0], wb[1], wb[2], wb[3]);
        *reinterpret_cast<uint4*>(tbg + 8192 + sw) = make_uint4(wb[0], wb[1], wb[2], wb[3]);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    named_sync(barid, 128);
    tc_fence_after();
    if (tid == 0) {
      // W = T diag(beta gamma) K, in rows 0-63 and again in rows 64-127 of the 128 x 128 result
      const uint32_t id = idesc_bf16(128, 128, false, true);
      const uint64_t a = sdesc_sw128(sb + S1_AT, 16, 1024);
      const uint64_t b = sdesc_sw128(sb + S1_QK, 16384, 1024);
#pragma unroll
      for (int ks = 0; ks < CT / 16; ++ks) mma_bf16(tbase, a + ks * 2, b + ks * 128, id, ks > 0 ? 1u : 0u);
      mma_commit(bar);
    }
    ok = mbar_wait(bar, ph & 1u, WAIT_LIMIT);
    if (!named_sync_or(barid, 128, !ok)) {
      tc_fence_after();
      {   // -W, swizzled, over the K tiles (the W product has read them): warps 0-1 columns
          // 0-63 of rows 0-63, warps 2-3 columns 64-127 of the copy
        const int half = tid >> 6;
        float v[64];
        tm_ld64(lane_base + half * 64, v);
#pragma unroll
        for (int i = 0; i < 64; ++i) v[i] = -v[i];
        st_row64(sm, S1_QK + half * 16384, tid & 63, v);
      }
      named_sync(barid, 128);
      // ... and out to the workspace in 512-byte runs per warp instruction (the row per
      // thread above would touch 32 lines per instruction)
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int i = tid + 128 * k;                  // 16-byte chunk of the two 8 KB boxes
        const uint32_t off = (uint32_t)(i >> 9) * 16384u + (uint32_t)(i & 511) * 16u;
        *reinterpret_cast<uint4*>(ws + WS_QW + off) = *reinterpret_cast<const uint4*>(sm + S1_QK + off);
      }
      named_sync(barid, 128);
      // the QK buffer is free: the next item's tiles may land there
      if (tid == 0 && nused) solve_load_tiles(sm, bar, tmq, tmk, p, nc0, nh);
      ahead.tiles = nused;
      done = true;
    }
  }
  ph += 1;
  if (!done && tid == 0) raise_error(p.err, kDevErrTimeout);
  // the next item may reuse this shared and tensor memory; thread 0 then fences for the
  // group (the barrier orders every thread's tile stores before its fence and flag) when a
  // flag publishes the tile (`publish`; the packed path's scans run in a later launch)
  tc_fence_before();
  named_sync(barid, 128);
  tc_fence_after();
  if (publish && tid == 0) asm volatile("fence.acq_rel.gpu;" ::: "memory");
  return done;
}

// Packed batches: persistent CTAs (three per SM) claim (chunk slot, value head) items
// in slot order from an atomic counter, one ahead, so that the next item's gate
// values and tiles load under the current one.
__global__ void __launch_bounds__(128, 3)
chunk_solve_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                   ChunkArgs p, int nitems, int* counter) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = tc::smem_aligned<1024>(smem_raw);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + S1_BAR);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + S1_BAR + 16);
  volatile int* item_slot = reinterpret_cast<volatile int*>(sm + S1_BAR + 32);   // two slots
  const int tid = threadIdx.x;
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_barrier_init();
  }
  if ((tid >> 5) == 0) tmem_alloc(tslot, 128);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  uint32_t ph = 0;
  // items claimed two ahead (see the one-sequence launch)
  if (tid == 0) {
    item_slot[0] = atomicAdd(counter, 1);
    item_slot[1] = atomicAdd(counter, 1);
  }
  __syncthreads();
  int item = item_slot[0], next = item_slot[1];
  SolveAhead ahead{false, false, 0.f, -1, 0, 0};
  int par = 0;
  while (item < nitems) {
    const int after = tid == 0 && next < nitems ? claim_item(counter) : nitems;
    const int nslot = next < nitems ? next / p.Nv : -1, nh = next < nitems ? next % p.Nv : 0;
    if (!solve_item(sm, tid, 1, bar, ph, *tslot, &tmq, &tmk, p, item / p.Nv, item % p.Nv, ahead, nslot, nh,
                    (size_t)(item / p.Nv), nullptr, 0, false))
      break;
    if (tid == 0) item_slot[par] = after;
    __syncthreads();
    item = next;
    next = item_slot[par];
    par ^= 1;
  }
  tc_fence_before();
  __syncthreads();
  if ((tid >> 5) == 0) tmem_dealloc(*tslot, 128);
}

// ---------------------------------------------------------------------------
// kernel 2: the scan over chunks
//   warp 0     PREP    [U~^T | 0] = V^T [T diag(beta); 0]^T once a chunk's v tiles land
//   warps 1-4  STATE   the S-dependent products and their epilogues
//   warps 5-8  OUT     the product O^T += U^T P^T (the STATE leader issues it when the
//                      gated norm is in the epilogue), then the output rows
//   warp 9     LOADER  (fused launch only) awaits each chunk's ready flag and issues its
//                      copies; without it PREP issues the v copies and OUT the stage copies
// The state lives in tensor memory transposed (lane dv, column dk, fp32).
// Per chunk, STATE writes S^T and U^T back into tensor memory as bf16 and
// every S-dependent product reads its A operand from there:
//   [U^T | O^T] += S^T [-W; Q~]^T          (N = 128, K = Dk)
//   S^T = gamma_L S^T + (U^T diag(dec)) K  (N = 128, K = 64; the scaling by gamma_L runs
//                                           in place while the product above is in flight)
//   O^T += U^T P^T                         (N = 64,  K = 64)
// ---------------------------------------------------------------------------
constexpr int NT2 = 288;
constexpr uint32_t STAGE_BYTES = 58368;     // [-W | Q~] 32 KB | K box0 | K box1 | P | dec, gamma_L
constexpr uint32_t SG_K = 32768, SG_P = 49152, SG_VEC = 57344;
constexpr uint32_t K2_ST = 0;                          // 2 stages
constexpr uint32_t K2_VT = 2 * STAGE_BYTES;            // 2 x [V box0 | V box1 | T diag(beta) | zeros]
constexpr uint32_t K2_OS = K2_VT + 2 * 32768;          // 2 x output tile (two 64 x 64 boxes)
constexpr uint32_t K2_RED = K2_OS + 2 * 16384;        // gated norm: weight (Dv floats, Dv bf16), row sums
constexpr uint32_t K2_BAR = K2_RED + 2048;
constexpr uint32_t K2_SMEM = K2_BAR + 256 + 1024;
static_assert(K2_SMEM <= 232448, "shared memory budget");
static_assert(SG_VEC + 512 <= STAGE_BYTES && WS_VEC == WS_P + 8192 && SG_VEC == SG_P + 8192, "stage layout");

// tensor memory columns
constexpr uint32_t TM_ACC = 0;     // 2 x [U^T (64) | O^T (64)], fp32
constexpr uint32_t TM_S = 256;     // S^T, fp32 (128)
constexpr uint32_t TM_SB = 384;    // S^T as bf16 pairs (64)
constexpr uint32_t TM_UD = 448;    // U^T diag(dec) as bf16 pairs (32)
constexpr uint32_t TM_UB = 480;    // U^T as bf16 pairs (32)

struct ScanBars {
  uint64_t stl[2];   // stage of a chunk landed ([-W | Q~], K, P, dec)
  uint64_t vt[2];    // v tiles and T diag(beta) of a chunk landed
  uint64_t ready[2]; // [U~^T | 0] of a chunk in its accumulator (MMA commit)
  uint64_t ob[2];    // O^T of a chunk complete (MMA commit)
  uint64_t of[2];    // OUT finished reading a chunk's accumulator
  uint64_t fg;       // [U^T | O^T] += S^T [-W; Q~]^T complete
  uint64_t gh;       // state update complete
  uint64_t zb[2];    // z tile of a chunk landed in its output buffer (gated norm)
  uint64_t ub[2];    // U^T of a chunk in tensor memory as bf16 and its S^T update issued
  uint64_t s0f;      // the initial state landed in shared memory (bulk copies)
  uint64_t s0c;      // the state role has moved it into tensor memory (128 arrivals)
  uint32_t tslot;
  int abort;
  int odone;         // side norm: chunks whose o stores have landed (the output role counts)
};
static_assert(sizeof(ScanBars) <= 256, "scan barriers fit their slot");

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, const WaitCtl& w) {
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1; i < POLL_CAP; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 1023u) == 0u && (*w.abort || global_ns() - t0 > w.limit_ns)) break;
  }
  *w.abort = 1;
  return false;
}

// Both phases at once: the two completed-phase tests are issued back to back.
__device__ __forceinline__ bool wait_bar2(uint64_t* b1, uint32_t p1, uint64_t* b2, uint32_t p2, const WaitCtl& w) {
  const bool t1 = mbar_test_wait(b1, p1), t2 = mbar_test_wait(b2, p2);
  if (t1 && t2) return true;
  return (t1 || wait_bar(b1, p1, w)) && (t2 || wait_bar(b2, p2, w));
}

// silu(z) = h + h tanh(h), h = z / 2, with the hardware tanh when the result is rounded
// to bf16, exact division for fp32.  The tanh's relative error (about 2^-11) leaves silu an
// absolute error of at most about 2^-11 |h|: within half a bf16 ulp of the result for z >= -2;
// below that silu is near zero and the error, though still far below the bf16 rounding of
// O(1) values, is no longer small relative to the result itself.
__device__ __forceinline__ float tanh_hw(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
template <typename Tout> __device__ __forceinline__ float silu_out(float z);
template <> __device__ __forceinline__ float silu_out<bf16>(float z) {
  const float hz = 0.5f * z;
  return fmaf(hz, tanh_hw(hz), hz);
}
template <> __device__ __forceinline__ float silu_out<float>(float z) { return silu_fast(z); }

// w silu(z) for two bf16 z values at once, in bf16x2 arithmetic (h + h tanh(h), h = z / 2,
// then times w): the gate of a bf16 output, whose own rounding is coarser than these steps.
__device__ __forceinline__ uint32_t gate_bf16x2(uint32_t z2, uint32_t w2) {
  uint32_t hz, t, s, g;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(hz) : "r"(z2), "r"(0x3F003F00u));     // z / 2
  asm("tanh.approx.bf16x2 %0, %1;" : "=r"(t) : "r"(hz));
  asm("fma.rn.bf16x2 %0, %1, %2, %1;" : "=r"(s) : "r"(hz), "r"(t));
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(g) : "r"(s), "r"(w2));
  return g;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h2 = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h2);
}

// Bounded wait until the solve of one (chunk slot, value head) published
// its workspace tiles (1), or reported a failure (-1).
__device__ __forceinline__ bool wait_flag(const int* f, const WaitCtl& w) {
  uint64_t t0 = 0;
  for (uint32_t i = 0; i < POLL_CAP; ++i) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
    if (v > 0) {
      asm volatile("fence.proxy.async.global;" ::: "memory");   // the tiles are read by the copy engine
      return true;
    }
    if (v < 0 || *w.abort) break;
    if ((i & 63u) == 63u) {
      const uint64_t now = global_ns();
      if (t0 == 0) t0 = now;
      else if (now - t0 > w.limit_ns) break;
    }
    __nanosleep(100);
  }
  *w.abort = 1;
  return false;
}

// What one scan CTA covers of its (sequence, value head): a range of its chunks,
// the state it starts from, and where its final state and output rows go.
//  - the whole sequence: S0 = the caller's initial state (or zeros), outputs to o;
//  - a later segment of a split sequence, from a zero state (its part of the state
//    and of the outputs that does not depend on the state it is entered with);
//  - that segment's transition map: the identity as the state (Dk = Dv) and no V
//    term, so that its "state" after chunk c is the product A_c ... A_first of the
//    chunk maps S -> A S of the homogeneous recurrence, and its "output" rows are
//    the response R of the chunk's outputs to the entry state (o += R S_entry).
struct ScanSeg {
  int c_begin, c_end;        // chunk range [c_begin, c_end) of the sequence (clipped to its end)
  const float* S0;           // initial state [Dk][Dv] of this (sequence, head), or null (zeros)
  bool identity;             // start from the identity instead (the transition map)
  bool zero_v;               // no V term: U~ = 0
  float* ST;                 // final state [Dk][Dv], or null (not written)
  void* out;                 // output rows [rows, Nv, Dv]: Tout, or bf16 when out_bf16
  bool out_bf16;             // the rows are bf16 whatever Tout is
  const CUtensorMap* tmo;    // bf16 map over `out` (used for bf16 rows of whole chunks)
  int row_off;               // token t is output row t - row_off
  int tile0, ring;           // workspace tiles: chunk c of the segment at position tile0 + c % ring
                             // (ring 0: one tile per chunk slot, at the sequence's slot + c)
  bool release;              // add one to a chunk's flag once its tiles are no longer needed
};

__device__ __forceinline__ void unpack8(const uint4 (&u)[1], float (&f)[8]) {   // 8 bf16
  const uint32_t w[4] = {u[0].x, u[0].y, u[0].z, u[0].w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
    f[2 * i] = a.x;
    f[2 * i + 1] = a.y;
  }
}
__device__ __forceinline__ void unpack8(const uint4 (&u)[2], float (&f)[8]) {   // 8 fp32
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    f[4 * j] = __uint_as_float(u[j].x);
    f[4 * j + 1] = __uint_as_float(u[j].y);
    f[4 * j + 2] = __uint_as_float(u[j].z);
    f[4 * j + 3] = __uint_as_float(u[j].w);
  }
}

// The gated RMSNorm of rows c0 .. c0 + len - 1 (len <= NB * NT / 16) of value head h, in
// place: y = o / sqrt(mean_dv o^2 + eps) * w * silu(z), o being the stored output row.  NT
// threads: thread (r, l) = (tid / 16, tid % 16) takes elements 8l .. 8l + 7 of rows
// r, r + NT/16, ...; every load is issued before the first use (one round trip; o is read
// from L2, where the scan's stores landed), and a row's sum of squares is a shuffle over
// its 16 lanes (one half-warp).
template <typename Tout, int NT, int NB>
__device__ __forceinline__ void norm_rows(const ChunkArgs& p, int c0, int len, int h, int tid, const float (&w)[8]) {
  constexpr int NR = sizeof(Tout) == 2 ? 1 : 2;      // 16-byte pieces of 8 output elements
  constexpr int RS = NT / 16;                         // rows per step
  const int l = tid & 15, r0 = tid >> 4;
  const unsigned half = (tid & 16) ? 0xffff0000u : 0x0000ffffu;
  uint4 ou[NB][NR], zu[NB];
#pragma unroll
  for (int i = 0; i < NB; ++i) {
    if (r0 + RS * i < len) {
      const size_t off = ((size_t)(c0 + r0 + RS * i) * p.Nv + h) * DV + 8 * l;
      const uint4* op = reinterpret_cast<const uint4*>(static_cast<const Tout*>(p.o) + off);
#pragma unroll
      for (int j = 0; j < NR; ++j) ou[i][j] = __ldcg(op + j);
      zu[i] = __ldg(reinterpret_cast<const uint4*>(static_cast<const bf16*>(p.z) + off));
    }
  }
#pragma unroll
  for (int i = 0; i < NB; ++i) {
    if (r0 + RS * i < len) {                           // (the same for the 16 lanes of a row)
      float x[8], z[8];
      unpack8(ou[i], x);
      const uint4 zz[1] = {zu[i]};
      unpack8(zz, z);
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
#pragma unroll
      for (int m = 8; m > 0; m >>= 1) ss += __shfl_xor_sync(half, ss, m);
      const float inv = rsqrtf(ss * (1.0f / DV) + p.norm_eps);
      float y[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) y[e] = x[e] * inv * w[e] * silu_out<Tout>(z[e]);
      store8(static_cast<Tout*>(p.o) + ((size_t)(c0 + r0 + RS * i) * p.Nv + h) * DV + 8 * l, y);
    }
  }
}

// The scan of one (sequence s, value head h) by the CTA's warps 0-9 (with the side
// norm of the one-sequence launch, warp 10 publishes the output blocks; other warps
// only join the final barrier).  sm is 1024-aligned
// shared memory of K2 bytes.  With `flags`, every chunk's workspace tiles are
// awaited before they are loaded (the solve runs concurrently in other CTAs).
template <typename Tout, bool NORM>
__device__ void scan_body(uint8_t* sm, const CUtensorMap* tmk, const CUtensorMap* tmv, const ScanSeg& sg,
                          const CUtensorMap* tmz, const ChunkArgs& p, int h, int s, const int* flags) {
  const CUtensorMap* tmo = sg.tmo;
  ScanBars* B = reinterpret_cast<ScanBars*>(sm + K2_BAR);
  volatile int* abort = &B->abort;
  const WaitCtl wc{abort, p.wait_ns};

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int dv = (warp & 3) * 32 + lane;        // this thread's tensor-memory lane

  const int hk = h / (p.Nv / p.Nk);
  int bos, eos;
  if (!seq_bounds(p.cu, p.num_seqs, p.total, s, bos, eos)) {
    if (tid == 0 && h == 0) raise_error(p.err, kDevErrSeqlens);
    return;
  }
  const int slot0 = slot_base(p, s) + sg.c_begin;
  {
    const int seq_bos = bos;
    bos = min(eos, seq_bos + sg.c_begin * CT);
    if (sg.c_end < (eos - seq_bos + CT - 1) / CT) eos = seq_bos + sg.c_end * CT;
  }
  const int n = (eos - bos + CT - 1) / CT;
  const uint8_t* wsb = static_cast<const uint8_t*>(p.workspace);
  int* flags_rw = const_cast<int*>(flags);
  auto ws_tile = [&](int c) {
    const size_t t = sg.ring ? (size_t)(sg.tile0 + c % sg.ring) : (size_t)(slot0 + c);
    return wsb + (t * p.Nv + h) * TILE_T_BYTES;
  };

  // The initial state arrives by four 16 KB bulk copies, issued by thread 0 as soon as their
  // mbarrier is initialised (a thread's 128 dependent-free column loads from global memory
  // took about 10 us at the start of a launch): rows 32q .. 32q + 31 into the second stage
  // buffer (q < 3) and into the head of the second v buffer (q = 3), away from the operand
  // rows zeroed below.  Both are first written by the loads of chunk 1, which wait until the
  // state role has moved the state into tensor memory (s0c).  (The host requires every
  // pointer to be 16-byte aligned, as the copies do.)
  const bool s0_bulk = sg.S0 != nullptr && !sg.identity;
  auto s0_part = [&](int q) -> uint8_t* {
    return sm + (q < 3 ? K2_ST + STAGE_BYTES + (uint32_t)q * 16384u : K2_VT + 32768u);
  };
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&B->stl[i], 1);
      mbar_init(&B->vt[i], 1);
      mbar_init(&B->ready[i], 1);
      mbar_init(&B->ob[i], 1);
      mbar_init(&B->of[i], 1);
      mbar_init(&B->ub[i], 1);
    }
    mbar_init(&B->fg, 1);
    mbar_init(&B->gh, 1);
    mbar_init(&B->zb[0], 1);
    mbar_init(&B->zb[1], 1);
    mbar_init(&B->s0f, 1);
    mbar_init(&B->s0c, 128);
    B->abort = 0;
    B->odone = 0;
    fence_barrier_init();
    if (s0_bulk) {
      mbar_arrive_expect_tx(&B->s0f, 65536);
      for (int q = 0; q < 4; ++q) bulk_load(s0_part(q), sg.S0 + (size_t)q * 32 * DV, 16384, &B->s0f);
    }
    prefetch_tmap(tmk);
    prefetch_tmap(tmv);
    prefetch_tmap(tmo);
  }
  if (warp == 0) tmem_alloc(&B->tslot, 512);
  for (int i = tid * 16; i < 2 * 8192; i += (int)blockDim.x * 16) {   // rows 64-127 of both [T diag(beta); 0] operands
    const uint32_t off = K2_VT + (uint32_t)(i >> 13) * 32768u + 24576u + (uint32_t)(i & 8191);
    *reinterpret_cast<uint4*>(sm + off) = make_uint4(0u, 0u, 0u, 0u);
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = B->tslot;
  const uint32_t lane_base = tbase + ((uint32_t)((warp & 3) * 32) << 16);
  const uint32_t sb = smem_u32(sm);


  // loads of a chunk: v tiles and T diag(beta) (for [U~^T | 0]), and the stage
  // Each buffer's mbarrier expects all of its bytes with the first of its copies, so that
  // the parts may be issued apart: the v tiles (issue_v) and the solve's T diag(beta)
  // (issue_tb); the k tiles (issue_k) and the solve's [-W; Q~] and P tiles (issue_ws).
  auto issue_v = [&](int c) {
    const int t = bos + c * CT;
    const uint32_t vt = K2_VT + (uint32_t)(c & 1) * 32768u;
    uint64_t* bar = &B->vt[c & 1];
    mbar_arrive_expect_tx(bar, 2 * 8192 + 8192);
    tma_load_2d(sm + vt, tmv, bar, h * DV, t);
    tma_load_2d(sm + vt + 8192, tmv, bar, h * DV + 64, t);
  };
  auto issue_tb = [&](int c) {
    const uint32_t vt = K2_VT + (uint32_t)(c & 1) * 32768u;
    bulk_load(sm + vt + 16384, ws_tile(c) + WS_TB, 8192, &B->vt[c & 1]);
  };
  auto issue_vt = [&](int c) {
    issue_v(c);
    issue_tb(c);
    return true;
  };
  auto issue_k = [&](int c) {
    const int t = bos + c * CT;
    const uint32_t st = K2_ST + (uint32_t)(c & 1) * STAGE_BYTES;
    uint64_t* bar = &B->stl[c & 1];
    mbar_arrive_expect_tx(bar, 32768 + 8192 + 512 + 2 * 8192);
    tma_load_2d(sm + st + SG_K, tmk, bar, hk * DK, t);
    tma_load_2d(sm + st + SG_K + 8192, tmk, bar, hk * DK + 64, t);
  };
  auto issue_ws = [&](int c) {
    const uint32_t st = K2_ST + (uint32_t)(c & 1) * STAGE_BYTES;
    uint64_t* bar = &B->stl[c & 1];
    const uint8_t* src = ws_tile(c);
    bulk_load(sm + st, src + WS_QW, 32768, bar);
    bulk_load(sm + st + SG_P, src + WS_P, 8192 + 512, bar);
  };
  auto issue_stage = [&](int c) {
    issue_k(c);
    issue_ws(c);
    return true;
  };
  // With `flags` (the fused launch) one LOADER thread (warp 9) awaits each chunk's
  // tiles and issues all of these loads, so no flag latency sits on PREP or OUT;
  // otherwise PREP issues the v loads and OUT the stage loads.
  const bool self_load = flags == nullptr;
  // O^T += U^T P^T is issued by the output role, right behind the state role's S^T update;
  // with the gated norm in the epilogue (NORM) the output role is the busier one, and the
  // state role issues it after the update completes
  constexpr bool out_issues_o = !NORM;

  if (warp == 9 && !self_load) {
    // ============================== LOADER ==============================
    if (lane == 0) {
      int st_issued = 0, vt_issued = 0, tb_issued = 0, ws_issued = 0;
      bool ok = true;
      for (int c = 0; c < n && ok; ++c) {
        // The v tiles first: their buffer frees (the [U~^T | 0] product of chunk c - 2) a
        // period before the stage buffer does.  The tiles read from q, k and v are issued
        // before the chunk's flag is awaited, the solve's tiles after it (the early chunks'
        // flags are set well after the scan has set up).
        if (!sg.zero_v) {
          // v tiles free (for c = 1: the state's copy in that buffer was read)
          if (c >= 2 || (c == 1 && s0_bulk))
            ok = c >= 2 ? wait_bar(&B->ready[c & 1], ((c - 2) >> 1) & 1, wc) : wait_bar(&B->s0c, 0, wc);
          if (!ok) break;
          issue_v(c);
          vt_issued = c + 1;
        }
        if (c < 2) {             // the stage buffers start free (for c = 1 after the wait above)
          issue_k(c);
          st_issued = c + 1;
        }
        ok = wait_flag(flags + (size_t)(slot0 + c) * p.Nv + h, wc);
        if (!ok) break;
        if (!sg.zero_v) {
          issue_tb(c);
          tb_issued = c + 1;
        }
        if (c >= 2) ok = wait_bar(&B->ob[c & 1], ((c - 2) >> 1) & 1, wc);           // stage free
        if (!ok) break;
        if (sg.release && c >= 2) {
          // chunk c - 2's tiles have been consumed (its stage and v buffers are free again: the
          // copies that read them completed before their products ran), so the solve of a later
          // chunk may overwrite them; a relaxed add keeps the loader from waiting on the fence
          // a release would need
          int* rel = flags_rw + (size_t)(slot0 + c - 2) * p.Nv + h;
          asm volatile("red.relaxed.gpu.global.add.s32 [%0], 1;" ::"l"(rel) : "memory");
        }
        if (c >= 2) issue_k(c);
        issue_ws(c);
        st_issued = ws_issued = c + 1;
      }
      if (!ok) {     // let the copies in flight land (the waits are bounded)
        // a buffer whose q/k/v tiles were issued but whose solve tiles never will be
        if (vt_issued > tb_issued) mbar_complete_tx(&B->vt[tb_issued & 1], 8192);
        if (st_issued > ws_issued) mbar_complete_tx(&B->stl[ws_issued & 1], 32768 + 8192 + 512);
        for (int k = max(st_issued - 2, 0); k < st_issued; ++k) mbar_wait(&B->stl[k & 1], (k >> 1) & 1, WAIT_LIMIT);
        for (int k = max(vt_issued - 2, 0); k < vt_issued; ++k) mbar_wait(&B->vt[k & 1], (k >> 1) & 1, WAIT_LIMIT);
      }
    }
  } else if (warp == 0 && sg.zero_v) {
    // ============================== PREP (no V term) ==============================
    // the [U^T | O^T] product starts its accumulator afresh; PREP only hands each
    // accumulator on once OUT has finished reading it
    if (lane == 0) {
      for (int c = 0; c < n; ++c) {
        const int b = c & 1;
        if (c >= 2 && !wait_bar(&B->of[b], ((c >> 1) - 1) & 1, wc)) break;
        mbar_arrive(&B->ready[b]);
      }
    }
  } else if (warp == 0) {
    // ============================== PREP ==============================
    if (lane == 0) {
      int issued = 0, committed = 0, c = 0;
      if (self_load && n > 0) {
        issue_vt(0);
        issued = 1;
        if (n > 1 && (!s0_bulk || wait_bar(&B->s0c, 0, wc))) {
          issue_vt(1);
          issued = 2;
        }
      }
      bool ok = true;
      for (; c < n; ++c) {
        const int b = c & 1;
        ok = wait_bar(&B->vt[b], (c >> 1) & 1, wc);
        if (ok && c >= 2) ok = wait_bar(&B->of[b], ((c >> 1) - 1) & 1, wc);   // accumulator b free
        if (!ok) break;
        tc_fence_after();
        // [U~^T | 0] = V^T [T diag(beta); 0]^T: A = V tiles read MN-major, B = [T diag(beta); 0]
        const uint32_t vt = K2_VT + (uint32_t)b * 32768u;
        const uint32_t id = idesc_bf16(128, 128, true, false);
        const uint64_t av = sdesc_sw128(sb + vt, 8192, 1024), bt = sdesc_sw128(sb + vt + 16384, 16, 1024);
#pragma unroll
        for (int ks = 0; ks < CT / 16; ++ks)
          mma_bf16(tbase + TM_ACC + b * 128, av + ks * 128, bt + ks * 2, id, ks > 0 ? 1u : 0u);
        mma_commit(&B->ready[b]);
        committed = c + 1;
        if (self_load && c + 2 < n) {
          ok = wait_bar(&B->ready[b], (c >> 1) & 1, wc) && issue_vt(c + 2);   // tiles b consumed
          if (!ok) break;
          issued = c + 3;
        }
      }
      if (!ok) {
        for (int k = c; k < issued; ++k) mbar_wait(&B->vt[k & 1], (k >> 1) & 1, WAIT_LIMIT);
        if (committed > 0) mbar_wait(&B->ready[(committed - 1) & 1], ((committed - 1) >> 1) & 1, WAIT_LIMIT);
      }
    }
  } else if (warp <= 4) {
    // ============================== STATE ==============================
    const bool leader = tid == 32;
    bool s0ok = true;
    if (s0_bulk) {
      // S^T <- the initial state from its shared-memory copy (S0 is [dk][dv]: thread dv
      // reads a column, conflict-free), 32 columns of tensor memory at a time
      s0ok = wait_bar(&B->s0f, 0, wc);
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        const float* src = reinterpret_cast<const float*>(s0_part(q)) + dv;
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = src[i * DV];
        tmem_st32(lane_base + TM_S + q * 32, v);
      }
      tmem_st_wait();
      mbar_arrive(&B->s0c);
    } else {
      // ... or the identity, or zeros
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = sg.identity && q * 32 + i == dv ? 1.f : 0.f;
        tmem_st32(lane_base + TM_S + q * 32, v);
      }
      tmem_st_wait();
    }
    int fg_issued = 0, gh_issued = 0, ob_issued = 0;
    bool fail = false;
    int c = 0;
    // ok carries each thread's waits of the chunk before (its S^T update, and this chunk's
    // stage and [U~^T | 0] product) into the barrier that precedes this chunk's first product
    bool ok = s0ok && (n == 0 || wait_bar2(&B->stl[0], 0, &B->ready[0], 0, wc));
    for (; c < n; ++c) {
      const int b = c & 1;
      const uint32_t st = K2_ST + (uint32_t)b * STAGE_BYTES;
      const float* vec = reinterpret_cast<const float*>(sm + st + SG_VEC);   // dec[0..63], gamma_L
      tc_fence_after();
      // E_S: bf16 copy of S^T (the A operand); only this sits before the product.  (This
      // loop and the rescale below are not unrolled: the scan's roles share one SM's
      // instruction caches, and the smaller loop body measured faster.)
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        float x[32], y[32], pk[32];
        tmem_ld32(lane_base + TM_S + half * 64, x);
        tmem_ld32(lane_base + TM_S + half * 64 + 32, y);
        tmem_ld_wait();
        tmem_ld_fence(x);
        tmem_ld_fence(y);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          pk[i] = __uint_as_float(pack_bf16(x[2 * i], x[2 * i + 1]));
          pk[16 + i] = __uint_as_float(pack_bf16(y[2 * i], y[2 * i + 1]));
        }
        tmem_st32(lane_base + TM_SB + half * 32, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      if (named_sync_or(2, 128, !ok)) { fail = true; break; }
      if (leader) {
        tc_fence_after();
        // [U^T | O^T] += S^T [-W; Q~]^T
        const uint32_t id = idesc_bf16(128, 128, false, false);
        const uint64_t bq = sdesc_sw128(sb + st, 16, 1024);
#pragma unroll
        for (int ks = 0; ks < DK / 16; ++ks)
          mma_bf16_ta(tbase + TM_ACC + b * 128, tbase + TM_SB + ks * 8, bq + (ks >> 2) * 1024 + (ks & 3) * 2, id,
                      (ks > 0 || !sg.zero_v) ? 1u : 0u);
        mma_commit(&B->fg);
        fg_issued = c + 1;
      }
      // S^T <- gamma_L S^T in place while the product runs (it reads the bf16 copy; the
      // S^T update below reads this)
      {
        const float gl = vec[CT];
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          float x[32], y[32];
          tmem_ld32(lane_base + TM_S + half * 64, x);
          tmem_ld32(lane_base + TM_S + half * 64 + 32, y);
          tmem_ld_wait();
          tmem_ld_fence(x);
          tmem_ld_fence(y);
#pragma unroll
          for (int i = 0; i < 32; ++i) { x[i] *= gl; y[i] *= gl; }
          tmem_st32(lane_base + TM_S + half * 64, x);
          tmem_st32(lane_base + TM_S + half * 64 + 32, y);
        }
      }
      // each thread awaits the product itself (and the chunk before's O product, which reads
      // the bf16 U^T rewritten below); a failed wait is carried by the barrier below
      ok = (!out_issues_o || c == 0) ? wait_bar(&B->fg, c & 1, wc)
                                     : wait_bar2(&B->fg, c & 1, &B->ob[(c - 1) & 1], ((c - 1) >> 1) & 1, wc);
      tc_fence_after();
      // E_U: U^T and U^T diag(dec) as bf16 pairs
      {
        float u[64], pu[32], pd[32];
        tm_ld64(lane_base + TM_ACC + b * 128, u);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          pu[i] = __uint_as_float(pack_bf16(u[2 * i], u[2 * i + 1]));
          pd[i] = __uint_as_float(pack_bf16(u[2 * i] * vec[2 * i], u[2 * i + 1] * vec[2 * i + 1]));
        }
        tmem_st32(lane_base + TM_UB, pu);
        tmem_st32(lane_base + TM_UD, pd);
      }
      tmem_st_wait();         // also the rescaled S^T
      tc_fence_before();
      if (named_sync_or(2, 128, !ok)) { fail = true; break; }
      if (leader) {
        tc_fence_after();
        // S^T += (U^T diag(dec)) K: B = K tiles read MN-major
        const uint32_t idh = idesc_bf16(128, 128, false, true);
        const uint64_t bk = sdesc_sw128(sb + st + SG_K, 8192, 1024);
#pragma unroll
        for (int ks = 0; ks < CT / 16; ++ks) mma_bf16_ta(tbase + TM_S, tbase + TM_UD + ks * 8, bk + ks * 128, idh, 1u);
        mma_commit(&B->gh);
        gh_issued = c + 1;
        if (out_issues_o) {
          tc_fence_before();
          mbar_arrive(&B->ub[b]);     // the output role issues O^T += U^T P^T
        }
      }
      // the next chunk's stage and [U~^T | 0] product (normally complete by now) while the
      // S^T update runs, then the update itself
      ok = c + 1 >= n || wait_bar2(&B->stl[b ^ 1], ((c + 1) >> 1) & 1, &B->ready[b ^ 1], ((c + 1) >> 1) & 1, wc);
      ok = ok && wait_bar(&B->gh, c & 1, wc);
      if (!out_issues_o && leader && ok) {
        // O^T += U^T P^T behind the S^T update (the next [U^T | O^T] product's commit covers
        // it before U^T is rewritten)
        tc_fence_after();
        const uint32_t idp = idesc_bf16(128, 64, false, false);
        const uint64_t bp = sdesc_sw128(sb + st + SG_P, 16, 1024);
#pragma unroll
        for (int ks = 0; ks < CT / 16; ++ks)
          mma_bf16_ta(tbase + TM_ACC + b * 128 + 64, tbase + TM_UB + ks * 8, bp + ks * 2, idp, 1u);
        mma_commit(&B->ob[b]);
        ob_issued = c + 1;
      }
    }
    if (!fail) fail = named_sync_or(2, 128, !ok);     // the last chunk's waits
    tc_fence_after();
    if (fail) {
      if (leader) {
        if (s0_bulk) mbar_wait(&B->s0f, 0, WAIT_LIMIT);       // the state's copies have landed
        if (fg_issued > 0) mbar_wait(&B->fg, (fg_issued - 1) & 1, WAIT_LIMIT);
        if (gh_issued > 0) mbar_wait(&B->gh, (gh_issued - 1) & 1, WAIT_LIMIT);
        if (ob_issued > 0) mbar_wait(&B->ob[(ob_issued - 1) & 1], ((ob_issued - 1) >> 1) & 1, WAIT_LIMIT);
      }
    } else if (sg.ST) {
      float* dst = sg.ST + dv;
#pragma unroll
      for (int c0 = 0; c0 < DK; c0 += 32) {
        float v[32];
        tmem_ld32(lane_base + TM_S + c0, v);
        tmem_ld_wait();
        tmem_ld_fence(v);
#pragma unroll
        for (int i = 0; i < 32; ++i) dst[(size_t)(c0 + i) * DV] = v[i];
      }
    }
  } else if (warp == 10 && p.side_norm && flags != nullptr) {
    // ============================== PUBLISHER ==============================
    // Side norm: publish each chunk's o block (a flag per (chunk, head)) once the output role
    // counts its stores as landed.  The gpu-scope fence this needs costs the thread that runs
    // it a memory round trip; here it holds up no other role (on the output role it cost the
    // chain about 30 us per 4096 tokens).  One fence covers every block counted since the last.
    if (lane == 0) {
      int* oflags = flags_rw + (size_t)((p.total + CT - 1) / CT) * p.Nv + 2;
      uint64_t t0 = global_ns();                 // time of the last progress
      int done = 0;
      for (uint32_t i = 0; done < n && i < POLL_CAP; ++i) {
        int avail;
        asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];" : "=r"(avail) : "r"(smem_u32(&B->odone)) : "memory");
        if (avail > done) {
          fence_proxy_async_global();
          asm volatile("fence.acq_rel.gpu;" ::: "memory");
          for (; done < avail; ++done) st_flag(oflags + (size_t)(slot0 + done) * p.Nv + h, 1);
          t0 = global_ns();
          continue;
        }
        // no progress within the wait bound: the scan failed (its own waits report it) or
        // stalled; the norm groups' bounded waits then end the call
        if (*abort || global_ns() - t0 > wc.limit_ns) break;
        __nanosleep(200);
      }
    }
  } else if (warp <= 8) {
    // ============================== OUT ==============================
    const bool leader = tid == 160;
    Tout* o = static_cast<Tout*>(sg.out);
    constexpr bool kBf16Out = sizeof(Tout) == 2;
    const bool rows_bf16 = kBf16Out || sg.out_bf16;
    int issued = 0;
    if (leader && self_load && n > 0) {
      issue_stage(0);
      issued = 1;
      if (n > 1 && (!s0_bulk || wait_bar(&B->s0c, 0, wc))) {
        issue_stage(1);
        issued = 2;
      }
    }
    // Gated RMSNorm in the epilogue (when z is given): y = o / sqrt(mean_dv o^2 + eps) * w * silu(z);
    // the mean over a row is a sum over this warpgroup's 128 lanes.  The z tile of a chunk
    // arrives by TMA in the output buffer its y tile is later written over, one chunk ahead.
    constexpr bool norm = NORM;
    int zissued = 0;
    auto issue_z = [&](int c) {
      uint8_t* os = sm + K2_OS + (uint32_t)(c & 1) * 16384u;
      mbar_arrive_expect_tx(&B->zb[c & 1], 16384);
      tma_load_2d(os, tmz, &B->zb[c & 1], h * DV, bos + c * CT);
      tma_load_2d(os + 8192, tmz, &B->zb[c & 1], h * DV + 64, bos + c * CT);
    };
    if (norm && leader && n > 0) {
      issue_z(0);
      zissued = 1;
    }
    bool fail = false;
    int c = 0, g2_issued = 0;
    if (norm) {     // the weight as fp32 and as bf16 pairs, read by the row phase
      reinterpret_cast<float*>(sm + K2_RED)[dv] = p.norm_w[dv];
      reinterpret_cast<bf16*>(sm + K2_RED + 512)[dv] = __float2bfloat16_rn(p.norm_w[dv]);
      named_sync(3, 128);
    }
    const int ot = tid - 160;                     // thread within OUT
    // Side norm (one-sequence launch with z): each chunk's o block is published with a flag
    // once its stores have landed -- a TMA-stored chunk when the next chunk's store has been
    // issued (one store group may stay in flight), a chunk of plain stores at once -- so that
    // spare solve groups can normalise it in place.
    const bool pub_o = p.side_norm && flags != nullptr;
    auto count_done = [&](int v) {               // (release at CTA scope: the publisher reads it)
      asm volatile("st.release.cta.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&B->odone)), "r"(v) : "memory");
    };
    // The TMA stores of o (and every wait on them) belong to a thread of another warp than
    // the leader, which issues the O products: a leader waiting on a store would hold back
    // the next O product, and with it the next chunk's E_U.
    const bool storer = tid == 192;
    for (; c < n; ++c) {
      const int b = c & 1;
      const int c0 = bos + c * CT, len = min(CT, eos - c0);
      const uint32_t st = K2_ST + (uint32_t)b * STAGE_BYTES;
      // O^T += U^T P^T once the state role has U^T as bf16 and its S^T update issued (the
      // update goes first to the tensor pipe: it is on the chain to the next chunk)
      bool ok = !out_issues_o || wait_bar(&B->ub[b], (c >> 1) & 1, wc);
      if (out_issues_o && leader && ok) {
        tc_fence_after();
        const uint32_t idp = idesc_bf16(128, 64, false, false);
        const uint64_t bp = sdesc_sw128(sb + st + SG_P, 16, 1024);
#pragma unroll
        for (int ks = 0; ks < CT / 16; ++ks)
          mma_bf16_ta(tbase + TM_ACC + b * 128 + 64, tbase + TM_UB + ks * 8, bp + ks * 2, idp, 1u);
        mma_commit(&B->ob[b]);
        g2_issued = c + 1;
      }
      ok = ok && wait_bar(&B->ob[b], (c >> 1) & 1, wc);
      if (named_sync_or(3, 128, !ok)) { fail = true; break; }
      tc_fence_after();
      if (self_load && leader && c + 2 < n && issue_stage(c + 2)) issued = c + 3;   // stage b is free now
      float v[64];
      tm_ld64(lane_base + TM_ACC + b * 128 + 64, v);   // lane dv holds O[0..63][dv]
      const bool use_tma = rows_bf16 && len == CT;
      if (storer) {
        // the stores that read the buffers have left them (with the norm, the other
        // buffer holds this chunk's o rows next)
        if (!norm && use_tma) bulk_wait_read<1>();
      }
      tc_fence_before();
      named_sync(3, 128);
      if (leader) mbar_arrive(&B->of[b]);
      uint8_t* os = sm + K2_OS + (uint32_t)b * 16384u;
      if (norm) {
        // o rows (bf16, the precision of a stored o) into the other output buffer, [r][dv] swizzled
        uint8_t* oscr = sm + K2_OS + (uint32_t)(b ^ 1) * 16384u;
        {
          uint8_t* box = oscr + (dv >> 6) * 8192;
          const uint32_t e = (uint32_t)(dv & 63);
#pragma unroll
          for (int r = 0; r < CT; ++r) {
            const uint32_t off = (uint32_t)r * 128u + ((((e >> 3) ^ (uint32_t)r) & 7u) << 4) + (e & 7u) * 2u;
            *reinterpret_cast<bf16*>(box + off) = __float2bfloat16_rn(p.scale * v[r]);
          }
        }
        const bool zok = wait_bar(&B->zb[b], (c >> 1) & 1, wc);   // z of this chunk in buffer b
        if (named_sync_or(3, 128, !zok)) { fail = true; break; }     // (also: the o rows are written)
        // row phase: thread (r, bx) = (ot % 64, ot / 64) owns the 64 Dv columns of row r in
        // box bx (a quarter-warp spans 8 rows of one box: conflict-free 16-byte accesses);
        // every load is issued before the arithmetic
        const int r = ot & 63, bx = ot >> 6;
        const uint32_t rowoff = (uint32_t)bx * 8192u + (uint32_t)r * 128u;
        const float* wsm = reinterpret_cast<const float*>(sm + K2_RED) + bx * 64;
        const uint8_t* wsm2 = sm + K2_RED + 512 + bx * 128;              // bf16 pairs
        uint4 xu[8], zu[8];
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          const uint32_t off = rowoff + ((((uint32_t)ch ^ (uint32_t)r) & 7u) << 4);
          xu[ch] = *reinterpret_cast<const uint4*>(oscr + off);
          zu[ch] = *reinterpret_cast<const uint4*>(os + off);
        }
        float ssp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          const uint32_t w4[4] = {xu[ch].x, xu[ch].y, xu[ch].z, xu[ch].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w4[i]));
            ssp[i] = fmaf(f.x, f.x, ssp[i]);
            ssp[i] = fmaf(f.y, f.y, ssp[i]);
          }
        }
        float* part = reinterpret_cast<float*>(sm + K2_RED + 768);     // the two halves' sums
        part[bx * 64 + r] = (ssp[0] + ssp[1]) + (ssp[2] + ssp[3]);
        named_sync(3, 128);
        const float inv = rsqrtf((part[r] + part[64 + r]) * (1.0f / DV) + p.norm_eps);
        Tout* yrow = o + ((size_t)(c0 + r) * p.Nv + h) * DV + bx * 64;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          const uint32_t xw[4] = {xu[ch].x, xu[ch].y, xu[ch].z, xu[ch].w};
          const uint32_t zw[4] = {zu[ch].x, zu[ch].y, zu[ch].z, zu[ch].w};
          float y[8];
          if (kBf16Out) {
            const uint4 wu = *reinterpret_cast<const uint4*>(wsm2 + ch * 16);
            const uint32_t wp[4] = {wu.x, wu.y, wu.z, wu.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint32_t g2 = gate_bf16x2(zw[i], wp[i]);
              const float2 gf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&g2));
              const float2 xf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xw[i]));
              y[2 * i] = xf.x * inv * gf.x;
              y[2 * i + 1] = xf.y * inv * gf.y;
            }
          } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 zf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&zw[i]));
              const float2 xf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xw[i]));
              const int j = ch * 8 + 2 * i;
              y[2 * i] = xf.x * inv * wsm[j] * silu_out<Tout>(zf.x);
              y[2 * i + 1] = xf.y * inv * wsm[j + 1] * silu_out<Tout>(zf.y);
            }
          }
          if (r < len) store8(yrow + ch * 8, y);   // 128 contiguous bytes per thread and row
        }
        fence_proxy_async_smem();      // the z tile and the o scratch are next written by the copy engine
        named_sync(3, 128);
        if (leader && c + 1 < n) {      // the next chunk's z goes into the scratch buffer
          issue_z(c + 1);
          zissued = c + 2;
        }
      } else if (use_tma) {
        uint8_t* box = os + (dv >> 6) * 8192;
        const uint32_t e = (uint32_t)(dv & 63);
#pragma unroll
        for (int r = 0; r < CT; ++r) {
          const uint32_t off = (uint32_t)r * 128u + ((((e >> 3) ^ (uint32_t)r) & 7u) << 4) + (e & 7u) * 2u;
          *reinterpret_cast<bf16*>(box + off) = __float2bfloat16_rn(p.scale * v[r]);
        }
        fence_proxy_async_smem();
        named_sync(3, 128);
        if (storer) {
          tma_store_2d(tmo, os, h * DV, c0 - sg.row_off);
          tma_store_2d(tmo, os + 8192, h * DV + 64, c0 - sg.row_off);
          bulk_commit_group();
        }
      } else {
        if (rows_bf16) {          // (bf16 rows with fp32 outputs: the map scan's response rows)
          bf16* dst = static_cast<bf16*>(sg.out) + ((size_t)(c0 - sg.row_off) * p.Nv + h) * DV + dv;
#pragma unroll
          for (int r = 0; r < CT; ++r)
            if (r < len) dst[(size_t)r * p.Nv * DV] = __float2bfloat16_rn(p.scale * v[r]);
        } else {
          // (for the side norm, o is normalised as a bf16 o would be stored, whatever the
          // output type: fp32 rows carry bf16-rounded values)
          Tout* dst = o + ((size_t)(c0 - sg.row_off) * p.Nv + h) * DV + dv;
#pragma unroll
          for (int r = 0; r < CT; ++r) {
            const float x = p.scale * v[r];
            if (r < len) dst[(size_t)r * p.Nv * DV] = from_f32<Tout>(pub_o ? __bfloat162float(__float2bfloat16_rn(x)) : x);
          }
        }
      }
      if (pub_o) {
        if (use_tma) {
          // chunks up to c - 1 have landed once at most this chunk's store group is pending
          if (storer && c >= 1) {
            bulk_wait_group<1>();
            count_done(c);
          }
        } else {
          named_sync(3, 128);                      // every OUT thread's plain stores are issued
          if (storer) {
            bulk_wait_all();
            count_done(c + 1);
          }
        }
      }
    }
    if (storer) {
      bulk_wait_all();
      if (pub_o && !fail) count_done(n);
    }
    if (leader && fail) {
      for (int k = c; k < issued; ++k) mbar_wait(&B->stl[k & 1], (k >> 1) & 1, WAIT_LIMIT);
      for (int k = c; k < zissued; ++k) mbar_wait(&B->zb[k & 1], (k >> 1) & 1, WAIT_LIMIT);
      if (g2_issued > 0) mbar_wait(&B->ob[(g2_issued - 1) & 1], ((g2_issued - 1) >> 1) & 1, WAIT_LIMIT);
    }
  }

  if (*abort && tid == 0) raise_error(p.err, kDevErrTimeout);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, 512);
}

// The whole of sequence s for value head h: the caller's states and output rows.
__device__ __forceinline__ ScanSeg whole_seq(const ChunkArgs& p, int h, int s, const CUtensorMap* tmo) {
  ScanSeg sg;
  const size_t hs = ((size_t)s * p.Nv + h) * DK * DV;
  sg.c_begin = 0;
  sg.c_end = 0x7fffffff;
  sg.S0 = p.S0 ? p.S0 + hs : nullptr;
  sg.identity = false;
  sg.zero_v = false;
  sg.ST = p.ST ? p.ST + hs : nullptr;
  sg.out = p.o;
  sg.out_bf16 = false;
  sg.tmo = tmo;
  sg.row_off = 0;
  sg.tile0 = 0;
  sg.ring = 0;
  sg.release = false;
  return sg;
}

// Packed batches: CTA i scans value head i % Nv of the sequence of length rank i / Nv
// (longest first, ties by index): CTAs start in index order, so the long chains start
// first and the short ones fill in behind them.
template <typename Tout, bool NORM>
__global__ void __launch_bounds__(NT2, 1)
chunk_scan_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                  const __grid_constant__ CUtensorMap tmo, const __grid_constant__ CUtensorMap tmz, ChunkArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = tc::smem_aligned<1024>(smem_raw);
  const int h = blockIdx.x % p.Nv, rank = blockIdx.x / p.Nv;
  volatile int* pick = reinterpret_cast<volatile int*>(sm + K2_BAR + 248);   // before the barriers' set-up
  if (threadIdx.x == 0) *pick = rank;                // (equal lengths: the identity)
  __syncthreads();
  if (p.cu != nullptr) {
    auto len = [&](int q) {
      const int a = __ldg(p.cu + q), b = __ldg(p.cu + q + 1);
      return b > a ? b - a : 0;
    };
    for (int q = threadIdx.x; q < p.num_seqs; q += blockDim.x) {
      const int lq = len(q);
      int r = 0;
      for (int o = 0; o < p.num_seqs; ++o) {
        const int lo = len(o);
        r += lo > lq || (lo == lq && o < q);
      }
      if (r == rank) *pick = q;
    }
  }
  __syncthreads();
  const int s = *pick;
  __syncthreads();
  const ScanSeg sg = whole_seq(p, h, s, &tmo);
  scan_body<Tout, NORM>(sm, &tmk, &tmv, sg, &tmz, p, h, s, nullptr);
}

// ---------------------------------------------------------------------------
// Solve and scan in one cooperative launch, for a single sequence: the first
// `nscan` CTAs run the scan of one value head each; every other CTA runs up to
// three independent 128-thread solve groups (own shared memory slice, 128
// tensor-memory columns, named barrier) that claim (chunk slot, value head)
// items in chunk order and publish a ready flag per item.  Groups on one SM
// slow each other down (an item takes about 2.5x as long with three as with
// one), so `ngroups` of them claim items: enough for the solve to stay ahead
// of the scans, and no more.  With z (the gated norm), the third group of every
// solve CTA normalises the published output blocks instead (the side norm).  A
// scan CTA awaits a chunk's flag before loading its tiles, so the solve of later
// chunks overlaps the scan of earlier ones.  All CTAs are resident at once
// (cooperative launch with one CTA per SM), so these waits always end; each is
// bounded anyway.
// ---------------------------------------------------------------------------
constexpr int NT3 = 384;
constexpr uint32_t S1_GROUP = (S1_BAR + 64 + 1023) & ~1023u;     // one solve group's shared memory
constexpr uint32_t K3_SMEM = (3 * S1_GROUP + 1024) > K2_SMEM ? (3 * S1_GROUP + 1024) : K2_SMEM;
static_assert(K3_SMEM <= 232448, "shared memory budget");

// A sequence split in two segments (nseg = 2): chunks [0, m) and [m, n).  Scratch in
// the workspace: the first segment's final state S_mid, the second's final state from
// zero Bst and its transition map Phi ([Nv][Dk][Dv] fp32 each), and the map scan's
// response rows R (bf16 [tokens - 64 m, Nv, Dk]).
struct SplitArgs {
  int nseg, m, n;
  int ring;               // tile positions per segment and head
  float* S_mid;
  float* Bst;
  float* Phi;
  bf16* R;
};

// Solve item k of the one-sequence launch -> (chunk, value head).  Split in two
// segments, the chunks of both are interleaved (chunk c of the first segment, then
// chunk m + c of the second), so that both segments' scans get their tiles in order.
__device__ __forceinline__ void item_chunk(const SplitArgs& sp, int Nv, int k, int& c, int& h) {
  if (sp.nseg == 1) {
    c = k / Nv;
    h = k % Nv;
    return;
  }
  const int n1 = sp.n - sp.m;                 // chunks of the second segment (<= m)
  const int inter = 2 * n1 * Nv;
  if (k < inter) {
    const int pr = k / (2 * Nv), seg = (k / Nv) & 1;
    h = k % Nv;
    c = seg ? sp.m + pr : pr;
  } else {
    const int k2 = k - inter;
    c = n1 + k2 / Nv;
    h = k2 % Nv;
  }
}

template <typename Tout, bool NORM>
__global__ void __launch_bounds__(NT3, 1)
chunk_fused_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmo,
                   const __grid_constant__ CUtensorMap tmz, const __grid_constant__ CUtensorMap tmr, ChunkArgs p,
                   SplitArgs sp, int nscan, int nitems, int* flags, int ngroups) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = tc::smem_aligned<1024>(smem_raw);
  // The solve CTAs' code comes first in the kernel: code near a kernel's entry runs at full
  // speed on its first pass, code further in is fetched on demand at its first pass (on a
  // GB300 about 14 us per 32 KB with a cold L2), and each solve SM's first item (the early
  // chunks every scan waits for) would pay that.  The scans meanwhile set up, load their
  // initial state and wait for chunk 0.
  if ((int)blockIdx.x >= nscan) {
    const int g = threadIdx.x >> 7, tid = threadIdx.x & 127;
    uint8_t* gsm = sm + g * S1_GROUP;
    uint64_t* bar = reinterpret_cast<uint64_t*>(gsm + S1_BAR);
    volatile int* item_slot = reinterpret_cast<volatile int*>(gsm + S1_BAR + 32);   // two slots
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + S1_BAR + 16);        // in group 0's slice
    const uint32_t barid = 1 + g;
    if (tid == 0) {
      mbar_init(bar, 1);
      fence_barrier_init();
    }
    if (threadIdx.x < 32) tmem_alloc(tslot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot + 128u * (uint32_t)g;
    int* counter = flags + nitems;
    uint32_t ph = 0;
    if (g < ngroups) {
      // Items are claimed two ahead: the next item's gate values and tiles load under the
      // current one, and the claim of the one after (a global atomic) is in flight meanwhile.
      // The first two items of every group are fixed: group i (numbered group-major over the
      // CTAs, so that consecutive items go to different SMs) takes items i and G + i, G the
      // number of groups; the counter hands out the items after 2G.  (With two atomic claims
      // per group at the start, an item of an early chunk could become some group's second
      // item and wait for its first.)
      const int nsolve = (int)gridDim.x - nscan;
      const int G = ngroups * nsolve;
      if (tid == 0) {
        const int gi = g * nsolve + ((int)blockIdx.x - nscan);
        item_slot[0] = gi;
        item_slot[1] = G + gi;
      }
      named_sync(barid, 128);
      int item = item_slot[0], next = item_slot[1];
      SolveAhead ahead{false, false, 0.f, -1, 0, 0};
      int par = 0;
      while (item < nitems) {
        const int after = tid == 0 && next < nitems ? 2 * G + claim_item(counter) : nitems;   // read after the item
        int c, h, nc = -1, nh = 0;
        item_chunk(sp, p.Nv, item, c, h);
        if (next < nitems) item_chunk(sp, p.Nv, next, nc, nh);
        // the chunk's ring position, and the chunk that used it before (same segment)
        const int seg = sp.nseg == 2 && c >= sp.m ? 1 : 0, cl = c - seg * sp.m;
        const int* rel = cl >= sp.ring ? flags + (size_t)(c - sp.ring) * p.Nv + h : nullptr;
        const bool ok = solve_item(gsm, tid, barid, bar, ph, tbase, &tmq, &tmk, p, c, h, ahead, nc, nh,
                                   (size_t)(seg * sp.ring + cl % sp.ring), rel, seg ? 3 : 2);
        if (tid == 0) {
          st_flag(flags + (size_t)c * p.Nv + h, ok ? 1 : -1);   // tiles visible (see solve_item)
          item_slot[par] = after;
        }
        if (!ok) break;
        named_sync(barid, 128);
        item = next;
        next = item_slot[par];
        par ^= 1;
      }
    } else if (p.side_norm && g == 2) {
      // The side norm: the third group of every solve CTA applies the gated RMSNorm to the
      // output blocks in chunk order, each once the scan has published it (its o rows sit in
      // the output buffer), claiming blocks from a counter of their own.  A block that is not
      // published within the wait bound (a failed scan) ends the group with the device error.
      int* ncount = flags + nitems + 1;
      const int* oflags = flags + nitems + 2;
      float w[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) w[i] = p.norm_w[8 * (tid & 15) + i];
      for (;;) {
        if (tid == 0) {
          int it = atomicAdd(ncount, 1);
          if (it < nitems && !wait_count(oflags + it, 1, p.wait_ns)) {
            raise_error(p.err, kDevErrTimeout);
            it = -1;
          }
          item_slot[0] = it;
        }
        named_sync(barid, 128);
        const int it = item_slot[0];
        named_sync(barid, 128);              // (the slot is written again next round)
        if (it < 0 || it >= nitems) break;
        const int c0 = (it / p.Nv) * CT;
        norm_rows<Tout, 128, 8>(p, c0, min(CT, p.total - c0), it % p.Nv, tid, w);
      }
    }
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x < 32) tmem_dealloc(*tslot, 512);
    return;
  }
  const int role = (int)blockIdx.x / p.Nv, h = (int)blockIdx.x % p.Nv;
  ScanSeg sg = whole_seq(p, h, 0, &tmo);
  sg.ring = sp.ring;
  sg.tile0 = role == 0 ? 0 : sp.ring;            // the second segment's ring follows the first's
  sg.release = true;
  if (sp.nseg == 2) {
    const size_t hs = (size_t)h * DK * DV;
    if (role == 0) {                       // first segment: the caller's initial state
      sg.c_end = sp.m;
      sg.ST = sp.S_mid + hs;
    } else if (role == 1) {                // second segment from a zero state
      sg.c_begin = sp.m;
      sg.S0 = nullptr;
      sg.ST = sp.Bst + hs;
    } else {                               // second segment's transition map
      sg.c_begin = sp.m;
      sg.S0 = nullptr;
      sg.identity = true;
      sg.zero_v = true;
      sg.ST = sp.Phi + hs;
      sg.out = sp.R;
      sg.out_bf16 = true;
      sg.tmo = &tmr;
      sg.row_off = sp.m * CT;
    }
  }
  scan_body<Tout, NORM>(sm, &tmk, &tmv, sg, &tmz, p, h, 0, flags);
}

// ---------------------------------------------------------------------------
// kernel 4: the fix-up of a sequence split in two segments.  With S_mid the state
// after the first segment (the state the second segment is entered with):
//   o[t] += R[t] S_mid   for the second segment's tokens (R: the map scan's rows);
//   S_T   = Bst + Phi S_mid.
// Output CTAs (the first nout): one value head and a run of 128-token blocks.  Per
// block D = R_blk S_mid on the tensor core (M = 128 tokens, N = Dv, K = Dk): R by TMA
// (K-major, two buffers), S_mid converted once to bf16 in shared memory (MN-major);
// thread t adds row t of D to its output row.  State CTAs: 16 rows of S_T of one
// head each, in fp32 on CUDA cores.
// ---------------------------------------------------------------------------
constexpr int NT4 = 128;
constexpr uint32_t K4_S = 0;                   // S_mid as bf16: two N blocks of 128 K rows x 128 B
constexpr uint32_t K4_R = 32768;               // 2 x R block: two K chunks x 128 rows x 128 B
constexpr uint32_t K4_BAR = K4_R + 2 * 32768;
constexpr uint32_t K4_SMEM = K4_BAR + 64 + 1024;

struct FixArgs {
  const float* S_mid;
  const float* Bst;
  const float* Phi;
  float* ST;              // [Nv][Dk][Dv], or null
  void* o;                // [T, Nv, Dv]
  int t1;                 // first token of the second segment
  int T, Nv;
  int nblk;               // 128-token blocks of the second segment
  int bpc;                // blocks per output CTA
  int cph;                // output CTAs per head
  int* err;
};

template <typename Tout>
__global__ void __launch_bounds__(NT4)
chunk_fixup_kernel(const __grid_constant__ CUtensorMap tmr, FixArgs f) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = tc::smem_aligned<1024>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int nout = f.cph * f.Nv;
  if ((int)blockIdx.x >= nout) {
    // ---- S_T = Bst + Phi S_mid: thread (row i, 16 columns from c0)
    if (f.ST == nullptr) return;
    const int id = blockIdx.x - nout;
    const int h = id >> 3, i = (id & 7) * 16 + (tid >> 3), c0 = (tid & 7) * 16;
    const size_t hs = (size_t)h * DK * DV;
    float acc[16];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 b4 = __ldg(reinterpret_cast<const float4*>(f.Bst + hs + (size_t)i * DV + c0) + q);
      acc[4 * q] = b4.x; acc[4 * q + 1] = b4.y; acc[4 * q + 2] = b4.z; acc[4 * q + 3] = b4.w;
    }
    const float* phi = f.Phi + hs + (size_t)i * DK;
#pragma unroll 4
    for (int j = 0; j < DK; ++j) {
      const float a = __ldg(phi + j);
      const float4* srow = reinterpret_cast<const float4*>(f.S_mid + hs + (size_t)j * DV + c0);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 s4 = __ldg(srow + q);
        acc[4 * q] = fmaf(a, s4.x, acc[4 * q]);
        acc[4 * q + 1] = fmaf(a, s4.y, acc[4 * q + 1]);
        acc[4 * q + 2] = fmaf(a, s4.z, acc[4 * q + 2]);
        acc[4 * q + 3] = fmaf(a, s4.w, acc[4 * q + 3]);
      }
    }
    float4* dst = reinterpret_cast<float4*>(f.ST + hs + (size_t)i * DV + c0);
#pragma unroll
    for (int q = 0; q < 4; ++q) dst[q] = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
    return;
  }
  // ---- o[t] += R[t] S_mid over blocks [b0, b1) of head h
  const int h = blockIdx.x / f.cph;
  const int b0 = (blockIdx.x % f.cph) * f.bpc, b1 = min(f.nblk, b0 + f.bpc);
  uint64_t* rbar = reinterpret_cast<uint64_t*>(sm + K4_BAR);      // [0], [1]: R buffers landed
  uint64_t* mbar = rbar + 2;                                        // product complete
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + K4_BAR + 32);
  if (tid == 0) {
    mbar_init(&rbar[0], 1);
    mbar_init(&rbar[1], 1);
    mbar_init(mbar, 1);
    fence_barrier_init();
    prefetch_tmap(&tmr);
  }
  if (warp == 0) tmem_alloc(tslot, 128);
  {   // S_mid of head h as the MN-major B operand: K row j = tid, N blocks of 64 columns
    const float* src = f.S_mid + (size_t)h * DK * DV + (size_t)tid * DV;
#pragma unroll
    for (int nb = 0; nb < 2; ++nb) {
      float v[64];
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const float4 x = __ldg(reinterpret_cast<const float4*>(src + nb * 64) + q);
        v[4 * q] = x.x; v[4 * q + 1] = x.y; v[4 * q + 2] = x.z; v[4 * q + 3] = x.w;
      }
      st_row64(sm, K4_S + nb * 16384, tid, v);
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  const uint32_t lane_base = tbase + ((uint32_t)(warp * 32) << 16);
  const uint32_t sb = smem_u32(sm);
  auto load_r = [&](int blk, int buf) {
    uint8_t* dst = sm + K4_R + (uint32_t)buf * 32768u;
    mbar_arrive_expect_tx(&rbar[buf], 32768);
#pragma unroll
    for (int kc = 0; kc < 2; ++kc)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf)
        tma_load_2d(dst + kc * 16384 + hf * 8192, &tmr, &rbar[buf], h * DK + kc * 64, blk * 128 + hf * 64);
  };
  // thread 0 tracks the R loads issued and landed and the products issued, so that a
  // failed wait still lets everything in flight land before the CTA exits
  int issued = 0, landed = 0, mma_issued = 0;
  if (tid == 0 && b0 < b1) {
    load_r(b0, 0);
    issued = 1;
  }
  bool ok = true;
  for (int b = b0; b < b1; ++b) {
    const int it = b - b0, buf = it & 1;
    bool good = true;
    if (tid == 0) {
      // the other buffer's product completed before the last epilogue: it is free
      if (b + 1 < b1) {
        load_r(b + 1, buf ^ 1);
        issued = it + 2;
      }
      good = mbar_wait(&rbar[buf], (it >> 1) & 1, WAIT_LIMIT);
      if (good) {
        landed = it + 1;
        tc_fence_after();
        const uint32_t id = idesc_bf16(128, 128, false, true);
        const uint64_t a = sdesc_sw128(sb + K4_R + (uint32_t)buf * 32768u, 16, 1024);
        const uint64_t bs = sdesc_sw128(sb + K4_S, 16384, 1024);
#pragma unroll
        for (int ks = 0; ks < DK / 16; ++ks)
          mma_bf16(tbase, a + (((ks >> 2) * 16384 + (ks & 3) * 32) >> 4), bs + ks * 128, id, ks > 0 ? 1u : 0u);
        mma_commit(mbar);
        mma_issued = it + 1;
      }
    }
    if (__syncthreads_or(!good)) { ok = false; break; }
    good = mbar_wait(mbar, it & 1, WAIT_LIMIT);
    if (__syncthreads_or(!good)) { ok = false; break; }
    tc_fence_after();
    const int t = f.t1 + b * 128 + tid;
    float d[4][32];
#pragma unroll
    for (int q = 0; q < 4; ++q) tmem_ld32(lane_base + q * 32, d[q]);
    tmem_ld_wait();
#pragma unroll
    for (int q = 0; q < 4; ++q) tmem_ld_fence(d[q]);
    if (t < f.T) {
      Tout* orow = static_cast<Tout*>(f.o) + ((size_t)t * f.Nv + h) * DV;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          float x[8];
          load8(orow + q * 32 + e, x);
#pragma unroll
          for (int u = 0; u < 8; ++u) x[u] += d[q][e + u];
          store8(orow + q * 32 + e, x);
        }
      }
    }
    tc_fence_before();
    __syncthreads();          // D is read out before the next product overwrites it
    tc_fence_after();
  }
  if (!ok && tid == 0) {
    raise_error(f.err, kDevErrTimeout);
    for (int k = landed; k < issued; ++k) mbar_wait(&rbar[k & 1], (k >> 1) & 1, WAIT_LIMIT);
    if (mma_issued > 0) mbar_wait(mbar, (mma_issued - 1) & 1, WAIT_LIMIT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, 128);
}

// ---- host: tensor maps and launch
// 2-D bf16 map over a token-major [rows, cols] matrix with a 64 x 64 box, 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* base, int rows, int cols) {
  return make_tmap_2d(map, base, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rows, cols, 64, 64,
                      CU_TENSOR_MAP_SWIZZLE_128B);
}

template <typename Tout>
cudaError_t launch_scan(const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mo, const CUtensorMap& mz,
                        const ChunkArgs& p, cudaStream_t s) {
  const auto fn = p.z != nullptr ? chunk_scan_kernel<Tout, true> : chunk_scan_kernel<Tout, false>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)K2_SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid(p.Nv * p.num_seqs);
  fn<<<grid, NT2, K2_SMEM, s>>>(mk, mv, mo, mz, p);
  return cudaGetLastError();
}

}  // namespace

bool chunk_tc_supported(const ChunkArgs& p) {
  return p.Dk == DK && p.Dv == DV && p.in_bf16 && tmap_encoder() != nullptr;
}

namespace {
// Per device: can one fused CTA stay resident on every SM (cooperative launch)?
struct FusedDevice {
  bool init = false;
  bool ok = false;
  int sms = 0;
};
std::mutex g_fused_mu;
FusedDevice g_fused[64];

// [bf16 out, fp32 out] x [plain, gated norm]
std::array<const void*, 4> fused_kernels() {
  return {reinterpret_cast<const void*>(chunk_fused_kernel<bf16, false>),
          reinterpret_cast<const void*>(chunk_fused_kernel<bf16, true>),
          reinterpret_cast<const void*>(chunk_fused_kernel<float, false>),
          reinterpret_cast<const void*>(chunk_fused_kernel<float, true>)};
}

bool fused_device(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lock(g_fused_mu);
  FusedDevice& f = g_fused[dev];
  if (!f.init) {
    f.init = true;
    int coop = 0, n = 0;
    bool ok = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) == cudaSuccess && coop &&
              cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess;
    for (const void* fn : fused_kernels()) {
      int nb = 0;
      ok = ok && cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)K3_SMEM) == cudaSuccess &&
           cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fn, NT3, K3_SMEM) == cudaSuccess && nb >= 1;
    }
    ok = ok &&
         cudaFuncSetAttribute(reinterpret_cast<const void*>(chunk_fixup_kernel<bf16>),
                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)K4_SMEM) == cudaSuccess &&
         cudaFuncSetAttribute(reinterpret_cast<const void*>(chunk_fixup_kernel<float>),
                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)K4_SMEM) == cudaSuccess;
    if (ok) {
      f.ok = true;
      f.sms = n;
    }
    cudaGetLastError();   // a refused query leaves no sticky error behind
  }
  *sms = f.sms;
  return f.ok;
}
}  // namespace

// ---- workspace plan
// One sequence on a device that holds the cooperative launch: the solve tiles go
// through a ring of kRing positions per segment and head (a solve item waits until
// the chunk that last used its position has been released by every scan that reads
// it), then one flag per (chunk, value head) -- 1 once the tiles are out, plus one per
// consumer that released them -- and the solve's item counter; then, for a sequence
// split in two segments (kSplitMinChunks chunks or more, and the SMs to hold the extra
// scans), the split's scratch: S_mid, Bst, Phi and the response rows R.  The size does
// not grow with the sequence beyond the flags (4 bytes per chunk and head) and R.
// Packed batches: the tiles of every (chunk slot, value head) and the item counter.
namespace {
constexpr int kSplitMinChunks = 32;
constexpr int kRing = 16;

struct ChunkPlan {
  bool fused;               // the one-sequence cooperative launch
  int nseg, n, m;           // segments; chunks; first chunk of the second segment (n: none)
  int ring;                 // tile positions per segment (0: one per chunk slot)
  size_t tiles, nflags;
  size_t flags_off, split_off, split_bytes, bytes;
};

ChunkPlan plan_chunk(int num_seqs, int total, int Nv, bool fused, bool split_ok) {
  ChunkPlan L{};
  L.n = (total + CT - 1) / CT;
  L.fused = fused && num_seqs == 1;
  if (L.fused) {
    L.nseg = split_ok && L.n >= kSplitMinChunks ? 2 : 1;
    L.m = L.nseg == 2 ? (L.n + 1) / 2 : L.n;
    L.ring = std::max(1, std::min(kRing, L.m));          // the first segment is the longer one
    L.tiles = (size_t)L.nseg * L.ring * Nv;
    // per (chunk, head): the ready / release count; the item counter; the side norm's block
    // counter; per (chunk, head): the side norm's o-ready flag
    L.nflags = 2 * (size_t)L.n * Nv + 2;
  } else {
    L.nseg = 1;
    L.m = L.n;
    L.ring = 0;
    L.tiles = ((size_t)(total / CT) + (size_t)num_seqs) * Nv;
    L.nflags = 1;
  }
  L.flags_off = L.tiles * TILE_T_BYTES;
  L.split_off = L.flags_off + (L.nflags * sizeof(int) + 255) / 256 * 256;
  if (L.nseg == 2) {
    const size_t st = (size_t)Nv * DK * DV * sizeof(float);
    L.split_bytes = 3 * st + ((size_t)(total - L.m * CT) * Nv * DV * sizeof(bf16) + 255) / 256 * 256;
  }
  L.bytes = L.split_off + L.split_bytes;
  return L;
}

// The plan a call takes on the current device.  A sequence is split when the SMs hold
// three scans per head and at least two solve CTAs per head beside them (the two
// segments' scans take twice the solve's output per period; with fewer solve SMs the
// split runs slower than one chain: 258 vs 151 us at 32 heads, T = 4096, and 5.1 vs
// 3.1 ms at T = 131072, on 152 SMs), and the output is the plain o (a gated norm applied
// to the blocks as they are scanned cannot be corrected afterwards).
ChunkPlan device_plan(int num_seqs, int total, int Nv, bool allow_split, int* sms_out) {
  int sms = 0;
  const bool fused = num_seqs == 1 && fused_device(&sms) && sms > Nv;
  if (sms_out) *sms_out = sms;
  return plan_chunk(num_seqs, total, Nv, fused, allow_split && sms >= 5 * Nv);
}
}  // namespace

size_t chunk_tc_workspace_bytes(int num_seqs, int total, int Nv, bool allow_split) {
  return device_plan(num_seqs, total, Nv, allow_split, nullptr).bytes;
}

cudaError_t launch_chunk_tc(const ChunkArgs& args, cudaStream_t s) {
  ChunkArgs p = args;
  if (p.wait_ns == 0) p.wait_ns = kDefaultWaitNs;
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
  CUtensorMap mz = mk;                                 // z tiles of the fused gated norm
  if (p.z != nullptr && !make_map(&mz, p.z, p.total, p.Nv * DV)) return cudaErrorInvalidValue;
  const int slots = p.total / CT + p.num_seqs;
  int sms = 0;
  const ChunkPlan L = device_plan(p.num_seqs, p.total, p.Nv, !p.no_split && p.z == nullptr, &sms);
  if (L.fused) {
    // one sequence: solve and scan overlap in one cooperative launch
    uint8_t* ws = static_cast<uint8_t*>(p.workspace);
    int nitems = L.n * p.Nv;
    int* flags = reinterpret_cast<int*>(ws + L.flags_off);
    cudaError_t e = cudaMemsetAsync(flags, 0, L.nflags * sizeof(int), s);
    if (e != cudaSuccess) return e;
    CUtensorMap mo = mk;                               // fp32 rows are stored directly
    if (p.out_bf16 && !make_map(&mo, p.o, p.total, p.Nv * DV)) return cudaErrorInvalidValue;
    SplitArgs sp{1, L.n, L.n, L.ring, nullptr, nullptr, nullptr, nullptr};
    CUtensorMap mr = mk;
    if (L.nseg == 2) {
      const size_t st = (size_t)p.Nv * DK * DV;
      float* scr = reinterpret_cast<float*>(ws + L.split_off);
      sp = SplitArgs{2, L.m, L.n, L.ring, scr, scr + st, scr + 2 * st, reinterpret_cast<bf16*>(scr + 3 * st)};
      if (!make_map(&mr, sp.R, p.total - L.m * CT, p.Nv * DV)) return cudaErrorInvalidValue;
    }
    int nscan = sp.nseg == 2 ? 3 * p.Nv : p.Nv;
    ChunkArgs pc = p;
    // With z, the scan stores o and the third group of every solve CTA applies the norm to
    // each published block in place (the norm in the scan's epilogue would pace the chain)
    pc.side_norm = p.z != nullptr ? 1 : 0;
    // Solve groups per CTA: the scans take Nv items per period (about 1.6 us); one group
    // per SM delivers an item per about 6.5 us, two groups one per about 11 us each, three
    // one per about 16 us each.  Take one group where the solve SMs outnumber the scans'
    // demand that much, else two (at 32 heads on 152 SMs two measured 1-2 % faster than
    // three on long sequences, the same at 4096 tokens: the third group adds little
    // throughput and every item's latency grows).
    const double per_scan = (double)(sms - nscan) / (double)(sp.nseg * p.Nv);
    int ngroups = per_scan >= 5.3 ? 1 : 2;
    if (p.no_solve) ngroups = 0;           // test hook: no flag is ever published
    void* args[] = {&mq, &mk, &mv, &mo, &mz, &mr, &pc, &sp, &nscan, &nitems, &flags, &ngroups};
    const void* fn = fused_kernels()[p.out_bf16 ? 0 : 2];
    e = cudaLaunchCooperativeKernel(fn, dim3(sms), dim3(NT3), args, K3_SMEM, s);
    if (e != cudaSuccess || sp.nseg == 1) return e;
    // the second segment's outputs and the final state from S_mid
    FixArgs f{};
    f.S_mid = sp.S_mid;
    f.Bst = sp.Bst;
    f.Phi = sp.Phi;
    f.ST = p.ST;
    f.o = p.o;
    f.t1 = sp.m * CT;
    f.T = p.total;
    f.Nv = p.Nv;
    f.nblk = (p.total - f.t1 + 127) / 128;
    const int target = 2 * sms;                        // output CTAs: about two per SM
    const int cph = std::max(1, std::min(f.nblk, target / p.Nv));
    f.bpc = (f.nblk + cph - 1) / cph;
    f.cph = (f.nblk + f.bpc - 1) / f.bpc;
    f.err = p.err;
    const int grid = f.cph * p.Nv + (p.ST ? 8 * p.Nv : 0);
    if (p.out_bf16)
      chunk_fixup_kernel<bf16><<<grid, NT4, K4_SMEM, s>>>(mr, f);
    else
      chunk_fixup_kernel<float><<<grid, NT4, K4_SMEM, s>>>(mr, f);
    return cudaGetLastError();
  }
  if (p.no_solve) return cudaErrorNotSupported;     // the test hook needs the one-sequence launch
  cudaError_t e = cudaFuncSetAttribute(chunk_solve_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)S1_SMEM);
  if (e != cudaSuccess) return e;
  // the item counter sits in the workspace's flag area
  const int nitems = slots * p.Nv;
  int* counter = reinterpret_cast<int*>(static_cast<uint8_t*>(p.workspace) + L.flags_off);
  e = cudaMemsetAsync(counter, 0, sizeof(int), s);
  if (e != cudaSuccess) return e;
  const int nsm = num_sms();
  chunk_solve_kernel<<<std::min(nitems, 3 * nsm), 128, S1_SMEM, s>>>(mq, mk, p, nitems, counter);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (!p.out_bf16) return launch_scan<float>(mk, mv, mk, mz, p, s);   // fp32 rows are stored directly
  CUtensorMap mo;
  if (!make_map(&mo, p.o, p.total, p.Nv * DV)) return cudaErrorInvalidValue;
  return launch_scan<bf16>(mk, mv, mo, mz, p, s);
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
