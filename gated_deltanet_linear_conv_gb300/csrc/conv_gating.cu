// Prefill front end of the Gated DeltaNet mixer: depthwise causal conv (K=4)
// with cached left context + SiLU, split into q/k/v heads, L2-norm of q and k,
// q scale, and the gates beta = sigmoid(b), g = -exp(A_log) softplus(a + dt_bias).
// ("Qwen3.5 Dense Model Architecture", section Linear Attention, forward
// listing; "Qwen3.5 Simulation Support Design Document", section 2.2 ops 2-3.)
//
// Memory-bound.  One warp owns a strip of 128 channels (4 per lane) over TB
// consecutive tokens and walks down them with the three previous rows in
// registers and the next PF rows already in flight, so each input row is read
// once from DRAM (plus a 3-row halo per TB tokens) with few registers and many
// resident warps.  Tokens in the first 3 positions of a sequence take their
// left context from the conv state.  A strip never straddles a q/k/v region
// and holds whole heads, so the per-head L2-norm is a shuffle reduction over
// Dk/4 lanes.

#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "tc_util.cuh"
#include "tmap.cuh"

namespace gdn {
namespace {

constexpr int WARPS = 8;
constexpr int TB = 32;      // tokens per warp work item

template <typename T> struct Row4;
template <> struct Row4<bf16> {
  static constexpr int PF = 8;        // rows prefetched ahead
  using R = uint2;
  static __device__ __forceinline__ R load(const bf16* p) { return *reinterpret_cast<const uint2*>(p); }
  static __device__ __forceinline__ R zero() { return make_uint2(0u, 0u); }
  static __device__ __forceinline__ void unpack(R u, float (&f)[4]) {
    float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
  }
};
template <> struct Row4<float> {
  static constexpr int PF = 4;
  using R = float4;
  static __device__ __forceinline__ R load(const float* p) { return *reinterpret_cast<const float4*>(p); }
  static __device__ __forceinline__ R zero() { return make_float4(0.f, 0.f, 0.f, 0.f); }
  static __device__ __forceinline__ void unpack(R u, float (&f)[4]) { f[0] = u.x; f[1] = u.y; f[2] = u.z; f[3] = u.w; }
};

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(WARPS * 32, 2)
conv_gating_kernel(ConvGatingArgs p) {
  using RW = Row4<Tin>;
  constexpr int PF = RW::PF;
  const int lane = threadIdx.x & 31;
  const int warp_global = blockIdx.x * WARPS + (threadIdx.x >> 5);
  const int nstrips = p.C / 128;
  const int ntb = (p.total + TB - 1) / TB;
  if (warp_global >= nstrips * ntb) return;
  const int strip = warp_global % nstrips;
  const int tb = warp_global / nstrips;
  const int t0 = tb * TB;
  const int t_end = min(t0 + TB, p.total);
  const int c0 = strip * 128 + lane * 4;           // first of my 4 channels
  const Tin* x = static_cast<const Tin*>(p.x) + c0;
  const size_t C = (size_t)p.C;

  // the next PF rows go in flight first
  typename RW::R buf[PF];
#pragma unroll
  for (int i = 0; i < PF; ++i) buf[i] = (t0 + i < t_end) ? RW::load(x + (size_t)(t0 + i) * C) : RW::zero();
  // the three rows before the block (a sequence start inside the window is patched below)
  float xm[3][4];
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    const int t = t0 - 3 + j;
    if (t >= 0) RW::unpack(RW::load(x + (size_t)t * C), xm[j]);
    else {
#pragma unroll
      for (int c = 0; c < 4; ++c) xm[j][c] = 0.f;
    }
  }
  float wt[4][4];                                  // [channel][tap]
#pragma unroll
  for (int c = 0; c < 4; ++c) load4(static_cast<const Tin*>(p.w) + (size_t)(c0 + c) * 4, wt[c]);
  float bias[4] = {0.f, 0.f, 0.f, 0.f};
  if (p.bias) load4(static_cast<const Tin*>(p.bias) + c0, bias);

  // tokens of this block in the first 3 positions of their sequence (bit r)
  uint32_t near_start = 0;
  {
    const int seq = find_seq(p.cu, p.num_seqs, p.total, max(t0 - 3, 0));
    for (int s = seq; s < p.num_seqs; ++s) {
      const int st = seq_start(p.cu, p.num_seqs, p.total, s);
      if (st >= t_end) break;
      for (int r = max(st - t0, 0); r < min(st + 3 - t0, TB); ++r) near_start |= 1u << r;
    }
  }

  const int kd = p.Nk * p.Dk;
  const int region = c0 < kd ? 0 : (c0 < 2 * kd ? 1 : 2);   // q, k, v
  const Tin* st_in = static_cast<const Tin*>(p.state_in);
  Tout* dst;
  size_t row_stride;
  if (region < 2) {
    dst = static_cast<Tout*>(region == 0 ? p.q : p.k) + (c0 - region * kd);
    row_stride = (size_t)kd;
  } else {
    dst = static_cast<Tout*>(p.v) + (c0 - 2 * kd);
    row_stride = (size_t)p.Nv * p.Dv;
  }
  const int lanes_per_head = p.Dk / 4;
  const float qs = region == 0 ? p.q_scale : 1.0f;

  const Tin* xnext = x + (size_t)(t0 + PF) * C;     // row t + PF, advanced one row per token
  Tout* const dst0 = dst;
  dst += (size_t)t0 * row_stride;                   // row t
#pragma unroll 1
  for (int tt = 0; tt < TB; tt += PF) {
#pragma unroll
    for (int i = 0; i < PF; ++i) {
      const int r = tt + i;
      const int t = t0 + r;
      float cur[4];
      RW::unpack(buf[i], cur);
      buf[i] = (r + PF < TB && t + PF < t_end) ? RW::load(xnext) : RW::zero();
      xnext += C;
      if (t < t_end) {
        float y[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float acc = bias[c];
          acc = fmaf(wt[c][0], xm[0][c], acc);
          acc = fmaf(wt[c][1], xm[1][c], acc);
          acc = fmaf(wt[c][2], xm[2][c], acc);
          y[c] = silu_fast(fmaf(wt[c][3], cur[c], acc));
        }
        if (region < 2) {
          float ss = y[0] * y[0] + y[1] * y[1] + y[2] * y[2] + y[3] * y[3];
          ss = group_sum(ss, lanes_per_head);
          const float inv = rsqrtf(ss + p.l2_eps) * qs;
#pragma unroll
          for (int c = 0; c < 4; ++c) y[c] *= inv;
        }
        store4(dst, y);
      }
      dst += row_stride;
#pragma unroll
      for (int c = 0; c < 4; ++c) { xm[0][c] = xm[1][c]; xm[1][c] = xm[2][c]; xm[2][c] = cur[c]; }
    }
  }

  // Tokens in the first 3 positions of a sequence were computed above with
  // the previous sequence's rows as left context; redo them with the conv state.
  while (near_start) {
    const int r = __ffs(near_start) - 1;
    near_start &= near_start - 1;
    const int t = t0 + r;
    const int seq = find_seq(p.cu, p.num_seqs, p.total, t);
    const int pos = t - seq_start(p.cu, p.num_seqs, p.total, seq);
    float y[4];
    float cur[4];
    RW::unpack(RW::load(x + (size_t)t * C), cur);
#pragma unroll
    for (int c = 0; c < 4; ++c) y[c] = fmaf(wt[c][3], cur[c], bias[c]);
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      const int si = pos + j;                 // index into [state(3) ; sequence]
      float xv[4];
      if (si < 3) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
          xv[c] = (st_in != nullptr && si >= 0) ? to_f32(st_in[((size_t)seq * C + c0 + c) * 3 + si]) : 0.f;
      } else {
        RW::unpack(RW::load(x + (size_t)(t - 3 + j) * C), xv);
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) y[c] = fmaf(wt[c][j], xv[c], y[c]);
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) y[c] = silu_fast(y[c]);
    if (region < 2) {
      float ss = y[0] * y[0] + y[1] * y[1] + y[2] * y[2] + y[3] * y[3];
      ss = group_sum(ss, lanes_per_head);
      const float inv = rsqrtf(ss + p.l2_eps) * qs;
#pragma unroll
      for (int c = 0; c < 4; ++c) y[c] *= inv;
    }
    store4(dst0 + (size_t)t * row_stride, y);
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

// Tiled variant for bf16 inputs with C a multiple of 1024, q/k regions of whole
// 256-channel strips and Dk 64 or 128.  A persistent CTA walks tiles of [3 + 16
// tokens] x [1024 channels] of mixed_qkv, staged in shared memory by four TMA box
// loads (the rows before the first token, including negative token indices,
// arrive as zeros) together with the block's weights, with the next tile's loads
// in flight while the current one is computed.  The channel block of a CTA's
// tiles rotates from round to round, so that the q and k blocks (with their L2
// norms) are spread over all CTAs.  Warp w walks 256-channel strip w % 4 (8
// channels per lane, 16-byte reads) down tokens 8 (w / 4) .. + 7 of the tile with
// a four-row register ring; the loop is unrolled so the ring never moves.
// Channel pairs go through the packed fp32x2 FMA (each lane holds an even/odd
// channel pair as one float2), which rounds each half as the scalar FMA does.
// Tokens in the first 3 positions of a sequence (but for a first sequence without
// a conv state in, whose zero left context the TMA fill supplies) are recomputed
// with their conv state afterwards.  The gates, which depend on the token and
// head only, are computed by all CTAs while their first tile is in flight.
constexpr int TT = 16;                         // tokens per tile
constexpr int TROWS = TT + 3;
constexpr int RPW = TT / 2;                    // tokens per warp
constexpr uint32_t STRIP_BYTES = TROWS * 512;  // 256 bf16 channels per row
constexpr uint32_t W_OFF = 4 * STRIP_BYTES;    // the block's conv weights [1024][4] bf16
constexpr uint32_t W_BYTES = 1024 * 4 * 2;
constexpr uint32_t B_OFF = W_OFF + W_BYTES;    // its bias [1024] bf16 (when there is one)
constexpr uint32_t B_BYTES = 1024 * 2;
constexpr uint32_t TILE_BYTES = B_OFF + B_BYTES;
static_assert(W_OFF % 16 == 0 && B_OFF % 16 == 0 && TILE_BYTES % 128 == 0, "bulk copy alignment");
constexpr uint32_t TILE_SMEM = 2 * TILE_BYTES + 64 + 128;

__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// SiLU for the tiled path: x sigmoid(x) = h + h tanh(h), h = x / 2, with the
// hardware tanh when the result is rounded to bf16, the exact-division form for
// fp32.  The tanh's relative error (about 2^-11) gives an absolute error of at
// most about 2^-11 |h|: within half a bf16 ulp of the result for x >= -2; for
// more negative x silu is near zero and the error, still far below the bf16
// rounding of O(1) values, is no longer small relative to the result.
// For bf16 outputs the tiled kernel computes the halved pre-activation h directly (its
// weights and bias scaled by 1/2, which is exact), so silu is h + h tanh(h) with no
// multiply before the tanh; for fp32 outputs the pre-activation is the plain one.
template <typename Tout> __device__ __forceinline__ float silu_pre(float v);
template <> __device__ __forceinline__ float silu_pre<bf16>(float h) { return fmaf(h, tanh_approx(h), h); }
template <> __device__ __forceinline__ float silu_pre<float>(float x) { return silu_fast(x); }
template <typename Tout> __device__ __forceinline__ float2 silu_pre2(float2 v);
template <> __device__ __forceinline__ float2 silu_pre2<bf16>(float2 h) {
  return __ffma2_rn(h, make_float2(tanh_approx(h.x), tanh_approx(h.y)), h);
}
template <> __device__ __forceinline__ float2 silu_pre2<float>(float2 x) {
  return make_float2(silu_fast(x.x), silu_fast(x.y));
}
template <typename Tout> constexpr float kPreScale = 1.0f;
template <> constexpr float kPreScale<bf16> = 0.5f;

__device__ __forceinline__ float2 bf2_to_f2(uint32_t w) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
}
// 8 consecutive bf16 channels from shared memory as 4 (even, odd) pairs
__device__ __forceinline__ void lds8x2(const uint8_t* p, float2 (&f)[4]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  f[0] = bf2_to_f2(u.x);
  f[1] = bf2_to_f2(u.y);
  f[2] = bf2_to_f2(u.z);
  f[3] = bf2_to_f2(u.w);
}
template <typename T> __device__ __forceinline__ void store8x2(T* p, const float2 (&y)[4]) {
  const float f[8] = {y[0].x, y[0].y, y[1].x, y[1].y, y[2].x, y[2].y, y[3].x, y[3].y};
  store8(p, f);
}
// L2-normalise (times qs) a head split over LPH lanes of 8 channels (a shuffle tree of
// fixed depth: no loop control between its steps)
template <int LPH>
__device__ __forceinline__ void l2norm8x2(float2 (&y)[4], float eps, float qs) {
  float2 ss2 = __fmul2_rn(y[0], y[0]);
#pragma unroll
  for (int i = 1; i < 4; ++i) ss2 = __ffma2_rn(y[i], y[i], ss2);
  float ss = ss2.x + ss2.y;
#pragma unroll
  for (int off = LPH / 2; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  const float inv = rsqrtf(ss + eps) * qs;
#pragma unroll
  for (int i = 0; i < 4; ++i) y[i] = __fmul2_rn(y[i], make_float2(inv, inv));
}

// Gates (token, head) items first .. n - 1 step `stride`, two per thread with all loads
// issued first.
__device__ __forceinline__ void gates_range(const ConvGatingArgs& p, int64_t first, int64_t stride) {
  const bf16* a = static_cast<const bf16*>(p.a);
  const bf16* b = static_cast<const bf16*>(p.b);
  const int64_t n = (int64_t)p.total * p.Nv;
  for (int64_t i0 = first; i0 < n; i0 += 2 * stride) {
    const int64_t i1 = i0 + stride;
    const bool has1 = i1 < n;
    const float a0 = __bfloat162float(a[i0]), b0 = __bfloat162float(b[i0]);
    const float a1 = has1 ? __bfloat162float(a[i1]) : 0.f, b1 = has1 ? __bfloat162float(b[i1]) : 0.f;
    const int h0 = (int)(i0 % p.Nv);
    p.beta[i0] = sigmoidf_(b0);
    p.g[i0] = -expf(p.A_log[h0]) * softplusf_(a0 + p.dt_bias[h0]);
    if (has1) {
      const int h1 = (int)(i1 % p.Nv);
      p.beta[i1] = sigmoidf_(b1);
      p.g[i1] = -expf(p.A_log[h1]) * softplusf_(a1 + p.dt_bias[h1]);
    }
  }
}

// LPH: lanes per q/k head (Dk / 8); BIAS: whether the conv has a bias.
template <typename Tout, int LPH, bool BIAS>
__global__ void __launch_bounds__(256, 2)
conv_gating_tile_kernel(const __grid_constant__ CUtensorMap tmx, ConvGatingArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = tc::smem_aligned<128>(smem_raw);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + 2 * TILE_BYTES);   // one per buffer
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sid = warp & 3, half = warp >> 2;
  const int nct = p.C / 1024;
  const int ntiles = ((p.total + TT - 1) / TT) * nct;
  const int kd = p.Nk * p.Dk;
  const bf16* st_in = static_cast<const bf16*>(p.state_in);
  // Tile L covers tokens TT (L / nct) .. and channel block (L + L / nct) % nct: over the
  // rounds of a persistent CTA (L advancing by the grid size) the block rotates, so that
  // the q and k blocks (with their L2 norms) are spread over all CTAs.
  auto tile_ct = [&](int tile) { return (tile + tile / nct) % nct; };
  auto issue = [&](int tile, int buf) {
    const int t0 = (tile / nct) * TT, ct = tile_ct(tile);
    tc::mbar_arrive_expect_tx(&bar[buf], W_OFF + W_BYTES + (BIAS ? B_BYTES : 0));
    for (int i = 0; i < 4; ++i)
      tc::tma_load_2d(sm + buf * TILE_BYTES + i * STRIP_BYTES, &tmx, &bar[buf], ct * 1024 + i * 256, t0 - 3);
    // the block's weights (and bias) come with its rows: the block changes from tile to tile
    tc::bulk_load(sm + buf * TILE_BYTES + W_OFF, static_cast<const uint8_t*>(p.w) + (size_t)ct * W_BYTES, W_BYTES,
                  &bar[buf]);
    if (BIAS)
      tc::bulk_load(sm + buf * TILE_BYTES + B_OFF, static_cast<const uint8_t*>(p.bias) + (size_t)ct * B_BYTES,
                    B_BYTES, &bar[buf]);
  };
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar[0], 1);
    tc::mbar_init(&bar[1], 1);
    tc::fence_barrier_init();
    if (blockIdx.x < ntiles) issue(blockIdx.x, 0);
  }
  // Without a state in, the new conv state comes from the staged rows of the tile holding a
  // sequence's last token (with one, a separate pass reads the old state first, so that it may
  // be updated in place).  Empty sequences keep a zero state: written here.
  const bool write_state = p.state_out != nullptr && p.state_in == nullptr;
  if (write_state) {
    for (int sq = blockIdx.x; sq < p.num_seqs; sq += gridDim.x) {
      int bos, eos;
      if (!seq_bounds(p.cu, p.num_seqs, p.total, sq, bos, eos)) {
        if (threadIdx.x == 0) raise_error(p.err, kDevErrSeqlens);
      } else if (bos == eos) {
        bf16* so = static_cast<bf16*>(p.state_out) + (size_t)sq * p.C * 3;
        for (int i = threadIdx.x; i < p.C * 3; i += blockDim.x) so[i] = __float2bfloat16_rn(0.f);
      }
    }
  }
  // The gates, which depend on the token and head only, while the first tile is in flight
  // (their loads are small beside it)
  gates_range(p, (int64_t)blockIdx.x * blockDim.x + threadIdx.x, (int64_t)gridDim.x * blockDim.x);
  __syncthreads();
  float2 wt[4][4], bias[4];                          // [channel pair][tap]
  int k = 0;
  for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++k) {
    const int buf = k & 1;
    const int tt = tile / nct, ct = tile_ct(tile);
    const int t0 = tt * TT, t_end = min(t0 + TT, p.total);
    // the other buffer was released by the barrier that ended the previous tile
    if (threadIdx.x == 0 && tile + (int)gridDim.x < ntiles) issue(tile + gridDim.x, buf ^ 1);
    const int strip0 = ct * 1024 + sid * 256;         // first channel of the warp's strip
    const int c0 = strip0 + lane * 8;
    const int region = strip0 < kd ? 0 : (strip0 < 2 * kd ? 1 : 2);
    const bool ok = tc::mbar_wait(&bar[buf], (uint32_t)(k >> 1) & 1u, 1u << 24);
    if (!__syncthreads_and(ok ? 1 : 0)) {
      if (threadIdx.x == 0) {
        raise_error(p.err, kDevErrTimeout);
        // let the copies in flight land before the CTA's shared memory goes away
        tc::mbar_wait(&bar[buf], (uint32_t)(k >> 1) & 1u, 1u << 24);
        if (tile + (int)gridDim.x < ntiles) tc::mbar_wait(&bar[buf ^ 1], (uint32_t)((k + 1) >> 1) & 1u, 1u << 24);
      }
      return;
    }
    {   // this lane's 8 channels: weights [channel][tap] (64 contiguous bytes) and bias
      const uint8_t* wsm = sm + buf * TILE_BYTES + W_OFF + (uint32_t)(sid * 256 + lane * 8) * 8u;
#pragma unroll
      for (int q = 0; q < 4; ++q) {             // 16 bytes: channels 2q, 2q + 1, four taps each
        const uint4 u = *reinterpret_cast<const uint4*>(wsm + 16 * q);
        const float2 e01 = bf2_to_f2(u.x), e23 = bf2_to_f2(u.y), o01 = bf2_to_f2(u.z), o23 = bf2_to_f2(u.w);
        const float2 k2 = make_float2(kPreScale<Tout>, kPreScale<Tout>);
        wt[q][0] = __fmul2_rn(make_float2(e01.x, o01.x), k2);
        wt[q][1] = __fmul2_rn(make_float2(e01.y, o01.y), k2);
        wt[q][2] = __fmul2_rn(make_float2(e23.x, o23.x), k2);
        wt[q][3] = __fmul2_rn(make_float2(e23.y, o23.y), k2);
      }
      if (BIAS) {
        lds8x2(sm + buf * TILE_BYTES + B_OFF + (uint32_t)(sid * 256 + lane * 8) * 2u, bias);
#pragma unroll
        for (int q = 0; q < 4; ++q) bias[q] = __fmul2_rn(bias[q], make_float2(kPreScale<Tout>, kPreScale<Tout>));
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) bias[q] = make_float2(0.f, 0.f);
      }
    }
    Tout* dst;
    size_t row_stride;
    if (region < 2) {
      dst = static_cast<Tout*>(region == 0 ? p.q : p.k) + (c0 - region * kd);
      row_stride = (size_t)kd;
    } else {
      dst = static_cast<Tout*>(p.v) + (c0 - 2 * kd);
      row_stride = (size_t)p.Nv * p.Dv;
    }
    Tout* const dst0 = dst;
    const float qs = region == 0 ? p.q_scale : 1.0f;
    const int r0 = RPW * half;                        // first token of this warp within the tile
    const uint8_t* rows = sm + buf * TILE_BYTES + sid * STRIP_BYTES + lane * 16 + r0 * 512;
    dst += (size_t)(t0 + r0) * row_stride;
    float2 ring[4][4];
#pragma unroll
    for (int j = 0; j < 3; ++j) lds8x2(rows + j * 512, ring[j]);
    // one output row (the ring index is static once the loop is unrolled)
    auto row_out = [&](int r, Tout* d) {
      float2(&cur)[4] = ring[(r + 3) & 3];
      lds8x2(rows + (r + 3) * 512, cur);
      const float2(&x0)[4] = ring[r & 3];
      const float2(&x1)[4] = ring[(r + 1) & 3];
      const float2(&x2)[4] = ring[(r + 2) & 3];
      float2 y[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float2 acc = BIAS ? __ffma2_rn(wt[q][0], x0[q], bias[q]) : __fmul2_rn(wt[q][0], x0[q]);
        acc = __ffma2_rn(wt[q][1], x1[q], acc);
        acc = __ffma2_rn(wt[q][2], x2[q], acc);
        y[q] = silu_pre2<Tout>(__ffma2_rn(wt[q][3], cur[q], acc));
      }
      if (region < 2) l2norm8x2<LPH>(y, p.l2_eps, qs);
      store8x2(d, y);
    };
    if (t_end - (t0 + r0) >= RPW) {          // every row of this warp is a token
#pragma unroll
      for (int r = 0; r < RPW; ++r) row_out(r, dst + (size_t)r * row_stride);
    } else {
#pragma unroll
      for (int r = 0; r < RPW; ++r) {
        if (t0 + r0 + r < t_end) {
          row_out(r, dst + (size_t)r * row_stride);
        } else {                             // (keeps the ring in step)
          lds8x2(rows + (r + 3) * 512, ring[(r + 3) & 3]);
        }
      }
    }
    // tokens of this warp in the first 3 positions of a sequence: redo with the conv state
    // (zeros without one) in place of the previous sequence's rows; the x rows of the
    // sequence itself are staged in the tile (row t - t0 + 3 holds token t).  A sequence
    // that starts at token 0 with no state in needs nothing: the rows before token 0 were
    // staged as zeros.
    const int ta = t0 + r0, tb = min(t0 + r0 + RPW, t_end);
    if (p.num_seqs > 1 || (ta < 3 && st_in != nullptr)) {
      const uint8_t* srow0 = sm + buf * TILE_BYTES + sid * STRIP_BYTES + lane * 16;
      auto lds8f = [&](int row, float (&f)[8]) {
        float2 pr[4];
        lds8x2(srow0 + row * 512, pr);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          f[2 * i] = pr[i].x;
          f[2 * i + 1] = pr[i].y;
        }
      };
      const int seq0 = find_seq(p.cu, p.num_seqs, p.total, max(ta - 3, 0));
      for (int sq = seq0; sq < p.num_seqs; ++sq) {
        int st, en;
        if (!seq_bounds(p.cu, p.num_seqs, p.total, sq, st, en)) {
          if (lane == 0) raise_error(p.err, kDevErrSeqlens);
          break;
        }
        if (st >= tb) break;
        if (st == 0 && st_in == nullptr) continue;
        for (int t = max(st, ta); t < min(min(st + 3, en), tb); ++t) {     // tokens of sequence sq only
          const int pos = t - st;
          float cur[8], y8[8];
          lds8f(t - t0 + 3, cur);
#pragma unroll
          for (int c = 0; c < 8; ++c)
            y8[c] = fmaf((c & 1) ? wt[c >> 1][3].y : wt[c >> 1][3].x, cur[c], (c & 1) ? bias[c >> 1].y : bias[c >> 1].x);
#pragma unroll
          for (int j = 0; j < 3; ++j) {
            const int si = pos + j;
            float xv[8];
            if (si < 3) {
#pragma unroll
              for (int c = 0; c < 8; ++c)
                xv[c] = st_in != nullptr ? __bfloat162float(st_in[((size_t)sq * p.C + c0 + c) * 3 + si]) : 0.f;
            } else {
              lds8f(t - t0 + j, xv);
            }
#pragma unroll
            for (int c = 0; c < 8; ++c) y8[c] = fmaf((c & 1) ? wt[c >> 1][j].y : wt[c >> 1][j].x, xv[c], y8[c]);
          }
          float2 y[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) y[q] = make_float2(silu_pre<Tout>(y8[2 * q]), silu_pre<Tout>(y8[2 * q + 1]));
          if (region < 2) l2norm8x2<LPH>(y, p.l2_eps, qs);
          store8x2(dst0 + (size_t)t * row_stride, y);
        }
      }
    }
    if (write_state && (p.num_seqs > 1 || t_end == p.total)) {
      // new conv state (no state in: zeros before a sequence's first token) of each non-empty
      // sequence whose last token is in this tile (all lie between the sequences of the
      // tile's first and last tokens), from the staged rows: thread = 4 channels of the 1024
      const int sa = find_seq(p.cu, p.num_seqs, p.total, t0);
      const int sb = find_seq(p.cu, p.num_seqs, p.total, t_end - 1);
      const int ch = threadIdx.x * 4;
      const uint8_t* box = sm + buf * TILE_BYTES + (ch >> 8) * STRIP_BYTES + (ch & 255) * 2;
      for (int sq = sa; sq <= sb; ++sq) {
        int bos, eos;
        if (!seq_bounds(p.cu, p.num_seqs, p.total, sq, bos, eos) || eos == bos || eos <= t0 || eos > t_end) continue;
        bf16* so = static_cast<bf16*>(p.state_out) + ((size_t)sq * p.C + ct * 1024 + ch) * 3;
#pragma unroll
        for (int j = 0; j < 3; ++j) {
          const int t = eos - 3 + j;                 // staged row t - t0 + 3
          const bool in_seq = t >= bos;
#pragma unroll
          for (int c = 0; c < 4; ++c)
            so[c * 3 + j] = in_seq ? *reinterpret_cast<const bf16*>(box + (t - t0 + 3) * 512 + c * 2)
                                   : __float2bfloat16_rn(0.f);
        }
      }
    }
    __syncthreads();     // the tile is read; the next TMA may overwrite it
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
  bool tiled = false;
  const int kd = p.Nk * p.Dk;
  if (std::is_same<Tin, bf16>::value && p.C % 1024 == 0 && kd % 256 == 0 && p.total > 0 &&
      (p.Dk == 64 || p.Dk == 128)) {
    CUtensorMap m;
    if (make_tmap_2d(&m, p.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.total, p.C, 256, TROWS,
                     CU_TENSOR_MAP_SWIZZLE_NONE)) {
      const bool bias = p.bias != nullptr;
      auto fn = p.Dk == 128 ? (bias ? conv_gating_tile_kernel<Tout, 16, true> : conv_gating_tile_kernel<Tout, 16, false>)
                            : (bias ? conv_gating_tile_kernel<Tout, 8, true> : conv_gating_tile_kernel<Tout, 8, false>);
      cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TILE_SMEM);
      if (e != cudaSuccess) return e;
      const int ntiles = ((p.total + TT - 1) / TT) * (p.C / 1024);
      const int blocks = std::min(ntiles, num_sms() * 2);
      fn<<<blocks, 256, TILE_SMEM, s>>>(m, p);
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
      tiled = true;
    }
  }
  if (!tiled) {
    const long long items = (long long)(p.C / 128) * ((p.total + TB - 1) / TB);
    if (items > 0) {
      const int blocks = (int)((items + WARPS - 1) / WARPS);
      conv_gating_kernel<Tin, Tout><<<blocks, WARPS * 32, 0, s>>>(p);
      cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
  }
  if (p.state_out != nullptr && !(tiled && p.state_in == nullptr)) {
    dim3 grid((p.C + 255) / 256, p.num_seqs);
    conv_state_kernel<Tin><<<grid, 256, 0, s>>>(p);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

}  // namespace

// ---------------------------------------------------------------------------
// conv state after every token (the rollback points of a draft + verify step):
// step_states[t] = the last three raw inputs up to and including token t of its
// sequence, oldest first, with the sequence's state in before its first token.
// One thread per (token, channel).
// ---------------------------------------------------------------------------
namespace {
template <typename Tin>
__global__ void conv_state_steps_kernel(ConvGatingArgs p, Tin* steps) {
  const int t = blockIdx.y;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= p.C) return;
  const int s = find_seq(p.cu, p.num_seqs, p.total, t);
  int bos, eos;
  if (!seq_bounds(p.cu, p.num_seqs, p.total, s, bos, eos) || t < bos || t >= eos) {
    if (c == 0) raise_error(p.err, kDevErrSeqlens);
    return;
  }
  const int i = t - bos;
  const Tin* x = static_cast<const Tin*>(p.x);
  const Tin* sin = static_cast<const Tin*>(p.state_in);
  Tin out[3];
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    const int q = i + 1 + j;                  // index into [state in (3) ; the sequence's inputs]
    out[j] = q >= 3 ? x[(size_t)(bos + q - 3) * p.C + c]
                    : (sin ? sin[((size_t)s * p.C + c) * 3 + q] : from_f32<Tin>(0.f));
  }
#pragma unroll
  for (int j = 0; j < 3; ++j) steps[((size_t)t * p.C + c) * 3 + j] = out[j];
}
}  // namespace

cudaError_t launch_conv_state_steps(const ConvGatingArgs& p, void* steps, cudaStream_t s) {
  if (p.total == 0) return cudaSuccess;
  dim3 grid((p.C + 255) / 256, p.total);
  if (p.in_bf16)
    conv_state_steps_kernel<bf16><<<grid, 256, 0, s>>>(p, static_cast<bf16*>(steps));
  else
    conv_state_steps_kernel<float><<<grid, 256, 0, s>>>(p, static_cast<float*>(steps));
  return cudaGetLastError();
}

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
