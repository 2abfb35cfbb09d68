/*
 * gdn.h -- C ABI of the GB300 (sm_103a) Gated DeltaNet token-mixer library.
 *
 * The mixer runs from the concatenated QKV / z / a / b projection outputs of
 * a Qwen3.5-style linear-attention layer to its gated output (the projections
 * themselves are not part of this library).  Sources, by page title and
 * section:
 *   [QDA]  "Qwen3.5 Dense Model Architecture", section "Linear Attention"
 *          (the forward listing) and section "Cache" (conv / recurrent state
 *          shapes).
 *   [RFC]  "Qwen3.5 Simulation Support Design Document", section 2.2 (the
 *          decomposed linear-attention ops), 2.4 (conv body vs conv-state
 *          update), 3.1.3 (state memory), Appendix B (chunk size 64).
 *
 * Conventions shared by every call
 * --------------------------------
 *  - All tensors are device pointers to contiguous, token-major arrays.
 *    Packed sequences are stored back to back; `cu_seqlens` (device, int32,
 *    [num_seqs + 1], cu_seqlens[0] = 0, non-decreasing, last = total_tokens)
 *    gives their bounds.  When `cu_seqlens` is NULL the tokens split into
 *    num_seqs equal sequences of total_tokens / num_seqs.
 *  - The caller owns every buffer.  The library never allocates, never frees
 *    and never synchronises: each call enqueues kernels on `stream` (a
 *    cudaStream_t passed as void*, NULL = legacy default stream) and returns.
 *  - Element types are chosen per argument with gdn_dtype.  Gates (g, beta),
 *    A_log, dt_bias, norm weights and recurrent states are always float32.
 *  - Every pointer must be 16-byte aligned.
 *  - Return value: GDN_OK, or an error code with nothing enqueued.  Argument
 *    errors are detected on the host before any launch.  A launch failure
 *    returns GDN_ERR_CUDA; gdn_last_error_string() describes the last error
 *    of the calling thread.  Inconsistent device-side metadata (a cu_seqlens
 *    that is not monotone or does not end at total_tokens) is detected on the
 *    device: the offending kernel skips the bad sequence and raises a sticky
 *    device error flag, read (and cleared) by gdn_check_device_error().
 *  - On its first use on a device the library looks up (once, with that device
 *    current) the device addresses of its own module variables: the error
 *    flag and the scratch array of gdn_chunk_prefill_static.  Those addresses
 *    belong to the device's primary context, so resetting the device
 *    (cudaDeviceReset) or destroying its primary context after the first call
 *    is not supported: later calls would use stale addresses.
 *
 * Supported sizes: Dk, Dv in {64, 128}; Nv a multiple of Nk; conv kernel 4;
 * chunk 64.  Other sizes return GDN_ERR_UNSUPPORTED.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GDN_OK = 0,
  GDN_ERR_INVALID_ARG = 1,  /* bad pointer, size, alignment or dtype        */
  GDN_ERR_UNSUPPORTED = 2,  /* a head size without a compiled kernel        */
  GDN_ERR_CUDA = 3,         /* a CUDA runtime error while enqueueing         */
  GDN_ERR_DEVICE = 4        /* the device error flag was raised (see above) */
} gdn_status;

typedef enum {
  GDN_BF16 = 0,  /* bfloat16 */
  GDN_F32 = 1    /* float32  */
} gdn_dtype;

/* Problem sizes shared by the calls.
 *   num_seqs      N, number of packed sequences (>= 1)
 *   total_tokens  tokens over all sequences (>= 0)
 *   num_k_heads   Nk, query/key heads;   head_k_dim Dk
 *   num_v_heads   Nv, value heads;       head_v_dim Dv
 * The concatenated projection has C = 2*Nk*Dk + Nv*Dv channels, ordered
 * [q heads | k heads | v heads] ([QDA] split of mixed_qkv).  Value head h
 * reads key head h / (Nv / Nk) (repeat_interleave of the key heads, [QDA]). */
typedef struct {
  int32_t num_seqs;
  int32_t total_tokens;
  int32_t num_k_heads;
  int32_t num_v_heads;
  int32_t head_k_dim;
  int32_t head_v_dim;
} gdn_dims;

/* Library version, (major << 16) | minor. */
int gdn_version(void);

/* Description of the last error returned on the calling thread. */
const char* gdn_last_error_string(void);

/* Synchronises `stream`, then reads and clears the device error flag.
 * Returns GDN_OK, GDN_ERR_DEVICE (flag was set) or GDN_ERR_CUDA. */
int gdn_check_device_error(void* stream);

/* ------------------------------------------------------------------------
 * gdn_conv_gating -- steps a1 + a2 + a3 of a prefill ([QDA] forward listing:
 * causal conv with cached left context, SiLU, split into heads, beta, g, and
 * the q/k L2-norm of [RFC] 2.2 op 3).
 *
 * Per sequence, with xpad = [conv_state_in (K-1 = 3 oldest-first inputs, or
 * zeros) ; x] along time and K = 4:
 *   y[t, c]  = silu( sum_j conv_w[c, j] * xpad[t + j, c] + conv_bias[c] )
 *   q[t, i]  = q_scale * y_q / sqrt(sum(y_q^2) + l2_eps)   per key head i
 *   k[t, i]  =           y_k / sqrt(sum(y_k^2) + l2_eps)   per key head i
 *   v[t, h]  = y_v                                          per value head h
 *   beta     = sigmoid(b);  g = -exp(A_log) * softplus(a + dt_bias)  (fp32)
 * On the tiled bf16 path (see the launches below) with bf16 outputs, silu(x) is
 * evaluated as h + h tanh(h), h = x / 2, with the hardware tanh: its absolute
 * error is at most about 2^-11 |h|, within half a bf16 ulp of the result for
 * x >= -2 (for more negative x the result is near zero and its relative error
 * grows); otherwise silu(x) = x / (1 + e^-x).
 *   conv_state_out[s] = the last 3 entries of xpad (raw inputs, oldest first)
 *
 *   mixed_qkv      [tokens, C]          in_dtype
 *   conv_w         [C, 4]               in_dtype (w[c,3] multiplies token t)
 *   conv_bias      [C] in_dtype, or NULL
 *   conv_state_in  [N, C, 3] in_dtype, or NULL (zero left context)
 *   conv_state_out [N, C, 3] in_dtype, or NULL (not written); may equal
 *                  conv_state_in for an in-place update
 *   a, b           [tokens, Nv]         in_dtype
 *   A_log, dt_bias [Nv]                 float32
 *   q, k           [tokens, Nk, Dk]     out_dtype
 *   v              [tokens, Nv, Dv]     out_dtype
 *   g, beta        [tokens, Nv]         float32
 * One kernel is enqueued for the conv/norm/gating pass.  A second one, the
 * conv-state update, follows when conv_state_out is not NULL and either
 * conv_state_in is not NULL (it reads the old state first, so the update may
 * be in place) or the inputs do not take the tiled bf16 path (C a multiple of
 * 1024, Nk*Dk a multiple of 256); otherwise the first kernel writes the new
 * state from its staged input rows.
 * ------------------------------------------------------------------------ */
int gdn_conv_gating(const gdn_dims* dims, const int32_t* cu_seqlens,
                    const void* mixed_qkv, int in_dtype,
                    const void* conv_w, const void* conv_bias,
                    const void* conv_state_in, void* conv_state_out,
                    const void* a, const void* b,
                    const float* A_log, const float* dt_bias,
                    float q_scale, float l2_eps,
                    void* q, void* k, void* v, int out_dtype,
                    float* g, float* beta, void* stream);

/* ------------------------------------------------------------------------
 * gdn_conv_state_steps -- the conv state after every token: the rollback
 * points of a multi-token (draft + verify) decode step, beside the recurrent
 * states of gdn_recurrent_decode_steps; a caller that accepts the first j + 1
 * tokens of a sequence keeps step_states[bos + j] as its conv state.  With
 * xpad = [conv_state_in (3 oldest-first inputs, or zeros) ; x] of a sequence
 * ([QDA] "Cache": the conv cache keeps the latest raw inputs), token i of it
 * gets step_states[bos + i] = xpad[i + 1 .. i + 3] (oldest first).  The last
 * token's entry equals the conv_state_out of gdn_conv_gating.
 *   mixed_qkv      [tokens, C]          in_dtype
 *   conv_state_in  [N, C, 3] in_dtype, or NULL (zeros); the state the tokens
 *                  follow -- read it before an in-place update of it
 *   step_states    [tokens, C, 3]       in_dtype, written
 * ------------------------------------------------------------------------ */
int gdn_conv_state_steps(const gdn_dims* dims, const int32_t* cu_seqlens, const void* mixed_qkv, int in_dtype,
                         const void* conv_state_in, void* step_states, void* stream);

/* ------------------------------------------------------------------------
 * gdn_gating -- step a3 alone, for callers that already hold q, k, v:
 *   beta[t, h] = sigmoid(b[t, h]);  g[t, h] = -exp(A_log[h]) * softplus(a[t, h] + dt_bias[h])
 *   a, b [rows, Nv] in_dtype; A_log, dt_bias [Nv] float32; g, beta [rows, Nv] float32.
 * ([QDA] forward listing: beta = b.sigmoid(), g in float32.)
 * ------------------------------------------------------------------------ */
int gdn_gating(int64_t rows, int32_t num_v_heads, const void* a, const void* b, int in_dtype,
               const float* A_log, const float* dt_bias, float* g, float* beta, void* stream);

/* ------------------------------------------------------------------------
 * gdn_chunk_prefill -- step a4: the chunked gated delta rule ([RFC] 2.2 op 4,
 * Appendix B: chunk 64, intra-chunk attention + inter-chunk recurrence;
 * [QDA] chunk_gated_delta_rule with initial_state / output_final_state).
 *
 * Computes exactly the recurrence of gdn_recurrent_decode over every token of
 * every sequence, chunk by chunk (chunks restart at each sequence start):
 *   S <- exp(g_t) S;  u = beta_t (v_t - S^T k_t);  S <- S + k_t u^T;
 *   o_t = S^T (scale * q_t),     S in [Dk, Dv] layout, fp32.
 * bf16 q, k, v with Dk = Dv = 128 run on the tensor cores (bf16 products,
 * fp32 accumulation and state); fp32 inputs and 64-wide heads run the fp32
 * CUDA-core kernel of gdn_chunk_prefill_fp32.
 *
 * Launches: on the tensor-core path, a memset of the workspace's flags and
 * then, for one sequence, a single cooperative launch (one CTA per SM; the
 * scan of each head overlaps the solve of later chunks), or, for packed
 * batches, a solve kernel and a scan kernel.  One long sequence (32 chunks or
 * more) runs split in two segments when the device holds three scans per head
 * and two solve CTAs per head beside them (with Nv = 32 that needs 160 SMs):
 * the second segment is scanned from a zero state and its transition map beside
 * the first, and a fix-up kernel adds the first segment's final state's share
 * to its outputs and to the final state.
 * The workspace of one sequence holds a ring of 16 solve-tile positions per
 * head (and segment), one flag per (chunk, head), and the split's scratch when
 * it splits: it grows by 4 bytes per chunk and head (plus, split, 128 bytes per
 * token and head), not by the 49,664-byte tile of every chunk.  Packed batches
 * keep one tile per (chunk, head).  The size is for the current device (its SM
 * count decides the split).  One workspace must not be shared by calls that
 * can run at the same time.
 *
 *   q, k           [tokens, Nk, Dk]     in_dtype
 *   v              [tokens, Nv, Dv]     in_dtype
 *   g, beta        [tokens, Nv]         float32
 *   scale          multiplies q (1.0 when q comes from gdn_conv_gating)
 *   initial_state  [N, Nv, Dk, Dv] float32, or NULL (zero state)
 *   final_state    [N, Nv, Dk, Dv] float32, or NULL (not written); may
 *                  equal initial_state (in-place update)
 *   o              [tokens, Nv, Dv]     out_dtype
 *   workspace      device scratch of gdn_chunk_prefill_workspace_size()
 *                  bytes (may be NULL when that size is 0)
 * ------------------------------------------------------------------------ */
int gdn_chunk_prefill_workspace_size(const gdn_dims* dims, size_t* bytes);

int gdn_chunk_prefill(const gdn_dims* dims, const int32_t* cu_seqlens,
                      const void* q, const void* k, const void* v, int in_dtype,
                      const float* g, const float* beta, float scale,
                      const float* initial_state, float* final_state,
                      void* o, int out_dtype,
                      void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * gdn_chunk_prefill_gated_norm -- steps a4 + a6 in one pass: the chunked
 * gated delta rule of gdn_chunk_prefill followed by the gated RMSNorm of
 * gdn_gated_rmsnorm on each (token, value head) row of its output
 * ([RFC] 2.2 ops 4 and 6; [QDA] forward listing: core output, then
 * self.norm(core_output, z)).  The core output o is rounded to bf16 (as a
 * stored bf16 o would be) and normalised:
 *   y[t, h] = o[t, h] / sqrt(mean(o[t, h]^2) + norm_eps) * norm_w * silu(z[t, h])
 * One sequence (the cooperative launch): the scan stores o into y and spare
 * solve groups normalise each 64-token block in place once it has landed, beside
 * the scan of later chunks (on one GB300, 119.2 us against 111.1 + 18.9 us for
 * gdn_chunk_prefill + gdn_gated_rmsnorm at 4096 tokens, 32 heads).  Packed
 * batches apply the norm in the scan's output epilogue (o is never stored; for
 * bf16 y the gate norm_w * silu(z) is evaluated in bf16x2 arithmetic), which is
 * slower than the two separate calls.  fp32 y keeps fp32 arithmetic.
 * Arguments as gdn_chunk_prefill, with o replaced by
 *   z              [tokens, Nv, Dv]     bf16 (else GDN_ERR_UNSUPPORTED)
 *   norm_w         [Dv]                 float32
 *   norm_eps       the RMSNorm epsilon
 *   y              [tokens, Nv, Dv]     out_dtype
 * Tensor-core shapes only (bf16 q/k/v, Dk = Dv = 128; else
 * GDN_ERR_UNSUPPORTED); same workspace as gdn_chunk_prefill.
 * ------------------------------------------------------------------------ */
int gdn_chunk_prefill_gated_norm(const gdn_dims* dims, const int32_t* cu_seqlens,
                                 const void* q, const void* k, const void* v, int in_dtype,
                                 const float* g, const float* beta, float scale,
                                 const float* initial_state, float* final_state,
                                 const void* z, int z_dtype, const float* norm_w, float norm_eps,
                                 void* y, int out_dtype,
                                 void* workspace, size_t workspace_bytes, void* stream);

/* gdn_chunk_prefill_fp32 -- the same computation as gdn_chunk_prefill, on
 * CUDA cores in fp32 throughout (q, k, v are not rounded to bf16).  Slower;
 * for callers that want fp32 accuracy of the chunk form.  Same arguments,
 * no workspace. */
int gdn_chunk_prefill_fp32(const gdn_dims* dims, const int32_t* cu_seqlens,
                           const void* q, const void* k, const void* v, int in_dtype,
                           const float* g, const float* beta, float scale,
                           const float* initial_state, float* final_state,
                           void* o, int out_dtype, void* stream);

/* gdn_chunk_prefill_static -- gdn_chunk_prefill for callers that cannot
 * allocate device memory: hosts that reserve the device's memory up front
 * (a serving engine's arena, another framework's plugin interface) and have
 * no allocator to hand out a workspace at call time.  No counterpart on the
 * source pages; this is a packaging choice of the library.
 *
 * Same arguments as gdn_chunk_prefill without the workspace: the library uses
 * its own fixed 32 MiB scratch array in device memory instead, which every
 * GPU that loads the library holds until the process exits.  This call never
 * allocates or frees.
 *   - Supported inputs: bf16 q/k/v with Dk = Dv = 128 (else
 *     GDN_ERR_UNSUPPORTED).
 *   - Size limit: the workspace of these dims, laid out without the split of a
 *     long sequence, must be at most 32 MiB.  One sequence of any length up to
 *     about 2 million tokens fits (its solve tiles go through a fixed ring; at
 *     32 value heads the ring takes 25.4 MB), but it never runs split.  Packed
 *     batches keep a tile per (chunk, head): at 32 value heads, about 1,200
 *     tokens in all.  Larger problems return GDN_ERR_INVALID_ARG and should use
 *     gdn_chunk_prefill.
 *   - The first call on a device looks up the scratch array's device address
 *     (once per device, with that device current); make that first call before
 *     any stream capture.
 *   - All calls share the one array and it keeps the last call's contents
 *     (every call rewrites what it reads, so nothing needs clearing).  Calls
 *     that overlap on the GPU (different streams, or different host threads)
 *     race on it: serialise them. */
int gdn_chunk_prefill_static(const gdn_dims* dims, const int32_t* cu_seqlens,
                             const void* q, const void* k, const void* v, int in_dtype,
                             const float* g, const float* beta, float scale,
                             const float* initial_state, float* final_state,
                             void* o, int out_dtype, void* stream);

/* ------------------------------------------------------------------------
 * gdn_recurrent_decode -- step a5: the token-by-token gated delta rule with
 * the fp32 state read-modify-written in place ([RFC] 2.2 op 5 and 3.1.3
 * state memory; [QDA] recurrent_gated_delta_rule).  For every sequence and
 * value head h (key head h / (Nv/Nk)), for each of its tokens in order:
 *   S <- exp(g_t) S;  u = beta_t (v_t - S^T k_t);  S <- S + k_t u^T;
 *   o_t = S^T (scale * q_t).
 *   q, k [tokens, Nk, Dk], v [tokens, Nv, Dv]   in_dtype
 *   g, beta [tokens, Nv] float32
 *   state  [N, Nv, Dk, Dv] float32, read and overwritten in place
 *   o      [tokens, Nv, Dv] out_dtype
 * Sequences may hold several tokens (multi-token decode / verify).
 * ------------------------------------------------------------------------ */
int gdn_recurrent_decode(const gdn_dims* dims, const int32_t* cu_seqlens,
                         const void* q, const void* k, const void* v, int in_dtype,
                         const float* g, const float* beta, float scale,
                         float* state, void* o, int out_dtype, void* stream);

/* ------------------------------------------------------------------------
 * gdn_recurrent_decode_steps -- gdn_recurrent_decode that also writes the
 * state after every token: the rollback points of a multi-token (draft +
 * verify) decode step, where a caller keeps the state after the last
 * accepted token by copying step_states[bos + j] into state.  No counterpart
 * on the source pages beyond the multi-token decode itself ([QDA]
 * recurrent_gated_delta_rule over several tokens).
 *   step_states    [tokens, Nv, Dk, Dv] float32, written: the state after
 *                  token t of its sequence (same [Dk, Dv] layout as state);
 *                  NULL returns GDN_ERR_INVALID_ARG
 * Other arguments and the in-place final state as gdn_recurrent_decode.
 * ------------------------------------------------------------------------ */
int gdn_recurrent_decode_steps(const gdn_dims* dims, const int32_t* cu_seqlens,
                               const void* q, const void* k, const void* v, int in_dtype,
                               const float* g, const float* beta, float scale,
                               float* state, float* step_states, void* o, int out_dtype,
                               void* stream);

/* ------------------------------------------------------------------------
 * gdn_gated_rmsnorm -- step a6 ([RFC] 2.2 op 6, [QDA] self.norm(core, z)):
 *   y[r, :] = x[r, :] / sqrt(mean(x[r, :]^2) + eps) * w * silu(z[r, :])
 *   x [rows, dim] x_dtype; z [rows, dim] z_dtype; w [dim] float32;
 *   y [rows, dim] out_dtype.  dim in {64, 128}.
 * silu(z) as in gdn_conv_gating: the hardware-tanh form for bf16 y (absolute
 * error at most about 2^-11 |z| / 2), z / (1 + e^-z) for fp32 y.
 * ------------------------------------------------------------------------ */
int gdn_gated_rmsnorm(int64_t rows, int32_t dim, const void* x, int x_dtype,
                      const void* z, int z_dtype, const float* w, float eps,
                      void* y, int out_dtype, void* stream);

/* ------------------------------------------------------------------------
 * gdn_decode_fused -- step a7: one decode step of the whole mixer for
 * num_seqs sequences with one new token each (total_tokens == num_seqs),
 * in one launch: conv-state update + conv + SiLU ([RFC] 2.4 conv-state
 * update), split / L2-norm / q scale, gating, one recurrent step with the
 * fp32 state updated in place, and the gated RMSNorm.
 *   mixed_qkv  [B, C] in_dtype;  conv_w [C, 4] in_dtype;  conv_bias [C] or NULL
 *   conv_state [B, C, 3] in_dtype, updated in place
 *   a, b [B, Nv] in_dtype;  A_log, dt_bias [Nv] float32
 *   state [B, Nv, Dk, Dv] float32, updated in place
 *   z [B, Nv, Dv] in_dtype;  norm_w [Dv] float32
 *   y [B, Nv, Dv] out_dtype
 * ------------------------------------------------------------------------ */
int gdn_decode_fused(const gdn_dims* dims,
                     const void* mixed_qkv, int in_dtype,
                     const void* conv_w, const void* conv_bias, void* conv_state,
                     const void* a, const void* b,
                     const float* A_log, const float* dt_bias,
                     float q_scale, float l2_eps,
                     float* state, const void* z, const float* norm_w, float norm_eps,
                     void* y, int out_dtype, void* stream);

/* ------------------------------------------------------------------------
 * Test hook (no counterpart on the source pages): failure detection of the
 * bounded device waits.  Every wait of the chunk-prefill scan on a ready flag
 * or an mbarrier gives up after a bound of device time (2 s in the calls
 * above); the CTA then lets its copies and products in flight land, releases
 * its tensor memory, raises the device error flag with code 2 ("bounded wait
 * timed out") and exits, and the context stays usable.
 *
 * gdn_test_chunk_wait_timeout enqueues the one-sequence chunk-prefill launch
 * of gdn_chunk_prefill with no solve work, so that no chunk's ready flag is
 * ever published, and with each wait bounded by wait_ns (1 ms .. 10 s): every
 * scan's first flag wait runs out while none of its copies or products is in
 * flight.  Arguments as gdn_chunk_prefill (one sequence, bf16 q/k/v and o,
 * Dk = Dv = 128, no states); o is not written.  The caller then reads
 * GDN_ERR_DEVICE from gdn_check_device_error().  Returns GDN_ERR_UNSUPPORTED
 * when the device cannot hold the one-sequence launch (fewer SMs than value
 * heads + 1, or no cooperative launch).
 * ------------------------------------------------------------------------ */
int gdn_test_chunk_wait_timeout(const gdn_dims* dims, const void* q, const void* k, const void* v,
                                const float* g, const float* beta, void* o, void* workspace,
                                size_t workspace_bytes, int64_t wait_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
