// Internal launcher interface between the C-ABI layer (api.cu) and the
// kernel translation units.  Arguments are already validated by the caller.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace gdn {

struct ConvGatingArgs {
  const void* x;          // mixed_qkv [T, C]
  const void* w;          // [C, 4]
  const void* bias;       // [C] or null
  const void* state_in;   // [N, C, 3] or null
  void* state_out;        // [N, C, 3] or null
  const void* a;          // [T, Nv]
  const void* b;          // [T, Nv]
  const float* A_log;     // [Nv]
  const float* dt_bias;   // [Nv]
  void* q;                // [T, Nk, Dk]
  void* k;                // [T, Nk, Dk]
  void* v;                // [T, Nv, Dv]
  float* g;               // [T, Nv]
  float* beta;            // [T, Nv]
  const int32_t* cu;      // [N + 1] or null
  int num_seqs, total, Nk, Nv, Dk, Dv, C;
  float q_scale, l2_eps;
  int in_bf16, out_bf16;
  int* err;
};
cudaError_t launch_conv_gating(const ConvGatingArgs& p, cudaStream_t s);
// The conv state after every token ([tokens, C, 3], the input element type).
cudaError_t launch_conv_state_steps(const ConvGatingArgs& p, void* steps, cudaStream_t s);

struct GatingArgs {
  const void* a; const void* b; const float* A_log; const float* dt_bias;
  float* g; float* beta; int64_t rows; int Nv; int in_bf16;
};
cudaError_t launch_gating(const GatingArgs& p, cudaStream_t s);

struct RmsNormArgs {
  const void* x; const void* z; const float* w; void* y;
  int64_t rows; int dim; float eps; int x_bf16, z_bf16, out_bf16;
};
cudaError_t launch_gated_rmsnorm(const RmsNormArgs& p, cudaStream_t s);

struct DecodeArgs {
  const void* q; const void* k; const void* v;   // [T, Nk, Dk] / [T, Nv, Dv]
  const float* g; const float* beta;             // [T, Nv]
  float* state;                                  // [N, Nv, Dk, Dv]
  void* o;                                       // [T, Nv, Dv]
  const int32_t* cu;
  int num_seqs, total, Nk, Nv, Dk, Dv;
  float scale;
  int in_bf16, out_bf16;
  int* err;
  float* step_states;                            // [T, Nv, Dk, Dv] state after each token, or null
};
cudaError_t launch_recurrent_decode(const DecodeArgs& p, cudaStream_t s);

struct DecodeFusedArgs {
  const void* x; const void* w; const void* bias; void* conv_state;
  const void* a; const void* b; const float* A_log; const float* dt_bias;
  float* state; const void* z; const float* norm_w; void* y;
  int B, Nk, Nv, Dk, Dv, C;
  float q_scale, l2_eps, norm_eps;
  int in_bf16, out_bf16;
};
cudaError_t launch_decode_fused(const DecodeFusedArgs& p, cudaStream_t s);

struct ChunkArgs {
  const void* q; const void* k; const void* v;   // [T, Nk, Dk] / [T, Nv, Dv]
  const float* g; const float* beta;             // [T, Nv]
  const float* S0;                               // [N, Nv, Dk, Dv] or null
  float* ST;                                     // [N, Nv, Dk, Dv] or null
  void* o;                                       // [T, Nv, Dv]
  const int32_t* cu;
  int num_seqs, total, Nk, Nv, Dk, Dv;
  float scale;
  int in_bf16, out_bf16;
  void* workspace; size_t workspace_bytes;
  int* err;
  // gated RMSNorm fused into the output (tensor-core path): o holds y then
  const void* z;                                 // [T, Nv, Dv] bf16, or null (plain o)
  const float* norm_w;                           // [Dv]
  float norm_eps;
  // bound of each wait of the scan on a flag or barrier, in ns of device time (0: the default)
  unsigned long long wait_ns;
  int no_solve;                                  // test hook: the one-sequence launch runs no solve
  int no_split;                                  // never split a long sequence (smaller workspace)
  // one-sequence launch with z: the scan writes o into o's buffer and spare solve groups apply
  // the gated norm in place, block by block (set by the launcher, not by callers)
  int side_norm;
};
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;
// Portable fp32 CUDA-core implementation of the chunk form.
cudaError_t launch_chunk_simt(const ChunkArgs& p, cudaStream_t s);
// tcgen05 tensor-core implementation (bf16 q/k/v, Dk = Dv = 128).
bool chunk_tc_supported(const ChunkArgs& p);
// Workspace bytes of a call on the current device (allow_split: a long single sequence may
// run split in two segments, which needs extra scratch).
size_t chunk_tc_workspace_bytes(int num_seqs, int total, int Nv, bool allow_split = true);
cudaError_t launch_chunk_tc(const ChunkArgs& p, cudaStream_t s);
// Fixed-size device scratch owned by the library (see gdn_chunk_prefill_static).
constexpr size_t kStaticScratchBytes = (size_t)32 << 20;
cudaError_t static_scratch(void** ptr);

}  // namespace gdn
