// C-ABI layer of the GB300 Gated DeltaNet library: argument validation on the
// host, then the launch of the kernels of each call.  Declarations and the
// contract of every entry point are in include/gdn.h.

#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "gdn.h"
#include "launch.h"

namespace {

thread_local char g_err[512] = "no error";

int fail(int code, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char* where) {
  return fail(GDN_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

// Sticky device error flag, one per device that loads the library.
__device__ int g_device_error;

constexpr int kMaxDevices = 64;
std::mutex g_flag_mu;
int* g_flag_ptr[kMaxDevices];

// Device address of the error flag on the current device (looked up once).
int get_flag(int** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(GDN_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::lock_guard<std::mutex> lock(g_flag_mu);
  if (g_flag_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_device_error);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(device error flag)");
    g_flag_ptr[dev] = static_cast<int*>(ptr);
  }
  *out = g_flag_ptr[dev];
  return GDN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool valid_dtype(int d) { return d == GDN_BF16 || d == GDN_F32; }

#define REQUIRE_PTR(p)                                                                  \
  do {                                                                                  \
    if ((p) == nullptr) return fail(GDN_ERR_INVALID_ARG, "%s: %s is NULL", fn, #p);    \
    if (!aligned16(p)) return fail(GDN_ERR_INVALID_ARG, "%s: %s is not 16-byte aligned", fn, #p); \
  } while (0)
#define OPTIONAL_PTR(p)                                                                 \
  do {                                                                                  \
    if ((p) != nullptr && !aligned16(p))                                                \
      return fail(GDN_ERR_INVALID_ARG, "%s: %s is not 16-byte aligned", fn, #p);      \
  } while (0)

int check_dims(const char* fn, const gdn_dims* d, const int32_t* cu) {
  if (d == nullptr) return fail(GDN_ERR_INVALID_ARG, "%s: dims is NULL", fn);
  if (d->num_seqs < 1) return fail(GDN_ERR_INVALID_ARG, "%s: num_seqs = %d < 1", fn, d->num_seqs);
  if (d->total_tokens < 0) return fail(GDN_ERR_INVALID_ARG, "%s: total_tokens < 0", fn);
  if (d->num_k_heads < 1 || d->num_v_heads < 1)
    return fail(GDN_ERR_INVALID_ARG, "%s: head counts must be >= 1", fn);
  if (d->num_v_heads % d->num_k_heads != 0)
    return fail(GDN_ERR_INVALID_ARG, "%s: num_v_heads (%d) is not a multiple of num_k_heads (%d)",
                fn, d->num_v_heads, d->num_k_heads);
  if ((d->head_k_dim != 64 && d->head_k_dim != 128) || (d->head_v_dim != 64 && d->head_v_dim != 128))
    return fail(GDN_ERR_UNSUPPORTED, "%s: head dims (%d, %d) not in {64, 128}", fn,
                d->head_k_dim, d->head_v_dim);
  if (cu == nullptr && d->total_tokens % d->num_seqs != 0)
    return fail(GDN_ERR_INVALID_ARG, "%s: total_tokens %% num_seqs != 0 without cu_seqlens", fn);
  OPTIONAL_PTR(cu);
  return GDN_OK;
}

}  // namespace

extern "C" {

int gdn_version(void) { return (1 << 16) | 0; }

const char* gdn_last_error_string(void) { return g_err; }

int gdn_check_device_error(void* stream) {
  int* flag = nullptr;
  int st = get_flag(&flag);
  if (st != GDN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int host = 0;
  e = cudaMemcpy(&host, flag, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read device error flag");
  if (host != 0) {
    const int zero = 0;
    e = cudaMemcpy(flag, &zero, sizeof(int), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "clear device error flag");
    return fail(GDN_ERR_DEVICE, "device error %d (%s)", host,
                host == 1 ? "inconsistent cu_seqlens" : host == 2 ? "bounded wait timed out" : "?");
  }
  return GDN_OK;
}

int gdn_conv_gating(const gdn_dims* dims, const int32_t* cu_seqlens, const void* mixed_qkv,
                    int in_dtype, const void* conv_w, const void* conv_bias,
                    const void* conv_state_in, void* conv_state_out, const void* a, const void* b,
                    const float* A_log, const float* dt_bias, float q_scale, float l2_eps,
                    void* q, void* k, void* v, int out_dtype, float* g, float* beta,
                    void* stream) {
  const char* fn = "gdn_conv_gating";
  int st = check_dims(fn, dims, cu_seqlens);
  if (st != GDN_OK) return st;
  if (!valid_dtype(in_dtype) || !valid_dtype(out_dtype))
    return fail(GDN_ERR_INVALID_ARG, "%s: bad dtype", fn);
  const int kd = dims->num_k_heads * dims->head_k_dim;
  const int vd = dims->num_v_heads * dims->head_v_dim;
  if (kd % 128 != 0 || vd % 128 != 0)
    return fail(GDN_ERR_UNSUPPORTED, "%s: Nk*Dk and Nv*Dv must be multiples of 128", fn);
  REQUIRE_PTR(conv_w);
  REQUIRE_PTR(A_log);
  REQUIRE_PTR(dt_bias);
  OPTIONAL_PTR(conv_bias);
  OPTIONAL_PTR(conv_state_in);
  OPTIONAL_PTR(conv_state_out);
  if (dims->total_tokens > 0) {
    REQUIRE_PTR(mixed_qkv);
    REQUIRE_PTR(a);
    REQUIRE_PTR(b);
    REQUIRE_PTR(q);
    REQUIRE_PTR(k);
    REQUIRE_PTR(v);
    REQUIRE_PTR(g);
    REQUIRE_PTR(beta);
  }
  int* flag = nullptr;
  st = get_flag(&flag);
  if (st != GDN_OK) return st;
  gdn::ConvGatingArgs p{};
  p.x = mixed_qkv; p.w = conv_w; p.bias = conv_bias;
  p.state_in = conv_state_in; p.state_out = conv_state_out;
  p.a = a; p.b = b; p.A_log = A_log; p.dt_bias = dt_bias;
  p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta;
  p.cu = cu_seqlens; p.num_seqs = dims->num_seqs; p.total = dims->total_tokens;
  p.Nk = dims->num_k_heads; p.Nv = dims->num_v_heads;
  p.Dk = dims->head_k_dim; p.Dv = dims->head_v_dim; p.C = 2 * kd + vd;
  p.q_scale = q_scale; p.l2_eps = l2_eps;
  p.in_bf16 = in_dtype == GDN_BF16; p.out_bf16 = out_dtype == GDN_BF16;
  p.err = flag;
  cudaError_t e = gdn::launch_conv_gating(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return GDN_OK;
}

int gdn_conv_state_steps(const gdn_dims* dims, const int32_t* cu_seqlens, const void* mixed_qkv, int in_dtype,
                         const void* conv_state_in, void* step_states, void* stream) {
  const char* fn = "gdn_conv_state_steps";
  int st = check_dims(fn, dims, cu_seqlens);
  if (st != GDN_OK) return st;
  if (!valid_dtype(in_dtype)) return fail(GDN_ERR_INVALID_ARG, "%s: bad dtype", fn);
  OPTIONAL_PTR(conv_state_in);
  if (dims->total_tokens > 0) {
    REQUIRE_PTR(mixed_qkv);
    REQUIRE_PTR(step_states);
  }
  int* flag = nullptr;
  st = get_flag(&flag);
  if (st != GDN_OK) return st;
  gdn::ConvGatingArgs p{};
  p.x = mixed_qkv;
  p.state_in = conv_state_in;
  p.cu = cu_seqlens;
  p.num_seqs = dims->num_seqs;
  p.total = dims->total_tokens;
  p.C = 2 * dims->num_k_heads * dims->head_k_dim + dims->num_v_heads * dims->head_v_dim;
  p.in_bf16 = in_dtype == GDN_BF16;
  p.err = flag;
  cudaError_t e = gdn::launch_conv_state_steps(p, step_states, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return GDN_OK;
}

int gdn_gating(int64_t rows, int32_t num_v_heads, const void* a, const void* b, int in_dtype,
               const float* A_log, const float* dt_bias, float* g, float* beta, void* stream) {
  const char* fn = "gdn_gating";
  if (rows < 0 || num_v_heads < 1) return fail(GDN_ERR_INVALID_ARG, "%s: bad sizes", fn);
  if (!valid_dtype(in_dtype)) return fail(GDN_ERR_INVALID_ARG, "%s: bad dtype", fn);
  REQUIRE_PTR(A_log);
  REQUIRE_PTR(dt_bias);
  if (rows > 0) {
    REQUIRE_PTR(a);
    REQUIRE_PTR(b);
    REQUIRE_PTR(g);
    REQUIRE_PTR(beta);
  }
  gdn::GatingArgs p{a, b, A_log, dt_bias, g, beta, rows, num_v_heads, in_dtype == GDN_BF16};
  cudaError_t e = gdn::launch_gating(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return GDN_OK;
}

int gdn_chunk_prefill_workspace_size(const gdn_dims* dims, size_t* bytes) {
  const char* fn = "gdn_chunk_prefill_workspace_size";
  if (dims == nullptr || bytes == nullptr) return fail(GDN_ERR_INVALID_ARG, "%s: NULL argument", fn);
  int st = check_dims(fn, dims, nullptr);
  if (st != GDN_OK && st != GDN_ERR_INVALID_ARG) return st;   // equal split not required here
  *bytes = (dims->head_k_dim == 128 && dims->head_v_dim == 128)
               ? gdn::chunk_tc_workspace_bytes(dims->num_seqs, dims->total_tokens, dims->num_v_heads)
               : 0;
  return GDN_OK;
}

static int chunk_common(const char* fn, const gdn_dims* dims, const int32_t* cu_seqlens,
                        const void* q, const void* k, const void* v, int in_dtype,
                        const float* g, const float* beta, const float* initial_state,
                        float* final_state, void* o, int out_dtype, gdn::ChunkArgs* p) {
  int st = check_dims(fn, dims, cu_seqlens);
  if (st != GDN_OK) return st;
  if (!valid_dtype(in_dtype) || !valid_dtype(out_dtype))
    return fail(GDN_ERR_INVALID_ARG, "%s: bad dtype", fn);
  OPTIONAL_PTR(initial_state);
  OPTIONAL_PTR(final_state);
  if (dims->total_tokens > 0) {
    REQUIRE_PTR(q);
    REQUIRE_PTR(k);
    REQUIRE_PTR(v);
    REQUIRE_PTR(g);
    REQUIRE_PTR(beta);
    REQUIRE_PTR(o);
  }
  int* flag = nullptr;
  st = get_flag(&flag);
  if (st != GDN_OK) return st;
  *p = gdn::ChunkArgs{};
  p->q = q; p->k = k; p->v = v; p->g = g; p->beta = beta;
  p->S0 = initial_state; p->ST = final_state; p->o = o;
  p->cu = cu_seqlens; p->num_seqs = dims->num_seqs; p->total = dims->total_tokens;
  p->Nk = dims->num_k_heads; p->Nv = dims->num_v_heads;
  p->Dk = dims->head_k_dim; p->Dv = dims->head_v_dim;
  p->in_bf16 = in_dtype == GDN_BF16; p->out_bf16 = out_dtype == GDN_BF16;
  p->err = flag;
  return GDN_OK;
}

int gdn_chunk_prefill(const gdn_dims* dims, const int32_t* cu_seqlens, const void* q,
                      const void* k, const void* v, int in_dtype, const float* g,
                      const float* beta, float scale, const float* initial_state,
                      float* final_state, void* o, int out_dtype, void* workspace,
                      size_t workspace_bytes, void* stream) {
  const char* fn = "gdn_chunk_prefill";
  gdn::ChunkArgs p;
  int st = chunk_common(fn, dims, cu_seqlens, q, k, v, in_dtype, g, beta, initial_state,
                        final_state, o, out_dtype, &p);
  if (st != GDN_OK) return st;
  p.scale = scale;
  p.workspace = workspace;
  p.workspace_bytes = workspace_bytes;
  // bf16 q/k/v with 128-wide heads run on the tensor cores; fp32 inputs and
  // other head sizes run the fp32 CUDA-core kernel.
  const bool tc = gdn::chunk_tc_supported(p);
  if (tc && dims->total_tokens > 0) {
    const size_t need = gdn::chunk_tc_workspace_bytes(dims->num_seqs, dims->total_tokens, dims->num_v_heads);
    if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace))
      return fail(GDN_ERR_INVALID_ARG, "%s: workspace of %zu bytes (16-byte aligned) required, got %zu", fn,
                  need, workspace_bytes);
  }
  cudaError_t e = tc ? gdn::launch_chunk_tc(p, static_cast<cudaStream_t>(stream))
                     : gdn::launch_chunk_simt(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return GDN_OK;
}

int gdn_chunk_prefill_gated_norm(const gdn_dims* dims, const int32_t* cu_seqlens, const void* q,
                                 const void* k, const void* v, int in_dtype, const float* g,
                                 const float* beta, float scale, const float* initial_state,
                                 float* final_state, const void* z, int z_dtype, const float* norm_w,
                                 float norm_eps, void* y, int out_dtype, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  const char* fn = "gdn_chunk_prefill_gated_norm";
  gdn::ChunkArgs p;
  int st = chunk_common(fn, dims, cu_seqlens, q, k, v, in_dtype, g, beta, initial_state,
                        final_state, y, out_dtype, &p);
  if (st != GDN_OK) return st;
  if (!valid_dtype(z_dtype)) return fail(GDN_ERR_INVALID_ARG, "%s: bad dtype", fn);
  if (!gdn::chunk_tc_supported(p))
    return fail(GDN_ERR_UNSUPPORTED, "%s: needs bf16 q/k/v and 128-wide heads", fn);
  if (z_dtype != GDN_BF16) return fail(GDN_ERR_UNSUPPORTED, "%s: z must be bf16", fn);
  REQUIRE_PTR(norm_w);
  if (dims->total_tokens > 0) {
    REQUIRE_PTR(z);
    const size_t need = gdn::chunk_tc_workspace_bytes(dims->num_seqs, dims->total_tokens, dims->num_v_heads);
    if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace))
      return fail(GDN_ERR_INVALID_ARG, "%s: workspace of %zu bytes (16-byte aligned) required, got %zu", fn,
                  need, workspace_bytes);
  }
  p.scale = scale;
  p.workspace = workspace;
  p.workspace_bytes = workspace_bytes;
  p.z = z;
  p.norm_w = norm_w;
  p.norm_eps = norm_eps;
  cudaError_t e = gdn::launch_chunk_tc(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return GDN_OK;
}

int gdn_chunk_prefill_fp32(const gdn_dims* dims, const int32_t* cu_seqlens, const void* q,
                           const void* k, const void* v, int in_dtype, const float* g,
                           const float* beta, float scale, const float* initial_state,
                           float* final_state, void* o, int out_dtype, void* stream) {
  const char* fn = "gdn_chunk_prefill_fp32";
  gdn::ChunkArgs p;
  int st = chunk_common(fn, dims, cu_seqlens, q, k, v, in_dtype, g, beta, initial_state,
                        final_state, o, out_dtype, &p);
  if (st != GDN_OK) return st;
  p.scale = scale;
  cudaError_t e = gdn::launch_chunk_simt(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return GDN_OK;
}

int gdn_chunk_prefill_static(const gdn_dims* dims, const int32_t* cu_seqlens, const void* q,
                             const void* k, const void* v, int in_dtype, const float* g,
                             const float* beta, float scale, const float* initial_state,
                             float* final_state, void* o, int out_dtype, void* stream) {
  const char* fn = "gdn_chunk_prefill_static";
  gdn::ChunkArgs p;
  int st = chunk_common(fn, dims, cu_seqlens, q, k, v, in_dtype, g, beta, initial_state,
                        final_state, o, out_dtype, &p);
  if (st != GDN_OK) return st;
  if (!gdn::chunk_tc_supported(p))
    return fail(GDN_ERR_UNSUPPORTED, "%s: needs bf16 q/k/v and 128-wide heads", fn);
  const size_t need = gdn::chunk_tc_workspace_bytes(dims->num_seqs, dims->total_tokens, dims->num_v_heads, false);
  if (need > gdn::kStaticScratchBytes)
    return fail(GDN_ERR_INVALID_ARG,
                "%s: this problem needs %zu bytes of scratch, more than the library's fixed %zu bytes; "
                "use gdn_chunk_prefill with a caller workspace", fn, need, gdn::kStaticScratchBytes);
  void* scratch = nullptr;
  cudaError_t e = gdn::static_scratch(&scratch);
  if (e != cudaSuccess) return cuda_fail(e, fn);
  p.scale = scale;
  p.workspace = scratch;
  p.workspace_bytes = gdn::kStaticScratchBytes;
  p.no_split = 1;                 // the layout checked above
  e = gdn::launch_chunk_tc(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return GDN_OK;
}

int gdn_test_chunk_wait_timeout(const gdn_dims* dims, const void* q, const void* k, const void* v,
                                const float* g, const float* beta, void* o, void* workspace,
                                size_t workspace_bytes, int64_t wait_ns, void* stream) {
  const char* fn = "gdn_test_chunk_wait_timeout";
  gdn::ChunkArgs p;
  int st = chunk_common(fn, dims, nullptr, q, k, v, GDN_BF16, g, beta, nullptr, nullptr, o, GDN_BF16, &p);
  if (st != GDN_OK) return st;
  if (dims->num_seqs != 1 || dims->total_tokens < 1 || !gdn::chunk_tc_supported(p))
    return fail(GDN_ERR_UNSUPPORTED, "%s: needs one sequence of bf16 q/k/v with 128-wide heads", fn);
  if (wait_ns < 1000000 || wait_ns > 10000000000ll)
    return fail(GDN_ERR_INVALID_ARG, "%s: wait_ns must lie in [1 ms, 10 s]", fn);
  const size_t need = gdn::chunk_tc_workspace_bytes(dims->num_seqs, dims->total_tokens, dims->num_v_heads);
  if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace))
    return fail(GDN_ERR_INVALID_ARG, "%s: workspace of %zu bytes (16-byte aligned) required", fn, need);
  p.scale = 1.0f;
  p.workspace = workspace;
  p.workspace_bytes = workspace_bytes;
  p.wait_ns = (unsigned long long)wait_ns;
  p.no_solve = 1;
  cudaError_t e = gdn::launch_chunk_tc(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return GDN_OK;
}

static int recurrent_decode(const char* fn, const gdn_dims* dims, const int32_t* cu_seqlens, const void* q,
                            const void* k, const void* v, int in_dtype, const float* g,
                            const float* beta, float scale, float* state, float* step_states, void* o,
                            int out_dtype, void* stream) {
  int st = check_dims(fn, dims, cu_seqlens);
  if (st != GDN_OK) return st;
  if (!valid_dtype(in_dtype) || !valid_dtype(out_dtype))
    return fail(GDN_ERR_INVALID_ARG, "%s: bad dtype", fn);
  REQUIRE_PTR(state);
  OPTIONAL_PTR(step_states);
  if (dims->total_tokens > 0) {
    REQUIRE_PTR(q);
    REQUIRE_PTR(k);
    REQUIRE_PTR(v);
    REQUIRE_PTR(g);
    REQUIRE_PTR(beta);
    REQUIRE_PTR(o);
  }
  int* flag = nullptr;
  st = get_flag(&flag);
  if (st != GDN_OK) return st;
  gdn::DecodeArgs p{};
  p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta; p.state = state; p.o = o;
  p.step_states = step_states;
  p.cu = cu_seqlens; p.num_seqs = dims->num_seqs; p.total = dims->total_tokens;
  p.Nk = dims->num_k_heads; p.Nv = dims->num_v_heads;
  p.Dk = dims->head_k_dim; p.Dv = dims->head_v_dim;
  p.scale = scale; p.in_bf16 = in_dtype == GDN_BF16; p.out_bf16 = out_dtype == GDN_BF16;
  p.err = flag;
  cudaError_t e = gdn::launch_recurrent_decode(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return GDN_OK;
}

int gdn_recurrent_decode(const gdn_dims* dims, const int32_t* cu_seqlens, const void* q,
                         const void* k, const void* v, int in_dtype, const float* g,
                         const float* beta, float scale, float* state, void* o, int out_dtype,
                         void* stream) {
  return recurrent_decode("gdn_recurrent_decode", dims, cu_seqlens, q, k, v, in_dtype, g, beta, scale, state,
                          nullptr, o, out_dtype, stream);
}

int gdn_recurrent_decode_steps(const gdn_dims* dims, const int32_t* cu_seqlens, const void* q,
                               const void* k, const void* v, int in_dtype, const float* g,
                               const float* beta, float scale, float* state, float* step_states, void* o,
                               int out_dtype, void* stream) {
  if (step_states == nullptr)
    return fail(GDN_ERR_INVALID_ARG, "gdn_recurrent_decode_steps: step_states is NULL");
  return recurrent_decode("gdn_recurrent_decode_steps", dims, cu_seqlens, q, k, v, in_dtype, g, beta, scale,
                          state, step_states, o, out_dtype, stream);
}

int gdn_gated_rmsnorm(int64_t rows, int32_t dim, const void* x, int x_dtype, const void* z,
                      int z_dtype, const float* w, float eps, void* y, int out_dtype,
                      void* stream) {
  const char* fn = "gdn_gated_rmsnorm";
  if (rows < 0) return fail(GDN_ERR_INVALID_ARG, "%s: rows < 0", fn);
  if (dim != 64 && dim != 128) return fail(GDN_ERR_UNSUPPORTED, "%s: dim %d not in {64, 128}", fn, dim);
  if (!valid_dtype(x_dtype) || !valid_dtype(z_dtype) || !valid_dtype(out_dtype))
    return fail(GDN_ERR_INVALID_ARG, "%s: bad dtype", fn);
  REQUIRE_PTR(w);
  if (rows > 0) {
    REQUIRE_PTR(x);
    REQUIRE_PTR(z);
    REQUIRE_PTR(y);
  }
  gdn::RmsNormArgs p{x, z, w, y, rows, dim, eps, x_dtype == GDN_BF16, z_dtype == GDN_BF16,
                     out_dtype == GDN_BF16};
  cudaError_t e = gdn::launch_gated_rmsnorm(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return GDN_OK;
}

int gdn_decode_fused(const gdn_dims* dims, const void* mixed_qkv, int in_dtype,
                     const void* conv_w, const void* conv_bias, void* conv_state, const void* a,
                     const void* b, const float* A_log, const float* dt_bias, float q_scale,
                     float l2_eps, float* state, const void* z, const float* norm_w,
                     float norm_eps, void* y, int out_dtype, void* stream) {
  const char* fn = "gdn_decode_fused";
  int st = check_dims(fn, dims, nullptr);
  if (st != GDN_OK) return st;
  if (dims->total_tokens != dims->num_seqs)
    return fail(GDN_ERR_INVALID_ARG, "%s: needs exactly one token per sequence", fn);
  if (dims->num_v_heads / dims->num_k_heads > 32)
    return fail(GDN_ERR_UNSUPPORTED, "%s: Nv/Nk > 32", fn);
  if (!valid_dtype(in_dtype) || !valid_dtype(out_dtype))
    return fail(GDN_ERR_INVALID_ARG, "%s: bad dtype", fn);
  REQUIRE_PTR(mixed_qkv);
  REQUIRE_PTR(conv_w);
  OPTIONAL_PTR(conv_bias);
  REQUIRE_PTR(conv_state);
  REQUIRE_PTR(a);
  REQUIRE_PTR(b);
  REQUIRE_PTR(A_log);
  REQUIRE_PTR(dt_bias);
  REQUIRE_PTR(state);
  REQUIRE_PTR(z);
  REQUIRE_PTR(norm_w);
  REQUIRE_PTR(y);
  gdn::DecodeFusedArgs p{};
  p.x = mixed_qkv; p.w = conv_w; p.bias = conv_bias; p.conv_state = conv_state;
  p.a = a; p.b = b; p.A_log = A_log; p.dt_bias = dt_bias;
  p.state = state; p.z = z; p.norm_w = norm_w; p.y = y;
  p.B = dims->num_seqs; p.Nk = dims->num_k_heads; p.Nv = dims->num_v_heads;
  p.Dk = dims->head_k_dim; p.Dv = dims->head_v_dim;
  p.C = 2 * p.Nk * p.Dk + p.Nv * p.Dv;
  p.q_scale = q_scale; p.l2_eps = l2_eps; p.norm_eps = norm_eps;
  p.in_bf16 = in_dtype == GDN_BF16; p.out_bf16 = out_dtype == GDN_BF16;
  cudaError_t e = gdn::launch_decode_fused(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return GDN_OK;
}

}  // extern "C"
