// abi.cu -- the extern "C" entry points of libnc: argument validation on the
// host, then the kernels. Nothing here reads device memory.
#include <cuda_runtime.h>
#include <float.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include "engine.h"
#include "kernels.h"

namespace nc {

static thread_local char g_err[512] = "";

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
}

nc_status fail(nc_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return s;
}

static Model* M(nc_model* m) { return reinterpret_cast<Model*>(m); }
static const Model* M(const nc_model* m) { return reinterpret_cast<const Model*>(m); }
static cudaStream_t S(void* s) { return static_cast<cudaStream_t>(s); }

static bool aligned16(const void* p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; }
// NULL or a multiple of n bytes: the widest access the kernels make through p.
static bool aligned(const void* p, uintptr_t n) { return reinterpret_cast<uintptr_t>(p) % n == 0; }

static nc_status launch_result(cudaError_t e, const char* what) {
  if (e != cudaSuccess) return fail(NC_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return NC_OK;
}

static nc_status check_gemv_shape(int B, int K, int N) {
  NC_CHECK(B >= 1 && B <= 16, NC_ERR_SHAPE, "batch %d outside [1, 16]", B);
  NC_CHECK(K >= 8 && K % 8 == 0, NC_ERR_SHAPE, "K = %d must be a positive multiple of 8", K);
  NC_CHECK(N >= 1, NC_ERR_SHAPE, "N = %d must be positive", N);
  return NC_OK;
}

}  // namespace nc

using namespace nc;

extern "C" {

const char* nc_status_string(nc_status s) {
  switch (s) {
    case NC_OK: return "NC_OK";
    case NC_ERR_INVALID_ARGUMENT: return "NC_ERR_INVALID_ARGUMENT";
    case NC_ERR_SHAPE: return "NC_ERR_SHAPE";
    case NC_ERR_DTYPE: return "NC_ERR_DTYPE";
    case NC_ERR_CAPACITY: return "NC_ERR_CAPACITY";
    case NC_ERR_POSITION: return "NC_ERR_POSITION";
    case NC_ERR_CUDA: return "NC_ERR_CUDA";
    case NC_ERR_TIMEOUT: return "NC_ERR_TIMEOUT";
    case NC_ERR_UNHEALTHY: return "NC_ERR_UNHEALTHY";
    case NC_ERR_UNSUPPORTED: return "NC_ERR_UNSUPPORTED";
  }
  return "NC_ERR_UNKNOWN";
}

const char* nc_last_error_message(void) { return g_err; }

int nc_abi_version(void) { return NC_ABI_VERSION; }

nc_status nc_model_create(const nc_config* cfg, const nc_weights* w, int max_batch, int max_ctx,
                          void* stream, nc_model** out) {
  Model* m = nullptr;
  nc_status st = model_create(cfg, w, max_batch, max_ctx, S(stream), &m);
  if (st == NC_OK) *out = reinterpret_cast<nc_model*>(m);
  return st;
}

nc_status nc_model_destroy(nc_model* m) {
  NC_CHECK(m, NC_ERR_INVALID_ARGUMENT, "model is NULL");
  delete M(m);
  return NC_OK;
}

nc_status nc_model_memory(const nc_model* m, size_t* weight_bytes, size_t* workspace_bytes) {
  NC_CHECK(m, NC_ERR_INVALID_ARGUMENT, "model is NULL");
  if (weight_bytes) *weight_bytes = M(m)->weight_bytes;
  if (workspace_bytes) *workspace_bytes = M(m)->workspace_bytes;
  return NC_OK;
}

nc_status nc_decode_step(nc_model* m, int batch, int32_t* tokens_dev, int32_t* positions_dev,
                         const int32_t* positions_host, const nc_kv_cache* kv, float* logits_dev,
                         int32_t* next_dev, int flags, void* stream) {
  return decode_step(M(m), batch, tokens_dev, positions_dev, positions_host, kv, logits_dev,
                     next_dev, flags, S(stream));
}

nc_status nc_block_forward(nc_model* m, int layer, int batch, float* x_dev,
                           const int32_t* positions_dev, const int32_t* positions_host,
                           const nc_kv_cache* kv, void* stream) {
  return block_forward(M(m), layer, batch, x_dev, positions_dev, positions_host, kv, S(stream));
}

nc_status nc_get_device_status(nc_model* m, void* stream, int* code) {
  NC_CHECK(m && code, NC_ERR_INVALID_ARGUMENT, "null argument");
  Model* mm = M(m);
  // Copy into the model's pinned host word, then clear the device word.
  cudaError_t e = cudaStreamSynchronize(S(stream));
  if (!e) e = cudaMemcpyAsync(mm->status_host, mm->status, sizeof(int), cudaMemcpyDeviceToHost,
                              S(stream));
  if (!e) e = cudaMemsetAsync(mm->status, 0, sizeof(int), S(stream));
  if (!e) e = cudaStreamSynchronize(S(stream));
  if (e) {
    mm->unhealthy = true;
    return fail(NC_ERR_CUDA, "reading the status word failed: %s", cudaGetErrorString(e));
  }
  *code = *mm->status_host;
  return NC_OK;
}

nc_status nc_decode_path(nc_model* m, int batch, const nc_kv_cache* kv, int flags, int* path) {
  NC_CHECK(m && kv && path, NC_ERR_INVALID_ARGUMENT, "null argument");
  NC_CHECK(batch >= 1 && batch <= M(m)->max_batch, NC_ERR_INVALID_ARGUMENT,
           "batch %d outside [1, %d]", batch, M(m)->max_batch);
  *path = use_persistent(M(m), batch, *kv, flags) ? NC_PATH_PERSISTENT : NC_PATH_STAGED;
  return NC_OK;
}

nc_status nc_debug_w8a8_codes(nc_model* m, int8_t* codes_dev, size_t codes_capacity,
                              float* scales_dev, size_t scales_capacity) {
  NC_CHECK(m, NC_ERR_INVALID_ARGUMENT, "model is NULL");
  Model* mm = M(m);
  NC_CHECK(mm->cfg.wtype != NC_BF16, NC_ERR_DTYPE, "the model's projections are not W8A8");
  NC_CHECK(codes_dev || !scales_dev, NC_ERR_INVALID_ARGUMENT, "scales need the codes buffer");
  NC_CHECK(aligned(scales_dev, 4), NC_ERR_INVALID_ARGUMENT, "scales must be 4-byte aligned");
  mm->dbg_codes = codes_dev;
  mm->dbg_scales = scales_dev;
  mm->dbg_codes_cap = codes_dev ? codes_capacity : 0;
  mm->dbg_scales_cap = scales_dev ? scales_capacity : 0;
  return NC_OK;
}

nc_status nc_profile_phases(nc_model* m, int enable) {
  NC_CHECK(m, NC_ERR_INVALID_ARGUMENT, "model is NULL");
  M(m)->prof_on = enable != 0;
  return NC_OK;
}

nc_status nc_read_phase_profile(nc_model* m, void* stream, unsigned long long* out_host,
                                int capacity, int* n) {
  NC_CHECK(m && out_host && n, NC_ERR_INVALID_ARGUMENT, "null argument");
  Model* mm = M(m);
  const int count = num_sms() * (int)prof_values(mm->cfg.n_layers);
  NC_CHECK(capacity >= count, NC_ERR_CAPACITY, "the profile holds %d values", count);
  cudaError_t e = cudaStreamSynchronize(S(stream));
  if (!e) e = cudaMemcpy(out_host, mm->prof, sizeof(unsigned long long) * count,
                         cudaMemcpyDeviceToHost);
  if (e) {
    mm->unhealthy = true;
    return fail(NC_ERR_CUDA, "reading the phase profile failed: %s", cudaGetErrorString(e));
  }
  *n = count;
  return NC_OK;
}

// The W8A8 form of a stage GEMV (NC_INT8): int8 rows with fp32 per-row
// scales, the per-token activation codes formed in the kernel.
static nc_status launch_stage_w8(Epi epi, const float* x, const void* gamma, float eps,
                                 const void* W, const float* w_scale, const void* bias, int B,
                                 int K, int N, float* y, int32_t* acc, cudaStream_t s,
                                 const char* what) {
  NC_CHECK(w_scale, NC_ERR_INVALID_ARGUMENT, "%s: NC_INT8 needs the per-row scales", what);
  NC_CHECK(aligned16(W) && aligned(x, 4) && aligned(gamma, 2) && aligned(w_scale, 4) &&
               aligned(bias, 2) && aligned(y, 4) && aligned(acc, 4),
           NC_ERR_INVALID_ARGUMENT,
           "%s: int8 W must be 16-byte aligned, fp32 and int32 pointers 4-byte, bf16 2-byte", what);
  NC_CHECK(B >= 1 && B <= 16, NC_ERR_SHAPE, "batch %d outside [1, 16]", B);
  const int bt = B <= 1 ? 1 : B <= 2 ? 2 : B <= 4 ? 4 : B <= 8 ? 8 : 16;  // batch tile
  NC_CHECK(K >= 16 && K % 16 == 0 && (size_t)bt * K <= 200000, NC_ERR_SHAPE,
           "%s: NC_INT8 needs K a positive multiple of 16 with (B rounded up to a power of 2) "
           "* K <= 200000", what);
  NC_CHECK(N >= 1, NC_ERR_SHAPE, "N must be positive");
  W8Args a{x, static_cast<const uint16_t*>(gamma), eps, static_cast<const int8_t*>(W), w_scale,
           static_cast<const uint16_t*>(bias), B, K, N, y, nullptr, nullptr, acc};
  return launch_result(launch_w8a8(epi, a, s), what);
}

nc_status nc_rmsnorm_gemv(const float* x, const void* gamma, float eps, const void* W,
                          nc_wtype wtype, const float* w_scale, const void* bias, int B, int K,
                          int N, float* y, int32_t* acc_i32_debug, void* stream) {
  NC_CHECK(x && W && y, NC_ERR_INVALID_ARGUMENT, "null pointer");
  NC_CHECK(wtype == NC_BF16 || wtype == NC_INT8, NC_ERR_DTYPE, "unknown weight type %d",
           (int)wtype);
  if (wtype == NC_INT8)
    return launch_stage_w8(Epi::Store, x, gamma, eps, W, w_scale, bias, B, K, N, y,
                           acc_i32_debug, S(stream), "nc_rmsnorm_gemv");
  NC_CHECK(!w_scale && !acc_i32_debug, NC_ERR_INVALID_ARGUMENT,
           "w_scale and acc_i32_debug apply to NC_INT8 weights only");
  NC_CHECK(aligned16(x) && aligned16(W), NC_ERR_INVALID_ARGUMENT, "x and W must be 16-byte aligned");
  NC_CHECK(aligned(gamma, 8) && aligned(bias, 2) && aligned(y, 4), NC_ERR_INVALID_ARGUMENT,
           "gamma must be 8-byte aligned, bias 2-byte and y 4-byte");
  nc_status st = check_gemv_shape(B, K, N);
  if (st) return st;
  GemvArgs a{x, static_cast<const uint16_t*>(gamma), eps, static_cast<const uint16_t*>(W),
             static_cast<const uint16_t*>(bias), B, K, N, y};
  return launch_result(launch_gemv(Epi::Store, a, S(stream)), "nc_rmsnorm_gemv");
}

nc_status nc_gemv_residual(const float* a_in, const void* W, nc_wtype wtype, const float* w_scale,
                           int B, int K, int N, float* x, void* stream) {
  NC_CHECK(a_in && W && x, NC_ERR_INVALID_ARGUMENT, "null pointer");
  NC_CHECK(wtype == NC_BF16 || wtype == NC_INT8, NC_ERR_DTYPE, "unknown weight type %d",
           (int)wtype);
  if (wtype == NC_INT8)
    return launch_stage_w8(Epi::Residual, a_in, nullptr, 0.f, W, w_scale, nullptr, B, K, N, x,
                           nullptr, S(stream), "nc_gemv_residual");
  NC_CHECK(!w_scale, NC_ERR_INVALID_ARGUMENT, "w_scale applies to NC_INT8 weights only");
  NC_CHECK(aligned16(a_in) && aligned16(W), NC_ERR_INVALID_ARGUMENT, "inputs must be 16-byte aligned");
  NC_CHECK(aligned(x, 4), NC_ERR_INVALID_ARGUMENT, "x must be 4-byte aligned");
  nc_status st = check_gemv_shape(B, K, N);
  if (st) return st;
  GemvArgs a{a_in, nullptr, 0.f, static_cast<const uint16_t*>(W), nullptr, B, K, N, x};
  return launch_result(launch_gemv(Epi::Residual, a, S(stream)), "nc_gemv_residual");
}

nc_status nc_swiglu_gemv(const float* x, const void* gamma, float eps, const void* W_gu,
                         nc_wtype wtype, const float* s_gu, int B, int K, int F, float* h,
                         void* stream) {
  NC_CHECK(x && W_gu && h, NC_ERR_INVALID_ARGUMENT, "null pointer");
  NC_CHECK(wtype == NC_BF16 || wtype == NC_INT8, NC_ERR_DTYPE, "unknown weight type %d",
           (int)wtype);
  if (wtype == NC_INT8)
    return launch_stage_w8(Epi::SwiGLU, x, gamma, eps, W_gu, s_gu, nullptr, B, K, F, h, nullptr,
                           S(stream), "nc_swiglu_gemv");
  NC_CHECK(!s_gu, NC_ERR_INVALID_ARGUMENT, "s_gu applies to NC_INT8 weights only");
  NC_CHECK(aligned16(x) && aligned16(W_gu), NC_ERR_INVALID_ARGUMENT, "inputs must be 16-byte aligned");
  NC_CHECK(aligned(gamma, 8) && aligned(h, 4), NC_ERR_INVALID_ARGUMENT,
           "gamma must be 8-byte aligned and h 4-byte");
  nc_status st = check_gemv_shape(B, K, F);
  if (st) return st;
  GemvArgs a{x, static_cast<const uint16_t*>(gamma), eps, static_cast<const uint16_t*>(W_gu),
             nullptr, B, K, F, h};
  return launch_result(launch_gemv(Epi::SwiGLU, a, S(stream)), "nc_swiglu_gemv");
}

nc_status nc_rope_qkv(const nc_model* m, int layer, int B, const float* qkv,
                      const int32_t* positions_dev, const int32_t* positions_host, float* q_out,
                      const nc_kv_cache* kv, void* stream) {
  NC_CHECK(m && qkv && positions_dev && q_out, NC_ERR_INVALID_ARGUMENT, "null pointer");
  const Model* mm = M(m);
  NC_CHECK(layer >= 0 && layer < mm->cfg.n_layers, NC_ERR_SHAPE, "layer out of range");
  NC_CHECK(B >= 1 && B <= mm->max_batch, NC_ERR_CAPACITY, "batch outside [1, max_batch]");
  nc_status st = validate_kv(mm, B, positions_host, kv);
  if (st) return st;
  const nc_config& c = mm->cfg;
  const LayerPacked& P = mm->layers[layer];
  RopeArgs a{qkv, positions_dev, mm->inv_freq, P.g_q, P.g_k, c.rms_eps, B, c.n_q_heads,
             c.n_kv_heads, c.head_dim, layer, q_out, kv_view(mm, *kv), mm->status};
  return launch_result(launch_rope_qkv(a, S(stream)), "nc_rope_qkv");
}

nc_status nc_attn_decode(const nc_model* m, int layer, int B, const float* q,
                         const int32_t* positions_dev, const int32_t* positions_host,
                         const nc_kv_cache* kv, float* out, void* stream) {
  NC_CHECK(m && q && positions_dev && out, NC_ERR_INVALID_ARGUMENT, "null pointer");
  const Model* mm = M(m);
  NC_CHECK(layer >= 0 && layer < mm->cfg.n_layers, NC_ERR_SHAPE, "layer out of range");
  NC_CHECK(B >= 1 && B <= mm->max_batch, NC_ERR_CAPACITY, "batch outside [1, max_batch]");
  nc_status st = validate_kv(mm, B, positions_host, kv);
  if (st) return st;
  const nc_config& c = mm->cfg;
  const int splits =
      attn_splits(B, c.n_kv_heads, c.head_dim, kv->dtype == NC_KV_BF16, kv_capacity(*kv));
  AttnArgs a{q, positions_dev, B, c.n_q_heads, c.n_kv_heads, c.head_dim, layer, splits,
             mm->part, out, kv_view(mm, *kv), mm->status, mm->atickets};
  return launch_result(launch_attn(a, S(stream)), "nc_attn_decode");
}

nc_status nc_lm_head_argmax(nc_model* m, const float* x, const void* gamma, float eps,
                            const void* W, int B, int K, int V, float* logits, int32_t* next,
                            void* stream) {
  NC_CHECK(m && x && gamma && W && logits, NC_ERR_INVALID_ARGUMENT, "null pointer");
  NC_CHECK(aligned16(x) && aligned16(W) && aligned(gamma, 8) && aligned(logits, 4) &&
               aligned(next, 4),
           NC_ERR_INVALID_ARGUMENT,
           "x and W must be 16-byte aligned, gamma 8-byte, logits and next 4-byte");
  Model* mm = M(m);
  NC_CHECK(!mm->unhealthy, NC_ERR_UNHEALTHY, "model saw an earlier CUDA failure");
  NC_CHECK(B >= 1 && B <= mm->max_batch, NC_ERR_CAPACITY, "batch outside [1, max_batch]");
  const int bt = B <= 1 ? 1 : B <= 2 ? 2 : B <= 4 ? 4 : B <= 8 ? 8 : 16;  // batch tile
  NC_CHECK(K % 8 == 0 && K >= 8 && (size_t)bt * K <= 51200, NC_ERR_SHAPE,
           "K must be a multiple of 8 with (B rounded up to a power of 2) * K <= 51200");
  NC_CHECK(V >= 1, NC_ERR_SHAPE, "V must be positive");
  LmHeadArgs a{x, static_cast<const uint16_t*>(gamma), eps, static_cast<const uint16_t*>(W), B, K,
               V, logits, next, mm->am_part, mm->ticket, mm->status, nullptr, nullptr};
  return launch_result(launch_lm_head(a, S(stream)), "nc_lm_head_argmax");
}

nc_status nc_quantize_weight(const void* W, int N, int K, int8_t* q, float* scale, void* stream) {
  NC_CHECK(W && q && scale, NC_ERR_INVALID_ARGUMENT, "null pointer");
  NC_CHECK(N >= 1 && K >= 1, NC_ERR_SHAPE, "sizes must be positive");
  return launch_result(
      launch_quantize_weight(static_cast<const uint16_t*>(W), N, K, q, scale, S(stream)),
      "nc_quantize_weight");
}

nc_status nc_w8a8_gemv(const float* x, const void* gamma, float eps, const int8_t* Wq,
                       const float* w_scale, const void* bias, int B, int K, int N, float* y,
                       int8_t* xq_out, float* sx_out, int32_t* acc_out, void* stream) {
  NC_CHECK(x && Wq && w_scale && y, NC_ERR_INVALID_ARGUMENT, "null pointer");
  NC_CHECK(aligned16(Wq), NC_ERR_INVALID_ARGUMENT, "Wq must be 16-byte aligned");
  NC_CHECK(aligned(x, 4) && aligned(gamma, 2) && aligned(w_scale, 4) && aligned(bias, 2) &&
               aligned(y, 4) && aligned(sx_out, 4) && aligned(acc_out, 4),
           NC_ERR_INVALID_ARGUMENT, "fp32 and int32 pointers must be 4-byte aligned, bf16 2-byte");
  NC_CHECK(B >= 1 && B <= 16, NC_ERR_SHAPE, "batch outside [1, 16]");
  const int bt = B <= 1 ? 1 : B <= 2 ? 2 : B <= 4 ? 4 : B <= 8 ? 8 : 16;  // batch tile
  NC_CHECK(K >= 16 && K % 16 == 0 && (size_t)bt * K <= 200000, NC_ERR_SHAPE,
           "K must be a positive multiple of 16 with (B rounded up to a power of 2) * K <= 200000");
  NC_CHECK(N >= 1, NC_ERR_SHAPE, "N must be positive");
  W8Args a{x, static_cast<const uint16_t*>(gamma), eps, Wq, w_scale,
           static_cast<const uint16_t*>(bias), B, K, N, y, xq_out, sx_out, acc_out};
  return launch_result(launch_w8a8(Epi::Store, a, S(stream)), "nc_w8a8_gemv");
}

nc_status nc_w8a8_gemv_b32(const float* x, const void* gamma, float eps, const int8_t* Wq,
                           const float* w_scale, const void* bias, int B, int K, int N, float* y,
                           int8_t* xq_out, float* sx_out, int32_t* acc_out, void* stream) {
  NC_CHECK(x && Wq && w_scale && y, NC_ERR_INVALID_ARGUMENT, "null pointer");
  NC_CHECK(aligned16(Wq) && aligned(x, 4) && aligned(gamma, 2) && aligned(w_scale, 4) &&
               aligned(bias, 2) && aligned(y, 4) && aligned(sx_out, 4) && aligned(acc_out, 4),
           NC_ERR_INVALID_ARGUMENT,
           "Wq must be 16-byte aligned, fp32 and int32 pointers 4-byte, bf16 2-byte");
  NC_CHECK(B >= 1 && B <= 8, NC_ERR_SHAPE, "batch %d outside [1, 8]", B);
  NC_CHECK(K >= 32 && K % 32 == 0, NC_ERR_SHAPE, "K = %d must be a positive multiple of 32", K);
  NC_CHECK(N >= 1, NC_ERR_SHAPE, "N must be positive");
  NC_CHECK(w8a8_b32_smem_bytes(B, K) + 4096 <= (size_t)max_smem_optin(), NC_ERR_SHAPE,
           "K = %d is too long to keep the batch's codes in shared memory", K);
  W8BArgs a{x, static_cast<const uint16_t*>(gamma), eps, Wq, w_scale,
            static_cast<const uint16_t*>(bias), B, K, N, y, xq_out, sx_out, acc_out};
  return launch_result(launch_w8a8_b32(Epi::Store, a, S(stream)), "nc_w8a8_gemv_b32");
}

nc_status nc_int4_gemv(const float* x, const void* gamma, float eps, const uint8_t* Wq,
                       const float* scales, int group, int B, int K, int N, float* y,
                       void* stream) {
  NC_CHECK(x && Wq && scales && y, NC_ERR_INVALID_ARGUMENT, "null pointer");
  NC_CHECK(aligned(x, 4) && aligned(gamma, 2) && aligned16(Wq) && aligned(scales, 4) &&
               aligned(y, 4),
           NC_ERR_INVALID_ARGUMENT,
           "Wq must be 16-byte aligned, x, scales and y 4-byte, gamma 2-byte");
  NC_CHECK(B >= 1 && B <= 8, NC_ERR_SHAPE, "batch %d outside [1, 8]", B);
  NC_CHECK(group == 32 || group == 64 || group == 128, NC_ERR_SHAPE,
           "group = %d must be 32, 64 or 128", group);
  NC_CHECK(K >= group && K % group == 0, NC_ERR_SHAPE, "K = %d must be a positive multiple of group %d",
           K, group);
  NC_CHECK(N >= 1, NC_ERR_SHAPE, "N must be positive");
  NC_CHECK(int4_smem_bytes(B, K) + 4096 <= (size_t)max_smem_optin(), NC_ERR_SHAPE,
           "K = %d is too long to keep the batch's activations in shared memory", K);
  Int4Args a{x, static_cast<const uint16_t*>(gamma), eps, Wq, scales, group, B, K, N, y};
  return launch_result(launch_int4_gemv(Epi::Store, a, S(stream)), "nc_int4_gemv");
}

size_t nc_prefill_scratch_bytes(const nc_model* m, int T) {
  if (!m || T < 1) return 0;
  return prefill_scratch_bytes(M(m), T);
}

nc_status nc_prefill(nc_model* m, int seq, int T, const int32_t* tokens_dev, int start_pos,
                     const nc_kv_cache* kv, float* logits_dev, int32_t* next_dev, void* scratch,
                     size_t scratch_bytes, void* stream) {
  return prefill(M(m), seq, T, tokens_dev, start_pos, kv, logits_dev, next_dev, scratch,
                 scratch_bytes, S(stream));
}

size_t nc_sample_scratch_bytes(int B, int V) {
  if (B < 1 || V < 1) return 0;
  return sample_scratch_bytes(B, V);
}

nc_status nc_sample(const float* logits, int B, int V, float temperature, int top_k, float top_p,
                    const double* u, int32_t* tokens, int32_t* kept, void* scratch,
                    size_t scratch_bytes, void* stream) {
  NC_CHECK(logits && tokens, NC_ERR_INVALID_ARGUMENT, "logits and tokens must not be NULL");
  NC_CHECK(aligned(logits, 4) && aligned(tokens, 4) && aligned(kept, 4) && aligned(u, 8),
           NC_ERR_INVALID_ARGUMENT, "logits, tokens and kept must be 4-byte aligned, u 8-byte");
  NC_CHECK(B >= 1 && B <= 65535, NC_ERR_SHAPE, "batch %d outside [1, 65535]", B);
  NC_CHECK(V >= 1 && V <= (1 << 24), NC_ERR_SHAPE, "V = %d outside [1, 2^24]", V);
  NC_CHECK(temperature >= 0.f && temperature <= FLT_MAX, NC_ERR_INVALID_ARGUMENT,
           "temperature must be finite and >= 0");
  NC_CHECK(top_k >= 0, NC_ERR_INVALID_ARGUMENT, "top_k = %d must be >= 0 (0: off)", top_k);
  NC_CHECK(top_p > 0.f && top_p <= 1.f, NC_ERR_INVALID_ARGUMENT,
           "top_p must lie in (0, 1] (1: off)");
  if (temperature > 0.f) {
    NC_CHECK(u, NC_ERR_INVALID_ARGUMENT, "u must not be NULL when temperature > 0");
    NC_CHECK(scratch && aligned16(scratch), NC_ERR_INVALID_ARGUMENT,
             "scratch must be a 16-byte aligned device buffer when temperature > 0");
    const size_t need = sample_scratch_bytes(B, V);
    NC_CHECK(scratch_bytes >= need, NC_ERR_CAPACITY, "scratch holds %zu bytes, %zu needed",
             scratch_bytes, need);
  }
  return launch_result(launch_sample(logits, B, V, temperature, top_k, top_p, u, tokens, kept,
                                     scratch, S(stream)),
                       "nc_sample");
}

}  // extern "C"
