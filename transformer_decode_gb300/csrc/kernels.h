// kernels.h -- launch interfaces of libnc's kernels (host side, internal).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "nc_internal.cuh"

namespace nc {

int num_sms();  // SM count of the current device (cached)

// Launch a stage kernel with programmatic stream serialisation: it may begin
// while the previous kernel in the stream drains, so it must call pdl_wait()
// before it touches memory that earlier kernels write. NC_PDL=0 in the
// environment launches every kernel the ordinary way.
bool pdl_enabled();
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ------------------------------------------------------------ streaming GEMV
enum class Epi : int { Store = 0, Residual = 1, SwiGLU = 2 };

struct GemvArgs {
  const float* x;         // [B, K] activations
  const uint16_t* gamma;  // [K] RMSNorm gain, or null (no norm)
  float eps;
  const uint16_t* W;      // [N, K] bf16; SwiGLU: [2N, K] (gate rows, then up rows)
  const uint16_t* bias;   // [N] bf16 or null (Store only)
  int B, K, N;
  float* y;               // [B, N]; Residual: updated in place
};
cudaError_t launch_gemv(Epi epi, const GemvArgs& a, cudaStream_t s);
// Batch 9..16 on the tensor cores (gemm16.cu); launch_gemv and launch_lm_head
// dispatch there when these report support.
bool gemm16_supported(Epi epi, int B, int K);
cudaError_t launch_gemm16(Epi epi, const GemvArgs& a, cudaStream_t s);

// Dense tiles on the tensor cores (umma.cu, tcgen05): y[t, n] = W[n, :] .
// xn[t, :] for T tokens, xn = rmsnorm(x[t]) * gamma when gamma is set. The
// activations are first written to xb as bf16 hi / lo planes.
struct UmmaArgs {
  const float* x;          // [T, K] fp32
  const uint16_t* gamma;   // [K] or null
  float eps;
  const uint16_t* W;       // [N, K] bf16; SwiGLU: [2N, K] (gate rows, then up rows)
  const uint16_t* bias;    // [N] or null (Store)
  int T, K, N;
  float* y;                // [T, ldy]; Residual: updated in place
  int ldy;
  uint16_t* xb;            // scratch of umma_act_bytes(T, K) bytes, 1024-byte aligned
  // LM head (Store with lm): per-CTA arg-max keys [T][ceil(N / 128)], the
  // ticket, and what the last CTA writes
  bool lm = false;
  unsigned long long* part = nullptr;
  unsigned int* ticket = nullptr;
  int32_t* next = nullptr;
  int* status = nullptr;
  int32_t* advance_tokens = nullptr;
  int32_t* advance_positions = nullptr;
};
bool umma_supported(int K);
int umma_tokens_per_tile(int T);
size_t umma_act_bytes(int T, int K);
cudaError_t launch_umma(Epi epi, const UmmaArgs& a, cudaStream_t s);

// LM head: logits = W rmsnorm(x) and the greedy token per sequence.
struct LmHeadArgs {
  const float* x;
  const uint16_t* gamma;
  float eps;
  const uint16_t* W;            // [V, K]
  int B, K, V;
  float* logits;                // [B, V]
  int32_t* next;                // [B] or null
  unsigned long long* part;     // [B, grid] arg-max partial keys (workspace)
  unsigned int* ticket;         // zero on entry; the last block resets it
  int* status;                  // device status word
  int32_t* advance_tokens;      // non-null: tokens[b] = greedy token after the step
  int32_t* advance_positions;   // non-null: positions[b] += 1 after the step
};
int lm_head_grid();
cudaError_t launch_lm_head(const LmHeadArgs& a, cudaStream_t s);
bool lm_head16_supported(int B, int K);
cudaError_t launch_lm_head16(const LmHeadArgs& a, cudaStream_t s);

// ------------------------------------------------------------ attention
struct RopeArgs {
  const float* qkv;         // [B, (Hq + 2 Hkv) D]
  const int32_t* positions; // [B]
  const float* inv_freq;    // [D/2]
  const uint16_t* g_q;      // [D] or null
  const uint16_t* g_k;      // [D] or null
  float eps;
  int B, Hq, Hkv, D, layer;
  float* q_out;             // [B, Hq D]
  KVView kv;
  int* status;              // device status word (NC_ERR_POSITION on a bad slot)
  // Prefill: seq >= 0 makes every row b a token of cache sequence `seq` at
  // position pos0 + b (positions is then unused).
  int seq = -1;
  int pos0 = 0;
};
cudaError_t launch_rope_qkv(const RopeArgs& a, cudaStream_t s);

// Causal attention of a prefill chunk (prefill.cu): T tokens of cache
// sequence `seq` at positions start .. start + T - 1 (their K/V already in the
// cache), each over slots 0 .. its own position; online softmax over tiles
// of 64 positions (Tang section 2.2).
struct PrefillAttnArgs {
  const float* q;           // [T, Hq D] rotated
  float* out;               // [T, Hq D]
  int T, start, seq, layer, Hq, Hkv, D;
  KVView kv;
  int pair = 0;             // set by the launcher: a CTA takes token blocks x and n - 1 - x
};
size_t prefill_attn_smem(int D);
cudaError_t launch_prefill_attn(const PrefillAttnArgs& a, cudaStream_t s);

struct AttnArgs {
  const float* q;           // [B, Hq D] rotated
  const int32_t* positions; // [B]
  int B, Hq, Hkv, D, layer, splits;
  float* part;              // [B, Hq, splits, D + 2] (m, l, acc[D])
  float* out;               // [B, Hq D]
  KVView kv;
  int* status;              // device status word (NC_ERR_POSITION on a bad slot)
  unsigned int* tickets;    // [B, Hkv], zero between launches (the merging CTA resets its own)
  // Non-null: RoPE (+ q/k norm) and the K/V append run inside the attention
  // launch, from the projections [B, (Hq + 2 Hkv) D]; q is then unused.
  const float* qkv = nullptr;
  const float* inv_freq = nullptr;  // [D/2]
  const uint16_t* g_q = nullptr;    // [D] or null
  const uint16_t* g_k = nullptr;    // [D] or null
  float eps = 0.f;
};
int attn_splits(int B, int Hkv, int D, bool kv16, int max_ctx);
size_t attn_part_floats(int B, int Hq, int D, int splits);
cudaError_t launch_attn(const AttnArgs& a, cudaStream_t s);

// ------------------------------------------------------------ W8A8
struct W8Args {
  const float* x;
  const uint16_t* gamma;
  float eps;
  const int8_t* Wq;       // [N, K]
  const float* w_scale;   // [N]
  const uint16_t* bias;   // [N] or null
  int B, K, N;
  float* y;               // [B, N] (Residual: in place)
  int8_t* xq_out;         // [B, K] or null
  float* sx_out;          // [B] or null
  int32_t* acc_out;       // [B, N] or null
};
cudaError_t launch_w8a8(Epi epi, const W8Args& a, cudaStream_t s);
cudaError_t launch_quantize_weight(const uint16_t* W, int N, int K, int8_t* q, float* scale,
                                   cudaStream_t s);

// W8A8 with activations quantised in blocks of 32 (w8a8_blocks.cu)
struct W8BArgs {
  const float* x;
  const uint16_t* gamma;
  float eps;
  const int8_t* Wq;       // [N, K]
  const float* w_scale;   // [N]
  const uint16_t* bias;   // [N] or null
  int B, K, N;
  float* y;               // [B, N]
  int8_t* xq_out;         // [B, K] or null
  float* sx_out;          // [B, K / 32] or null
  int32_t* acc_out;       // [B, R N, K / 32] or null (R = 2 for SwiGLU)
  // non-null part: the LM head -- y are the logits, and the arg-max of each
  // sequence goes to next (and, when non-null, the greedy feedback)
  unsigned long long* part = nullptr;  // [B, lm_head_grid()] (workspace)
  unsigned int* ticket = nullptr;      // zero on entry; the last CTA resets it
  int32_t* next = nullptr;
  int* status = nullptr;
  int32_t* advance_tokens = nullptr;
  int32_t* advance_positions = nullptr;
};
size_t w8a8_b32_smem_bytes(int B, int K);
cudaError_t launch_w8a8_b32(Epi epi, const W8BArgs& a, cudaStream_t s);
cudaError_t launch_embed_i8(const int8_t* q, const float* sc, const int32_t* tokens, int B, int H,
                            int V, float* x, int* status, cudaStream_t s);
// ------------------------------------------------------------ INT4 weights
struct Int4Args {
  const float* x;         // [B, K]
  const uint16_t* gamma;  // [K] RMSNorm gain, or null (no norm)
  float eps;
  const uint8_t* Wq;      // [N, K / 2]: two codes a byte, the even index in the low nibble
  const float* scales;    // [N, K / group]
  int group, B, K, N;
  float* y;               // [B, N] (Residual: in place); SwiGLU: Wq and scales hold 2N rows
  const uint16_t* bias = nullptr;  // [N] bf16 or null (Store only)
};
size_t int4_smem_bytes(int B, int K);  // the activations kept in shared memory
cudaError_t launch_int4_gemv(Epi epi, const Int4Args& a, cudaStream_t s);
cudaError_t launch_quantize_int4(const uint16_t* W, int N, int K, int group, uint8_t* q,
                                 float* sc, cudaStream_t s);

// ------------------------------------------------------------ sampling
// Scratch of nc_sample: per row five arrays of V rounded up to 64 words.
size_t sample_scratch_bytes(int B, int V);
cudaError_t launch_sample(const float* logits, int B, int V, float temperature, int top_k,
                          float top_p, const double* u, int32_t* tokens, int32_t* kept,
                          void* scratch, cudaStream_t s);

// ------------------------------------------------------------ misc
// x[b] = widen(E[tokens[b]]); a token outside [0, V) reads row 0 and sets *status.
cudaError_t launch_embed(const uint16_t* E, const int32_t* tokens, int B, int H, int V, float* x,
                         int* status, cudaStream_t s);

// Raise a kernel's dynamic shared memory limit to the device's opt-in maximum,
// once per kernel (outside any stream capture on the first call).
int max_smem_optin();
// The limit is the opt-in maximum less the kernel's static shared memory.
template <auto Kern>
cudaError_t ensure_smem() {
  static const cudaError_t e = [] {
    cudaFuncAttributes fa;
    cudaError_t r = cudaFuncGetAttributes(&fa, Kern);
    if (r != cudaSuccess) return r;
    return cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                max_smem_optin() - (int)fa.sharedSizeBytes);
  }();
  return e;
}

}  // namespace nc
