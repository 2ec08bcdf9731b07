/*
 * oracle.h -- CPU oracle for the single-token decode step of a Qwen2-style
 * decoder (pre-norm blocks, grouped-query attention with RoPE, SwiGLU MLP,
 * tied or untied LM head, greedy argmax).
 *
 * TEST INFRASTRUCTURE. This library defines what the decode step computes, in
 * plain, slow loops: every sum runs in index order, nothing is blocked, fused
 * or reordered. Only the tests, the smoke check and the benchmark's CPU
 * baseline may load it. It shares no code, header or table with the CUDA
 * library and never links it.
 *
 * Sources (web pages; cited by title and section):
 *   nanoinfer  -- "Model architecture" (pre-norm block, GQA repeat, RoPE
 *                 half-split, causal mask j <= i, tied embeddings, QKV bias
 *                 without o-proj bias, final norm before the head),
 *                 "KV cache" (rotate once on insert, positions continue past
 *                 the cache), "Sampling" (temperature 0 is argmax),
 *                 "Quantization" (symmetric per-channel int8, range
 *                 [-127, 127], round half away from zero), "Weights"
 *                 (bf16 widen by shift, narrow by round-half-to-even),
 *                 "Phase 8" sigmoid form e = exp(-|x|).
 *   nanocompile -- "Phase 1" (mean square is a sum then a divide, the norm
 *                 takes sqrt then reciprocal, RoPE angles are f32 products).
 *   Tang       -- section 2.2 (online softmax and arg-max are monoids; the
 *                 oracle uses the plain two-pass softmax they must equal).
 *
 * Readings where the pages are silent (each listed in the design notes):
 *   attention scale 1/sqrt(D); RMSNorm (x * r) * g with r = 1/sqrt(ss/n + eps);
 *   inv_freq[i] = float(1 / theta^(2i/D)) computed in double; angle is the
 *   fp32 product float(pos) * inv_freq[i]; the cache stores K and V in fp32
 *   (nanoinfer's cache), or in bf16 when asked (rounded to nearest even on
 *   store, in the cached and the uncached forward alike); per-head q/k
 *   RMSNorm (8B shape) is applied before RoPE with gains [D] shared by all
 *   heads; argmax takes the lowest index on ties.
 *
 * Precision: every function exists as _f32 (the oracle) and _f64 (the same
 * definition in double, used to show the oracle's own rounding is far below
 * the parity tolerance). Weights, biases, gains and the KV cache are bf16
 * bit patterns (uint16_t); activations are REAL.
 */
#ifndef NC_ORACLE_H
#define NC_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int hidden;          /* H */
  int n_q_heads;       /* Hq */
  int n_kv_heads;      /* Hkv; query head h reads kv head h / (Hq/Hkv) */
  int head_dim;        /* D (even) */
  int ffn;             /* F */
  int n_layers;        /* L */
  int vocab;           /* V */
  double rms_eps;
  double rope_theta;
  int qkv_bias;        /* q, k, v projections carry a bias */
  int qk_norm;         /* per-head RMSNorm of q and k before RoPE */
  int tie_embeddings;  /* logits = embed @ x (no separate head) */
} orc_config;

/* One block. Matrices are [out, in] row-major bf16. Pointers that a shape
 * does not use are NULL. The q8_* / s_* fields hold the W8A8 form of the
 * seven projections (int8 rows and one fp32 scale per output row). */
typedef struct {
  const uint16_t *wq, *wk, *wv, *bq, *bk, *bv, *wo, *wg, *wu, *wd;
  const uint16_t *g_attn, *g_mlp, *g_q, *g_k;
  const int8_t *q8_wq, *q8_wk, *q8_wv, *q8_wo, *q8_wg, *q8_wu, *q8_wd;
  const float *s_wq, *s_wk, *s_wv, *s_wo, *s_wg, *s_wu, *s_wd;
  /* INT4 form (orc_model.int4_group > 0): packed codes [out, in / 2], two a
   * byte with the even index in the low nibble, and fp32 scales
   * [out, in / group] */
  const uint8_t *q4_wq, *q4_wk, *q4_wv, *q4_wo, *q4_wg, *q4_wu, *q4_wd;
  const float *s4_wq, *s4_wk, *s4_wv, *s4_wo, *s4_wg, *s4_wu, *s4_wd;
} orc_layer;

typedef struct {
  orc_config cfg;
  const uint16_t *embed;    /* [V, H] */
  const uint16_t *lm_head;  /* [V, H]; NULL when tied */
  const uint16_t *g_final;  /* [H] */
  const orc_layer *layers;  /* [L] */
  int w8a8;                 /* projections use the int8 fields */
  int act_block;            /* w8a8: 0 = one activation scale per token; n > 0 = one per
                               block of n values (nanoinfer, INT8 activation section:
                               "one per 32") */
  const int8_t* q8_embed;   /* [V, H] int8 rows with one fp32 scale each (s_embed), or
                               NULL: the embedding, and the tied head, stored int8 */
  const float* s_embed;     /* [V] */
  int int4_group;           /* > 0: the projections use the INT4 fields, one scale per
                               group of this many weights (nanoinfer "Quantization") */
} orc_model;

/* Logical KV cache: k, v are [L][B][Hkv][max_ctx][D] of fp32 (bf16 = 0, the
 * nanoinfer cache: "24 KiB per token at fp32") or of bf16 bit patterns
 * (bf16 = 1, rounded to nearest even when stored). */
typedef struct {
  int batch;
  int max_ctx;
  int bf16;
  void *k;
  void *v;
} orc_kv;

/* ---- bf16 ---- */
float orc_bf16_to_f32(uint16_t b);
uint16_t orc_f32_to_bf16(float f);          /* round half to even; NaN -> 0x7FC0 */
void orc_bf16_to_f32_n(const uint16_t* b, float* out, long n);
void orc_f32_to_bf16_n(const float* f, uint16_t* out, long n);

/* ---- int8 (W8A8) ---- */
/* Symmetric per-vector quantisation: s = amax / 127, q = clamp(round_half_away(v / s)).
 * amax = 0 gives s = 0 and q = 0. Returns s. */
float orc_quantize_row_f32(const float* v, int n, int8_t* q);
/* Per-output-row weight quantisation of a bf16 [N, K] matrix. */
void orc_quantize_weight_f32(const uint16_t* w, int n, int k, int8_t* q, float* scale);
/* acc[j] = sum_k W[j,k] * x[k] with an int64 accumulator; returns 0, or -1 if
 * some sum leaves the int32 range. */
int orc_matvec_i8(const int8_t* w, int n, int k, const int8_t* x, int32_t* acc);

/* ---- argmax: lowest index on ties; -1 if any NaN ---- */
int orc_argmax_f32(const float* v, int n);
int orc_argmax_f64(const double* v, int n);

/* ---- RoPE frequency table (float(1 / theta^(2i/D)), i < D/2) ---- */
void orc_rope_inv_freq(double theta, int d, float* inv_freq);

#define ORC_DECLARE(REAL, SFX)                                                        \
  void orc_rmsnorm_##SFX(const REAL* x, int n, const uint16_t* g, double eps, REAL* out); \
  void orc_matvec_bf16_##SFX(const uint16_t* w, int n, int k, const REAL* x, REAL* y);  \
  void orc_rope_##SFX(REAL* v, int d, int pos, double theta);                           \
  void orc_rope_interleaved_##SFX(REAL* v, int d, int pos, double theta);               \
  REAL orc_silu_##SFX(REAL x);                                                          \
  void orc_softmax_##SFX(const REAL* s, int n, REAL* p);                                \
  void orc_attention_head_##SFX(const REAL* q, const void* k, const void* v, int kv_bf16, \
                                int n_pos, int d, REAL* out);                            \
  void orc_linear_w8a8_##SFX(const int8_t* w, const float* sw, const uint16_t* bias,     \
                             int n, int k, const REAL* x, REAL* y);                       \
  void orc_linear_w8a8_blocked_##SFX(const int8_t* w, const float* sw,                   \
                                     const uint16_t* bias, int n, int k, int block,       \
                                     const REAL* x, REAL* y);                             \
  void orc_linear_int4_##SFX(const uint8_t* w4, const float* s4, int group,              \
                             const uint16_t* bias, int n, int k, const REAL* x, REAL* y); \
  void orc_block_decode_##SFX(const orc_model* m, int layer, orc_kv* kv, int b, int pos,  \
                              REAL* x);                                                  \
  int orc_decode_step_##SFX(const orc_model* m, orc_kv* kv, int batch,                   \
                            const int32_t* tokens, const int32_t* positions,              \
                            REAL* logits, int32_t* next, REAL* hidden);                   \
  int orc_forward_chunk_##SFX(const orc_model* m, orc_kv* kv, int b, int n,               \
                              const int32_t* tokens, int start_pos, REAL* logits);        \
  int orc_forward_full_##SFX(const orc_model* m, int t, const int32_t* tokens,           \
                             int kv_bf16, REAL* logits);

ORC_DECLARE(float, f32)
ORC_DECLARE(double, f64)

void orc_set_threads(int n);
int orc_get_threads(void);

#ifdef __cplusplus
}
#endif
#endif
