/*
 * oracle_impl.h -- the oracle's definitions, written once against REAL and
 * included twice by oracle.c (REAL = float, SFX = f32; REAL = double,
 * SFX = f64). TEST INFRASTRUCTURE; see oracle.h for sources and readings.
 *
 * Every reduction below is a plain loop in index order. OpenMP only splits
 * independent outputs (rows of a matrix-vector product, heads of attention),
 * so the bits do not depend on the thread count.
 */
#define CAT2(a, b) a##_##b
#define CAT(a, b) CAT2(a, b)
#define F(name) CAT(name, SFX)

static REAL F(widen)(uint16_t b) { return (REAL)orc_bf16_to_f32(b); }

static REAL F(sqrtr)(REAL x) {
  return sizeof(REAL) == sizeof(float) ? (REAL)sqrtf((float)x) : (REAL)sqrt((double)x);
}

static uint16_t F(narrow)(REAL v) { return orc_f32_to_bf16((float)v); }

/* Element i of a K/V array stored as bf16 (kv_bf16 = 1) or fp32. */
static REAL F(kv_get)(const void* p, int kv_bf16, long i) {
  return kv_bf16 ? F(widen)(((const uint16_t*)p)[i]) : (REAL)((const float*)p)[i];
}
static void F(kv_put)(void* p, int kv_bf16, long i, REAL v) {
  if (kv_bf16)
    ((uint16_t*)p)[i] = F(narrow)(v);
  else
    ((float*)p)[i] = (float)v;
}

/* nanocompile "Phase 1": the mean square is a sum then a divide; the norm is
 * a sqrt then a reciprocal; the gain multiplies the normalised value. */
void F(orc_rmsnorm)(const REAL* x, int n, const uint16_t* g, double eps, REAL* out) {
  REAL ss = 0;
  for (int i = 0; i < n; ++i) ss += x[i] * x[i];
  REAL ms = ss / (REAL)n;
  REAL r = (REAL)1 / F(sqrtr)(ms + (REAL)eps);
  for (int i = 0; i < n; ++i) out[i] = (x[i] * r) * F(widen)(g[i]);
}

/* y[j] = sum_k W[j, k] * x[k], W bf16 [n, k] row-major (x @ W.T). */
void F(orc_matvec_bf16)(const uint16_t* w, int n, int k, const REAL* x, REAL* y) {
#pragma omp parallel for schedule(static)
  for (int j = 0; j < n; ++j) {
    const uint16_t* row = w + (long)j * k;
    REAL acc = 0;
    for (int i = 0; i < k; ++i) acc += F(widen)(row[i]) * x[i];
    y[j] = acc;
  }
}

static REAL F(cosr)(float a) {
  return sizeof(REAL) == sizeof(float) ? (REAL)cosf(a) : (REAL)cos((double)a);
}
static REAL F(sinr)(float a) {
  return sizeof(REAL) == sizeof(float) ? (REAL)sinf(a) : (REAL)sin((double)a);
}

/* nanoinfer "Model architecture": half-split RoPE pairs component i with
 * i + d/2. The angle is the fp32 product float(pos) * inv_freq[i]
 * (nanocompile "Phase 1": RoPE's angles are f32 products). */
void F(orc_rope)(REAL* v, int d, int pos, double theta) {
  float inv_freq[1024];
  orc_rope_inv_freq(theta, d, inv_freq);
  int half = d / 2;
  for (int i = 0; i < half; ++i) {
    float angle = (float)pos * inv_freq[i];
    REAL c = F(cosr)(angle), s = F(sinr)(angle);
    REAL a = v[i], b = v[i + half];
    v[i] = a * c - b * s;
    v[i + half] = b * c + a * s;
  }
}

/* The interleaved convention (pairs 2i, 2i+1). Not used by the model: it
 * exists so a test can show the two conventions differ. */
void F(orc_rope_interleaved)(REAL* v, int d, int pos, double theta) {
  float inv_freq[1024];
  orc_rope_inv_freq(theta, d, inv_freq);
  for (int i = 0; i < d / 2; ++i) {
    float angle = (float)pos * inv_freq[i];
    REAL c = F(cosr)(angle), s = F(sinr)(angle);
    REAL a = v[2 * i], b = v[2 * i + 1];
    v[2 * i] = a * c - b * s;
    v[2 * i + 1] = b * c + a * s;
  }
}

static REAL F(expr)(REAL x) {
  return sizeof(REAL) == sizeof(float) ? (REAL)expf((float)x) : (REAL)exp((double)x);
}

/* nanoinfer "Phase 8": both halves of the sigmoid share e = exp(-|x|);
 * sigmoid is 1/(1+e) for x >= 0 and e/(1+e) otherwise. silu = x * sigmoid. */
REAL F(orc_silu)(REAL x) {
  REAL e = F(expr)(-(x < 0 ? -x : x));
  REAL sig = x >= 0 ? (REAL)1 / ((REAL)1 + e) : e / ((REAL)1 + e);
  return x * sig;
}

/* Two-pass softmax: max, then exp and sum, then divide. */
void F(orc_softmax)(const REAL* s, int n, REAL* p) {
  REAL m = s[0];
  for (int i = 1; i < n; ++i)
    if (s[i] > m) m = s[i];
  REAL l = 0;
  for (int i = 0; i < n; ++i) {
    p[i] = F(expr)(s[i] - m);
    l += p[i];
  }
  for (int i = 0; i < n; ++i) p[i] = p[i] / l;
}

/* One query head against n_pos cached keys/values ([n_pos, d], bf16 or fp32):
 * s_t = (q . k_t) / sqrt(d), p = softmax(s), out = sum_t p_t v_t. */
void F(orc_attention_head)(const REAL* q, const void* k, const void* v, int kv_bf16,
                           int n_pos, int d, REAL* out) {
  REAL* s = (REAL*)malloc(sizeof(REAL) * (size_t)n_pos);
  REAL* p = (REAL*)malloc(sizeof(REAL) * (size_t)n_pos);
  REAL scale = (REAL)1 / F(sqrtr)((REAL)d);
  for (int t = 0; t < n_pos; ++t) {
    REAL dot = 0;
    for (int i = 0; i < d; ++i) dot += q[i] * F(kv_get)(k, kv_bf16, (long)t * d + i);
    s[t] = dot * scale;
  }
  F(orc_softmax)(s, n_pos, p);
  for (int i = 0; i < d; ++i) {
    REAL acc = 0;
    for (int t = 0; t < n_pos; ++t) acc += p[t] * F(kv_get)(v, kv_bf16, (long)t * d + i);
    out[i] = acc;
  }
  free(s);
  free(p);
}

/* W8A8 linear (nanoinfer "Quantization"; per-token activation scale):
 * quantise x, integer dot products, y[j] = float(acc[j]) * (sw[j] * sx) (+ bias). */
void F(orc_linear_w8a8)(const int8_t* w, const float* sw, const uint16_t* bias, int n,
                        int k, const REAL* x, REAL* y) {
  float* xf = (float*)malloc(sizeof(float) * (size_t)k);
  int8_t* xq = (int8_t*)malloc((size_t)k);
  int32_t* acc = (int32_t*)malloc(sizeof(int32_t) * (size_t)n);
  for (int i = 0; i < k; ++i) xf[i] = (float)x[i];
  float sx = orc_quantize_row_f32(xf, k, xq);
  if (orc_matvec_i8(w, n, k, xq, acc) != 0) abort();
  for (int j = 0; j < n; ++j) {
    REAL yj = (REAL)acc[j] * ((REAL)sw[j] * (REAL)sx);
    if (bias) yj += F(widen)(bias[j]);
    y[j] = yj;
  }
  free(xf);
  free(xq);
  free(acc);
}

/* W8A8 with activations in blocks of `block` values (nanoinfer, INT8
 * activation section: one scale per 32, so an outlier widens only its own
 * block): each block is quantised as a row is, acc[j, b] is the int32 sum of
 * block b (int64, checked), and y[j] = sum_b float(acc[j, b]) * (sw[j] * sx[b])
 * in block order, then + bias. A ragged last block is shorter. */
void F(orc_linear_w8a8_blocked)(const int8_t* w, const float* sw, const uint16_t* bias, int n,
                                int k, int block, const REAL* x, REAL* y) {
  const int nb = (k + block - 1) / block;
  float* xf = (float*)malloc(sizeof(float) * (size_t)k);
  int8_t* xq = (int8_t*)malloc((size_t)k);
  float* sx = (float*)malloc(sizeof(float) * (size_t)nb);
  for (int i = 0; i < k; ++i) xf[i] = (float)x[i];
  for (int b = 0; b < nb; ++b) {
    const int len = k - b * block < block ? k - b * block : block;
    sx[b] = orc_quantize_row_f32(xf + (long)b * block, len, xq + (long)b * block);
  }
  int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
  for (int j = 0; j < n; ++j) {
    REAL t = 0;
    for (int b = 0; b < nb; ++b) {
      const int i1 = (b + 1) * block < k ? (b + 1) * block : k;
      int64_t acc = 0;
      for (int i = b * block; i < i1; ++i) acc += (int64_t)w[(long)j * k + i] * (int64_t)xq[i];
      if (acc > INT32_MAX || acc < INT32_MIN) bad = 1;
      t += (REAL)(int32_t)acc * ((REAL)sw[j] * (REAL)sx[b]);
    }
    if (bias) t += F(widen)(bias[j]);
    y[j] = t;
  }
  if (bad) abort();
  free(xf);
  free(xq);
  free(sx);
}

/* INT4 group-wise weights (nanoinfer "Quantization": fifteen symmetric levels,
 * one fp32 scale per group of `group` weights of a row; two codes a byte, the
 * even index in the low nibble): y[j] = sum_i float(q[j, i] * s[j, i / group])
 * * x[i] in index order (the dequantised weight rounded to fp32, as in the
 * page's quantise-dequantise evaluation), then + bias. */
void F(orc_linear_int4)(const uint8_t* w4, const float* s4, int group, const uint16_t* bias,
                        int n, int k, const REAL* x, REAL* y) {
  const int ng = (k + group - 1) / group;
#pragma omp parallel for schedule(static)
  for (int j = 0; j < n; ++j) {
    REAL t = 0;
    for (int i = 0; i < k; ++i) {
      const uint8_t byte = w4[(long)j * (k / 2) + i / 2];
      int q = (i & 1) ? (byte >> 4) : (byte & 0xF);
      if (q >= 8) q -= 16;
      const float wd = (float)q * s4[(long)j * ng + i / group];
      t += (REAL)wd * x[i];
    }
    if (bias) t += F(widen)(bias[j]);
    y[j] = t;
  }
}

/* The W8A8 product in the model's activation mode. */
static void F(linear_i8)(const orc_model* m, const int8_t* w8, const float* sw,
                         const uint16_t* bias, int n, int k, const REAL* x, REAL* y) {
  if (m->act_block > 0)
    F(orc_linear_w8a8_blocked)(w8, sw, bias, n, k, m->act_block, x, y);
  else
    F(orc_linear_w8a8)(w8, sw, bias, n, k, x, y);
}

/* The residual row of a token: the bf16 embedding widened, or an int8 row
 * times its scale (the product rounded to fp32). */
static void F(embed_row)(const orc_model* m, int tok, REAL* x) {
  const int H = m->cfg.hidden;
  if (m->q8_embed) {
    for (int i = 0; i < H; ++i)
      x[i] = (REAL)((float)m->q8_embed[(long)tok * H + i] * m->s_embed[tok]);
    return;
  }
  for (int i = 0; i < H; ++i) x[i] = F(widen)(m->embed[(long)tok * H + i]);
}

/* y = W x + b for one of a layer's projections, bf16 or W8A8. */
static void F(project)(const orc_model* m, const uint16_t* w, const int8_t* w8,
                       const float* sw, const uint8_t* w4, const float* s4,
                       const uint16_t* bias, int n, int k, const REAL* x, REAL* y) {
  if (m->w8a8) {
    F(linear_i8)(m, w8, sw, bias, n, k, x, y);
    return;
  }
  if (m->int4_group > 0) {
    F(orc_linear_int4)(w4, s4, m->int4_group, bias, n, k, x, y);
    return;
  }
  F(orc_matvec_bf16)(w, n, k, x, y);
  if (bias)
    for (int j = 0; j < n; ++j) y[j] += F(widen)(bias[j]);
}

static long F(kv_off)(const orc_config* c, const orc_kv* kv, int layer, int b, int g) {
  return ((((long)layer * kv->batch + b) * c->n_kv_heads + g) * kv->max_ctx) * c->head_dim;
}

/* q, k, v of one token at one layer: norm, projections, optional per-head
 * q/k norm, RoPE at pos (nanoinfer "Model architecture", "KV cache"). */
static void F(qkv_token)(const orc_model* m, int layer, const REAL* x, int pos, REAL* q,
                         REAL* k, REAL* v) {
  const orc_config* c = &m->cfg;
  const orc_layer* w = &m->layers[layer];
  int H = c->hidden, D = c->head_dim, qd = c->n_q_heads * D, kd = c->n_kv_heads * D;
  REAL* n = (REAL*)malloc(sizeof(REAL) * (size_t)H);
  F(orc_rmsnorm)(x, H, w->g_attn, c->rms_eps, n);
  F(project)(m, w->wq, w->q8_wq, w->s_wq, w->q4_wq, w->s4_wq, c->qkv_bias ? w->bq : NULL, qd, H, n, q);
  F(project)(m, w->wk, w->q8_wk, w->s_wk, w->q4_wk, w->s4_wk, c->qkv_bias ? w->bk : NULL, kd, H, n, k);
  F(project)(m, w->wv, w->q8_wv, w->s_wv, w->q4_wv, w->s4_wv, c->qkv_bias ? w->bv : NULL, kd, H, n, v);
  if (c->qk_norm) {
    for (int h = 0; h < c->n_q_heads; ++h) F(orc_rmsnorm)(q + h * D, D, w->g_q, c->rms_eps, q + h * D);
    for (int h = 0; h < c->n_kv_heads; ++h) F(orc_rmsnorm)(k + h * D, D, w->g_k, c->rms_eps, k + h * D);
  }
  for (int h = 0; h < c->n_q_heads; ++h) F(orc_rope)(q + h * D, D, pos, c->rope_theta);
  for (int h = 0; h < c->n_kv_heads; ++h) F(orc_rope)(k + h * D, D, pos, c->rope_theta);
  free(n);
}

/* x += W_o a; then x += W_d (silu(W_g n2) * (W_u n2)) with n2 = rmsnorm(x). */
static void F(post_attention)(const orc_model* m, int layer, const REAL* a, REAL* x) {
  const orc_config* c = &m->cfg;
  const orc_layer* w = &m->layers[layer];
  int H = c->hidden, Fd = c->ffn, qd = c->n_q_heads * c->head_dim;
  REAL* o = (REAL*)malloc(sizeof(REAL) * (size_t)H);
  REAL* n2 = (REAL*)malloc(sizeof(REAL) * (size_t)H);
  REAL* gate = (REAL*)malloc(sizeof(REAL) * (size_t)Fd);
  REAL* up = (REAL*)malloc(sizeof(REAL) * (size_t)Fd);
  F(project)(m, w->wo, w->q8_wo, w->s_wo, w->q4_wo, w->s4_wo, NULL, H, qd, a, o);
  for (int i = 0; i < H; ++i) x[i] = x[i] + o[i];
  F(orc_rmsnorm)(x, H, w->g_mlp, c->rms_eps, n2);
  F(project)(m, w->wg, w->q8_wg, w->s_wg, w->q4_wg, w->s4_wg, NULL, Fd, H, n2, gate);
  F(project)(m, w->wu, w->q8_wu, w->s_wu, w->q4_wu, w->s4_wu, NULL, Fd, H, n2, up);
  for (int j = 0; j < Fd; ++j) gate[j] = F(orc_silu)(gate[j]) * up[j];
  F(project)(m, w->wd, w->q8_wd, w->s_wd, w->q4_wd, w->s4_wd, NULL, H, Fd, gate, o);
  for (int i = 0; i < H; ++i) x[i] = x[i] + o[i];
  free(o);
  free(n2);
  free(gate);
  free(up);
}

/* Address of element `off` of a cache array (fp32 or bf16 elements). */
static const void* F(kv_at)(const orc_kv* kv, const void* p, long off) {
  return (const char*)p + off * (kv->bf16 ? 2 : 4);
}

/* One block for one token of sequence b at position pos (pos = number of
 * tokens already cached). K and V are stored in slot pos (fp32, or rounded
 * to bf16); query head h attends with kv head h / (Hq/Hkv) over slots 0..pos. */
void F(orc_block_decode)(const orc_model* m, int layer, orc_kv* kv, int b, int pos, REAL* x) {
  const orc_config* c = &m->cfg;
  int D = c->head_dim, G = c->n_q_heads / c->n_kv_heads;
  int qd = c->n_q_heads * D, kd = c->n_kv_heads * D;
  REAL* q = (REAL*)malloc(sizeof(REAL) * (size_t)qd);
  REAL* k = (REAL*)malloc(sizeof(REAL) * (size_t)kd);
  REAL* v = (REAL*)malloc(sizeof(REAL) * (size_t)kd);
  REAL* a = (REAL*)malloc(sizeof(REAL) * (size_t)qd);
  F(qkv_token)(m, layer, x, pos, q, k, v);
  for (int g = 0; g < c->n_kv_heads; ++g) {
    long base = F(kv_off)(c, kv, layer, b, g) + (long)pos * D;
    for (int i = 0; i < D; ++i) {
      F(kv_put)(kv->k, kv->bf16, base + i, k[g * D + i]);
      F(kv_put)(kv->v, kv->bf16, base + i, v[g * D + i]);
    }
  }
#pragma omp parallel for schedule(static)
  for (int h = 0; h < c->n_q_heads; ++h) {
    long base = F(kv_off)(c, kv, layer, b, h / G);
    F(orc_attention_head)(q + h * D, F(kv_at)(kv, kv->k, base), F(kv_at)(kv, kv->v, base),
                          kv->bf16, pos + 1, D, a + h * D);
  }
  F(post_attention)(m, layer, a, x);
  free(q);
  free(k);
  free(v);
  free(a);
}

/* Final norm and head: logits = W_head rmsnorm(x) (W_head = embed when tied). */
static void F(head)(const orc_model* m, const REAL* x, REAL* logits) {
  const orc_config* c = &m->cfg;
  REAL* n = (REAL*)malloc(sizeof(REAL) * (size_t)c->hidden);
  F(orc_rmsnorm)(x, c->hidden, m->g_final, c->rms_eps, n);
  if (m->q8_embed && c->tie_embeddings)  /* the int8 embedding is the head */
    F(linear_i8)(m, m->q8_embed, m->s_embed, NULL, c->vocab, c->hidden, n, logits);
  else
    F(orc_matvec_bf16)(c->tie_embeddings ? m->embed : m->lm_head, c->vocab, c->hidden, n,
                       logits);
  free(n);
}

/* One decode step for a batch: token tokens[b] enters sequence b at position
 * positions[b]. Writes logits [B, V] and, if next != NULL, the greedy token
 * (argmax, lowest index on ties). hidden (nullable) receives, per sequence,
 * the residual stream after the embedding and after every layer:
 * [B][L + 1][H]. Returns 0, or -1 on an invalid position or NaN logits. */
int F(orc_decode_step)(const orc_model* m, orc_kv* kv, int batch, const int32_t* tokens,
                       const int32_t* positions, REAL* logits, int32_t* next, REAL* hidden) {
  const orc_config* c = &m->cfg;
  int H = c->hidden, L = c->n_layers;
  REAL* x = (REAL*)malloc(sizeof(REAL) * (size_t)H);
  int rc = 0;
  for (int b = 0; b < batch; ++b) {
    if (positions[b] < 0 || positions[b] >= kv->max_ctx || tokens[b] < 0 || tokens[b] >= c->vocab) {
      rc = -1;
      break;
    }
    F(embed_row)(m, tokens[b], x);
    if (hidden) memcpy(hidden + ((long)b * (L + 1)) * H, x, sizeof(REAL) * (size_t)H);
    for (int l = 0; l < L; ++l) {
      F(orc_block_decode)(m, l, kv, b, positions[b], x);
      if (hidden) memcpy(hidden + ((long)b * (L + 1) + l + 1) * H, x, sizeof(REAL) * (size_t)H);
    }
    REAL* lg = logits + (long)b * c->vocab;
    F(head)(m, x, lg);
    if (next) {
      int t = sizeof(REAL) == sizeof(float) ? orc_argmax_f32((const float*)lg, c->vocab)
                                            : orc_argmax_f64((const double*)lg, c->vocab);
      next[b] = t;
      if (t < 0) rc = -1;
    }
  }
  free(x);
  return rc;
}

/* n tokens of sequence b at positions start_pos .. start_pos + n - 1, layer by
 * layer: every token's K/V of a layer is cached before that layer's attention,
 * and token i attends over slots 0 .. start_pos + i. logits: [n, V]. */
int F(orc_forward_chunk)(const orc_model* m, orc_kv* kv, int b, int n, const int32_t* tokens,
                         int start_pos, REAL* logits) {
  const orc_config* c = &m->cfg;
  int H = c->hidden, D = c->head_dim, G = c->n_q_heads / c->n_kv_heads;
  int qd = c->n_q_heads * D, kd = c->n_kv_heads * D;
  if (start_pos < 0 || start_pos + n > kv->max_ctx) return -1;
  REAL* x = (REAL*)malloc(sizeof(REAL) * (size_t)n * H);
  REAL* q = (REAL*)malloc(sizeof(REAL) * (size_t)n * qd);
  REAL* k = (REAL*)malloc(sizeof(REAL) * (size_t)kd);
  REAL* v = (REAL*)malloc(sizeof(REAL) * (size_t)kd);
  REAL* a = (REAL*)malloc(sizeof(REAL) * (size_t)qd);
  for (int i = 0; i < n; ++i)
    F(embed_row)(m, tokens[i], x + (long)i * H);
  for (int l = 0; l < c->n_layers; ++l) {
    for (int i = 0; i < n; ++i) {
      F(qkv_token)(m, l, x + (long)i * H, start_pos + i, q + (long)i * qd, k, v);
      for (int g = 0; g < c->n_kv_heads; ++g) {
        long base = F(kv_off)(c, kv, l, b, g) + (long)(start_pos + i) * D;
        for (int e = 0; e < D; ++e) {
          F(kv_put)(kv->k, kv->bf16, base + e, k[g * D + e]);
          F(kv_put)(kv->v, kv->bf16, base + e, v[g * D + e]);
        }
      }
    }
    for (int i = 0; i < n; ++i) {
      for (int h = 0; h < c->n_q_heads; ++h) {
        long base = F(kv_off)(c, kv, l, b, h / G);
        F(orc_attention_head)(q + (long)i * qd + h * D, F(kv_at)(kv, kv->k, base),
                              F(kv_at)(kv, kv->v, base), kv->bf16, start_pos + i + 1, D,
                              a + h * D);
      }
      F(post_attention)(m, l, a, x + (long)i * H);
    }
  }
  for (int i = 0; i < n; ++i) F(head)(m, x + (long)i * H, logits + (long)i * c->vocab);
  free(x);
  free(q);
  free(k);
  free(v);
  free(a);
  return 0;
}

/* The uncached forward over a whole sequence of t tokens at positions
 * 0 .. t-1: per layer, all keys and values are computed from that layer's
 * input, the t x t score matrix is masked causally (key j visible to query i
 * iff j <= i) and softmaxed row by row. K and V are rounded exactly as a cache
 * of that type stores them (fp32, or bf16 when kv_bf16). logits: [t, V]. */
int F(orc_forward_full)(const orc_model* m, int t, const int32_t* tokens, int kv_bf16,
                        REAL* logits) {
  const orc_config* c = &m->cfg;
  int H = c->hidden, D = c->head_dim, G = c->n_q_heads / c->n_kv_heads;
  int qd = c->n_q_heads * D, kd = c->n_kv_heads * D;
  REAL* x = (REAL*)malloc(sizeof(REAL) * (size_t)t * H);
  REAL* q = (REAL*)malloc(sizeof(REAL) * (size_t)t * qd);
  REAL* k = (REAL*)malloc(sizeof(REAL) * (size_t)t * kd);
  REAL* v = (REAL*)malloc(sizeof(REAL) * (size_t)t * kd);
  REAL* a = (REAL*)malloc(sizeof(REAL) * (size_t)t * qd);
  REAL* s = (REAL*)malloc(sizeof(REAL) * (size_t)t);
  REAL* p = (REAL*)malloc(sizeof(REAL) * (size_t)t);
  REAL scale = (REAL)1 / F(sqrtr)((REAL)D);
  for (int i = 0; i < t; ++i)
    F(embed_row)(m, tokens[i], x + (long)i * H);
  for (int l = 0; l < c->n_layers; ++l) {
    for (int i = 0; i < t; ++i) {
      F(qkv_token)(m, l, x + (long)i * H, i, q + (long)i * qd, k + (long)i * kd, v + (long)i * kd);
      for (int e = 0; e < kd; ++e) {
        const long j = (long)i * kd + e;
        k[j] = kv_bf16 ? F(widen)(F(narrow)(k[j])) : (REAL)(float)k[j];
        v[j] = kv_bf16 ? F(widen)(F(narrow)(v[j])) : (REAL)(float)v[j];
      }
    }
    for (int i = 0; i < t; ++i) {
      for (int h = 0; h < c->n_q_heads; ++h) {
        int g = h / G;
        const REAL* qi = q + (long)i * qd + h * D;
        /* full row of scores with the causal mask applied as exclusion */
        REAL mx = 0;
        int first = 1;
        for (int j = 0; j < t; ++j) {
          REAL dot = 0;
          for (int e = 0; e < D; ++e) dot += qi[e] * k[(long)j * kd + g * D + e];
          s[j] = dot * scale;
          if (j <= i && (first || s[j] > mx)) {
            mx = s[j];
            first = 0;
          }
        }
        REAL sum = 0;
        for (int j = 0; j < t; ++j) {
          p[j] = j <= i ? F(expr)(s[j] - mx) : (REAL)0;
          sum += p[j];
        }
        for (int e = 0; e < D; ++e) {
          REAL acc = 0;
          for (int j = 0; j < t; ++j) acc += (p[j] / sum) * v[(long)j * kd + g * D + e];
          a[(long)i * qd + h * D + e] = acc;
        }
      }
    }
    for (int i = 0; i < t; ++i) F(post_attention)(m, l, a + (long)i * qd, x + (long)i * H);
  }
  for (int i = 0; i < t; ++i) F(head)(m, x + (long)i * H, logits + (long)i * c->vocab);
  free(x);
  free(q);
  free(k);
  free(v);
  free(a);
  free(s);
  free(p);
  return 0;
}

#undef F
#undef CAT
#undef CAT2
