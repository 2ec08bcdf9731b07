/*
 * nc.h -- C ABI of libnc: the single-token decode step of a Qwen2-style
 * decoder on one GB300 (sm_103a), as hand-written CUDA kernels.
 *
 * The model: pre-norm blocks x += attn(rmsnorm(x)); x += mlp(rmsnorm(x))
 * (nanoinfer, "Model architecture"); grouped-query attention where query head
 * h reads kv head h / (Hq/Hkv) (same section: repeat, not tile); half-split
 * RoPE pairing i with i + D/2, applied once when K enters the cache (nanoinfer,
 * "KV cache"); QKV bias and no o-proj bias; SwiGLU down(silu(gate) * up);
 * tied embedding head after a final norm; greedy = argmax, lowest index on
 * ties (nanoinfer, "Sampling": temperature 0).
 *
 * Conventions for every entry point:
 *   - Pointers named *_dev, and every tensor pointer unless stated, are DEVICE
 *     pointers owned by the caller; libnc never frees them. *_host pointers
 *     are host memory read synchronously during the call.
 *   - bf16 tensors are raw bf16 bit patterns (2 bytes, round-to-nearest-even
 *     when libnc narrows); activations are fp32; matrices are [out, in]
 *     row-major (y = W x), rows 16-byte aligned (in * 2 % 16 == 0).
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). Work is
 *     enqueued asynchronously; nothing is read back from the device during a
 *     call (validation uses host-side sizes and *_host copies only).
 *   - Invalid input returns an error code before anything is enqueued and
 *     leaves all state untouched. A CUDA error latches the model UNHEALTHY:
 *     every later call on it returns NC_ERR_UNHEALTHY.
 *   - nc_last_error_message() gives a thread-local description of the last
 *     failure.
 */
#ifndef NC_H
#define NC_H
#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define NC_ABI_VERSION 1

typedef enum {
  NC_OK = 0,
  NC_ERR_INVALID_ARGUMENT = 1, /* null pointer, bad flag */
  NC_ERR_SHAPE = 2,            /* sizes inconsistent or unsupported */
  NC_ERR_DTYPE = 3,            /* weight type not supported by this call */
  NC_ERR_CAPACITY = 4,         /* batch or positions beyond what was reserved */
  NC_ERR_POSITION = 5,         /* a position outside [0, capacity) or a block-table hole */
  NC_ERR_CUDA = 6,             /* a CUDA runtime call failed (model now unhealthy) */
  NC_ERR_TIMEOUT = 7,          /* a bounded device-side wait expired */
  NC_ERR_UNHEALTHY = 8,        /* the model saw an earlier CUDA failure */
  NC_ERR_UNSUPPORTED = 9
} nc_status;

/* Weight storage of the seven projections (nanoinfer "Quantization").
 * NC_INT8: int8 per output row, activations quantised per token (W8A8).
 * NC_INT8_B32: the same projections with activations quantised per block of
 * 32 values, and the embedding stored int8 per row too, which is also the
 * tied head (nanoinfer, INT8 activation section and its "INT8 + embeddings"
 * level); needs tie_embeddings and hidden, ffn, n_q_heads * head_dim
 * multiples of 32. NC_INT4_G32 / NC_INT4_G128: INT4 codes in [-7, 7] with
 * one fp32 scale per group of 32 / 128 weights of a row, fp32 activations;
 * hidden, ffn and n_q_heads * head_dim must be multiples of the group. In
 * the other types the embedding and the head stay bf16. */
typedef enum {
  NC_BF16 = 0,
  NC_INT8 = 1,
  NC_INT8_B32 = 2,
  NC_INT4_G32 = 3,
  NC_INT4_G128 = 4
} nc_wtype;

/* Hyperparameters. head_dim must be 64 or 128; n_q_heads a multiple of
 * n_kv_heads with group <= 8; hidden, ffn, n_q_heads*head_dim multiples of 8. */
typedef struct {
  int hidden;          /* H */
  int n_q_heads;       /* Hq */
  int n_kv_heads;      /* Hkv */
  int head_dim;        /* D */
  int ffn;             /* F */
  int n_layers;        /* L */
  int vocab;           /* V */
  float rms_eps;       /* RMSNorm epsilon */
  float rope_theta;    /* RoPE base */
  int qkv_bias;        /* 1: q, k, v projections carry a bias (Qwen2) */
  int qk_norm;         /* 1: per-head RMSNorm of q and k before RoPE (gains [D]) */
  int tie_embeddings;  /* 1: logits use the embedding matrix */
  nc_wtype wtype;      /* NC_INT8: the seven projections run W8A8 */
} nc_config;

/* One block's weights in checkpoint layout (device, bf16, caller-owned; read
 * only during nc_model_create, which keeps its own packed copy). */
typedef struct {
  const void *wq, *wk, *wv;     /* [Hq*D, H], [Hkv*D, H], [Hkv*D, H] */
  const void *bq, *bk, *bv;     /* [Hq*D], [Hkv*D], [Hkv*D]; NULL unless qkv_bias */
  const void *wo;               /* [H, Hq*D] */
  const void *wg, *wu;          /* [F, H] */
  const void *wd;               /* [H, F] */
  const void *g_attn, *g_mlp;   /* [H] */
  const void *g_q, *g_k;        /* [D]; NULL unless qk_norm */
} nc_layer_weights;

typedef struct {
  const void* embed;               /* [V, H] */
  const void* lm_head;             /* [V, H]; NULL when tie_embeddings */
  const void* g_final;             /* [H] */
  const nc_layer_weights* layers;  /* HOST array of n_layers entries */
} nc_weights;

/* Element type of the KV cache. fp32 is nanoinfer's cache ("24 KiB per token
 * at fp32" for the 0.5B shape) and the default; bf16 halves the cache traffic
 * and rounds K and V to nearest even when they are stored. */
typedef enum { NC_KV_F32 = 0, NC_KV_BF16 = 1 } nc_kv_dtype;

/* KV cache (caller-owned device memory of `dtype`). K and V of the new token
 * are written at slot `position` of its sequence; attention reads slots
 * 0..position.
 *   contiguous (paged = 0): k, v are [L][batch_capacity][Hkv][max_ctx][D].
 *   paged (paged = 1):      k, v are [L][num_blocks][Hkv][block_size][D];
 *     position p of sequence b lives in block block_table[b][p / block_size]
 *     at offset p % block_size (vLLM-style gather; Tang section 2.1 "paged KV
 *     caches" as a gather view). block_table is int32 [batch][max_blocks_per_seq]
 *     on the device, with an identical host copy used for validation. */
typedef struct {
  int paged;
  nc_kv_dtype dtype;
  int batch_capacity;      /* contiguous: sequences reserved */
  int max_ctx;             /* contiguous: slots per sequence; paged: max_blocks_per_seq*block_size */
  int block_size;          /* paged */
  int num_blocks;          /* paged: physical blocks per layer */
  int max_blocks_per_seq;  /* paged */
  void* k;
  void* v;
  const int32_t* block_table;       /* device, paged only */
  const int32_t* block_table_host;  /* host, paged only */
} nc_kv_cache;

typedef struct nc_model nc_model; /* opaque: packed weights, workspace, graphs */

const char* nc_status_string(nc_status s);
const char* nc_last_error_message(void);
int nc_abi_version(void);

/* Build a model: validates cfg, packs the weights into model-owned device
 * memory (QKV rows concatenated, gate and up concatenated; NC_INT8 quantises
 * the seven projections per output row, nanoinfer "Quantization"), and
 * reserves the workspace for up to max_batch sequences of up to max_ctx
 * positions. Synchronises `stream` before returning. */
nc_status nc_model_create(const nc_config* cfg, const nc_weights* w, int max_batch, int max_ctx,
                          void* stream, nc_model** out);
nc_status nc_model_destroy(nc_model* m);
/* Bytes of packed weights and of workspace held by the model (the static
 * memory plan of nanocompile's phase 7: everything a step touches is
 * reserved at creation; the pages give no call of this kind). Either
 * pointer may be NULL. */
nc_status nc_model_memory(const nc_model* m, size_t* weight_bytes, size_t* workspace_bytes);

/* Flags of nc_decode_step. */
#define NC_STEP_GRAPH 1   /* replay a CUDA graph captured on first use for this
                             (batch, kv layout, buffer pointers); else launch
                             the kernels directly */
#define NC_STEP_ADVANCE 2 /* after the step, on the device: positions_dev[b] += 1
                             and tokens_dev[b] = the greedy token, so the next
                             call continues greedy decoding with no host work
                             (the caller then passes positions_host + 1) */
#define NC_STEP_STAGED 4  /* use the per-stage kernels even where the persistent
                             decode kernel applies. By default a step with bf16
                             weights and batch <= 4 runs as one persistent,
                             cooperative kernel (one launch, no graph; any cache
                             length: long scans are split over the grid); other
                             steps run the per-stage kernels. */

/* One decode step for `batch` sequences (nanoinfer "Model architecture" and
 * "KV cache"; the one-call-per-token step of nanocompile's phase 7): token
 * tokens_dev[b] enters sequence b at position positions[b] (= tokens already
 * cached). Every layer writes K/V at that slot; logits_dev [batch, V] fp32
 * receives the head output and next_dev [batch] int32 (nullable) the argmax
 * (lowest index on ties; -1 if a logit is NaN). positions_host must equal
 * positions_dev. tokens_dev and positions_dev are written only under
 * NC_STEP_ADVANCE. */
nc_status nc_decode_step(nc_model* m, int batch, int32_t* tokens_dev, int32_t* positions_dev,
                         const int32_t* positions_host, const nc_kv_cache* kv, float* logits_dev,
                         int32_t* next_dev, int flags, void* stream);

/* One block (layer `layer`) for `batch` sequences: x_dev [batch, H] fp32 is
 * the residual stream, updated in place; K/V are appended at positions. */
nc_status nc_block_forward(nc_model* m, int layer, int batch, float* x_dev,
                           const int32_t* positions_dev, const int32_t* positions_host,
                           const nc_kv_cache* kv, void* stream);

/* ---------------- prefill (a prompt chunk as one forward pass) ------------- */

/* Bytes of caller-owned device scratch nc_prefill needs for a chunk of T
 * tokens (the chunk's activations and the tensor cores' input planes). 0 for
 * an invalid model or T. */
size_t nc_prefill_scratch_bytes(const nc_model* m, int T);

/* The T tokens tokens_dev [T] int32 enter cache sequence `seq` at positions
 * start_pos .. start_pos + T - 1, as one causal forward pass instead of T
 * decode steps (the nanoinfer page's batched prefill: each weight row read
 * once for the whole prompt; Tang section 2.3: attention fused under the
 * online-softmax monoid). Per layer: the projections of all T tokens as
 * tensor-core GEMMs (tcgen05, fp32 accumulation, activations as bf16 hi / lo
 * planes), RoPE and the K/V append of every token, and a flash-style
 * attention where token i sees slots 0 .. start_pos + i (the cache's earlier
 * positions and the chunk's tokens up to itself). logits_dev [V] fp32
 * receives the last token's logits and next_dev [1] int32 (nullable) their
 * arg-max (lowest index on ties; -1 on NaN). Positions after the chunk are
 * untouched; a following nc_decode_step continues at start_pos + T.
 * bf16 models only (NC_ERR_UNSUPPORTED otherwise); hidden, ffn and
 * n_q_heads * head_dim must be multiples of 64. scratch: device memory of at
 * least nc_prefill_scratch_bytes(m, T) bytes, 16-byte aligned, owned by the
 * caller. Validation uses host data: start_pos + T within the cache's
 * capacity, seq within batch_capacity (contiguous) or every block of the
 * chunk in the pool (paged), else NC_ERR_POSITION / NC_ERR_CAPACITY before
 * anything is enqueued. Uses the model's workspace (non-reentrant). */
nc_status nc_prefill(nc_model* m, int seq, int T, const int32_t* tokens_dev, int start_pos,
                     const nc_kv_cache* kv, float* logits_dev, int32_t* next_dev, void* scratch,
                     size_t scratch_bytes, void* stream);

/* Device watchdog word (0 = fine, else an nc_status set by a kernel, e.g. a
 * NaN in the logits or an expired bounded wait). Synchronises `stream`,
 * reads the word and clears it. It is how device-side failures reach the
 * host without a read-back inside a step (nanoserve: host read-backs were
 * the graph breaks, so the step never reads the device itself; ForgeML
 * "Leader/worker protocol and failure semantics": after a backend failure
 * the engine goes unhealthy and fails later calls). */
nc_status nc_get_device_status(nc_model* m, void* stream, int* code);

/* Which implementation nc_decode_step runs for these arguments (nothing is
 * launched; the pages have no counterpart: it reports a dispatch decision of
 * this library): NC_PATH_PERSISTENT, the whole step as one cooperative
 * persistent kernel (bf16 weights, batch <= 4, shape within its
 * shared-memory plan, NC_STEP_STAGED not set), else
 * NC_PATH_STAGED, the per-stage kernels (2 + 5 per layer launches, in a CUDA
 * graph with NC_STEP_GRAPH). */
typedef enum { NC_PATH_STAGED = 0, NC_PATH_PERSISTENT = 1 } nc_path;
nc_status nc_decode_path(nc_model* m, int batch, const nc_kv_cache* kv, int flags, int* path);

/* W8A8 diagnostic (nanoinfer "Quantization": the per-token activation codes;
 * for checking every code a whole-model W8A8 step used against the oracle's).
 * While set, every nc_decode_step and nc_block_forward of this W8A8 model
 * (NC_INT8 or NC_INT8_B32) writes the activation codes of its W8A8 products
 * (and, NC_INT8 only, their per-token scales) to the caller's device
 * buffers, and a decode step runs its kernels directly (no graph). Layout
 * for a step at batch B, per layer l of L:
 *   codes_dev + l * B * (2 H + Hq D + F): the codes [B][H] of the QKV
 *     product, then [B][Hq D] of the o-proj, [B][H] of gate|up, [B][F] of
 *     the down product (nc_block_forward writes layer `layer`'s slot);
 *     NC_INT8_B32 then the int8 head's codes [B][H] after the L layers;
 *   scales_dev (nullable; NC_INT8) + (l * 4 + p) * B: the B scales of
 *     product p in that order.
 * Capacities are in elements; a step that needs more returns
 * NC_ERR_CAPACITY. A NULL codes_dev turns it off. NC_ERR_DTYPE for a bf16
 * model. */
nc_status nc_debug_w8a8_codes(nc_model* m, int8_t* codes_dev, size_t codes_capacity,
                              float* scales_dev, size_t scales_capacity);

/* Phase profile of the persistent decode kernel (a per-phase step profile in
 * the spirit of nanocompile's per-primitive profile of one step). While
 * enabled, every persistent step records %globaltimer (ns) in each CTA at the
 * start of each phase and when the phase's input had arrived; phases are, per
 * layer, QKV, attention, o-proj, gate|up, down, then the LM head.
 * nc_read_phase_profile synchronises `stream` and copies the last step's
 * record: for each of the n_sm CTAs (one per SM) 2 * P + 2 + 8 * n_layers
 * values, P = 5 * n_layers + 1: [2p] start of phase p, [2p + 1] its input
 * in, then the CTA's start and end (the CTA that finishes the step: the
 * step's end), then per layer l eight values of the CTA's first attention
 * item: [2P + 2 + 8l] its split's softmax states combined, [+1] its output
 * (or split partials and ticket) published, [+2] the merge of the splits
 * done (0 unless this CTA merged), [+3] and [+4] the first and the last K/V
 * chunk in shared memory (as the first scan warp saw them), [+5] that
 * warp's scan done, [+6] and [+7] (head size 64, the block-wide scan) the
 * first chunk's scores and weights done. *n receives the count; a smaller
 * capacity returns NC_ERR_CAPACITY. */
nc_status nc_profile_phases(nc_model* m, int enable);
nc_status nc_read_phase_profile(nc_model* m, void* stream, unsigned long long* out_host,
                                int capacity, int* n);

/* ---------------- per-stage entry points (no model needed unless named) ---- */

/* The weight-type argument of the stage GEMVs (nanoinfer "Quantization"):
 *   NC_BF16: W is bf16 [N, K] (raw bits); the scale argument and
 *     acc_i32_debug must be NULL.
 *   NC_INT8: W is int8 [N, K] (16-byte aligned) with fp32 per-row scales
 *     w_scale [N] (as nc_quantize_weight makes them). The kernel quantises
 *     each sequence's (normed) input per token: s_x = amax / 127, codes
 *     round-half-away(v / s_x) in [-127, 127]; accumulates acc = sum_k
 *     W[n, k] * code_k in int32 (exact: |acc| <= K * 127^2); and dequantises
 *     y = float(acc) * (w_scale[n] * s_x), each product rounded on its own,
 *     then + bias. K must be a multiple of 16.
 * Any other value returns NC_ERR_DTYPE. */

/* y[b, n] = sum_k W[n, k] * xn[b, k] (+ bias[n]), xn = rmsnorm(x[b]) * gamma
 * when gamma != NULL (nanocompile: the five passes of rms_norm fused into one,
 * and the norm fused into the GEMV that follows), else xn = x: the QKV
 * projection with its bias. x [B, K] fp32, gamma [K] bf16, W [N, K] of
 * `wtype`, w_scale [N] fp32 (NC_INT8), bias [N] bf16 or NULL, y [B, N] fp32.
 * acc_i32_debug (NC_INT8, nullable): [B, N] int32 receives the accumulators,
 * for bit-exact checks. B <= 16. */
nc_status nc_rmsnorm_gemv(const float* x, const void* gamma, float eps, const void* W,
                          nc_wtype wtype, const float* w_scale, const void* bias, int B, int K,
                          int N, float* y, int32_t* acc_i32_debug, void* stream);

/* x[b, n] += sum_k W[n, k] * a[b, k]: the o-proj and down projections with
 * the residual add fused in (nanocompile, "Phase 3": "output projection with
 * its residual add"). a [B, K], x [B, N] fp32 in place, W [N, K] of `wtype`,
 * w_scale [N] fp32 (NC_INT8, else NULL). */
nc_status nc_gemv_residual(const float* a, const void* W, nc_wtype wtype, const float* w_scale,
                           int B, int K, int N, float* x, void* stream);

/* h[b, f] = silu(g_f) * u_f with g = W_gate xn, u = W_up xn and xn the
 * normed x (Tang section 2.3: sibling reductions gate|up merged; nanoinfer
 * "Phase 8" sigmoid form). W_gu is [2F, K] of `wtype`: rows 0..F-1 gate,
 * F..2F-1 up; s_gu [2F] fp32 their scales (NC_INT8, else NULL).
 * x [B, K], h [B, F] fp32. */
nc_status nc_swiglu_gemv(const float* x, const void* gamma, float eps, const void* W_gu,
                         nc_wtype wtype, const float* s_gu, int B, int K, int F, float* h,
                         void* stream);

/* RoPE (half-split) on q and k of layer `layer` at positions, optional
 * per-head q/k RMSNorm before it, then K and V rounded to bf16 and stored at
 * slot positions[b] (nanoinfer "KV cache": rotate once on insert).
 * qkv [B, (Hq + 2 Hkv) D] fp32 (bias already added), q_out [B, Hq D] fp32. */
nc_status nc_rope_qkv(const nc_model* m, int layer, int B, const float* qkv,
                      const int32_t* positions_dev, const int32_t* positions_host,
                      float* q_out, const nc_kv_cache* kv, void* stream);

/* Split-K GQA decode attention (Tang section 2.2: online softmax is a monoid
 * on (max, rescaled sum, weighted values); section 2.5: split is valid for
 * any associative monoid): for query head h of sequence b, softmax over
 * slots 0..positions[b] of q.k_t / sqrt(D), weighted sum of v_t. Partials of
 * each split go to the model's workspace and are merged into out
 * [B, Hq D] fp32. q [B, Hq D] fp32 (already rotated). */
nc_status nc_attn_decode(const nc_model* m, int layer, int B, const float* q,
                         const int32_t* positions_dev, const int32_t* positions_host,
                         const nc_kv_cache* kv, float* out, void* stream);

/* The same attention as nc_attn_decode, for callers that cannot allocate
 * device memory (the pages have no counterpart of this entry point). Such
 * callers include code running while a stream of the process is in
 * global-mode graph capture, where cudaMalloc is not permitted; code whose
 * device memory is owned by a framework allocator that forbids raw
 * cudaMalloc; and latency-critical loops that cannot afford cudaMalloc's
 * implicit synchronisation. It needs no model and allocates nothing: the
 * split partials live in a static device array of 1,048,576 floats (4 MiB)
 * that every GPU loading libnc holds until the process exits, beside 1,024
 * static merge counters (zero at load; each call returns the ones it used to
 * zero) and one static status word. A request whose partials,
 * n_q_heads * splits * (head_dim + 2) floats with splits >= B (the splits of
 * one kv head are shared out among the sequences), exceed the array, or
 * whose B * n_kv_heads exceeds the counters, returns NC_ERR_CAPACITY before
 * anything is enqueued. The first call on each device looks up the array's
 * device address (cudaGetSymbolAddress, with that device current); make that
 * first call before any stream capture. Later calls whose stream is not
 * capturing look the address up again (a context re-created after a device
 * reset is then picked up); a capturing call reuses the last lookup. All
 * calls share the array: calls that overlap on the GPU (on different
 * streams, or from different threads) race and must be serialised by the
 * caller. Every scratch element a call reads is written earlier in the same
 * call, so what the previous call left there does not matter. Errors the
 * kernel detects on the device (an expired bounded wait: NC_ERR_TIMEOUT; a
 * block-table entry or position the device copy disagrees on:
 * NC_ERR_POSITION) leave `out` undefined for the affected heads and are
 * recorded in the static status word; nc_attn_decode_static_status reads it.
 * n_layers is the cache's layer count (bounds `layer`); other arguments as
 * for nc_attn_decode. */
nc_status nc_attn_decode_static(int n_q_heads, int n_kv_heads, int head_dim, int n_layers,
                                int layer, int B, const float* q, const int32_t* positions_dev,
                                const int32_t* positions_host, const nc_kv_cache* kv, float* out,
                                void* stream);

/* Synchronises `stream`, then reads the static status word of
 * nc_attn_decode_static into *code (0 = no device-side error since the last
 * read, else the first nc_status a kernel recorded) and clears it. Copies
 * between the word and host memory only; allocates nothing. */
nc_status nc_attn_decode_static_status(void* stream, int* code);

/* logits[b, v] = sum_k W[v, k] * xn[b, k] with xn = rmsnorm(x[b]) * gamma,
 * and next[b] = argmax_v logits[b, v], lowest index on ties, -1 on NaN
 * (Tang section 2.2: arg-max is a monoid on (value, index)). next nullable.
 * Needs scratch for per-block partials: uses the model's workspace. */
nc_status nc_lm_head_argmax(nc_model* m, const float* x, const void* gamma, float eps,
                            const void* W, int B, int K, int V, float* logits, int32_t* next,
                            void* stream);

/* ---------------- INT4 weights (nanoinfer "Quantization": group-wise INT4) --- */

/* y[b, n] = sum_k (q[n, k] * scales[n, k / group]) * xn[b, k], each
 * dequantised weight rounded to fp32, with xn = rmsnorm(x[b]) * gamma when
 * gamma != NULL, else xn = x (nanoinfer, "Quantization": INT4 codes in
 * [-7, 7], one fp32 scale per group of `group` consecutive weights of a row).
 * Wq [N, K / 2] bytes: two codes a byte, the even index in the low nibble,
 * two's-complement nibbles; scales [N, K / group] fp32; x [B, K] fp32,
 * gamma [K] bf16 or NULL, y [B, N] fp32. B in [1, 8], group 32, 64 or 128,
 * K a multiple of group, the batch's activations within shared memory
 * (8 rows of K up to ~5,500). Errors (before anything is enqueued): NULL or
 * misaligned pointers -> NC_ERR_INVALID_ARGUMENT, other sizes -> NC_ERR_SHAPE. */
nc_status nc_int4_gemv(const float* x, const void* gamma, float eps, const uint8_t* Wq,
                       const float* scales, int group, int B, int K, int N, float* y,
                       void* stream);

/* ---------------- sampling (nanoinfer, sampling section) -------------------- */

/* Bytes of device scratch nc_sample needs for B rows of V logits at
 * temperature > 0: 20 * B * (V rounded up to 64). 0 for invalid sizes. */
size_t nc_sample_scratch_bytes(int B, int V);

/* One token per row of logits [B, V] fp32 (nanoinfer, sampling section:
 * "temperature, top-k, top-p, seeded draw", in that order, then the softmax
 * of what is left and an inverse-CDF draw):
 *   temperature == 0: the arg-max, lowest index on ties (greedy);
 *   else s = logits / temperature (fp32 IEEE division); top_k > 0 keeps the
 *   tokens whose s is >= the k-th largest (ties at the k-th place stay;
 *   0 or >= V keeps all); top_p < 1 orders the kept tokens by ascending s,
 *   equal s in index order, and drops each one whose running fp32 sum of
 *   exp(s - max) / total is <= 1 - top_p (the largest always stays); then
 *   tokens[b] is the first kept token, in index order, whose running sum of
 *   the weights exp(s - max) (fp32 values, fp64 sums) exceeds u[b] times
 *   their total.
 * u [B] fp64 on the device holds the caller's uniform numbers in [0, 1)
 * (unused at temperature 0); kept [B, 2] int32 (nullable) receives the
 * number of tokens kept after top-k and after top-p ((1, 1) at temperature
 * 0). A row with a NaN logit, or at temperature > 0 a score of +inf or only
 * scores of -inf, gets token -1 and kept (0, 0); a -inf logit is a masked
 * token that is never drawn. scratch: device memory of at least
 * nc_sample_scratch_bytes(B, V) bytes, 16-byte aligned, owned by the caller
 * (NULL allowed at temperature 0); its contents on entry do not matter.
 * One CTA per row; calls sharing a scratch buffer must not overlap on the
 * GPU. Errors: NULL pointers or temperature < 0 / not finite, top_k < 0,
 * top_p outside (0, 1] -> NC_ERR_INVALID_ARGUMENT; B outside [1, 65535] or
 * V outside [1, 2^24] -> NC_ERR_SHAPE; scratch smaller than needed ->
 * NC_ERR_CAPACITY; all before anything is enqueued. */
nc_status nc_sample(const float* logits, int B, int V, float temperature, int top_k, float top_p,
                    const double* u, int32_t* tokens, int32_t* kept, void* scratch,
                    size_t scratch_bytes, void* stream);

/* ---------------- W8A8 (nanoinfer "Quantization", per-token activations) ---- */

/* Per-output-row symmetric weight quantisation: scale[n] = amax_n / 127,
 * q[n, k] = clamp(round_half_away(W[n, k] / scale[n]), -127, 127); a zero row
 * gets scale 0 and q = 0. W [N, K] bf16, q [N, K] int8, scale [N] fp32. */
nc_status nc_quantize_weight(const void* W, int N, int K, int8_t* q, float* scale, void* stream);

/* y[b, n] = float(acc[b, n]) * (w_scale[n] * sx[b]) (+ bias[n]) with
 * acc = sum_k Wq[n, k] * xq[b, k] in int32, xq/sx the per-token quantisation
 * of xn (normed when gamma != NULL). The optional outputs expose xq [B, K]
 * int8, sx [B] fp32 and acc [B, N] int32 for bit-exact checks. */
nc_status nc_w8a8_gemv(const float* x, const void* gamma, float eps, const int8_t* Wq,
                       const float* w_scale, const void* bias, int B, int K, int N, float* y,
                       int8_t* xq_out, float* sx_out, int32_t* acc_out, void* stream);

/* The same product with activations quantised per block of 32 consecutive
 * values instead of per token (nanoinfer, INT8 activation section: "one per
 * 32", so an outlier widens only its own block): sx[b, j] = amax of block j
 * of xn[b] / 127, xq = clamp(round_half_away(xn / sx), -127, 127);
 * acc[b, n, j] = sum over block j of Wq[n, k] * xq[b, k] in int32;
 * y[b, n] = sum_j float(acc[b, n, j]) * (w_scale[n] * sx[b, j]) (+ bias[n]).
 * B in [1, 8], K a multiple of 32. The optional outputs expose xq [B, K] int8,
 * sx [B, K / 32] fp32 and acc [B, N, K / 32] int32 for bit-exact checks.
 * Errors as for nc_w8a8_gemv. */
nc_status nc_w8a8_gemv_b32(const float* x, const void* gamma, float eps, const int8_t* Wq,
                           const float* w_scale, const void* bias, int B, int K, int N, float* y,
                           int8_t* xq_out, float* sx_out, int32_t* acc_out, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* NC_H */
