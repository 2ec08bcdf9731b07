// engine.cu -- the model object, weight packing, and the decode step.
//
// nc_model_create packs the caller's checkpoint-layout weights once into
// model-owned device memory (nanocompile "Phase 4": the runtime packs each
// weight once): QKV rows concatenated into one [(Hq + 2 Hkv) D, H] matrix
// (one wide GEMV, ForgeML "shared-projection fusion"), gate and up stacked
// into [2F, H] (Tang section 2.3, merge_siblings), or, for W8A8, the int8
// rows and per-row scales. The workspace (residual stream, q/k/v, attention
// partials, gate|up output, arg-max partials, status word) is reserved here
// too, so a decode step allocates nothing (nanocompile phase 7: one call per
// token, a static memory plan).
//
// A step launches: embed -> L x [QKV GEMV, RoPE+append, attention, o-proj +
// residual, gate|up + SiLU, down + residual] -> LM head + arg-max. With
// use_graph the sequence is captured once per (batch, buffers) and replayed
// as one CUDA graph: control crosses from host to device once per token and
// never back inside the step (nanoserve day 49: host readbacks were the
// graph breaks).
#include <cuda_runtime.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include <algorithm>

#include "engine.h"
#include "kernels.h"

namespace nc {

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Bump allocator over one cudaMalloc; with a null base it only measures.
struct Arena {
  char* base = nullptr;
  size_t used = 0;
  template <class T>
  T* take(size_t n) {
    used = align_up(used, 256);
    T* p = reinterpret_cast<T*>(reinterpret_cast<uintptr_t>(base) + used);
    used += n * sizeof(T);
    return p;
  }
};

Model::~Model() {
  for (auto& kv : graphs) cudaGraphExecDestroy(kv.second.exec);
  if (cap_stream) cudaStreamDestroy(cap_stream);
  if (status_host) cudaFreeHost(status_host);
  if (weights) cudaFree(weights);
  if (workspace) cudaFree(workspace);
}

bool valid_config(const nc_config& c, std::string* why) {
  char buf[256];
  auto bad = [&](const char* m) {
    snprintf(buf, sizeof buf, "%s", m);
    *why = buf;
    return false;
  };
  if (c.hidden <= 0 || c.n_q_heads <= 0 || c.n_kv_heads <= 0 || c.ffn <= 0 || c.n_layers <= 0 ||
      c.vocab <= 0)
    return bad("all sizes must be positive");
  if (c.head_dim != 64 && c.head_dim != 128) return bad("head_dim must be 64 or 128");
  if (c.n_q_heads % c.n_kv_heads != 0) return bad("n_q_heads must be a multiple of n_kv_heads");
  if (c.n_q_heads / c.n_kv_heads > 8) return bad("GQA group above 8 is unsupported");
  if (c.hidden % 16 || c.ffn % 16) return bad("hidden and ffn must be multiples of 16");
  if (c.hidden > 16384 || c.ffn > 65536) return bad("hidden or ffn too large");
  if (!(c.rms_eps > 0) || !(c.rope_theta > 1)) return bad("rms_eps must be > 0 and rope_theta > 1");
  if (c.wtype != NC_BF16 && c.wtype != NC_INT8 && c.wtype != NC_INT8_B32 &&
      c.wtype != NC_INT4_G32 && c.wtype != NC_INT4_G128)
    return bad("unknown weight type");
  if (c.wtype == NC_INT8_B32 &&
      (!c.tie_embeddings || c.hidden % 32 || c.ffn % 32 || (c.n_q_heads * c.head_dim) % 32))
    return bad("NC_INT8_B32 needs a tied head and hidden, ffn, n_q_heads * head_dim multiples of 32");
  if (c.wtype == NC_INT4_G32 || c.wtype == NC_INT4_G128) {
    const int g = c.wtype == NC_INT4_G32 ? 32 : 128;
    if (c.hidden % g || c.ffn % g || (c.n_q_heads * c.head_dim) % g)
      return bad("INT4 weights need hidden, ffn and n_q_heads * head_dim multiples of the group");
  }
  return true;
}

static nc_status check_ptr(const void* p, const char* name) {
  if (!p) return fail(NC_ERR_INVALID_ARGUMENT, "weight pointer %s is NULL", name);
  if (reinterpret_cast<uintptr_t>(p) % 16)
    return fail(NC_ERR_INVALID_ARGUMENT, "weight pointer %s is not 16-byte aligned", name);
  return NC_OK;
}

nc_status model_create(const nc_config* cfg, const nc_weights* w, int max_batch, int max_ctx,
                       cudaStream_t s, Model** out) {
  NC_CHECK(cfg && w && out && w->layers, NC_ERR_INVALID_ARGUMENT, "null argument");
  std::string why;
  NC_CHECK(valid_config(*cfg, &why), NC_ERR_SHAPE, "invalid config: %s", why.c_str());
  NC_CHECK(max_batch >= 1 && max_batch <= 16, NC_ERR_CAPACITY, "max_batch must be in [1, 16]");
  NC_CHECK(cfg->wtype != NC_INT8_B32 || max_batch <= 8, NC_ERR_CAPACITY,
           "NC_INT8_B32 models take at most 8 sequences");
  NC_CHECK(max_ctx >= 1 && max_ctx <= (1 << 20), NC_ERR_CAPACITY, "max_ctx out of range");
  const nc_config& c = *cfg;
  const int bt = max_batch <= 1 ? 1 : max_batch <= 2 ? 2 : max_batch <= 4 ? 4 : max_batch <= 8 ? 8 : 16;
  const int g4 = c.wtype == NC_INT4_G32 ? 32 : c.wtype == NC_INT4_G128 ? 128 : 0;
  if (g4) {
    NC_CHECK(max_batch <= 8, NC_ERR_CAPACITY, "INT4 models take at most 8 sequences");
    const int kmax = std::max(std::max(c.hidden, c.ffn), c.n_q_heads * c.head_dim);
    NC_CHECK(int4_smem_bytes(max_batch, kmax) + 4096 <= (size_t)max_smem_optin(), NC_ERR_SHAPE,
             "the INT4 GEMV keeps %d sequences of %d activations in shared memory: too many",
             max_batch, kmax);
  }
  NC_CHECK(bt * c.hidden <= 51200, NC_ERR_SHAPE,
           "max_batch (rounded up to a power of 2) * hidden must be <= 51200 for the LM head");
  nc_status st;
  if ((st = check_ptr(w->embed, "embed")) || (st = check_ptr(w->g_final, "g_final"))) return st;
  if (!c.tie_embeddings && (st = check_ptr(w->lm_head, "lm_head"))) return st;
  for (int l = 0; l < c.n_layers; ++l) {
    const nc_layer_weights& L = w->layers[l];
    const void* req[] = {L.wq, L.wk, L.wv, L.wo, L.wg, L.wu, L.wd, L.g_attn, L.g_mlp};
    for (const void* p : req)
      if ((st = check_ptr(p, "layer projection or norm"))) return st;
    if (c.qkv_bias)
      for (const void* p : {L.bq, L.bk, L.bv})
        if ((st = check_ptr(p, "qkv bias"))) return st;
    if (c.qk_norm)
      for (const void* p : {L.g_q, L.g_k})
        if ((st = check_ptr(p, "q/k norm gain"))) return st;
  }

  auto m = new Model();
  m->cfg = c;
  m->max_batch = max_batch;
  m->max_ctx = max_ctx;
  const int H = c.hidden, D = c.head_dim, F = c.ffn, Hq = c.n_q_heads, Hkv = c.n_kv_heads;
  const size_t qd = (size_t)Hq * D, kd = (size_t)Hkv * D, nqkv = qd + 2 * kd;
  const bool i8 = c.wtype == NC_INT8 || c.wtype == NC_INT8_B32;
  const bool b32 = c.wtype == NC_INT8_B32;

  // Two passes over one layout function: first with null bases to size the
  // arenas, then with the real allocations to assign every pointer.
  size_t part_max = 0;
  for (int b = 1; b <= max_batch; ++b) {
    const int sp = std::max(attn_splits(b, Hkv, D, false, max_ctx), attn_splits(b, Hkv, D, true, max_ctx));
    const size_t pf = attn_part_floats(b, Hq, D, sp);
    if (pf > part_max) part_max = pf;
  }
  auto layout = [&](Arena& A, Arena& W) {
    m->layers.assign(c.n_layers, LayerPacked{});
    for (int l = 0; l < c.n_layers; ++l) {
      LayerPacked& P = m->layers[l];
      if (g4) {
        P.p4_qkv = A.take<uint8_t>(nqkv * H / 2);
        P.p4_o = A.take<uint8_t>(qd * H / 2);
        P.p4_gu = A.take<uint8_t>((size_t)F * H);
        P.p4_d = A.take<uint8_t>((size_t)H * F / 2);
        P.s4_qkv = A.take<float>(nqkv * (H / g4));
        P.s4_o = A.take<float>((size_t)H * (qd / g4));
        P.s4_gu = A.take<float>(2 * (size_t)F * (H / g4));
        P.s4_d = A.take<float>((size_t)H * (F / g4));
      } else if (!i8) {
        P.w_qkv = A.take<uint16_t>(nqkv * H);
        P.w_o = A.take<uint16_t>(qd * H);
        P.w_gu = A.take<uint16_t>(2 * (size_t)F * H);
        P.w_d = A.take<uint16_t>((size_t)H * F);
      } else {
        P.q_qkv = A.take<int8_t>(nqkv * H);
        P.q_o = A.take<int8_t>(qd * H);
        P.q_gu = A.take<int8_t>(2 * (size_t)F * H);
        P.q_d = A.take<int8_t>((size_t)H * F);
        P.s_qkv = A.take<float>(nqkv);
        P.s_o = A.take<float>(H);
        P.s_gu = A.take<float>(2 * (size_t)F);
        P.s_d = A.take<float>(H);
      }
      P.b_qkv = c.qkv_bias ? A.take<uint16_t>(nqkv) : nullptr;
      P.g_attn = A.take<uint16_t>(H);
      P.g_mlp = A.take<uint16_t>(H);
      P.g_q = c.qk_norm ? A.take<uint16_t>(D) : nullptr;
      P.g_k = c.qk_norm ? A.take<uint16_t>(D) : nullptr;
    }
    if (b32) {  // the int8 rows replace the bf16 table (and serve as the head)
      m->q_embed = A.take<int8_t>((size_t)c.vocab * H);
      m->s_embed = A.take<float>(c.vocab);
    } else {
      m->embed = A.take<uint16_t>((size_t)c.vocab * H);
      m->head = c.tie_embeddings ? m->embed : A.take<uint16_t>((size_t)c.vocab * H);
    }
    m->g_final = A.take<uint16_t>(H);
    m->inv_freq = A.take<float>(D / 2);

    m->x = W.take<float>((size_t)max_batch * H);
    m->qkv = W.take<float>((size_t)max_batch * nqkv);
    m->q = W.take<float>((size_t)max_batch * qd);
    m->attn = W.take<float>((size_t)max_batch * qd);
    m->part = W.take<float>(part_max);
    m->h = W.take<float>((size_t)max_batch * F);
    // arg-max partial keys: one per CTA of the LM head (the tensor-core head
    // at batch 9..16 runs one CTA per 128 vocabulary rows)
    m->am_part = W.take<unsigned long long>(
        (size_t)max_batch * std::max(lm_head_grid(), (c.vocab + 127) / 128));
    // bf16 hi / lo activation planes of the tensor-core projections
    m->xb = max_batch > 8 && !i8 && !g4
                ? W.take<uint16_t>(umma_act_bytes(max_batch, std::max(std::max(H, F), (int)qd)) / 2 +
                                   512)
                : nullptr;
    m->ticket = W.take<unsigned int>(1);
    m->atickets = W.take<unsigned int>((size_t)max_batch * Hkv);
    m->status = W.take<int>(1);
    const size_t pb = max_batch < kPMaxBatch ? max_batch : kPMaxBatch;
    m->xw = W.take<uint64_t>(pb * H);
    m->qkvw = W.take<uint64_t>(pb * nqkv);
    m->aw = W.take<uint64_t>(pb * qd);
    m->apart = W.take<float>((size_t)kPMaxBatch * kPMaxSplits * c.n_q_heads * (D + 4));
    m->atick = W.take<unsigned int>((size_t)c.n_layers * kPMaxBatch * Hkv);
    m->hw = W.take<uint64_t>(pb * F);
    m->pticket = W.take<unsigned int>(1);
    m->seq = W.take<unsigned int>(1);
    m->prof = W.take<unsigned long long>((size_t)num_sms() * prof_values(c.n_layers));
    m->players = A.take<PLayer>(c.n_layers);
  };
  Arena A0, W0;
  layout(A0, W0);
  const size_t wb = A0.used, ws = W0.used;

  cudaError_t e = cudaMalloc(&m->weights, wb);
  if (e == cudaSuccess) e = cudaMalloc(&m->workspace, ws);
  if (e == cudaSuccess) e = cudaMallocHost(&m->status_host, sizeof(int));
  if (e != cudaSuccess) {
    delete m;
    return fail(NC_ERR_CUDA, "cudaMalloc of %zu + %zu bytes failed: %s", wb, ws,
                cudaGetErrorString(e));
  }
  m->weight_bytes = wb;
  m->workspace_bytes = ws;
  Arena A{static_cast<char*>(m->weights)}, W{static_cast<char*>(m->workspace)};
  layout(A, W);

  auto copy = [&](void* dst, const void* src, size_t bytes) -> cudaError_t {
    return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, s);
  };
  e = cudaSuccess;
  for (int l = 0; l < c.n_layers && e == cudaSuccess; ++l) {
    const nc_layer_weights& L = w->layers[l];
    const LayerPacked& P = m->layers[l];
    const uint16_t* wq = static_cast<const uint16_t*>(L.wq);
    const uint16_t* wk = static_cast<const uint16_t*>(L.wk);
    const uint16_t* wv = static_cast<const uint16_t*>(L.wv);
    const uint16_t* wo = static_cast<const uint16_t*>(L.wo);
    const uint16_t* wg = static_cast<const uint16_t*>(L.wg);
    const uint16_t* wu = static_cast<const uint16_t*>(L.wu);
    const uint16_t* wd = static_cast<const uint16_t*>(L.wd);
    if (g4) {
      auto q4 = [&](const uint16_t* src, int rows, int k, uint8_t* p, float* sc) {
        if (!e) e = launch_quantize_int4(src, rows, k, g4, p, sc, s);
      };
      q4(wq, (int)qd, H, P.p4_qkv, P.s4_qkv);
      q4(wk, (int)kd, H, P.p4_qkv + qd * H / 2, P.s4_qkv + qd * (H / g4));
      q4(wv, (int)kd, H, P.p4_qkv + (qd + kd) * H / 2, P.s4_qkv + (qd + kd) * (H / g4));
      q4(wo, H, (int)qd, P.p4_o, P.s4_o);
      q4(wg, F, H, P.p4_gu, P.s4_gu);
      q4(wu, F, H, P.p4_gu + (size_t)F * H / 2, P.s4_gu + (size_t)F * (H / g4));
      q4(wd, H, F, P.p4_d, P.s4_d);
    } else if (!i8) {
      if (!e) e = copy(P.w_qkv, wq, qd * H * 2);
      if (!e) e = copy(P.w_qkv + qd * H, wk, kd * H * 2);
      if (!e) e = copy(P.w_qkv + (qd + kd) * H, wv, kd * H * 2);
      if (!e) e = copy(P.w_o, wo, qd * H * 2);
      if (!e) e = copy(P.w_gu, wg, (size_t)F * H * 2);
      if (!e) e = copy(P.w_gu + (size_t)F * H, wu, (size_t)F * H * 2);
      if (!e) e = copy(P.w_d, wd, (size_t)H * F * 2);
    } else {
      if (!e) e = launch_quantize_weight(wq, (int)qd, H, P.q_qkv, P.s_qkv, s);
      if (!e) e = launch_quantize_weight(wk, (int)kd, H, P.q_qkv + qd * H, P.s_qkv + qd, s);
      if (!e) e = launch_quantize_weight(wv, (int)kd, H, P.q_qkv + (qd + kd) * H, P.s_qkv + qd + kd, s);
      if (!e) e = launch_quantize_weight(wo, H, (int)qd, P.q_o, P.s_o, s);
      if (!e) e = launch_quantize_weight(wg, F, H, P.q_gu, P.s_gu, s);
      if (!e) e = launch_quantize_weight(wu, F, H, P.q_gu + (size_t)F * H, P.s_gu + F, s);
      if (!e) e = launch_quantize_weight(wd, H, F, P.q_d, P.s_d, s);
    }
    if (c.qkv_bias) {
      if (!e) e = copy(P.b_qkv, L.bq, qd * 2);
      if (!e) e = copy(P.b_qkv + qd, L.bk, kd * 2);
      if (!e) e = copy(P.b_qkv + qd + kd, L.bv, kd * 2);
    }
    if (!e) e = copy(P.g_attn, L.g_attn, (size_t)H * 2);
    if (!e) e = copy(P.g_mlp, L.g_mlp, (size_t)H * 2);
    if (c.qk_norm) {
      if (!e) e = copy(P.g_q, L.g_q, (size_t)D * 2);
      if (!e) e = copy(P.g_k, L.g_k, (size_t)D * 2);
    }
  }
  if (b32) {
    if (!e)
      e = launch_quantize_weight(static_cast<const uint16_t*>(w->embed), c.vocab, H, m->q_embed,
                                 m->s_embed, s);
  } else if (!e) {
    e = copy(m->embed, w->embed, (size_t)c.vocab * H * 2);
  }
  if (!c.tie_embeddings && !e) e = copy(m->head, w->lm_head, (size_t)c.vocab * H * 2);
  if (!e) e = copy(m->g_final, w->g_final, (size_t)H * 2);
  // RoPE frequencies: float(1 / theta^(2i/D)), evaluated in double on the host.
  std::vector<float> inv(D / 2);
  for (int i = 0; i < D / 2; ++i) inv[i] = (float)(1.0 / pow((double)c.rope_theta, (2.0 * i) / D));
  if (!e) e = cudaMemcpyAsync(m->inv_freq, inv.data(), inv.size() * 4, cudaMemcpyHostToDevice, s);
  // per-layer pointers for the persistent kernel
  std::vector<PLayer> pl(c.n_layers);
  for (int l = 0; l < c.n_layers; ++l) {
    const LayerPacked& P = m->layers[l];
    pl[l] = PLayer{P.w_qkv, P.b_qkv, P.w_o, P.w_gu, P.w_d, P.g_attn, P.g_mlp, P.g_q, P.g_k};
  }
  if (!e) e = cudaMemcpyAsync(m->players, pl.data(), pl.size() * sizeof(PLayer),
                              cudaMemcpyHostToDevice, s);
  if (!e) e = cudaMemsetAsync(m->workspace, 0, ws, s);
  // The step sequence starts at 1: epoch 0 would match the zeroed hand-over words.
  const unsigned one = 1u;
  if (!e) e = cudaMemcpyAsync(m->seq, &one, sizeof one, cudaMemcpyHostToDevice, s);
  if (!e) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    delete m;
    return fail(NC_ERR_CUDA, "packing the weights failed: %s", cudaGetErrorString(e));
  }
  *out = m;
  return NC_OK;
}

// The persistent kernel serves bf16 weights and small batches, at any cache
// length (long scans are split over the grid).
bool use_persistent(const Model* m, int batch, const nc_kv_cache& kv, int flags) {
  const nc_config& c = m->cfg;
  (void)kv;
  return !(flags & NC_STEP_STAGED) && c.wtype == NC_BF16 && batch <= kPMaxBatch &&
         persistent_supported(c.n_layers, c.hidden, c.n_q_heads * c.head_dim, c.ffn, c.head_dim,
                              c.n_q_heads / c.n_kv_heads, batch);
}

static cudaError_t enqueue_persistent(Model* m, int batch, int32_t* tokens, int32_t* positions,
                                      float* logits, int32_t* next, bool advance,
                                      const KVView& kvv, cudaStream_t s) {
  const nc_config& c = m->cfg;
  PersistArgs a{};
  a.layers = m->players;
  a.L = c.n_layers;
  a.embed = m->embed;
  a.head = m->head;
  a.g_final = m->g_final;
  a.inv_freq = m->inv_freq;
  a.H = c.hidden;
  a.Hq = c.n_q_heads;
  a.Hkv = c.n_kv_heads;
  a.D = c.head_dim;
  a.F = c.ffn;
  a.V = c.vocab;
  a.nqkv = (c.n_q_heads + 2 * c.n_kv_heads) * c.head_dim;
  a.eps = c.rms_eps;
  a.B = batch;
  a.tokens = tokens;
  a.positions = positions;
  a.logits = logits;
  a.next = next;
  a.advance = advance ? 1 : 0;
  a.kv = kvv;
  a.xw = m->xw;
  a.qkvw = m->qkvw;
  a.aw = m->aw;
  a.apart = m->apart;
  a.atick = m->atick;
  a.hw = m->hw;
  a.am_part = m->am_part;
  a.ticket = m->pticket;
  a.seq = m->seq;
  a.status = m->status;
  a.timeout_ns = 200ull * 1000 * 1000;  // 200 ms; a step takes well under 10 ms
  a.grid = num_sms();
  a.prof = m->prof_on ? m->prof : nullptr;
  return launch_persistent(a, s);
}

// ------------------------------------------------------------------ step
KVView kv_view(const Model* m, const nc_kv_cache& kv) {
  KVView v;
  v.k = kv.k;
  v.v = kv.v;
  v.block_table = kv.block_table;
  v.paged = kv.paged;
  v.bf16 = kv.dtype == NC_KV_BF16;
  v.batch_capacity = kv.batch_capacity;
  v.max_ctx = kv.max_ctx;
  v.block_size = kv.block_size;
  v.num_blocks = kv.num_blocks;
  v.max_blocks_per_seq = kv.max_blocks_per_seq;
  v.n_kv_heads = m->cfg.n_kv_heads;
  v.head_dim = m->cfg.head_dim;
  return v;
}

int kv_capacity(const nc_kv_cache& kv) {
  return kv.paged ? kv.max_blocks_per_seq * kv.block_size : kv.max_ctx;
}

nc_status validate_kv(const Model* m, int batch, const int32_t* positions_host,
                      const nc_kv_cache* kv) {
  NC_CHECK(kv && kv->k && kv->v, NC_ERR_INVALID_ARGUMENT, "kv cache pointers are NULL");
  NC_CHECK(kv->dtype == NC_KV_F32 || kv->dtype == NC_KV_BF16, NC_ERR_DTYPE,
           "unknown kv dtype %d", (int)kv->dtype);
  NC_CHECK(reinterpret_cast<uintptr_t>(kv->k) % 16 == 0 && reinterpret_cast<uintptr_t>(kv->v) % 16 == 0,
           NC_ERR_INVALID_ARGUMENT, "kv cache pointers must be 16-byte aligned");
  NC_CHECK(positions_host, NC_ERR_INVALID_ARGUMENT, "positions_host is NULL");
  const int cap = kv_capacity(*kv);
  NC_CHECK(cap >= 1 && cap <= m->max_ctx, NC_ERR_CAPACITY,
           "kv capacity %d outside [1, %d] reserved at model creation", cap, m->max_ctx);
  if (!kv->paged) {
    NC_CHECK(kv->batch_capacity >= batch, NC_ERR_CAPACITY, "kv batch_capacity %d < batch %d",
             kv->batch_capacity, batch);
  } else {
    NC_CHECK(kv->block_table && kv->block_table_host, NC_ERR_INVALID_ARGUMENT,
             "paged cache needs block_table and block_table_host");
    NC_CHECK(kv->block_size >= 1 && kv->num_blocks >= 1 && kv->max_blocks_per_seq >= 1,
             NC_ERR_SHAPE, "paged cache sizes must be positive");
  }
  for (int b = 0; b < batch; ++b) {
    const int p = positions_host[b];
    NC_CHECK(p >= 0 && p < cap, NC_ERR_POSITION, "position %d of sequence %d outside [0, %d)", p,
             b, cap);
    if (kv->paged) {
      for (int i = 0; i <= p / kv->block_size; ++i) {
        const int blk = kv->block_table_host[(size_t)b * kv->max_blocks_per_seq + i];
        NC_CHECK(blk >= 0 && blk < kv->num_blocks, NC_ERR_POSITION,
                 "block table entry %d of sequence %d is %d (pool has %d blocks)", i, b, blk,
                 kv->num_blocks);
      }
    }
  }
  return NC_OK;
}

// The W8A8 diagnostic's layout for one step at `batch`: per layer the codes
// of the four products [qkv: B x H][o: B x Hq D][gate|up: B x H][down: B x F]
// and their scales [4][B].
size_t dbg_codes_per_step(const Model* m, int batch) {
  const nc_config& c = m->cfg;
  // the blocked mode's int8 head quantises the final norm too: [B][H] last
  return (size_t)c.n_layers * batch *
             (2 * (size_t)c.hidden + (size_t)c.n_q_heads * c.head_dim + c.ffn) +
         (c.wtype == NC_INT8_B32 ? (size_t)batch * c.hidden : 0);
}
size_t dbg_scales_per_step(const Model* m, int batch) {
  // per-token scales (the blocked mode's per-block scales are not captured)
  return m->cfg.wtype == NC_INT8 ? (size_t)m->cfg.n_layers * 4 * batch : 0;
}

// Batch 9..16 with bf16 weights runs the projections and the LM head on the
// tensor cores (tcgen05); NC_UMMA=0 in the environment uses the CUDA-core
// and mma.sync stage kernels instead (for comparison).
static bool umma_enabled() {
  static const bool on = [] {
    const char* e = getenv("NC_UMMA");
    return !(e && e[0] == '0');
  }();
  return on;
}
static bool use_umma(const Model* m, int batch) {
  const nc_config& c = m->cfg;
  return umma_enabled() && m->xb && batch > 8 && c.wtype == NC_BF16 && umma_supported(c.hidden) &&
         umma_supported(c.ffn) && umma_supported(c.n_q_heads * c.head_dim);
}
// The tensor-core scratch, aligned for TMA (1024 bytes).
static uint16_t* xb_aligned(const Model* m) {
  return reinterpret_cast<uint16_t*>((reinterpret_cast<uintptr_t>(m->xb) + 1023) &
                                     ~uintptr_t(1023));
}

static cudaError_t enqueue_block(Model* m, int layer, int batch, const int32_t* positions,
                                 const KVView& kvv, int splits, cudaStream_t s) {
  const nc_config& c = m->cfg;
  const LayerPacked& P = m->layers[layer];
  const int H = c.hidden, D = c.head_dim, F = c.ffn, Hq = c.n_q_heads, Hkv = c.n_kv_heads;
  const int nqkv = (Hq + 2 * Hkv) * D;
  const bool i8 = c.wtype == NC_INT8 || c.wtype == NC_INT8_B32;
  const bool b32 = c.wtype == NC_INT8_B32;
  // the W8A8 diagnostic's slots of this layer (null when it is off)
  int8_t* dq[4] = {nullptr, nullptr, nullptr, nullptr};
  float* ds[4] = {nullptr, nullptr, nullptr, nullptr};
  if (i8 && m->dbg_codes) {
    const size_t per = (size_t)batch * (2 * (size_t)H + (size_t)Hq * D + F);
    int8_t* base = m->dbg_codes + (size_t)layer * per;
    dq[0] = base;
    dq[1] = dq[0] + (size_t)batch * H;
    dq[2] = dq[1] + (size_t)batch * Hq * D;
    dq[3] = dq[2] + (size_t)batch * H;
    if (!b32 && m->dbg_scales)
      for (int k = 0; k < 4; ++k) ds[k] = m->dbg_scales + ((size_t)layer * 4 + k) * batch;
  }
  const int g4 = c.wtype == NC_INT4_G32 ? 32 : c.wtype == NC_INT4_G128 ? 128 : 0;
  cudaError_t e;
  if (g4) {
    Int4Args a{m->x, P.g_attn, c.rms_eps, P.p4_qkv, P.s4_qkv, g4, batch, H, nqkv, m->qkv, P.b_qkv};
    e = launch_int4_gemv(Epi::Store, a, s);
  } else if (!i8 && use_umma(m, batch)) {
    UmmaArgs u{m->x, P.g_attn, c.rms_eps, P.w_qkv, P.b_qkv, batch, H, nqkv, m->qkv, nqkv,
               xb_aligned(m)};
    e = launch_umma(Epi::Store, u, s);
  } else if (!i8) {
    e = launch_gemv(Epi::Store, {m->x, P.g_attn, c.rms_eps, P.w_qkv, P.b_qkv, batch, H, nqkv, m->qkv}, s);
  } else if (b32) {
    W8BArgs a{m->x, P.g_attn, c.rms_eps, P.q_qkv, P.s_qkv, P.b_qkv, batch, H, nqkv, m->qkv,
              dq[0], nullptr, nullptr};
    e = launch_w8a8_b32(Epi::Store, a, s);
  } else {
    W8Args a{m->x, P.g_attn, c.rms_eps, P.q_qkv, P.s_qkv, P.b_qkv, batch, H, nqkv, m->qkv,
             dq[0], ds[0], nullptr};
    e = launch_w8a8(Epi::Store, a, s);
  }
  if (e) return e;
  // RoPE (+ q/k norm) and the K/V append run inside the attention launch
  AttnArgs at{m->q, positions, batch, Hq, Hkv, D, layer, splits, m->part, m->attn, kvv, m->status,
              m->atickets};
  at.qkv = m->qkv;
  at.inv_freq = m->inv_freq;
  at.g_q = P.g_q;
  at.g_k = P.g_k;
  at.eps = c.rms_eps;
  if ((e = launch_attn(at, s))) return e;
  if (g4) {
    Int4Args o{m->attn, nullptr, 0.f, P.p4_o, P.s4_o, g4, batch, Hq * D, H, m->x};
    if ((e = launch_int4_gemv(Epi::Residual, o, s))) return e;
    Int4Args gu{m->x, P.g_mlp, c.rms_eps, P.p4_gu, P.s4_gu, g4, batch, H, F, m->h};
    if ((e = launch_int4_gemv(Epi::SwiGLU, gu, s))) return e;
    Int4Args dn{m->h, nullptr, 0.f, P.p4_d, P.s4_d, g4, batch, F, H, m->x};
    return launch_int4_gemv(Epi::Residual, dn, s);
  }
  if (!i8 && use_umma(m, batch)) {
    uint16_t* xb = xb_aligned(m);
    UmmaArgs o{m->attn, nullptr, 0.f, P.w_o, nullptr, batch, Hq * D, H, m->x, H, xb};
    if ((e = launch_umma(Epi::Residual, o, s))) return e;
    UmmaArgs gu{m->x, P.g_mlp, c.rms_eps, P.w_gu, nullptr, batch, H, F, m->h, F, xb};
    if ((e = launch_umma(Epi::SwiGLU, gu, s))) return e;
    UmmaArgs dn{m->h, nullptr, 0.f, P.w_d, nullptr, batch, F, H, m->x, H, xb};
    return launch_umma(Epi::Residual, dn, s);
  }
  if (!i8) {
    if ((e = launch_gemv(Epi::Residual, {m->attn, nullptr, 0.f, P.w_o, nullptr, batch, Hq * D, H, m->x}, s)))
      return e;
    if ((e = launch_gemv(Epi::SwiGLU, {m->x, P.g_mlp, c.rms_eps, P.w_gu, nullptr, batch, H, F, m->h}, s)))
      return e;
    return launch_gemv(Epi::Residual, {m->h, nullptr, 0.f, P.w_d, nullptr, batch, F, H, m->x}, s);
  }
  if (b32) {
    W8BArgs o{m->attn, nullptr, 0.f, P.q_o, P.s_o, nullptr, batch, Hq * D, H, m->x,
              dq[1], nullptr, nullptr};
    if ((e = launch_w8a8_b32(Epi::Residual, o, s))) return e;
    W8BArgs gu{m->x, P.g_mlp, c.rms_eps, P.q_gu, P.s_gu, nullptr, batch, H, F, m->h,
               dq[2], nullptr, nullptr};
    if ((e = launch_w8a8_b32(Epi::SwiGLU, gu, s))) return e;
    W8BArgs dn{m->h, nullptr, 0.f, P.q_d, P.s_d, nullptr, batch, F, H, m->x,
               dq[3], nullptr, nullptr};
    return launch_w8a8_b32(Epi::Residual, dn, s);
  }
  W8Args o{m->attn, nullptr, 0.f, P.q_o, P.s_o, nullptr, batch, Hq * D, H, m->x, dq[1], ds[1], nullptr};
  if ((e = launch_w8a8(Epi::Residual, o, s))) return e;
  W8Args gu{m->x, P.g_mlp, c.rms_eps, P.q_gu, P.s_gu, nullptr, batch, H, F, m->h, dq[2], ds[2], nullptr};
  if ((e = launch_w8a8(Epi::SwiGLU, gu, s))) return e;
  W8Args dn{m->h, nullptr, 0.f, P.q_d, P.s_d, nullptr, batch, F, H, m->x, dq[3], ds[3], nullptr};
  return launch_w8a8(Epi::Residual, dn, s);
}

struct StepIO {
  int32_t* tokens;
  int32_t* positions;
  float* logits;
  int32_t* next;
  bool advance;
};

static cudaError_t enqueue_step(Model* m, int batch, const StepIO& io, const KVView& kvv,
                                int splits, cudaStream_t s) {
  const nc_config& c = m->cfg;
  const bool b32 = c.wtype == NC_INT8_B32;
  cudaError_t e = b32 ? launch_embed_i8(m->q_embed, m->s_embed, io.tokens, batch, c.hidden,
                                        c.vocab, m->x, m->status, s)
                      : launch_embed(m->embed, io.tokens, batch, c.hidden, c.vocab, m->x,
                                     m->status, s);
  if (e) return e;
  for (int l = 0; l < c.n_layers; ++l)
    if ((e = enqueue_block(m, l, batch, io.positions, kvv, splits, s))) return e;
  if (b32) {  // the int8 head: the blocked W8A8 product of the final norm, with the arg-max
    int8_t* hq = m->dbg_codes
                     ? m->dbg_codes + (size_t)c.n_layers * batch *
                                          (2 * (size_t)c.hidden + (size_t)c.n_q_heads * c.head_dim + c.ffn)
                     : nullptr;  // the W8A8 diagnostic's head slot
    W8BArgs h{m->x, m->g_final, c.rms_eps, m->q_embed, m->s_embed, nullptr, batch, c.hidden,
              c.vocab, io.logits, hq, nullptr, nullptr};
    h.part = m->am_part;
    h.ticket = m->ticket;
    h.next = io.next;
    h.status = m->status;
    h.advance_tokens = io.advance ? io.tokens : nullptr;
    h.advance_positions = io.advance ? io.positions : nullptr;
    return launch_w8a8_b32(Epi::Store, h, s);
  }
  if (use_umma(m, batch)) {  // logits and the arg-max on the tensor cores
    UmmaArgs u{m->x, m->g_final, c.rms_eps, m->head, nullptr, batch, c.hidden, c.vocab,
               io.logits, c.vocab, xb_aligned(m)};
    u.lm = true;
    u.part = m->am_part;
    u.ticket = m->ticket;
    u.next = io.next;
    u.status = m->status;
    u.advance_tokens = io.advance ? io.tokens : nullptr;
    u.advance_positions = io.advance ? io.positions : nullptr;
    return launch_umma(Epi::Store, u, s);
  }
  LmHeadArgs a{m->x, m->g_final, c.rms_eps, m->head, batch, c.hidden, c.vocab, io.logits, io.next,
               m->am_part, m->ticket, m->status, io.advance ? io.tokens : nullptr,
               io.advance ? io.positions : nullptr};
  return launch_lm_head(a, s);
}

nc_status decode_step(Model* m, int batch, int32_t* tokens, int32_t* positions,
                      const int32_t* positions_host, const nc_kv_cache* kv, float* logits,
                      int32_t* next, int flags, cudaStream_t s) {
  NC_CHECK(m, NC_ERR_INVALID_ARGUMENT, "model is NULL");
  NC_CHECK(!m->unhealthy, NC_ERR_UNHEALTHY, "model saw an earlier CUDA failure");
  NC_CHECK(batch >= 1 && batch <= m->max_batch, NC_ERR_CAPACITY, "batch %d outside [1, %d]",
           batch, m->max_batch);
  NC_CHECK(tokens && positions && logits, NC_ERR_INVALID_ARGUMENT, "null device pointer");
  NC_CHECK(reinterpret_cast<uintptr_t>(tokens) % 4 == 0 &&
               reinterpret_cast<uintptr_t>(positions) % 4 == 0 &&
               reinterpret_cast<uintptr_t>(logits) % 4 == 0 &&
               reinterpret_cast<uintptr_t>(next) % 4 == 0,
           NC_ERR_INVALID_ARGUMENT, "tokens, positions, logits and next must be 4-byte aligned");
  NC_CHECK((flags & ~(NC_STEP_GRAPH | NC_STEP_ADVANCE | NC_STEP_STAGED)) == 0,
           NC_ERR_INVALID_ARGUMENT,
           "unknown flags 0x%x", flags);
  nc_status st = validate_kv(m, batch, positions_host, kv);
  if (st) return st;
  const KVView kvv = kv_view(m, *kv);
  const int splits = attn_splits(batch, m->cfg.n_kv_heads, m->cfg.head_dim, kv->dtype == NC_KV_BF16,
                                 kv_capacity(*kv));
  const StepIO io{tokens, positions, logits, next, (flags & NC_STEP_ADVANCE) != 0};
  if (m->dbg_codes) {
    NC_CHECK(dbg_codes_per_step(m, batch) <= m->dbg_codes_cap &&
                 (!m->dbg_scales || dbg_scales_per_step(m, batch) <= m->dbg_scales_cap),
             NC_ERR_CAPACITY, "the W8A8 diagnostic buffers are too small for batch %d", batch);
    flags &= ~NC_STEP_GRAPH;  // the diagnostic runs the kernels directly
  }
  cudaError_t e;
  if (use_persistent(m, batch, *kv, flags)) {
    e = enqueue_persistent(m, batch, tokens, positions, logits, next, io.advance, kvv, s);
  } else if (!(flags & NC_STEP_GRAPH)) {
    e = enqueue_step(m, batch, io, kvv, splits, s);
  } else {
    GraphKey key{batch, tokens, positions, logits, next, kv->k, kv->v, kv->block_table,
                 kv->paged, kv->batch_capacity, kv->max_ctx, kv->block_size, kv->num_blocks,
                 kv->max_blocks_per_seq, (int)io.advance, (int)kv->dtype};
    auto it = m->graphs.find(key);
    if (it == m->graphs.end()) {
      if (m->graphs.size() >= kMaxGraphs) {
        // evict the least recently used graph; a launch of it may still be
        // in flight on another stream, so the device drains first (rare)
        auto old = m->graphs.begin();
        for (auto g = m->graphs.begin(); g != m->graphs.end(); ++g)
          if (g->second.used < old->second.used) old = g;
        e = cudaDeviceSynchronize();
        if (!e) e = cudaGraphExecDestroy(old->second.exec);
        if (e) {
          m->unhealthy = true;
          return fail(NC_ERR_CUDA, "evicting a step graph failed: %s", cudaGetErrorString(e));
        }
        m->graphs.erase(old);
      }
      // First use: launch once eagerly (sets per-kernel attributes), then capture.
      e = enqueue_step(m, batch, io, kvv, splits, s);
      if (!e) e = cudaStreamSynchronize(s);
      if (e) {
        m->unhealthy = true;
        return fail(NC_ERR_CUDA, "decode step launch failed: %s", cudaGetErrorString(e));
      }
      cudaGraph_t g = nullptr;
      cudaGraphExec_t ge = nullptr;
      // Capture on the model's own stream: the legacy default stream cannot be
      // captured, and capturing executes nothing.
      if (!e && !m->cap_stream) e = cudaStreamCreateWithFlags(&m->cap_stream, cudaStreamNonBlocking);
      if (!e) e = cudaStreamBeginCapture(m->cap_stream, cudaStreamCaptureModeThreadLocal);
      if (!e) {
        cudaError_t e2 = enqueue_step(m, batch, io, kvv, splits, m->cap_stream);
        e = cudaStreamEndCapture(m->cap_stream, &g);
        if (!e) e = e2;
      }
      if (!e) e = cudaGraphInstantiate(&ge, g, 0);
      if (g) cudaGraphDestroy(g);
      if (e) {
        m->unhealthy = true;
        return fail(NC_ERR_CUDA, "graph capture failed: %s", cudaGetErrorString(e));
      }
      it = m->graphs.emplace(key, Model::GraphEntry{ge, ++m->graph_clock}).first;
      // The eager launch above already performed this step; its KV writes and
      // logits are identical to a replay, so the replay is skipped.
      return NC_OK;
    }
    it->second.used = ++m->graph_clock;
    e = cudaGraphLaunch(it->second.exec, s);
  }
  if (e) {
    m->unhealthy = true;
    return fail(NC_ERR_CUDA, "decode step launch failed: %s", cudaGetErrorString(e));
  }
  return NC_OK;
}

nc_status block_forward(Model* m, int layer, int batch, float* x, const int32_t* positions,
                        const int32_t* positions_host, const nc_kv_cache* kv, cudaStream_t s) {
  NC_CHECK(m, NC_ERR_INVALID_ARGUMENT, "model is NULL");
  NC_CHECK(!m->unhealthy, NC_ERR_UNHEALTHY, "model saw an earlier CUDA failure");
  NC_CHECK(layer >= 0 && layer < m->cfg.n_layers, NC_ERR_SHAPE, "layer %d outside [0, %d)", layer,
           m->cfg.n_layers);
  NC_CHECK(batch >= 1 && batch <= m->max_batch, NC_ERR_CAPACITY, "batch %d outside [1, %d]",
           batch, m->max_batch);
  NC_CHECK(x && positions, NC_ERR_INVALID_ARGUMENT, "null device pointer");
  NC_CHECK(reinterpret_cast<uintptr_t>(positions) % 4 == 0, NC_ERR_INVALID_ARGUMENT,
           "positions must be 4-byte aligned");
  nc_status st = validate_kv(m, batch, positions_host, kv);
  if (st) return st;
  NC_CHECK(!m->dbg_codes || (dbg_codes_per_step(m, batch) <= m->dbg_codes_cap &&
                             (!m->dbg_scales ||
                              dbg_scales_per_step(m, batch) <= m->dbg_scales_cap)),
           NC_ERR_CAPACITY, "the W8A8 diagnostic buffers are too small for batch %d", batch);
  const KVView kvv = kv_view(m, *kv);
  const int splits = attn_splits(batch, m->cfg.n_kv_heads, m->cfg.head_dim, kv->dtype == NC_KV_BF16,
                                 kv_capacity(*kv));
  cudaError_t e = cudaMemcpyAsync(m->x, x, (size_t)batch * m->cfg.hidden * 4,
                                  cudaMemcpyDeviceToDevice, s);
  if (!e) e = enqueue_block(m, layer, batch, positions, kvv, splits, s);
  if (!e)
    e = cudaMemcpyAsync(x, m->x, (size_t)batch * m->cfg.hidden * 4, cudaMemcpyDeviceToDevice, s);
  if (e) {
    m->unhealthy = true;
    return fail(NC_ERR_CUDA, "block launch failed: %s", cudaGetErrorString(e));
  }
  return NC_OK;
}

}  // namespace nc

// ------------------------------------------------------------------ prefill
namespace nc {

// Scratch of a prefill chunk of T tokens: residual x [T][H], projections
// [T][(Hq + 2 Hkv) D], rotated q and attention output [T][Hq D], SiLU * up
// [T][F], and the tensor-core activation planes; pieces 1024-byte aligned.
struct PrefillPlan {
  size_t x, qkv, q, attn, h, xb, total;
};
static PrefillPlan prefill_plan(const Model* m, int T) {
  const nc_config& c = m->cfg;
  const size_t qd = (size_t)c.n_q_heads * c.head_dim, nqkv = qd + 2 * (size_t)c.n_kv_heads * c.head_dim;
  const int kmax = std::max(std::max(c.hidden, c.ffn), (int)qd);
  PrefillPlan p{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, 1024);
    return at;
  };
  p.x = take((size_t)T * c.hidden * 4);
  p.qkv = take((size_t)T * nqkv * 4);
  p.q = take((size_t)T * qd * 4);
  p.attn = take((size_t)T * qd * 4);
  p.h = take((size_t)T * c.ffn * 4);
  p.xb = take(umma_act_bytes(T, kmax));
  p.total = off + 1024;  // room to align the caller's base
  return p;
}

size_t prefill_scratch_bytes(const Model* m, int T) { return prefill_plan(m, T).total; }

nc_status prefill(Model* m, int seq, int T, const int32_t* tokens, int start,
                  const nc_kv_cache* kv, float* logits, int32_t* next, void* scratch,
                  size_t scratch_bytes, cudaStream_t s) {
  NC_CHECK(m, NC_ERR_INVALID_ARGUMENT, "model is NULL");
  NC_CHECK(!m->unhealthy, NC_ERR_UNHEALTHY, "model saw an earlier CUDA failure");
  const nc_config& c = m->cfg;
  NC_CHECK(c.wtype == NC_BF16, NC_ERR_UNSUPPORTED, "prefill runs bf16 weights only");
  NC_CHECK(umma_supported(c.hidden) && umma_supported(c.ffn) &&
               umma_supported(c.n_q_heads * c.head_dim),
           NC_ERR_SHAPE, "prefill needs hidden, ffn and n_q_heads * head_dim multiples of 64");
  NC_CHECK(tokens && logits && scratch, NC_ERR_INVALID_ARGUMENT, "null pointer");
  NC_CHECK(reinterpret_cast<uintptr_t>(tokens) % 4 == 0 && reinterpret_cast<uintptr_t>(logits) % 4 == 0 &&
               reinterpret_cast<uintptr_t>(next) % 4 == 0 &&
               reinterpret_cast<uintptr_t>(scratch) % 16 == 0,
           NC_ERR_INVALID_ARGUMENT,
           "tokens, logits and next must be 4-byte aligned, scratch 16-byte aligned");
  NC_CHECK(T >= 1 && T <= 32768, NC_ERR_SHAPE, "T = %d outside [1, 32768]", T);
  NC_CHECK(start >= 0, NC_ERR_POSITION, "start position %d is negative", start);
  NC_CHECK(kv && kv->k && kv->v, NC_ERR_INVALID_ARGUMENT, "kv cache pointers are NULL");
  NC_CHECK(kv->dtype == NC_KV_F32 || kv->dtype == NC_KV_BF16, NC_ERR_DTYPE, "unknown kv dtype");
  NC_CHECK(reinterpret_cast<uintptr_t>(kv->k) % 16 == 0 && reinterpret_cast<uintptr_t>(kv->v) % 16 == 0,
           NC_ERR_INVALID_ARGUMENT, "kv cache pointers must be 16-byte aligned");
  const int cap = kv_capacity(*kv);
  NC_CHECK(cap >= 1 && cap <= m->max_ctx, NC_ERR_CAPACITY,
           "kv capacity %d outside [1, %d] reserved at model creation", cap, m->max_ctx);
  NC_CHECK((long long)start + T <= cap, NC_ERR_POSITION,
           "positions %d .. %d do not fit the cache's %d slots", start, start + T - 1, cap);
  NC_CHECK(seq >= 0, NC_ERR_INVALID_ARGUMENT, "sequence %d is negative", seq);
  if (!kv->paged) {
    NC_CHECK(seq < kv->batch_capacity, NC_ERR_CAPACITY, "sequence %d beyond batch_capacity %d",
             seq, kv->batch_capacity);
  } else {
    NC_CHECK(kv->block_table && kv->block_table_host && kv->block_size >= 1 &&
                 kv->num_blocks >= 1 && kv->max_blocks_per_seq >= 1,
             NC_ERR_INVALID_ARGUMENT, "paged cache needs block tables and positive sizes");
    for (int i = 0; i <= (start + T - 1) / kv->block_size; ++i) {
      const int blk = kv->block_table_host[(size_t)seq * kv->max_blocks_per_seq + i];
      NC_CHECK(blk >= 0 && blk < kv->num_blocks, NC_ERR_POSITION,
               "block table entry %d of sequence %d is %d (pool has %d blocks)", i, seq, blk,
               kv->num_blocks);
    }
  }
  const PrefillPlan p = prefill_plan(m, T);
  NC_CHECK(scratch_bytes >= p.total, NC_ERR_CAPACITY, "scratch holds %zu bytes, %zu needed",
           scratch_bytes, p.total);
  char* base = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(scratch) + 1023) &
                                       ~uintptr_t(1023));
  float* x = reinterpret_cast<float*>(base + p.x);
  float* qkv = reinterpret_cast<float*>(base + p.qkv);
  float* q = reinterpret_cast<float*>(base + p.q);
  float* attn = reinterpret_cast<float*>(base + p.attn);
  float* h = reinterpret_cast<float*>(base + p.h);
  uint16_t* xb = reinterpret_cast<uint16_t*>(base + p.xb);
  const int H = c.hidden, D = c.head_dim, F = c.ffn, Hq = c.n_q_heads, Hkv = c.n_kv_heads;
  const int qd = Hq * D, nqkv = (Hq + 2 * Hkv) * D;
  const KVView kvv = kv_view(m, *kv);

  cudaError_t e = launch_embed(m->embed, tokens, T, H, c.vocab, x, m->status, s);
  for (int l = 0; l < c.n_layers && !e; ++l) {
    const LayerPacked& P = m->layers[l];
    UmmaArgs u{x, P.g_attn, c.rms_eps, P.w_qkv, P.b_qkv, T, H, nqkv, qkv, nqkv, xb};
    if ((e = launch_umma(Epi::Store, u, s))) break;
    RopeArgs r{qkv, nullptr, m->inv_freq, P.g_q, P.g_k, c.rms_eps, T, Hq, Hkv, D, l, q, kvv,
               m->status};
    r.seq = seq;
    r.pos0 = start;
    if ((e = launch_rope_qkv(r, s))) break;
    PrefillAttnArgs at{q, attn, T, start, seq, l, Hq, Hkv, D, kvv};
    if ((e = launch_prefill_attn(at, s))) break;
    UmmaArgs o{attn, nullptr, 0.f, P.w_o, nullptr, T, qd, H, x, H, xb};
    if ((e = launch_umma(Epi::Residual, o, s))) break;
    UmmaArgs gu{x, P.g_mlp, c.rms_eps, P.w_gu, nullptr, T, H, F, h, F, xb};
    if ((e = launch_umma(Epi::SwiGLU, gu, s))) break;
    UmmaArgs dn{h, nullptr, 0.f, P.w_d, nullptr, T, F, H, x, H, xb};
    if ((e = launch_umma(Epi::Residual, dn, s))) break;
  }
  if (!e) {
    // logits of the last token only: the next token is all a prompt yields
    LmHeadArgs a{x + (size_t)(T - 1) * H, m->g_final, c.rms_eps, m->head, 1, H, c.vocab, logits,
                 next, m->am_part, m->ticket, m->status, nullptr, nullptr};
    e = launch_lm_head(a, s);
  }
  if (e) {
    m->unhealthy = true;
    return fail(NC_ERR_CUDA, "prefill launch failed: %s", cudaGetErrorString(e));
  }
  return NC_OK;
}

}  // namespace nc
