// engine.h -- the model object behind nc_model (internal).
#pragma once
#include <cuda_runtime.h>

#include <map>
#include <string>
#include <tuple>
#include <vector>

#include "kernels.h"
#include "persistent.h"

namespace nc {

constexpr size_t kMaxGraphs = 16;  // captured step graphs a model keeps

struct LayerPacked {
  uint16_t* w_qkv = nullptr;  // [(Hq + 2 Hkv) D, H] bf16 (NC_BF16)
  uint16_t* b_qkv = nullptr;  // [(Hq + 2 Hkv) D] or null
  uint16_t* w_o = nullptr;    // [H, Hq D]
  uint16_t* w_gu = nullptr;   // [2F, H]: gate rows then up rows
  uint16_t* w_d = nullptr;    // [H, F]
  int8_t *q_qkv = nullptr, *q_o = nullptr, *q_gu = nullptr, *q_d = nullptr;  // NC_INT8 rows
  float *s_qkv = nullptr, *s_o = nullptr, *s_gu = nullptr, *s_d = nullptr;   // per-row scales
  // NC_INT4_*: packed codes [rows, in / 2] and per-group scales [rows, in / group]
  uint8_t *p4_qkv = nullptr, *p4_o = nullptr, *p4_gu = nullptr, *p4_d = nullptr;
  float *s4_qkv = nullptr, *s4_o = nullptr, *s4_gu = nullptr, *s4_d = nullptr;
  uint16_t *g_attn = nullptr, *g_mlp = nullptr, *g_q = nullptr, *g_k = nullptr;
};

using GraphKey = std::tuple<int, const void*, const void*, const void*, const void*, const void*,
                            const void*, const void*, int, int, int, int, int, int, int, int>;

struct Model {
  nc_config cfg{};
  int max_batch = 0, max_ctx = 0;
  void* weights = nullptr;    // packed weight arena
  void* workspace = nullptr;  // workspace arena
  size_t weight_bytes = 0, workspace_bytes = 0;
  std::vector<LayerPacked> layers;
  uint16_t *embed = nullptr, *head = nullptr, *g_final = nullptr;
  int8_t* q_embed = nullptr;  // NC_INT8_B32: int8 embedding rows (also the tied head)
  float* s_embed = nullptr;   // [V] their scales
  float* inv_freq = nullptr;
  // workspace
  float *x = nullptr, *qkv = nullptr, *q = nullptr, *attn = nullptr, *part = nullptr, *h = nullptr;
  unsigned long long* am_part = nullptr;
  uint16_t* xb = nullptr;  // tensor-core activation planes (batch 9..16), or null
  unsigned int* ticket = nullptr;
  unsigned int* atickets = nullptr;  // [max_batch, Hkv] split-attention merge tickets
  int* status = nullptr;
  // persistent decode kernel: epoch-tagged hand-over words, its ticket, the
  // step sequence number and the device copy of the per-layer pointers
  uint64_t *xw = nullptr, *qkvw = nullptr, *aw = nullptr, *hw = nullptr;
  float* apart = nullptr;          // attention split partials
  unsigned int* atick = nullptr;   // attention split tickets [L][kPMaxBatch][Hkv]
  unsigned int *pticket = nullptr, *seq = nullptr;
  PLayer* players = nullptr;
  unsigned long long* prof = nullptr;  // phase profile [2 * (5L + 1) + 2]
  // W8A8 diagnostic (nc_debug_w8a8_codes): caller-owned device buffers that
  // receive every step's activation codes and scales, or null
  int8_t* dbg_codes = nullptr;
  float* dbg_scales = nullptr;
  size_t dbg_codes_cap = 0, dbg_scales_cap = 0;
  bool prof_on = false;
  bool unhealthy = false;
  cudaStream_t cap_stream = nullptr;  // private stream used only for graph capture
  int* status_host = nullptr;         // pinned host copy of the status word
  // Captured step graphs by (batch, buffers, cache layout), each with the
  // stamp of its last use; at most kMaxGraphs are kept (least recently used
  // evicted), so a caller that rotates buffers does not grow the cache.
  struct GraphEntry {
    cudaGraphExec_t exec;
    unsigned long long used;
  };
  std::map<GraphKey, GraphEntry> graphs;
  unsigned long long graph_clock = 0;
  ~Model();
};

bool valid_config(const nc_config& c, std::string* why);
nc_status model_create(const nc_config* cfg, const nc_weights* w, int max_batch, int max_ctx,
                       cudaStream_t s, Model** out);
KVView kv_view(const Model* m, const nc_kv_cache& kv);
int kv_capacity(const nc_kv_cache& kv);
nc_status validate_kv(const Model* m, int batch, const int32_t* positions_host,
                      const nc_kv_cache* kv);
nc_status decode_step(Model* m, int batch, int32_t* tokens, int32_t* positions,
                      const int32_t* positions_host, const nc_kv_cache* kv, float* logits,
                      int32_t* next, int flags, cudaStream_t s);
// True when a decode step with these arguments runs as the persistent kernel.
bool use_persistent(const Model* m, int batch, const nc_kv_cache& kv, int flags);
nc_status block_forward(Model* m, int layer, int batch, float* x, const int32_t* positions,
                        const int32_t* positions_host, const nc_kv_cache* kv, cudaStream_t s);
// A prompt chunk of T tokens of sequence `seq` at positions start .. start +
// T - 1 as one forward pass (tensor-core projections, flash-style causal
// attention); logits of the last token. Scratch is caller-owned.
size_t prefill_scratch_bytes(const Model* m, int T);
nc_status prefill(Model* m, int seq, int T, const int32_t* tokens, int start,
                  const nc_kv_cache* kv, float* logits, int32_t* next, void* scratch,
                  size_t scratch_bytes, cudaStream_t s);
// Codes and scales the W8A8 diagnostic holds for one step at this batch.
size_t dbg_codes_per_step(const Model* m, int batch);
size_t dbg_scales_per_step(const Model* m, int batch);

}  // namespace nc
