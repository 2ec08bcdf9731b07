// persistent.h -- launch interface of the persistent decode kernel (internal).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "nc_internal.cuh"

namespace nc {

constexpr int kMaxSlots = 8;           // weight ring slots (shared memory)
constexpr int kPMaxBatch = 4;          // sequences per persistent step
constexpr int kPSlots = 3;                // weight ring slots; they share what shared memory is left
constexpr int kPMinSlotBytes = 32 * 1024; // smallest slot the kernel is run with
constexpr int kPMaxRows = 128;         // rows of H one CTA may own (H <= 128 * grid)
constexpr int kPMaxLayers = 64;        // layers the persistent kernel handles
constexpr int kPMaxSplits = 32;        // attention position splits per (sequence, kv head)
constexpr int kPMaxHeads = 64;         // query heads

// Per-layer packed weights as the persistent kernel reads them.
struct PLayer {
  const uint16_t *w_qkv, *b_qkv, *w_o, *w_gu, *w_d, *g_attn, *g_mlp, *g_q, *g_k;
};

struct PersistArgs {
  const PLayer* layers;  // device array [L]
  int L;
  const uint16_t* embed;
  const uint16_t* head;
  const uint16_t* g_final;
  const float* inv_freq;
  int H, Hq, Hkv, D, F, V, nqkv;
  float eps;
  int B;
  int32_t* tokens;
  int32_t* positions;
  float* logits;
  int32_t* next;
  int advance;
  KVView kv;
  // epoch-tagged hand-over words (value in the low half, epoch in the high)
  uint64_t* xw;    // [kPMaxBatch][H] residual stream
  uint64_t* qkvw;  // [kPMaxBatch][nqkv]
  uint64_t* aw;    // [kPMaxBatch][Hq D] attention output (merged over the position splits)
  float* apart;    // [kPMaxBatch][kPMaxSplits][Hq][D + 4] split partials (o = acc / l, m, l)
  unsigned int* atick;  // [L][kPMaxBatch][Hkv] split arrivals, zeroed by the step's last CTA
  uint64_t* hw;    // [kPMaxBatch][F] SiLU(gate) * up
  unsigned long long* am_part;  // [B][grid] arg-max partial keys
  unsigned int* ticket;         // zero between steps
  unsigned int* seq;            // step sequence number (starts at 1)
  int* status;
  unsigned long long timeout_ns;  // bound of every wait
  int grid;                       // CTAs (one per SM)
  // Optional phase profile (null: off), [grid][prof_values(L)]: each CTA
  // records %globaltimer at the start of every phase (2*ph) and when its
  // input is in (2*ph + 1); then its own start (2*nph) and end (2*nph + 1;
  // for the CTA that finishes the step, the end of the step); then per layer
  // kProfAttnMarks marks of its first attention item (2*nph + 2 +
  // kProfAttnMarks*layer + k): the scan's states combined (k = 0), its
  // output or partials published (k = 1), the merge done (k = 2; 0 unless
  // this CTA merged), scan warp 0's first and last K/V chunk in shared
  // memory (k = 3, 4), its scan done (k = 5), and for the block-wide scan
  // the first chunk's scores and weights done (k = 6, 7).
  unsigned long long* prof;
  // shared-memory plan (filled by launch_persistent)
  int slot_bytes, nslots, ring_offset, xs_offset, attn_offset, attn_bytes;
};

// Values per CTA in the phase profile of an L-layer step.
constexpr int kProfAttnMarks = 8;
__host__ __device__ inline size_t prof_values(int L) {
  return 2 * (5 * (size_t)L + 1) + 2 + kProfAttnMarks * (size_t)L;
}

// True when the persistent kernel fits this shape (shared memory, batch,
// head_dim, GQA group).
bool persistent_supported(int L, int H, int qd, int F, int D, int G, int B);
cudaError_t launch_persistent(PersistArgs a, cudaStream_t s);

}  // namespace nc
