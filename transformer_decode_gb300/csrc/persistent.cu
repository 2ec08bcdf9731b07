// persistent.cu -- the whole decode step as one persistent kernel.
//
// At batch 1 the step is a chain of ~5 dependent phases per layer (QKV,
// attention, o-proj, gate|up, down; nanocompile's 13 kernels per block fused
// down), each moving only 1-17 MB: as separate launches it is bound by
// launch latency and per-kernel ramp-up, not by HBM. Here one CTA per SM runs
// the whole step:
//
//  * Weights do not depend on activations, so warp 0 of every CTA streams the
//    CTA's future weight tiles -- its rows of every projection of every layer,
//    then of the LM head, in the order the consumers will use them -- into a
//    ring of shared-memory slots with TMA bulk copies (cp.async.bulk, mbarrier
//    completion). HBM stays busy while the dependency chain advances.
//  * Warps 1..11 consume: per phase they gather the phase's input vector,
//    compute the RMSNorm where one precedes the projection, and reduce their
//    tile rows against it; the epilogue (bias, residual, SiLU * up, logits
//    and arg-max) runs on the reducing lane (Tang section 2.3).
//  * Phases hand values over through 64-bit global words holding (value,
//    epoch): a reader spins until the epoch of the word equals the one it
//    expects, so no separate flag or grid barrier is needed. Epochs carry the
//    step sequence number, so values of an earlier step never match.
//  * Attention runs one CTA per (sequence, kv head): RoPE (and q/k norm) of
//    its heads, the K/V append, and the online-softmax scan over the cached
//    positions in chunks (Tang section 2.2, the monoid on (m, l, acc)).
//  * Every spin is bounded by %globaltimer. On expiry the CTA writes
//    NC_ERR_TIMEOUT to the status word, stops issuing copies, waits (bounded)
//    for the copies in flight and leaves through the final ticket, so the
//    kernel always ends.
//
// The launch is cooperative: all CTAs must be resident together.
#include <cuda_runtime.h>
#include <math.h>

#include "kernels.h"
#include "persistent.h"

namespace nc {

constexpr int kPThreads = 384;
constexpr int kPConsumerWarps = kPThreads / kWarp - 1;
constexpr int kPConsumerThreads = kPConsumerWarps * kWarp;
constexpr int kPhasesPerLayer = 5;
enum PhaseKind : int { kQKV = 0, kATTN = 1, kOPROJ = 2, kGU = 3, kDOWN = 4, kHEAD = 5 };

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ uint64_t global_timer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ uint64_t ld_word(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_word(uint64_t* p, float v, uint32_t epoch) {
  const uint64_t w = (static_cast<uint64_t>(epoch) << 32) | __float_as_uint(v);
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}

// ------------------------------------------------------------------ shared state
struct PShared {
  uint64_t full[kMaxSlots];
  uint64_t empty[kMaxSlots];
  int abort;        // set once a bounded wait expired in this CTA
  unsigned issued;  // tiles the producer issued
  int pos[kPMaxBatch];
  int tok[kPMaxBatch];
  float rn[kPMaxBatch];
  float red[kPConsumerWarps][kPMaxBatch];
  unsigned long long best[kPConsumerWarps][kPMaxBatch];
  float xold[kPMaxBatch][kPMaxRows];  // residual rows the o-proj/down epilogue adds to
  float kred[kPConsumerWarps][2][kPMaxBatch];  // k-segment partial sums of a tile
  bool last;
};

// Deadline-bounded wait context for one CTA.
struct Spin {
  uint64_t deadline;
  int* abort;
  int* status;
  __device__ bool expired() {
    if (*reinterpret_cast<volatile int*>(abort)) return true;
    if (global_timer() > deadline) {
      atomicExch(abort, 1);
      if (status) atomicCAS(status, 0, (int)NC_ERR_TIMEOUT);
      return true;
    }
    return false;
  }
};

// Spin until the word at p carries `epoch`; returns its value (0 on abort).
__device__ __forceinline__ float ll_get(const uint64_t* p, uint32_t epoch, Spin& sp) {
  uint64_t w = ld_word(p);
  int n = 0;
  while (static_cast<uint32_t>(w >> 32) != epoch) {
    if ((++n & 63) == 0 && sp.expired()) return 0.f;
    w = ld_word(p);
  }
  return __uint_as_float(static_cast<uint32_t>(w));
}

// Read `count` words p[0], p[stride], ... (count <= kLLBatch) with all loads
// in flight at once, then re-poll only the words whose epoch is stale.
constexpr int kLLBatch = 8;
__device__ __forceinline__ void ll_get_batch(const uint64_t* p, int stride, int count,
                                             uint32_t epoch, float* out, Spin& sp) {
  uint64_t w[kLLBatch];
#pragma unroll
  for (int u = 0; u < kLLBatch; ++u)
    if (u < count) w[u] = ld_word(p + (size_t)u * stride);
#pragma unroll
  for (int u = 0; u < kLLBatch; ++u) {
    if (u >= count) break;
    int n = 0;
    while (static_cast<uint32_t>(w[u] >> 32) != epoch) {
      if ((++n & 63) == 0 && sp.expired()) {
        w[u] = 0;
        break;
      }
      w[u] = ld_word(p + (size_t)u * stride);
    }
    out[u] = __uint_as_float(static_cast<uint32_t>(w[u]));
  }
}

__device__ __forceinline__ uint32_t epoch_of(uint32_t seq, int phase) {
  return ((seq & 0xFFFFFFu) << 8) | static_cast<uint32_t>(phase);
}

// Rows of phase `ph` given to CTA `cta` and the tile shape used to stream them.
struct Rows {
  int r0, r1, R;          // rows [r0, r1), R rows per tile
  int K;                  // elements per row
  const uint16_t* m0;     // matrix (gate block for gate|up)
  const uint16_t* m1;     // up block, or null
};

__device__ __forceinline__ Rows phase_rows(const PersistArgs& a, int ph, int cta, int grid,
                                           int slot_bytes) {
  Rows r{0, 0, 1, 0, nullptr, nullptr};
  int N = 0;
  if (ph == kPhasesPerLayer * a.L) {
    N = a.V;
    r.K = a.H;
    r.m0 = a.head;
  } else {
    const PLayer& P = a.layers[ph / kPhasesPerLayer];
    switch (ph % kPhasesPerLayer) {
      case kQKV: N = a.nqkv; r.K = a.H; r.m0 = P.w_qkv; break;
      case kOPROJ: N = a.H; r.K = a.Hq * a.D; r.m0 = P.w_o; break;
      case kGU:
        N = a.F; r.K = a.H; r.m0 = P.w_gu; r.m1 = P.w_gu + (size_t)a.F * a.H; break;
      case kDOWN: N = a.H; r.K = a.F; r.m0 = P.w_d; break;
      default: return r;  // attention streams no weights
    }
  }
  r.r0 = (int)(((long long)cta * N) / grid);
  r.r1 = (int)(((long long)(cta + 1) * N) / grid);
  const int row_bytes = r.K * 2 * (r.m1 ? 2 : 1);
  r.R = slot_bytes / row_bytes;
  if (r.R > kPConsumerWarps) r.R = kPConsumerWarps;  // one unit per consumer warp
  if (r.R < 1) r.R = 1;
  return r;
}

// ------------------------------------------------------------------ producer
template <bool KV16>
__device__ bool produce_kv(const PersistArgs& a, PShared& S, char* ring, int slot_bytes,
                           int nslots, int layer, int b, int g, int npos, uint32_t& iter,
                           Spin& sp);

template <bool KV16>
__device__ void producer(const PersistArgs& a, PShared& S, char* ring, int slot_bytes, int nslots,
                         Spin& sp) {
  const int nph = kPhasesPerLayer * a.L + 1;
  uint32_t iter = 0;
  for (int ph = 0; ph < nph; ++ph) {
    if (ph < kPhasesPerLayer * a.L && ph % kPhasesPerLayer == kATTN) {
      for (int it = blockIdx.x; it < a.B * a.Hkv; it += gridDim.x) {
        const int b = it / a.Hkv, g = it % a.Hkv;
        const int npos = a.kv.slot_ok(b, S.pos[b]) ? S.pos[b] : 0;
        if (!produce_kv<KV16>(a, S, ring, slot_bytes, nslots, ph / kPhasesPerLayer, b, g, npos,
                              iter, sp))
          return;
      }
      continue;
    }
    const Rows r = phase_rows(a, ph, blockIdx.x, gridDim.x, slot_bytes);
    for (int row = r.r0; row < r.r1; row += r.R) {
      const int n = min(r.R, r.r1 - row);
      const int s = iter % nslots;
      if (iter >= (uint32_t)nslots) {
        const uint32_t par = ((iter / nslots) - 1) & 1;
        int k = 0;
        while (!mbar_try_wait(&S.empty[s], par))
          if ((++k & 15) == 0 && sp.expired()) return;
      }
      if (*reinterpret_cast<volatile int*>(&S.abort)) return;
      const uint32_t bytes = (uint32_t)n * r.K * 2;
      char* dst = ring + (size_t)s * slot_bytes;
      mbar_expect_tx(&S.full[s], bytes * (r.m1 ? 2u : 1u));
      bulk_g2s(dst, r.m0 + (size_t)row * r.K, bytes, &S.full[s]);
      if (r.m1) bulk_g2s(dst + bytes, r.m1 + (size_t)row * r.K, bytes, &S.full[s]);
      S.issued = ++iter;
    }
  }
}

// ------------------------------------------------------------------ consumer helpers
// Named barrier over the consumer warps only (the producer never joins).
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kPConsumerThreads) : "memory");
}
// The same barrier with an OR reduction: every consumer thread gets the same
// answer, so a decision taken on it keeps the named barriers uniform.
__device__ __forceinline__ bool consumer_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 1, %2, p;\n"
      " selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(kPConsumerThreads)
      : "memory");
  return r != 0;
}

// Gather the phase input [B][n] from epoch-tagged words into xs (fp32);
// with gamma, also compute the RMSNorm factor per sequence and scale xs.
template <int BT>
__device__ void gather_input(const PersistArgs& a, PShared& S, const uint64_t* src, int n,
                             uint32_t epoch, const uint16_t* embed_rows, const uint16_t* gamma,
                             float* xs, Spin& sp) {
  const int ct = threadIdx.x - kWarp, warp = ct / kWarp, lane = ct % kWarp;
#pragma unroll 1
  for (int b = 0; b < BT; ++b) {
    float ss = 0.f;
    for (int i0 = ct; i0 < n; i0 += kLLBatch * kPConsumerThreads) {
      const int count = min(kLLBatch, (n - i0 + kPConsumerThreads - 1) / kPConsumerThreads);
      float v[kLLBatch];
      if (b >= a.B) {
#pragma unroll
        for (int u = 0; u < kLLBatch; ++u) v[u] = 0.f;
      } else if (embed_rows) {
#pragma unroll
        for (int u = 0; u < kLLBatch; ++u)
          if (u < count)
            v[u] = bf16_to_f32(embed_rows[(size_t)S.tok[b] * n + i0 + u * kPConsumerThreads]);
      } else {
        ll_get_batch(src + (size_t)b * n + i0, kPConsumerThreads, count, epoch, v, sp);
      }
#pragma unroll
      for (int u = 0; u < kLLBatch; ++u) {
        if (u >= count) break;
        xs[b * n + i0 + u * kPConsumerThreads] = v[u];
        ss = fmaf(v[u], v[u], ss);
      }
    }
    if (gamma) {
      ss = warp_sum(ss);
      if (lane == 0) S.red[warp][b] = ss;
    }
  }
  if (!gamma) {
    consumer_sync();
    return;
  }
  consumer_sync();
  if (ct < BT) {
    float t = 0.f;
    for (int w = 0; w < kPConsumerWarps; ++w) t += S.red[w][ct];
    S.rn[ct] = 1.f / sqrtf(t / (float)n + a.eps);
  }
  consumer_sync();
  for (int i = ct; i < n; i += kPConsumerThreads) {
    const float g = bf16_to_f32(gamma[i]);
#pragma unroll
    for (int b = 0; b < BT; ++b) xs[b * n + i] = (xs[b * n + i] * S.rn[b]) * g;
  }
  consumer_sync();
}

__device__ __forceinline__ float silu_mul_p(float g, float u) {
  const float e = expf(-fabsf(g));
  const float sig = g >= 0.f ? 1.f / (1.f + e) : e / (1.f + e);
  return (g * sig) * u;
}

// Input chunks kept in registers per lane at batch 1 (8 floats each).
constexpr int kXReg = 4;

// 8 bf16 weights (one 16-byte chunk) times 8 fp32 inputs held in registers.
__device__ __forceinline__ float dot8r(const uint4& w, const float (&x)[8]) {
  float s = bf16_lo(w.x) * x[0];
  s = fmaf(bf16_hi(w.x), x[1], s);
  s = fmaf(bf16_lo(w.y), x[2], s);
  s = fmaf(bf16_hi(w.y), x[3], s);
  s = fmaf(bf16_lo(w.z), x[4], s);
  s = fmaf(bf16_hi(w.z), x[5], s);
  s = fmaf(bf16_lo(w.w), x[6], s);
  s = fmaf(bf16_hi(w.w), x[7], s);
  return s;
}

// Epilogue of output row j of sequence b on the reducing thread: bias, the
// residual add, silu(gate) * up, or the logit and its arg-max key.
template <int BT>
__device__ __forceinline__ void tile_epilogue(const PersistArgs& a, const PShared& S, int kind,
                                              const PLayer* P, int r0, int j, int b, float v0,
                                              float v1, uint32_t ep,
                                              unsigned long long (&best)[BT]) {
  if (kind == kQKV) {
    if (P->b_qkv) v0 += bf16_to_f32(P->b_qkv[j]);
    st_word(a.qkvw + (size_t)b * a.nqkv + j, v0, ep);
  } else if (kind == kOPROJ || kind == kDOWN) {
    st_word(a.xw + (size_t)b * a.H + j, S.xold[b][j - r0] + v0, ep);
  } else if (kind == kGU) {
    st_word(a.hw + (size_t)b * a.F + j, silu_mul_p(v0, v1), ep);
  } else {
    a.logits[(size_t)b * a.V + j] = v0;
    const unsigned long long key = argmax_key(v0, (uint32_t)j);
#pragma unroll
    for (int bb = 0; bb < BT; ++bb)
      if (bb == b) best[bb] = key > best[bb] ? key : best[bb];
  }
}

// ------------------------------------------------------------------ attention item
// The producer streams the cached K and V of slots 0..pos-1 of every
// attention item this CTA owns through the ring, as chunk tiles holding the K
// rows then the V rows of up to attn_chunk positions; the new position's K/V
// never leaves shared memory.
constexpr int kAttnMaxChunk = 128;
__host__ __device__ __forceinline__ int attn_chunk(int slot_bytes, int D, int es) {
  return slot_bytes / (2 * D * es);
}

// Producer: issue the chunk tiles of (layer, b, g) for slots [0, npos).
template <bool KV16>
__device__ bool produce_kv(const PersistArgs& a, PShared& S, char* ring, int slot_bytes,
                           int nslots, int layer, int b, int g, int npos, uint32_t& iter,
                           Spin& sp) {
  constexpr int ES = KV16 ? 2 : 4;
  const int D = a.D, CP = attn_chunk(slot_bytes, D, ES);
  const int bs = a.kv.paged ? a.kv.block_size : npos;
  for (int t0 = 0; t0 < npos; t0 += CP) {
    const int n = min(CP, npos - t0);
    const int s = iter % nslots;
    if (iter >= (uint32_t)nslots) {
      const uint32_t par = ((iter / nslots) - 1) & 1;
      int k = 0;
      while (!mbar_try_wait(&S.empty[s], par))
        if ((++k & 15) == 0 && sp.expired()) return false;
    }
    if (*reinterpret_cast<volatile int*>(&S.abort)) return false;
    // runs of positions contiguous in the cache: the whole chunk when the
    // cache is contiguous, a block's worth when it is paged
    uint32_t bytes = 0;
    for (int t = t0; t < t0 + n;) {
      const int len = min(t0 + n - t, bs - t % bs);
      if (a.kv.slot_ok(b, t)) bytes += 2u * len * D * ES;
      t += len;
    }
    mbar_expect_tx(&S.full[s], bytes);
    char* dst = ring + (size_t)s * slot_bytes;
    for (int t = t0; t < t0 + n;) {
      const int len = min(t0 + n - t, bs - t % bs);
      if (a.kv.slot_ok(b, t)) {
        const size_t off = a.kv.offset(layer, b, g, t) * ES;
        const uint32_t nb = (uint32_t)len * D * ES;
        bulk_g2s(dst + (size_t)(t - t0) * D * ES, static_cast<const char*>(a.kv.k) + off, nb,
                 &S.full[s]);
        bulk_g2s(dst + (size_t)(CP + t - t0) * D * ES, static_cast<const char*>(a.kv.v) + off,
                 nb, &S.full[s]);
      }
      t += len;
    }
    S.issued = ++iter;
  }
  return true;
}

template <bool KV16>
__device__ __forceinline__ float kv_smem(const char* base, int idx) {
  if constexpr (KV16) return bf16_to_f32(reinterpret_cast<const uint16_t*>(base)[idx]);
  else return reinterpret_cast<const float*>(base)[idx];
}

// Consumer: one (sequence b, kv head g). RoPE (+ q/k norm) of the G query
// heads and the key, K/V append at slot pos, then the online-softmax scan:
// the new position first, then the cached chunks from the ring.
template <int D, bool KV16>
__device__ void attention_item(const PersistArgs& a, PShared& S, int b, int g, int layer,
                               uint32_t ep_qkv, uint32_t ep_out, float* scratch, char* ring,
                               int slot_bytes, int nslots, uint32_t& iter, Spin& sp) {
  constexpr int GM = 8, ES = KV16 ? 2 : 4;
  const int ct = threadIdx.x - kWarp, warp = ct / kWarp, lane = ct % kWarp;
  const int G = a.Hq / a.Hkv;
  const int CP = attn_chunk(slot_bytes, D, ES);
  const int pos = S.pos[b];
  float* qs = scratch;                    // [GM][D]
  float* kn = qs + GM * D;                // [D]
  float* vn = kn + D;                     // [D]
  float* sc = vn + D;                     // [GM][kAttnMaxChunk]
  float* mrun = sc + GM * kAttnMaxChunk;  // [GM] running max
  float* lrun = mrun + GM;                // [GM] running sum
  float* resc = lrun + GM;                // [GM] rescale of the chunk
  const PLayer& P = a.layers[layer];
  const uint64_t* qkv = a.qkvw + (size_t)b * a.nqkv;

  // gather q heads, k, v of this group
  for (int i = ct; i < (G + 2) * D; i += kPConsumerThreads) {
    const int h = i / D, d = i % D;
    int src;
    if (h < G) src = (g * G + h) * D + d;
    else if (h == G) src = (a.Hq + g) * D + d;
    else src = (a.Hq + a.Hkv + g) * D + d;
    const float v = ll_get(qkv + src, ep_qkv, sp);
    if (h < G) qs[h * D + d] = v;
    else if (h == G) kn[d] = v;
    else vn[d] = v;
  }
  consumer_sync();
  // per-head RMSNorm (q/k norm) and RoPE, one warp per head (G is the key)
  for (int hh = warp; hh <= G; hh += kPConsumerWarps) {
    float* v = hh < G ? qs + hh * D : kn;
    constexpr int E = D / 32;
    float e[E];
#pragma unroll
    for (int j = 0; j < E; ++j) e[j] = v[lane + 32 * j];
    const uint16_t* gain = hh < G ? P.g_q : P.g_k;
    if (gain) {
      float ss = 0.f;
#pragma unroll
      for (int j = 0; j < E; ++j) ss = fmaf(e[j], e[j], ss);
      ss = warp_sum(ss);
      const float r = 1.f / sqrtf(ss / (float)D + a.eps);
#pragma unroll
      for (int j = 0; j < E; ++j) e[j] = (e[j] * r) * bf16_to_f32(gain[lane + 32 * j]);
    }
#pragma unroll
    for (int j = 0; j < E / 2; ++j) {
      const int i = lane + 32 * j;
      const float angle = __fmul_rn((float)pos, a.inv_freq[i]);
      float sn, cs;
      sincosf(angle, &sn, &cs);
      const float x0 = e[j], x1 = e[j + E / 2];
      e[j] = __fsub_rn(__fmul_rn(x0, cs), __fmul_rn(x1, sn));
      e[j + E / 2] = __fadd_rn(__fmul_rn(x1, cs), __fmul_rn(x0, sn));
    }
#pragma unroll
    for (int j = 0; j < E; ++j) v[lane + 32 * j] = e[j];
  }
  consumer_sync();
  // append K/V at slot pos; the scan reads slot pos from kn/vn as stored
  const bool pos_ok = a.kv.slot_ok(b, pos);
  if (!pos_ok && ct == 0 && a.status) atomicCAS(a.status, 0, (int)NC_ERR_POSITION);
  if (ct < D) {
    float k_st = kn[ct], v_st = vn[ct];
    if (pos_ok) {
      const size_t off = a.kv.offset(layer, b, g, pos);
      kv_store<KV16>(a.kv.k, off + ct, k_st);
      kv_store<KV16>(a.kv.v, off + ct, v_st);
    }
    if (KV16) {
      k_st = bf16_to_f32(f32_to_bf16(k_st));
      v_st = bf16_to_f32(f32_to_bf16(v_st));
    }
    kn[ct] = k_st;
    vn[ct] = v_st;
  }
  consumer_sync();
  const float scale = 1.f / sqrtf((float)D);
  // the new position opens the running state: m = its score, l = 1, acc = v
  for (int h = warp; h < G; h += kPConsumerWarps) {
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < D / 32; ++j) s = fmaf(qs[h * D + lane + 32 * j], kn[lane + 32 * j], s);
    s = warp_sum(s) * scale;
    if (lane == 0) {
      mrun[h] = pos_ok ? s : -INFINITY;
      lrun[h] = pos_ok ? 1.f : 0.f;
    }
  }
  const int npair = G * (D / 2);
  const int my_h = ct / (D / 2), my_d2 = ct % (D / 2);
  float acc0 = 0.f, acc1 = 0.f;
  if (ct < npair && pos_ok) {
    acc0 = vn[2 * my_d2];
    acc1 = vn[2 * my_d2 + 1];
  }
  consumer_sync();
  const int npos = pos_ok ? pos : 0;
  for (int t0 = 0; t0 < npos; t0 += CP) {
    const int n = min(CP, npos - t0);
    const int s = iter % nslots;
    {
      const uint32_t par = (iter / nslots) & 1;
      int k = 0;
      while (!mbar_try_wait(&S.full[s], par))
        if ((++k & 15) == 0 && sp.expired()) break;
    }
    const char* Ks = ring + (size_t)s * slot_bytes;
    const char* Vs = Ks + (size_t)CP * D * ES;
    // scores: warp -> (head, 32 positions); lane l reads its row from column
    // (d + l) mod D so the 32 rows of a warp fall in different banks
    const int blocks = (n + 31) / 32;
    for (int wb = warp; wb < G * blocks; wb += kPConsumerWarps) {
      const int h = wb % G, p = (wb / G) * 32 + lane;
      if (p < n) {
        float sv = -INFINITY;
        if (a.kv.slot_ok(b, t0 + p)) {
          float acc = 0.f;
#pragma unroll 8
          for (int d = 0; d < D; ++d) {
            const int dd = (d + lane) & (D - 1);
            acc = fmaf(qs[h * D + dd], kv_smem<KV16>(Ks, p * D + dd), acc);
          }
          sv = acc * scale;
        }
        sc[h * kAttnMaxChunk + p] = sv;
      }
    }
    consumer_sync();
    for (int h = warp; h < G; h += kPConsumerWarps) {
      float m = -INFINITY;
      for (int t = lane; t < n; t += kWarp) m = fmaxf(m, sc[h * kAttnMaxChunk + t]);
      m = warp_max(m);
      const float m_new = fmaxf(mrun[h], m);
      float l = 0.f;
      for (int t = lane; t < n; t += kWarp) {
        const float x = sc[h * kAttnMaxChunk + t];
        const float p = x == -INFINITY ? 0.f : expf(x - m_new);
        sc[h * kAttnMaxChunk + t] = p;
        l += p;
      }
      l = warp_sum(l);
      if (lane == 0) {
        const float r = mrun[h] == -INFINITY ? 0.f : expf(mrun[h] - m_new);
        resc[h] = r;
        lrun[h] = lrun[h] * r + l;
        mrun[h] = m_new;
      }
    }
    consumer_sync();
    if (ct < npair) {
      const float r = resc[my_h];
      acc0 *= r;
      acc1 *= r;
      for (int t = 0; t < n; ++t) {
        const float p = sc[my_h * kAttnMaxChunk + t];
        if (p == 0.f) continue;
        acc0 = fmaf(p, kv_smem<KV16>(Vs, t * D + 2 * my_d2), acc0);
        acc1 = fmaf(p, kv_smem<KV16>(Vs, t * D + 2 * my_d2 + 1), acc1);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[s]);
    ++iter;
    consumer_sync();  // sc is rewritten by the next chunk
  }
  if (ct < npair) {
    const float inv = lrun[my_h] > 0.f ? 1.f / lrun[my_h] : 0.f;
    uint64_t* out = a.aw + (size_t)b * a.Hq * D + (size_t)(g * G + my_h) * D + 2 * my_d2;
    st_word(out, acc0 * inv, ep_out);
    st_word(out + 1, acc1 * inv, ep_out);
  }
  consumer_sync();  // the scratch is reused by the next item
}

// ------------------------------------------------------------------ the kernel
template <int BT, int D, bool KV16>
__global__ void __launch_bounds__(kPThreads, 1) k_decode_persistent(PersistArgs a) {
  extern __shared__ __align__(128) char smem[];
  PShared& S = *reinterpret_cast<PShared*>(smem);
  const int slot_bytes = a.slot_bytes, nslots = a.nslots;
  char* ring = smem + a.ring_offset;
  float* xs = reinterpret_cast<float*>(smem + a.xs_offset);
  float* scratch = reinterpret_cast<float*>(smem + a.attn_offset);
  const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;

  if (threadIdx.x == 0) {
    for (int s = 0; s < nslots; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], kPConsumerWarps);
    }
    S.abort = 0;
    S.issued = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (threadIdx.x < BT) {
    const int b = threadIdx.x;
    S.pos[b] = b < a.B ? a.positions[b] : 0;
    int t = b < a.B ? a.tokens[b] : 0;
    if (t < 0 || t >= a.V) {
      if (a.status) atomicCAS(a.status, 0, (int)NC_ERR_INVALID_ARGUMENT);
      t = 0;
    }
    S.tok[b] = t;
  }
  __syncthreads();
  const uint32_t seq = *reinterpret_cast<volatile const unsigned*>(a.seq);
  Spin sp{global_timer() + a.timeout_ns, &S.abort, a.status};
  if (a.prof && blockIdx.x == 0 && threadIdx.x == 0)
    a.prof[2 * (kPhasesPerLayer * a.L + 1)] = global_timer();

  if (warp == 0) {
    if (lane == 0) producer<KV16>(a, S, ring, slot_bytes, nslots, sp);
  } else {
    const int ct = threadIdx.x - kWarp, cw = ct / kWarp;
    const int L = a.L, nph = kPhasesPerLayer * L + 1;
    uint32_t iter = 0;
    unsigned long long best[BT];
#pragma unroll
    for (int b = 0; b < BT; ++b) best[b] = 0ull;
    float xr[kXReg][8];      // batch 1: this lane's input chunks (see the tile loop)
    int xr_ks = -1, xr_seg = -1;
    for (int ph = 0; ph < nph; ++ph) {
      // Uniform across the consumer warps, and a barrier: no warp overwrites
      // the shared input vector while another still reduces against it.
      if (consumer_any(*reinterpret_cast<volatile int*>(&S.abort) != 0)) break;
      const bool prof = a.prof && blockIdx.x == 0 && ct == 0;
      if (prof) a.prof[2 * ph] = global_timer();
      const int layer = ph / kPhasesPerLayer;
      const int kind = ph == kPhasesPerLayer * L ? kHEAD : ph % kPhasesPerLayer;
      const uint32_t ep = epoch_of(seq, ph);
      if (kind == kATTN) {
        const int items = a.B * a.Hkv;
        for (int it = blockIdx.x; it < items; it += gridDim.x)
          attention_item<D, KV16>(a, S, it / a.Hkv, it % a.Hkv, layer, epoch_of(seq, ph - 1),
                                  ep, scratch, ring, slot_bytes, nslots, iter, sp);
        if (prof) a.prof[2 * ph + 1] = global_timer();
        continue;
      }
      const Rows r = phase_rows(a, ph, blockIdx.x, gridDim.x, slot_bytes);
      if (r.r0 >= r.r1) continue;
      // phase input
      const PLayer* P = kind == kHEAD ? nullptr : &a.layers[layer];
      const int K = r.K;
      if (kind == kOPROJ || kind == kDOWN) {
        // The residual rows this CTA updates are older than the phase input,
        // so reading them first overlaps their round trip with the wait.
        const int nr = r.r1 - r.r0;
        const uint32_t ep_old = epoch_of(seq, kind == kOPROJ ? ph - 3 : ph - 2);
        for (int i = ct; i < nr * BT; i += kPConsumerThreads) {
          const int b = i / nr, jr = i % nr, j = r.r0 + jr;
          float old = 0.f;
          if (b < a.B)
            old = (kind == kOPROJ && layer == 0)
                      ? bf16_to_f32(a.embed[(size_t)S.tok[b] * a.H + j])
                      : ll_get(a.xw + (size_t)b * a.H + j, ep_old, sp);
          S.xold[b][jr] = old;
        }
      }
      if (kind == kQKV) {
        gather_input<BT>(a, S, a.xw, K, epoch_of(seq, ph - 1), layer == 0 ? a.embed : nullptr,
                         P->g_attn, xs, sp);
      } else if (kind == kOPROJ) {
        gather_input<BT>(a, S, a.aw, K, epoch_of(seq, ph - 1), nullptr, nullptr, xs, sp);
      } else if (kind == kGU) {
        gather_input<BT>(a, S, a.xw, K, epoch_of(seq, ph - 1), nullptr, P->g_mlp, xs, sp);
      } else if (kind == kDOWN) {
        gather_input<BT>(a, S, a.hw, K, epoch_of(seq, ph - 1), nullptr, nullptr, xs, sp);
      } else {
        gather_input<BT>(a, S, a.xw, K, epoch_of(seq, ph - 1), nullptr, a.g_final, xs, sp);
      }
      if (prof) a.prof[2 * ph + 1] = global_timer();
      xr_ks = -1;  // a new input vector: reload the register copy
      const int two = r.m1 ? 2 : 1;
      for (int row = r.r0; row < r.r1; row += r.R) {
        const int n = min(r.R, r.r1 - row);
        const int s = iter % nslots;
        {
          const uint32_t par = (iter / nslots) & 1;
          int k = 0;
          while (!mbar_try_wait(&S.full[s], par))
            if ((++k & 15) == 0 && sp.expired()) break;
        }
        if (*reinterpret_cast<volatile int*>(&S.abort)) break;
        const uint16_t* tile = reinterpret_cast<const uint16_t*>(ring + (size_t)s * slot_bytes);
        // Work split: an output unit (a row; a gate|up pair) is cut into KS
        // k-segments and each warp takes one (unit, segment), so a tile of few
        // long rows still keeps every warp busy on a short chain. Tiles hold
        // at most kPConsumerWarps units.
        const int KS = n >= kPConsumerWarps ? 1 : kPConsumerWarps / n;
        const int C = K / 8;  // 16-byte chunks per row
        const bool active = cw < n * KS;
        const int ui = cw / KS, seg = cw % KS;
        float acc[2][BT];
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
          for (int b = 0; b < BT; ++b) acc[u][b] = 0.f;
        if (active && BT == 1) {
          // batch 1: this lane's input chunks stay in registers across the
          // phase's tiles; only the weights are read from shared memory
          const int c0 = (seg * C) / KS, c1 = ((seg + 1) * C) / KS;
          if (KS != xr_ks || seg != xr_seg) {
#pragma unroll
            for (int jj = 0; jj < kXReg; ++jj) {
              const int c = c0 + lane + jj * kWarp;
              if (c < c1) {
                const float4 p0 = *reinterpret_cast<const float4*>(xs + c * 8);
                const float4 p1 = *reinterpret_cast<const float4*>(xs + c * 8 + 4);
                xr[jj][0] = p0.x; xr[jj][1] = p0.y; xr[jj][2] = p0.z; xr[jj][3] = p0.w;
                xr[jj][4] = p1.x; xr[jj][5] = p1.y; xr[jj][6] = p1.z; xr[jj][7] = p1.w;
              }
            }
            xr_ks = KS;
            xr_seg = seg;
          }
          for (int u = 0; u < two; ++u) {
            const uint16_t* w = tile + ((size_t)u * n + ui) * K;
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int jj = 0; jj < kXReg; jj += 2) {
              const int c = c0 + lane + jj * kWarp;
              if (c < c1) a0 += dot8r(*reinterpret_cast<const uint4*>(w + c * 8), xr[jj]);
              if (jj + 1 < kXReg && c + kWarp < c1)
                a1 += dot8r(*reinterpret_cast<const uint4*>(w + (c + kWarp) * 8), xr[jj + 1]);
            }
            for (int c = c0 + lane + kXReg * kWarp; c < c1; c += kWarp)  // beyond the registers
              a0 += dot8(*reinterpret_cast<const uint4*>(w + c * 8), xs + c * 8);
            acc[u][0] = warp_sum(a0 + a1);
          }
        } else if (active) {
          const int c0 = (seg * C) / KS, c1 = ((seg + 1) * C) / KS;
          for (int u = 0; u < two; ++u) {
            const uint16_t* w = tile + ((size_t)u * n + ui) * K;
            float acc2[BT];
#pragma unroll
            for (int b = 0; b < BT; ++b) acc2[b] = 0.f;
            int c = c0 + lane;
            for (; c + kWarp < c1; c += 2 * kWarp) {  // two independent chains
              const uint4 w0 = *reinterpret_cast<const uint4*>(w + c * 8);
              const uint4 w1 = *reinterpret_cast<const uint4*>(w + (c + kWarp) * 8);
#pragma unroll
              for (int b = 0; b < BT; ++b) {
                acc[u][b] += dot8(w0, xs + b * K + c * 8);
                acc2[b] += dot8(w1, xs + b * K + (c + kWarp) * 8);
              }
            }
            if (c < c1) {
              const uint4 w0 = *reinterpret_cast<const uint4*>(w + c * 8);
#pragma unroll
              for (int b = 0; b < BT; ++b) acc[u][b] += dot8(w0, xs + b * K + c * 8);
            }
#pragma unroll
            for (int b = 0; b < BT; ++b) acc[u][b] = warp_sum(acc[u][b] + acc2[b]);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.empty[s]);  // this warp is done with the slot
        ++iter;
        if (KS == 1) {
          if (active && lane < BT && lane < a.B) {
            float v0 = acc[0][0], v1 = acc[1][0];
#pragma unroll
            for (int bb = 1; bb < BT; ++bb)
              if (lane == bb) {
                v0 = acc[0][bb];
                v1 = acc[1][bb];
              }
            tile_epilogue<BT>(a, S, kind, P, r.r0, row + ui, lane, v0, v1, ep, best);
          }
        } else {
          if (active && lane == 0)
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
              for (int b = 0; b < BT; ++b) S.kred[cw][u][b] = acc[u][b];
          consumer_sync();
          for (int t = ct; t < n * BT; t += kPConsumerThreads) {
            const int i = t / BT, b = t % BT;
            if (b >= a.B) continue;
            float v0 = 0.f, v1 = 0.f;
            for (int sg = 0; sg < KS; ++sg) {
              v0 += S.kred[i * KS + sg][0][b];
              v1 += S.kred[i * KS + sg][1][b];
            }
            tile_epilogue<BT>(a, S, kind, P, r.r0, row + i, b, v0, v1, ep, best);
          }
          consumer_sync();  // kred is rewritten by the next tile
        }
      }
    }
    // per-CTA arg-max partials (any lane of a warp may hold a row's key)
#pragma unroll
    for (int b = 0; b < BT; ++b) {
      unsigned long long m = best[b];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long t = __shfl_xor_sync(0xFFFFFFFFu, m, o);
        m = t > m ? t : m;
      }
      if (lane == 0) S.best[cw][b] = m;
    }
  }
  __syncthreads();
  // Drain: copies issued but never consumed (only after an abort) must land
  // before the CTA exits. Only the last fill of each slot can be pending: tile
  // t fills slot t % nslots for the (t / nslots)-th time. Waits are bounded.
  if (threadIdx.x == 0 && S.abort) {
    const uint64_t dl = global_timer() + a.timeout_ns;
    const unsigned issued = S.issued;
    for (unsigned t = issued > (unsigned)nslots ? issued - nslots : 0u; t < issued; ++t) {
      while (!mbar_try_wait(&S.full[t % nslots], (t / nslots) & 1))
        if (global_timer() > dl) break;
    }
  }
  if (threadIdx.x < BT && threadIdx.x < a.B) {
    unsigned long long m = 0ull;
    for (int w = 0; w < kPConsumerWarps; ++w) m = S.best[w][threadIdx.x] > m ? S.best[w][threadIdx.x] : m;
    a.am_part[(size_t)threadIdx.x * gridDim.x + blockIdx.x] = S.abort ? ~0ull : m;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) S.last = atomicAdd(a.ticket, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!S.last) return;
  __threadfence();
  if (warp < BT && warp < a.B) {
    const int b = warp;
    unsigned long long m = 0ull;
    for (int i = lane; i < (int)gridDim.x; i += kWarp) {
      const unsigned long long k = __ldcg(a.am_part + (size_t)b * gridDim.x + i);
      m = k > m ? k : m;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long t = __shfl_xor_sync(0xFFFFFFFFu, m, o);
      m = t > m ? t : m;
    }
    if (lane == 0) {
      const bool bad = m == ~0ull;
      const int32_t tok = bad ? -1 : (int32_t)(0xFFFFFFFFu - (uint32_t)(m & 0xFFFFFFFFull));
      if (a.next) a.next[b] = tok;
      if (bad && a.status) atomicCAS(a.status, 0, (int)NC_ERR_INVALID_ARGUMENT);
      if (a.advance) {
        a.tokens[b] = bad ? 0 : tok;
        a.positions[b] = S.pos[b] + 1;
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    *a.seq = seq + 1;  // next step's epochs
    if (a.prof) a.prof[2 * (kPhasesPerLayer * a.L + 1) + 1] = global_timer();
    *a.ticket = 0u;
    __threadfence();
  }
}

// ------------------------------------------------------------------ host side
// Shared-memory plan: PShared, the input vector [BT][max(H, Hq D, F)] fp32,
// the attention scratch, then the weight ring in the rest.
static int bt_of(int B) { return B <= 1 ? 1 : B <= 2 ? 2 : 4; }
static int kmax_of(int H, int qd, int F) { return H > qd ? (H > F ? H : F) : (qd > F ? qd : F); }
static size_t round128(size_t x) { return (x + 127) / 128 * 128; }

static size_t persistent_fixed_smem(int H, int qd, int F, int D, int BT) {
  size_t off = round128(sizeof(PShared));
  off = round128(off + (size_t)BT * kmax_of(H, qd, F) * 4);
  off += sizeof(float) * (8 * D + 2 * D + 8 * kAttnMaxChunk + 3 * 8);
  return round128(off);
}

template <int BT, int D, bool KV16>
static cudaError_t launch_bt(const PersistArgs& a, size_t smem, cudaStream_t s) {
  auto kern = k_decode_persistent<BT, D, KV16>;
  static const cudaError_t attr =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem_optin());
  if (attr != cudaSuccess) return attr;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(a.grid);
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeCooperative;
  attrs[0].val.cooperative = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int BT>
static cudaError_t launch_b(const PersistArgs& a, size_t smem, cudaStream_t s) {
  if (a.D == 64) return a.kv.bf16 ? launch_bt<BT, 64, true>(a, smem, s) : launch_bt<BT, 64, false>(a, smem, s);
  return a.kv.bf16 ? launch_bt<BT, 128, true>(a, smem, s) : launch_bt<BT, 128, false>(a, smem, s);
}

cudaError_t launch_persistent(PersistArgs a, cudaStream_t s) {
  const int qd = a.Hq * a.D, BT = bt_of(a.B);
  const size_t fixed = persistent_fixed_smem(a.H, qd, a.F, a.D, BT);
  const size_t pshared = round128(sizeof(PShared));
  a.xs_offset = (int)pshared;
  a.attn_offset = (int)round128(pshared + (size_t)BT * kmax_of(a.H, qd, a.F) * 4);
  a.ring_offset = (int)fixed;
  const size_t avail = (size_t)max_smem_optin();
  if (fixed + (size_t)a.slot_bytes * 2 > avail) return cudaErrorInvalidConfiguration;
  int nslots = (int)((avail - fixed) / a.slot_bytes);
  if (nslots > kMaxSlots) nslots = kMaxSlots;
  a.nslots = nslots;
  const size_t smem = fixed + (size_t)nslots * a.slot_bytes;
  if (BT == 1) return launch_b<1>(a, smem, s);
  if (BT == 2) return launch_b<2>(a, smem, s);
  return launch_b<4>(a, smem, s);
}

bool persistent_supported(int H, int qd, int F, int D, int G, int B) {
  if (B < 1 || B > kPMaxBatch || (D != 64 && D != 128)) return false;
  if (G < 1 || G > 8 || G * (D / 2) > kPConsumerThreads) return false;
  if (H % 8 || qd % 8 || F % 8) return false;
  if ((H + num_sms() - 1) / num_sms() > kPMaxRows) return false;
  const size_t fixed = persistent_fixed_smem(H, qd, F, D, bt_of(B));
  return fixed + 2 * (size_t)kPSlotBytes <= (size_t)max_smem_optin();
}

}  // namespace nc
