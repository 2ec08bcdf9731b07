// attention.cu -- RoPE + KV append, and split-K grouped-query decode attention.
//
// RoPE (nanoinfer "Model architecture", "KV cache"): half-split pairs
// (i, i + D/2), angle = float(pos) * inv_freq[i] as an fp32 product, applied
// once to K on insert; K and V are rounded to bf16 when stored.
//
// Attention (Tang section 2.2: online softmax is the monoid on (m, l, acc);
// section 2.5: split is valid for any associative monoid): the positions
// 0..pos of one (sequence, kv head) are cut into `splits` chunks. Each CTA
// reads its chunk of K and V once for all G query heads of the group (the
// repeat_kv expansion folded into indexing, nanocompile "Phase 3"), produces
// the partial (m, l, acc[D]) per head, and a merge combines the partials:
//   M = max_c m_c,  out = sum_c acc_c e^(m_c - M) / sum_c l_c e^(m_c - M).
#include <cuda_runtime.h>
#include <math.h>

#include "kernels.h"

namespace nc {

// ------------------------------------------------------------------ RoPE
template <int D, bool KV16>
__global__ void __launch_bounds__(256) k_rope_qkv(RopeArgs a) {
  constexpr int E = D / 32;  // elements per lane
  const int b = blockIdx.x;
  const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
  const int pos = a.positions[b];
  if (!a.kv.slot_ok(b, pos)) {
    if (threadIdx.x == 0 && a.status) atomicCAS(a.status, 0, (int)NC_ERR_POSITION);
    return;
  }
  const int qkv_dim = (a.Hq + 2 * a.Hkv) * D;
  const float* src = a.qkv + (size_t)b * qkv_dim;
  for (int hh = warp; hh < a.Hq + a.Hkv; hh += blockDim.x / kWarp) {
    const bool is_q = hh < a.Hq;
    const float* v = src + (size_t)hh * D;
    float e[E];
#pragma unroll
    for (int j = 0; j < E; ++j) e[j] = v[lane + 32 * j];
    const uint16_t* gain = is_q ? a.g_q : a.g_k;
    if (gain) {  // per-head RMSNorm over D
      float ss = 0.f;
#pragma unroll
      for (int j = 0; j < E; ++j) ss = fmaf(e[j], e[j], ss);
      ss = warp_sum(ss);
      const float r = 1.f / sqrtf(ss / (float)D + a.eps);
#pragma unroll
      for (int j = 0; j < E; ++j) e[j] = (e[j] * r) * bf16_to_f32(gain[lane + 32 * j]);
    }
    // element lane + 32 j pairs with lane + 32 (j + E/2)
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
    if (is_q) {
#pragma unroll
      for (int j = 0; j < E; ++j) a.q_out[((size_t)b * a.Hq + hh) * D + lane + 32 * j] = e[j];
    } else {
      const int g = hh - a.Hq;
      const size_t off = a.kv.offset(a.layer, b, g, pos);
      const float* vv = src + (size_t)(a.Hq + a.Hkv + g) * D;
#pragma unroll
      for (int j = 0; j < E; ++j) {
        kv_store<KV16>(a.kv.k, off + lane + 32 * j, e[j]);
        kv_store<KV16>(a.kv.v, off + lane + 32 * j, vv[lane + 32 * j]);
      }
    }
  }
}

cudaError_t launch_rope_qkv(const RopeArgs& a, cudaStream_t s) {
  if (a.D == 64)
    (a.kv.bf16 ? k_rope_qkv<64, true> : k_rope_qkv<64, false>)<<<a.B, 256, 0, s>>>(a);
  else
    (a.kv.bf16 ? k_rope_qkv<128, true> : k_rope_qkv<128, false>)<<<a.B, 256, 0, s>>>(a);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ attention
constexpr int kAttnThreads = 256;
constexpr int kMaxChunk = 512;

int attn_splits(int B, int Hkv, int max_ctx) {
  const int target = 2 * num_sms();
  int s = (target + B * Hkv - 1) / (B * Hkv);
  const int lo = (max_ctx + kMaxChunk - 1) / kMaxChunk;
  const int hi = (max_ctx + 15) / 16;
  if (s > hi) s = hi;
  if (s < lo) s = lo;
  if (s > 256) s = 256;
  return s < 1 ? 1 : s;
}

size_t attn_part_floats(int B, int Hq, int D, int splits) {
  return (size_t)B * Hq * splits * (D + 2);
}

template <int D, int GM, bool KV16>
__global__ void __launch_bounds__(kAttnThreads) k_attn_split(AttnArgs a, int cap) {
  extern __shared__ float p_s[];  // [GM][cap] scores, then probabilities; then [cap] row offsets
  size_t* off_s = reinterpret_cast<size_t*>(p_s + ((GM * cap + 1) & ~1));  // 8-byte aligned
  __shared__ float q_s[GM][D];
  __shared__ float m_s[GM], l_s[GM];
  const int c = blockIdx.x, g = blockIdx.y, b = blockIdx.z, S = gridDim.x;
  const int G = a.Hq / a.Hkv;
  const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
  const int pos = a.positions[b];
  if ((pos < 0 || pos >= a.kv.capacity()) && threadIdx.x == 0 && c == 0 && g == 0 && a.status)
    atomicCAS(a.status, 0, (int)NC_ERR_POSITION);
  const int n = max(0, min(pos + 1, a.kv.capacity()));
  const int chunk = (n + S - 1) / S;
  const int t0 = c * chunk;
  const int len = max(0, min(n, t0 + chunk) - t0);
  float* part = a.part + ((size_t)b * a.Hq + (size_t)g * G) * S * (D + 2);

  for (int i = threadIdx.x; i < GM * D; i += kAttnThreads) {
    const int h = i / D;
    q_s[h][i % D] = h < G ? a.q[((size_t)b * a.Hq + g * G + h) * D + i % D] : 0.f;
  }
  __syncthreads();
  const float scale = 1.f / sqrtf((float)D);

  // scores: one position per thread, its K row read once for all heads
  for (int t = threadIdx.x; t < len; t += kAttnThreads) {
    if (!a.kv.slot_ok(b, t0 + t)) {  // excluded from the softmax
      if (a.status) atomicCAS(a.status, 0, (int)NC_ERR_POSITION);
#pragma unroll
      for (int h = 0; h < GM; ++h) p_s[h * cap + t] = -INFINITY;
      off_s[t] = 0;  // never dereferenced with a nonzero weight
      continue;
    }
    const size_t kr = a.kv.offset(a.layer, b, g, t0 + t);
    off_s[t] = kr;  // the row's offset, for the value pass
    float s[GM];
#pragma unroll
    for (int h = 0; h < GM; ++h) s[h] = 0.f;
#pragma unroll
    for (int ch = 0; ch < D / 8; ++ch) {
      float kf[8];
      kv_load8<KV16>(a.kv.k, kr + ch * 8, kf);
#pragma unroll
      for (int h = 0; h < GM; ++h)
#pragma unroll
        for (int e = 0; e < 8; ++e) s[h] = fmaf(q_s[h][ch * 8 + e], kf[e], s[h]);
    }
#pragma unroll
    for (int h = 0; h < GM; ++h) p_s[h * cap + t] = s[h] * scale;
  }
  __syncthreads();

  // softmax statistics of the chunk, one warp per head
  for (int h = warp; h < G; h += kAttnThreads / kWarp) {
    float m = -INFINITY;
    for (int t = lane; t < len; t += kWarp) m = fmaxf(m, p_s[h * cap + t]);
    m = warp_max(m);
    float l = 0.f;
    for (int t = lane; t < len; t += kWarp) {
      const float p = expf(p_s[h * cap + t] - m);
      p_s[h * cap + t] = p;
      l += p;
    }
    l = warp_sum(l);
    if (lane == 0) {
      m_s[h] = m;
      l_s[h] = l;
    }
  }
  __syncthreads();

  // weighted values: one thread per (head, pair of dims). The row offsets
  // come from shared memory, so the loads of several positions are in flight
  // together (a per-position block-table lookup before each load would
  // serialise them).
  for (int idx = threadIdx.x; idx < G * (D / 2); idx += kAttnThreads) {
    const int h = idx / (D / 2), d2 = idx % (D / 2);
    float acc0 = 0.f, acc1 = 0.f;
#pragma unroll 8
    for (int t = 0; t < len; ++t) {
      const float p = p_s[h * cap + t];
      const float2 w = kv_load2<KV16>(a.kv.v, off_s[t] + 2 * d2);
      // an excluded slot (p = 0) is not multiplied: its row may be anything
      acc0 = fmaf(p, p == 0.f ? 0.f : w.x, acc0);
      acc1 = fmaf(p, p == 0.f ? 0.f : w.y, acc1);
    }
    float* ph = part + ((size_t)h * S + c) * (D + 2);
    ph[2 + 2 * d2] = acc0;
    ph[3 + 2 * d2] = acc1;
    if (d2 == 0) {
      ph[0] = len > 0 ? m_s[h] : -INFINITY;
      ph[1] = len > 0 ? l_s[h] : 0.f;
    }
  }
}

template <int D>
__global__ void k_attn_merge(AttnArgs a) {
  const int h = blockIdx.x, b = blockIdx.y, d = threadIdx.x, S = a.splits;
  const float* ph = a.part + ((size_t)b * a.Hq + h) * S * (D + 2);
  float M = -INFINITY;
  for (int c = 0; c < S; ++c) M = fmaxf(M, ph[(size_t)c * (D + 2)]);
  float num = 0.f, den = 0.f;
  for (int c = 0; c < S; ++c) {
    const float mc = ph[(size_t)c * (D + 2)];
    if (mc == -INFINITY) continue;
    const float w = expf(mc - M);
    den = fmaf(ph[(size_t)c * (D + 2) + 1], w, den);
    num = fmaf(ph[(size_t)c * (D + 2) + 2 + d], w, num);
  }
  a.out[((size_t)b * a.Hq + h) * D + d] = num / den;
}

template <int D, int GM, bool KV16>
static cudaError_t attn_split(const AttnArgs& a, int cap, cudaStream_t s) {
  const size_t smem = sizeof(float) * (size_t)((GM * cap + 1) & ~1) + sizeof(size_t) * (size_t)cap;
  cudaError_t e = ensure_smem<k_attn_split<D, GM, KV16>>();
  if (e != cudaSuccess) return e;
  k_attn_split<D, GM, KV16><<<dim3(a.splits, a.Hkv, a.B), kAttnThreads, smem, s>>>(a, cap);
  return cudaGetLastError();
}

template <int D, int GM>
static cudaError_t attn_dg(const AttnArgs& a, int cap, cudaStream_t s) {
  cudaError_t e = a.kv.bf16 ? attn_split<D, GM, true>(a, cap, s) : attn_split<D, GM, false>(a, cap, s);
  if (e != cudaSuccess) return e;
  k_attn_merge<D><<<dim3(a.Hq, a.B), D, 0, s>>>(a);
  return cudaGetLastError();
}

template <int D>
static cudaError_t attn_d(const AttnArgs& a, int cap, cudaStream_t s) {
  const int G = a.Hq / a.Hkv;
  if (G <= 1) return attn_dg<D, 1>(a, cap, s);
  if (G <= 2) return attn_dg<D, 2>(a, cap, s);
  if (G <= 4) return attn_dg<D, 4>(a, cap, s);
  return attn_dg<D, 8>(a, cap, s);
}

cudaError_t launch_attn(const AttnArgs& a, cudaStream_t s) {
  const int max_ctx = a.kv.paged ? a.kv.max_blocks_per_seq * a.kv.block_size : a.kv.max_ctx;
  const int cap = (max_ctx + a.splits - 1) / a.splits;
  return a.D == 64 ? attn_d<64>(a, cap, s) : attn_d<128>(a, cap, s);
}

}  // namespace nc
