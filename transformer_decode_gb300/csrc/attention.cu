// attention.cu -- RoPE + KV append, and split-K grouped-query decode attention.
//
// RoPE (nanoinfer "Model architecture", "KV cache"): half-split pairs
// (i, i + D/2), angle = float(pos) * inv_freq[i] as an fp32 product, applied
// once to K on insert; K and V are rounded to bf16 when stored.
//
// Attention (Tang section 2.2: online softmax is the monoid on (m, l, acc);
// section 2.5: split is valid for any associative monoid): the positions
// 0..pos of one (sequence, kv head) are cut into `splits` ranges. Each CTA
// reads its range of K and V once for all G query heads of the group (the
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
  pdl_wait();
  const int b = blockIdx.x;
  const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
  const int pos = a.positions[b];
  if (!a.kv.slot_ok(b, pos)) {
    if (threadIdx.x == 0 && blockIdx.y == 0 && a.status) atomicCAS(a.status, 0, (int)NC_ERR_POSITION);
    return;
  }
  const int qkv_dim = (a.Hq + 2 * a.Hkv) * D;
  const float* src = a.qkv + (size_t)b * qkv_dim;
  // blockIdx.y picks this CTA's heads: one per warp, so the heads run side by side
  for (int hh = blockIdx.y * (blockDim.x / kWarp) + warp; hh < a.Hq + a.Hkv;
       hh += gridDim.y * (blockDim.x / kWarp)) {
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
  const dim3 grid(a.B, (a.Hq + a.Hkv + 7) / 8);  // 8 warps per CTA, one head each
  const auto kern = a.D == 64 ? (a.kv.bf16 ? k_rope_qkv<64, true> : k_rope_qkv<64, false>)
                              : (a.kv.bf16 ? k_rope_qkv<128, true> : k_rope_qkv<128, false>);
  return launch_pdl(kern, grid, dim3(256), 0, s, a);
}

// ------------------------------------------------------------------ attention
constexpr int kAttnThreads = 256;
constexpr int kMaxChunk = 512;
constexpr int kMaxSplits = 128;  // splits of one (sequence, kv head); the merge keeps one weight each

int attn_splits(int B, int Hkv, int max_ctx) {
  const int target = 2 * num_sms();
  int s = (target + B * Hkv - 1) / (B * Hkv);
  const int lo = (max_ctx + kMaxChunk - 1) / kMaxChunk;
  const int hi = (max_ctx + 15) / 16;
  if (s > hi) s = hi;
  if (s < lo) s = lo;
  if (s > kMaxSplits) s = kMaxSplits;
  return s < 1 ? 1 : s;
}

size_t attn_part_floats(int B, int Hq, int D, int splits) {
  return (size_t)B * Hq * splits * (D + 2);
}

// Positions per chunk staged in shared memory.
constexpr int kAttnChunk = 64;

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// One CTA per (split c, kv head g, sequence b). The split's positions are
// scanned in chunks of kAttnChunk: the chunk's K and V rows are copied into
// shared memory with asynchronous 16-byte copies (the next chunk's copies in
// flight while this one is used), so the cache is read with coalesced
// transfers instead of per-thread row walks. Scores: one position per thread
// for all G heads (K rows padded by 16 bytes so the threads' equal-column
// reads fall in different banks; q reads are broadcasts). Softmax statistics
// run online over the chunks, one warp per head; values: one thread per
// (head, pair of dims), the running sums rescaled at each chunk.
template <int D, int GM, bool KV16>
__global__ void __launch_bounds__(kAttnThreads) k_attn_split(AttnArgs a, int cap) {
  constexpr int ES = KV16 ? 2 : 4;
  constexpr int RS = D + 16 / ES;  // padded row, elements
  constexpr int PPR = D * ES / 16; // 16-byte pieces per row
  extern __shared__ __align__(16) unsigned char sm[];
  unsigned char* kbuf = sm;                                   // [2][kAttnChunk][RS]
  unsigned char* vbuf = kbuf + 2 * kAttnChunk * RS * ES;      // [2][kAttnChunk][RS]
  float* p_s = reinterpret_cast<float*>(vbuf + 2 * kAttnChunk * RS * ES);  // [GM][kAttnChunk]
  size_t* off_s = reinterpret_cast<size_t*>(p_s + GM * kAttnChunk);      // [cap] row offsets
  __shared__ float q_s[GM][D];
  __shared__ float m_s[GM], l_s[GM], r_s[GM];
  const int c = blockIdx.x, g = blockIdx.y, b = blockIdx.z, S = gridDim.x;
  const int G = a.Hq / a.Hkv;
  const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
  pdl_wait();
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
  // row offsets of the split (the block table read once); ~0 marks a slot
  // outside the cache: its row is not copied and its score is -inf
  for (int t = threadIdx.x; t < len; t += kAttnThreads) {
    if (a.kv.slot_ok(b, t0 + t)) {
      off_s[t] = a.kv.offset(a.layer, b, g, t0 + t);
    } else {
      off_s[t] = ~(size_t)0;
      if (a.status) atomicCAS(a.status, 0, (int)NC_ERR_POSITION);
    }
  }
  if (threadIdx.x < GM) {
    m_s[threadIdx.x] = -INFINITY;
    l_s[threadIdx.x] = 0.f;
  }
  __syncthreads();

  const int nchunks = (len + kAttnChunk - 1) / kAttnChunk;
  const auto issue = [&](int ci) {
    const int q0 = ci * kAttnChunk, m = min(kAttnChunk, len - q0);
    unsigned char* kd = kbuf + (size_t)(ci & 1) * kAttnChunk * RS * ES;
    unsigned char* vd = vbuf + (size_t)(ci & 1) * kAttnChunk * RS * ES;
    for (int i = threadIdx.x; i < m * PPR; i += kAttnThreads) {
      const int row = i / PPR, piece = i % PPR;
      const size_t off = off_s[q0 + row];
      if (off == ~(size_t)0) continue;
      const size_t src = off * ES + (size_t)piece * 16;
      cp_async16(kd + (size_t)row * RS * ES + piece * 16,
                 static_cast<const unsigned char*>(a.kv.k) + src);
      cp_async16(vd + (size_t)row * RS * ES + piece * 16,
                 static_cast<const unsigned char*>(a.kv.v) + src);
    }
    cp_async_commit();
  };
  const float scale = 1.f / sqrtf((float)D);
  const int h_pv = threadIdx.x / (D / 2), d2 = threadIdx.x % (D / 2);
  const bool pv = threadIdx.x < G * (D / 2);
  float acc0 = 0.f, acc1 = 0.f;
  if (nchunks > 0) issue(0);
  for (int ci = 0; ci < nchunks; ++ci) {
    if (ci + 1 < nchunks) {
      issue(ci + 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const int q0 = ci * kAttnChunk, m = min(kAttnChunk, len - q0);
    const unsigned char* kc = kbuf + (size_t)(ci & 1) * kAttnChunk * RS * ES;
    const unsigned char* vc = vbuf + (size_t)(ci & 1) * kAttnChunk * RS * ES;
    // scores of every head for one position per thread
    for (int t = threadIdx.x; t < m; t += kAttnThreads) {
      if (off_s[q0 + t] == ~(size_t)0) {
#pragma unroll
        for (int h = 0; h < GM; ++h) p_s[h * kAttnChunk + t] = -INFINITY;
        continue;
      }
      float sc[GM];
#pragma unroll
      for (int h = 0; h < GM; ++h) sc[h] = 0.f;
#pragma unroll 4
      for (int k4 = 0; k4 < D / 4; ++k4) {
        float kf[4];
        if constexpr (KV16) {
          const uint2 w = *reinterpret_cast<const uint2*>(kc + ((size_t)t * RS + 4 * k4) * ES);
          kf[0] = bf16_lo(w.x); kf[1] = bf16_hi(w.x); kf[2] = bf16_lo(w.y); kf[3] = bf16_hi(w.y);
        } else {
          const float4 w = *reinterpret_cast<const float4*>(kc + ((size_t)t * RS + 4 * k4) * ES);
          kf[0] = w.x; kf[1] = w.y; kf[2] = w.z; kf[3] = w.w;
        }
#pragma unroll
        for (int h = 0; h < GM; ++h) {
          const float4 qv = *reinterpret_cast<const float4*>(&q_s[h][4 * k4]);
          sc[h] = fmaf(qv.x, kf[0], sc[h]);
          sc[h] = fmaf(qv.y, kf[1], sc[h]);
          sc[h] = fmaf(qv.z, kf[2], sc[h]);
          sc[h] = fmaf(qv.w, kf[3], sc[h]);
        }
      }
#pragma unroll
      for (int h = 0; h < GM; ++h) p_s[h * kAttnChunk + t] = sc[h] * scale;
    }
    __syncthreads();
    // running softmax statistics, one warp per head
    for (int h = warp; h < G; h += kAttnThreads / kWarp) {
      float mx = -INFINITY;
      for (int t = lane; t < m; t += kWarp) mx = fmaxf(mx, p_s[h * kAttnChunk + t]);
      mx = warp_max(mx);
      const float m_new = fmaxf(m_s[h], mx);
      float l = 0.f;
      for (int t = lane; t < m; t += kWarp) {
        const float x = p_s[h * kAttnChunk + t];
        const float p = x == -INFINITY ? 0.f : expf(x - m_new);
        p_s[h * kAttnChunk + t] = p;
        l += p;
      }
      l = warp_sum(l);
      if (lane == 0) {
        const float r = m_s[h] == -INFINITY ? 0.f : expf(m_s[h] - m_new);
        r_s[h] = r;
        l_s[h] = l_s[h] * r + l;
        m_s[h] = m_new;
      }
    }
    __syncthreads();
    // values, running sums rescaled by the chunk's factor
    if (pv) {
      float e0 = 0.f, e1 = 0.f;
#pragma unroll 4
      for (int t = 0; t < m; ++t) {
        const float p = p_s[h_pv * kAttnChunk + t];
        float2 v;
        if constexpr (KV16) {
          const uint32_t w = *reinterpret_cast<const uint32_t*>(vc + ((size_t)t * RS + 2 * d2) * ES);
          v = make_float2(bf16_lo(w), bf16_hi(w));
        } else {
          v = *reinterpret_cast<const float2*>(vc + ((size_t)t * RS + 2 * d2) * ES);
        }
        // a slot outside the cache (p = 0) left its row stale: not multiplied
        e0 = fmaf(p, p == 0.f ? 0.f : v.x, e0);
        e1 = fmaf(p, p == 0.f ? 0.f : v.y, e1);
      }
      const float r = r_s[h_pv];
      acc0 = fmaf(acc0, r, e0);
      acc1 = fmaf(acc1, r, e1);
    }
    __syncthreads();  // the buffers of this chunk are refilled two chunks on
  }
  if (pv) {
    float* ph = part + ((size_t)h_pv * S + c) * (D + 2);
    ph[2 + 2 * d2] = acc0;
    ph[3 + 2 * d2] = acc1;
    if (d2 == 0) {
      ph[0] = len > 0 ? m_s[h_pv] : -INFINITY;
      ph[1] = len > 0 ? l_s[h_pv] : 0.f;
    }
  }
}

template <int D>
__global__ void k_attn_merge(AttnArgs a) {
  // M = max_c m_c and the split weights w_c = e^(m_c - M) are formed once and
  // shared; each thread then sums its dimension over the splits with the
  // loads independent of one another
  __shared__ float w_s[kMaxSplits];
  __shared__ float red[2][D / kWarp];
  const int h = blockIdx.x, b = blockIdx.y, d = threadIdx.x, S = a.splits;
  const int warp = d / kWarp, lane = d % kWarp;
  pdl_wait();
  const float* ph = a.part + ((size_t)b * a.Hq + h) * S * (D + 2);
  float M = -INFINITY;
  for (int c = d; c < S; c += D) M = fmaxf(M, ph[(size_t)c * (D + 2)]);
  M = warp_max(M);
  if (lane == 0) red[0][warp] = M;
  __syncthreads();
  M = red[0][0];
  for (int i = 1; i < D / kWarp; ++i) M = fmaxf(M, red[0][i]);
  float den = 0.f;
  for (int c = d; c < S; c += D) {
    const float m = ph[(size_t)c * (D + 2)];
    const float w = m == -INFINITY ? 0.f : expf(m - M);
    w_s[c] = w;
    den = fmaf(ph[(size_t)c * (D + 2) + 1], w, den);
  }
  den = warp_sum(den);
  if (lane == 0) red[1][warp] = den;
  __syncthreads();
  den = 0.f;
  for (int i = 0; i < D / kWarp; ++i) den += red[1][i];
  float num = 0.f;
#pragma unroll 8
  for (int c = 0; c < S; ++c) num = fmaf(ph[(size_t)c * (D + 2) + 2 + d], w_s[c], num);
  a.out[((size_t)b * a.Hq + h) * D + d] = num / den;
}

template <int D, int GM, bool KV16>
static cudaError_t attn_split(const AttnArgs& a, int cap, cudaStream_t s) {
  constexpr int ES = KV16 ? 2 : 4, RS = D + 16 / ES;
  const size_t smem = (size_t)4 * kAttnChunk * RS * ES + sizeof(float) * GM * kAttnChunk +
                      sizeof(size_t) * (size_t)cap;
  cudaError_t e = ensure_smem<k_attn_split<D, GM, KV16>>();
  if (e != cudaSuccess) return e;
  return launch_pdl(k_attn_split<D, GM, KV16>, dim3(a.splits, a.Hkv, a.B), dim3(kAttnThreads), smem,
                    s, a, cap);
}

template <int D, int GM>
static cudaError_t attn_dg(const AttnArgs& a, int cap, cudaStream_t s) {
  cudaError_t e = a.kv.bf16 ? attn_split<D, GM, true>(a, cap, s) : attn_split<D, GM, false>(a, cap, s);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_attn_merge<D>, dim3(a.Hq, a.B), dim3(D), 0, s, a);
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
