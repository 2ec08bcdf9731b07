// prefill.cu -- causal attention of a prefill chunk, flash style.
//
// A prompt run as one forward pass (the nanoinfer page's batched prefill:
// the token loop inside the weight-row loop, so each weight row is read once
// per prompt) needs, per layer, the attention of every prompt token over the
// cached positions and the prompt tokens before it (the causal mask j <= i,
// nanoinfer "Model architecture"). Tang section 2.3 derives the fused form:
// the softmax is the monoid on (m, l, acc) (section 2.2), so the scores of a
// query never have to exist all at once: the keys and values stream through
// in tiles and each query row keeps its running state.
//
// One CTA takes 64 query rows, (token, head) pairs of one kv head's group
// (64 / G consecutive tokens x the G heads; the repeat of K/V across the
// group folded into indexing), and streams the sequence's K and V through
// shared memory in tiles of 64 positions (fp32 or widened bf16), up to the
// last position any of its tokens sees. Each warp owns 8 rows, processed 4
// at a time: scores of 2 positions per lane against 4 rows, a warp-wide max
// and sum per row, the probabilities through shared memory, then P V with
// the lane holding D / 32 output dimensions of each row.
#include <cuda_runtime.h>
#include <math.h>

#include "kernels.h"

namespace nc {

constexpr int kPFRows = 64;      // query rows per CTA
constexpr int kPFTile = 64;      // positions per K/V tile
constexpr int kPFThreads = 256;  // 8 warps x 8 rows

size_t prefill_attn_smem(int D) {
  return sizeof(float) * ((size_t)kPFRows * D + (size_t)kPFTile * (D + 4) + (size_t)kPFTile * D +
                          (size_t)(kPFThreads / kWarp) * kPFTile * 4);
}

template <int D, bool KV16>
__global__ void __launch_bounds__(kPFThreads) k_prefill_attn(const PrefillAttnArgs a) {
  constexpr int E = D / 32;          // output dimensions per lane
  constexpr int KS = D + 4;          // padded K row (conflict-free row-per-lane reads)
  extern __shared__ float4 pf_raw[];
  float* qs = reinterpret_cast<float*>(pf_raw);  // [64][D]
  float* ks = qs + kPFRows * D;                  // [64][D + 4]
  float* vs = ks + kPFTile * KS;                 // [64][D]
  float* ps = vs + kPFTile * D;                  // [8 warps][64 positions][4 rows]
  pdl_wait();
  const int G = a.Hq / a.Hkv, g = blockIdx.y;
  const int qt = kPFRows / G;                    // tokens per CTA
  const int i0 = blockIdx.x * qt, i1 = min(a.T, i0 + qt);
  const int nrows = (i1 - i0) * G;
  const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
  const float scale = 1.f / sqrtf((float)D);

  // the CTA's query rows: row r = token i0 + r / G, head g G + r % G
  for (int e = threadIdx.x; e < kPFRows * D / 4; e += kPFThreads) {
    const int r = e / (D / 4), c = e % (D / 4);
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r < nrows) {
      const int t = i0 + r / G, h = g * G + r % G;
      v = *reinterpret_cast<const float4*>(a.q + ((size_t)t * a.Hq + h) * D + 4 * c);
    }
    *reinterpret_cast<float4*>(qs + r * D + 4 * c) = v;
  }

  float m[8], l[8], o[8][E];
#pragma unroll
  for (int rr = 0; rr < 8; ++rr) {
    m[rr] = -INFINITY;
    l[rr] = 0.f;
#pragma unroll
    for (int j = 0; j < E; ++j) o[rr][j] = 0.f;
  }
  const int kv_end = a.start + i1;  // positions [0, kv_end) are seen by some row
  float* pw = ps + warp * kPFTile * 4;
  for (int base = 0; base < kv_end; base += kPFTile) {
    __syncthreads();  // the previous tile is no longer read
    for (int e = threadIdx.x; e < kPFTile * D / 8; e += kPFThreads) {
      const int p = e / (D / 8), c = e % (D / 8), pos = base + p;
      float f[8];
      if (pos < kv_end && a.kv.slot_ok(a.seq, pos)) {
        const size_t off = a.kv.offset(a.layer, a.seq, g, pos) + 8 * c;
        kv_load8<KV16>(a.kv.k, off, f);
#pragma unroll
        for (int u = 0; u < 8; ++u) ks[p * KS + 8 * c + u] = f[u];
        kv_load8<KV16>(a.kv.v, off, f);
#pragma unroll
        for (int u = 0; u < 8; ++u) vs[p * D + 8 * c + u] = f[u];
      } else {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          ks[p * KS + 8 * c + u] = 0.f;
          vs[p * D + 8 * c + u] = 0.f;
        }
      }
    }
    __syncthreads();
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
      const int r0 = warp * 8 + blk * 4;
      // scores of positions lane and lane + 32 against rows r0 .. r0 + 3
      float s[4][2];
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) s[rr][0] = s[rr][1] = 0.f;
#pragma unroll 4
      for (int d = 0; d < D; d += 4) {
        const float4 k0 = *reinterpret_cast<const float4*>(ks + lane * KS + d);
        const float4 k1 = *reinterpret_cast<const float4*>(ks + (lane + 32) * KS + d);
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
          const float4 q = *reinterpret_cast<const float4*>(qs + (r0 + rr) * D + d);
          s[rr][0] = fmaf(q.x, k0.x, fmaf(q.y, k0.y, fmaf(q.z, k0.z, fmaf(q.w, k0.w, s[rr][0]))));
          s[rr][1] = fmaf(q.x, k1.x, fmaf(q.y, k1.y, fmaf(q.z, k1.z, fmaf(q.w, k1.w, s[rr][1]))));
        }
      }
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        const int r = r0 + rr;
        const int qpos = a.start + i0 + r / G;  // the row's own position
        const bool row_ok = r < nrows;
        float p2[2];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int pos = base + lane + 32 * c;
          p2[c] = row_ok && pos <= qpos ? s[rr][c] * scale : -INFINITY;
        }
        const float mt = warp_max(fmaxf(p2[0], p2[1]));
        const int ri = blk * 4 + rr;
        const float mn = fmaxf(m[ri], mt);
        // a row with nothing seen yet keeps m = -inf and contributes nothing
        const float corr = m[ri] == -INFINITY ? 0.f : expf(m[ri] - mn);
#pragma unroll
        for (int c = 0; c < 2; ++c) p2[c] = p2[c] == -INFINITY ? 0.f : expf(p2[c] - mn);
        l[ri] = l[ri] * corr + warp_sum(p2[0] + p2[1]);
        m[ri] = mn;
#pragma unroll
        for (int j = 0; j < E; ++j) o[ri][j] *= corr;
        pw[lane * 4 + rr] = p2[0];
        pw[(lane + 32) * 4 + rr] = p2[1];
      }
      __syncwarp();
      // P V: output dimension lane + 32 j of the 4 rows
#pragma unroll 4
      for (int p = 0; p < kPFTile; ++p) {
        const float4 pr = *reinterpret_cast<const float4*>(pw + p * 4);
#pragma unroll
        for (int j = 0; j < E; ++j) {
          const float v = vs[p * D + lane + 32 * j];
          o[blk * 4 + 0][j] = fmaf(pr.x, v, o[blk * 4 + 0][j]);
          o[blk * 4 + 1][j] = fmaf(pr.y, v, o[blk * 4 + 1][j]);
          o[blk * 4 + 2][j] = fmaf(pr.z, v, o[blk * 4 + 2][j]);
          o[blk * 4 + 3][j] = fmaf(pr.w, v, o[blk * 4 + 3][j]);
        }
      }
      __syncwarp();  // pw is rewritten by the next block
    }
  }
#pragma unroll
  for (int ri = 0; ri < 8; ++ri) {
    const int r = warp * 8 + ri;
    if (r >= nrows) continue;
    const int t = i0 + r / G, h = g * G + r % G;
    const float inv = l[ri] > 0.f ? 1.f / l[ri] : 0.f;
#pragma unroll
    for (int j = 0; j < E; ++j) a.out[((size_t)t * a.Hq + h) * D + lane + 32 * j] = o[ri][j] * inv;
  }
}

cudaError_t launch_prefill_attn(const PrefillAttnArgs& a, cudaStream_t s) {
  const int G = a.Hq / a.Hkv, qt = kPFRows / G;
  const dim3 grid((a.T + qt - 1) / qt, a.Hkv);
  const size_t smem = prefill_attn_smem(a.D);
  auto kern = a.D == 64 ? (a.kv.bf16 ? k_prefill_attn<64, true> : k_prefill_attn<64, false>)
                        : (a.kv.bf16 ? k_prefill_attn<128, true> : k_prefill_attn<128, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, grid, dim3(kPFThreads), smem, s, a);
}

}  // namespace nc
