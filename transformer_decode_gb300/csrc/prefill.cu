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
// last position any of its tokens sees. The 256 threads tile each 64 x 64
// block of scores as 16 x 16 blocks of 4 x 4: thread (rb, cb) holds rows
// 4 rb .. 4 rb + 3 against positions 4 cb .. 4 cb + 3, with q and k stored
// transposed ([dim][row], [dim][position]) so that each step of the dot
// products is two 16-byte loads for 16 multiply-adds. The row's running
// (max, sum) is reduced over the 16 threads of its row block; the
// probabilities go through shared memory by rows (one 16-byte store per row
// and thread), and the same thread accumulates rows 4 rb .. 4 rb + 3 of the
// output over dims D/16 cb .., four positions per step.
#include <cuda_runtime.h>
#include <math.h>

#include "kernels.h"

namespace nc {

constexpr int kPFRows = 64;      // query rows per CTA
constexpr int kPFTile = 64;      // positions per K/V tile
constexpr int kPFThreads = 256;  // 16 row blocks x 16 column blocks

size_t prefill_attn_smem(int D) {
  // qT [D][64], kT [D][64], V [64][D], P [64 rows][64 positions]
  return sizeof(float) * ((size_t)D * kPFRows + (size_t)D * kPFTile + (size_t)kPFTile * D +
                          (size_t)kPFTile * kPFRows);
}

template <int D, bool KV16>
__global__ void __launch_bounds__(kPFThreads, 2) k_prefill_attn(const PrefillAttnArgs a) {
  constexpr int DC = D / 16;  // output dims per thread
  extern __shared__ float4 pf_raw[];
  float* qT = reinterpret_cast<float*>(pf_raw);  // [D][64]
  float* kT = qT + D * kPFRows;                  // [D][64]
  float* vs = kT + D * kPFTile;                  // [64][D]
  float* ps = vs + kPFTile * D;                  // [64 rows][64 positions]
  pdl_wait();
  const int G = a.Hq / a.Hkv, g = blockIdx.y;
  const int qt = kPFRows / G;  // tokens per block
  const int nblk = (a.T + qt - 1) / qt;
  const int tid = threadIdx.x, rb = tid / 16, cb = tid % 16;
  const float scale = 1.f / sqrtf((float)D);
  // With a.pair the CTA takes token blocks x and nblk - 1 - x: a block late
  // in the prompt (many positions to scan) with an early one, so the CTAs'
  // work is about even.
  for (int pass = 0; pass < (a.pair ? 2 : 1); ++pass) {
  const int blk = pass == 0 ? (int)blockIdx.x : nblk - 1 - (int)blockIdx.x;
  if (pass == 1 && blk <= (int)blockIdx.x) break;  // the middle block, or none
  const int i0 = blk * qt, i1 = min(a.T, i0 + qt);
  const int nrows = (i1 - i0) * G;
  __syncthreads();  // the previous block's shared memory is no longer read

  // the CTA's query rows, transposed: row r = token i0 + r / G, head g G + r % G
  for (int e = tid; e < kPFRows * (D / 4); e += kPFThreads) {
    const int r = e % kPFRows, c = e / kPFRows;  // consecutive threads: consecutive rows
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r < nrows)
      v = *reinterpret_cast<const float4*>(a.q + ((size_t)(i0 + r / G) * a.Hq + g * G + r % G) * D + 4 * c);
    qT[(4 * c + 0) * kPFRows + r] = v.x;
    qT[(4 * c + 1) * kPFRows + r] = v.y;
    qT[(4 * c + 2) * kPFRows + r] = v.z;
    qT[(4 * c + 3) * kPFRows + r] = v.w;
  }
  int qpos[4];
  bool rok[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = 4 * rb + i;
    rok[i] = r < nrows;
    qpos[i] = a.start + i0 + r / G;  // the row's own position
  }
  float m[4], l[4], o[4][DC];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.f;
#pragma unroll
    for (int c = 0; c < DC; ++c) o[i][c] = 0.f;
  }
  const int kv_end = a.start + i1;  // positions [0, kv_end) are seen by some row
  for (int base = 0; base < kv_end; base += kPFTile) {
    __syncthreads();  // the previous tile (and, first, nothing) is no longer read
    // K, transposed (consecutive threads: consecutive positions, so the
    // column stores hit consecutive banks), then V by rows; each loop is
    // unrolled so a thread's loads are all in flight before its stores
#pragma unroll
    for (int e = tid; e < kPFTile * (D / 8); e += kPFThreads) {
      const int p = e % kPFTile, c = e / kPFTile, pos = base + p;
      float f[8];
      if (pos < kv_end && a.kv.slot_ok(a.seq, pos)) {
        kv_load8<KV16>(a.kv.k, a.kv.offset(a.layer, a.seq, g, pos) + 8 * c, f);
      } else {
#pragma unroll
        for (int u = 0; u < 8; ++u) f[u] = 0.f;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) kT[(8 * c + u) * kPFTile + p] = f[u];
    }
#pragma unroll
    for (int e = tid; e < kPFTile * (D / 8); e += kPFThreads) {
      const int c = e % (D / 8), p = e / (D / 8), pos = base + p;
      float f[8];
      if (pos < kv_end && a.kv.slot_ok(a.seq, pos)) {
        kv_load8<KV16>(a.kv.v, a.kv.offset(a.layer, a.seq, g, pos) + 8 * c, f);
      } else {
#pragma unroll
        for (int u = 0; u < 8; ++u) f[u] = 0.f;
      }
      *reinterpret_cast<float4*>(vs + p * D + 8 * c) = make_float4(f[0], f[1], f[2], f[3]);
      *reinterpret_cast<float4*>(vs + p * D + 8 * c + 4) = make_float4(f[4], f[5], f[6], f[7]);
    }
    __syncthreads();
    // scores of rows 4 rb + i against positions 4 cb + j
    float sc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) sc[i][j] = 0.f;
#pragma unroll 8
    for (int d = 0; d < D; ++d) {
      const float4 q4 = *reinterpret_cast<const float4*>(qT + d * kPFRows + 4 * rb);
      const float4 k4 = *reinterpret_cast<const float4*>(kT + d * kPFTile + 4 * cb);
      const float qv[4] = {q4.x, q4.y, q4.z, q4.w}, kv[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) sc[i][j] = fmaf(qv[i], kv[j], sc[i][j]);
    }
    // the causal mask and the online softmax of each row (its 64 scores on
    // the 16 threads of the row block); the weights to ps
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float pv[4], mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int pos = base + 4 * cb + j;
        pv[j] = rok[i] && pos <= qpos[i] ? sc[i][j] * scale : -INFINITY;
        mx = fmaxf(mx, pv[j]);
      }
#pragma unroll
      for (int off = 1; off < 16; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
      const float mn = fmaxf(m[i], mx);
      // a row with nothing seen yet keeps m = -inf and contributes nothing
      const float corr = m[i] == -INFINITY ? 0.f : expf(m[i] - mn);
      float sum = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        pv[j] = pv[j] == -INFINITY ? 0.f : expf(pv[j] - mn);
        sum += pv[j];
      }
#pragma unroll
      for (int off = 1; off < 16; off <<= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, off);
      l[i] = l[i] * corr + sum;
      m[i] = mn;
#pragma unroll
      for (int c = 0; c < DC; ++c) o[i][c] *= corr;
      *reinterpret_cast<float4*>(ps + (4 * rb + i) * kPFTile + 4 * cb) =
          make_float4(pv[0], pv[1], pv[2], pv[3]);
    }
    __syncthreads();  // the weights of every row
    // P V: rows 4 rb + i, dims DC cb .. DC cb + DC - 1 (a masked or empty
    // position has weight 0 over a zero or finite value)
#pragma unroll 2
    for (int p4 = 0; p4 < kPFTile; p4 += 4) {
      float pw[4][4];  // [row i][position p4 + j]
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 pr = *reinterpret_cast<const float4*>(ps + (4 * rb + i) * kPFTile + p4);
        pw[i][0] = pr.x;
        pw[i][1] = pr.y;
        pw[i][2] = pr.z;
        pw[i][3] = pr.w;
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float v[DC];
#pragma unroll
        for (int c = 0; c < DC; c += 4) {
          const float4 v4 = *reinterpret_cast<const float4*>(vs + (p4 + j) * D + DC * cb + c);
          v[c] = v4.x;
          v[c + 1] = v4.y;
          v[c + 2] = v4.z;
          v[c + 3] = v4.w;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int c = 0; c < DC; ++c) o[i][c] = fmaf(pw[i][j], v[c], o[i][c]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = 4 * rb + i;
    if (r >= nrows) continue;
    const float inv = l[i] > 0.f ? 1.f / l[i] : 0.f;
    float* dst = a.out + ((size_t)(i0 + r / G) * a.Hq + g * G + r % G) * D + DC * cb;
#pragma unroll
    for (int c = 0; c < DC; c += 4)
      *reinterpret_cast<float4*>(dst + c) =
          make_float4(o[i][c] * inv, o[i][c + 1] * inv, o[i][c + 2] * inv, o[i][c + 3] * inv);
  }
  }  // pass
}

cudaError_t launch_prefill_attn(const PrefillAttnArgs& args, cudaStream_t s) {
  PrefillAttnArgs a = args;
  const int G = a.Hq / a.Hkv, qt = kPFRows / G;
  const int nblk = (a.T + qt - 1) / qt;
  // pair early and late token blocks when the blocks outnumber the SMs
  a.pair = nblk * a.Hkv > num_sms() ? 1 : 0;
  const dim3 grid(a.pair ? (nblk + 1) / 2 : nblk, a.Hkv);
  const size_t smem = prefill_attn_smem(a.D);
  auto kern = a.D == 64 ? (a.kv.bf16 ? k_prefill_attn<64, true> : k_prefill_attn<64, false>)
                        : (a.kv.bf16 ? k_prefill_attn<128, true> : k_prefill_attn<128, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, grid, dim3(kPFThreads), smem, s, a);
}

}  // namespace nc
