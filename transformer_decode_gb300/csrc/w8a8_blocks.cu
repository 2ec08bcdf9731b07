// w8a8_blocks.cu -- W8A8 with activations quantised in blocks of 32.
//
// nanoinfer, INT8 activation section: one activation scale per 32 values
// ("one per 32"), so an outlier only widens its own block: per-row scales
// cost 4.97% activation error on a 4864-wide vector against 0.90% per 32.
// Weights stay int8 with one scale per output row, range [-127, 127], round
// half away from zero. For each row n and block b the int32 sum
// acc[n, b] = sum over the block of Wq[n, k] * xq[k] is exact (dp4a), and
// y[n] = sum_b float(acc[n, b]) * (w_scale[n] * sx[b]) (+ bias) in fp32.
//
// Layout of the work: a 16-byte weight chunk is 16 codes, half a block, and
// lane l streams chunks l, l + 32, ...: the two halves of a block sit on the
// lanes 2j and 2j + 1 of a pair, which add their int32 sums with one
// shuffle; the even lane then owns the block's fp32 term.
#include <cuda_runtime.h>
#include <math.h>

#include "kernels.h"

namespace nc {
namespace {

constexpr int kB32Threads = 256;
constexpr int kB32Warps = kB32Threads / kWarp;
constexpr int kActBlock = 32;

__device__ __forceinline__ int8_t quant_code(float v, float s) {
  if (s == 0.f) return 0;
  float r = roundf(__fdiv_rn(v, s));
  r = fminf(fmaxf(r, -127.f), 127.f);
  return (int8_t)(int)r;
}

__device__ __forceinline__ float silu_mul_b32(float g, float u) {
  const float e = expf(-fabsf(g));  // nanoinfer "Phase 8" sigmoid form
  const float sig = g >= 0.f ? 1.f / (1.f + e) : e / (1.f + e);
  return (g * sig) * u;
}

// Block i owns the rows [N i / grid, N (i + 1) / grid) (one wave). EPI:
// Store (+ bias), Residual (y += ...), SwiGLU (rows n and N + n are gate and
// up: y = silu(gate) * up). ARGMAX: also the arg-max of each sequence's y
// (the logits), lowest index on ties, combined by the last CTA to finish.
template <int BT, Epi EPI, bool ARGMAX>
__global__ void __launch_bounds__(kB32Threads) k_w8a8_b32(const __grid_constant__ W8BArgs a) {
  extern __shared__ int4 smem_i4[];
  const int K = a.K, nblk = K / kActBlock;
  int8_t* xq = reinterpret_cast<int8_t*>(smem_i4);                   // [BT][K]
  float* sx = reinterpret_cast<float*>(xq + (size_t)BT * K);          // [BT][nblk]
  __shared__ float rn[BT];
  __shared__ float part[kB32Warps][BT];
  __shared__ unsigned long long best_s[kB32Warps][BT];
  __shared__ bool last_s;
  constexpr int R = EPI == Epi::SwiGLU ? 2 : 1;
  constexpr int U = 4;  // 16-byte chunks per row in flight
  const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
  const int r0 = (int)((long long)a.N * blockIdx.x / gridDim.x);
  const int r1 = (int)((long long)a.N * (blockIdx.x + 1) / gridDim.x);

  // RMSNorm factor per sequence (partials added in a fixed order)
  if (a.gamma) {
#pragma unroll 1
    for (int b = 0; b < BT; ++b) {
      float ss = 0.f;
      if (b < a.B)
        for (int k = threadIdx.x; k < K; k += kB32Threads) {
          const float v = a.x[(size_t)b * K + k];
          ss = fmaf(v, v, ss);
        }
      ss = warp_sum(ss);
      if (lane == 0) part[warp][b] = ss;
    }
    __syncthreads();
  }
  if (threadIdx.x < BT) {
    float r = 1.f;
    if (a.gamma) {
      float ss = 0.f;
      for (int w = 0; w < kB32Warps; ++w) ss += part[w][threadIdx.x];
      r = 1.f / sqrtf(ss / (float)K + a.eps);
    }
    rn[threadIdx.x] = r;
  }
  __syncthreads();
  // one thread per (sequence, block): the block's amax, its scale and codes
  for (int i = threadIdx.x; i < BT * nblk; i += kB32Threads) {
    const int b = i / nblk, blk = i - b * nblk;
    float v[kActBlock];
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < kActBlock; ++j) {
      const int k = blk * kActBlock + j;
      float t = 0.f;
      if (b < a.B) {
        t = a.x[(size_t)b * K + k];
        if (a.gamma) t = (t * rn[b]) * bf16_to_f32(a.gamma[k]);
      }
      v[j] = t;
      amax = fmaxf(amax, fabsf(t));
    }
    const float s = __fdiv_rn(amax, 127.f);
    sx[i] = s;
    if (blockIdx.x == 0 && a.sx_out && b < a.B) a.sx_out[(size_t)b * nblk + blk] = s;
#pragma unroll
    for (int j = 0; j < kActBlock; ++j) {
      const int8_t q = quant_code(v[j], s);
      xq[(size_t)b * K + blk * kActBlock + j] = q;
      if (blockIdx.x == 0 && a.xq_out && b < a.B) a.xq_out[(size_t)b * K + blk * kActBlock + j] = q;
    }
  }
  __syncthreads();

  const int nchunk = K / 16;  // even: K is a multiple of 32
  unsigned long long best[BT];
#pragma unroll
  for (int b = 0; b < BT; ++b) best[b] = 0ull;
  for (int n = r0 + warp; n < r1; n += kB32Warps) {  // no block barrier below
    float yf[R][BT];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int b = 0; b < BT; ++b) yf[r][b] = 0.f;
    const int8_t* rows[R];
    float sw[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      rows[r] = a.Wq + ((size_t)r * a.N + n) * K;
      sw[r] = a.w_scale[(size_t)r * a.N + n];
    }
    // the trip count is the same on every lane (the pair shuffle below needs
    // the whole warp); chunks past the row are predicated off
    for (int cb = 0; cb < nchunk; cb += U * kWarp) {
      const int c0 = cb + lane;
      uint4 w[R][U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + u * kWarp;
#pragma unroll
        for (int r = 0; r < R; ++r)
          w[r][u] = c < nchunk ? ld_stream(rows[r] + (size_t)c * 16) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + u * kWarp;  // the pair (2j, 2j + 1) is in range together
        const int blk = c >> 1;
#pragma unroll
        for (int b = 0; b < BT; ++b) {
          int4 xv = make_int4(0, 0, 0, 0);
          if (c < nchunk) xv = *reinterpret_cast<const int4*>(xq + (size_t)b * K + (size_t)c * 16);
#pragma unroll
          for (int r = 0; r < R; ++r) {
            int acc = 0;
            acc = __dp4a((int)w[r][u].x, xv.x, acc);
            acc = __dp4a((int)w[r][u].y, xv.y, acc);
            acc = __dp4a((int)w[r][u].z, xv.z, acc);
            acc = __dp4a((int)w[r][u].w, xv.w, acc);
            acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 1);  // the block's exact int32 sum
            if ((lane & 1) == 0 && c < nchunk && b < a.B) {
              yf[r][b] = fmaf((float)acc, sw[r] * sx[b * nblk + blk], yf[r][b]);
              if (a.acc_out) a.acc_out[((size_t)b * R * a.N + (size_t)r * a.N + n) * nblk + blk] = acc;
            }
          }
        }
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int b = 0; b < BT; ++b) yf[r][b] = warp_sum(yf[r][b]);
    if constexpr (ARGMAX) {
#pragma unroll
      for (int b = 0; b < BT; ++b)
        if (b < a.B) {
          const unsigned long long key = argmax_key(yf[0][b], (uint32_t)n);
          best[b] = key > best[b] ? key : best[b];
        }
    }
    if (lane < BT && lane < a.B) {
      float v[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        v[r] = yf[r][0];
#pragma unroll
        for (int b = 1; b < BT; ++b)
          if (lane == b) v[r] = yf[r][b];
      }
      float* yp = a.y + (size_t)lane * a.N + n;
      if constexpr (EPI == Epi::Store) {
        *yp = a.bias ? v[0] + bf16_to_f32(a.bias[n]) : v[0];
      } else if constexpr (EPI == Epi::Residual) {
        *yp = *yp + v[0];
      } else {
        *yp = silu_mul_b32(v[0], v[R - 1]);
      }
    }
  }
  if constexpr (ARGMAX) {
    // per-CTA best keys, then the last CTA to finish combines them (a max over
    // integer keys: the order of the CTAs does not matter)
    if (lane == 0)
#pragma unroll
      for (int b = 0; b < BT; ++b) best_s[warp][b] = best[b];
    __syncthreads();
    if (threadIdx.x < BT && threadIdx.x < a.B) {
      unsigned long long m = 0ull;
      for (int w = 0; w < kB32Warps; ++w) m = best_s[w][threadIdx.x] > m ? best_s[w][threadIdx.x] : m;
      a.part[(size_t)threadIdx.x * gridDim.x + blockIdx.x] = m;
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) last_s = atomicAdd(a.ticket, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!last_s) return;
    __threadfence();
    for (int b = warp; b < a.B; b += kB32Warps) {
      unsigned long long m = 0ull;
      for (int i = lane; i < (int)gridDim.x; i += kWarp) {
        const unsigned long long k = __ldcg(a.part + (size_t)b * gridDim.x + i);
        m = k > m ? k : m;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long t = __shfl_xor_sync(0xFFFFFFFFu, m, o);
        m = t > m ? t : m;
      }
      if (lane == 0) {
        const bool nan = m == ~0ull;
        const int32_t tok = nan ? -1 : (int32_t)(0xFFFFFFFFu - (uint32_t)(m & 0xFFFFFFFFull));
        if (a.next) a.next[b] = tok;
        if (nan && a.status) atomicCAS(a.status, 0, (int)NC_ERR_INVALID_ARGUMENT);
        if (a.advance_tokens) a.advance_tokens[b] = nan ? 0 : tok;
        if (a.advance_positions) a.advance_positions[b] += 1;
      }
    }
    if (threadIdx.x == 0) *a.ticket = 0u;
  }
}

template <int BT, Epi EPI, bool ARGMAX>
cudaError_t launch_bt(const W8BArgs& a, cudaStream_t s) {
  const size_t smem = w8a8_b32_smem_bytes(BT, a.K);
  cudaError_t e = ensure_smem<k_w8a8_b32<BT, EPI, ARGMAX>>();
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_w8a8_b32<BT, EPI, ARGMAX>,
                                                    kB32Threads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  int grid = per_sm * num_sms();
  const int rows_cta = (a.N + kB32Warps - 1) / kB32Warps;
  grid = grid < rows_cta ? grid : rows_cta;
  if (ARGMAX && grid > lm_head_grid()) grid = lm_head_grid();  // the partials hold that many
  k_w8a8_b32<BT, EPI, ARGMAX><<<grid, kB32Threads, smem, s>>>(a);
  return cudaGetLastError();
}

template <Epi EPI, bool ARGMAX>
cudaError_t launch_epi(const W8BArgs& a, cudaStream_t s) {
  if (a.B <= 1) return launch_bt<1, EPI, ARGMAX>(a, s);
  if (a.B <= 2) return launch_bt<2, EPI, ARGMAX>(a, s);
  if (a.B <= 4) return launch_bt<4, EPI, ARGMAX>(a, s);
  return launch_bt<8, EPI, ARGMAX>(a, s);
}

// x[b] = q[tokens[b]] * s[tokens[b]] (int8 embedding rows); a token outside
// [0, V) reads row 0 and sets *status.
__global__ void k_embed_i8(const int8_t* q, const float* sc, const int32_t* tokens, int B, int H,
                           int V, float* x, int* status) {
  const int b = blockIdx.y;
  int tok = tokens[b];
  if (tok < 0 || tok >= V) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && status) atomicCAS(status, 0, (int)NC_ERR_INVALID_ARGUMENT);
    tok = 0;
  }
  const float s = sc[tok];
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < H; i += gridDim.x * blockDim.x)
    x[(size_t)b * H + i] = (float)q[(size_t)tok * H + i] * s;
}

}  // namespace

size_t w8a8_b32_smem_bytes(int B, int K) {
  const int bt = B <= 1 ? 1 : B <= 2 ? 2 : B <= 4 ? 4 : 8;
  return (size_t)bt * K + (size_t)bt * (K / kActBlock) * sizeof(float);
}

cudaError_t launch_w8a8_b32(Epi epi, const W8BArgs& a, cudaStream_t s) {
  if (a.part) return launch_epi<Epi::Store, true>(a, s);
  switch (epi) {
    case Epi::Store: return launch_epi<Epi::Store, false>(a, s);
    case Epi::Residual: return launch_epi<Epi::Residual, false>(a, s);
    default: return launch_epi<Epi::SwiGLU, false>(a, s);
  }
}

cudaError_t launch_embed_i8(const int8_t* q, const float* sc, const int32_t* tokens, int B, int H,
                            int V, float* x, int* status, cudaStream_t s) {
  k_embed_i8<<<dim3((H + 255) / 256, B), 256, 0, s>>>(q, sc, tokens, B, H, V, x, status);
  return cudaGetLastError();
}

}  // namespace nc
