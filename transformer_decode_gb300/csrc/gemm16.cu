// gemm16.cu -- the decode projections and the LM head at batch 9..16 on the
// tensor cores.
//
// At 16 sequences a projection does 32 flop per weight element (16 FMAs per
// bf16), about 11 flop per byte of the step: at HBM speed that is about the
// whole fp32 CUDA-core rate, so the contraction moves to the tensor cores
// (mma.sync m16n8k16, bf16 in, fp32 accumulate), still HBM-bound there.
//
//  * Weights are the A operand: a warp owns 16 output rows and streams them
//    from HBM with 16-byte loads straight into fragment registers. The k
//    positions of an MMA are a permutation of the physical ones (the same for
//    A and B, so the dot products are unchanged): lane l covers 16 consecutive
//    k of its rows per 64-k group, i.e. two 16-byte loads per row.
//  * Activations are the B operand: each CTA normalises its 16 sequences
//    (RMSNorm when the projection has a gain), splits every value into a
//    bf16 high part and the bf16 rounding of the remainder, and keeps both
//    planes in shared memory; two MMAs (hi, lo) per step give ~16 mantissa
//    bits of the fp32 input.
//  * The four warps of a CTA split its k range; their accumulators are summed
//    through shared memory and the epilogue (bias, residual add, SiLU * up,
//    logits and arg-max) runs on the summed values. A residual projection may
//    also split k across CTAs (atomic adds into the residual).
#include <cuda_runtime.h>

#include "kernels.h"

namespace nc {

namespace {

constexpr int kGThreads = 128;
constexpr int kGWarps = kGThreads / kWarp;
constexpr int kGMaxK = 2048;  // k range of one CTA (its activation planes live in shared memory)
constexpr int kGPad = 8;      // plane row padding (bf16): the B-fragment loads are conflict free

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float silu_mul16(float g, float u) {
  const float e = expf(-fabsf(g));
  const float sig = g >= 0.f ? 1.f / (1.f + e) : e / (1.f + e);
  return (g * sig) * u;
}

// rn[b] = 1 / sqrt(mean(x[b]^2) + eps) for the 16 sequences (0 past B).
__device__ void norms16(const float* x, int B, int K, float eps, float* rn) {
  const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
  for (int b = warp; b < 16; b += kGWarps) {
    float ss = 0.f;
    if (b < B) {
      const float* xb = x + (size_t)b * K;
      for (int k = lane * 4; k < K; k += kWarp * 4) {
        const float4 v = *reinterpret_cast<const float4*>(xb + k);
        ss = fmaf(v.x, v.x, ss);
        ss = fmaf(v.y, v.y, ss);
        ss = fmaf(v.z, v.z, ss);
        ss = fmaf(v.w, v.w, ss);
      }
    }
    ss = warp_sum(ss);
    if (lane == 0) rn[b] = b < B ? 1.f / sqrtf(ss / (float)K + eps) : 0.f;
  }
}

// The hi and lo bf16 planes [16][stride] of xn[b][k0 .. k0 + kr), xn = x or
// (x * rn) * gamma; rows of absent sequences are zero.
__device__ void build_planes(const float* x, const uint16_t* gamma, const float* rn, int B,
                             int K, int k0, int kr, int stride, uint16_t* hi, uint16_t* lo) {
  const int q = kr / 4;  // float4 per row
  for (int i = threadIdx.x; i < 16 * q; i += kGThreads) {
    const int b = i / q, kk = (i - b * q) * 4;
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    if (b < B) {
      const float4 f = *reinterpret_cast<const float4*>(x + (size_t)b * K + k0 + kk);
      v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
      if (gamma) {
        const uint2 g = *reinterpret_cast<const uint2*>(gamma + k0 + kk);
        v[0] = (v[0] * rn[b]) * bf16_lo(g.x);
        v[1] = (v[1] * rn[b]) * bf16_hi(g.x);
        v[2] = (v[2] * rn[b]) * bf16_lo(g.y);
        v[3] = (v[3] * rn[b]) * bf16_hi(g.y);
      }
    }
    uint16_t h[4], l[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      h[e] = f32_to_bf16(v[e]);
      l[e] = f32_to_bf16(v[e] - bf16_to_f32(h[e]));
    }
    uint2 hv, lv;
    hv.x = h[0] | (uint32_t)h[1] << 16;
    hv.y = h[2] | (uint32_t)h[3] << 16;
    lv.x = l[0] | (uint32_t)l[1] << 16;
    lv.y = l[2] | (uint32_t)l[3] << 16;
    *reinterpret_cast<uint2*>(hi + b * stride + kk) = hv;
    *reinterpret_cast<uint2*>(lo + b * stride + kk) = lv;
  }
}

__device__ __forceinline__ void words8(const uint4& a, const uint4& b, uint32_t (&w)[8]) {
  w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
  w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
}

// One warp: 16 rows (and, with PAIR, the 16 rows ldw * n_up further) over
// the 64-k groups [g0, g1) of the CTA's range. acc[m][j][.] is the C fragment
// of matrix m (gate / up) and tokens 8 j .. 8 j + 7.
template <bool PAIR>
__device__ __forceinline__ void warp_tiles(const uint16_t* W0, const uint16_t* W1, int K,
                                           int rows_valid, const uint16_t* hi, const uint16_t* lo,
                                           int stride, int g0, int g1, float (&acc)[2][2][4]) {
  const int lane = threadIdx.x % kWarp, t4 = lane % 4, r = lane / 4;
  // rows past the matrix re-read its last row (results unused)
  const int ra = min(r, rows_valid - 1), rb = min(r + 8, rows_valid - 1);
  const uint16_t* A0 = W0 + (size_t)ra * K;
  const uint16_t* A1 = W0 + (size_t)rb * K;
  const uint16_t* U0 = PAIR ? W1 + (size_t)ra * K : nullptr;
  const uint16_t* U1 = PAIR ? W1 + (size_t)rb * K : nullptr;
  // the next group's weights are loaded while this one multiplies
  uint4 cur[2][4], nxt[2][4];
  const auto load = [&](int c, uint4 (&w)[2][4]) {
    const int kb = c * 64 + 16 * t4;  // the lane's 16 k of group c
    w[0][0] = ld_stream(A0 + kb);
    w[0][1] = ld_stream(A0 + kb + 8);
    w[0][2] = ld_stream(A1 + kb);
    w[0][3] = ld_stream(A1 + kb + 8);
    if (PAIR) {
      w[1][0] = ld_stream(U0 + kb);
      w[1][1] = ld_stream(U0 + kb + 8);
      w[1][2] = ld_stream(U1 + kb);
      w[1][3] = ld_stream(U1 + kb + 8);
    }
  };
  if (g0 < g1) load(g0, cur);
  for (int c = g0; c < g1; ++c) {
    const int kb = c * 64 + 16 * t4;  // the lane's 16 k of this group
    if (c + 1 < g1) load(c + 1, nxt);
    uint32_t wa[8], wb[8], ua[8], ub[8];
    words8(cur[0][0], cur[0][1], wa);
    words8(cur[0][2], cur[0][3], wb);
    if (PAIR) {
      words8(cur[1][0], cur[1][1], ua);
      words8(cur[1][2], cur[1][3], ub);
    }
    uint32_t bh[2][8], bl[2][8];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int row = (r + 8 * j) * stride + kb;
      words8(*reinterpret_cast<const uint4*>(hi + row), *reinterpret_cast<const uint4*>(hi + row + 8),
             bh[j]);
      words8(*reinterpret_cast<const uint4*>(lo + row), *reinterpret_cast<const uint4*>(lo + row + 8),
             bl[j]);
    }
#pragma unroll
    for (int s = 0; s < 4; ++s) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        mma16816(acc[0][j], wa[2 * s], wb[2 * s], wa[2 * s + 1], wb[2 * s + 1], bh[j][2 * s],
                 bh[j][2 * s + 1]);
        mma16816(acc[0][j], wa[2 * s], wb[2 * s], wa[2 * s + 1], wb[2 * s + 1], bl[j][2 * s],
                 bl[j][2 * s + 1]);
        if (PAIR) {
          mma16816(acc[1][j], ua[2 * s], ub[2 * s], ua[2 * s + 1], ub[2 * s + 1], bh[j][2 * s],
                   bh[j][2 * s + 1]);
          mma16816(acc[1][j], ua[2 * s], ub[2 * s], ua[2 * s + 1], ub[2 * s + 1], bl[j][2 * s],
                   bl[j][2 * s + 1]);
        }
      }
    }
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int q = 0; q < 4; ++q) cur[m][q] = nxt[m][q];
  }
}

// The four warps' C fragments summed: red[m][row][token] (padded).
struct Red {
  float v[2][16][17];
};

__device__ __forceinline__ void reduce_warps(const float (&acc)[2][2][4], bool pair, Red* red) {
  const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp, t4 = lane % 4, r = lane / 4;
  for (int w = 0; w < kGWarps; ++w) {
    if (warp == w) {
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        if (m == 1 && !pair) break;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int n = 8 * j + 2 * t4;
          float* p0 = &red->v[m][r][n];
          float* p1 = &red->v[m][r + 8][n];
          if (w == 0) {
            p0[0] = acc[m][j][0]; p0[1] = acc[m][j][1];
            p1[0] = acc[m][j][2]; p1[1] = acc[m][j][3];
          } else {
            p0[0] += acc[m][j][0]; p0[1] += acc[m][j][1];
            p1[0] += acc[m][j][2]; p1[1] += acc[m][j][3];
          }
        }
      }
    }
    __syncthreads();
  }
}

template <Epi EPI>
__global__ void __launch_bounds__(kGThreads) k_gemm16(GemvArgs a, int KR) {
  extern __shared__ __align__(16) uint16_t gsm[];
  __shared__ float rn[16];
  __shared__ Red red;
  constexpr bool PAIR = EPI == Epi::SwiGLU;
  const int K = a.K, N = a.N;
  const int r0 = blockIdx.x * 16;
  const int k0 = blockIdx.y * KR, kr = min(KR, K - k0);
  const int stride = KR + kGPad;
  uint16_t* hi = gsm;
  uint16_t* lo = gsm + 16 * stride;

  // warm L2 with this tile's weights (no earlier kernel writes them), then
  // wait for the activations
  if (threadIdx.x < 16 && r0 + (int)threadIdx.x < N) {
    prefetch_l2(a.W + (size_t)(r0 + threadIdx.x) * K + k0, (uint32_t)kr * 2);
    if (PAIR) prefetch_l2(a.W + ((size_t)N + r0 + threadIdx.x) * K + k0, (uint32_t)kr * 2);
  }
  pdl_wait();
  if (a.gamma) norms16(a.x, a.B, K, a.eps, rn);
  __syncthreads();
  build_planes(a.x, a.gamma, rn, a.B, K, k0, kr, stride, hi, lo);
  __syncthreads();

  const int warp = threadIdx.x / kWarp;
  const int groups = kr / 64;
  const int g0 = (warp * groups) / kGWarps, g1 = ((warp + 1) * groups) / kGWarps;
  float acc[2][2][4] = {};
  const uint16_t* W0 = a.W + (size_t)r0 * K + k0;
  const uint16_t* W1 = PAIR ? a.W + ((size_t)N + r0) * K + k0 : nullptr;
  warp_tiles<PAIR>(W0, W1, K, min(16, N - r0), hi, lo, stride, g0, g1, acc);
  reduce_warps(acc, PAIR, &red);

  for (int i = threadIdx.x; i < 256; i += kGThreads) {
    const int row = i / 16, b = i % 16, n = r0 + row;
    if (b >= a.B || n >= N) continue;
    const float v = red.v[0][row][b];
    float* yp = a.y + (size_t)b * N + n;
    if constexpr (EPI == Epi::Store) {
      *yp = a.bias ? v + bf16_to_f32(a.bias[n]) : v;
    } else if constexpr (EPI == Epi::Residual) {
      if (gridDim.y == 1) *yp = *yp + v;
      else atomicAdd(yp, v);  // k split across CTAs: each adds its share
    } else {
      *yp = silu_mul16(v, red.v[1][row][b]);
    }
  }
}

// LM head: logits and per-sequence arg-max keys, tiles of 16 vocabulary rows
// over a grid-stride loop; the last CTA combines the per-CTA keys.
__global__ void __launch_bounds__(kGThreads) k_lm_head16(LmHeadArgs a) {
  extern __shared__ __align__(16) uint16_t gsm[];
  __shared__ float rn[16];
  __shared__ Red red;
  __shared__ unsigned long long best_s[kGThreads];
  __shared__ bool last_s;
  const int K = a.K, V = a.V;
  const int stride = K + kGPad;
  uint16_t* hi = gsm;
  uint16_t* lo = gsm + 16 * stride;
  if (threadIdx.x < 16 && blockIdx.x * 16 + (int)threadIdx.x < V)
    prefetch_l2(a.W + (size_t)(blockIdx.x * 16 + threadIdx.x) * K, (uint32_t)K * 2);
  pdl_wait();
  norms16(a.x, a.B, K, a.eps, rn);
  __syncthreads();
  build_planes(a.x, a.gamma, rn, a.B, K, 0, K, stride, hi, lo);
  __syncthreads();

  const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
  const int groups = K / 64;
  const int g0 = (warp * groups) / kGWarps, g1 = ((warp + 1) * groups) / kGWarps;
  const int tiles = (V + 15) / 16;
  unsigned long long best = 0ull;  // this thread's token is threadIdx.x % 16
  for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
    const int r0 = t * 16;
    float acc[2][2][4] = {};
    warp_tiles<false>(a.W + (size_t)r0 * K, nullptr, K, min(16, V - r0), hi, lo, stride, g0, g1,
                      acc);
    reduce_warps(acc, false, &red);
    for (int i = threadIdx.x; i < 256; i += kGThreads) {
      const int row = i / 16, b = i % 16, n = r0 + row;
      if (b < a.B && n < V) {
        const float v = red.v[0][row][b];
        a.logits[(size_t)b * V + n] = v;
        const unsigned long long key = argmax_key(v, (uint32_t)n);
        best = key > best ? key : best;
      }
    }
    __syncthreads();  // red is rewritten by the next tile
  }
  (void)lane;
  best_s[threadIdx.x] = best;
  __syncthreads();
  if (threadIdx.x < 16 && threadIdx.x < a.B) {
    unsigned long long m = 0ull;
    for (int i = threadIdx.x; i < kGThreads; i += 16) m = best_s[i] > m ? best_s[i] : m;
    a.part[(size_t)threadIdx.x * gridDim.x + blockIdx.x] = m;
  }
  // the last CTA combines the per-CTA keys (max over integer keys: order-free)
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last_s = atomicAdd(a.ticket, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!last_s) return;
  __threadfence();
  for (int b = warp; b < a.B; b += kGWarps) {
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

size_t planes_bytes(int kr) { return sizeof(uint16_t) * 2 * 16 * (size_t)(kr + kGPad); }

}  // namespace

bool gemm16_supported(Epi epi, int B, int K) {
  if (B <= 8 || B > 16 || K % 64) return false;
  return epi == Epi::Residual || K <= kGMaxK;
}

bool lm_head16_supported(int B, int K) { return B > 8 && B <= 16 && K % 64 == 0 && K <= kGMaxK; }

template <Epi EPI>
static cudaError_t gemm16_epi(const GemvArgs& a, cudaStream_t s) {
  const int tiles = (a.N + 15) / 16;
  int ks = 1;
  if (EPI == Epi::Residual) {
    // enough CTAs to keep every SM streaming, k ranges of at least 256
    ks = (2 * num_sms() + tiles - 1) / tiles;
    if (ks > a.K / 256) ks = a.K / 256;
    const int need = (a.K + kGMaxK - 1) / kGMaxK;
    if (ks < need) ks = need;
    if (ks < 1) ks = 1;
  }
  const int groups = a.K / 64;
  const int KR = ((groups + ks - 1) / ks) * 64;
  ks = (a.K + KR - 1) / KR;
  auto kern = k_gemm16<EPI>;
  cudaError_t e = ensure_smem<k_gemm16<EPI>>();
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(tiles, ks), dim3(kGThreads), planes_bytes(KR), s, a, KR);
}

cudaError_t launch_gemm16(Epi epi, const GemvArgs& a, cudaStream_t s) {
  switch (epi) {
    case Epi::Store: return gemm16_epi<Epi::Store>(a, s);
    case Epi::Residual: return gemm16_epi<Epi::Residual>(a, s);
    default: return gemm16_epi<Epi::SwiGLU>(a, s);
  }
}

cudaError_t launch_lm_head16(const LmHeadArgs& a, cudaStream_t s) {
  cudaError_t e = ensure_smem<k_lm_head16>();
  if (e != cudaSuccess) return e;
  return launch_pdl(k_lm_head16, dim3(lm_head_grid()), dim3(kGThreads), planes_bytes(a.K), s, a);
}

}  // namespace nc
