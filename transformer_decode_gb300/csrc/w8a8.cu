// w8a8.cu -- int8 weights and activations with int32 accumulation.
//
// nanoinfer "Quantization": symmetric per-output-row weight scales, range
// [-127, 127], round half away from zero. Activations are quantised per token
// (one scale per input vector) in each consuming CTA: amax is an
// order-independent max, so every CTA derives bit-identical int8 inputs.
// acc = sum_k Wq[n,k] xq[k] is exact in int32 (|acc| <= K * 127^2 < 2^31 for
// K <= 133,000), computed four products at a time with dp4a, so the integer
// result does not depend on the summation order. The fp epilogue is
// y = float(acc) * (w_scale[n] * sx) (+ bias).
#include <cuda_runtime.h>
#include <math.h>

#include "kernels.h"

namespace nc {

constexpr int kW8Threads = 256;
constexpr int kW8Warps = kW8Threads / kWarp;

__device__ __forceinline__ int8_t quant1(float v, float s) {
  if (s == 0.f) return 0;
  float r = roundf(__fdiv_rn(v, s));
  r = fminf(fmaxf(r, -127.f), 127.f);
  return (int8_t)(int)r;
}

__device__ __forceinline__ float silu_mul8(float g, float u) {
  const float e = expf(-fabsf(g));
  const float sig = g >= 0.f ? 1.f / (1.f + e) : e / (1.f + e);
  return (g * sig) * u;
}

template <int BT, Epi EPI>
__global__ void __launch_bounds__(kW8Threads) k_w8a8(W8Args a) {
  extern __shared__ int4 smem_i4[];
  int8_t* xq = reinterpret_cast<int8_t*>(smem_i4);  // [BT][K]
  __shared__ float rn[BT], sx[BT];
  constexpr int R = EPI == Epi::SwiGLU ? 2 : 1;
  const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
  const int K = a.K;

  // RMSNorm factor and amax of the normed row, one warp per sequence
  for (int b = warp; b < BT; b += kW8Warps) {
    float r = 1.f;
    float amax = 0.f;
    if (b < a.B) {
      const float* xb = a.x + (size_t)b * K;
      if (a.gamma) {
        float ss = 0.f;
        for (int k = lane; k < K; k += kWarp) ss = fmaf(xb[k], xb[k], ss);
        ss = warp_sum(ss);
        r = 1.f / sqrtf(ss / (float)K + a.eps);
      }
      for (int k = lane; k < K; k += kWarp) {
        const float v = a.gamma ? (xb[k] * r) * bf16_to_f32(a.gamma[k]) : xb[k];
        amax = fmaxf(amax, fabsf(v));
      }
      amax = warp_max(amax);
    }
    if (lane == 0) {
      rn[b] = r;
      sx[b] = __fdiv_rn(amax, 127.f);
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < BT * K; i += kW8Threads) {
    const int b = i / K, k = i - b * K;
    int8_t q = 0;
    if (b < a.B) {
      const float xv = a.x[(size_t)b * K + k];
      const float v = a.gamma ? (xv * rn[b]) * bf16_to_f32(a.gamma[k]) : xv;
      q = quant1(v, sx[b]);
      if (blockIdx.x == 0 && a.xq_out) a.xq_out[(size_t)b * K + k] = q;
    }
    xq[i] = q;
  }
  if (blockIdx.x == 0 && a.sx_out && threadIdx.x < a.B) a.sx_out[threadIdx.x] = sx[threadIdx.x];
  __syncthreads();

  const int nchunk = K / 16;
  const int groups = (a.N + kW8Warps - 1) / kW8Warps;
  for (int grp = blockIdx.x; grp < groups; grp += gridDim.x) {
    const int n = grp * kW8Warps + warp;
    if (n >= a.N) continue;  // warp-uniform; no block barrier below
    int acc[R][BT];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int b = 0; b < BT; ++b) acc[r][b] = 0;
    const int8_t* rows[R];
    rows[0] = a.Wq + (size_t)n * K;
    if constexpr (R == 2) rows[1] = a.Wq + ((size_t)a.N + n) * K;
    for (int c = lane; c < nchunk; c += kWarp) {
      uint4 w[R];
#pragma unroll
      for (int r = 0; r < R; ++r) w[r] = ld_stream(rows[r] + (size_t)c * 16);
#pragma unroll
      for (int b = 0; b < BT; ++b) {
        const int4 xv = *reinterpret_cast<const int4*>(xq + (size_t)b * K + c * 16);
#pragma unroll
        for (int r = 0; r < R; ++r) {
          acc[r][b] = __dp4a((int)w[r].x, xv.x, acc[r][b]);
          acc[r][b] = __dp4a((int)w[r].y, xv.y, acc[r][b]);
          acc[r][b] = __dp4a((int)w[r].z, xv.z, acc[r][b]);
          acc[r][b] = __dp4a((int)w[r].w, xv.w, acc[r][b]);
        }
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int b = 0; b < BT; ++b) acc[r][b] = warp_sum_i(acc[r][b]);
    if (lane < BT && lane < a.B) {
      int v[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        v[r] = acc[r][0];
#pragma unroll
        for (int b = 1; b < BT; ++b)
          if (lane == b) v[r] = acc[r][b];
      }
      const float s = sx[lane];
      if (a.acc_out) {
        a.acc_out[(size_t)lane * R * a.N + n] = v[0];
        if constexpr (R == 2) a.acc_out[(size_t)lane * R * a.N + a.N + n] = v[1];
      }
      float* yp = a.y + (size_t)lane * a.N + n;
      const float y0 = (float)v[0] * (a.w_scale[n] * s);
      if constexpr (EPI == Epi::Store) {
        *yp = a.bias ? y0 + bf16_to_f32(a.bias[n]) : y0;
      } else if constexpr (EPI == Epi::Residual) {
        *yp = *yp + y0;
      } else {
        const float y1 = (float)v[R - 1] * (a.w_scale[a.N + n] * s);
        *yp = silu_mul8(y0, y1);
      }
    }
  }
}

template <int BT, Epi EPI>
static cudaError_t w8_bt(const W8Args& a, cudaStream_t s) {
  const size_t smem = (size_t)BT * a.K;
  cudaError_t e = ensure_smem<k_w8a8<BT, EPI>>();
  if (e != cudaSuccess) return e;
  const int groups = (a.N + kW8Warps - 1) / kW8Warps;
  const int grid = groups < num_sms() * 8 ? groups : num_sms() * 8;
  k_w8a8<BT, EPI><<<grid, kW8Threads, smem, s>>>(a);
  return cudaGetLastError();
}

template <Epi EPI>
static cudaError_t w8_epi(const W8Args& a, cudaStream_t s) {
  if (a.B <= 1) return w8_bt<1, EPI>(a, s);
  if (a.B <= 2) return w8_bt<2, EPI>(a, s);
  if (a.B <= 4) return w8_bt<4, EPI>(a, s);
  if (a.B <= 8) return w8_bt<8, EPI>(a, s);
  return w8_bt<16, EPI>(a, s);
}

cudaError_t launch_w8a8(Epi epi, const W8Args& a, cudaStream_t s) {
  switch (epi) {
    case Epi::Store: return w8_epi<Epi::Store>(a, s);
    case Epi::Residual: return w8_epi<Epi::Residual>(a, s);
    default: return w8_epi<Epi::SwiGLU>(a, s);
  }
}

// One warp per row: scale = amax / 127, q = clamp(round_half_away(w / scale)).
__global__ void k_quantize_weight(const uint16_t* W, int N, int K, int8_t* q, float* scale) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) / kWarp, lane = threadIdx.x % kWarp;
  if (warp >= N) return;
  const uint16_t* row = W + (size_t)warp * K;
  float amax = 0.f;
  for (int k = lane; k < K; k += kWarp) amax = fmaxf(amax, fabsf(bf16_to_f32(row[k])));
  amax = warp_max(amax);
  const float s = __fdiv_rn(amax, 127.f);
  for (int k = lane; k < K; k += kWarp) q[(size_t)warp * K + k] = quant1(bf16_to_f32(row[k]), s);
  if (lane == 0) scale[warp] = s;
}

cudaError_t launch_quantize_weight(const uint16_t* W, int N, int K, int8_t* q, float* scale,
                                   cudaStream_t s) {
  const int warps_per_block = 8;
  k_quantize_weight<<<(N + warps_per_block - 1) / warps_per_block, warps_per_block * kWarp, 0, s>>>(
      W, N, K, q, scale);
  return cudaGetLastError();
}

}  // namespace nc
