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

// Block i owns the rows [N i / grid, N (i + 1) / grid) (an even split; one wave).
template <int BT, Epi EPI>
__global__ void __launch_bounds__(kW8Threads) k_w8a8(W8Args a) {
  extern __shared__ int4 smem_i4[];
  int8_t* xq = reinterpret_cast<int8_t*>(smem_i4);  // [BT][K]
  __shared__ float rn[BT], sx[BT];
  __shared__ float part[kW8Warps][BT];
  constexpr int R = EPI == Epi::SwiGLU ? 2 : 1;
  constexpr int U = 4;  // 16-byte chunks per row in flight
  const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
  const int K = a.K;
  const int r0 = (int)((long long)a.N * blockIdx.x / gridDim.x);
  const int r1 = (int)((long long)a.N * (blockIdx.x + 1) / gridDim.x);

  // the int8 weights depend on no earlier kernel: warm L2 with this warp's
  // first row(s) while the previous kernel drains
  if (lane == 0 && r0 + warp < r1) {
    const uint32_t nb = (uint32_t)min(K, 32768);
    prefetch_l2(a.Wq + (size_t)(r0 + warp) * K, nb);
    if constexpr (R == 2) prefetch_l2(a.Wq + ((size_t)a.N + r0 + warp) * K, nb);
  }
  pdl_wait();

  // RMSNorm factor per sequence: every warp sums a slice, the partials are
  // added in a fixed order
  if (a.gamma) {
#pragma unroll 1
    for (int b = 0; b < BT; ++b) {
      float ss = 0.f;
      if (b < a.B) {
        const float* xb = a.x + (size_t)b * K;
        for (int k = threadIdx.x; k < K; k += kW8Threads) ss = fmaf(xb[k], xb[k], ss);
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
      for (int w = 0; w < kW8Warps; ++w) ss += part[w][threadIdx.x];
      r = 1.f / sqrtf(ss / (float)K + a.eps);
    }
    rn[threadIdx.x] = r;
  }
  __syncthreads();
  // amax of each normed row (a max: the order of the partials does not matter)
#pragma unroll 1
  for (int b = 0; b < BT; ++b) {
    float amax = 0.f;
    if (b < a.B) {
      const float* xb = a.x + (size_t)b * K;
      const float r = rn[b];
      for (int k = threadIdx.x; k < K; k += kW8Threads) {
        const float v = a.gamma ? (xb[k] * r) * bf16_to_f32(a.gamma[k]) : xb[k];
        amax = fmaxf(amax, fabsf(v));
      }
    }
    amax = warp_max(amax);
    __syncwarp();
    if (lane == 0) part[warp][b] = amax;
  }
  __syncthreads();
  if (threadIdx.x < BT) {
    float amax = 0.f;
    for (int w = 0; w < kW8Warps; ++w) amax = fmaxf(amax, part[w][threadIdx.x]);
    sx[threadIdx.x] = __fdiv_rn(amax, 127.f);
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
  for (int n = r0 + warp; n < r1; n += kW8Warps) {  // no block barrier below
    int acc[R][BT];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int b = 0; b < BT; ++b) acc[r][b] = 0;
    const int8_t* rows[R];
    rows[0] = a.Wq + (size_t)n * K;
    if constexpr (R == 2) rows[1] = a.Wq + ((size_t)a.N + n) * K;
    for (int c = lane; c < nchunk; c += U * kWarp) {
      uint4 w[R][U];
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int r = 0; r < R; ++r)
          w[r][u] = c + u * kWarp < nchunk ? ld_stream(rows[r] + (size_t)(c + u * kWarp) * 16)
                                           : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (c + u * kWarp >= nchunk) break;
#pragma unroll
        for (int b = 0; b < BT; ++b) {
          const int4 xv = *reinterpret_cast<const int4*>(xq + (size_t)b * K + (c + u * kWarp) * 16);
#pragma unroll
          for (int r = 0; r < R; ++r) {
            acc[r][b] = __dp4a((int)w[r][u].x, xv.x, acc[r][b]);
            acc[r][b] = __dp4a((int)w[r][u].y, xv.y, acc[r][b]);
            acc[r][b] = __dp4a((int)w[r][u].z, xv.z, acc[r][b]);
            acc[r][b] = __dp4a((int)w[r][u].w, xv.w, acc[r][b]);
          }
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
      // each product and the bias add rounded on its own (no contraction), so
      // the dequantised value is the IEEE result of float(acc) * (s_w * s_x) + b
      const float y0 = __fmul_rn(__int2float_rn(v[0]), __fmul_rn(a.w_scale[n], s));
      if constexpr (EPI == Epi::Store) {
        *yp = a.bias ? __fadd_rn(y0, bf16_to_f32(a.bias[n])) : y0;
      } else if constexpr (EPI == Epi::Residual) {
        *yp = __fadd_rn(*yp, y0);
      } else {
        const float y1 = __fmul_rn(__int2float_rn(v[R - 1]), __fmul_rn(a.w_scale[a.N + n], s));
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
  // one wave: the resident blocks per SM at this shared-memory size, times the SMs
  static size_t occ_smem = ~(size_t)0;
  static int occ = 1;
  if (occ_smem != smem) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_w8a8<BT, EPI>, kW8Threads, smem) !=
            cudaSuccess ||
        n < 1)
      n = 1;
    occ = n;
    occ_smem = smem;
  }
  const int groups = (a.N + kW8Warps - 1) / kW8Warps;
  const int grid = groups < num_sms() * occ ? groups : num_sms() * occ;
  return launch_pdl(k_w8a8<BT, EPI>, dim3(grid), dim3(kW8Threads), smem, s, a);
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
