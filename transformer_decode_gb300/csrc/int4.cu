// int4.cu -- the GEMV over group-wise INT4 weights.
//
// nanoinfer, "Quantization": INT4 weights with one scale per group of 32 or
// 128 consecutive weights of a row, fifteen symmetric levels [-7, 7] (no zero
// point), so a weight is q * scale. Two codes share a byte, the even index in
// the low nibble, each nibble two's complement. The dequantised weight is
// q * scale rounded to fp32 and multiplied by the activation, as in the
// page's quantise-dequantise evaluation; the kernel only never stores it.
//
// At batch 1 a row of K weights is K / 2 bytes plus K / group fp32 scales:
// a quarter of the bf16 bytes (plus 3% or 12.5% for the scales), so the
// kernel is bound by HBM like the bf16 GEMV. Design: the RMSNorm of the
// input rows in the prologue (each CTA computes it), the normalised
// activations in shared memory with one pad word per 32 (a lane reads the 32
// activations of its own 16-byte weight chunk; the pad puts the 32 lanes on
// 32 banks); one warp per output row, lanes striding the row in 16-byte
// chunks of 32 codes, all of a chunk in one group (group is a multiple of 32).
#include <cuda_runtime.h>

#include "kernels.h"

namespace nc {
namespace {

constexpr int kI4Threads = 256;
constexpr int kI4Warps = kI4Threads / kWarp;
constexpr int kI4Unroll = 4;  // chunks of a row in flight per lane

__device__ __forceinline__ int xs_pad(int k) { return k + (k >> 5); }

__device__ __forceinline__ float silu_mul_i4(float g, float u) {
  const float e = expf(-fabsf(g));  // nanoinfer "Phase 8" sigmoid form
  const float sig = g >= 0.f ? 1.f / (1.f + e) : e / (1.f + e);
  return (g * sig) * u;
}

// EPI: Store (+ bias), Residual (y += ...), SwiGLU (rows n and N + n are gate
// and up: y = silu(gate) * up).
template <int BT, Epi EPI>
__global__ void __launch_bounds__(kI4Threads) k_int4_gemv(const __grid_constant__ Int4Args a) {
  constexpr int R = EPI == Epi::SwiGLU ? 2 : 1;
  constexpr int U = R == 2 ? (BT >= 8 ? 1 : 2) : kI4Unroll;
  extern __shared__ float xs[];  // [BT][K + K / 32]
  __shared__ float part[kI4Warps][BT];
  __shared__ float rn[BT];
  const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
  const int K = a.K, ld = K + K / 32;

  // RMSNorm factor of each input row: r = 1 / sqrt(sum(x^2) / K + eps)
  if (a.gamma) {
#pragma unroll
    for (int b = 0; b < BT; ++b) {
      float ss = 0.f;
      if (b < a.B)
        for (int k = threadIdx.x; k < K; k += kI4Threads) {
          const float v = a.x[(size_t)b * K + k];
          ss = fmaf(v, v, ss);
        }
      ss = warp_sum(ss);
      if (lane == 0) part[warp][b] = ss;
    }
    __syncthreads();
    if (threadIdx.x < BT) {
      float t = 0.f;
      for (int w = 0; w < kI4Warps; ++w) t += part[w][threadIdx.x];
      rn[threadIdx.x] = 1.f / sqrtf(t / (float)K + a.eps);
    }
    __syncthreads();
  }
  for (int b = 0; b < BT; ++b)
    for (int k = threadIdx.x; k < K; k += kI4Threads) {
      float v = 0.f;
      if (b < a.B) {
        v = a.x[(size_t)b * K + k];
        if (a.gamma) v = (v * rn[b]) * bf16_to_f32(a.gamma[k]);
      }
      xs[b * ld + xs_pad(k)] = v;
    }
  __syncthreads();

  const int nchunk = K / 32;  // 16 bytes = 32 codes
  const int ng = K / a.group;
  for (int n = blockIdx.x * kI4Warps + warp; n < a.N; n += gridDim.x * kI4Warps) {
    const uint8_t* wr[R];
    const float* sr[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      wr[r] = a.Wq + ((size_t)r * a.N + n) * (K / 2);
      sr[r] = a.scales + ((size_t)r * a.N + n) * ng;
    }
    float acc[R][BT];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int b = 0; b < BT; ++b) acc[r][b] = 0.f;
    for (int c0 = lane; c0 < nchunk; c0 += U * kWarp) {
      uint4 w[R][U];
      float s[R][U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + u * kWarp;
#pragma unroll
        for (int r = 0; r < R; ++r) {
          if (c < nchunk) {
            w[r][u] = ld_stream(wr[r] + (size_t)c * 16);
            s[r][u] = sr[r][(c * 32) / a.group];
          } else {
            w[r][u] = make_uint4(0, 0, 0, 0);
            s[r][u] = 0.f;
          }
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + u * kWarp;
        if (c >= nchunk) break;
        const int p0 = xs_pad(c * 32);  // the chunk's 32 activations, contiguous after the pad
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const uint32_t words[4] = {w[r][u].x, w[r][u].y, w[r][u].z, w[r][u].w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              int q = (int)((words[j] >> (4 * t)) & 0xFu);
              q = q >= 8 ? q - 16 : q;
              const float wv = (float)q * s[r][u];
#pragma unroll
              for (int b = 0; b < BT; ++b)
                acc[r][b] = fmaf(wv, xs[b * ld + p0 + 8 * j + t], acc[r][b]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int b = 0; b < BT; ++b) {
      float v[R];
#pragma unroll
      for (int r = 0; r < R; ++r) v[r] = warp_sum(acc[r][b]);
      if (lane == 0 && b < a.B) {
        float* yp = a.y + (size_t)b * a.N + n;
        if constexpr (EPI == Epi::Store) {
          *yp = a.bias ? v[0] + bf16_to_f32(a.bias[n]) : v[0];
        } else if constexpr (EPI == Epi::Residual) {
          *yp = *yp + v[0];
        } else {
          *yp = silu_mul_i4(v[0], v[R - 1]);
        }
      }
    }
  }
}

// Group-wise INT4 quantisation of a bf16 [N, K] matrix, one thread per (row,
// group): s = amax / 7 (IEEE division), q = clamp(round_half_away(w / s),
// -7, 7) (a zero group: s = 0, codes 0), two codes a byte, the even index in
// the low nibble. The same operations as the oracle's quantiser, so the codes
// and scales agree bit for bit.
__global__ void k_quantize_int4(const uint16_t* W, int N, int K, int group, uint8_t* q,
                                float* sc) {
  const int ng = K / group;
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)N * ng) return;
  const int n = (int)(i / ng), g = (int)(i % ng);
  const uint16_t* w = W + (size_t)n * K + (size_t)g * group;
  float amax = 0.f;
  for (int j = 0; j < group; ++j) amax = fmaxf(amax, fabsf(bf16_to_f32(w[j])));
  const float s = __fdiv_rn(amax, 7.f);
  sc[i] = s;
  uint8_t* out = q + (size_t)n * (K / 2) + (size_t)g * (group / 2);
  for (int j = 0; j < group; j += 2) {
    int c[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float r = 0.f;
      if (s != 0.f) r = fminf(fmaxf(roundf(__fdiv_rn(bf16_to_f32(w[j + h]), s)), -7.f), 7.f);
      c[h] = (int)r;
    }
    out[j / 2] = (uint8_t)((c[0] & 0xF) | ((c[1] & 0xF) << 4));
  }
}

template <int BT, Epi EPI>
cudaError_t launch_bt(const Int4Args& a, cudaStream_t s) {
  const size_t smem = (size_t)BT * (a.K + a.K / 32) * sizeof(float);
  cudaError_t attr = ensure_smem<k_int4_gemv<BT, EPI>>();
  if (attr != cudaSuccess) return attr;
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_int4_gemv<BT, EPI>,
                                                                 kI4Threads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  const int rows_per_cta = kI4Warps;
  int grid = (a.N + rows_per_cta - 1) / rows_per_cta;
  grid = grid < per_sm * num_sms() ? grid : per_sm * num_sms();
  k_int4_gemv<BT, EPI><<<grid, kI4Threads, smem, s>>>(a);
  return cudaGetLastError();
}

template <Epi EPI>
cudaError_t launch_epi(const Int4Args& a, cudaStream_t s) {
  if (a.B <= 1) return launch_bt<1, EPI>(a, s);
  if (a.B <= 2) return launch_bt<2, EPI>(a, s);
  if (a.B <= 4) return launch_bt<4, EPI>(a, s);
  return launch_bt<8, EPI>(a, s);
}

}  // namespace

size_t int4_smem_bytes(int B, int K) {
  const int bt = B <= 1 ? 1 : B <= 2 ? 2 : B <= 4 ? 4 : 8;
  return (size_t)bt * (K + K / 32) * sizeof(float);
}

cudaError_t launch_int4_gemv(Epi epi, const Int4Args& a, cudaStream_t s) {
  switch (epi) {
    case Epi::Store: return launch_epi<Epi::Store>(a, s);
    case Epi::Residual: return launch_epi<Epi::Residual>(a, s);
    default: return launch_epi<Epi::SwiGLU>(a, s);
  }
}

cudaError_t launch_quantize_int4(const uint16_t* W, int N, int K, int group, uint8_t* q,
                                 float* sc, cudaStream_t s) {
  const long long n = (long long)N * (K / group);
  k_quantize_int4<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(W, N, K, group, q, sc);
  return cudaGetLastError();
}

}  // namespace nc
