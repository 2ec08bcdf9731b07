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

// Block i owns the rows [N i / grid, N (i + 1) / grid) (one wave).
template <int BT>
__global__ void __launch_bounds__(kB32Threads) k_w8a8_b32(const __grid_constant__ W8BArgs a) {
  extern __shared__ int4 smem_i4[];
  const int K = a.K, nblk = K / kActBlock;
  int8_t* xq = reinterpret_cast<int8_t*>(smem_i4);                   // [BT][K]
  float* sx = reinterpret_cast<float*>(xq + (size_t)BT * K);          // [BT][nblk]
  __shared__ float rn[BT];
  __shared__ float part[kB32Warps][BT];
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
  for (int n = r0 + warp; n < r1; n += kB32Warps) {  // no block barrier below
    float yf[BT];
#pragma unroll
    for (int b = 0; b < BT; ++b) yf[b] = 0.f;
    const int8_t* row = a.Wq + (size_t)n * K;
    const float sw = a.w_scale[n];
    for (int c0 = lane; c0 < nchunk; c0 += U * kWarp) {
      uint4 w[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + u * kWarp;
        w[u] = c < nchunk ? ld_stream(row + (size_t)c * 16) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + u * kWarp;  // the pair (2j, 2j + 1) is in range together
        const int blk = c >> 1;
#pragma unroll
        for (int b = 0; b < BT; ++b) {
          int acc = 0;
          if (c < nchunk) {
            const int4 xv = *reinterpret_cast<const int4*>(xq + (size_t)b * K + (size_t)c * 16);
            acc = __dp4a((int)w[u].x, xv.x, acc);
            acc = __dp4a((int)w[u].y, xv.y, acc);
            acc = __dp4a((int)w[u].z, xv.z, acc);
            acc = __dp4a((int)w[u].w, xv.w, acc);
          }
          acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 1);  // the block's exact int32 sum
          if ((lane & 1) == 0 && c < nchunk && b < a.B) {
            yf[b] = fmaf((float)acc, sw * sx[b * nblk + blk], yf[b]);
            if (a.acc_out) a.acc_out[((size_t)b * a.N + n) * nblk + blk] = acc;
          }
        }
      }
    }
#pragma unroll
    for (int b = 0; b < BT; ++b) yf[b] = warp_sum(yf[b]);
    if (lane < BT && lane < a.B) {
      float v = yf[0];
#pragma unroll
      for (int b = 1; b < BT; ++b)
        if (lane == b) v = yf[b];
      a.y[(size_t)lane * a.N + n] = a.bias ? v + bf16_to_f32(a.bias[n]) : v;
    }
  }
}

template <int BT>
cudaError_t launch_bt(const W8BArgs& a, cudaStream_t s) {
  const size_t smem = w8a8_b32_smem_bytes(BT, a.K);
  cudaError_t e = ensure_smem<k_w8a8_b32<BT>>();
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_w8a8_b32<BT>, kB32Threads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  int grid = per_sm * num_sms();
  const int rows_cta = (a.N + kB32Warps - 1) / kB32Warps;
  grid = grid < rows_cta ? grid : rows_cta;
  k_w8a8_b32<BT><<<grid, kB32Threads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

size_t w8a8_b32_smem_bytes(int B, int K) {
  const int bt = B <= 1 ? 1 : B <= 2 ? 2 : B <= 4 ? 4 : 8;
  return (size_t)bt * K + (size_t)bt * (K / kActBlock) * sizeof(float);
}

cudaError_t launch_w8a8_b32(const W8BArgs& a, cudaStream_t s) {
  if (a.B <= 1) return launch_bt<1>(a, s);
  if (a.B <= 2) return launch_bt<2>(a, s);
  if (a.B <= 4) return launch_bt<4>(a, s);
  return launch_bt<8>(a, s);
}

}  // namespace nc
