// gemv.cu -- streaming matrix-vector products for the decode step.
//
// Decode at small batch is a GEMV per projection: every weight byte is read
// once per step and used B times, so these kernels are bound by HBM
// bandwidth (nanoinfer, "Phase 4": decode is bandwidth-bound). Design:
//   * prologue: each CTA computes the RMSNorm of its input rows itself
//     (nanocompile: the five passes of rms_norm become one, fused into the
//     GEMV) and keeps the normalised activations in shared memory;
//   * body: one warp per output row (two rows, gate and up, for SwiGLU --
//     Tang section 2.3, sibling reductions merged); lanes stride the row in
//     16-byte chunks with four chunks per row in flight, read with
//     L1::no_allocate streaming loads;
//   * epilogue on the reducing warp (Tang section 2.3, "epilogues run on the
//     reducing thread"): bias, residual add, or silu(gate) * up;
//   * LM head: the same body plus the arg-max monoid on (value, index) per
//     block, combined by the last block to finish (Tang section 2.2).
#include <cuda_runtime.h>

#include <cstdlib>

#include "kernels.h"

namespace nc {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / kWarp;
constexpr int kXsFloats = 16384;  // activations kept in shared memory per K tile (64 KB)
constexpr int kRowPrefetchBytes = 32768;  // L2 warm-up per weight row before the wait

__device__ __forceinline__ float silu_mul(float g, float u) {
  // nanoinfer "Phase 8": both sigmoid halves share e = exp(-|g|).
  const float e = expf(-fabsf(g));
  const float sig = g >= 0.f ? 1.f / (1.f + e) : e / (1.f + e);
  return (g * sig) * u;
}

// Per-row RMSNorm factors r[b] = 1 / sqrt(sum(x^2) / K + eps) into rn[] (shared):
// every warp sums a slice of each row, the partials are added in a fixed order.
template <int BT>
__device__ __forceinline__ void row_norms(const float* x, int B, int K, float eps,
                                          float (*part)[BT], float* rn) {
  const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
  const int nv = K / 4;
#pragma unroll 1
  for (int b = 0; b < BT; ++b) {
    float ss = 0.f;
    if (b < B) {
      const float4* xb = reinterpret_cast<const float4*>(x + (size_t)b * K);
#pragma unroll 4
      for (int i = threadIdx.x; i < nv; i += kThreads) {
        const float4 v = xb[i];
        ss = fmaf(v.x, v.x, ss);
        ss = fmaf(v.y, v.y, ss);
        ss = fmaf(v.z, v.z, ss);
        ss = fmaf(v.w, v.w, ss);
      }
    }
    ss = warp_sum(ss);
    if (lane == 0) part[warp][b] = ss;
  }
  __syncthreads();
  if (threadIdx.x < BT) {
    float ss = 0.f;
    for (int w = 0; w < kWarps; ++w) ss += part[w][threadIdx.x];
    rn[threadIdx.x] = 1.f / sqrtf(ss / (float)K + eps);
  }
}

// xs[b][kk] = x[b][k0 + kk] * r[b] * gamma[k0 + kk] for kk < kt (zero for b >= B),
// four elements per thread and step (kt a multiple of 4).
template <int BT>
__device__ __forceinline__ void fill_xs(const float* x, const uint16_t* gamma, const float* rn,
                                        int B, int K, int k0, int kt, float* xs) {
  const int kt4 = kt / 4;
  const bool g8 = (reinterpret_cast<uintptr_t>(gamma) & 7) == 0;
#pragma unroll 4
  for (int i = threadIdx.x; i < BT * kt4; i += kThreads) {
    const int b = i / kt4, kk = (i - b * kt4) * 4;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (b < B) {
      v = *reinterpret_cast<const float4*>(x + (size_t)b * K + k0 + kk);
      if (gamma) {
        const uint16_t* gp = gamma + k0 + kk;
        float g0, g1, g2, g3;
        if (g8) {
          const uint2 gw = *reinterpret_cast<const uint2*>(gp);
          g0 = bf16_lo(gw.x); g1 = bf16_hi(gw.x); g2 = bf16_lo(gw.y); g3 = bf16_hi(gw.y);
        } else {
          g0 = bf16_to_f32(gp[0]); g1 = bf16_to_f32(gp[1]);
          g2 = bf16_to_f32(gp[2]); g3 = bf16_to_f32(gp[3]);
        }
        const float r = rn[b];
        v.x = (v.x * r) * g0;
        v.y = (v.y * r) * g1;
        v.z = (v.z * r) * g2;
        v.w = (v.w * r) * g3;
      }
    }
    *reinterpret_cast<float4*>(xs + (size_t)b * kt + kk) = v;
  }
}

// acc[r][b] += W_r[tile] . xs[b][tile] for the R rows of one warp; lanes take
// 16-byte chunks lane, lane+32, ...; U chunks per row (eight at batch 1) are
// loaded before use, the ones past the row's end predicated off.
template <int BT, int R>
__device__ __forceinline__ void warp_dot(const uint16_t* const (&row)[R], int nchunk,
                                         const float* xs, int kt, float (&acc)[R][BT]) {
  const int lane = threadIdx.x % kWarp;
  constexpr int U = BT == 1 ? 8 : 4;  // chunks per row in flight
  for (int c = lane; c < nchunk; c += U * kWarp) {
    uint4 w[R][U];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int r = 0; r < R; ++r)
        w[r][u] = c + u * kWarp < nchunk ? ld_stream(row[r] + (size_t)(c + u * kWarp) * 8)
                                         : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (c + u * kWarp < nchunk)
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int b = 0; b < BT; ++b)
            acc[r][b] += dot8(w[r][u], xs + b * kt + (c + u * kWarp) * 8);
  }
}

__host__ __device__ constexpr int tile_k(int K, int BT) {
  return K <= kXsFloats / BT ? K : (kXsFloats / BT) / 256 * 256;
}

// Block i owns the rows [N i / grid, N (i + 1) / grid): an even split, so every
// SM streams the same bytes; the grid is one wave of resident blocks.
template <int BT, Epi EPI>
__global__ void __launch_bounds__(kThreads) k_gemv(GemvArgs a) {
  extern __shared__ float4 smem4[];
  float* xs = reinterpret_cast<float*>(smem4);
  __shared__ float part[kWarps][BT];
  __shared__ float rn[BT];
  constexpr int R = EPI == Epi::SwiGLU ? 2 : 1;
  const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
  const int K = a.K, kt = tile_k(K, BT);
  const bool one_tile = kt >= K;
  const int r0 = (int)((long long)a.N * blockIdx.x / gridDim.x);
  const int r1 = (int)((long long)a.N * (blockIdx.x + 1) / gridDim.x);

  // the weights depend on no earlier kernel: pull this warp's first row(s)
  // into L2 while the previous kernel drains
  if (lane == 0 && r0 + warp < r1) {
    const uint32_t nb = (uint32_t)min((size_t)K * 2, (size_t)kRowPrefetchBytes);
    prefetch_l2(a.W + (size_t)(r0 + warp) * K, nb);
    if constexpr (R == 2) prefetch_l2(a.W + ((size_t)a.N + r0 + warp) * K, nb);
  }
  pdl_wait();

  if (a.gamma) row_norms<BT>(a.x, a.B, K, a.eps, part, rn);
  __syncthreads();
  if (one_tile) {
    fill_xs<BT>(a.x, a.gamma, rn, a.B, K, 0, K, xs);
    __syncthreads();
  }
  const int iters = (r1 - r0 + kWarps - 1) / kWarps;  // the same for every warp (barriers below)
  for (int it = 0; it < iters; ++it) {
    const int n = r0 + it * kWarps + warp;
    const bool live = n < r1;
    float acc[R][BT];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int b = 0; b < BT; ++b) acc[r][b] = 0.f;
    for (int k0 = 0; k0 < K; k0 += kt) {
      const int cur = min(kt, K - k0);
      if (!one_tile) {
        __syncthreads();
        fill_xs<BT>(a.x, a.gamma, rn, a.B, K, k0, cur, xs);
        __syncthreads();
      }
      if (live) {
        const uint16_t* rows[R];
        rows[0] = a.W + (size_t)n * K + k0;
        if constexpr (R == 2) rows[1] = a.W + ((size_t)a.N + n) * K + k0;
        warp_dot<BT, R>(rows, cur / 8, xs, cur, acc);
      }
    }
    if (!live) continue;  // warp-uniform
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int b = 0; b < BT; ++b) acc[r][b] = warp_sum(acc[r][b]);
    if (lane < BT && lane < a.B) {
      float v[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        v[r] = acc[r][0];
#pragma unroll
        for (int b = 1; b < BT; ++b)
          if (lane == b) v[r] = acc[r][b];
      }
      float* yp = a.y + (size_t)lane * a.N + n;
      if constexpr (EPI == Epi::Store) {
        *yp = a.bias ? v[0] + bf16_to_f32(a.bias[n]) : v[0];
      } else if constexpr (EPI == Epi::Residual) {
        *yp = *yp + v[0];
      } else {
        *yp = silu_mul(v[0], v[R - 1]);
      }
    }
  }
}

bool pdl_enabled() {
  static const bool on = [] {
    const char* e = getenv("NC_PDL");
    return !(e && e[0] == '0');
  }();
  return on;
}

int max_smem_optin() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
        n <= 0)
      n = 48 * 1024;
  }
  return n;
}

int num_sms() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = kNumSMs;
  }
  return n;
}

template <int BT, Epi EPI>
static cudaError_t gemv_bt(const GemvArgs& a, cudaStream_t s) {
  const int kt = tile_k(a.K, BT);
  const size_t smem = sizeof(float) * (size_t)BT * (kt < a.K ? kt : a.K);
  auto kern = k_gemv<BT, EPI>;
  cudaError_t e = ensure_smem<k_gemv<BT, EPI>>();
  if (e != cudaSuccess) return e;
  // one wave: the resident blocks per SM at this shared-memory size, times the SMs
  static size_t occ_smem = ~(size_t)0;
  static int occ = 1;
  if (occ_smem != smem) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kThreads, smem) != cudaSuccess || n < 1)
      n = 1;
    occ = n;
    occ_smem = smem;
  }
  const int groups = (a.N + kWarps - 1) / kWarps;
  const int grid = groups < num_sms() * occ ? groups : num_sms() * occ;
  return launch_pdl(kern, dim3(grid), dim3(kThreads), smem, s, a);
}

template <Epi EPI>
static cudaError_t gemv_epi(const GemvArgs& a, cudaStream_t s) {
  if (a.B <= 1) return gemv_bt<1, EPI>(a, s);
  if (a.B <= 2) return gemv_bt<2, EPI>(a, s);
  if (a.B <= 4) return gemv_bt<4, EPI>(a, s);
  if (a.B <= 8) return gemv_bt<8, EPI>(a, s);
  return gemv_bt<16, EPI>(a, s);
}

cudaError_t launch_gemv(Epi epi, const GemvArgs& a, cudaStream_t s) {
  if (gemm16_supported(epi, a.B, a.K)) return launch_gemm16(epi, a, s);
  switch (epi) {
    case Epi::Store: return gemv_epi<Epi::Store>(a, s);
    case Epi::Residual: return gemv_epi<Epi::Residual>(a, s);
    default: return gemv_epi<Epi::SwiGLU>(a, s);
  }
}

// ------------------------------------------------------------------ LM head
template <int BT>
__global__ void __launch_bounds__(kThreads) k_lm_head(LmHeadArgs a) {
  extern __shared__ float4 smem4[];
  float* xs = reinterpret_cast<float*>(smem4);
  __shared__ float rn[BT];
  __shared__ unsigned long long best_s[kWarps][BT];
  __shared__ bool last_s;
  __shared__ float part[kWarps][BT];
  const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
  const int K = a.K;
  {
    const int n = blockIdx.x * kWarps + warp;
    if (lane == 0 && n < a.V)
      prefetch_l2(a.W + (size_t)n * K, (uint32_t)min((size_t)K * 2, (size_t)kRowPrefetchBytes));
  }
  pdl_wait();
  row_norms<BT>(a.x, a.B, K, a.eps, part, rn);
  __syncthreads();
  fill_xs<BT>(a.x, a.gamma, rn, a.B, K, 0, K, xs);
  __syncthreads();

  unsigned long long best[BT];
#pragma unroll
  for (int b = 0; b < BT; ++b) best[b] = 0ull;
  const int groups = (a.V + kWarps - 1) / kWarps;
  for (int grp = blockIdx.x; grp < groups; grp += gridDim.x) {
    const int n = grp * kWarps + warp;
    if (n >= a.V) continue;  // warp-uniform
    float acc[1][BT];
#pragma unroll
    for (int b = 0; b < BT; ++b) acc[0][b] = 0.f;
    const uint16_t* rows[1] = {a.W + (size_t)n * K};
    warp_dot<BT, 1>(rows, K / 8, xs, K, acc);
#pragma unroll
    for (int b = 0; b < BT; ++b) {
      const float v = warp_sum(acc[0][b]);
      if (b < a.B) {
        if (lane == b) a.logits[(size_t)b * a.V + n] = v;
        const unsigned long long key = argmax_key(v, (uint32_t)n);
        best[b] = key > best[b] ? key : best[b];
      }
    }
  }
  if (lane == 0)
#pragma unroll
    for (int b = 0; b < BT; ++b) best_s[warp][b] = best[b];
  __syncthreads();
  if (threadIdx.x < BT && threadIdx.x < a.B) {
    unsigned long long m = 0ull;
    for (int w = 0; w < kWarps; ++w) m = best_s[w][threadIdx.x] > m ? best_s[w][threadIdx.x] : m;
    a.part[(size_t)threadIdx.x * gridDim.x + blockIdx.x] = m;
  }
  // Last block to finish combines the per-block partials (deterministic:
  // max over integer keys is order-independent).
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last_s = atomicAdd(a.ticket, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!last_s) return;
  __threadfence();
  for (int b = warp; b < a.B; b += kWarps) {
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
      // Greedy feedback for the next step: every kernel of this step that
      // reads tokens or positions ran before this one (stream order).
      if (a.advance_tokens) a.advance_tokens[b] = nan ? 0 : tok;
      if (a.advance_positions) a.advance_positions[b] += 1;
    }
  }
  if (threadIdx.x == 0) *a.ticket = 0u;
}

int lm_head_grid() { return num_sms() * 4; }

template <int BT>
static cudaError_t lm_bt(const LmHeadArgs& a, cudaStream_t s) {
  const size_t smem = sizeof(float) * (size_t)BT * a.K;
  cudaError_t e = ensure_smem<k_lm_head<BT>>();
  if (e != cudaSuccess) return e;
  return launch_pdl(k_lm_head<BT>, dim3(lm_head_grid()), dim3(kThreads), smem, s, a);
}

cudaError_t launch_lm_head(const LmHeadArgs& a, cudaStream_t s) {
  if (lm_head16_supported(a.B, a.K)) return launch_lm_head16(a, s);
  if (a.B <= 1) return lm_bt<1>(a, s);
  if (a.B <= 2) return lm_bt<2>(a, s);
  if (a.B <= 4) return lm_bt<4>(a, s);
  if (a.B <= 8) return lm_bt<8>(a, s);
  return lm_bt<16>(a, s);
}

// ------------------------------------------------------------------ embedding
__global__ void k_embed(const uint16_t* E, const int32_t* tokens, int B, int H, int V, float* x,
                        int* status) {
  pdl_wait();
  const int b = blockIdx.y;
  int tok = tokens[b];
  if (tok < 0 || tok >= V) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && status) atomicCAS(status, 0, (int)NC_ERR_INVALID_ARGUMENT);
    tok = 0;
  }
  const uint16_t* row = E + (size_t)tok * H;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < H; i += gridDim.x * blockDim.x)
    x[(size_t)b * H + i] = bf16_to_f32(row[i]);
}

cudaError_t launch_embed(const uint16_t* E, const int32_t* tokens, int B, int H, int V, float* x,
                         int* status, cudaStream_t s) {
  return launch_pdl(k_embed, dim3((H + 255) / 256, B), dim3(256), 0, s, E, tokens, B, H, V, x,
                    status);
}

}  // namespace nc
