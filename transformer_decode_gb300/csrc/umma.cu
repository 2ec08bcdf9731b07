// umma.cu -- dense contractions on the 5th-generation tensor cores.
//
// Y[t, n] = sum_k W[n, k] X[t, k] for T tokens at once: the projections of a
// batch of 9..16 sequences and of a prompt run as one prefill. Matrix-shaped
// tiles belong on the tensor cores (Tang section 5); at one token a GEMV
// stays on the CUDA cores.
//
// One CTA computes a tile of 128 weight rows by NT tokens:
//  * warp 0 (one lane) streams the tiles with TMA (cp.async.bulk.tensor, 2-D
//    tensor maps over this GPU's own memory): per 64-wide k block, 128 rows of
//    W (two boxes of 64 rows: for gate|up, 64 gate rows and the 64 up rows
//    that pair with them) and the k block of the activations, all in the
//    128-byte swizzled layout the tensor core reads, into a ring of stages
//    with mbarrier completion;
//  * warp 1 holds the accumulator in tensor memory (tcgen05.alloc) and one
//    lane issues tcgen05.mma (kind::f16, bf16 inputs, fp32 accumulation),
//    four k16 steps per stage, committing each stage back to the producer;
//  * the activations enter as two bf16 planes, hi = bf16(x) and lo =
//    bf16(x - hi), stacked as the 2 NT columns of the B operand, so the
//    product keeps the fp32 input's precision: the epilogue adds column t and
//    column NT + t;
//  * all four warps read their 32 TMEM lanes (tcgen05.ld) and apply the
//    epilogue: bias, residual add (atomic when k is split over CTAs),
//    SiLU(gate) * up, or logits with the arg-max keys.
// Every wait is bounded by %globaltimer: on expiry the CTA records
// NC_ERR_TIMEOUT, stops issuing, drains what it issued and frees its TMEM.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>

#include "kernels.h"

namespace nc {

constexpr int kUThreads = 128;
constexpr int kUKBlock = 64;         // k elements per stage (128 bytes of bf16)
constexpr int kURows = 128;          // weight rows per CTA (the MMA's M)
constexpr int kUAStage = kURows * kUKBlock * 2;  // 16 KB

// ------------------------------------------------------------------ PTX
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void umma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
// 16 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor of a K-major operand tile in the 128-byte
// swizzled layout (rows of 128 bytes, 8-row groups 1024 bytes apart): start
// address, leading offset unused for this layout (1), stride offset 1024
// bytes, descriptor version 1, swizzle mode 2 (128 bytes).
__device__ __forceinline__ uint64_t sw128_desc(const void* tile) {
  const uint64_t a = (smem_addr(tile) & 0x3FFFFu) >> 4;
  return a | (uint64_t(1) << 16) | (uint64_t(1024 >> 4) << 32) | (uint64_t(1) << 46) |
         (uint64_t(2) << 61);
}
// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, N and M encoded as N / 8 and M / 16.
__host__ __device__ constexpr uint32_t umma_idesc(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// ------------------------------------------------------------------ kernel
struct UArgs {
  int N;             // output rows (SwiGLU: F, the gate|up pairs)
  int K;
  int T;             // tokens
  int kb_per_cta;    // k blocks of 64 per CTA (k split over gridDim.z)
  int up_row0;       // SwiGLU: first up row in the W map (= F)
  const uint16_t* bias;  // [N] or null (Store)
  float* y;          // [T, ldy]
  int ldy;
  // LM head: per-CTA arg-max keys [T][grid.x], the ticket and the outputs of
  // the last CTA (lm == 1)
  int lm;
  unsigned long long* part;
  unsigned int* ticket;
  int32_t* next;
  int* status;
  int32_t* advance_tokens;
  int32_t* advance_positions;
  unsigned long long timeout_ns;
};

template <int NT>
__host__ __device__ constexpr int ustage_bytes() {
  return kUAStage + 2 * NT * kUKBlock * 2;
}
// Token tiles of 64 or more (prefill) run two CTAs per SM, so one CTA's
// epilogue overlaps the other's products: half the shared memory (and at
// most 256 tensor-memory columns) each. Smaller tiles keep one CTA per SM.
template <int NT>
__host__ __device__ constexpr int uctas_per_sm() { return NT >= 64 ? 2 : 1; }
template <int NT>
__host__ __device__ constexpr int ustages() {
  constexpr int budget = (uctas_per_sm<NT>() == 2 ? 100 : 200) * 1024;
  return budget / ustage_bytes<NT>() > 8 ? 8 : budget / ustage_bytes<NT>();
}
template <int NT>
__host__ __device__ constexpr uint32_t utmem_cols() {
  return 2 * NT <= 32 ? 32u : (2 * NT <= 64 ? 64u : (2 * NT <= 128 ? 128u : 256u));
}

struct UShared {
  uint64_t full[8], empty[8], done;
  uint32_t tmem;
  int abort;
  int last;
  unsigned long long best[4][128];  // LM head: per-warp arg-max key per token
};

template <Epi EPI, int NT>
__global__ void __launch_bounds__(kUThreads, uctas_per_sm<NT>())
    k_umma(const __grid_constant__ CUtensorMap tw, const __grid_constant__ CUtensorMap tx,
           const UArgs a) {
  constexpr int S = ustages<NT>();
  constexpr int SB = ustage_bytes<NT>();
  constexpr uint32_t COLS = utmem_cols<NT>();
  extern __shared__ uint8_t usm_raw[];
  // stage buffers 1024-byte aligned (the swizzle pattern follows the address)
  uint8_t* usm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(usm_raw) + sizeof(UShared) + 1023) & ~uintptr_t(1023));
  UShared& U = *reinterpret_cast<UShared*>(usm_raw);
  const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
  const int n0 = blockIdx.x * (EPI == Epi::SwiGLU ? kURows / 2 : kURows);
  const int t0 = blockIdx.y * NT;
  const int nkb_all = a.K / kUKBlock;
  const int kb0 = blockIdx.z * a.kb_per_cta;
  const int nkb = min(a.kb_per_cta, nkb_all - kb0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&U.full[s], 1);
      mbar_init(&U.empty[s], 1);
    }
    mbar_init(&U.done, 1);
    U.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tw)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tx)) : "memory");
  }
  if (warp == 1) tmem_alloc(&U.tmem, COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // No kernel writes the weights: the first stages' weight boxes are issued
  // before the wait, so their round trip overlaps the activation kernel
  // (which lets this grid launch once its own wait is over, so every kernel
  // before it has completed).
  const int pre = nkb < S ? nkb : S;
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < pre; ++i) {
      uint8_t* st = usm + (size_t)i * SB;
      const int kx = (kb0 + i) * kUKBlock;
      mbar_expect_tx(&U.full[i], (uint32_t)SB);
      tma_load_2d(st, &tw, kx, n0, &U.full[i]);
      tma_load_2d(st + kUAStage / 2, &tw,
                  kx, EPI == Epi::SwiGLU ? a.up_row0 + n0 : n0 + kURows / 2, &U.full[i]);
    }
  }
  // the activation planes and (residual form) the output come from earlier
  // kernels: every thread waits for them to be complete and visible
  pdl_wait();
  const uint32_t tmem = U.tmem;
  const uint64_t deadline = global_timer() + a.timeout_ns;
  auto expired = [&]() {
    if (*reinterpret_cast<volatile int*>(&U.abort)) return true;
    if (global_timer() > deadline) {
      atomicExch(&U.abort, 1);
      if (a.status) atomicCAS(a.status, 0, (int)NC_ERR_TIMEOUT);
      return true;
    }
    return false;
  };
  auto wait_bar = [&](uint64_t* bar, uint32_t par) {
    int k = 0;
    while (!mbar_try_wait(bar, par))
      if ((++k & 63) == 0 && expired()) return false;
    return true;
  };

  int issued = 0;  // stages the producer filled (for the drain)
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < nkb; ++i) {
      const int s = i % S;
      uint8_t* st = usm + (size_t)s * SB;
      const int kx = (kb0 + i) * kUKBlock;
      if (i >= pre) {  // the first stages' weights are in flight already
        if (i >= S && !wait_bar(&U.empty[s], ((i / S) - 1) & 1)) break;
        if (*reinterpret_cast<volatile int*>(&U.abort)) break;
        mbar_expect_tx(&U.full[s], (uint32_t)SB);
        tma_load_2d(st, &tw, kx, n0, &U.full[s]);
        tma_load_2d(st + kUAStage / 2, &tw,
                    kx, EPI == Epi::SwiGLU ? a.up_row0 + n0 : n0 + kURows / 2, &U.full[s]);
      }
      tma_load_2d(st + kUAStage, &tx, kx, blockIdx.y * 2 * NT, &U.full[s]);
      issued = i + 1;
    }
  } else if (warp == 1 && lane == 0) {
    constexpr uint32_t idesc = umma_idesc(kURows, 2 * NT);
    int i = 0;
    for (; i < nkb; ++i) {
      const int s = i % S;
      if (!wait_bar(&U.full[s], (i / S) & 1)) break;
      tc_fence_after();
      const uint8_t* st = usm + (size_t)s * SB;
      const uint64_t ad = sw128_desc(st), bd = sw128_desc(st + kUAStage);
#pragma unroll
      for (int k = 0; k < kUKBlock / 16; ++k)  // 16 k = 32 bytes = 2 descriptor units
        umma_f16(tmem, ad + 2 * k, bd + 2 * k, idesc, (i > 0 || k > 0) ? 1u : 0u);
      umma_commit(&U.empty[s]);
    }
    umma_commit(&U.done);  // arrives once every issued product has completed
  }
  __syncwarp();
  // every thread: the accumulator is complete (bounded; after an abort the
  // commit above still arrives once the issued products drain)
  wait_bar(&U.done, 0);
  tc_fence_after();
  const bool ok = !*reinterpret_cast<volatile int*>(&U.abort) && nkb > 0;
  pdl_trigger();  // the next kernel's launch overlaps this epilogue

  // ---------------------------------------------------------------- epilogue
  // thread (warp w, lane l) owns TMEM lane 32 w + l = weight row r of the tile
  const int r = warp * 32 + lane;
  const uint32_t lane_addr = tmem + (uint32_t(warp * 32) << 16);
  float* xch = reinterpret_cast<float*>(usm);  // SwiGLU: up values [64][16]
  for (int tb = 0; tb < NT; tb += 16) {
    float hi[16], lo[16], v[16];
    tmem_ld16(lane_addr + tb, hi);
    tmem_ld16(lane_addr + NT + tb, lo);
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = hi[j] + lo[j];
    if constexpr (EPI == Epi::SwiGLU) {
      // rows 64..127 are the up rows of rows 0..63
      __syncthreads();  // the stage buffers (and the previous round's xch) are free
      if (warp >= 2)
#pragma unroll
        for (int j = 0; j < 16; ++j) xch[(r - 64) * 16 + j] = v[j];
      __syncthreads();
      if (warp < 2 && ok) {
        const int n = n0 + r;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int t = t0 + tb + j;
          if (n < a.N && t < a.T) {
            const float g = v[j], u = xch[r * 16 + j];
            const float e = expf(-fabsf(g));
            const float sig = g >= 0.f ? 1.f / (1.f + e) : e / (1.f + e);
            a.y[(size_t)t * a.ldy + n] = (g * sig) * u;
          }
        }
      }
    } else {
      const int n = n0 + r;
      if (ok && n < a.N) {
        const float b = (EPI == Epi::Store && a.bias) ? bf16_to_f32(a.bias[n]) : 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int t = t0 + tb + j;
          if (t >= a.T) break;
          float* yp = a.y + (size_t)t * a.ldy + n;
          if constexpr (EPI == Epi::Residual) {
            if (gridDim.z > 1) atomicAdd(yp, v[j]);
            else *yp = *yp + v[j];
          } else if (gridDim.z > 1) {  // k split: y was zeroed; the first slice adds the bias
            atomicAdd(yp, blockIdx.z == 0 ? v[j] + b : v[j]);
          } else {
            *yp = v[j] + b;
          }
        }
        if (a.lm) {
          // arg-max keys of this row for the tile's tokens, max over the warp
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            unsigned long long key = t0 + tb + j < a.T ? argmax_key(v[j], (uint32_t)n) : 0ull;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
              const unsigned long long q = __shfl_xor_sync(0xFFFFFFFFu, key, o);
              key = q > key ? q : key;
            }
            if (lane == 0) U.best[warp][tb + j] = key;
          }
        }
      } else if (a.lm) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          unsigned long long key = 0ull;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long q = __shfl_xor_sync(0xFFFFFFFFu, key, o);
            key = q > key ? q : key;
          }
          if (lane == 0) U.best[warp][tb + j] = key;
        }
      }
    }
  }

  // drain: copies issued but not consumed (only after an abort) land before
  // the CTA exits; then the accumulator is released
  if (warp == 0 && lane == 0 && *reinterpret_cast<volatile int*>(&U.abort)) {
    const uint64_t dl = global_timer() + a.timeout_ns;
    for (int t = issued > S ? issued - S : 0; t < issued; ++t)
      while (!mbar_try_wait(&U.full[t % S], (t / S) & 1))
        if (global_timer() > dl) break;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, COLS);

  if constexpr (EPI == Epi::Store) {
    if (!a.lm) return;
    // LM head: the CTA's key per token, then the last CTA combines them
    if (threadIdx.x < NT && t0 + (int)threadIdx.x < a.T) {
      unsigned long long m = 0ull;
      for (int w = 0; w < 4; ++w) m = U.best[w][threadIdx.x] > m ? U.best[w][threadIdx.x] : m;
      a.part[(size_t)(t0 + threadIdx.x) * gridDim.x + blockIdx.x] = ok ? m : ~0ull;
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0)
      U.last = atomicAdd(a.ticket, 1u) == gridDim.x * gridDim.y - 1;
    __syncthreads();
    if (!U.last) return;
    __threadfence();
    for (int t = warp; t < a.T; t += kUThreads / kWarp) {
      unsigned long long m = 0ull;
      for (int i = lane; i < (int)gridDim.x; i += kWarp) {
        const unsigned long long k = __ldcg(a.part + (size_t)t * gridDim.x + i);
        m = k > m ? k : m;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long q = __shfl_xor_sync(0xFFFFFFFFu, m, o);
        m = q > m ? q : m;
      }
      if (lane == 0) {
        const bool nan = m == ~0ull;
        const int32_t tok = nan ? -1 : (int32_t)(0xFFFFFFFFu - (uint32_t)(m & 0xFFFFFFFFull));
        if (a.next) a.next[t] = tok;
        if (nan && a.status) atomicCAS(a.status, 0, (int)NC_ERR_INVALID_ARGUMENT);
        if (a.advance_tokens) a.advance_tokens[t] = nan ? 0 : tok;
        if (a.advance_positions) a.advance_positions[t] += 1;
      }
    }
    if (threadIdx.x == 0) *a.ticket = 0u;
  }
}

// ------------------------------------------------------------------ activations
// xb [T_tiles][2][NT][K] bf16: per tile of NT tokens the hi plane then the
// lo plane of the (normed) activations; rows past T are zero. One CTA per
// token: the RMSNorm factor (when gamma is set) from the row's sum of squares.
// One pass: every thread loads its 16-byte chunks of the token's row at once
// (kActChunks per thread covers rows up to 256 * 4 * kActChunks), forms the
// RMSNorm factor from them, and writes the hi / lo planes from registers.
// With yz set it also zeroes the product's output rows yz[t][0, yN) (stride
// yld), which a k-split store then accumulates into.
constexpr int kActChunks = 12;
constexpr int kActMaxK = 256 * 4 * kActChunks;
__global__ void __launch_bounds__(256) k_umma_act(const float* x, const uint16_t* gamma, float eps,
                                                  int T, int K, int NT, uint16_t* xb, float* yz,
                                                  int yN, int yld) {
  pdl_wait();
  pdl_trigger();  // the product kernel may launch and fetch its weights meanwhile
  const int t = blockIdx.x;
  if (yz && t < T)
    for (int n = threadIdx.x; n < yN; n += 256) yz[(size_t)t * yld + n] = 0.f;
  const int tile = t / NT, tt = t % NT;
  uint16_t* hi = xb + ((size_t)tile * 2 * NT + tt) * K;
  uint16_t* lo = hi + (size_t)NT * K;
  __shared__ float red[8];
  const int C4 = K / 4;  // 16-byte chunks of the row
  float4 v[kActChunks];
#pragma unroll
  for (int j = 0; j < kActChunks; ++j) {
    const int c = threadIdx.x + j * 256;
    v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (t < T && c < C4) v[j] = reinterpret_cast<const float4*>(x + (size_t)t * K)[c];
  }
  float r = 1.f;
  if (t < T && gamma) {
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < kActChunks; ++j)
      ss = fmaf(v[j].x, v[j].x, fmaf(v[j].y, v[j].y, fmaf(v[j].z, v[j].z, fmaf(v[j].w, v[j].w, ss))));
    ss = warp_sum(ss);
    if (threadIdx.x % kWarp == 0) red[threadIdx.x / kWarp] = ss;
    __syncthreads();
    float tot = 0.f;
    for (int w = 0; w < (int)blockDim.x / kWarp; ++w) tot += red[w];
    r = 1.f / sqrtf(tot / (float)K + eps);
  }
#pragma unroll
  for (int j = 0; j < kActChunks; ++j) {
    const int c = threadIdx.x + j * 256;
    if (c >= C4) break;
    float f[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
    uint16_t h[4], l[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float u = f[e];
      if (gamma && t < T) u = (u * r) * bf16_to_f32(gamma[4 * c + e]);
      h[e] = f32_to_bf16(u);
      l[e] = f32_to_bf16(u - bf16_to_f32(h[e]));
    }
    reinterpret_cast<uint2*>(hi)[c] = make_uint2(h[0] | ((uint32_t)h[1] << 16), h[2] | ((uint32_t)h[3] << 16));
    reinterpret_cast<uint2*>(lo)[c] = make_uint2(l[0] | ((uint32_t)l[1] << 16), l[2] | ((uint32_t)l[3] << 16));
  }
}

// ------------------------------------------------------------------ host
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiled encode_fn() {
  static EncodeTiled fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiled>(nullptr);
    return reinterpret_cast<EncodeTiled>(p);
  }();
  return fn;
}

// A 2-D bf16 tensor map over rows of `cols` elements, `rows` rows, with a box
// of 64 elements by box_rows rows in the 128-byte swizzled layout; reads
// past the edges are zero.
static cudaError_t make_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows,
                            uint32_t box_rows) {
  EncodeTiled enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kUKBlock, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

int umma_tokens_per_tile(int T) { return T <= 16 ? 16 : (T <= 32 ? 32 : (T <= 64 ? 64 : 128)); }

size_t umma_act_bytes(int T, int K) {
  const int NT = umma_tokens_per_tile(T);
  return (size_t)((T + NT - 1) / NT) * 2 * NT * K * 2;
}

template <Epi EPI, int NT>
static cudaError_t launch_umma_nt(const UmmaArgs& g, const CUtensorMap& tw, const CUtensorMap& tx,
                                  int ks, cudaStream_t s) {
  auto kern = k_umma<EPI, NT>;
  const int smem = (int)sizeof(UShared) + 1024 + ustages<NT>() * ustage_bytes<NT>();
  static const cudaError_t attr =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (attr != cudaSuccess) return attr;
  UArgs a{};
  a.N = g.N;
  a.K = g.K;
  a.T = g.T;
  const int nkb = g.K / kUKBlock;
  a.kb_per_cta = (nkb + ks - 1) / ks;
  a.up_row0 = g.N;
  a.bias = g.bias;
  a.y = g.y;
  a.ldy = g.ldy;
  a.lm = g.lm ? 1 : 0;
  a.part = g.part;
  a.ticket = g.ticket;
  a.next = g.next;
  a.status = g.status;
  a.advance_tokens = g.advance_tokens;
  a.advance_positions = g.advance_positions;
  a.timeout_ns = 200ull * 1000 * 1000;
  const int rows_per_cta = EPI == Epi::SwiGLU ? kURows / 2 : kURows;
  dim3 grid((g.N + rows_per_cta - 1) / rows_per_cta, (g.T + NT - 1) / NT,
            (nkb + a.kb_per_cta - 1) / a.kb_per_cta);
  return launch_pdl(kern, grid, dim3(kUThreads), (size_t)smem, s, tw, tx, a);
}

template <Epi EPI>
static cudaError_t launch_umma_epi(const UmmaArgs& g, const CUtensorMap& tw, const CUtensorMap& tx,
                                   int NT, int ks, cudaStream_t s) {
  switch (NT) {
    case 16: return launch_umma_nt<EPI, 16>(g, tw, tx, ks, s);
    case 32: return launch_umma_nt<EPI, 32>(g, tw, tx, ks, s);
    case 64: return launch_umma_nt<EPI, 64>(g, tw, tx, ks, s);
    default: return launch_umma_nt<EPI, 128>(g, tw, tx, ks, s);
  }
}

bool umma_supported(int K) {
  return K >= kUKBlock && K % kUKBlock == 0 && K <= kActMaxK && encode_fn() != nullptr;
}

cudaError_t launch_umma(Epi epi, const UmmaArgs& g, cudaStream_t s) {
  const int NT = umma_tokens_per_tile(g.T);
  const int tiles = (g.T + NT - 1) / NT;
  // the activation planes (normed when gamma is set)
  // k split over CTAs when the tiles alone leave most SMs idle, for the
  // residual form and the plain store (atomic adds; the store's output is
  // zeroed by the activation kernel first), not for the LM head (its arg-max
  // wants finished logits)
  int ks = 1;
  if (epi == Epi::Residual || (epi == Epi::Store && !g.lm)) {
    const int ctas = ((g.N + kURows - 1) / kURows) * tiles;
    const int nkb = g.K / kUKBlock;
    ks = (num_sms() + ctas - 1) / ctas;
    if (ks > nkb / 2) ks = nkb / 2;
    if (ks < 1) ks = 1;
  }
  const bool zero = epi == Epi::Store && ks > 1;
  cudaError_t e = launch_pdl(k_umma_act, dim3(tiles * NT), dim3(256), 0, s, g.x, g.gamma, g.eps,
                             g.T, g.K, NT, g.xb, zero ? g.y : nullptr, g.N, g.ldy);
  if (e != cudaSuccess) return e;
  CUtensorMap tw, tx;
  const uint64_t wrows = epi == Epi::SwiGLU ? 2 * (uint64_t)g.N : (uint64_t)g.N;
  if ((e = make_map(&tw, g.W, g.K, wrows, kURows / 2)) != cudaSuccess) return e;
  if ((e = make_map(&tx, g.xb, g.K, (uint64_t)tiles * 2 * NT, 2 * NT)) != cudaSuccess) return e;
  switch (epi) {
    case Epi::Store: return launch_umma_epi<Epi::Store>(g, tw, tx, NT, ks, s);
    case Epi::Residual: return launch_umma_epi<Epi::Residual>(g, tw, tx, NT, ks, s);
    default: return launch_umma_epi<Epi::SwiGLU>(g, tw, tx, NT, 1, s);
  }
}

}  // namespace nc
