// nc_internal.cuh -- helpers shared by libnc's kernels and host code.
//
// Nothing here is numerics beyond bf16 widening (exact: a bf16 value is the
// top half of an fp32 word) and fp32 reductions.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include <cstdio>
#include <string>

#include "../../include/nc.h"

namespace nc {

constexpr int kWarp = 32;
constexpr int kNumSMs = 152;  // GB300; the host code queries the real count

// ---------------------------------------------------------------- errors
void set_error(const char* fmt, ...);
nc_status fail(nc_status s, const char* fmt, ...);

#define NC_CUDA_TRY(expr)                                                              \
  do {                                                                                 \
    cudaError_t _e = (expr);                                                           \
    if (_e != cudaSuccess)                                                             \
      return ::nc::fail(NC_ERR_CUDA, "%s failed: %s (%s:%d)", #expr, cudaGetErrorString(_e), \
                        __FILE__, __LINE__);                                            \
  } while (0)

#define NC_CHECK(cond, status, ...)                      \
  do {                                                   \
    if (!(cond)) return ::nc::fail((status), __VA_ARGS__); \
  } while (0)

// ---------------------------------------------------------------- device helpers
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}
// Round to nearest even (the hardware conversion).
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
  unsigned short r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(f));
  return r;
}

// 16-byte streaming load of data read once (weights): no L1 allocation.
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Programmatic dependent launch. Stage kernels are launched so that the next
// kernel in the stream may start once every CTA of this one has exited (or
// called pdl_trigger), before the grid's completion is flushed: its prologue
// does only work that reads no output of an earlier kernel and writes no
// global memory (warming L2 with its weights, or loading weight tiles), then
// waits for the earlier kernels to complete and their writes to be visible
// (pdl_wait). Launched the ordinary way, the wait is a no-op. Only the
// tensor-core activation and product kernels trigger early; for the GEMV
// kernels an early trigger from the top measured slower (the successor's L2
// warm-up then runs too far ahead of use).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Let the next kernel in the stream launch before this one exits (once every
// CTA of this grid has called it or exited). A kernel calls it only after its
// own pdl_wait, so everything before it in the stream is complete when the
// successor's prologue runs; the successor still waits in pdl_wait for this
// grid's writes.
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Fetch [p, p + bytes) into L2 without waiting (p 16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}
__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// 8 bf16 (one 16-byte chunk) times 8 fp32 from shared memory.
__device__ __forceinline__ float dot8(const uint4& w, const float* x) {
  const float4 a = *reinterpret_cast<const float4*>(x);
  const float4 b = *reinterpret_cast<const float4*>(x + 4);
  float s = bf16_lo(w.x) * a.x;
  s = fmaf(bf16_hi(w.x), a.y, s);
  s = fmaf(bf16_lo(w.y), a.z, s);
  s = fmaf(bf16_hi(w.y), a.w, s);
  s = fmaf(bf16_lo(w.z), b.x, s);
  s = fmaf(bf16_hi(w.z), b.y, s);
  s = fmaf(bf16_lo(w.w), b.z, s);
  s = fmaf(bf16_hi(w.w), b.w, s);
  return s;
}

// Order-preserving map of a float to uint32 (larger float -> larger key).
__device__ __forceinline__ uint32_t float_order_key(float f) {
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
// Arg-max key: value in the high word, (0xFFFFFFFF - index) in the low word so
// that equal values resolve to the lowest index under max. NaN -> all ones.
__device__ __forceinline__ unsigned long long argmax_key(float v, uint32_t idx) {
  if (v != v) return ~0ull;
  return (static_cast<unsigned long long>(float_order_key(v)) << 32) |
         static_cast<unsigned long long>(0xFFFFFFFFu - idx);
}

// ---------------------------------------------------------------- async copies
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ uint64_t global_timer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Sums each of the N values of a lane over the warp in N - 1 + (5 - log2 N)
// shuffles instead of 5 N: every butterfly step swaps half of the values
// with the partner lane, so the number a lane carries halves. Afterwards
// v[0] of lane i * (32 / N) holds the warp total of value i.
template <int N>
__device__ __forceinline__ void warp_sum_many(float (&v)[N]) {
  static_assert(N >= 1 && N <= kWarp && (N & (N - 1)) == 0, "N must be a power of two");
  const int lane = threadIdx.x % kWarp;
  int o = kWarp / 2;
#pragma unroll
  for (int half = N / 2; half >= 1; half /= 2, o /= 2) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int k = 0; k < half; ++k) {
      const float send = upper ? v[k] : v[k + half];
      const float keep = upper ? v[k + half] : v[k];
      v[k] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, o);
    }
  }
#pragma unroll
  for (; o > 0; o /= 2) v[0] += __shfl_xor_sync(0xFFFFFFFFu, v[0], o);
}

// ---------------------------------------------------------------- KV addressing
struct KVView {
  void* k;  // fp32 or bf16 elements (bf16 != 0)
  void* v;
  const int32_t* block_table;  // paged only
  int paged;
  int bf16;
  int batch_capacity;
  int max_ctx;
  int block_size;
  int num_blocks;
  int max_blocks_per_seq;
  int n_kv_heads;
  int head_dim;
  __device__ __forceinline__ int capacity() const {
    return paged ? max_blocks_per_seq * block_size : max_ctx;
  }
  // True when slot t of sequence b exists: t inside the capacity and, when
  // paged, its block-table entry inside the pool. The host validates the same
  // facts from its copies; this guards against device copies that disagree.
  __device__ __forceinline__ bool slot_ok(int b, int t) const {
    if (t < 0 || t >= capacity()) return false;
    if (!paged) return true;
    const int blk = block_table[(size_t)b * max_blocks_per_seq + t / block_size];
    return blk >= 0 && blk < num_blocks;
  }
  // element offset of (layer, seq b, kv head g, position t)
  __device__ __forceinline__ size_t offset(int layer, int b, int g, int t) const {
    if (!paged) {
      return ((((size_t)layer * batch_capacity + b) * n_kv_heads + g) * max_ctx + t) *
             (size_t)head_dim;
    }
    const int blk = block_table[(size_t)b * max_blocks_per_seq + t / block_size];
    return ((((size_t)layer * num_blocks + blk) * n_kv_heads + g) * block_size +
            t % block_size) *
           (size_t)head_dim;
  }
};

// Eight consecutive cache elements (16-byte aligned start) widened to fp32.
template <bool KV16>
__device__ __forceinline__ void kv_load8(const void* base, size_t off, float (&f)[8]) {
  if constexpr (KV16) {
    const uint4 w = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + off);
    f[0] = bf16_lo(w.x); f[1] = bf16_hi(w.x); f[2] = bf16_lo(w.y); f[3] = bf16_hi(w.y);
    f[4] = bf16_lo(w.z); f[5] = bf16_hi(w.z); f[6] = bf16_lo(w.w); f[7] = bf16_hi(w.w);
  } else {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + off);
    const float4 a = p[0], b = p[1];
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  }
}
// Two consecutive cache elements (8-byte aligned for fp32, 4 for bf16).
template <bool KV16>
__device__ __forceinline__ float2 kv_load2(const void* base, size_t off) {
  if constexpr (KV16) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(static_cast<const uint16_t*>(base) + off);
    return make_float2(bf16_lo(w), bf16_hi(w));
  } else {
    return *reinterpret_cast<const float2*>(static_cast<const float*>(base) + off);
  }
}
// Store one cache element (bf16: round to nearest even).
template <bool KV16>
__device__ __forceinline__ void kv_store(void* base, size_t off, float v) {
  if constexpr (KV16)
    static_cast<uint16_t*>(base)[off] = f32_to_bf16(v);
  else
    static_cast<float*>(base)[off] = v;
}

}  // namespace nc
