// attention.cu -- RoPE + KV append, and split-K grouped-query decode attention.
//
// RoPE (nanoinfer "Model architecture", "KV cache"): half-split pairs
// (i, i + D/2), angle = float(pos) * inv_freq[i] as an fp32 product, applied
// once to K on insert; K and V are rounded to bf16 when stored.
//
// Attention (Tang section 2.2: online softmax is the monoid on (m, l, acc);
// section 2.5: split is valid for any associative monoid): the positions
// 0..pos of one (sequence, kv head) are cut into `splits` ranges. Each CTA
// reads its range of K and V once for all G query heads of the group (the
// repeat_kv expansion folded into indexing, nanocompile "Phase 3"), produces
// the partial (m, l, acc[D]) per head, and the last CTA of the group to
// finish combines the partials:
//   M = max_c m_c,  out = sum_c acc_c e^(m_c - M) / sum_c l_c e^(m_c - M).
#include <cuda_runtime.h>
#include <math.h>

#include "kernels.h"

namespace nc {

// ------------------------------------------------------------------ RoPE
template <int D, bool KV16>
__global__ void __launch_bounds__(256) k_rope_qkv(RopeArgs a) {
  constexpr int E = D / 32;  // elements per lane
  pdl_wait();
  const int b = blockIdx.x;
  const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
  const int pos = a.seq >= 0 ? a.pos0 + b : a.positions[b];
  const int kb = a.seq >= 0 ? a.seq : b;  // the cache sequence of row b
  if (!a.kv.slot_ok(kb, pos)) {
    if (threadIdx.x == 0 && blockIdx.y == 0 && a.status) atomicCAS(a.status, 0, (int)NC_ERR_POSITION);
    return;
  }
  const int qkv_dim = (a.Hq + 2 * a.Hkv) * D;
  const float* src = a.qkv + (size_t)b * qkv_dim;
  // blockIdx.y picks this CTA's heads: one per warp, so the heads run side by side
  for (int hh = blockIdx.y * (blockDim.x / kWarp) + warp; hh < a.Hq + a.Hkv;
       hh += gridDim.y * (blockDim.x / kWarp)) {
    const bool is_q = hh < a.Hq;
    const float* v = src + (size_t)hh * D;
    float e[E];
#pragma unroll
    for (int j = 0; j < E; ++j) e[j] = v[lane + 32 * j];
    const uint16_t* gain = is_q ? a.g_q : a.g_k;
    if (gain) {  // per-head RMSNorm over D
      float ss = 0.f;
#pragma unroll
      for (int j = 0; j < E; ++j) ss = fmaf(e[j], e[j], ss);
      ss = warp_sum(ss);
      const float r = 1.f / sqrtf(ss / (float)D + a.eps);
#pragma unroll
      for (int j = 0; j < E; ++j) e[j] = (e[j] * r) * bf16_to_f32(gain[lane + 32 * j]);
    }
    // element lane + 32 j pairs with lane + 32 (j + E/2)
#pragma unroll
    for (int j = 0; j < E / 2; ++j) {
      const int i = lane + 32 * j;
      const float angle = __fmul_rn((float)pos, a.inv_freq[i]);
      float sn, cs;
      sincosf(angle, &sn, &cs);
      const float x0 = e[j], x1 = e[j + E / 2];
      e[j] = __fsub_rn(__fmul_rn(x0, cs), __fmul_rn(x1, sn));
      e[j + E / 2] = __fadd_rn(__fmul_rn(x1, cs), __fmul_rn(x0, sn));
    }
    if (is_q) {
#pragma unroll
      for (int j = 0; j < E; ++j) a.q_out[((size_t)b * a.Hq + hh) * D + lane + 32 * j] = e[j];
    } else {
      const int g = hh - a.Hq;
      const size_t off = a.kv.offset(a.layer, kb, g, pos);
      const float* vv = src + (size_t)(a.Hq + a.Hkv + g) * D;
#pragma unroll
      for (int j = 0; j < E; ++j) {
        kv_store<KV16>(a.kv.k, off + lane + 32 * j, e[j]);
        kv_store<KV16>(a.kv.v, off + lane + 32 * j, vv[lane + 32 * j]);
      }
    }
  }
}

cudaError_t launch_rope_qkv(const RopeArgs& a, cudaStream_t s) {
  const dim3 grid(a.B, (a.Hq + a.Hkv + 7) / 8);  // 8 warps per CTA, one head each
  const auto kern = a.D == 64 ? (a.kv.bf16 ? k_rope_qkv<64, true> : k_rope_qkv<64, false>)
                              : (a.kv.bf16 ? k_rope_qkv<128, true> : k_rope_qkv<128, false>);
  return launch_pdl(kern, grid, dim3(256), 0, s, a);
}

// ------------------------------------------------------------------ attention
constexpr int kAttnThreads = 256;
constexpr int kAttnWarps = kAttnThreads / kWarp;
constexpr int kAttnCh = 64;      // positions per staged chunk
constexpr int kAttnStages = 3;   // chunks in shared memory: two in flight while one is used
constexpr int kMaxSplits = 256;  // splits of one (sequence, kv head); the merge keeps one weight each
constexpr uint64_t kAttnWaitNs = 1000000000ull;  // bound on any wait for a staged chunk
constexpr int kAttnMinPer = 32;  // positions per split at least (shorter scans are not split)

template <int D, bool KV16>
struct AttnGeo {
  static constexpr int ES = KV16 ? 2 : 4;
  static constexpr size_t kRow = (size_t)D * ES;          // bytes of one cached row
  static constexpr size_t kStage = 2 * kAttnCh * kRow;    // a chunk's K rows, then its V rows
  static constexpr size_t kSmem = kAttnStages * kStage + sizeof(uint64_t) * kAttnStages;
  static_assert(kAttnStages * kStage >= sizeof(float) * (8 * 8 * D + 2 * 8 * 8),
                "the warps' states are combined in the spent stages");
  static_assert(kAttnStages * kStage >= sizeof(float) * 8 * kMaxSplits,
                "the merge's split weights fit in the spent stages");
};

// CTAs of the split kernel one SM holds (shared memory bound), cached per shape.
template <int D, bool KV16>
static int attn_occupancy();

// CTAs per kv head (the grid's x): one wave of resident CTAs over the kv
// heads, at most one per kAttnMinPer positions a full batch could scan, at
// least one per sequence; the kernel deals them to the sequences by length.
int attn_splits(int B, int Hkv, int D, bool kv16, int max_ctx) {
  const int occ = D == 64 ? (kv16 ? attn_occupancy<64, true>() : attn_occupancy<64, false>())
                          : (kv16 ? attn_occupancy<128, true>() : attn_occupancy<128, false>());
  long long s = (long long)num_sms() * occ / Hkv;
  const long long hi = (long long)B * ((max_ctx + kAttnMinPer - 1) / kAttnMinPer);
  if (s > hi) s = hi;
  if (s > kMaxSplits) s = kMaxSplits;
  if (s < B) s = B;
  return (int)s;
}

// Partials of one launch: [Hkv][splits][G][D + 2] = Hq x splits x (D + 2) floats.
size_t attn_part_floats(int B, int Hq, int D, int splits) {
  (void)B;
  return (size_t)Hq * splits * (D + 2);
}

// E consecutive cached elements (E = 2 or 4) of one staged row, widened to fp32.
template <int E, bool KV16>
__device__ __forceinline__ void load_row(const unsigned char* p, float (&f)[E]) {
  if constexpr (KV16) {
    if constexpr (E == 4) {
      const uint2 w = *reinterpret_cast<const uint2*>(p);
      f[0] = bf16_lo(w.x); f[1] = bf16_hi(w.x); f[2] = bf16_lo(w.y); f[3] = bf16_hi(w.y);
    } else {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
      f[0] = bf16_lo(w); f[1] = bf16_hi(w);
    }
  } else {
    if constexpr (E == 4) {
      const float4 w = *reinterpret_cast<const float4*>(p);
      f[0] = w.x; f[1] = w.y; f[2] = w.z; f[3] = w.w;
    } else {
      const float2 w = *reinterpret_cast<const float2*>(p);
      f[0] = w.x; f[1] = w.y;
    }
  }
}

// Head size 64 with groups of 8 heads: lane (position p = lane / 8, slice
// s = lane % 8) holds 8 dims of the position's K row and of every query head:
// fp32 dims 4s..4s+3 and 32+4s..32+4s+3 (two 16-byte loads, the 8 lanes of a
// load phase on 8 bank groups), bf16 dims 8s..8s+7 (one 16-byte load).
template <bool KV16>
__host__ __device__ __forceinline__ int slice_dim(int s, int j) {
  return KV16 ? 8 * s + j : (j < 4 ? 4 * s + j : 32 + 4 * s + (j - 4));
}
template <bool KV16>
__device__ __forceinline__ void load_slice(const unsigned char* row, int s, float (&f)[8]) {
  if constexpr (KV16) {
    const uint4 w = *reinterpret_cast<const uint4*>(row + 16 * s);
    f[0] = bf16_lo(w.x); f[1] = bf16_hi(w.x); f[2] = bf16_lo(w.y); f[3] = bf16_hi(w.y);
    f[4] = bf16_lo(w.z); f[5] = bf16_hi(w.z); f[6] = bf16_lo(w.w); f[7] = bf16_hi(w.w);
  } else {
    const float4 a = *reinterpret_cast<const float4*>(row + 16 * s);
    const float4 b = *reinterpret_cast<const float4*>(row + 128 + 16 * s);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  }
}
// Sum v[i] over the N lanes of each aligned group of N, value i landing in
// the group's lane i (a reduce-scatter of N - 1 shuffles).
template <int N>
__device__ __forceinline__ void group_sum_scatter(float (&v)[N]) {
  const int lane = threadIdx.x % kWarp;
  int o = N / 2;
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
}

// One CTA per (split c, kv head g, sequence b). Thread 0 streams the split's
// positions through a ring of kAttnStages shared-memory stages with bulk
// copies (one per run of positions contiguous in the cache: the whole chunk
// when the cache is contiguous, one block's worth when it is paged), so the
// next chunks are in flight while one is used. Scores: each warp takes
// 32 / GM positions at a time, a lane holding D / 32 dimensions of every
// query head in registers and of the position's K row, the G x (32 / GM)
// partial dots summed over the warp in one reduce-scatter. Each warp keeps
// its own online-softmax state (m, l, acc) over the positions it scored and
// accumulates their values at once, a lane holding D / 32 dims of every head,
// so a chunk needs no block barrier but the one that frees its stage; the
// warps' states are combined at the end (Tang section 2.2: the online softmax
// is a monoid on (m, l, acc), so any grouping merges exactly). The last CTA
// of (b, g) to finish merges the splits' partials the same way:
//   M = max_c m_c,  out = sum_c acc_c e^(m_c - M) / sum_c l_c e^(m_c - M).
// ROPE: the CTA starts from the projections instead (a.qkv, as the QKV GEMV
// left them) and does what k_rope_qkv would: q/k norm and RoPE of its G query
// heads (every split of the group recomputes them); split 0 also rotates the
// new key, appends K and V at slot pos and opens its running state with the
// new position, so the scan covers the cached positions 0..pos-1 only and
// nothing reads the appended row in this launch.
template <int D, int GM, bool KV16, bool ROPE>
__global__ void __launch_bounds__(kAttnThreads) k_attn_split(AttnArgs a) {
  using Geo = AttnGeo<D, KV16>;
  constexpr int ES = Geo::ES, E = D / kWarp;      // elements of a row per lane
  constexpr int NP = kWarp / GM;                  // positions per warp step of the scores
  extern __shared__ __align__(128) unsigned char sm[];
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + kAttnStages * Geo::kStage);  // [kAttnStages]
  __shared__ float den_s[GM];
  __shared__ unsigned long long valid_s[kAttnStages];  // positions of each stage that were copied
  __shared__ bool last_s;
  __shared__ int left_s[kAttnStages];  // warps yet to finish the chunk a stage holds
  __shared__ int issued_s;             // chunks issued so far
  __shared__ int abort_s;              // a chunk never landed
  __shared__ float q_s[ROPE ? GM : 1][D], kn_s[ROPE ? D : 1], vn_s[ROPE ? D : 1];
  __shared__ int plan_s[5];  // sequence (-1: idle), split, the sequence's splits, its first, position
  const int g = blockIdx.y, NB = gridDim.x;
  const int G = a.Hq / a.Hkv;
  const int tid = threadIdx.x, warp = tid / kWarp, lane = tid % kWarp;
  if (tid == 0) {
    for (int s = 0; s < kAttnStages; ++s) {
      mbar_init(&full[s], 1);
      left_s[s] = kAttnWarps;
    }
    issued_s = 0;
    abort_s = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  const int cap = a.kv.capacity();
  pdl_wait();
  if (warp == 0) {
    // The plan (every CTA derives the same one): the NB CTAs of kv head g are
    // dealt to the sequences in proportion to the positions each scans, at
    // least one each and at most one per kAttnMinPer positions; a sequence's
    // splits are consecutive CTAs. CTAs past the last split stay idle.
    int nb = 0, pb = 0;
    if (lane < a.B) {
      pb = a.positions[lane];
      nb = ROPE ? max(0, min(pb, cap)) : max(0, min(pb + 1, cap));
    }
    const int total = warp_sum_i(nb);
    int sb = 0;
    if (lane < a.B) {
      sb = total > 0 ? 1 + (int)((long long)(NB - a.B) * nb / total) : 1;
      sb = min(sb, max(1, (nb + kAttnMinPer - 1) / kAttnMinPer));
    }
    int incl = sb;
#pragma unroll
    for (int o = 1; o < kWarp; o <<= 1) {
      const int t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += t;
    }
    const int j0 = incl - sb, j = blockIdx.x;
    const bool mine = lane < a.B && j >= j0 && j < j0 + sb;
    if (mine) {
      plan_s[0] = lane;
      plan_s[1] = j - j0;
      plan_s[2] = sb;
      plan_s[3] = j0;
      plan_s[4] = pb;
    }
    if (__ballot_sync(0xFFFFFFFFu, mine) == 0u && lane == 0) plan_s[0] = -1;
  }
  __syncthreads();  // barriers initialised, plan in shared memory
  const int b = plan_s[0];
  if (b < 0) return;  // idle: no copy issued, no ticket taken
  const int c = plan_s[1], S = plan_s[2];
  const int pos = plan_s[4];
  const bool pos_ok = ROPE ? a.kv.slot_ok(b, pos) : (pos >= 0 && pos < cap);
  if (!pos_ok && tid == 0 && c == 0 && g == 0 && a.status)
    atomicCAS(a.status, 0, (int)NC_ERR_POSITION);
  const int n = ROPE ? max(0, min(pos, cap)) : max(0, min(pos + 1, cap));
  const int per = (n + S - 1) / S;
  const int t0 = min(n, c * per);
  const int len = max(0, min(n, t0 + per) - t0);
  const int nch = (len + kAttnCh - 1) / kAttnCh;
  // partials of (b, g): splits plan_s[3] .. + S of kv head g, [S][G][D + 2]
  float* part = a.part + ((size_t)g * NB + plan_s[3]) * G * (D + 2);
  const size_t cs = (size_t)G * (D + 2);  // split stride

  // Warp 0 fills stage ci % kAttnStages with chunk ci: lane i takes the
  // chunk's i-th run of positions inside one cache block (the whole chunk
  // when the cache is contiguous), so the block-table reads run side by side.
  // Positions whose block-table entry is a hole are not copied; the stage's
  // mask of copied positions goes to valid_s before the barrier's arrive.
  const int bs = a.kv.paged ? a.kv.block_size : (1 << 30);
  const auto issue = [&](int ci) {
    const int st = ci % kAttnStages;
    unsigned char* kd = sm + (size_t)st * Geo::kStage;
    unsigned char* vd = kd + kAttnCh * Geo::kRow;
    const int q0 = t0 + ci * kAttnCh, m = min(kAttnCh, len - ci * kAttnCh);
    const int pg0 = q0 / bs, npg = (q0 + m - 1) / bs - pg0 + 1;
    uint32_t bytes = 0;
    unsigned long long vmask = 0ull;
    for (int i = lane; i < npg; i += kWarp) {
      const int s0 = max(q0, (pg0 + i) * bs);
      const int s1 = (int)min((long long)(q0 + m), (long long)(pg0 + i + 1) * bs);
      if (a.kv.slot_ok(b, s0)) {
        bytes += 2u * (uint32_t)(s1 - s0) * (uint32_t)Geo::kRow;
        const int nrun = s1 - s0;
        vmask |= (nrun >= 64 ? ~0ull : ((1ull << nrun) - 1ull)) << (s0 - q0);
      } else if (a.status) {
        atomicCAS(a.status, 0, (int)NC_ERR_POSITION);
      }
    }
    bytes = __reduce_add_sync(0xFFFFFFFFu, bytes);
    const uint32_t vlo = __reduce_or_sync(0xFFFFFFFFu, (uint32_t)vmask);
    const uint32_t vhi = __reduce_or_sync(0xFFFFFFFFu, (uint32_t)(vmask >> 32));
    if (lane == 0) {
      valid_s[st] = ((unsigned long long)vhi << 32) | vlo;
      issued_s = ci + 1;
      mbar_expect_tx(&full[st], bytes);
    }
    __syncwarp();
    for (int i = lane; i < npg; i += kWarp) {
      const int s0 = max(q0, (pg0 + i) * bs);
      const int s1 = (int)min((long long)(q0 + m), (long long)(pg0 + i + 1) * bs);
      if (a.kv.slot_ok(b, s0)) {
        const size_t off = a.kv.offset(a.layer, b, g, s0) * ES;
        const uint32_t nb = (uint32_t)(s1 - s0) * (uint32_t)Geo::kRow;
        bulk_g2s(kd + (size_t)(s0 - q0) * Geo::kRow, static_cast<const char*>(a.kv.k) + off, nb,
                 &full[st]);
        bulk_g2s(vd + (size_t)(s0 - q0) * Geo::kRow, static_cast<const char*>(a.kv.v) + off, nb,
                 &full[st]);
      }
    }
  };
  // the copies depend on the positions only: issue them before the q work
  if (warp == 0)
    for (int ci = 0; ci < nch && ci < kAttnStages; ++ci) issue(ci);

  if constexpr (ROPE) {
    // warp w < G: query head w; then (split 0 only) warp G % 8 the key and
    // the next warp the value. Lane l holds dims l + 32 j: a RoPE pair
    // (i, i + D/2) sits in one lane. Same arithmetic as k_rope_qkv.
    constexpr int EJ = D / kWarp;
    const float* src = a.qkv + (size_t)b * (a.Hq + 2 * a.Hkv) * D;
    for (int hh = warp; hh < G + 2; hh += kAttnWarps) {
      if (hh >= G && c != 0) continue;  // warp-uniform
      const float* v = src + (size_t)(hh < G ? g * G + hh : (hh == G ? a.Hq + g : a.Hq + a.Hkv + g)) * D;
      float e[EJ];
#pragma unroll
      for (int j = 0; j < EJ; ++j) e[j] = v[lane + 32 * j];
      const uint16_t* gain = hh < G ? a.g_q : (hh == G ? a.g_k : nullptr);
      if (gain) {  // per-head RMSNorm over D
        float ss = 0.f;
#pragma unroll
        for (int j = 0; j < EJ; ++j) ss = fmaf(e[j], e[j], ss);
        ss = warp_sum(ss);
        const float r = 1.f / sqrtf(ss / (float)D + a.eps);
#pragma unroll
        for (int j = 0; j < EJ; ++j) e[j] = (e[j] * r) * bf16_to_f32(gain[lane + 32 * j]);
      }
      if (hh <= G) {
#pragma unroll
        for (int j = 0; j < EJ / 2; ++j) {
          const float angle = __fmul_rn((float)pos, a.inv_freq[lane + 32 * j]);
          float sn, cs;
          sincosf(angle, &sn, &cs);
          const float x0 = e[j], x1 = e[j + EJ / 2];
          e[j] = __fsub_rn(__fmul_rn(x0, cs), __fmul_rn(x1, sn));
          e[j + EJ / 2] = __fadd_rn(__fmul_rn(x1, cs), __fmul_rn(x0, sn));
        }
      }
      if (hh >= G && KV16)  // k and v as the cache stores them
#pragma unroll
        for (int j = 0; j < EJ; ++j) e[j] = bf16_to_f32(f32_to_bf16(e[j]));
      float* dst = hh < G ? q_s[hh] : (hh == G ? kn_s : vn_s);
#pragma unroll
      for (int j = 0; j < EJ; ++j) dst[lane + 32 * j] = e[j];
      if (hh >= G && pos_ok) {
        const size_t off = a.kv.offset(a.layer, b, g, pos);
        void* cache = hh == G ? a.kv.k : a.kv.v;
#pragma unroll
        for (int j = 0; j < EJ; ++j) kv_store<KV16>(cache, off + lane + 32 * j, e[j]);
      }
    }
  }
  __syncthreads();  // the rotated heads in shared memory

  // The scores' layout. Sliced (head size 64, groups of 8): the 8 dims of
  // slice lane % 8 of every query head; otherwise dims [lane E, lane E + E)
  // of every query head, the 32 lanes' partial dots summed over the warp.
  constexpr bool SLICED = D == 64 && GM == 8;
  constexpr int QE = SLICED ? 8 : E;
  float qr[GM][QE];
#pragma unroll
  for (int h = 0; h < GM; ++h)
#pragma unroll
    for (int e = 0; e < QE; ++e) {
      const int d = SLICED ? slice_dim<KV16>(lane % GM, e) : lane * E + e;
      qr[h][e] = h >= G ? 0.f
                 : ROPE ? q_s[ROPE ? h : 0][d]
                        : a.q[((size_t)b * a.Hq + g * G + h) * D + d];
    }


  // Each warp keeps its own online-softmax state over the positions it
  // scores: (m, l) of head lane % GM in every lane of that head's lane group,
  // acc[h][e] of dims lane E + e of every head. No block barrier inside a
  // chunk; the warps' states are combined once at the end.
  const float scale = 1.f / sqrtf((float)D);
  const int hl = lane % GM;  // the head whose (m, l) this lane carries
  float m_run = -INFINITY, l_run = 0.f;
  float acc[GM][E];
#pragma unroll
  for (int h = 0; h < GM; ++h)
#pragma unroll
    for (int e = 0; e < E; ++e) acc[h][e] = 0.f;
  if constexpr (ROPE) {
    if (c == 0 && pos_ok && warp == 0) {  // the new position opens warp 0 of split 0
      for (int h = 0; h < G; ++h) {
        float sc = 0.f;
#pragma unroll
        for (int j = 0; j < D / kWarp; ++j) sc = fmaf(q_s[h][lane + 32 * j], kn_s[lane + 32 * j], sc);
        sc = warp_sum(sc);
        if (hl == h) {
          m_run = sc * scale;
          l_run = 1.f;
        }
#pragma unroll
        for (int hh = 0; hh < GM; ++hh)
          if (hh == h)
#pragma unroll
            for (int e = 0; e < E; ++e) acc[hh][e] = vn_s[lane * E + e];
      }
    }
  }
  // No block barrier between chunks: each warp takes the chunks in order,
  // and the warp that finishes a stage's chunk last refills the stage with
  // chunk ci + kAttnStages (a shared-memory count of the warps still at it).
  // A chunk that never lands ends the scan of the warp that waited for it;
  // the CTA then keeps no partial.
  const uint64_t deadline = global_timer() + kAttnWaitNs;
  for (int ci = 0; ci < nch; ++ci) {
    const int st = ci % kAttnStages;
    bool late = false;
    while (!mbar_try_wait(&full[st], (uint32_t)(ci / kAttnStages) & 1u))
      if (global_timer() > deadline || *reinterpret_cast<volatile int*>(&abort_s)) {
        late = true;
        break;
      }
    if (late) {
      if (lane == 0) abort_s = 1;
      break;
    }
    const unsigned char* kc = sm + (size_t)st * Geo::kStage;
    const unsigned char* vc = kc + kAttnCh * Geo::kRow;
    const int m = min(kAttnCh, len - ci * kAttnCh);
    const unsigned long long valid = valid_s[st];
    for (int p0 = warp * NP; p0 < m; p0 += kAttnWarps * NP) {
      // scores of NP positions x GM heads; lane i ends with value i =
      // (position i / GM, head i % GM)
      float v[SLICED ? GM : GM * NP];
      if constexpr (SLICED) {
        // a row past the chunk's end is stale shared memory inside the
        // stage; its score is masked below
        float kf[8];
        load_slice<KV16>(kc + (size_t)(p0 + lane / GM) * Geo::kRow, lane % GM, kf);
#pragma unroll
        for (int h = 0; h < GM; ++h) {
          float d = 0.f;
#pragma unroll
          for (int e = 0; e < 8; ++e) d = fmaf(qr[h][e], kf[e], d);
          v[h] = d;
        }
        group_sum_scatter<GM>(v);
      } else {
#pragma unroll
        for (int p = 0; p < NP; ++p) {
          float kf[E];
          load_row<E, KV16>(kc + (size_t)(p0 + p) * Geo::kRow + (size_t)lane * E * ES, kf);
#pragma unroll
          for (int h = 0; h < GM; ++h) {
            float d = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) d = fmaf(qr[h][e], kf[e], d);
            v[p * GM + h] = d;
          }
        }
        warp_sum_many<GM * NP>(v);
      }
      const int t = p0 + lane / GM;
      // a block-table hole (no row copied) scores -inf
      const float sc = hl < G && t < m && ((valid >> t) & 1ull) ? v[0] * scale : -INFINITY;
      // this warp's running max and sum of head hl: lanes hl, hl + GM, ...
      float mx = sc;
#pragma unroll
      for (int o = GM; o < kWarp; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
      const float m_new = fmaxf(m_run, mx);
      const float pr = sc == -INFINITY ? 0.f : expf(sc - m_new);
      float ls = pr;
#pragma unroll
      for (int o = GM; o < kWarp; o <<= 1) ls += __shfl_xor_sync(0xFFFFFFFFu, ls, o);
      const float r = m_run == -INFINITY ? 0.f : expf(m_run - m_new);
      l_run = fmaf(l_run, r, ls);
      m_run = m_new;
#pragma unroll
      for (int h = 0; h < GM; ++h) {
        const float rh = __shfl_sync(0xFFFFFFFFu, r, h);
#pragma unroll
        for (int e = 0; e < E; ++e) acc[h][e] *= rh;
      }
      // values: position p's weights come from lanes p GM .. p GM + GM - 1;
      // a hole (no row copied, weight 0) left its row unwritten, so its
      // value is replaced, not multiplied: only steps with a hole take that
      // path (the mask is the chunk's, the test warp-uniform)
      const unsigned long long stepm = (NP >= 64 ? ~0ull : ((1ull << NP) - 1ull)) << p0;
      const bool hole = (valid & stepm) != stepm;
      if (hole) {
#pragma unroll
        for (int p = 0; p < NP; ++p) {
          if (p0 + p >= m) break;  // warp-uniform
          float vf[E];
          load_row<E, KV16>(vc + (size_t)(p0 + p) * Geo::kRow + (size_t)lane * E * ES, vf);
#pragma unroll
          for (int h = 0; h < GM; ++h) {
            const float w = __shfl_sync(0xFFFFFFFFu, pr, p * GM + h);
#pragma unroll
            for (int e = 0; e < E; ++e) acc[h][e] = fmaf(w, w == 0.f ? 0.f : vf[e], acc[h][e]);
          }
        }
      } else {
#pragma unroll
        for (int p = 0; p < NP; ++p) {
          if (p0 + p >= m) break;  // warp-uniform
          float vf[E];
          load_row<E, KV16>(vc + (size_t)(p0 + p) * Geo::kRow + (size_t)lane * E * ES, vf);
#pragma unroll
          for (int h = 0; h < GM; ++h) {
            const float w = __shfl_sync(0xFFFFFFFFu, pr, p * GM + h);
#pragma unroll
            for (int e = 0; e < E; ++e) acc[h][e] = fmaf(w, vf[e], acc[h][e]);
          }
        }
      }
    }
    // this warp is done with the stage; the last one refills it
    __syncwarp();
    int last = 0;
    if (lane == 0) {
      __threadfence_block();  // this warp's reads of the stage come first
      last = atomicSub(&left_s[st], 1) == 1;
      if (last) {
        left_s[st] = kAttnWarps;
        __threadfence_block();
      }
    }
    last = __shfl_sync(0xFFFFFFFFu, last, 0);
    if (last && ci + kAttnStages < nch) issue(ci + kAttnStages);
  }
  __syncthreads();
  if (abort_s) {
    // abandoned: let the copies already issued land (bounded) before the
    // shared memory is reused or released; this split contributes nothing
    if (tid == 0) {
      if (a.status) atomicCAS(a.status, 0, (int)NC_ERR_TIMEOUT);
      const uint64_t dl = global_timer() + kAttnWaitNs;
      const int is = issued_s;
      for (int ci = is > kAttnStages ? is - kAttnStages : 0; ci < is; ++ci)
        while (!mbar_try_wait(&full[ci % kAttnStages], (uint32_t)(ci / kAttnStages) & 1u))
          if (global_timer() > dl) break;
    }
    m_run = -INFINITY;
    l_run = 0.f;
#pragma unroll
    for (int h = 0; h < GM; ++h)
#pragma unroll
      for (int e = 0; e < E; ++e) acc[h][e] = 0.f;
  }
  // combine the warps' states into the CTA's partial (the stages are spent)
  __syncthreads();
  float* wacc = reinterpret_cast<float*>(sm);        // [warps][GM][D]
  float* wm = wacc + kAttnWarps * GM * D;            // [warps][GM]
  float* wl = wm + kAttnWarps * GM;                  // [warps][GM]
  if (lane < GM) {
    wm[warp * GM + lane] = m_run;
    wl[warp * GM + lane] = l_run;
  }
#pragma unroll
  for (int h = 0; h < GM; ++h)
#pragma unroll
    for (int e = 0; e < E; ++e) wacc[(warp * GM + h) * D + lane * E + e] = acc[h][e];
  __syncthreads();
  for (int i = tid; i < G * D; i += kAttnThreads) {
    const int h = i / D, d = i % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, wm[w * GM + h]);
    float num = 0.f, den = 0.f;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) {
      const float mw = wm[w * GM + h];
      const float f = mw == -INFINITY ? 0.f : expf(mw - M);
      num = fmaf(wacc[(w * GM + h) * D + d], f, num);
      den = fmaf(wl[w * GM + h], f, den);
    }
    float* ph = part + ((size_t)c * G + h) * (D + 2);
    ph[2 + d] = num;
    if (d == 0) {  // (-inf, 0) when the split saw no position
      ph[0] = M;
      ph[1] = den;
    }
  }

  // the last CTA of (b, g) merges the S partials of its G heads
  __threadfence();
  __syncthreads();
  unsigned int* ticket = a.tickets + (size_t)b * a.Hkv + g;
  if (tid == 0) last_s = atomicAdd(ticket, 1u) == (unsigned int)(S - 1);
  __syncthreads();
  if (!last_s) return;
  __threadfence();
  // The values of the first kMB splits are loaded up front, so their round
  // trip overlaps the (m, l) pass.
  constexpr int kMB = 16;
  constexpr int NIT = (GM * D + kAttnThreads - 1) / kAttnThreads;  // (head, dim) items per thread
  float av[NIT][kMB];
#pragma unroll
  for (int it = 0; it < NIT; ++it) {
    const int i = tid + it * kAttnThreads, h = i / D, d = i % D;
    const float* ph = part + (size_t)h * (D + 2) + 2 + d;
#pragma unroll
    for (int cc = 0; cc < kMB; ++cc)
      av[it][cc] = h < G && cc < S ? __ldcg(ph + (size_t)cc * cs) : 0.f;
  }
  float* w_s = reinterpret_cast<float*>(sm);  // [GM][kMaxSplits]; the stages are spent
  for (int h = warp; h < G; h += kAttnWarps) {
    const float* ph = part + (size_t)h * (D + 2);
    float M = -INFINITY;
    for (int cc = lane; cc < S; cc += kWarp) M = fmaxf(M, __ldcg(ph + (size_t)cc * cs));
    M = warp_max(M);
    float den = 0.f;
    for (int cc = lane; cc < S; cc += kWarp) {
      const float mc = __ldcg(ph + (size_t)cc * cs);
      const float w = mc == -INFINITY ? 0.f : expf(mc - M);
      w_s[h * kMaxSplits + cc] = w;
      den = fmaf(__ldcg(ph + (size_t)cc * cs + 1), w, den);
    }
    den = warp_sum(den);
    if (lane == 0) den_s[h] = den;
  }
  __syncthreads();
#pragma unroll
  for (int it = 0; it < NIT; ++it) {
    const int i = tid + it * kAttnThreads, h = i / D, d = i % D;
    if (h >= G) continue;
    const float* ph = part + (size_t)h * (D + 2) + 2 + d;
    float num = 0.f;
#pragma unroll
    for (int cc = 0; cc < kMB; ++cc)
      if (cc < S) num = fmaf(av[it][cc], w_s[h * kMaxSplits + cc], num);
#pragma unroll 8
    for (int cc = kMB; cc < S; ++cc) num = fmaf(__ldcg(ph + (size_t)cc * cs), w_s[h * kMaxSplits + cc], num);
    a.out[((size_t)b * a.Hq + g * G + h) * D + d] = num / den_s[h];
  }
  if (tid == 0) *ticket = 0u;  // ready for the next launch
}

template <int D, bool KV16>
static int attn_occupancy() {
  static const int occ = [] {
    int n = 0;
    const auto kern = k_attn_split<D, 8, KV16, true>;  // the larger static shared memory
    if (ensure_smem<k_attn_split<D, 8, KV16, true>>() != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kAttnThreads, AttnGeo<D, KV16>::kSmem) !=
            cudaSuccess ||
        n < 1)
      n = 1;
    return n;
  }();
  return occ;
}

template <int D, int GM, bool KV16, bool ROPE>
static cudaError_t attn_launch(const AttnArgs& a, cudaStream_t s) {
  cudaError_t e = ensure_smem<k_attn_split<D, GM, KV16, ROPE>>();
  if (e != cudaSuccess) return e;
  return launch_pdl(k_attn_split<D, GM, KV16, ROPE>, dim3(a.splits, a.Hkv),
                    dim3(kAttnThreads), AttnGeo<D, KV16>::kSmem, s, a);
}

template <int D, int GM, bool KV16>
static cudaError_t attn_split(const AttnArgs& a, cudaStream_t s) {
  return a.qkv ? attn_launch<D, GM, KV16, true>(a, s) : attn_launch<D, GM, KV16, false>(a, s);
}

template <int D>
static cudaError_t attn_d(const AttnArgs& a, cudaStream_t s) {
  const int G = a.Hq / a.Hkv;
  const bool h = a.kv.bf16;
  if (G <= 1) return h ? attn_split<D, 1, true>(a, s) : attn_split<D, 1, false>(a, s);
  if (G <= 2) return h ? attn_split<D, 2, true>(a, s) : attn_split<D, 2, false>(a, s);
  if (G <= 4) return h ? attn_split<D, 4, true>(a, s) : attn_split<D, 4, false>(a, s);
  return h ? attn_split<D, 8, true>(a, s) : attn_split<D, 8, false>(a, s);
}

cudaError_t launch_attn(const AttnArgs& a, cudaStream_t s) {
  if (a.splits < a.B || a.splits > kMaxSplits || a.B > kWarp) return cudaErrorInvalidValue;
  return a.D == 64 ? attn_d<64>(a, s) : attn_d<128>(a, s);
}

}  // namespace nc
