// persistent.cu -- the whole decode step as one persistent kernel.
//
// At batch 1 the step is a chain of ~5 dependent phases per layer (QKV,
// attention, o-proj, gate|up, down; nanocompile's 13 kernels per block fused
// down), each moving only 1-17 MB: as separate launches it is bound by
// launch latency and per-kernel ramp-up, not by HBM. Here one CTA per SM runs
// the whole step:
//
//  * Weights do not depend on activations, so warp 0 of every CTA streams the
//    CTA's future weight tiles -- its rows of every projection of every layer,
//    then of the LM head, in the order the consumers will use them -- into a
//    ring of shared-memory slots with TMA bulk copies (cp.async.bulk, mbarrier
//    completion). HBM stays busy while the dependency chain advances.
//  * Warps 1..11 consume: per phase they gather the phase's input vector,
//    compute the RMSNorm where one precedes the projection, and reduce their
//    tile rows against it; the epilogue (bias, residual, SiLU * up, logits
//    and arg-max) runs on the reducing lane (Tang section 2.3).
//  * Phases hand values over through 64-bit global words holding (value,
//    epoch): a reader spins until the epoch of the word equals the one it
//    expects, so no separate flag or grid barrier is needed. Epochs carry the
//    step sequence number, so values of an earlier step never match.
//  * Attention runs one CTA per (sequence, kv head, position split): RoPE
//    (and q/k norm) of its heads, the K/V append, and the online-softmax scan
//    over the split's cached positions in chunks (Tang section 2.2, the
//    monoid on (m, l, acc)). Long caches are split over the whole grid; the
//    last split of each (sequence, kv head) to finish merges the partials
//    (section 2.5: a split is valid for any associative monoid).
//  * Every spin is bounded by %globaltimer. On expiry the CTA writes
//    NC_ERR_TIMEOUT to the status word, stops issuing copies, waits (bounded)
//    for the copies in flight and leaves through the final ticket, so the
//    kernel always ends.
//
// The launch is cooperative: all CTAs must be resident together.
#include <cuda_runtime.h>
#include <math.h>
#include <stdlib.h>

#include "kernels.h"
#include "persistent.h"

namespace nc {

constexpr int kPThreads = 384;
constexpr int kPConsumerWarps = kPThreads / kWarp - 1;
constexpr int kPConsumerThreads = kPConsumerWarps * kWarp;
constexpr int kPhasesPerLayer = 5;
constexpr int kUnitsPerWarp = 4;  // output units (rows, gate|up pairs) a warp takes per tile
// ... at batch BT: fewer at larger batches, where every unit holds BT sums
__host__ __device__ constexpr int units_per_warp(int BT) { return BT == 1 ? 4 : (BT == 2 ? 2 : 1); }
__host__ __device__ constexpr int bt_of_batch(int B) { return B <= 1 ? 1 : (B <= 2 ? 2 : 4); }
enum PhaseKind : int { kQKV = 0, kATTN = 1, kOPROJ = 2, kGU = 3, kDOWN = 4, kHEAD = 5 };

// ------------------------------------------------------------------ PTX helpers
// 16-byte asynchronous copy global -> shared (L2, not L1: the words may have
// been written by other SMs); completion by cp_async_wait_all.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ uint64_t ld_word(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_word(uint64_t* p, float v, uint32_t epoch) {
  const uint64_t w = (static_cast<uint64_t>(epoch) << 32) | __float_as_uint(v);
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}

// Rows of one phase given to a CTA and the tile shape used to stream them.
struct Rows {
  int r0, r1, R;          // rows [r0, r1), R rows per tile
  int K;                  // elements per row
  const uint16_t* m0;     // matrix (gate block for gate|up)
  const uint16_t* m1;     // up block, or null
};

// ------------------------------------------------------------------ shared state
struct PShared {
  // residual words (value, epoch) of the rows the o-proj/down epilogue adds
  // to, from row r0 rounded down to even; raw bf16 QKV bias of this CTA's
  // rows, from r0 rounded down to a multiple of 8 (both copied 16 bytes at a
  // time while the phase input is polled)
  alignas(16) uint64_t xoldw[kPMaxBatch][kPMaxRows + 2];
  alignas(16) uint16_t biasr[kPMaxRows + 16];
  PLayer layers[kPMaxLayers];  // per-layer pointers, read once per step
  Rows rows[kHEAD + 1];        // this CTA's rows and tile shape per phase kind
  int nsplit[kPMaxBatch];      // attention: position splits per sequence
  int item0[kPMaxBatch + 1];   // attention: first item of each sequence (items = sum Hkv * splits)
  uint64_t full[kMaxSlots];
  uint64_t empty[kMaxSlots];
  int abort;        // set once a bounded wait expired in this CTA
  int merge;        // attention: this CTA's split arrived last and merges
  unsigned issued;  // tiles the producer issued
  int pos[kPMaxBatch];
  float rope_cs[kPMaxBatch][64], rope_sn[kPMaxBatch][64];  // RoPE cos / sin at each position (D/2 <= 64)
  int tok[kPMaxBatch];
  float rn[kPMaxBatch];
  float red[kPConsumerWarps][kPMaxBatch];
  unsigned long long best[kPConsumerWarps][kPMaxBatch];
  float kred[2][kUnitsPerWarp * kPConsumerWarps][2 * kPMaxBatch];  // k-segment partials, 2 buffers
  bool last;
};

// Deadline-bounded wait context for one CTA.
struct Spin {
  uint64_t deadline;
  int* abort;
  int* status;
  __device__ bool expired() {
    if (*reinterpret_cast<volatile int*>(abort)) return true;
    if (global_timer() > deadline) {
      atomicExch(abort, 1);
      if (status) atomicCAS(status, 0, (int)NC_ERR_TIMEOUT);
      return true;
    }
    return false;
  }
};

// Spin until the word at p carries `epoch`; returns its value (0 on abort).
__device__ __forceinline__ float ll_get(const uint64_t* p, uint32_t epoch, Spin& sp) {
  uint64_t w = ld_word(p);
  int n = 0;
  while (static_cast<uint32_t>(w >> 32) != epoch) {
    if ((++n & 63) == 0 && sp.expired()) return 0.f;
    w = ld_word(p);
  }
  return __uint_as_float(static_cast<uint32_t>(w));
}

// Words w[u] = *addr(u) (bit u of `valid` set) were loaded once; re-load, in rounds
// with every stale word's load in flight together, until all carry `epoch`.
// One round costs one memory round trip however many words are stale (a
// word-by-word re-poll would pay one per word). On expiry the stale words
// read as 0.
constexpr unsigned kPollPauseNs = 128;
template <int N, class Addr>
__device__ __forceinline__ void ll_settle(const Addr& addr, uint32_t valid, uint32_t epoch,
                                          uint64_t (&w)[N], Spin& sp) {
  for (int round = 1;; ++round) {
    bool stale = false;
#pragma unroll
    for (int u = 0; u < N; ++u)
      if (((valid >> u) & 1u) && static_cast<uint32_t>(w[u] >> 32) != epoch) stale = true;
    if (!stale) return;
    if ((round & 15) == 0 && sp.expired()) {
#pragma unroll
      for (int u = 0; u < N; ++u)
        if (((valid >> u) & 1u) && static_cast<uint32_t>(w[u] >> 32) != epoch) w[u] = 0;
      return;
    }
    // a short pause before the next round, longer once the wait is long:
    // every consumer thread of every CTA polls at once, and back-to-back
    // rounds crowd the L2 the weight stream goes through
    __nanosleep(round < 8 ? kPollPauseNs : 4 * kPollPauseNs);
#pragma unroll
    for (int u = 0; u < N; ++u)
      if (((valid >> u) & 1u) && static_cast<uint32_t>(w[u] >> 32) != epoch) w[u] = ld_word(addr(u));
  }
}

// Read `count` words p[0], p[stride], ... (count <= kLLBatch): all loads in
// flight at once, then settle the stale ones.
constexpr int kLLBatch = 16;
__device__ __forceinline__ void ll_get_batch(const uint64_t* p, int stride, int count,
                                             uint32_t epoch, float* out, Spin& sp) {
  uint64_t w[kLLBatch];
  const auto addr = [p, stride](int u) { return p + (size_t)u * stride; };
#pragma unroll
  for (int u = 0; u < kLLBatch; ++u)
    if (u < count) w[u] = ld_word(addr(u));
  ll_settle<kLLBatch>(addr, (1u << count) - 1u, epoch, w, sp);
#pragma unroll
  for (int u = 0; u < kLLBatch; ++u)
    if (u < count) out[u] = __uint_as_float(static_cast<uint32_t>(w[u]));
}

__device__ __forceinline__ uint32_t epoch_of(uint32_t seq, int phase) {
  return ((seq & 0xFFFFFFu) << 8) | static_cast<uint32_t>(phase);
}

// Position in the slot ring: tiles passed, the slot, and the parity of the
// slot's current fill. Producer and consumers walk the same sequence.
struct RingPos {
  uint32_t n = 0;
  int s = 0;
  uint32_t par = 0;
  __device__ __forceinline__ void next(int nslots) {
    ++n;
    if (++s == nslots) {
      s = 0;
      par ^= 1u;
    }
  }
};

// Bounded wait for phase `par` of an mbarrier; false once the CTA gave up.
__device__ __forceinline__ bool ring_wait(uint64_t* bar, uint32_t par, Spin& sp) {
  int k = 0;
  while (!mbar_try_wait(bar, par))
    if ((++k & 15) == 0 && sp.expired()) return false;
  return true;
}


// Cached positions sequence b attends to in this step (slot pos itself comes
// from the step's own k/v): pos, or 0 when pos is outside the cache.
__device__ __forceinline__ int cached_positions(const PersistArgs& a, int b, int pos) {
  return a.kv.slot_ok(b, pos) ? pos : 0;
}

// Attention work plan: the cached positions of each (sequence, kv head) are
// split into up to kPMaxSplits ranges of at least kAttnSplitMin positions,
// each range one item on its own CTA (split-K over positions; the last split
// to finish merges the partial softmax states). Items of all sequences
// together stay within the grid, so a long cache streams through every SM.
// Returns the item count.
constexpr int kAttnSplitMin = 128;  // one chunk: shorter scans are not split
__device__ int attn_plan(const PersistArgs& a, int grid, int (&nsplit)[kPMaxBatch],
                         int (&item0)[kPMaxBatch + 1]) {
  int cap = grid / (a.B * a.Hkv);
  if (cap > kPMaxSplits) cap = kPMaxSplits;
  if (cap < 1) cap = 1;
  item0[0] = 0;
  for (int b = 0; b < kPMaxBatch; ++b) {
    int ns = 0;
    if (b < a.B) {
      const int np = cached_positions(a, b, a.positions[b]);
      ns = (np + kAttnSplitMin - 1) / kAttnSplitMin;
      if (ns > cap) ns = cap;
      if (ns < 1) ns = 1;
    }
    nsplit[b] = ns;
    item0[b + 1] = item0[b] + a.Hkv * ns;
  }
  return item0[kPMaxBatch];
}

// Item `it` of the plan: sequence b, kv head g, split sp of ns, and its range
// of cached positions [p0, p1).
struct AttnItem {
  int b, g, sp, ns, p0, p1;
};
__device__ __forceinline__ AttnItem attn_item_of(const PShared& S, int Hkv, int it) {
  AttnItem t{0, 0, 0, 1, 0, 0};
  int b = 0;
  while (b + 1 < kPMaxBatch && it >= S.item0[b + 1]) ++b;
  const int r = it - S.item0[b];
  t.b = b;
  t.ns = S.nsplit[b];
  t.g = r / t.ns;
  t.sp = r % t.ns;
  return t;
}

// CTAs that run attention items (item i on CTA i) and hold no o-proj rows.
__device__ __forceinline__ int attn_ctas(const PersistArgs& a, int grid) {
  int ns[kPMaxBatch], i0[kPMaxBatch + 1];
  const int items = attn_plan(a, grid, ns, i0);
  return items < grid / 2 ? items : 0;
}

// The row range and tile shape of one phase kind for CTA `cta` (the same in
// every layer); the matrix pointers are left null.
__device__ Rows kind_rows(const PersistArgs& a, int kind, int cta, int grid, int slot_bytes) {
  Rows r{0, 0, 1, 0, nullptr, nullptr};
  int N = 0;
  bool pair = false;
  switch (kind) {
    case kQKV: N = a.nqkv; r.K = a.H; break;
    case kOPROJ: N = a.H; r.K = a.Hq * a.D; break;
    case kGU: N = a.F; r.K = a.H; pair = true; break;
    case kDOWN: N = a.H; r.K = a.F; break;
    case kHEAD: N = a.V; r.K = a.H; break;
    default: return r;  // attention streams no weights
  }
  if (kind == kOPROJ) {
    // the CTAs that ran the attention items come out of it last: the o-proj
    // rows go to the others, which are idle meanwhile
    const int na = attn_ctas(a, grid);
    if (cta < na) return r;
    cta -= na;
    grid -= na;
  }
  r.r0 = (int)(((long long)cta * N) / grid);
  r.r1 = (int)(((long long)(cta + 1) * N) / grid);
  const int row_bytes = r.K * 2 * (pair ? 2 : 1);
  int rmax = slot_bytes / row_bytes;
  const int umax = units_per_warp(bt_of_batch(a.B)) * kPConsumerWarps;
  if (rmax > umax) rmax = umax;
  if (rmax < 1) rmax = 1;
  // tiles of (nearly) equal size: the fewest tiles that fit, rows spread evenly
  const int nr = r.r1 - r.r0;
  const int nt = nr > 0 ? (nr + rmax - 1) / rmax : 1;
  r.R = nr > 0 ? (nr + nt - 1) / nt : 1;
  return r;
}

// Rows of phase `ph` for this CTA: the per-kind shape computed once per step
// (kept in shared memory) plus this layer's matrices.
__device__ __forceinline__ Rows phase_rows(const PersistArgs& a, const PShared& S, int ph) {
  const int L = a.L;
  const int kind = ph == kPhasesPerLayer * L ? kHEAD : ph % kPhasesPerLayer;
  Rows r = S.rows[kind];
  if (kind == kHEAD) {
    r.m0 = a.head;
  } else {
    const PLayer& P = S.layers[ph / kPhasesPerLayer];
    switch (kind) {
      case kQKV: r.m0 = P.w_qkv; break;
      case kOPROJ: r.m0 = P.w_o; break;
      case kGU: r.m0 = P.w_gu; r.m1 = P.w_gu + (size_t)a.F * a.H; break;
      case kDOWN: r.m0 = P.w_d; break;
      default: break;
    }
  }
  return r;
}

// ------------------------------------------------------------------ producer
template <bool KV16>
__device__ bool produce_kv(const PersistArgs& a, PShared& S, char* ring, int slot_bytes,
                           int nslots, int layer, int b, int g, int p0, int p1, RingPos& rp,
                           Spin& sp);

template <bool KV16>
__device__ void producer(const PersistArgs& a, PShared& S, char* ring, int slot_bytes, int nslots,
                         Spin& sp) {
  const int nph = kPhasesPerLayer * a.L + 1;
  RingPos rp;
  for (int ph = 0; ph < nph; ++ph) {
    if (ph < kPhasesPerLayer * a.L && ph % kPhasesPerLayer == kATTN) {
      for (int it = blockIdx.x; it < S.item0[kPMaxBatch]; it += gridDim.x) {
        AttnItem t = attn_item_of(S, a.Hkv, it);
        const int np = cached_positions(a, t.b, S.pos[t.b]);
        t.p0 = (int)(((long long)t.sp * np) / t.ns);
        t.p1 = (int)(((long long)(t.sp + 1) * np) / t.ns);
        if (!produce_kv<KV16>(a, S, ring, slot_bytes, nslots, ph / kPhasesPerLayer, t.b, t.g,
                              t.p0, t.p1, rp, sp))
          return;
      }
      continue;
    }
    const Rows r = phase_rows(a, S, ph);
    for (int row = r.r0; row < r.r1; row += r.R) {
      const int n = min(r.R, r.r1 - row);
      const int s = rp.s;
      if (rp.n >= (uint32_t)nslots && !ring_wait(&S.empty[s], rp.par ^ 1u, sp)) return;
      if (*reinterpret_cast<volatile int*>(&S.abort)) return;
      const uint32_t bytes = (uint32_t)n * r.K * 2;
      char* dst = ring + (size_t)s * slot_bytes;
      mbar_expect_tx(&S.full[s], bytes * (r.m1 ? 2u : 1u));
      bulk_g2s(dst, r.m0 + (size_t)row * r.K, bytes, &S.full[s]);
      if (r.m1) bulk_g2s(dst + bytes, r.m1 + (size_t)row * r.K, bytes, &S.full[s]);
      rp.next(nslots);
      S.issued = rp.n;
    }
  }
}

// ------------------------------------------------------------------ consumer helpers
// Named barrier over the consumer warps only (the producer never joins).
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kPConsumerThreads) : "memory");
}
// The same barrier with an OR reduction: every consumer thread gets the same
// answer, so a decision taken on it keeps the named barriers uniform.
__device__ __forceinline__ bool consumer_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 1, %2, p;\n"
      " selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(kPConsumerThreads)
      : "memory");
  return r != 0;
}

// Where element i of an input row of n (a multiple of 8) sits in shared
// memory: the first four elements of every 8-element chunk in the lower half,
// the last four in the upper half. A lane reading chunk c then reads two
// float4 at a 16-byte stride across the warp, which no two lanes of a load
// phase share a bank group in.
__device__ __forceinline__ int xs_at(int i, int n) {
  return ((i & 4) ? (n >> 1) : 0) + ((i >> 3) << 2) + (i & 3);
}

// Gather the phase input [B][n] (sequences src_stride words apart) from
// epoch-tagged words into xs (fp32);
// with gamma, also compute the RMSNorm factor per sequence and scale xs.
// The gains are copied asynchronously before the words are polled, so their
// round trip overlaps the wait for the previous phase.
template <int BT>
__device__ __noinline__ void gather_input(const PersistArgs& a, const uint64_t* src, int n,
                                          size_t src_stride, uint32_t epoch,
                                          const uint16_t* embed_rows, const uint16_t* gamma,
                                          Spin& sp) {
  // shared-memory pointers are derived from the dynamic shared array here, so
  // the compiler addresses them as shared, not generic
  extern __shared__ __align__(128) char smem[];
  PShared& S = *reinterpret_cast<PShared*>(smem);
  float* xs = reinterpret_cast<float*>(smem + a.xs_offset);
  // the gains go to the attention scratch (idle during a projection phase),
  // copied asynchronously while the input words are polled
  uint16_t* gs = reinterpret_cast<uint16_t*>(smem + a.attn_offset);
  const int nb = a.B;
  const float eps = a.eps;
  const int ct = threadIdx.x - kWarp, warp = ct / kWarp, lane = ct % kWarp;
  const bool gain_smem = gamma && n * 2 <= a.attn_bytes;
  if (gain_smem) {
    for (int c = ct; c < n / 8; c += kPConsumerThreads) cp_async16(gs + 8 * c, gamma + 8 * c);
    cp_async_commit();
  }
#pragma unroll 1
  for (int b = 0; b < BT; ++b) {
    float ss = 0.f;
    for (int i0 = ct; i0 < n; i0 += kLLBatch * kPConsumerThreads) {
      const int count = min(kLLBatch, (n - i0 + kPConsumerThreads - 1) / kPConsumerThreads);
      float v[kLLBatch];
      if (b >= nb) {
#pragma unroll
        for (int u = 0; u < kLLBatch; ++u) v[u] = 0.f;
      } else if (embed_rows) {
#pragma unroll
        for (int u = 0; u < kLLBatch; ++u)
          if (u < count)
            v[u] = bf16_to_f32(embed_rows[(size_t)S.tok[b] * n + i0 + u * kPConsumerThreads]);
      } else {
        ll_get_batch(src + (size_t)b * src_stride + i0, kPConsumerThreads, count, epoch, v, sp);
      }
#pragma unroll
      for (int u = 0; u < kLLBatch; ++u) {
        if (u >= count) break;
        xs[b * n + xs_at(i0 + u * kPConsumerThreads, n)] = v[u];
        ss = fmaf(v[u], v[u], ss);
      }
    }
    if (gamma) {
      ss = warp_sum(ss);
      if (lane == 0) S.red[warp][b] = ss;
    }
  }
  // this thread's asynchronous copies (the caller's too) have landed; the
  // barrier makes everyone's visible
  cp_async_wait_all();
  consumer_sync();
  if (!gamma) return;
  // every thread forms the norm factors itself: no single-thread step and no
  // second barrier before the scaling
  float rn[BT];
#pragma unroll
  for (int b = 0; b < BT; ++b) {
    float t = 0.f;
    for (int w = 0; w < kPConsumerWarps; ++w) t += S.red[w][b];
    rn[b] = 1.f / sqrtf(t / (float)n + eps);
  }
  for (int i = ct; i < n; i += kPConsumerThreads) {
    const float g = bf16_to_f32(gain_smem ? gs[i] : gamma[i]);
#pragma unroll
    for (int b = 0; b < BT; ++b) {
      float* x = xs + b * n + xs_at(i, n);
      *x = (*x * rn[b]) * g;
    }
  }
  consumer_sync();
}

__device__ __forceinline__ float silu_mul_p(float g, float u) {
  const float e = expf(-fabsf(g));
  const float sig = g >= 0.f ? 1.f / (1.f + e) : e / (1.f + e);
  return (g * sig) * u;
}

// An empty asm with a memory clobber: the compiler moves no memory access
// across it (scheduling only; it emits no instruction).
__device__ __forceinline__ void compiler_fence() { asm volatile("" ::: "memory"); }

// Input chunks kept in registers per lane at batch 1 (8 floats each).
constexpr int kXReg = 4;

// 8 bf16 weights (one 16-byte chunk) times 8 fp32 inputs held in registers.
__device__ __forceinline__ float dot8r(const uint4& w, const float (&x)[8]) {
  float s = bf16_lo(w.x) * x[0];
  s = fmaf(bf16_hi(w.x), x[1], s);
  s = fmaf(bf16_lo(w.y), x[2], s);
  s = fmaf(bf16_hi(w.y), x[3], s);
  s = fmaf(bf16_lo(w.z), x[4], s);
  s = fmaf(bf16_hi(w.z), x[5], s);
  s = fmaf(bf16_lo(w.w), x[6], s);
  s = fmaf(bf16_hi(w.w), x[7], s);
  return s;
}

// U <= 4 units of a tile (rows cw, cw + W, ... from w0; with PAIR also their up
// rows, ms elements further) times the input held in registers (the lane's
// chunks lane, lane + 32, ...): per-lane partials into v[2 u + m]. All loads of
// one chunk position are independent, so the U (x 2) chains run side by side.
template <bool PAIR>
__device__ __forceinline__ void units_xreg(const uint16_t* w0, int U, int K, size_t ms,
                                           const float (&xr)[kXReg][8], int C, int lane,
                                           float (&v)[2 * kUnitsPerWarp]) {
#pragma unroll
  for (int jj = 0; jj < kXReg; ++jj) {
    const int c = lane + jj * kWarp;
    if (c < C) {
#pragma unroll
      for (int u = 0; u < kUnitsPerWarp; ++u) {
        if (u < U) {
          const uint16_t* w = w0 + (size_t)u * kPConsumerWarps * K + c * 8;
          v[2 * u] += dot8r(*reinterpret_cast<const uint4*>(w), xr[jj]);
          if (PAIR) v[2 * u + 1] += dot8r(*reinterpret_cast<const uint4*>(w + ms), xr[jj]);
        }
      }
    }
    // one chunk position's loads at a time: keeps the compiler from hoisting
    // all 32 of them (and their registers) to the top
    compiler_fence();
  }
}

// Chunks [c0, c1) of NR <= 8 rows of a tile (row r = unit r / two, matrix r % two;
// units from w0, up rows ms elements further) times the input in shared
// memory: per-lane partials into o[r]. The input chunk is loaded once for all
// NR rows.
__device__ __forceinline__ void seg_rows(const uint16_t* w0, int NR, int K, size_t ms, int two,
                                         const float* xs, int c0, int c1, int lane,
                                         float (&o)[8]) {
  int wr[8];  // element offsets of the rows (a tile holds well under 2^31 elements)
#pragma unroll
  for (int r = 0; r < 8; ++r) wr[r] = (r / two) * K + (r % two) * (int)ms;
#pragma unroll 2
  for (int c = c0 + lane; c < c1; c += kWarp) {
    float xb[8];
    const float4 p0 = *reinterpret_cast<const float4*>(xs + c * 4);
    const float4 p1 = *reinterpret_cast<const float4*>(xs + K / 2 + c * 4);
    xb[0] = p0.x; xb[1] = p0.y; xb[2] = p0.z; xb[3] = p0.w;
    xb[4] = p1.x; xb[5] = p1.y; xb[6] = p1.z; xb[7] = p1.w;
#pragma unroll
    for (int r = 0; r < 8; ++r)
      if (r < NR) o[r] += dot8r(*reinterpret_cast<const uint4*>(w0 + wr[r] + c * 8), xb);
    compiler_fence();
  }
}

// Batch > 1, whole rows: U <= UPW units (rows cw, cw + W, ... from w0, with
// their up rows ms elements further when pair) times the input [BT][K] in
// shared memory. Each chunk of the input is loaded once for all units:
// partials into v[(2 u + m) BT + b].
template <int BT, int UPW>
__device__ __forceinline__ void units_smem(const uint16_t* w0, int U, int K, size_t ms, bool pair,
                                           const float* xs, int C, int lane,
                                           float (&v)[UPW * 2 * BT]) {
  for (int c = lane; c < C; c += kWarp) {
    float xb[BT][8];
#pragma unroll
    for (int b = 0; b < BT; ++b) {
      const float4 p0 = *reinterpret_cast<const float4*>(xs + b * K + c * 4);
      const float4 p1 = *reinterpret_cast<const float4*>(xs + b * K + K / 2 + c * 4);
      xb[b][0] = p0.x; xb[b][1] = p0.y; xb[b][2] = p0.z; xb[b][3] = p0.w;
      xb[b][4] = p1.x; xb[b][5] = p1.y; xb[b][6] = p1.z; xb[b][7] = p1.w;
    }
#pragma unroll
    for (int u = 0; u < UPW; ++u) {
      if (u < U) {
        const uint16_t* w = w0 + (size_t)u * kPConsumerWarps * K + c * 8;
        const uint4 wa = *reinterpret_cast<const uint4*>(w);
#pragma unroll
        for (int b = 0; b < BT; ++b) v[(2 * u) * BT + b] += dot8r(wa, xb[b]);
        if (pair) {
          const uint4 wb = *reinterpret_cast<const uint4*>(w + ms);
#pragma unroll
          for (int b = 0; b < BT; ++b) v[(2 * u + 1) * BT + b] += dot8r(wb, xb[b]);
        }
      }
    }
    compiler_fence();
  }
}

// Chunks [c0, c1) of one row (and of its up row when w1 is set) times the
// input [BT][K] in shared memory: per-lane partials into o[m * BT + b].
template <int BT>
__device__ __forceinline__ void row_dot_smem(const uint16_t* w0, const uint16_t* w1,
                                             const float* xs, int K, int c0, int c1, int lane,
                                             float* o) {
#pragma unroll 2
  for (int c = c0 + lane; c < c1; c += kWarp) {
    const uint4 wa = *reinterpret_cast<const uint4*>(w0 + c * 8);
    const uint4 wb = w1 ? *reinterpret_cast<const uint4*>(w1 + c * 8) : uint4{};
#pragma unroll
    for (int b = 0; b < BT; ++b) {
      float xb[8];
      const float4 p0 = *reinterpret_cast<const float4*>(xs + b * K + c * 4);
      const float4 p1 = *reinterpret_cast<const float4*>(xs + b * K + K / 2 + c * 4);
      xb[0] = p0.x; xb[1] = p0.y; xb[2] = p0.z; xb[3] = p0.w;
      xb[4] = p1.x; xb[5] = p1.y; xb[6] = p1.z; xb[7] = p1.w;
      o[b] += dot8r(wa, xb);
      if (w1) o[BT + b] += dot8r(wb, xb);
    }
  }
}

// Where a phase's outputs go, read from the arguments once per phase: the
// tile loop then touches no argument field (after every asm statement with a
// memory clobber the compiler would have to load those again).
struct PhaseOut {
  uint64_t* words;  // epoch-tagged outputs [B][stride] (QKV, residual, SiLU * up)
  float* logits;    // [B][stride] (LM head)
  int stride;
  int base;         // first row held in xoldw / biasr
  uint32_t ep_old;  // epoch of the residual words the o-proj/down epilogue adds to
  bool bias;        // QKV bias present
};

// Epilogue of output row j of sequence b on the reducing thread: bias, the
// residual add, silu(gate) * up, or the logit and its arg-max key.
template <int BT>
__device__ __forceinline__ void tile_epilogue(const PShared& S, int kind, const PhaseOut& po,
                                              int r0, int j, int b, float v0, float v1,
                                              uint32_t ep, unsigned long long (&best)[BT],
                                              Spin& sp) {
  if (kind == kQKV) {
    const float bias = po.bias ? bf16_to_f32(S.biasr[j - po.base]) : 0.f;
    st_word(po.words + (size_t)b * po.stride + j, v0 + bias, ep);
  } else if (kind == kOPROJ || kind == kDOWN) {
    uint64_t* dst = po.words + (size_t)b * po.stride + j;
    const uint64_t w = S.xoldw[b][j - po.base];
    // complete before this phase began (its readers checked), so the epoch
    // matches; a mismatch falls back to polling the word
    const float old = static_cast<uint32_t>(w >> 32) == po.ep_old
                          ? __uint_as_float(static_cast<uint32_t>(w))
                          : ll_get(dst, po.ep_old, sp);
    st_word(dst, old + v0, ep);
  } else if (kind == kGU) {
    st_word(po.words + (size_t)b * po.stride + j, silu_mul_p(v0, v1), ep);
  } else {
    po.logits[(size_t)b * po.stride + j] = v0;
    const unsigned long long key = argmax_key(v0, (uint32_t)j);
#pragma unroll
    for (int bb = 0; bb < BT; ++bb)
      if (bb == b) best[bb] = key > best[bb] ? key : best[bb];
  }
}

// ------------------------------------------------------------------ attention item
// The producer streams the cached K and V of slots 0..pos-1 of every
// attention item this CTA owns through the ring, as chunk tiles holding the K
// rows then the V rows of up to attn_chunk positions; the new position's K/V
// never leaves shared memory.
constexpr int kAttnMaxChunk = 128;
__host__ __device__ __forceinline__ int attn_chunk(int slot_bytes, int D, int es) {
  const int cp = slot_bytes / (2 * D * es);
  return cp < kAttnMaxChunk ? cp : kAttnMaxChunk;
}

// Producer: issue the chunk tiles of (layer, b, g) for cached slots [p0, p1).
template <bool KV16>
__device__ bool produce_kv(const PersistArgs& a, PShared& S, char* ring, int slot_bytes,
                           int nslots, int layer, int b, int g, int p0, int p1, RingPos& rp,
                           Spin& sp) {
  constexpr int ES = KV16 ? 2 : 4;
  const int D = a.D, CP = attn_chunk(slot_bytes, D, ES);
  const int bs = a.kv.paged ? a.kv.block_size : (1 << 30);
  for (int t0 = p0; t0 < p1; t0 += CP) {
    const int n = min(CP, p1 - t0);
    const int s = rp.s;
    if (rp.n >= (uint32_t)nslots && !ring_wait(&S.empty[s], rp.par ^ 1u, sp)) return false;
    if (*reinterpret_cast<volatile int*>(&S.abort)) return false;
    // runs of positions contiguous in the cache: the whole chunk when the
    // cache is contiguous, a block's worth when it is paged
    uint32_t bytes = 0;
    for (int t = t0; t < t0 + n;) {
      const int len = min(t0 + n - t, bs - t % bs);
      if (a.kv.slot_ok(b, t)) bytes += 2u * len * D * ES;
      t += len;
    }
    mbar_expect_tx(&S.full[s], bytes);
    char* dst = ring + (size_t)s * slot_bytes;
    for (int t = t0; t < t0 + n;) {
      const int len = min(t0 + n - t, bs - t % bs);
      if (a.kv.slot_ok(b, t)) {
        const size_t off = a.kv.offset(layer, b, g, t) * ES;
        const uint32_t nb = (uint32_t)len * D * ES;
        bulk_g2s(dst + (size_t)(t - t0) * D * ES, static_cast<const char*>(a.kv.k) + off, nb,
                 &S.full[s]);
        bulk_g2s(dst + (size_t)(CP + t - t0) * D * ES, static_cast<const char*>(a.kv.v) + off,
                 nb, &S.full[s]);
      }
      t += len;
    }
    rp.next(nslots);
    S.issued = rp.n;
  }
  return true;
}

template <bool KV16>
__device__ __forceinline__ float kv_smem(const char* base, int idx) {
  if constexpr (KV16) return bf16_to_f32(reinterpret_cast<const uint16_t*>(base)[idx]);
  else return reinterpret_cast<const float*>(base)[idx];
}

// Elements idx .. idx + 3 (idx a multiple of 4) in one 16- or 8-byte load.
template <bool KV16>
__device__ __forceinline__ void kv_smem4(const char* base, int idx, float (&o)[4]) {
  if constexpr (KV16) {
    const uint2 w = *reinterpret_cast<const uint2*>(base + (size_t)idx * 2);
    o[0] = bf16_lo(w.x); o[1] = bf16_hi(w.x); o[2] = bf16_lo(w.y); o[3] = bf16_hi(w.y);
  } else {
    const float4 v = *reinterpret_cast<const float4*>(base + (size_t)idx * 4);
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
  }
}
// Elements idx, idx + 1 (idx even) in one load.
template <bool KV16>
__device__ __forceinline__ float2 kv_smem2(const char* base, int idx) {
  if constexpr (KV16) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(base + (size_t)idx * 2);
    return make_float2(bf16_lo(w), bf16_hi(w));
  } else {
    return *reinterpret_cast<const float2*>(base + (size_t)idx * 4);
  }
}

// Elements idx .. idx + E - 1 (E = 2 or 4, idx a multiple of E) in one load.
template <bool KV16, int E>
__device__ __forceinline__ void kv_smemE(const char* base, int idx, float (&o)[E]) {
  if constexpr (E == 4) {
    kv_smem4<KV16>(base, idx, o);
  } else {
    const float2 v = kv_smem2<KV16>(base, idx);
    o[0] = v.x;
    o[1] = v.y;
  }
}

// One attention item is split `split` of the ns splits of (sequence b, kv
// head g): RoPE (+ q/k norm) of the G query heads and the key; split 0
// appends K/V at slot pos and opens the online-softmax state with the new
// position; then the scan over the split's cached positions [p0, p1), in
// chunks from the ring. An unsplit scan writes its output o = acc / l as the
// attention output words. A split writes its state (m, l and o per head) to
// the partials and takes a ticket; the split that arrives last merges all
// of them (Tang section 2.2: per head M = max_s m_s, weights
// w_s = exp(m_s - M) l_s, out = sum_s (w_s / sum_t w_t) o_s; one split gives
// weight l / l = 1 and out = o exactly) and writes the output words.
//
// The attention scratch: qs [GM][D] (the query heads; after the scan the
// normalised outputs), kn [D], vn [D], then sc: the scan's score buffers or
// per-warp states, the merge's (m, l) and weights, and from sc + kAttnFin the
// heads' final (m, l).
constexpr int kAttnFin = 2 * 8 * kAttnMaxChunk;

// The item's inputs: warp w < G gathers query head w, warp G the key, warp
// G + 1 the value; lane l holds dims l + 32 j, so a RoPE pair (i, i + D/2)
// sits in one lane: the q/k norm and the rotation run in registers (angles
// from the per-step table), then K and V go to the cache straight from the
// owning warps. Returns whether this item owns the new position.
template <int D, bool KV16>
__device__ __forceinline__ bool attn_inputs(const PersistArgs& a, int b, int g, int split,
                                            int layer, uint32_t ep_qkv, Spin& sp) {
  // shared-memory pointers are derived from the dynamic shared array here, so
  // the compiler addresses them as shared, not generic
  extern __shared__ __align__(128) char smem[];
  PShared& S = *reinterpret_cast<PShared*>(smem);
  float* scratch = reinterpret_cast<float*>(smem + a.attn_offset);
  constexpr int GM = 8, E = D / 32;
  const int ct = threadIdx.x - kWarp, warp = ct / kWarp, lane = ct % kWarp;
  const KVView kv = a.kv;
  const int Hq = a.Hq, Hkv = a.Hkv;
  const float eps = a.eps;
  int* const status = a.status;
  const int G = Hq / Hkv;
  const int pos = S.pos[b];
  float* qs = scratch;
  float* kn = qs + GM * D;
  float* vn = kn + D;
  const PLayer& P = S.layers[layer];
  const bool pos_ok = kv.slot_ok(b, pos);
  const bool own_new = pos_ok && split == 0;  // the new position belongs to split 0
  if (!pos_ok && split == 0 && ct == 0 && status) atomicCAS(status, 0, (int)NC_ERR_POSITION);
  const uint16_t* gq = P.g_q;
  const uint16_t* gk = P.g_k;
  if (warp < G + 2) {
    const uint64_t* qkv = a.qkvw + (size_t)b * a.nqkv;
    const uint64_t* src =
        qkv + (warp < G ? (g * G + warp) * D : (warp == G ? (Hq + g) * D : (Hq + Hkv + g) * D));
    const auto addr = [src, lane](int j) { return src + lane + 32 * j; };
    uint64_t w[E];
#pragma unroll
    for (int j = 0; j < E; ++j) w[j] = ld_word(addr(j));
    const uint16_t* gain = warp < G ? gq : (warp == G ? gk : nullptr);
    float gn[E];
#pragma unroll
    for (int j = 0; j < E; ++j) gn[j] = gain ? bf16_to_f32(gain[lane + 32 * j]) : 1.f;
    ll_settle<E>(addr, (1u << E) - 1u, ep_qkv, w, sp);
    float e[E];
#pragma unroll
    for (int j = 0; j < E; ++j) e[j] = __uint_as_float(static_cast<uint32_t>(w[j]));
    if (gain) {  // per-head RMSNorm over D
      float ss = 0.f;
#pragma unroll
      for (int j = 0; j < E; ++j) ss = fmaf(e[j], e[j], ss);
      ss = warp_sum(ss);
      const float r = 1.f / sqrtf(ss / (float)D + eps);
#pragma unroll
      for (int j = 0; j < E; ++j) e[j] = (e[j] * r) * gn[j];
    }
    if (warp <= G) {  // RoPE on q and k
#pragma unroll
      for (int j = 0; j < E / 2; ++j) {
        const float cs = S.rope_cs[b][lane + 32 * j], sn = S.rope_sn[b][lane + 32 * j];
        const float x0 = e[j], x1 = e[j + E / 2];
        e[j] = __fsub_rn(__fmul_rn(x0, cs), __fmul_rn(x1, sn));
        e[j + E / 2] = __fadd_rn(__fmul_rn(x1, cs), __fmul_rn(x0, sn));
      }
    }
    if (KV16 && warp >= G)  // k and v as the cache stores them
#pragma unroll
      for (int j = 0; j < E; ++j) e[j] = bf16_to_f32(f32_to_bf16(e[j]));
    float* dst = warp < G ? qs + warp * D : (warp == G ? kn : vn);
#pragma unroll
    for (int j = 0; j < E; ++j) dst[lane + 32 * j] = e[j];
    if (warp >= G && own_new) {  // append at slot pos
      const size_t off = kv.offset(layer, b, g, pos);
      void* cache = warp == G ? kv.k : kv.v;
#pragma unroll
      for (int j = 0; j < E; ++j) kv_store<KV16>(cache, off + lane + 32 * j, e[j]);
    }
  }
  consumer_sync();
  return own_new;
}

// The item's end: the normalised outputs ofin [G][D] and the heads' (m, l)
// are in shared memory (behind a barrier). An unsplit item writes the output
// words; a split publishes its partials, takes the ticket, and the last
// split merges.
template <int D>
__device__ __forceinline__ void attn_finish(const PersistArgs& a, int b, int g, int split, int ns,
                                            int layer, uint32_t ep_out,
                                            unsigned long long* prof_sub) {
  // shared-memory pointers are derived from the dynamic shared array here, so
  // the compiler addresses them as shared, not generic
  extern __shared__ __align__(128) char smem[];
  PShared& S = *reinterpret_cast<PShared*>(smem);
  float* scratch = reinterpret_cast<float*>(smem + a.attn_offset);
  constexpr int GM = 8;
  const int ct = threadIdx.x - kWarp, warp = ct / kWarp, lane = ct % kWarp;
  const int Hq = a.Hq, Hkv = a.Hkv;
  const int G = Hq / Hkv;
  const float* ofin = scratch;      // [G][D]
  float* sc = scratch + (GM + 2) * D;
  const float* mfin = sc + kAttnFin;  // [G]
  const float* lfin = mfin + GM;      // [G]
  if (prof_sub && ct == 0) {
    prof_sub[0] = global_timer();
    prof_sub[2] = 0ull;
  }
  uint64_t* const aout = a.aw + (size_t)b * Hq * D + (size_t)g * G * D;  // [G][D] words
  // split partials [G][DP] per head of this (b, g, split): o[D], then m, l
  // (rows padded to a 16-byte multiple, so the merge can stage them with
  // 16-byte asynchronous copies)
  constexpr int DP = D + 4;
  float* const parts = a.apart + ((size_t)b * kPMaxSplits * Hq + (size_t)g * G) * DP;
  const size_t sstride = (size_t)Hq * DP;  // from one split's partials to the next
  float* const mine = parts + split * sstride;
  for (int i = ct; i < G * D; i += kPConsumerThreads) {
    const int h = i / D, d = i % D;
    if (ns == 1) {
      st_word(aout + i, ofin[i], ep_out);
    } else {
      mine[h * DP + d] = ofin[i];
      if (d == 0) *reinterpret_cast<float2*>(mine + h * DP + D) = make_float2(mfin[h], lfin[h]);
    }
  }
  if (ns == 1) {
    consumer_sync();  // the scratch is reused by the next item
    if (prof_sub && ct == 0) prof_sub[1] = global_timer();
    return;
  }
  // The ticket. The barrier orders every thread's partials before thread
  // 0's fence, which publishes them GPU-wide (cumulatively) before its
  // arrival; the split that arrives last fences again before the barrier
  // that lets its threads read the others' partials.
  consumer_sync();
  unsigned int* const tick = a.atick + ((size_t)layer * kPMaxBatch + b) * Hkv + g;
  if (ct == 0) {
    __threadfence();
    const bool last = atomicAdd(tick, 1u) == (unsigned)(ns - 1);
    if (last) __threadfence();
    S.merge = last;
  }
  consumer_sync();
  if (prof_sub && ct == 0) prof_sub[1] = global_timer();
  if (!S.merge) return;  // uniform: read after the barrier
  // The splits' outputs are staged into the (idle) input-vector region in
  // rounds of as many splits as it holds. The first round's copies are in
  // flight while the (m, l) of every (split, head) are loaded (one load
  // each); then warp h forms head h's merge weights, lane t that of split t:
  // M = max_t m_t, w_t = e^(m_t - M) l_t, coef_t = w_t / sum w (a division,
  // not a reciprocal, as in the single-split case). Every thread accumulates
  // its elements over the splits in index order.
  float* ml = sc;                          // [ns][G][2]
  float* coef = sc + 2 * kPMaxSplits * GM;  // [G][kPMaxSplits] merge weights
  float* stage = reinterpret_cast<float*>(smem + a.xs_offset);
  const int per_split = G * DP;  // floats of one split's block
  const int span = (a.attn_offset - a.xs_offset) / (per_split * 4);
  const auto stage_round = [&](int t0) {
    const int chunks = min(span, ns - t0) * (per_split / 4);
    for (int c = ct; c < chunks; c += kPConsumerThreads) {
      const int t = c / (per_split / 4), r = c % (per_split / 4);
      cp_async16(stage + t * per_split + 4 * r, parts + (t0 + t) * sstride + 4 * r);
    }
    cp_async_commit();
  };
  stage_round(0);
  if (ct < ns * G) {
    const int t = ct / G, h = ct % G;
    const float2 v = __ldcg(reinterpret_cast<const float2*>(parts + t * sstride + h * DP + D));
    ml[2 * ct] = v.x;
    ml[2 * ct + 1] = v.y;
  }
  consumer_sync();
  if (warp < G) {
    const float m = lane < ns ? ml[2 * (lane * G + warp)] : -INFINITY;
    const float l = lane < ns ? ml[2 * (lane * G + warp) + 1] : 0.f;
    const float M = warp_max(m);
    const float w = m == -INFINITY ? 0.f : expf(m - M) * l;
    const float L = warp_sum(w);
    if (lane < ns) coef[warp * kPMaxSplits + lane] = L > 0.f ? w / L : 0.f;
  }
  constexpr int EPT = (8 * 128 + kPConsumerThreads - 1) / kPConsumerThreads;  // outputs a thread owns
  float o[EPT];
#pragma unroll
  for (int e = 0; e < EPT; ++e) o[e] = 0.f;
  for (int t0 = 0; t0 < ns; t0 += span) {
    const int nt = min(span, ns - t0);
    if (t0 > 0) stage_round(t0);
    cp_async_wait_all();
    consumer_sync();  // staged (and, in the first round, coef written)
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
      const int i = ct + e * kPConsumerThreads;
      if (i < G * D) {
        const int h = i / D, d = i % D;
        for (int t = 0; t < nt; ++t)
          o[e] = fmaf(coef[h * kPMaxSplits + t0 + t], stage[t * per_split + h * DP + d], o[e]);
      }
    }
    consumer_sync();  // the staging area is rewritten by the next round
  }
#pragma unroll
  for (int e = 0; e < EPT; ++e) {
    const int i = ct + e * kPConsumerThreads;
    if (i < G * D) st_word(aout + i, o[e], ep_out);
  }
  if (prof_sub && ct == 0) prof_sub[2] = global_timer();
}


// Scan with per-warp states (head size 128). Warps 0 .. SW - 1 each keep
// their own online-softmax state of every query head over the positions
// they take, with no block barrier inside a chunk: lane l holds dims
// l E .. l E + E - 1 of each head in registers; a group of PG = 32 / GP
// positions (GP = G rounded up to a power of two) gives 32 partial dot
// products per lane, which one reduce-scatter turns into lane i's score of
// (position i / GP, head i % GP). The warps' states are combined once, after
// the scan.
template <int D, bool KV16, int GP>
__device__ __noinline__ void attention_item(const PersistArgs& a, int b, int g, int split, int ns,
                                            int p0, int p1, int layer, uint32_t ep_qkv,
                                            uint32_t ep_out, int nslots, RingPos& rp, Spin& sp,
                                            unsigned long long* prof_in,
                                            unsigned long long* prof_sub) {
  const bool own_new = attn_inputs<D, KV16>(a, b, g, split, layer, ep_qkv, sp);
  if (prof_in) *prof_in = global_timer();  // the phase input (q, k, v) is in
  // shared-memory pointers are derived from the dynamic shared array here, so
  // the compiler addresses them as shared, not generic
  extern __shared__ __align__(128) char smem[];
  PShared& S = *reinterpret_cast<PShared*>(smem);
  float* scratch = reinterpret_cast<float*>(smem + a.attn_offset);
  constexpr int GM = 8, E = D / 32;
  const int ct = threadIdx.x - kWarp, warp = ct / kWarp, lane = ct % kWarp;
  char* ring = smem + a.ring_offset;
  const int slot_bytes = a.slot_bytes;
  constexpr int ES = KV16 ? 2 : 4;
  const KVView kv = a.kv;
  const int G = a.Hq / a.Hkv;
  const int CP = attn_chunk(slot_bytes, D, ES);
  float* qs = scratch;
  float* kn = qs + GM * D;
  float* vn = kn + D;
  float* sc = vn + D;
  constexpr int SW = kPConsumerWarps;  // scan warps: all of them
  constexpr int PG = kWarp / GP;       // positions per group
  const float scale = 1.f / sqrtf((float)D);
  float qr[GP][E], acc[GP][E], mh[GP], lh[GP];
#pragma unroll
  for (int h = 0; h < GP; ++h) {
    mh[h] = -INFINITY;
    lh[h] = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      acc[h][e] = 0.f;
      qr[h][e] = h < G ? qs[h * D + lane * E + e] : 0.f;
    }
  }
  // the new position opens warp 0's state: m = its score, l = 1, acc = v
  if (warp == 0 && own_new) {
#pragma unroll
    for (int h = 0; h < GP; ++h) {
      float d = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) d = fmaf(qr[h][e], kn[lane * E + e], d);
      d = warp_sum(d) * scale;
      if (h < G) {
        mh[h] = d;
        lh[h] = 1.f;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[h][e] = vn[lane * E + e];
      }
    }
  }
  const int hl = lane % GP, pl = lane / GP;  // what lane holds after the reduce
  unsigned long long* const mark = prof_sub && ct == 0 ? prof_sub : nullptr;
  // Groups are numbered across the chunks and warp w takes the groups
  // congruent to w modulo SW, so a chunk of fewer than SW groups leaves the
  // other warps to the next chunk (the ring holds several) instead of idle.
  int gbase = 0;  // groups of the earlier chunks
  for (int t0 = p0; t0 < p1; t0 += CP) {
    const int n = min(CP, p1 - t0);
    const int s = rp.s;
    ring_wait(&S.full[s], rp.par, sp);
    if (mark) mark[t0 == p0 ? 3 : 4] = global_timer();
    const char* Ks = ring + (size_t)s * slot_bytes;
    const char* Vs = Ks + (size_t)CP * D * ES;
    {
      for (int g0 = ((warp - gbase % SW + SW) % SW) * PG; g0 < n; g0 += SW * PG) {
        float part[kWarp];
#pragma unroll
        for (int p = 0; p < PG; ++p) {
          float k[E];
          kv_smemE<KV16, E>(Ks, (g0 + p < n ? g0 + p : 0) * D + lane * E, k);
#pragma unroll
          for (int h = 0; h < GP; ++h) {
            float d = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) d = fmaf(qr[h][e], k[e], d);
            part[p * GP + h] = d;
          }
        }
        warp_sum_many<kWarp>(part);
        const int pp = g0 + pl;
        const bool ok = pp < n && hl < G && kv.slot_ok(b, t0 + pp);
        const float sv = ok ? part[0] * scale : -INFINITY;
        float mx = sv;  // the group's max of each head, over the lanes holding it
#pragma unroll
        for (int o = GP; o < kWarp; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
        float corr[GP], mine_m = -INFINITY;
#pragma unroll
        for (int h = 0; h < GP; ++h) {
          const float mn = fmaxf(mh[h], __shfl_sync(0xFFFFFFFFu, mx, h));
          corr[h] = mh[h] == -INFINITY ? 0.f : expf(mh[h] - mn);
          mh[h] = mn;
          if (h == hl) mine_m = mn;
        }
        const float pr = sv == -INFINITY ? 0.f : expf(sv - mine_m);
        float sm = pr;
#pragma unroll
        for (int o = GP; o < kWarp; o <<= 1) sm += __shfl_xor_sync(0xFFFFFFFFu, sm, o);
#pragma unroll
        for (int h = 0; h < GP; ++h) {
          lh[h] = lh[h] * corr[h] + __shfl_sync(0xFFFFFFFFu, sm, h);
#pragma unroll
          for (int e = 0; e < E; ++e) acc[h][e] *= corr[h];
        }
#pragma unroll
        for (int p = 0; p < PG; ++p) {
          float v[E];
          kv_smemE<KV16, E>(Vs, (g0 + p < n ? g0 + p : 0) * D + lane * E, v);
#pragma unroll
          for (int h = 0; h < GP; ++h) {
            const float ph = __shfl_sync(0xFFFFFFFFu, pr, p * GP + h);
            // a masked position (weight 0) may sit over stale shared memory,
            // so its value is replaced, not multiplied
#pragma unroll
            for (int e = 0; e < E; ++e) acc[h][e] = fmaf(ph, ph == 0.f ? 0.f : v[e], acc[h][e]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[s]);
    rp.next(nslots);
    gbase += (n + PG - 1) / PG;
  }
  if (mark) {
    const unsigned long long now = global_timer();
    if (p1 <= p0) mark[3] = now;           // nothing to scan
    if (p1 - p0 <= CP) mark[4] = mark[3];  // one chunk: the first is the last
    mark[5] = now;
  }
  // combine the scan warps' states per head: M = max_w m_w, weights
  // c_w = e^(m_w - M), L = sum_w c_w l_w, O = sum_w c_w acc_w (warps in order)
  float* cmb = reinterpret_cast<float*>(smem + a.xs_offset);  // [SW][G][D] (idle now)
  float* mlw = sc;                                            // [SW][GM][2]
  if (warp < SW) {
#pragma unroll
    for (int h = 0; h < GP; ++h)
      if (h < G) {
#pragma unroll
        for (int e = 0; e < E; ++e) cmb[(warp * G + h) * D + lane * E + e] = acc[h][e];
        if (lane == 0) {
          mlw[(warp * GM + h) * 2] = mh[h];
          mlw[(warp * GM + h) * 2 + 1] = lh[h];
        }
      }
  }
  consumer_sync();
  // the heads' combined states: normalised outputs to qs (idle after the
  // scan), (M, L) after the merge's buffers
  float* mfin = sc + kAttnFin;
  float* lfin = mfin + GM;
  for (int i = ct; i < G * D; i += kPConsumerThreads) {
    const int h = i / D, d = i % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < SW; ++w) M = fmaxf(M, mlw[(w * GM + h) * 2]);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < SW; ++w) {
      const float m = mlw[(w * GM + h) * 2];
      const float c = m == -INFINITY ? 0.f : expf(m - M);
      L = fmaf(c, mlw[(w * GM + h) * 2 + 1], L);
      O = fmaf(c, cmb[(w * G + h) * D + d], O);
    }
    qs[i] = L > 0.f ? O / L : 0.f;
    if (d == 0) {
      mfin[h] = M;
      lfin[h] = L;
    }
  }
  consumer_sync();
  attn_finish<D>(a, b, g, split, ns, layer, ep_out, prof_sub);
}

// Scan with block-wide steps (head size 64, short rows and up to 8 heads a
// group, where every (head, dim pair) has a thread of its own): per chunk the
// warps compute the scores of (head, 32 positions) blocks, one warp per head
// updates that head's running (m, l) and turns the scores into weights, and
// thread (h, d pair) accumulates its two output dims over the chunk.
template <int D, bool KV16>
__device__ __noinline__ void attention_item_block(const PersistArgs& a, int b, int g, int split,
                                                  int ns, int p0, int p1, int layer,
                                                  uint32_t ep_qkv, uint32_t ep_out, int nslots,
                                                  RingPos& rp, Spin& sp,
                                                  unsigned long long* prof_in,
                                                  unsigned long long* prof_sub) {
  const bool own_new = attn_inputs<D, KV16>(a, b, g, split, layer, ep_qkv, sp);
  if (prof_in) *prof_in = global_timer();  // the phase input (q, k, v) is in
  extern __shared__ __align__(128) char smem[];
  PShared& S = *reinterpret_cast<PShared*>(smem);
  float* scratch = reinterpret_cast<float*>(smem + a.attn_offset);
  constexpr int GM = 8, E = D / 32, ES = KV16 ? 2 : 4;
  const int ct = threadIdx.x - kWarp, warp = ct / kWarp, lane = ct % kWarp;
  char* ring = smem + a.ring_offset;
  const int slot_bytes = a.slot_bytes;
  const KVView kv = a.kv;
  const int G = a.Hq / a.Hkv;
  const int CP = attn_chunk(slot_bytes, D, ES);
  float* qs = scratch;
  float* kn = qs + GM * D;
  float* vn = kn + D;
  float* sc = vn + D;                 // [2][GM][kAttnMaxChunk] scores, by chunk parity
  float* mrun = sc + kAttnFin;        // [GM] running max (the final m)
  float* lrun = mrun + GM;            // [GM] running sum (the final l)
  float* resc = lrun + GM;            // [GM] rescale of the chunk
  unsigned long long* const mark = prof_sub && ct == 0 ? prof_sub : nullptr;
  // the new position opens the running state: m = its score, l = 1, acc = v
  const float scale = 1.f / sqrtf((float)D);
  for (int h = warp; h < G; h += kPConsumerWarps) {
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < E; ++j) s = fmaf(qs[h * D + lane + 32 * j], kn[lane + 32 * j], s);
    s = warp_sum(s) * scale;
    if (lane == 0) {
      mrun[h] = own_new ? s : -INFINITY;
      lrun[h] = own_new ? 1.f : 0.f;
    }
  }
  const int npair = G * (D / 2);
  const int my_h = ct / (D / 2), my_d2 = ct % (D / 2);
  float acc0 = 0.f, acc1 = 0.f;
  if (ct < npair && own_new) {
    acc0 = vn[2 * my_d2];
    acc1 = vn[2 * my_d2 + 1];
  }
  consumer_sync();
  int cpar = 0;
  for (int t0 = p0; t0 < p1; t0 += CP, cpar ^= 1) {
    const int n = min(CP, p1 - t0);
    const int s = rp.s;
    ring_wait(&S.full[s], rp.par, sp);
    if (mark) mark[t0 == p0 ? 3 : 4] = global_timer();
    const char* Ks = ring + (size_t)s * slot_bytes;
    const char* Vs = Ks + (size_t)CP * D * ES;
    float* scc = sc + cpar * GM * kAttnMaxChunk;  // the other buffer may still be read
    // scores: warp -> (head, 32 positions); lane l reads its row from column
    // (d + l) mod D so the 32 rows of a warp fall in different banks
    const int blocks = (n + 31) / 32;
    for (int wb = warp; wb < G * blocks; wb += kPConsumerWarps) {
      const int h = wb % G, p = (wb / G) * 32 + lane;
      if (p < n) {
        float sv = -INFINITY;
        if (kv.slot_ok(b, t0 + p)) {
          // 4-element columns, skewed by lane: the 8 lanes of each 16-byte
          // load phase read 8 different bank groups
          float s4[4] = {0.f, 0.f, 0.f, 0.f};
          const float* qh = qs + h * D;
#pragma unroll
          for (int j = 0; j < D / 4; ++j) {
            const int c = ((j + lane) & (D / 4 - 1)) * 4;
            const float4 q4 = *reinterpret_cast<const float4*>(qh + c);
            float k4[4];
            kv_smem4<KV16>(Ks, p * D + c, k4);
            s4[0] = fmaf(q4.x, k4[0], s4[0]);
            s4[1] = fmaf(q4.y, k4[1], s4[1]);
            s4[2] = fmaf(q4.z, k4[2], s4[2]);
            s4[3] = fmaf(q4.w, k4[3], s4[3]);
          }
          sv = ((s4[0] + s4[1]) + (s4[2] + s4[3])) * scale;
        }
        scc[h * kAttnMaxChunk + p] = sv;
      }
    }
    consumer_sync();
    if (mark && t0 == p0) mark[6] = global_timer();  // the first chunk's scores
    for (int h = warp; h < G; h += kPConsumerWarps) {
      float m = -INFINITY;
      for (int t = lane; t < n; t += kWarp) m = fmaxf(m, scc[h * kAttnMaxChunk + t]);
      m = warp_max(m);
      const float m_new = fmaxf(mrun[h], m);
      float l = 0.f;
      for (int t = lane; t < n; t += kWarp) {
        const float x = scc[h * kAttnMaxChunk + t];
        const float p = x == -INFINITY ? 0.f : expf(x - m_new);
        scc[h * kAttnMaxChunk + t] = p;
        l += p;
      }
      l = warp_sum(l);
      if (lane == 0) {
        const float r = mrun[h] == -INFINITY ? 0.f : expf(mrun[h] - m_new);
        resc[h] = r;
        lrun[h] = lrun[h] * r + l;
        mrun[h] = m_new;
      }
    }
    consumer_sync();
    if (mark && t0 == p0) mark[7] = global_timer();  // ... and its weights
    if (ct < npair) {
      const float r = resc[my_h];
      // two interleaved chains per output; a masked position (p = 0) may sit
      // over stale shared memory, so its value is replaced, not multiplied
      float e0 = 0.f, e1 = 0.f, o0 = 0.f, o1 = 0.f;
      const float* ph = scc + my_h * kAttnMaxChunk;
      int t = 0;
#pragma unroll 4
      for (; t + 1 < n; t += 2) {
        const float pa = ph[t], pb = ph[t + 1];
        const float2 va = kv_smem2<KV16>(Vs, t * D + 2 * my_d2);
        const float2 vb = kv_smem2<KV16>(Vs, (t + 1) * D + 2 * my_d2);
        e0 = fmaf(pa, pa == 0.f ? 0.f : va.x, e0);
        e1 = fmaf(pa, pa == 0.f ? 0.f : va.y, e1);
        o0 = fmaf(pb, pb == 0.f ? 0.f : vb.x, o0);
        o1 = fmaf(pb, pb == 0.f ? 0.f : vb.y, o1);
      }
      if (t < n) {
        const float pa = ph[t];
        const float2 va = kv_smem2<KV16>(Vs, t * D + 2 * my_d2);
        e0 = fmaf(pa, pa == 0.f ? 0.f : va.x, e0);
        e1 = fmaf(pa, pa == 0.f ? 0.f : va.y, e1);
      }
      acc0 = fmaf(acc0, r, e0 + o0);
      acc1 = fmaf(acc1, r, e1 + o1);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[s]);
    rp.next(nslots);
    // no barrier here: the next chunk writes the other score buffer, and the
    // one after it is behind that chunk's two barriers
  }
  if (mark) {
    const unsigned long long now = global_timer();
    if (p1 <= p0) mark[3] = mark[6] = mark[7] = now;  // nothing to scan
    if (p1 - p0 <= CP) mark[4] = mark[3];             // one chunk: the first is the last
    mark[5] = now;
  }
  // normalised outputs to qs (no score step reads it any more: the last
  // chunk's scores are behind two barriers)
  if (ct < npair) {
    const float inv = lrun[my_h] > 0.f ? 1.f / lrun[my_h] : 0.f;
    qs[my_h * D + 2 * my_d2] = acc0 * inv;
    qs[my_h * D + 2 * my_d2 + 1] = acc1 * inv;
  }
  consumer_sync();
  attn_finish<D>(a, b, g, split, ns, layer, ep_out, prof_sub);
}

// The tiles of one projection phase (see gemv_phase). MODE 0: batch 1, rows of
// at most 1024 (input in registers); 1: batch 1, longer rows (k segments
// across warps); 3: batch 1, longer rows, whole rows per warp; 2: batch > 1. Inlined: a call here would save and restore
// the live registers of all 352 consumer threads through local memory, which
// with ~28 KB of L1 next to the ring spills to L2 and costs a round trip.
template <int BT, int MODE>
__device__ __forceinline__ void gemv_tiles(const PersistArgs& a, const Rows& rin,
                                        const PhaseOut& poin, int kind, uint32_t ep,
                                        RingPos& rp_io, int& kb_io,
                                        unsigned long long (&best_io)[BT], Spin& sp) {
  extern __shared__ __align__(128) char smem[];
  PShared& S = *reinterpret_cast<PShared*>(smem);
  char* ring = smem + a.ring_offset;
  float* xs = reinterpret_cast<float*>(smem + a.xs_offset);
  const int slot_bytes = a.slot_bytes, nslots = a.nslots;
  const int ct = threadIdx.x - kWarp, cw = ct / kWarp, lane = threadIdx.x % kWarp;
  const Rows r = rin;
  PhaseOut po = poin;
  const int K = r.K;
  RingPos rp = rp_io;
  int kb = kb_io;
  unsigned long long best[BT];
#pragma unroll
  for (int b = 0; b < BT; ++b) best[b] = best_io[b];
  const int two = r.m1 ? 2 : 1;
  const int nb = a.B;
  const int C = K / 8;  // 16-byte chunks per row
  // batch 1 and rows of at most 1024: every lane keeps its chunks of the
  // input in registers for the whole phase, and each unit is one row (or
  // one gate|up pair) reduced by one warp
  const bool xreg = MODE == 0;
  float xr[kXReg][8];
  if (xreg) {
#pragma unroll
    for (int jj = 0; jj < kXReg; ++jj) {
      const int c = lane + jj * kWarp;
      float4 p0 = make_float4(0.f, 0.f, 0.f, 0.f), p1 = p0;
      if (c < C) {  // two 16-byte loads, not eight scalar ones
        p0 = *reinterpret_cast<const float4*>(xs + c * 4);
        p1 = *reinterpret_cast<const float4*>(xs + K / 2 + c * 4);
      }
      xr[jj][0] = p0.x; xr[jj][1] = p0.y; xr[jj][2] = p0.z; xr[jj][3] = p0.w;
      xr[jj][4] = p1.x; xr[jj][5] = p1.y; xr[jj][6] = p1.z; xr[jj][7] = p1.w;
    }
  }
  for (int row = r.r0; row < r.r1; row += r.R) {
    const int n = min(r.R, r.r1 - row);
    ring_wait(&S.full[rp.s], rp.par, sp);  // on expiry the tile is garbage; the step is failed
    const uint16_t* tile =
        reinterpret_cast<const uint16_t*>(ring + (size_t)rp.s * slot_bytes);
    const size_t ms = (size_t)n * K;  // the up rows follow the n gate rows
    // How the warps share the tile:
    //  batch 1, rows of at most 1024: warp w reduces whole units w, w + W, ...
    //    against the input held in registers;
    //  batch 1, longer rows: the k range is cut into W segments, warp w
    //    reduces segment w of every unit (each input chunk loaded once for
    //    all of them) and the partials are summed across warps;
    //  batch > 1: units are cut into KS segments as needed, the input is
    //    read from shared memory.
    if constexpr (BT == 1 && MODE == 3) {
      // unit u of the phase (a row, or a gate|up pair) belongs to warp u % W:
      // the warp reduces its units of this tile over the whole k range
      // against the input in shared memory, one lane per 16-byte chunk, with
      // no barrier and no cross-warp sum; units of later tiles keep the other
      // warps busy meanwhile
      const int first = (cw - (row - r.r0) % kPConsumerWarps + kPConsumerWarps) % kPConsumerWarps;
      for (int i = first; i < n; i += kPConsumerWarps) {
        const uint16_t* w0 = tile + (size_t)i * K;
        // four chunks per lane in flight, each with its own partial sums
        float g[4] = {0.f, 0.f, 0.f, 0.f}, u[4] = {0.f, 0.f, 0.f, 0.f};
        const auto chunk = [&](int cc, float& gs, float& us) {
          float xb[8];
          const float4 p0 = *reinterpret_cast<const float4*>(xs + cc * 4);
          const float4 p1 = *reinterpret_cast<const float4*>(xs + K / 2 + cc * 4);
          xb[0] = p0.x; xb[1] = p0.y; xb[2] = p0.z; xb[3] = p0.w;
          xb[4] = p1.x; xb[5] = p1.y; xb[6] = p1.z; xb[7] = p1.w;
          gs += dot8r(*reinterpret_cast<const uint4*>(w0 + cc * 8), xb);
          if (two == 2) us += dot8r(*reinterpret_cast<const uint4*>(w0 + ms + cc * 8), xb);
        };
        int c = lane;
        for (; c + 3 * kWarp < C; c += 4 * kWarp) {
#pragma unroll
          for (int q = 0; q < 4; ++q) chunk(c + q * kWarp, g[q], u[q]);
          compiler_fence();
        }
        for (; c < C; c += kWarp) chunk(c, g[0], u[0]);
        float v[2] = {(g[0] + g[1]) + (g[2] + g[3]), (u[0] + u[1]) + (u[2] + u[3])};
        warp_sum_many<2>(v);  // value i in lane 16 i
        const float vup = __shfl_sync(0xFFFFFFFFu, v[0], 16);
        if (lane == 0 && nb > 0)
          tile_epilogue<BT>(S, kind, po, r.r0, row + i, 0, v[0], vup, ep, best, sp);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty[rp.s]);  // this warp is done with the slot
      rp.next(nslots);
    } else if constexpr (BT == 1) {
      if (xreg) {
        const int U = cw < n ? (n - cw + kPConsumerWarps - 1) / kPConsumerWarps : 0;
        float v[2 * kUnitsPerWarp];
#pragma unroll
        for (int i = 0; i < 2 * kUnitsPerWarp; ++i) v[i] = 0.f;
        const uint16_t* wt = tile + (size_t)cw * K;
        if (two == 2) units_xreg<true>(wt, U, K, ms, xr, C, lane, v);
        else units_xreg<false>(wt, U, K, ms, xr, C, lane, v);
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.empty[rp.s]);  // this warp is done with the slot
        rp.next(nslots);
        if (U > 0) {
          warp_sum_many<2 * kUnitsPerWarp>(v);  // value i = (unit i / 2, matrix i % 2) in lane 4 i
          const float vup = __shfl_down_sync(0xFFFFFFFFu, v[0], 4);
          const int i = lane / 4, u = i / 2, it = cw + u * kPConsumerWarps;
          if (lane % 4 == 0 && (i & 1) == 0 && u < U && nb > 0)
            tile_epilogue<BT>(S, kind, po, r.r0, row + it, 0, v[0], vup, ep, best, sp);
        }
      } else {
        // segment w of the k range, all units in passes of up to 8 rows
        const int KS = C >= kPConsumerWarps * kWarp ? kPConsumerWarps : max(1, C / kWarp);
        const int seg = cw;
        const int c0 = (seg * C) / KS, c1 = ((seg + 1) * C) / KS;
        const int upp = 8 / two;  // units per pass
        for (int g0 = 0; g0 < n; g0 += upp) {
          const int nu = min(upp, n - g0), nr = nu * two;
          float o[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) o[i] = 0.f;
          if (seg < KS) {
            const uint16_t* wt = tile + (size_t)g0 * K;
            seg_rows(wt, nr, K, ms, two, xs, c0, c1, lane, o);
          }
          if (g0 + upp >= n) {  // the slot is no longer read by this warp
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.empty[rp.s]);
          }
          warp_sum_many<8>(o);  // row i of the pass in lane 4 i
          if (lane % 4 == 0) S.kred[kb][seg][lane / 4] = seg < KS ? o[0] : 0.f;
          consumer_sync();
          for (int u = ct; u < nu; u += kPConsumerThreads) {
            float v0 = 0.f, v1 = 0.f;
#pragma unroll
            for (int sg = 0; sg < kPConsumerWarps; ++sg)  // independent loads, one chain of adds
              if (sg < KS) {
                v0 += S.kred[kb][sg][u * two];
                if (two == 2) v1 += S.kred[kb][sg][u * two + 1];
              }
            if (nb > 0)
              tile_epilogue<BT>(S, kind, po, r.r0, row + g0 + u, 0, v0, v1, ep, best, sp);
          }
          kb ^= 1;  // the next pass writes the other buffer: no second barrier
        }
        rp.next(nslots);
      }
    } else {
      // batch > 1: long rows are cut into KS k-segments when the tile has few
      // units, so the work spreads over all warps (up to kUnitsPerWarp items
      // each); a segment keeps at least 64 chunks, two per lane
      int KS = 1;
      constexpr int UPW = units_per_warp(BT);
      if (n < kPConsumerWarps) {
        KS = UPW * kPConsumerWarps / n;
        const int kmax = C / 64;
        if (KS > kmax) KS = kmax;
        if (KS < 1) KS = 1;
      }
      const int items = n * KS;  // warp cw takes items cw, cw + W, ...
      constexpr int NV = UPW * 2 * BT;  // [item u][matrix m][sequence b]
      float v[NV];
#pragma unroll
      for (int i = 0; i < NV; ++i) v[i] = 0.f;
      if (KS == 1) {
        // whole rows: the warp's units share each input chunk (loaded once)
        const int U = cw < n ? min(UPW, (n - cw + kPConsumerWarps - 1) / kPConsumerWarps) : 0;
        units_smem<BT, UPW>(tile + (size_t)cw * K, U, K, ms, two == 2, xs, C, lane, v);
      } else {
#pragma unroll
        for (int u = 0; u < UPW; ++u) {
          const int it = cw + u * kPConsumerWarps;
          if (it >= items) break;  // uniform across the warp
          const int ui = it / KS, seg = it % KS;
          const int c0 = (seg * C) / KS, c1 = ((seg + 1) * C) / KS;
          const uint16_t* w0 = tile + (size_t)ui * K;
          row_dot_smem<BT>(w0, two == 2 ? w0 + ms : nullptr, xs, K, c0, c1, lane,
                           v + 2 * u * BT);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty[rp.s]);  // this warp is done with the slot
      rp.next(nslots);
      // value i of the warp ends up in lane i * hl
      constexpr int hl = kWarp / NV;
      warp_sum_many<NV>(v);
      const int i = lane / hl, b = i % BT, m = (i / BT) & 1, u = i / (2 * BT);
      const int it = cw + u * kPConsumerWarps;
      if (KS == 1) {
        const float vup = __shfl_down_sync(0xFFFFFFFFu, v[0], BT * hl);  // the up partner
        if (lane % hl == 0 && m == 0 && b < nb && it < items)
          tile_epilogue<BT>(S, kind, po, r.r0, row + it, b, v[0], vup, ep, best, sp);
      } else {
        if (lane % hl == 0 && it < items) S.kred[kb][it][m * BT + b] = v[0];
        consumer_sync();
        for (int t = ct; t < n * BT; t += kPConsumerThreads) {
          const int ui = t / BT, bb = t % BT;
          if (bb >= nb) continue;
          float v0 = 0.f, v1 = 0.f;
#pragma unroll
          for (int sg = 0; sg < kPConsumerWarps; ++sg)  // independent loads, one chain of adds
            if (sg < KS) {
              v0 += S.kred[kb][ui * KS + sg][bb];
              v1 += S.kred[kb][ui * KS + sg][BT + bb];
            }
          tile_epilogue<BT>(S, kind, po, r.r0, row + ui, bb, v0, v1, ep, best, sp);
        }
        kb ^= 1;  // the next split tile writes the other buffer: no second barrier
      }
    }
  }
  rp_io = rp;
  kb_io = kb;
#pragma unroll
  for (int b = 0; b < BT; ++b) best_io[b] = best[b];
}

// One projection phase (QKV, o-proj, gate|up, down or the LM head) on the
// consumer warps: the epilogue's asynchronous prefetches, the input gather
// (out of line) and the tiles (per mode). The ring position, the
// split-buffer parity and the arg-max keys are carried in and out.
template <int BT>
__device__ __forceinline__ void gemv_phase(const PersistArgs& a, int ph, uint32_t seq,
                                           RingPos& rp_io, int& kb_io,
                                           unsigned long long (&best_io)[BT],
                                           unsigned long long* prof, Spin& sp) {
  extern __shared__ __align__(128) char smem[];
  PShared& S = *reinterpret_cast<PShared*>(smem);
  const int ct = threadIdx.x - kWarp;
  const int L = a.L;
  const int layer = ph / kPhasesPerLayer;
  const int kind = ph == kPhasesPerLayer * L ? kHEAD : ph % kPhasesPerLayer;
  const uint32_t ep = epoch_of(seq, ph);
  const Rows r = phase_rows(a, S, ph);
  if (r.r0 >= r.r1) return;
  // phase input
  const PLayer* P = kind == kHEAD ? nullptr : &S.layers[layer];
  const int K = r.K;
  PhaseOut po;
  po.base = 0;
  po.ep_old = 0;
  po.bias = false;
  // Rows this phase's epilogue needs that do not wait on the phase input
  // are copied asynchronously now; the gather waits for them before its
  // first barrier.
  if (kind == kOPROJ || kind == kDOWN) {
    // the residual rows this CTA updates: complete since an earlier phase
    po.ep_old = epoch_of(seq, kind == kOPROJ ? ph - 3 : ph - 2);
    po.base = r.r0 & ~1;
    if (kind == kOPROJ && layer == 0) {
      const int nr = r.r1 - po.base;
      for (int i = ct; i < nr * BT; i += kPConsumerThreads) {
        const int b = i / nr, jr = i % nr;
        const float old = b < a.B ? bf16_to_f32(a.embed[(size_t)S.tok[b] * a.H + po.base + jr]) : 0.f;
        S.xoldw[b][jr] = (static_cast<uint64_t>(po.ep_old) << 32) | __float_as_uint(old);
      }
    } else {
      const int npair = (r.r1 - po.base + 1) / 2;
      for (int i = ct; i < npair * BT; i += kPConsumerThreads) {
        const int b = i / npair, q = i % npair;
        if (b < a.B) cp_async16(&S.xoldw[b][2 * q], a.xw + (size_t)b * a.H + po.base + 2 * q);
      }
    }
  }
  if (kind == kQKV && P->b_qkv) {
    po.base = r.r0 & ~7;
    po.bias = true;
    const int nchunk = (r.r1 - po.base + 7) / 8;
    for (int i = ct; i < nchunk; i += kPConsumerThreads)
      cp_async16(&S.biasr[8 * i], P->b_qkv + po.base + 8 * i);
  }
  cp_async_commit();
  if (kind == kQKV) {
    gather_input<BT>(a, a.xw, K, K, epoch_of(seq, ph - 1), layer == 0 ? a.embed : nullptr,
                     P->g_attn, sp);
  } else if (kind == kOPROJ) {
    // the attention output words, merged over the position splits
    gather_input<BT>(a, a.aw, K, K, epoch_of(seq, ph - 1), nullptr, nullptr, sp);
  } else if (kind == kGU) {
    gather_input<BT>(a, a.xw, K, K, epoch_of(seq, ph - 1), nullptr, P->g_mlp, sp);
  } else if (kind == kDOWN) {
    gather_input<BT>(a, a.hw, K, K, epoch_of(seq, ph - 1), nullptr, nullptr, sp);
  } else {
    gather_input<BT>(a, a.xw, K, K, epoch_of(seq, ph - 1), nullptr, a.g_final, sp);
  }
  if (prof) prof[2 * ph + 1] = global_timer();
  po.words = kind == kQKV ? a.qkvw : (kind == kGU ? a.hw : a.xw);
  po.logits = a.logits;
  po.stride = kind == kQKV ? a.nqkv : (kind == kGU ? a.F : (kind == kHEAD ? a.V : a.H));
  if constexpr (BT == 1) {
    // rows of at most 1024: input in registers; longer rows: whole rows per
    // warp when the phase gives every warp at least two units, else the k
    // range split over the warps (a few long rows on the latency chain)
    if (K / 8 <= kXReg * kWarp) gemv_tiles<1, 0>(a, r, po, kind, ep, rp_io, kb_io, best_io, sp);
    else if (r.r1 - r.r0 >= 2 * kPConsumerWarps)
      gemv_tiles<1, 3>(a, r, po, kind, ep, rp_io, kb_io, best_io, sp);
    else gemv_tiles<1, 1>(a, r, po, kind, ep, rp_io, kb_io, best_io, sp);
  } else {
    gemv_tiles<BT, 2>(a, r, po, kind, ep, rp_io, kb_io, best_io, sp);
  }
}

// ------------------------------------------------------------------ the kernel
// The attention phase of one CTA: its items. Head size 64 takes the
// block-wide scan; head size 128 the per-warp scan, instantiated for the
// group size rounded up to a power of two, at most 4 (an 8-head instance's
// registers would crowd the projection phases' code out of registers;
// persistent_supported keeps such shapes on the stage path). A function of
// its own, so that the kernel's loop keeps few values live across the call.
template <int D, bool KV16>
__device__ __noinline__ void attention_phase(const PersistArgs& a, int ph, int layer, uint32_t seq,
                                             uint32_t ep, int nslots, RingPos& rp, Spin& sp,
                                             unsigned long long* prof) {
  extern __shared__ __align__(128) char smem[];
  const PShared& S = *reinterpret_cast<const PShared*>(smem);
  const uint32_t eq = epoch_of(seq, ph - 1);
  const int G = a.Hq / a.Hkv;
  bool first = true;
  for (int it = blockIdx.x; it < S.item0[kPMaxBatch]; it += gridDim.x) {
    const AttnItem t = attn_item_of(S, a.Hkv, it);
    const int np = cached_positions(a, t.b, S.pos[t.b]);
    const int p0 = (int)(((long long)t.sp * np) / t.ns);
    const int p1 = (int)(((long long)(t.sp + 1) * np) / t.ns);
    unsigned long long* const pin = first && prof ? prof + 2 * ph + 1 : nullptr;
    unsigned long long* const psub =
        pin ? prof + 2 * (kPhasesPerLayer * a.L + 1) + 2 + kProfAttnMarks * layer : nullptr;
    if constexpr (D == 64) {
      attention_item_block<D, KV16>(a, t.b, t.g, t.sp, t.ns, p0, p1, layer, eq, ep, nslots, rp, sp,
                                    pin, psub);
    } else {
      if (G <= 2)
        attention_item<D, KV16, 2>(a, t.b, t.g, t.sp, t.ns, p0, p1, layer, eq, ep, nslots, rp, sp,
                                   pin, psub);
      else
        attention_item<D, KV16, 4>(a, t.b, t.g, t.sp, t.ns, p0, p1, layer, eq, ep, nslots, rp, sp,
                                   pin, psub);
    }
    first = false;
  }
  if (prof && first) prof[2 * ph + 1] = global_timer();  // a CTA with no item
}

template <int BT, int D, bool KV16>
__global__ void __launch_bounds__(kPThreads, 1) k_decode_persistent(const __grid_constant__ PersistArgs a) {
  extern __shared__ __align__(128) char smem[];
  PShared& S = *reinterpret_cast<PShared*>(smem);
  const int slot_bytes = a.slot_bytes, nslots = a.nslots;
  char* ring = smem + a.ring_offset;
  const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;

  if (threadIdx.x == 0) {
    for (int s = 0; s < nslots; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], kPConsumerWarps);
    }
    S.abort = 0;
    S.issued = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (threadIdx.x < BT) {
    const int b = threadIdx.x;
    S.pos[b] = b < a.B ? a.positions[b] : 0;
    int t = b < a.B ? a.tokens[b] : 0;
    if (t < 0 || t >= a.V) {
      if (a.status) atomicCAS(a.status, 0, (int)NC_ERR_INVALID_ARGUMENT);
      t = 0;
    }
    S.tok[b] = t;
  }
  if (threadIdx.x < kHEAD + 1)
    S.rows[threadIdx.x] = kind_rows(a, threadIdx.x, blockIdx.x, gridDim.x, a.slot_bytes);
  if (threadIdx.x == kWarp) attn_plan(a, gridDim.x, S.nsplit, S.item0);
  {  // the per-layer pointer table, copied once
    const int words = a.L * (int)(sizeof(PLayer) / sizeof(uint64_t));
    const uint64_t* src = reinterpret_cast<const uint64_t*>(a.layers);
    uint64_t* dst = reinterpret_cast<uint64_t*>(S.layers);
    for (int i = threadIdx.x; i < words; i += blockDim.x) dst[i] = src[i];
  }
  __syncthreads();
  const uint32_t seq = *reinterpret_cast<volatile const unsigned*>(a.seq);
  Spin sp{global_timer() + a.timeout_ns, &S.abort, a.status};
  const int nph_all = kPhasesPerLayer * a.L + 1;
  unsigned long long* const prof_cta =
      a.prof ? a.prof + (size_t)blockIdx.x * prof_values(a.L) : nullptr;
  if (prof_cta && threadIdx.x == 0) prof_cta[2 * nph_all] = global_timer();

  if (warp == 0) {
    if (lane == 0) producer<KV16>(a, S, ring, slot_bytes, nslots, sp);
  } else {
    const int ct = threadIdx.x - kWarp, cw = ct / kWarp;
    const int L = a.L, nph = kPhasesPerLayer * L + 1;
    // RoPE angles of this step's positions, read by the attention items
    for (int i = ct; i < BT * (D / 2); i += kPConsumerThreads) {
      const int b = i / (D / 2), j = i % (D / 2);
      float sn, cs;
      sincosf(__fmul_rn((float)S.pos[b], a.inv_freq[j]), &sn, &cs);
      S.rope_cs[b][j] = cs;
      S.rope_sn[b][j] = sn;
    }
    consumer_sync();
    RingPos rp;
    int kb = 0;  // k-split partial-sum buffer of the next split tile
    unsigned long long best[BT];
#pragma unroll
    for (int b = 0; b < BT; ++b) best[b] = 0ull;
    for (int ph = 0; ph < nph; ++ph) {
      // Uniform across the consumer warps, and a barrier: no warp overwrites
      // the shared input vector while another still reduces against it.
      if (consumer_any(*reinterpret_cast<volatile int*>(&S.abort) != 0)) break;
      unsigned long long* const prof = ct == 0 ? prof_cta : nullptr;
      if (prof) prof[2 * ph] = global_timer();
      const int layer = ph / kPhasesPerLayer;
      const int kind = ph == kPhasesPerLayer * L ? kHEAD : ph % kPhasesPerLayer;
      const uint32_t ep = epoch_of(seq, ph);
      if (kind == kATTN) {
        attention_phase<D, KV16>(a, ph, layer, seq, ep, nslots, rp, sp, prof);
        continue;
      }
      gemv_phase<BT>(a, ph, seq, rp, kb, best, prof, sp);
    }
    // per-CTA arg-max partials (any lane of a warp may hold a row's key)
#pragma unroll
    for (int b = 0; b < BT; ++b) {
      unsigned long long m = best[b];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long t = __shfl_xor_sync(0xFFFFFFFFu, m, o);
        m = t > m ? t : m;
      }
      if (lane == 0) S.best[cw][b] = m;
    }
  }
  __syncthreads();
  // Drain: copies issued but never consumed (only after an abort) must land
  // before the CTA exits. Only the last fill of each slot can be pending: tile
  // t fills slot t % nslots for the (t / nslots)-th time. Waits are bounded.
  if (threadIdx.x == 0 && S.abort) {
    const uint64_t dl = global_timer() + a.timeout_ns;
    const unsigned issued = S.issued;
    for (unsigned t = issued > (unsigned)nslots ? issued - nslots : 0u; t < issued; ++t) {
      while (!mbar_try_wait(&S.full[t % nslots], (t / nslots) & 1))
        if (global_timer() > dl) break;
    }
  }
  if (threadIdx.x < BT && threadIdx.x < a.B) {
    unsigned long long m = 0ull;
    for (int w = 0; w < kPConsumerWarps; ++w) m = S.best[w][threadIdx.x] > m ? S.best[w][threadIdx.x] : m;
    a.am_part[(size_t)threadIdx.x * gridDim.x + blockIdx.x] = S.abort ? ~0ull : m;
  }
  __threadfence();
  __syncthreads();
  if (prof_cta && threadIdx.x == 0) prof_cta[2 * nph_all + 1] = global_timer();
  if (threadIdx.x == 0) S.last = atomicAdd(a.ticket, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!S.last) return;
  __threadfence();
  if (warp < BT && warp < a.B) {
    const int b = warp;
    unsigned long long m = 0ull;
    for (int i = lane; i < (int)gridDim.x; i += kWarp) {
      const unsigned long long k = __ldcg(a.am_part + (size_t)b * gridDim.x + i);
      m = k > m ? k : m;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long t = __shfl_xor_sync(0xFFFFFFFFu, m, o);
      m = t > m ? t : m;
    }
    if (lane == 0) {
      const bool bad = m == ~0ull;
      const int32_t tok = bad ? -1 : (int32_t)(0xFFFFFFFFu - (uint32_t)(m & 0xFFFFFFFFull));
      if (a.next) a.next[b] = tok;
      if (bad && a.status) atomicCAS(a.status, 0, (int)NC_ERR_INVALID_ARGUMENT);
      if (a.advance) {
        a.tokens[b] = bad ? 0 : tok;
        a.positions[b] = S.pos[b] + 1;
      }
    }
  }
  // the split tickets of every layer start the next step at zero (also
  // after an abort left some of them short)
  for (int i = threadIdx.x; i < a.L * kPMaxBatch * a.Hkv; i += blockDim.x) a.atick[i] = 0u;
  __syncthreads();
  if (threadIdx.x == 0) {
    *a.seq = seq + 1;  // next step's epochs
    if (prof_cta) prof_cta[2 * nph_all + 1] = global_timer();
    *a.ticket = 0u;
    __threadfence();
  }
}

// ------------------------------------------------------------------ host side
// Shared-memory plan: PShared, the input vector [BT][max(H, Hq D, F)] fp32,
// the attention scratch, then the weight ring in the rest.
static int bt_of(int B) { return B <= 1 ? 1 : B <= 2 ? 2 : 4; }
static int kmax_of(int H, int qd, int F) { return H > qd ? (H > F ? H : F) : (qd > F ? qd : F); }
static size_t round128(size_t x) { return (x + 127) / 128 * 128; }

static size_t attn_scratch_bytes(int D) {
  return sizeof(float) * (8 * D + 2 * D + 2 * 8 * kAttnMaxChunk + 3 * 8);
}
// The longest row a ring slot must hold: a gate|up pair (2 rows of H), a
// down row (F), an o-proj row (Hq D) or a QKV / LM-head row (H), bf16.
static size_t max_row_bytes(int H, int qd, int F) {
  size_t m = (size_t)4 * H;
  if ((size_t)2 * F > m) m = (size_t)2 * F;
  if ((size_t)2 * qd > m) m = (size_t)2 * qd;
  return m;
}

// Ring slots (NC_PERSIST_SLOTS in the environment, read once; kPSlots by
// default): the same shared memory cut into more, smaller tiles.
static int persist_slots() {
  static const int n = [] {
    const char* e = getenv("NC_PERSIST_SLOTS");
    int v = e ? atoi(e) : kPSlots;
    return v < kPSlots ? kPSlots : (v > kMaxSlots ? kMaxSlots : v);
  }();
  return n;
}

// The input-vector region: BT rows of the longest input, and at least one
// split's partial block (G heads of D + 4 floats), which the attention merge
// stages there.
static size_t xs_bytes(int H, int qd, int F, int D, int G, int BT) {
  // also the attention scan's combine buffer [consumer warps][G][D]
  size_t v = (size_t)BT * kmax_of(H, qd, F) * 4;
  const size_t p = (size_t)G * (D + 4) * 4, c = (size_t)kPConsumerWarps * G * D * 4;
  if (p > v) v = p;
  return c > v ? c : v;
}
static size_t persistent_fixed_smem(int H, int qd, int F, int D, int G, int BT) {
  size_t off = round128(sizeof(PShared));
  off = round128(off + xs_bytes(H, qd, F, D, G, BT));
  off += attn_scratch_bytes(D);
  return round128(off);
}

template <int BT, int D, bool KV16>
static cudaError_t launch_bt(const PersistArgs& a, size_t smem, cudaStream_t s) {
  auto kern = k_decode_persistent<BT, D, KV16>;
  static const cudaError_t attr =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem_optin());
  if (attr != cudaSuccess) return attr;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(a.grid);
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeCooperative;
  attrs[0].val.cooperative = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int BT>
static cudaError_t launch_b(const PersistArgs& a, size_t smem, cudaStream_t s) {
  if (a.D == 64) return a.kv.bf16 ? launch_bt<BT, 64, true>(a, smem, s) : launch_bt<BT, 64, false>(a, smem, s);
  return a.kv.bf16 ? launch_bt<BT, 128, true>(a, smem, s) : launch_bt<BT, 128, false>(a, smem, s);
}

cudaError_t launch_persistent(PersistArgs a, cudaStream_t s) {
  const int qd = a.Hq * a.D, BT = bt_of(a.B), G = a.Hq / a.Hkv;
  const size_t fixed = persistent_fixed_smem(a.H, qd, a.F, a.D, G, BT);
  const size_t pshared = round128(sizeof(PShared));
  a.xs_offset = (int)pshared;
  a.attn_offset = (int)round128(pshared + xs_bytes(a.H, qd, a.F, a.D, G, BT));
  a.ring_offset = (int)fixed;
  a.attn_bytes = (int)attn_scratch_bytes(a.D);
  const size_t avail = (size_t)max_smem_optin();
  if (fixed + (size_t)kPMinSlotBytes * kPSlots > avail) return cudaErrorInvalidConfiguration;
  // the rest of shared memory as equal slots (multiples of 128 bytes), each
  // holding at least one row of every matrix: NC_PERSIST_SLOTS slots
  // (default kPSlots), fewer when a row would not fit
  const size_t row_max = max_row_bytes(a.H, qd, a.F);
  int ns = persist_slots();
  while (ns > kPSlots && ((avail - fixed) / ns / 128 * 128 < row_max ||
                          (avail - fixed) / ns < (size_t)kPMinSlotBytes))
    --ns;
  a.nslots = ns;
  a.slot_bytes = (int)(((avail - fixed) / ns) / 128 * 128);
  if ((size_t)a.slot_bytes < row_max) return cudaErrorInvalidConfiguration;
  const size_t smem = fixed + (size_t)a.nslots * a.slot_bytes;
  if (BT == 1) return launch_b<1>(a, smem, s);
  if (BT == 2) return launch_b<2>(a, smem, s);
  return launch_b<4>(a, smem, s);
}

bool persistent_supported(int L, int H, int qd, int F, int D, int G, int B) {
  if (B < 1 || B > kPMaxBatch || (D != 64 && D != 128)) return false;
  if (L < 1 || L > kPMaxLayers) return false;
  if (G < 1 || G > 8 || G * (D / 2) > kPConsumerThreads) return false;
  if (D == 128 && G > 4) return false;  // the scan instances (attention_phase)
  if (H % 8 || qd % 8 || F % 8) return false;
  if (G + 2 > kPConsumerWarps) return false;  // one gathering warp per q head, k and v
  if (qd / D > kPMaxHeads) return false;
  // rows one CTA may own: the o-proj rows go to at least half of the CTAs
  const int grid = num_sms(), half = grid - grid / 2;
  const long long nqkv = (long long)qd + 2LL * (qd / G);
  if ((H + half - 1) / half > kPMaxRows || (nqkv + grid - 1) / grid > kPMaxRows) return false;
  const size_t fixed = persistent_fixed_smem(H, qd, F, D, G, bt_of(B));
  if (fixed + (size_t)kPMinSlotBytes * kPSlots > (size_t)max_smem_optin()) return false;
  // every row of every matrix fits one slot
  return ((size_t)max_smem_optin() - fixed) / kPSlots / 128 * 128 >= max_row_bytes(H, qd, F);
}

}  // namespace nc
