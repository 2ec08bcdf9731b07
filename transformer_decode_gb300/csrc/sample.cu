// sample.cu -- token sampling from rows of logits: temperature, top-k, top-p
// and an inverse-CDF draw, one CTA of 1024 threads per row.
//
// nanoinfer, sampling section ("sampling.py: temperature, top-k, top-p,
// seeded draw"): the order is temperature -> top-k -> top-p -> softmax ->
// draw, and temperature 0 is the arg-max (lowest index on ties). The
// truncations are the transformers warpers the page checks against: top-k
// keeps every score >= the k-th largest (ties at the k-th place stay); top-p
// orders the kept scores ascending, stable (equal scores in index order), and
// drops each token whose running fp32 softmax sum is <= 1 - p, the largest
// always staying. The draw is the first kept token whose running weight
// exceeds u times the total (the page: an inverse-CDF search, which needs no
// weights summing to exactly one).
//
// Precision and order, chosen so every integer decision is taken the way
// the definition states it:
//   * s = v / T is an IEEE fp32 division; its order key folds -0 into +0.
//   * top-p's weights e = expf(s - max) are fp32; their total and the running
//     sums are folded by one warp in the sorted order, one fp32 addition at a
//     time (all lanes carry the same chain), each addend e_j / total an IEEE
//     division.
//   * the draw uses the same fp32 weights summed in fp64 in index order
//     (per-thread segments, then a block scan), so only its association
//     differs from a serial fp64 sum.
//
// After both truncations the kept set is {i : (key_i << 32 | i) >= C} for one
// 64-bit threshold C, which is all the draw needs.
//
// Work per row: pass 0 writes the scores' keys to scratch and, with top-k,
// a histogram of their top 12 bits (warp-aggregated shared atomics: scores
// crowd into few bins). When the bins holding the k largest keys hold at
// most 8192 tokens (the usual case: top-k 20 keeps tens), one more pass
// gathers those candidates into shared memory and everything else (the
// k-th key, top-p, the draw) runs on them there. Otherwise top-k finishes
// as a radix select over the keys (10 more bits per pass); top-p sorts the
// kept (key, index) pairs in shared memory (bitonic) up to 8192 of them,
// else with a stable 4-bit LSD radix sort in scratch; the draw reads the
// keys once more. Invalid rows (NaN logits; at T > 0 a +inf score or all
// scores -inf) give token -1.
#include <float.h>

#include "kernels.h"

namespace nc {
namespace {

constexpr int kT = 1024;           // threads per CTA (one row)
constexpr int kWarps = kT / kWarp;
constexpr int kSmallCap = 8192;    // kept sets sorted in shared memory
constexpr int kBins0 = 4096;       // first select pass: the keys' top 12 bits
// comp (pairs) + e (weights) + dr (index-ordered draw list); the candidate
// path's bucket counters (33 x kT u16) alias comp and e
constexpr size_t kDynSmem = (size_t)kSmallCap * (2 * sizeof(unsigned long long) + sizeof(float));
constexpr unsigned kFull = 0xFFFFFFFFu;

struct SampleShared {
  uint32_t hist[kBins0];
  uint32_t red32[kWarps];
  unsigned long long red64[kWarps];
  double redd[kWarps];
  uint32_t bc[8];
  uint32_t btot[33];
  unsigned long long bc64;
};

// Order key of a score (larger score -> larger key); -0 and +0 share a key.
__device__ __forceinline__ uint32_t score_key(float s) {
  uint32_t u = __float_as_uint(s);
  if ((u & 0x7FFFFFFFu) == 0) u = 0;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_score(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}
__device__ __forceinline__ unsigned long long pair_key(uint32_t k, uint32_t i) {
  return (static_cast<unsigned long long>(k) << 32) | i;
}

// One pass over a row of V elements: U coalesced loads per thread are
// issued before any is used (one load in flight per warp would leave a pass
// waiting on L2 latency), then f(i, value) runs for each, in order; lanes
// past the end get i >= V and value 0 (every lane calls f, so f may use
// warp-wide votes).
template <int U, typename T, typename F>
__device__ __forceinline__ void row_pass(const T* x, int V, F&& f) {
  for (int base = 0; base < V; base += U * kT) {
    T v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * kT + (int)threadIdx.x;
      v[u] = i < V ? x[i] : T(0);  // plain loads: keys are written earlier in this kernel
    }
#pragma unroll
    for (int u = 0; u < U; ++u) f(base + u * kT + (int)threadIdx.x, v[u]);
  }
}
constexpr int kUnroll = 16;

// ---------------------------------------------------------------- block reductions
// Every thread of the CTA calls these and receives the result; the scratch
// word array is free again when they return.
__device__ uint32_t block_max_u32(uint32_t v, uint32_t* sh) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(kFull, v, o));
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = v;
  __syncthreads();
  v = sh[threadIdx.x & 31];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(kFull, v, o));
  __syncthreads();
  return v;
}
__device__ uint32_t block_min_u32(uint32_t v, uint32_t* sh) {
  return ~block_max_u32(~v, sh);
}
__device__ unsigned long long block_max_u64(unsigned long long v, unsigned long long* sh) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(kFull, v, o));
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = v;
  __syncthreads();
  v = sh[threadIdx.x & 31];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(kFull, v, o));
  __syncthreads();
  return v;
}
// Exclusive prefix sum over the CTA in thread order; *total gets the sum.
__device__ uint32_t block_excl_scan_u32(uint32_t v, uint32_t* sh, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh[warp] = x;
  __syncthreads();
  const uint32_t w = sh[lane];
  uint32_t wi = w;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(kFull, wi, o);
    if (lane >= o) wi += y;
  }
  const uint32_t wex = __shfl_sync(kFull, wi - w, warp);
  *total = __shfl_sync(kFull, wi, 31);
  __syncthreads();
  return wex + x - v;
}
// The same in fp64 (a fixed association, so the result is deterministic);
// *incl gets this thread's inclusive sum.
__device__ double block_excl_scan_f64(double v, double* sh, double* incl, double* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  double x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  double xe = __shfl_up_sync(kFull, x, 1);
  if (lane == 0) xe = 0.0;
  if (lane == 31) sh[warp] = x;
  __syncthreads();
  double wi = sh[lane];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_up_sync(kFull, wi, o);
    if (lane >= o) wi += y;
  }
  double wprev = __shfl_up_sync(kFull, wi, 1);
  if (lane == 0) wprev = 0.0;
  const double wex = __shfl_sync(kFull, wprev, warp);
  *total = __shfl_sync(kFull, wi, 31);
  *incl = wex + x;
  __syncthreads();
  return wex + xe;
}

// ---------------------------------------------------------------- the serial folds
// Run by one whole warp: every lane carries the same fp32 chain, fed the
// values in order through shuffles, so the result is the plain left-to-right
// sum e[0] + e[1] + ... of the definition.
__device__ float warp_serial_sum(const float* e, int n) {
  const int lane = threadIdx.x & 31;
  float acc = 0.f;
  for (int base = 0; base < n; base += 32) {
    const float v = base + lane < n ? e[base + lane] : 0.f;
    const int cnt = min(32, n - base);
#pragma unroll
    for (int q = 0; q < 32; ++q) {
      const float y = __shfl_sync(kFull, v, q);
      if (q < cnt) acc = __fadd_rn(acc, y);
    }
  }
  return acc;
}
// The top-p cut over ascending weights e[0..n): the first j < n - 1 whose
// running sum c_j = c_{j-1} + e_j / tot exceeds thr, else n - 1. Tokens
// before the cut are dropped.
__device__ int warp_cut(const float* e, int n, float tot, float thr) {
  const int lane = threadIdx.x & 31;
  float c = 0.f;
  for (int base = 0; base < n - 1; base += 32) {
    const int j = base + lane;
    const float pj = j < n - 1 ? __fdiv_rn(e[j], tot) : 0.f;
    const int cnt = min(32, n - 1 - base);
#pragma unroll
    for (int q = 0; q < 32; ++q) {
      const float y = __shfl_sync(kFull, pj, q);
      if (q < cnt) {
        c = __fadd_rn(c, y);
        if (c > thr) return base + q;  // the same in every lane
      }
    }
  }
  return n - 1;
}

// The bin, among BPT * kT counts, that holds the need-th largest key (bins
// scanned from the top): sh.bc = {bin, count in higher bins, count in bin}.
template <int BPT>
__device__ void select_bin(const uint32_t* hist, uint32_t need, SampleShared& sh) {
  constexpr int nb = BPT * kT;
  uint32_t c[BPT], sum = 0;
#pragma unroll
  for (int j = 0; j < BPT; ++j) {
    c[j] = hist[nb - 1 - (BPT * (int)threadIdx.x + j)];
    sum += c[j];
  }
  uint32_t total;
  const uint32_t exc = block_excl_scan_u32(sum, sh.red32, &total);
  if (exc < need && exc + sum >= need) {  // exactly one thread
    uint32_t above = exc, bin = 0, cnt = 0;
    bool found = false;
#pragma unroll
    for (int j = 0; j < BPT; ++j) {
      if (!found) {
        if (above + c[j] >= need) {
          found = true;
          bin = nb - 1 - (BPT * threadIdx.x + j);
          cnt = c[j];
        } else {
          above += c[j];
        }
      }
    }
    sh.bc[0] = bin;
    sh.bc[1] = above;
    sh.bc[2] = cnt;
  }
  __syncthreads();
}

// Ascending bitonic sort of n2 (a power of two, >= 2) 64-bit words in shared memory.
__device__ void bitonic_sort_u64(unsigned long long* a, int n2) {
  for (int size = 2; size <= n2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      __syncthreads();
      for (int t = threadIdx.x; t < (n2 >> 1); t += kT) {
        const int lo = 2 * t - (t & (stride - 1));
        const int hi = lo + stride;
        const bool up = (lo & size) == 0;
        const unsigned long long x = a[lo], y = a[hi];
        if ((x > y) == up) {
          a[lo] = y;
          a[hi] = x;
        }
      }
    }
  }
  __syncthreads();
}

// Stable ascending sort of n (key, index) pairs by key: 4-bit LSD radix,
// each thread owning a contiguous segment, digit counters in shared memory
// (cnt: 16 x kT words). Returns which buffer holds the result (0: k0/i0).
__device__ int radix_sort_pairs(uint32_t* k0, uint32_t* i0, uint32_t* k1, uint32_t* i1, int n,
                                uint32_t* cnt, uint32_t* red) {
  const int tid = threadIdx.x;
  const int seg = (n + kT - 1) / kT;
  const int lo = min(n, tid * seg), hi = min(n, lo + seg);
  int cur = 0;
  for (int pass = 0; pass < 8; ++pass) {
    const int shift = 4 * pass;
    uint32_t* sk = cur ? k1 : k0;
    uint32_t* si = cur ? i1 : i0;
    uint32_t* dk = cur ? k0 : k1;
    uint32_t* di = cur ? i0 : i1;
#pragma unroll
    for (int d = 0; d < 16; ++d) cnt[d * kT + tid] = 0;
    for (int i = lo; i < hi; ++i) cnt[((sk[i] >> shift) & 15u) * kT + tid] += 1;
    __syncthreads();
    // Exclusive scan of the counters in digit-major order (digit, thread):
    // thread t scans the 16 consecutive entries [16 t, 16 t + 16).
    uint32_t loc[16];
    uint32_t s = 0;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      loc[j] = cnt[16 * tid + j];
      s += loc[j];
    }
    uint32_t total;
    uint32_t base = block_excl_scan_u32(s, red, &total);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      cnt[16 * tid + j] = base;
      base += loc[j];
    }
    __syncthreads();
    // A digit holding every element leaves the order as it is.
    bool skip = false;
#pragma unroll
    for (int d = 0; d < 16; ++d) {
      const uint32_t start = cnt[d * kT];
      const uint32_t end = d < 15 ? cnt[(d + 1) * kT] : (uint32_t)n;
      skip |= (end - start) == (uint32_t)n;
    }
    __syncthreads();
    if (!skip) {
      for (int i = lo; i < hi; ++i) {
        const uint32_t k = sk[i];
        const uint32_t dst = cnt[((k >> shift) & 15u) * kT + tid]++;
        dk[dst] = k;
        di[dst] = si[i];
      }
      cur ^= 1;
    }
    __syncthreads();
  }
  return cur;
}

struct SampleArgs {
  const float* logits;  // [B, V]
  int B, V;
  float temperature;
  int top_k;
  float top_p;
  const double* u;      // [B] uniforms in [0, 1)
  int32_t* tokens;      // [B]
  int32_t* kept;        // [B, 2] or null: kept after top-k, after top-p
  uint32_t* scratch;    // B rows of row_stride words: keys, then k0, i0, k1, i1
  size_t vpad;          // V rounded up to 64 (one scratch array)
};

__device__ void finish(const SampleArgs& a, int row, int tok, uint32_t nk, uint32_t np) {
  a.tokens[row] = tok;
  if (a.kept) {
    a.kept[2 * row] = (int32_t)nk;
    a.kept[2 * row + 1] = (int32_t)np;
  }
}

// fp64 inverse-CDF draw over n (index << 32 | fp32 weight bits) words sorted
// by index: per-thread contiguous segments, a block scan, and the thread
// whose segment crosses u * total walks it. Returns the token to thread 0
// through sh.bc[6].
__device__ void draw_list(const unsigned long long* dr, int n, double u, SampleShared& sh) {
  const int tid = threadIdx.x;
  const int seg = (n + kT - 1) / kT;
  const int lo = min(n, tid * seg), hi = min(n, lo + seg);
  double part = 0.0;
  int last = -1;
  for (int t = lo; t < hi; ++t) {
    const float w = __uint_as_float((uint32_t)dr[t]);
    if (w > 0.f) {
      part += (double)w;
      last = (int)(dr[t] >> 32);
    }
  }
  double incl, total;
  const double excl = block_excl_scan_f64(part, sh.redd, &incl, &total);
  const double r = u * total;
  const uint32_t win = block_min_u32(part > 0.0 && incl > r ? (uint32_t)tid : kFull, sh.red32);
  const uint32_t lastpos = block_max_u32((uint32_t)(last + 1), sh.red32);
  if (win == kFull) {
    if (tid == 0) sh.bc[6] = lastpos - 1;
  } else if ((uint32_t)tid == win) {
    double c = excl;
    int tok = -1, lastw = -1;
    for (int t = lo; t < hi; ++t) {
      const float w = __uint_as_float((uint32_t)dr[t]);
      if (w > 0.f) {
        c += (double)w;
        lastw = (int)(dr[t] >> 32);
        if (c > r) {
          tok = lastw;
          break;
        }
      }
    }
    sh.bc[6] = (uint32_t)(tok >= 0 ? tok : lastw);
  }
  __syncthreads();
}

// The candidate path, for 0 < k <= kSmallCap. s = v / T rounds a monotone
// map, so the k largest scores belong to the k largest logits; the buckets
// of log2 distance (in order keys) from the largest logit are counted
// (pass B: per-thread u16 counters in shared memory, no atomics), and the
// tokens of the fewest leading buckets that hold at least k are gathered
// (pass C, dividing only those by T) into shared memory and sorted ascending
// by (score key, index). The k-th largest key K, the kept suffix, the top-p
// cut and the draw then all work there. A token outside the gathered set
// has a logit key <= lkmax - 2^B, so its score key is at most that of
// v_out / T; the path is taken only when K is above that (else a tie across
// the boundary is possible) and the gathered set fits: returns false, with
// nothing written, otherwise.
__device__ bool sample_candidates(const SampleArgs& a, int row, const float* x, uint32_t lkmax,
                                  float m, SampleShared& sh, unsigned char* dyn) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = a.V;
  // pass B: bucket 0 holds distance 0, bucket b >= 1 distances [2^(b-1), 2^b)
  uint16_t* cnt = reinterpret_cast<uint16_t*>(dyn);  // [33][kT], dead after the totals
#pragma unroll
  for (int b = 0; b < 33; ++b) cnt[b * kT + tid] = 0;
  row_pass<kUnroll>(x, V, [&](int i, float v) {
    if (i < V) {
      const uint32_t d = lkmax - score_key(v);
      const int b = d == 0 ? 0 : 32 - __clz(d);
      cnt[b * kT + tid] += 1;
    }
  });
  __syncthreads();
  for (int b = warp; b < 33; b += kWarps) {
    uint32_t t = 0;
    for (int j = lane; j < kT; j += 32) t += cnt[b * kT + j];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(kFull, t, o);
    if (lane == 0) sh.btot[b] = t;
  }
  __syncthreads();
  if (tid == 0) {
    uint32_t cum = 0;
    int B = 32;
    for (int b = 0; b < 33; ++b) {
      cum += sh.btot[b];
      if (cum >= (uint32_t)a.top_k) {
        B = b;
        break;
      }
    }
    sh.bc[0] = (uint32_t)B;
    sh.bc[1] = cum;
    sh.bc[3] = 0;
  }
  __syncthreads();
  const int B = (int)sh.bc[0];
  const uint32_t n_c = sh.bc[1];
  if (n_c > (uint32_t)kSmallCap) return false;
  const unsigned long long lim = 1ull << B;  // candidates: distance < lim

  unsigned long long* comp = reinterpret_cast<unsigned long long*>(dyn);
  float* e = reinterpret_cast<float*>(dyn + (size_t)kSmallCap * sizeof(unsigned long long));
  unsigned long long* dr = reinterpret_cast<unsigned long long*>(
      dyn + (size_t)kSmallCap * (sizeof(unsigned long long) + sizeof(float)));
  // pass C: gather (a warp takes its slots with one shared atomic)
  row_pass<kUnroll>(x, V, [&](int i, float v) {
    const bool take = i < V && (unsigned long long)(lkmax - score_key(v)) < lim;
    const unsigned bal = __ballot_sync(kFull, take);
    if (bal) {
      uint32_t slot0 = 0;
      if (lane == 0) slot0 = atomicAdd(&sh.bc[3], (uint32_t)__popc(bal));
      slot0 = __shfl_sync(kFull, slot0, 0);
      if (take) {
        const uint32_t slot = slot0 + __popc(bal & ((1u << lane) - 1u));
        if (slot < (uint32_t)kSmallCap)
          comp[slot] = pair_key(score_key(__fdiv_rn(v, a.temperature)), (uint32_t)i);
      }
    }
  });
  __syncthreads();
  const int nc = (int)n_c;
  int n2 = 2;
  while (n2 < nc) n2 <<= 1;
  for (int j = nc + tid; j < n2; j += kT) comp[j] = ~0ull;
  bitonic_sort_u64(comp, n2);
  // the k-th largest score key, and whether a token outside can reach it
  const uint32_t K = (uint32_t)(comp[nc - a.top_k] >> 32);
  const uint32_t kNegInf = 0x007FFFFFu;  // order key of -inf: the smallest non-NaN key
  if ((unsigned long long)lkmax >= lim + kNegInf) {
    const float v_out = key_score(lkmax - (uint32_t)lim);
    if (K <= score_key(__fdiv_rn(v_out, a.temperature))) return false;
  }
  // the first position holding K: the kept suffix after top-k
  for (int j = tid; j < nc; j += kT) {
    const uint32_t kj = (uint32_t)(comp[j] >> 32);
    if (kj >= K && (j == 0 || (uint32_t)(comp[j - 1] >> 32) < K)) sh.bc[5] = (uint32_t)j;
  }
  __syncthreads();
  const int j0 = (int)sh.bc[5];
  const int nk = nc - j0;
  int j1 = j0;
  if (a.top_p < 1.f && nk > 1) {
    for (int t = tid; t < nk; t += kT)
      e[t] = expf(__fsub_rn(key_score((uint32_t)(comp[j0 + t] >> 32)), m));
    __syncthreads();
    if (warp == 0) {
      const float tot = warp_serial_sum(e, nk);
      const int cut = warp_cut(e, nk, tot, __fsub_rn(1.f, a.top_p));
      if (lane == 0) sh.bc[4] = (uint32_t)cut;
    }
    __syncthreads();
    j1 = j0 + (int)sh.bc[4];
  }
  // the draw over the kept tokens in index order
  const int np = nc - j1;
  int np2 = 1;
  while (np2 < np) np2 <<= 1;
  for (int t = tid; t < np2; t += kT) {
    if (t < np) {
      const unsigned long long c = comp[j1 + t];
      const float w = expf(__fsub_rn(key_score((uint32_t)(c >> 32)), m));
      dr[t] = (c << 32) | __float_as_uint(w);
    } else {
      dr[t] = ~0ull;
    }
  }
  if (np2 >= 2) bitonic_sort_u64(dr, np2);
  __syncthreads();
  draw_list(dr, np, a.u[row], sh);
  if (tid == 0) finish(a, row, (int)sh.bc[6], (uint32_t)nk, (uint32_t)np);
  return true;
}

__global__ void __launch_bounds__(kT, 1) k_sample(const __grid_constant__ SampleArgs a) {
  __shared__ SampleShared sh;
  extern __shared__ __align__(16) unsigned char dyn[];
  const int row = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = a.V;
  const float* x = a.logits + (size_t)row * V;

  // ---- temperature 0: the arg-max, lowest index on ties
  if (a.temperature == 0.f) {
    unsigned long long best = 0;
    uint32_t nan = 0;
    row_pass<kUnroll>(x, V, [&](int i, float v) {
      if (i < V) {
        if (v != v) nan = 1;
        best = max(best, pair_key(score_key(v), 0xFFFFFFFFu - (uint32_t)i));
      }
    });
    nan = block_max_u32(nan, sh.red32);
    best = block_max_u64(best, sh.red64);
    if (tid == 0) {
      if (nan)
        finish(a, row, -1, 0, 0);
      else
        finish(a, row, (int)(0xFFFFFFFFu - (uint32_t)best), 1, 1);
    }
    return;
  }

  // ---- pass A: validity and the largest logit. s = v / T rounds a monotone
  // map, so the largest score is the largest logit's (and is +inf iff some
  // score is; -inf iff every score is).
  uint32_t lkmax = 0, bad = 0;
  row_pass<kUnroll>(x, V, [&](int i, float v) {
    if (i < V) {
      if (v != v) bad = 1;
      lkmax = max(lkmax, score_key(v));
    }
  });
  bad = block_max_u32(bad, sh.red32);
  lkmax = block_max_u32(lkmax, sh.red32);
  const float m = key_score(score_key(__fdiv_rn(key_score(lkmax), a.temperature)));
  if (bad || fabsf(m) == __int_as_float(0x7f800000)) {
    if (tid == 0) finish(a, row, -1, 0, 0);
    return;
  }
  const bool topk = a.top_k > 0 && a.top_k < V;
  if (topk && a.top_k <= kSmallCap && sample_candidates(a, row, x, lkmax, m, sh, dyn)) return;

  // ---- general path, pass 0: every score key to scratch; with top-k, a
  // histogram of their top 12 bits
  uint32_t* keys = a.scratch + (size_t)row * 5 * a.vpad;
  if (topk) {
    for (int j = tid; j < kBins0; j += kT) sh.hist[j] = 0;
    __syncthreads();
  }
  row_pass<kUnroll>(x, V, [&](int i, float v) {
    if (i < V) {
      const uint32_t k = score_key(__fdiv_rn(v, a.temperature));
      keys[i] = k;
      if (topk) atomicAdd(&sh.hist[k >> 20], 1u);
    }
  });
  __syncthreads();

  uint32_t K = 0, nk = (uint32_t)V;
  if (topk) {
    select_bin<kBins0 / kT>(sh.hist, (uint32_t)a.top_k, sh);
    const uint32_t b0 = sh.bc[0], above0 = sh.bc[1], cnt0 = sh.bc[2];
    // ---- the rest of the radix select over the keys, 10 bits per pass
    uint32_t prefix = b0 << 20, pmask = 0xFFF00000u, need = (uint32_t)a.top_k - above0;
    uint32_t ngt = above0, neq = cnt0;
    for (int shift = 10; shift >= 0; shift -= 10) {
      sh.hist[tid] = 0;
      __syncthreads();
      row_pass<kUnroll>(keys, V, [&](int i, uint32_t k) {
        if (i < V && (k & pmask) == prefix) atomicAdd(&sh.hist[(k >> shift) & 1023u], 1u);
      });
      __syncthreads();
      select_bin<1>(sh.hist, need, sh);
      const uint32_t bin = sh.bc[0], above = sh.bc[1];
      neq = sh.bc[2];
      ngt += above;
      need -= above;
      prefix |= bin << shift;
      pmask |= 1023u << shift;
      __syncthreads();
    }
    K = prefix;
    nk = ngt + neq;
  }

  // ---- top-p: ascending (key, index) order of the kept set, serial fp32 folds
  unsigned long long C = pair_key(K, 0);
  uint32_t np = nk;
  if (a.top_p < 1.f && nk > 1) {
    const float thr = __fsub_rn(1.f, a.top_p);
    if (nk <= (uint32_t)kSmallCap) {
      unsigned long long* comp = reinterpret_cast<unsigned long long*>(dyn);
      float* e = reinterpret_cast<float*>(dyn + (size_t)kSmallCap * sizeof(unsigned long long));
      if (tid == 0) sh.bc[3] = 0;
      __syncthreads();
      for (int i = tid; i < V; i += kT) {
        const uint32_t k = keys[i];
        if (k >= K) {
          const uint32_t slot = atomicAdd(&sh.bc[3], 1u);
          if (slot < (uint32_t)kSmallCap) comp[slot] = pair_key(k, (uint32_t)i);
        }
      }
      __syncthreads();
      int n2 = 2;
      while (n2 < (int)nk) n2 <<= 1;
      for (int j = (int)nk + tid; j < n2; j += kT) comp[j] = ~0ull;
      bitonic_sort_u64(comp, n2);
      for (int j = tid; j < (int)nk; j += kT)
        e[j] = expf(__fsub_rn(key_score((uint32_t)(comp[j] >> 32)), m));
      __syncthreads();
      if (warp == 0) {
        const float tot = warp_serial_sum(e, (int)nk);
        const int cut = warp_cut(e, (int)nk, tot, thr);
        if (lane == 0) {
          sh.bc64 = comp[cut];
          sh.bc[4] = (uint32_t)cut;
        }
      }
      __syncthreads();
    } else {
      uint32_t* k0 = keys + a.vpad;
      uint32_t* i0 = keys + 2 * a.vpad;
      uint32_t* k1 = keys + 3 * a.vpad;
      uint32_t* i1 = keys + 4 * a.vpad;
      // kept pairs in index order (a stable compaction)
      const int seg = (V + kT - 1) / kT;
      const int lo = min(V, tid * seg), hi = min(V, lo + seg);
      uint32_t cnt = 0;
      for (int i = lo; i < hi; ++i) cnt += keys[i] >= K;
      uint32_t total;
      uint32_t off = block_excl_scan_u32(cnt, sh.red32, &total);
      for (int i = lo; i < hi; ++i) {
        const uint32_t k = keys[i];
        if (k >= K) {
          k0[off] = k;
          i0[off] = (uint32_t)i;
          ++off;
        }
      }
      __syncthreads();
      const int n = (int)nk;
      const int cur = radix_sort_pairs(k0, i0, k1, i1, n, reinterpret_cast<uint32_t*>(dyn),
                                       sh.red32);
      const uint32_t* sk = cur ? k1 : k0;
      const uint32_t* si = cur ? i1 : i0;
      float* e = reinterpret_cast<float*>(cur ? k0 : k1);  // the free key buffer
      for (int j = tid; j < n; j += kT) e[j] = expf(__fsub_rn(key_score(sk[j]), m));
      __syncthreads();
      if (warp == 0) {
        const float tot = warp_serial_sum(e, n);
        const int cut = warp_cut(e, n, tot, thr);
        if (lane == 0) {
          sh.bc64 = pair_key(sk[cut], si[cut]);
          sh.bc[4] = (uint32_t)cut;
        }
      }
      __syncthreads();
    }
    C = sh.bc64;
    np = nk - sh.bc[4];
  }

  // ---- the draw: fp32 weights of the kept tokens, fp64 sums in index order
  const int seg = (V + kT - 1) / kT;
  const int lo = min(V, tid * seg), hi = min(V, lo + seg);
  double part = 0.0;
  int last = -1;
  for (int i = lo; i < hi; ++i) {
    const uint32_t k = keys[i];
    if (pair_key(k, (uint32_t)i) >= C) {
      const float w = expf(__fsub_rn(key_score(k), m));
      if (w > 0.f) {
        part += (double)w;
        last = i;
      }
    }
  }
  double incl, total;
  const double excl = block_excl_scan_f64(part, sh.redd, &incl, &total);
  const double r = a.u[row] * total;
  const uint32_t win = block_min_u32(part > 0.0 && incl > r ? (uint32_t)tid : kFull, sh.red32);
  const uint32_t lastpos = block_max_u32((uint32_t)(last + 1), sh.red32);  // 0: none
  if (win == kFull) {
    // rounding left u * total at or past every running sum
    if (tid == 0) finish(a, row, (int)lastpos - 1, nk, np);
  } else if ((uint32_t)tid == win) {
    double c = excl;
    int tok = -1, lastw = -1;
    for (int i = lo; i < hi; ++i) {
      const uint32_t k = keys[i];
      if (pair_key(k, (uint32_t)i) >= C) {
        const float w = expf(__fsub_rn(key_score(k), m));
        if (w > 0.f) {
          c += (double)w;
          lastw = i;
          if (c > r) {
            tok = i;
            break;
          }
        }
      }
    }
    finish(a, row, tok >= 0 ? tok : lastw, nk, np);
  }
}

}  // namespace

size_t sample_scratch_bytes(int B, int V) {
  const size_t vpad = ((size_t)V + 63) & ~(size_t)63;
  return (size_t)B * 5 * vpad * sizeof(uint32_t);
}

cudaError_t launch_sample(const float* logits, int B, int V, float temperature, int top_k,
                          float top_p, const double* u, int32_t* tokens, int32_t* kept,
                          void* scratch, cudaStream_t s) {
  cudaError_t e = ensure_smem<k_sample>();
  if (e != cudaSuccess) return e;
  SampleArgs a{logits, B, V, temperature, top_k, top_p, u, tokens, kept,
               static_cast<uint32_t*>(scratch), ((size_t)V + 63) & ~(size_t)63};
  k_sample<<<B, kT, kDynSmem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace nc
