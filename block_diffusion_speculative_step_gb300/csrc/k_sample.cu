// k_sample.cu -- sampling-mode verification: the lossless-in-distribution
// variant of the greedy acceptance ("DFlash：块扩散加速的 LLM 推测解码技术",
// section 7: the path is walked greedily or by sampling, and rejection
// sampling keeps the output distribution exactly the target's).  It is
// speculative sampling at temperature T: drafts are draws from
// q = softmax(draft logits / T); draft d is accepted iff log u < log p(d) -
// log q(d) with p = softmax(target logits / T); the first rejection emits a
// draw from max(0, p - q), and if every draft is accepted a bonus draw from
// the last target row is emitted.
//
// A categorical draw from weights w is the argmax over v of log w_v + g_v
// with g_v Gumbel(0, 1) (Gumbel-max; the exponential race for unnormalised
// weights).  Random numbers: Philox4x32-10 (Salmon, Moraes, Dror, Shaw,
// "Parallel random numbers: as easy as 1, 2, 3", SC'11), key (seed low, seed
// high), counter (vocabulary entry, position, sequence << 8 | purpose,
// cycle); u = ((x0 >> 8) + 1/2) 2^-24.  Every reduction runs in a fixed
// order: the row is cut into kSplit contiguous slices, one CTA each, and the
// last CTA of a row merges the slices in slice order.
#include <limits.h>

#include "common.cuh"
#include "internal.h"
#include "launch.cuh"
#include "rng.cuh"

namespace dfl {

constexpr int kSampleThreads = 256;
constexpr int kSplit = 16;  // CTAs per vocabulary row

// Running state of one slice: log-sum-exp pieces (m, s: sum exp(x - m)) and
// the best draw (score, index; lower index on equal scores).
struct RowAcc {
  float m, s, best;
  int idx;
};

__device__ __forceinline__ RowAcc acc_empty() { return RowAcc{-INFINITY, 0.f, -INFINITY, INT_MAX}; }

__device__ __forceinline__ void acc_lse(RowAcc& a, float x) {
  if (x == -INFINITY) return;  // exp(-inf) adds nothing
  if (x > a.m) {
    a.s = a.s * expf(a.m - x) + 1.f;
    a.m = x;
  } else {
    a.s += expf(x - a.m);
  }
}

__device__ __forceinline__ void acc_draw(RowAcc& a, float sc, int v) {
  if (sc > a.best || (sc == a.best && v < a.idx)) {
    a.best = sc;
    a.idx = v;
  }
}

// Associative merge (the order of merges is fixed by the callers).
__device__ __forceinline__ RowAcc acc_merge(const RowAcc& a, const RowAcc& b) {
  RowAcc r;
  if (b.m == -INFINITY) {
    r.m = a.m;
    r.s = a.s;
  } else if (a.m == -INFINITY) {
    r.m = b.m;
    r.s = b.s;
  } else if (a.m >= b.m) {
    r.m = a.m;
    r.s = a.s + b.s * expf(b.m - a.m);
  } else {
    r.m = b.m;
    r.s = b.s + a.s * expf(a.m - b.m);
  }
  const bool tb = b.best > a.best || (b.best == a.best && b.idx < a.idx);
  r.best = tb ? b.best : a.best;
  r.idx = tb ? b.idx : a.idx;
  return r;
}

// Block-wide merge in a fixed order: lanes by a butterfly, then warps in order.
__device__ __forceinline__ RowAcc block_merge(RowAcc a, RowAcc* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    RowAcc b;
    b.m = __shfl_xor_sync(0xffffffffu, a.m, o);
    b.s = __shfl_xor_sync(0xffffffffu, a.s, o);
    b.best = __shfl_xor_sync(0xffffffffu, a.best, o);
    b.idx = __shfl_xor_sync(0xffffffffu, a.idx, o);
    a = acc_merge(a, b);
  }
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) red[w] = a;
  __syncthreads();
  RowAcc t = red[0];
  for (int i = 1; i < (int)(blockDim.x >> 5); ++i) t = acc_merge(t, red[i]);
  __syncthreads();
  return t;
}

// Last of kSplit slice CTAs of `row` to arrive (its slice partial stored).
__device__ __forceinline__ bool slice_last(uint32_t* ctr, int* s_last) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const uint32_t old = atomicAdd(ctr, 1u);
    *s_last = (old == (uint32_t)kSplit - 1);
    if (*s_last) *ctr = 0u;
  }
  __syncthreads();
  if (*s_last) __threadfence();
  return *s_last != 0;
}

// ---------------------------------------------------- top-k / top-p filter
//
// The kept set of a row: entries ordered by logit (descending, lower index
// first on equal logits), the first top_k of them, then the shortest prefix
// of those whose renormalised softmax(l / T) mass reaches top_p.  It is a
// prefix of that order, held as its last entry (key, idx): v is kept iff
// key(l_v) > key, or key(l_v) == key and v <= idx.  One CTA per row finds it
// by radix selection on the order-preserving key of the logits (four 8-bit
// rounds over the entries that match the key bits chosen so far) and, among
// equal logits, on the index.  Top-p counts masses as integers, w_v =
// floor(exp((l_v - max) / T) 2^32), summed by 64-bit integer atomics, so the
// selection is the same whatever the order of the additions.
constexpr int kFiltThreads = 1024;

__device__ __forceinline__ uint32_t okey(float x) {
  const uint32_t b = __float_as_uint(x);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ bool filt_kept(const RowFilter* f, float l, int v) {
  if (l != l) return false;
  if (f == nullptr) return true;
  const uint32_t k = okey(l);
  return k > f->key || (k == f->key && v <= f->idx);
}

__device__ __forceinline__ unsigned long long filt_mass(float l, float mx, float invT) {
  return __float2ull_rd(expf((l - mx) * invT) * 4294967296.0f);
}

// Histogram of one radix round: one private 256-bin histogram per warp;
// the lanes of a warp that hit the same bin are combined first (match +
// add, the 64-bit weight added as two 16-bit halves, each sum < 2^21) and
// one lane adds the group's total, so no bin is ever updated by two threads
// at once and no atomics are needed (logits concentrate in a few key bytes,
// which made shared atomics on one address the bottleneck).  Integer sums:
// the result does not depend on the order of the additions.
constexpr int kFiltWarps = kFiltThreads / 32;

template <typename In, typename W, typename Bin>
__device__ void filt_hist(const float* l, int V, In in, W weight, Bin bin_of, unsigned long long* hist,
                          unsigned long long* whist) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long* mine = whist + warp * 256;
  for (int i = threadIdx.x; i < kFiltWarps * 256; i += blockDim.x) whist[i] = 0ull;
  __syncthreads();
  // eight elements per thread loaded before any is processed: the warp
  // intrinsics below keep the compiler from moving later loads ahead
  constexpr int U = 8;
  for (int base = warp * 32 * U; base < V; base += blockDim.x * U) {
    float xs[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = base + u * 32 + lane;
      xs[u] = v < V ? l[v] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = base + u * 32 + lane;
      int bin = -1;
      unsigned long long w = 0ull;
      if (v < V && in(xs[u], v)) {
        bin = bin_of(xs[u], v);
        if (bin >= 0) w = weight(xs[u]);
      }
      if (w == 0ull) bin = -1;
      const unsigned peers = __match_any_sync(0xffffffffu, bin);
      const unsigned hi = __reduce_add_sync(peers, (unsigned)(w >> 16));
      const unsigned lo = __reduce_add_sync(peers, (unsigned)(w & 0xFFFFull));
      if (bin >= 0 && lane == __ffs(peers) - 1) mine[bin] += ((unsigned long long)hi << 16) + lo;
      __syncwarp();
    }
  }
  __syncthreads();
  for (int b = threadIdx.x; b < 256; b += blockDim.x) {
    unsigned long long t = 0ull;
    for (int g = 0; g < kFiltWarps; ++g) t += whist[g * 256 + b];
    hist[b] = t;
  }
  __syncthreads();
}

// One warp finds the bin at which the running total of hist -- from bin 255
// down (desc) or from bin 0 up -- first reaches nd (>= 1): lane l sums its 8
// bins, a shuffle scan locates the lane, that lane walks its bins and
// writes the bin, the need left inside it and the bin's own total to shared
// memory (the last bin takes whatever is left, as a serial walk would).
__device__ __forceinline__ void filt_find_bin(const unsigned long long* hist, unsigned long long nd, bool desc,
                                              int* s_bin, unsigned long long* s_need, unsigned long long* s_binv) {
  const int lane = threadIdx.x & 31;
  unsigned long long t = 0ull;
#pragma unroll
  for (int e = 0; e < 8; ++e) t += hist[desc ? 255 - (8 * lane + e) : 8 * lane + e];
  unsigned long long inc = t;  // inclusive scan over lanes
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  const unsigned hit = __ballot_sync(0xffffffffu, inc >= nd);
  const int src = hit ? __ffs(hit) - 1 : 31;
  if (lane == src) {
    unsigned long long acc = inc - t;
    int k = 0;
    for (; k < 7; ++k) {
      const unsigned long long h = hist[desc ? 255 - (8 * lane + k) : 8 * lane + k];
      if (acc + h >= nd) break;
      acc += h;
    }
    const int bn = desc ? 255 - (8 * lane + k) : 8 * lane + k;
    *s_bin = bn;
    *s_need = nd - acc;
    *s_binv = hist[bn];
  }
}

// Among the entries v passing `in(v)`, select by `weight(v)` (1 for counts,
// the integer mass for top-p) the entry at which the running total in the
// order (key descending, index ascending) first reaches `need` (>= 1): its
// key and index.  Radix rounds on the key from the top byte; then, only when
// the boundary falls inside a group of equal logits, on the index
// (ascending) among that group (idx = INT_MAX: the whole group is kept).
template <typename In, typename W>
__device__ void filt_select(const float* l, int V, In in, W weight, unsigned long long need, uint32_t* key_out,
                            int* idx_out, unsigned long long* whist) {
  __shared__ unsigned long long hist[256];
  __shared__ unsigned long long s_need, s_binv;
  __shared__ int s_bin;
  if (threadIdx.x == 0) s_need = need;
  __syncthreads();
  uint32_t prefix = 0u, mask = 0u;
  for (int shift = 24; shift >= 0; shift -= 8) {
    filt_hist(l, V, in, weight,
              [prefix, mask, shift](float x, int) {
                const uint32_t k = okey(x);
                return (k & mask) == prefix ? (int)((k >> shift) & 255u) : -1;
              },
              hist, whist);
    if (threadIdx.x < 32) filt_find_bin(hist, s_need, true, &s_bin, &s_need, &s_binv);
    __syncthreads();
    prefix |= (uint32_t)s_bin << shift;
    mask |= 255u << shift;
  }
  const uint32_t key = prefix;
  // the group of entries with this key has equal weights e: it holds
  // s_binv / e entries, of which ceil(s_need / e) are kept
  const uint32_t kb = (key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key;
  const unsigned long long e = weight(__uint_as_float(kb));
  const unsigned long long n_grp = e ? s_binv / e : 0ull;
  const unsigned long long n_need = e ? (s_need + e - 1) / e : 0ull;
  int idx = INT_MAX;
  if (n_need < n_grp) {
    __syncthreads();
    if (threadIdx.x == 0) s_need = n_need;
    __syncthreads();
    int ip = 0, imask = 0;
    for (int shift = 16; shift >= 0; shift -= 8) {
      filt_hist(l, V, in, [](float) { return 1ull; },
                [key, imask, ip, shift](float x, int v) {
                  return (okey(x) == key && (v & imask) == ip) ? ((v >> shift) & 255) : -1;
                },
                hist, whist);
      if (threadIdx.x < 32) filt_find_bin(hist, s_need, false, &s_bin, &s_need, &s_binv);
      __syncthreads();
      ip |= s_bin << shift;
      imask |= 255 << shift;
    }
    idx = ip;
  }
  if (threadIdx.x == 0) {
    *key_out = key;
    *idx_out = idx;
  }
  __syncthreads();
}

// Top-p inside a top-k set of at most kFiltCompact entries: the k kept
// entries are gathered into shared memory (one pass over the row), sorted by
// (key descending, index ascending) as 64-bit words, and the prefix whose
// integer mass first reaches `need` is found by a block scan.  The row's
// maximum is the first sorted entry.  The result names the last kept entry
// exactly (its key and index), so entries that share its logit but fell
// outside the top-k set stay out.
constexpr int kFiltCompact = kFiltWarps * 256;  // u64 words of the histogram space

__device__ void filt_top_p_compact(const float* l, int V, const RowFilter& fk, int top_k, float invT, float top_p,
                                   unsigned long long* cand, RowFilter* s_f) {
  __shared__ int s_cnt;
  __shared__ unsigned long long s_part[kFiltThreads / 32];
  __shared__ unsigned long long s_z;
  if (threadIdx.x == 0) s_cnt = 0;
  __syncthreads();
  for (int v = threadIdx.x; v < V; v += blockDim.x) {
    const float x = l[v];
    if (filt_kept(&fk, x, v)) {
      const int slot = atomicAdd(&s_cnt, 1);
      if (slot < kFiltCompact) cand[slot] = ((unsigned long long)(~okey(x)) << 32) | (uint32_t)v;
    }
  }
  __syncthreads();
  const int cnt = min(s_cnt, kFiltCompact);  // == top_k
  int n = 1;
  while (n < cnt) n <<= 1;
  for (int i = cnt + threadIdx.x; i < n; i += blockDim.x) cand[i] = ~0ull;
  __syncthreads();
  // bitonic sort, ascending
  for (int size = 2; size <= n; size <<= 1)
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int j = i ^ stride;
        if (j > i) {
          const unsigned long long a = cand[i], b = cand[j];
          const bool up = (i & size) == 0;
          if ((a > b) == up) {
            cand[i] = b;
            cand[j] = a;
          }
        }
      }
      __syncthreads();
    }
  auto logit_of = [](unsigned long long c) {
    const uint32_t k = ~(uint32_t)(c >> 32);
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
  };
  const float mx = logit_of(cand[0]);
  // each thread a contiguous segment of the sorted entries
  const int E = (cnt + blockDim.x - 1) / blockDim.x;
  const int b0 = threadIdx.x * E, b1 = min(cnt, b0 + E);
  unsigned long long mine = 0ull;
  for (int i = b0; i < b1; ++i) mine += filt_mass(logit_of(cand[i]), mx, invT);
  // exclusive scan of the segment sums over the block
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long inc = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) s_part[warp] = inc;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long t = 0ull;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
      const unsigned long long x = s_part[w];
      s_part[w] = t;
      t += x;
    }
    s_z = t;
  }
  __syncthreads();
  const unsigned long long excl = s_part[warp] + inc - mine;
  unsigned long long need = (unsigned long long)ceil((double)top_p * (double)s_z);
  if (need < 1ull) need = 1ull;
  if (excl < need && need <= excl + mine) {
    unsigned long long acc = excl;
    for (int i = b0; i < b1; ++i) {
      acc += filt_mass(logit_of(cand[i]), mx, invT);
      if (acc >= need) {
        *s_f = RowFilter{~(uint32_t)(cand[i] >> 32), (int)(uint32_t)cand[i]};
        break;
      }
    }
  }
  __syncthreads();
  (void)top_k;
}

// Rows [0, rows_a) of logits_a and then the rows of logits_b (two row sets
// in one launch); one CTA per row.
__global__ void __launch_bounds__(kFiltThreads) row_filter_kernel(const float* logits_a, int rows_a, RowFilter* out_a,
                                                                  const float* logits_b, RowFilter* out_b, int V,
                                                                  float invT, int top_k, float top_p, uint32_t* status) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ float red[kFiltThreads / 32];
  __shared__ unsigned long long redu[kFiltThreads / 32];
  __shared__ RowFilter s_f;
  extern __shared__ unsigned long long filt_sm[];  // [kFiltWarps][256] private histograms
  const bool in_a = (int)blockIdx.x < rows_a;
  const int row = in_a ? (int)blockIdx.x : (int)blockIdx.x - rows_a;
  const float* l = (in_a ? logits_a : logits_b) + (size_t)row * V;
  RowFilter* out = in_a ? out_a : out_b;
  if (threadIdx.x == 0) s_f = RowFilter{0u, INT_MAX};
  __syncthreads();
  const bool use_k = top_k > 0 && top_k < V, use_p = top_p > 0.f && top_p < 1.f;
  if (use_k) {
    uint32_t k;
    int i;
    filt_select(l, V, [](float x, int) { return x == x; }, [](float) { return 1ull; }, (unsigned long long)top_k, &k,
                &i, filt_sm);
    if (threadIdx.x == 0) s_f = RowFilter{k, i};
    __syncthreads();
  }
  if (use_p && use_k && top_k <= kFiltCompact) {
    const RowFilter fk = s_f;
    __syncthreads();
    filt_top_p_compact(l, V, fk, top_k, invT, top_p, filt_sm, &s_f);
  } else if (use_p) {
    float mx = -INFINITY;
    for (int v = threadIdx.x; v < V; v += blockDim.x) {
      const float x = l[v];
      if (x == x) mx = fmaxf(mx, x);
    }
    mx = warp_max(mx);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
    __syncthreads();
    mx = red[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) mx = fmaxf(mx, red[w]);
    const RowFilter fk = s_f;
    auto in = [fk](float x, int v) { return filt_kept(&fk, x, v); };
    auto mass = [mx, invT](float x) { return filt_mass(x, mx, invT); };
    unsigned long long z = 0ull;
    for (int v = threadIdx.x; v < V; v += blockDim.x) {
      const float x = l[v];
      if (in(x, v)) z += mass(x);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    if ((threadIdx.x & 31) == 0) redu[threadIdx.x >> 5] = z;
    __syncthreads();
    z = 0ull;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) z += redu[w];
    unsigned long long need = (unsigned long long)ceil((double)top_p * (double)z);
    if (need < 1ull) need = 1ull;
    uint32_t k;
    int i;
    filt_select(l, V, in, mass, need, &k, &i, filt_sm);
    // a boundary group kept whole (i = INT_MAX) holds only its members inside
    // the top-k set: on the top-k boundary key, cap at the top-k index
    if (use_k && k == fk.key && i > fk.idx) i = fk.idx;
    if (threadIdx.x == 0) s_f = RowFilter{k, i};
    __syncthreads();
  }
  if (threadIdx.x == 0) out[row] = s_f;
  (void)status;
}

// One vocabulary row per blockIdx.x (row = s * rows_per_seq + i), slice
// blockIdx.y.  lse_out[row] = log sum exp(l / T); with draw != 0 also
// tok_out[row] = a Gumbel-max draw from softmax(l / T) at position
// base_pos[s] + first_pos + i.
__global__ void __launch_bounds__(kSampleThreads) row_sample_kernel(const __grid_constant__ SampleDesc d,
                                                                    const float* logits, int rows_per_seq,
                                                                    int first_pos, int draw, float* lse_out,
                                                                    int32_t* tok_out, const RowFilter* filt) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ RowAcc red[kSampleThreads / 32];
  __shared__ int s_last;
  const int row = blockIdx.x, sl = blockIdx.y;
  const int s = row / rows_per_seq, i = row % rows_per_seq;
  const int V = d.V;
  const float invT = 1.f / d.T;
  const float* l = logits + (size_t)row * V;
  const int per = (V + kSplit - 1) / kSplit;
  const int v0 = sl * per, v1 = min(V, v0 + per);
  const uint32_t pos = (uint32_t)(d.base_pos[s] + first_pos + i);
  const RowFilter* f = filt ? filt + row : nullptr;
  RowAcc a = acc_empty();
  for (int v = v0 + threadIdx.x; v < v1; v += blockDim.x) {
    const float x = l[v] * invT;
    if (x != x) {
      raise_status(d.status, ST_NUMERIC);
      continue;
    }
    if (!filt_kept(f, l[v], v)) continue;
    acc_lse(a, x);
    if (draw) acc_draw(a, x + rng_gumbel(d.seed, (uint32_t)v, pos, (uint32_t)s, RNG_DRAFT, (uint32_t)d.cycle), v);
  }
  a = block_merge(a, red);
  RowAcc* part = static_cast<RowAcc*>(d.part) + (size_t)row * kSplit;
  if (threadIdx.x == 0) part[sl] = a;
  if (!slice_last(d.counters + row, &s_last)) return;
  if (threadIdx.x == 0) {
    RowAcc t = part[0];
    for (int k = 1; k < kSplit; ++k) {
      RowAcc p;
      p.m = __ldcg(&part[k].m);
      p.s = __ldcg(&part[k].s);
      p.best = __ldcg(&part[k].best);
      p.idx = __ldcg(&part[k].idx);
      t = acc_merge(t, p);
    }
    lse_out[row] = t.m + logf(t.s);
    if (draw) tok_out[row] = t.idx == INT_MAX ? 0 : t.idx;
  }
}

// One warp per sequence: the acceptance tests of the block, then the row of
// the final draw (its index into the target rows, or -1 for none).
__global__ void spec_accept_kernel(const __grid_constant__ SampleDesc d, const float* lse_t) {
  pdl_wait();
  pdl_launch_dependents();
  const int s = blockIdx.x;
  if (threadIdx.x != 0) return;
  const int B = d.block, V = d.V;
  const float invT = 1.f / d.T;
  const int P = d.base_pos[s];
  int k = 0;
  for (int j = 1; j <= B - 1; ++j) {
    const int dj = d.drafts[(size_t)s * (B - 1) + j - 1];
    if (dj < 0 || dj >= V) {
      raise_status(d.status, ST_RANGE);
      break;
    }
    const float lt_dj = d.target_logits[((size_t)s * B + j - 1) * V + dj];
    const float lp = filt_kept(d.filt_t ? d.filt_t + (size_t)s * B + j - 1 : nullptr, lt_dj, dj)
                         ? lt_dj * invT - lse_t[(size_t)s * B + j - 1]
                         : -INFINITY;
    float lq;
    if (d.qcand) {  // the sampled path walk's proposal: log q of d_j among the row's candidates
      lq = -INFINITY;
      const size_t o = ((size_t)s * (B - 1) + j - 1) * d.qk;
      for (int q = 0; q < d.qk; ++q)
        if (d.qcand[o + q] == dj) {
          lq = d.qlogq[o + q];
          break;
        }
    } else {
      lq = d.draft_logits[((size_t)s * (B - 1) + j - 1) * V + dj] * invT - d.draft_lse[(size_t)s * (B - 1) + j - 1];
    }
    const float lu = logf(rng_uniform(d.seed, 0u, (uint32_t)(P + j), (uint32_t)s, RNG_ACCEPT, (uint32_t)d.cycle));
    if (!(lu < lp - lq)) break;
    d.out_tokens[(size_t)s * B + k] = dj;
    ++k;
  }
  d.seq_k[s] = k;
}

// Final draw of each sequence (blockIdx.x), slice blockIdx.y: from
// max(0, p - q) at the rejected row, or from p (every draft accepted, or
// p == q there); the last slice CTA writes the token and the cycle state.
__global__ void __launch_bounds__(kSampleThreads) resample_kernel(const __grid_constant__ SampleDesc d,
                                                                  const float* lse_t) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ RowAcc red[kSampleThreads / 32];
  __shared__ int s_last;
  __shared__ int s_qc[16];  // the sparse proposal of the rejected row (<= 16 candidates)
  __shared__ float s_ql[16];
  const int s = blockIdx.x, sl = blockIdx.y;
  const int B = d.block, V = d.V;
  const float invT = 1.f / d.T;
  const int k = d.seq_k[s];
  const int P = d.base_pos[s];
  const bool resid = k < B - 1;
  const int trow = resid ? k : B - 1;
  const float* tl = d.target_logits + ((size_t)s * B + trow) * V;
  const bool sparse = d.qcand != nullptr;
  const float* dl = (resid && !sparse) ? d.draft_logits + ((size_t)s * (B - 1) + k) * V : nullptr;
  const float lt = lse_t[(size_t)s * B + trow];
  const float ld = (resid && !sparse) ? d.draft_lse[(size_t)s * (B - 1) + k] : 0.f;
  if (sparse && resid && threadIdx.x < d.qk) {
    s_qc[threadIdx.x] = d.qcand[((size_t)s * (B - 1) + k) * d.qk + threadIdx.x];
    s_ql[threadIdx.x] = d.qlogq[((size_t)s * (B - 1) + k) * d.qk + threadIdx.x];
  }
  __syncthreads();
  const uint32_t pos = (uint32_t)(P + trow + 1);
  const int per = (V + kSplit - 1) / kSplit;
  const int v0 = sl * per, v1 = min(V, v0 + per);
  const RowFilter* ft = d.filt_t ? d.filt_t + (size_t)s * B + trow : nullptr;
  const RowFilter* fd = (resid && d.filt_d) ? d.filt_d + (size_t)s * (B - 1) + k : nullptr;
  RowAcc ar = acc_empty();  // the residual draw
  RowAcc ap = acc_empty();  // the draw from p (used when no residual weight is positive)
  for (int v = v0 + threadIdx.x; v < v1; v += blockDim.x) {
    if (!filt_kept(ft, tl[v], v)) continue;  // p = 0 here
    const float a = tl[v] * invT - lt;
    if (resid) {
      float b = -INFINITY;
      if (sparse) {
        for (int q = 0; q < d.qk; ++q)
          if (s_qc[q] == v) {
            b = s_ql[q];
            break;
          }
      } else if (filt_kept(fd, dl[v], v)) {
        b = dl[v] * invT - ld;
      }
      if (a > b)
        acc_draw(ar, (b == -INFINITY ? a : a + log1pf(-expf(b - a))) +
                         rng_gumbel(d.seed, (uint32_t)v, pos, (uint32_t)s, RNG_RESID, (uint32_t)d.cycle), v);
      acc_draw(ap, tl[v] * invT + rng_gumbel(d.seed, (uint32_t)v, pos, (uint32_t)s, RNG_RESID, (uint32_t)d.cycle), v);
    } else {
      acc_draw(ap, tl[v] * invT + rng_gumbel(d.seed, (uint32_t)v, pos, (uint32_t)s, RNG_BONUS, (uint32_t)d.cycle), v);
    }
  }
  ar = block_merge(ar, red);
  ap = block_merge(ap, red);
  RowAcc* part = static_cast<RowAcc*>(d.part) + (size_t)s * 2 * kSplit;
  if (threadIdx.x == 0) {
    part[sl] = ar;
    part[kSplit + sl] = ap;
  }
  if (!slice_last(d.counters + s, &s_last)) return;
  if (threadIdx.x == 0) {
    RowAcc r = part[0], q = part[kSplit];
    for (int i = 1; i < kSplit; ++i) {
      RowAcc x, y;
      x.m = -INFINITY;
      x.s = 0.f;
      x.best = __ldcg(&part[i].best);
      x.idx = __ldcg(&part[i].idx);
      y.m = -INFINITY;
      y.s = 0.f;
      y.best = __ldcg(&part[kSplit + i].best);
      y.idx = __ldcg(&part[kSplit + i].idx);
      r = acc_merge(r, x);
      q = acc_merge(q, y);
    }
    const int x = (resid && r.idx != INT_MAX) ? r.idx : (q.idx == INT_MAX ? 0 : q.idx);
    d.out_tokens[(size_t)s * B + k] = x;
    for (int j = k + 1; j < B; ++j) d.out_tokens[(size_t)s * B + j] = -1;
    d.accept_len[s] = k;
    if (d.next_anchor) d.next_anchor[s] = x;
    if (d.update_base) {
      if (d.commit_base) d.commit_base[s] = P;
      d.base_pos[s] = P + k + 1;
    }
    if (d.commit_count) d.commit_count[s] = k + 1;
  }
}

constexpr size_t kFiltSmem = (size_t)kFiltWarps * 256 * sizeof(unsigned long long);

static cudaError_t filter_smem_attr() {
  return cudaFuncSetAttribute(row_filter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFiltSmem);
}

static bool filtering(const SampleDesc& d) {
  return (d.top_k > 0 && d.top_k < d.V) || (d.top_p > 0.f && d.top_p < 1.f);
}

cudaError_t launch_sample_drafts(const SampleDesc& d, cudaStream_t st) {
  const int rows = d.n_seqs * (d.block - 1);
  if (rows == 0) return cudaSuccess;
  const RowFilter* fd = nullptr;
  if (filtering(d)) {
    cudaError_t e = filter_smem_attr();
    if (e != cudaSuccess) return e;
    e = launch_pdl(row_filter_kernel, dim3(rows), dim3(kFiltThreads), kFiltSmem, st, d.draft_logits, rows,
                   d.filt_d_out, (const float*)nullptr, (RowFilter*)nullptr, d.V, 1.f / d.T, d.top_k, d.top_p,
                   d.status);
    if (e != cudaSuccess) return e;
    fd = d.filt_d_out;
  }
  return launch_pdl(row_sample_kernel, dim3(rows, kSplit), dim3(kSampleThreads), 0, st, d, d.draft_logits,
                    d.block - 1, 1, 1, d.draft_lse_out, d.drafts_out, fd);
}

cudaError_t launch_sample_accept(const SampleDesc& d, float* lse_t, cudaStream_t st) {
  if (d.n_seqs == 0) return cudaSuccess;
  cudaError_t e;
  if (filtering(d)) {  // one launch: the target rows' and (again, identically) the draft rows' kept sets
    e = filter_smem_attr();
    if (e != cudaSuccess) return e;
    const int rt = d.n_seqs * d.block, rd = d.qcand ? 0 : d.n_seqs * (d.block - 1);  // a sparse proposal is not filtered
    e = launch_pdl(row_filter_kernel, dim3(rt + rd), dim3(kFiltThreads), kFiltSmem, st, d.target_logits, rt,
                   const_cast<RowFilter*>(d.filt_t), d.draft_logits, const_cast<RowFilter*>(d.filt_d), d.V, 1.f / d.T,
                   d.top_k, d.top_p, d.status);
    if (e != cudaSuccess) return e;
  }
  e = launch_pdl(row_sample_kernel, dim3(d.n_seqs * d.block, kSplit), dim3(kSampleThreads), 0, st, d,
                 d.target_logits, d.block, 0, 0, lse_t, (int32_t*)nullptr, d.filt_t);
  if (e != cudaSuccess) return e;
  e = launch_pdl(spec_accept_kernel, dim3(d.n_seqs), dim3(32), 0, st, d, (const float*)lse_t);
  if (e != cudaSuccess) return e;
  return launch_pdl(resample_kernel, dim3(d.n_seqs, kSplit), dim3(kSampleThreads), 0, st, d, (const float*)lse_t);
}

size_t sample_part_bytes(int rows) { return (size_t)rows * 2 * kSplit * sizeof(RowAcc); }

}  // namespace dfl
