// head_common.cuh -- per-token greedy argmax state of the LM head and the
// last-CTA finish (global merge in CTA order, acceptance rule, outputs).
#pragma once
#include <limits.h>

#include "common.cuh"
#include "internal.h"

namespace dfl {

constexpr int kHeadMaxM = 1024;  // token rows per LM-head launch

struct Top2 {
  float v1;  // best logit
  int i1;    // its vocab index (lowest on ties)
  float v2;  // best logit among the other indices
};

__device__ __forceinline__ Top2 top2_empty() { return Top2{-INFINITY, INT_MAX, -INFINITY}; }

__device__ __forceinline__ bool beats(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

// Top-k mode (path selector candidates): per (tile, token row) the k best
// (logit, index) pairs of the tile, best first (greater logit, then lower
// index); index INT_MAX marks an empty entry.
constexpr int kMaxTopK = 16;
struct Cand {
  float v;
  int i;
};

__device__ __forceinline__ void top2_push(Top2& t, float v, int i, uint32_t* status) {
  if (v != v) {  // NaN never wins; flag it
    raise_status(status, ST_NUMERIC);
    return;
  }
  if (beats(v, i, t.v1, t.i1)) {
    t.v2 = t.v1;
    t.v1 = v;
    t.i1 = i;
  } else if (v > t.v2) {
    t.v2 = v;
  }
}

__device__ __forceinline__ Top2 top2_merge(const Top2& a, const Top2& b) {
  if (beats(b.v1, b.i1, a.v1, a.i1)) return Top2{b.v1, b.i1, fmaxf(b.v2, a.v1)};
  return Top2{a.v1, a.i1, fmaxf(a.v2, b.v1)};
}

// Draft mode skips block row 0 (the anchor row predicts nothing).
__device__ __forceinline__ bool head_row_used(const HeadDesc& h, int m) {
  return h.mode == 1 || (m % h.block) != 0;
}

__device__ __forceinline__ void head_store_logit(const HeadDesc& h, int m, int v, float val) {
  size_t row;
  if (h.mode == 1) {
    row = (size_t)m;
  } else {
    int s = m / h.block, j = m % h.block;
    row = (size_t)s * (h.block - 1) + (j - 1);
  }
  h.logits[row * h.V + v] = val;
}

__device__ __forceinline__ Top2 ldcg_top2(const Top2* p) {
  Top2 t;
  t.v1 = __ldcg(&p->v1);
  t.i1 = __ldcg(&p->i1);
  t.v2 = __ldcg(&p->v2);
  return t;
}

// Called by every CTA (all its threads) once its per-token triples are stored
// in part[M][n_parts] (CTA b's triple of row m at m * n_parts + b).  The last
// of n_arrivals CTAs to arrive merges them and writes
// the mode's outputs.  The merge (greater value wins, lower index on equal
// values; second = the largest other value) is associative and commutative,
// so the warp-parallel reduction below gives the same result in any order.
__device__ __forceinline__ void head_finish(const HeadDesc& h, int n_arrivals, int n_parts, const Top2* part,
                                            int* s_last) {
  __shared__ int s_arg[kHeadMaxM];
  if (h.mode == 2) return;  // top-k mode: candidates are merged by their own kernel
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t* ctr = h.counters + kCtrHead;
    uint32_t old = atomicAdd(ctr, 1u);
    *s_last = (old == (uint32_t)n_arrivals - 1);
    if (*s_last) *ctr = 0u;
  }
  __syncthreads();
  if (!*s_last) return;
  __threadfence();
  const int M = h.M, B = h.block;
  const int lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  // part is [M][n_parts]: a warp reads a row's triples as contiguous bytes.
  // RG rows per warp at a time, QB parts per lane per row in flight: the
  // loads of RG rows overlap instead of one row's round trip after another.
  constexpr int RG = 8, QB = 5;
  for (int m0 = (threadIdx.x >> 5) * RG; m0 < M; m0 += nwarps * RG) {
    Top2 t[RG];
#pragma unroll
    for (int g = 0; g < RG; ++g) t[g] = top2_empty();
    for (int b0 = 0; b0 < n_parts; b0 += 32 * QB) {
      Top2 x[RG][QB];
#pragma unroll
      for (int g = 0; g < RG; ++g)
#pragma unroll
        for (int q = 0; q < QB; ++q) {
          const int b = b0 + 32 * q + lane, m = m0 + g;
          x[g][q] = (b < n_parts && m < M) ? ldcg_top2(part + (size_t)m * n_parts + b) : top2_empty();
        }
#pragma unroll
      for (int g = 0; g < RG; ++g)
#pragma unroll
        for (int q = 0; q < QB; ++q) t[g] = top2_merge(t[g], x[g][q]);
    }
#pragma unroll
    for (int g = 0; g < RG; ++g)
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        Top2 u;
        u.v1 = __shfl_xor_sync(0xffffffffu, t[g].v1, o);
        u.i1 = __shfl_xor_sync(0xffffffffu, t[g].i1, o);
        u.v2 = __shfl_xor_sync(0xffffffffu, t[g].v2, o);
        t[g] = top2_merge(t[g], u);
      }
    // lane g writes row m0 + g
    Top2 tl = t[0];
#pragma unroll
    for (int g = 1; g < RG; ++g)
      if (lane == g) tl = t[g];
    const int m = m0 + lane;
    if (lane >= RG || m >= M || !head_row_used(h, m)) continue;
    int idx = (tl.i1 == INT_MAX) ? 0 : tl.i1;
    s_arg[m] = idx;
    if (h.mode == 1) {
      h.argmax[m] = idx;
      if (h.margin) h.margin[m] = tl.v1 - tl.v2;
    } else {
      const int s = m / B, j = m % B;
      h.drafts_out[(size_t)s * (B - 1) + j - 1] = idx;
      if (h.margin) h.margin[(size_t)s * (B - 1) + j - 1] = tl.v1 - tl.v2;
    }
  }
  __syncthreads();
  if (h.mode != 1) return;
  // greedy longest-prefix acceptance, one thread per sequence
  for (int s = threadIdx.x; s < h.n_seqs; s += blockDim.x) {
    const int* g = s_arg + (size_t)s * B;
    const int32_t* dr = h.drafts ? h.drafts + (size_t)s * (B - 1) : nullptr;
    int k = 0;
    while (k < B - 1 && dr[k] == g[k]) ++k;
    int32_t* out = h.out_tokens + (size_t)s * B;
    for (int j = 0; j < B; ++j) out[j] = (j < k) ? dr[j] : (j == k ? g[k] : -1);
    h.accept_len[s] = k;
    if (h.next_anchor) h.next_anchor[s] = g[k];
    if (h.base_pos) {
      int p = h.base_pos[s];
      if (h.commit_base) h.commit_base[s] = p;
      h.base_pos[s] = p + k + 1;
    } else if (h.commit_base) {
      h.commit_base[s] = 0;
    }
    if (h.commit_count) h.commit_count[s] = k + 1;
  }
}

}  // namespace dfl
