// k_head.cu -- shared LM head with fused greedy argmax (lowest index on
// ties, top1 - top2 margin), the cross-CTA reduction, and the acceptance
// rule / draft-token output, plus the DFlash 2 path-selector walk.
//
// CUDA-core variant (fp32 path and any shape): a CTA owns a contiguous range
// of vocabulary rows, a warp one row at a time for every token row; per-token
// (best value, best index, second value) triples are merged warp by warp,
// then CTA by CTA in index order by the last CTA to arrive, which also runs
// the acceptance rule.  No CTA ever waits on another.
#include "common.cuh"
#include "head_common.cuh"
#include "internal.h"
#include "rng.cuh"
#include "launch.cuh"

namespace dfl {

constexpr int kHeadWarps = 8;
constexpr int kHeadTok = 8;

template <typename T>
__global__ void __launch_bounds__(kHeadWarps * 32) head_simt_kernel(const __grid_constant__ HeadDesc h) {
  pdl_wait();
  pdl_launch_dependents();
  extern __shared__ Top2 tsm[];  // [warps][M]
  __shared__ int s_last;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int M = h.M, H = h.H, V = h.V;
  Top2* mine = tsm + (size_t)warp * M;
  for (int m = lane; m < M; m += 32) mine[m] = top2_empty();
  __syncwarp();
  const int per = (V + gridDim.x - 1) / gridDim.x;
  const int v0 = blockIdx.x * per, v1 = min(V, v0 + per);
  const T* X = reinterpret_cast<const T*>(h.x);
  for (int v = v0 + warp; v < v1; v += kHeadWarps) {
    const T* w = reinterpret_cast<const T*>(h.w) + (size_t)v * H;
    for (int m0 = 0; m0 < M; m0 += kHeadTok) {
      float acc[kHeadTok];
#pragma unroll
      for (int t = 0; t < kHeadTok; ++t) acc[t] = 0.f;
      for (int k = lane * 8; k < H; k += 256) {
        float fw[8];
        load8<T>(w + k, fw);
#pragma unroll
        for (int t = 0; t < kHeadTok; ++t) {
          if (m0 + t < M && head_row_used(h, m0 + t)) {
            float x[8];
            load8<T>(X + (size_t)(m0 + t) * H + k, x);
            float s = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) s = fmaf(fw[i], x[i], s);
            acc[t] += s;
          }
        }
      }
#pragma unroll
      for (int t = 0; t < kHeadTok; ++t) acc[t] = warp_sum(acc[t]);
#pragma unroll
      for (int t = 0; t < kHeadTok; ++t) {
        const int m = m0 + t;
        if (lane == t && m < M && head_row_used(h, m)) {
          float val = acc[t];
          if (h.logits) head_store_logit(h, m, v, val);
          top2_push(mine[m], val, v, reinterpret_cast<uint32_t*>(h.status));
        }
      }
    }
  }
  __syncthreads();
  // merge warps in order -> this CTA's triple per token
  Top2* part = reinterpret_cast<Top2*>(h.partials);
  for (int m = threadIdx.x; m < M; m += blockDim.x) {
    Top2 t = tsm[m];
    for (int w = 1; w < kHeadWarps; ++w) t = top2_merge(t, tsm[(size_t)w * M + m]);
    part[(size_t)m * gridDim.x + blockIdx.x] = t;  // [M][G]: a row's triples contiguous
  }
  head_finish(h, gridDim.x, gridDim.x, part, &s_last);
}

size_t head_workspace(const HeadDesc& h, int num_sms) {
  size_t simt = (size_t)(2 * num_sms) * h.M * sizeof(Top2) + 256;
  size_t tc = head_tc_workspace(h, num_sms);
  return simt > tc ? simt : tc;
}

cudaError_t launch_head_simt(const HeadDesc& h, int num_sms, cudaStream_t st) {
  int grid = 2 * num_sms;
  size_t smem = (size_t)kHeadWarps * h.M * sizeof(Top2);
  if (h.dtype == DFLASH_BF16) {
    auto k = head_simt_kernel<__nv_bfloat16>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    return launch_pdl(k, dim3(grid), dim3(kHeadWarps * 32), smem, st, h);
  } else {
    auto k = head_simt_kernel<float>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    return launch_pdl(k, dim3(grid), dim3(kHeadWarps * 32), smem, st, h);
  }
  return cudaGetLastError();
}

cudaError_t launch_head(const HeadDesc& h, int num_sms, cudaStream_t st) {
  if (head_tc_supported(h)) return launch_head_tc(h, num_sms, st);
  return launch_head_simt(h, num_sms, st);
}

// ------------------------------------------------- top-k candidate merge

// Insert (v, i) into a register list of the 16 best pairs, best first.
__device__ __forceinline__ void cand_insert(float (&lv)[kMaxTopK], int (&li)[kMaxTopK], float v, int i) {
  if (!beats(v, i, lv[kMaxTopK - 1], li[kMaxTopK - 1])) return;
  bool done = false;
#pragma unroll
  for (int q = kMaxTopK - 1; q > 0; --q) {
    if (!done) {
      if (beats(v, i, lv[q - 1], li[q - 1])) {
        lv[q] = lv[q - 1];
        li[q] = li[q - 1];
      } else {
        lv[q] = v;
        li[q] = i;
        done = true;
      }
    }
  }
  if (!done) {
    lv[0] = v;
    li[0] = i;
  }
}

// One warp per draft row: every lane keeps the 16 best pairs of its share
// (tiles lane, lane+32, .. or vocabulary entries), then k rounds take the
// best list head of the warp.  The order (greater logit, then lower index)
// is total, so the result does not depend on how the pairs were split.
__global__ void topk_merge_kernel(const __grid_constant__ HeadDesc h, const Cand* tlist, int n_tiles) {
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int B = h.block;
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);  // s * (B-1) + j - 1
  if (row >= h.n_seqs * (B - 1)) return;  // whole warp
  const int m = (row / (B - 1)) * B + row % (B - 1) + 1;
  float lv[kMaxTopK];
  int li[kMaxTopK];
#pragma unroll
  for (int q = 0; q < kMaxTopK; ++q) {
    lv[q] = -INFINITY;
    li[q] = INT_MAX;
  }
  if (tlist) {
    for (int t = lane; t < n_tiles; t += 32) {
      const Cand* c = tlist + ((size_t)t * h.M + m) * h.topk;
      for (int q = 0; q < h.topk; ++q) {
        const float v = __ldcg(&c[q].v);
        const int i = __ldcg(&c[q].i);
        if (i == INT_MAX) break;
        cand_insert(lv, li, v, i);
      }
    }
  } else {
    const float* lr = h.logits + (size_t)row * h.V;
    for (int v = lane; v < h.V; v += 32) {
      const float x = lr[v];
      if (x != x) {
        raise_status(h.status, ST_NUMERIC);
        continue;
      }
      cand_insert(lv, li, x, v);
    }
  }
  int32_t* out = h.cand_out + (size_t)row * h.topk;
  for (int q = 0; q < h.topk; ++q) {
    float rv = lv[0];
    int ri = li[0];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, rv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, ri, o);
      if (beats(ov, oi, rv, ri)) {
        rv = ov;
        ri = oi;
      }
    }
    if (ri != INT_MAX && li[0] == ri) {  // this lane's head was taken
#pragma unroll
      for (int z = 0; z < kMaxTopK - 1; ++z) {
        lv[z] = lv[z + 1];
        li[z] = li[z + 1];
      }
      lv[kMaxTopK - 1] = -INFINITY;
      li[kMaxTopK - 1] = INT_MAX;
    }
    if (lane == 0) out[q] = (ri == INT_MAX) ? 0 : ri;
  }
}

cudaError_t launch_topk_merge(const HeadDesc& h, const void* tlist, int n_tiles, cudaStream_t st) {
  const int rows = h.n_seqs * (h.block - 1);
  if (rows <= 0) return cudaSuccess;
  constexpr int kWarps = 4;
  return launch_pdl(topk_merge_kernel, dim3((rows + kWarps - 1) / kWarps), dim3(kWarps * 32), 0, st, h,
                    static_cast<const Cand*>(tlist), n_tiles);
}

// ------------------------------------------------------------ path selector
//
// score(a -> b) = (U e_a) . (V e_b).  The projections of the anchor and of
// every candidate do not depend on the walk, so they are formed first, one
// CTA per token slot; the walk then needs rank-long dot products only.

constexpr int kPathThreads = 256;

// proj[s][slot][0..R) = U e_tok, [R..2R) = V e_tok; slot 0 is the anchor,
// slot 1 + j*topk + q is candidate q of draft row j.  Fixed-order sums.
template <typename T>
__global__ void __launch_bounds__(kPathThreads) path_proj_kernel(const __grid_constant__ PathDesc p) {
  pdl_wait();
  pdl_launch_dependents();
  const int s = blockIdx.y, slot = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int nslot = 1 + (p.block - 1) * p.topk, R = p.rank, H = p.H;
  int tok = slot == 0 ? p.anchor[s] : p.cand[(size_t)s * (p.block - 1) * p.topk + (slot - 1)];
  float* dst = p.proj + ((size_t)s * nslot + slot) * 2 * R;
  if (tok < 0 || tok >= p.V) {  // never read outside the embedding table
    if (threadIdx.x == 0) raise_status(p.status, ST_RANGE);
    for (int o = threadIdx.x; o < 2 * R; o += blockDim.x) dst[o] = 0.f;
    return;
  }
  const T* e = reinterpret_cast<const T*>(p.embed) + (size_t)tok * H;
  for (int o = warp; o < 2 * R; o += nw) {
    const T* w = reinterpret_cast<const T*>(o < R ? p.u : p.v) + (size_t)(o < R ? o : o - R) * H;
    float acc = 0.f;
    for (int k = lane * 8; k < H; k += 256) {
      float fw[8], fe[8];
      load8<T>(w + k, fw);
      load8<T>(e + k, fe);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc = fmaf(fw[i], fe[i], acc);
    }
    acc = warp_sum(acc);
    if (lane == 0) dst[o] = acc;
  }
}

// One warp per sequence: lane q scores candidate q of row j from p_{j-1};
// the greatest score wins, the lower rank on ties (the candidates are ranked
// by draft logit).  Sampled walk (T > 0): the proposal over the candidates
// is softmax(score / T); p_j is a Gumbel-max draw from it (purpose
// RNG_PATH, entry = candidate rank, position base_pos + j + 1), lower rank
// on equal draw scores; logq receives log q_j per candidate.
__global__ void path_walk_kernel(const __grid_constant__ PathDesc p) {
  pdl_wait();
  pdl_launch_dependents();
  const int s = blockIdx.x, lane = threadIdx.x & 31;
  const int K = p.topk, R = p.rank, B = p.block, nslot = 1 + (B - 1) * K;
  const float* base = p.proj + (size_t)s * nslot * 2 * R;
  int prev = 0;  // slot of p_{j-1}
  for (int j = 0; j < B - 1; ++j) {
    const float* ue = base + (size_t)prev * 2 * R;
    float sc = -INFINITY;
    if (lane < K) {
      const float* ve = base + (size_t)(1 + j * K + lane) * 2 * R + R;
      float acc = 0.f;
      for (int r = 0; r < R; ++r) acc = fmaf(ue[r], ve[r], acc);
      if (acc != acc) {
        raise_status(p.status, ST_NUMERIC);
        acc = -INFINITY;
      }
      sc = acc;
    }
    if (p.T > 0.f) {
      const float z = sc / p.T;
      float mx = warp_max(lane < K ? z : -INFINITY);
      const float lse = mx + logf(warp_sum(lane < K ? expf(z - mx) : 0.f));
      const size_t o = ((size_t)s * (B - 1) + j) * K + lane;
      if (lane < K && p.logq) p.logq[o] = z - lse;
      sc = lane < K ? z + rng_gumbel(p.seed, (uint32_t)lane, (uint32_t)(p.base_pos[s] + j + 1), (uint32_t)s, RNG_PATH,
                                     (uint32_t)p.cycle)
                    : -INFINITY;
    }
    if (lane < K && p.cand_out) p.cand_out[((size_t)s * (B - 1) + j) * K + lane] = p.cand[((size_t)s * (B - 1) + j) * K + lane];
    float bv = sc;
    int bq = lane < K ? lane : 64;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oq = __shfl_xor_sync(0xffffffffu, bq, o);
      if (ov > bv || (ov == bv && oq < bq)) {
        bv = ov;
        bq = oq;
      }
    }
    bq = __shfl_sync(0xffffffffu, bq, 0);
    bq = bq < K ? bq : 0;
    float sv = (lane < K && lane != bq) ? sc : -INFINITY;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sv = fmaxf(sv, __shfl_xor_sync(0xffffffffu, sv, o));
    if (lane == 0) {
      p.path[(size_t)s * (B - 1) + j] = p.cand[((size_t)s * (B - 1) + j) * K + bq];
      if (p.margin) p.margin[(size_t)s * (B - 1) + j] = bv - sv;
    }
    prev = 1 + j * K + bq;
  }
}

cudaError_t launch_path_select(const PathDesc& p, cudaStream_t st) {
  if (p.n_seqs == 0 || p.block < 2) return cudaSuccess;
  const dim3 grid(1 + (p.block - 1) * p.topk, p.n_seqs);
  cudaError_t e;
  if (p.dtype == DFLASH_BF16)
    e = launch_pdl(path_proj_kernel<__nv_bfloat16>, grid, dim3(kPathThreads), 0, st, p);
  else
    e = launch_pdl(path_proj_kernel<float>, grid, dim3(kPathThreads), 0, st, p);
  if (e != cudaSuccess) return e;
  return launch_pdl(path_walk_kernel, dim3(p.n_seqs), dim3(32), 0, st, p);
}

}  // namespace dfl
