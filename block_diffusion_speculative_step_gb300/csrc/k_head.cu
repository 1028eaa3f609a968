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
    part[(size_t)blockIdx.x * M + m] = t;
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

// ------------------------------------------------------------ path selector

// One CTA per sequence.  ue = U e_prev, then for each candidate b of row j,
// score = ue . (V e_b); walk greedily.  Scores are fp32 with fixed-order sums.
template <typename T>
__global__ void path_select_kernel(const __grid_constant__ PathDesc p) {
  pdl_wait();
  pdl_launch_dependents();
  extern __shared__ float psm[];
  float* ue = psm;                            // [rank]
  int* park = reinterpret_cast<int*>(psm + p.rank);  // chosen token of the step
  float* sc = psm + p.rank + 1;               // [topk]
  const int s = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const T* E = reinterpret_cast<const T*>(p.embed);
  const T* U = reinterpret_cast<const T*>(p.u);
  const T* Vm = reinterpret_cast<const T*>(p.v);
  int prev = p.anchor[s];
  for (int j = 0; j < p.block - 1; ++j) {
    for (int r = warp; r < p.rank; r += nw) {
      float acc = 0.f;
      for (int k = lane; k < p.H; k += 32) acc = fmaf(to_f<T>(U[(size_t)r * p.H + k]), to_f<T>(E[(size_t)prev * p.H + k]), acc);
      acc = warp_sum(acc);
      if (lane == 0) ue[r] = acc;
    }
    __syncthreads();
    const int32_t* cj = p.cand + ((size_t)s * (p.block - 1) + j) * p.topk;
    for (int q = warp; q < p.topk; q += nw) {
      const int b = cj[q];
      float tot = 0.f;
      for (int r = 0; r < p.rank; ++r) {
        float acc = 0.f;
        for (int k = lane; k < p.H; k += 32)
          acc = fmaf(to_f<T>(Vm[(size_t)r * p.H + k]), to_f<T>(E[(size_t)b * p.H + k]), acc);
        acc = warp_sum(acc);
        tot = fmaf(ue[r], acc, tot);
      }
      if (lane == 0) sc[q] = tot;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int bi = 0;
      float best = sc[0], second = -INFINITY;
      for (int q = 1; q < p.topk; ++q) {
        if (sc[q] > best) {
          second = best;
          best = sc[q];
          bi = q;
        } else if (sc[q] > second) {
          second = sc[q];
        }
      }
      p.path[(size_t)s * (p.block - 1) + j] = cj[bi];
      if (p.margin) p.margin[(size_t)s * (p.block - 1) + j] = best - second;
      *park = cj[bi];
    }
    __syncthreads();
    prev = *park;
    __syncthreads();
  }
}

cudaError_t launch_path_select(const PathDesc& p, cudaStream_t st) {
  if (p.n_seqs == 0 || p.block < 2) return cudaSuccess;
  size_t smem = (size_t)(p.rank + 1 + p.topk) * sizeof(float);
  if (p.dtype == DFLASH_BF16)
    return launch_pdl(path_select_kernel<__nv_bfloat16>, dim3(p.n_seqs), dim3(256), smem, st, p);
  else
    return launch_pdl(path_select_kernel<float>, dim3(p.n_seqs), dim3(256), smem, st, p);
  return cudaGetLastError();
}

}  // namespace dfl
