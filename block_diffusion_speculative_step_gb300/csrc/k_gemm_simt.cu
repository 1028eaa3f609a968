// k_gemm_simt.cu -- CUDA-core GEMM Y = X W^T with fused epilogues.  Serves
// the fp32 path and shapes the tcgen05 kernel does not tile.  One warp owns
// one output unit (a row, or a RoPE / SwiGLU row pair) for every token row;
// each lane accumulates k = 8*lane + 256*j in order and the warp reduces with
// a fixed xor tree, so a token row's result does not depend on M.
#include "common.cuh"
#include "epilogue.cuh"
#include "internal.h"
#include "launch.cuh"

namespace dfl {

constexpr int kSimtWarps = 8;
constexpr int kSimtTok = 8;

template <typename T>
__global__ void __launch_bounds__(kSimtWarps * 32) gemm_simt_kernel(const __grid_constant__ GemmDesc g) {
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int U = epi_units(g);
  const long total = (long)g.nseg * U;
  const T* X = reinterpret_cast<const T*>(g.X);
  const bool pair = (g.kind == EPI_QKV || g.kind == EPI_SWIGLU);
  for (long unit = (long)blockIdx.x * kSimtWarps + warp; unit < total; unit += (long)gridDim.x * kSimtWarps) {
    const int seg = (int)(unit / U), u = (int)(unit % U);
    int ra, rb;
    epi_unit_rows(g, u, ra, rb);
    const T* W = reinterpret_cast<const T*>(g.seg_w[seg]);
    const Epi ep = make_epi(g, seg);
    const T* wa = W + (size_t)ra * g.K;
    const T* wb = pair ? W + (size_t)rb * g.K : wa;
    for (int m0 = 0; m0 < g.M; m0 += kSimtTok) {
      float acc_a[kSimtTok], acc_b[kSimtTok];
#pragma unroll
      for (int t = 0; t < kSimtTok; ++t) acc_a[t] = acc_b[t] = 0.f;
      for (int k = lane * 8; k < g.K; k += 256) {
        float fa[8], fb[8];
        load8<T>(wa + k, fa);
        if (pair) load8<T>(wb + k, fb);
#pragma unroll
        for (int t = 0; t < kSimtTok; ++t) {
          if (m0 + t < g.M) {
            float x[8];
            load8<T>(X + (size_t)(m0 + t) * g.K + k, x);
            float sa = 0.f, sb = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              sa = fmaf(fa[i], x[i], sa);
              if (pair) sb = fmaf(fb[i], x[i], sb);
            }
            acc_a[t] += sa;
            if (pair) acc_b[t] += sb;
          }
        }
      }
#pragma unroll
      for (int t = 0; t < kSimtTok; ++t) {
        acc_a[t] = warp_sum(acc_a[t]);
        if (pair) acc_b[t] = warp_sum(acc_b[t]);
      }
#pragma unroll
      for (int t = 0; t < kSimtTok; ++t) {
        if (lane == t && m0 + t < g.M) {
          if (pair)
            epi_pair<T>(ep, u, m0 + t, acc_a[t], acc_b[t]);
          else
            epi_single<T>(ep, ra - g.seg_row0, m0 + t, acc_a[t]);
        }
      }
    }
  }
}

int gemm_out_rows(const GemmDesc& g) { return g.nseg * epi_units(g); }

cudaError_t launch_gemm_simt(const GemmDesc& g, cudaStream_t st) {
  if (g.M == 0) return cudaSuccess;
  long units = (long)g.nseg * epi_units(g);
  long blocks = (units + kSimtWarps - 1) / kSimtWarps;
  if (blocks > 65535) blocks = 65535;
  if (g.dtype == DFLASH_BF16)
    return launch_pdl(gemm_simt_kernel<__nv_bfloat16>, dim3((int)blocks), dim3(kSimtWarps * 32), 0, st, g);
  else
    return launch_pdl(gemm_simt_kernel<float>, dim3((int)blocks), dim3(kSimtWarps * 32), 0, st, g);
  return cudaGetLastError();
}

}  // namespace dfl
