// k_conv.cu -- DFlash 2 two-tap dynamic depthwise convolution of the draft
// layers ("DFlash: block-diffusion accelerated LLM speculative decoding"
// guide, section 7: a two-tap convolution over the current and the previous
// position, before and after attention and the MLP of every draft layer; the
// block head reads the last verified token).  The page fixes neither the tap
// generator nor the form of the layer; the reading implemented here, for the
// token rows u_t of one block (rows per sequence = the block size):
//
//   z_t       = SiLU(W1 u_t)          W1 [r][H]
//   (a_t,b_t) = W2 z_t                W2 [2H][r]: rows 0..H-1 give a, H..2H-1 give b
//   y_t       = u_t + a_t u_t + b_t u_{t-1}   per channel, u_{-1} = 0
//
// Block row 0 (the anchor) has no predecessor in the block; row 1, the first
// drafted position, reads the anchor, the last verified token.
//
// Two kernels: conv_z_kernel forms z (a reduction over H per token row, one
// CTA per generator row j and 16 token rows), conv_apply_kernel the taps
// and the output (one CTA per 64 channels and 16 token rows, the 64 x r tap
// generator rows held transposed in shared memory).  Every sum runs in a
// fixed order that does not depend on how many rows share the launch.  The
// output is either stored (rounded to the compute type: the input of the
// next projection) or added to the fp32 residual stream.
#include "common.cuh"
#include "internal.h"
#include "launch.cuh"

namespace dfl {

constexpr int kConvRows = 16;     // token rows per CTA
constexpr int kConvThreads = 256;
constexpr int kConvCh = 64;       // channels per CTA of the apply kernel
constexpr int kConvChPad = kConvCh + 1;
constexpr int kConvPer = kConvRows * kConvCh / kConvThreads;  // outputs per thread

__device__ __forceinline__ float conv_silu(float s) { return s / (1.f + expf(-s)); }

// Eight consecutive elements held raw (one 16-byte load for bf16, two for
// fp32), converted when used, so that many loads can be in flight at once.
template <typename T>
struct Raw8;
template <>
struct Raw8<__nv_bfloat16> {
  uint4 v;
  __device__ __forceinline__ void load(const __nv_bfloat16* p) { v = *reinterpret_cast<const uint4*>(p); }
  __device__ __forceinline__ float get(int e) const {
    const uint32_t w = e < 2 ? v.x : e < 4 ? v.y : e < 6 ? v.z : v.w;
    return __uint_as_float((e & 1) ? (w & 0xffff0000u) : (w << 16));
  }
};
template <>
struct Raw8<float> {
  float4 a, b;
  __device__ __forceinline__ void load(const float* p) {
    a = *reinterpret_cast<const float4*>(p);
    b = *reinterpret_cast<const float4*>(p + 4);
  }
  __device__ __forceinline__ float get(int e) const {
    const float4& q = e < 4 ? a : b;
    const int f = e & 3;
    return f == 0 ? q.x : f == 1 ? q.y : f == 2 ? q.z : q.w;
  }
};

// z[m][j] = SiLU(sum_k W1[j][k] u[m][k]).  Thread t takes the 8-element
// groups t, t + 256, ... of k in order (the weight group and the 16 rows'
// groups are loaded before any product); then a fixed xor tree in the warp
// and the warps in order.  H % 8 == 0.
template <typename TW, typename TU>
__global__ void __launch_bounds__(kConvThreads) conv_z_kernel(const TW* __restrict__ W1, const TU* __restrict__ u,
                                                              int H, int M, int r, float* __restrict__ z) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ float red[kConvThreads / 32][kConvRows];
  const int j = blockIdx.x;
  const int m0 = blockIdx.y * kConvRows;
  const int nr = min(kConvRows, M - m0);
  const TW* w = W1 + (size_t)j * H;
  const TU* ub = u + (size_t)m0 * H;
  float acc[kConvRows];
#pragma unroll
  for (int i = 0; i < kConvRows; ++i) acc[i] = 0.f;
  for (int g = threadIdx.x; 8 * g < H; g += kConvThreads) {
    Raw8<TW> wv;
    wv.load(w + 8 * g);
    Raw8<TU> xv[kConvRows];
#pragma unroll
    for (int i = 0; i < kConvRows; ++i)
      if (i < nr) xv[i].load(ub + (size_t)i * H + 8 * g);
#pragma unroll
    for (int i = 0; i < kConvRows; ++i)
      if (i < nr) {
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[i] = fmaf(wv.get(e), xv[i].get(e), acc[i]);
      }
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int i = 0; i < kConvRows; ++i) {
    const float v = warp_sum(acc[i]);
    if (lane == 0) red[warp][i] = v;
  }
  __syncthreads();
  if (threadIdx.x < nr) {
    float s = 0.f;
#pragma unroll
    for (int w8 = 0; w8 < kConvThreads / 32; ++w8) s += red[w8][threadIdx.x];
    z[(size_t)(m0 + threadIdx.x) * r + j] = conv_silu(s);
  }
}

// a = W2[n] . z_m, b = W2[H + n] . z_m (j in order), y = u + a u + b u_prev.
// resid: out is the fp32 residual and receives += y; else out[m][n] = y
// rounded to TO.  r % 8 == 0.
template <typename TW, typename TU, typename TO>
__global__ void __launch_bounds__(kConvThreads) conv_apply_kernel(const TW* __restrict__ W2, const float* __restrict__ z,
                                                                  const TU* __restrict__ u, int H, int M, int r,
                                                                  int rows, TO* __restrict__ out, int resid) {
  pdl_wait();
  pdl_launch_dependents();
  extern __shared__ float conv_sm[];
  float* wa = conv_sm;                  // [r][kConvChPad]: W2 row c0 + ch, entry j at wa[j][ch]
  float* wb = wa + r * kConvChPad;      // [r][kConvChPad]: W2 row H + c0 + ch
  float* zs = wb + r * kConvChPad;      // [kConvRows][r]
  const int c0 = blockIdx.x * kConvCh, m0 = blockIdx.y * kConvRows;
  const int nc = min(kConvCh, H - c0), nr = min(kConvRows, M - m0);
  // the outputs' inputs first: they do not depend on the taps
  float ut[kConvPer], up[kConvPer];
#pragma unroll
  for (int q = 0; q < kConvPer; ++q) {
    const int t = threadIdx.x + q * kConvThreads;
    ut[q] = up[q] = 0.f;
    if (t < nr * nc) {
      const int m = m0 + t / nc, n = c0 + t % nc;
      ut[q] = to_f(u[(size_t)m * H + n]);
      if (m % rows != 0) up[q] = to_f(u[(size_t)(m - 1) * H + n]);
    }
  }
  // tap generator rows of this CTA's channels, transposed, and the rows' z
  const int r8 = r / 8, nv = nc * r8;
  for (int t0 = threadIdx.x; t0 < nv; t0 += 2 * kConvThreads) {
    Raw8<TW> va[2], vb[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int t = t0 + q * kConvThreads;
      if (t < nv) {
        const int ch = t / r8, j8 = 8 * (t % r8);
        va[q].load(W2 + (size_t)(c0 + ch) * r + j8);
        vb[q].load(W2 + (size_t)(H + c0 + ch) * r + j8);
      }
    }
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int t = t0 + q * kConvThreads;
      if (t < nv) {
        const int ch = t / r8, j8 = 8 * (t % r8);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          wa[(j8 + e) * kConvChPad + ch] = va[q].get(e);
          wb[(j8 + e) * kConvChPad + ch] = vb[q].get(e);
        }
      }
    }
  }
  for (int t = threadIdx.x; t < nr * r / 4; t += kConvThreads)
    reinterpret_cast<float4*>(zs)[t] = reinterpret_cast<const float4*>(z + (size_t)m0 * r)[t];
  __syncthreads();
#pragma unroll
  for (int q = 0; q < kConvPer; ++q) {
    const int t = threadIdx.x + q * kConvThreads;
    if (t >= nr * nc) break;
    const int i = t / nc, ch = t % nc;
    const int m = m0 + i, n = c0 + ch;
    float a = 0.f, b = 0.f;
    for (int j = 0; j < r; ++j) {
      const float zj = zs[i * r + j];
      a = fmaf(wa[j * kConvChPad + ch], zj, a);
      b = fmaf(wb[j * kConvChPad + ch], zj, b);
    }
    const float y = ut[q] + a * ut[q] + b * up[q];
    if (resid)
      reinterpret_cast<float*>(out)[(size_t)m * H + n] += y;
    else
      out[(size_t)m * H + n] = from_f<TO>(y);
  }
}

size_t conv_apply_smem(int r) { return (size_t)(2 * r * kConvChPad + kConvRows * r) * sizeof(float); }

namespace {

template <typename TW, typename TU, typename TO>
cudaError_t launch_conv_t(const ConvDesc& c, cudaStream_t st) {
  const dim3 gz(c.r, (c.M + kConvRows - 1) / kConvRows);
  cudaError_t e = launch_pdl(conv_z_kernel<TW, TU>, gz, dim3(kConvThreads), 0, st, (const TW*)c.w1, (const TU*)c.u,
                             c.H, c.M, c.r, c.z);
  if (e != cudaSuccess) return e;
  auto k = conv_apply_kernel<TW, TU, TO>;
  const size_t smem = conv_apply_smem(c.r);
  e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const dim3 ga((c.H + kConvCh - 1) / kConvCh, (c.M + kConvRows - 1) / kConvRows);
  return launch_pdl(k, ga, dim3(kConvThreads), smem, st, (const TW*)c.w2, (const float*)c.z, (const TU*)c.u, c.H,
                    c.M, c.r, c.rows, (TO*)c.out, c.resid);
}

}  // namespace

cudaError_t launch_dyn_conv(const ConvDesc& c, cudaStream_t st) {
  if (c.M == 0) return cudaSuccess;
  if (c.dtype == DFLASH_BF16) {
    if (c.resid) return launch_conv_t<__nv_bfloat16, float, float>(c, st);
    return launch_conv_t<__nv_bfloat16, __nv_bfloat16, __nv_bfloat16>(c, st);
  }
  return launch_conv_t<float, float, float>(c, st);
}

}  // namespace dfl
