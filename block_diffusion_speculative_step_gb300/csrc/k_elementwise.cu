// k_elementwise.cu -- RoPE table, embedding gather, RMSNorm, tap store.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "launch.cuh"

namespace dfl {

// cos_sin[p][i] = (cos(p w_i), sin(p w_i)), w_i = theta^(-2i/d), evaluated in
// double so large positions keep full float accuracy.
__global__ void rope_table_kernel(double theta, int d, int max_pos, float* cs) {
  pdl_wait();
  pdl_launch_dependents();
  int half = d / 2;
  long n = (long)max_pos * half;
  for (long t = blockIdx.x * (long)blockDim.x + threadIdx.x; t < n; t += (long)gridDim.x * blockDim.x) {
    int p = (int)(t / half), i = (int)(t % half);
    double w = pow(theta, -2.0 * (double)i / (double)d);
    double a = (double)p * w;
    cs[2 * t] = (float)cos(a);
    cs[2 * t + 1] = (float)sin(a);
  }
}

cudaError_t launch_rope_table(float theta, int d, int max_pos, float* cs, cudaStream_t st) {
  long n = (long)max_pos * (d / 2);
  int blocks = (int)((n + 255) / 256);
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  return launch_pdl(rope_table_kernel, dim3(blocks), dim3(256), 0, st, (double)theta, d, max_pos, cs);
  return cudaGetLastError();
}

// 4 consecutive elements as floats / from floats (16-byte fp32, 8-byte bf16).
__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 ld4(const __nv_bfloat16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ void st4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ void st4(__nv_bfloat16* p, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = u;
}

constexpr int kRowThreads = 256;
constexpr int kRowVec = 8;  // 4-element groups per thread: rows up to 8192 elements stay in registers

// h[m][:] = E[token(m)][:] as fp32 (4 elements per access).  A token id
// outside [0, V) raises the range status and reads row 0 instead, so no
// access leaves the table.
template <typename T>
__global__ void __launch_bounds__(kRowThreads) embed_kernel(const T* __restrict__ E, int H, int V, int rows,
                                                            const int32_t* __restrict__ first,
                                                            const int32_t* __restrict__ rest, int fill,
                                                            float* __restrict__ h, uint32_t* status) {
  pdl_wait();
  pdl_launch_dependents();
  const int m = blockIdx.x;
  const int s = m / rows, i = m % rows;
  int tok = (i == 0) ? first[s] : (rest ? rest[s * (rows - 1) + i - 1] : fill);
  if (tok < 0 || tok >= V) {
    if (threadIdx.x == 0) raise_status(status, ST_RANGE);
    tok = 0;
  }
  const T* e = E + (size_t)tok * H;
  float* o = h + (size_t)m * H;
  for (int k = 4 * threadIdx.x; k < H; k += 4 * kRowThreads) st4(o + k, ld4(e + k));
}

cudaError_t launch_embed(int dtype, const void* E, int H, int V, int n_seqs, int rows, const int32_t* first,
                         const int32_t* rest, int fill, float* h, uint32_t* status, cudaStream_t st) {
  int M = n_seqs * rows;
  if (M == 0) return cudaSuccess;
  if (dtype == DFLASH_BF16)
    return launch_pdl(embed_kernel<__nv_bfloat16>, dim3(M), dim3(kRowThreads), 0, st, (const __nv_bfloat16*)E,
                      H, V, rows, first, rest, fill, h, status);
  return launch_pdl(embed_kernel<float>, dim3(M), dim3(kRowThreads), 0, st, (const float*)E, H, V, rows, first,
                    rest, fill, h, status);
}

// x[m] = round(h[m] * rsqrt(mean(h[m]^2) + eps) * g), one block per row, the
// row held in registers between the two passes.  The sum of squares runs in
// a fixed order (per-thread groups in index order, then a fixed tree), so a
// row's result does not depend on M.  Rows longer than 4*256*8 elements use
// the strided loop.
template <typename T>
__global__ void __launch_bounds__(kRowThreads) rmsnorm_kernel(const float* __restrict__ h, const T* __restrict__ g,
                                                              int H, float eps, T* __restrict__ x) {
  const bool fits = H <= 4 * kRowThreads * kRowVec;
  float4 gg[kRowVec];  // the gain is no kernel's output: loaded before the wait
  if (fits) {
#pragma unroll
    for (int i = 0; i < kRowVec; ++i) {
      const int k = 4 * (threadIdx.x + i * kRowThreads);
      gg[i] = k < H ? ld4(g + k) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  pdl_wait();
  pdl_launch_dependents();
  __shared__ float red[32];
  const float* r = h + (size_t)blockIdx.x * H;
  T* o = x + (size_t)blockIdx.x * H;
  float4 v[kRowVec];
  float ss = 0.f;
  if (fits) {
#pragma unroll
    for (int i = 0; i < kRowVec; ++i) {
      const int k = 4 * (threadIdx.x + i * kRowThreads);
      v[i] = k < H ? ld4(r + k) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int i = 0; i < kRowVec; ++i) ss += v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z + v[i].w * v[i].w;
  } else {
    for (int k = threadIdx.x; k < H; k += kRowThreads) ss += r[k] * r[k];
  }
  ss = warp_sum(ss);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) red[w] = ss;
  __syncthreads();
  if (w == 0) {
    float t = (l < (int)(blockDim.x >> 5)) ? red[l] : 0.f;
    t = warp_sum(t);
    if (l == 0) red[0] = t;
  }
  __syncthreads();
  const float inv = rsqrtf(red[0] / (float)H + eps);
  if (fits) {
#pragma unroll
    for (int i = 0; i < kRowVec; ++i) {
      const int k = 4 * (threadIdx.x + i * kRowThreads);
      if (k < H)
        st4(o + k, make_float4(v[i].x * inv * gg[i].x, v[i].y * inv * gg[i].y, v[i].z * inv * gg[i].z,
                               v[i].w * inv * gg[i].w));
    }
  } else {
    for (int k = threadIdx.x; k < H; k += kRowThreads) o[k] = from_f<T>(r[k] * inv * to_f<T>(g[k]));
  }
}

cudaError_t launch_rmsnorm(int dtype, const float* h, const void* g, int M, int H, float eps, void* x,
                           cudaStream_t st) {
  if (M == 0) return cudaSuccess;
  if (dtype == DFLASH_BF16)
    return launch_pdl(rmsnorm_kernel<__nv_bfloat16>, dim3(M), dim3(kRowThreads), 0, st, h,
                      (const __nv_bfloat16*)g, H, eps, (__nv_bfloat16*)x);
  return launch_pdl(rmsnorm_kernel<float>, dim3(M), dim3(kRowThreads), 0, st, h, (const float*)g, H, eps, (float*)x);
}

// tap[m*stride + offset + k] = round(h[m][k]).
template <typename T>
__global__ void __launch_bounds__(kRowThreads) store_tap_kernel(const float* __restrict__ h, int H,
                                                                T* __restrict__ tap, int stride, int offset) {
  pdl_wait();
  pdl_launch_dependents();
  const float* r = h + (size_t)blockIdx.x * H;
  T* o = tap + (size_t)blockIdx.x * stride + offset;
  for (int k = 4 * threadIdx.x; k < H; k += 4 * kRowThreads) st4(o + k, ld4(r + k));
}

cudaError_t launch_store_tap(int dtype, const float* h, int M, int H, void* tap, int stride, int offset,
                             cudaStream_t st) {
  if (M == 0) return cudaSuccess;
  if (dtype == DFLASH_BF16)
    return launch_pdl(store_tap_kernel<__nv_bfloat16>, dim3(M), dim3(kRowThreads), 0, st, h, H,
                      (__nv_bfloat16*)tap, stride, offset);
  return launch_pdl(store_tap_kernel<float>, dim3(M), dim3(kRowThreads), 0, st, h, H, (float*)tap, stride, offset);
}

template <typename T>
__global__ void to_f32_kernel(const T* __restrict__ src, size_t n, float* __restrict__ dst) {
  pdl_wait();
  pdl_launch_dependents();
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    dst[i] = to_f<T>(src[i]);
}

cudaError_t launch_to_f32(int dtype, const void* src, size_t n, float* dst, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  int blocks = (int)std::min<size_t>((n + 255) / 256, 4096);
  if (dtype == DFLASH_BF16)
    return launch_pdl(to_f32_kernel<__nv_bfloat16>, dim3(blocks), dim3(256), 0, st, (const __nv_bfloat16*)src, n, dst);
  else
    return launch_pdl(to_f32_kernel<float>, dim3(blocks), dim3(256), 0, st, (const float*)src, n, dst);
  return cudaGetLastError();
}

// Paged KV caches: row m of the block scratch (sequence s = m / rows, in-block
// index i = m % rows) goes to its slot's page, KV head by KV head, in 16-byte
// pieces.  Grid: (S * rows, n_layers); one CTA moves one row's K and V.
template <typename T>
__global__ void __launch_bounds__(128) kv_page_scatter_kernel(const __grid_constant__ KvScatter k) {
  pdl_wait();
  pdl_launch_dependents();
  const int m = blockIdx.x, layer = blockIdx.y;
  const int s = m / k.rows, i = m % k.rows;
  if (k.valid && i >= __ldg(k.valid + s)) return;
  const int pos = __ldg(k.base_pos + s) + i;
  if (pos < 0 || pos >= k.rope_max_pos) return;
  const int slot = k.window > 0 ? pos % k.window : pos;
  if (slot >= k.cap) return;
  const KvMap km{k.pages[layer], k.cap, k.ps, k.max_pages, k.pool, k.nkv};
  bool bad = false;
  const size_t r0 = km.row0(s, slot, &bad);
  if (bad) {
    if (threadIdx.x == 0) raise_status(k.status, ST_RANGE);
    return;
  }
  const int per_head = k.d * (int)sizeof(T) / 16;  // 16-byte pieces per head row
  for (int t = threadIdx.x; t < 2 * k.nkv * per_head; t += blockDim.x) {
    const int is_v = t / (k.nkv * per_head), rem = t % (k.nkv * per_head);
    const int g = rem / per_head, piece = rem % per_head;
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const T*>(is_v ? k.vb[layer] : k.kb[layer]) +
                                                      (((size_t)s * k.nkv + g) * k.rows + i) * k.d) + piece;
    uint4* dst = reinterpret_cast<uint4*>(static_cast<T*>(is_v ? k.vpool[layer] : k.kpool[layer]) +
                                          (r0 + (size_t)g * k.ps) * k.d) + piece;
    *dst = *src;
  }
}

cudaError_t launch_kv_page_scatter(const KvScatter& k, cudaStream_t st) {
  if (k.S == 0 || k.rows == 0) return cudaSuccess;
  const dim3 grid(k.S * k.rows, k.n_layers);
  if (k.dtype == DFLASH_BF16) return launch_pdl(kv_page_scatter_kernel<__nv_bfloat16>, grid, dim3(128), 0, st, k);
  return launch_pdl(kv_page_scatter_kernel<float>, grid, dim3(128), 0, st, k);
}

}  // namespace dfl
