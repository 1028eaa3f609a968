// k_attention.cu -- GQA softmax attention for the draft block (bidirectional
// over injected context + block) and for target verification (causal over
// the cache), split over fixed chunks of key slots.
//
// Grid: x = key chunk (chunk c covers slots [c*CH, (c+1)*CH)), y = (kv head,
// query tile), z = sequence.  Each CTA writes, for each query vector of its
// tile, the chunk's softmax partial (running max m, denominator l, unnormalised
// output o) in log2 units; the last CTA to arrive for a (sequence, kv head,
// query tile) merges the chunks in chunk order.  Chunk boundaries sit at fixed
// slot offsets and chunks past a row's last visible key contribute exact
// zeros, so a row's output does not depend on how many rows share the launch.
#include "common.cuh"
#include "internal.h"

namespace dfl {

constexpr int kAttnCH = 64;     // keys per chunk
constexpr int kAttnQT = 64;     // query vectors per CTA
constexpr int kAttnWarps = 4;
constexpr float kLog2e = 1.4426950408889634f;

struct AttnGeom {
  int grp, nqv, n_qt, nch;
};

__host__ __device__ __forceinline__ AttnGeom attn_geom(const AttnDesc& a) {
  AttnGeom g;
  g.grp = a.nq / a.nkv;
  g.nqv = a.rows * g.grp;
  g.n_qt = (g.nqv + kAttnQT - 1) / kAttnQT;
  if (a.mode == DFLASH_ATTN_CAUSAL) {
    g.nch = (a.max_pos + kAttnCH - 1) / kAttnCH;
  } else {
    int ctx = a.window > 0 ? (a.window < a.max_pos ? a.window : a.max_pos) : a.max_pos;
    g.nch = (ctx + kAttnCH - 1) / kAttnCH + 1;  // + the block chunk
  }
  return g;
}

// Per-sequence chunk structure.
struct SeqKeys {
  int n_ctx;      // context slots visible (bidir) or cache slots in use (causal)
  int n_ctx_ch;   // chunks over those slots
  int n_ch;       // chunks this sequence uses (bidir: + block chunk)
};

// Slots beyond the cache or beyond the chunks the grid covers are never read
// (positions past max_pos are a caller error; they are clamped, not read).
__device__ __forceinline__ SeqKeys seq_keys(const AttnDesc& a, int P, int grid_ch) {
  SeqKeys k;
  if (a.mode == DFLASH_ATTN_CAUSAL) {
    k.n_ctx = min(max(P + a.rows, 0), min(a.cap, grid_ch * kAttnCH));
    k.n_ctx_ch = (k.n_ctx + kAttnCH - 1) / kAttnCH;
    k.n_ch = k.n_ctx_ch;
  } else {
    k.n_ctx = a.window > 0 ? min(P, a.window) : P;
    k.n_ctx = min(max(k.n_ctx, 0), min(a.cap, (grid_ch - 1) * kAttnCH));
    k.n_ctx_ch = (k.n_ctx + kAttnCH - 1) / kAttnCH;
    k.n_ch = k.n_ctx_ch + 1;
  }
  return k;
}

template <typename T>
__global__ void __launch_bounds__(kAttnWarps * 32) attn_simt_kernel(const __grid_constant__ AttnDesc a,
                                                                     int n_qt) {
  extern __shared__ float sm[];
  const int d = a.d;
  float* Ks = sm;                       // [CH][d]
  float* Vs = Ks + kAttnCH * d;         // [CH][d]
  float* qs = Vs + kAttnCH * d;         // [warps][d]
  float* ps = qs + kAttnWarps * d;      // [warps][CH]
  __shared__ int s_last;

  const int c = blockIdx.x;
  const int g = blockIdx.y / n_qt, qt = blockIdx.y % n_qt;
  const int s = blockIdx.z;
  const int grp = a.nq / a.nkv;
  const int nqv = a.rows * grp;
  const int QD = a.nq * d;
  const int P = a.base_pos[s];
  const SeqKeys sk = seq_keys(a, P, gridDim.x);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int qv0 = qt * kAttnQT;
  const int nq_tile = min(kAttnQT, nqv - qv0);
  const size_t grp_id = ((size_t)s * a.nkv + g) * n_qt + qt;
  const int stride_c = kAttnQT * (d + 2);
  float* part = a.partials + grp_id * (size_t)gridDim.x * stride_c;

  if (c < sk.n_ch) {
    // ---- which keys this chunk holds
    const T* kp;
    const T* vp;
    int nk, slot0;
    bool block_chunk = (a.mode == DFLASH_ATTN_BLOCK_BIDIR && c == sk.n_ctx_ch);
    if (block_chunk) {
      kp = reinterpret_cast<const T*>(a.kb) + ((size_t)s * a.nkv + g) * a.rows * d;
      vp = reinterpret_cast<const T*>(a.vb) + ((size_t)s * a.nkv + g) * a.rows * d;
      nk = a.rows;
      slot0 = 0;
    } else {
      slot0 = c * kAttnCH;
      kp = reinterpret_cast<const T*>(a.kc) + (((size_t)s * a.nkv + g) * a.cap + slot0) * d;
      vp = reinterpret_cast<const T*>(a.vc) + (((size_t)s * a.nkv + g) * a.cap + slot0) * d;
      nk = min(kAttnCH, sk.n_ctx - slot0);
    }
    for (int t = threadIdx.x; t < kAttnCH * d; t += blockDim.x) {
      int j = t / d;
      Ks[t] = j < nk ? to_f<T>(kp[t]) : 0.f;
      Vs[t] = j < nk ? to_f<T>(vp[t]) : 0.f;
    }
    __syncthreads();
    const float scale = rsqrtf((float)d) * kLog2e;
    for (int qi = warp; qi < nq_tile; qi += kAttnWarps) {
      const int qv = qv0 + qi;
      const int row = qv / grp, head = g * grp + qv % grp;
      const int m = s * a.rows + row;
      const T* q = reinterpret_cast<const T*>(a.q) + (size_t)m * QD + (size_t)head * d;
      for (int e = lane; e < d; e += 32) qs[warp * d + e] = to_f<T>(q[e]);
      __syncwarp();
      const int limit = (a.mode == DFLASH_ATTN_CAUSAL) ? (P + row - slot0) : nk - 1;  // last visible key
      float mx = -INFINITY;
      for (int j = lane; j < kAttnCH; j += 32) {
        float sc = -INFINITY;
        if (j < nk && j <= limit) {
          float acc = 0.f;
          for (int e = 0; e < d; ++e) acc = fmaf(qs[warp * d + e], Ks[j * d + e], acc);
          sc = acc * scale;
        }
        ps[warp * kAttnCH + j] = sc;
        mx = fmaxf(mx, sc);
      }
      mx = warp_max(mx);
      float l = 0.f;
      for (int j = lane; j < kAttnCH; j += 32) {
        float sc = ps[warp * kAttnCH + j];
        float p = (mx == -INFINITY || sc == -INFINITY) ? 0.f : exp2f(sc - mx);
        ps[warp * kAttnCH + j] = p;
        l += p;
      }
      l = warp_sum(l);
      __syncwarp();
      float* out = part + (size_t)c * stride_c + (size_t)qi * (d + 2);
      for (int e = lane; e < d; e += 32) {
        float o = 0.f;
        for (int j = 0; j < kAttnCH; ++j) o = fmaf(ps[warp * kAttnCH + j], Vs[j * d + e], o);
        out[2 + e] = o;
      }
      if (lane == 0) {
        out[0] = mx;
        out[1] = l;
      }
      __syncwarp();
    }
  }
  // ---- arrival; the last CTA of this (seq, head, tile) merges the chunks
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t* ctr = a.counters + kCtrAttn + grp_id;
    uint32_t old = atomicAdd(ctr, 1u);
    s_last = (old == gridDim.x - 1);
    if (s_last) *ctr = 0u;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  T* outp = reinterpret_cast<T*>(a.out);
  for (int t = threadIdx.x; t < nq_tile * d; t += blockDim.x) {
    const int qi = t / d, e = t % d;
    const int qv = qv0 + qi;
    const int row = qv / grp, head = g * grp + qv % grp;
    float M = -INFINITY;
    for (int cc = 0; cc < sk.n_ch; ++cc) M = fmaxf(M, __ldcg(part + (size_t)cc * stride_c + (size_t)qi * (d + 2)));
    float L = 0.f, O = 0.f;
    for (int cc = 0; cc < sk.n_ch; ++cc) {
      const float* pp = part + (size_t)cc * stride_c + (size_t)qi * (d + 2);
      float mc = __ldcg(pp);
      float w = (mc == -INFINITY) ? 0.f : exp2f(mc - M);
      L = fmaf(__ldcg(pp + 1), w, L);
      O = fmaf(__ldcg(pp + 2 + e), w, O);
    }
    float v = (L > 0.f) ? O / L : 0.f;
    outp[((size_t)s * a.rows + row) * QD + (size_t)head * d + e] = from_f<T>(v);
  }
}

size_t attn_workspace(const AttnDesc& a) {
  AttnGeom g = attn_geom(a);
  return (size_t)a.n_seqs * a.nkv * g.n_qt * g.nch * kAttnQT * (a.d + 2) * sizeof(float);
}

cudaError_t launch_attention(const AttnDesc& a, cudaStream_t st) {
  AttnGeom g = attn_geom(a);
  if (a.n_seqs == 0 || a.rows == 0) return cudaSuccess;
  dim3 grid(g.nch, a.nkv * g.n_qt, a.n_seqs);
  size_t smem = (size_t)(2 * kAttnCH * a.d + kAttnWarps * a.d + kAttnWarps * kAttnCH) * sizeof(float);
  if (a.dtype == DFLASH_BF16) {
    auto k = attn_simt_kernel<__nv_bfloat16>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    k<<<grid, kAttnWarps * 32, smem, st>>>(a, g.n_qt);
  } else {
    auto k = attn_simt_kernel<float>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    k<<<grid, kAttnWarps * 32, smem, st>>>(a, g.n_qt);
  }
  return cudaGetLastError();
}

}  // namespace dfl
