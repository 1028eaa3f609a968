// epilogue.cuh -- per-element GEMM epilogues shared by the SIMT and the
// tcgen05 GEMMs: residual add, RoPE + Q/K/V scatter into the query buffer and
// the KV destinations, SwiGLU.
#pragma once
#include "common.cuh"
#include "internal.h"

namespace dfl {

__device__ __forceinline__ RowMap rowmap_of(const GemmDesc& g) {
  RowMap r;
  r.base_pos = g.base_pos;
  r.valid = g.valid;
  r.rows = g.rows;
  return r;
}

// Output units per segment: row pairs for QKV (RoPE partners i, i + d/2) and
// SwiGLU (gate j, up j); single rows otherwise.
__host__ __device__ __forceinline__ int epi_units(const GemmDesc& g) {
  if (g.kind == EPI_QKV) return g.seg_rows / 2;
  if (g.kind == EPI_SWIGLU) return g.inter;
  return g.seg_rows;
}

// Weight rows (relative to the segment's weights) of unit u.
__host__ __device__ __forceinline__ void epi_unit_rows(const GemmDesc& g, int u, int& ra, int& rb) {
  if (g.kind == EPI_QKV) {
    int half = g.d / 2;
    ra = g.seg_row0 + (u / half) * g.d + (u % half);
    rb = ra + half;
  } else if (g.kind == EPI_SWIGLU) {
    ra = u;
    rb = g.inter + u;
  } else {
    ra = g.seg_row0 + u;
    rb = -1;
  }
}

template <typename T>
__device__ __forceinline__ void epi_single(const GemmDesc& g, int n, int m, float v) {
  RowMap rm = rowmap_of(g);
  if (!rm.live(m)) return;
  float* o = g.out_f32 + (size_t)m * g.ldo + n;
  if (g.kind == EPI_RESID)
    *o += v;
  else
    *o = v;
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.f + expf(-z)); }

// Pair epilogue for unit u of segment seg, token row m, accumulators (va, vb).
template <typename T>
__device__ __forceinline__ void epi_pair(const GemmDesc& g, int seg, int u, int m, float va, float vb) {
  RowMap rm = rowmap_of(g);
  if (!rm.live(m)) return;
  if (g.kind == EPI_SWIGLU) {
    T* act = reinterpret_cast<T*>(g.act_out);
    act[(size_t)m * g.inter + u] = from_f<T>(silu_f(va) * vb);
    return;
  }
  // EPI_QKV
  const int d = g.d, half = d / 2;
  const int QD = g.nq * d, KD = g.nkv * d;
  int ra, rb;
  epi_unit_rows(g, u, ra, rb);
  const int e = ra % d;  // < half
  const int pos = rm.pos(m);
  if (pos < 0 || pos >= g.rope_max_pos) return;  // outside the RoPE table: nothing is written
  if (ra < QD + KD) {  // Q or K: rotate the pair (e, e + d/2) by pos * w_e
    const float* cs = g.rope_cs + ((size_t)pos * half + e) * 2;
    float c = cs[0], s = cs[1];
    float lo = va * c - vb * s;
    float hi = vb * c + va * s;
    va = lo;
    vb = hi;
  }
  if (ra < QD) {
    T* q = reinterpret_cast<T*>(g.q_out) + (size_t)m * QD + ra;
    q[0] = from_f<T>(va);
    q[half] = from_f<T>(vb);
    return;
  }
  const bool is_k = ra < QD + KD;
  const int r = is_k ? ra - QD : ra - QD - KD;
  const int head = r / d;
  const int s_idx = rm.seq(m);
  int slot;
  if (g.kv_slot_mode == 1)
    slot = g.kv_window > 0 ? pos % g.kv_window : pos;
  else
    slot = rm.idx(m);
  if (slot >= g.kv_cap) return;
  T* dst = reinterpret_cast<T*>(is_k ? g.k_dst[seg] : g.v_dst[seg]) +
           (((size_t)s_idx * g.nkv + head) * g.kv_cap + slot) * d + e;
  dst[0] = from_f<T>(va);
  dst[half] = from_f<T>(vb);
}

}  // namespace dfl
