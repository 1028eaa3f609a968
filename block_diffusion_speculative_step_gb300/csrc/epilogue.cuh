// epilogue.cuh -- per-element GEMM epilogues shared by the SIMT and the
// tcgen05 GEMMs: residual add, RoPE + Q/K/V scatter into the query buffer and
// the KV destinations, SwiGLU.
#pragma once
#include "common.cuh"
#include "internal.h"

namespace dfl {

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

// The epilogue's operands as plain scalars and pointers, built once per tile
// so the per-element code never re-reads the (large) launch descriptor.
struct Epi {
  int kind, seg_row0, d, half, QD, KD, nkv, kv_cap, kv_window, kv_slot_mode, rope_max_pos, inter, ldo, rows;
  const int32_t* base_pos;
  const int32_t* valid;
  float* out_f32;
  void* q_out;
  void* k_dst;
  void* v_dst;
  const float* rope_cs;
  void* act_out;
};

__device__ __forceinline__ Epi make_epi(const GemmDesc& g, int seg) {
  Epi e;
  e.kind = g.kind;
  e.seg_row0 = g.seg_row0;
  e.d = g.d;
  e.half = g.d / 2;
  e.QD = g.nq * g.d;
  e.KD = g.nkv * g.d;
  e.nkv = g.nkv;
  e.kv_cap = g.kv_cap;
  e.kv_window = g.kv_window;
  e.kv_slot_mode = g.kv_slot_mode;
  e.rope_max_pos = g.rope_max_pos;
  e.inter = g.inter;
  e.ldo = g.ldo;
  e.rows = g.rows;
  e.base_pos = g.base_pos;
  e.valid = g.valid;
  e.out_f32 = g.out_f32;
  e.q_out = g.q_out;
  e.k_dst = g.k_dst[seg];
  e.v_dst = g.v_dst[seg];
  e.rope_cs = g.rope_cs;
  e.act_out = g.act_out;
  return e;
}

__device__ __forceinline__ bool epi_live(const Epi& e, int m) {
  return e.valid == nullptr || (m % e.rows) < e.valid[m / e.rows];
}

template <typename T>
__device__ __forceinline__ void epi_single(const Epi& e, int n, int m, float v) {
  if (!epi_live(e, m)) return;
  float* o = e.out_f32 + (size_t)m * e.ldo + n;
  if (e.kind == EPI_RESID)
    *o += v;
  else
    *o = v;
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.f + expf(-z)); }

// Pair epilogue for unit u, token row m, accumulators (va, vb): SwiGLU, or
// RoPE of the pair (e, e + d/2) followed by the Q / K / V scatter.
template <typename T>
__device__ __forceinline__ void epi_pair(const Epi& e, int u, int m, float va, float vb) {
  if (!epi_live(e, m)) return;
  if (e.kind == EPI_SWIGLU) {
    reinterpret_cast<T*>(e.act_out)[(size_t)m * e.inter + u] = from_f<T>(silu_f(va) * vb);
    return;
  }
  const int d = e.d, half = e.half;
  const int ra = e.seg_row0 + (u / half) * d + (u % half);
  const int col = ra % d;  // < half
  const int s_idx = m / e.rows, idx = m % e.rows;
  const int pos = e.base_pos[s_idx] + idx;
  if (pos < 0 || pos >= e.rope_max_pos) return;  // outside the RoPE table: nothing is written
  if (ra < e.QD + e.KD) {  // Q or K: rotate the pair by pos * w_col
    const float2 cs = *reinterpret_cast<const float2*>(e.rope_cs + ((size_t)pos * half + col) * 2);
    const float lo = va * cs.x - vb * cs.y;
    const float hi = vb * cs.x + va * cs.y;
    va = lo;
    vb = hi;
  }
  if (ra < e.QD) {
    T* q = reinterpret_cast<T*>(e.q_out) + (size_t)m * e.QD + ra;
    q[0] = from_f<T>(va);
    q[half] = from_f<T>(vb);
    return;
  }
  const bool is_k = ra < e.QD + e.KD;
  const int r = is_k ? ra - e.QD : ra - e.QD - e.KD;
  const int head = r / d;
  int slot;
  if (e.kv_slot_mode == 1)
    slot = e.kv_window > 0 ? pos % e.kv_window : pos;
  else
    slot = idx;
  if (slot >= e.kv_cap) return;
  T* dst = reinterpret_cast<T*>(is_k ? e.k_dst : e.v_dst) + (((size_t)s_idx * e.nkv + head) * e.kv_cap + slot) * d + col;
  dst[0] = from_f<T>(va);
  dst[half] = from_f<T>(vb);
}

// ---- 16-column forms used by the tensor-core kernel: every load of the 16
// columns is issued before any store, so the columns do not serialise on
// load latency (the compiler cannot prove the stores leave them untouched).

__device__ __forceinline__ void epi_live16(const Epi& e, int c0, int M, bool (&live)[16]) {
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int m = c0 + j;
    live[j] = m < M && (e.valid == nullptr || (m % e.rows) < __ldg(e.valid + m / e.rows));
  }
}

// Residual add / store of output column n for token rows c0 .. c0+15.
__device__ __forceinline__ void epi_single16(const Epi& e, int n, int c0, int M, const float (&v)[16]) {
  bool live[16];
  epi_live16(e, c0, M, live);
  float old[16];
  if (e.kind == EPI_RESID) {
#pragma unroll
    for (int j = 0; j < 16; ++j) old[j] = live[j] ? e.out_f32[(size_t)(c0 + j) * e.ldo + n] : 0.f;
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j) old[j] = 0.f;
  }
#pragma unroll
  for (int j = 0; j < 16; ++j)
    if (live[j]) e.out_f32[(size_t)(c0 + j) * e.ldo + n] = old[j] + v[j];
}

// Pair epilogue (SwiGLU, or RoPE + Q/K/V scatter) of unit u for token rows
// c0 .. c0+15.
template <typename T>
__device__ __forceinline__ void epi_pair16(const Epi& e, int u, int c0, int M, const float (&va)[16],
                                           const float (&vb)[16]) {
  bool live[16];
  epi_live16(e, c0, M, live);
  if (e.kind == EPI_SWIGLU) {
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (live[j])
        reinterpret_cast<T*>(e.act_out)[(size_t)(c0 + j) * e.inter + u] = from_f<T>(silu_f(va[j]) * vb[j]);
    return;
  }
  const int d = e.d, half = e.half;
  const int ra = e.seg_row0 + (u / half) * d + (u % half);
  const int col = ra % d;  // < half
  const bool rotate = ra < e.QD + e.KD;
  int pos[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int m = c0 + j;
    pos[j] = live[j] ? __ldg(e.base_pos + m / e.rows) + m % e.rows : -1;
    if (pos[j] < 0 || pos[j] >= e.rope_max_pos) live[j] = false;  // outside the RoPE table: nothing is written
  }
  float2 cs[16];
#pragma unroll
  for (int j = 0; j < 16; ++j)
    cs[j] = (live[j] && rotate) ? __ldg(reinterpret_cast<const float2*>(e.rope_cs) + (size_t)pos[j] * half + col)
                                : make_float2(1.f, 0.f);
  float lo[16], hi[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    lo[j] = va[j] * cs[j].x - vb[j] * cs[j].y;
    hi[j] = vb[j] * cs[j].x + va[j] * cs[j].y;
  }
  if (ra < e.QD) {
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (live[j]) {
        T* q = reinterpret_cast<T*>(e.q_out) + (size_t)(c0 + j) * e.QD + ra;
        q[0] = from_f<T>(lo[j]);
        q[half] = from_f<T>(hi[j]);
      }
    return;
  }
  const bool is_k = ra < e.QD + e.KD;
  const int r = is_k ? ra - e.QD : ra - e.QD - e.KD;
  const int head = r / d;
  T* base = reinterpret_cast<T*>(is_k ? e.k_dst : e.v_dst);
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    if (!live[j]) continue;
    const int m = c0 + j;
    const int s_idx = m / e.rows, idx = m % e.rows;
    const int slot = e.kv_slot_mode == 1 ? (e.kv_window > 0 ? pos[j] % e.kv_window : pos[j]) : idx;
    if (slot >= e.kv_cap) continue;
    T* dst = base + (((size_t)s_idx * e.nkv + head) * e.kv_cap + slot) * d + col;
    dst[0] = from_f<T>(lo[j]);
    dst[half] = from_f<T>(hi[j]);
  }
}

}  // namespace dfl
