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
  int M;             // token rows of the launch
  long long kv_rows; // head-dim vectors the K/V destinations hold: (M / rows) * nkv * kv_cap
  uint32_t* status;  // the checked build's bounds assertions report here (may be null)
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
  e.M = g.M;
  e.kv_rows = g.rows > 0 ? (long long)(g.M / g.rows) * g.nkv * g.kv_cap : 0;
  e.status = nullptr;
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

// SiLU z * sigmoid(z) with the fast exponential and division intrinsics (a
// few fp32 ulp, far below the bf16 output rounding): the IEEE division's
// slow-path branch kept the 16 quotients of an epilogue chunk from
// overlapping (about 1 us per chunk).  For z below about -88 the
// denominator is +inf and the quotient 0.
__device__ __forceinline__ float silu_f(float z) { return __fdividef(z, 1.f + __expf(-z)); }

// Rotation of one RoPE pair by (c, s) = (cos, sin): every product and sum
// rounded on its own (no fused multiply-add), so every epilogue that applies
// it gets the same bits whatever code surrounds it: a token row's K/V and
// queries do not depend on how many rows share the launch.
__device__ __forceinline__ void rope_rot(float va, float vb, float c, float s, float& lo, float& hi) {
  lo = __fsub_rn(__fmul_rn(va, c), __fmul_rn(vb, s));
  hi = __fadd_rn(__fmul_rn(vb, c), __fmul_rn(va, s));
}

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
    float lo, hi;
    rope_rot(va, vb, cs.x, cs.y, lo, hi);
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
  if (!DFL_CHECK(((long long)s_idx * e.nkv + head) * e.kv_cap + slot < e.kv_rows, e.status)) return;
  T* dst = reinterpret_cast<T*>(is_k ? e.k_dst : e.v_dst) + (((size_t)s_idx * e.nkv + head) * e.kv_cap + slot) * d + col;
  dst[0] = from_f<T>(va);
  dst[half] = from_f<T>(vb);
}

// ---- 16-column forms used by the tensor-core kernel.  Every load the
// epilogue of one output row needs is issued early, while the accumulator is
// still being computed, so the tail after the last MMA holds only arithmetic
// and stores:
//   epi_preload_rows -- liveness, token positions, RoPE (cos, sin) for the
//     row's rotation column.  With tiles aligned to heads these depend only on
//     the row within the head, never on the tile, so one load serves every
//     tile of the run.
//   epi_preload_tile -- per output column: the residual being added to, or
//     an L2 prefetch of the store destination.

struct EpiRows {
  uint32_t live;    // bit j: token row c0 + j is written
  uint32_t inpos;   // QKV, bit j: the row's position lies inside the RoPE table
  uint32_t kvr[16]; // QKV: K/V destination row (sequence, head 0, slot) of token row c0 + j; ~0u: none
  float2 cs[16];    // QKV: rotation (cos, sin) of the row's column
};

__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Rotation column of QKV unit u (the pair (col, col + d/2) of one head).
__device__ __forceinline__ int epi_rope_col(const Epi& e, int u) {
  return (e.seg_row0 + (u / e.half) * e.d + (u % e.half)) % e.d;
}

__device__ __forceinline__ void epi_preload_rows(const Epi& e, int u, int c0, int M, EpiRows& p) {
  p.live = 0u;
  p.inpos = 0u;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int m = c0 + j;
    const bool lv = m < M && (e.valid == nullptr || (m % e.rows) < __ldg(e.valid + m / e.rows));
    p.live |= lv ? (1u << j) : 0u;
    p.kvr[j] = ~0u;
    p.cs[j] = make_float2(1.f, 0.f);
  }
  if (e.kind != EPI_QKV) return;
  const int col = epi_rope_col(e, u);
  int pos[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int m = c0 + j;
    pos[j] = (p.live >> j) & 1u ? __ldg(e.base_pos + m / e.rows) + m % e.rows : -1;
  }
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    if (pos[j] < 0 || pos[j] >= e.rope_max_pos) continue;  // outside the RoPE table: nothing is written
    p.inpos |= 1u << j;
    p.cs[j] = __ldg(reinterpret_cast<const float2*>(e.rope_cs) + (size_t)pos[j] * e.half + col);
    const int m = c0 + j;
    const int slot = e.kv_slot_mode == 1 ? (e.kv_window > 0 ? pos[j] % e.kv_window : pos[j]) : m % e.rows;
    if (slot < e.kv_cap) p.kvr[j] = (uint32_t)((m / e.rows) * e.nkv) * (uint32_t)e.kv_cap + (uint32_t)slot;
  }
}

// n: output column (single kinds) or unit (pair kinds).
__device__ __forceinline__ void epi_preload_tile(const Epi& e, int n, int c0, const EpiRows& rw, float (&old)[16]) {
#pragma unroll
  for (int j = 0; j < 16; ++j) old[j] = 0.f;
  if (!(rw.live & 1u)) return;
  if (e.kind == EPI_RESID) {
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if ((rw.live >> j) & 1u) old[j] = e.out_f32[(size_t)(c0 + j) * e.ldo + n];
  } else if (e.kind == EPI_STORE) {
    prefetch_l2(e.out_f32 + (size_t)c0 * e.ldo + n);
  } else if (e.kind == EPI_SWIGLU) {
    if (e.act_out) prefetch_l2(static_cast<const char*>(e.act_out) + ((size_t)c0 * e.inter + n) * 2);
  } else if (rw.inpos & 1u) {
    const int ra = e.seg_row0 + (n / e.half) * e.d + (n % e.half);
    if (ra < e.QD) {
      prefetch_l2(static_cast<const char*>(e.q_out) + ((size_t)c0 * e.QD + ra) * 2);
    } else if (rw.kvr[0] != ~0u) {
      const bool is_k = ra < e.QD + e.KD;
      const int r = is_k ? ra - e.QD : ra - e.QD - e.KD;
      prefetch_l2(static_cast<const char*>(is_k ? e.k_dst : e.v_dst) +
                  (((size_t)rw.kvr[0] + (size_t)(r / e.d) * e.kv_cap) * e.d + ra % e.d) * 2);
    }
  }
}

// Residual add / store of output column n for token rows c0 .. c0+15.
__device__ __forceinline__ void epi_single16(const Epi& e, int n, int c0, const float (&v)[16], const EpiRows& rw,
                                             const float (&old)[16]) {
#pragma unroll
  for (int j = 0; j < 16; ++j)
    if ((rw.live >> j) & 1u) e.out_f32[(size_t)(c0 + j) * e.ldo + n] = old[j] + v[j];
}

// Pair epilogue (SwiGLU, or RoPE + Q/K/V scatter) of unit u for token rows
// c0 .. c0+15.
template <typename T>
__device__ __forceinline__ void epi_pair16(const Epi& e, int u, int c0, const float (&va)[16], const float (&vb)[16],
                                           const EpiRows& rw) {
  if (e.kind == EPI_SWIGLU) {
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if ((rw.live >> j) & 1u)
        reinterpret_cast<T*>(e.act_out)[(size_t)(c0 + j) * e.inter + u] = from_f<T>(silu_f(va[j]) * vb[j]);
    return;
  }
  const int d = e.d, half = e.half;
  const int ra = e.seg_row0 + (u / half) * d + (u % half);
  const int col = ra % d;  // < half
  const bool rotate = ra < e.QD + e.KD;  // Q and K rows turn by pos * w_col; V rows do not
  float lo[16], hi[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float2 cs = rotate ? rw.cs[j] : make_float2(1.f, 0.f);
    rope_rot(va[j], vb[j], cs.x, cs.y, lo[j], hi[j]);
  }
  if (ra < e.QD) {
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (((rw.inpos >> j) & 1u) && DFL_CHECK(c0 + j < e.M, e.status)) {
        T* q = reinterpret_cast<T*>(e.q_out) + (size_t)(c0 + j) * e.QD + ra;
        q[0] = from_f<T>(lo[j]);
        q[half] = from_f<T>(hi[j]);
      }
    return;
  }
  const bool is_k = rotate;
  const int r = is_k ? ra - e.QD : ra - e.QD - e.KD;
  T* base = reinterpret_cast<T*>(is_k ? e.k_dst : e.v_dst) + (size_t)(r / d) * e.kv_cap * d + col;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    if (rw.kvr[j] == ~0u) continue;
    if (!DFL_CHECK((long long)rw.kvr[j] + (long long)(r / d) * e.kv_cap < e.kv_rows, e.status)) continue;
    T* dst = base + (size_t)rw.kvr[j] * d;
    dst[0] = from_f<T>(lo[j]);
    dst[half] = from_f<T>(hi[j]);
  }
}

}  // namespace dfl
