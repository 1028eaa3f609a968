// k_attention.cu -- GQA softmax attention for the draft block (bidirectional
// over injected context + block) and for target verification (causal over
// the cache), split over fixed chunks of key slots.
//
// Grid: x = key chunk (chunk c covers slots [c*CH, (c+1)*CH)), y = (kv head,
// query tile), z = sequence.  Each CTA writes, for each query vector of its
// tile, the chunk's softmax partial (max m, denominator l, unnormalised output
// o, in log2 units); the last CTA to arrive for a (sequence, kv head, query
// tile) merges the chunks in chunk order.  Chunk boundaries sit at fixed slot
// offsets and chunks past a row's last visible key contribute exact zeros, so
// a row's output does not depend on how many rows share the launch.
//
// fp32 path: CUDA-core dot products, chunk partials in the workspace, merged
// by the last CTA of the group.
//
// bf16 path: a thread-block cluster of NC CTAs per (sequence, kv head, query
// tile).  CTA rank r owns chunks r, r + NC, r + 2 NC, ... (CH = 128 key slots
// each, at fixed absolute offsets), streams them through double-buffered TMA
// loads (128-byte swizzled boxes) and runs mma.sync m16n8k16 tiles with an
// online softmax over its chunks in order: S = Q K^T, then O += P V with P
// carried as a bf16 pair (hi + lo) so the product keeps about 16 bits of P.
// The NC partials are then merged in rank order through distributed shared
// memory; cluster barriers are hardware barriers over co-scheduled CTAs, so
// nothing spins and nothing round-trips through HBM.
//
// For head dimension 128 the bf16 path runs attn_tc_kernel instead, which
// computes the same function on the tcgen05 tensor cores: the query tile
// arrives as one 3-D TMA box per 64 dims, S and O are TMEM accumulators, the
// 64 query rows are duplicated into MMA rows 64..127 so that the softmax
// warps on all four TMEM lane quadrants share the rows, and each rank pushes
// its partial rows into their owner's shared memory for a local merge (same
// arithmetic and order as the pulled merge).  With more (sequence, KV head)
// items than clusters fit at once, clusters of half the width run them, each
// CTA taking two of the logical ranks into two TMEM output accumulators; the
// chunk split and the merge order do not change, nor do the results.
// DFLASH_ATTN_MMASYNC=1 in the environment selects the mma.sync kernel for
// head dimension 128 too.
#include <cooperative_groups.h>
#include <stdlib.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "launch.cuh"
#include "tc_ptx.cuh"
#include "tmap.h"

namespace dfl {

constexpr int kAttnQT = 64;      // query vectors per CTA
constexpr int kAttnWarps = 4;
constexpr int kSimtCH = 64;      // keys per chunk, fp32 path
constexpr int kMmaCH = 128;      // keys per chunk, bf16 tensor-core path
constexpr float kLog2e = 1.4426950408889634f;

__host__ __device__ __forceinline__ int attn_ch(const AttnDesc& a) {
  return a.dtype == DFLASH_BF16 ? kMmaCH : kSimtCH;
}

struct AttnGeom {
  int grp, nqv, n_qt, nch;
};

__host__ __device__ __forceinline__ AttnGeom attn_geom(const AttnDesc& a) {
  const int CH = attn_ch(a);
  AttnGeom g;
  g.grp = a.nq / a.nkv;
  g.nqv = a.rows * g.grp;
  g.n_qt = (g.nqv + kAttnQT - 1) / kAttnQT;
  if (a.mode == DFLASH_ATTN_CAUSAL) {
    g.nch = (a.max_pos + CH - 1) / CH;
  } else {
    int ctx = a.window > 0 ? (a.window < a.max_pos ? a.window : a.max_pos) : a.max_pos;
    g.nch = (ctx + CH - 1) / CH + 1;  // + the block chunk
  }
  return g;
}

struct SeqKeys {
  int n_ctx;     // context slots visible (bidir) or cache slots in use (causal)
  int n_ctx_ch;  // chunks over those slots
  int n_ch;      // chunks this sequence uses (bidir: + block chunk)
};

// Slots beyond the cache or beyond the chunks the grid covers are never read
// (positions past max_pos are a caller error; they are clamped, not read).
__device__ __forceinline__ SeqKeys seq_keys(const AttnDesc& a, int P, int grid_ch, int CH) {
  SeqKeys k;
  if (a.mode == DFLASH_ATTN_CAUSAL) {
    k.n_ctx = min(max(P + a.rows, 0), min(a.cap, grid_ch * CH));
    k.n_ctx_ch = (k.n_ctx + CH - 1) / CH;
    k.n_ch = k.n_ctx_ch;
  } else {
    k.n_ctx = a.window > 0 ? min(P, a.window) : P;
    k.n_ctx = min(max(k.n_ctx, 0), min(a.cap, (grid_ch - 1) * CH));
    k.n_ctx_ch = (k.n_ctx + CH - 1) / CH;
    k.n_ch = k.n_ctx_ch + 1;
  }
  return k;
}

// The key chunks of a sequence whose block starts at position P (the tensor-core
// kernels read the cache up to its capacity; 128-key chunks).
__device__ __forceinline__ SeqKeys tc_seq_keys(const AttnDesc& a, int P) {
  SeqKeys k;
  if (a.mode == DFLASH_ATTN_CAUSAL) {
    k.n_ctx = min(max(P + a.rows, 0), a.cap);
    k.n_ctx_ch = (k.n_ctx + kMmaCH - 1) / kMmaCH;
    k.n_ch = k.n_ctx_ch;
  } else {
    k.n_ctx = min(max(a.window > 0 ? min(P, a.window) : P, 0), a.cap);
    k.n_ctx_ch = (k.n_ctx + kMmaCH - 1) / kMmaCH;
    k.n_ch = k.n_ctx_ch + 1;
  }
  return k;
}

// Keys of chunk c: base pointers, count, first slot.
template <typename T>
__device__ __forceinline__ void chunk_keys(const AttnDesc& a, const SeqKeys& sk, int s, int g, int c, int CH,
                                           const T*& kp, const T*& vp, int& nk, int& slot0) {
  const int d = a.d;
  if (a.mode == DFLASH_ATTN_BLOCK_BIDIR && c == sk.n_ctx_ch) {
    kp = reinterpret_cast<const T*>(a.kb) + ((size_t)s * a.nkv + g) * a.rows * d;
    vp = reinterpret_cast<const T*>(a.vb) + ((size_t)s * a.nkv + g) * a.rows * d;
    nk = min(a.rows, CH);
    slot0 = -1;  // block chunk: every key visible
  } else {
    slot0 = c * CH;
    const KvMap km{a.pages, a.cap, a.ps, a.max_pages, a.pool, a.nkv};
    bool bad = false;
    const size_t row = (size_t)km.row0(s, slot0, &bad) + (size_t)g * km.head_rows();
    if (bad) raise_status(a.status, ST_RANGE);  // read from page 0 instead
    kp = reinterpret_cast<const T*>(a.kc) + row * d;
    vp = reinterpret_cast<const T*>(a.vc) + row * d;
    nk = min(CH, sk.n_ctx - slot0);
  }
}

// Arrival + merge of the chunk partials by the last CTA of the group.
template <typename T>
__device__ __forceinline__ void attn_finish(const AttnDesc& a, const float* part, size_t grp_id, int stride_c,
                                            int nq_tile, int qv0, int g, int s, int n_ch, int* s_last) {
  const int d = a.d, grp = a.nq / a.nkv, QD = a.nq * d;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t* ctr = a.counters + kCtrAttn + grp_id;
    const uint32_t old = atomicAdd(ctr, 1u);
    *s_last = (old == gridDim.x - 1);
    if (*s_last) *ctr = 0u;
  }
  __syncthreads();
  if (!*s_last) return;
  __threadfence();
  T* outp = reinterpret_cast<T*>(a.out);
  for (int t = threadIdx.x; t < nq_tile * d; t += blockDim.x) {
    const int qi = t / d, e = t % d;
    const int qv = qv0 + qi;
    const int row = qv / grp, head = g * grp + qv % grp;
    float M = -INFINITY;
    for (int cc = 0; cc < n_ch; ++cc) M = fmaxf(M, __ldcg(part + (size_t)cc * stride_c + (size_t)qi * (d + 2)));
    float L = 0.f, O = 0.f;
    for (int cc = 0; cc < n_ch; ++cc) {
      const float* pp = part + (size_t)cc * stride_c + (size_t)qi * (d + 2);
      const float mc = __ldcg(pp);
      const float w = (mc == -INFINITY) ? 0.f : exp2f(mc - M);
      L = fmaf(__ldcg(pp + 1), w, L);
      O = fmaf(__ldcg(pp + 2 + e), w, O);
    }
    const float v = (L > 0.f) ? O / L : 0.f;
    outp[((size_t)s * a.rows + row) * QD + (size_t)head * d + e] = from_f<T>(v);
  }
}

// ------------------------------------------------------------- fp32 path

template <typename T>
__global__ void __launch_bounds__(kAttnWarps * 32) attn_simt_kernel(const __grid_constant__ AttnDesc a, int n_qt) {
  pdl_wait();
  pdl_launch_dependents();
  extern __shared__ float sm[];
  constexpr int CH = kSimtCH;
  const int d = a.d, ld = d + 1;  // padded rows: lanes reading different keys hit different banks
  float* Ks = sm;                  // [CH][d+1]
  float* Vs = Ks + CH * ld;        // [CH][d+1]
  float* qs = Vs + CH * ld;        // [warps][d]
  float* ps = qs + kAttnWarps * d; // [warps][CH]
  __shared__ int s_last;

  const int c = blockIdx.x;
  const int g = blockIdx.y / n_qt, qt = blockIdx.y % n_qt;
  const int s = blockIdx.z;
  const int grp = a.nq / a.nkv;
  const int nqv = a.rows * grp;
  const int QD = a.nq * d;
  const int P = a.base_pos[s];
  const SeqKeys sk = seq_keys(a, P, gridDim.x, CH);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int qv0 = qt * kAttnQT;
  const int nq_tile = min(kAttnQT, nqv - qv0);
  const size_t grp_id = ((size_t)s * a.nkv + g) * n_qt + qt;
  const int stride_c = kAttnQT * (d + 2);
  float* part = a.partials + grp_id * (size_t)gridDim.x * stride_c;

  if (c < sk.n_ch) {
    const T* kp;
    const T* vp;
    int nk, slot0;
    chunk_keys<T>(a, sk, s, g, c, CH, kp, vp, nk, slot0);
    for (int t = threadIdx.x; t < CH * d; t += blockDim.x) {
      const int j = t / d, e = t % d;
      Ks[j * ld + e] = j < nk ? to_f<T>(kp[t]) : 0.f;
      Vs[j * ld + e] = j < nk ? to_f<T>(vp[t]) : 0.f;
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
      // last visible key of this chunk for this row
      const int limit = (a.mode == DFLASH_ATTN_CAUSAL) ? (P + row - slot0) : nk - 1;
      float mx = -INFINITY;
      for (int j = lane; j < CH; j += 32) {
        float sc = -INFINITY;
        if (j < nk && j <= limit) {
          float acc = 0.f;
          for (int e = 0; e < d; ++e) acc = fmaf(qs[warp * d + e], Ks[j * ld + e], acc);
          sc = acc * scale;
        }
        ps[warp * CH + j] = sc;
        mx = fmaxf(mx, sc);
      }
      mx = warp_max(mx);
      float l = 0.f;
      for (int j = lane; j < CH; j += 32) {
        const float sc = ps[warp * CH + j];
        const float p = (mx == -INFINITY || sc == -INFINITY) ? 0.f : exp2f(sc - mx);
        ps[warp * CH + j] = p;
        l += p;
      }
      l = warp_sum(l);
      __syncwarp();
      float* out = part + (size_t)c * stride_c + (size_t)qi * (d + 2);
      for (int e = lane; e < d; e += 32) {
        float o = 0.f;
        for (int j = 0; j < CH; ++j) o = fmaf(ps[warp * CH + j], Vs[j * ld + e], o);
        out[2 + e] = o;
      }
      if (lane == 0) {
        out[0] = mx;
        out[1] = l;
      }
      __syncwarp();
    }
  }
  attn_finish<T>(a, part, grp_id, stride_c, nq_tile, qv0, g, s, sk.n_ch, &s_last);
}

// ------------------------------------------------- bf16 tensor-core path

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void cp_async16(uint32_t saddr, const void* g) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(saddr), "l"(g) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// (x, y) as a bf16 pair hi plus the bf16 pair of the remainders lo: hi + lo
// carries the fp32 values to about 2^-17 relative, so a product with
// bf16 operands keeps the probabilities at fp32-like precision.
__device__ __forceinline__ void split_bf16(float x, float y, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
  const float2 hf = __bfloat1622float2(h);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = pack_bf16(x - hf.x, y - hf.y);
}

// Byte offset of (row, 16-byte chunk) in a [rows][D] bf16 tile whose chunk
// index is XOR-swizzled by the row, so ldmatrix row sets are bank-conflict free.
template <int D>
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return (uint32_t)(row * (D * 2) + ((chunk ^ (row & 7)) << 4));
}

namespace cg = cooperative_groups;

constexpr int kClusterWarps = 16;  // 4 row tiles x 4 key quarters of every chunk
constexpr int kClQT = 64;          // query vectors per cluster CTA
constexpr int kMaxNC = 16;

struct AttnTma {
  CUtensorMap kc, vc;  // cache [S*nkv*cap][D], box 64 dims x 128 keys, 128-byte swizzle
  CUtensorMap kb, vb;  // block scratch [S*nkv*rows][D] (bidirectional mode)
  CUtensorMap q3;      // queries [M][nq][D], box 64 dims x grp heads x 64/grp tokens (q_tma)
  int q_tma;           // the GQA group divides 64: a query tile is one 3-D box per 64 dims
  AttnDesc a;
};

// Byte offset of (key row j, 16-byte chunk ch) in a 128-key tile written by
// two (D = 128) or one (D = 64) TMA boxes of 64 dims with 128-byte swizzle.
__device__ __forceinline__ uint32_t kv_off(int j, int ch) {
  return (uint32_t)((ch >> 3) * (kMmaCH * 128) + j * 128 + (((ch & 7) ^ (j & 7)) << 4));
}

// Merge of the NC rank partials of one 64-query tile, in rank order; rank r
// writes rows [r*RP, (r+1)*RP) of the tile.  psm: this CTA's partial
// [64][D+4] (O, then m and l, log2 units), read by every rank through
// distributed shared memory; scratch: local shared memory.  The per-(row,
// rank) weights are formed once; then every output element reads its NC
// partial values with independent loads.
template <int D>
__device__ __forceinline__ void rank_merge(cg::cluster_group& cl, float* psm, float* scratch, int NC, int rank,
                                           int nq_tile, int qv0, int grp, int g, int s, int rows, int QD,
                                           void* out, uint32_t* status) {
  constexpr int PST = D + 4;
  const int RP = (nq_tile + NC - 1) / NC;
  const int q_lo = rank * RP;
  const int nrow = max(0, min(nq_tile, q_lo + RP) - q_lo);
  float* mw = scratch;               // [RP][kMaxNC] partial maxima, then weights
  float* lw = mw + RP * kMaxNC;      // [RP][kMaxNC] partial sums
  float* Ls = lw + RP * kMaxNC;      // [RP] merged sums
  for (int t = threadIdx.x; t < nrow * NC; t += blockDim.x) {
    const int i = t / NC, r = t % NC;
    const float* pr = cl.map_shared_rank(psm, r) + (size_t)(q_lo + i) * PST;
    mw[i * kMaxNC + r] = pr[D];
    lw[i * kMaxNC + r] = pr[D + 1];
  }
  __syncthreads();
  for (int i = threadIdx.x; i < nrow; i += blockDim.x) {
    float M = -INFINITY;
    for (int r = 0; r < NC; ++r) M = fmaxf(M, mw[i * kMaxNC + r]);
    float L = 0.f;
    for (int r = 0; r < NC; ++r) {
      const float mr = mw[i * kMaxNC + r];
      const float w = (mr == -INFINITY) ? 0.f : exp2f(mr - M);
      mw[i * kMaxNC + r] = w;
      L = fmaf(lw[i * kMaxNC + r], w, L);
    }
    Ls[i] = L;
  }
  __syncthreads();
  __nv_bfloat16* outp = reinterpret_cast<__nv_bfloat16*>(out);
  for (int t = threadIdx.x; t < nrow * (D / 4); t += blockDim.x) {
    const int i = t / (D / 4), e4 = 4 * (t % (D / 4));
    float4 v[kMaxNC];
#pragma unroll
    for (int r = 0; r < kMaxNC; ++r)
      if (r < NC) v[r] = *reinterpret_cast<const float4*>(cl.map_shared_rank(psm, r) + (size_t)(q_lo + i) * PST + e4);
    float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
#pragma unroll
    for (int r = 0; r < kMaxNC; ++r)
      if (r < NC) {
        const float w = mw[i * kMaxNC + r];
        o0 = fmaf(v[r].x, w, o0);
        o1 = fmaf(v[r].y, w, o1);
        o2 = fmaf(v[r].z, w, o2);
        o3 = fmaf(v[r].w, w, o3);
      }
    const float L = Ls[i];
    const int qv = qv0 + q_lo + i;
    const int row = qv / grp, head = g * grp + qv % grp;
    if (!DFL_CHECK(row < rows && head * D + e4 + 4 <= QD, status)) continue;
    __nv_bfloat162* dst = reinterpret_cast<__nv_bfloat162*>(outp + ((size_t)s * rows + row) * QD + (size_t)head * D + e4);
    dst[0] = __floats2bfloat162_rn(L > 0.f ? o0 / L : 0.f, L > 0.f ? o1 / L : 0.f);
    dst[1] = __floats2bfloat162_rn(L > 0.f ? o2 / L : 0.f, L > 0.f ? o3 / L : 0.f);
  }
}

// The normalised quad, rounded to bf16 (a row that saw no key gives zeros).
__device__ __forceinline__ void store_quad(__nv_bfloat16* dst, const float (&o)[4], float L) {
  __nv_bfloat162* d2 = reinterpret_cast<__nv_bfloat162*>(dst);
  d2[0] = __floats2bfloat162_rn(L > 0.f ? o[0] / L : 0.f, L > 0.f ? o[1] / L : 0.f);
  d2[1] = __floats2bfloat162_rn(L > 0.f ? o[2] / L : 0.f, L > 0.f ? o[3] / L : 0.f);
}

// The same merge with the partials pushed instead of pulled: after a
// cluster barrier (every rank's chunks done, its K/V buffers free), each
// rank stores its partial rows into their owner's shared memory (recv, on
// the owner, away from psm); after a second barrier each owner merges its
// rows from local shared memory, with the arithmetic and order of
// rank_merge, and nothing reads a peer's memory any more.  With E = 2 each
// CTA holds two logical ranks (rank and rank + NC; partials psm[0], psm[1])
// and owns the rows of both: the merge runs over the NL = E NC logical ranks
// in the same order as a cluster of NL CTAs.  recv: [E owned][NL][RP][D+4].
template <int D>
__device__ __forceinline__ void push_merge(cg::cluster_group& cl, const float* psm, float* recv, int NC, int E,
                                           int rank, int nq_tile, int qv0, int grp, int g, int s, int rows, int QD,
                                           void* out, uint32_t* status) {
  constexpr int PST = D + 4;
  const int NL = NC * E;
  const int RP = (nq_tile + NL - 1) / NL;
  for (int e = 0; e < E; ++e) {
    const float* pe = psm + (size_t)e * kClQT * PST;
    const int lr = rank + e * NC;  // logical rank of this partial
    for (int t = threadIdx.x; t < nq_tile * (PST / 4); t += blockDim.x) {
      const int qr = t / (PST / 4), c4 = t % (PST / 4);
      const int lo = qr / RP, i = qr - lo * RP;  // logical owner of the row
      const float4 v = *reinterpret_cast<const float4*>(pe + (size_t)qr * PST + 4 * c4);
      float* r = cl.map_shared_rank(recv, lo % NC) + (((size_t)(lo / NC) * NL + lr) * RP + i) * PST;
      *reinterpret_cast<float4*>(r + 4 * c4) = v;
    }
  }
  cl.sync();
  for (int sl = 0; sl < E; ++sl) {
  const float* rv = recv + (size_t)sl * NL * RP * PST;
  const int q_lo = (rank + sl * NC) * RP;
  const int nrow = max(0, min(nq_tile, q_lo + RP) - q_lo);
  __nv_bfloat16* outp = reinterpret_cast<__nv_bfloat16*>(out);
  for (int t = threadIdx.x; t < nrow * (D / 4); t += blockDim.x) {
    const int i = t / (D / 4), e4 = 4 * (t % (D / 4));
    // the arithmetic and order of the streaming kernel's merge phase
    float M = -INFINITY;
    for (int r = 0; r < NL; ++r) M = fmaxf(M, rv[((size_t)r * RP + i) * PST + D]);
    float L = 0.f, o[4] = {0.f, 0.f, 0.f, 0.f};
    for (int r = 0; r < NL; ++r) {
      const float* pr = rv + ((size_t)r * RP + i) * PST;
      const float mr = pr[D];
      const float w = (mr == -INFINITY) ? 0.f : exp2f(mr - M);
      L = fmaf(pr[D + 1], w, L);
      const float4 v = *reinterpret_cast<const float4*>(pr + e4);
      o[0] = fmaf(v.x, w, o[0]);
      o[1] = fmaf(v.y, w, o[1]);
      o[2] = fmaf(v.z, w, o[2]);
      o[3] = fmaf(v.w, w, o[3]);
    }
    const int qv = qv0 + q_lo + i;
    const int row = qv / grp, head = g * grp + qv % grp;
    if (!DFL_CHECK(row < rows && head * D + e4 + 4 <= QD, status)) continue;
    store_quad(outp + ((size_t)s * rows + row) * QD + (size_t)head * D + e4, o, L);
  }
  }
}

template <int D>
__global__ void __launch_bounds__(kClusterWarps * 32, 1) attn_cluster_kernel(const __grid_constant__ AttnTma p,
                                                                              int n_qt) {
  constexpr int CH = kMmaCH;
  constexpr int QK = CH / 4;         // keys per warp and chunk
  constexpr int CPR = D / 8;         // 16-byte chunks per row
  constexpr int TILE = CH * D * 2;   // one K or V chunk tile, bytes
  constexpr int PST = D + 4;         // floats per row of a partial (16-byte aligned rows)
  extern __shared__ __align__(1024) uint8_t smem_att[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_att) + 1023) & ~uintptr_t(1023));
  uint8_t* KV = sm;                        // buffer b: K at KV + 2*b*TILE, V at KV + (2*b+1)*TILE
  uint8_t* Qs = KV + 4 * TILE;             // [64][D]
  uint64_t* full = reinterpret_cast<uint64_t*>(Qs + kClQT * D * 2);  // [2]
  float* psm = reinterpret_cast<float*>(sm);         // [64][PST] CTA partial (after the chunk loop)
  float* qsm = psm + kClQT * PST;                    // [3][64][PST] key-quarter partials 1..3

  const AttnDesc& a = p.a;
  cg::cluster_group cl = cg::this_cluster();
  const int NC = (int)cl.num_blocks();
  const int rank = (int)cl.block_rank();
  const int g = blockIdx.y / n_qt, qt = blockIdx.y % n_qt;
  const int s = blockIdx.z;
  const int mode = a.mode, rows = a.rows, cap = a.cap, nkv = a.nkv;
  const int grp = a.nq / a.nkv;
  const int nqv = rows * grp;
  const int QD = a.nq * D;
  uint32_t* status = a.status;
  // base_pos is written only by the acceptance step, never by the kernel that
  // precedes attention inside a call, so it may be read before the PDL wait.
  const int P = a.base_pos[s];
  SeqKeys sk;
  if (mode == DFLASH_ATTN_CAUSAL) {
    sk.n_ctx = min(max(P + rows, 0), cap);
    sk.n_ctx_ch = (sk.n_ctx + CH - 1) / CH;
    sk.n_ch = sk.n_ctx_ch;
  } else {
    sk.n_ctx = min(max(a.window > 0 ? min(P, a.window) : P, 0), cap);
    sk.n_ctx_ch = (sk.n_ctx + CH - 1) / CH;
    sk.n_ch = sk.n_ctx_ch + 1;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int wq = warp & 3, kq = warp >> 2;
  const int qv0 = qt * kClQT;
  const int nq_tile = min(kClQT, nqv - qv0);
  const int nmine = sk.n_ch > rank ? (sk.n_ch - rank + NC - 1) / NC : 0;
  const uint32_t qb = __cvta_generic_to_shared(Qs);
  const uint32_t kvb = __cvta_generic_to_shared(KV);

  // chunk c -> (is block chunk, first tensor row)
  const KvMap km{a.pages, cap, a.ps, a.max_pages, a.pool, nkv};
  const uint64_t lim = wait_limit_ns(status);
  const bool stall = stall_kv_loads(status);  // test switch: issue no K/V copy
  auto chunk_row = [&](int c, bool& blk) -> int {
    blk = (mode == DFLASH_ATTN_BLOCK_BIDIR && c == sk.n_ctx_ch);
    if (blk) return (s * nkv + g) * rows;
    bool bad = false;
    const int r = (int)(km.row0(s, c * CH, &bad) + (uint32_t)g * (uint32_t)km.head_rows());
    if (bad) raise_status(status, ST_RANGE);  // read from page 0 instead
    return r;
  };
  auto issue = [&](int c, int buf) {  // one thread
    if (stall) return;
    bool blk;
    const int row = chunk_row(c, blk);
    const CUtensorMap* km = blk ? &p.kb : &p.kc;
    const CUtensorMap* vm = blk ? &p.vb : &p.vc;
    uint8_t* Kt = KV + 2 * buf * TILE;
    tc::mbar_arrive_expect_tx(&full[buf], 2 * TILE);
    const uint64_t pol = tc::policy_evict_first();
#pragma unroll
    for (int h = 0; h < D / 64; ++h) {
      tc::tma_load_2d(Kt + h * (CH * 128), km, 64 * h, row, &full[buf], pol);
      tc::tma_load_2d(Kt + TILE + h * (CH * 128), vm, 64 * h, row, &full[buf], pol);
    }
  };
  // a chunk the preceding kernel cannot have written (context below P)
  auto early_ok = [&](int c) { return c < sk.n_ctx_ch && (mode == DFLASH_ATTN_BLOCK_BIDIR || (c + 1) * CH <= P); };

  if (threadIdx.x == 0) {
    tc::mbar_init(&full[0], 1);
    tc::mbar_init(&full[1], 1);
    tc::fence_mbar_init();
    tc::tma_prefetch_desc(&p.kc);
    tc::tma_prefetch_desc(&p.vc);
  }
  __syncthreads();
  bool pre0 = false, pre1 = false;
  int issued = 0;  // chunks thread 0 issued (stalled: none)
  if (threadIdx.x == 0) {
    if (nmine > 0 && early_ok(rank)) { issue(rank, 0); pre0 = true; }
    if (nmine > 1 && early_ok(rank + NC)) { issue(rank + NC, 1); pre1 = true; }
    issued = stall ? 0 : (nmine < 2 ? nmine : 2);
  }
  pdl_wait();
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    if (nmine > 0 && !pre0) issue(rank, 0);
    if (nmine > 1 && !pre1) issue(rank + NC, 1);
  }
  // ---- Q (rows >= nq_tile zero)
  for (int t = threadIdx.x; t < kClQT * CPR; t += blockDim.x) {
    const int qi = t / CPR, ch = t % CPR;
    if (qi < nq_tile) {
      const int qv = qv0 + qi;
      const int row = qv / grp, head = g * grp + qv % grp;
      const __nv_bfloat16* q =
          reinterpret_cast<const __nv_bfloat16*>(a.q) + ((size_t)s * rows + row) * QD + (size_t)head * D;
      cp_async16(qb + swz<D>(qi, ch), q + ch * 8);
    } else {
      *reinterpret_cast<uint4*>(Qs + swz<D>(qi, ch)) = make_uint4(0, 0, 0, 0);
    }
  }
  cp_async_wait_all();
  __syncthreads();

  const int r0 = 16 * wq;  // this warp's 16 query vectors
  const bool warp_on = r0 < nq_tile;
  const int qa = r0 + (lane >> 2), qb2 = qa + 8;  // the two rows this thread holds
  const int row_a = (qv0 + qa) / grp, row_b = (qv0 + qb2) / grp;
  const float scale = rsqrtf((float)D) * kLog2e;
  float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;
  float O[D / 8][4];
#pragma unroll
  for (int t = 0; t < D / 8; ++t) O[t][0] = O[t][1] = O[t][2] = O[t][3] = 0.f;
  bool failed = false;

  for (int i = 0; i < nmine; ++i) {
    const int c = rank + i * NC, buf = i & 1;
    if (!failed && !tc::mbar_wait(&full[buf], (uint32_t)(i >> 1) & 1u, nullptr, lim)) {
      raise_status(status, ST_TIMEOUT);
      failed = true;
    }
    const uint32_t kb = kvb + 2 * buf * TILE, vb = kb + TILE;
    bool blk;
    chunk_row(c, blk);
    const int slot0 = blk ? -1 : c * CH;
    const int nk = blk ? min(rows, CH) : min(CH, sk.n_ctx - c * CH);
    if (nk < CH) {
      // Rows past the last key hold whatever follows in memory (unwritten
      // cache slots may be NaN); zero V there so that P = 0 contributes 0.
      uint8_t* Vt = KV + (2 * buf + 1) * TILE;
      for (int t = threadIdx.x; t < (CH - nk) * (D / 8); t += blockDim.x) {
        const int j = nk + t / (D / 8), ch = t % (D / 8);
        *reinterpret_cast<uint4*>(Vt + kv_off(j, ch)) = make_uint4(0, 0, 0, 0);
      }
      tc::fence_proxy_async_smem();
      __syncthreads();
    }
    if (!failed && warp_on && QK * kq < nk) {
      // S = Q K^T over this warp's quarter of the chunk (keys QK*kq .. QK*kq + QK)
      float S[QK / 8][4];
#pragma unroll
      for (int t = 0; t < QK / 8; ++t) S[t][0] = S[t][1] = S[t][2] = S[t][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(qb + swz<D>(r0 + (lane & 15), 2 * ks + (lane >> 4)), a0, a1, a2, a3);
#pragma unroll
        for (int nt = 0; nt < QK / 16; ++nt) {
          uint32_t b0, b1, b2, b3;
          const int key = QK * kq + 16 * nt + (lane & 7) + ((lane >> 4) << 3);
          ldsm_x4(kb + kv_off(key, 2 * ks + ((lane >> 3) & 1)), b0, b1, b2, b3);
          mma_16816(S[2 * nt], a0, a1, a2, a3, b0, b1);
          mma_16816(S[2 * nt + 1], a0, a1, a2, a3, b2, b3);
        }
      }
      // mask, scale to log2 units, maxima over this quarter
      const bool causal = mode == DFLASH_ATTN_CAUSAL && slot0 >= 0;
      const int lim_a = causal ? P + row_a - slot0 : CH;
      const int lim_b = causal ? P + row_b - slot0 : CH;
      float cm_a = -INFINITY, cm_b = -INFINITY;
#pragma unroll
      for (int t = 0; t < QK / 8; ++t) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int j = QK * kq + 8 * t + 2 * (lane & 3) + e;  // key index within the chunk
          S[t][e] = (j < nk && j <= lim_a) ? S[t][e] * scale : -INFINITY;
          S[t][2 + e] = (j < nk && j <= lim_b) ? S[t][2 + e] * scale : -INFINITY;
          cm_a = fmaxf(cm_a, S[t][e]);
          cm_b = fmaxf(cm_b, S[t][2 + e]);
        }
      }
      cm_a = fmaxf(cm_a, __shfl_xor_sync(0xffffffffu, cm_a, 1));
      cm_a = fmaxf(cm_a, __shfl_xor_sync(0xffffffffu, cm_a, 2));
      cm_b = fmaxf(cm_b, __shfl_xor_sync(0xffffffffu, cm_b, 1));
      cm_b = fmaxf(cm_b, __shfl_xor_sync(0xffffffffu, cm_b, 2));
      // online softmax: rescale the running state to the new maximum
      const float mn_a = fmaxf(m_a, cm_a), mn_b = fmaxf(m_b, cm_b);
      const float al_a = (m_a == -INFINITY) ? 0.f : exp2f(m_a - mn_a);
      const float al_b = (m_b == -INFINITY) ? 0.f : exp2f(m_b - mn_b);
      float sl_a = 0.f, sl_b = 0.f;
#pragma unroll
      for (int t = 0; t < QK / 8; ++t) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float pa = (S[t][e] == -INFINITY) ? 0.f : exp2f(S[t][e] - mn_a);
          const float pb = (S[t][2 + e] == -INFINITY) ? 0.f : exp2f(S[t][2 + e] - mn_b);
          S[t][e] = pa;
          S[t][2 + e] = pb;
          sl_a += pa;
          sl_b += pb;
        }
      }
      sl_a += __shfl_xor_sync(0xffffffffu, sl_a, 1);
      sl_a += __shfl_xor_sync(0xffffffffu, sl_a, 2);
      sl_b += __shfl_xor_sync(0xffffffffu, sl_b, 1);
      sl_b += __shfl_xor_sync(0xffffffffu, sl_b, 2);
      l_a = fmaf(l_a, al_a, sl_a);
      l_b = fmaf(l_b, al_b, sl_b);
      m_a = mn_a;
      m_b = mn_b;
#pragma unroll
      for (int t = 0; t < D / 8; ++t) {
        O[t][0] *= al_a;
        O[t][1] *= al_a;
        O[t][2] *= al_b;
        O[t][3] *= al_b;
      }
      // O += P V over the quarter.  The probabilities stay fp32 (softmax is
      // not a rounding point): P = P_hi + P_lo as two bf16 operands.
#pragma unroll
      for (int kk = 0; kk < QK / 16; ++kk) {
        uint32_t a0, a1, a2, a3, l0, l1, l2, l3;
        split_bf16(S[2 * kk][0], S[2 * kk][1], a0, l0);
        split_bf16(S[2 * kk][2], S[2 * kk][3], a1, l1);
        split_bf16(S[2 * kk + 1][0], S[2 * kk + 1][1], a2, l2);
        split_bf16(S[2 * kk + 1][2], S[2 * kk + 1][3], a3, l3);
#pragma unroll
        for (int dt = 0; dt < D / 16; ++dt) {
          uint32_t b0, b1, b2, b3;
          const int key = QK * kq + 16 * kk + (lane & 7) + (((lane >> 3) & 1) << 3);
          ldsm_x4_t(vb + kv_off(key, 2 * dt + (lane >> 4)), b0, b1, b2, b3);
          mma_16816(O[2 * dt], a0, a1, a2, a3, b0, b1);
          mma_16816(O[2 * dt + 1], a0, a1, a2, a3, b2, b3);
          mma_16816(O[2 * dt], l0, l1, l2, l3, b0, b1);
          mma_16816(O[2 * dt + 1], l0, l1, l2, l3, b2, b3);
        }
      }
    }
    __syncthreads();  // every warp is done with this buffer
    if (threadIdx.x == 0 && i + 2 < nmine && !failed) {
      issue(rank + (i + 2) * NC, buf);
      if (!stall) ++issued;
    }
  }
  // every issued copy has landed before the partials overwrite the buffers
  if (threadIdx.x == 0)
    for (int i = issued > 2 ? issued - 2 : 0; i < issued; ++i)
      tc::mbar_wait(&full[i & 1], (uint32_t)(i >> 1) & 1u, nullptr, lim);
  __syncthreads();

  // ---- merge the four key quarters in order, then this CTA's partial
  if (warp_on && kq > 0) {
    float* pa = qsm + ((size_t)(kq - 1) * kClQT + qa) * PST;
    float* pb = qsm + ((size_t)(kq - 1) * kClQT + qb2) * PST;
#pragma unroll
    for (int t = 0; t < D / 8; ++t) {
      const int col = 8 * t + 2 * (lane & 3);
      pa[col] = O[t][0];
      pa[col + 1] = O[t][1];
      pb[col] = O[t][2];
      pb[col + 1] = O[t][3];
    }
    pa[D + (lane & 3)] = (lane & 3) == 0 ? m_a : l_a;  // lanes 0/1 of the quad hold m / l
    pb[D + (lane & 3)] = (lane & 3) == 0 ? m_b : l_b;
  }
  __syncthreads();
  if (warp_on && kq == 0) {
    float Ma = m_a, Mb = m_b;
#pragma unroll
    for (int qq = 0; qq < 3; ++qq) {
      Ma = fmaxf(Ma, qsm[((size_t)qq * kClQT + qa) * PST + D]);
      Mb = fmaxf(Mb, qsm[((size_t)qq * kClQT + qb2) * PST + D]);
    }
    float wa[4], wb[4];
    wa[0] = (m_a == -INFINITY) ? 0.f : exp2f(m_a - Ma);
    wb[0] = (m_b == -INFINITY) ? 0.f : exp2f(m_b - Mb);
    float La = l_a * wa[0], Lb = l_b * wb[0];
#pragma unroll
    for (int qq = 0; qq < 3; ++qq) {
      const float* ha = qsm + ((size_t)qq * kClQT + qa) * PST;
      const float* hb = qsm + ((size_t)qq * kClQT + qb2) * PST;
      wa[qq + 1] = (ha[D] == -INFINITY) ? 0.f : exp2f(ha[D] - Ma);
      wb[qq + 1] = (hb[D] == -INFINITY) ? 0.f : exp2f(hb[D] - Mb);
      La = fmaf(ha[D + 1], wa[qq + 1], La);
      Lb = fmaf(hb[D + 1], wb[qq + 1], Lb);
    }
    float* pa = psm + (size_t)qa * PST;
    float* pb = psm + (size_t)qb2 * PST;
#pragma unroll
    for (int t = 0; t < D / 8; ++t) {
      const int col = 8 * t + 2 * (lane & 3);
      float oa0 = O[t][0] * wa[0], oa1 = O[t][1] * wa[0], ob0 = O[t][2] * wb[0], ob1 = O[t][3] * wb[0];
#pragma unroll
      for (int qq = 0; qq < 3; ++qq) {
        const float* ha = qsm + ((size_t)qq * kClQT + qa) * PST;
        const float* hb = qsm + ((size_t)qq * kClQT + qb2) * PST;
        oa0 = fmaf(ha[col], wa[qq + 1], oa0);
        oa1 = fmaf(ha[col + 1], wa[qq + 1], oa1);
        ob0 = fmaf(hb[col], wb[qq + 1], ob0);
        ob1 = fmaf(hb[col + 1], wb[qq + 1], ob1);
      }
      pa[col] = oa0;
      pa[col + 1] = oa1;
      pb[col] = ob0;
      pb[col + 1] = ob1;
    }
    if ((lane & 3) == 0) {
      pa[D] = Ma;
      pa[D + 1] = La;
      pb[D] = Mb;
      pb[D + 1] = Lb;
    }
  }
  cl.sync();

  rank_merge<D>(cl, psm, qsm, NC, rank, nq_tile, qv0, grp, g, s, rows, QD, a.out, status);
  cl.sync();  // peers keep their shared memory until every rank has read it
}

// ---------------------------------------------------------- tcgen05 variant
//
// Same work split as attn_cluster_kernel (one cluster of NC CTAs per
// (sequence, KV head, 64-query tile), rank r owns chunks r, r+NC, ...), with
// both products on the 5th-generation tensor cores: per 128-key chunk
// S = Q K^T (M = 128 MMA rows: the 64 query rows of the tile, then the same
// 64 again; N = 128 keys; K = 128 dims) into one of two TMEM accumulators.
// The softmax warps (sixteen: 2..17), four per key group and one of each
// group on every TMEM lane quadrant, read S: the thread on TMEM lane l of key
// group k takes query row l mod 64 and the KP = 16 keys of piece 2k + l / 64,
// so every row is shared by 8 threads, which exchange their maxima and sums
// through shared memory in piece order.  P
// goes to shared memory as a bf16 pair (P_hi, P_lo), the running output O is
// rescaled in TMEM, then O += P_hi V + P_lo V (V as an MN-major operand).
// Roles: warp 0 issues the K/V TMA copies, one lane of warp 1 the MMAs; S of
// chunk i+1 is computed while the softmax of chunk i runs.  Every wait is
// bounded.
// Sixteen softmax warps (KP = 16 keys per thread, 96 registers) measured
// faster than eight (KP = 32: each chunk's softmax is a chain of dependent
// instructions, which four warps per sub-partition hide better than two) and
// than four.
#ifndef DFLASH_TC_ATTN_SOFT_WARPS
#define DFLASH_TC_ATTN_SOFT_WARPS 16
#endif
constexpr int kTcAttnSoftWarps = DFLASH_TC_ATTN_SOFT_WARPS;  // 4 per TMEM lane quadrant x key groups
constexpr int kTcAttnSoft = kTcAttnSoftWarps * 32;
constexpr int kTcAttnThreads = 64 + kTcAttnSoft;
constexpr int kTcAttnRows = 128;                          // MMA rows (the 64-query tile, twice)
constexpr int kTcAttnGroups = kTcAttnSoftWarps / 4;       // key groups
constexpr int kTcAttnPieces = 2 * kTcAttnGroups;          // key pieces of a chunk (x 2 row copies)
constexpr int kTcAttnKP = kMmaCH / kTcAttnPieces;         // keys per softmax thread
static_assert(kTcAttnSoftWarps % 4 == 0 && kTcAttnKP % 16 == 0, "whole 16-column TMEM loads");
// P_hi and P_lo are [128 rows][128 keys] operands (two 64-key boxes of 128
// rows), but only rows 0..63 are ever written: P_lo starts 64 rows after P_hi,
// so the rows 64..127 the PV MMA reads (and whose output is discarded) fall on
// the other operand's live rows, and the pair takes 40 KB instead of 64.
constexpr int kTcAttnPloOff = 64 * 128;
constexpr int kTcAttnPBytes = kTcAttnPloOff + 2 * kTcAttnRows * 128;

__host__ __device__ constexpr size_t tc_attn_smem(int d) {
  return 4 * (size_t)kMmaCH * d * 2             // two K/V chunk buffers
         + (size_t)kTcAttnRows * d * 2          // Q
         + (size_t)kTcAttnPBytes                // P_hi, P_lo
         + 128                                  // barriers
         + 2 * 2 * kTcAttnPieces * 64 * 4       // row max / sum exchange, double-buffered
         + 1024;                                // alignment
}

// The softmax steps of one thread's KP keys, shared by the tcgen05 kernels so
// that they compute the same values.  Scores: scaled to log2 units, keys past
// the chunk's last key or the causal limit masked to -inf; the maximum is
// taken over four interleaved partial maxima (exact in any order).
template <int KP>
__device__ __forceinline__ float soft_scores(float (&sc)[KP], int j0, int nk, int lim, float scale) {
  float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int t = 0; t < KP; ++t) {
    const int j = j0 + t;  // key index in the chunk
    sc[t] = (j < nk && j <= lim) ? sc[t] * scale : -INFINITY;
    m4[t & 3] = fmaxf(m4[t & 3], sc[t]);
  }
  return fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
}

// One thread's KP scores of a chunk from TMEM (one load, one wait).
template <int KP>
__device__ __forceinline__ void tmem_ld_scores(uint32_t taddr, float (&sc)[KP]) {
  static_assert(KP == 16 || KP == 32, "16 or 32 keys per softmax thread");
  if constexpr (KP == 32) tc::tmem_ld32(taddr, sc);
  else tc::tmem_ld16(taddr, sc);
}

// N consecutive fp32 columns of this thread's TMEM lane (one load, one wait).
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&v)[N]) {
  static_assert(N == 16 || N == 32 || N == 64, "16, 32 or 64 columns");
  if constexpr (N == 64) tc::tmem_ld64(taddr, v);
  else if constexpr (N == 32) tc::tmem_ld32(taddr, v);
  else tc::tmem_ld16(taddr, v);
}

// 2^x by the hardware approximation (PTX ex2.approx.ftz; results below the
// normal range flush to 0): the arguments are at most 8, and P is carried as
// a bf16 pair (about 16 bits) anyway.
__device__ __forceinline__ float ex2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// P = 2^(s - m_new) in place, and its sum: four interleaved partial sums,
// added pairwise.
template <int KP>
__device__ __forceinline__ float soft_exp(float (&sc)[KP], float m_new) {
  float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int t = 0; t < KP; ++t) {
    const float pj = (sc[t] == -INFINITY) ? 0.f : ex2_fast(sc[t] - m_new);
    sc[t] = pj;
    s4[t & 3] += pj;
  }
  return (s4[0] + s4[1]) + (s4[2] + s4[3]);
}

// Byte offset of (row, 16-byte chunk) in a [128 rows][64 x nbox] bf16 operand
// stored as nbox 128-byte swizzled boxes of 128 rows (the TMA layout).
__device__ __forceinline__ uint32_t op_off(int row, int ch) {
  return (uint32_t)((ch >> 3) * (kTcAttnRows * 128) + row * 128 + (((ch & 7) ^ (row & 7)) << 4));
}

// E: logical ranks per CTA (1, or 2 on clusters of half the logical width).
template <int D, int E>
__global__ void __launch_bounds__(kTcAttnThreads, 1) attn_tc_kernel(const __grid_constant__ AttnTma p, int n_qt) {
  static_assert(E == 1 || E == 2, "one or two logical ranks per CTA");
  static_assert(D == 128, "two 64-dim boxes per row");
  constexpr int CH = kMmaCH;
  constexpr int TILE = CH * D * 2;
  constexpr int QB = kTcAttnRows * D * 2;
  constexpr int PST = D + 4;
  constexpr int KP = kTcAttnKP;
  constexpr int OC = D / kTcAttnGroups;  // output columns per owner thread
  static_assert(CH == 128 && OC % 16 == 0, "whole 16-column TMEM loads");
  extern __shared__ __align__(1024) uint8_t smem_att[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_att) + 1023) & ~uintptr_t(1023));
  uint8_t* KV = sm;  // buffer b: K at KV + 2*b*TILE, V at KV + (2*b+1)*TILE
  uint8_t* Qs = KV + 4 * TILE;
  uint8_t* Ph = Qs + QB;
  uint8_t* Pl = Ph + kTcAttnPloOff;
  uint64_t* full = reinterpret_cast<uint64_t*>(Ph + kTcAttnPBytes);  // [2] K/V chunk landed
  uint64_t* empty = full + 2;                             // [2] K/V chunk consumed
  uint64_t* sfull = empty + 2;                            // [2] S in TMEM
  uint64_t* pdone = sfull + 2;                            // [2] P written, O rescaled
  uint64_t* ofull = pdone + 2;                            // P V done
  uint64_t* qfull = ofull + 1;                            // Q landed (TMA path)
  uint32_t* tslot = reinterpret_cast<uint32_t*>(qfull + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tslot + 1);
  // [2 chunk parities][8 pieces][64 rows] each
  float* xmax = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(full) + 128);
  float* xsum = xmax + 2 * kTcAttnPieces * 64;
  float* psm = reinterpret_cast<float*>(sm);   // [E][64][PST] CTA partials (after the chunk loop)

  const AttnDesc& a = p.a;
  cg::cluster_group cl = cg::this_cluster();
  const int NC = (int)cl.num_blocks();
  const int rank = (int)cl.block_rank();
  // Logical ranks: NL = E x the cluster width; this CTA runs logical ranks
  // rank and (E = 2) rank + NC one after the other, each an online softmax
  // over its own chunks with its own output accumulator.
  const int NL = E * NC;
  const int g = blockIdx.y / n_qt, qt = blockIdx.y % n_qt;
  const int s = blockIdx.z;
  const int mode = a.mode, rows = a.rows, cap = a.cap, nkv = a.nkv;
  const int grp = a.nq / a.nkv;
  const int nqv = rows * grp;
  const int QD = a.nq * D;
  uint32_t* status = a.status;
  // base_pos is written only by the acceptance step, never by the kernel that
  // precedes attention inside a call, so it may be read before the PDL wait.
  const int P = a.base_pos[s];
  const SeqKeys sk = tc_seq_keys(a, P);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int qv0 = qt * kClQT;
  const int nq_tile = min(kClQT, nqv - qv0);
  const int rB = rank + NC;  // second logical rank (E = 2)
  const int nA = sk.n_ch > rank ? (sk.n_ch - rank + NL - 1) / NL : 0;
  const int nB = (E > 1 && sk.n_ch > rB) ? (sk.n_ch - rB + NL - 1) / NL : 0;
  const int nmine = nA + nB;
  auto chunk_of = [&](int i) { return i < nA ? rank + i * NL : rB + (i - nA) * NL; };

  const KvMap km{a.pages, cap, a.ps, a.max_pages, a.pool, nkv};
  const uint64_t lim_ns = wait_limit_ns(status);  // (lim is the causal key limit below)
  const bool stall = stall_kv_loads(status);  // test switch: issue no K/V copy
  auto chunk_row = [&](int c, bool& blk) -> int {
    blk = (mode == DFLASH_ATTN_BLOCK_BIDIR && c == sk.n_ctx_ch);
    if (blk) return (s * nkv + g) * rows;
    bool bad = false;
    const int r = (int)(km.row0(s, c * CH, &bad) + (uint32_t)g * (uint32_t)km.head_rows());
    if (bad) raise_status(status, ST_RANGE);  // read from page 0 instead
    return r;
  };
  auto issue = [&](int c, int buf) {  // one thread
    if (stall) return;
    bool blk;
    const int row = chunk_row(c, blk);
    const CUtensorMap* km = blk ? &p.kb : &p.kc;
    const CUtensorMap* vm = blk ? &p.vb : &p.vc;
    uint8_t* Kt = KV + 2 * buf * TILE;
    tc::mbar_arrive_expect_tx(&full[buf], 2 * TILE);
    const uint64_t pol = tc::policy_evict_first();
#pragma unroll
    for (int h = 0; h < D / 64; ++h) {
      tc::tma_load_2d(Kt + h * (CH * 128), km, 64 * h, row, &full[buf], pol);
      tc::tma_load_2d(Kt + TILE + h * (CH * 128), vm, 64 * h, row, &full[buf], pol);
    }
  };
  auto early_ok = [&](int c) { return c < sk.n_ctx_ch && (mode == DFLASH_ATTN_BLOCK_BIDIR || (c + 1) * CH <= P); };

  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&full[b], 1);
      tc::mbar_init(&empty[b], 1);
      tc::mbar_init(&sfull[b], 1);
      tc::mbar_init(&pdone[b], kTcAttnSoft);
    }
    tc::mbar_init(ofull, 1);
    tc::mbar_init(qfull, 1);
    *abort = 0;
    tc::fence_mbar_init();
    tc::tma_prefetch_desc(&p.kc);
    tc::tma_prefetch_desc(&p.vc);
    if (p.q_tma) tc::tma_prefetch_desc(&p.q3);
  }
  if (warp == 1) tc::tmem_alloc(tslot, 512);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tslot;
  bool pre0 = false, pre1 = false;
  if (threadIdx.x == 0) {
    if (nmine > 0 && early_ok(chunk_of(0))) { issue(chunk_of(0), 0); pre0 = true; }
    if (nmine > 1 && early_ok(chunk_of(1))) { issue(chunk_of(1), 1); pre1 = true; }
  }
  pdl_wait();
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    if (nmine > 0 && !pre0) issue(chunk_of(0), 0);
    if (nmine > 1 && !pre1) issue(chunk_of(1), 1);
  }
  // ---- Q: the tile's query vectors in rows 0..63 and again in rows 64..127
  // (TMEM lanes 64..127 then hold a copy of every score row, so the softmax
  // warps on all four lane quadrants share the rows).  When the GQA group
  // divides 64 the tile (64 / grp tokens x grp heads) is one 3-D TMA box per
  // 64 dims, loaded twice; rows past the tile's last query vector then hold
  // other queries or zeros, whose rows of S, P and O are never used.
  const uint32_t qb = __cvta_generic_to_shared(Qs);
  if (p.q_tma) {
    if (threadIdx.x == 0) {
      tc::mbar_arrive_expect_tx(qfull, 4 * kClQT * 128);
      const int z = s * rows + qv0 / grp, y = g * grp;
#pragma unroll
      for (int h = 0; h < D / 64; ++h)
#pragma unroll
        for (int dup = 0; dup < 2; ++dup)
          tc::tma_load_3d(Qs + h * (kTcAttnRows * 128) + dup * (kClQT * 128), &p.q3, 64 * h, y, z, qfull);
    }
  } else {
    for (int t = threadIdx.x; t < kTcAttnRows * (D / 8); t += blockDim.x) {
      const int qrow = t / (D / 8), ch = t % (D / 8);
      const int qi = qrow & (kClQT - 1);
      if (qi < nq_tile) {
        const int qv = qv0 + qi;
        const int row = qv / grp, head = g * grp + qv % grp;
        const __nv_bfloat16* q =
            reinterpret_cast<const __nv_bfloat16*>(a.q) + ((size_t)s * rows + row) * QD + (size_t)head * D;
        cp_async16(qb + op_off(qrow, ch), q + ch * 8);
      } else {
        *reinterpret_cast<uint4*>(Qs + op_off(qrow, ch)) = make_uint4(0, 0, 0, 0);
      }
    }
    cp_async_wait_all();
    tc::fence_proxy_async_smem();
  }
  __syncthreads();

  const uint32_t kvb = __cvta_generic_to_shared(KV);
  const uint32_t phb = __cvta_generic_to_shared(Ph), plb = __cvta_generic_to_shared(Pl);
  if (warp == 0) {
    if (lane == 0) {
      // ---------------- K/V producer: chunk i into buffer i & 1 once P V of chunk i-2 is done
      int issued = stall ? 0 : (nmine < 2 ? nmine : 2);  // this thread issued chunks 0 and 1 above
      for (int i = 2; i < nmine; ++i) {
        if (!tc::mbar_wait(&empty[i & 1], (uint32_t)((i - 2) >> 1) & 1u, abort, lim_ns)) {
          raise_status(status, ST_TIMEOUT);
          *abort = 1;
          break;
        }
        issue(chunk_of(i), i & 1);
        if (!stall) ++issued;
      }
      // Every copy this CTA issued has landed before its shared memory goes
      // away, also when a wait gave up (the last copy into each buffer).
      for (int i = issued > 2 ? issued - 2 : 0; i < issued; ++i)
        tc::mbar_wait(&full[i & 1], (uint32_t)(i >> 1) & 1u, nullptr, lim_ns);
      if (p.q_tma) tc::mbar_wait(qfull, 0u, nullptr, lim_ns);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      constexpr uint32_t idS = tc::idesc_bf16_f32(kTcAttnRows, CH);
      constexpr uint32_t idV = tc::idesc_bf16_f32_bmn(kTcAttnRows, D);
      bool ok = true;
      auto wait = [&](uint64_t* bar, uint32_t par) {
        if (ok && !tc::mbar_wait(bar, par, abort, lim_ns)) {
          raise_status(status, ST_TIMEOUT);
          *abort = 1;
          ok = false;
        }
        return ok;
      };
      auto issue_s = [&](int i) {
        const int b = i & 1;
        if (!wait(&full[b], (uint32_t)(i >> 1) & 1u)) return;
        tc::tc_fence_after();
        const uint32_t kb = kvb + 2 * b * TILE;
#pragma unroll
        for (int j = 0; j < D / 16; ++j) {
          const uint32_t off = (uint32_t)((j >> 2) * (kTcAttnRows * 128) + (j & 3) * 32);
          const uint32_t koff = (uint32_t)((j >> 2) * (CH * 128) + (j & 3) * 32);
          tc::mma_bf16(tmem + (uint32_t)(b * CH), tc::sdesc_sw128(qb + off), tc::sdesc_sw128(kb + koff), idS,
                       j > 0 ? 1u : 0u);
        }
        tc::mma_commit(&sfull[b]);
      };
      if (p.q_tma) wait(qfull, 0u);  // a timeout raises the abort flag: the loops below then stop
      // S of the first two chunks up front; then P V of chunk i as soon as its
      // P is written, and S of chunk i+2 after it (its K/V buffer and S
      // accumulator are the ones chunk i used), so that a chunk's load
      // latency hides behind the softmax of the chunk before it.
      // S of chunk ns is issued once its K/V has landed, and at the latest
      // before the wait for the softmax of that chunk; an S whose K is still
      // on its way never holds up the P V of the chunk before it.
      int ns = 0;
      for (; ns < nmine && ns < 2; ++ns) issue_s(ns);
      for (int i = 0; i < nmine && ok; ++i) {
        for (; ns <= i && ok; ++ns) issue_s(ns);
        if (!wait(&pdone[i & 1], (uint32_t)(i >> 1) & 1u)) break;
        tc::tc_fence_after();
        const uint32_t vb = kvb + (2 * (i & 1) + 1) * TILE;
        const int li = i < nA ? i : i - nA;                          // chunk within its logical rank
        const uint32_t od = tmem + (uint32_t)((i < nA ? 2 : 3) * CH);  // that rank's output accumulator
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const uint32_t pb = half ? plb : phb;
#pragma unroll
          for (int j = 0; j < CH / 16; ++j) {
            const uint32_t poff = (uint32_t)((j >> 2) * (kTcAttnRows * 128) + (j & 3) * 32);
            tc::mma_bf16(od, tc::sdesc_sw128(pb + poff),
                         tc::sdesc_sw128_mn(vb + (uint32_t)j * 2048u, CH * 128, 1024), idV,
                         (li > 0 || half > 0 || j > 0) ? 1u : 0u);
          }
        }
        tc::mma_commit(&empty[i & 1]);
        tc::mma_commit(ofull);
        if (ns == i + 2 && ns < nmine && tc::mbar_test(&full[ns & 1], (uint32_t)(ns >> 1) & 1u)) issue_s(ns++);
      }
    }
  } else {
    // ---------------- softmax, warps 2..17: TMEM lane L holds score row L;
    // rows 0..63 and their copies 64..127 are the same query row q = L & 63.
    // Warp w reads the lanes of quadrant w & 3; its key group kg = (w - 2) / 4
    // and the row copy h = L >> 6 pick the KP keys of piece 2 kg + h.
    const int sw = warp - 2;
    const int L = (warp & 3) * 32 + lane;
    const int qr = L & (kClQT - 1), h = L >> 6;
    const int kg = sw >> 2, piece = 2 * kg + h;
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const bool o_owner = h == 0;  // lanes 0..63 hold the output rows; this thread takes columns OC kg ..
    const int row_tok = (qv0 + qr) / grp;
    const float scale = rsqrtf((float)D) * kLog2e;
    float m_run = -INFINITY, l_run = 0.f;
    float mA = -INFINITY, lA = 0.f;  // the first logical rank's state once the second starts
    bool ok = true;
    for (int i = 0; i < nmine; ++i) {
      const int c = chunk_of(i), b = i & 1;
      const int li = i < nA ? i : i - nA;
      if (i == nA) {  // the second logical rank starts from scratch
        mA = m_run;
        lA = l_run;
        m_run = -INFINITY;
        l_run = 0.f;
      }
      float* xm = xmax + b * (kTcAttnPieces * 64);
      float* xs = xsum + b * (kTcAttnPieces * 64);
      bool blk;
      chunk_row(c, blk);
      const int slot0 = blk ? -1 : c * CH;
      const int nk = blk ? min(rows, CH) : min(CH, sk.n_ctx - c * CH);
      const bool causal = mode == DFLASH_ATTN_CAUSAL && slot0 >= 0;
      const int lim = causal ? P + row_tok - slot0 : CH;
      if (ok && !tc::mbar_wait(&sfull[b], (uint32_t)(i >> 1) & 1u, abort, lim_ns)) {
        raise_status(status, ST_TIMEOUT);
        *abort = 1;
        ok = false;
      }
      __syncwarp();  // the TMEM load below is warp-collective
      tc::tc_fence_after();
      float sc[KP];
      tmem_ld_scores(lane_base + (uint32_t)(b * CH + KP * piece), sc);
      const float cmax = soft_scores(sc, KP * piece, nk, lim, scale);
      xm[piece * 64 + qr] = cmax;
      tc::named_bar(2, kTcAttnSoft);
      float m_cand = m_run;
#pragma unroll
      for (int pc = 0; pc < kTcAttnPieces; ++pc) m_cand = fmaxf(m_cand, xm[pc * 64 + qr]);
      // The reference maximum moves only when the chunk's maximum exceeds it
      // by more than 8 (log2 units, a factor 256): P then stays below 2^8, and
      // most chunks skip rescaling O in TMEM (alpha = 1 exactly).  O and l
      // are kept against the same reference, so the result is unchanged.
      const float m_new = (m_run == -INFINITY || m_cand > m_run + 8.f) ? m_cand : m_run;
      const float alpha = (m_run == -INFINITY) ? 0.f : exp2f(m_run - m_new);
      xs[piece * 64 + qr] = soft_exp(sc, m_new);
      // P has one buffer: the P V products of the chunk before must have
      // finished reading it (S of this chunk was issued ahead of them).
      if (i > 0 && ok && !tc::mbar_wait(ofull, (uint32_t)(i - 1) & 1u, abort, lim_ns)) {
        raise_status(status, ST_TIMEOUT);
        *abort = 1;
        ok = false;
      }
      // P = P_hi + P_lo: this thread's KP keys of row q, 8 per 16-byte chunk
#pragma unroll
      for (int cc = 0; cc < KP / 8; ++cc) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) split_bf16(sc[8 * cc + 2 * e], sc[8 * cc + 2 * e + 1], hi[e], lo[e]);
        const int ch = (KP / 8) * piece + cc;
        *reinterpret_cast<uint4*>(Ph + op_off(qr, ch)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(Pl + op_off(qr, ch)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
      if (nk < CH) {
        // Rows past the last key hold whatever follows in memory (unwritten
        // cache slots may be NaN); zero V there so that P = 0 contributes 0.
        uint8_t* Vt = KV + (2 * b + 1) * TILE;
        for (int t = sw * 32 + lane; t < (CH - nk) * (D / 8); t += kTcAttnSoft) {
          const int j = nk + t / (D / 8), ch = t % (D / 8);
          *reinterpret_cast<uint4*>(Vt + kv_off(j, ch)) = make_uint4(0, 0, 0, 0);
        }
      }
      tc::named_bar(2, kTcAttnSoft);
      float lsum = 0.f;
#pragma unroll
      for (int pc = 0; pc < kTcAttnPieces; ++pc) lsum += xs[pc * 64 + qr];
      l_run = fmaf(l_run, alpha, lsum);
      // O (lanes 0..63) holds the chunks before this one (their P V products
      // have completed: waited above): rescale this thread's OC columns to the
      // new maximum.  TMEM accesses are warp-collective: the whole warp takes
      // the branch when any of its rows needs it (alpha = 1 keeps a row).
      if (o_owner && li > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        __syncwarp();
        tc::tc_fence_after();
#pragma unroll
        for (int q = 0; q < OC / 16; ++q) {
          float o16[16];
          const uint32_t col = (uint32_t)((i < nA ? 2 : 3) * CH + OC * kg + 16 * q);
          tc::tmem_ld16(lane_base + col, o16);
#pragma unroll
          for (int t = 0; t < 16; ++t) o16[t] *= alpha;
          tc::tmem_st16(lane_base + col, o16);
        }
      }
      m_run = m_new;
      // This thread's P (and V zero) stores and TMEM stores are done: release
      // them to the MMA issuer (pdone counts every softmax thread).
      tc::fence_proxy_async_smem();
      tc::tc_fence_before();
      tc::mbar_arrive(&pdone[b]);
    }
    // ---- this CTA's partial of its 64 rows (lanes 0..63, OC columns per thread)
    if (o_owner && nmine > 0) {
      if (ok && !tc::mbar_wait(ofull, (uint32_t)(nmine - 1) & 1u, abort, lim_ns)) {
        raise_status(status, ST_TIMEOUT);
        *abort = 1;
        ok = false;
      }
    }
    float mB = -INFINITY, lB = 0.f;
    if (nB > 0) {
      mB = m_run;
      lB = l_run;
    } else {
      mA = m_run;
      lA = l_run;
    }
    // psm overlays the K/V buffers: every MMA (the last P V) has completed here
    tc::named_bar(2, kTcAttnSoft);
    if (o_owner) {
      __syncwarp();
      tc::tc_fence_after();
      for (int e = 0; e < E; ++e) {
        float* pr = psm + ((size_t)e * kClQT + qr) * PST;
        const bool any = (e == 0 ? nA : nB) > 0;  // uniform over the CTA
        constexpr int NC_ = OC < 64 ? OC : 64;  // columns per TMEM load
#pragma unroll
        for (int q = 0; q < OC / NC_; ++q) {
          float o64[NC_];
          if (any) {
            tmem_ld_cols(lane_base + (uint32_t)((2 + e) * CH + OC * kg + NC_ * q), o64);
          } else {
#pragma unroll
            for (int t = 0; t < NC_; ++t) o64[t] = 0.f;
          }
#pragma unroll
          for (int t = 0; t < NC_; t += 4)
            *reinterpret_cast<float4*>(pr + OC * kg + NC_ * q + t) = make_float4(o64[t], o64[t + 1], o64[t + 2], o64[t + 3]);
        }
        if (kg == 0) {
          pr[D] = e == 0 ? mA : mB;
          pr[D + 1] = e == 0 ? lA : lB;
        }
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
  cl.sync();  // every rank's chunks are done: its K/V buffers may receive
  // recv follows the E partials (E = 2: 67.6 KB + 76 KB, inside the K/V, Q and P space)
  push_merge<D>(cl, psm, psm + (size_t)E * kClQT * PST, NC, E, rank, nq_tile, qv0, grp, g, s, rows, QD, a.out,
                 status);
}

// ------------------------------------------------ tcgen05 streaming variant
//
// With more (sequence, KV head, query tile) items than clusters fit at once,
// the same function runs as a grid of one CTA per SM without clusters.  The
// work is cut into units, one per (item, logical rank): a unit is that
// rank's chunks of the item under the split of the cluster kernels (NL
// logical ranks, rank r owning chunks r, r + NL, ...), and the units are
// ordered by item, then rank.  CTA b takes the units whose first chunk falls
// in the b-th equal share of all the launch's chunks, so every CTA streams
// about the same number of K/V chunks whatever the context lengths.  A unit
// runs the online softmax of its logical rank from scratch; its partial
// (O, m, l) goes from TMEM to the workspace, and the CTA that completes the
// last unit of an item merges the item's NL partials in rank order with the
// arithmetic of push_merge.  The outputs are therefore bit for bit those of
// the cluster kernels.  The K/V pipeline runs on across unit and item
// boundaries; the query tile is reloaded when the item changes (one buffer:
// the load waits until the item's last S = Q K^T has completed).

// A CTA's units walked chunk by chunk: every role keeps its own copy.
struct UnitCursor {
  const AttnDesc* a;
  int ips, NL;          // items per sequence, logical ranks
  int s, it, r, k;      // sequence, item of the sequence, logical rank, chunk of the rank
  int P, nle, q, rem;   // block position; ranks with chunks; chunks per rank = q + (r < rem)
  SeqKeys sk;
  __device__ __forceinline__ void load() {
    P = a->base_pos[s];
    sk = tc_seq_keys(*a, P);
    nle = min(NL, sk.n_ch);
    q = sk.n_ch / NL;
    rem = sk.n_ch - q * NL;
  }
  __device__ __forceinline__ int cnt() const { return q + (r < rem ? 1 : 0); }
  __device__ __forceinline__ int chunk() const { return r + k * NL; }
  __device__ __forceinline__ bool item_first() const { return k == 0 && r == 0; }
  __device__ __forceinline__ bool item_last() const { return k + 1 == cnt() && r + 1 == nle; }
  __device__ __forceinline__ int item() const { return s * ips + it; }
  __device__ __forceinline__ void next() {
    if (++k < cnt()) return;
    k = 0;
    if (++r < nle) return;
    r = 0;
    if (++it < ips) return;
    it = 0;
    if (++s < a->n_seqs) load();
  }
};

// Chunks of sequence s over all its items.
__device__ __forceinline__ long long seq_units_chunks(const AttnDesc& a, int s, int ips) {
  return (long long)tc_seq_keys(a, a.base_pos[s]).n_ch * ips;
}

// The first unit whose first chunk is at or after chunk x of the launch's
// chunk order: (s, it, r) and its first chunk t; s = n_seqs when there is
// none (t is then the total).  Run by a whole warp, the same result in every
// lane.
__device__ void find_unit(const AttnDesc& a, int ips, int NL, long long x, int lane, int& s_out, int& it_out,
                          int& r_out, long long& t_out) {
  long long cum = 0;  // chunks of the sequences before s0
  for (int s0 = 0; s0 < a.n_seqs; s0 += 32) {
    const int sl = s0 + lane;
    const long long v = sl < a.n_seqs ? seq_units_chunks(a, sl, ips) : 0;
    long long incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, sl < a.n_seqs && cum + incl > x);
    if (hit) {
      const int l = __ffs(hit) - 1;
      const long long base = cum + __shfl_sync(0xffffffffu, incl - v, l);  // first chunk of sequence s
      const int s = s0 + l;
      const int n_ch = tc_seq_keys(a, a.base_pos[s]).n_ch;
      const long long off = x - base;  // 0 <= off < n_ch * ips
      int it = (int)(off / n_ch);
      const int o2 = (int)(off - (long long)it * n_ch);
      const int q = n_ch / NL, rem = n_ch - q * NL, nle = min(NL, n_ch);
      int r = 0;
      while (r < nle && r * q + min(r, rem) < o2) ++r;
      if (r < nle) {
        s_out = s;
        it_out = it;
        r_out = r;
        t_out = base + (long long)it * n_ch + r * q + min(r, rem);
      } else if (it + 1 < ips) {  // the next item's first unit
        s_out = s;
        it_out = it + 1;
        r_out = 0;
        t_out = base + (long long)(it + 1) * n_ch;
      } else {  // the next sequence's first unit (or none)
        s_out = s + 1;
        it_out = 0;
        r_out = 0;
        t_out = base + (long long)ips * n_ch;
      }
      return;
    }
    cum += __shfl_sync(0xffffffffu, incl, 31);
  }
  s_out = a.n_seqs;
  it_out = 0;
  r_out = 0;
  t_out = cum;
}

// Threads of the streaming kernel: warp 0 loads K (and the query tiles),
// warp 1 issues the MMAs, the softmax warps follow, and the last warp loads V.
constexpr int kTcStreamThreads = kTcAttnThreads + 32;
// One unit's partial (head dim 128): four blocks of 16 query rows, each
// O [32 column quads][16 rows][4] then m[16], l[16] -- 8320 contiguous bytes,
// one bulk copy in the merge.
constexpr int kRbRows = 16;
constexpr int kRbFloats = (128 + 2) * kRbRows;
constexpr int kRbBytes = kRbFloats * 4;
constexpr int kPartFloats = kRbFloats * (kClQT / kRbRows);
constexpr int kTcStreamVWarp = kTcAttnThreads / 32;

template <int D>
__global__ void __launch_bounds__(kTcStreamThreads, 1) attn_tc_stream_kernel(const __grid_constant__ AttnTma p,
                                                                             int n_qt, int NL) {
  static_assert(D == 128, "two 64-dim boxes per row");
  constexpr int CH = kMmaCH;
  constexpr int TILE = CH * D * 2;
  constexpr int KP = kTcAttnKP;
  constexpr int OC = D / kTcAttnGroups;  // output columns per owner thread
  static_assert(CH == 128 && OC % 16 == 0, "whole 16-column TMEM loads");
  static_assert((D + 2) * kClQT == kPartFloats, "partial size");
  static_assert(kRbBytes % 16 == 0, "bulk copies of whole 16-byte units");
  extern __shared__ __align__(1024) uint8_t smem_att[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_att) + 1023) & ~uintptr_t(1023));
  uint8_t* KV = sm;  // slot b: K at KV + 2*b*TILE, V at KV + (2*b+1)*TILE
  uint8_t* Qs = KV + 4 * TILE;
  uint8_t* Ph = Qs + kTcAttnRows * D * 2;
  uint8_t* Pl = Ph + kTcAttnPloOff;
  uint64_t* kfull = reinterpret_cast<uint64_t*>(Ph + kTcAttnPBytes);  // [2] K of a chunk landed
  uint64_t* vfull = kfull + 2;                            // [2] V of a chunk landed
  uint64_t* kempty = vfull + 2;                           // [2] S = Q K^T done: the K slot is free
  uint64_t* vempty = kempty + 2;                          // [2] P V done: the V slot is free
  uint64_t* sfull = vempty + 2;                           // [2] S in TMEM
  uint64_t* pdone = sfull + 2;                            // [2] P written, O rescaled
  uint64_t* ofull = pdone + 2;                            // P V done
  uint64_t* qfull = ofull + 1;                            // query tile landed
  uint64_t* qempty = qfull + 1;                           // the item's last S done: Q may be replaced
  uint32_t* tslot = reinterpret_cast<uint32_t*>(qempty + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tslot + 1);
  int* sched = const_cast<int*>(abort) + 1;  // [4] first unit (s, it, r), chunk count; [4] last-arriver flag
  // [2 chunk parities][pieces][64 rows] each
  float* xmax = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(kfull) + 160);
  float* xsum = xmax + 2 * kTcAttnPieces * 64;

  const AttnDesc& a = p.a;
  const int ips = a.nkv * n_qt;
  const int mode = a.mode, rows = a.rows;
  const int grp = a.nq / a.nkv;
  const int nqv = rows * grp;
  const int QD = a.nq * D;
  uint32_t* status = a.status;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint64_t lim_ns = wait_limit_ns(status);
  const bool stall = stall_kv_loads(status);  // test switch: issue no K/V copy
  const KvMap km{a.pages, a.cap, a.ps, a.max_pages, a.pool, a.nkv};
  float* part = a.partials;  // [items][NL][kPartFloats]

  // ---- this CTA's units (base_pos is not written by the kernel before this
  // one inside a call, so it may be read before the PDL wait)
  if (warp == 0) {
    long long T = 0;
    for (int s0 = 0; s0 < a.n_seqs; s0 += 32) {
      long long v = s0 + lane < a.n_seqs ? seq_units_chunks(a, s0 + lane, ips) : 0;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      T += v;
    }
    const long long lo = (long long)blockIdx.x * T / gridDim.x, hi = (long long)(blockIdx.x + 1) * T / gridDim.x;
    int s0, it0, r0, s1, it1, r1;
    long long t0, t1;
    find_unit(a, ips, NL, lo, lane, s0, it0, r0, t0);
    find_unit(a, ips, NL, hi, lane, s1, it1, r1, t1);
    if (lane == 0) {
      sched[0] = s0;
      sched[1] = it0;
      sched[2] = r0;
      sched[3] = (int)(t1 - t0);
    }
  }
  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&kfull[b], 1);
      tc::mbar_init(&vfull[b], 1);
      tc::mbar_init(&kempty[b], 1);
      tc::mbar_init(&vempty[b], 1);
      tc::mbar_init(&sfull[b], 1);
      tc::mbar_init(&pdone[b], kTcAttnSoft);
    }
    tc::mbar_init(ofull, 1);
    tc::mbar_init(qfull, 1);
    tc::mbar_init(qempty, 1);
    *abort = 0;
    tc::fence_mbar_init();
    tc::tma_prefetch_desc(&p.kc);
    tc::tma_prefetch_desc(&p.vc);
    tc::tma_prefetch_desc(&p.q3);
  }
  if (warp == 1) tc::tmem_alloc(tslot, 512);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tslot;
  const int nmine = sched[3];
  UnitCursor start;
  start.a = &a;
  start.ips = ips;
  start.NL = NL;
  start.s = sched[0];
  start.it = sched[1];
  start.r = sched[2];
  start.k = 0;
  if (nmine > 0) start.load();

  auto chunk_row = [&](const UnitCursor& u, bool& blk) -> int {
    const int c = u.chunk(), g = u.it / n_qt;
    blk = (mode == DFLASH_ATTN_BLOCK_BIDIR && c == u.sk.n_ctx_ch);
    if (blk) return (u.s * a.nkv + g) * rows;
    bool bad = false;
    const int r = (int)(km.row0(u.s, c * CH, &bad) + (uint32_t)g * (uint32_t)km.head_rows());
    if (bad) raise_status(status, ST_RANGE);  // read from page 0 instead
    return r;
  };
  // One operand tile (K: v = 0, V: v = 1) of chunk u into slot buf; one thread.
  auto issue = [&](const UnitCursor& u, int buf, int v) -> bool {
    if (stall) return false;
    bool blk;
    const int row = chunk_row(u, blk);
    const CUtensorMap* map = v ? (blk ? &p.vb : &p.vc) : (blk ? &p.kb : &p.kc);
    uint64_t* bar = v ? &vfull[buf] : &kfull[buf];
    uint8_t* dst = KV + (2 * buf + v) * TILE;
    tc::mbar_arrive_expect_tx(bar, TILE);
    const uint64_t pol = tc::policy_evict_first();
#pragma unroll
    for (int h = 0; h < D / 64; ++h) tc::tma_load_2d(dst + h * (CH * 128), map, 64 * h, row, bar, pol);
    return true;
  };
  auto early_ok = [&](const UnitCursor& u) {
    const int c = u.chunk();
    return c < u.sk.n_ctx_ch && (mode == DFLASH_ATTN_BLOCK_BIDIR || (c + 1) * CH <= u.P);
  };
  // Context chunks that the kernel before this one does not write may load
  // before the PDL wait: K by thread 0, V by the V loader.
  const bool loader = (warp == 0 || warp == kTcStreamVWarp) && lane == 0;
  const int vsel = warp == kTcStreamVWarp ? 1 : 0;
  bool pre0 = false, pre1 = false;
  if (loader && nmine > 0) {
    if (early_ok(start)) pre0 = issue(start, 0, vsel);
    if (nmine > 1) {
      UnitCursor u1 = start;
      u1.next();
      if (early_ok(u1)) pre1 = issue(u1, 1, vsel);
    }
  }
  pdl_wait();
  pdl_launch_dependents();

  const uint32_t kvb = __cvta_generic_to_shared(KV);
  const uint32_t qb = __cvta_generic_to_shared(Qs);
  const uint32_t phb = __cvta_generic_to_shared(Ph), plb = __cvta_generic_to_shared(Pl);
  if (loader) {
    // ---------------- loaders: chunk i's K (V) into slot i & 1 once S (P V)
    // of chunk i-2 is done; the K loader also loads each new item's query tile
    uint64_t* fullb = vsel ? vfull : kfull;
    uint64_t* emptyb = vsel ? vempty : kempty;
    UnitCursor u = start;
    int issued = 0, nq = 0;
    bool ok = true;
    for (int i = 0; i < nmine && ok; ++i, u.next()) {
      if (!vsel && (i == 0 || u.item_first())) {
        if (nq > 0 && !tc::mbar_wait(qempty, (uint32_t)(nq - 1) & 1u, abort, lim_ns)) {
          ok = false;
          break;
        }
        tc::mbar_arrive_expect_tx(qfull, 4 * kClQT * 128);
        const int g = u.it / n_qt, qt = u.it % n_qt;
        const int z = u.s * rows + (qt * kClQT) / grp, y = g * grp;
#pragma unroll
        for (int h = 0; h < D / 64; ++h)
#pragma unroll
          for (int dup = 0; dup < 2; ++dup)
            tc::tma_load_3d(Qs + h * (kTcAttnRows * 128) + dup * (kClQT * 128), &p.q3, 64 * h, y, z, qfull);
        ++nq;
      }
      if (i < 2 && (i == 0 ? pre0 : pre1)) {
        ++issued;
        continue;
      }
      if (i >= 2 && !tc::mbar_wait(&emptyb[i & 1], (uint32_t)((i - 2) >> 1) & 1u, abort, lim_ns)) {
        ok = false;
        break;
      }
      if (issue(u, i & 1, vsel)) ++issued;
    }
    if (!ok) {
      raise_status(status, ST_TIMEOUT);
      *abort = 1;
    }
    // Every copy this thread issued has landed before the CTA's shared memory
    // goes away, also when a wait gave up (the last copy into each slot).
    for (int i = issued > 2 ? issued - 2 : 0; i < issued; ++i)
      tc::mbar_wait(&fullb[i & 1], (uint32_t)(i >> 1) & 1u, nullptr, lim_ns);
    if (nq > 0) tc::mbar_wait(qfull, (uint32_t)(nq - 1) & 1u, nullptr, lim_ns);
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      constexpr uint32_t idS = tc::idesc_bf16_f32(kTcAttnRows, CH);
      constexpr uint32_t idV = tc::idesc_bf16_f32_bmn(kTcAttnRows, D);
      bool ok = true;
      auto wait = [&](uint64_t* bar, uint32_t par) {
        if (ok && !tc::mbar_wait(bar, par, abort, lim_ns)) {
          raise_status(status, ST_TIMEOUT);
          *abort = 1;
          ok = false;
        }
        return ok;
      };
      UnitCursor us = start;  // next chunk whose S is issued
      int nqs = 0;
      auto issue_s = [&](int i) {
        const int b = i & 1;
        if ((i == 0 || us.item_first()) && !wait(qfull, (uint32_t)(nqs++) & 1u)) return;
        if (!wait(&kfull[b], (uint32_t)(i >> 1) & 1u)) return;
        tc::tc_fence_after();
        const uint32_t kb = kvb + 2 * b * TILE;
#pragma unroll
        for (int j = 0; j < D / 16; ++j) {
          const uint32_t off = (uint32_t)((j >> 2) * (kTcAttnRows * 128) + (j & 3) * 32);
          const uint32_t koff = (uint32_t)((j >> 2) * (CH * 128) + (j & 3) * 32);
          tc::mma_bf16(tmem + (uint32_t)(b * CH), tc::sdesc_sw128(qb + off), tc::sdesc_sw128(kb + koff), idS,
                       j > 0 ? 1u : 0u);
        }
        tc::mma_commit(&sfull[b]);
        tc::mma_commit(&kempty[b]);
        if (i + 1 < nmine && us.item_last()) tc::mma_commit(qempty);  // the next chunk starts another item
        us.next();
      };
      UnitCursor uv = start;  // chunk whose P V is issued
      int unit = 0;           // this CTA's unit of that chunk: output accumulator 2 + (unit & 1)
      // S of chunk i+2 right after P V of chunk i: its K slot frees only when
      // it completes, so deferring it would slow the K ring.
      if (nmine > 0) issue_s(0);
      if (nmine > 1) issue_s(1);
      for (int i = 0; i < nmine && ok; ++i, uv.next()) {
        if (i > 0 && uv.k == 0) ++unit;
        if (!wait(&pdone[i & 1], (uint32_t)(i >> 1) & 1u)) break;
        if (!wait(&vfull[i & 1], (uint32_t)(i >> 1) & 1u)) break;
        tc::tc_fence_after();
        const uint32_t vb = kvb + (2 * (i & 1) + 1) * TILE;
        const uint32_t od = tmem + (uint32_t)((2 + (unit & 1)) * CH);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const uint32_t pb = half ? plb : phb;
#pragma unroll
          for (int j = 0; j < CH / 16; ++j) {
            const uint32_t poff = (uint32_t)((j >> 2) * (kTcAttnRows * 128) + (j & 3) * 32);
            tc::mma_bf16(od, tc::sdesc_sw128(pb + poff),
                         tc::sdesc_sw128_mn(vb + (uint32_t)j * 2048u, CH * 128, 1024), idV,
                         (uv.k > 0 || half > 0 || j > 0) ? 1u : 0u);
          }
        }
        tc::mma_commit(&vempty[i & 1]);
        tc::mma_commit(ofull);
        if (i + 2 < nmine) issue_s(i + 2);
      }
    }
  } else if (warp >= 2 && warp < kTcStreamVWarp) {
    // ---------------- softmax warps: the thread roles of attn_tc_kernel
    const int sw = warp - 2;
    const int L = (warp & 3) * 32 + lane;
    const int qr = L & (kClQT - 1), h = L >> 6;
    const int kg = sw >> 2, piece = 2 * kg + h;
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const bool o_owner = h == 0;  // lanes 0..63 hold the output rows; this thread takes columns OC kg ..
    const float scale = rsqrtf((float)D) * kLog2e;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    // Unit u is complete (its last P V has finished; its output accumulator
    // is ob): O from TMEM, m and l to its partial (a warp's 32 rows store
    // two 256-byte runs per instruction).
    auto flush = [&](const UnitCursor& u, int ob, float m_fin, float l_fin) {
      if (o_owner) {
        float* pb = part + (size_t)(u.item() * NL + u.r) * kPartFloats + (qr / kRbRows) * kRbFloats;
        const int ri = qr % kRbRows;
        const uint64_t keep = tc::policy_evict_last();  // read back by the merge: keep in L2
        __syncwarp();
        tc::tc_fence_after();
        constexpr int NC_ = OC < 64 ? OC : 64;  // columns per TMEM load
#pragma unroll
        for (int q = 0; q < OC / NC_; ++q) {
          float o64[NC_];
          tmem_ld_cols(lane_base + (uint32_t)(ob * CH + OC * kg + NC_ * q), o64);
#pragma unroll
          for (int t = 0; t < NC_; t += 4) {
            const int quad = (OC * kg + NC_ * q + t) / 4;
            tc::st_global_hint(pb + (quad * kRbRows + ri) * 4, make_float4(o64[t], o64[t + 1], o64[t + 2], o64[t + 3]),
                               keep);
          }
        }
        if (kg == 0) {
          tc::st_global_hint(pb + D * kRbRows + ri, m_fin, keep);
          tc::st_global_hint(pb + D * kRbRows + kRbRows + ri, l_fin, keep);
        }
      }
    };
    UnitCursor u = start, prev = start;
    int unit = 0;
    float m_fin = -INFINITY, l_fin = 0.f;
    for (int i = 0; i < nmine; ++i) {
      const int c = u.chunk(), b = i & 1;
      const int li = u.k;
      if (li == 0 && i > 0) {  // a new logical rank starts from scratch
        m_fin = m_run;
        l_fin = l_run;
        m_run = -INFINITY;
        l_run = 0.f;
        ++unit;
      }
      const uint32_t ocol = (uint32_t)((2 + (unit & 1)) * CH);  // this unit's output accumulator
      const int qv0 = (u.it % n_qt) * kClQT;
      const int row_tok = (qv0 + qr) / grp;
      float* xm = xmax + b * (kTcAttnPieces * 64);
      float* xs = xsum + b * (kTcAttnPieces * 64);
      bool blk;
      chunk_row(u, blk);
      const int slot0 = blk ? -1 : c * CH;
      const int nk = blk ? min(rows, CH) : min(CH, u.sk.n_ctx - c * CH);
      const bool causal = mode == DFLASH_ATTN_CAUSAL && slot0 >= 0;
      const int lim = causal ? u.P + row_tok - slot0 : CH;
      if (ok && !tc::mbar_wait(&sfull[b], (uint32_t)(i >> 1) & 1u, abort, lim_ns)) {
        raise_status(status, ST_TIMEOUT);
        *abort = 1;
        ok = false;
      }
      __syncwarp();  // the TMEM load below is warp-collective
      tc::tc_fence_after();
      float sc[KP];
      tmem_ld_scores(lane_base + (uint32_t)(b * CH + KP * piece), sc);
      const float cmax = soft_scores(sc, KP * piece, nk, lim, scale);
      xm[piece * 64 + qr] = cmax;
      tc::named_bar(2, kTcAttnSoft);
      float m_cand = m_run;
#pragma unroll
      for (int pc = 0; pc < kTcAttnPieces; ++pc) m_cand = fmaxf(m_cand, xm[pc * 64 + qr]);
      // the reference maximum moves only by more than 8 (attn_tc_kernel)
      const float m_new = (m_run == -INFINITY || m_cand > m_run + 8.f) ? m_cand : m_run;
      const float alpha = (m_run == -INFINITY) ? 0.f : exp2f(m_run - m_new);
      xs[piece * 64 + qr] = soft_exp(sc, m_new);
      // P has one buffer: the P V products of the chunk before must have
      // finished reading it (and, for the unit before, writing its output).
      if (i > 0 && ok && !tc::mbar_wait(ofull, (uint32_t)(i - 1) & 1u, abort, lim_ns)) {
        raise_status(status, ST_TIMEOUT);
        *abort = 1;
        ok = false;
      }
#pragma unroll
      for (int cc = 0; cc < KP / 8; ++cc) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) split_bf16(sc[8 * cc + 2 * e], sc[8 * cc + 2 * e + 1], hi[e], lo[e]);
        const int ch = (KP / 8) * piece + cc;
        *reinterpret_cast<uint4*>(Ph + op_off(qr, ch)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(Pl + op_off(qr, ch)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
      if (nk < CH) {
        // rows past the last key: zero V (once it has landed) so that P = 0
        // contributes 0
        if (ok && !stall && !tc::mbar_wait(&vfull[b], (uint32_t)(i >> 1) & 1u, abort, lim_ns)) {
          raise_status(status, ST_TIMEOUT);
          *abort = 1;
          ok = false;
        }
        uint8_t* Vt = KV + (2 * b + 1) * TILE;
        for (int t = sw * 32 + lane; t < (CH - nk) * (D / 8); t += kTcAttnSoft) {
          const int j = nk + t / (D / 8), ch = t % (D / 8);
          *reinterpret_cast<uint4*>(Vt + kv_off(j, ch)) = make_uint4(0, 0, 0, 0);
        }
      }
      tc::named_bar(2, kTcAttnSoft);
      float lsum = 0.f;
#pragma unroll
      for (int pc = 0; pc < kTcAttnPieces; ++pc) lsum += xs[pc * 64 + qr];
      l_run = fmaf(l_run, alpha, lsum);
      if (o_owner && li > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        __syncwarp();
        tc::tc_fence_after();
#pragma unroll
        for (int q = 0; q < OC / 16; ++q) {
          float o16[16];
          const uint32_t col = ocol + (uint32_t)(OC * kg + 16 * q);
          tc::tmem_ld16(lane_base + col, o16);
#pragma unroll
          for (int t = 0; t < 16; ++t) o16[t] *= alpha;
          tc::tmem_st16(lane_base + col, o16);
        }
      }
      m_run = m_new;
      tc::fence_proxy_async_smem();
      tc::tc_fence_before();
      tc::mbar_arrive(&pdone[b]);
      // The unit before this one finished with chunk i-1 (its P V completed:
      // waited above) in the other accumulator, which the MMAs of this unit
      // do not touch: write it out while P V of chunk i runs.
      if (i > 0 && li == 0) flush(prev, 2 + ((unit - 1) & 1), m_fin, l_fin);
      prev = u;
      u.next();
    }
    if (nmine > 0) {
      if (ok && !tc::mbar_wait(ofull, (uint32_t)(nmine - 1) & 1u, abort, lim_ns)) {
        raise_status(status, ST_TIMEOUT);
        *abort = 1;
        ok = false;
      }
      flush(prev, 2 + (unit & 1), m_run, l_run);
      if (o_owner) __threadfence();  // this thread's partial rows, before the grid barrier
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 512);
  }

  // ---- every CTA's partials are written (grid barrier: the grid is one CTA
  // per SM, all resident); then the merges, split evenly over the CTAs in
  // tasks of (item, 16-row block): the NL partial blocks of a task arrive by
  // bulk copy, double-buffered when two tasks' blocks fit.
  if (threadIdx.x == 0) {
    uint32_t* ctr = a.counters + kCtrAttnGrid;
    volatile uint32_t* gen = ctr + 1;
    const uint32_t g0 = *gen;
    __threadfence();
    if (atomicAdd(ctr, 1u) == gridDim.x - 1) {
      *ctr = 0u;  // every CTA has arrived: ready for the next launch
      __threadfence();
      atomicAdd(ctr + 1, 1u);
    } else {
      const uint64_t t0 = global_ns();
      while (*gen == g0) {
        if (global_ns() - t0 > lim_ns) {
          raise_status(status, ST_TIMEOUT);
          break;
        }
        __nanosleep(64);
      }
    }
    __threadfence();
    // the K barriers are idle (every K copy has landed): they now count the merge copies
    tc::mbar_init(&kfull[0], 1);
    tc::mbar_init(&kfull[1], 1);
    tc::fence_mbar_init();
  }
  __syncthreads();
  constexpr int kMergeSmem = 4 * TILE + kTcAttnRows * D * 2 + kTcAttnPBytes;  // K/V, Q and P space
  static_assert((kRbRows * kMaxNC + kRbRows) * 4 <= 2 * 2 * kTcAttnPieces * 64 * 4, "weights fit the exchange space");
  const int NB = 2 * NL * kRbBytes + kRbRows * D * 2 <= kMergeSmem ? 2 : 1;
  __nv_bfloat16* Ob = reinterpret_cast<__nv_bfloat16*>(sm + (size_t)NB * NL * kRbBytes);  // [16][D] output rows
  float* W = xmax;                   // [16][kMaxNC] rank weights (the softmax exchange space)
  float* Ls = W + kRbRows * kMaxNC;  // [16] denominators
  __nv_bfloat16* outp = reinterpret_cast<__nv_bfloat16*>(a.out);
  const int n_tasks = a.n_seqs * ips * (kClQT / kRbRows);
  auto task_geom = [&](int task, int& item, int& rb, int& nle, int& nrow) {
    item = task / (kClQT / kRbRows);
    rb = task % (kClQT / kRbRows);
    const int s = item / ips, it = item % ips;
    nle = min(NL, tc_seq_keys(a, a.base_pos[s]).n_ch);
    nrow = min(kRbRows, nqv - (it % n_qt) * kClQT - rb * kRbRows);
  };
  auto issue_task = [&](int task, int buf) {  // one thread
    int item, rb, nle, nrow;
    task_geom(task, item, rb, nle, nrow);
    if (nrow <= 0) {
      tc::mbar_arrive(&kfull[buf]);
      return;
    }
    tc::mbar_arrive_expect_tx(&kfull[buf], (uint32_t)(nle * kRbBytes));
    const uint64_t drop = tc::policy_evict_first();  // read once
    for (int r = 0; r < nle; ++r)
      tc::bulk_load_hint(sm + (size_t)(buf * NL + r) * kRbBytes,
                         part + ((size_t)item * NL + r) * kPartFloats + (size_t)rb * kRbFloats, kRbBytes, &kfull[buf],
                         drop);
  };
  if (threadIdx.x == 0 && (int)blockIdx.x < n_tasks) issue_task(blockIdx.x, 0);
  int k = 0;
  for (int task = blockIdx.x; task < n_tasks; task += gridDim.x, ++k) {
    const int buf = NB == 2 ? (k & 1) : 0;
    const uint32_t par = (uint32_t)(NB == 2 ? (k >> 1) : k) & 1u;
    if (NB == 2 && threadIdx.x == 0 && task + (int)gridDim.x < n_tasks) issue_task(task + gridDim.x, buf ^ 1);
    int item, rb, nle, nrow;
    task_geom(task, item, rb, nle, nrow);
    if (!tc::mbar_wait(&kfull[buf], par, nullptr, lim_ns)) raise_status(status, ST_TIMEOUT);
    const float* B = reinterpret_cast<const float*>(sm + (size_t)buf * NL * kRbBytes);
    // the rank weights of each query row (the arithmetic of push_merge)
    if ((int)threadIdx.x < nrow) {
      const int i = threadIdx.x;
      float mr[kMaxNC], lr[kMaxNC];
#pragma unroll
      for (int r = 0; r < kMaxNC; ++r) {
        mr[r] = r < nle ? B[(size_t)r * kRbFloats + D * kRbRows + i] : -INFINITY;
        lr[r] = r < nle ? B[(size_t)r * kRbFloats + D * kRbRows + kRbRows + i] : 0.f;
      }
      float M = -INFINITY;
#pragma unroll
      for (int r = 0; r < kMaxNC; ++r)
        if (r < NL) M = fmaxf(M, mr[r]);
      float Lr = 0.f;
#pragma unroll
      for (int r = 0; r < kMaxNC; ++r) {
        if (r < NL) {
          const float w = (mr[r] == -INFINITY) ? 0.f : exp2f(mr[r] - M);
          W[i * kMaxNC + r] = w;
          Lr = fmaf(lr[r], w, Lr);
        }
      }
      Ls[i] = Lr;
    }
    __syncthreads();
    // the weighted sums: consecutive threads take consecutive rows of a quad
    for (int t = threadIdx.x; t < kRbRows * (D / 4); t += blockDim.x) {
      const int i = t % kRbRows, quad = t / kRbRows;
      if (i >= nrow) continue;
      float o[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int r = 0; r < kMaxNC; ++r) {
        if (r < NL) {
          const float4 v = r < nle ? *reinterpret_cast<const float4*>(B + (size_t)r * kRbFloats + (quad * kRbRows + i) * 4)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
          const float w = W[i * kMaxNC + r];
          o[0] = fmaf(v.x, w, o[0]);
          o[1] = fmaf(v.y, w, o[1]);
          o[2] = fmaf(v.z, w, o[2]);
          o[3] = fmaf(v.w, w, o[3]);
        }
      }
      store_quad(Ob + i * D + 4 * quad, o, Ls[i]);
    }
    __syncthreads();
    // the block's rows to the output, 16 bytes per thread
    const int s = item / ips, it = item % ips;
    const int g = it / n_qt, qv_b = (it % n_qt) * kClQT + rb * kRbRows;
    for (int t = threadIdx.x; t < nrow * (D / 8); t += blockDim.x) {
      const int i = t / (D / 8), c8 = 8 * (t % (D / 8));
      const int qv = qv_b + i;
      const int row = qv / grp, head = g * grp + qv % grp;
      if (!DFL_CHECK(row < rows && head * D + c8 + 8 <= QD, status)) continue;
      *reinterpret_cast<uint4*>(outp + ((size_t)s * rows + row) * QD + (size_t)head * D + c8) =
          *reinterpret_cast<const uint4*>(Ob + i * D + c8);
    }
    __syncthreads();
    if (NB == 1 && threadIdx.x == 0 && task + (int)gridDim.x < n_tasks) issue_task(task + gridDim.x, 0);
  }
}

// ------------------------------------------------------------------- host

namespace {

size_t cluster_smem(int d) {
  const size_t kv = 4 * (size_t)kMmaCH * d * 2, q = (size_t)kClQT * d * 2;
  const size_t parts = 4 * (size_t)kClQT * (d + 4) * sizeof(float);
  return (kv + q > parts ? kv + q : parts) + 64 + 1024;
}

template <int D>
cudaLaunchConfig_t cluster_cfg(int nc, dim3 grid, cudaStream_t st, cudaLaunchAttribute* at) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kClusterWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = cluster_smem(D);
  cfg.stream = st;
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = nc;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  return cfg;
}

// How many clusters of width nc this device runs at once (cached per device).
template <int D>
int clusters_resident(int nc) {
  static std::mutex mu;
  static int cache[64][kMaxNC + 1];
  static bool init[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (!init[dev]) {
    auto k = attn_cluster_kernel<D>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)cluster_smem(D));
    cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    for (int w = 1; w <= kMaxNC; ++w) {
      cudaLaunchAttribute at[2];
      cudaLaunchConfig_t cfg = cluster_cfg<D>(w, dim3(w, 1, 1), nullptr, at);
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess) n = 0;
      cache[dev][w] = n;
    }
    cudaGetLastError();
    init[dev] = true;
  }
  return cache[dev][nc];
}

// Cluster width: the widest (<= 16) for which the clusters of one sequence
// (one per KV head) all run at once, at least 8.  It depends on the KV-head
// count and the device only -- never on the row or sequence count -- so a
// token row's attention is computed the same way whatever else is in the
// launch (decode and verification, one sequence or a batch).
template <int D>
int pick_nc(long groups) {
  for (int nc = kMaxNC; nc > 8; --nc)
    if (clusters_resident<D>(nc) >= groups) return nc;
  return 8;
}

// Tensor maps of the context cache and (bidirectional mode) the block K/V:
// [rows][D] bf16, boxes of 64 dims x 128 keys, 128-byte swizzle.
template <int D>
bool attn_maps(const AttnDesc& a, AttnTma& p) {
  memset(&p, 0, sizeof(p));
  p.a = a;
  const uint64_t crow = a.pages ? (uint64_t)a.pool * a.nkv * a.ps : (uint64_t)a.n_seqs * a.nkv * a.cap;
  if (!make_tmap_bf16(&p.kc, a.kc, D, crow, kMmaCH) || !make_tmap_bf16(&p.vc, a.vc, D, crow, kMmaCH)) return false;
  const int grp = a.nq / a.nkv;
  p.q_tma = 0;
  if (D == 128 && grp <= 64 && kClQT % grp == 0)
    p.q_tma = make_tmap3_bf16(&p.q3, a.q, D, a.nq, (uint64_t)a.n_seqs * a.rows, grp, kClQT / grp) ? 1 : 0;
  if (a.mode == DFLASH_ATTN_BLOCK_BIDIR) {
    const uint64_t brow = (uint64_t)a.n_seqs * a.nkv * a.rows;
    if (!make_tmap_bf16(&p.kb, a.kb, D, brow, kMmaCH) || !make_tmap_bf16(&p.vb, a.vb, D, brow, kMmaCH)) return false;
  } else {
    p.kb = p.kc;
    p.vb = p.vc;
  }
  return true;
}

template <int D>
cudaError_t launch_cluster(const AttnDesc& a, int n_qt, cudaStream_t st) {
  auto k = attn_cluster_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)cluster_smem(D));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  AttnTma p;
  if (!attn_maps<D>(a, p)) return cudaErrorInvalidValue;
  const int nc = pick_nc<D>((long)a.nkv);
  cudaLaunchAttribute at[2];
  cudaLaunchConfig_t cfg = cluster_cfg<D>(nc, dim3(nc, a.nkv * n_qt, a.n_seqs), st, at);
  trace_kernel();
  return cudaLaunchKernelEx(&cfg, k, p, n_qt);
}

// The tcgen05 variant: the number of logical ranks comes from the same
// residency query (both kernels hold one CTA per SM), so it too depends on
// the KV-head count and the device only.  When there are more (sequence, KV
// head, query tile) items than clusters of that width fit at once, the
// items run on clusters of half the width, each CTA taking two logical
// ranks: the chunk split and the merge order are those of the full width,
// so every output is the same bit for bit, and the narrower clusters pack
// the GPCs more fully.
template <int D, int E>
cudaError_t launch_tc_e(const AttnTma& p, int nc, int n_qt, cudaStream_t st) {
  auto k = attn_tc_kernel<D, E>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tc_attn_smem(D));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  const AttnDesc& a = p.a;
  cudaLaunchAttribute at[2];
  cudaLaunchConfig_t cfg = cluster_cfg<D>(nc, dim3(nc, a.nkv * n_qt, a.n_seqs), st, at);
  cfg.blockDim = dim3(kTcAttnThreads, 1, 1);
  cfg.dynamicSmemBytes = tc_attn_smem(D);
  trace_kernel();
  return cudaLaunchKernelEx(&cfg, k, p, n_qt);
}

// The streaming variant: one CTA per SM, the NL logical ranks of the
// cluster kernels as units (NL from the same residency query).
template <int D>
cudaError_t launch_tc_stream(const AttnTma& p, int nl, int n_qt, cudaStream_t st) {
  auto k = attn_tc_stream_kernel<D>;
  const size_t smem = tc_attn_smem(D) + 64;  // 32 more bytes of barriers and schedule than attn_tc_kernel
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sms, 1, 1);
  cfg.blockDim = dim3(kTcStreamThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  trace_kernel();
  return cudaLaunchKernelEx(&cfg, k, p, n_qt, nl);
}

// DFLASH_ATTN_STREAM in the environment (read at every launch): "0" never
// runs the streaming variant, "1" runs it whenever it applies; unset, it runs
// when there are more items than clusters of the logical width fit at once.
// All choices compute the same outputs bit for bit.
static int stream_override() {
  const char* v = getenv("DFLASH_ATTN_STREAM");
  if (v == nullptr || v[0] == 0) return -1;
  return v[0] == '1' ? 1 : 0;
}

template <int D>
cudaError_t launch_tc(const AttnDesc& a, int n_qt, cudaStream_t st) {
  AttnTma p;
  if (!attn_maps<D>(a, p)) return cudaErrorInvalidValue;
  const int nl = pick_nc<D>((long)a.nkv);
  const long items = (long)a.nkv * n_qt * a.n_seqs;
  const int force = stream_override();
  if (p.q_tma && a.partials && a.counters && nl <= kMaxNC && force != 0 &&
      (force == 1 || items > clusters_resident<D>(nl)))
    return launch_tc_stream<D>(p, nl, n_qt, st);
  if (nl % 2 == 0 && items > clusters_resident<D>(nl) && clusters_resident<D>(nl / 2) > clusters_resident<D>(nl))
    return launch_tc_e<D, 2>(p, nl / 2, n_qt, st);
  return launch_tc_e<D, 1>(p, nl, n_qt, st);
}

}  // namespace

size_t attn_workspace(const AttnDesc& a) {
  AttnGeom g = attn_geom(a);
  if (a.dtype == DFLASH_BF16) {
    // the streaming variant's partials, [items][NL <= kMaxNC][64][d + 4]
    // (the cluster kernels merge on chip)
    if (a.d != 128) return 0;
    return (size_t)a.n_seqs * a.nkv * g.n_qt * kMaxNC * kClQT * (a.d + 4) * sizeof(float);
  }
  return (size_t)a.n_seqs * a.nkv * g.n_qt * g.nch * kAttnQT * (a.d + 2) * sizeof(float);
}

// Head dimension 128 runs the tcgen05 kernel unless DFLASH_ATTN_MMASYNC=1 is
// set in the environment (read once per process); both compute the same
// function, and the tcgen05 one measured faster in the whole cycle.
static bool use_tc_attention() {
  static const bool on = [] {
    const char* v = getenv("DFLASH_ATTN_MMASYNC");
    return !(v != nullptr && v[0] == '1');
  }();
  return on;
}

cudaError_t launch_attention(const AttnDesc& a, cudaStream_t st) {
  AttnGeom g = attn_geom(a);
  if (a.n_seqs == 0 || a.rows == 0) return cudaSuccess;
  if (a.dtype == DFLASH_BF16) {
    const int n_qt = (g.nqv + kClQT - 1) / kClQT;
    if (a.d == 128 && use_tc_attention()) return launch_tc<128>(a, n_qt, st);
    return a.d == 128 ? launch_cluster<128>(a, n_qt, st) : launch_cluster<64>(a, n_qt, st);
  }
  dim3 grid(g.nch, a.nkv * g.n_qt, a.n_seqs);
  const size_t smem = (size_t)(2 * kSimtCH * (a.d + 1) + kAttnWarps * a.d + kAttnWarps * kSimtCH) * sizeof(float);
  auto k = attn_simt_kernel<float>;
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  return launch_pdl(k, grid, dim3(kAttnWarps * 32), smem, st, a, g.n_qt);
}

}  // namespace dfl
