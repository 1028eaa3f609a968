// k_gemm_tc.cu -- persistent stream-K tcgen05 kernel for every weight-
// streaming product of the cycle: the layer GEMMs Y[m][n] = sum_k X[m][k]
// W[n][k] (fused epilogues: RoPE + Q/KV scatter, SwiGLU, residual add, store)
// and the LM head with the greedy argmax fused into its epilogue.
//
// Swap-AB: a 128-row weight tile is the MMA's A operand (M = 128) and the
// token rows are the B operand (N = BN in 16..256); at small batch the one
// bf16 weight stream is the whole HBM traffic.  One CTA per SM (its shared
// memory ring is sized so no second CTA fits).  The
// (tile, 64-wide k-block) space is cut into contiguous runs, one per CTA; a
// run's piece inside one tile accumulates in TMEM.  Roles per CTA: warp 0 streams W and X boxes with TMA (128-byte
// swizzle) through a STAGES-deep mbarrier ring, warp 1 allocates TMEM and one
// lane issues tcgen05.mma into one of two TMEM accumulators, warps 2-5 drain
// the other accumulator with tcgen05.ld, so a piece's epilogue overlaps the
// next piece's loads.  A tile split over several CTAs is finished by the
// piece that completes its k range, summing the fp32 partials in k order:
// the run boundaries depend only on (tiles, K, SM count), never on M, so a
// token row's result does not depend on the other rows in the launch.
// Weight loads for the first stages are issued before griddepcontrol.wait,
// overlapping the predecessor kernel's tail.  Every wait is bounded.
//
// Tiles of more than 16 token rows finish in 16-column chunks; their
// column-independent row operands are staged once per CTA in shared memory
// (RowTab), so a chunk costs one global round trip.  From 128 token rows on,
// every piece only stores its accumulator (a tile that one run covers, into
// a slot of its own) and tc_fixup_kernel, launched behind the GEMM, finishes
// every tile with one CTA per 16-column chunk (same k-order sum, same
// epilogue), so no CTA holds a whole tile's epilogue past its last MMA; two
// 256-row parts of a projection run as one launch of tc_pair_kernel, which
// feeds each weight k-block to the MMAs of both.  The LM head keeps, per
// CTA, each token row's best (logit, index) and runner-up over the tiles the
// CTA finishes; the last CTA merges one triple per CTA.
#include <cudaTypedefs.h>

#include "epilogue.cuh"
#include "head_common.cuh"
#include "internal.h"
#include "launch.cuh"
#include "tc_ptx.cuh"
#include "tmap.h"

namespace dfl {

constexpr int kTcThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kTcA = 128 * 128;  // one 128 x 64 bf16 weight box, bytes

enum TcMode : int { TC_GEMM = 0, TC_HEAD = 1 };

struct TcParams {  // the CUtensorMap members keep it 64-byte aligned
  CUtensorMap wmap[kMaxSeg];
  CUtensorMap xmap;
  GemmDesc g;
  HeadDesc h;
  int mode;
  int tiles_per_seg;
  int n_tiles;
  int nkb;        // k-blocks per tile (K / 64)
  long long T;    // n_tiles * nkb
  int G;          // CTAs (runs)
  int M;          // token rows
  int defer;      // GEMM, BN >= 128: split tiles are finished by tc_fixup_kernel, not by their last piece
  int M_b;        // tc_pair_kernel: token rows of the second 256-row part (its X box starts at row 256)
  float* part_b;  // tc_pair_kernel: the second part's slots (same layout as `part`)
  float* part;    // partial slots [2 G (+ n_tiles when deferred)][BN][128] (piece_slot, tile_slot)
  Top2* tops;     // LM head: per-CTA triples [M][G] (a row's G triples contiguous for the final merge)
  Cand* tlist;    // LM head, top-k mode: per-tile lists [n_tiles][M][topk]
  uint32_t* counters;
  uint32_t* status;
};

template <int BN>
struct TcCfg {
  static constexpr int STAGE = kTcA + BN * 128;
  // Deep enough that one CTA needs more than half of an SM's shared memory:
  // the block scheduler then places exactly one CTA (one run) on every SM.
  static constexpr int BUDGET = BN <= 64 ? 128 * 1024 : 200 * 1024;
  static constexpr int STAGES = (BUDGET / STAGE) > 10 ? 10 : (BUDGET / STAGE);
  static constexpr int ACC = BN < 32 ? 32 : BN;  // columns of one accumulator
  static constexpr int TMEM_COLS = 2 * ACC;       // double-buffered
  static constexpr int XCH = 16 * 128 * 4;        // epilogue exchange tile
  static constexpr bool WIDE = BN > 16;           // several 16-column chunks per tile
  static constexpr int TAB = WIDE ? 2304 : 0;     // RowTab, 256-byte multiple
  static constexpr int SMEM = STAGES * STAGE + XCH + 256 + TAB + 1024;
  static_assert(SMEM > 117 * 1024, "a second CTA must not fit on the SM");
  static_assert(SMEM + 17 * 1024 <= 232448, "with the kernel's ~16.5 KB of static shared memory, one SM");
};

// Run c of the G equal contiguous runs of the (tile, k-block) line [0, T).
__host__ __device__ __forceinline__ long long run_start(long long T, int G, int c) { return (T * c) / G; }

__device__ __forceinline__ int run_of(long long p, long long T, int G) {
  int c = (int)((p * G) / T);
  while (c + 1 <= G && run_start(T, G, c + 1) <= p) ++c;
  while (c > 0 && run_start(T, G, c) > p) --c;
  return c;
}

// Offset (floats) within a partial slot [BN][128] of accumulator row r's
// columns c0 + 4 j4 .. c0 + 4 j4 + 3 (c0 a multiple of 16): per 16-column
// chunk, four [128 rows][4] blocks, so a warp's 16-byte stores and loads of
// one block cover 512 contiguous bytes.
__host__ __device__ __forceinline__ size_t part_off(int c0, int j4, int r) {
  return (size_t)c0 * 128 + (size_t)j4 * 512 + (size_t)r * 4;
}

// Partial slot of run c's piece of a tile.  A run is contiguous, so only its
// first piece (slot 2c) and its last piece (slot 2c + 1, when the run began
// in an earlier tile) can be parts of split tiles: 2 slots per run, whatever
// the tile count.  Of the runs first..last covering a tile, only `first` can
// have begun in an earlier tile (first_tail: run_start(first) < the tile's
// first k-block), so the slots need one 64-bit division per tile, not one
// per piece.
__device__ __forceinline__ size_t piece_slot(int c, int first, bool first_tail) {
  return 2 * (size_t)c + ((c == first && first_tail) ? 1u : 0u);
}

// Slot of tile t's accumulator when one run covers the tile in a deferred
// launch: after the 2 G piece slots.
__host__ __device__ __forceinline__ size_t tile_slot(int G, int t) { return 2 * (size_t)G + (size_t)t; }

__device__ __forceinline__ void tc_timeout(uint32_t* status, volatile int* abort) {
  raise_status(status, ST_TIMEOUT);
  *abort = 1;
}

// Launch scalars held in registers: the inline-asm memory clobbers of the
// pipeline would otherwise force every use to re-read the parameter block.
struct TcLocal {
  int mode, M, tps, nkb, G, n_tiles, kind, d, inter, row0, defer;
  long long T;
  int V, hmode, hblock, topk;
  float* logits;
  Top2* tops;
  Cand* tlist;
  float* part;
  uint32_t* counters;
  uint32_t* status;
};

__device__ __forceinline__ TcLocal tc_local(const TcParams& p) {
  TcLocal L;
  L.mode = p.mode;
  L.M = p.M;
  L.defer = p.defer;
  L.tps = p.tiles_per_seg;
  L.nkb = p.nkb;
  L.G = p.G;
  L.n_tiles = p.n_tiles;
  L.T = p.T;
  L.kind = p.g.kind;
  L.d = p.g.d;
  L.inter = p.g.inter;
  L.row0 = p.g.seg_row0;
  L.V = p.h.V;
  L.hmode = p.h.mode;
  L.hblock = p.h.block;
  L.topk = p.h.topk;
  L.logits = p.h.logits;
  L.tops = p.tops;
  L.tlist = p.tlist;
  L.part = p.part;
  L.counters = p.counters;
  L.status = p.status;
  return L;
}

__device__ __forceinline__ bool row_used(const TcLocal& L, int m) { return L.hmode == 1 || (m % L.hblock) != 0; }

// Output unit of this thread's accumulator row r in tile t: the output
// column (store / residual kinds) or the RoPE / SwiGLU pair unit, whose
// partner row lives in another warp.  False for pair partners (r % blk >= half).
__device__ __forceinline__ bool tc_unit(const TcLocal& L, int t, int r, int& unit) {
  const int tile = t % L.tps;
  if (L.kind == EPI_STORE || L.kind == EPI_RESID) {
    unit = tile * 128 + r;
    return true;
  }
  const int half = (L.kind == EPI_SWIGLU) ? 64 : L.d / 2;
  const int blk = (L.kind == EPI_SWIGLU) ? 128 : L.d;
  if ((r % blk) >= half) return false;
  if (L.kind == EPI_SWIGLU) {
    unit = tile * 64 + r;
  } else {
    const int rr = tile * 128 + r;
    unit = (rr / L.d) * half + rr % L.d;
  }
  return true;
}

// Final epilogue of 16 accumulator columns [c0, c0+16) of tile t for the
// weight row r of this thread (128 epilogue threads, uniform control flow).
// rw / old hold the epilogue's loads for columns 0..15, issued while the
// accumulator was being computed; later column groups load here.
__device__ __forceinline__ void final_chunk(const TcLocal& L, const Epi& e, int t, int c0, int r, int et,
                                            float (&v)[16], float* xch, const EpiRows& rw, const float (&old)[16],
                                            Top2* s_top) {
  const int M = L.M;
  if (L.mode == TC_HEAD) {
    const int vrow = t * 128 + r;
    if (L.logits && vrow < L.V) {
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int m = c0 + j;
        if (m < M && row_used(L, m)) {
          size_t row;
          if (L.hmode == 1) {
            row = (size_t)m;
          } else {
            row = (size_t)(m / L.hblock) * (L.hblock - 1) + (m % L.hblock) - 1;
          }
          L.logits[row * L.V + vrow] = v[j];
        }
      }
    }
    if (L.topk == 0) {
      // Greedy: each warp reduces its 32 rows' (logit, index) pairs of the
      // 16 columns by a butterfly that halves the columns a lane holds at
      // every step (48 shuffles in all), then merges the column's best into
      // its own running selection s_top[warp][m]: no barrier, no shared
      // memory exchange.  top2_merge is associative and commutative, so the
      // grouping does not change the result.
      const bool vr = vrow < L.V;
      bool nan = false;
#pragma unroll
      for (int j = 0; j < 16; ++j) nan |= vr && v[j] != v[j];
      if (nan) raise_status(L.status, ST_NUMERIC);  // NaN never wins; flag it
      float a1[16], a2[16];
      int i1[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const bool ok = vr && v[j] == v[j];
        a1[j] = ok ? v[j] : -INFINITY;
        i1[j] = ok ? vrow : INT_MAX;
        a2[j] = -INFINITY;
      }
      const int lane = r & 31;
#pragma unroll
      for (int o = 16, n = 16; o >= 2; o >>= 1, n >>= 1) {
        const bool hi = (lane & o) != 0;  // keeps the upper half of its n columns
#pragma unroll
        for (int q = 0; q < n / 2; ++q) {
          const float sv = hi ? a1[q] : a1[q + n / 2], sv2 = hi ? a2[q] : a2[q + n / 2];
          const int si = hi ? i1[q] : i1[q + n / 2];
          const Top2 mine = hi ? Top2{a1[q + n / 2], i1[q + n / 2], a2[q + n / 2]} : Top2{a1[q], i1[q], a2[q]};
          const Top2 got{__shfl_xor_sync(0xffffffffu, sv, o), __shfl_xor_sync(0xffffffffu, si, o),
                         __shfl_xor_sync(0xffffffffu, sv2, o)};
          const Top2 mm = top2_merge(mine, got);
          a1[q] = mm.v1;
          i1[q] = mm.i1;
          a2[q] = mm.v2;
        }
      }
      Top2 tp{a1[0], i1[0], a2[0]};  // column c0 + lane / 2, over this lane pair
      const Top2 u{__shfl_xor_sync(0xffffffffu, tp.v1, 1), __shfl_xor_sync(0xffffffffu, tp.i1, 1),
                   __shfl_xor_sync(0xffffffffu, tp.v2, 1)};
      tp = top2_merge(tp, u);
      const int m = c0 + (lane >> 1);
      if ((lane & 1) == 0 && m < M && row_used(L, m)) {
        Top2* st = s_top + (r >> 5) * 256 + m;
        *st = top2_merge(*st, tp);
      }
      return;
    }
    // top-k mode: k rounds over the column's 8 threads, through shared memory
    tc::named_bar(1, 128);
#pragma unroll
    for (int j = 0; j < 16; ++j) xch[j * 128 + r] = v[j];
    tc::named_bar(1, 128);
    const int jc = et >> 3, g8 = et & 7;  // column jc, rows 16*g8 .. 16*g8+15
    const int m = c0 + jc;
    {
      // k rounds: each of the column's 8 threads offers its best unselected
      // row; the winner over the 8 (greater logit, then lower index) is taken.
      const bool used = m < M && row_used(L, m);
      uint32_t taken = 0u;
      Cand* out = L.tlist + ((size_t)t * M + m) * L.topk;
      for (int q = 0; q < L.topk; ++q) {
        float bv = -INFINITY;
        int bi = INT_MAX, brr = -1;
        if (used) {
#pragma unroll
          for (int rr = 0; rr < 16; ++rr) {
            const int vi = t * 128 + 16 * g8 + rr;
            const float x = xch[jc * 128 + 16 * g8 + rr];
            if (vi >= L.V || ((taken >> rr) & 1u)) continue;
            if (x != x) {  // NaN never wins; flag it
              if (q == 0) raise_status(L.status, ST_NUMERIC);
              continue;
            }
            if (beats(x, vi, bv, bi)) {
              bv = x;
              bi = vi;
              brr = rr;
            }
          }
        }
        float rv = bv;
        int ri = bi;
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, rv, o);
          const int oi = __shfl_xor_sync(0xffffffffu, ri, o);
          if (beats(ov, oi, rv, ri)) {
            rv = ov;
            ri = oi;
          }
        }
        if (brr >= 0 && bi == ri) taken |= 1u << brr;
        if (g8 == 0 && used) out[q] = Cand{rv, ri};
      }
      return;
    }
  }
  int unit = 0;
  const bool works = tc_unit(L, t, r, unit);
  if (L.kind == EPI_STORE || L.kind == EPI_RESID) {
    if (c0 == 0) {
      epi_single16(e, unit, c0, v, rw, old);
    } else {
      EpiRows rw2;
      float old2[16];
      epi_preload_rows(e, unit, c0, M, rw2);
      epi_preload_tile(e, unit, c0, rw2, old2);
      epi_single16(e, unit, c0, v, rw2, old2);
    }
    return;
  }
  // pair epilogues: partner row r + half lives in another warp
  const int half = (L.kind == EPI_SWIGLU) ? 64 : L.d / 2;
  tc::named_bar(1, 128);
#pragma unroll
  for (int j = 0; j < 16; ++j) xch[j * 128 + r] = v[j];
  tc::named_bar(1, 128);
  if (works) {
    float w[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) w[j] = xch[j * 128 + r + half];
    if (c0 == 0) {
      epi_pair16<__nv_bfloat16>(e, unit, c0, v, w, rw);
    } else {
      EpiRows rw2;
      epi_preload_rows(e, unit, c0, M, rw2);
      epi_pair16<__nv_bfloat16>(e, unit, c0, v, w, rw2);
    }
  }
}

// ---- wide tiles (more than 16 token rows).  The operands of a token row
// that do not depend on the output column (liveness, position, K/V slot) are
// resolved once per CTA into shared memory, and each 16-column chunk issues
// its few global loads -- the residual being added to, or the rotation of the
// unit's column -- all at once, before its accumulator values are read: one
// round trip per chunk instead of a chain of dependent loads.  The arithmetic
// and the set of writes are those of the 16-column forms.
struct RowTab {
  uint32_t live[8];  // bit m % 32 of word m / 32: token row m is written
  int32_t pos[256];  // QKV: position of a live row inside the RoPE table, else -1
  uint32_t kvr[256]; // QKV: K/V destination row (sequence, head 0, slot); ~0u: none
};
static_assert(sizeof(RowTab) <= 2304, "row table");

// All 128 epilogue threads (et = 0..127) call this: it holds named barriers.
__device__ __forceinline__ void row_tab_build(const Epi& e, int M, int et, RowTab* tb) {
  const int lane = et & 31;
#pragma unroll
  for (int m0 = 0; m0 < 256; m0 += 128) {
    const int m = m0 + et;
    const bool lv = m < M && (e.valid == nullptr || (m % e.rows) < __ldg(e.valid + m / e.rows));
    const uint32_t bits = __ballot_sync(0xffffffffu, lv);
    if (lane == 0) tb->live[m >> 5] = bits;
    int pos = -1;
    uint32_t kvr = ~0u;
    if (e.kind == EPI_QKV && lv) {
      const int q = __ldg(e.base_pos + m / e.rows) + m % e.rows;
      if (q >= 0 && q < e.rope_max_pos) {
        pos = q;
        const int slot = e.kv_slot_mode == 1 ? (e.kv_window > 0 ? q % e.kv_window : q) : m % e.rows;
        if (slot < e.kv_cap) kvr = (uint32_t)((m / e.rows) * e.nkv) * (uint32_t)e.kv_cap + (uint32_t)slot;
      }
    }
    tb->pos[m] = pos;
    tb->kvr[m] = kvr;
  }
  tc::named_bar(1, 128);
}

// The global loads of chunk [c0, c0+16) for output unit `unit`: residual
// rows (EPI_RESID; rows < M are in the buffer whether live or not) or the
// (cos, sin) pairs of the unit's column (EPI_QKV, Q and K rows).
__device__ __forceinline__ void wide_loads(const Epi& e, const RowTab* tb, int unit, bool works, int c0, int M,
                                           float (&pre)[32]) {
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    pre[2 * j] = 0.f;
    pre[2 * j + 1] = 0.f;
  }
  if (e.kind == EPI_RESID) {
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (c0 + j < M) pre[j] = e.out_f32[(size_t)(c0 + j) * e.ldo + unit];
  } else if (e.kind == EPI_QKV) {
#pragma unroll
    for (int j = 0; j < 16; ++j) pre[2 * j] = 1.f;  // (1, 0): V rows are not rotated
    const int ra = e.seg_row0 + (unit / e.half) * e.d + (unit % e.half);
    if (works && ra < e.QD + e.KD) {
      const float2* cs = reinterpret_cast<const float2*>(e.rope_cs) + ra % e.d;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int q = tb->pos[c0 + j];
        const float2 c = q >= 0 ? __ldg(cs + (size_t)q * e.half) : make_float2(1.f, 0.f);
        pre[2 * j] = c.x;
        pre[2 * j + 1] = c.y;
      }
    }
  }
}

// Epilogue of chunk [c0, c0+16) of tile t for accumulator row r, with the
// chunk's loads in `pre` (all 128 epilogue threads: pair kinds exchange rows).
__device__ __forceinline__ void final_wide(const TcLocal& L, const Epi& e, const RowTab* tb, int t, int c0, int r,
                                           const float (&v)[16], float* xch, const float (&pre)[32]) {
  int unit = 0;
  const bool works = tc_unit(L, t, r, unit);
  const uint32_t live = (tb->live[c0 >> 5] >> (c0 & 31)) & 0xffffu;
  if (L.kind == EPI_STORE || L.kind == EPI_RESID) {
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if ((live >> j) & 1u) e.out_f32[(size_t)(c0 + j) * e.ldo + unit] = pre[j] + v[j];
    return;
  }
  const int half = (L.kind == EPI_SWIGLU) ? 64 : L.d / 2;
  tc::named_bar(1, 128);
#pragma unroll
  for (int j = 0; j < 16; ++j) xch[j * 128 + r] = v[j];
  tc::named_bar(1, 128);
  if (!works) return;
  float w[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) w[j] = xch[j * 128 + r + half];
  if (L.kind == EPI_SWIGLU) {
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if ((live >> j) & 1u)
        reinterpret_cast<__nv_bfloat16*>(e.act_out)[(size_t)(c0 + j) * e.inter + unit] =
            from_f<__nv_bfloat16>(silu_f(v[j]) * w[j]);
    return;
  }
  const int d = e.d;
  const int ra = e.seg_row0 + (unit / half) * d + (unit % half);
  const int col = ra % d;
  float lo[16], hi[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    // pre holds (1, 0) for V rows and rows outside the RoPE table
    rope_rot(v[j], w[j], pre[2 * j], pre[2 * j + 1], lo[j], hi[j]);
  }
  if (ra < e.QD) {
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (tb->pos[c0 + j] >= 0 && DFL_CHECK(c0 + j < e.M, e.status)) {
        __nv_bfloat16* q = reinterpret_cast<__nv_bfloat16*>(e.q_out) + (size_t)(c0 + j) * e.QD + ra;
        q[0] = from_f<__nv_bfloat16>(lo[j]);
        q[half] = from_f<__nv_bfloat16>(hi[j]);
      }
    return;
  }
  const bool is_k = ra < e.QD + e.KD;
  const int rr = is_k ? ra - e.QD : ra - e.QD - e.KD;
  __nv_bfloat16* base =
      reinterpret_cast<__nv_bfloat16*>(is_k ? e.k_dst : e.v_dst) + (size_t)(rr / d) * e.kv_cap * d + col;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const uint32_t kv = tb->kvr[c0 + j];
    if (kv == ~0u) continue;
    if (!DFL_CHECK((long long)kv + (long long)(rr / d) * e.kv_cap < e.kv_rows, e.status)) continue;
    __nv_bfloat16* dst = base + (size_t)kv * d;
    dst[0] = from_f<__nv_bfloat16>(lo[j]);
    dst[half] = from_f<__nv_bfloat16>(hi[j]);
  }
}

template <int BN>
__global__ void __launch_bounds__(kTcThreads, 1) tc_stream_kernel(const __grid_constant__ TcParams p) {
  using Cfg = TcCfg<BN>;
  constexpr int ST = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_last_head;
  __shared__ Top2 s_top[4 * 256];  // LM head: per epilogue warp, best (logit, index) and runner-up of each token row so far
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* xch = reinterpret_cast<float*>(smem + ST * Cfg::STAGE);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + ST * Cfg::STAGE + Cfg::XCH);
  uint64_t* empty = full + ST;
  uint64_t* accf = empty + ST;  // [2] accumulator full  (MMA -> epilogue)
  uint64_t* acce = accf + 2;    // [2] accumulator empty (epilogue -> MMA)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acce + 2);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_flag = reinterpret_cast<int*>(tmem_slot + 2);
  RowTab* tab = reinterpret_cast<RowTab*>(smem + ST * Cfg::STAGE + Cfg::XCH + 256);

  const TcLocal L = tc_local(p);
  const CUtensorMap* wmaps = p.wmap;
  const CUtensorMap* xmap = &p.xmap;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = L.nkb;
  const long long p0 = run_start(L.T, L.G, blockIdx.x), p1 = run_start(L.T, L.G, blockIdx.x + 1);
  const int n_my = (int)(p1 - p0);
  const uint64_t lim = wait_limit_ns(L.status);

  if (threadIdx.x == 0) {
    for (int s = 0; s < ST; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&accf[b], 1);
      tc::mbar_init(&acce[b], 1);
    }
    *abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    const int nmaps = L.mode == TC_GEMM ? p.g.nseg : 1;
    for (int s = 0; s < nmaps; ++s) tc::tma_prefetch_desc(wmaps + s);
    tc::tma_prefetch_desc(xmap);
  }
  if (warp == 1) tc::tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      const uint64_t pol_w = tc::policy_evict_first();
      const uint64_t pol_x = tc::policy_evict_last();
      const bool head = L.mode == TC_HEAD, swiglu = L.kind == EPI_SWIGLU;
      const int tps = L.tps, inter = L.inter, row0 = L.row0;
      int t = (int)(p0 / nkb), kb = (int)(p0 - (long long)t * nkb);  // position of load i
      int t_x = t, kb_x = kb;                                          // position of the next X load
      auto load_w = [&](int i) {
        uint8_t* a = smem + (i % ST) * Cfg::STAGE;
        const int kx = kb * 64;
        if (head) {
          tc::tma_load_2d(a, wmaps, kx, t * 128, &full[i % ST], pol_w);
        } else {
          const int seg = t / tps, tile = t - seg * tps;
          if (swiglu) {
            tc::tma_load_2d(a, wmaps + seg, kx, tile * 64, &full[i % ST], pol_w);
            tc::tma_load_2d(a + kTcA / 2, wmaps + seg, kx, inter + tile * 64, &full[i % ST], pol_w);
          } else {
            tc::tma_load_2d(a, wmaps + seg, kx, row0 + tile * 128, &full[i % ST], pol_w);
          }
        }
        if (++kb == nkb) {
          kb = 0;
          ++t;
        }
      };
      auto load_x = [&](int i) {
        tc::tma_load_2d(smem + (i % ST) * Cfg::STAGE + kTcA, xmap, kb_x * 64, 0, &full[i % ST], pol_x);
        if (++kb_x == nkb) {
          kb_x = 0;
          ++t_x;
        }
      };
      // weights depend on nothing upstream: fill the ring before the wait
      const int pre = n_my < ST ? n_my : ST;
      for (int i = 0; i < pre; ++i) {
        tc::mbar_arrive_expect_tx(&full[i], Cfg::STAGE);
        load_w(i);
      }
      pdl_wait();
      for (int i = 0; i < pre; ++i) load_x(i);
      int issued = pre;
      for (int i = pre; i < n_my; ++i) {
        const int s = i % ST;
        if (!tc::mbar_wait(&empty[s], ((uint32_t)(i / ST) & 1u) ^ 1u, abort, lim)) {
          tc_timeout(L.status, abort);
          break;
        }
        tc::mbar_arrive_expect_tx(&full[s], Cfg::STAGE);
        load_w(i);
        load_x(i);
        ++issued;
      }
      // every issued copy has landed before this CTA's shared memory goes away
      for (int i = (issued > ST ? issued - ST : 0); i < issued; ++i)
        tc::mbar_wait(&full[i % ST], (uint32_t)(i / ST) & 1u, nullptr, lim);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer, one accumulator per piece, alternating
      constexpr uint32_t idesc = tc::idesc_bf16_f32(128, BN);
      const uint32_t sbase = tc::smem_u32(smem);
      long long pos = p0;
      int i = 0, k = 0;
      bool stop = false;
      while (pos < p1 && !stop) {
        const int t = (int)(pos / nkb);
        const long long end = p1 < (long long)(t + 1) * nkb ? p1 : (long long)(t + 1) * nkb;
        const int b = k & 1;
        if (!tc::mbar_wait(&acce[b], ((uint32_t)(k >> 1) & 1u) ^ 1u, abort, lim)) {
          tc_timeout(L.status, abort);
          break;
        }
        tc::tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(b * Cfg::ACC);
        for (long long q = pos; q < end; ++q, ++i) {
          const int s = i % ST;
          if (!tc::mbar_wait(&full[s], (uint32_t)(i / ST) & 1u, abort, lim)) {
            tc_timeout(L.status, abort);
            stop = true;
            break;
          }
          tc::tc_fence_after();
          const uint32_t a = sbase + (uint32_t)(s * Cfg::STAGE);
          const uint32_t bb = a + kTcA;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            tc::mma_bf16(d, tc::sdesc_sw128(a + 32 * j), tc::sdesc_sw128(bb + 32 * j), idesc,
                         (q > pos || j > 0) ? 1u : 0u);
          tc::mma_commit(&empty[s]);
        }
        tc::mma_commit(&accf[b]);  // arrives when this piece's MMAs completed
        pos = end;
        ++k;
      }
    }
  } else {
    // ---------------- epilogue: warps 2..5 (TMEM lanes 32*(warp%4) ..)
    pdl_wait();
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;  // accumulator row = weight row within the tile
    const int et = threadIdx.x - 64;
    const int ncol = min(BN, ((L.M + 15) / 16) * 16);
    const uint32_t acce0 = tc::smem_u32(&acce[0]);
    long long pos = p0;
    int k = 0;
    int seg_built = -1;
    Epi e;
    EpiRows rows;  // columns 0..15: the same for every tile of the run
    float old[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) old[j] = 0.f;
    rows.live = 0u;
    if (L.mode == TC_HEAD)
      for (int m = et; m < 4 * 256; m += 128) s_top[m] = top2_empty();  // ordered by the barrier after accf
    if (L.mode == TC_GEMM && p0 < p1) {
      // Nothing loaded here is written before this run's pieces are added:
      // a tile's outputs are written once, by the piece completing its k range.
      const int t = (int)(p0 / nkb);
      seg_built = t / L.tps;
      e = make_epi(p.g, seg_built);
      e.status = L.status;
      if constexpr (Cfg::WIDE) {
        row_tab_build(e, L.M, et, tab);
      } else {
        int unit = 0;
        if (tc_unit(L, t, r, unit)) {
          epi_preload_rows(e, unit, 0, L.M, rows);
          epi_preload_tile(e, unit, 0, rows, old);
        }
      }
    }
    while (pos < p1) {
      const int t = (int)(pos / nkb);
      const long long tbeg = (long long)t * nkb, tend = tbeg + nkb;
      const long long end = p1 < tend ? p1 : tend;
      const bool whole = (pos == tbeg && end == tend);
      const int b = k & 1;
      if (L.mode == TC_GEMM && t / L.tps != seg_built) {
        seg_built = t / L.tps;
        e = make_epi(p.g, seg_built);
        e.status = L.status;
      e.status = L.status;
      }
      if (!tc::mbar_wait(&accf[b], (uint32_t)(k >> 1) & 1u, abort, lim)) tc_timeout(L.status, abort);
      tc::named_bar(1, 128);
      if (*abort) break;  // uniform: read after the barrier
      tc::tc_fence_after();
      // the next piece's per-tile loads go out before this piece's stores
      float old_next[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) old_next[j] = 0.f;
      if (!Cfg::WIDE && L.mode == TC_GEMM && end < p1) {
        const int t2 = (int)(end / nkb);
        Epi e2 = (t2 / L.tps != seg_built) ? make_epi(p.g, t2 / L.tps) : e;
        e2.status = L.status;
        int unit2 = 0;
        if (tc_unit(L, t2, r, unit2)) epi_preload_tile(e2, unit2, 0, rows, old_next);
      }
      const uint32_t trow = tmem + (uint32_t)(b * Cfg::ACC) + ((uint32_t)(q4 * 32) << 16);
      const bool deferred = Cfg::WIDE && L.defer;
      if (whole && !deferred) {
        for (int c0 = 0; c0 < ncol; c0 += 16) {
          float v[16];
          if (Cfg::WIDE && L.mode == TC_GEMM) {
            float pre[32];
            int unit = 0;
            const bool works = tc_unit(L, t, r, unit);
            wide_loads(e, tab, unit, works, c0, L.M, pre);
            tc::tmem_ld16(trow + c0, v);
            final_wide(L, e, tab, t, c0, r, v, xch, pre);
            continue;
          }
          tc::tmem_ld16(trow + c0, v);
          final_chunk(L, e, t, c0, r, et, v, xch, rows, old, s_top);
        }
        tc::tc_fence_before();
        tc::named_bar(1, 128);
        if (et == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(acce0 + 8u * b) : "memory");
      } else {
        // piece_slot of this piece; a deferred whole tile has a slot of its own
        const size_t slot = whole ? tile_slot(L.G, t) : 2 * (size_t)blockIdx.x + (p0 < tbeg ? 1u : 0u);
        float* dst0 = L.part + slot * BN * 128;
        for (int c0 = 0; c0 < ncol; c0 += 16) {
          float v[16];
          tc::tmem_ld16(trow + c0, v);
#pragma unroll
          for (int j4 = 0; j4 < 4; ++j4)
            *reinterpret_cast<float4*>(dst0 + part_off(c0, j4, r)) =
                make_float4(v[4 * j4], v[4 * j4 + 1], v[4 * j4 + 2], v[4 * j4 + 3]);
        }
        tc::tc_fence_before();
        // bar.sync orders every epilogue thread's partial stores before the
        // release of the one thread that publishes the piece; its acquire
        // (and the barrier after it) orders the fixup's loads after the
        // other pieces' stores.
        tc::named_bar(1, 128);
        if (deferred) {  // finished by tc_fixup_kernel once the grid has completed
          if (et == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(acce0 + 8u * b) : "memory");
          pos = end;
          ++k;
          continue;
        }
        if (et == 0) {
          asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(acce0 + 8u * b) : "memory");
          uint32_t* ctr = L.counters + kCtrGemm + t;
          const uint32_t add = (uint32_t)(end - pos);
          uint32_t old_ctr;
          asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old_ctr) : "l"(ctr), "r"(add) : "memory");
          *s_flag = (old_ctr + add == (uint32_t)nkb);
          if (*s_flag) *ctr = 0u;
        }
        tc::named_bar(1, 128);
        if (*s_flag) {
          const int first = run_of(tbeg, L.T, L.G);
          const int last = run_of(tend - 1, L.T, L.G);
          const bool first_tail = run_start(L.T, L.G, first) < tbeg;
          for (int c0 = 0; c0 < ncol; c0 += 16) {
            float v[16];
            float pre[32];
            if (Cfg::WIDE && L.mode == TC_GEMM) {  // in flight with the partial loads
              int unit = 0;
              const bool works = tc_unit(L, t, r, unit);
              wide_loads(e, tab, unit, works, c0, L.M, pre);
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = 0.f;
            // the pieces' partial slots in k order (runs first..last); each
            // batch of up to 4 slots is loaded at once
            for (int sb = first; sb <= last; sb += 4) {
              float pv[4][16];
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const int c = sb + q <= last ? sb + q : last;
                const float* src = L.part + piece_slot(c, first, first_tail) * BN * 128;
#pragma unroll
                for (int j4 = 0; j4 < 4; ++j4) {
                  const float4 x = (sb + q <= last) ? __ldcg(reinterpret_cast<const float4*>(src + part_off(c0, j4, r)))
                                                    : make_float4(0.f, 0.f, 0.f, 0.f);
                  pv[q][4 * j4] = x.x;
                  pv[q][4 * j4 + 1] = x.y;
                  pv[q][4 * j4 + 2] = x.z;
                  pv[q][4 * j4 + 3] = x.w;
                }
              }
#pragma unroll
              for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int j = 0; j < 16; ++j)
                  if (sb + q <= last) v[j] += pv[q][j];
            }
            if (Cfg::WIDE && L.mode == TC_GEMM)
              final_wide(L, e, tab, t, c0, r, v, xch, pre);
            else
              final_chunk(L, e, t, c0, r, et, v, xch, rows, old, s_top);
          }
        }
        tc::named_bar(1, 128);  // s_flag is rewritten by the next piece
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) old[j] = old_next[j];
      pos = end;
      ++k;
    }
    if (L.mode == TC_HEAD && L.topk == 0) {
      tc::named_bar(1, 128);
      for (int m = et; m < L.M; m += 128)
        L.tops[(size_t)m * gridDim.x + blockIdx.x] =
            top2_merge(top2_merge(s_top[m], s_top[256 + m]), top2_merge(s_top[512 + m], s_top[768 + m]));
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, Cfg::TMEM_COLS);
  }
  if (L.mode == TC_HEAD) head_finish(p.h, gridDim.x, gridDim.x, L.tops, &s_last_head);
}

// Two 256-row parts of a deferred projection in one launch: each weight
// k-block lands in shared memory once and feeds the MMAs of both parts (two
// accumulators of 256 columns: all 512 TMEM columns), so the weights cross
// HBM once for up to 512 token rows.  The run partition, every piece's k
// range and the partial slots are those of two separate launches, so the
// fixup and every row's bits are unchanged; with both accumulators in use,
// a piece's MMAs wait until the epilogue has stored the previous piece's
// partials.  Rings: kPairW weight k-blocks and kPairX token-row half blocks
// (a k-block takes two), each slot freed by the MMAs that read it.
constexpr int kPairW = 4, kPairX = 4;
struct PairCfg {
  static constexpr int WB = kTcA;       // one 128 x 64 weight box pair, bytes
  static constexpr int XB = 256 * 128;  // 256 token rows x 64, bytes
  static constexpr int RING = kPairW * WB + kPairX * XB;
  static constexpr int SMEM = RING + 256 + 1024;
  static_assert(SMEM > 117 * 1024 && SMEM <= 227 * 1024, "one CTA per SM");
  static_assert((2 * kPairW + 2 * kPairX + 2) * 8 + 8 <= 256, "barriers fit their 256 bytes");
  static_assert(kPairX % 2 == 0, "a k-block's two halves take consecutive slots");
};

__global__ void __launch_bounds__(kTcThreads, 1) tc_pair_kernel(const __grid_constant__ TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* xring = smem + kPairW * PairCfg::WB;
  uint64_t* wfull = reinterpret_cast<uint64_t*>(smem + PairCfg::RING);
  uint64_t* wempty = wfull + kPairW;
  uint64_t* xfull = wempty + kPairW;
  uint64_t* xempty = xfull + kPairX;
  uint64_t* accf = xempty + kPairX;  // both accumulators hold a finished piece (MMA -> epilogue)
  uint64_t* acce = accf + 1;         // both drained (epilogue -> MMA)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acce + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const TcLocal L = tc_local(p);
  const CUtensorMap* wmaps = p.wmap;
  const CUtensorMap* xmap = &p.xmap;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = L.nkb;
  const long long p0 = run_start(L.T, L.G, blockIdx.x), p1 = run_start(L.T, L.G, blockIdx.x + 1);
  const int n_my = (int)(p1 - p0);
  const uint64_t lim = wait_limit_ns(L.status);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPairW; ++s) {
      tc::mbar_init(&wfull[s], 1);
      tc::mbar_init(&wempty[s], 1);
    }
    for (int s = 0; s < kPairX; ++s) {
      tc::mbar_init(&xfull[s], 1);
      tc::mbar_init(&xempty[s], 1);
    }
    tc::mbar_init(accf, 1);
    tc::mbar_init(acce, 1);
    *abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < p.g.nseg; ++s) tc::tma_prefetch_desc(wmaps + s);
    tc::tma_prefetch_desc(xmap);
  }
  if (warp == 1) tc::tmem_alloc(tmem_slot, 512);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      const uint64_t pol_w = tc::policy_evict_first();
      const uint64_t pol_x = tc::policy_evict_last();
      const bool swiglu = L.kind == EPI_SWIGLU;
      const bool stall = stall_weight_loads(L.status);  // test switch: issue no weight copy
      const int tps = L.tps, inter = L.inter, row0 = L.row0;
      int t = (int)(p0 / nkb), kb = (int)(p0 - (long long)t * nkb);  // position of the next W load
      int kb_x = kb;                                                   // k-block of the next X load
      auto load_w = [&](int i) {
        uint8_t* a = smem + (i % kPairW) * PairCfg::WB;
        uint64_t* bar = &wfull[i % kPairW];
        const int kx = kb * 64, seg = t / tps, tile = t - seg * tps;
        if (++kb == nkb) {
          kb = 0;
          ++t;
        }
        if (stall) return;
        tc::mbar_arrive_expect_tx(bar, PairCfg::WB);
        if (swiglu) {
          tc::tma_load_2d(a, wmaps + seg, kx, tile * 64, bar, pol_w);
          tc::tma_load_2d(a + kTcA / 2, wmaps + seg, kx, inter + tile * 64, bar, pol_w);
        } else {
          tc::tma_load_2d(a, wmaps + seg, kx, row0 + tile * 128, bar, pol_w);
        }
      };
      auto load_x = [&](int i) {  // both 256-row halves of k-block i
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int sl = (2 * i + h) % kPairX;
          tc::mbar_arrive_expect_tx(&xfull[sl], PairCfg::XB);
          tc::tma_load_2d(xring + sl * PairCfg::XB, xmap, kb_x * 64, 256 * h, &xfull[sl], pol_x);
        }
        if (++kb_x == nkb) kb_x = 0;
      };
      // weights depend on nothing upstream: fill their ring before the wait
      const int prw = n_my < kPairW ? n_my : kPairW, prx = n_my < kPairX / 2 ? n_my : kPairX / 2;
      for (int i = 0; i < prw; ++i) load_w(i);
      pdl_wait();
      for (int i = 0; i < prx; ++i) load_x(i);
      // the MMAs of k-block j free its two X slots (for k-block j + kPairX / 2)
      // and its W slot (for k-block j + kPairW); the X halves are needed first
      int iw = prw, ix = prx;
      bool ok = true;
      while (ok && (ix < n_my || iw < n_my)) {
        if (ix < n_my) {
          for (int h = 0; h < 2 && ok; ++h) {
            const int u = 2 * ix + h;
            if (!tc::mbar_wait(&xempty[u % kPairX], ((uint32_t)(u / kPairX) & 1u) ^ 1u, abort, lim)) {
              tc_timeout(L.status, abort);
              ok = false;
            }
          }
          if (!ok) break;
          load_x(ix++);
        }
        if (iw < n_my) {
          if (!tc::mbar_wait(&wempty[iw % kPairW], ((uint32_t)(iw / kPairW) & 1u) ^ 1u, abort, lim)) {
            tc_timeout(L.status, abort);
            break;
          }
          load_w(iw++);
        }
      }
      // every issued copy has landed before this CTA's shared memory goes away
      for (int i = (iw > kPairW ? iw - kPairW : 0); i < iw && !stall; ++i)
        tc::mbar_wait(&wfull[i % kPairW], (uint32_t)(i / kPairW) & 1u, nullptr, lim);
      for (int u = (2 * ix > kPairX ? 2 * ix - kPairX : 0); u < 2 * ix; ++u)
        tc::mbar_wait(&xfull[u % kPairX], (uint32_t)(u / kPairX) & 1u, nullptr, lim);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer: both parts of every k-block of a piece
      constexpr uint32_t idesc = tc::idesc_bf16_f32(128, 256);
      const uint32_t wbase = tc::smem_u32(smem), xbase = tc::smem_u32(xring);
      long long pos = p0;
      int i = 0, k = 0;
      bool stop = false;
      while (pos < p1 && !stop) {
        const int t = (int)(pos / nkb);
        const long long end = p1 < (long long)(t + 1) * nkb ? p1 : (long long)(t + 1) * nkb;
        if (!tc::mbar_wait(acce, ((uint32_t)k & 1u) ^ 1u, abort, lim)) {
          tc_timeout(L.status, abort);
          break;
        }
        tc::tc_fence_after();
        for (long long q = pos; q < end; ++q, ++i) {
          const int sw = i % kPairW, sx0 = (2 * i) % kPairX, sx1 = (2 * i + 1) % kPairX;
          if (!tc::mbar_wait(&wfull[sw], (uint32_t)(i / kPairW) & 1u, abort, lim) ||
              !tc::mbar_wait(&xfull[sx0], (uint32_t)((2 * i) / kPairX) & 1u, abort, lim) ||
              !tc::mbar_wait(&xfull[sx1], (uint32_t)((2 * i + 1) / kPairX) & 1u, abort, lim)) {
            tc_timeout(L.status, abort);
            stop = true;
            break;
          }
          tc::tc_fence_after();
          const uint32_t a = wbase + (uint32_t)(sw * PairCfg::WB);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t bb = xbase + (uint32_t)((h ? sx1 : sx0) * PairCfg::XB);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              tc::mma_bf16(tmem + (uint32_t)(h * 256), tc::sdesc_sw128(a + 32 * j), tc::sdesc_sw128(bb + 32 * j),
                           idesc, (q > pos || j > 0) ? 1u : 0u);
          }
          tc::mma_commit(&wempty[sw]);
          tc::mma_commit(&xempty[sx0]);
          tc::mma_commit(&xempty[sx1]);
        }
        tc::mma_commit(accf);  // arrives when this piece's MMAs completed
        pos = end;
        ++k;
      }
    }
  } else {
    // ---------------- epilogue: warps 2..5 store both accumulators of each piece
    pdl_wait();  // the slots may still be read by the fixup of the launch before
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;  // accumulator row = weight row within the tile
    const int et = threadIdx.x - 64;
    const int ncol[2] = {min(256, ((p.M + 15) / 16) * 16), min(256, ((p.M_b + 15) / 16) * 16)};
    long long pos = p0;
    int k = 0;
    while (pos < p1) {
      const int t = (int)(pos / nkb);
      const long long tbeg = (long long)t * nkb, tend = tbeg + nkb;
      const long long end = p1 < tend ? p1 : tend;
      const bool whole = (pos == tbeg && end == tend);
      if (!tc::mbar_wait(accf, (uint32_t)k & 1u, abort, lim)) tc_timeout(L.status, abort);
      tc::named_bar(1, 128);
      if (*abort) break;  // uniform: read after the barrier
      tc::tc_fence_after();
      // piece_slot of this piece; a whole tile has a slot of its own
      const size_t slot = whole ? tile_slot(L.G, t) : 2 * (size_t)blockIdx.x + (p0 < tbeg ? 1u : 0u);
#pragma unroll
      const uint64_t keep = tc::policy_evict_last();
      for (int h = 0; h < 2; ++h) {
        float* dst0 = (h ? p.part_b : L.part) + slot * 256 * 128;
        const uint32_t trow = tmem + (uint32_t)(h * 256) + ((uint32_t)(q4 * 32) << 16);
        int c0 = 0;
        for (; c0 + 64 <= ncol[h]; c0 += 64) {  // four chunks per TMEM load: one wait instead of four
          float v[64];
          tc::tmem_ld64(trow + c0, v);
#pragma unroll
          for (int j = 0; j < 16; ++j)
            tc::st_global_hint(dst0 + part_off(c0 + 16 * (j >> 2), j & 3, r),
                               make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]), keep);
        }
        for (; c0 < ncol[h]; c0 += 16) {
          float v[16];
          tc::tmem_ld16(trow + c0, v);
#pragma unroll
          for (int j4 = 0; j4 < 4; ++j4)
            tc::st_global_hint(dst0 + part_off(c0, j4, r), make_float4(v[4 * j4], v[4 * j4 + 1], v[4 * j4 + 2], v[4 * j4 + 3]), keep);
        }
      }
      tc::tc_fence_before();
      tc::named_bar(1, 128);
      if (et == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc::smem_u32(acce)) : "memory");
      pos = end;
      ++k;
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}

// Tiles of a deferred launch (BN >= 128), once the GEMM grid has completed:
// one CTA of 128 threads per (part, tile, 16-column chunk); thread r sums
// accumulator row r's partial slots in k order and runs the chunk's epilogue
// -- the arithmetic and order of a last piece finishing its tile inline (a
// tile that one run covers: its accumulator as it is), spread over every SM
// instead of one CTA per tile.  Each thread first copies its own 16-byte
// blocks of the slots into shared memory (cp.async), then the row table is
// built, so the two latencies overlap and the slots cost no registers.
constexpr int kFixBatch = 8;  // most slots held in shared memory (more: in batches)

// The deferred launches finished by one fixup launch: a projection of more
// than 256 token rows runs as several GEMM launches (whole sequences each)
// and one fixup behind the last of them.
constexpr int kMaxFixParts = 4;
struct FixPart {
  GemmDesc g;
  float* part;
  long long T;
  int M, tps, n_tiles, nkb, G;
  int blocks;  // fixup CTAs of this part: n_tiles x 16-column chunks
};
struct FixParams {
  FixPart q[kMaxFixParts];
  int nparts;
  int pb;  // slots held in shared memory ([pb][4][128] float4)
  uint32_t* status;
};
static_assert(sizeof(FixParams) <= 4000, "fixup parameters fit the classic 4 KB parameter space");

__device__ __forceinline__ void part_copy16(void* sdst, const void* g) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(tc::smem_u32(sdst)), "l"(g) : "memory");
}

template <int BN>
__global__ void __launch_bounds__(128, 6) tc_fixup_kernel(const __grid_constant__ FixParams fp) {
  extern __shared__ float4 s_part[];  // [pb][4][128]: slot q's block j4 of row r at (q * 4 + j4) * 128 + r
  __shared__ RowTab s_tab;
  __shared__ float s_xch[16 * 128];
  int bid = (int)blockIdx.x, pi = 0;
  while (pi + 1 < fp.nparts && bid >= fp.q[pi].blocks) bid -= fp.q[pi++].blocks;
  const FixPart& P = fp.q[pi];
  TcLocal L;
  memset(&L, 0, sizeof(L));
  L.mode = TC_GEMM;
  L.M = P.M;
  L.defer = 1;
  L.tps = P.tps;
  L.nkb = P.nkb;
  L.G = P.G;
  L.n_tiles = P.n_tiles;
  L.T = P.T;
  L.kind = P.g.kind;
  L.d = P.g.d;
  L.inter = P.g.inter;
  L.row0 = P.g.seg_row0;
  L.part = P.part;
  L.status = fp.status;
  const int nkb = L.nkb, PB = fp.pb;
  const int nch = min(BN, ((L.M + 15) / 16) * 16) / 16;
  const int t = bid / nch, c0 = (bid % nch) * 16;
  const long long tbeg = (long long)t * nkb, tend = tbeg + nkb;
  const int first = run_of(tbeg, L.T, L.G), last = run_of(tend - 1, L.T, L.G);
  const bool first_tail = run_start(L.T, L.G, first) < tbeg;
  const int r = threadIdx.x, lane = r & 31;
  const int np = last - first + 1;  // pieces, in k order
  uint32_t dyn;
  asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
  if (PB < 1 || (size_t)PB * 4 * 128 * 16 > dyn) {  // uniform
    if (r == 0) raise_status(L.status, ST_RANGE);
    return;
  }
  auto copy_batch = [&](int q0) {  // slots q0 .. q0 + PB - 1, one cp.async group
    for (int q = q0; q < np && q < q0 + PB; ++q) {
      const size_t slot = np == 1 ? tile_slot(L.G, t) : piece_slot(first + q, first, first_tail);
      const float* src = L.part + slot * BN * 128;
#pragma unroll
      for (int j4 = 0; j4 < 4; ++j4) part_copy16(&s_part[((q - q0) * 4 + j4) * 128 + r], src + part_off(c0, j4, r));
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  // The row table and the RoPE operands come from inputs (positions, valid
  // lengths, the RoPE table) that no kernel of the call writes: resolved
  // before the wait, while the GEMM still runs.
  Epi e = make_epi(P.g, t / L.tps);
  e.status = L.status;
  // row operands of the 32-row word holding the chunk (warp 0)
  if (r < 32) {
    const int m = (c0 & ~31) + lane;
    const bool in = m < L.M;
    const int sq = in ? m / e.rows : 0;
    const int bp = (in && e.kind == EPI_QKV) ? __ldg(e.base_pos + sq) : 0;  // issued with the valid load
    const bool lv = in && (e.valid == nullptr || (m % e.rows) < __ldg(e.valid + sq));
    const uint32_t bits = __ballot_sync(0xffffffffu, lv);
    if (lane == 0) s_tab.live[c0 >> 5] = bits;
    int pos = -1;
    uint32_t kvr = ~0u;
    if (e.kind == EPI_QKV && lv) {
      const int q = bp + m % e.rows;
      if (q >= 0 && q < e.rope_max_pos) {
        pos = q;
        const int slot = e.kv_slot_mode == 1 ? (e.kv_window > 0 ? q % e.kv_window : q) : m % e.rows;
        if (slot < e.kv_cap) kvr = (uint32_t)((m / e.rows) * e.nkv) * (uint32_t)e.kv_cap + (uint32_t)slot;
      }
    }
    s_tab.pos[m] = pos;
    s_tab.kvr[m] = kvr;
  }
  __syncthreads();
  float pre[32];
  int unit = 0;
  const bool works = tc_unit(L, t, r, unit);
  if (e.kind == EPI_QKV) wide_loads(e, &s_tab, unit, works, c0, L.M, pre);
  pdl_wait();
  pdl_launch_dependents();
  copy_batch(0);
  if (e.kind != EPI_QKV) wide_loads(e, &s_tab, unit, works, c0, L.M, pre);  // the residual: the GEMM's predecessors' output
  float v[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = 0.f;
  for (int q0 = 0; q0 < np; q0 += PB) {
    if (q0 > 0) copy_batch(q0);
    asm volatile("cp.async.wait_all;" ::: "memory");  // this thread's own copies: no barrier needed
    for (int q = q0; q < np && q < q0 + PB; ++q) {
#pragma unroll
      for (int j4 = 0; j4 < 4; ++j4) {
        const float4 x = s_part[((q - q0) * 4 + j4) * 128 + r];
        if (np == 1) {  // the tile's accumulator as it is (no 0 + x)
          v[4 * j4] = x.x;
          v[4 * j4 + 1] = x.y;
          v[4 * j4 + 2] = x.z;
          v[4 * j4 + 3] = x.w;
        } else {
          v[4 * j4] += x.x;
          v[4 * j4 + 1] += x.y;
          v[4 * j4 + 2] += x.z;
          v[4 * j4 + 3] += x.w;
        }
      }
    }
  }
  final_wide(L, e, &s_tab, t, c0, r, v, s_xch, pre);
}

// ------------------------------------------------------------------- host

namespace {

bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  return make_tmap_bf16(m, base, inner, rows, box_rows);
}

int pick_bn(int M) {
  if (M <= 16) return 16;
  if (M <= 32) return 32;
  if (M <= 64) return 64;
  if (M <= 128) return 128;
  return 256;
}

int gemm_tiles_per_seg(const GemmDesc& g) { return g.kind == EPI_SWIGLU ? g.inter / 64 : g.seg_rows / 128; }

int runs_for(long long T, int num_sms) { return (int)(T < num_sms ? T : num_sms); }

// Split-K partial slots: two per run (piece_slot), and in a deferred launch
// (BN >= 128) one per tile as well (tile_slot).
size_t part_bytes(int G, int bn, int n_tiles = 0) {
  return ((size_t)2 * G + (bn >= 128 ? (size_t)n_tiles : 0)) * bn * 128 * sizeof(float);
}

// Two 256-row parts of a projection as one paired launch (tc_pair_kernel).
#ifndef DFLASH_GEMM_PAIR
#define DFLASH_GEMM_PAIR 1
#endif
constexpr bool kGemmPair = DFLASH_GEMM_PAIR != 0;

// Most pieces any tile has: runs are at least floor(T / G) k-blocks long.
int max_pieces(long long T, int G, int nkb) {
  const long long lmin = T / G;
  return (int)((nkb - 1 + lmin - 1) / lmin) + 1;
}

template <int BN>
cudaError_t launch_bn(const TcParams& p, cudaStream_t st) {
  auto k = tc_stream_kernel<BN>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, TcCfg<BN>::SMEM);
  if (e != cudaSuccess) return e;
  return launch_pdl(k, dim3(p.G), dim3(kTcThreads), TcCfg<BN>::SMEM, st, p);
}

cudaError_t launch_params(const TcParams& p, cudaStream_t st) {
  switch (pick_bn(p.M)) {
    case 16: return launch_bn<16>(p, st);
    case 32: return launch_bn<32>(p, st);
    case 64: return launch_bn<64>(p, st);
    case 128: return launch_bn<128>(p, st);
    default: return launch_bn<256>(p, st);
  }
}

template <int BN>
cudaError_t launch_fixup(FixParams& f, int pb, cudaStream_t st) {
  f.pb = pb;
  int blocks = 0;
  for (int i = 0; i < f.nparts; ++i) {
    FixPart& q = f.q[i];
    q.blocks = q.n_tiles * ((q.M < BN ? (q.M + 15) / 16 * 16 : BN) / 16);
    blocks += q.blocks;
  }
  const size_t smem = (size_t)f.pb * 4 * 128 * 16;
  cudaError_t e = cudaFuncSetAttribute(tc_fixup_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kFixBatch * 4 * 128 * 16);
  if (e != cudaSuccess) return e;
  return launch_pdl(tc_fixup_kernel<BN>, dim3(blocks), dim3(128), smem, st, f);
}

}  // namespace

bool gemm_tc_supported(const GemmDesc& g) {
  if (g.dtype != DFLASH_BF16 || g.M < 1 || g.K % 64 != 0 || g.nseg < 1 || g.nseg > kMaxSeg) return false;
  if (g.M > 256 && g.rows > 256) return false;  // launches of <= 256 rows split at sequence boundaries
  if ((reinterpret_cast<uintptr_t>(g.X) & 15) != 0) return false;
  switch (g.kind) {
    case EPI_STORE:
    case EPI_RESID:
      return g.seg_row0 == 0 && g.seg_rows % 128 == 0;
    case EPI_QKV:
      return (g.d == 64 || g.d == 128) && g.seg_rows % 128 == 0 && g.seg_row0 % 128 == 0;
    case EPI_SWIGLU:
      return g.inter % 64 == 0 && g.seg_rows == 2 * g.inter;
  }
  return false;
}

// Token rows of each launch: more than 256 rows run as launches of whole
// sequences (<= 256 rows each).
int launch_rows(const GemmDesc& g) {
  if (g.M <= 256) return g.M;
  const int per = g.rows > 0 ? g.rows : 1;
  return (256 / per) * per;
}

size_t gemm_tc_workspace(const GemmDesc& g, int num_sms) {
  const int n_tiles = g.nseg * gemm_tiles_per_seg(g);
  const long long T = (long long)n_tiles * (g.K / 64);
  const int G = runs_for(T, num_sms), mc = launch_rows(g);
  if (mc < 1) return 0;
  size_t b = 0;  // every launch has its own slots: one fixup reads them all
  for (int m0 = 0; m0 < g.M; m0 += mc) b += part_bytes(G, pick_bn(std::min(mc, g.M - m0)), n_tiles);
  return b;
}

namespace {

// The launch parameters of one part of <= 256 token rows, its slots at ws.
cudaError_t part_params(const GemmDesc& g, void* ws, size_t ws_bytes, uint32_t* counters, uint32_t* status,
                        int num_sms, TcParams& p) {
  memset(&p, 0, sizeof(p));
  p.mode = TC_GEMM;
  p.g = g;
  p.M = g.M;
  p.tiles_per_seg = gemm_tiles_per_seg(g);
  p.n_tiles = g.nseg * p.tiles_per_seg;
  p.nkb = g.K / 64;
  p.T = (long long)p.n_tiles * p.nkb;
  p.G = runs_for(p.T, num_sms);
  if (p.n_tiles > 8192) return cudaErrorInvalidValue;
  if (ws_bytes < part_bytes(p.G, pick_bn(g.M), p.n_tiles)) return cudaErrorInvalidValue;
  p.part = static_cast<float*>(ws);
  p.counters = counters;
  p.status = status;
  p.defer = pick_bn(g.M) >= 128 ? 1 : 0;
  const uint64_t wrows = g.kind == EPI_SWIGLU ? (uint64_t)2 * g.inter : (uint64_t)(g.seg_row0 + g.seg_rows);
  const uint32_t box_rows = g.kind == EPI_SWIGLU ? 64 : 128;
  for (int s = 0; s < g.nseg; ++s)
    if (!make_map(&p.wmap[s], g.seg_w[s], g.K, wrows, box_rows)) return cudaErrorInvalidValue;
  if (!make_map(&p.xmap, g.X, g.K, g.M, pick_bn(g.M))) return cudaErrorInvalidValue;
  return cudaSuccess;
}

}  // namespace

// The GEMM launches of every part first, then one fixup for the deferred
// parts (BN >= 128), so a part's GEMM does not wait for the previous part's
// fixup.  A row's result does not depend on the launch it is in: the
// k-partition is a function of the tiles and K only.
cudaError_t launch_gemm_tc(const GemmDesc& g, void* ws, size_t ws_bytes, uint32_t* counters, uint32_t* status,
                           int num_sms, cudaStream_t st) {
  if (g.M == 0) return cudaSuccess;
  const int per = g.rows > 0 ? g.rows : 1;
  const int mc = launch_rows(g);
  if (mc < 1) return cudaErrorInvalidValue;
  FixParams f;
  memset(&f, 0, sizeof(f));
  f.status = status;
  auto add_part = [&](const GemmDesc& c, const TcParams& p, float* part) {
    FixPart& fp = f.q[f.nparts++];
    fp.g = c;
    fp.part = part;
    fp.T = p.T;
    fp.M = c.M;
    fp.tps = p.tiles_per_seg;
    fp.n_tiles = p.n_tiles;
    fp.nkb = p.nkb;
    fp.G = p.G;
  };
  int f_bn = 0, f_pb = 1;
  auto flush = [&]() -> cudaError_t {
    if (f.nparts == 0) return cudaSuccess;
    const cudaError_t e = f_bn == 256 ? launch_fixup<256>(f, f_pb, st) : launch_fixup<128>(f, f_pb, st);
    f.nparts = 0;
    f_pb = 1;
    return e;
  };
  // Two 256-row parts (more than 384 and at most 512 rows, whole sequences
  // of a 256-row boundary): one paired launch, the weights read once.
  if (kGemmPair && mc == 256 && g.M > 384 && g.M <= 512) {
    GemmDesc c0 = g, c1 = g;
    c0.M = 256;
    c1.M = g.M - 256;
    const int sq = 256 / per;
    c1.X = static_cast<const char*>(g.X) + (size_t)256 * g.K * 2;
    if (g.base_pos) c1.base_pos = g.base_pos + sq;
    if (g.valid) c1.valid = g.valid + sq;
    if (g.out_f32) c1.out_f32 = g.out_f32 + (size_t)256 * g.ldo;
    if (g.q_out) c1.q_out = static_cast<char*>(g.q_out) + (size_t)256 * g.nq * g.d * 2;
    if (g.act_out) c1.act_out = static_cast<char*>(g.act_out) + (size_t)256 * g.inter * 2;
    for (int q = 0; q < g.nseg; ++q) {
      const size_t kv = (size_t)sq * g.nkv * g.kv_cap * g.d * 2;
      if (g.k_dst[q]) c1.k_dst[q] = static_cast<char*>(g.k_dst[q]) + kv;
      if (g.v_dst[q]) c1.v_dst[q] = static_cast<char*>(g.v_dst[q]) + kv;
    }
    TcParams p;
    cudaError_t e = part_params(c0, ws, ws_bytes, counters, status, num_sms, p);
    if (e != cudaSuccess) return e;
    const size_t b0 = part_bytes(p.G, 256, p.n_tiles);
    if (ws_bytes < 2 * b0) return cudaErrorInvalidValue;
    p.M_b = c1.M;
    p.part_b = reinterpret_cast<float*>(static_cast<char*>(ws) + b0);
    if (!make_map(&p.xmap, g.X, g.K, g.M, 256)) return cudaErrorInvalidValue;  // both halves
    e = cudaFuncSetAttribute(tc_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, PairCfg::SMEM);
    if (e != cudaSuccess) return e;
    e = launch_pdl(tc_pair_kernel, dim3(p.G), dim3(kTcThreads), PairCfg::SMEM, st, p);
    if (e != cudaSuccess) return e;
    add_part(c0, p, p.part);
    add_part(c1, p, p.part_b);
    return launch_fixup<256>(f, std::min(max_pieces(p.T, p.G, p.nkb), kFixBatch), st);
  }
  size_t off = 0;
  for (int m0 = 0; m0 < g.M; m0 += mc) {
    GemmDesc c = g;
    const int sq = m0 / per;  // first sequence of the launch
    c.M = g.M - m0 < mc ? g.M - m0 : mc;
    if (m0 > 0) {
      c.X = static_cast<const char*>(g.X) + (size_t)m0 * g.K * 2;
      if (g.base_pos) c.base_pos = g.base_pos + sq;
      if (g.valid) c.valid = g.valid + sq;
      if (g.out_f32) c.out_f32 = g.out_f32 + (size_t)m0 * g.ldo;
      if (g.q_out) c.q_out = static_cast<char*>(g.q_out) + (size_t)m0 * g.nq * g.d * 2;
      if (g.act_out) c.act_out = static_cast<char*>(g.act_out) + (size_t)m0 * g.inter * 2;
      for (int q = 0; q < g.nseg; ++q) {
        const size_t kv = (size_t)sq * g.nkv * g.kv_cap * g.d * 2;
        if (g.k_dst[q]) c.k_dst[q] = static_cast<char*>(g.k_dst[q]) + kv;
        if (g.v_dst[q]) c.v_dst[q] = static_cast<char*>(g.v_dst[q]) + kv;
      }
    }
    TcParams p;
    if (off > ws_bytes) return cudaErrorInvalidValue;
    cudaError_t e = part_params(c, static_cast<char*>(ws) + off, ws_bytes - off, counters, status, num_sms, p);
    if (e != cudaSuccess) return e;
    const int bn = pick_bn(c.M);
    off += part_bytes(p.G, bn, p.n_tiles);
    e = launch_params(p, st);
    if (e != cudaSuccess) return e;
    if (!p.defer) continue;
    if (f.nparts == kMaxFixParts || (f.nparts > 0 && f_bn != bn)) {
      e = flush();
      if (e != cudaSuccess) return e;
    }
    add_part(c, p, p.part);
    f_bn = bn;
    f_pb = std::max(f_pb, std::min(max_pieces(p.T, p.G, p.nkb), kFixBatch));
  }
  return flush();
}

// ------------------------------------------------------------- LM head

bool head_tc_supported(const HeadDesc& h) {
  return h.dtype == DFLASH_BF16 && h.M >= 1 && h.M <= 256 && h.H % 64 == 0 &&
         (h.mode != 2 || (h.topk >= 1 && h.topk <= kMaxTopK)) &&
         (reinterpret_cast<uintptr_t>(h.x) & 15) == 0 && (h.V + 127) / 128 <= 8192;
}

// Selections of the LM head: one triple per (CTA, token row), or the top-k
// lists of every (tile, token row).
size_t head_sel_bytes(const HeadDesc& h, int n_tiles, int G) {
  const size_t t2 = (size_t)G * h.M * sizeof(Top2);  // one selection per CTA
  const size_t tk = (size_t)n_tiles * h.M * (h.topk > 0 ? h.topk : 0) * sizeof(Cand);
  return t2 > tk ? t2 : tk;
}

size_t head_tc_workspace(const HeadDesc& h, int num_sms) {
  const int n_tiles = (h.V + 127) / 128;
  const long long T = (long long)n_tiles * (h.H / 64);
  return ((part_bytes(runs_for(T, num_sms), pick_bn(h.M)) + 255) & ~size_t(255)) +
         head_sel_bytes(h, n_tiles, runs_for(T, num_sms)) + 256;
}

const void* head_tc_tlist(const HeadDesc& h, int num_sms, int* n_tiles) {
  const int nt = (h.V + 127) / 128;
  const long long T = (long long)nt * (h.H / 64);
  const size_t pb = part_bytes(runs_for(T, num_sms), pick_bn(h.M));
  *n_tiles = nt;
  return reinterpret_cast<const char*>(h.partials) + ((pb + 255) & ~size_t(255));
}

cudaError_t launch_head_tc(const HeadDesc& h, int num_sms, cudaStream_t st) {
  TcParams p;
  memset(&p, 0, sizeof(p));
  p.mode = TC_HEAD;
  p.h = h;
  p.M = h.M;
  p.tiles_per_seg = (h.V + 127) / 128;
  p.n_tiles = p.tiles_per_seg;
  p.nkb = h.H / 64;
  p.T = (long long)p.n_tiles * p.nkb;
  p.G = runs_for(p.T, num_sms);
  const size_t pb = part_bytes(p.G, pick_bn(h.M));
  p.part = h.partials;
  p.tops = reinterpret_cast<Top2*>(reinterpret_cast<char*>(h.partials) + ((pb + 255) & ~size_t(255)));
  p.tlist = reinterpret_cast<Cand*>(p.tops);
  p.counters = h.counters;
  p.status = h.status;
  if (!make_map(&p.wmap[0], h.w, h.H, h.V, 128)) return cudaErrorInvalidValue;
  if (!make_map(&p.xmap, h.x, h.H, h.M, pick_bn(h.M))) return cudaErrorInvalidValue;
  return launch_params(p, st);
}

}  // namespace dfl
