// k_gemm_tc.cu -- tcgen05 GEMM Y[m][n] = sum_k X[m][k] W[n][k] for small
// token counts (M <= 256), with the same fused epilogues as the SIMT GEMM.
//
// Swap-AB: the weight tile (128 output rows x 64 k) is the MMA's A operand
// (M = 128) and the token rows are the B operand (N = BN in 16..256), so the
// one bf16 weight stream -- the dominant HBM traffic at small batch -- fills
// the 128-row tensor-core side.  Per CTA: warp 0 issues TMA loads (128-byte
// swizzle) into a STAGES-deep mbarrier ring, warp 1 allocates TMEM and one
// lane issues tcgen05.mma into an fp32 TMEM accumulator, warps 2-5 drain TMEM
// with tcgen05.ld and run the epilogue.  K is split over `splits` CTAs per
// tile; the split count depends only on (tiles, K, SM count), never on M, and
// the last CTA of a tile sums the fp32 partials in split order, so a token
// row's result is the same whatever other rows share the launch.  No CTA waits
// on another.  Every mbarrier wait is bounded (ST_TIMEOUT).
#include <cudaTypedefs.h>

#include "epilogue.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace dfl {

constexpr int kTcThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kTcA = 128 * 128;  // one 128 x 64 bf16 weight tile, bytes

struct TcParams {  // CUtensorMap members keep it 64-byte aligned
  CUtensorMap wmap[kMaxSeg];
  CUtensorMap xmap;
  GemmDesc g;
  int tiles_per_seg;
  int splits;
  int nkb;  // K / 64
  float* part;
  uint32_t* counters;
  uint32_t* status;
};

template <int BN>
struct TcCfg {
  static constexpr int B = BN * 128;
  static constexpr int STAGE = kTcA + B;
  static constexpr int BUDGET = BN <= 64 ? 100 * 1024 : 200 * 1024;
  static constexpr int STAGES = (BUDGET / STAGE) > 8 ? 8 : (BUDGET / STAGE);
  static constexpr int TMEM_COLS = BN < 32 ? 32 : BN;
  static constexpr int XCH = 16 * 128 * 4;  // epilogue exchange tile
  static constexpr int SMEM = STAGES * STAGE + XCH + 256 + 1024;
};

__device__ __forceinline__ void tc_timeout(uint32_t* status, volatile int* abort) {
  raise_status(status, ST_TIMEOUT);
  *abort = 1;
}

template <int BN>
__global__ void __launch_bounds__(kTcThreads, 1) gemm_tc_kernel(const __grid_constant__ TcParams p) {
  using Cfg = TcCfg<BN>;
  constexpr int ST = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* xch = reinterpret_cast<float*>(smem + ST * Cfg::STAGE);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + ST * Cfg::STAGE + Cfg::XCH);
  uint64_t* empty = full + ST;
  uint64_t* done = empty + ST;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_last = reinterpret_cast<int*>(tmem_slot + 2);

  const GemmDesc& g = p.g;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile_g = blockIdx.x / p.splits;
  const int split = blockIdx.x % p.splits;
  const int seg = tile_g / p.tiles_per_seg;
  const int tile = tile_g % p.tiles_per_seg;
  const int kb0 = split * p.nkb / p.splits;
  const int nk = (split + 1) * p.nkb / p.splits - kb0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < ST; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    tc::mbar_init(done, 1);
    *abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tc::tma_prefetch_desc(&p.wmap[seg]);
    tc::tma_prefetch_desc(&p.xmap);
  }
  if (warp == 1) tc::tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      const uint64_t pol_w = tc::policy_evict_first();
      const uint64_t pol_x = tc::policy_evict_last();
      int issued = 0;
      for (int i = 0; i < nk; ++i) {
        const int s = i % ST;
        const uint32_t ph = (uint32_t)(i / ST) & 1u;
        if (!tc::mbar_wait(&empty[s], ph ^ 1u, abort)) {
          tc_timeout(p.status, abort);
          break;
        }
        uint8_t* a = smem + s * Cfg::STAGE;
        tc::mbar_arrive_expect_tx(&full[s], Cfg::STAGE);
        const int kx = (kb0 + i) * 64;
        if (g.kind == EPI_SWIGLU) {
          tc::tma_load_2d(a, &p.wmap[seg], kx, tile * 64, &full[s], pol_w);
          tc::tma_load_2d(a + kTcA / 2, &p.wmap[seg], kx, g.inter + tile * 64, &full[s], pol_w);
        } else {
          tc::tma_load_2d(a, &p.wmap[seg], kx, g.seg_row0 + tile * 128, &full[s], pol_w);
        }
        tc::tma_load_2d(a + kTcA, &p.xmap, kx, 0, &full[s], pol_x);
        ++issued;
      }
      // every issued copy has landed before this CTA's shared memory goes away
      for (int i = (issued > ST ? issued - ST : 0); i < issued; ++i)
        tc::mbar_wait(&full[i % ST], (uint32_t)(i / ST) & 1u, nullptr);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      constexpr uint32_t idesc = tc::idesc_bf16_f32(128, BN);
      for (int i = 0; i < nk; ++i) {
        const int s = i % ST;
        const uint32_t ph = (uint32_t)(i / ST) & 1u;
        if (!tc::mbar_wait(&full[s], ph, abort)) {
          tc_timeout(p.status, abort);
          break;
        }
        tc::tc_fence_after();
        const uint32_t a = tc::smem_u32(smem + s * Cfg::STAGE);
        const uint32_t b = a + kTcA;
#pragma unroll
        for (int j = 0; j < 4; ++j)
          tc::mma_bf16(tmem, tc::sdesc_sw128(a + 32 * j), tc::sdesc_sw128(b + 32 * j), idesc,
                       (i > 0 || j > 0) ? 1u : 0u);
        tc::mma_commit(&empty[s]);
      }
      tc::mma_commit(done);  // arrives once every issued MMA has completed
    }
  } else {
    // ---------------- epilogue: warps 2..5, TMEM lanes 32*(warp%4) ..
    const int q = warp & 3;
    const int r = q * 32 + lane;  // accumulator row = weight row within the tile
    const int et = threadIdx.x - 64;
    if (!tc::mbar_wait(done, 0, nullptr)) tc_timeout(p.status, abort);
    tc::named_bar(1, 128);
    const bool ok = (*abort == 0);  // same value in every epilogue thread
    tc::tc_fence_after();
    const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
    const int M = g.M;
    const int ncol = min(BN, ((M + 15) / 16) * 16);
    float* part_tile = p.part + (size_t)tile_g * p.splits * BN * 128;
    bool active = ok;
    if (active && p.splits > 1) {
      for (int c0 = 0; c0 < ncol; c0 += 16) {
        float v[16];
        tc::tmem_ld16(trow + c0, v);
        float* dst = part_tile + ((size_t)split * BN + c0) * 128 + r;
#pragma unroll
        for (int j = 0; j < 16; ++j) dst[(size_t)j * 128] = v[j];
      }
      __threadfence();
      tc::named_bar(1, 128);
      if (et == 0) {
        uint32_t* ctr = p.counters + kCtrGemm + tile_g;
        const uint32_t old = atomicAdd(ctr, 1u);
        *s_last = (old == (uint32_t)p.splits - 1);
        if (*s_last) *ctr = 0u;
      }
      tc::named_bar(1, 128);
      active = *s_last != 0;
      if (active) __threadfence();
    }
    if (active) {
      const bool pair = (g.kind == EPI_QKV || g.kind == EPI_SWIGLU);
      const int half = (g.kind == EPI_SWIGLU) ? 64 : g.d / 2;
      const int blk = (g.kind == EPI_SWIGLU) ? 128 : g.d;
      for (int c0 = 0; c0 < ncol; c0 += 16) {
        float v[16];
        if (p.splits > 1) {
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = 0.f;
          for (int s = 0; s < p.splits; ++s) {
            const float* src = part_tile + ((size_t)s * BN + c0) * 128 + r;
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] += __ldcg(src + (size_t)j * 128);
          }
        } else {
          tc::tmem_ld16(trow + c0, v);
        }
        if (!pair) {
          const int n = tile * 128 + r;
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (c0 + j < M) epi_single<__nv_bfloat16>(g, n, c0 + j, v[j]);
        } else {
          tc::named_bar(1, 128);
#pragma unroll
          for (int j = 0; j < 16; ++j) xch[j * 128 + r] = v[j];
          tc::named_bar(1, 128);
          if ((r % blk) < half) {
            int u;
            if (g.kind == EPI_SWIGLU) {
              u = tile * 64 + r;
            } else {
              const int rr = tile * 128 + r;
              u = (rr / g.d) * half + rr % g.d;
            }
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (c0 + j < M) epi_pair<__nv_bfloat16>(g, seg, u, c0 + j, v[j], xch[j * 128 + r + half]);
          }
        }
      }
    }
    (void)et;
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, Cfg::TMEM_COLS);
  }
}

// ------------------------------------------------------------------- host

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// Row-major bf16 [rows][inner] tensor, box = 64 (inner) x box_rows, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int pick_bn(int M) {
  if (M <= 16) return 16;
  if (M <= 32) return 32;
  if (M <= 64) return 64;
  if (M <= 128) return 128;
  return 256;
}

int tiles_per_seg(const GemmDesc& g) { return g.kind == EPI_SWIGLU ? g.inter / 64 : g.seg_rows / 128; }

// Split count from the tile count, K and the SM count only (never M): the
// most even fill of two resident CTAs per SM, at least two k-blocks each.
int pick_splits(int n_tiles, int nkb, int sms) {
  const long slots = 2L * sms;
  int best = 1;
  double best_eff = 0.0;
  const int max_s = nkb / 2 < 32 ? nkb / 2 : 32;
  for (int s = 1; s <= (max_s > 0 ? max_s : 1); ++s) {
    const long units = (long)n_tiles * s;
    const long waves = (units + slots - 1) / slots;
    const double eff = (double)units / (double)(waves * slots);
    if (eff > best_eff + 0.01) {
      best_eff = eff;
      best = s;
    }
  }
  return best;
}

template <int BN>
cudaError_t launch_bn(const TcParams& p, int grid, cudaStream_t st) {
  auto k = gemm_tc_kernel<BN>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, TcCfg<BN>::SMEM);
  if (e != cudaSuccess) return e;
  k<<<grid, kTcThreads, TcCfg<BN>::SMEM, st>>>(p);
  return cudaGetLastError();
}

}  // namespace

bool gemm_tc_supported(const GemmDesc& g) {
  if (g.dtype != DFLASH_BF16 || g.M < 1 || g.M > 256 || g.K % 64 != 0 || g.nseg < 1 || g.nseg > kMaxSeg)
    return false;
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

size_t gemm_tc_workspace(const GemmDesc& g, int num_sms) {
  const int n_tiles = g.nseg * tiles_per_seg(g);
  const int splits = pick_splits(n_tiles, g.K / 64, num_sms);
  if (splits <= 1) return 0;
  return (size_t)n_tiles * splits * pick_bn(g.M) * 128 * sizeof(float);
}

cudaError_t launch_gemm_tc(const GemmDesc& g, void* ws, size_t ws_bytes, uint32_t* counters, uint32_t* status,
                           int num_sms, cudaStream_t st) {
  if (g.M == 0) return cudaSuccess;
  TcParams p;
  memset(&p, 0, sizeof(p));
  p.g = g;
  p.tiles_per_seg = tiles_per_seg(g);
  p.nkb = g.K / 64;
  const int n_tiles = g.nseg * p.tiles_per_seg;
  if (n_tiles > 8192) return cudaErrorInvalidValue;
  p.splits = pick_splits(n_tiles, p.nkb, num_sms);
  const int bn = pick_bn(g.M);
  if (p.splits > 1 && ws_bytes < (size_t)n_tiles * p.splits * bn * 128 * sizeof(float)) return cudaErrorInvalidValue;
  p.part = static_cast<float*>(ws);
  p.counters = counters;
  p.status = status;
  const uint64_t wrows = g.kind == EPI_SWIGLU ? (uint64_t)2 * g.inter : (uint64_t)(g.seg_row0 + g.seg_rows);
  const uint32_t box_rows = g.kind == EPI_SWIGLU ? 64 : 128;
  for (int s = 0; s < g.nseg; ++s)
    if (!make_map(&p.wmap[s], g.seg_w[s], g.K, wrows, box_rows)) return cudaErrorInvalidValue;
  if (!make_map(&p.xmap, g.X, g.K, g.M, bn)) return cudaErrorInvalidValue;
  const int grid = n_tiles * p.splits;
  switch (bn) {
    case 16: return launch_bn<16>(p, grid, st);
    case 32: return launch_bn<32>(p, grid, st);
    case 64: return launch_bn<64>(p, grid, st);
    case 128: return launch_bn<128>(p, grid, st);
    default: return launch_bn<256>(p, grid, st);
  }
}

}  // namespace dfl
