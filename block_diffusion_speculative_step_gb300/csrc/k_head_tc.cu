// k_head_tc.cu -- tcgen05 LM head with the greedy argmax fused into the
// epilogue (swap-AB like the GEMM: 128 vocabulary rows on the MMA M side,
// the token rows on N).  One CTA per 128-row vocabulary tile streams the
// tile's full hidden dimension through a TMA/mbarrier ring; the epilogue
// reduces the tile's logits to one (best, index, second) triple per token and
// stores it; the last CTA merges all tiles and runs acceptance (head_finish).
// Logits never reach HBM unless the caller asks for them.
#include <cudaTypedefs.h>

#include "head_common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace dfl {

constexpr int kHtThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kHtA = 128 * 128;

struct HeadTcParams {
  CUtensorMap wmap;
  CUtensorMap xmap;
  HeadDesc h;
  int nkb;
};

template <int BN>
struct HtCfg {
  static constexpr int STAGE = kHtA + BN * 128;
  static constexpr int BUDGET = BN <= 64 ? 100 * 1024 : 200 * 1024;
  static constexpr int STAGES = (BUDGET / STAGE) > 8 ? 8 : (BUDGET / STAGE);
  static constexpr int TMEM_COLS = BN < 32 ? 32 : BN;
  static constexpr int XCH = 16 * 128 * 4;
  static constexpr int SMEM = STAGES * STAGE + XCH + 256 + 1024;
};

template <int BN>
__global__ void __launch_bounds__(kHtThreads, 1) head_tc_kernel(const __grid_constant__ HeadTcParams p) {
  using Cfg = HtCfg<BN>;
  constexpr int ST = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_last;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* xch = reinterpret_cast<float*>(smem + ST * Cfg::STAGE);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + ST * Cfg::STAGE + Cfg::XCH);
  uint64_t* empty = full + ST;
  uint64_t* done = empty + ST;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const HeadDesc& h = p.h;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x;
  const int nk = p.nkb;

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
    tc::tma_prefetch_desc(&p.wmap);
    tc::tma_prefetch_desc(&p.xmap);
  }
  if (warp == 1) tc::tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol_w = tc::policy_evict_first();
      const uint64_t pol_x = tc::policy_evict_last();
      int issued = 0;
      for (int i = 0; i < nk; ++i) {
        const int s = i % ST;
        const uint32_t ph = (uint32_t)(i / ST) & 1u;
        if (!tc::mbar_wait(&empty[s], ph ^ 1u, abort)) {
          raise_status(h.status, ST_TIMEOUT);
          *abort = 1;
          break;
        }
        uint8_t* a = smem + s * Cfg::STAGE;
        tc::mbar_arrive_expect_tx(&full[s], Cfg::STAGE);
        tc::tma_load_2d(a, &p.wmap, i * 64, tile * 128, &full[s], pol_w);
        tc::tma_load_2d(a + kHtA, &p.xmap, i * 64, 0, &full[s], pol_x);
        ++issued;
      }
      for (int i = (issued > ST ? issued - ST : 0); i < issued; ++i)
        tc::mbar_wait(&full[i % ST], (uint32_t)(i / ST) & 1u, nullptr);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(128, BN);
      for (int i = 0; i < nk; ++i) {
        const int s = i % ST;
        const uint32_t ph = (uint32_t)(i / ST) & 1u;
        if (!tc::mbar_wait(&full[s], ph, abort)) {
          raise_status(h.status, ST_TIMEOUT);
          *abort = 1;
          break;
        }
        tc::tc_fence_after();
        const uint32_t a = tc::smem_u32(smem + s * Cfg::STAGE);
        const uint32_t b = a + kHtA;
#pragma unroll
        for (int j = 0; j < 4; ++j)
          tc::mma_bf16(tmem, tc::sdesc_sw128(a + 32 * j), tc::sdesc_sw128(b + 32 * j), idesc,
                       (i > 0 || j > 0) ? 1u : 0u);
        tc::mma_commit(&empty[s]);
      }
      tc::mma_commit(done);
    }
  } else {
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const int et = threadIdx.x - 64;  // 0..127
    if (!tc::mbar_wait(done, 0, nullptr)) {
      raise_status(h.status, ST_TIMEOUT);
      *abort = 1;
    }
    tc::named_bar(1, 128);
    const bool ok = (*abort == 0);
    tc::tc_fence_after();
    const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
    const int M = h.M;
    const int ncol = min(BN, ((M + 15) / 16) * 16);
    const int vrow = tile * 128 + r;  // this thread's vocabulary row
    Top2* part = reinterpret_cast<Top2*>(h.partials) + (size_t)tile * M;
    // reduction roles: column jc of the 16-column chunk, rows 16*g8 .. 16*g8+15
    const int jc = et >> 3, g8 = et & 7;
    for (int c0 = 0; c0 < ncol; c0 += 16) {
      float v[16];
      if (ok) {
        tc::tmem_ld16(trow + c0, v);
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = 0.f;
      }
      if (h.logits && vrow < h.V) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int m = c0 + j;
          if (m < M && head_row_used(h, m)) head_store_logit(h, m, vrow, v[j]);
        }
      }
      tc::named_bar(1, 128);
#pragma unroll
      for (int j = 0; j < 16; ++j) xch[j * 128 + r] = v[j];
      tc::named_bar(1, 128);
      const int m = c0 + jc;
      Top2 t = top2_empty();
      if (m < M && head_row_used(h, m)) {
        for (int rr = 16 * g8; rr < 16 * g8 + 16; ++rr) {
          const int vi = tile * 128 + rr;
          if (vi < h.V) top2_push(t, xch[jc * 128 + rr], vi, h.status);
        }
      }
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) {
        Top2 u;
        u.v1 = __shfl_xor_sync(0xffffffffu, t.v1, o);
        u.i1 = __shfl_xor_sync(0xffffffffu, t.i1, o);
        u.v2 = __shfl_xor_sync(0xffffffffu, t.v2, o);
        t = top2_merge(t, u);
      }
      if (g8 == 0 && m < M) part[m] = t;
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, Cfg::TMEM_COLS);
  }
  head_finish(h, gridDim.x, reinterpret_cast<const Top2*>(h.partials), &s_last);
}

// ------------------------------------------------------------------- host

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN>
cudaError_t launch_ht(const HeadTcParams& p, int grid, cudaStream_t st) {
  auto k = head_tc_kernel<BN>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, HtCfg<BN>::SMEM);
  if (e != cudaSuccess) return e;
  k<<<grid, kHtThreads, HtCfg<BN>::SMEM, st>>>(p);
  return cudaGetLastError();
}

}  // namespace

bool head_tc_supported(const HeadDesc& h) {
  return h.dtype == DFLASH_BF16 && h.M >= 1 && h.M <= 256 && h.H % 64 == 0 && h.mode != 2 &&
         (reinterpret_cast<uintptr_t>(h.x) & 15) == 0;
}

size_t head_tc_workspace(const HeadDesc& h) { return (size_t)((h.V + 127) / 128) * h.M * sizeof(Top2) + 256; }

cudaError_t launch_head_tc(const HeadDesc& h, cudaStream_t st) {
  HeadTcParams p;
  memset(&p, 0, sizeof(p));
  p.h = h;
  p.nkb = h.H / 64;
  const int grid = (h.V + 127) / 128;
  const int bn = h.M <= 16 ? 16 : h.M <= 32 ? 32 : h.M <= 64 ? 64 : h.M <= 128 ? 128 : 256;
  if (!make_map(&p.wmap, h.w, h.H, h.V, 128)) return cudaErrorInvalidValue;
  if (!make_map(&p.xmap, h.x, h.H, h.M, bn)) return cudaErrorInvalidValue;
  switch (bn) {
    case 16: return launch_ht<16>(p, grid, st);
    case 32: return launch_ht<32>(p, grid, st);
    case 64: return launch_ht<64>(p, grid, st);
    case 128: return launch_ht<128>(p, grid, st);
    default: return launch_ht<256>(p, grid, st);
  }
}

}  // namespace dfl
