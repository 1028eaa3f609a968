// common.cuh -- device helpers shared by the DFlash kernels (sm_103a).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dflash.h"

namespace dfl {

// Device status word bits (first word of every workspace).
enum : uint32_t {
  ST_NUMERIC = 1u,  // NaN reached an argmax
  ST_TIMEOUT = 2u,  // a bounded wait gave up
  ST_RANGE = 4u,    // a token id (vocabulary) or KV page id (pool) read on the device was out of range
  ST_CHECK = 8u,    // a device bounds assertion of the checked build failed (the access was skipped)
};

// Workspace header: status word + arrival counters of the last-CTA reductions.
constexpr size_t kHeaderBytes = 256;
constexpr int kNumCounters = 32768;
constexpr size_t kCounterBytes = kNumCounters * sizeof(uint32_t);
constexpr size_t kReservedBytes = kHeaderBytes + kCounterBytes;

// Counter regions (indices into the counter array) per kernel family.
constexpr int kCtrGemm = 0;        // 8192 tiles
constexpr int kCtrAttn = 8192;     // 16384 (seq, head, query-tile) groups
constexpr int kCtrHead = 24576;    // LM-head reduction (1)
constexpr int kCtrHeadEnd = 24577;
constexpr int kCtrAttnGrid = 24592;  // streaming attention's grid barrier: count, generation
constexpr int kCtrSample = 25600;  // sampling-mode slice arrivals, one per row (<= 1024)

__device__ __forceinline__ void raise_status(uint32_t* status, uint32_t bits) {
  if (status) atomicOr(status, bits);
}

// Device bounds assertions of the checked build (compiled with
// DFLASH_CHECKED): a failed one raises ST_CHECK in the status word and the
// guarded access is skipped instead of trapping, so the context stays
// usable.  In the normal build the condition is not evaluated.
__device__ __forceinline__ bool check_bound(bool ok, uint32_t* status) {
  if (!ok) raise_status(status, ST_CHECK);
  return ok;
}
#ifdef DFLASH_CHECKED
#define DFL_CHECK(cond, status) (::dfl::check_bound((cond), (status)))
#else
#define DFL_CHECK(cond, status) (true)
#endif

template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T>
__device__ __forceinline__ T from_f(float v);
template <>
__device__ __forceinline__ float from_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// Round a float to the storage type and back (the value a consumer reads).
template <typename T>
__device__ __forceinline__ float round_to(float v) { return to_f<T>(from_f<T>(v)); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Load 8 consecutive elements as floats (16-byte aligned for bf16, 2x16 for f32).
template <typename T>
__device__ __forceinline__ void load8(const T* p, float (&o)[8]);
template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* p, float (&o)[8]) {
  uint4 u = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __bfloat1622float2(b[i]);
    o[2 * i] = f.x;
    o[2 * i + 1] = f.y;
  }
}
template <>
__device__ __forceinline__ void load8<float>(const float* p, float (&o)[8]) {
  float4 a = *reinterpret_cast<const float4*>(p);
  float4 b = *reinterpret_cast<const float4*>(p + 4);
  o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
  o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
}

// Token row m -> sequence, in-block index and absolute position.
struct RowMap {
  const int32_t* base_pos;  // [n_seqs]
  const int32_t* valid;     // [n_seqs] or null
  int32_t rows;             // rows per sequence
  __device__ __forceinline__ int seq(int m) const { return m / rows; }
  __device__ __forceinline__ int idx(int m) const { return m % rows; }
  __device__ __forceinline__ int pos(int m) const { return base_pos[m / rows] + m % rows; }
  __device__ __forceinline__ bool live(int m) const {
    return valid == nullptr || (m % rows) < valid[m / rows];
  }
};

// Where cache slot `slot` of sequence s lives.  Contiguous caches
// [S][nkv][cap][d] (pages == nullptr), or paged pools [pool][nkv][ps][d]
// with the page table pages[s * max_pages + slot / ps].  row0() is the row
// (in head_dim vectors) of KV head 0; KV head g adds g * head_rows().  An
// unmapped page id (outside [0, pool)) sets *bad and maps to page 0, so no
// access leaves the pool.
struct KvMap {
  const int32_t* pages;
  int cap, ps, max_pages, pool, nkv;
  __host__ __device__ __forceinline__ int head_rows() const { return pages ? ps : cap; }
  __device__ __forceinline__ uint32_t row0(int s, int slot, bool* bad) const {
    if (!pages) return (uint32_t)(s * nkv) * (uint32_t)cap + (uint32_t)slot;
    int pg = __ldg(pages + (size_t)s * max_pages + slot / ps);
    if (pg < 0 || pg >= pool) {
      *bad = true;
      pg = 0;
    }
    return (uint32_t)(pg * nkv) * (uint32_t)ps + (uint32_t)(slot % ps);
  }
};

// Programmatic dependent launch: wait for the previous grid's results /
// allow the next grid to start its independent prologue.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded waits give up after a limit and raise ST_TIMEOUT.  The limit and
// a test switch live in the workspace header right after the status word
// (dflash_workspace_control): bytes 8..15 the limit in ns (0: the default,
// 1 s), bytes 16..19 a nonzero word that makes the attention kernels issue
// no K/V copies, so that their waits expire with nothing in flight.
constexpr uint64_t kDefaultWaitNs = 1000000000ull;  // 1 s

__device__ __forceinline__ uint64_t wait_limit_ns(const uint32_t* status) {
  if (status == nullptr) return kDefaultWaitNs;
  const uint64_t v = *reinterpret_cast<const volatile uint64_t*>(status + 2);
  return v != 0 ? v : kDefaultWaitNs;
}

// Test switches (bits of the workspace's stall word): bit 0, the attention
// kernels issue no K/V copy; bit 1, the paired GEMM issues no weight copy.
__device__ __forceinline__ bool stall_kv_loads(const uint32_t* status) {
  return status != nullptr && (*reinterpret_cast<const volatile uint32_t*>(status + 4) & 1u) != 0u;
}
__device__ __forceinline__ bool stall_weight_loads(const uint32_t* status) {
  return status != nullptr && (*reinterpret_cast<const volatile uint32_t*>(status + 4) & 2u) != 0u;
}

}  // namespace dfl
