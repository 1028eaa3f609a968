// trace.cu -- opt-in kernel tracing: while on (per host thread), every kernel
// the library launches is bracketed by two CUDA events on its stream.  Event
// records are stream operations, so they are captured into CUDA graphs too;
// after a replay the pairs hold that replay's per-kernel durations.
#include <string.h>

#include <vector>

#include "../../include/dflash.h"
#include "trace.h"

namespace dfl {

namespace {
struct Rec {
  int family;
  int kernels;  // kernels the traced call launched
  double bytes;
  cudaEvent_t a, b;
};
struct TraceState {
  bool on = false;
  int cap = 0;
  std::vector<cudaEvent_t> pool;
  std::vector<Rec> recs;
  int open_family = -1;
  cudaEvent_t open_a = nullptr;
  long long kernels = 0;  // kernel launches on this host thread
  long long open_k = 0;
};
thread_local TraceState g_trace;

const char* kFamilyNames[kTraceFamilies] = {"embed",      "rmsnorm", "gemm_simt", "gemm_tc",
                                            "attention",  "lm_head", "path",      "rope_table",
                                            "tap_store",  "convert", "sample",  "conv",   "kv_page"};
}  // namespace

// Inside stream capture an external record becomes an event node of the
// graph; outside capture a plain record is used.
cudaError_t record(cudaEvent_t e, cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) cs = cudaStreamCaptureStatusNone;
  return cs == cudaStreamCaptureStatusActive ? cudaEventRecordWithFlags(e, st, cudaEventRecordExternal)
                                             : cudaEventRecord(e, st);
}

void trace_pre(cudaStream_t st, int family) {
  TraceState& t = g_trace;
  if (!t.on || (int)t.recs.size() >= t.cap) return;
  cudaEvent_t a = t.pool[2 * t.recs.size()];
  if (record(a, st) == cudaSuccess) {
    t.open_family = family;
    t.open_a = a;
    t.open_k = t.kernels;
  }
}

void trace_kernel() { ++g_trace.kernels; }

void trace_post(cudaStream_t st, double bytes) {
  TraceState& t = g_trace;
  if (!t.on || t.open_a == nullptr) return;
  cudaEvent_t b = t.pool[2 * t.recs.size() + 1];
  if (record(b, st) == cudaSuccess)
    t.recs.push_back(Rec{t.open_family, (int)(t.kernels - t.open_k), bytes, t.open_a, b});
  t.open_a = nullptr;
}

}  // namespace dfl

using namespace dfl;

extern "C" {

int dflash_trace_begin(int32_t max_launches) {
  TraceState& t = g_trace;
  if (max_launches <= 0 || max_launches > (1 << 20)) return DFLASH_ERR_INVALID_ARG;
  for (auto e : t.pool) cudaEventDestroy(e);
  t.pool.assign(2 * (size_t)max_launches, nullptr);
  for (auto& e : t.pool)
    if (cudaEventCreate(&e) != cudaSuccess) return DFLASH_ERR_CUDA;
  t.cap = max_launches;
  t.recs.clear();
  t.open_a = nullptr;
  t.on = true;
  return DFLASH_OK;
}

int dflash_trace_pause(void) {
  g_trace.on = false;
  return DFLASH_OK;
}

int dflash_trace_read(dflash_trace_stat* stats, int32_t n_stats) {
  TraceState& t = g_trace;
  if (!stats || n_stats < kTraceFamilies) return DFLASH_ERR_INVALID_ARG;
  for (int f = 0; f < kTraceFamilies; ++f) {
    memset(&stats[f], 0, sizeof(stats[f]));
    strncpy(stats[f].name, kFamilyNames[f], sizeof(stats[f].name) - 1);
  }
  for (const Rec& r : t.recs) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) {
      cudaGetLastError();
      return DFLASH_ERR_CUDA;
    }
    dflash_trace_stat& s = stats[r.family];
    s.launches += r.kernels;
    s.total_ms += ms;
    s.bytes += r.bytes;
  }
  return kTraceFamilies;
}

int dflash_trace_launches(float* ms, int32_t* family, int32_t n) {
  TraceState& t = g_trace;
  if (n < 0 || (n > 0 && (!ms || !family))) return DFLASH_ERR_INVALID_ARG;
  const int count = (int)t.recs.size();
  for (int i = 0; i < count && i < n; ++i) {
    float v = 0.f;
    if (cudaEventElapsedTime(&v, t.recs[i].a, t.recs[i].b) != cudaSuccess) {
      cudaGetLastError();
      return DFLASH_ERR_CUDA;
    }
    ms[i] = v;
    family[i] = t.recs[i].family;
  }
  return count;
}

int dflash_trace_end(void) {
  TraceState& t = g_trace;
  for (auto e : t.pool) cudaEventDestroy(e);
  t.pool.clear();
  t.recs.clear();
  t.on = false;
  t.cap = 0;
  return DFLASH_OK;
}

}  // extern "C"
