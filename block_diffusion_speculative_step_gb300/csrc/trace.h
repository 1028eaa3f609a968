// trace.h -- kernel-launch tracing hooks used by the ABI layer.
#pragma once
#include <cuda_runtime.h>

namespace dfl {

enum TraceFamily : int {
  TF_EMBED = 0,
  TF_RMSNORM = 1,
  TF_GEMM_SIMT = 2,
  TF_GEMM_TC = 3,
  TF_ATTN = 4,
  TF_HEAD = 5,
  TF_PATH = 6,
  TF_ROPE = 7,
  TF_TAP = 8,
  TF_CONVERT = 9,
  TF_SAMPLE = 10,
  TF_CONV = 11,
  TF_PAGE = 12,
  kTraceFamilies = 13
};

void trace_pre(cudaStream_t st, int family);
void trace_post(cudaStream_t st, double bytes);
// Called at every kernel launch: a traced call counts the kernels it launched.
void trace_kernel();

}  // namespace dfl
