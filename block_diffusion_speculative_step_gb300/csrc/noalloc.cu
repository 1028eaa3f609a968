// noalloc.cu -- dflash_verify_accept_noalloc: verification + acceptance with
// its scratch in a fixed device array of the library instead of a caller
// workspace, for callers that cannot allocate device memory when they call.
#include <stdio.h>

#include <mutex>

#include "../../include/dflash.h"
#include "common.cuh"

namespace dfl {
int abi_fail(int code, const char* msg);
int verify_check(const dflash_verify_args* a, const char* who);
}

namespace {

constexpr size_t kStaticScratchBytes = size_t(8) << 20;  // 8 MiB
constexpr int kMaxDevices = 64;

// The scratch itself.  In host code this name is only a stand-in for the
// symbol: its device address comes from cudaGetSymbolAddress, per device.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of the array on the current device, looked up once per device.
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return dfl::abi_fail(DFLASH_ERR_CUDA, "dflash_verify_accept_noalloc: no current CUDA device");
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return dfl::abi_fail(DFLASH_ERR_CUDA, "dflash_verify_accept_noalloc: cudaGetSymbolAddress failed");
    }
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return DFLASH_OK;
}

}  // namespace

extern "C" int dflash_verify_accept_noalloc(const dflash_verify_args* a, int32_t* status_out,
                                            dflash_stream_t stream) {
  // the checks of dflash_verify_accept first, so that bad arguments report
  // DFLASH_ERR_INVALID_ARG as they do there, never a scratch size
  int rc = dfl::verify_check(a, "dflash_verify_accept_noalloc");
  if (rc) return rc;
  const size_t need = dflash_workspace_bytes(DFLASH_OP_VERIFY, a);
  if (need > kStaticScratchBytes) {
    char msg[200];
    snprintf(msg, sizeof(msg),
             "dflash_verify_accept_noalloc: these shapes need %zu bytes of scratch; the static scratch holds "
             "%zu (8 MiB) -- use dflash_verify_accept with a workspace",
             need, kStaticScratchBytes);
    return dfl::abi_fail(DFLASH_ERR_WORKSPACE, msg);
  }
  void* ws = nullptr;
  rc = scratch_address(&ws);
  if (rc) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  // status word and arrival counters must start at zero
  if (cudaMemsetAsync(ws, 0, dfl::kReservedBytes, st) != cudaSuccess) {
    cudaGetLastError();
    return dfl::abi_fail(DFLASH_ERR_CUDA, "dflash_verify_accept_noalloc: clearing the scratch header failed");
  }
  rc = dflash_verify_accept(a, ws, kStaticScratchBytes, stream);
  if (rc) return rc;
  if (status_out && cudaMemcpyAsync(status_out, ws, sizeof(int32_t), cudaMemcpyDeviceToDevice, st) != cudaSuccess) {
    cudaGetLastError();
    return dfl::abi_fail(DFLASH_ERR_CUDA, "dflash_verify_accept_noalloc: copying the status word failed");
  }
  return DFLASH_OK;
}
