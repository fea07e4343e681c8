// Allocation-free forward: eas_lmhead_fwd with its scratch in a static device
// array instead of a caller-provided workspace.
//
// Some callers cannot allocate device memory when they need the forward:
// a host that hands every byte of the GPU to its own pool allocator at start-up
// and gives libraries no way to draw from it, an embedded or real-time host
// that forbids allocation once it is running, or a plugin interface that passes
// only input and output buffers.  This entry point serves them with a fixed
// scratch area compiled into the library: every GPU that loads the library
// reserves it until the process exits.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "../../include/eas.h"
#include "eas_kernels.h"

namespace {

constexpr size_t kStaticScratchBytes = EAS_STATIC_SCRATCH_BYTES;

// The scratch area.  In host code this name is only a stand-in for the
// device symbol: its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch area on the current device, looked up once
// per device (with that device current) and cached.
eas_status static_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof(msg), "cudaGetDevice: %s", cudaGetErrorString(e));
    eas::set_last_error(msg);
    return EAS_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    eas::set_last_error("device ordinal out of range for the static scratch table");
    return EAS_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || p == nullptr) {
      char msg[256];
      snprintf(msg, sizeof(msg), "cudaGetSymbolAddress(static scratch): %s",
               cudaGetErrorString(e));
      eas::set_last_error(msg);
      return EAS_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return EAS_OK;
}

}  // namespace

extern "C" {

eas_status eas_lmhead_fwd_noalloc(const void* hidden, const void* weight,
                                  const int32_t* targets, const uint8_t* mask,
                                  const int32_t* spans, const int32_t* num_spans, int64_t cap,
                                  int64_t T, int64_t H, int64_t V, eas_dtype dtype,
                                  uint32_t flags, float* logprob, float* entropy, float* lse,
                                  void* stream) {
  const size_t need = eas::lmhead_fwd_workspace_bytes(T, H, V, static_cast<int>(dtype));
  if (need > kStaticScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "eas_lmhead_fwd_noalloc: T=%lld H=%lld V=%lld needs %zu bytes of scratch; the "
             "static scratch holds %zu (use eas_lmhead_fwd with a workspace)",
             static_cast<long long>(T), static_cast<long long>(H), static_cast<long long>(V),
             need, kStaticScratchBytes);
    eas::set_last_error(msg);
    return EAS_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  const eas_status st = static_scratch(&scratch);
  if (st != EAS_OK) return st;
  return eas_lmhead_fwd(hidden, weight, targets, mask, spans, num_spans, cap, T, H, V, dtype,
                        flags, logprob, entropy, lse, scratch, kStaticScratchBytes, stream);
}

}  // extern "C"
