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
#include <cuda.h>
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

// Device address of the scratch area in the context current on this thread.
//
// Module addresses belong to a context.  The primary context of a device, a
// context the host created through the driver API and made current, and the
// primary context re-created after cudaDeviceReset each hold their own copy of
// the array at their own address.  The address is therefore looked up once per
// context (for most callers: once per device, in its primary context), with
// that context current, and cached under the context's unique ID, which the
// driver never hands out twice in a process; a call made in a context not seen
// before looks the address up again.  The lookup allocates nothing, but the
// first one in a context loads the library's device code into that context,
// so the first call in a context should come before any stream capture.

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

struct CtxApi {
  CtxGetCurrentFn get_current = nullptr;
  CtxGetIdFn get_id = nullptr;
};

const CtxApi& ctx_api() {
  static CtxApi api;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      api.get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      api.get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  return api;
}

// Unique ID of the context current on this thread; false if there is none.
bool current_ctx_id(const CtxApi& api, unsigned long long* id) {
  CUcontext ctx = nullptr;
  if (api.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return api.get_id(ctx, id) == CUDA_SUCCESS;
}

constexpr int kCacheSlots = 64;
struct CacheSlot {
  unsigned long long ctx_id;
  void* ptr;
};
std::mutex g_mu;
CacheSlot g_cache[kCacheSlots] = {};
int g_cache_next = 0;

eas_status lookup_error(cudaError_t e) {
  char msg[256];
  snprintf(msg, sizeof(msg), "cudaGetSymbolAddress(static scratch): %s", cudaGetErrorString(e));
  eas::set_last_error(msg);
  return EAS_ERR_CUDA;
}

eas_status static_scratch(void** out) {
  const CtxApi& api = ctx_api();
  if (!api.get_current || !api.get_id) {
    eas::set_last_error("cuCtxGetCurrent / cuCtxGetId unavailable from the driver");
    return EAS_ERR_CUDA;
  }
  unsigned long long id = 0;
  bool have_ctx = current_ctx_id(api, &id);
  std::lock_guard<std::mutex> lk(g_mu);
  if (have_ctx) {
    for (const CacheSlot& c : g_cache)
      if (c.ptr != nullptr && c.ctx_id == id) {
        *out = c.ptr;
        return EAS_OK;
      }
  }
  // set-up in this context: with no context current yet, the lookup makes the
  // current device's primary context current first
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
  if (e != cudaSuccess || p == nullptr) return lookup_error(e);
  if (!have_ctx) have_ctx = current_ctx_id(api, &id);
  if (have_ctx) {
    g_cache[g_cache_next] = CacheSlot{id, p};
    g_cache_next = (g_cache_next + 1) % kCacheSlots;
  }
  *out = p;
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
