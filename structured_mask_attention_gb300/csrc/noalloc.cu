// noalloc.cu -- a backward entry point for callers that cannot allocate
// device memory.
//
// Some callers have no way to obtain scratch memory for the library: plugin
// hosts that hand a library only its input and output buffers, runtimes that
// reserve all device memory up front and forbid further cudaMalloc, and
// latency-critical code that avoids cudaMalloc because it may synchronize the
// device.  bdlm_attn_bwd_noalloc serves them: it runs the ordinary backward
// (bdlm_attn_bwd) with its workspace placed in a fixed-size array in device
// global memory that this file declares, so the caller passes only inputs and
// outputs and the library calls no allocator.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>
#include <string>

#include "../../include/bdlm_attn.h"
#include "kernels.h"

namespace {

// Workspace of the backward: the status word plus the row statistic D of
// both streams, 2 * Hq * L fp32.  32 MiB covers Hq * L up to 4,194,272
// (e.g. 16 query heads at L = 131072, or 8 at L = 262144).
constexpr size_t kNoAllocScratchBytes = (size_t)32 << 20;

// Loaded with this file's module and held by every GPU that loads it until
// the process exits.  Host code must not pass &g_noalloc_scratch to a kernel:
// on the host the name is only a stand-in; the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// The array's device address, cached per device for the CUDA context it was
// looked up in.  A context is identified by the driver's context id, which
// is unique for the life of the process, so after cudaDeviceReset (a new
// primary context, in which the module and its array are loaded afresh) the
// address is looked up again instead of reusing a stale one.
struct ScratchSlot {
  unsigned long long ctx_id = 0;
  void* addr = nullptr;
};
std::mutex g_mu;
ScratchSlot g_slot[64];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Id of the current context, or 0 when the driver cannot say (then the
// address is looked up on every call: a lookup, never an allocation).
unsigned long long current_ctx_id() {
  static std::once_flag once;
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(f);
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  unsigned long long id = 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the scratch array on the current device.  The first call
// on a device (and the first after its context was re-created) looks it up
// with that device current; cudaGetSymbolAddress may load the library's
// device code then, which is why that first call belongs before any stream
// capture.
bdlm_status scratch_address(void** out, const char* who) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) {
    bdlm::set_last_error(std::string(who) + ": no current CUDA device (" + cudaGetErrorString(e) + ")");
    return BDLM_ERR_CUDA;
  }
  // (id 0: no context current yet, or the driver cannot say; the lookup
  // below then creates the device's primary context, and its id is read
  // afterwards)
  const unsigned long long id = current_ctx_id();
  std::lock_guard<std::mutex> lock(g_mu);
  ScratchSlot& slot = g_slot[dev];
  if (!slot.addr || id == 0 || slot.ctx_id != id) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
      slot = ScratchSlot{};
      bdlm::set_last_error(std::string(who) + ": cudaGetSymbolAddress failed (" + cudaGetErrorString(e) + ")");
      return BDLM_ERR_CUDA;
    }
    slot.addr = p;
    slot.ctx_id = id ? id : current_ctx_id();
  }
  *out = slot.addr;
  return BDLM_OK;
}

}  // namespace

extern "C" bdlm_status bdlm_attn_bwd_noalloc(const void* Qc, const void* Kc, const void* Vc, const void* Qn,
                                             const void* Kn, const void* Vn, const void* Oc, const void* On,
                                             const void* dOc, const void* dOn, const float* LSEc,
                                             const float* LSEn, int64_t L, int64_t B, int Hq, int Hkv, int d,
                                             float scale, void* dQc, void* dKc, void* dVc, void* dQn, void* dKn,
                                             void* dVn, bdlm_dtype g_dtype, bdlm_stream stream) {
  try {
    const size_t need = bdlm_workspace_size(BDLM_OP_BWD, L, B, Hq, Hkv, d, 1);
    if (need == 0) {
      // invalid shape: let the ordinary entry point report which check failed
      return bdlm_attn_bwd(Qc, Kc, Vc, Qn, Kn, Vn, Oc, On, dOc, dOn, LSEc, LSEn, L, B, Hq, Hkv, d, scale, dQc, dKc,
                           dVc, dQn, dKn, dVn, g_dtype, nullptr, 0, stream);
    }
    if (need > kNoAllocScratchBytes) {
      char buf[256];
      snprintf(buf, sizeof(buf),
               "bdlm_attn_bwd_noalloc: shape needs %zu bytes of scratch, above the fixed %zu-byte array "
               "(Hq * L must be <= %zu); use bdlm_attn_bwd with a caller workspace",
               need, kNoAllocScratchBytes, (kNoAllocScratchBytes - 256) / 8);
      bdlm::set_last_error(buf);
      return BDLM_ERR_WORKSPACE;
    }
    // a null or misaligned pointer: the ordinary entry point reports it (it
    // checks pointers before the workspace), before any device call here
    const void* ptrs[] = {Qc, Kc, Vc, Qn, Kn, Vn, Oc, On, dOc, dOn, LSEc, LSEn, dQc, dKc, dVc, dQn, dKn, dVn};
    for (const void* q : ptrs)
      if (!q || (reinterpret_cast<uintptr_t>(q) & 15u))
        return bdlm_attn_bwd(Qc, Kc, Vc, Qn, Kn, Vn, Oc, On, dOc, dOn, LSEc, LSEn, L, B, Hq, Hkv, d, scale, dQc,
                             dKc, dVc, dQn, dKn, dVn, g_dtype, nullptr, 0, stream);
    void* ws = nullptr;
    const bdlm_status s = scratch_address(&ws, "bdlm_attn_bwd_noalloc");
    if (s != BDLM_OK) return s;
    return bdlm_attn_bwd(Qc, Kc, Vc, Qn, Kn, Vn, Oc, On, dOc, dOn, LSEc, LSEn, L, B, Hq, Hkv, d, scale, dQc, dKc,
                         dVc, dQn, dKn, dVn, g_dtype, ws, kNoAllocScratchBytes, stream);
  } catch (...) {
    bdlm::set_last_error("bdlm_attn_bwd_noalloc: internal exception");
    return BDLM_ERR_INVALID_ARG;
  }
}

extern "C" bdlm_status bdlm_sync_status_noalloc(bdlm_stream stream) {
  try {
    void* ws = nullptr;
    const bdlm_status s = scratch_address(&ws, "bdlm_sync_status_noalloc");
    if (s != BDLM_OK) return s;
    return bdlm_sync_status(ws, stream);
  } catch (...) {
    bdlm::set_last_error("bdlm_sync_status_noalloc: internal exception");
    return BDLM_ERR_INVALID_ARG;
  }
}

extern "C" bdlm_status bdlm_watchdog_selftest_noalloc(uint32_t limit_us, bdlm_stream stream) {
  try {
    void* ws = nullptr;
    const bdlm_status s = scratch_address(&ws, "bdlm_watchdog_selftest_noalloc");
    if (s != BDLM_OK) return s;
    return bdlm_watchdog_selftest(ws, kNoAllocScratchBytes, limit_us, stream);
  } catch (...) {
    bdlm::set_last_error("bdlm_watchdog_selftest_noalloc: internal exception");
    return BDLM_ERR_INVALID_ARG;
  }
}
