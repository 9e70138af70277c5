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

std::mutex g_mu;
void* g_scratch_addr[64] = {};

// Device address of the scratch array on the current device, looked up once
// per device with that device current.
bdlm_status scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) {
    bdlm::set_last_error(std::string("bdlm_attn_bwd_noalloc: no current CUDA device (") + cudaGetErrorString(e) + ")");
    return BDLM_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
      bdlm::set_last_error(std::string("bdlm_attn_bwd_noalloc: cudaGetSymbolAddress failed (") +
                           cudaGetErrorString(e) + ")");
      return BDLM_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
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
    void* ws = nullptr;
    const bdlm_status s = scratch_address(&ws);
    if (s != BDLM_OK) return s;
    return bdlm_attn_bwd(Qc, Kc, Vc, Qn, Kn, Vn, Oc, On, dOc, dOn, LSEc, LSEn, L, B, Hq, Hkv, d, scale, dQc, dKc,
                         dVc, dQn, dKn, dVn, g_dtype, ws, kNoAllocScratchBytes, stream);
  } catch (...) {
    bdlm::set_last_error("bdlm_attn_bwd_noalloc: internal exception");
    return BDLM_ERR_INVALID_ARG;
  }
}
