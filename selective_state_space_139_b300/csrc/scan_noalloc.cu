// Prefill scan for callers that cannot allocate device memory.
//
// The regular entry point, ssm_scan_fwd, asks the caller for a device workspace whenever its
// schedule needs scratch (the carries of the balanced schedule, the chunk aggregates of the chunked
// one).  Some callers have no way to provide it: code that runs where cudaMalloc is forbidden or
// unavailable (inside a host callback or a driver/plugin hook that must not allocate, a process
// whose allocator is owned by another framework, memory-capped sandboxes), or code that cannot
// afford an allocation on its latency path.  ssm_scan_fwd_noalloc serves them: its scratch is a
// fixed array in this library's device memory, reserved when the library's module loads on a GPU
// and held until the process exits.  The call itself allocates nothing.
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "internal.h"
#include "ssm.h"

namespace {

// Fixed scratch shared by every ssm_scan_fwd_noalloc call on a device.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;   // 8 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// The array's device address, looked up once per CUDA context with that context current.  The
// context is identified by its driver-assigned unique id, which is never reused: after a
// cudaDeviceReset, or in another context of the same device, the module is loaded anew and the
// array may sit elsewhere, so a new id triggers a new lookup.
struct ScratchEntry {
  unsigned long long ctx_id;
  void* addr;
};
constexpr int kCacheEntries = 64;
ScratchEntry g_cache[kCacheEntries] = {};
int g_cache_next = 0;
std::mutex g_scratch_mu;

using PfnCtxGetCurrent = CUresult (*)(CUcontext*);
using PfnCtxGetId = CUresult (*)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current context, or 0 if there is none or it cannot be read.
unsigned long long current_context_id() {
  static PfnCtxGetCurrent get_current = nullptr;
  static PfnCtxGetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PfnCtxGetCurrent>(f);
    else
      cudaGetLastError();
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PfnCtxGetId>(f);
    else
      cudaGetLastError();
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// The array's device address in the current context (set-up on the first call in a context).
cudaError_t scratch_address(void** out) {
  const unsigned long long id = current_context_id();
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (id != 0) {
    for (const ScratchEntry& e : g_cache)
      if (e.ctx_id == id) {
        *out = e.addr;
        return cudaSuccess;
      }
  }
  // the host-side name of the array is not a device pointer: translate it with the context current
  void* addr = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&addr, g_noalloc_scratch);
  if (e != cudaSuccess) return e;
  // the runtime creates the context on its first call: the id may only be readable now
  const unsigned long long id2 = id != 0 ? id : current_context_id();
  if (id2 != 0) {
    g_cache[g_cache_next] = ScratchEntry{id2, addr};
    g_cache_next = (g_cache_next + 1) % kCacheEntries;
  }
  *out = addr;
  return cudaSuccess;
}

}  // namespace

extern "C" {

size_t ssm_scan_fwd_noalloc_max_scratch(void) { return kNoAllocScratchBytes; }

ssm_status ssm_scan_fwd_noalloc(const void* u, const void* delta, const float* A, const void* B, const void* C,
                                const float* D, const void* z, const float* delta_bias, int softplus_flag, void* y,
                                float* last_state, int batch, int dim, int dstate, int64_t seqlen,
                                ssm_dtype io_dtype, const ssm_scan_options* opts, cudaStream_t stream) {
  // sizes whose schedule needs more scratch than the fixed array are refused before anything else
  const size_t need = ssm_scan_fwd_workspace_size_ex(batch, dim, dstate, seqlen, io_dtype, opts);
  if (need > kNoAllocScratchBytes) {
    ssm::set_last_error("ssm_scan_fwd_noalloc: this shape needs %zu bytes of scratch, above the fixed %zu bytes; "
                        "use ssm_scan_fwd with a caller workspace",
                        need, kNoAllocScratchBytes);
    return SSM_ERR_UNSUPPORTED;
  }
  void* scratch = nullptr;
  const cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) {
    ssm::set_last_error("ssm_scan_fwd_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    return SSM_ERR_CUDA;
  }
  // The existing entry point does the rest: its schedules write every scratch word they read in the
  // same call (the balanced schedule clears its flags first; the chunked one writes its aggregates
  // and carries before reading them), so the previous call's contents never leak into a result.
  return ssm_scan_fwd_ex(u, delta, A, B, C, D, z, delta_bias, softplus_flag, y, last_state, batch, dim, dstate,
                         seqlen, io_dtype, scratch, kNoAllocScratchBytes, opts, stream);
}

}  // extern "C"
