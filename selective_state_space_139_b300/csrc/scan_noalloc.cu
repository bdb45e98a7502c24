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
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "internal.h"
#include "ssm.h"

namespace {

// Fixed scratch shared by every ssm_scan_fwd_noalloc call on a device.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;   // 8 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// The array's device address, looked up once per device with that device current.
constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

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
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    ssm::set_last_error("ssm_scan_fwd_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
    return SSM_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    ssm::set_last_error("ssm_scan_fwd_noalloc: device ordinal %d above %d", dev, kMaxDevices - 1);
    return SSM_ERR_UNSUPPORTED;
  }
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
      // first call on this device: translate the symbol to its device address (the host-side name
      // of the array is not a device pointer)
      void* addr = nullptr;
      e = cudaGetSymbolAddress(&addr, g_noalloc_scratch);
      if (e != cudaSuccess) {
        ssm::set_last_error("ssm_scan_fwd_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        return SSM_ERR_CUDA;
      }
      g_scratch_addr[dev] = addr;
    }
    scratch = g_scratch_addr[dev];
  }
  // The existing entry point does the rest: its schedules write every scratch word they read in the
  // same call (the balanced schedule clears its flags first; the chunked one writes its aggregates
  // and carries before reading them), so the previous call's contents never leak into a result.
  return ssm_scan_fwd_ex(u, delta, A, B, C, D, z, delta_bias, softplus_flag, y, last_state, batch, dim, dstate,
                         seqlen, io_dtype, scratch, kNoAllocScratchBytes, opts, stream);
}

}  // extern "C"
