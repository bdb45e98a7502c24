// Self-test of the device failure path: a bounded wait that nothing can complete.
//
// Every kernel of this library that waits on the device (an mbarrier phase of a TMA pipeline, the
// publication flag of the CTA-to-CTA carry) gives up after a time limit, records kStatusTimeout in a
// status word and returns, so that the failure reaches the host through ssm_device_status() while
// the CUDA context stays usable.  Those waits never run out in correct operation; this kernel makes
// each kind run out on purpose, with the same helpers and the same status word protocol, so that the
// path can be tested without faulting, trapping or hanging a GPU.
//
// In the checked build a second kernel asks checked() for an index one past a 32-element buffer: the
// check redirects the store to its sink and records kStatusBounds, which the next
// ssm_device_status() reports as SSM_ERR_CHECK.  The ordinary build has no such kernel.
#include "internal.h"
#include "ssm_device.cuh"

namespace ssm {
namespace {

__device__ unsigned int g_selftest_status = 0;
__device__ unsigned int g_never_set = 0;   // a flag that no kernel writes

__global__ void bounded_wait_selftest_kernel(int which, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  if (which == 0) {
    // an mbarrier expecting one arrival that never comes: phase 0 does not complete
    mbar_init(&bar, 1);
    fence_mbar_init();
    (void)mbar_wait_bounded(&bar, 0u, &g_selftest_status, limit_ns);
  } else {
    // a publication flag that nothing sets, polled as the carry wait polls its predecessor's flag
    const uint64_t t0 = globaltimer_ns();
    while (true) {
      unsigned v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(&g_never_set) : "memory");
      if (v != 0u) break;
      if (globaltimer_ns() - t0 > limit_ns) {
        atomicOr(&g_selftest_status, kStatusTimeout);
        break;
      }
      __nanosleep(1000);
    }
  }
}

#if SSM_CHECK
__device__ float g_check_probe[32];

__global__ void index_check_selftest_kernel() {
  *checked(g_check_probe, 32 + static_cast<int64_t>(threadIdx.x), 32) = 1.0f;
}
#endif

}  // namespace

cudaError_t selftest_index_check_launch(cudaStream_t stream) {
#if SSM_CHECK
  index_check_selftest_kernel<<<1, 1, 0, stream>>>();
  return cudaGetLastError();
#else
  (void)stream;
  return cudaErrorNotSupported;
#endif
}

cudaError_t selftest_bounded_wait_launch(int which, unsigned long long limit_ns, cudaStream_t stream) {
  bounded_wait_selftest_kernel<<<1, 32, 0, stream>>>(which, limit_ns);
  return cudaGetLastError();
}

cudaError_t selftest_status_read_and_clear(unsigned int* out) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_selftest_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  e = cudaMemcpyToSymbol(g_selftest_status, &zero, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  unsigned int c = 0;
  e = tu_check_read_and_clear(&c);
  *out |= c;
  return e;
}

}  // namespace ssm
