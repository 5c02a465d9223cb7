// selftest.cu -- exercises the bounded-wait path of the kernels without a fault.
//
// One thread initialises an mbarrier that nothing ever arrives on and waits on
// it with the library's bounded wait (mbar_wait_for, the loop every kernel's
// waits use), for a caller-chosen limit.  The wait gives up, the kernel
// records ATTN_ERR_TIMEOUT in the device status word exactly as a kernel whose
// producer had stalled would, and it returns; the context stays usable.
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

__global__ void wait_selftest_kernel(uint64_t limit_ns, int* status, uint64_t* waited_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  ptx::mbar_init(&bar, 1);
  ptx::fence_mbar_init();
  const uint64_t t0 = ptx::globaltimer();
  const bool ok = ptx::mbar_wait_for(&bar, 0, limit_ns);
  if (waited_ns != nullptr) *waited_ns = ptx::globaltimer() - t0;
  if (!ok && status != nullptr) atomicCAS(status, 0, ATTN_ERR_TIMEOUT);
}

}  // namespace

cudaError_t launch_wait_selftest(uint64_t limit_ns, int* status, uint64_t* waited_ns,
                                 cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns, status, waited_ns);
  return cudaGetLastError();
}

}  // namespace attn
