// kvp_selftest.cu -- exercises the bounded mbarrier wait that every pipeline
// wait of the library goes through: a barrier that nothing arrives on, a
// short limit, and the status word the host reads afterwards.  The GPU and
// the context stay usable; nothing faults or hangs.
#include "kvp_device.cuh"
#include "kvp_internal.h"

namespace kvp {
namespace {

__global__ void selftest_wait_kernel(int32_t* status, uint64_t limit_ns) {
  using namespace dev;
  __shared__ uint64_t bar;  // one arrival expected; none comes
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait_bounded(smem_addr(&bar), 0, limit_ns))
    set_status(status, kErrTimeout);
}

}  // namespace

cudaError_t launch_selftest_wait(int32_t* status, uint64_t limit_ns, cudaStream_t s) {
  selftest_wait_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace kvp
