// kvp_selftest.cu -- exercises the bounded mbarrier wait that every pipeline
// wait of the library goes through: barriers that nothing arrives on, a
// short limit, the shared abort flag that ends the other waits of the CTA,
// and the status word the host reads afterwards.  The GPU and the context
// stay usable; nothing faults or hangs.
#include "kvp_device.cuh"
#include "kvp_internal.h"

namespace kvp {
namespace {

__global__ void selftest_wait_kernel(int32_t* status, uint64_t limit_ns) {
  using namespace dev;
  // two barriers, one arrival expected on each; none comes.  Warp 0 waits
  // with the caller's limit, warp 1 with the default 2 s; both poll one abort
  // flag, so warp 1 gives up right after warp 0 does (within 16 tries), the
  // way every role of a pipeline stops once one of its waits has failed.
  __shared__ uint64_t bar[2];
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar[0]), 1);
    mbar_init(smem_addr(&bar[1]), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    const bool ok = mbar_wait_bounded(smem_addr(&bar[warp]), 0,
                                      warp == 0 ? limit_ns : kWaitTimeoutNs, &abort_flag);
    if (!ok) set_status(status, kErrTimeout);
  }
}

}  // namespace

cudaError_t launch_selftest_wait(int32_t* status, uint64_t limit_ns, cudaStream_t s) {
  selftest_wait_kernel<<<1, 64, 0, s>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace kvp
