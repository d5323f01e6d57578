// Failure-path self-test of the bounded device waits (moe_selftest_wait_timeout).
//
// One CTA of two warps waits on a shared-memory mbarrier that nothing ever
// completes, through the same bounded wait the layer's kernels use.  Warp 0
// waits with the caller's short limit and gives up first: it sets the shared
// abort flag and bit 0 of the status words.  Warp 1 waits with the layer's ~2 s
// limit and must leave through the abort flag, as the other roles of a GEMM
// kernel do when one of them times out.  No memory beyond the status words and
// one counter is touched, nothing faults, and the context stays usable.
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"
#include "sm100_ptx.cuh"

namespace gbmoe {

using namespace sm100;

constexpr long long kLayerWaitLimit = 4000000000LL;  // the GEMM kernels' limit (~2 s of SM clocks)

__global__ void __launch_bounds__(64) wait_timeout_kernel(DeviceStatus* status, long long limit, int32_t* gave_up) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    status->bad_ids = 0;
    status->flags = 0;
    *gave_up = 0;
    fence_barrier_init();
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    volatile int* abort = &abort_flag;
    const bool ok = mbar_wait(&bar, 0, abort, status, warp == 0 ? limit : kLayerWaitLimit);
    if (!ok) atomicAdd(gave_up, 1);
  }
}

cudaError_t launch_wait_timeout(DeviceStatus* status, long long limit, int32_t* gave_up, cudaStream_t s) {
  wait_timeout_kernel<<<1, 64, 0, s>>>(status, limit, gave_up);
  return cudaGetLastError();
}

}  // namespace gbmoe
