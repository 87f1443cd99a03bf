// A kernel that exercises the bounded-wait error path on its own: one warp
// waits on a shared-memory mbarrier that nothing arrives at, through the same
// bounded wait the layer's kernels use, with a caller-chosen wall-clock
// limit.  When the limit passes, the wait records kErrTimeout in the handle's
// error flag and the kernel returns; no TMA copy, MMA or tensor memory is in
// flight, so nothing else needs to unwind.
#include "common.cuh"
#include "lmoe_internal.h"

namespace lmoe {
namespace {

__global__ void wait_timeout_probe_kernel(int* err, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, err, kErrTimeout, limit_ns);   // nothing arrives: times out
  __syncwarp();
}

}  // namespace

cudaError_t launch_wait_timeout_probe(int* err, unsigned long long limit_ns, cudaStream_t s) {
  wait_timeout_probe_kernel<<<1, 32, 0, s>>>(err, limit_ns);
  return cudaGetLastError();
}

}  // namespace lmoe
