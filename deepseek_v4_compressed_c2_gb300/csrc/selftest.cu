// Self-test of the bounded waits every pipelined kernel uses: one CTA waits
// on an mbarrier that nothing ever arrives on, through the same
// mbar_wait_bounded helper, and must give up after `polls` polls, report
// kFaultTimeout in the caller's fault counter and return -- no trap, no hang.
// A second warp waits on the same barrier and must notice the first one's
// abort flag and give up too.
#include "internal.cuh"
#include "tma.cuh"

namespace dsv4kv {

__global__ void bounded_wait_selftest_kernel(uint32_t polls, int* err, int* gave_up) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);       // count 1, and no thread ever arrives
    abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  if ((threadIdx.x & 31) == 0) {
    // the second waiter's own limit is 4x longer: it must leave through the
    // first one's abort flag (a single timeout fault), not its own limit
    const bool ok = mbar_wait_bounded(&bar, 0u, &abort_flag, err,
                                      threadIdx.x == 0 ? polls : 4u * polls);
    if (!ok) atomicAdd(gave_up, 1);
  }
}

cudaError_t launch_bounded_wait_selftest(uint32_t polls, int* err, int* gave_up,
                                         cudaStream_t stream) {
  bounded_wait_selftest_kernel<<<1, 64, 0, stream>>>(polls, err, gave_up);
  return cudaGetLastError();
}

}  // namespace dsv4kv
