// Self-test of the bounded waits every pipelined kernel uses: one CTA waits
// on an mbarrier that nothing ever arrives on, through the same
// mbar_wait_bounded helper, and must give up after `polls` polls, report
// kFaultTimeout in the caller's fault counter and return -- no trap, no hang.
// A second warp waits on the same barrier and must notice the first one's
// abort flag and give up too.
#include "internal.cuh"
#include "quant.cuh"
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

// The FP4 quantizer's division x / s (s a positive e4m3 value): the fast
// reciprocal-and-correction form next to the IEEE division, for a test that
// compares them bit for bit.  Element i uses the divisor e4m3 code
// scale_codes[i].
__global__ void fp4_quotient_selftest_kernel(const float* x, const unsigned char* scale_codes,
                                             long long n, float* q_fast, float* q_ieee) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const float s = e4m3_to_f32(scale_codes[i]);
    q_fast[i] = div_by_recip(x[i], s, __frcp_rn(s));
    q_ieee[i] = __fdiv_rn(x[i], s);
  }
}

cudaError_t launch_fp4_quotient_selftest(const float* x, const unsigned char* scale_codes,
                                         long long n, float* q_fast, float* q_ieee,
                                         cudaStream_t stream) {
  const long long want = (n + 255) / 256;
  const int grid = (int)(want < 4096 ? want : 4096);
  fp4_quotient_selftest_kernel<<<grid, 256, 0, stream>>>(x, scale_codes, n, q_fast, q_ieee);
  return cudaGetLastError();
}

}  // namespace dsv4kv
