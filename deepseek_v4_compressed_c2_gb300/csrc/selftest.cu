// Self-test of the bounded waits every pipelined kernel uses: one CTA waits
// on an mbarrier that nothing ever arrives on, through the same
// mbar_wait_bounded helper, and must give up after `polls` polls, report
// kFaultTimeout in the caller's fault counter and return -- no trap, no hang.
// A second warp waits on the same barrier and must notice the first one's
// abort flag and give up too.
#include "internal.cuh"
#include "launchers.cuh"
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
  // elements 2j and 2j + 1 go through the paired form used by the FP4 store,
  // each with its own divisor
  const long long pairs = (n + 1) / 2;
  for (long long j = (long long)blockIdx.x * blockDim.x + threadIdx.x; j < pairs;
       j += (long long)gridDim.x * blockDim.x) {
    const long long i = 2 * j;
    const bool has0 = i < n, has1 = i + 1 < n;
    const uint32_t c0 = has0 ? scale_codes[i] : 1u, c1 = has1 ? scale_codes[i + 1] : 1u;
    const float s0 = e4m3_to_f32(c0), s1 = e4m3_to_f32(c1);
    const float y0 = e4m3_recip(s0), y1 = e4m3_recip(s1);
    float a, b;
    f2_split(div2_by_recip(f2(has0 ? x[i] : 0.f, has1 ? x[i + 1] : 0.f), f2(-s0, -s1), f2(y0, y1)),
             a, b);
    if (has0) {
      q_fast[i] = a;
      q_ieee[i] = __fdiv_rn(x[i], s0);
    }
    if (has1) {
      q_fast[i + 1] = b;
      q_ieee[i + 1] = __fdiv_rn(x[i + 1], s1);
    }
  }
}

// The FP4 quantizer's reciprocal of an e4m3 value next to the IEEE
// reciprocal: element i is the value of code codes[i].
__global__ void e4m3_recip_selftest_kernel(const unsigned char* codes, long long n, float* y_fast,
                                           float* y_ieee) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const float s = e4m3_to_f32(codes[i]);
    y_fast[i] = e4m3_recip(s);
    y_ieee[i] = __frcp_rn(s);
  }
}

cudaError_t launch_e4m3_recip_selftest(const unsigned char* codes, long long n, float* y_fast,
                                       float* y_ieee, cudaStream_t stream) {
  const long long want = (n + 255) / 256;
  const int grid = (int)(want < 1024 ? want : 1024);
  e4m3_recip_selftest_kernel<<<grid, 256, 0, stream>>>(codes, n, y_fast, y_ieee);
  return cudaGetLastError();
}

cudaError_t launch_fp4_quotient_selftest(const float* x, const unsigned char* scale_codes,
                                         long long n, float* q_fast, float* q_ieee,
                                         cudaStream_t stream) {
  const long long want = ((n + 1) / 2 + 255) / 256;
  const int grid = (int)(want < 4096 ? want : 4096);
  fp4_quotient_selftest_kernel<<<grid, 256, 0, stream>>>(x, scale_codes, n, q_fast, q_ieee);
  return cudaGetLastError();
}

}  // namespace dsv4kv
