// Kernel parameters and device helpers shared between the kernel files and
// the C-ABI layer (the launchers are declared in launchers.cuh).  Everything
// here is device-pointer plumbing; argument checks happen in capi.cu before
// any launcher is reached.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace dsv4kv {

// request slots per compress_store call (the plan lives in shared memory)
constexpr int kMaxSlots = 4096;

struct StoreParams {
  const __nv_bfloat16* rows;   // [n_rows, row_stride]
  long long n_rows;
  long long row_stride;        // elements
  const __nv_bfloat16* score;  // nullptr: rows + 512 (fused | kv | score |)
  long long score_stride;
  const int* ext;              // [2, n_slots]
  int n_slots;
  const int* page_table;       // [n_slots, max_pages] or nullptr (out_loc given)
  int max_pages;
  int page_bits;
  const __nv_bfloat16* norm_w; // [512] or nullptr
  float eps;
  const float* freqs;          // [max_pos, 64] or nullptr
  int max_pos;
  const int* out_loc;          // [n_out] or nullptr
  int n_out;
  uint8_t* pool;
  long long pool_rows;
  __nv_bfloat16* latent_out;   // [n_out, 512] or nullptr
  float* prequant_out;         // [n_out, 512] or nullptr
  int* err;                    // device fault counter or nullptr
  const int* start_pos;        // [n_slots] position of each slot's first new token, or nullptr (0)
  __nv_bfloat16* ring;         // [n_slots, ring_size, 1024] pair-state ring (ratio 2) or nullptr
  int ring_size;
};

// Launch with programmatic stream serialization: the kernel may be scheduled
// while the previous kernel in the stream finishes; it waits
// (grid_dependency_wait) before touching global memory.
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kern)(Params...), int grid, int block, size_t smem,
                             cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Streaming 16-byte global load that bypasses L1 (inputs read exactly once).
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

__device__ __forceinline__ uint2 ld_stream_v2(const void* p) {
  uint2 v;
  asm("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ld_stream_u32(const void* p) {
  uint32_t v;
  asm("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// Multiprocessor count of the current device (cached), for persistent grids.
int device_sm_count();

}  // namespace dsv4kv
