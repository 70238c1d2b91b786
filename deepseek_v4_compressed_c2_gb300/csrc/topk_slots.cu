// Request-local top-k compressed ids -> physical pool slots, plus the count
// of valid slots per row.
//
// flashinfer_sparse.py, _compressed_topk_to_slots (single-rank branch,
// compute_global_topk_indices_and_lens): the indexer's request-local ids map
// through the request's block table; compressed pages hold
// block_size // compress_ratio states (here 2^page_bits rows); empty entries
// become -1; CUDA-graph padding rows (is_valid_token == 0) attend nothing.
//
#include "internal.cuh"
#include "launchers.cuh"

namespace dsv4kv {

constexpr int kTopkThreads = 512;

__device__ __forceinline__ int topk_slot(int id, bool tok_ok, int r, const int* __restrict__ page_table,
                                         int max_pages, int page_bits, unsigned mask, int* err) {
  if (!tok_ok || id < 0) return -1;
  const int lp = id >> page_bits;
  if (lp >= max_pages) {
    if (err) atomicAdd(err, 1);
    return -1;
  }
  // 64-bit slot: a negative entry or a slot past int32 is no page (fault)
  const int phys = page_table[(long long)r * max_pages + lp];
  const long long slot = phys < 0 ? -1LL : ((long long)phys << page_bits) | ((unsigned)id & mask);
  if (slot < 0 || slot > 2147483647LL) {
    if (err) atomicAdd(err, 1);
    return -1;
  }
  return (int)slot;
}

// One CTA per token row; each thread maps 4 consecutive entries with 16-byte
// loads and stores when the rows are 16-byte aligned (k % 4 == 0 and aligned
// base pointers), so a row of 2048 ids is one pass.
__global__ void __launch_bounds__(kTopkThreads)
topk_to_slots_kernel(const int* __restrict__ topk, int n_tok, int k,
                     const int* __restrict__ token_to_req, const unsigned char* __restrict__ is_valid,
                     const int* __restrict__ page_table, int n_req, int max_pages, int page_bits,
                     int* __restrict__ slots, int* __restrict__ lens, int* err) {
  __shared__ int s_cnt[kTopkThreads / 32];
  const unsigned mask = (1u << page_bits) - 1u;
  const bool vec = (k & 3) == 0 && ((reinterpret_cast<uintptr_t>(topk) | reinterpret_cast<uintptr_t>(slots)) & 15) == 0;
  for (int t = blockIdx.x; t < n_tok; t += gridDim.x) {
    const int r = token_to_req[t];
    const bool bad_req = r < 0 || r >= n_req;
    const bool tok_ok = !bad_req && (is_valid == nullptr || is_valid[t] != 0);
    if (bad_req && threadIdx.x == 0 && err) atomicAdd(err, 1);
    int cnt = 0;
    const long long rowoff = (long long)t * k;
    if (vec) {
      const int4* in4 = reinterpret_cast<const int4*>(topk + rowoff);
      int4* out4 = reinterpret_cast<int4*>(slots + rowoff);
      for (int c = threadIdx.x; c < (k >> 2); c += blockDim.x) {
        const int4 id = __ldg(in4 + c);
        int4 sl;
        sl.x = topk_slot(id.x, tok_ok, r, page_table, max_pages, page_bits, mask, err);
        sl.y = topk_slot(id.y, tok_ok, r, page_table, max_pages, page_bits, mask, err);
        sl.z = topk_slot(id.z, tok_ok, r, page_table, max_pages, page_bits, mask, err);
        sl.w = topk_slot(id.w, tok_ok, r, page_table, max_pages, page_bits, mask, err);
        out4[c] = sl;
        cnt += (sl.x >= 0) + (sl.y >= 0) + (sl.z >= 0) + (sl.w >= 0);
      }
    } else {
      for (int c = threadIdx.x; c < k; c += blockDim.x) {
        const int sl = topk_slot(topk[rowoff + c], tok_ok, r, page_table, max_pages, page_bits, mask, err);
        slots[rowoff + c] = sl;
        cnt += sl >= 0;
      }
    }
    if (lens) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
      if ((threadIdx.x & 31) == 0) s_cnt[threadIdx.x >> 5] = cnt;
      __syncthreads();
      if (threadIdx.x == 0) {
        int sum = 0;
        for (int w = 0; w < kTopkThreads / 32; ++w) sum += s_cnt[w];
        lens[t] = sum;
      }
      __syncthreads();
    }
  }
}

cudaError_t launch_topk_to_slots(const int* topk, int n_tok, int k, const int* token_to_req,
                                 const unsigned char* is_valid, const int* page_table, int n_req,
                                 int max_pages, int page_bits, int* slots, int* lens, int* err,
                                 cudaStream_t stream) {
  const int grid = n_tok < 65535 * 4 ? n_tok : 65535 * 4;
  topk_to_slots_kernel<<<grid, kTopkThreads, 0, stream>>>(topk, n_tok, k, token_to_req, is_valid,
                                                          page_table, n_req, max_pages, page_bits,
                                                          slots, lens, err);
  return cudaGetLastError();
}

// Short-context ids (sglang PR #39652's test table: fill_all_compressed_indices;
// flashinfer_sparse.py: the "short-context bypass" of the indexer): every
// compressed row a token can see is selected, out[t][j] = j for
// j < min(lens[t], k), -1 after.  One CTA per token row, 4 entries per thread
// with 16-byte stores when the rows are 16-byte aligned.
__global__ void __launch_bounds__(kTopkThreads)
fill_all_indices_kernel(int* __restrict__ out, int n_tok, int k, const int* __restrict__ lens) {
  const bool vec = (k & 3) == 0 && (reinterpret_cast<uintptr_t>(out) & 15) == 0;
  for (int t = blockIdx.x; t < n_tok; t += gridDim.x) {
    const int len = __ldg(lens + t);
    const long long rowoff = (long long)t * k;
    if (vec) {
      int4* out4 = reinterpret_cast<int4*>(out + rowoff);
      for (int c = threadIdx.x; c < (k >> 2); c += blockDim.x) {
        const int j = 4 * c;
        out4[c] = make_int4(j < len ? j : -1, j + 1 < len ? j + 1 : -1, j + 2 < len ? j + 2 : -1,
                            j + 3 < len ? j + 3 : -1);
      }
    } else {
      for (int j = threadIdx.x; j < k; j += blockDim.x) out[rowoff + j] = j < len ? j : -1;
    }
  }
}

cudaError_t launch_fill_all_indices(int* out, int n_tok, int k, const int* lens,
                                    cudaStream_t stream) {
  const int grid = n_tok < 65535 * 4 ? n_tok : 65535 * 4;
  fill_all_indices_kernel<<<grid, kTopkThreads, 0, stream>>>(out, n_tok, k, lens);
  return cudaGetLastError();
}

}  // namespace dsv4kv
