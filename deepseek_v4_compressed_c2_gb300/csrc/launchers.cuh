// Host launchers of the kernels, called by the C-ABI layer (capi.cu) after
// its argument checks; each kernel file defines its own.  Device-side
// parameters and helpers are in internal.cuh.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "internal.cuh"

namespace dsv4kv {

cudaError_t launch_compress_store(const StoreParams& p, int layout, int ratio, cudaStream_t stream);

// ratio-2 steps with start positions / the ring of at most kDecodeRowsPerCta
// output rows per SM (decode, speculative-verify and short chunked-prefill
// steps): one CTA per chunk of at most kDecodeMaxChunk request slots
// (compress_decode.cu).  decode_grid: the launch's CTA count, 0 when the
// step does not fit the form.
constexpr int kDecodeRowsPerCta = 16;
constexpr int kDecodeMaxChunk = 32;
constexpr int kDecodeMaxGrid = 256;
int decode_grid(int n_slots, int n_out, int sms);
cudaError_t launch_compress_decode(const StoreParams& p, int layout, int grid, cudaStream_t stream);

cudaError_t launch_dequant_gather(int layout, const uint8_t* pool, long long pool_rows,
                                  const int* ids, long long n, __nv_bfloat16* out, int* err,
                                  cudaStream_t stream);

// topk == nullptr: the short-context form, ids j < fill_len[t] (else -1)
cudaError_t launch_dequant_gather_topk(int layout, const uint8_t* pool, long long pool_rows,
                                       const int* topk, const int* fill_len, int n_tok, int k,
                                       const int* token_to_req, const unsigned char* is_valid,
                                       const int* page_table, int n_req, int max_pages,
                                       int page_bits, __nv_bfloat16* out, int* lens, int* err,
                                       cudaStream_t stream);

cudaError_t launch_fill_all_indices(int* out, int n_tok, int k, const int* lens,
                                    cudaStream_t stream);

cudaError_t launch_fake_quant(int layout, const __nv_bfloat16* in, long long n,
                              long long in_stride, __nv_bfloat16* out, cudaStream_t stream);

cudaError_t launch_topk_to_slots(const int* topk, int n_tok, int k, const int* token_to_req,
                                 const unsigned char* is_valid, const int* page_table, int n_req,
                                 int max_pages, int page_bits, int* slots, int* lens, int* err,
                                 cudaStream_t stream);

cudaError_t launch_bounded_wait_selftest(uint32_t polls, int* err, int* gave_up,
                                         cudaStream_t stream);

cudaError_t launch_fp4_quotient_selftest(const float* x, const unsigned char* scale_codes,
                                         long long n, float* q_fast, float* q_ieee,
                                         cudaStream_t stream);

cudaError_t launch_e4m3_recip_selftest(const unsigned char* codes, long long n, float* y_fast,
                                       float* y_ieee, cudaStream_t stream);

}  // namespace dsv4kv
