// KVLayout and PagedKV: the paged main-KV row formats and the one address
// rule every writer and reader uses.
//
// sglang PR #39652 "dsv4.1: compression, KV I/O, and metadata kernels",
// Summary (KVLayout bullet): V4 is 584 B (448 fp8 nope + 64 bf16 rope + ue8m0
// scales), V41 is 528 B (every dim fp8, one ue8m0 scale per 32 dims), V41_FP4
// is 288 B (e2m1 codes, one e4m3 scale per 16 dims); PagedKV<layout,
// page_bits>::row gives every writer the same address arithmetic.
//
// Row order inside a row (the pages do not spell it out): codes first, then
// scales.  Both parts start on a 16-byte boundary (512 and 256 are multiples
// of 16, and so are 528 and 288), so rows and their scale blocks can be moved
// with 16-byte vector accesses.
#pragma once
#include <cstdint>

namespace dsv4kv {

constexpr int kDim = 512;       // latent width
constexpr int kNopeDim = 448;   // dims 0..447
constexpr int kRopeDim = 64;    // dims 448..511, 32 interleaved complex pairs

enum KVLayout : int { kV4 = 0, kV41 = 1, kV41Fp4 = 2 };

template <int L> struct LayoutTraits;

// V4 (the pages give the sizes only; the order follows their wording):
// bytes 0..447 e4m3 codes of dims 0..447, 448..575 the 64 rope dims as bf16,
// 576..582 one ue8m0 scale per 64 nope dims, 583 zero.  Rows are 8-byte
// aligned (584 = 8 * 73), so V4 rows move with 8-byte accesses.
template <> struct LayoutTraits<kV4> {
  static constexpr int kGroup = 64;                           // nope dims per ue8m0 scale
  static constexpr int kCodeBytes = kNopeDim + 2 * kRopeDim;  // fp8 nope + bf16 rope
  static constexpr int kScaleBytes = 8;                       // 7 scales + 1 zero byte
  static constexpr int kRowBytes = kCodeBytes + kScaleBytes;
};

template <> struct LayoutTraits<kV41> {
  static constexpr int kGroup = 32;                           // dims per ue8m0 scale
  static constexpr int kCodeBytes = kDim;                     // one e4m3 per dim
  static constexpr int kScaleBytes = kDim / kGroup;           // 16
  static constexpr int kRowBytes = kCodeBytes + kScaleBytes;  // 528
};

template <> struct LayoutTraits<kV41Fp4> {
  static constexpr int kGroup = 16;                           // dims per e4m3 scale
  static constexpr int kCodeBytes = kDim / 2;                 // two e2m1 per byte
  static constexpr int kScaleBytes = kDim / kGroup;           // 32
  static constexpr int kRowBytes = kCodeBytes + kScaleBytes;  // 288
};

static_assert(LayoutTraits<kV4>::kRowBytes == 584, "V4 row is 584 B");
static_assert(LayoutTraits<kV41>::kRowBytes == 528, "V41 row is 528 B");
static_assert(LayoutTraits<kV41Fp4>::kRowBytes == 288, "V41_FP4 row is 288 B");
static_assert(LayoutTraits<kV41>::kRowBytes % 16 == 0 && LayoutTraits<kV41Fp4>::kRowBytes % 16 == 0,
              "rows stay 16-byte aligned");

__host__ __device__ constexpr int row_bytes_of(int layout) {
  return layout == kV4 ? LayoutTraits<kV4>::kRowBytes
       : layout == kV41 ? LayoutTraits<kV41>::kRowBytes
       : layout == kV41Fp4 ? LayoutTraits<kV41Fp4>::kRowBytes : -1;
}

// slot -> (page, row in page) -> byte address.  Pages are unpadded runs of
// 2^page_bits rows, so the address equals base + slot * kRowBytes; it is
// written out as page/offset to keep the paged meaning visible.
template <int L>
struct PagedKV {
  uint8_t* base;
  int page_bits;
  // pages are unpadded, so row (page, off) sits at (page * 2^page_bits + off)
  // = slot rows from the base
  __device__ __forceinline__ uint8_t* row(long long slot) const {
    return base + slot * LayoutTraits<L>::kRowBytes;
  }
};

}  // namespace dsv4kv
