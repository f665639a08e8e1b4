// Device-side helpers shared by the kernels of the MXFP4 sparse paged decode
// library (sm_103a).  Page geometry follows "vllm.models.minimax_m3.amd.ops.
// mxfp4_pages" (module description): per page and head, 128 token rows of
// 64 B e2m1 data followed by 128 rows of 4 B e8m0 scales, 8704 B in all.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "mx4sp.h"

namespace mx4 {

constexpr int kPageTokens = 128;
constexpr int kHeadDim = 128;
constexpr int kRowDataBytes = 64;                          // 128 elements, two a byte
constexpr int kRowScaleBytes = 4;                          // one e8m0 per 32 elements
constexpr int kScaleOffset = kPageTokens * kRowDataBytes;  // 8192: start of the scale rows
constexpr int kPageBytes = kPageTokens * (kRowDataBytes + kRowScaleBytes);  // 8704
static_assert(kPageBytes == MX4_PAGE_BYTES, "page geometry");

// Value of an e8m0 scale byte as an fp32 bit pattern: 2^(b - 127).  b = 0 is
// the subnormal 2^-127, b = 255 is NaN.
__device__ __forceinline__ float e8m0_to_float(uint32_t b) {
  uint32_t bits = (b == 0u) ? 0x00400000u : (b == 255u ? 0x7FC00000u : (b << 23));
  return __uint_as_float(bits);
}

// Value of one e2m1 code (low 4 bits of c) as fp32.  The magnitude bits
// (exponent e, mantissa m) give 0.5*m for e == 0 and (1 + m/2) * 2^(e-1)
// otherwise; bit 3 is the sign.
__device__ __forceinline__ float e2m1_to_float(uint32_t c) {
  uint32_t e = (c >> 1) & 3u, m = c & 1u;
  float mag = (e == 0u) ? 0.5f * (float)m : __uint_as_float(((e + 126u) << 23) | (m << 22));
  return __uint_as_float(__float_as_uint(mag) | ((c & 8u) << 28));
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) {
  return __uint_as_float(b << 16);
}

__device__ __forceinline__ void flag(uint32_t* status, uint32_t bit) {
  if (status) atomicOr(status, bit);
}

}  // namespace mx4
