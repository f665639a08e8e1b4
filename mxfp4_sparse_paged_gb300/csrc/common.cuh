// Device-side helpers shared by the kernels of the MXFP4 sparse paged decode
// library (sm_103a).  Page geometry follows "vllm.models.minimax_m3.amd.ops.
// mxfp4_pages" (module description): per page and head, 128 token rows of
// 64 B e2m1 data followed by 128 rows of 4 B e8m0 scales, 8704 B in all.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
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

// Programmatic dependent launch.  Every kernel of the library is launched with
// launch_pdl and signals its dependents as soon as it starts, so the next kernel
// in the stream can be scheduled while this one drains.  A kernel may run code
// before pdl_wait() only if it reads inputs no kernel of the library writes
// (sequence lengths, block tables) and writes nothing but shared memory;
// pdl_wait() returns once the previous kernel in the stream has completed and
// its writes are visible (at once when there is none).
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) {
  return __uint_as_float(b << 16);
}

__device__ __forceinline__ void flag(uint32_t* status, uint32_t bit) {
  if (status) atomicOr(status, bit);
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier and bulk-copy (TMA engine) helpers ---------------------------

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
// Make initialised barriers visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}\n" ::"r"(
          bar),
      "r"(bytes)
      : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}\n" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0u;
}
// Wait for the phase of `parity` to complete, giving up after a bounded number
// of polls (each poll may itself suspend for a while).  Returns false on time-out.
constexpr uint32_t kWaitPolls = 1u << 22;
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (uint32_t i = 0; i < kWaitPolls; ++i)
    if (mbar_test(bar, parity)) return true;
  return false;
}
// Bulk copy global -> this CTA's shared memory, completing `bytes` of
// transaction count on `bar`.  Addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// The four bytes of w, each an e2m1 pair -> f16x2 (low nibble -> low half).
// The hardware conversion gives the exact E2M1 grid value.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&r)[4]) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(w));
}

__device__ __forceinline__ void mma_m16n8k16_f16(float (&c)[4], uint32_t a0, uint32_t a1,
                                                 uint32_t a2, uint32_t a3, uint32_t b0,
                                                 uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

}  // namespace mx4
