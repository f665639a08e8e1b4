// mx4_insert: quantise each new token's K, V and index-K rows into MXFP4 page
// rows through the shared page-128 slot mapping.
//
// Format: "vllm.models.minimax_m3.amd.ops.mxfp4_pages" (module description):
// 64 B of e2m1 codes per 128-element row, element 2n in the low nibble of byte
// n, then one e8m0 scale per 32 elements in the page's scale rows.  Rule: OCP
// MX v1.0 conversion -- shared exponent floor(log2(amax)) - 2 per 32-element
// block, elements rounded to the nearest E2M1 value, ties to even, saturating.
// Slot mapping: "vllm.models.minimax_m3.amd.mono.dispatch", _slots_shared.
//
// One warp quantises one row.  Lane l owns elements 4l .. 4l+3 (a float4), so
// the 8 lanes 8b .. 8b+7 hold block b; the block maximum is an xor-shuffle
// over those 8 lanes.  Each lane writes its 2 code bytes (the warp writes the
// 64 data bytes contiguously) and lane 0 writes the row's 4 scale bytes.
#include <cuda_bf16.h>

#include "common.cuh"

namespace mx4 {

// E2M1 magnitude code (0..7) of a = |y| < 8: the number of rounding thresholds
// that a lies above.  A tie sits exactly on a threshold and goes to the
// neighbour with an even mantissa bit, so the comparison is strict (>) where
// the even neighbour is the lower one (0.25, 1.25, 2.5, 5) and non-strict (>=)
// where it is the upper one (0.75, 1.75, 3.5).  Values above 6 saturate to 7.
__device__ __forceinline__ uint32_t e2m1_magnitude_code(float a) {
  return (uint32_t)(a > 0.25f) + (uint32_t)(a >= 0.75f) + (uint32_t)(a > 1.25f) +
         (uint32_t)(a >= 1.75f) + (uint32_t)(a > 2.5f) + (uint32_t)(a >= 3.5f) +
         (uint32_t)(a > 5.0f);
}

// Shared exponent E = floor(log2(amax)) - 2 clamped to [-127, 127], read from
// the fp32 exponent field (exact).  amax == 0 and subnormal amax give -127;
// finite amax never exceeds E = 125.
__device__ __forceinline__ int block_exponent(float amax) {
  uint32_t ef = (__float_as_uint(amax) >> 23) & 0xFFu;
  int E = (int)ef - 127 - 2;
  return (ef == 0u || E < -127) ? -127 : E;
}

// One 128-element row held by a warp (lane l: elements 4l .. 4l+3) -> its 64 code
// bytes and 4 scale bytes at token row `row` of the page (head) at `dst`.
// Non-finite input sets MX4_STATUS_BAD_VALUE.
__device__ __forceinline__ void quantize_store_row(float4 x, int lane, uint8_t* dst, int row,
                                                   uint32_t* status) {
  const bool finite = isfinite(x.x) && isfinite(x.y) && isfinite(x.z) && isfinite(x.w);
  if (!__all_sync(0xFFFFFFFFu, finite) && lane == 0) flag(status, MX4_STATUS_BAD_VALUE);

  float amax = fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w)));
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
  const int E = block_exponent(amax);
  // 2^-E is a normal fp32 for every E in [-127, 125]; the product is exact.
  const float inv = __uint_as_float((uint32_t)(127 - E) << 23);

  const float xs[4] = {x.x, x.y, x.z, x.w};
  uint32_t packed = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const uint32_t code = e2m1_magnitude_code(fabsf(xs[e] * inv)) |
                          ((__float_as_uint(xs[e]) >> 28) & 8u);
    packed |= code << (4 * e);
  }
  reinterpret_cast<uint16_t*>(dst + row * kRowDataBytes)[lane] = (uint16_t)packed;

  // scale bytes of blocks 0..3 live in lanes 0, 8, 16, 24
  const uint32_t sb = (uint32_t)(E + 127);
  const uint32_t s1 = __shfl_sync(0xFFFFFFFFu, sb, 8);
  const uint32_t s2 = __shfl_sync(0xFFFFFFFFu, sb, 16);
  const uint32_t s3 = __shfl_sync(0xFFFFFFFFu, sb, 24);
  if (lane == 0)
    *reinterpret_cast<uint32_t*>(dst + kScaleOffset + row * kRowScaleBytes) =
        sb | (s1 << 8) | (s2 << 16) | (s3 << 24);
}

__global__ void __launch_bounds__(256)
insert_kernel(const float* __restrict__ k, const float* __restrict__ v,
              const float* __restrict__ idx_k, int64_t T, int Hkv,
              const int64_t* __restrict__ slot_mapping, uint8_t* __restrict__ k_pages,
              uint8_t* __restrict__ v_pages, int64_t kv_page_stride, int64_t kv_head_stride,
              uint8_t* __restrict__ idx_pages, int64_t idx_page_stride, int64_t num_pages,
              uint32_t* status) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int rows_per_token = 2 * Hkv + 1;  // K heads, V heads, index key
  const int64_t warp = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (warp >= T * rows_per_token) return;
  const int64_t t = warp / rows_per_token;
  const int r = (int)(warp % rows_per_token);

  // the row and the slot are independent loads: both in flight at once
  const float* src = r < Hkv       ? k + (t * Hkv + r) * kHeadDim
                     : r < 2 * Hkv ? v + (t * Hkv + (r - Hkv)) * kHeadDim
                                   : idx_k + t * kHeadDim;
  const float4 x = reinterpret_cast<const float4*>(src)[lane];
  const int64_t slot = slot_mapping[t];
  if (slot < 0) return;
  const int64_t page = slot / kPageTokens;
  const int row = (int)(slot % kPageTokens);
  if (page >= num_pages) {
    if (lane == 0) flag(status, MX4_STATUS_BAD_SLOT);
    return;
  }
  uint8_t* const dst =
      r < Hkv       ? k_pages + page * kv_page_stride + (int64_t)r * kv_head_stride
      : r < 2 * Hkv ? v_pages + page * kv_page_stride + (int64_t)(r - Hkv) * kv_head_stride
                    : idx_pages + page * idx_page_stride;
  quantize_store_row(x, lane, dst, row, status);
}

cudaError_t launch_insert(const float* k, const float* v, const float* idx_k, int64_t T, int Hkv,
                          const int64_t* slot_mapping, uint8_t* k_pages, uint8_t* v_pages,
                          int64_t kv_page_stride, int64_t kv_head_stride, uint8_t* idx_pages,
                          int64_t idx_page_stride, int64_t num_pages, uint32_t* status,
                          cudaStream_t stream) {
  const int64_t warps = T * (2 * Hkv + 1);
  const int threads = 256;
  const int64_t blocks = (warps + (threads / 32) - 1) / (threads / 32);
  return launch_pdl(insert_kernel, dim3((unsigned)blocks), dim3(threads), 0, stream, k, v, idx_k,
                    T, Hkv, slot_mapping, k_pages, v_pages, kv_page_stride, kv_head_stride,
                    idx_pages, idx_page_stride, num_pages, status);
}

// ---------------------------------------------------------------------------
// mx4_norm_rope_insert: the writer in front of the insert ("vllm.models.
// minimax_m3.amd.mono.weights", SparseMoeLayer: norm weights g_q, g_k, g_iq,
// g_ik and the rotary table cos_sin; no formula is printed, so the plainest
// reading is taken): each q, index-q, k and index-k head row is RMS-normed over
// its 128 dims, times its weight, then turned pairwise -- dims i and i+64
// (i < 64) by the angle with cosine cos_sin[pos][i] and sine cos_sin[pos][64+i].
// q and index-q go out as bf16 (round to nearest even); k and index-k are then
// quantised into their page rows, and V is quantised as it comes.
//
// One warp per row.  Lane l holds dims 4l .. 4l+3, so the rotation partner of
// lane l < 16 is lane l + 16 (one xor-shuffle).

// RMS norm of the warp's row, times g, then (rope) the pairwise turn by cs.
__device__ __forceinline__ float4 norm_rope_row(float4 x, int lane, const float* __restrict__ g,
                                                const float* __restrict__ cs, float eps,
                                                bool rope) {
  float p = x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) p += __shfl_xor_sync(0xFFFFFFFFu, p, o);
  const float inv = 1.0f / sqrtf(p * (1.0f / 128.0f) + eps);  // IEEE sqrt and divide
  const float4 gw = reinterpret_cast<const float4*>(g)[lane];
  const float4 z = make_float4(x.x * inv * gw.x, x.y * inv * gw.y, x.z * inv * gw.z,
                               x.w * inv * gw.w);
  if (!rope) return z;
  const float4 w = make_float4(__shfl_xor_sync(0xFFFFFFFFu, z.x, 16),
                               __shfl_xor_sync(0xFFFFFFFFu, z.y, 16),
                               __shfl_xor_sync(0xFFFFFFFFu, z.z, 16),
                               __shfl_xor_sync(0xFFFFFFFFu, z.w, 16));
  const float4 c = reinterpret_cast<const float4*>(cs)[lane & 15];
  const float4 sn = reinterpret_cast<const float4*>(cs + kHeadDim / 2)[lane & 15];
  if (lane < 16)  // first halves: z c - partner s
    return make_float4(z.x * c.x - w.x * sn.x, z.y * c.y - w.y * sn.y, z.z * c.z - w.z * sn.z,
                       z.w * c.w - w.w * sn.w);
  return make_float4(z.x * c.x + w.x * sn.x, z.y * c.y + w.y * sn.y, z.z * c.z + w.z * sn.z,
                     z.w * c.w + w.w * sn.w);
}

__global__ void __launch_bounds__(256)
norm_rope_insert_kernel(const float* __restrict__ q, const float* __restrict__ iq,
                        const float* __restrict__ k, const float* __restrict__ v,
                        const float* __restrict__ idx_k, int64_t T, int H, int Hkv,
                        const int64_t* __restrict__ positions, const float* __restrict__ cos_sin,
                        int64_t max_pos, const float* __restrict__ g_q,
                        const float* __restrict__ g_k, const float* __restrict__ g_iq,
                        const float* __restrict__ g_ik, float eps,
                        const int64_t* __restrict__ slot_mapping, uint8_t* __restrict__ k_pages,
                        uint8_t* __restrict__ v_pages, int64_t kv_page_stride,
                        int64_t kv_head_stride, uint8_t* __restrict__ idx_pages,
                        int64_t idx_page_stride, int64_t num_pages, uint16_t* __restrict__ q_out,
                        uint16_t* __restrict__ iq_out, uint32_t* status) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int rows_per_token = H + 1 + 2 * Hkv + 1;  // q heads, index-q, K heads, V heads, index-k
  const int64_t warp = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (warp >= T * rows_per_token) return;
  const int64_t t = warp / rows_per_token;
  const int r = (int)(warp % rows_per_token);
  const int rk = r - H - 1;  // 0 .. 2 Hkv: K heads, V heads, index-k
  // the row, the position and the slot are independent loads: all in flight at once
  const float* src = r < H          ? q + (t * H + r) * kHeadDim
                     : r == H       ? iq + t * kHeadDim
                     : rk < Hkv     ? k + (t * Hkv + rk) * kHeadDim
                     : rk < 2 * Hkv ? v + (t * Hkv + (rk - Hkv)) * kHeadDim
                                    : idx_k + t * kHeadDim;
  const float4 xr = reinterpret_cast<const float4*>(src)[lane];
  const int64_t pos = positions[t];
  const int64_t slot = r > H ? slot_mapping[t] : 0;
  if (pos < 0 || pos >= max_pos) {
    if (lane == 0) flag(status, MX4_STATUS_BAD_INDEX);
    return;
  }
  const float* cs = cos_sin + pos * kHeadDim;

  if (r <= H) {  // q head r, or (r == H) the index-q head: bf16 out
    const bool isq = r < H;
    uint16_t* dst = isq ? q_out + (t * H + r) * kHeadDim : iq_out + t * kHeadDim;
    const float4 y = norm_rope_row(xr, lane, isq ? g_q : g_iq, cs, eps, true);
    const __nv_bfloat162 lo = __floats2bfloat162_rn(y.x, y.y), hi = __floats2bfloat162_rn(y.z, y.w);
    reinterpret_cast<uint2*>(dst)[lane] =
        make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
    return;
  }

  if (slot < 0) return;
  const int64_t page = slot / kPageTokens;
  const int row = (int)(slot % kPageTokens);
  if (page >= num_pages) {
    if (lane == 0) flag(status, MX4_STATUS_BAD_SLOT);
    return;
  }
  float4 x;
  uint8_t* dst;
  if (rk < Hkv) {
    x = norm_rope_row(xr, lane, g_k, cs, eps, true);
    dst = k_pages + page * kv_page_stride + (int64_t)rk * kv_head_stride;
  } else if (rk < 2 * Hkv) {
    x = xr;
    dst = v_pages + page * kv_page_stride + (int64_t)(rk - Hkv) * kv_head_stride;
  } else {
    x = norm_rope_row(xr, lane, g_ik, cs, eps, true);
    dst = idx_pages + page * idx_page_stride;
  }
  quantize_store_row(x, lane, dst, row, status);
}

cudaError_t launch_norm_rope_insert(const float* q, const float* iq, const float* k,
                                    const float* v, const float* idx_k, int64_t T, int H, int Hkv,
                                    const int64_t* positions, const float* cos_sin,
                                    int64_t max_pos, const float* g_q, const float* g_k,
                                    const float* g_iq, const float* g_ik, float eps,
                                    const int64_t* slot_mapping, uint8_t* k_pages,
                                    uint8_t* v_pages, int64_t kv_page_stride,
                                    int64_t kv_head_stride, uint8_t* idx_pages,
                                    int64_t idx_page_stride, int64_t num_pages, uint16_t* q_out,
                                    uint16_t* iq_out, uint32_t* status, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const int64_t warps = T * (H + 2 + 2 * Hkv);
  const int threads = 256;
  const int64_t blocks = (warps + (threads / 32) - 1) / (threads / 32);
  return launch_pdl(norm_rope_insert_kernel, dim3((unsigned)blocks), dim3(threads), 0, stream, q,
                    iq, k, v, idx_k, T, H, Hkv, positions, cos_sin, max_pos, g_q, g_k, g_iq, g_ik,
                    eps, slot_mapping, k_pages, v_pages, kv_page_stride, kv_head_stride, idx_pages,
                    idx_page_stride, num_pages, q_out, iq_out, status);
}

}  // namespace mx4
