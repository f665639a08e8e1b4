// The fp8 index-K cache variant: insert and scorer.
//
// The other revision of the layer keeps the index keys in an fp8 cache of shape
// [blocks, block, head_dim] with shared block ids ("vllm.models.minimax_m3.amd.
// mono.weights", SparseMoeLayer.index_cache; "vllm.models.minimax_m3.amd.mono.
// dispatch", _config_refusal requires the fp8 index dtype).  A token row is 128
// OCP E4M3 bytes and a page 128 rows = 16384 B.  The layout has no room for
// scales, so one fp32 scale S > 0 per cache is an argument: a key element is
// stored as E4M3(fl32(x / S)) (round to nearest even, saturating at 448) and
// reads back as its E4M3 value times S.
//
// fp8_index_insert_kernel: one warp per new token row, 4 elements a lane.
//
// index_score_fp8: the shared scorer pipeline (score_pipeline.cuh: pages of all
// sequences cut into equal contiguous ranges, one per CTA; a producer warp
// streams each page plus the sequence's index-q rows into a shared-memory ring
// with bulk copies completing on mbarriers; bounded waits, drained on exit) with
// the fp8 tile math: on the tensor cores (mma m16n8k16, f16 in, fp32
// accumulate), A = 16 key rows decoded by the hardware e4m3 -> f16 conversion
// (exact), thread t of a quad owning dims 32t .. 32t+31; B = index-q, bf16
// scaled into f16 by a power of two (exact), output column n = query n.  The
// score is C * 2^-sigma * S.
#include <cuda_fp8.h>

#include "score_pipeline.cuh"

namespace mx4 {

constexpr int kFp8RowBytes = kHeadDim;                        // one E4M3 byte per element
constexpr int kFp8PageBytes = kPageTokens * kFp8RowBytes;     // 16384
static_assert(kFp8PageBytes == MX4_FP8_PAGE_BYTES, "fp8 page geometry");

// ---------------------------------------------------------------------------
// insert

__global__ void __launch_bounds__(256)
fp8_index_insert_kernel(const float* __restrict__ idx_k, int64_t T,
                        const int64_t* __restrict__ slot_mapping, float scale,
                        uint8_t* __restrict__ pages, int64_t page_stride, int64_t num_pages,
                        uint32_t* status) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  const int64_t slot = slot_mapping[t];
  if (slot < 0) return;
  const int64_t page = slot / kPageTokens;
  const int row = (int)(slot % kPageTokens);
  if (page >= num_pages) {
    if (lane == 0) flag(status, MX4_STATUS_BAD_SLOT);
    return;
  }
  const float4 x = reinterpret_cast<const float4*>(idx_k + t * kHeadDim)[lane];
  const bool finite = isfinite(x.x) && isfinite(x.y) && isfinite(x.z) && isfinite(x.w);
  if (!__all_sync(0xFFFFFFFFu, finite) && lane == 0) flag(status, MX4_STATUS_BAD_VALUE);
  const float xs[4] = {x.x, x.y, x.z, x.w};
  uint32_t packed = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    // IEEE-rounded quotient, then the hardware conversion (nearest even, saturating);
    // the sign bit is kept for a quotient that rounds to zero.
    const uint32_t code =
        (uint32_t)__nv_cvt_float_to_fp8(__fdiv_rn(xs[e], scale), __NV_SATFINITE, __NV_E4M3) |
        ((__float_as_uint(xs[e]) >> 24) & 0x80u);
    packed |= code << (8 * e);
  }
  reinterpret_cast<uint32_t*>(pages + page * page_stride + (int64_t)row * kFp8RowBytes)[lane] =
      packed;
}

cudaError_t launch_fp8_index_insert(const float* idx_k, int64_t T, const int64_t* slot_mapping,
                                    float scale, uint8_t* pages, int64_t page_stride,
                                    int64_t num_pages, uint32_t* status, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t blocks = (T + (threads / 32) - 1) / (threads / 32);
  return launch_pdl(fp8_index_insert_kernel, dim3((unsigned)blocks), dim3(threads), 0, stream,
                    idx_k, T, slot_mapping, scale, pages, page_stride, num_pages, status);
}

// ---------------------------------------------------------------------------
// scorer

// Two E4M3 pairs of w -> two f16x2 (the low byte of each pair -> the low half).
__device__ __forceinline__ void e4m3x4_to_f16x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n .reg .b16 h0, h1;\n mov.b32 {h0, h1}, %2;\n"
      " cvt.rn.f16x2.e4m3x2 %0, h0;\n cvt.rn.f16x2.e4m3x2 %1, h1;\n}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

__device__ __forceinline__ uint32_t f8_pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

struct Fp8Fmt {
  static constexpr int kPageBytes = kFp8PageBytes;
  static constexpr int kConsumers = 8;  // one 16-row tile of each page per warp
  static constexpr int kStages = 4;
  static constexpr int kStageDataBytes = kPageBytes;
  static constexpr int kStageAlign = 16;
  static constexpr int kFullCount = 1;             // the producer's expect-tx arrival
  static constexpr int kEmptyCount = kConsumers;    // one arrival per consumer warp
  static constexpr int kExtraBytes = 0;
  static constexpr bool kWholePage = false;
  static constexpr int ctas_per_sm(int) { return 2; }

  template <int Q>
  struct Tile {
    uint32_t breg[8][2];
    float osc[2];  // 2^-sigma * S of this thread's queries 2 tig, 2 tig + 1

    // index-q of the sequence -> f16 B fragments, scaled by 2^sigma per query so
    // the largest magnitude sits in [2^14, 2^15) (bf16 -> f16 then exact)
    __device__ __forceinline__ void set_queries(const uint16_t* qs, int lane, float scale) {
      const int g = lane >> 2, tig = lane & 3;
      float f = 0.f;  // 2^sigma of query g (0 for a column past the queries)
      osc[0] = osc[1] = scale;
#pragma unroll
      for (int qq = 0; qq < Q; ++qq) {
        const uint2 v = *reinterpret_cast<const uint2*>(qs + qq * kHeadDim + 4 * lane);
        uint32_t am = max(max((v.x << 17) >> 1, v.x & 0x7FFF0000u),
                          max((v.y << 17) >> 1, v.y & 0x7FFF0000u));
        am = __reduce_max_sync(0xFFFFFFFFu, am);
        const int sigma = (am == 0u) ? 0 : min(100, max(-113, 14 - ((int)(am >> 23) - 127)));
        const float down = __uint_as_float((uint32_t)(127 - sigma) << 23) * scale;
        if (qq == g) f = __uint_as_float((uint32_t)(127 + sigma) << 23);
        if (qq == 2 * tig) osc[0] = down;
        if (qq == 2 * tig + 1) osc[1] = down;
      }
      // thread (g, tig) holds column n = g: dims 32 tig + 4j .. +1 (b0), +2 .. +3 (b1)
      const bool active = g < Q;
      const uint16_t* qv = qs + (active ? g : 0) * kHeadDim + 32 * tig;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint2 v = *reinterpret_cast<const uint2*>(qv + 4 * j);
        breg[j][0] = active ? f8_pack_half2(bf16_bits_to_float(v.x & 0xFFFFu) * f,
                                            bf16_bits_to_float(v.x >> 16) * f)
                            : 0u;
        breg[j][1] = active ? f8_pack_half2(bf16_bits_to_float(v.y & 0xFFFFu) * f,
                                            bf16_bits_to_float(v.y >> 16) * f)
                            : 0u;
      }
    }

    // rows r0 .. r0 + 15 of the page: emit(query, row, score).  Rows g and g + 8
    // are 128 B apart (the same banks): a thread of an odd row reads the two
    // 16-byte halves of its 32 bytes in the other order, so the 8 lanes of a
    // quarter-warp hit all 32 banks, then swaps them back in registers.
    template <class Emit>
    __device__ __forceinline__ void run(const uint8_t* page, int r0, int lane, Emit& emit) {
      const int g = lane >> 2, tig = lane & 3;
      const int swap = g & 1;
      const uint8_t* rx = page + (r0 + g) * kFp8RowBytes + 32 * tig;
      const uint8_t* ry = rx + 8 * kFp8RowBytes;
      uint4 x0 = *reinterpret_cast<const uint4*>(rx + 16 * swap);
      uint4 x1 = *reinterpret_cast<const uint4*>(rx + 16 * (1 - swap));
      uint4 y0 = *reinterpret_cast<const uint4*>(ry + 16 * swap);
      uint4 y1 = *reinterpret_cast<const uint4*>(ry + 16 * (1 - swap));
      if (swap) {
        const uint4 tx = x0, ty = y0;
        x0 = x1;
        x1 = tx;
        y0 = y1;
        y1 = ty;
      }
      const uint32_t xw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
      const uint32_t yw[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
      float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint32_t ax0, ax2, ay1, ay3;
        e4m3x4_to_f16x2(xw[j], ax0, ax2);
        e4m3x4_to_f16x2(yw[j], ay1, ay3);
        mma_m16n8k16_f16(c, ax0, ay1, ax2, ay3, breg[j][0], breg[j][1]);
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int qq = 2 * tig + h;
        if (qq < Q) {
          emit(qq, r0 + g, c[h] * osc[h]);
          emit(qq, r0 + g + 8, c[2 + h] * osc[h]);
        }
      }
    }
  };
};

cudaError_t launch_index_score_fp8(const uint16_t* iq, int q, const uint8_t* pages,
                                   int64_t page_stride, int64_t num_pages,
                                   const int32_t* block_table, int B, int64_t bt_width,
                                   const int32_t* seq_lens, float scale, float* scores,
                                   int64_t ld, uint32_t* status, int num_sms,
                                   cudaStream_t stream) {
  ScoreArgs a{iq, pages, page_stride, num_pages, block_table, B, bt_width, seq_lens,
              scores, ld, status, scale};
  switch (q) {
    case 1: return launch_score<Fp8Fmt, 1>(a, num_sms, stream);
    case 2: return launch_score<Fp8Fmt, 2>(a, num_sms, stream);
    case 3: return launch_score<Fp8Fmt, 3>(a, num_sms, stream);
    case 4: return launch_score<Fp8Fmt, 4>(a, num_sms, stream);
    case 5: return launch_score<Fp8Fmt, 5>(a, num_sms, stream);
    case 6: return launch_score<Fp8Fmt, 6>(a, num_sms, stream);
    case 7: return launch_score<Fp8Fmt, 7>(a, num_sms, stream);
    case 8: return launch_score<Fp8Fmt, 8>(a, num_sms, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mx4
