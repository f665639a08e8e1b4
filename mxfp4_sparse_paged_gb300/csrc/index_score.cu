// index_score: dot every cached index key of a sequence with the index-q head
// of each of its decode tokens, over the MXFP4 index-K cache [pages, 8704]
// ("vllm.models.minimax_m3.amd.ops.mxfp4_pages", mxfp4_page_views: the
// [pages, 128, 64] / [pages, 128, 4] pair the index scorers read).  The page
// streaming is the shared scorer pipeline (score_pipeline.cuh); this file holds
// the MXFP4 tile math.
//
// Math (per 16-row tile, tensor cores): A = 16 index-key rows x 128 dims, decoded
// by the hardware e2m1 -> f16 conversion (exact); thread t of a quad owns the 32
// dims of scale block t.  B = index-q, bf16 scaled by a power of two into f16
// (exact), laid out so that output column n = 4*query + block: a column only
// sees the dims of its own block, so C holds per-block partial dots.  The
// scores are then sum_b C[row][4q+b] * 2^(scale_b - 127) in fp32 (exact
// scaling), combined across the quad with one shuffle.
#include "score_pipeline.cuh"

namespace mx4 {

__device__ __forceinline__ float e8m0_fast(uint32_t word, uint32_t sel) {
  return fmaxf(__uint_as_float(__byte_perm(word, 0u, sel) >> 1), 0x1p-127f);
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

struct Mxfp4Fmt {
  static constexpr int kPageBytes = mx4::kPageBytes;
  static constexpr int kConsumers = 8;  // one 16-row tile of each page per warp
  static constexpr int kStages = 4;
  static constexpr int kStageDataBytes = kPageBytes;
  static constexpr int kStageAlign = 16;
  static constexpr int kFullCount = 1;             // the producer's expect-tx arrival
  static constexpr int kEmptyCount = kConsumers;    // one arrival per consumer warp
  static constexpr int kExtraBytes = 0;
  static constexpr bool kWholePage = false;
  static constexpr int ctas_per_sm(int Q) { return Q <= 2 ? 4 : (Q <= 6 ? 2 : 1); }

  template <int Q>
  struct Tile {
    static constexpr int NT = (Q + 1) / 2;  // n8 tiles: 4 block-columns per query
    uint32_t breg[NT][8][2];
    float isc[NT];  // 2^-sigma of this lane's query in n8 tile nt: 2 nt + (tig >> 1)

    // index-q of the sequence -> f16 B fragments, scaled by 2^sigma per query so
    // its largest magnitude lands in [2^14, 2^15)
    __device__ __forceinline__ void set_queries(const uint16_t* qs, int lane, float) {
      const int g = lane >> 2, tig = lane & 3;
      float sc[Q], inv[Q];
#pragma unroll
      for (int qq = 0; qq < Q; ++qq) {
        const uint2 v = *reinterpret_cast<const uint2*>(qs + qq * kHeadDim + 4 * lane);
        uint32_t am = max(max((v.x << 17) >> 1, v.x & 0x7FFF0000u),
                          max((v.y << 17) >> 1, v.y & 0x7FFF0000u));
        am = __reduce_max_sync(0xFFFFFFFFu, am);
        const int sigma = (am == 0u) ? 0 : min(100, max(-113, 14 - ((int)(am >> 23) - 127)));
        sc[qq] = __uint_as_float((uint32_t)(127 + sigma) << 23);
        inv[qq] = __uint_as_float((uint32_t)(127 - sigma) << 23);
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {  // selected once, without lane-dependent indexing
        const int qq = 2 * nt + (tig >> 1);
        isc[nt] = inv[0];
#pragma unroll
        for (int q2 = 1; q2 < Q; ++q2)
          if (q2 == qq) isc[nt] = inv[q2];
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int qq = 2 * nt + (g >> 2);
        const bool active = ((g & 3) == tig) && qq < Q;
        const uint16_t* qv = qs + (qq < Q ? qq : 0) * kHeadDim + 32 * tig;
        float f = 0.f;  // sc[qq] without a lane-dependent index (which would go to local memory)
#pragma unroll
        for (int q2 = 0; q2 < Q; ++q2)
          if (active && q2 == qq) f = sc[q2];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint2 v = *reinterpret_cast<const uint2*>(qv + 4 * j);
          breg[nt][j][0] = active ? pack_half2(bf16_bits_to_float(v.x & 0xFFFFu) * f,
                                               bf16_bits_to_float(v.x >> 16) * f)
                                  : 0u;
          breg[nt][j][1] = active ? pack_half2(bf16_bits_to_float(v.y & 0xFFFFu) * f,
                                               bf16_bits_to_float(v.y >> 16) * f)
                                  : 0u;
        }
      }
    }

    // rows r0 .. r0 + 15 of the page: emit(query, row, score)
    template <class Emit>
    __device__ __forceinline__ void run(const uint8_t* page, int r0, int lane, Emit& emit) {
      const int g = lane >> 2, tig = lane & 3;
      // byte-permute selectors: scale byte 2 (tig & 1) (+1) of a word to byte 3
      const uint32_t sel0 = 0x0444u | ((uint32_t)(2 * (tig & 1)) << 12);
      const uint32_t sel1 = 0x0444u | ((uint32_t)(2 * (tig & 1) + 1) << 12);
      const uint4 x = *reinterpret_cast<const uint4*>(page + (r0 + g) * kRowDataBytes + 16 * tig);
      const uint4 y =
          *reinterpret_cast<const uint4*>(page + (r0 + g + 8) * kRowDataBytes + 16 * tig);
      const uint32_t sx = *reinterpret_cast<const uint32_t*>(page + kScaleOffset + (r0 + g) * 4);
      const uint32_t sy =
          *reinterpret_cast<const uint32_t*>(page + kScaleOffset + (r0 + g + 8) * 4);
      const uint32_t xw[4] = {x.x, x.y, x.z, x.w}, yw[4] = {y.x, y.y, y.z, y.w};
      float c[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) c[nt][0] = c[nt][1] = c[nt][2] = c[nt][3] = 0.f;
#pragma unroll
      for (int wi = 0; wi < 4; ++wi) {
        uint32_t fx[4], fy[4];
        e2m1x8_to_f16x2(xw[wi], fx);
        e2m1x8_to_f16x2(yw[wi], fy);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          mma_m16n8k16_f16(c[nt], fx[0], fy[0], fx[1], fy[1], breg[nt][2 * wi][0],
                           breg[nt][2 * wi][1]);
          mma_m16n8k16_f16(c[nt], fx[2], fy[2], fx[3], fy[3], breg[nt][2 * wi + 1][0],
                           breg[nt][2 * wi + 1][1]);
        }
      }
      // scale bytes b0, b0+1 of the two rows -> fp32 2^(byte - 127): the byte goes
      // to bits 31..24 (byte permute), then to the exponent field (>> 1); the max
      // with 2^-127 gives byte 0 its subnormal value.  Byte 255 gives +inf, so a
      // poisoned scale still yields a non-finite score.
      const float sx0 = e8m0_fast(sx, sel0), sx1 = e8m0_fast(sx, sel1);
      const float sy0 = e8m0_fast(sy, sel0), sy1 = e8m0_fast(sy, sel1);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float vg = c[nt][0] * sx0 + c[nt][1] * sx1;
        float vg8 = c[nt][2] * sy0 + c[nt][3] * sy1;
        vg += __shfl_xor_sync(0xFFFFFFFFu, vg, 1);
        vg8 += __shfl_xor_sync(0xFFFFFFFFu, vg8, 1);
        const int qq = 2 * nt + (tig >> 1);
        if ((tig & 1) == 0 && qq < Q) {
          emit(qq, r0 + g, vg * isc[nt]);
          emit(qq, r0 + g + 8, vg8 * isc[nt]);
        }
      }
    }
  };
};

cudaError_t launch_index_score(const uint16_t* iq, int q, const uint8_t* idx_pages,
                               int64_t idx_page_stride, int64_t num_pages,
                               const int32_t* block_table, int B, int64_t bt_width,
                               const int32_t* seq_lens, float* scores, int64_t ld,
                               uint32_t* status, int num_sms, cudaStream_t stream) {
  const ScoreArgs a{iq, idx_pages, idx_page_stride, num_pages, block_table, B, bt_width,
                    seq_lens, scores, ld, status, 1.f};
  switch (q) {
    case 1: return launch_score<Mxfp4Fmt, 1>(a, num_sms, stream);
    case 2: return launch_score<Mxfp4Fmt, 2>(a, num_sms, stream);
    case 3: return launch_score<Mxfp4Fmt, 3>(a, num_sms, stream);
    case 4: return launch_score<Mxfp4Fmt, 4>(a, num_sms, stream);
    case 5: return launch_score<Mxfp4Fmt, 5>(a, num_sms, stream);
    case 6: return launch_score<Mxfp4Fmt, 6>(a, num_sms, stream);
    case 7: return launch_score<Mxfp4Fmt, 7>(a, num_sms, stream);
    case 8: return launch_score<Mxfp4Fmt, 8>(a, num_sms, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mx4
