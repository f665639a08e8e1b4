// index_score_mxq: the index scorer in its block-scaled tensor-core mode.  The
// MXFP4 index keys ("vllm.models.minimax_m3.amd.ops.mxfp4_pages": [pages, 128,
// 64] e2m1 rows + [pages, 128, 4] e8m0 scales) go into a block-scaled MMA as
// they are; the index-q row is first converted to MXFP8 (per 32-element block a
// shared exponent floor(log2 amax) - 8, elements to E4M3), the other MX operand
// format of the pages' scaled matrix core ("vllm.models.minimax_m3.amd.mono.
// weights", module description and mxfp8_a_tiles: the f8f6f4 MFMA with e8m0
// scales).  The score is the MXFP8 query dotted with the dequantised key,
// accumulated in fp32 by the tensor core.
//
// One page per MMA group: M = the page's 128 token rows, N = 16 (the q <= 8
// queries of the sequence, the rest zero), K = 128 as four K = 32 steps of
//   tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X
// with A = e2m1, B = e4m3 and UE8M0 scales; step kb picks byte kb of each
// row's 32-bit scale word, which is the page's own scale row.
//
// Operand layouts (K-major, no swizzle, 8-row x 16-byte core matrices):
//   A: the 16 codes of K-chunk j of row m take the first 8 bytes of a 16-byte
//      slot at (m/8)*1024 + j*128 + (m%8)*16 (the e2m1 operand of this MMA kind
//      is packed two a byte, low nibble first, in 16-byte slots of which the
//      last 8 bytes are ignored), so a page row's 64 bytes are spread as eight
//      8-byte pieces; LBO (next K-chunk) = 128, SBO (next 8 rows) = 1024.
//   B: the 16 E4M3 bytes of K-chunk j of query n at (n/8)*1024 + j*128 + (n%8)*16.
//   Scales in tensor memory: row m's word at lane m, column kColSfa + m/32;
//   query n's word at lane n of every lane quarter (each quarter of the
//   accumulator reads the query scales from its own 32 lanes), column kColSfb.
//   Accumulator: lane m = page row m, column n = query n (fp32).
//
// Roles: the pipeline's producer warp streams pages into the stage ring; four
// consumer warps (one per tensor-memory lane quarter) copy each page into the A
// tile and its scale words into tensor memory, free the stage, and thread 0
// issues the four MMAs; the warps read the accumulator back with tcgen05.ld and
// write the scores.  Every wait is bounded and every exit frees the tensor
// memory the CTA allocated.
#include "score_pipeline.cuh"

namespace mx4 {

namespace mxq {

constexpr int kATileBytes = 128 * 8 * 16;  // 128 rows x 8 K-chunks x 16-byte slots
constexpr int kBTileBytes = 16 * 8 * 16;   // 16 query rows x 8 K-chunks x 16 bytes
constexpr int kTmemCols = 32;              // the smallest allocation
constexpr int kColD = 0;                   // accumulator: columns 0 .. 15
constexpr int kColSfa = 16;                // key scales: columns 16 .. 19
constexpr int kColSfb = 24;                // query scales: column 24
// format region: A tile | B tile | MMA barrier | tensor-memory address | query scale bytes
constexpr int kBarOff = kATileBytes + kBTileBytes;
constexpr int kTaddrOff = kBarOff + 8;
constexpr int kSfbOff = kTaddrOff + 8;
constexpr int kRegionBytes = (kSfbOff + 16 * 4 + 127) / 128 * 128;

__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((addr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version; base offset 0, no swizzle
  return d;
}

// Instruction descriptor of K-step kb: A e2m1 (5), B e4m3 (0), UE8M0 scales,
// N = 16, M = 128, scale byte kb of both scale words.
__host__ __device__ constexpr uint32_t idesc(uint32_t kb) {
  return (kb << 4) | (5u << 7) | (0u << 10) | ((16u >> 3) << 17) | (1u << 23) |
         ((128u >> 4) << 24) | (kb << 29);
}

__device__ __forceinline__ void named_sync() { asm volatile("bar.sync 1, 128;\n" ::: "memory"); }

// AND of v over the 128 consumer threads (all of them must call it).
__device__ __forceinline__ bool all_consumers(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
      " barrier.cta.red.and.pred q, 1, 128, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0u;
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};\n" ::"r"(taddr), "r"(v) : "memory");
}

// E4M3 codes of four fp32 values (nearest, ties to even, saturating at 448),
// x0 in the low byte.
__device__ __forceinline__ uint32_t e4m3x4(float x0, float x1, float x2, float x3) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %2, %1;\n" : "=h"(lo) : "f"(x0), "f"(x1));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %2, %1;\n" : "=h"(hi) : "f"(x2), "f"(x3));
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

}  // namespace mxq

struct MxqFmt {
  static constexpr int kPageBytes = mx4::kPageBytes;
  static constexpr int kConsumers = 4;  // one warp per tensor-memory lane quarter
  static constexpr int kStages = 4;
  static constexpr int kExtraBytes = mxq::kRegionBytes;
  static constexpr bool kWholePage = true;
  static constexpr int ctas_per_sm(int) { return 3; }

  // The sequence's index-q rows (bf16, in the stage after the page) -> MXFP8:
  // the B tile and the query scale words (written by each warp into its own lane
  // quarter).  Thread t converts the 16 elements of
  // K-chunk j = t % 8 of query n = t / 8; the two threads of a 32-element block
  // share its largest magnitude.
  template <int Q>
  static __device__ __forceinline__ void set_queries(const uint16_t* qs, uint8_t* region,
                                                     uint32_t tm, int tid, int warp, int lane) {
    const int n = tid >> 3, j = tid & 7;
    uint32_t w[8];
    float amax = 0.f;
    if (n < Q) {
      const uint4 u0 = *reinterpret_cast<const uint4*>(qs + n * kHeadDim + 16 * j);
      const uint4 u1 = *reinterpret_cast<const uint4*>(qs + n * kHeadDim + 16 * j + 8);
      w[0] = u0.x; w[1] = u0.y; w[2] = u0.z; w[3] = u0.w;
      w[4] = u1.x; w[5] = u1.y; w[6] = u1.z; w[7] = u1.w;
#pragma unroll
      for (int i = 0; i < 8; ++i)
        amax = fmaxf(amax, fmaxf(fabsf(bf16_bits_to_float(w[i] & 0xFFFFu)),
                                 fabsf(bf16_bits_to_float(w[i] >> 16))));
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
    // shared exponent floor(log2 amax) - 8 in [-127, 127]; -127 for a zero block
    // (or one below the normal range, whose floor(log2) is below -126)
    const int efield = (int)(__float_as_uint(amax) >> 23);
    const int E = (amax == 0.f) ? -127 : max(-127, min(127, efield - 127 - 8));
    const float inv = __uint_as_float((uint32_t)(127 - E) << 23);  // 2^-E, normal for E >= -127
    uint4 codes = make_uint4(0u, 0u, 0u, 0u);
    if (n < Q) {
      float x[16];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        x[2 * i] = bf16_bits_to_float(w[i] & 0xFFFFu) * inv;  // exact: power-of-two scaling
        x[2 * i + 1] = bf16_bits_to_float(w[i] >> 16) * inv;
      }
      codes.x = mxq::e4m3x4(x[0], x[1], x[2], x[3]);
      codes.y = mxq::e4m3x4(x[4], x[5], x[6], x[7]);
      codes.z = mxq::e4m3x4(x[8], x[9], x[10], x[11]);
      codes.w = mxq::e4m3x4(x[12], x[13], x[14], x[15]);
    }
    *reinterpret_cast<uint4*>(region + mxq::kATileBytes + (n >> 3) * 1024 + j * 128 +
                              (n & 7) * 16) = codes;
    uint8_t* sfb = region + mxq::kSfbOff;
    if ((j & 1) == 0) sfb[n * 4 + (j >> 1)] = (uint8_t)(n < Q ? E + 127 : 127);
    mxq::named_sync();
    const uint32_t word = *reinterpret_cast<const uint32_t*>(sfb + (lane & 15) * 4);
    mxq::tmem_st1(tm + ((uint32_t)(32 * warp) << 16) + mxq::kColSfb, word);
  }

  template <int Q>
  static __device__ void consume(const ScoreArgs& a, const StageRing& ring, uint8_t* region,
                                 int n, int warp, int lane) {
    constexpr int S = kStages;
    const int tid = warp * 32 + lane;
    if (n == 0) return;  // no pages for this CTA: nothing allocated
    uint8_t* atile = region;
    uint64_t* mma_bar = reinterpret_cast<uint64_t*>(region + mxq::kBarOff);
    uint32_t* taddr_slot = reinterpret_cast<uint32_t*>(region + mxq::kTaddrOff);
    const uint32_t bar = smem_addr(mma_bar);
    if (tid == 0) {
      mbar_init(bar, 1);
      fence_barrier_init();
    }
    if (warp == 0) {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                       smem_addr(taddr_slot)),
                   "r"(mxq::kTmemCols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    mxq::tc_fence_before();
    mxq::named_sync();
    mxq::tc_fence_after();
    const uint32_t tm = *taddr_slot;
    const uint32_t lane_base = tm + ((uint32_t)(32 * warp) << 16);
    const uint32_t a_addr = smem_addr(atile), b_addr = a_addr + mxq::kATileBytes;

    int cur_seq = -1;
    uint32_t mma_phase = 0;
    bool mma_pending = false;  // an MMA group whose completion was not seen
    for (int kk = 0; kk < n; ++kk) {
      const int st = kk % S, round = kk / S;
      bool landed = false;
      for (uint32_t i = 0; i < kWaitPolls && !landed; ++i) {
        landed = mbar_test(smem_addr(&ring.full[st]), round & 1);
        if (!landed && *ring.abort_flag) break;
      }
      if (!mxq::all_consumers(landed)) {
        if (tid == 0) flag(a.status, MX4_STATUS_TIMEOUT);
        *ring.abort_flag = 1;
        break;
      }
      const int seq = ring.seq[st], pg = ring.page[st], L = ring.len[st];
      const bool ok = ring.ok[st] != 0;
      const uint8_t* page = ring.base + st * ring.stage_bytes;
      if (ok) {
        if (seq != cur_seq) {
          set_queries<Q>(reinterpret_cast<const uint16_t*>(page + kPageBytes), region, tm, tid,
                         warp, lane);
          cur_seq = seq;
        }
        // page rows -> A tile: 16-byte piece p (row p/4, K-chunks 2(p%4), 2(p%4)+1)
#pragma unroll
        for (int it = 0; it < 4; ++it) {
          const int p = it * 128 + tid, r = p >> 2, c = p & 3;
          const uint4 v = *reinterpret_cast<const uint4*>(page + p * 16);
          uint8_t* dst = atile + (r >> 3) * 1024 + (2 * c) * 128 + (r & 7) * 16;
          *reinterpret_cast<uint2*>(dst) = make_uint2(v.x, v.y);
          *reinterpret_cast<uint2*>(dst + 128) = make_uint2(v.z, v.w);
        }
        // this lane quarter's scale words: row 32*warp + lane at column kColSfa + warp
        const uint32_t sw =
            *reinterpret_cast<const uint32_t*>(page + kScaleOffset + 4 * (32 * warp + lane));
        mxq::tmem_st1(lane_base + mxq::kColSfa + warp, sw);
        asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
      }
      mxq::tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&ring.empty[st]));  // the page is copied out
      if (!ok) continue;
      mxq::named_sync();
      if (tid == 0) {
        mxq::tc_fence_after();
#pragma unroll
        for (uint32_t kb = 0; kb < 4; ++kb) {
          const uint64_t ad = mxq::smem_desc(a_addr + kb * 256, 128, 1024);
          const uint64_t bd = mxq::smem_desc(b_addr + kb * 256, 128, 1024);
          asm volatile(
              "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
              " tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, "
              "%3, [%4], [%5], p;\n}\n" ::"r"(tm + mxq::kColD),
              "l"(ad), "l"(bd), "r"(mxq::idesc(kb)), "r"(tm + mxq::kColSfa),
              "r"(tm + mxq::kColSfb), "r"(kb)
              : "memory");
        }
        asm volatile(
            "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
                bar)
            : "memory");
      }
      mma_pending = true;
      const bool done = mbar_wait(bar, mma_phase);
      if (!mxq::all_consumers(done)) {
        if (tid == 0) flag(a.status, MX4_STATUS_TIMEOUT);
        *ring.abort_flag = 1;
        break;
      }
      mma_pending = false;
      mma_phase ^= 1u;
      mxq::tc_fence_after();
      uint32_t d[8];
      asm volatile(
          "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];\n"
          : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3]), "=r"(d[4]), "=r"(d[5]), "=r"(d[6]),
            "=r"(d[7])
          : "r"(lane_base + mxq::kColD)
          : "memory");
      asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
      const int row = 32 * warp + lane;
      const int64_t i_g = (int64_t)pg * kPageTokens + row;
      if (i_g < L) {
#pragma unroll
        for (int qq = 0; qq < Q; ++qq) {
          const int64_t p = (int64_t)L - Q + qq;
          a.scores[((int64_t)seq * Q + qq) * a.ld + i_g] =
              (i_g <= p) ? __uint_as_float(d[qq]) : -INFINITY;
        }
      }
      mxq::tc_fence_before();
    }
    // teardown: every consumer gets here (the loop's exits are taken by all 128)
    if (mma_pending && !mbar_wait(bar, mma_phase) && tid == 0) flag(a.status, MX4_STATUS_TIMEOUT);
    mxq::tc_fence_before();
    mxq::named_sync();
    mxq::tc_fence_after();
    if (warp == 0)
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tm),
                   "r"(mxq::kTmemCols)
                   : "memory");
  }
};

cudaError_t launch_index_score_mxq(const uint16_t* iq, int q, const uint8_t* idx_pages,
                                   int64_t idx_page_stride, int64_t num_pages,
                                   const int32_t* block_table, int B, int64_t bt_width,
                                   const int32_t* seq_lens, float* scores, int64_t ld,
                                   uint32_t* status, int num_sms, cudaStream_t stream) {
  const ScoreArgs a{iq, idx_pages, idx_page_stride, num_pages, block_table, B, bt_width,
                    seq_lens, scores, ld, status, 1.f};
  switch (q) {
    case 1: return launch_score<MxqFmt, 1>(a, num_sms, stream);
    case 2: return launch_score<MxqFmt, 2>(a, num_sms, stream);
    case 3: return launch_score<MxqFmt, 3>(a, num_sms, stream);
    case 4: return launch_score<MxqFmt, 4>(a, num_sms, stream);
    case 5: return launch_score<MxqFmt, 5>(a, num_sms, stream);
    case 6: return launch_score<MxqFmt, 6>(a, num_sms, stream);
    case 7: return launch_score<MxqFmt, 7>(a, num_sms, stream);
    case 8: return launch_score<MxqFmt, 8>(a, num_sms, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mx4
