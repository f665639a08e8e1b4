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
// Operand layouts (K-major):
//   A: the e2m1 operand of this MMA kind takes 16 codes (packed two a byte, low
//      nibble first) in the first 8 bytes of a 16-byte slot, the other 8 bytes
//      unread.  A tensor copy of the pool with the 4-bit type that writes exactly
//      that (16U4_ALIGN16B) and 128-byte swizzle puts a page's 128 rows into the A
//      tile as 8-row x 128-byte atoms, the 16-byte slots of row r XOR-permuted by
//      r % 8; the descriptor's SBO (next 8 rows) is 1024 and K-step kb starts 32
//      bytes along the row.  The A tile is the stage itself.
//   B: no swizzle, 8-row x 16-byte core matrices: the 16 E4M3 bytes of K-chunk j of
//      query n at (n/8)*1024 + j*128 + (n%8)*16; LBO = 128, SBO = 1024.
//   Scales in tensor memory: row m's word at lane m, column (key scales) + m/32;
//   query n's word at lane n of every lane quarter (each quarter of the
//   accumulator reads the query scales from its own 32 lanes).
//   Accumulator: lane m = page row m, column n = query n (fp32).
//
// Stage (1024-byte aligned): A tile (16384 B) | the page's 512 scale bytes | the
// sequence's index-q rows.  Its full barrier completes when the tensor copy (8192
// bytes read) and the bulk copies (transaction-counted) have landed; the MMA group's
// commit frees it.
//
// Consumers (four warps, one per tensor-memory lane quarter): per page, write
// its scale words into tensor memory, and thread 0 issues the four MMAs into
// one of two accumulators; then read back and store the previous page's
// scores, whose MMAs ran meanwhile.  Every wait is bounded and every exit waits
// for the MMAs in flight and frees the tensor memory the CTA allocated.
#include <cudaTypedefs.h>  // PFN_cuTensorMapEncodeTiled

#include "score_pipeline.cuh"

namespace mx4 {

namespace mxq {

constexpr int kATileBytes = 128 * 8 * 16;  // 128 rows x 8 K-chunks x 16-byte slots
constexpr int kScaleBytes = 128 * 4;
constexpr int kBTileBytes = 16 * 8 * 16;   // 16 query rows x 8 K-chunks x 16 bytes
constexpr int kTmemCols = 64;              // an allocation is a power of two >= 32
constexpr int kColD = 0;                   // accumulators: columns 0..15 and 16..31
constexpr int kColSfa = 32;                // key scales: columns 32..35 and 36..39
constexpr int kColSfb = 40;                // query scales
// format region: B tile | MMA barriers [2] | tensor-memory address | query scale bytes
constexpr int kBarOff = kBTileBytes;
constexpr int kTaddrOff = kBarOff + 16;
constexpr int kSfbOff = kTaddrOff + 16;
constexpr int kRegionBytes = (kSfbOff + 16 * 4 + 127) / 128 * 128;

__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((addr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version; base offset 0, no swizzle
  return d;
}

// Descriptor of a K-major operand in 128-byte swizzle atoms (8 rows x 128 bytes,
// the 16-byte chunks of row r XOR-permuted by r % 8, as the tensor copy writes them):
// SBO = 1024 to the next 8 rows; a K-step starts 32 bytes further along the row.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
  return smem_desc(addr, 16, 1024) | ((uint64_t)2 << 61);
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
__device__ __forceinline__ void commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
                   bar)
               : "memory");
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
  static constexpr int kStageDataBytes = mxq::kATileBytes + mxq::kScaleBytes;
  static constexpr int kStageAlign = 1024;  // the A tile's 128-byte swizzle atoms
  static constexpr int kConsumers = 4;      // one warp per tensor-memory lane quarter
  static constexpr int kStages = 2;
  static constexpr int kFullCount = 1;   // the producer's expect-tx arrival
  static constexpr int kEmptyCount = 1;  // the MMA group's commit (or a skip)
  static constexpr int kExtraBytes = (mxq::kRegionBytes + kStageAlign - 1) / kStageAlign * kStageAlign;
  static constexpr bool kWholePage = true;
  // Two stages and five CTAs an SM (as many as the shared memory holds): the page
  // rate follows the CTAs working at once more than the stages each keeps in flight
  // (measured on the b256 workload, stages x CTAs: 5 x 2 65 us, 3 x 3 53 us,
  // 2 x 4 49 us, 2 x 5 47 us, 1 x 6 56 us).
  static constexpr int ctas_per_sm(int) { return 5; }

  // Producer warp: for each page of the CTA's range, once its stage is free, one
  // tensor copy of the page's 128 data rows into the A tile (the pool's tensor map:
  // 4-bit elements, 16 to a 16-byte slot, 128-byte swizzle), and bulk copies of the
  // scale row and the sequence's index-q rows.  The tensor copy counts the 8192 bytes
  // it reads in the barrier's transaction count.
  template <int Q>
  static __device__ void produce(const ScoreArgs& a, const StageRing& ring, const int* pref,
                                 int p0, int n, int lane) {
    constexpr int S = kStages;
    for (int base = 0; base < n; base += 32) {
      if (__any_sync(0xFFFFFFFFu, *ring.abort_flag != 0)) break;
      PageRef pr{a.pages, -1, 0, 0, 0, 0};
      if (base + lane < n) pr = resolve_page(a, pref, p0 + base + lane);
      const int cnt = min(32, n - base);
      for (int l = 0; l < cnt; ++l) {
        if (lane == l) {
          const int kk = base + l, st = kk % S, round = kk / S;
          bool go = !*ring.abort_flag;
          if (go && round > 0 && !mbar_wait(smem_addr(&ring.empty[st]), (round - 1) & 1)) {
            flag(a.status, MX4_STATUS_TIMEOUT);
            *ring.abort_flag = 1;
            go = false;
          }
          if (go) {
            ring.seq[st] = pr.seq;
            ring.page[st] = pr.page;
            ring.len[st] = pr.len;
            ring.ok[st] = pr.ok;
            const uint32_t fb = smem_addr(&ring.full[st]);
            const uint32_t d0 = smem_addr(ring.base + st * ring.stage_bytes);
            if (pr.ok) {
              mbar_arrive_expect_tx(fb, kRowDataBytes * kPageTokens + mxq::kScaleBytes +
                                            Q * kHeadDim * 2);
              asm volatile(
                  "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::"
                  "bytes [%0], [%1, {%2, %3, %4}], [%5];\n" ::"r"(d0),
                  "l"(reinterpret_cast<uint64_t>(&a.tmap)), "r"(0), "r"(0), "r"(pr.pid), "r"(fb)
                  : "memory");
              bulk_copy_g2s(d0 + mxq::kATileBytes, pr.src + kScaleOffset, mxq::kScaleBytes, fb);
              bulk_copy_g2s(d0 + kStageDataBytes, a.iq + (int64_t)pr.seq * Q * kHeadDim,
                            Q * kHeadDim * 2, fb);
            } else {
              mbar_arrive(fb);
            }
            *ring.issued = kk + 1;
          }
        }
        __syncwarp();
      }
    }
  }

  // The sequence's index-q rows (bf16, in the stage) -> MXFP8: the B tile and the
  // query scale words (written by each warp into its own lane quarter).  Thread t
  // converts the 16 elements of K-chunk j = t % 8 of query n = t / 8; the two
  // threads of a 32-element block share its largest magnitude.
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
    *reinterpret_cast<uint4*>(region + (n >> 3) * 1024 + j * 128 + (n & 7) * 16) = codes;
    uint8_t* sfb = region + mxq::kSfbOff;
    if ((j & 1) == 0) sfb[n * 4 + (j >> 1)] = (uint8_t)(n < Q ? E + 127 : 127);
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");  // the B tile, for the MMA
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
    uint64_t* mma_bar = reinterpret_cast<uint64_t*>(region + mxq::kBarOff);  // one per accumulator
    uint32_t* taddr_slot = reinterpret_cast<uint32_t*>(region + mxq::kTaddrOff);
    if (tid == 0) {
      mbar_init(smem_addr(&mma_bar[0]), 1);
      mbar_init(smem_addr(&mma_bar[1]), 1);
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
    const uint32_t b_addr = smem_addr(region);

    int cur_seq = -1;
    uint32_t phases = 0;   // bit b: the phase of mma_bar[b] to wait for next
    uint32_t groups = 0;   // MMA groups issued; group g accumulates in buffer g & 1
    uint32_t running = 0;  // bit b: buffer b's last group has not been waited for
    bool pending = false;  // a group issued and not read back yet: (p_seq, p_pg, p_len, p_buf)
    int p_seq = 0, p_pg = 0, p_len = 0;
    uint32_t p_buf = 0;
    bool failed = false;
    bool bad = false;  // this thread saw a time-out (read back)

    // Wait for the pending group, read its accumulator and store its scores.
    // Warp-local (tcgen05.ld is a warp's own): a time-out sets `bad`, which the next
    // page's vote turns into a stop for all consumers.
    auto read_back = [&]() {
      if (bad) return;  // this warp already gave up: the teardown waits (bounded) once more
      const bool done = mbar_wait(smem_addr(&mma_bar[p_buf]), (phases >> p_buf) & 1u);
      if (!__all_sync(0xFFFFFFFFu, done)) {
        bad = true;
        return;
      }
      phases ^= 1u << p_buf;
      running &= ~(1u << p_buf);
      pending = false;
      mxq::tc_fence_after();
      uint32_t d[8];
      asm volatile(
          "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];\n"
          : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3]), "=r"(d[4]), "=r"(d[5]), "=r"(d[6]),
            "=r"(d[7])
          : "r"(lane_base + mxq::kColD + 16u * p_buf)
          : "memory");
      asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
      const int64_t i_g = (int64_t)p_pg * kPageTokens + 32 * warp + lane;
      if (i_g < p_len) {
#pragma unroll
        for (int qq = 0; qq < Q; ++qq) {
          const int64_t p = (int64_t)p_len - Q + qq;
          a.scores[((int64_t)p_seq * Q + qq) * a.ld + i_g] =
              (i_g <= p) ? __uint_as_float(d[qq]) : -INFINITY;
        }
      }
      mxq::tc_fence_before();
    };

    for (int kk = 0; kk < n; ++kk) {
      const int st = kk % S, round = kk / S;
      bool landed = false;
      for (uint32_t i = 0; i < kWaitPolls && !landed; ++i) {
        landed = mbar_test(smem_addr(&ring.full[st]), round & 1);
        if (!landed && *ring.abort_flag) break;
      }
      if (!mxq::all_consumers(landed && !bad)) {
        failed = true;
        break;
      }
      // the producer's 8-byte copies and bulk copies are visible from here; make
      // them visible to the tensor core's reads too
      asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
      const int seq = ring.seq[st], pg = ring.page[st], L = ring.len[st];
      const bool ok = ring.ok[st] != 0;
      const uint8_t* stage = ring.base + st * ring.stage_bytes;
      if (ok && seq != cur_seq && pending) read_back();  // the B tile is about to change
      if (ok) {
        if (seq != cur_seq) {
          set_queries<Q>(reinterpret_cast<const uint16_t*>(stage + kStageDataBytes), region, tm,
                         tid, warp, lane);
          cur_seq = seq;
        }
        const uint32_t buf = groups & 1u;
        // this lane quarter's key scale words: row 32*warp + lane, column + warp
        const uint32_t sw =
            *reinterpret_cast<const uint32_t*>(stage + mxq::kATileBytes + 4 * (32 * warp + lane));
        mxq::tmem_st1(lane_base + mxq::kColSfa + 4u * buf + warp, sw);
        asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
        mxq::tc_fence_before();
        mxq::named_sync();
        if (tid == 0) {
          mxq::tc_fence_after();
          const uint32_t a_addr = smem_addr(stage);
#pragma unroll
          for (uint32_t kb = 0; kb < 4; ++kb) {
            const uint64_t ad = mxq::smem_desc_sw128(a_addr + kb * 32);
            const uint64_t bd = mxq::smem_desc(b_addr + kb * 256, 128, 1024);
            asm volatile(
                "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
                " tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, "
                "%2, %3, [%4], [%5], p;\n}\n" ::"r"(tm + mxq::kColD + 16u * buf),
                "l"(ad), "l"(bd), "r"(mxq::idesc(kb)), "r"(tm + mxq::kColSfa + 4u * buf),
                "r"(tm + mxq::kColSfb), "r"(kb)
                : "memory");
          }
          mxq::commit(smem_addr(&mma_bar[buf]));
          mxq::commit(smem_addr(&ring.empty[st]));  // the stage is free once the group is done
        }
        ++groups;
        running |= 1u << buf;
      } else if (tid == 0) {
        mbar_arrive(smem_addr(&ring.empty[st]));
      }
      if (pending) read_back();
      if (ok) {
        pending = true;
        p_seq = seq;
        p_pg = pg;
        p_len = L;
        p_buf = (groups - 1u) & 1u;
      }
    }
    if (!failed && pending) read_back();
    if (failed || bad) {
      flag(a.status, MX4_STATUS_TIMEOUT);
      *ring.abort_flag = 1;
    }
    // teardown (every consumer gets here): no MMA group may still run when the
    // tensor memory is freed (a buffer holds at most one group not waited for)
    for (uint32_t b = 0; b < 2; ++b)
      if (((running >> b) & 1u) && !mbar_wait(smem_addr(&mma_bar[b]), (phases >> b) & 1u) &&
          tid == 0)
        flag(a.status, MX4_STATUS_TIMEOUT);
    mxq::tc_fence_before();
    mxq::named_sync();
    mxq::tc_fence_after();
    if (warp == 0)
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tm),
                   "r"(mxq::kTmemCols)
                   : "memory");
  }
};

// The pool's data rows as a 3-d tensor for the tensor copy: 128 4-bit elements a
// row (64 bytes), 128 rows a page (64 bytes apart), num_pages pages (page_stride
// apart); a box is one page.  The 4-bit type writes 16 elements to each 16-byte
// slot.  Needs the pool 32-byte aligned and the page stride a multiple of 32.
// The encoder is the driver's, found through the runtime (no link to the driver
// library).
static cudaError_t encode_pool(const uint8_t* pages, int64_t page_stride, int64_t num_pages,
                               CUtensorMap* tm) {
  static PFN_cuTensorMapEncodeTiled_v12000 enc = [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      fn = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {(cuuint64_t)2 * kRowDataBytes, (cuuint64_t)kPageTokens,
                              (cuuint64_t)num_pages};
  const cuuint64_t strides[2] = {(cuuint64_t)kRowDataBytes, (cuuint64_t)page_stride};
  const cuuint32_t box[3] = {2 * kRowDataBytes, kPageTokens, 1};
  const cuuint32_t elem_strides[3] = {1, 1, 1};
  const CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3,
                         const_cast<uint8_t*>(pages), dims, strides, box, elem_strides,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_index_score_mxq(const uint16_t* iq, int q, const uint8_t* idx_pages,
                                   int64_t idx_page_stride, int64_t num_pages,
                                   const int32_t* block_table, int B, int64_t bt_width,
                                   const int32_t* seq_lens, float* scores, int64_t ld,
                                   uint32_t* status, int num_sms, cudaStream_t stream) {
  ScoreArgs a{iq, idx_pages, idx_page_stride, num_pages, block_table, B, bt_width,
              seq_lens, scores, ld, status, 1.f, {}};
  if (cudaError_t e = encode_pool(idx_pages, idx_page_stride, num_pages, &a.tmap)) return e;
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
