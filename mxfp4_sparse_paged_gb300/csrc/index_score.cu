// index_score: dot every cached index key of a sequence with the index-q head
// of each of its decode tokens.
//
// The index key cache is [pages, 8704] ("vllm.models.minimax_m3.amd.ops.
// mxfp4_pages", mxfp4_page_views: the [pages, 128, 64] / [pages, 128, 4] pair
// the index scorers read); pages are found through the block table shared with
// the K/V cache ("vllm.models.minimax_m3.amd.mono.dispatch", _slots_shared).
//
// Work: the pages of all sequences, flattened in order, are cut into equal
// contiguous ranges, one per CTA (a block-wide prefix sum over seq_lens in
// shared memory maps a flat page number to (sequence, page)).  All q decode
// tokens of a sequence are scored in one pass over its pages.
//
// Pipeline: warp 4 is the producer.  It resolves pages through the block table
// (32 lanes at a time) and streams each 8704-byte page, plus the sequence's
// index-q rows, into a 4-stage shared-memory ring with bulk copies (TMA engine)
// that complete on the stage's "full" mbarrier.  Warps 0-3 consume: each takes
// two 16-row tiles of the page.  Four CTAs run per SM.
//
// Math (per tile, tensor cores): A = 16 index-key rows x 128 dims, decoded by
// the hardware e2m1 -> f16 conversion (exact); thread t of a quad owns the 32
// dims of scale block t.  B = index-q, bf16 scaled by a power of two into f16
// (exact), laid out so that output column n = 4*query + block: a column only
// sees the dims of its own block, so C holds per-block partial dots.  The
// scores are then sum_b C[row][4q+b] * 2^(scale_b - 127) in fp32 (exact
// scaling), combined across the quad with one shuffle.
#include "common.cuh"

namespace mx4 {

constexpr int kScoreConsumers = 4;
constexpr int kScoreThreads = (kScoreConsumers + 1) * 32;
constexpr int kScoreStages = 4;
constexpr int kMaxQ = 8;
constexpr int kStageIqBytes = kMaxQ * kHeadDim * 2;
constexpr int kScoreStageBytes = kPageBytes + kStageIqBytes;  // 10752, a multiple of 16
constexpr int kScoreMaxBatch = 2048;                           // sequences per launch
static_assert(kScoreStageBytes % 16 == 0, "bulk-copy alignment");

struct ScoreSmem {
  uint8_t stage[kScoreStages][kScoreStageBytes];
  int pref[kScoreMaxBatch];  // inclusive prefix sum of pages per sequence
  int info_seq[kScoreStages];
  int info_page[kScoreStages];
  int info_len[kScoreStages];
  int info_ok[kScoreStages];
  int warp_sum[kScoreThreads / 32];
  unsigned long long full[kScoreStages];
  unsigned long long empty[kScoreStages];
  volatile int abort_flag;
  int issued;  // pages whose copies (or bare arrival) the producer has issued
};

__device__ __forceinline__ float e8m0_fast(uint32_t word, uint32_t sel) {
  return fmaxf(__uint_as_float(__byte_perm(word, 0u, sel) >> 1), 0x1p-127f);
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

template <int Q>
__global__ void __launch_bounds__(kScoreThreads)
index_score_kernel(const uint16_t* __restrict__ iq, const uint8_t* __restrict__ idx_pages,
                   int64_t idx_page_stride, int64_t num_pages,
                   const int32_t* __restrict__ block_table, int B, int64_t bt_width,
                   const int32_t* __restrict__ seq_lens, float* __restrict__ scores, int64_t ld,
                   uint32_t* status) {
  constexpr int NT = (Q + 1) / 2;  // n8 tiles: 4 block-columns per query
  extern __shared__ __align__(128) uint8_t smem_raw[];
  ScoreSmem& s = *reinterpret_cast<ScoreSmem*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_launch_dependents();

  // ---- pages per sequence and their prefix sum (contiguous segment per thread)
  {
    const int per = (B + kScoreThreads - 1) / kScoreThreads;
    const int s0 = min(B, tid * per), s1 = min(B, s0 + per);
    int sum = 0;
    for (int sq = s0; sq < s1; ++sq) {
      const int64_t L = seq_lens[sq];
      const bool ok = L >= Q && L <= bt_width * kPageTokens && L <= ld;
      if (!ok && blockIdx.x == 0) flag(status, MX4_STATUS_BAD_LEN);
      sum += ok ? (int)((L + kPageTokens - 1) / kPageTokens) : 0;
    }
    int inc = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
      if (lane >= o) inc += y;
    }
    if (lane == 31) s.warp_sum[warp] = inc;
    __syncthreads();
    int before = inc - sum;
    for (int w = 0; w < warp; ++w) before += s.warp_sum[w];
    for (int sq = s0; sq < s1; ++sq) {
      const int64_t L = seq_lens[sq];
      const bool ok = L >= Q && L <= bt_width * kPageTokens && L <= ld;
      before += ok ? (int)((L + kPageTokens - 1) / kPageTokens) : 0;
      s.pref[sq] = before;
    }
  }
  if (tid == 0) {
    for (int i = 0; i < kScoreStages; ++i) {
      mbar_init(smem_addr(&s.full[i]), 1);
      mbar_init(smem_addr(&s.empty[i]), kScoreConsumers);
    }
    s.abort_flag = 0;
    s.issued = 0;
    fence_barrier_init();
  }
  __syncthreads();
  pdl_wait();  // pages (written by mx4_insert) and scores are touched from here on

  const int total = B > 0 ? s.pref[B - 1] : 0;
  const int G = gridDim.x;
  const int p0 = (int)((int64_t)total * blockIdx.x / G);
  const int n = (int)((int64_t)total * (blockIdx.x + 1) / G) - p0;

  if (warp == kScoreConsumers) {
    // ================= producer
    for (int base = 0; base < n; base += 32) {
      if (__any_sync(0xFFFFFFFFu, s.abort_flag != 0)) break;
      const int k = base + lane;
      int seqk = 0, jk = 0, lenk = 0, okk = 0;
      const uint8_t* src = idx_pages;
      if (k < n) {
        const int P = p0 + k;
        int lo = 0, hi = B - 1;
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (s.pref[mid] > P) hi = mid; else lo = mid + 1;
        }
        seqk = lo;
        jk = P - (lo > 0 ? s.pref[lo - 1] : 0);
        lenk = seq_lens[seqk];
        const int32_t pid = block_table[(int64_t)seqk * bt_width + jk];
        okk = (pid >= 0 && pid < num_pages) ? 1 : 0;
        if (!okk) flag(status, MX4_STATUS_BAD_PAGE);
        else src = idx_pages + (int64_t)pid * idx_page_stride;
      }
      const int cnt = min(32, n - base);
      for (int l = 0; l < cnt; ++l) {
        if (lane == l) {
          const int kk = base + l, st = kk % kScoreStages, round = kk / kScoreStages;
          bool go = !s.abort_flag;
          if (go && round > 0 && !mbar_wait(smem_addr(&s.empty[st]), (round - 1) & 1)) {
            flag(status, MX4_STATUS_TIMEOUT);
            s.abort_flag = 1;
            go = false;
          }
          if (go) {
            s.info_seq[st] = seqk;
            s.info_page[st] = jk;
            s.info_len[st] = lenk;
            s.info_ok[st] = okk;
            const uint32_t fb = smem_addr(&s.full[st]);
            if (okk) {
              mbar_arrive_expect_tx(fb, kPageBytes + Q * kHeadDim * 2);
              bulk_copy_g2s(smem_addr(&s.stage[st][0]), src, kPageBytes, fb);
              bulk_copy_g2s(smem_addr(&s.stage[st][kPageBytes]),
                            iq + (int64_t)seqk * Q * kHeadDim, Q * kHeadDim * 2, fb);
            } else {
              mbar_arrive(fb);
            }
            s.issued = kk + 1;
          }
        }
        __syncwarp();
      }
    }
    // Drain: wait (bounded) until the copies of the last stages issued have landed,
    // so none is in flight when the CTA exits, also after a time-out.
    __syncwarp();
    if (lane == 0) {
      const int iss = s.issued;
      for (int kk = max(0, iss - kScoreStages); kk < iss; ++kk)
        if (!mbar_wait(smem_addr(&s.full[kk % kScoreStages]), (kk / kScoreStages) & 1))
          flag(status, MX4_STATUS_TIMEOUT);
    }
    return;
  }

  // ================= consumers
  const int g = lane >> 2, tig = lane & 3;
  // byte-permute selectors: scale byte 2 (tig & 1) (+1) of a word to byte 3, zeros below
  const uint32_t sel0 = 0x0444u | ((uint32_t)(2 * (tig & 1)) << 12);
  const uint32_t sel1 = 0x0444u | ((uint32_t)(2 * (tig & 1) + 1) << 12);
  uint32_t breg[NT][8][2];
  float inv_scale[Q];
  int cur_seq = -1;
#pragma unroll
  for (int qq = 0; qq < Q; ++qq) inv_scale[qq] = 1.f;

  for (int kk = 0; kk < n; ++kk) {
    const int st = kk % kScoreStages, round = kk / kScoreStages;
    bool landed = false;
    for (uint32_t i = 0; i < kWaitPolls && !landed; ++i) {
      landed = mbar_test(smem_addr(&s.full[st]), round & 1);
      if (!landed && s.abort_flag) break;
    }
    if (!__all_sync(0xFFFFFFFFu, landed)) {
      if (lane == 0) flag(status, MX4_STATUS_TIMEOUT);
      s.abort_flag = 1;
      break;
    }
    const int seq = s.info_seq[st], pg = s.info_page[st], L = s.info_len[st];
    if (s.info_ok[st]) {
      const uint8_t* page = &s.stage[st][0];
      if (seq != cur_seq) {
        // index-q of this sequence -> f16 B fragments, scaled by 2^sigma per query
        const uint16_t* qs = reinterpret_cast<const uint16_t*>(page + kPageBytes);
        float sc[Q];
#pragma unroll
        for (int qq = 0; qq < Q; ++qq) {
          const uint2 v = *reinterpret_cast<const uint2*>(qs + qq * kHeadDim + 4 * lane);
          uint32_t a = max(max((v.x << 17) >> 1, v.x & 0x7FFF0000u),
                           max((v.y << 17) >> 1, v.y & 0x7FFF0000u));
          a = __reduce_max_sync(0xFFFFFFFFu, a);
          const int sigma = (a == 0u) ? 0 : min(127, max(-126, 14 - ((int)(a >> 23) - 127)));
          sc[qq] = __uint_as_float((uint32_t)(127 + sigma) << 23);
          inv_scale[qq] = __uint_as_float((uint32_t)(127 - sigma) << 23);
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int qq = 2 * nt + (g >> 2);
          const bool active = ((g & 3) == tig) && qq < Q;
          const uint16_t* qv = qs + (qq < Q ? qq : 0) * kHeadDim + 32 * tig;
          const float f = active ? sc[qq < Q ? qq : 0] : 0.f;
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
        cur_seq = seq;
      }
#pragma unroll
      for (int tt = 0; tt < kPageTokens / 16 / kScoreConsumers; ++tt) {
        const int r0 = (warp + kScoreConsumers * tt) * 16;
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
        const int64_t i_g = (int64_t)pg * kPageTokens + r0 + g;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float vg = c[nt][0] * sx0 + c[nt][1] * sx1;
          float vg8 = c[nt][2] * sy0 + c[nt][3] * sy1;
          vg += __shfl_xor_sync(0xFFFFFFFFu, vg, 1);
          vg8 += __shfl_xor_sync(0xFFFFFFFFu, vg8, 1);
          const int qq = 2 * nt + (tig >> 1);
          if ((tig & 1) == 0 && qq < Q) {
            const float isc = inv_scale[qq < Q ? qq : 0];
            const int64_t p = (int64_t)L - Q + qq;
            float* out = scores + ((int64_t)seq * Q + qq) * ld;
            if (i_g < L) out[i_g] = (i_g <= p) ? vg * isc : -INFINITY;
            if (i_g + 8 < L) out[i_g + 8] = (i_g + 8 <= p) ? vg8 * isc : -INFINITY;
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&s.empty[st]));
  }
}

template <int Q>
static cudaError_t launch_q(int grid, const uint16_t* iq, const uint8_t* idx_pages,
                            int64_t idx_page_stride, int64_t num_pages,
                            const int32_t* block_table, int B, int64_t bt_width,
                            const int32_t* seq_lens, float* scores, int64_t ld, uint32_t* status,
                            cudaStream_t stream) {
  const int smem = (int)sizeof(ScoreSmem);
  cudaError_t err = cudaFuncSetAttribute(index_score_kernel<Q>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  for (int b0 = 0; b0 < B; b0 += kScoreMaxBatch) {
    const int nb = min(kScoreMaxBatch, B - b0);
    err = launch_pdl(index_score_kernel<Q>, dim3(grid), dim3(kScoreThreads), smem, stream,
                     iq + (int64_t)b0 * Q * kHeadDim, idx_pages, idx_page_stride, num_pages,
                     block_table + (int64_t)b0 * bt_width, nb, bt_width, seq_lens + b0,
                     scores + (int64_t)b0 * Q * ld, ld, status);
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

cudaError_t launch_index_score(const uint16_t* iq, int q, const uint8_t* idx_pages,
                               int64_t idx_page_stride, int64_t num_pages,
                               const int32_t* block_table, int B, int64_t bt_width,
                               const int32_t* seq_lens, float* scores, int64_t ld,
                               uint32_t* status, int num_sms, cudaStream_t stream) {
  const int grid = num_sms * 4;  // 4 CTAs of ~51 KB shared memory per SM
  switch (q) {
    case 1: return launch_q<1>(grid, iq, idx_pages, idx_page_stride, num_pages, block_table, B,
                               bt_width, seq_lens, scores, ld, status, stream);
    case 2: return launch_q<2>(grid, iq, idx_pages, idx_page_stride, num_pages, block_table, B,
                               bt_width, seq_lens, scores, ld, status, stream);
    case 3: return launch_q<3>(grid, iq, idx_pages, idx_page_stride, num_pages, block_table, B,
                               bt_width, seq_lens, scores, ld, status, stream);
    case 4: return launch_q<4>(grid, iq, idx_pages, idx_page_stride, num_pages, block_table, B,
                               bt_width, seq_lens, scores, ld, status, stream);
    case 5: return launch_q<5>(grid, iq, idx_pages, idx_page_stride, num_pages, block_table, B,
                               bt_width, seq_lens, scores, ld, status, stream);
    case 6: return launch_q<6>(grid, iq, idx_pages, idx_page_stride, num_pages, block_table, B,
                               bt_width, seq_lens, scores, ld, status, stream);
    case 7: return launch_q<7>(grid, iq, idx_pages, idx_page_stride, num_pages, block_table, B,
                               bt_width, seq_lens, scores, ld, status, stream);
    case 8: return launch_q<8>(grid, iq, idx_pages, idx_page_stride, num_pages, block_table, B,
                               bt_width, seq_lens, scores, ld, status, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mx4
