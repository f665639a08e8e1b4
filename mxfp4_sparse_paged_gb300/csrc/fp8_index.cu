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
// index_score_fp8_kernel: the same pipeline as the MXFP4 scorer -- pages of all
// sequences cut into equal contiguous ranges, one per CTA; warp 4 streams each
// page plus the sequence's index-q rows into a 4-stage shared-memory ring with
// bulk copies completing on mbarriers (bounded waits, drained on exit); warps
// 0-3 consume two 16-row tiles each.  Tile math on the tensor cores
// (mma m16n8k16, f16 in, fp32 accumulate): A = 16 key rows decoded by the
// hardware e4m3 -> f16 conversion (exact), thread t of a quad owning dims
// 32t .. 32t+31; B = index-q, bf16 scaled into f16 by a power of two (exact),
// output column n = query n.  The score is C * 2^-sigma * S.
#include <cuda_fp8.h>

#include "common.cuh"

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

constexpr int kF8Consumers = 4;
constexpr int kF8Threads = (kF8Consumers + 1) * 32;
constexpr int kF8Stages = 4;
constexpr int kF8MaxQ = 8;
constexpr int kF8StageBytes = kFp8PageBytes + kF8MaxQ * kHeadDim * 2;  // 18432
constexpr int kF8MaxBatch = 2048;                                       // sequences per launch
static_assert(kF8StageBytes % 16 == 0, "bulk-copy alignment");

struct F8ScoreSmem {
  uint8_t stage[kF8Stages][kF8StageBytes];
  int pref[kF8MaxBatch];  // inclusive prefix sum of pages per sequence
  int info_seq[kF8Stages];
  int info_page[kF8Stages];
  int info_len[kF8Stages];
  int info_ok[kF8Stages];
  int warp_sum[kF8Threads / 32];
  unsigned long long full[kF8Stages];
  unsigned long long empty[kF8Stages];
  volatile int abort_flag;
  int issued;  // pages whose copies (or bare arrival) the producer has issued
};

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

template <int Q>
__global__ void __launch_bounds__(kF8Threads, 2)
index_score_fp8_kernel(const uint16_t* __restrict__ iq, const uint8_t* __restrict__ pages,
                       int64_t page_stride, int64_t num_pages,
                       const int32_t* __restrict__ block_table, int B, int64_t bt_width,
                       const int32_t* __restrict__ seq_lens, float scale,
                       float* __restrict__ scores, int64_t ld, uint32_t* status) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  F8ScoreSmem& s = *reinterpret_cast<F8ScoreSmem*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_launch_dependents();

  // ---- pages per sequence and their prefix sum (contiguous segment per thread)
  {
    const int per = (B + kF8Threads - 1) / kF8Threads;
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
    for (int i = 0; i < kF8Stages; ++i) {
      mbar_init(smem_addr(&s.full[i]), 1);
      mbar_init(smem_addr(&s.empty[i]), kF8Consumers);
    }
    s.abort_flag = 0;
    s.issued = 0;
    fence_barrier_init();
  }
  __syncthreads();
  pdl_wait();  // pages (written by the insert) and scores are touched from here on

  const int total = B > 0 ? s.pref[B - 1] : 0;
  const int G = gridDim.x;
  const int p0 = (int)((int64_t)total * blockIdx.x / G);
  const int n = (int)((int64_t)total * (blockIdx.x + 1) / G) - p0;

  if (warp == kF8Consumers) {
    // ================= producer
    for (int base = 0; base < n; base += 32) {
      if (__any_sync(0xFFFFFFFFu, s.abort_flag != 0)) break;
      const int k = base + lane;
      int seqk = 0, jk = 0, lenk = 0, okk = 0;
      const uint8_t* src = pages;
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
        else src = pages + (int64_t)pid * page_stride;
      }
      const int cnt = min(32, n - base);
      for (int l = 0; l < cnt; ++l) {
        if (lane == l) {
          const int kk = base + l, st = kk % kF8Stages, round = kk / kF8Stages;
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
              mbar_arrive_expect_tx(fb, kFp8PageBytes + Q * kHeadDim * 2);
              bulk_copy_g2s(smem_addr(&s.stage[st][0]), src, kFp8PageBytes, fb);
              bulk_copy_g2s(smem_addr(&s.stage[st][kFp8PageBytes]),
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
      for (int kk = max(0, iss - kF8Stages); kk < iss; ++kk)
        if (!mbar_wait(smem_addr(&s.full[kk % kF8Stages]), (kk / kF8Stages) & 1))
          flag(status, MX4_STATUS_TIMEOUT);
    }
    return;
  }

  // ================= consumers
  const int g = lane >> 2, tig = lane & 3;
  // Rows g and g+8 of a tile are 128 B apart (the same banks): a thread of an odd
  // row reads the two 16-byte halves of its 32 bytes in the other order, so the
  // 8 lanes of a quarter-warp hit all 32 banks, then swaps them back in registers.
  const int swap = g & 1;
  uint32_t breg[8][2];
  float osc[2] = {scale, scale};  // 2^-sigma * S of this thread's queries 2 tig, 2 tig + 1
  int cur_seq = -1;

  for (int kk = 0; kk < n; ++kk) {
    const int st = kk % kF8Stages, round = kk / kF8Stages;
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
        // so the largest magnitude sits near 2^14 (bf16 -> f16 then exact)
        const uint16_t* qs = reinterpret_cast<const uint16_t*>(page + kFp8PageBytes);
        float f = 0.f;  // 2^sigma of query g (0 for a column past the queries)
#pragma unroll
        for (int qq = 0; qq < Q; ++qq) {
          const uint2 v = *reinterpret_cast<const uint2*>(qs + qq * kHeadDim + 4 * lane);
          uint32_t a = max(max((v.x << 17) >> 1, v.x & 0x7FFF0000u),
                           max((v.y << 17) >> 1, v.y & 0x7FFF0000u));
          a = __reduce_max_sync(0xFFFFFFFFu, a);
          const int sigma = (a == 0u) ? 0 : min(127, max(-126, 14 - ((int)(a >> 23) - 127)));
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
        cur_seq = seq;
      }
#pragma unroll
      for (int tt = 0; tt < kPageTokens / 16 / kF8Consumers; ++tt) {
        const int r0 = (warp + kF8Consumers * tt) * 16;
        const uint8_t* rx = page + (r0 + g) * kFp8RowBytes + 32 * tig;
        const uint8_t* ry = rx + 8 * kFp8RowBytes;
        uint4 x0 = *reinterpret_cast<const uint4*>(rx + 16 * swap);
        uint4 x1 = *reinterpret_cast<const uint4*>(rx + 16 * (1 - swap));
        uint4 y0 = *reinterpret_cast<const uint4*>(ry + 16 * swap);
        uint4 y1 = *reinterpret_cast<const uint4*>(ry + 16 * (1 - swap));
        if (swap) {
          const uint4 tx = x0, ty = y0;
          x0 = x1; x1 = tx;
          y0 = y1; y1 = ty;
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
        const int64_t i_g = (int64_t)pg * kPageTokens + r0 + g;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int qq = 2 * tig + h;
          if (qq < Q) {
            const int64_t p = (int64_t)L - Q + qq;
            float* out = scores + ((int64_t)seq * Q + qq) * ld;
            if (i_g < L) out[i_g] = (i_g <= p) ? c[h] * osc[h] : -INFINITY;
            if (i_g + 8 < L) out[i_g + 8] = (i_g + 8 <= p) ? c[2 + h] * osc[h] : -INFINITY;
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&s.empty[st]));
  }
}

template <int Q>
static cudaError_t launch_fp8_q(int grid, const uint16_t* iq, const uint8_t* pages,
                                int64_t page_stride, int64_t num_pages,
                                const int32_t* block_table, int B, int64_t bt_width,
                                const int32_t* seq_lens, float scale, float* scores, int64_t ld,
                                uint32_t* status, cudaStream_t stream) {
  const int smem = (int)sizeof(F8ScoreSmem);
  cudaError_t err = cudaFuncSetAttribute(index_score_fp8_kernel<Q>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  for (int b0 = 0; b0 < B; b0 += kF8MaxBatch) {
    const int nb = min(kF8MaxBatch, B - b0);
    err = launch_pdl(index_score_fp8_kernel<Q>, dim3(grid), dim3(kF8Threads), smem, stream,
                     iq + (int64_t)b0 * Q * kHeadDim, pages, page_stride, num_pages,
                     block_table + (int64_t)b0 * bt_width, nb, bt_width, seq_lens + b0, scale,
                     scores + (int64_t)b0 * Q * ld, ld, status);
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

cudaError_t launch_index_score_fp8(const uint16_t* iq, int q, const uint8_t* pages,
                                   int64_t page_stride, int64_t num_pages,
                                   const int32_t* block_table, int B, int64_t bt_width,
                                   const int32_t* seq_lens, float scale, float* scores,
                                   int64_t ld, uint32_t* status, int num_sms,
                                   cudaStream_t stream) {
  const int grid = num_sms * 2;  // 2 CTAs of ~82 KB shared memory per SM
#define MX4_FP8_Q(QQ)                                                                       \
  case QQ:                                                                                 \
    return launch_fp8_q<QQ>(grid, iq, pages, page_stride, num_pages, block_table, B,       \
                            bt_width, seq_lens, scale, scores, ld, status, stream);
  switch (q) {
    MX4_FP8_Q(1)
    MX4_FP8_Q(2)
    MX4_FP8_Q(3)
    MX4_FP8_Q(4)
    MX4_FP8_Q(5)
    MX4_FP8_Q(6)
    MX4_FP8_Q(7)
    MX4_FP8_Q(8)
    default: return cudaErrorInvalidValue;
  }
#undef MX4_FP8_Q
}

}  // namespace mx4
