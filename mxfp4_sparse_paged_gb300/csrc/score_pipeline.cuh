// The index-scorer pipeline shared by the MXFP4 index-K cache ("vllm.models.
// minimax_m3.amd.ops.mxfp4_pages": [pages, 128, 64] e2m1 rows + [pages, 128, 4]
// e8m0 scales) and the fp8 one of the other revision ("vllm.models.minimax_m3.
// amd.mono.weights", SparseMoeLayer.index_cache).  Pages are found through the
// block table shared with the K/V cache ("vllm.models.minimax_m3.amd.mono.
// dispatch", _slots_shared).
//
// Work: the pages of all sequences, flattened in order, are cut into equal
// contiguous ranges, one per CTA (a block-wide prefix sum over seq_lens in
// shared memory maps a flat page number to (sequence, page)).  All q decode
// tokens of a sequence are scored in one pass over its pages.
//
// The last warp is the producer: it resolves pages through the block table (32
// lanes at a time) and streams each page, plus the sequence's index-q rows, into
// a ring of shared-memory stages with bulk copies (TMA engine) that complete on
// the stage's "full" mbarrier.  The other warps consume, one 16-row tile of each
// page per warp (the format's tile math), and arrive on the stage's "empty"
// mbarrier.  Every wait is bounded: on time-out the kernel sets
// MX4_STATUS_TIMEOUT, stops, and drains the copies in flight before exiting.
//
// A format whose tile math takes a whole page at once (kWholePage: the
// block-scaled tensor-core scorer) gets a region of kExtraBytes of shared memory
// for its operand tiles and runs its own producer and consumer loops over the
// same stage ring, prefix scan, page resolution and drain.  A format sets the
// bytes of a stage before the index-q rows (kStageDataBytes) and the arrival
// counts of its full and empty barriers.
#pragma once

#include <algorithm>

#include <cuda.h>  // CUtensorMap (a type only: the map is encoded through the runtime)

#include "common.cuh"

namespace mx4 {

constexpr int kScoreMaxBatch = 2048;  // sequences per launch

// Order-preserving uint32 key of an fp32 score (larger score -> larger key); -0
// and +0 share one key.  The top-k selection uses the same map.
__device__ __forceinline__ uint32_t score_key(float f) {
  const uint32_t u = __float_as_uint(f + 0.0f);  // -0 + 0 = +0
  return u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
}

struct ScoreArgs {
  const uint16_t* iq;          // bf16 [B * Q, 128]
  const uint8_t* pages;        // page p at pages + p * page_stride
  int64_t page_stride;
  int64_t num_pages;
  const int32_t* block_table;  // [B, bt_width]
  int B;
  int64_t bt_width;
  const int32_t* seq_lens;     // [B]
  float* scores;               // [B * Q, ld]
  int64_t ld;
  uint32_t* status;
  float scale;                 // the fp8 cache's scale (1 for MXFP4)
  CUtensorMap tmap;            // the pool as a tensor map, for a format that loads pages by one
};

// Shared-memory layout of the kernel, in bytes: format region | stages |
// barriers | stage info | warp sums, flags | per-sequence page prefix [B].
template <class F, int Q>
struct ScoreLayout {
  static constexpr int kStageBytes =
      (F::kStageDataBytes + Q * kHeadDim * 2 + F::kStageAlign - 1) / F::kStageAlign * F::kStageAlign;
  static_assert(kStageBytes % 16 == 0, "bulk-copy alignment");
  static_assert(F::kExtraBytes % 128 == 0 && F::kExtraBytes % F::kStageAlign == 0,
                "format region alignment");
  static constexpr int kStagesOff = F::kExtraBytes;
  static constexpr int kBarOff = kStagesOff + F::kStages * kStageBytes;  // full[S], empty[S]
  static constexpr int kInfoOff = kBarOff + 2 * F::kStages * 8;
  static constexpr int kWarpSumOff = kInfoOff + 4 * F::kStages * 4;
  static constexpr int kFlagOff = kWarpSumOff + 32 * 4;  // abort, issued
  static constexpr int kPrefOff = (kFlagOff + 8 + 15) / 16 * 16;
  // (plus the slack that aligns the dynamic shared memory to a stage alignment above 128)
  static size_t bytes(int B) {
    return (size_t)kPrefOff + (size_t)B * 4 + (F::kStageAlign > 128 ? F::kStageAlign : 0);
  }
};

// The stage ring as a whole-page format sees it: stage st holds a page (and the
// sequence's index-q rows after kStageDataBytes) once full[st] completes its
// phase; the consumer frees it with the format's arrivals on empty[st].
struct StageRing {
  uint8_t* base;
  int stage_bytes;
  uint64_t* full;
  uint64_t* empty;
  int* seq;
  int* page;
  int* len;
  int* ok;
  volatile int* abort_flag;
  int* issued;  // stages the producer has filled (for the drain)
};

// Page P of the flattened page list: its sequence, its page number within the
// sequence, the sequence's length and its address.  ok = 0 (and the status bit
// set) for a page id outside the pool.
struct PageRef {
  const uint8_t* src;
  int seq, page, len, ok;
  int pid;  // the page id (0 when not ok)
};
__device__ __forceinline__ PageRef resolve_page(const ScoreArgs& a, const int* pref, int P) {
  int lo = 0, hi = a.B - 1;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (pref[mid] > P) hi = mid; else lo = mid + 1;
  }
  PageRef r;
  r.seq = lo;
  r.page = P - (lo > 0 ? pref[lo - 1] : 0);
  r.len = a.seq_lens[lo];
  const int32_t pid = a.block_table[(int64_t)lo * a.bt_width + r.page];
  r.ok = (pid >= 0 && pid < a.num_pages) ? 1 : 0;
  if (!r.ok) flag(a.status, MX4_STATUS_BAD_PAGE);
  r.src = r.ok ? a.pages + (int64_t)pid * a.page_stride : a.pages;
  r.pid = r.ok ? pid : 0;
  return r;
}

template <class F, int Q>
__global__ void __launch_bounds__((F::kConsumers + 1) * 32, F::ctas_per_sm(Q))
score_kernel(const __grid_constant__ ScoreArgs a) {
  using Lay = ScoreLayout<F, Q>;
  constexpr int S = F::kStages, NC = F::kConsumers, NTHR = (NC + 1) * 32;
  extern __shared__ __align__(128) uint8_t smem_dyn[];
  uint8_t* const smem_raw =
      F::kStageAlign > 128
          ? reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + F::kStageAlign - 1) &
                                       ~static_cast<uintptr_t>(F::kStageAlign - 1))
          : smem_dyn;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem_raw + Lay::kBarOff);
  uint64_t* empty = full + S;
  int* info_seq = reinterpret_cast<int*>(smem_raw + Lay::kInfoOff);
  int* info_page = info_seq + S;
  int* info_len = info_page + S;
  int* info_ok = info_len + S;
  int* warp_sum = reinterpret_cast<int*>(smem_raw + Lay::kWarpSumOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem_raw + Lay::kFlagOff);
  int* issued = reinterpret_cast<int*>(smem_raw + Lay::kFlagOff + 4);
  int* pref = reinterpret_cast<int*>(smem_raw + Lay::kPrefOff);
  const int B = a.B;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_launch_dependents();

  // ---- pages per sequence and their prefix sum (contiguous segment per thread)
  {
    const int per = (B + NTHR - 1) / NTHR;
    const int s0 = min(B, tid * per), s1 = min(B, s0 + per);
    int sum = 0;
    for (int sq = s0; sq < s1; ++sq) {
      const int64_t L = a.seq_lens[sq];
      const bool ok = L >= Q && L <= a.bt_width * kPageTokens && L <= a.ld;
      if (!ok && blockIdx.x == 0) flag(a.status, MX4_STATUS_BAD_LEN);
      sum += ok ? (int)((L + kPageTokens - 1) / kPageTokens) : 0;
    }
    int inc = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
      if (lane >= o) inc += y;
    }
    if (lane == 31) warp_sum[warp] = inc;
    __syncthreads();
    int before = inc - sum;
    for (int w = 0; w < warp; ++w) before += warp_sum[w];
    for (int sq = s0; sq < s1; ++sq) {
      const int64_t L = a.seq_lens[sq];
      const bool ok = L >= Q && L <= a.bt_width * kPageTokens && L <= a.ld;
      before += ok ? (int)((L + kPageTokens - 1) / kPageTokens) : 0;
      pref[sq] = before;
    }
  }
  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(smem_addr(&full[i]), F::kFullCount);
      mbar_init(smem_addr(&empty[i]), F::kEmptyCount);
    }
    *abort_flag = 0;
    *issued = 0;
    fence_barrier_init();
  }
  __syncthreads();
  pdl_wait();  // pages (written by the insert) and scores are touched from here on

  const int total = B > 0 ? pref[B - 1] : 0;
  const int G = gridDim.x;
  const int p0 = (int)((int64_t)total * blockIdx.x / G);
  const int n = (int)((int64_t)total * (blockIdx.x + 1) / G) - p0;

  const StageRing ring{smem_raw + Lay::kStagesOff, Lay::kStageBytes, full, empty, info_seq,
                       info_page, info_len, info_ok, abort_flag, issued};
  if (warp == NC) {
    // ================= producer
    if constexpr (F::kWholePage) {
      F::template produce<Q>(a, ring, pref, p0, n, lane);
    } else {
      for (int base = 0; base < n; base += 32) {
        if (__any_sync(0xFFFFFFFFu, *abort_flag != 0)) break;
        const int k = base + lane;
        PageRef pr{a.pages, -1, 0, 0, 0, 0};
        if (k < n) pr = resolve_page(a, pref, p0 + k);
        const int seqk = pr.seq, jk = pr.page, lenk = pr.len, okk = pr.ok;
        const uint8_t* src = pr.src;
        const int cnt = min(32, n - base);
        for (int l = 0; l < cnt; ++l) {
          if (lane == l) {
            const int kk = base + l, st = kk % S, round = kk / S;
            bool go = !*abort_flag;
            if (go && round > 0 && !mbar_wait(smem_addr(&empty[st]), (round - 1) & 1)) {
              flag(a.status, MX4_STATUS_TIMEOUT);
              *abort_flag = 1;
              go = false;
            }
            if (go) {
              info_seq[st] = seqk;
              info_page[st] = jk;
              info_len[st] = lenk;
              info_ok[st] = okk;
              const uint32_t fb = smem_addr(&full[st]);
              const uint32_t dst = smem_addr(smem_raw + Lay::kStagesOff + st * Lay::kStageBytes);
              if (okk) {
                mbar_arrive_expect_tx(fb, F::kPageBytes + Q * kHeadDim * 2);
                bulk_copy_g2s(dst, src, F::kPageBytes, fb);
                bulk_copy_g2s(dst + F::kPageBytes, a.iq + (int64_t)seqk * Q * kHeadDim,
                              Q * kHeadDim * 2, fb);
              } else {
                mbar_arrive(fb);
              }
              *issued = kk + 1;
            }
          }
          __syncwarp();
        }
      }
    }
    // Drain: wait (bounded) until the copies of the last stages issued have landed,
    // so none is in flight when the CTA exits, also after a time-out.
    __syncwarp();
    if (lane == 0) {
      const int iss = *issued;
      for (int kk = max(0, iss - S); kk < iss; ++kk)
        if (!mbar_wait(smem_addr(&full[kk % S]), (kk / S) & 1)) flag(a.status, MX4_STATUS_TIMEOUT);
    }
    return;
  }

  // ================= consumers
  if constexpr (F::kWholePage) {
    F::template consume<Q>(a, ring, smem_raw, n, warp, lane);
  } else {
    typename F::template Tile<Q> tile;
    int cur_seq = -1;
    for (int kk = 0; kk < n; ++kk) {
      const int st = kk % S, round = kk / S;
      bool landed = false;
      for (uint32_t i = 0; i < kWaitPolls && !landed; ++i) {
        landed = mbar_test(smem_addr(&full[st]), round & 1);
        if (!landed && *abort_flag) break;
      }
      if (!__all_sync(0xFFFFFFFFu, landed)) {
        if (lane == 0) flag(a.status, MX4_STATUS_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      const int seq = info_seq[st], pg = info_page[st], L = info_len[st];
      if (info_ok[st]) {
        const uint8_t* page = smem_raw + Lay::kStagesOff + st * Lay::kStageBytes;
        if (seq != cur_seq) {
          tile.set_queries(reinterpret_cast<const uint16_t*>(page + F::kPageBytes), lane, a.scale);
          cur_seq = seq;
        }
        // score of row r of this page for query qq: -inf past the token's position
        // (L - Q + qq); rows at or past L are not written.  With three or more
        // queries, the page's first score of query 0 and the limits relative to the
        // page are taken once per page (measured: faster for q = 4, slower for q = 1).
        float* const base = a.scores + (int64_t)seq * Q * a.ld + (int64_t)pg * kPageTokens;
        const int nrows = min(kPageTokens, L - pg * kPageTokens);
        const int last0 = L - Q - pg * kPageTokens;  // query 0's last finite row
        auto emit = [&](int qq, int r, float v) {
          if constexpr (Q >= 3) {
            if (r < nrows) base[qq * a.ld + r] = (r <= last0 + qq) ? v : -INFINITY;
          } else {
            const int64_t i_g = (int64_t)pg * kPageTokens + r;
            const int64_t p = (int64_t)L - Q + qq;
            if (i_g < L)
              a.scores[((int64_t)seq * Q + qq) * a.ld + i_g] = (i_g <= p) ? v : -INFINITY;
          }
        };
#pragma unroll
        for (int tt = 0; tt < kPageTokens / 16 / NC; ++tt)
          tile.run(page, (warp + NC * tt) * 16, lane, emit);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&empty[st]));
    }
  }
}

// CTAs of `kern` with `threads` threads and `smem` bytes of dynamic shared memory
// that fit on one SM of the current device at once.
inline cudaError_t resident_ctas(const void* kern, int threads, size_t smem, int* out) {
  cudaFuncAttributes fa;
  cudaError_t err = cudaFuncGetAttributes(&fa, kern);
  if (err != cudaSuccess) return err;
  int dev = 0, smem_sm = 0, reserved = 0, regs_sm = 0, threads_sm = 0, blocks_sm = 0;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  if ((err = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor,
                                    dev)) != cudaSuccess ||
      (err = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev)) !=
          cudaSuccess ||
      (err = cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev)) !=
          cudaSuccess ||
      (err = cudaDeviceGetAttribute(&threads_sm, cudaDevAttrMaxThreadsPerMultiProcessor, dev)) !=
          cudaSuccess ||
      (err = cudaDeviceGetAttribute(&blocks_sm, cudaDevAttrMaxBlocksPerMultiprocessor, dev)) !=
          cudaSuccess)
    return err;
  const size_t per_block = smem + fa.sharedSizeBytes + (size_t)reserved;
  const int warps = (threads + 31) / 32;
  const int regs_warp = (fa.numRegs * 32 + 255) / 256 * 256;  // allocated per warp, 256 at a time
  int n = blocks_sm;
  n = std::min(n, (int)((size_t)smem_sm / per_block));
  n = std::min(n, regs_warp > 0 ? regs_sm / (regs_warp * warps) : n);
  n = std::min(n, threads_sm / (warps * 32));
  *out = n;
  return cudaSuccess;
}

// Launch over batches of at most kScoreMaxBatch sequences (the prefix array).
template <class F, int Q>
cudaError_t launch_score(ScoreArgs a, int num_sms, cudaStream_t stream) {
  using Lay = ScoreLayout<F, Q>;
  auto kern = score_kernel<F, Q>;
  const int B = a.B;
  const size_t smem = Lay::bytes(min(B, kScoreMaxBatch));
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)Lay::bytes(kScoreMaxBatch));
  if (err != cudaSuccess) return err;
  // all of the SM's unified memory that can be shared memory (the stages are filled
  // by bulk and tensor copies, not through L1)
  err = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  if (err != cudaSuccess) return err;
  // CTAs per SM: the format's figure, or fewer when this launch's shared memory
  // (which grows with the batch) lets fewer reside, so the grid is one wave.  The
  // residency is taken from the SM's shared memory, registers and threads and the
  // kernel's own use of them.
  int resident = 0;
  err = resident_ctas(reinterpret_cast<const void*>(kern), (F::kConsumers + 1) * 32, smem,
                      &resident);
  if (err != cudaSuccess) return err;
  const int grid = num_sms * max(1, min(F::ctas_per_sm(Q), resident));
  for (int b0 = 0; b0 < B; b0 += kScoreMaxBatch) {
    ScoreArgs c = a;
    c.B = min(kScoreMaxBatch, B - b0);
    c.iq = a.iq + (int64_t)b0 * Q * kHeadDim;
    c.block_table = a.block_table + (int64_t)b0 * a.bt_width;
    c.seq_lens = a.seq_lens + b0;
    c.scores = a.scores + (int64_t)b0 * Q * a.ld;
    err = launch_pdl(kern, dim3(grid), dim3((F::kConsumers + 1) * 32), smem, stream, c);
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

}  // namespace mx4
