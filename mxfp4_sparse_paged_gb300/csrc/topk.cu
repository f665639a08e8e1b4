// topk_select: per decode token, the k cached tokens with the largest index
// scores (ties to the lower token index), returned in ascending index order.
//
// The selection step sits between the index scorer and the MXFP4 pa_decode
// reader ("vllm.models.minimax_m3.amd.ops.mxfp4_pages", module description:
// the scorers and pa_decode read the same pages).  The rule for ties and the
// output order are fixed by this library's contract (header mx4sp.h).
//
// Scores are compared as order-preserving uint32 keys (-0 folded to +0).  Rows
// of more than kCand scores go through a candidate filter first:
// topk_threshold_kernel -- one 512-thread CTA per such row: an evenly spaced
//   sample of 2048 keys of the row and, as threshold, the sample key at a rank
//   a few binomial standard deviations past the k-th (radix select).
// topk_filter_kernel -- persistent CTAs over 16384-score segments of those
//   rows: the segment's keys >= threshold are compacted in index order (warp
//   scans, block scan over warps) and appended to the row's candidate list in
//   the workspace at an offset taken with one atomic per segment, which records
//   (offset, count).
// topk_kernel -- one 512-thread CTA per decode token:
//   1. Candidates in shared memory, in index order.  Rows of up to kCand scores
//      take every score.  Longer rows gather the filter's segments in index
//      order when their total is in [k, kCand]; otherwise (unlucky sample,
//      massive ties, k > kCand) the CTA runs its own threshold / candidate
//      passes over the row and, if the candidates still do not fit, the exact
//      global path below.
//   2. Exact k-th key.  A radix select over the candidate keys (held in
//      registers, 11 bits per pass below the bits all keys share) gives the
//      k-th largest key K* and `want` = how many keys equal to K* are taken.
//   3. Ordered output.  Each warp owns a contiguous run of candidates; warp
//      ballots select every key > K* and the `want` lowest-index keys == K*.
// Global path: a radix select, 8 bits per pass, over the row in global memory,
// then an ordered compaction over the row.
#include "common.cuh"

namespace mx4 {

constexpr int kTopkThreads = 512;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kCand = 8192;
constexpr int kSample = 2048;
constexpr int kUnroll = 4;                            // row loads in flight per lane (fallback)
constexpr int kSeg = 16384;                           // scores per filter segment
constexpr int kSegIters = kSeg / (kTopkWarps * 128);  // 16-byte loads per lane per segment
constexpr int kMaxSeg = kTopkThreads;                 // segments per row (rows up to 8 M)
constexpr int kRadixBits = 11;
constexpr int kBins = 1 << kRadixBits;
constexpr int kCandPer = kCand / kTopkThreads;        // candidate keys per thread
constexpr int kSamplePer = kSample / kTopkThreads;    // sample keys per thread
static_assert(kTopkWarps <= 32 && kTopkThreads >= 256, "one scan warp; 256 radix bins");
static_assert(kSeg == kSegIters * kTopkWarps * 128, "segment = warps x iterations x 128");
static_assert(kBins == 4 * kTopkThreads, "4 radix bins per thread");
static_assert(kCand == kCandPer * kTopkThreads && kSample == kSamplePer * kTopkThreads, "");

// Shared state of the radix select.
struct RadixSmem {
  uint32_t hist[kBins];
  int tmp[32];
  uint32_t red_and[kTopkWarps], red_or[kTopkWarps], wsum[kTopkWarps];
  uint32_t bc_digit, bc_want, bc_count, bc_key;
};

struct TopkSmem : RadixSmem {
  uint32_t ckey[kCand];
  uint32_t cidx[kCand];
  int warp_base[kTopkWarps];
  int wgt[kTopkWarps], weq[kTopkWarps];
  int seg_off[kMaxSeg + 1];
  int seg_base[kMaxSeg];
};

struct FilterSmem {
  int tmp[32];
  int warp_base[kTopkWarps];
  int chunk_pref[kTopkThreads];
  long long rown[kTopkThreads];  // row lengths when every row has its own thread
  uint32_t rthr[kTopkThreads];   // and their thresholds
  int base;
};

// Workspace of the filter, per decode token t: the candidate count, the
// threshold, (offset, count) of each segment, and up to kCand (key, index)
// candidates.
struct TopkWs {
  int* count;     // [T]
  uint32_t* thr;  // [T]
  int2* seg;      // [T][nseg]
  uint32_t* key;  // [T][kCand]
  int32_t* idx;   // [T][kCand]
  int nseg;
};

__host__ __device__ inline int64_t align16(int64_t x) { return (x + 15) / 16 * 16; }

// Rows that take the filter (the same test in all kernels).
__device__ __forceinline__ bool use_filter(int64_t n, int64_t ld, int k) {
  return n > kCand && n <= ld && k < n && k <= kCand;
}
// Threshold rank in the sample: m = k * 2048 / n sample keys are expected at or
// above the k-th largest score; taking rank m + 4 sqrt(m) + 8 leaves fewer than k
// candidates only with a probability below ~1e-5 (binomial tail), and such a row
// falls back to the exact paths.
__device__ __forceinline__ int sample_rank(int64_t n, int k) {
  const double m = (double)k * kSample / (double)n;
  return min(kSample - 1, (int)(m + 4.0 * sqrt(m)) + 8);
}
__device__ __forceinline__ int64_t row_len(const int32_t* seq_lens, int64_t t, int Q) {
  return (int64_t)seq_lens[t / Q] - Q + (t % Q) + 1;
}

__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f + 0.0f);  // -0 + 0 = +0
  return u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
}

__device__ __forceinline__ void red_add_shared(uint32_t* p, uint32_t v) {
  asm volatile("red.shared.add.u32 [%0], %1;\n" ::"r"(smem_addr(p)), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Exclusive scan of one int per thread over the whole block; also returns the
// block total.  `s_tmp` holds 32 ints.
__device__ __forceinline__ int block_exclusive_scan(int x, int* s_tmp, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  int inc = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) s_tmp[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nwarps ? s_tmp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, w, o);
      if (lane >= o) w += y;
    }
    s_tmp[lane] = w;
  }
  __syncthreads();
  total = s_tmp[nwarps - 1];
  const int res = inc - x + (warp > 0 ? s_tmp[warp - 1] : 0);
  __syncthreads();
  return res;
}

// Radix select over keys held in registers: thread tid holds kv[u] for
// u < nv (any distribution of the C keys over the threads).  *kth = the
// rank-th largest key (1 <= rank <= C), *want = how many of the keys equal to
// it are needed to make up `rank` (the rest are strictly larger).  The leading
// bits common to all keys (block AND / OR) are skipped; the rest are resolved
// kRadixBits per pass from the top, and a pass whose chosen bin holds a single
// key ends the search.  Each pass: non-returning shared adds into the
// histogram, then a two-level search (warp sums, then one warp's scan).
template <int N>
__device__ void radix_select_reg(const uint32_t (&kv)[N], int nv, uint32_t rank, uint32_t* kth,
                                 uint32_t* want, RadixSmem& s) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
#pragma unroll
  for (int u = 0; u < 4; ++u) s.hist[4 * tid + u] = 0u;
  uint32_t a = 0xFFFFFFFFu, o = 0u;
#pragma unroll
  for (int u = 0; u < N; ++u)
    if (u < nv) {
      a &= kv[u];
      o |= kv[u];
    }
  a = __reduce_and_sync(0xFFFFFFFFu, a);
  o = __reduce_or_sync(0xFFFFFFFFu, o);
  if (lane == 0) {
    s.red_and[warp] = a;
    s.red_or[warp] = o;
  }
  __syncthreads();
  a = 0xFFFFFFFFu;
  o = 0u;
#pragma unroll
  for (int w = 0; w < kTopkWarps; ++w) {
    a &= s.red_and[w];
    o |= s.red_or[w];
  }
  const uint32_t diff = a ^ o;
  uint32_t w = rank, prefix = a, mask = 0xFFFFFFFFu;
  int top = -1;  // all keys equal: the answer is that key
  if (diff != 0u) {
    top = 31 - __clz(diff);  // highest bit on which the keys differ
    mask = top == 31 ? 0u : ~((2u << top) - 1u);
    prefix = a & mask;
  }
  while (top >= 0) {
    const int bits = min(kRadixBits, top + 1);
    const int shift = top + 1 - bits;
    const uint32_t nbm = (1u << bits) - 1u;
#pragma unroll
    for (int u = 0; u < N; ++u)
      if (u < nv && (kv[u] & mask) == prefix) red_add_shared(&s.hist[(kv[u] >> shift) & nbm], 1u);
    __syncthreads();
    // descending digits: thread tid owns nbm - 4 tid .. nbm - 4 tid - 3 (and clears them)
    uint32_t c[4], local = 0u;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int d = (int)nbm - (4 * tid + u);
      c[u] = 0u;
      if (d >= 0) {
        c[u] = s.hist[d];
        s.hist[d] = 0u;
      }
      local += c[u];
    }
    const uint32_t wtot = __reduce_add_sync(0xFFFFFFFFu, local);
    if (lane == 0) s.wsum[warp] = wtot;
    __syncthreads();
    uint32_t before = 0u;
    for (int v = 0; v < warp; ++v) before += s.wsum[v];
    if (before < w && w <= before + wtot) {  // this warp holds the rank-w bin
      uint32_t inc = local;
#pragma unroll
      for (int of = 1; of < 32; of <<= 1) {
        const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, inc, of);
        if (lane >= of) inc += y;
      }
      uint32_t run = before + inc - local;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t ge = run + c[u];
        if (c[u] > 0u && run < w && w <= ge) {
          s.bc_digit = nbm - (uint32_t)(4 * tid + u);
          s.bc_want = w - run;
          s.bc_count = c[u];
        }
        run = ge;
      }
    }
    __syncthreads();
    prefix |= s.bc_digit << shift;
    mask |= nbm << shift;
    w = s.bc_want;
    top = shift - 1;
    if (s.bc_count == 1u && top >= 0) {  // the one key with this prefix is the answer
#pragma unroll
      for (int u = 0; u < N; ++u)
        if (u < nv && (kv[u] & mask) == prefix) s.bc_key = kv[u];
      __syncthreads();
      prefix = s.bc_key;
      break;
    }
  }
  *kth = prefix;
  *want = w;
  __syncthreads();
}

// Keys of the (up to) 4 scores at i .. i+3 of the row (i a multiple of 4), in
// k[0..m); scores at or beyond n are not loaded.
template <bool VEC>
__device__ __forceinline__ int load4_keys(const float* row, int64_t i, int64_t n,
                                          uint32_t (&k)[4]) {
  if (VEC && i + 3 < n) {
    const float4 v = *reinterpret_cast<const float4*>(row + i);
    k[0] = order_key(v.x);
    k[1] = order_key(v.y);
    k[2] = order_key(v.z);
    k[3] = order_key(v.w);
    return 4;
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) k[e] = (i + e < n) ? order_key(row[i + e]) : 0u;
  const int64_t m = n - i;
  return m <= 0 ? 0 : (int)min(m, (int64_t)4);
}

// Keys of the 4 (VEC) or 1 elements at i .. of the row, in k[0..m); elements at
// or beyond n are not loaded.  Returns m.  (Static indexing only, so the keys
// stay in registers.)
template <bool VEC>
__device__ __forceinline__ int load_keys(const float* row, int64_t i, int64_t n, uint32_t (&k)[4]) {
  if (VEC && i + 3 < n) {
    const float4 v = *reinterpret_cast<const float4*>(row + i);
    k[0] = order_key(v.x);
    k[1] = order_key(v.y);
    k[2] = order_key(v.z);
    k[3] = order_key(v.w);
    return 4;
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) k[e] = (e < (VEC ? 4 : 1) && i + e < n) ? order_key(row[i + e]) : 0u;
  const int64_t m = n - i;
  return m <= 0 ? 0 : (int)min(m, (int64_t)(VEC ? 4 : 1));
}

// The evenly spaced sample of the row: thread tid holds sample tid + u*512.
__device__ __forceinline__ void load_sample(const float* row, int64_t n,
                                            uint32_t (&smp)[kSamplePer]) {
#pragma unroll
  for (int u = 0; u < kSamplePer; ++u)
    smp[u] = order_key(row[(int64_t)(threadIdx.x + u * kTopkThreads) * n / kSample]);
}

// ============================================================ filter kernels

__global__ void __launch_bounds__(kTopkThreads)
topk_threshold_kernel(const float* __restrict__ scores, int64_t ld,
                      const int32_t* __restrict__ seq_lens, int Q, int k, TopkWs ws) {
  __shared__ RadixSmem s;
  pdl_launch_dependents();
  const int64_t t = blockIdx.x;
  const int64_t n = row_len(seq_lens, t, Q);
  if (!use_filter(n, ld, k)) return;
  pdl_wait();
  uint32_t smp[kSamplePer];
  load_sample(scores + t * ld, n, smp);
  uint32_t thr, unused;
  radix_select_reg<kSamplePer>(smp, kSamplePer, (uint32_t)sample_rank(n, k) + 1, &thr, &unused, s);
  if (threadIdx.x == 0) {
    ws.thr[t] = thr;
    ws.count[t] = 0;
  }
}

// Filter segments of token t's row (0 when the row does not take the filter).
__device__ __forceinline__ int row_segments(const int32_t* seq_lens, int64_t t, int Q, int64_t ld,
                                            int k) {
  const int64_t n = row_len(seq_lens, t, Q);
  return use_filter(n, ld, k) ? (int)((n + kSeg - 1) / kSeg) : 0;
}

// Persistent CTAs over the filter items (the segments of the rows that take the
// filter, in row order); each CTA maps an item number to (row, segment) through
// a block-wide prefix over per-thread chunks of rows.
template <bool VEC>
__global__ void __launch_bounds__(kTopkThreads, 2)
topk_filter_kernel(const float* __restrict__ scores, int64_t ld,
                   const int32_t* __restrict__ seq_lens, int64_t T, int Q, int k, TopkWs ws) {
  __shared__ FilterSmem s;
  pdl_launch_dependents();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // With at most one row per thread, every row's length (and below, threshold) is
  // kept in shared memory, so an item is mapped to (row, segment) without loads.
  const bool small = T <= kTopkThreads;
  const int64_t per = (T + kTopkThreads - 1) / kTopkThreads;
  const int64_t r0 = min(T, (int64_t)tid * per), r1 = min(T, r0 + per);
  int cnt = 0;
  if (small) {
    const int64_t n = tid < T ? row_len(seq_lens, tid, Q) : 0;
    cnt = (tid < T && use_filter(n, ld, k)) ? (int)((n + kSeg - 1) / kSeg) : 0;
    s.rown[tid] = n;
  } else {
    for (int64_t t = r0; t < r1; ++t) cnt += row_segments(seq_lens, t, Q, ld, k);
  }
  int items;
  s.chunk_pref[tid] = block_exclusive_scan(cnt, s.tmp, items);
  pdl_wait();  // scores, thresholds and counts are touched from here on
  if (small && cnt > 0) s.rthr[tid] = ws.thr[tid];
  __syncthreads();

  for (int item = blockIdx.x; item < items; item += gridDim.x) {
    int lo = 0, hi = kTopkThreads - 1;  // last chunk whose prefix is <= item
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s.chunk_pref[mid] <= item) lo = mid; else hi = mid - 1;
    }
    int64_t t = (int64_t)lo * per;
    int sg = item - s.chunk_pref[lo];
    int64_t n;
    uint32_t thr;
    if (small) {
      n = s.rown[lo];
      thr = s.rthr[lo];
    } else {
      for (;;) {
        const int ns = row_segments(seq_lens, t, Q, ld, k);
        if (sg < ns) break;
        sg -= ns;
        ++t;
      }
      n = row_len(seq_lens, t, Q);
      thr = ws.thr[t];
    }
    const int64_t s0 = (int64_t)sg * kSeg, s1 = min(n, s0 + kSeg);
    const float* row = scores + t * ld;

    // the segment's keys, all loads in flight
    uint32_t key[kSegIters][4];
    int m[kSegIters];
    const int64_t w0 = s0 + (int64_t)warp * (kSegIters * 128) + 4 * lane;
#pragma unroll
    for (int j = 0; j < kSegIters; ++j) m[j] = load4_keys<VEC>(row, w0 + 128 * j, s1, key[j]);

    // index-ordered compaction of the keys >= thr
    int pos[kSegIters];
    int wtot = 0;
#pragma unroll
    for (int j = 0; j < kSegIters; ++j) {
      int c = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) c += (e < m[j] && key[j][e] >= thr) ? 1 : 0;
      int inc = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
        if (lane >= o) inc += y;
      }
      pos[j] = wtot + inc - c;
      wtot += __shfl_sync(0xFFFFFFFFu, inc, 31);
    }
    if (lane == 0) s.warp_base[warp] = wtot;
    __syncthreads();
    if (warp == 0) {
      const int v = lane < kTopkWarps ? s.warp_base[lane] : 0;
      int inc = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
        if (lane >= o) inc += y;
      }
      if (lane < kTopkWarps) s.warp_base[lane] = inc - v;
      if (lane == 31) {
        const int base = inc > 0 ? atomicAdd(&ws.count[t], inc) : 0;
        s.base = base;
        ws.seg[t * ws.nseg + sg] = make_int2(base, inc);
      }
    }
    __syncthreads();
    const int base = s.base + s.warp_base[warp];
    uint32_t* ck = ws.key + t * kCand;
    int32_t* ci = ws.idx + t * kCand;
#pragma unroll
    for (int j = 0; j < kSegIters; ++j) {
      int p = base + pos[j];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (e < m[j] && key[j][e] >= thr) {
          if (p < kCand) {
            ck[p] = key[j][e];
            ci[p] = (int32_t)(w0 + 128 * j + e);
          }
          ++p;
        }
    }
    __syncthreads();
  }
}

// ============================================================ per-row select

// Candidate pass over the row: keys >= thr, in index order.  Returns the total
// count; writes (key, index) pairs only while they fit in kCand.
template <bool VEC>
__device__ int collect_candidates(const float* row, int64_t n, uint32_t thr, TopkSmem& s) {
  constexpr int E = VEC ? 4 : 1;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t per_it = 32 * E;
  const int64_t chunk = ((n + kTopkWarps - 1) / kTopkWarps + per_it - 1) / per_it * per_it;
  const int64_t c0 = min(n, (int64_t)warp * chunk), c1 = min(n, c0 + chunk);
  // counting pass (kUnroll loads in flight per lane)
  int cnt = 0;
  for (int64_t b = c0; b < c1; b += per_it * kUnroll) {
    uint32_t k[kUnroll][4];
    int m[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      m[u] = load_keys<VEC>(row, b + per_it * u + (int64_t)lane * E, c1, k[u]);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
#pragma unroll
      for (int e = 0; e < 4; ++e) cnt += (e < m[u] && k[u][e] >= thr) ? 1 : 0;
  }
  cnt = __reduce_add_sync(0xFFFFFFFFu, cnt);
  if (lane == 0) s.warp_base[warp] = cnt;
  __syncthreads();
  if (warp == 0) {
    const int v = lane < kTopkWarps ? s.warp_base[lane] : 0;
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
      if (lane >= o) inc += y;
    }
    if (lane < kTopkWarps) s.warp_base[lane] = inc - v;
    if (lane == 31) s.tmp[0] = inc;
  }
  __syncthreads();
  const int total = s.tmp[0];
  if (total <= kCand) {
    int pos = s.warp_base[warp];
    for (int64_t b = c0; b < c1; b += per_it * kUnroll) {
      uint32_t k[kUnroll][4];
      int m[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
        m[u] = load_keys<VEC>(row, b + per_it * u + (int64_t)lane * E, c1, k[u]);
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t i0 = b + per_it * u + (int64_t)lane * E;
        int mine = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) mine += (e < m[u] && k[u][e] >= thr) ? 1 : 0;
        int inc = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
          if (lane >= o) inc += y;
        }
        int w = pos + inc - mine;
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (e < m[u] && k[u][e] >= thr) {
            s.ckey[w] = k[u][e];
            s.cidx[w] = (uint32_t)(i0 + e);
            ++w;
          }
        pos += __shfl_sync(0xFFFFFFFFu, inc, 31);
      }
    }
  }
  __syncthreads();
  return total;
}

// Exact selection over the row in global memory (rows whose candidates do not
// fit in shared memory): radix select of the k-th key, then ordered compaction.
__device__ void topk_global_path(const float* row, int64_t n, int k, int32_t* o, TopkSmem& s) {
  const int tid = threadIdx.x;
  uint32_t prefix = 0, mask = 0, want = (uint32_t)k;
  for (int shift = 24; shift >= 0; shift -= 8) {
    if (tid < 256) s.hist[tid] = 0;
    __syncthreads();
    for (int64_t i = tid; i < n; i += kTopkThreads) {
      const uint32_t key = order_key(row[i]);
      if ((key & mask) == prefix) atomicAdd(&s.hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    const int d = 255 - tid;
    const int c = (tid < 256) ? (int)s.hist[d] : 0;
    int total;
    const int before = block_exclusive_scan(c, s.tmp, total);
    if (tid < 256) {
      const uint32_t gt = (uint32_t)before, ge = gt + (uint32_t)c;
      if (gt < want && want <= ge) {
        s.bc_digit = (uint32_t)d;
        s.bc_want = want - gt;
      }
    }
    __syncthreads();
    prefix |= s.bc_digit << shift;
    mask |= 255u << shift;
    want = s.bc_want;
    __syncthreads();
  }
  const uint32_t kth = prefix;
  const int64_t seg = (n + kTopkThreads - 1) / kTopkThreads;
  const int64_t lo = tid * seg, hi = min(n, lo + seg);
  int gt = 0, eq = 0;
  for (int64_t i = lo; i < hi; ++i) {
    const uint32_t key = order_key(row[i]);
    gt += key > kth;
    eq += key == kth;
  }
  int total;
  const int eq_before = block_exclusive_scan(eq, s.tmp, total);
  const int take_eq = max(0, min(eq, (int)want - eq_before));
  int off = block_exclusive_scan(gt + take_eq, s.tmp, total);
  int taken = 0;
  for (int64_t i = lo; i < hi; ++i) {
    const uint32_t key = order_key(row[i]);
    if (key > kth || (key == kth && taken < take_eq)) {
      taken += key == kth;
      o[off++] = (int32_t)i;
    }
  }
}

template <bool VEC>
__global__ void __launch_bounds__(kTopkThreads)
topk_kernel(const float* __restrict__ scores, int64_t ld, const int32_t* __restrict__ seq_lens,
            int Q, int k, int32_t* __restrict__ out, TopkWs ws, uint32_t* status) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  TopkSmem& s = *reinterpret_cast<TopkSmem*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_launch_dependents();
  const int64_t t = blockIdx.x;
  const int64_t n = row_len(seq_lens, t, Q);
  int32_t* o = out + t * (int64_t)k;
  pdl_wait();  // scores and the filter's workspace are touched from here on

  if (n < 1 || n > ld) {
    for (int i = tid; i < k; i += kTopkThreads) o[i] = -1;
    if (tid == 0) flag(status, MX4_STATUS_BAD_LEN);
    return;
  }
  if (n <= k) {
    for (int i = tid; i < k; i += kTopkThreads) o[i] = (i < n) ? i : -1;
    return;
  }
  const float* row = scores + t * ld;

  // ---- 1. candidates in shared memory, in index order
  int C = -1;
  if (n <= kCand) {
    // every score (16-byte loads, all in flight)
    constexpr int kV = kCand / (4 * kTopkThreads);
    uint32_t kk[kV][4];
    int mm[kV];
#pragma unroll
    for (int u = 0; u < kV; ++u) mm[u] = load4_keys<VEC>(row, 4 * (tid + u * kTopkThreads), n, kk[u]);
#pragma unroll
    for (int u = 0; u < kV; ++u)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (e < mm[u]) {
          const int i = 4 * (tid + u * kTopkThreads) + e;
          s.ckey[i] = kk[u][e];
          s.cidx[i] = (uint32_t)i;
        }
    C = (int)n;
    __syncthreads();
  } else if (use_filter(n, ld, k) && ws.count != nullptr) {
    // the filter's segments, in index order: sources, then all loads, then stores
    const int nseg = (int)((n + kSeg - 1) / kSeg);
    const int total = ws.count[t];
    int c = 0;
    if (tid < nseg) {
      const int2 sgm = ws.seg[t * ws.nseg + tid];
      s.seg_base[tid] = sgm.x;
      c = sgm.y;
    }
    int sum;
    const int off = block_exclusive_scan(c, s.tmp, sum);
    if (total >= k && total <= kCand && nseg <= kMaxSeg) {
      if (tid < nseg) s.seg_off[tid] = off;
      __syncthreads();
      const uint32_t* ck = ws.key + t * kCand;
      const int32_t* ci = ws.idx + t * kCand;
      int src[kCandPer];
#pragma unroll
      for (int u = 0; u < kCandPer; ++u) {
        const int i = tid + u * kTopkThreads;
        src[u] = -1;
        if (i < total) {
          int lo = 0, hi = nseg - 1;  // last segment with seg_off <= i
          while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s.seg_off[mid] <= i) lo = mid; else hi = mid - 1;
          }
          src[u] = s.seg_base[lo] + (i - s.seg_off[lo]);
        }
      }
      uint32_t kv[kCandPer];
      int32_t iv[kCandPer];
#pragma unroll
      for (int u = 0; u < kCandPer; ++u)
        if (src[u] >= 0) {
          kv[u] = ck[src[u]];
          iv[u] = ci[src[u]];
        }
#pragma unroll
      for (int u = 0; u < kCandPer; ++u)
        if (src[u] >= 0) {
          s.ckey[tid + u * kTopkThreads] = kv[u];
          s.cidx[tid + u * kTopkThreads] = (uint32_t)iv[u];
        }
      C = total;
      __syncthreads();
    }
  }
  if (C < 0) {
    // own threshold and candidate passes over the row
    uint32_t thr = 0u;
    int r = -1;
    uint32_t smp[kSamplePer];
    if (n > kCand) {
      load_sample(row, n, smp);
      r = sample_rank(n, k);
      uint32_t unused;
      radix_select_reg<kSamplePer>(smp, kSamplePer, (uint32_t)r + 1, &thr, &unused, s);
    }
    for (;;) {
      C = collect_candidates<VEC>(row, n, thr, s);
      if (C >= k && C <= kCand) break;
      if (C > kCand || r < 0 || r >= kSample - 1) {
        topk_global_path(row, n, k, o, s);
        return;
      }
      r = min(kSample - 1, 2 * r + 64);  // too few candidates: lower the threshold
      if (r >= kSample - 1) {
        thr = 0u;
      } else {
        uint32_t unused;
        radix_select_reg<kSamplePer>(smp, kSamplePer, (uint32_t)r + 1, &thr, &unused, s);
      }
    }
  }

  // ---- 2. exact k-th key among the candidates
  uint32_t kth, want_u;
  {
    uint32_t kv[kCandPer];
    const int nv = C > tid ? (C - tid + kTopkThreads - 1) / kTopkThreads : 0;
#pragma unroll
    for (int u = 0; u < kCandPer; ++u) kv[u] = u < nv ? s.ckey[tid + u * kTopkThreads] : 0u;
    radix_select_reg<kCandPer>(kv, nv, (uint32_t)k, &kth, &want_u, s);
  }
  const int want = (int)want_u;  // keys equal to K* that are taken (lowest indices)

  // ---- 3. ordered output: warp w owns candidates [w cw, (w+1) cw)
  const int cw = (C + kTopkWarps * 32 - 1) / (kTopkWarps * 32) * 32;
  const int i0 = min(C, warp * cw), i1 = min(C, i0 + cw);
  int ngt = 0, neq = 0;
  for (int b = i0; b < i1; b += 32) {
    const int i = b + lane;
    const uint32_t key = i < i1 ? s.ckey[i] : 0u;
    ngt += __popc(__ballot_sync(0xFFFFFFFFu, i < i1 && key > kth));
    neq += __popc(__ballot_sync(0xFFFFFFFFu, i < i1 && key == kth));
  }
  if (lane == 0) {
    s.wgt[warp] = ngt;
    s.weq[warp] = neq;
  }
  __syncthreads();
  int eq_before = 0, out_base = 0, take = 0;
  for (int v = 0; v < kTopkWarps; ++v) {
    const int tv = max(0, min(s.weq[v], want - eq_before));
    if (v == warp) {
      take = tv;
      break;
    }
    out_base += s.wgt[v] + tv;
    eq_before += s.weq[v];
  }
  const uint32_t lt = lanemask_lt();
  int eq_run = 0, out_run = 0;
  for (int b = i0; b < i1; b += 32) {
    const int i = b + lane;
    const bool valid = i < i1;
    const uint32_t key = valid ? s.ckey[i] : 0u;
    const bool e = valid && key == kth;
    const uint32_t eb = __ballot_sync(0xFFFFFFFFu, e);
    const bool sel = (valid && key > kth) || (e && eq_run + __popc(eb & lt) < take);
    const uint32_t sb = __ballot_sync(0xFFFFFFFFu, sel);
    if (sel) o[out_base + out_run + __popc(sb & lt)] = (int32_t)s.cidx[i];
    out_run += __popc(sb);
    eq_run += __popc(eb);
  }
}

// Workspace: count [T] | thr [T] | seg [T][nseg] | key [T][kCand] | idx [T][kCand],
// each section 16-byte aligned; none when no row can take the filter.
size_t topk_workspace_bytes(int64_t T, int k, int64_t ld) {
  if (ld <= kCand || k > kCand || T <= 0) return 0;
  const int64_t nseg = (ld + kSeg - 1) / kSeg;
  return (size_t)(2 * align16(T * 4) + align16(T * nseg * 8) + 2 * align16(T * kCand * 4));
}

template <bool VEC>
static cudaError_t launch_topk_v(const float* scores, int64_t ld, const int32_t* seq_lens,
                                 int64_t T, int Q, int k, int32_t* out, const TopkWs& ws,
                                 uint32_t* status, int num_sms, cudaStream_t stream) {
  const int smem = (int)sizeof(TopkSmem);
  cudaError_t err =
      cudaFuncSetAttribute(topk_kernel<VEC>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  if (ws.count != nullptr) {
    err = launch_pdl(topk_threshold_kernel, dim3((unsigned)T), dim3(kTopkThreads), 0, stream,
                     scores, ld, seq_lens, Q, k, ws);
    if (err != cudaSuccess) return err;
    const int64_t grid = min(T * (int64_t)ws.nseg, (int64_t)num_sms * 2);
    err = launch_pdl(topk_filter_kernel<VEC>, dim3((unsigned)grid), dim3(kTopkThreads), 0, stream,
                     scores, ld, seq_lens, T, Q, k, ws);
    if (err != cudaSuccess) return err;
  }
  return launch_pdl(topk_kernel<VEC>, dim3((unsigned)T), dim3(kTopkThreads), (size_t)smem, stream,
                    scores, ld, seq_lens, Q, k, out, ws, status);
}

cudaError_t launch_topk(const float* scores, int64_t ld, const int32_t* seq_lens, int64_t T, int Q,
                        int k, int32_t* out, void* wsp, uint32_t* status, int num_sms,
                        cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  TopkWs ws{nullptr, nullptr, nullptr, nullptr, nullptr, 0};
  if (topk_workspace_bytes(T, k, ld) > 0) {
    const int64_t nseg = (ld + kSeg - 1) / kSeg;
    if (T > 65535 || nseg > kMaxSeg) return cudaErrorInvalidValue;
    uint8_t* p = static_cast<uint8_t*>(wsp);
    ws.count = reinterpret_cast<int*>(p);
    p += align16(T * 4);
    ws.thr = reinterpret_cast<uint32_t*>(p);
    p += align16(T * 4);
    ws.seg = reinterpret_cast<int2*>(p);
    p += align16(T * nseg * 8);
    ws.key = reinterpret_cast<uint32_t*>(p);
    p += align16(T * kCand * 4);
    ws.idx = reinterpret_cast<int32_t*>(p);
    ws.nseg = (int)nseg;
  }
  const bool vec = (reinterpret_cast<uintptr_t>(scores) % 16 == 0) && (ld % 4 == 0);
  return vec ? launch_topk_v<true>(scores, ld, seq_lens, T, Q, k, out, ws, status, num_sms, stream)
             : launch_topk_v<false>(scores, ld, seq_lens, T, Q, k, out, ws, status, num_sms,
                                    stream);
}

}  // namespace mx4
