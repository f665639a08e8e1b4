// topk_select: per decode token, the k cached tokens with the largest index
// scores (ties to the lower token index), returned in ascending index order.
//
// The selection step sits between the index scorer and the MXFP4 pa_decode
// reader ("vllm.models.minimax_m3.amd.ops.mxfp4_pages", module description:
// the scorers and pa_decode read the same pages).  The rule for ties and the
// output order are fixed by this library's contract (header mx4sp.h).
//
// One 512-thread CTA per decode token; scores are compared as order-preserving
// uint32 keys (-0 folded to +0).
//   1. Threshold.  Rows of up to kCand scores take every score as a candidate.
//      Longer rows take an evenly spaced sample of 2048 keys and, as threshold,
//      the sample key at a rank that leaves about 1.3 k candidates plus a
//      margin (radix select in shared memory).
//   2. Candidates.  Each warp owns a contiguous chunk of the row; a counting pass
//      and a writing pass (ballot/scan compaction, coalesced reads) store the
//      keys >= threshold, with their indices, in index order in shared memory.
//      Too few candidates lowers the threshold and repeats; more than kCand
//      (only possible with massive ties) takes the exact global path below.
//   3. Exact k-th key.  A radix select over the candidate keys in shared memory
//      (8 bits per pass) gives the k-th largest key K* and `want` = how many keys
//      equal to K* are taken (the lowest indices).
//   4. Ordered output.  A block scan over the index-ordered candidates writes
//      every key > K* and the first `want` keys == K*.
// Global path (fallback for rows whose candidates do not fit): a radix select,
// 8 bits per pass, over the row in global memory, then the same ordered
// compaction over the row.
#include "common.cuh"

namespace mx4 {

constexpr int kTopkThreads = 512;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kCand = 8192;
constexpr int kSample = 2048;
constexpr int kUnroll = 4;  // row loads in flight per lane in the candidate passes
static_assert(kTopkWarps <= 32 && kTopkThreads >= 256, "one scan warp; 256 radix bins");

struct TopkSmem {
  uint32_t ckey[kCand];
  uint32_t cidx[kCand];
  uint32_t sbuf[kSample];
  int tmp[32];
  uint32_t hist[256];
  int warp_base[kTopkWarps];
  uint32_t bc_digit, bc_want;
};

__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f + 0.0f);  // -0 + 0 = +0
  return u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
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

// Radix select over keys[0..C) in shared memory, 8 bits per pass from the top:
// *kth = the rank-th largest key (rank >= 1), *want = how many of the keys equal
// to it are needed to make up `rank` (the rest are strictly larger).
__device__ void radix_select_smem(const uint32_t* keys, int C, uint32_t rank, uint32_t* kth,
                                  uint32_t* want, TopkSmem& s) {
  const int tid = threadIdx.x;
  uint32_t prefix = 0, mask = 0, w = rank;
  for (int shift = 24; shift >= 0; shift -= 8) {
    if (tid < 256) s.hist[tid] = 0;
    __syncthreads();
    for (int i = tid; i < C; i += kTopkThreads) {
      const uint32_t key = keys[i];
      if ((key & mask) == prefix) atomicAdd(&s.hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    const int d = 255 - tid;
    const int c = (tid < 256) ? (int)s.hist[d] : 0;
    int total;
    const int before = block_exclusive_scan(c, s.tmp, total);
    if (tid < 256) {
      const uint32_t gt = (uint32_t)before, ge = gt + (uint32_t)c;
      if (gt < w && w <= ge) {
        s.bc_digit = (uint32_t)d;
        s.bc_want = w - gt;
      }
    }
    __syncthreads();
    prefix |= s.bc_digit << shift;
    mask |= 255u << shift;
    w = s.bc_want;
    __syncthreads();
  }
  *kth = prefix;
  *want = w;
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
            int Q, int k, int32_t* __restrict__ out, uint32_t* status) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  TopkSmem& s = *reinterpret_cast<TopkSmem*>(smem_raw);
  const int tid = threadIdx.x;
  const int64_t t = blockIdx.x;
  const int64_t L = seq_lens[t / Q];
  const int64_t n = L - Q + (t % Q) + 1;
  int32_t* o = out + t * (int64_t)k;

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

  // ---- 1. threshold
  uint32_t thr = 0;
  int r = -1;
  if (n > kCand) {
    for (int i = tid; i < kSample; i += kTopkThreads)
      s.sbuf[i] = order_key(row[(int64_t)i * n / kSample]);
    __syncthreads();
    r = min(kSample - 1, (int)(1.3 * (double)k * kSample / (double)n) + 32);
    uint32_t unused;
    radix_select_smem(s.sbuf, kSample, (uint32_t)r + 1, &thr, &unused, s);
  }
  // ---- 2. candidates
  int C;
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
      radix_select_smem(s.sbuf, kSample, (uint32_t)r + 1, &thr, &unused, s);
    }
  }
  // ---- 3. exact k-th key among the candidates
  uint32_t kth, want_u;
  radix_select_smem(s.ckey, C, (uint32_t)k, &kth, &want_u, s);
  const int want = (int)want_u;  // keys equal to K* that are taken (lowest indices)
  // ---- 4. ordered output over the index-ordered candidates
  const int seg = (C + kTopkThreads - 1) / kTopkThreads;
  const int lo = min(C, tid * seg), hi = min(C, lo + seg);
  int gt = 0, eq = 0;
  for (int i = lo; i < hi; ++i) {
    gt += s.ckey[i] > kth;
    eq += s.ckey[i] == kth;
  }
  int total;
  const int eq_before = block_exclusive_scan(eq, s.tmp, total);
  const int take_eq = max(0, min(eq, want - eq_before));
  int off = block_exclusive_scan(gt + take_eq, s.tmp, total);
  int taken = 0;
  for (int i = lo; i < hi; ++i) {
    const uint32_t key = s.ckey[i];
    if (key > kth || (key == kth && taken < take_eq)) {
      taken += key == kth;
      o[off++] = (int32_t)s.cidx[i];
    }
  }
}

cudaError_t launch_topk(const float* scores, int64_t ld, const int32_t* seq_lens, int64_t T, int Q,
                        int k, int32_t* out, uint32_t* status, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const int smem = (int)sizeof(TopkSmem);
  const bool vec = (reinterpret_cast<uintptr_t>(scores) % 16 == 0) && (ld % 4 == 0);
  cudaError_t err;
  if (vec) {
    err = cudaFuncSetAttribute(topk_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               smem);
    if (err != cudaSuccess) return err;
    topk_kernel<true><<<(unsigned)T, kTopkThreads, smem, stream>>>(scores, ld, seq_lens, Q, k,
                                                                   out, status);
  } else {
    err = cudaFuncSetAttribute(topk_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               smem);
    if (err != cudaSuccess) return err;
    topk_kernel<false><<<(unsigned)T, kTopkThreads, smem, stream>>>(scores, ld, seq_lens, Q, k,
                                                                    out, status);
  }
  return cudaGetLastError();
}

}  // namespace mx4
