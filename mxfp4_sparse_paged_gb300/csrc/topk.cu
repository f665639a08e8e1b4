// topk_select: per decode token, the k cached tokens with the largest index
// scores (ties to the lower token index), returned in ascending index order.
//
// The selection step sits between the index scorer and the MXFP4 pa_decode
// reader ("vllm.models.minimax_m3.amd.ops.mxfp4_pages", module description:
// the scorers and pa_decode read the same pages).  The rule for ties and the
// output order are fixed by this library's contract (header mx4sp.h).
//
// Algorithm (one CTA per decode token):
//   1. Map each fp32 score to an order-preserving uint32 key (-0 folded to +0).
//   2. Radix select, 8 bits per pass from the top: a shared-memory histogram of
//      the keys that match the digits chosen so far gives the digit of the
//      k-th largest key.  After four passes the threshold key K* is exact and
//      `want` = how many keys equal to K* belong to the selection.
//   3. Ordered compaction: thread t owns a contiguous segment of the row; it
//      counts keys > K* and == K*, a block scan hands the `want` equal keys to
//      the lowest indices and gives every thread its output offset, and a
//      second pass over the segment writes the indices in order.
#include "common.cuh"

namespace mx4 {

constexpr int kTopkThreads = 1024;

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
    s_tmp[lane] = w;  // inclusive warp prefix
  }
  __syncthreads();
  total = s_tmp[nwarps - 1];
  const int res = inc - x + (warp > 0 ? s_tmp[warp - 1] : 0);
  __syncthreads();
  return res;
}

__global__ void __launch_bounds__(kTopkThreads)
topk_kernel(const float* __restrict__ scores, int64_t ld, const int32_t* __restrict__ seq_lens,
            int Q, int k, int32_t* __restrict__ out, uint32_t* status) {
  __shared__ uint32_t hist[256];
  __shared__ int s_tmp[32];
  __shared__ uint32_t s_digit, s_want;

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

  // ---- radix select of the k-th largest key
  uint32_t prefix = 0, mask = 0, want = (uint32_t)k;
  for (int shift = 24; shift >= 0; shift -= 8) {
    if (tid < 256) hist[tid] = 0;
    __syncthreads();
    for (int64_t i = tid; i < n; i += kTopkThreads) {
      const uint32_t key = order_key(row[i]);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    // cum_ge(d) = #keys with digit >= d; scan the bins from the top digit down
    const int d = 255 - tid;
    const int c = (tid < 256) ? (int)hist[d] : 0;
    int total;
    const int before = block_exclusive_scan(c, s_tmp, total);  // = cum_gt(d) for tid < 256
    if (tid < 256) {
      const uint32_t gt = (uint32_t)before, ge = gt + (uint32_t)c;
      if (gt < want && want <= ge) {
        s_digit = (uint32_t)d;
        s_want = want - gt;
      }
    }
    __syncthreads();
    prefix |= s_digit << shift;
    mask |= 255u << shift;
    want = s_want;
    __syncthreads();
  }
  const uint32_t kth = prefix;

  // ---- ordered compaction
  const int64_t seg = (n + kTopkThreads - 1) / kTopkThreads;
  const int64_t lo = tid * seg, hi = min(n, lo + seg);
  int gt = 0, eq = 0;
  for (int64_t i = lo; i < hi; ++i) {
    const uint32_t key = order_key(row[i]);
    gt += key > kth;
    eq += key == kth;
  }
  int total;
  const int eq_before = block_exclusive_scan(eq, s_tmp, total);
  const int take_eq = max(0, min(eq, (int)want - eq_before));
  int off = block_exclusive_scan(gt + take_eq, s_tmp, total);
  int taken = 0;
  for (int64_t i = lo; i < hi; ++i) {
    const uint32_t key = order_key(row[i]);
    if (key > kth || (key == kth && taken < take_eq)) {
      taken += key == kth;
      o[off++] = (int32_t)i;
    }
  }
  // total == k here; nothing to pad
}

cudaError_t launch_topk(const float* scores, int64_t ld, const int32_t* seq_lens, int64_t T, int Q,
                        int k, int32_t* out, uint32_t* status, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  topk_kernel<<<(unsigned)T, kTopkThreads, 0, stream>>>(scores, ld, seq_lens, Q, k, out, status);
  return cudaGetLastError();
}

}  // namespace mx4
