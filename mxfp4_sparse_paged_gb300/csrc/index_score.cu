// index_score: dot every cached index key of a sequence with the index-q head
// of each of its decode tokens.
//
// The index key cache is [pages, 8704] ("vllm.models.minimax_m3.amd.ops.
// mxfp4_pages", mxfp4_page_views: the [pages, 128, 64] / [pages, 128, 4] pair
// the index scorers read); pages are found through the block table shared with
// the K/V cache ("vllm.models.minimax_m3.amd.mono.dispatch", _slots_shared).
//
// Work decomposition: a work item is (sequence, chunk of kChunkPages pages).
// Persistent CTAs walk the items round-robin; the item -> sequence map is a
// block-wide prefix sum over seq_lens, recomputed by each CTA tile by tile,
// so the call needs no workspace and no host knowledge of the lengths.  All q
// decode tokens of a sequence are scored in the same pass over its pages.
//
// Inside an item a warp reads 8 token rows per step: lane l takes row l/4 and
// block b = l%4 (16 data bytes = 32 elements as one 16-B load, plus that
// block's scale byte).  The 32-element partial dot is scaled by 2^(scale-127)
// and the four blocks of a row are summed with two xor-shuffles.
#include "common.cuh"

namespace mx4 {

constexpr int kScoreThreads = 256;
constexpr int kChunkPages = 2;

template <int Q>
__device__ __forceinline__ void score_rows(const uint8_t* __restrict__ page, int row, int b,
                                           const float* __restrict__ s_iq, float (&acc)[Q]) {
  const uint4 d = *reinterpret_cast<const uint4*>(page + row * kRowDataBytes + b * 16);
  const float sc = e8m0_to_float(page[kScaleOffset + row * kRowScaleBytes + b]);
  const uint32_t w[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
  for (int qq = 0; qq < Q; ++qq) acc[qq] = 0.f;
#pragma unroll
  for (int wi = 0; wi < 4; ++wi) {
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      const int j = wi * 8 + n;  // element 32b + j of the row
      const float f = e2m1_to_float(w[wi] >> (4 * n));
#pragma unroll
      for (int qq = 0; qq < Q; ++qq) acc[qq] = fmaf(s_iq[qq * kHeadDim + j * 4 + b], f, acc[qq]);
    }
  }
#pragma unroll
  for (int qq = 0; qq < Q; ++qq) acc[qq] *= sc;
}

template <int Q>
__global__ void __launch_bounds__(kScoreThreads)
index_score_kernel(const uint16_t* __restrict__ iq, const uint8_t* __restrict__ idx_pages,
                   int64_t idx_page_stride, int64_t num_pages,
                   const int32_t* __restrict__ block_table, int B, int64_t bt_width,
                   const int32_t* __restrict__ seq_lens, float* __restrict__ scores, int64_t ld,
                   uint32_t* status) {
  __shared__ int s_pref[kScoreThreads];      // inclusive prefix of items in this tile
  __shared__ float s_iq[Q * kHeadDim];       // [q][j][b]: element 32b+j at j*4+b
  __shared__ int s_warp[kScoreThreads / 32];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t grid = gridDim.x;
  int64_t base_item = 0;

  for (int tile = 0; tile < B; tile += kScoreThreads) {
    // items of the sequences tile .. tile+255
    const int s = tile + tid;
    int n = 0;
    if (s < B) {
      const int64_t L = seq_lens[s];
      const bool ok = L >= Q && L <= bt_width * kPageTokens && L <= ld;
      if (!ok && blockIdx.x == 0) flag(status, MX4_STATUS_BAD_LEN);
      const int64_t pages = (L + kPageTokens - 1) / kPageTokens;
      n = ok ? (int)((pages + kChunkPages - 1) / kChunkPages) : 0;
    }
    // block inclusive scan of n
    int x = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int w = lane < kScoreThreads / 32 ? s_warp[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, w, o);
        if (lane >= o) w += y;
      }
      if (lane < kScoreThreads / 32) s_warp[lane] = w;
    }
    __syncthreads();
    s_pref[tid] = x + (warp > 0 ? s_warp[warp - 1] : 0);
    __syncthreads();
    const int64_t total = s_pref[kScoreThreads - 1];

    // this CTA's items in [base_item, base_item + total)
    int64_t it = base_item + (((int64_t)blockIdx.x - base_item) % grid + grid) % grid;
    for (; it < base_item + total; it += grid) {
      const int local = (int)(it - base_item);
      int lo = 0, hi = kScoreThreads - 1;  // first index with s_pref > local
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (s_pref[mid] > local) hi = mid; else lo = mid + 1;
      }
      const int seq = tile + lo;
      const int chunk = local - (lo > 0 ? s_pref[lo - 1] : 0);
      const int64_t L = seq_lens[seq];

      __syncthreads();  // previous item's readers of s_iq are done
      for (int e = tid; e < Q * kHeadDim; e += kScoreThreads) {
        const int qq = e / kHeadDim, d = e % kHeadDim;
        s_iq[qq * kHeadDim + (d % 32) * 4 + d / 32] =
            bf16_bits_to_float(iq[((int64_t)seq * Q + qq) * kHeadDim + d]);
      }
      __syncthreads();

      const int64_t npages = (L + kPageTokens - 1) / kPageTokens;
      for (int cp = 0; cp < kChunkPages; ++cp) {
        const int64_t pg = (int64_t)chunk * kChunkPages + cp;
        if (pg >= npages) break;
        const int32_t pid = block_table[(int64_t)seq * bt_width + pg];
        if (pid < 0 || pid >= num_pages) {
          if (tid == 0) flag(status, MX4_STATUS_BAD_PAGE);
          continue;
        }
        const uint8_t* page = idx_pages + (int64_t)pid * idx_page_stride;
        for (int r0 = warp * 8; r0 < kPageTokens; r0 += kScoreThreads / 4) {
          const int row = r0 + (lane >> 2), b = lane & 3;
          const int64_t i = pg * kPageTokens + row;
          float acc[Q];
          score_rows<Q>(page, row, b, s_iq, acc);
#pragma unroll
          for (int qq = 0; qq < Q; ++qq) {
            acc[qq] += __shfl_xor_sync(0xFFFFFFFFu, acc[qq], 1);
            acc[qq] += __shfl_xor_sync(0xFFFFFFFFu, acc[qq], 2);
          }
          if (b == 0 && i < L) {
#pragma unroll
            for (int qq = 0; qq < Q; ++qq) {
              const int64_t p = L - Q + qq;
              scores[((int64_t)seq * Q + qq) * ld + i] = (i <= p) ? acc[qq] : -INFINITY;
            }
          }
        }
      }
    }
    base_item += total;
    __syncthreads();
  }
}

template <int Q>
static cudaError_t launch_q(int grid, const uint16_t* iq, const uint8_t* idx_pages,
                            int64_t idx_page_stride, int64_t num_pages,
                            const int32_t* block_table, int B, int64_t bt_width,
                            const int32_t* seq_lens, float* scores, int64_t ld, uint32_t* status,
                            cudaStream_t stream) {
  index_score_kernel<Q><<<grid, kScoreThreads, 0, stream>>>(
      iq, idx_pages, idx_page_stride, num_pages, block_table, B, bt_width, seq_lens, scores, ld,
      status);
  return cudaGetLastError();
}

cudaError_t launch_index_score(const uint16_t* iq, int q, const uint8_t* idx_pages,
                               int64_t idx_page_stride, int64_t num_pages,
                               const int32_t* block_table, int B, int64_t bt_width,
                               const int32_t* seq_lens, float* scores, int64_t ld,
                               uint32_t* status, int num_sms, cudaStream_t stream) {
  const int grid = num_sms * 8;
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
