// sparse_paged_decode: GQA decode attention (16 query heads sharing one KV head,
// head_dim 128) over the selected tokens' MXFP4 K/V rows, split over the
// selected list with an online softmax per split and a merge kernel.
//
// K/V pages are [pages, heads, 8704] ("vllm.models.minimax_m3.amd.ops.
// mxfp4_pages", mxfp4_page_views: the [pages, heads, 128, 64] /
// [pages, heads, 128, 4] pair pa_decode takes).  Head geometry: one rank's
// q(2048) | k(128) | v(128) rows ("vllm.models.minimax_m3.amd.mono.weights",
// _build_cp_qkv), i.e. 16 query heads over one KV head.
//
// split kernel: one CTA per (decode token, split of kSplitTokens selected
//   entries).  Phase 1 resolves the split's indices to page rows; phase 2
//   gathers those K and V rows (data + scales) into shared memory with
//   independent 16-byte loads; phase 3 runs the online softmax.  Thread
//   (h, part) owns query head h = tid/8 and dims 16*part .. 16*part+15: it
//   dots its 16 dims, the 8 threads of a head combine with xor-shuffles, and
//   it accumulates its 16 output dims.  The split writes its unnormalised
//   output, running max (log2 units) and running sum to the workspace.
// merge kernel: one CTA per decode token combines the splits of each head.
#include "common.cuh"

namespace mx4 {

constexpr int kSplitTokens = 256;
constexpr int kDecThreads = 128;  // 16 heads x 8 parts
constexpr int kHeads = 16;
constexpr float kLog2e = 1.4426950408889634f;

__global__ void __launch_bounds__(kDecThreads)
decode_split_kernel(const uint16_t* __restrict__ q, int Q, const uint8_t* __restrict__ k_pages,
                    const uint8_t* __restrict__ v_pages, int64_t kv_page_stride,
                    int64_t num_pages, const int32_t* __restrict__ block_table, int64_t bt_width,
                    const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ topk,
                    int kw, float scale_log2, int S, float* __restrict__ ws_o,
                    float* __restrict__ ws_ml, uint32_t* status) {
  __shared__ __align__(16) uint8_t sK[kSplitTokens][kRowDataBytes];
  __shared__ __align__(16) uint8_t sV[kSplitTokens][kRowDataBytes];
  __shared__ uint32_t sKs[kSplitTokens], sVs[kSplitTokens];
  __shared__ int64_t s_off[kSplitTokens];  // page byte offset, or -1 to skip
  __shared__ int s_row[kSplitTokens];

  const int tid = threadIdx.x;
  const int64_t t = blockIdx.x / S;
  const int sp = blockIdx.x % S;
  const int64_t seq = t / Q;
  const int64_t p = (int64_t)seq_lens[seq] - Q + (t % Q);
  const int begin = sp * kSplitTokens;
  const int cnt = max(0, min(kSplitTokens, kw - begin));

  // phase 1: indices -> page rows
  for (int r = tid; r < cnt; r += kDecThreads) {
    const int32_t i = topk[t * kw + begin + r];
    int64_t off = -1;
    if (i >= 0) {
      if (i > p || (int64_t)i / kPageTokens >= bt_width) {
        flag(status, MX4_STATUS_BAD_INDEX);
      } else {
        const int32_t pid = block_table[seq * bt_width + i / kPageTokens];
        if (pid < 0 || pid >= num_pages) flag(status, MX4_STATUS_BAD_PAGE);
        else off = (int64_t)pid * kv_page_stride;
      }
    }
    s_off[r] = off;
    s_row[r] = (i >= 0) ? (i % kPageTokens) : 0;
  }
  __syncthreads();

  // phase 2: gather the rows (4 x 16 B of data per row and tensor, 4 B of scales)
  for (int e = tid; e < cnt * 4; e += kDecThreads) {
    const int r = e >> 2, part = e & 3;
    const int64_t off = s_off[r];
    if (off < 0) continue;
    const int64_t base = off + s_row[r] * kRowDataBytes + part * 16;
    *reinterpret_cast<uint4*>(&sK[r][part * 16]) = *reinterpret_cast<const uint4*>(k_pages + base);
    *reinterpret_cast<uint4*>(&sV[r][part * 16]) = *reinterpret_cast<const uint4*>(v_pages + base);
  }
  for (int r = tid; r < cnt; r += kDecThreads) {
    const int64_t off = s_off[r];
    if (off < 0) continue;
    const int64_t so = off + kScaleOffset + s_row[r] * kRowScaleBytes;
    sKs[r] = *reinterpret_cast<const uint32_t*>(k_pages + so);
    sVs[r] = *reinterpret_cast<const uint32_t*>(v_pages + so);
  }
  __syncthreads();

  // phase 3: online softmax over the split
  const int h = tid >> 3, part = tid & 7;
  float qv[16], o[16];
  {
    const uint16_t* qh = q + (t * kHeads + h) * kHeadDim + part * 16;
#pragma unroll
    for (int d = 0; d < 16; ++d) {
      qv[d] = bf16_bits_to_float(qh[d]) * scale_log2;
      o[d] = 0.f;
    }
  }
  float m = -INFINITY, l = 0.f;
  const int blk = part >> 1;  // scale block of dims 16*part .. 16*part+15
  for (int r = 0; r < cnt; ++r) {
    if (s_off[r] < 0) continue;
    const uint2 kd = *reinterpret_cast<const uint2*>(&sK[r][part * 8]);
    const float ks = e8m0_to_float((sKs[r] >> (8 * blk)) & 0xFFu);
    float dot = 0.f;
#pragma unroll
    for (int d = 0; d < 16; ++d) {
      const uint32_t w = d < 8 ? kd.x : kd.y;
      dot = fmaf(qv[d], e2m1_to_float(w >> (4 * (d & 7))), dot);
    }
    dot *= ks;  // this thread's 16 dims share one scale block
    dot += __shfl_xor_sync(0xFFFFFFFFu, dot, 1);
    dot += __shfl_xor_sync(0xFFFFFFFFu, dot, 2);
    dot += __shfl_xor_sync(0xFFFFFFFFu, dot, 4);
    const float logit = dot;  // log2 units
    const float m_new = fmaxf(m, logit);
    const float corr = exp2f(m - m_new);
    const float pw = exp2f(logit - m_new);
    l = l * corr + pw;
    m = m_new;
    const uint2 vd = *reinterpret_cast<const uint2*>(&sV[r][part * 8]);
    const float vs = e8m0_to_float((sVs[r] >> (8 * blk)) & 0xFFu) * pw;
#pragma unroll
    for (int d = 0; d < 16; ++d) {
      const uint32_t w = d < 8 ? vd.x : vd.y;
      o[d] = fmaf(e2m1_to_float(w >> (4 * (d & 7))), vs, o[d] * corr);
    }
  }
  const int64_t slot = (t * S + sp) * kHeads + h;
  float* wo = ws_o + slot * kHeadDim + part * 16;
#pragma unroll
  for (int d = 0; d < 16; d += 4)
    *reinterpret_cast<float4*>(wo + d) = make_float4(o[d], o[d + 1], o[d + 2], o[d + 3]);
  if (part == 0) {
    ws_ml[slot * 2 + 0] = m;
    ws_ml[slot * 2 + 1] = l;
  }
}

__global__ void __launch_bounds__(kHeadDim)
decode_merge_kernel(const float* __restrict__ ws_o, const float* __restrict__ ws_ml, int S,
                    float* __restrict__ out) {
  const int64_t t = blockIdx.x;
  const int d = threadIdx.x;
  for (int h = 0; h < kHeads; ++h) {
    float m = -INFINITY;
    for (int sp = 0; sp < S; ++sp) m = fmaxf(m, ws_ml[((t * S + sp) * kHeads + h) * 2]);
    float l = 0.f, acc = 0.f;
    if (m != -INFINITY) {
      for (int sp = 0; sp < S; ++sp) {
        const int64_t slot = (t * S + sp) * kHeads + h;
        const float ms = ws_ml[slot * 2];
        if (ms == -INFINITY) continue;
        const float w = exp2f(ms - m);
        l = fmaf(ws_ml[slot * 2 + 1], w, l);
        acc = fmaf(ws_o[slot * kHeadDim + d], w, acc);
      }
    }
    out[(t * kHeads + h) * kHeadDim + d] = (l > 0.f) ? acc / l : 0.f;
  }
}

int decode_splits(int kw) { return (kw + kSplitTokens - 1) / kSplitTokens; }

size_t decode_workspace_bytes(int64_t T, int kw) {
  const int64_t S = decode_splits(kw);
  return (size_t)(T * S * kHeads) * (kHeadDim + 2) * sizeof(float);
}

cudaError_t launch_decode(const uint16_t* q, int64_t T, int Q, const uint8_t* k_pages,
                          const uint8_t* v_pages, int64_t kv_page_stride, int64_t num_pages,
                          const int32_t* block_table, int64_t bt_width, const int32_t* seq_lens,
                          const int32_t* topk, int kw, float scale, float* out, void* ws,
                          uint32_t* status, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const int S = decode_splits(kw);
  float* ws_o = static_cast<float*>(ws);
  float* ws_ml = ws_o + T * S * kHeads * kHeadDim;
  decode_split_kernel<<<(unsigned)(T * S), kDecThreads, 0, stream>>>(
      q, Q, k_pages, v_pages, kv_page_stride, num_pages, block_table, bt_width, seq_lens, topk, kw,
      scale * kLog2e, S, ws_o, ws_ml, status);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  decode_merge_kernel<<<(unsigned)T, kHeadDim, 0, stream>>>(ws_o, ws_ml, S, out);
  return cudaGetLastError();
}

}  // namespace mx4
