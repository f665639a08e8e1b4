// sparse_paged_decode: GQA decode attention (16 query heads sharing one KV head,
// head_dim 128) over the selected tokens' MXFP4 K/V rows, split over the
// selected list with an online softmax per split and a merge kernel.
//
// K/V pages are [pages, heads, 8704] ("vllm.models.minimax_m3.amd.ops.
// mxfp4_pages", mxfp4_page_views: the [pages, heads, 128, 64] /
// [pages, heads, 128, 4] pair pa_decode takes).  Head geometry: one rank's
// q(2048) | k(128) | v(128) rows ("vllm.models.minimax_m3.amd.mono.weights",
// _build_cp_qkv), i.e. 16 query heads over one KV head, which makes the 16
// heads the M = 16 side of a tensor-core MMA.
//
// split kernel -- one CTA of 8 warps per (decode token, split of up to 512
// selected entries); warp w owns the 16-entry tiles w, w+8, w+16, w+24:
//   1. The sequence's block-table row goes to shared memory and warp 0 turns Q
//      into f16 MMA A fragments (bf16 scaled by a power of two, exact), kept in
//      shared memory.  Each warp then resolves its tiles' entries to page rows
//      and issues the gathers of all their scale words (one cp.async group),
//      then of each tile's 64 B K and V rows (one group per tile; rows padded
//      to 80 B so the fragment loads are bank-conflict free).
//   2. When the scale words land, the warp derives, for its 64 entries, the V
//      reference per 32-dim block (largest scale byte), K factors
//      2^(scale - 127) and exact f16 V multipliers 2^(scale - reference).
//   3. Each tile is processed as soon as its rows land, with no block-wide
//      step: S = Q K^T with mma.sync m16n8k16 (K = hardware e2m1 -> f16,
//      exact), one accumulator per 32-dim scale block, so the K scales are
//      applied exactly in fp32; online softmax in fp32 (log2 units, lazy
//      rescaling; weights scaled by 2^7 so the f16 P stays normal); P split
//      into f16 hi + lo parts so P V keeps ~22 bits; O += P V with mma.sync, V
//      fragments built by zipping the nibbles of two entries so one cvt yields
//      an (entry, entry) pair, times the V multipliers.
//   4. The 8 warps' (max, sum, O) are merged in shared memory, one float4 per
//      lane and MMA n-tile (bank-conflict free), and the split writes its
//      unnormalised [head][dim] output plus its running max (log2 units) and
//      sum per head.
// merge kernel -- one CTA per decode token combines the splits.
#include "common.cuh"

namespace mx4 {

constexpr int kHeads = 16;
constexpr int kDecWarps = 8;
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kSplitTokens = 512;                   // selected entries per CTA
constexpr int kTile = 16;                           // entries per MMA tile
constexpr int kTiles = kSplitTokens / kTile;        // 32
constexpr int kTilesPerWarp = kTiles / kDecWarps;   // 4
constexpr int kRowPitch = 80;                       // staged row pitch (64 B + 16 B pad)
constexpr int kTileV = kTile * kRowPitch;           // V rows follow the K rows
constexpr int kTileSw = 2 * kTile * kRowPitch;      // then 16 K and 16 V scale words
constexpr int kTileBytes = kTileSw + 2 * kTile * 4; // 2688 B
constexpr int kBtCache = 2048;                      // block-table entries kept in smem
constexpr int kFrag = kHeads * kHeadDim;            // 2048 outputs per split
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kPScale = 128.f;  // p' = 2^(logit - m) * 2^7, at most 2^15 in f16
constexpr float kLazy = 8.f;      // rescale only when the max grows by more than this
static_assert(kTilesPerWarp * kDecWarps == kTiles && kTilesPerWarp == 4, "split geometry");
static_assert(kTileBytes % 16 == 0, "16-byte aligned tiles");
static_assert(kDecWarps * kFrag * 4 <= kDecWarps * kTilesPerWarp * kTileBytes,
              "merge buffer fits in the tiles");

struct DecodeSmem {
  uint8_t tile[kDecWarps][kTilesPerWarp][kTileBytes];  // 84 KB; reused by the final merge
  uint4 qfrag[8][32];                                  // Q A fragments, per k16 slice and lane
  float4 kf[kDecWarps][kTilesPerWarp][kTile];          // K scale factors 2^(s_b - 127) * cQ
  uint16_t vm16[kDecWarps][kTilesPerWarp][4][kTile];   // f16 V multipliers [tile][block][entry]
  int32_t bt[kBtCache];                                // the sequence's block-table row
  float red_m[kDecWarps][kHeads];
  float red_l[kDecWarps][kHeads];
  int sigma;
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0));
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src),
               "r"(valid ? 4 : 0));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }
// wait until at most N of this thread's cp.async groups are pending
template <int N>
__device__ __forceinline__ void cp_async_wait_pending() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;\n" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t lop_merge(uint32_t a, uint32_t b, uint32_t m) {
  return (a & m) | (b & ~m);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ float f16_lo(uint32_t v) {
  return __half2float(__ushort_as_half((unsigned short)(v & 0xFFFFu)));
}
__device__ __forceinline__ float f16_hi(uint32_t v) {
  return __half2float(__ushort_as_half((unsigned short)(v >> 16)));
}

// f16 bit pattern of 2^e for e <= 0: normal down to 2^-14, subnormal down to
// 2^-24, 0 below.  A scale byte of 255 (NaN) gives an f16 NaN.
__device__ __forceinline__ uint32_t f16_pow2(uint32_t byte, uint32_t ref) {
  if (byte == 255u) return 0x7E00u;
  const int e = (int)byte - (int)ref;
  if (e >= -14) return (uint32_t)(e + 15) << 10;
  if (e >= -24) return 1u << (e + 24);
  return 0u;
}

// bytes equal to 0xFF (NaN scales) do not take part in the reference maximum
__device__ __forceinline__ uint32_t drop_nan_bytes(uint32_t w) {
  return w & ~__vcmpeq4(w, 0xFFFFFFFFu);
}

__global__ void __launch_bounds__(kDecThreads, 2)
decode_split_kernel(const uint16_t* __restrict__ q, int Q, const uint8_t* __restrict__ k_pages,
                    const uint8_t* __restrict__ v_pages, int64_t kv_page_stride,
                    int64_t num_pages, const int32_t* __restrict__ block_table, int64_t bt_width,
                    const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ topk,
                    int kw, float scale, int S, float* __restrict__ ws_o,
                    float* __restrict__ ws_ml, uint32_t* status) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  DecodeSmem& s = *reinterpret_cast<DecodeSmem*>(smem_raw);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_launch_dependents();
  const int g = lane >> 2, tig = lane & 3;
  const int64_t t = blockIdx.x / S;
  const int sp = blockIdx.x % S;
  const int64_t seq = t / Q;
  const int64_t p = (int64_t)seq_lens[seq] - Q + (t % Q);
  const int begin = sp * kSplitTokens;
  const int cnt = max(0, min(kSplitTokens, kw - begin));

  // ---- 1a. block-table row; Q as f16 A fragments (warp 0), scaled by 2^sigma
  // so that bf16 fits f16 exactly
  const int64_t npg = min(bt_width, max((int64_t)0, p / kPageTokens + 1));
  for (int j = tid; j < min(npg, (int64_t)kBtCache); j += kDecThreads)
    s.bt[j] = block_table[seq * bt_width + j];
  if (warp == 0) {
    uint4 qraw[2][4];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh)
#pragma unroll
      for (int b = 0; b < 4; ++b)
        qraw[hh][b] = *reinterpret_cast<const uint4*>(
            q + (t * kHeads + g + 8 * hh) * kHeadDim + 32 * b + 8 * tig);
    uint32_t amax = 0;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh)
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const uint32_t w[4] = {qraw[hh][b].x, qraw[hh][b].y, qraw[hh][b].z, qraw[hh][b].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          amax = max(amax, (w[j] << 17) >> 1);     // |low bf16| as fp32 bits
          amax = max(amax, (w[j] & 0x7FFF0000u));  // |high bf16|
        }
      }
    amax = __reduce_max_sync(0xFFFFFFFFu, amax);
    const int e = (int)(amax >> 23) - 127;
    const int sigma = (amax == 0u) ? 0 : min(127, max(-126, 14 - e));
    const float sc = __uint_as_float((uint32_t)(127 + sigma) << 23);
#pragma unroll
    for (int b = 0; b < 4; ++b)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        // slice 2b+h: k = 2tig,2tig+1 <-> dims 32b+8tig+4h+{0,1}; k = 2tig+8,+9 <-> +{2,3}
        const uint32_t w0 = h ? qraw[0][b].z : qraw[0][b].x, w1 = h ? qraw[0][b].w : qraw[0][b].y;
        const uint32_t u0 = h ? qraw[1][b].z : qraw[1][b].x, u1 = h ? qraw[1][b].w : qraw[1][b].y;
        s.qfrag[2 * b + h][lane] = make_uint4(
            pack_f16x2(bf16_bits_to_float(w0 & 0xFFFFu) * sc, bf16_bits_to_float(w0 >> 16) * sc),
            pack_f16x2(bf16_bits_to_float(u0 & 0xFFFFu) * sc, bf16_bits_to_float(u0 >> 16) * sc),
            pack_f16x2(bf16_bits_to_float(w1 & 0xFFFFu) * sc, bf16_bits_to_float(w1 >> 16) * sc),
            pack_f16x2(bf16_bits_to_float(u1 & 0xFFFFu) * sc, bf16_bits_to_float(u1 >> 16) * sc));
      }
    if (lane == 0) s.sigma = sigma;
  }
  pdl_wait();  // top-k indices and pages are touched from here on

  // ---- 1b. this warp's entries: lane l takes entry l/2 of each tile, its K row
  // and K scale word (even l) or its V row and V scale word (odd l)
  const int r = lane >> 1;
  const bool isv = (lane & 1) != 0;
  int32_t idx[kTilesPerWarp];
#pragma unroll
  for (int u = 0; u < kTilesPerWarp; ++u) {
    const int e = (warp + kDecWarps * u) * kTile + r;
    idx[u] = (e < cnt) ? topk[t * kw + begin + e] : -1;
  }
  __syncthreads();  // block-table row and Q fragments
  uint32_t okm[kTilesPerWarp];
  int rows[kTilesPerWarp];
  const uint8_t* srcs[kTilesPerWarp];
#pragma unroll
  for (int u = 0; u < kTilesPerWarp; ++u) {
    const int32_t i = idx[u];
    bool ok = false;
    const uint8_t* src = isv ? v_pages : k_pages;
    if (i >= 0) {
      if (i > p || (int64_t)i / kPageTokens >= bt_width) {
        flag(status, MX4_STATUS_BAD_INDEX);
      } else {
        const int64_t slot = i / kPageTokens;
        const int32_t pid = slot < kBtCache ? s.bt[slot] : block_table[seq * bt_width + slot];
        if (pid < 0 || pid >= num_pages) {
          flag(status, MX4_STATUS_BAD_PAGE);
        } else {
          src += (int64_t)pid * kv_page_stride;
          ok = true;
        }
      }
    }
    rows[u] = ok ? (i % kPageTokens) : -1;
    srcs[u] = src;
    okm[u] = __ballot_sync(0xFFFFFFFFu, ok);  // bit 2e: entry e of the tile is valid
    cp_async4(smem_addr(&s.tile[warp][u][0]) + kTileSw + (isv ? kTile * 4 : 0) + r * 4,
              src + kScaleOffset + (ok ? rows[u] : 0) * kRowScaleBytes, ok);
  }
  cp_async_commit();  // group: the scale words of all four tiles
#pragma unroll
  for (int u = 0; u < kTilesPerWarp; ++u) {
    const bool ok = rows[u] >= 0;
    const uint32_t dst = smem_addr(&s.tile[warp][u][0]) + (isv ? kTileV : 0) + r * kRowPitch;
    const uint8_t* src = srcs[u] + (ok ? rows[u] : 0) * kRowDataBytes;
#pragma unroll
    for (int c = 0; c < 4; ++c) cp_async16(dst + 16 * c, src + 16 * c, ok);
    cp_async_commit();  // group: the K and V rows of tile u
  }

  // logit (log2 units) = sum_b S_b * 2^(scale_b - 127) * cQ
  const float cQ = ldexpf(scale * kLog2e, -s.sigma);

  // ---- 1c. scale tables of the warp's 64 entries (while the rows are in flight):
  // the V reference per 32-dim block (largest valid scale byte, NaN excluded),
  // K factors 2^(s_b - 127) * cQ and f16 V multipliers 2^(s_b - ref_b)
  cp_async_wait_pending<kTilesPerWarp>();
  __syncwarp();
  uint32_t refV = 0u;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int u = (lane >> 4) + 2 * h, er = lane & 15;  // entries lane and lane + 32
    const uint32_t* sw = reinterpret_cast<const uint32_t*>(&s.tile[warp][u][kTileSw]);
    if ((okm[u] >> (2 * er)) & 1u) refV = __vmaxu4(refV, drop_nan_bytes(sw[kTile + er]));
  }
#pragma unroll
  for (int of = 16; of > 0; of >>= 1) refV = __vmaxu4(refV, __shfl_xor_sync(0xFFFFFFFFu, refV, of));
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int u = (lane >> 4) + 2 * h, er = lane & 15;
    const uint32_t* sw = reinterpret_cast<const uint32_t*>(&s.tile[warp][u][kTileSw]);
    const uint32_t kw4 = sw[er], vw4 = sw[kTile + er];
    s.kf[warp][u][er] = make_float4(e8m0_to_float(kw4 & 0xFFu) * cQ,
                                    e8m0_to_float((kw4 >> 8) & 0xFFu) * cQ,
                                    e8m0_to_float((kw4 >> 16) & 0xFFu) * cQ,
                                    e8m0_to_float(kw4 >> 24) * cQ);
#pragma unroll
    for (int b = 0; b < 4; ++b)
      s.vm16[warp][u][b][er] =
          (uint16_t)f16_pow2((vw4 >> (8 * b)) & 0xFFu, (refV >> (8 * b)) & 0xFFu);
  }
  __syncwarp();

  // ---- 3. this warp's tiles
  float o[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float m_used[2] = {-INFINITY, -INFINITY};
  float lsum[2] = {0.f, 0.f};

#pragma unroll
  for (int u = 0; u < kTilesPerWarp; ++u) {
    if ((warp + kDecWarps * u) * kTile >= cnt) break;
    if (u == 0) cp_async_wait_pending<3>();  // row groups of tiles u+1 .. 3 may be pending
    else if (u == 1) cp_async_wait_pending<2>();
    else if (u == 2) cp_async_wait_pending<1>();
    else cp_async_wait_pending<0>();
    __syncwarp();
    const uint8_t* sk = &s.tile[warp][u][0];
    const uint8_t* sv = sk + kTileV;
    const uint16_t* vm = &s.vm16[warp][u][0][0];
    const uint32_t okb = okm[u];

    // S = Q K^T per 32-dim scale block, two n8 tiles of entries
    float acc[2][4][4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint4 qa0 = s.qfrag[2 * b][lane], qa1 = s.qfrag[2 * b + 1][lane];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        acc[nt][b][0] = acc[nt][b][1] = acc[nt][b][2] = acc[nt][b][3] = 0.f;
        uint32_t f[4];
        e2m1x8_to_f16x2(
            *reinterpret_cast<const uint32_t*>(sk + (nt * 8 + g) * kRowPitch + (4 * b + tig) * 4),
            f);
        mma_m16n8k16_f16(acc[nt][b], qa0.x, qa0.y, qa0.z, qa0.w, f[0], f[1]);
        mma_m16n8k16_f16(acc[nt][b], qa1.x, qa1.y, qa1.z, qa1.w, f[2], f[3]);
      }
    }
    // logits of this thread's entries nt*8 + 2 tig + cc (heads g and g + 8)
    float lg[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int en = nt * 8 + 2 * tig + cc;
        const float4 kf = s.kf[warp][u][en];
        const float f[4] = {kf.x, kf.y, kf.z, kf.w};
        float d0 = 0.f, d1 = 0.f;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          d0 = fmaf(acc[nt][b][cc], f[b], d0);
          d1 = fmaf(acc[nt][b][cc + 2], f[b], d1);
        }
        const bool valid = (okb >> (2 * en)) & 1u;
        lg[nt][cc] = valid ? d0 : -INFINITY;
        lg[nt][cc + 2] = valid ? d1 : -INFINITY;
      }
    float mx[2];
    mx[0] = fmaxf(fmaxf(lg[0][0], lg[0][1]), fmaxf(lg[1][0], lg[1][1]));
    mx[1] = fmaxf(fmaxf(lg[0][2], lg[0][3]), fmaxf(lg[1][2], lg[1][3]));
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xFFFFFFFFu, mx[rr], 1));
      mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xFFFFFFFFu, mx[rr], 2));
    }
    const bool need = mx[0] > m_used[0] + kLazy || mx[1] > m_used[1] + kLazy;
    if (__any_sync(0xFFFFFFFFu, need)) {
      float corr[2];
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const float nm = mx[rr] > m_used[rr] + kLazy ? mx[rr] : m_used[rr];
        corr[rr] = (nm == m_used[rr]) ? 1.f : exp2f(m_used[rr] - nm);
        m_used[rr] = nm;
        lsum[rr] *= corr[rr];
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        o[j][0] *= corr[0];
        o[j][1] *= corr[0];
        o[j][2] *= corr[1];
        o[j][3] *= corr[1];
      }
    }
    // p' = 2^(logit - m) * 2^7: the largest logit gets exactly 128
    const float mb0 = (m_used[0] == -INFINITY) ? 0.f : m_used[0];
    const float mb1 = (m_used[1] == -INFINITY) ? 0.f : m_used[1];
    float pw[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      pw[nt][0] = exp2f(lg[nt][0] - mb0) * kPScale;
      pw[nt][1] = exp2f(lg[nt][1] - mb0) * kPScale;
      pw[nt][2] = exp2f(lg[nt][2] - mb1) * kPScale;
      pw[nt][3] = exp2f(lg[nt][3] - mb1) * kPScale;
    }
    lsum[0] += (pw[0][0] + pw[0][1]) + (pw[1][0] + pw[1][1]);
    lsum[1] += (pw[0][2] + pw[0][3]) + (pw[1][2] + pw[1][3]);
    // P = hi + lo, both f16
    uint32_t ph[4], pl[4];
    ph[0] = pack_f16x2(pw[0][0], pw[0][1]);
    ph[1] = pack_f16x2(pw[0][2], pw[0][3]);
    ph[2] = pack_f16x2(pw[1][0], pw[1][1]);
    ph[3] = pack_f16x2(pw[1][2], pw[1][3]);
    pl[0] = pack_f16x2(pw[0][0] - f16_lo(ph[0]), pw[0][1] - f16_hi(ph[0]));
    pl[1] = pack_f16x2(pw[0][2] - f16_lo(ph[1]), pw[0][3] - f16_hi(ph[1]));
    pl[2] = pack_f16x2(pw[1][0] - f16_lo(ph[2]), pw[1][1] - f16_hi(ph[2]));
    pl[3] = pack_f16x2(pw[1][2] - f16_lo(ph[3]), pw[1][3] - f16_hi(ph[3]));

    // O += P V: dim tile j = 8h + i, column g <-> dim 8(g + 8h) + i (block (g>>2) + 2h)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int wi = (g + 8 * h) * 4;
      const int bh = (g >> 2) + 2 * h;
      const uint32_t m01 = *reinterpret_cast<const uint32_t*>(&vm[bh * kTile + 2 * tig]);
      const uint32_t m89 = *reinterpret_cast<const uint32_t*>(&vm[bh * kTile + 8 + 2 * tig]);
      const uint32_t wA = *reinterpret_cast<const uint32_t*>(sv + (2 * tig) * kRowPitch + wi);
      const uint32_t wB = *reinterpret_cast<const uint32_t*>(sv + (2 * tig + 1) * kRowPitch + wi);
      const uint32_t wC = *reinterpret_cast<const uint32_t*>(sv + (2 * tig + 8) * kRowPitch + wi);
      const uint32_t wD = *reinterpret_cast<const uint32_t*>(sv + (2 * tig + 9) * kRowPitch + wi);
      // nibble zip: byte q of ze = (A.dim 2q) | (B.dim 2q) << 4; zo likewise for 2q+1
      uint32_t ze01[4], zo01[4], ze89[4], zo89[4];
      e2m1x8_to_f16x2(lop_merge(wA, wB << 4, 0x0F0F0F0Fu), ze01);
      e2m1x8_to_f16x2(lop_merge(wA >> 4, wB, 0x0F0F0F0Fu), zo01);
      e2m1x8_to_f16x2(lop_merge(wC, wD << 4, 0x0F0F0F0Fu), ze89);
      e2m1x8_to_f16x2(lop_merge(wC >> 4, wD, 0x0F0F0F0Fu), zo89);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t b0 = hmul2((i & 1) ? zo01[i >> 1] : ze01[i >> 1], m01);
        const uint32_t b1 = hmul2((i & 1) ? zo89[i >> 1] : ze89[i >> 1], m89);
        mma_m16n8k16_f16(o[8 * h + i], ph[0], ph[1], ph[2], ph[3], b0, b1);
        mma_m16n8k16_f16(o[8 * h + i], pl[0], pl[1], pl[2], pl[3], b0, b1);
      }
    }
  }
  cp_async_wait_all();  // gathers of tiles past the end land before the merge reuses them

  // ---- 4. merge the warps' partial results (fragment order, conflict free)
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    lsum[rr] += __shfl_xor_sync(0xFFFFFFFFu, lsum[rr], 1);
    lsum[rr] += __shfl_xor_sync(0xFFFFFFFFu, lsum[rr], 2);
  }
  __syncthreads();  // every warp is done with its tiles
  if (tig == 0) {
    s.red_m[warp][g] = m_used[0];
    s.red_m[warp][g + 8] = m_used[1];
    s.red_l[warp][g] = lsum[0];
    s.red_l[warp][g + 8] = lsum[1];
  }
  __syncthreads();
  float M[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int w = 0; w < kDecWarps; ++w) {
    M[0] = fmaxf(M[0], s.red_m[w][g]);
    M[1] = fmaxf(M[1], s.red_m[w][g + 8]);
  }
  float fw[2];
#pragma unroll
  for (int rr = 0; rr < 2; ++rr)
    fw[rr] = (m_used[rr] == -INFINITY) ? 0.f : exp2f(m_used[rr] - M[rr]);
  float fv[4];
#pragma unroll
  for (int b = 0; b < 4; ++b) fv[b] = ldexpf(1.f, (int)((refV >> (8 * b)) & 0xFFu) - 127);
  // elements (j, 0..3) of lane l live in one float4 at red4[warp][j * 32 + l]
  float4* red4 = reinterpret_cast<float4*>(&s.tile[0][0][0]);
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float f = fv[(2 * tig + 8 * (j >> 3)) >> 2];
    const float f0 = fw[0] * f, f1 = fw[1] * f;
    red4[warp * (kFrag / 4) + j * 32 + lane] =
        make_float4(o[j][0] * f0, o[j][1] * f0, o[j][2] * f1, o[j][3] * f1);
  }
  __syncthreads();
  // float4 x = j * 32 + lane -> element c: head = g + 8 (c/2) (g = lane/4),
  // dim = 8 (2 tig + c%2 + 8 (j/8)) + j%8 (tig = lane%4)
  const int64_t split = t * S + sp;
  for (int x = tid; x < kFrag / 4; x += kDecThreads) {
    float4 acc = red4[x];
#pragma unroll
    for (int w = 1; w < kDecWarps; ++w) {
      const float4 y = red4[w * (kFrag / 4) + x];
      acc.x += y.x;
      acc.y += y.y;
      acc.z += y.z;
      acc.w += y.w;
    }
    const int ln = x & 31, j = x >> 5;
    const int h0 = ln >> 2;
    const int d0 = 8 * (2 * (ln & 3) + 8 * (j >> 3)) + (j & 7);
    float* dst = ws_o + split * kFrag;
    dst[h0 * kHeadDim + d0] = acc.x;
    dst[h0 * kHeadDim + d0 + 8] = acc.y;
    dst[(h0 + 8) * kHeadDim + d0] = acc.z;
    dst[(h0 + 8) * kHeadDim + d0 + 8] = acc.w;
  }
  if (tid < kHeads) {
    float Mh = -INFINITY;
    for (int w = 0; w < kDecWarps; ++w) Mh = fmaxf(Mh, s.red_m[w][tid]);
    float l = 0.f;
    if (Mh != -INFINITY)
      for (int w = 0; w < kDecWarps; ++w)
        if (s.red_m[w][tid] != -INFINITY) l += s.red_l[w][tid] * exp2f(s.red_m[w][tid] - Mh);
    ws_ml[(split * kHeads + tid) * 2 + 0] = Mh;
    ws_ml[(split * kHeads + tid) * 2 + 1] = l;
  }
}

// One CTA per decode token; thread (h, part) combines dims 4*part .. 4*part+3 of
// head h over the splits: out = sum_s O_s 2^(m_s - M) / sum_s l_s 2^(m_s - M),
// with O_s the split's unnormalised [head][dim] output and (m_s, l_s) its
// running max (log2 units) and sum for the head.
constexpr int kMergeThreads = kHeads * (kHeadDim / 4);  // 512
constexpr int kMaxSplits = 128;
__global__ void __launch_bounds__(kMergeThreads)
decode_merge_kernel(const float* __restrict__ ws_o, const float* __restrict__ ws_ml, int S,
                    float* __restrict__ out) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t t = blockIdx.x;
  const int h = threadIdx.x / (kHeadDim / 4), d0 = 4 * (threadIdx.x % (kHeadDim / 4));
  float M = -INFINITY;
  for (int sp = 0; sp < S; ++sp) M = fmaxf(M, ws_ml[((t * S + sp) * kHeads + h) * 2]);
  float l = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (M != -INFINITY) {
    for (int sp = 0; sp < S; ++sp) {
      const int64_t slot = (t * S + sp) * kHeads + h;
      const float ms = ws_ml[slot * 2];
      if (ms == -INFINITY) continue;
      const float w = exp2f(ms - M);
      l = fmaf(ws_ml[slot * 2 + 1], w, l);
      const float4 x = *reinterpret_cast<const float4*>(ws_o + slot * kHeadDim + d0);
      acc.x = fmaf(x.x, w, acc.x);
      acc.y = fmaf(x.y, w, acc.y);
      acc.z = fmaf(x.z, w, acc.z);
      acc.w = fmaf(x.w, w, acc.w);
    }
  }
  float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
  if (l > 0.f) r = make_float4(acc.x / l, acc.y / l, acc.z / l, acc.w / l);
  *reinterpret_cast<float4*>(out + (t * kHeads + h) * kHeadDim + d0) = r;
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
  if (S > kMaxSplits) return cudaErrorInvalidValue;
  float* ws_o = static_cast<float*>(ws);
  float* ws_ml = ws_o + T * S * kFrag;
  const int smem = (int)sizeof(DecodeSmem);
  cudaError_t err =
      cudaFuncSetAttribute(decode_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  err = launch_pdl(decode_split_kernel, dim3((unsigned)(T * S)), dim3(kDecThreads), smem, stream,
                   q, Q, k_pages, v_pages, kv_page_stride, num_pages, block_table, bt_width,
                   seq_lens, topk, kw, scale, S, ws_o, ws_ml, status);
  if (err != cudaSuccess) return err;
  return launch_pdl(decode_merge_kernel, dim3((unsigned)T), dim3(kMergeThreads), 0, stream,
                    (const float*)ws_o, (const float*)ws_ml, S, out);
}

}  // namespace mx4
