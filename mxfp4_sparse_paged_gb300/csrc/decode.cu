// sparse_paged_decode: GQA decode attention (16 query heads sharing one KV head,
// head_dim 128) over the selected tokens' MXFP4 K/V rows, with an online
// softmax over each run of selected entries and a merge of the runs.
//
// K/V pages are [pages, heads, 8704] ("vllm.models.minimax_m3.amd.ops.
// mxfp4_pages", mxfp4_page_views: the [pages, heads, 128, 64] /
// [pages, heads, 128, 4] pair pa_decode takes).  Head geometry: one rank's
// q(2048) | k(128) | v(128) rows ("vllm.models.minimax_m3.amd.mono.weights",
// _build_cp_qkv), i.e. 16 query heads over one KV head, which makes the 16
// heads the M = 16 side of a tensor-core MMA.
//
// Work.  The selected lists of all decode tokens are cut into tiles of 16
// entries (ceil(k / 16) tiles per token), and the tiles, token after token, into
// equal contiguous ranges, one per warp of a persistent grid (one CTA of 8 warps
// per SM).  Each warp streams its range through a ring of kRing shared-memory
// tile slots with cp.async, so the gathers of the next kRing - 1 tiles are in
// flight while it computes one.  The address of a selected row takes two
// dependent loads (top-k index, then block-table entry); they run one and two
// tiles ahead of the copies, so no wait sits on the critical path.
//
// On this GPU a random 64-byte row read costs a 128-byte DRAM access, so a
// sparse selection moves up to twice the layout's 68 bytes per row; keeping
// many rows in flight is what the kernel can do about it.
//
// Math per tile (tensor cores, mma.sync m16n8k16, fp32 accumulation):
//   S = Q K^T with one accumulator per 32-dim scale block (K codes by the exact
//   hardware e2m1 -> f16 conversion; the K scales applied in fp32);
//   online softmax in log2 units with lazy rescaling (weights scaled by 2^7 so
//   the f16 P stays normal; powers of two by the hardware's approximate exp2); P split into f16 hi + lo parts so P V keeps about
//   22 bits; O += P V with V fragments built by zipping the nibbles of two
//   entries, times exact f16 multipliers 2^(scale - reference), where the
//   reference is the warp's running largest scale byte per 32-dim block (O is
//   rescaled by a power of two when it grows).
// At each token boundary of its range a warp writes its run's partial result
// (unnormalised O, running max and sum per head) to the workspace; the merge
// kernel combines the runs of each token.
#include <algorithm>

#include "common.cuh"

namespace mx4 {

constexpr int kHeads = 16;
constexpr int kDecWarps = 8;                        // warps per CTA (one CTA per SM)
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kRing = 4;                            // tile slots per warp
constexpr int kTile = 16;                           // entries per MMA tile
constexpr int kRowPitch = 80;                       // staged row pitch (64 B + 16 B pad)
constexpr int kTileV = kTile * kRowPitch;           // V rows follow the K rows
constexpr int kTileSw = 2 * kTile * kRowPitch;      // then 16 K and 16 V scale words
constexpr int kTileBytes = kTileSw + 2 * kTile * 4; // 2688 B
constexpr int kFrag = kHeads * kHeadDim;            // 2048 outputs per token
constexpr int kRecFloats = kFrag + 2 * kHeads;      // partial record: O, max, sum
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kPScale = 128.f;  // p' = 2^(logit - m) * 2^7, at most 2^15 in f16
constexpr float kLazy = 8.f;      // rescale only when the max grows by more than this
static_assert(kTileBytes % 16 == 0, "16-byte aligned tiles");

struct WarpSmem {
  uint8_t slot[kRing][kTileBytes];  // the ring of gathered tiles
  float4 kf[kTile];                 // K scale factors 2^(s_b - 127) * cQ of the tile computed
  uint16_t vm16[4][kTile];          // f16 V multipliers [block][entry] of that tile
  uint32_t okm[kRing];              // valid-entry mask (bit 2e) of each slot
};
struct DecodeSmem {
  WarpSmem w[kDecWarps];
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

// f16 bit pattern of 2^(byte - ref) for byte <= ref: normal down to 2^-14,
// subnormal down to 2^-24, 0 below.  A scale byte of 255 (NaN) gives an f16 NaN.
__device__ __forceinline__ uint16_t f16_pow2(uint32_t byte, int ref) {
  if (byte == 255u) return 0x7E00u;
  const int e = (int)byte - ref;
  if (e >= -14) return (uint16_t)((e + 15) << 10);
  if (e >= -24) return (uint16_t)(1u << (e + 24));
  return 0u;
}

// First tile of the range of warp g: the T * NT tiles cut into NW equal ranges.
__host__ __device__ __forceinline__ int64_t warp_tile_begin(int64_t g, int64_t U, int64_t NW) {
  return U * g / NW;
}

// Per-launch constants of the split kernel.
struct DecodeArgs {
  const uint16_t* q;
  const uint8_t* k_pages;
  const uint8_t* v_pages;
  int64_t kv_page_stride;
  int64_t num_pages;
  const int32_t* block_table;
  int64_t bt_width;
  const int32_t* seq_lens;
  const int32_t* topk;
  float* ws;  // partial records [NW + T][kRecFloats]
  uint32_t* status;
  int64_t U;  // tiles in all
  int NT;     // tiles per token
  int kw;     // top-k width (entries per token)
  int Q;      // decode tokens per sequence
  float scale;
};

// Q of token t as this lane's f16 A fragments (qf[k16 slice]), held in registers for
// the token's tiles: bf16 scaled by 2^sigma so the largest magnitude lands in
// [2^14, 2^15).  The conversion is exact for every element whose exponent is at most
// 31 below the largest one's; smaller elements round on the f16 subnormal grid
// (2^-24 after scaling).  Returns sigma.
__device__ __forceinline__ int load_q_fragments(const uint16_t* __restrict__ q, int64_t t,
                                                uint4 (&qf)[8], int lane) {
  const int g = lane >> 2, tig = lane & 3;
  uint4 qraw[2][4];
#pragma unroll
  for (int hh = 0; hh < 2; ++hh)
#pragma unroll
    for (int b = 0; b < 4; ++b)
      qraw[hh][b] = *reinterpret_cast<const uint4*>(q + (t * kHeads + g + 8 * hh) * kHeadDim +
                                                    32 * b + 8 * tig);
  uint32_t amax = 0;
#pragma unroll
  for (int hh = 0; hh < 2; ++hh)
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint32_t x[4] = {qraw[hh][b].x, qraw[hh][b].y, qraw[hh][b].z, qraw[hh][b].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        amax = max(amax, (x[j] << 17) >> 1);     // |low bf16| as fp32 bits
        amax = max(amax, (x[j] & 0x7FFF0000u));  // |high bf16|
      }
    }
  amax = __reduce_max_sync(0xFFFFFFFFu, amax);
  const int e = (int)(amax >> 23) - 127;
  // sigma puts the largest |q| near 2^14 (never above it, so no f16 overflow); the
  // upper clamp keeps 2^-sigma, folded into the K factors, a normal fp32 number
  const int sigma = (amax == 0u) ? 0 : min(100, max(-113, 14 - e));
  const float sc = __uint_as_float((uint32_t)(127 + sigma) << 23);
#pragma unroll
  for (int b = 0; b < 4; ++b)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      // slice 2b+h: k = 2tig,2tig+1 <-> dims 32b+8tig+4h+{0,1}; k = 2tig+8,+9 <-> +{2,3}
      const uint32_t w0 = h ? qraw[0][b].z : qraw[0][b].x, w1 = h ? qraw[0][b].w : qraw[0][b].y;
      const uint32_t u0 = h ? qraw[1][b].z : qraw[1][b].x, u1 = h ? qraw[1][b].w : qraw[1][b].y;
      qf[2 * b + h] = make_uint4(
          pack_f16x2(bf16_bits_to_float(w0 & 0xFFFFu) * sc, bf16_bits_to_float(w0 >> 16) * sc),
          pack_f16x2(bf16_bits_to_float(u0 & 0xFFFFu) * sc, bf16_bits_to_float(u0 >> 16) * sc),
          pack_f16x2(bf16_bits_to_float(w1 & 0xFFFFu) * sc, bf16_bits_to_float(w1 >> 16) * sc),
          pack_f16x2(bf16_bits_to_float(u1 & 0xFFFFu) * sc, bf16_bits_to_float(u1 >> 16) * sc));
    }
  return sigma;
}

// 2^x by the hardware's approximate base-2 exponential (PTX ex2.approx, flushing
// subnormal results to zero); 2^-inf = +0.
__device__ __forceinline__ float ex2_hw(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// 2^e as fp32 for e <= 127 (0 below the normal range).
__device__ __forceinline__ float pow2f(int e) {
  return e >= -126 ? __uint_as_float((uint32_t)(127 + e) << 23) : 0.f;
}

__global__ void __launch_bounds__(kDecThreads, 1) decode_split_kernel(const DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  DecodeSmem& sm = *reinterpret_cast<DecodeSmem*>(smem_raw);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  WarpSmem& w = sm.w[warp];
  pdl_launch_dependents();
  const int g = lane >> 2, tig = lane & 3;
  const int r = lane >> 1;           // entry of a tile whose row this lane gathers
  const bool isv = (lane & 1) != 0;  // its V row and scale word (odd lanes) or K's (even)
  const int64_t NW = (int64_t)gridDim.x * kDecWarps;
  const int64_t gw = (int64_t)blockIdx.x * kDecWarps + warp;
  const int64_t u0 = warp_tile_begin(gw, a.U, NW), u1 = warp_tile_begin(gw + 1, a.U, NW);
  pdl_wait();  // top-k indices (and q, pages) are touched from here on
  if (u0 >= u1) return;  // no CTA-wide barrier in this kernel

  // ---- the address pipeline: top-k index -> block-table entry -> copies.  Each
  // stage walks the tiles in order, so its (token, tile of the token, sequence,
  // position) advances by one tile at a time without divisions.
  struct Pos {
    int64_t u;
    int t, j, seq;
    int64_t p;  // the token's position: it attends to cached tokens 0 .. p
  };
  auto at = [&](int64_t u) {
    Pos x;
    x.u = u;
    x.t = (int)(u / a.NT);
    x.j = (int)(u - (int64_t)x.t * a.NT);
    x.seq = x.t / a.Q;
    x.p = u < u1 ? (int64_t)__ldg(a.seq_lens + x.seq) - a.Q + (x.t - x.seq * a.Q) : -1;
    return x;
  };
  auto next = [&](Pos& x) {
    ++x.u;
    if (++x.j == a.NT) {
      x.j = 0;
      ++x.t;
      x.seq = x.t / a.Q;
      x.p = x.u < u1 ? (int64_t)__ldg(a.seq_lens + x.seq) - a.Q + (x.t - x.seq * a.Q) : -1;
    }
  };
  auto load_idx = [&](const Pos& x) -> int32_t {
    if (x.u >= u1) return -1;
    const int e = x.j * kTile + r;
    return e < a.kw ? __ldg(a.topk + (int64_t)x.t * a.kw + e) : -1;
  };
  auto resolve = [&](const Pos& x, int32_t i, int32_t& row) -> int32_t {
    row = -1;
    if (i < 0 || x.u >= u1) return -1;
    const uint32_t slot = (uint32_t)i >> 7;
    if ((int64_t)i > x.p || (int64_t)slot >= a.bt_width) {
      if (!isv) flag(a.status, MX4_STATUS_BAD_INDEX);
      return -1;
    }
    row = i & (kPageTokens - 1);
    return __ldg(a.block_table + (int64_t)x.seq * a.bt_width + slot);
  };
  auto issue = [&](int64_t u, int sl, int32_t pid, int32_t row) {
    if (u < u1) {
      bool ok = false;
      const uint8_t* src = isv ? a.v_pages : a.k_pages;
      if (row >= 0) {
        if (pid < 0 || pid >= a.num_pages) {
          if (!isv) flag(a.status, MX4_STATUS_BAD_PAGE);
        } else {
          src += (int64_t)pid * a.kv_page_stride;
          ok = true;
        }
      }
      const uint32_t okm = __ballot_sync(0xFFFFFFFFu, ok);  // bit 2e: entry e valid
      if (lane == 0) w.okm[sl] = okm;
      const uint32_t base = smem_addr(&w.slot[sl][0]);
      cp_async4(base + kTileSw + (isv ? kTile * 4 : 0) + r * 4,
                src + kScaleOffset + (ok ? row : 0) * kRowScaleBytes, ok);
      const uint32_t dst = base + (isv ? kTileV : 0) + r * kRowPitch;
      const uint8_t* rs = src + (ok ? row : 0) * kRowDataBytes;
#pragma unroll
      for (int c = 0; c < 4; ++c) cp_async16(dst + 16 * c, rs + 16 * c, ok);
    }
    cp_async_commit();  // one group per tile (empty past the range)
  };

  // prologue: the first kRing tiles' indices and pages (independent loads), the
  // copies of the first kRing - 1
  int32_t pid_b, row_b, i_a;
  Pos x_res, x_idx;  // the tiles whose page / index the loop looks up next
  {
    int32_t ii[kRing], pp[kRing], rr[kRing];
    Pos x = at(u0);
    Pos xs[kRing];
#pragma unroll
    for (int s = 0; s < kRing; ++s) {
      xs[s] = x;
      ii[s] = load_idx(x);
      next(x);
    }
#pragma unroll
    for (int s = 0; s < kRing; ++s) pp[s] = resolve(xs[s], ii[s], rr[s]);
#pragma unroll
    for (int s = 0; s < kRing - 1; ++s) issue(u0 + s, s, pp[s], rr[s]);
    pid_b = pp[kRing - 1];
    row_b = rr[kRing - 1];
    x_res = x;  // tile u0 + kRing
    i_a = load_idx(x_res);
    x_idx = x_res;
    next(x_idx);  // tile u0 + kRing + 1
  }

  // ---- per-run state
  float o[16][4];
  float m_used[2] = {-INFINITY, -INFINITY}, lsum[2] = {0.f, 0.f};
  int ref[4] = {0, 0, 0, 0};  // largest valid V scale byte per 32-dim block so far
  float cQ = 0.f;
  int64_t cur_t = -1;
  uint4 qf[8];  // Q fragments of the current token
  const int blo = tig >> 1;  // scale block of this lane's O columns j < 8 (blo + 2 for j >= 8)

  auto flush = [&](int64_t t) {
    float l0 = lsum[0], l1 = lsum[1];
    l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, 1);
    l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, 2);
    l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, 1);
    l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, 2);
    float* rec = a.ws + (gw + t) * kRecFloats;
    const float flo = pow2f((blo ? ref[1] : ref[0]) - 127), fhi = pow2f((blo ? ref[3] : ref[2]) - 127);
    float4* r4 = reinterpret_cast<float4*>(rec);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float f = j < 8 ? flo : fhi;
      r4[j * 32 + lane] = make_float4(o[j][0] * f, o[j][1] * f, o[j][2] * f, o[j][3] * f);
    }
    if (tig == 0) {
      rec[kFrag + g] = m_used[0];
      rec[kFrag + g + 8] = m_used[1];
      rec[kFrag + kHeads + g] = l0;
      rec[kFrag + kHeads + g + 8] = l1;
    }
  };

  int sl = 0;  // slot of tile u
  int t_prev = -1;
  int t = u0 / a.NT, jt = (int)(u0 - (int64_t)t * a.NT);  // token and tile of token of u
  for (int64_t u = u0; u < u1; ++u) {
    // copies of tile u + kRing - 1 (into the slot tile u - 1 used), its page looked
    // up last iteration; the page of tile u + kRing; the index of tile u + kRing + 1
    issue(u + kRing - 1, sl == 0 ? kRing - 1 : sl - 1, pid_b, row_b);
    pid_b = resolve(x_res, i_a, row_b);
    i_a = load_idx(x_idx);
    next(x_res);
    next(x_idx);

    if (t != t_prev) {  // a new run: flush the last one, take this token's Q
      if (cur_t >= 0) flush(cur_t);
      cur_t = t;
      t_prev = t;
#pragma unroll
      for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
      m_used[0] = m_used[1] = -INFINITY;
      lsum[0] = lsum[1] = 0.f;
      ref[0] = ref[1] = ref[2] = ref[3] = 0;
      const int sigma = load_q_fragments(a.q, t, qf, lane);
      cQ = a.scale * kLog2e * pow2f(-sigma);  // logit (log2 units) = sum_b S_b 2^(s_b-127) cQ
    }
    cp_async_wait_pending<kRing - 1>();  // tile u has landed
    __syncwarp();
    const uint32_t okb = w.okm[sl];
    if (okb != 0u) {
      const uint8_t* sk = &w.slot[sl][0];
      const uint8_t* sv = sk + kTileV;
      const uint32_t* sw = reinterpret_cast<const uint32_t*>(sk + kTileSw);
      // ---- scale tables of the tile: V reference, K factors, V multipliers.  Lane l
      // takes entry l % 16 and the scale blocks 2 (l / 16) and 2 (l / 16) + 1.
      {
        const int er = lane & 15, bp = lane >> 4;
        const uint32_t kwd = sw[er], vwd = sw[kTile + er];
        const bool ev = (okb >> (2 * er)) & 1u;
        int nref[4];
        bool grow = false;
#pragma unroll
        for (int b = 0; b < 4; ++b) {  // largest valid scale byte of the tile (NaN excluded)
          uint32_t x = (vwd >> (8 * b)) & 0xFFu;
          x = __reduce_max_sync(0xFFFFFFFFu, (ev && x != 0xFFu) ? x : 0u);
          nref[b] = max(ref[b], (int)x);
          grow |= nref[b] != ref[b];
        }
        if (grow) {  // warp-uniform: bring O to the larger reference
          const float flo = pow2f((blo ? ref[1] : ref[0]) - (blo ? nref[1] : nref[0]));
          const float fhi = pow2f((blo ? ref[3] : ref[2]) - (blo ? nref[3] : nref[2]));
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float f = j < 8 ? flo : fhi;
            o[j][0] *= f;
            o[j][1] *= f;
            o[j][2] *= f;
            o[j][3] *= f;
          }
#pragma unroll
          for (int b = 0; b < 4; ++b) ref[b] = nref[b];
        }
        const int sh = 16 * bp;
        *reinterpret_cast<float2*>(&w.kf[er].x + 2 * bp) =
            make_float2(e8m0_to_float((kwd >> sh) & 0xFFu) * cQ,
                        e8m0_to_float((kwd >> (sh + 8)) & 0xFFu) * cQ);
        w.vm16[2 * bp][er] = f16_pow2((vwd >> sh) & 0xFFu, bp ? ref[2] : ref[0]);
        w.vm16[2 * bp + 1][er] = f16_pow2((vwd >> (sh + 8)) & 0xFFu, bp ? ref[3] : ref[1]);
        __syncwarp();
      }
      const uint16_t* vm = &w.vm16[0][0];

      // ---- S = Q K^T per 32-dim scale block, two n8 tiles of entries
      float acc[2][4][4];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const uint4 qa0 = qf[2 * b], qa1 = qf[2 * b + 1];
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
          const float4 kf = w.kf[en];
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
          corr[rr] = (nm == m_used[rr]) ? 1.f : ex2_hw(m_used[rr] - nm);
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
        pw[nt][0] = ex2_hw(lg[nt][0] - mb0) * kPScale;
        pw[nt][1] = ex2_hw(lg[nt][1] - mb0) * kPScale;
        pw[nt][2] = ex2_hw(lg[nt][2] - mb1) * kPScale;
        pw[nt][3] = ex2_hw(lg[nt][3] - mb1) * kPScale;
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

      // ---- O += P V: dim tile j = 8h + i, column g <-> dim 8(g + 8h) + i (block (g>>2) + 2h)
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
    __syncwarp();  // the slot of tile u is reused by the next iteration's copies
    sl = (sl == kRing - 1) ? 0 : sl + 1;
    if (++jt == a.NT) {
      jt = 0;
      ++t;
    }
  }
  flush(cur_t);
  asm volatile("cp.async.wait_all;\n" ::: "memory");  // no copy in flight at exit
}

// gridDim.y CTAs per decode token (1 or 4), each 4 / gridDim.y quarters of the
// fragment order (quarter y: fragments j of 4 y .. 4 y + 3), thread x = (j, lane)
// of the fragment order: combines
// the runs of the token, out = sum_r O_r 2^(m_r - M) / sum_r l_r 2^(m_r - M), with
// O_r the run's unnormalised output and (m_r, l_r) its running max (log2 units)
// and sum per head; the runs are those of the warps whose ranges meet the token's
// tiles.  A quarter is 16 heads x 32 dims of the output, in runs of 4 dims: it goes
// through shared memory to 16-byte stores.  A token met by many warps (many
// records) takes 4 CTAs, so the records of few tokens spread over the SMs.
constexpr int kMergeQuarter = kFrag / 4 / 4;  // 128 float4 of the fragment order
constexpr int kMergeSplitRuns = 8;            // more runs per token than this: 4 CTAs

// SPLIT CTAs per token of 512 / SPLIT threads; runs whose loads are in flight
// together: 6 at 512 threads (two CTAs per SM), 8 at 128.
template <int SPLIT>
__global__ void __launch_bounds__(4 * kMergeQuarter / SPLIT, SPLIT == 1 ? 2 : 1)
decode_merge_kernel(const float* __restrict__ ws, int64_t U, int64_t NW, int NT,
                    float* __restrict__ out) {
  constexpr int kMergeUnroll = SPLIT == 1 ? 6 : 8;
  __shared__ __align__(16) float so[4][kHeads][32];
  __shared__ int64_t s_g[2];
  pdl_launch_dependents();
  const int64_t t = blockIdx.x;
  const int x = blockIdx.y * blockDim.x + threadIdx.x, j = x >> 5, lane = x & 31;
  const int qy = x / kMergeQuarter, lq = threadIdx.x / kMergeQuarter;  // quarter, local
  const int h0 = lane >> 2, tig = lane & 3;
  if (threadIdx.x < 2) {
    // the warp whose range holds the token's first (0) or last (1) tile: the last
    // g with begin(g) <= tile
    const int64_t tile = threadIdx.x == 0 ? t * NT : (t + 1) * NT - 1;
    int64_t lo = 0, hi = NW - 1;
    while (lo < hi) {
      const int64_t mid = (lo + hi + 1) >> 1;
      if (warp_tile_begin(mid, U, NW) <= tile) lo = mid; else hi = mid - 1;
    }
    s_g[threadIdx.x] = lo;
  }
  __syncthreads();
  pdl_wait();
  const int64_t g0 = s_g[0], g1 = s_g[1];
  const bool gaps = U < NW;  // only then can a warp's range be empty (no run record)
  auto live = [&](int64_t gw) {
    return !gaps || warp_tile_begin(gw, U, NW) != warp_tile_begin(gw + 1, U, NW);
  };
  // one pass over the runs, kMergeUnroll of them in flight: the running max per
  // head rescales what is summed so far when a run raises it
  float M0 = -INFINITY, M1 = -INFINITY;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float L0 = 0.f, L1 = 0.f;
  for (int64_t gw = g0; gw <= g1; gw += kMergeUnroll) {
    float m0[kMergeUnroll], m1[kMergeUnroll], l0[kMergeUnroll], l1[kMergeUnroll];
    float4 v[kMergeUnroll];
#pragma unroll
    for (int u = 0; u < kMergeUnroll; ++u) {
      const int64_t g = gw + u;
      const bool ok = g <= g1 && live(g);
      const float* rec = ws + (ok ? g + t : g0 + t) * kRecFloats;
      m0[u] = ok ? rec[kFrag + h0] : -INFINITY;
      m1[u] = ok ? rec[kFrag + h0 + 8] : -INFINITY;
      l0[u] = rec[kFrag + kHeads + h0];
      l1[u] = rec[kFrag + kHeads + h0 + 8];
      v[u] = reinterpret_cast<const float4*>(rec)[x];
    }
    float N0 = M0, N1 = M1;
#pragma unroll
    for (int u = 0; u < kMergeUnroll; ++u) {
      N0 = fmaxf(N0, m0[u]);
      N1 = fmaxf(N1, m1[u]);
    }
    // what is summed so far is 0 while the max is still -inf
    const float r0 = (M0 == -INFINITY) ? 0.f : exp2f(M0 - N0);
    const float r1 = (M1 == -INFINITY) ? 0.f : exp2f(M1 - N1);
    L0 *= r0;
    L1 *= r1;
    acc.x *= r0;
    acc.y *= r0;
    acc.z *= r1;
    acc.w *= r1;
    M0 = N0;
    M1 = N1;
#pragma unroll
    for (int u = 0; u < kMergeUnroll; ++u) {
      // a run with no valid entry has max -inf, sum 0 and O 0: weight 0
      const float w0 = (m0[u] == -INFINITY) ? 0.f : exp2f(m0[u] - M0);
      const float w1 = (m1[u] == -INFINITY) ? 0.f : exp2f(m1[u] - M1);
      L0 = fmaf(l0[u], w0, L0);
      L1 = fmaf(l1[u], w1, L1);
      acc.x = fmaf(v[u].x, w0, acc.x);
      acc.y = fmaf(v[u].y, w0, acc.y);
      acc.z = fmaf(v[u].z, w1, acc.z);
      acc.w = fmaf(v[u].w, w1, acc.w);
    }
  }
  // element c: head h0 + 8 (c >> 1), dim 8 (2 tig + (c & 1) + 8 (j >> 3)) + (j & 7);
  // within the quarter (dims 64 (qy >> 1) + 8 col + 4 (qy & 1) + e, e = j & 3): the
  // column 4 col + e of so
  const int e = j & 3;
  so[lq][h0][4 * (2 * tig) + e] = L0 > 0.f ? acc.x / L0 : 0.f;
  so[lq][h0][4 * (2 * tig + 1) + e] = L0 > 0.f ? acc.y / L0 : 0.f;
  so[lq][h0 + 8][4 * (2 * tig) + e] = L1 > 0.f ? acc.z / L1 : 0.f;
  so[lq][h0 + 8][4 * (2 * tig + 1) + e] = L1 > 0.f ? acc.w / L1 : 0.f;
  __syncthreads();
  const int r = threadIdx.x & (kMergeQuarter - 1), hh = r >> 3, col = r & 7;
  const int d = 64 * (qy >> 1) + 8 * col + 4 * (qy & 1);
  *reinterpret_cast<float4*>(out + t * kFrag + hh * kHeadDim + d) =
      *reinterpret_cast<const float4*>(&so[lq][hh][4 * col]);
}

// Grid of the split kernel: one CTA per SM, fewer when the warps would get fewer
// than kMinWarpTiles tiles each (a run's partial record costs a 8 KB write and
// read, worth it only over a few tiles).
constexpr int kMinWarpTiles = 4;
static int64_t decode_grid(int64_t U, int num_sms) {
  const int64_t want = U / (kDecWarps * kMinWarpTiles);
  return std::max<int64_t>(1, std::min<int64_t>(want, num_sms > 0 ? num_sms : 1));
}

size_t decode_workspace_bytes(int64_t T, int kw, int num_sms) {
  if (T <= 0 || kw < 1) return 0;
  const int64_t NT = (kw + kTile - 1) / kTile;
  const int64_t NW = decode_grid(T * NT, num_sms) * kDecWarps;
  return (size_t)(NW + T) * kRecFloats * sizeof(float);
}

cudaError_t launch_decode(const uint16_t* q, int64_t T, int Q, const uint8_t* k_pages,
                          const uint8_t* v_pages, int64_t kv_page_stride, int64_t num_pages,
                          const int32_t* block_table, int64_t bt_width, const int32_t* seq_lens,
                          const int32_t* topk, int kw, float scale, float* out, void* ws,
                          uint32_t* status, int num_sms, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  DecodeArgs a;
  a.q = q;
  a.k_pages = k_pages;
  a.v_pages = v_pages;
  a.kv_page_stride = kv_page_stride;
  a.num_pages = num_pages;
  a.block_table = block_table;
  a.bt_width = bt_width;
  a.seq_lens = seq_lens;
  a.topk = topk;
  a.ws = static_cast<float*>(ws);
  a.status = status;
  a.NT = (kw + kTile - 1) / kTile;
  a.U = T * a.NT;
  a.kw = kw;
  a.Q = Q;
  a.scale = scale;
  const int64_t G = decode_grid(a.U, num_sms);
  const int smem = (int)sizeof(DecodeSmem);
  cudaError_t err =
      cudaFuncSetAttribute(decode_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  err = launch_pdl(decode_split_kernel, dim3((unsigned)G), dim3(kDecThreads), smem, stream, a);
  if (err != cudaSuccess) return err;
  if (G * kDecWarps > (int64_t)kMergeSplitRuns * T)
    return launch_pdl(decode_merge_kernel<4>, dim3((unsigned)T, 4), dim3(kMergeQuarter), 0, stream,
                      (const float*)a.ws, a.U, G * kDecWarps, a.NT, out);
  return launch_pdl(decode_merge_kernel<1>, dim3((unsigned)T, 1), dim3(4 * kMergeQuarter), 0,
                    stream,
                    (const float*)a.ws, a.U, G * kDecWarps, a.NT, out);
}

}  // namespace mx4
