/*
 * mx4sp.h -- C ABI of the GB300 (sm_103a) library for sparse-attention decode
 * over an MXFP4 paged KV cache.
 *
 * The cache format is the one described on "vllm.models.minimax_m3.amd.ops.
 * mxfp4_pages" (module description and mxfp4_page_views): one page holds 128
 * token rows of one head as
 *
 *     [128 tokens x 64 B e2m1 data][128 tokens x 4 B e8m0 scale] = 8704 B
 *
 * two elements a byte (the low nibble is the even element), one e8m0 scale per
 * 32 consecutive elements, no global scale.  A page tensor is
 * [pages, heads, 8704] for K and V and [pages, 8704] for the index key, with
 * arbitrary page/head strides and a contiguous byte axis.  K/V and the index
 * key are written through one page-128 slot mapping and read through one
 * block table ("vllm.models.minimax_m3.amd.mono.dispatch", _slots_shared,
 * _step_refusal).
 *
 * Conventions shared by every entry point
 *   - All pointers to tensors are DEVICE pointers on the current CUDA device,
 *     except where stated.  The caller owns every buffer, workspaces included;
 *     no call allocates, frees or synchronises (mx4_check_status excepted), so
 *     every call can be recorded into a CUDA graph.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     All work is enqueued on it, asynchronously.
 *   - bf16 tensors are passed as uint16_t bit patterns.
 *   - Return value: MX4_OK, or a negative mx4_status.  On error nothing has been
 *     enqueued and mx4_last_error() returns the reason (thread-local).  Argument
 *     checks that need device data (block-table entries, slots, sequence lengths,
 *     top-k indices) are done by the kernels: a bad entry is skipped, its output
 *     is left as described per call, and a bit is set in a device status word
 *     that mx4_check_status() reads and clears.
 *   - Page pointers must be 16-byte aligned and page/head strides multiples of
 *     16 bytes; fp32/bf16 row tensors must be contiguous and 16-byte aligned.
 *   - Sequence s of a batch holds seq_lens[s] cached tokens; its q decode tokens
 *     are t = s*q + j (j = 0..q-1) at positions seq_lens[s] - q + j, and token j
 *     attends to cached positions 0 .. seq_lens[s] - q + j.
 */
#ifndef MX4SP_H
#define MX4SP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MX4_OK = 0,
    MX4_ERR_INVALID = -1,     /* a NULL pointer, a negative size, a misaligned buffer */
    MX4_ERR_UNSUPPORTED = -2, /* a geometry this library does not implement */
    MX4_ERR_WORKSPACE = -3,   /* workspace too small */
    MX4_ERR_CUDA = -4,        /* a CUDA runtime error (launch or copy) */
    MX4_ERR_BOUNDS = -5       /* reported by mx4_check_status: a kernel skipped bad data */
} mx4_status;

/* Bits of the device status word (mx4_check_status). */
#define MX4_STATUS_BAD_SLOT 0x1u   /* slot >= num_pages * 128 */
#define MX4_STATUS_BAD_PAGE 0x2u   /* block-table entry outside [0, num_pages) */
#define MX4_STATUS_BAD_LEN 0x4u    /* seq_len < q, or beyond the block table / ld */
#define MX4_STATUS_BAD_INDEX 0x8u  /* top-k index outside [0, position] */
#define MX4_STATUS_BAD_VALUE 0x10u /* non-finite fp32 input to mx4_insert */
#define MX4_STATUS_TIMEOUT 0x20u   /* a kernel gave up a bounded wait (should not happen) */

#define MX4_PAGE_TOKENS 128
#define MX4_HEAD_DIM 128
#define MX4_PAGE_BYTES 8704
#define MX4_FP8_PAGE_BYTES 16384 /* fp8 index-K cache page: 128 rows x 128 E4M3 bytes */

/* Reason for the last non-OK return on this thread ("" if none). */
const char *mx4_last_error(void);

/* Bytes of one page of one head: 8704. */
size_t mx4_page_bytes(void);

/* ---------------------------------------------------------------------------
 * mx4_insert -- quantise-on-insert (page description of "mxfp4_pages"; slot
 * mapping of _slots_shared).
 *
 * For each new token t with slot = slot_mapping[t] >= 0, quantise its K row (per
 * KV head), V row (per KV head) and index-K row, 128 fp32 values each, into
 * MXFP4 and write them to row slot % 128 of page slot / 128 of k_pages, v_pages
 * and idx_pages.  Each 32-element block gets the shared exponent
 * E = floor(log2(amax)) - 2 clamped to [-127, 127] (-127 when amax == 0), scale
 * byte E + 127, and every element the E2M1 code of x / 2^E rounded to nearest,
 * ties to even, saturating at 6, with the sign of x (OCP MX v1.0 conversion).
 *
 *   k, v         fp32 [T, Hkv, 128], contiguous
 *   idx_k        fp32 [T, 128], contiguous
 *   slot_mapping int64 [T]; a negative slot skips the token
 *   k_pages, v_pages  uint8, page p head h at base + p*kv_page_stride
 *                     + h*kv_head_stride (bytes); written in place
 *   idx_pages    uint8, page p at base + p*idx_page_stride; written in place
 *   num_pages    pages in each pool (slots must be < num_pages * 128)
 * Bad slot: the token is skipped and MX4_STATUS_BAD_SLOT is set.  Non-finite
 * inputs are out of contract: their bytes are unspecified and
 * MX4_STATUS_BAD_VALUE is set.  1 <= Hkv <= 8.
 * ------------------------------------------------------------------------- */
int mx4_insert(const float *k, const float *v, const float *idx_k, int64_t T, int Hkv,
               const int64_t *slot_mapping, uint8_t *k_pages, uint8_t *v_pages,
               int64_t kv_page_stride, int64_t kv_head_stride, uint8_t *idx_pages,
               int64_t idx_page_stride, int64_t num_pages, void *stream);

/* ---------------------------------------------------------------------------
 * mx4_norm_rope_insert -- the writer in front of mx4_insert: norm and rotary
 * embedding of the new token's heads, then the MXFP4 insert ("vllm.models.
 * minimax_m3.amd.mono.weights", SparseMoeLayer: g_q, g_k, g_iq, g_ik, cos_sin;
 * the formula is not printed -- the plainest reading is taken).
 *
 * For token t at position pos = positions[t], every q head, the index-q head,
 * every K head and the index-K head row x (128 fp32) becomes
 *     z = x * g / sqrt(mean(x^2) + eps),
 *     y[i] = z[i] c[i] - z[i+64] s[i],  y[i+64] = z[i+64] c[i] + z[i] s[i]  (i < 64)
 * with c[i] = cos_sin[pos*128 + i], s[i] = cos_sin[pos*128 + 64 + i] and g the
 * head kind's weight.  q and index-q are written as bf16 (round to nearest
 * even) to q_out and iq_out.  K and index-K are quantised like mx4_insert into
 * their page rows, and so is V, unchanged.  Computed in fp32.
 *
 *   q            fp32 [T, H, 128];  iq fp32 [T, 128]
 *   k, v         fp32 [T, Hkv, 128]; idx_k fp32 [T, 128]   (all contiguous)
 *   positions    int64 [T]; cos_sin fp32 [max_pos, 128]
 *   g_q, g_k, g_iq, g_ik  fp32 [128]; eps >= 0
 *   slot_mapping, pages   as mx4_insert
 *   q_out        bf16 [T, H, 128]; iq_out bf16 [T, 128]  (outputs)
 * fp32 arrays 16-byte aligned, q_out / iq_out 8-byte aligned.  A position
 * outside [0, max_pos) skips every row of that token and sets
 * MX4_STATUS_BAD_INDEX.  Slots behave as in mx4_insert; a negative slot skips
 * only the token's page rows (its q_out and iq_out rows are still written).
 * Non-finite values set MX4_STATUS_BAD_VALUE when they reach a page row.
 * 1 <= H <= 64, 1 <= Hkv <= 8.
 * ------------------------------------------------------------------------- */
int mx4_norm_rope_insert(const float *q, const float *iq, const float *k, const float *v,
                         const float *idx_k, int64_t T, int H, int Hkv, const int64_t *positions,
                         const float *cos_sin, int64_t max_pos, const float *g_q,
                         const float *g_k, const float *g_iq, const float *g_ik, float eps,
                         const int64_t *slot_mapping, uint8_t *k_pages, uint8_t *v_pages,
                         int64_t kv_page_stride, int64_t kv_head_stride, uint8_t *idx_pages,
                         int64_t idx_page_stride, int64_t num_pages, uint16_t *q_out,
                         uint16_t *iq_out, void *stream);

/* ---------------------------------------------------------------------------
 * index_score -- the index scorer (the scorers that read [pages, 128, 64] /
 * [pages, 128, 4] index-key views, "mxfp4_pages" / mxfp4_page_views).
 *
 * For decode token t = s*q + j at position p = seq_lens[s] - q + j:
 *     scores[t*ld_scores + i] = sum_d iq[t][d] * dequant(indexK[s, i])[d]
 * for 0 <= i <= p, computed in fp32, and -inf for p < i < seq_lens[s]; entries
 * at i >= seq_lens[s] are not written.  dequant = e2m1 value x 2^(scale - 127).
 * Token i of sequence s is row i % 128 of page block_table[s*bt_width + i/128].
 * The q decode tokens of a sequence share one pass over its pages.
 *
 *   iq          bf16 [T, 128] with T = B * q_per_seq, contiguous
 *   idx_pages   uint8 [num_pages, 8704] at stride idx_page_stride
 *   block_table int32 [B, bt_width], row-contiguous
 *   seq_lens    int32 [B]
 *   scores      fp32 [T, ld_scores]
 * 1 <= q_per_seq <= 8, B <= 65535.  A sequence with seq_len < q, seq_len >
 * bt_width*128 or seq_len > ld_scores is skipped (MX4_STATUS_BAD_LEN); a page
 * id outside [0, num_pages) skips that page (MX4_STATUS_BAD_PAGE).
 * ------------------------------------------------------------------------- */
int index_score(const uint16_t *iq, int64_t T, int q_per_seq, const uint8_t *idx_pages,
                int64_t idx_page_stride, int64_t num_pages, const int32_t *block_table,
                int64_t B, int64_t bt_width, const int32_t *seq_lens, float *scores,
                int64_t ld_scores, void *stream);

/* ---------------------------------------------------------------------------
 * index_score_mxq -- the index scorer in block-scaled mode: the MXFP4 keys are
 * the A operand of a block-scaled tensor-core product as stored (e2m1 codes,
 * e8m0 scale per 32 dims), and each index-q row is first converted to MXFP8,
 * the other MX operand format of the pages' scaled matrix core ("vllm.models.
 * minimax_m3.amd.mono.weights", module description and mxfp8_a_tiles: the
 * f8f6f4 MFMA with e8m0 scales).  Per 32-dim block b of iq[t]:
 *     E_b = floor(log2 max|x|) - 8, clamped to [-127, 127] (-127 for a zero block)
 *     code = E4M3(x * 2^-E_b), nearest, ties to even, saturating at 448
 * and then
 *     scores[t*ld_scores + i] = sum_b 2^E_b * sum_{d in b} E4M3value(code_d) * dequant(indexK[s, i])[d]
 * for 0 <= i <= p, accumulated in fp32 by the tensor core; -inf and unwritten
 * entries as index_score.  Arguments, layouts, limits, ownership and status
 * bits are those of index_score, except that idx_pages must be 32-byte aligned
 * and idx_page_stride a multiple of 32 (MX4_ERR_INVALID otherwise: the pages are
 * read by tensor copies of the pool).  An opt-in mode: it differs from index_score
 * by the query's MXFP8 rounding (a relative error of at most 2^-4 per element).
 * ------------------------------------------------------------------------- */
int index_score_mxq(const uint16_t *iq, int64_t T, int q_per_seq, const uint8_t *idx_pages,
                    int64_t idx_page_stride, int64_t num_pages, const int32_t *block_table,
                    int64_t B, int64_t bt_width, const int32_t *seq_lens, float *scores,
                    int64_t ld_scores, void *stream);

/* ---------------------------------------------------------------------------
 * topk_select -- per-token top-k selection of the tokens to attend.
 *
 * For decode token t with n = p + 1 valid scores (p as above): the min(k, n)
 * indices i in [0, n) with the largest scores[t*ld_scores + i], ties broken
 * towards the lower index (the order is: larger score first, then lower index;
 * -0.0 and +0.0 are equal), written in ascending index order to
 * topk_idx[t*k ...]; the remaining entries up to k are -1.
 *
 *   scores   fp32 [T, ld_scores], T = B * q_per_seq; must be finite on [0, n)
 *   seq_lens int32 [B]
 *   topk_idx int32 [T, k] (output)
 *   ws       workspace of topk_select_workspace(T, k, ld_scores) bytes (may be
 *            NULL when that is 0)
 * 1 <= k <= 65536, 1 <= q_per_seq <= 8.  A bad seq_len (n < 1 or n > ld_scores)
 * writes a row of -1 and sets MX4_STATUS_BAD_LEN.
 * ------------------------------------------------------------------------- */
int topk_select(const float *scores, int64_t ld_scores, const int32_t *seq_lens, int64_t B,
                int q_per_seq, int k, int32_t *topk_idx, void *ws, size_t ws_bytes,
                void *stream);
size_t topk_select_workspace(int64_t T, int k, int64_t ld_scores);

/* ---------------------------------------------------------------------------
 * index_topk -- index_score and topk_select in one call, the scorer -> selection
 * chain in front of pa_decode ("mxfp4_pages", module description: the index
 * scorers and pa_decode read the same pages).
 *
 * Same arguments and results as index_score (scores, -inf past each token's
 * position) followed by topk_select (topk_idx [T, k], ascending, -1 padded, ties
 * to the lower index), with the same kernels: the scores stay in L2 between the
 * scorer and the selection (12 MB for 256 tokens of 11.6k cached tokens on
 * average, against a 129 MB L2), and the caller makes one call and provides one
 * workspace.
 *
 *   ws   workspace of index_topk_workspace(T, k, ld_scores) bytes (the same as
 *        topk_select_workspace), 16-byte aligned
 * Limits and status bits as index_score and topk_select (B <= 65535,
 * T <= 65535, 1 <= q_per_seq <= 8, 1 <= k <= 65536, ld_scores <= 8388608).
 * ------------------------------------------------------------------------- */
int index_topk(const uint16_t *iq, int64_t T, int q_per_seq, const uint8_t *idx_pages,
               int64_t idx_page_stride, int64_t num_pages, const int32_t *block_table,
               int64_t B, int64_t bt_width, const int32_t *seq_lens, float *scores,
               int64_t ld_scores, int k, int32_t *topk_idx, void *ws, size_t ws_bytes,
               void *stream);
size_t index_topk_workspace(int64_t T, int k, int64_t ld_scores);

/* ---------------------------------------------------------------------------
 * sparse_paged_decode -- GQA decode attention over the selected tokens (the
 * pa_decode reader of [pages, heads, 128, 64] / [pages, heads, 128, 4] K/V
 * views, "mxfp4_pages" / mxfp4_page_views), with a split-K merge.
 *
 * For decode token t of sequence s and query head h (KV head h / (H / Hkv)):
 *     l_i = scale * sum_d q[t][h][d] * dequant(K[s, i])[d],
 *     out[t][h][:] = sum_i softmax(l)_i * dequant(V[s, i])[:]
 * over the indices i of topk_idx[t*k ...] that are >= 0 (negative entries are
 * skipped, so the -1 padding of topk_select is ignored).
 * Logits and the softmax are fp32.  The selected lists are cut into runs of
 * entries, one run per warp of a persistent grid and token; each run keeps a
 * running max and sum (online softmax) and writes its partial result to the
 * workspace, and a merge kernel combines the runs of each token.
 *
 *   q         bf16 [T, H, 128], contiguous
 *   k_pages, v_pages  uint8 [num_pages, Hkv, 8704] at the given strides
 *   block_table int32 [B, bt_width]; seq_lens int32 [B]
 *   topk_idx  int32 [T, k], ascending indices then -1 padding
 *   out       fp32 [T, H, 128] (output)
 *   ws        workspace of sparse_paged_decode_workspace(T, k) bytes, 16-byte
 *             aligned; the size depends on the current device's SM count (the
 *             grid has one CTA per SM), so query it with that device current
 * H == 16 and Hkv == 1 in this library (else MX4_ERR_UNSUPPORTED).  An index
 * outside [0, p] or a bad page id skips that token and sets
 * MX4_STATUS_BAD_INDEX / MX4_STATUS_BAD_PAGE.  A token with no selected index
 * gets a zero output.
 * ------------------------------------------------------------------------- */
int sparse_paged_decode(const uint16_t *q, int64_t T, int q_per_seq, int H, int Hkv,
                        const uint8_t *k_pages, const uint8_t *v_pages, int64_t kv_page_stride,
                        int64_t kv_head_stride, int64_t num_pages, const int32_t *block_table,
                        int64_t B, int64_t bt_width, const int32_t *seq_lens,
                        const int32_t *topk_idx, int k, float scale, float *out, void *ws,
                        size_t ws_bytes, void *stream);
size_t sparse_paged_decode_workspace(int64_t T, int k);

/* ---------------------------------------------------------------------------
 * sparse_paged_decode_noalloc -- sparse_paged_decode without a caller
 * workspace.  The pages this library follows ("vllm.models.minimax_m3.amd.ops.
 * mxfp4_pages", "vllm.models.minimax_m3.amd.mono.dispatch") have no counterpart
 * for it: it exists for callers that cannot allocate device memory (a host
 * framework that owns all device memory and gives an extension only the
 * operation's inputs and outputs, or a C or foreign-language runtime with no
 * device allocator).  Same arguments, result and errors as
 * sparse_paged_decode, minus ws/ws_bytes.
 *
 * The run workspace lives in a fixed array inside the library of
 * MX4_NOALLOC_SCRATCH_BYTES (32 MiB) of device memory, which every GPU that
 * loads the library holds until the process exits.  A call whose workspace
 * (sparse_paged_decode_workspace(T, k)) exceeds it returns MX4_ERR_WORKSPACE
 * without launching.  The call allocates and frees nothing.  The first call on
 * a device looks up the array's device address (cudaGetSymbolAddress) with
 * that device current: make it before any stream capture.  All calls on a
 * device share the array, so calls that overlap on the GPU race; nothing in it
 * needs clearing between calls.  The looked-up address (like the device
 * address of the status word every call uses) is kept for the life of the
 * process: do not use the library across a cudaDeviceReset of that device.
 * ------------------------------------------------------------------------- */
#define MX4_NOALLOC_SCRATCH_BYTES (32u << 20)
int sparse_paged_decode_noalloc(const uint16_t *q, int64_t T, int q_per_seq, int H, int Hkv,
                                const uint8_t *k_pages, const uint8_t *v_pages,
                                int64_t kv_page_stride, int64_t kv_head_stride,
                                int64_t num_pages, const int32_t *block_table, int64_t B,
                                int64_t bt_width, const int32_t *seq_lens,
                                const int32_t *topk_idx, int k, float scale, float *out,
                                void *stream);

/* ---------------------------------------------------------------------------
 * The fp8 index-K cache variant ("vllm.models.minimax_m3.amd.mono.weights",
 * SparseMoeLayer.index_cache: [blocks, block, head_dim] fp8 with the block ids
 * of the K/V cache; "vllm.models.minimax_m3.amd.mono.dispatch",
 * _config_refusal: the index cache dtype is fp8).  A page holds 128 token rows
 * of 128 OCP E4M3 bytes (MX4_FP8_PAGE_BYTES), row r at byte r*128.  The layout
 * has no scale bytes: one fp32 scale S > 0 per cache is an argument.
 *
 * fp8_index_insert -- for each new token t with slot s = slot_mapping[t] >= 0,
 * byte d of row s%128 of page s/128 becomes E4M3(fl32(idx_k[t][d] / S)):
 * the IEEE fp32 quotient rounded to the nearest E4M3 value, ties to even,
 * magnitudes past 448 saturating to 448, the sign kept for a quotient that
 * rounds to zero.  Negative slots are skipped; a slot past the pool skips the
 * token (MX4_STATUS_BAD_SLOT); a non-finite input is written as the conversion
 * gives it and sets MX4_STATUS_BAD_VALUE.
 *
 *   idx_k         fp32 [T, 128], contiguous, 16-byte aligned
 *   slot_mapping  int64 [T]
 *   pages         uint8 [num_pages, 16384] at byte stride page_stride
 *                 (a multiple of 16, at least 16384), written in place
 *
 * index_score_fp8 -- index_score over the fp8 cache: for decode token
 * t = s*q + j at position p = seq_lens[s] - q + j,
 *     scores[t*ld_scores + i] = S * sum_d iq[t][d] * E4M3value(row i)[d]
 * for 0 <= i <= p, computed in fp32, -inf for p < i < seq_lens[s], entries at
 * i >= seq_lens[s] not written.  Arguments, limits and status bits as
 * index_score, with pages [num_pages, 16384] at page_stride.  An E4M3 NaN byte
 * (0x7F, 0xFF: the poison of a never-written row) gives a NaN score.
 * ------------------------------------------------------------------------- */
int fp8_index_insert(const float *idx_k, int64_t T, const int64_t *slot_mapping, float scale,
                     uint8_t *pages, int64_t page_stride, int64_t num_pages, void *stream);
int index_score_fp8(const uint16_t *iq, int64_t T, int q_per_seq, const uint8_t *pages,
                    int64_t page_stride, int64_t num_pages, const int32_t *block_table,
                    int64_t B, int64_t bt_width, const int32_t *seq_lens, float scale,
                    float *scores, int64_t ld_scores, void *stream);

/* ---------------------------------------------------------------------------
 * mx4_decode_step -- one whole decode step from host memory to host memory:
 * the step's inputs are copied from one packed host buffer to the device, the
 * new tokens' K/V/index-K rows are inserted (mx4_insert), the index keys are
 * scored and the top-k selected (index_topk), attention computed
 * (sparse_paged_decode), and the output copied back to host memory.  This is
 * the chain the scorer and pa_decode form over the same pages
 * ("vllm.models.minimax_m3.amd.ops.mxfp4_pages", module description), with the
 * insert through the shared slot mapping first ("vllm.models.minimax_m3.amd.
 * mono.dispatch", _slots_shared).
 *
 *   h_inputs   HOST buffer of mx4_decode_step_input_bytes(T, n_new) bytes laid
 *              out as mx4_decode_step_input_offsets gives: q bf16 [T, 16, 128],
 *              iq bf16 [T, 128], k_new fp32 [n_new, 128], v_new fp32
 *              [n_new, 128], idx_k_new fp32 [n_new, 128], slots int64 [n_new]
 *              (n_new = 0: no insert).  Page-locked memory makes the copy
 *              asynchronous; pageable memory works but the copy blocks the host.
 *   d_staging  DEVICE buffer of at least the same size (the copy's target)
 *   caches, tables, q_per_seq, k, scale: as the four calls above (H = 16,
 *              Hkv = 1); T = B * q_per_seq
 *   d_scores   fp32 [T, ld_scores]; d_topk_idx int32 [T, k]; d_out fp32
 *              [T, 16, 128] (device); topk_ws the index_topk workspace
 *              (index_topk_workspace(T, k, ld_scores) bytes; may be NULL when
 *              that is 0), dec_ws the sparse_paged_decode one
 *   h_out      HOST fp32 [T, 16, 128]: receives the step's attention output
 * Everything is enqueued on `stream` and the call returns without waiting:
 * h_out holds the result once the stream reaches this point (synchronise the
 * stream or record an event).  Errors as the four calls; the first failing
 * stage's status is returned and nothing after it is enqueued.
 * ------------------------------------------------------------------------- */
size_t mx4_decode_step_input_bytes(int64_t T, int64_t n_new);
/* offsets[0..5] = byte offsets of q, iq, k_new, v_new, idx_k_new, slots in the
 * packed input buffer (each a multiple of 256). */
void mx4_decode_step_input_offsets(int64_t T, int64_t n_new, size_t offsets[6]);
int mx4_decode_step(const void *h_inputs, int64_t n_new, void *d_staging, size_t staging_bytes,
                    uint8_t *k_pages, uint8_t *v_pages, int64_t kv_page_stride,
                    int64_t kv_head_stride, uint8_t *idx_pages, int64_t idx_page_stride,
                    int64_t num_pages, const int32_t *block_table, int64_t B, int64_t bt_width,
                    const int32_t *seq_lens, int q_per_seq, int k, float scale, float *d_scores,
                    int64_t ld_scores, int32_t *d_topk_idx, void *topk_ws, size_t topk_ws_bytes,
                    void *dec_ws, size_t dec_ws_bytes, float *d_out, float *h_out,
                    void *stream);

/* ---------------------------------------------------------------------------
 * mx4_decode_steps -- n_steps decode steps in order, host memory to host
 * memory, with the copies of neighbouring steps overlapping the compute: step
 * i's inputs go to the device on h2d_stream while step i-1 computes on
 * `stream`, and step i's output comes back on d2h_stream while step i+1
 * computes.  Each step is exactly mx4_decode_step (insert, index_topk,
 * sparse_paged_decode on the shared page caches, in step order, so every
 * step's insert lands before the next step reads the caches).
 *
 *   h_inputs   HOST packed inputs of step i at h_inputs + i * h_inputs_stride
 *              (stride 0: the same inputs every step); page-locked memory is
 *              needed for the copies to overlap
 *   d_staging  DEVICE, two input sets: set b at d_staging + b * S, S =
 *              mx4_decode_step_input_bytes(T, n_new) rounded up to 256;
 *              staging_bytes >= 2 * S, 256-byte aligned
 *   d_out      DEVICE fp32, two output sets [2][T, 16, 128]
 *   h_out      HOST fp32: step i's output [T, 16, 128] at byte offset
 *              i * h_out_stride (stride 0: every step into the same buffer, in
 *              step order)
 *   stream, h2d_stream, d2h_stream  the compute stream (may be the default
 *              stream) and two copy streams for the inputs and the outputs, of
 *              the caller: distinct, the copy streams not the default stream
 *   the rest   as mx4_decode_step (one set of scores, top-k indices and
 *              workspaces, reused by every step)
 * The copies start after the work already on `stream`, and `stream` waits for
 * the last copy at the end: once `stream` reaches this point every h_out
 * holds its step's result.  The call returns without waiting; it creates and
 * releases its own events.  Errors as mx4_decode_step, checked for both sets
 * before anything is enqueued; MX4_ERR_INVALID for missing or equal streams.
 * ------------------------------------------------------------------------- */
int mx4_decode_steps(int64_t n_steps, const void *h_inputs, size_t h_inputs_stride,
                     int64_t n_new, void *d_staging, size_t staging_bytes, uint8_t *k_pages,
                     uint8_t *v_pages, int64_t kv_page_stride, int64_t kv_head_stride,
                     uint8_t *idx_pages, int64_t idx_page_stride, int64_t num_pages,
                     const int32_t *block_table, int64_t B, int64_t bt_width,
                     const int32_t *seq_lens, int q_per_seq, int k, float scale, float *d_scores,
                     int64_t ld_scores, int32_t *d_topk_idx, void *topk_ws, size_t topk_ws_bytes,
                     void *dec_ws, size_t dec_ws_bytes, float *d_out, float *h_out,
                     size_t h_out_stride, void *stream, void *h2d_stream, void *d2h_stream);

/* ---------------------------------------------------------------------------
 * mx4_check_status -- synchronise `stream`, return MX4_OK if no kernel of this
 * library has flagged bad data on the current device since the last check,
 * else MX4_ERR_BOUNDS with the flagged MX4_STATUS_* bits in *bits (if bits is
 * not NULL) and in mx4_last_error().  Clears the word.  This is the only call
 * that synchronises.
 * ------------------------------------------------------------------------- */
int mx4_check_status(void *stream, uint32_t *bits);

#ifdef __cplusplus
}
#endif

#endif /* MX4SP_H */
