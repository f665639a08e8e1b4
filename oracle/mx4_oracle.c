/*
 * mx4_oracle.c -- the CPU oracle for sparse-attention decode over an MXFP4 paged
 * KV cache.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check and
 * the benchmark's CPU-baseline leg load this library.  The CUDA library neither
 * links nor calls it, and the two share no source, header, table or helper.
 *
 * Everything here is plain, slow and written to be checked by eye against its
 * definition: scalar loops, float64 arithmetic, no blocking, no fusion, no
 * reordering beyond the definition, no threads.
 *
 * Sources (cited by page title and section):
 *   [pages]  "vllm.models.minimax_m3.amd.ops.mxfp4_pages" -- module description
 *            (page geometry: [128 tokens x 64 B e2m1 data][128 tokens x 4 B e8m0
 *            scale] = 8704 B; two elements a byte, low nibble the even one; one
 *            scale per 32 elements; no global scale) and mxfp4_page_views (data
 *            view at byte 0 with rows 64 B apart, scale view at byte 128*64 with
 *            rows 4 B apart).
 *   [slots]  "vllm.models.minimax_m3.amd.mono.dispatch" -- _slots_shared (K/V and
 *            the index key are inserted through one page-128 slot mapping) and
 *            _step_refusal (int32 row-contiguous block_table and seq_lens, int64
 *            slot mapping, decode_query_len tokens per request).
 *   [heads]  "vllm.models.minimax_m3.amd.mono.weights" -- _build_cp_qkv (one
 *            rank's rows q(2048) | k(128) | v(128) | index_q(128) | index_k(128):
 *            16 query heads, one KV head, one index head, head_dim 128).
 *   [layer]  "vllm.models.minimax_m3.amd.mono.weights" -- SparseMoeLayer (the norm
 *            weights g_q, g_k, g_iq, g_ik and the rotary table cos_sin a layer's
 *            kernels read).
 *   [fp8]    "vllm.models.minimax_m3.amd.mono.weights" -- SparseMoeLayer (index_cache
 *            [blocks, block, head_dim] fp8, shared block ids) and
 *            "vllm.models.minimax_m3.amd.mono.dispatch" -- _config_refusal (the
 *            index cache dtype must be fp8): the other revision's index-K cache.
 *   [OCP]    OCP Microscaling Formats (MX) v1.0 -- the FP4 E2M1 element type
 *            (1 sign, 2 exponent bits with bias 1, 1 mantissa bit, no inf/NaN),
 *            the E8M0 scale type (2^(byte-127), 0xFF = NaN) and the conversion of
 *            a 32-element block: shared exponent floor(log2(amax)) - emax_elem
 *            with emax_elem = 2 for E2M1, elements rounded to nearest, ties to
 *            even, saturating at the largest normal; and the FP8 E4M3 element
 *            type (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no
 *            inf, S.1111.111 = NaN, largest normal 448).
 *
 * Readings taken where the pages are silent:
 *   R1  scale b of a row covers the contiguous elements 32b .. 32b+31;
 *   R2  amax == 0 gives shared exponent -127 (scale byte 0x00);
 *   R3  the exponent is clamped to [-127, 127];
 *   R4  the element code keeps the sign of x even when the magnitude rounds to
 *       zero (x < 0 -> code 0x8);
 *   R6  a negative slot means "do not insert this token";
 *   R7  token j (0-based) of a sequence with q decode tokens sits at position
 *       seq_len - q + j and sees cached tokens 0 .. that position;
 *   R8  the index score is the plain dot product of the index-q head with the
 *       dequantised index key (no weight, no activation, no scale);
 *   R9  top-k ties go to the lower token index; the selected indices are
 *       returned in ascending order, padded with -1;
 *   R10 attention is softmax(scale * q.K) V over the selected tokens only.
 *   R14 the writer in front of the insert ([layer] SparseMoeLayer: g_q, g_k,
 *       g_iq, g_ik, cos_sin; no formula printed): each q, k, index-q and
 *       index-k head row is RMS-normed over its 128 dims (mean of squares plus
 *       eps, times the weight g) and then rotated: dims i and i+64 (i < 64) are
 *       a pair turned by the angle whose cosine and sine are cos_sin[pos][i]
 *       and cos_sin[pos][64+i]; V is neither normed nor rotated.
 *   R15 the fp8 of the [fp8] index cache is OCP E4M3 (the MX element type of
 *       the same pages' MXFP8 weights), one byte per element, a token row 128 B
 *       and a page of 128 rows 16384 B;
 *   R16 that layout has no room for scales, so one fp32 scale S > 0 per cache
 *       is an argument: the stored code is E4M3(fl32(x / S)), rounded to
 *       nearest, ties to even, saturating at 448; the element reads back as
 *       E4M3 value times S.
 *   R17 the block-scaled score mode (an MX operand format for the query, as a
 *       block-scaled tensor-core product needs): the bf16 index-q row is
 *       converted to MXFP8 per [OCP] -- per 32-element block, shared exponent
 *       floor(log2(amax)) - 8 (8 = the largest E4M3 exponent), clamped to
 *       [-127, 127], -127 for amax == 0; elements x * 2^-E to E4M3, nearest,
 *       ties to even, saturating at 448 -- and dotted with the dequantised key.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_PAGE_TOKENS 128
#define ORC_ROW_ELEMS 128
#define ORC_DATA_BYTES 64   /* per token row: 128 elements, two a byte  [pages] */
#define ORC_SCALE_BYTES 4   /* per token row: one e8m0 per 32 elements  [pages] */
#define ORC_PAGE_BYTES (ORC_PAGE_TOKENS * (ORC_DATA_BYTES + ORC_SCALE_BYTES))
#define ORC_BLOCK 32

enum { ORC_OK = 0, ORC_ERR_INVALID = -1, ORC_ERR_BOUNDS = -5 };

int orc_page_bytes(void) { return ORC_PAGE_BYTES; }

/* ------------------------------------------------------------------------- */
/* Element and scale types  [OCP]                                             */
/* ------------------------------------------------------------------------- */

/* Value of a 4-bit E2M1 code: bit 3 sign, bits 2..1 exponent (bias 1), bit 0
 * mantissa.  Exponent field 0 is subnormal: 0.m * 2^(1-1).  Otherwise
 * 1.m * 2^(e-1). */
double orc_e2m1_value(int code)
{
    int sign = (code >> 3) & 1;
    int e = (code >> 1) & 3;
    int m = code & 1;
    double mag;
    if (e == 0)
        mag = (m ? 0.5 : 0.0);
    else
        mag = ldexp(1.0 + 0.5 * m, e - 1);
    return sign ? -mag : mag;
}

/* Value of an E8M0 scale byte: 2^(byte-127); 0xFF is NaN. */
double orc_e8m0_value(int byte)
{
    if (byte == 255) return NAN;
    return ldexp(1.0, byte - 127);
}

/* ------------------------------------------------------------------------- */
/* Quantisation of one 32-element block  [OCP], readings R2-R4               */
/* ------------------------------------------------------------------------- */

/* Shared exponent E of a block with largest magnitude amax:
 * floor(log2(amax)) - 2, clamped to [-127, 127]; -127 for amax == 0.
 * floor(log2) is taken exactly with frexp (amax = f * 2^e, 0.5 <= f < 1). */
int orc_block_exponent(double amax)
{
    int e, E;
    if (amax == 0.0) return -127;
    (void)frexp(amax, &e);
    E = (e - 1) - 2;
    if (E < -127) E = -127;
    if (E > 127) E = 127;
    return E;
}

/* Nearest E2M1 magnitude code (0..7) to |y|; on a tie, the code whose
 * mantissa bit (bit 0) is 0.  Brute force over the eight magnitudes. */
int orc_e2m1_round_magnitude(double ay)
{
    int c, best = 0;
    double best_d = fabs(ay - orc_e2m1_value(0));
    for (c = 1; c < 8; ++c) {
        double d = fabs(ay - orc_e2m1_value(c));
        if (d < best_d || (d == best_d && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_d = d;
        }
    }
    return best;
}

/* Quantise x[0..31] (finite) to 32 E2M1 codes and one E8M0 scale byte.
 * Returns ORC_ERR_INVALID on a non-finite input. */
int orc_quantize_block(const float *x, uint8_t *codes, uint8_t *scale_byte)
{
    double amax = 0.0;
    int i, E;
    for (i = 0; i < ORC_BLOCK; ++i) {
        if (!isfinite(x[i])) return ORC_ERR_INVALID;
        if (fabs((double)x[i]) > amax) amax = fabs((double)x[i]);
    }
    E = orc_block_exponent(amax);
    *scale_byte = (uint8_t)(E + 127);
    for (i = 0; i < ORC_BLOCK; ++i) {
        double y = ldexp((double)x[i], -E); /* exact: a power-of-two scaling */
        int mag = orc_e2m1_round_magnitude(fabs(y));
        int sign = signbit(x[i]) ? 1 : 0;
        codes[i] = (uint8_t)((sign << 3) | mag);
    }
    return ORC_OK;
}

/* Quantise one 128-element row into its 64 data bytes and 4 scale bytes.
 * Element 2n goes to the low nibble of byte n, element 2n+1 to the high
 * nibble [pages]; scale b covers elements 32b..32b+31 (R1). */
int orc_quantize_row(const float *x, uint8_t *data, uint8_t *scale)
{
    uint8_t codes[ORC_ROW_ELEMS];
    int b, n, rc;
    for (b = 0; b < ORC_ROW_ELEMS / ORC_BLOCK; ++b) {
        rc = orc_quantize_block(x + b * ORC_BLOCK, codes + b * ORC_BLOCK, &scale[b]);
        if (rc) return rc;
    }
    for (n = 0; n < ORC_DATA_BYTES; ++n)
        data[n] = (uint8_t)(codes[2 * n] | (codes[2 * n + 1] << 4));
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* Page addressing and dequantisation  [pages]                               */
/* ------------------------------------------------------------------------- */

/* Data bytes of token row `row` of a page start at row*64; its scale bytes at
 * 128*64 + row*4 (the offsets of the data and scale views). */
static const uint8_t *row_data(const uint8_t *page, int row)
{
    return page + (size_t)row * ORC_DATA_BYTES;
}
static const uint8_t *row_scale(const uint8_t *page, int row)
{
    return page + (size_t)ORC_PAGE_TOKENS * ORC_DATA_BYTES + (size_t)row * ORC_SCALE_BYTES;
}

/* Element j of token row `row` of one page, dequantised. */
double orc_dequant_element(const uint8_t *page, int row, int j)
{
    uint8_t byte = row_data(page, row)[j / 2];
    int code = (j % 2 == 0) ? (byte & 0xF) : (byte >> 4);
    int sb = row_scale(page, row)[j / ORC_BLOCK];
    return orc_e2m1_value(code) * orc_e8m0_value(sb);
}

void orc_dequant_row(const uint8_t *page, int row, double *out)
{
    int j;
    for (j = 0; j < ORC_ROW_ELEMS; ++j) out[j] = orc_dequant_element(page, row, j);
}

/* ------------------------------------------------------------------------- */
/* a1: quantise-on-insert through the shared page-128 slot mapping  [slots]  */
/* ------------------------------------------------------------------------- */

static int write_row(uint8_t *page, int row, const float *x)
{
    return orc_quantize_row(x, page + (size_t)row * ORC_DATA_BYTES,
                            page + (size_t)ORC_PAGE_TOKENS * ORC_DATA_BYTES +
                                (size_t)row * ORC_SCALE_BYTES);
}

/* For each new token t with slot s = slot_mapping[t] >= 0: page s/128, row
 * s%128 of the K pages (every KV head h), the V pages and the index-K pages.
 * k, v: [T, Hkv, 128] fp32; idx_k: [T, 128] fp32.  Page tensors are addressed
 * as base + page*page_stride (+ h*head_stride) bytes.  Any of the three caches
 * may be skipped by passing its rows pointer as NULL. */
int orc_mx4_insert(const float *k, const float *v, const float *idx_k, int64_t T, int Hkv,
                   const int64_t *slot_mapping, uint8_t *k_pages, uint8_t *v_pages,
                   int64_t kv_page_stride, int64_t kv_head_stride, uint8_t *idx_pages,
                   int64_t idx_page_stride, int64_t num_pages)
{
    int64_t t;
    int h, rc;
    for (t = 0; t < T; ++t) {
        int64_t s = slot_mapping[t], page;
        int row;
        if (s < 0) continue;                                  /* R6 */
        page = s / ORC_PAGE_TOKENS;
        row = (int)(s % ORC_PAGE_TOKENS);
        if (page >= num_pages) return ORC_ERR_BOUNDS;
        for (h = 0; h < Hkv; ++h) {
            if (k) {
                rc = write_row(k_pages + page * kv_page_stride + h * kv_head_stride, row,
                               k + ((size_t)t * Hkv + h) * ORC_ROW_ELEMS);
                if (rc) return rc;
            }
            if (v) {
                rc = write_row(v_pages + page * kv_page_stride + h * kv_head_stride, row,
                               v + ((size_t)t * Hkv + h) * ORC_ROW_ELEMS);
                if (rc) return rc;
            }
        }
        if (idx_k) {
            rc = write_row(idx_pages + page * idx_page_stride, row,
                           idx_k + (size_t)t * ORC_ROW_ELEMS);
            if (rc) return rc;
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* Logical token -> physical page row through the block table  [slots]       */
/* ------------------------------------------------------------------------- */

/* Physical page of logical token i of sequence s; -1 when out of bounds. */
static int64_t page_of(const int32_t *block_table, int64_t bt_width, int64_t s, int64_t i,
                       int64_t num_pages)
{
    int64_t slot = i / ORC_PAGE_TOKENS, p;
    if (slot >= bt_width) return -1;
    p = block_table[s * bt_width + slot];
    if (p < 0 || p >= num_pages) return -1;
    return p;
}

static double bf16_to_double(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------------- */
/* a2: index scores, readings R7, R8                                          */
/* ------------------------------------------------------------------------- */

/* For decode token t = s*q + j (position p = seq_len[s] - q + j):
 *   score[t][i] = sum_j iq[t][j] * dequant(idxK[i][j])   for 0 <= i <= p,
 *   score[t][i] = -inf                                    for p < i < ld.
 * iq is bf16 bits [T, 128].  If `mag` is not NULL it receives
 * sum_j |iq[t][j] * dequant(idxK[i][j])| (for error bounds of other
 * implementations), with 0 outside 0..p. */
int orc_index_score(const uint16_t *iq, int64_t B, int q, const uint8_t *idx_pages,
                    int64_t idx_page_stride, int64_t num_pages, const int32_t *block_table,
                    int64_t bt_width, const int32_t *seq_lens, double *scores, double *mag,
                    int64_t ld)
{
    int64_t s, i;
    int j, d;
    for (s = 0; s < B; ++s) {
        int64_t L = seq_lens[s];
        if (L < q || L > ld || L > bt_width * ORC_PAGE_TOKENS) return ORC_ERR_BOUNDS;
        for (j = 0; j < q; ++j) {
            int64_t t = s * q + j;
            int64_t p = L - q + j;
            const uint16_t *qt = iq + t * ORC_ROW_ELEMS;
            for (i = 0; i < ld; ++i) {
                double acc = 0.0, acc_abs = 0.0;
                int64_t pg;
                const uint8_t *page;
                if (i > p) {
                    scores[t * ld + i] = -INFINITY;
                    if (mag) mag[t * ld + i] = 0.0;
                    continue;
                }
                pg = page_of(block_table, bt_width, s, i, num_pages);
                if (pg < 0) return ORC_ERR_BOUNDS;
                page = idx_pages + pg * idx_page_stride;
                for (d = 0; d < ORC_ROW_ELEMS; ++d) {
                    double term = bf16_to_double(qt[d]) *
                                  orc_dequant_element(page, (int)(i % ORC_PAGE_TOKENS), d);
                    acc += term;
                    acc_abs += fabs(term);
                }
                scores[t * ld + i] = acc;
                if (mag) mag[t * ld + i] = acc_abs;
            }
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* a3: top-k selection, reading R9                                            */
/* ------------------------------------------------------------------------- */

/* One candidate of the selection: its score and its token index. */
struct orc_cand {
    double score;
    int64_t index;
};

/* Order for qsort: larger score first, then lower index (R9).  The order is
 * total, so the result does not depend on the sort's stability. */
static int cand_order(const void *pa, const void *pb)
{
    const struct orc_cand *a = (const struct orc_cand *)pa;
    const struct orc_cand *b = (const struct orc_cand *)pb;
    if (a->score != b->score) return (a->score > b->score) ? -1 : 1;
    return (a->index < b->index) ? -1 : (a->index > b->index);
}

static int index_order(const void *pa, const void *pb)
{
    int32_t a = *(const int32_t *)pa, b = *(const int32_t *)pb;
    return (a > b) - (a < b);
}

/* For each decode token t with n = p + 1 valid scores: sort the candidates
 * by (score descending, index ascending), keep the first min(k, n), write
 * their indices in ascending order to out[t][0..], and -1 in the rest of
 * out[t][0..k). */
int orc_topk_select(const double *scores, int64_t ld, const int32_t *seq_lens, int64_t B, int q,
                    int k, int32_t *out)
{
    int64_t s, i;
    int j;
    struct orc_cand *c = (struct orc_cand *)malloc((size_t)ld * sizeof *c);
    if (!c) return ORC_ERR_INVALID;
    for (s = 0; s < B; ++s) {
        for (j = 0; j < q; ++j) {
            int64_t t = s * q + j;
            int64_t n = (int64_t)seq_lens[s] - q + j + 1;
            int64_t kk = (n < k) ? n : k, w;
            int32_t *o = out + t * k;
            if (n < 1 || n > ld) {
                free(c);
                return ORC_ERR_BOUNDS;
            }
            for (i = 0; i < n; ++i) {
                c[i].score = scores[t * ld + i];
                c[i].index = i;
            }
            qsort(c, (size_t)n, sizeof *c, cand_order);
            for (w = 0; w < kk; ++w) o[w] = (int32_t)c[w].index;
            qsort(o, (size_t)kk, sizeof *o, index_order);
            for (; w < k; ++w) o[w] = -1;
        }
    }
    free(c);
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* a4: GQA attention over the selected tokens, reading R10                    */
/* ------------------------------------------------------------------------- */

/* For decode token t of sequence s and query head h (KV head h / (H/Hkv)):
 *   l_i = scale * sum_d q[t][h][d] * K_i[d]      over i in the selected set,
 *   out[t][h][:] = sum_i softmax(l)_i * V_i[:].
 * q is bf16 bits [T, H, 128]; out is float64 [T, H, 128]; topk is int32
 * [T, kw], -1 entries ignored.  K/V pages are [pages, Hkv, 8704] at
 * base + page*page_stride + h*head_stride.  The result is the plain
 * definition: no split, no online rescaling. */
int orc_sparse_paged_decode(const uint16_t *qh, int64_t B, int q, int H, int Hkv,
                            const uint8_t *k_pages, const uint8_t *v_pages,
                            int64_t kv_page_stride, int64_t kv_head_stride, int64_t num_pages,
                            const int32_t *block_table, int64_t bt_width,
                            const int32_t *seq_lens, const int32_t *topk, int kw, double scale,
                            double *out)
{
    int64_t s;
    int j, h, r, d;
    double kd[ORC_ROW_ELEMS], vd[ORC_ROW_ELEMS];
    double *lg;
    int rc = ORC_OK;
    if (Hkv <= 0 || H % Hkv || kw <= 0) return ORC_ERR_INVALID;
    lg = (double *)malloc((size_t)kw * sizeof *lg);
    if (!lg) return ORC_ERR_INVALID;
    for (s = 0; s < B; ++s) {
        for (j = 0; j < q; ++j) {
            int64_t t = s * q + j;
            int64_t p = (int64_t)seq_lens[s] - q + j;
            const int32_t *sel = topk + t * kw;
            for (h = 0; h < H; ++h) {
                int hk = h / (H / Hkv);
                const uint16_t *qv = qh + (t * H + h) * ORC_ROW_ELEMS;
                double m = -INFINITY, l = 0.0;
                double *o = out + (t * H + h) * ORC_ROW_ELEMS;
                int n = 0;
                for (d = 0; d < ORC_ROW_ELEMS; ++d) o[d] = 0.0;
                /* logits */
                for (r = 0; r < kw; ++r) {
                    int64_t i = sel[r], pg;
                    double acc = 0.0;
                    if (i < 0) continue;
                    pg = page_of(block_table, bt_width, s, i, num_pages);
                    if (i > p || pg < 0) {
                        rc = ORC_ERR_BOUNDS;
                        goto done;
                    }
                    orc_dequant_row(k_pages + pg * kv_page_stride + hk * kv_head_stride,
                                    (int)(i % ORC_PAGE_TOKENS), kd);
                    for (d = 0; d < ORC_ROW_ELEMS; ++d) acc += bf16_to_double(qv[d]) * kd[d];
                    lg[r] = scale * acc;
                    if (lg[r] > m) m = lg[r];
                    ++n;
                }
                if (n == 0) continue; /* nothing selected: zero output */
                /* softmax weights and weighted sum of V */
                for (r = 0; r < kw; ++r) {
                    int64_t i = sel[r], pg;
                    double w;
                    if (i < 0) continue;
                    pg = page_of(block_table, bt_width, s, i, num_pages);
                    w = exp(lg[r] - m);
                    l += w;
                    orc_dequant_row(v_pages + pg * kv_page_stride + hk * kv_head_stride,
                                    (int)(i % ORC_PAGE_TOKENS), vd);
                    for (d = 0; d < ORC_ROW_ELEMS; ++d) o[d] += w * vd[d];
                }
                for (d = 0; d < ORC_ROW_ELEMS; ++d) o[d] /= l;
            }
        }
    }
done:
    free(lg);
    return rc;
}

/* ------------------------------------------------------------------------- */
/* The writer's norm and rotary embedding, R14 ([layer] SparseMoeLayer):
 *   z_j = x_j * g_j / sqrt(mean_j x_j^2 + eps)
 *   y_i = z_i c_i - z_{i+64} s_i,  y_{i+64} = z_{i+64} c_i + z_i s_i   (i < 64)
 * with c_i = cos_sin[pos][i], s_i = cos_sin[pos][64 + i]; rope = 0 skips the
 * rotation.  x: n rows of 128 fp32; out: n rows of 128 float64.  A position
 * outside [0, max_pos) is refused.                                            */
int orc_norm_rope(const float *x, int64_t n, const float *g, const float *cos_sin,
                  int64_t max_pos, const int64_t *pos, double eps, int rope, double *out)
{
    for (int64_t r = 0; r < n; ++r) {
        const float *xr = x + r * ORC_ROW_ELEMS;
        double *yr = out + r * ORC_ROW_ELEMS;
        double ss = 0.0;
        for (int j = 0; j < ORC_ROW_ELEMS; ++j) ss += (double)xr[j] * (double)xr[j];
        const double inv = 1.0 / sqrt(ss / ORC_ROW_ELEMS + eps);
        double z[ORC_ROW_ELEMS];
        for (int j = 0; j < ORC_ROW_ELEMS; ++j) z[j] = (double)xr[j] * inv * (double)g[j];
        if (!rope) {
            memcpy(yr, z, sizeof z);
            continue;
        }
        if (pos[r] < 0 || pos[r] >= max_pos) return ORC_ERR_BOUNDS;
        const float *cs = cos_sin + pos[r] * ORC_ROW_ELEMS;
        for (int i = 0; i < ORC_ROW_ELEMS / 2; ++i) {
            const double c = cs[i], sn = cs[ORC_ROW_ELEMS / 2 + i];
            yr[i] = z[i] * c - z[i + ORC_ROW_ELEMS / 2] * sn;
            yr[i + ORC_ROW_ELEMS / 2] = z[i + ORC_ROW_ELEMS / 2] * c + z[i] * sn;
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* The fp8 index cache variant  [fp8], [OCP], readings R15, R16               */
/* ------------------------------------------------------------------------- */

/* Value of an E4M3 code: bit 7 sign, bits 6..3 exponent (bias 7), bits 2..0
 * mantissa.  Exponent field 0 is subnormal: m/8 * 2^(1-7).  Otherwise
 * (1 + m/8) * 2^(e-7); S.1111.111 is NaN and there is no infinity. */
double orc_e4m3_value(int code)
{
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 15;
    int m = code & 7;
    double mag;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        mag = ldexp((double)m, -9);
    else
        mag = ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/* Round a non-negative double to the nearest integer, ties to the even one. */
static double round_half_even(double a)
{
    double f = floor(a), r = a - f;
    if (r > 0.5 || (r == 0.5 && fmod(f, 2.0) != 0.0)) f += 1.0;
    return f;
}

/* E4M3 code of a finite y (R16): nearest value, ties to the even mantissa,
 * magnitudes above 448 saturate to 448; the sign bit is kept for values that
 * round to zero.  Subnormals step by 2^-9; normals with exponent e (2^e <=
 * |y| < 2^(e+1), -6 <= e <= 8) step by 2^(e-3). */
int orc_e4m3_encode(float y)
{
    int sign = signbit(y) ? 0x80 : 0;
    double a = fabs((double)y);
    int e, code;
    if (a > 448.0) return sign | 0x7E;
    if (a < ldexp(1.0, -6)) {
        code = (int)round_half_even(ldexp(a, 9));            /* 0 .. 8; 8 is 2^-6 */
    } else {
        double mant;
        int m;
        (void)frexp(a, &e);
        e -= 1;                                               /* 2^e <= a < 2^(e+1) */
        mant = ldexp(a, -e);                                  /* [1, 2), exact */
        m = (int)round_half_even((mant - 1.0) * 8.0);        /* 0 .. 8 */
        if (m == 8) { m = 0; e += 1; }
        code = ((e + 7) << 3) | m;                            /* <= 0x7E as a <= 448 */
    }
    return sign | code;
}

/* Insert the index-K rows of new tokens into the fp8 cache: for each t with
 * slot s = slot_mapping[t] >= 0, byte d of row s%128 of page s/128 is
 * E4M3(fl32(idx_k[t][d] / scale)).  The quotient is rounded to fp32 first,
 * as an fp32 implementation divides (the precision the code is decided in).
 * Pages are addressed as base + page*page_stride, rows 128 B apart. */
int orc_fp8_index_insert(const float *idx_k, int64_t T, const int64_t *slot_mapping,
                         float scale, uint8_t *pages, int64_t page_stride, int64_t num_pages)
{
    int64_t t;
    int d;
    if (!(scale > 0.0f) || !isfinite(scale)) return ORC_ERR_INVALID;
    for (t = 0; t < T; ++t) {
        int64_t s = slot_mapping[t], page;
        uint8_t *row;
        if (s < 0) continue;                                  /* R6 */
        page = s / ORC_PAGE_TOKENS;
        if (page >= num_pages) return ORC_ERR_BOUNDS;
        row = pages + page * page_stride + (s % ORC_PAGE_TOKENS) * ORC_ROW_ELEMS;
        for (d = 0; d < ORC_ROW_ELEMS; ++d) {
            float x = idx_k[t * ORC_ROW_ELEMS + d];
            float y;
            if (!isfinite(x)) return ORC_ERR_INVALID;
            y = x / scale;
            row[d] = (uint8_t)orc_e4m3_encode(y);
        }
    }
    return ORC_OK;
}

/* Index scores over the fp8 cache: as orc_index_score, with the key element
 * read back as E4M3 value times scale (R16). */
int orc_index_score_fp8(const uint16_t *iq, int64_t B, int q, const uint8_t *pages,
                        int64_t page_stride, int64_t num_pages, const int32_t *block_table,
                        int64_t bt_width, const int32_t *seq_lens, float scale,
                        double *scores, double *mag, int64_t ld)
{
    int64_t s, i;
    int j, d;
    for (s = 0; s < B; ++s) {
        int64_t L = seq_lens[s];
        if (L < q || L > ld || L > bt_width * ORC_PAGE_TOKENS) return ORC_ERR_BOUNDS;
        for (j = 0; j < q; ++j) {
            int64_t t = s * q + j;
            int64_t p = L - q + j;
            const uint16_t *qt = iq + t * ORC_ROW_ELEMS;
            for (i = 0; i < ld; ++i) {
                double acc = 0.0, acc_abs = 0.0;
                int64_t pg;
                const uint8_t *row;
                if (i > p) {
                    scores[t * ld + i] = -INFINITY;
                    if (mag) mag[t * ld + i] = 0.0;
                    continue;
                }
                pg = page_of(block_table, bt_width, s, i, num_pages);
                if (pg < 0) return ORC_ERR_BOUNDS;
                row = pages + pg * page_stride + (i % ORC_PAGE_TOKENS) * ORC_ROW_ELEMS;
                for (d = 0; d < ORC_ROW_ELEMS; ++d) {
                    double term = bf16_to_double(qt[d]) * (orc_e4m3_value(row[d]) * scale);
                    acc += term;
                    acc_abs += fabs(term);
                }
                scores[t * ld + i] = acc;
                if (mag) mag[t * ld + i] = acc_abs;
            }
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* Block-scaled score mode: the index-q row in MXFP8  [OCP], reading R17     */
/* ------------------------------------------------------------------------- */

/* Shared exponent of an MXFP8 (E4M3) block with largest magnitude amax:
 * floor(log2(amax)) - 8, clamped to [-127, 127]; -127 for amax == 0. */
int orc_mxfp8_block_exponent(double amax)
{
    int e, E;
    if (amax == 0.0) return -127;
    (void)frexp(amax, &e);
    E = (e - 1) - 8;
    if (E < -127) E = -127;
    if (E > 127) E = 127;
    return E;
}

/* Quantise x[0..31] (finite) to 32 E4M3 codes and one E8M0 scale byte. */
int orc_mxfp8_quantize_block(const float *x, uint8_t *codes, uint8_t *scale_byte)
{
    double amax = 0.0;
    int i, E;
    for (i = 0; i < ORC_BLOCK; ++i) {
        if (!isfinite(x[i])) return ORC_ERR_INVALID;
        if (fabs((double)x[i]) > amax) amax = fabs((double)x[i]);
    }
    E = orc_mxfp8_block_exponent(amax);
    *scale_byte = (uint8_t)(E + 127);
    for (i = 0; i < ORC_BLOCK; ++i) {
        /* exact: a power-of-two scaling of an fp32 value, below 512 in magnitude;
         * parts below the smallest fp32 subnormal would round to code 0 anyway */
        codes[i] = (uint8_t)orc_e4m3_encode((float)ldexp((double)x[i], -E));
    }
    return ORC_OK;
}

/* Index scores with the index-q row in MXFP8 (R17): as orc_index_score, with
 * iq[t] replaced by its MXFP8 value sum_b E4M3(code_j) * 2^(scale_b - 127). */
int orc_index_score_mxq(const uint16_t *iq, int64_t B, int q, const uint8_t *idx_pages,
                        int64_t idx_page_stride, int64_t num_pages, const int32_t *block_table,
                        int64_t bt_width, const int32_t *seq_lens, double *scores, double *mag,
                        int64_t ld)
{
    int64_t s, i;
    int j, d, b;
    for (s = 0; s < B; ++s) {
        int64_t L = seq_lens[s];
        if (L < q || L > ld || L > bt_width * ORC_PAGE_TOKENS) return ORC_ERR_BOUNDS;
        for (j = 0; j < q; ++j) {
            int64_t t = s * q + j;
            int64_t p = L - q + j;
            float x[ORC_ROW_ELEMS];
            double qv[ORC_ROW_ELEMS];
            uint8_t codes[ORC_BLOCK], sb;
            for (d = 0; d < ORC_ROW_ELEMS; ++d)
                x[d] = (float)bf16_to_double(iq[t * ORC_ROW_ELEMS + d]);
            for (b = 0; b < ORC_ROW_ELEMS / ORC_BLOCK; ++b) {
                int rc = orc_mxfp8_quantize_block(x + b * ORC_BLOCK, codes, &sb);
                if (rc) return rc;
                for (d = 0; d < ORC_BLOCK; ++d)
                    qv[b * ORC_BLOCK + d] = orc_e4m3_value(codes[d]) * orc_e8m0_value(sb);
            }
            for (i = 0; i < ld; ++i) {
                double acc = 0.0, acc_abs = 0.0;
                int64_t pg;
                const uint8_t *page;
                if (i > p) {
                    scores[t * ld + i] = -INFINITY;
                    if (mag) mag[t * ld + i] = 0.0;
                    continue;
                }
                pg = page_of(block_table, bt_width, s, i, num_pages);
                if (pg < 0) return ORC_ERR_BOUNDS;
                page = idx_pages + pg * idx_page_stride;
                for (d = 0; d < ORC_ROW_ELEMS; ++d) {
                    double term = qv[d] * orc_dequant_element(page, (int)(i % ORC_PAGE_TOKENS), d);
                    acc += term;
                    acc_abs += fabs(term);
                }
                scores[t * ld + i] = acc;
                if (mag) mag[t * ld + i] = acc_abs;
            }
        }
    }
    return ORC_OK;
}
