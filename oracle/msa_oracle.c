/*
 * msa_oracle.c -- plain CPU reference of block-sparse paged decode attention.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg call this code; the library never does.  It
 * shares no code, header, table or helper with the CUDA path.
 *
 * Sources.  The method is described in prose on three TensorRT-LLM pull
 * request pages about MiniMax-M3 serving:
 *   [M3-DECODE]  "MiniMax-M3 NVFP4 low-latency decode megakernel for
 *                modeling_v2 for Blackwell", sections "The TP4 decode target",
 *                "The TP8 decode target" and "Step-loop runtime hooks";
 *   [M31-RUBIN]  "Add Rubin (sm_107) MiniMax-M3.1 low-latency decode targets",
 *                section "Items and numerics", section "Disclosures and known
 *                gaps", and its commit messages on the MSA selector/decode
 *                hooks, the long-context select, the prefill select tile and
 *                the q8kv4 indexer over an NVFP4 index-K mirror;
 *   [M3-P128]    "MiniMax-M3: native P128 draft KV view for the NVFP4 hybrid
 *                cache", section "Description".
 * The pages fix the structure (index score, per-block max, top-k block
 * selection with a smaller-index tie-break and an ascending -1-padded table,
 * GQA attention over the selected 128-token pages) but print no formula.
 * Where they are silent this file takes the plainest reading, marked READING.
 *
 * Everything is computed in double precision with plain loops, one token at
 * a time, in the order the definition states.  No blocking, no fusion.
 *
 * Layouts are those of the synthetic-input module (row-major; Hi index
 * heads, Hs selection heads: Hs = 1 when Hi = 1, else Hs = Hkv):
 *   q_idx       bf16 bits  [T][Hi][Di]
 *   idxk_pool   bf16 bits  [pages][Hi][P][Di]  or NVFP4 bytes [pages][Hi][P][Di/2]
 *   idxk_scales E4M3 codes [pages][Hi][P][Di/16]   (NVFP4 only)
 *   q           bf16 bits  [T][Hq][D]
 *   kv_pool     bf16 bits or E4M3 codes [pages][2][Hkv][P][D]  (K then V)
 *   block_table int32      [R][max_blocks]
 *   seq_lens    int32      [R]
 *   selected    int32      [T][Hs][topk]
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct oracle_shape {
    int32_t num_requests;
    int32_t q_per_req;
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t index_dim;
    int32_t page_size;
    int32_t num_pages;
    int32_t max_blocks;
    int32_t topk;
    int32_t kv_fp8;      /* 0: bf16 K/V; 1: E4M3 K/V with per-tensor scales; 2: NVFP4 K/V */
    int32_t index_nvfp4; /* 0: bf16 index keys; 1: NVFP4 codes + E4M3 scales */
    double softmax_scale;
    double k_scale;
    double v_scale;
    int32_t num_index_heads; /* Hi: 1, or a multiple of num_kv_heads */
    int32_t init_blocks;     /* first blocks every token keeps (0: none) */
    int32_t local_blocks;    /* most recent blocks every token keeps (0: none) */
} oracle_shape;

enum {
    ORACLE_OK = 0,
    ORACLE_BAD_PAGE = 1,
    ORACLE_BAD_SEQ_LEN = 2,
    ORACLE_BAD_SELECTION = 3,
    ORACLE_NO_MEMORY = 4,
    ORACLE_BAD_SHAPE = 5,
};

/* Selection heads: one table per token shared by every KV head when there is
 * one index head, else one table per KV head.  [M31-RUBIN] selector-hook
 * commit: the selector is offered "KV-head-reduced scores"; the select op's
 * table is [tokens, heads, topk]; [M3-DECODE] restructure of the targets:
 * "4 KV / index heads".  READING: index head i belongs to KV head
 * i / (Hi / Hkv) (consecutive, as for query heads). */
static int selection_heads(const oracle_shape *s)
{
    return s->num_index_heads == 1 ? 1 : s->num_kv_heads;
}

/* ---- element decoders --------------------------------------------------- */

/* bf16: the upper 16 bits of an IEEE binary32. */
double oracle_bf16(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* FP8 E4M3 ("fn" variant: no infinities, S.1111.111 is NaN): 1 sign bit,
 * 4 exponent bits with bias 7, 3 mantissa bits; exponent 0 is subnormal.
 * [M31-RUBIN] "Items and numerics" and [M3-DECODE] "The TP4 decode target"
 * use FP8 KV; the pages name the format only. */
double oracle_e4m3(uint8_t code)
{
    int sign = code >> 7;
    int e = (code >> 3) & 15;
    int m = code & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);          /* m/8 * 2^(1-7) */
    else
        v = ldexp((double)(8 + m), e - 10); /* (1 + m/8) * 2^(e-7) */
    return sign ? -v : v;
}

/* FP4 E2M1: 1 sign bit, 2 exponent bits with bias 1, 1 mantissa bit;
 * exponent 0 is subnormal (0 or 0.5).  The NVFP4 index-K pages of
 * [M31-RUBIN] (indexer_kv_dtype='nvfp4') hold these codes. */
double oracle_e2m1(uint8_t nibble)
{
    int sign = (nibble >> 3) & 1;
    int e = (nibble >> 1) & 3;
    int m = nibble & 1;
    double v;
    if (e == 0)
        v = 0.5 * m;
    else
        v = ldexp((double)(2 + m), e - 2); /* (1 + m/2) * 2^(e-1) */
    return sign ? -v : v;
}

/* ---- element encoders (the KV / index-key update) ----------------------- */

/* Nearest code of a non-negative magnitude among the codes 0..top (whose
 * values increase with the code), ties to the even code; values above the
 * largest one saturate to it.  Round to nearest, ties to even, saturating:
 * the rounding NVIDIA's FP8 / FP4 conversions name (satfinite). */
static int nearest_code(double mag, double (*decode)(uint8_t), int top)
{
    if (!(mag < decode((uint8_t)top)))
        return top;
    int best = 0;
    for (int c = 1; c <= top; ++c) {
        double d_best = fabs(decode((uint8_t)best) - mag), d = fabs(decode((uint8_t)c) - mag);
        if (d < d_best || (d == d_best && (c & 1) == 0 && (best & 1) == 1))
            best = c;
    }
    return best;
}

/* E4M3 code of x (largest finite magnitude 448 = code 0x7E).  A value that
 * rounds to zero is stored as +0. */
uint8_t oracle_encode_e4m3(double x)
{
    int c = nearest_code(fabs(x), oracle_e4m3, 0x7E);
    return (uint8_t)(c == 0 ? 0 : (signbit(x) ? 0x80 | c : c));
}

/* E2M1 code of x (largest magnitude 6 = code 7); zero is stored as +0. */
uint8_t oracle_encode_e2m1(double x)
{
    int c = nearest_code(fabs(x), oracle_e2m1, 7);
    return (uint8_t)(c == 0 ? 0 : (signbit(x) ? 8 | c : c));
}

/* ---- paged gather ------------------------------------------------------- */

/* Page holding logical block b of request r, or -1 if the table entry is out
 * of the pool.  [M3-P128] "Description": one block table row per request
 * maps each 128-token block to its page. */
static int64_t page_of(const oracle_shape *s, const int32_t *block_table, int r, int64_t b)
{
    if (b < 0 || b >= s->max_blocks)
        return -1;
    int64_t page = block_table[(int64_t)r * s->max_blocks + b];
    if (page < 0 || page >= s->num_pages)
        return -1;
    return page;
}

/* Index key of token `tok` of `page`, dimension d, dequantised.
 * READING for NVFP4 (the pages give no byte layout): dimension 2i is the
 * low nibble of byte i, one E4M3 scale covers 16 consecutive dimensions,
 * and there is no second-level (global) scale. */
static double index_key(const oracle_shape *s, const void *pool, const uint8_t *scales,
                        int64_t page, int head, int tok, int d)
{
    int64_t row = (page * s->num_index_heads + head) * s->page_size + tok;
    if (!s->index_nvfp4)
        return oracle_bf16(((const uint16_t *)pool)[row * s->index_dim + d]);
    uint8_t byte = ((const uint8_t *)pool)[row * (s->index_dim / 2) + d / 2];
    uint8_t code = (d & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15);
    double scale = oracle_e4m3(scales[row * (s->index_dim / 16) + d / 16]);
    return oracle_e2m1(code) * scale;
}

/* Bytes of one NVFP4 K or V tile (one page, one KV head): e2m1 codes
 * [P][D/2] then E4M3 scales [P][D/16]. */
static int64_t nvfp4_tile_bytes(const oracle_shape *s)
{
    return (int64_t)s->page_size * (s->head_dim / 2 + s->head_dim / 16);
}

/* Element d of token tok of the K (kv = 0) or V (kv = 1) page of KV head g.
 * READING for NVFP4 K/V (the pages name the dtype, "Q8KV4", and give no
 * layout): the K tile of (page, g) then the V tiles, as for bf16 / FP8, each
 * tile [P][D/2] e2m1 pairs (dimension 2i in the low nibble) followed by
 * [P][D/16] E4M3 scales, one per 16 consecutive dimensions; k_scale and
 * v_scale are the second-level (per-tensor) scales. */
static double kv_elem(const oracle_shape *s, const void *kv_pool, int64_t page, int kv, int g,
                      int tok, int d)
{
    int64_t tile = (page * 2 + kv) * s->num_kv_heads + g;
    if (s->kv_fp8 == 2) {
        const uint8_t *t = (const uint8_t *)kv_pool + tile * nvfp4_tile_bytes(s);
        uint8_t byte = t[(int64_t)tok * (s->head_dim / 2) + d / 2];
        uint8_t code = (d & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15);
        uint8_t sc = t[(int64_t)s->page_size * (s->head_dim / 2) + (int64_t)tok * (s->head_dim / 16) + d / 16];
        return oracle_e2m1(code) * oracle_e4m3(sc) * (kv ? s->v_scale : s->k_scale);
    }
    int64_t idx = (tile * (int64_t)s->page_size + tok) * s->head_dim + d;
    if (!s->kv_fp8)
        return oracle_bf16(((const uint16_t *)kv_pool)[idx]);
    return oracle_e4m3(((const uint8_t *)kv_pool)[idx]) * (kv ? s->v_scale : s->k_scale);
}

/* Causal limit: query token j of request r sees positions 0 .. seq_len+j-1.
 * READING: a speculative step appends q_per_req tokens; token j is the j-th
 * of them, so seq_lens[r] counts the positions its first token sees. */
static int64_t visible(const oracle_shape *s, const int32_t *seq_lens, int t)
{
    int r = t / s->q_per_req, j = t % s->q_per_req;
    return (int64_t)seq_lens[r] + j;
}

static int check_request(const oracle_shape *s, const int32_t *seq_lens, int r)
{
    int64_t cached = (int64_t)seq_lens[r] + s->q_per_req - 1;
    if (seq_lens[r] < 1)
        return ORACLE_BAD_SEQ_LEN;
    if ((cached + s->page_size - 1) / s->page_size > s->max_blocks)
        return ORACLE_BAD_SEQ_LEN;
    return ORACLE_OK;
}

/* ---- (a) index score and per-block max ---------------------------------- */

/* out[b] = max over visible positions pos of block b of the dot product of
 * the token's index query of index head `head` with that head's index key
 * at pos; -inf for a block with no visible position.  [M3-DECODE] "The TP4 decode target" (index scorer
 * over index-K pages) and [M31-RUBIN] prefill-select commit (per-block
 * "proxy" max score).  READING: the score is the plain dot product (no
 * weights, activation or scaling appear on the pages). */
int oracle_block_scores(const oracle_shape *s, const uint16_t *q_idx, const void *idxk_pool,
                        const uint8_t *idxk_scales, const int32_t *block_table,
                        const int32_t *seq_lens, int t, int head, double *out)
{
    int r = t / s->q_per_req;
    if (head < 0 || head >= s->num_index_heads)
        return ORACLE_BAD_SHAPE;
    int rc = check_request(s, seq_lens, r);
    if (rc)
        return rc;
    for (int b = 0; b < s->max_blocks; ++b)
        out[b] = -INFINITY;
    int64_t L = visible(s, seq_lens, t);
    const uint16_t *qi = q_idx + ((int64_t)t * s->num_index_heads + head) * s->index_dim;
    for (int64_t pos = 0; pos < L; ++pos) {
        int64_t b = pos / s->page_size;
        int64_t page = page_of(s, block_table, r, b);
        if (page < 0)
            return ORACLE_BAD_PAGE;
        double score = 0.0;
        for (int d = 0; d < s->index_dim; ++d)
            score += oracle_bf16(qi[d])
                     * index_key(s, idxk_pool, idxk_scales, page, head, (int)(pos % s->page_size), d);
        if (score > out[b])
            out[b] = score;
    }
    return ORACLE_OK;
}

/* ---- (b) top-k block selection ------------------------------------------ */

static const double *g_sort_scores; /* qsort context; guarded by the caller */

static int by_score_then_index(const void *pa, const void *pb)
{
    int a = *(const int *)pa, b = *(const int *)pb;
    double sa = g_sort_scores[a], sb = g_sort_scores[b];
    if (sa > sb)
        return -1;
    if (sa < sb)
        return 1;
    return (a > b) - (a < b);
}

static int ascending(const void *pa, const void *pb)
{
    int a = *(const int *)pa, b = *(const int *)pb;
    return (a > b) - (a < b);
}

/* Top-k selection with forced blocks.  Forced: the first min(init, n_valid)
 * blocks and the last min(local, n_valid) of blocks 0..n_valid-1
 * ([M31-RUBIN] prefill-select commit: the tile select reproduces the stock
 * table "including tie order and init / local forcing").  READING: forced
 * blocks are always kept (the pages give no further rule), init + local <= k,
 * and the remaining k - |forced| places go to the other blocks in the order
 * (score descending, block index ascending) ([M3-DECODE] "The TP4 decode
 * target": ties go to the smaller block).  The kept blocks are written in
 * ascending order followed by -1 up to k ([M31-RUBIN] q8kv4 indexer commit:
 * "the ascending, -1-padded contract").  READING: only blocks that hold a
 * visible position (finite score) are candidates. */
int oracle_select_forced(const double *scores, int n_valid, int k, int init, int local,
                         int32_t *sel)
{
    if (init < 0 || local < 0 || init + local > k)
        return ORACLE_BAD_SHAPE;
    int *order = (int *)malloc(sizeof(int) * (size_t)(n_valid > 0 ? n_valid : 1));
    char *forced = (char *)calloc((size_t)(n_valid > 0 ? n_valid : 1), 1);
    if (!order || !forced) {
        free(order);
        free(forced);
        return ORACLE_NO_MEMORY;
    }
    int n_forced = 0;
    for (int b = 0; b < n_valid; ++b) {
        forced[b] = (char)(b < init || b >= n_valid - local);
        n_forced += forced[b];
    }
    /* the other blocks, best first */
    int n_other = 0;
    for (int b = 0; b < n_valid; ++b)
        if (!forced[b])
            order[n_other++] = b;
#ifdef _OPENMP
#pragma omp critical(oracle_qsort)
#endif
    {
        g_sort_scores = scores;
        qsort(order, (size_t)n_other, sizeof(int), by_score_then_index);
    }
    int room = k - n_forced;
    int keep_other = n_other < room ? n_other : room;
    /* kept = forced blocks + the best keep_other others, in ascending order */
    int keep = 0;
    for (int b = 0; b < n_valid; ++b)
        if (forced[b])
            sel[keep++] = b;
    for (int i = 0; i < keep_other; ++i)
        sel[keep++] = order[i];
    qsort(sel, (size_t)keep, sizeof(int32_t), ascending);
    for (int i = keep; i < k; ++i)
        sel[i] = -1;
    free(order);
    free(forced);
    return ORACLE_OK;
}

/* The plain top-k: no forced blocks. */
int oracle_select(const double *scores, int n_valid, int k, int32_t *sel)
{
    return oracle_select_forced(scores, n_valid, k, 0, 0, sel);
}

/* Scores of selection head gs: for each block the maximum over the group's
 * index heads i = gs * r .. gs * r + r - 1 (r = Hi / Hs) of their block
 * scores.  READING: the pages name "KV-head-reduced scores" without the
 * reduction; max keeps a block score the largest index score of any
 * position in the block under any index head of the group, as the per-block
 * max does for one head.  scores_by_head: [Hi][max_blocks]. */
void oracle_reduce_heads(const oracle_shape *s, const double *scores_by_head, int gs, double *out)
{
    int r = s->num_index_heads / selection_heads(s);
    for (int b = 0; b < s->max_blocks; ++b) {
        double m = -INFINITY;
        for (int i = gs * r; i < gs * r + r; ++i) {
            double v = scores_by_head[(int64_t)i * s->max_blocks + b];
            if (v > m)
                m = v;
        }
        out[b] = m;
    }
}

/* Block selection of many query rows from a head-major score buffer
 * scores[Hs][max_blocks][n_rows] (the row index innermost): row t of
 * selection head gs sees blocks 0 .. n_visible[t] - 1, and its table
 * sel[t][gs][0..k) is what oracle_select_forced gives for that row.
 * [M31-RUBIN] prefill-select commit: context rows take a tile select over a
 * [heads, max_k_tiles, tokens] max-score block, with the "same table bit
 * for bit, including tie order and init / local forcing" as the per-token
 * select. */
int oracle_select_rows(const double *scores, int hs, int max_blocks, int n_rows,
                       const int32_t *n_visible, int k, int init, int local, int32_t *sel)
{
    double *row = (double *)malloc(sizeof(double) * (size_t)(max_blocks > 0 ? max_blocks : 1));
    if (!row)
        return ORACLE_NO_MEMORY;
    int rc = ORACLE_OK;
    for (int t = 0; t < n_rows && !rc; ++t)
        for (int gs = 0; gs < hs && !rc; ++gs) {
            int n = n_visible[t];
            if (n < 0 || n > max_blocks) {
                rc = ORACLE_BAD_SHAPE;
                break;
            }
            for (int b = 0; b < n; ++b)
                row[b] = scores[((int64_t)gs * max_blocks + b) * n_rows + t];
            rc = oracle_select_forced(row, n, k, init, local, sel + ((int64_t)t * hs + gs) * k);
        }
    free(row);
    return rc;
}

/* ---- (c) attention over the selected pages ------------------------------ */

/* For every query head h (KV head g = h / (Hq/Hkv); READING: consecutive
 * query heads share a KV head) attend over the visible positions of the
 * selected blocks:
 *   z_pos = softmax_scale * sum_d q[t,h,d] * K[g,pos,d]
 *   O     = sum_pos e^(z_pos - M) V[g,pos,:] / sum_pos e^(z_pos - M)
 *   LSE   = M + ln sum_pos e^(z_pos - M),   M = max_pos z_pos
 * READING: the pages never define the LSE; this is the natural log of the
 * softmax denominator of the scaled logits.  FP8 K and V are dequantised
 * with their own per-tensor scale.  [M31-RUBIN] "Items and numerics"
 * checks the split-K merge against a float64 reference; this is that
 * reference with no split at all.  sel holds the token's tables
 * [Hs][topk] of block indices (ascending, -1 padded), as produced by
 * oracle_select_forced; query head h reads the table of its KV head g when
 * Hs > 1 ([M31-RUBIN]: the select op's table is [tokens, heads, topk]). */
int oracle_attend(const oracle_shape *s, const uint16_t *q, const void *kv_pool,
                  const int32_t *block_table, const int32_t *seq_lens, int t,
                  const int32_t *sel, double *out, double *lse)
{
    int r = t / s->q_per_req;
    int rc = check_request(s, seq_lens, r);
    if (rc)
        return rc;
    int64_t L = visible(s, seq_lens, t);
    int P = s->page_size, D = s->head_dim;
    int group = s->num_q_heads / s->num_kv_heads;

    /* positions attended by the heads of one table: the visible positions
     * of its selected blocks (rebuilt when the table changes) */
    int64_t npos = 0;
    int64_t *pos_page = (int64_t *)malloc(sizeof(int64_t) * (size_t)s->topk * P);
    int *pos_tok = (int *)malloc(sizeof(int) * (size_t)s->topk * P);
    double *z = (double *)malloc(sizeof(double) * (size_t)s->topk * P);
    if (!pos_page || !pos_tok || !z) {
        free(pos_page); free(pos_tok); free(z);
        return ORACLE_NO_MEMORY;
    }
    int hs = selection_heads(s), table = -1;
    for (int h = 0; h < s->num_q_heads; ++h) {
        int g = h / group;
        int gs = hs > 1 ? g : 0;
        if (gs != table) {
            table = gs;
            npos = 0;
            const int32_t *sl = sel + (int64_t)gs * s->topk;
            for (int i = 0; i < s->topk; ++i) {
                int32_t b = sl[i];
                if (b < 0)
                    continue;
                int64_t page = page_of(s, block_table, r, b);
                if (page < 0 || (int64_t)b * P >= L) {
                    free(pos_page); free(pos_tok); free(z);
                    return page < 0 ? ORACLE_BAD_PAGE : ORACLE_BAD_SELECTION;
                }
                for (int tok = 0; tok < P; ++tok) {
                    if ((int64_t)b * P + tok >= L)
                        break;
                    pos_page[npos] = page;
                    pos_tok[npos] = tok;
                    ++npos;
                }
            }
        }
        const uint16_t *qh = q + ((int64_t)t * s->num_q_heads + h) * D;
        double M = -INFINITY;
        for (int64_t n = 0; n < npos; ++n) {
            double acc = 0.0;
            for (int d = 0; d < D; ++d)
                acc += oracle_bf16(qh[d]) * kv_elem(s, kv_pool, pos_page[n], 0, g, pos_tok[n], d);
            z[n] = s->softmax_scale * acc;
            if (z[n] > M)
                M = z[n];
        }
        double denom = 0.0;
        double *o = out + (int64_t)h * D;
        for (int d = 0; d < D; ++d)
            o[d] = 0.0;
        for (int64_t n = 0; n < npos; ++n) {
            double w = exp(z[n] - M);
            denom += w;
            for (int d = 0; d < D; ++d)
                o[d] += w * kv_elem(s, kv_pool, pos_page[n], 1, g, pos_tok[n], d);
        }
        for (int d = 0; d < D; ++d)
            o[d] /= denom;
        lse[h] = M + log(denom);
    }
    free(pos_page);
    free(pos_tok);
    free(z);
    return ORACLE_OK;
}

/* ---- (d) KV / index-key update ------------------------------------------ */

/* One row of n bf16 values x (each divided by `scale` first, in binary32)
 * as NVFP4: per group of 16, scale code c = e4m3(amax / 6), codes
 * e2m1(y / value(c)) (0 when value(c) = 0), quotients in binary32,
 * dimension 2i in the low nibble of codes[i]. */
static void nvfp4_group_row(const uint16_t *x, int n, float scale, uint8_t *codes, uint8_t *scales)
{
    for (int grp = 0; grp < n / 16; ++grp) {
        float y[16], amax = 0.0f;
        for (int i = 0; i < 16; ++i) {
            y[i] = (float)oracle_bf16(x[16 * grp + i]) / scale;
            if (fabsf(y[i]) > amax)
                amax = fabsf(y[i]);
        }
        uint8_t sc = oracle_encode_e4m3((double)(amax / 6.0f));
        scales[grp] = sc;
        float S = (float)oracle_e4m3(sc);
        for (int i = 0; i < 16; i += 2) {
            uint8_t lo = S > 0.0f ? oracle_encode_e2m1((double)(y[i] / S)) : 0;
            uint8_t hi = S > 0.0f ? oracle_encode_e2m1((double)(y[i + 1] / S)) : 0;
            codes[8 * grp + i / 2] = (uint8_t)(lo | (hi << 4));
        }
    }
}

/* Writes this step's keys, values and index keys into their pages, in place.
 * [M3-DECODE] "The TP4 decode target": the attention megakernels carry "the
 * KV update"; [M31-RUBIN] q8kv4 indexer commit: the NVFP4 index-K copy is
 * "refreshed from this step's slots".  READING (the pages give neither the
 * slot nor the quantiser):
 *   - new token j of request r sits at position pos = seq_lens[r] - 1 + j
 *     (the last position it sees), row pos % P of page
 *     block_table[r][pos / P];
 *   - bf16 pools take the bf16 inputs as they are;
 *   - FP8 pools: code = e4m3(x / k_scale) for K and e4m3(x / v_scale) for V,
 *     the quotient in binary32 (the pages fix no precision; binary32 is the
 *     kernel's, so both sides take the rounding decision alike);
 *   - NVFP4 K / V pools: y = x / k_scale (x / v_scale) in binary32, then the
 *     index keys' group recipe below on y;
 *   - NVFP4 index keys, per group of 16 consecutive dimensions: scale code
 *     c = e4m3(amax / 6) with amax the largest |x| of the group and 6 the
 *     largest e2m1 magnitude, S its value, element codes e2m1(x / S) (0 when
 *     S = 0), quotients in binary32; no second-level scale, as for the
 *     decoder above.
 * Inputs (bf16 bits): k_new, v_new [T][Hkv][D], idxk_new [T][Hi][Di]. */
int oracle_kv_update(const oracle_shape *s, const uint16_t *k_new, const uint16_t *v_new,
                     const uint16_t *idxk_new, const int32_t *block_table,
                     const int32_t *seq_lens, void *kv_pool, void *idxk_pool,
                     uint8_t *idxk_scales)
{
    int T = s->num_requests * s->q_per_req;
    int Hkv = s->num_kv_heads, Hi = s->num_index_heads, D = s->head_dim, Di = s->index_dim;
    int P = s->page_size;
    for (int t = 0; t < T; ++t) {
        int r = t / s->q_per_req, j = t % s->q_per_req;
        int rc = check_request(s, seq_lens, r);
        if (rc)
            return rc;
        int64_t pos = (int64_t)seq_lens[r] - 1 + j;
        int64_t page = page_of(s, block_table, r, pos / P);
        if (page < 0)
            return ORACLE_BAD_PAGE;
        int row = (int)(pos % P);
        for (int kv = 0; kv < 2; ++kv) {
            const uint16_t *src = kv ? v_new : k_new;
            float scale = (float)(kv ? s->v_scale : s->k_scale);
            if (s->kv_fp8 == 2) {
                /* NVFP4 K / V: the group recipe of the index keys below on
                 * y = x / scale (binary32) */
                for (int g = 0; g < Hkv; ++g) {
                    uint8_t *tile = (uint8_t *)kv_pool + ((page * 2 + kv) * Hkv + g) * nvfp4_tile_bytes(s);
                    const uint16_t *x = src + ((int64_t)t * Hkv + g) * D;
                    nvfp4_group_row(x, D, scale, tile + (int64_t)row * (D / 2),
                                    tile + (int64_t)P * (D / 2) + (int64_t)row * (D / 16));
                }
                continue;
            }
            for (int g = 0; g < Hkv; ++g)
                for (int d = 0; d < D; ++d) {
                    uint16_t bits = src[((int64_t)t * Hkv + g) * D + d];
                    int64_t idx = (((page * 2 + kv) * Hkv + g) * (int64_t)P + row) * D + d;
                    if (!s->kv_fp8)
                        ((uint16_t *)kv_pool)[idx] = bits;
                    else
                        ((uint8_t *)kv_pool)[idx] =
                            oracle_encode_e4m3((double)((float)oracle_bf16(bits) / scale));
                }
        }
        for (int i = 0; i < Hi; ++i) {
            const uint16_t *src = idxk_new + ((int64_t)t * Hi + i) * Di;
            int64_t prow = (page * Hi + i) * (int64_t)P + row;
            if (!s->index_nvfp4) {
                for (int d = 0; d < Di; ++d)
                    ((uint16_t *)idxk_pool)[prow * Di + d] = src[d];
                continue;
            }
            nvfp4_group_row(src, Di, 1.0f, (uint8_t *)idxk_pool + prow * (Di / 2),
                            idxk_scales + prow * (Di / 16));
        }
    }
    return ORACLE_OK;
}

/* ---- the whole step ------------------------------------------------------ */

/* Runs (a), (b) and (c) for each token in tokens[0..n_tokens) and writes
 * row i of every output for tokens[i]:
 *   block_scores [n][Hi][max_blocks] float (every score is exact in
 *                binary32: integer-valued or NVFP4 inputs; the test suite
 *                checks this)
 *   selected     [n][Hs][topk]
 *   out          [n][Hq][D] double,  lse [n][Hq] double
 * num_threads > 1 spreads tokens over OpenMP threads (each token is still
 * computed by one thread in the same order). */
int oracle_decode_step(const oracle_shape *s, const uint16_t *q_idx, const void *idxk_pool,
                       const uint8_t *idxk_scales, const uint16_t *q, const void *kv_pool,
                       const int32_t *block_table, const int32_t *seq_lens,
                       const int32_t *tokens, int n_tokens, int num_threads,
                       float *block_scores, int32_t *selected, double *out, double *lse)
{
    int Hi = s->num_index_heads, hs = selection_heads(s);
    if (Hi < 1 || (Hi > 1 && Hi % s->num_kv_heads != 0))
        return ORACLE_BAD_SHAPE;
    int err = ORACLE_OK;
#ifdef _OPENMP
    if (num_threads < 1)
        num_threads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads)
#endif
    for (int i = 0; i < n_tokens; ++i) {
        int t = tokens[i];
        double *bs = (double *)malloc(sizeof(double) * (size_t)s->max_blocks * (size_t)Hi);
        double *red = (double *)malloc(sizeof(double) * (size_t)s->max_blocks);
        int rc = (bs && red) ? ORACLE_OK : ORACLE_NO_MEMORY;
        for (int head = 0; head < Hi && !rc; ++head)
            rc = oracle_block_scores(s, q_idx, idxk_pool, idxk_scales, block_table, seq_lens, t,
                                     head, bs + (int64_t)head * s->max_blocks);
        int32_t *sel_t = selected + (int64_t)i * hs * s->topk;
        if (!rc) {
            int64_t L = visible(s, seq_lens, t);
            int n_valid = (int)((L + s->page_size - 1) / s->page_size);
            for (int64_t x = 0; x < (int64_t)Hi * s->max_blocks; ++x)
                block_scores[(int64_t)i * Hi * s->max_blocks + x] = (float)bs[x];
            for (int gs = 0; gs < hs && !rc; ++gs) {
                oracle_reduce_heads(s, bs, gs, red);
                rc = oracle_select_forced(red, n_valid, s->topk, s->init_blocks, s->local_blocks,
                                          sel_t + (int64_t)gs * s->topk);
            }
        }
        if (!rc)
            rc = oracle_attend(s, q, kv_pool, block_table, seq_lens, t, sel_t,
                               out + (int64_t)i * s->num_q_heads * s->head_dim,
                               lse + (int64_t)i * s->num_q_heads);
        free(bs);
        free(red);
        if (rc) {
#ifdef _OPENMP
#pragma omp critical(oracle_err)
#endif
            err = rc;
        }
    }
    return err;
}

/* Threads the OpenMP runtime would use by default (1 without OpenMP). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
