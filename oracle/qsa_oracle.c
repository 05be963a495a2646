/*
 * QSA token-indexer CPU oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, single-threaded, obviously-correct restatement of what the QSA
 * token indexer computes.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library; the product path never
 * does.  It shares no code, header, table builder or constant with the CUDA
 * library: every helper below is written here for the oracle alone.
 *
 * Sources (the pages this restates):
 *  [SCORE]  pegainfer PR #1160 "feat(qwen4): score QSA token-indexer blocks in
 *           native CUDA": description (pooling, (1+w) RMSNorm, partial RoPE at
 *           the block's first token, sum_h relu(q_h . k_b) / sqrt(hd), relu as a
 *           comparison so NaN propagates, explicit score_cols, entries past a
 *           row's prefix untouched); review mutation table (the rounding points);
 *           "Tolerance" section (the reference rounds float32 reductions).
 *  [SELECT] pegainfer PR #1178 "select QSA indexer blocks": "Exact semantics"
 *           (blocks/tail/keep arithmetic, canonical tie order, mask contents,
 *           +-0 tie, non-finite is an error, empty launch is a no-op).
 *  [LAYER]  metrale layers/qsa.rs: module doc (mean-pool, norm, rope at the
 *           block's first position), decode_select (host sort by (-score, idx);
 *           the selected token list and the gather of its K/V rows from the
 *           paged cache into a contiguous scratch).
 *  [PREFILL] atlas layers/qsa_select.rs prefill_select: rows at or past the
 *           inert bound get their attention context replaced by attention
 *           over exactly their selected set (kept blocks' tokens and the tail),
 *           read from the paged K/V cache through the sequence's block table,
 *           with nq query heads over nkv KV heads and a 1/sqrt(d) scale;
 *           before scoring, the indexer's fused q|k row comes from a dense bf16
 *           projection of the normed hidden states (hidden -> 640) in slabs of
 *           2048 rows.
 *
 * Readings taken where the pages are silent:
 *  R1  bf16 <-> f32: widening is exact; narrowing is round-to-nearest-even,
 *      NaN stays NaN.
 *  R2  RoPE table: inv_freq[j] = f32(1 / theta^(2j/64)), angle = f32(p * inv_freq[j])
 *      (one f32 product), cos/sin taken in double and rounded to f32 then to
 *      bf16; row layout [c0..c31, c0..c31] (rotate-half pairing (i, i+32)).
 *  R3  Reductions the pages call "float32" (the 4-token mean, the mean square
 *      inside the norm) are taken as the exact sum rounded once to f32; the
 *      elementwise steps are single f32 operations in the reference's order:
 *      ms = f32(sum m^2 / 128); r = 1 / sqrt(ms + eps) (two IEEE f32 ops);
 *      y = (m * r) * (1 + w) (f32); then bf16.
 *  R4  RoPE on bf16 tensors rounds every elementwise op to bf16:
 *      out_i = bf16(bf16(x_i c_i) - bf16(x_{i+32} s_i)),
 *      out_{i+32} = bf16(bf16(x_{i+32} c_i) + bf16(x_i s_i)).
 *  R5  Query heads are prepared exactly like a pooled key (norm with q_norm_w,
 *      RoPE at the row's own position) and kept in bf16.
 *  R6  Each head's dot q_h . k_b is exact (double accumulation of 128 bf16 x bf16
 *      products), rounded once to f32; relu_h = (d < 0) ? 0 : d; the head sum is
 *      ((r0 + r1) + r2) + r3 in f32; score = f32(sum / sqrt(128)).
 *  R7  Selection compares real values, with -0.0 equal to +0.0; the canonical
 *      order is descending score then ascending block index.
 *  R8  Sparse attention is softmax attention restricted to the selected
 *      tokens: query head h reads KV head h / (nq / nkv) (consecutive query
 *      heads share a KV head); logits s_j = (q_h . k_j) * scale with the dot
 *      exact in double; weights exp(s_j - max s) in double; output
 *      sum_j w_j v_j / sum_j w_j in double, rounded to f32 and then to bf16
 *      (the attention output's dtype).  A row with no selected token gets zeros.
 *  R9  The projection y = x W^T (W stored [out, in], as a linear layer keeps
 *      it) sums the exact bf16 x bf16 products in double, rounds to f32, then
 *      to bf16 (the output dtype; the pages call it a bf16 dense projection).
 *
 * Build: plain C11, no fast-math, no FMA contraction (-ffp-contract=off).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_HEADS 4
#define ORC_HD 128
#define ORC_RATIO 4
#define ORC_ROT 64
#define ORC_HALF 32

enum {
    ORC_OK = 0,
    ORC_ERR_INVALID_VALUE = 1,
    ORC_ERR_ROW_RANGE = 3,
    ORC_ERR_NONFINITE = 4
};

/* ---- R1: bf16 helpers ---------------------------------------------------- */

static float orc_widen(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

static uint16_t orc_narrow(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u)          /* NaN: keep it a (quiet) NaN */
        return (uint16_t)((u >> 16) | 0x0040u);
    /* round to nearest, ties to even, on the bit pattern */
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static float orc_round_bf16(float f) { return orc_widen(orc_narrow(f)); }

uint16_t orc_f32_to_bf16(float f) { return orc_narrow(f); }

/* ---- R2: the RoPE cos/sin tables ----------------------------------------- */

int orc_rope_table(int32_t max_pos, double theta, uint16_t *cos_t, uint16_t *sin_t)
{
    float inv_freq[ORC_HALF];
    if (max_pos < 0 || !(theta > 0.0))
        return ORC_ERR_INVALID_VALUE;
    for (int j = 0; j < ORC_HALF; ++j)
        inv_freq[j] = (float)(1.0 / pow(theta, (double)(2 * j) / (double)ORC_ROT));
    for (int64_t p = 0; p < max_pos; ++p) {
        for (int j = 0; j < ORC_HALF; ++j) {
            float ang = (float)p * inv_freq[j];
            uint16_t c = orc_narrow((float)cos((double)ang));
            uint16_t s = orc_narrow((float)sin((double)ang));
            cos_t[p * ORC_ROT + j] = c;
            cos_t[p * ORC_ROT + j + ORC_HALF] = c;
            sin_t[p * ORC_ROT + j] = s;
            sin_t[p * ORC_ROT + j + ORC_HALF] = s;
        }
    }
    return ORC_OK;
}

/* ---- R3 + R4: (1 + w) RMSNorm then partial RoPE at position P ------------ */

static void orc_norm_rope(const float *x, const uint16_t *w, int64_t P,
                          const uint16_t *cos_t, const uint16_t *sin_t, float eps,
                          uint16_t *out)
{
    double ss = 0.0;
    float n[ORC_HD];
    for (int d = 0; d < ORC_HD; ++d)
        ss += (double)x[d] * (double)x[d];
    float ms = (float)(ss / (double)ORC_HD);
    float r = 1.0f / sqrtf(ms + eps);
    for (int d = 0; d < ORC_HD; ++d) {
        float scaled = x[d] * r;
        float gain = 1.0f + orc_widen(w[d]);
        n[d] = orc_round_bf16(scaled * gain);
    }
    const uint16_t *crow = cos_t + P * ORC_ROT;
    const uint16_t *srow = sin_t + P * ORC_ROT;
    for (int i = 0; i < ORC_HALF; ++i) {
        float c = orc_widen(crow[i]);
        float s = orc_widen(srow[i]);
        float x1 = n[i];
        float x2 = n[i + ORC_HALF];
        float a = orc_round_bf16(x1 * c);
        float b = orc_round_bf16(x2 * s);
        float e = orc_round_bf16(x2 * c);
        float f = orc_round_bf16(x1 * s);
        out[i] = orc_narrow(a - b);
        out[i + ORC_HALF] = orc_narrow(e + f);
    }
    for (int d = ORC_ROT; d < ORC_HD; ++d)
        out[d] = orc_narrow(n[d]);
}

/* ---- Pooling: one bf16 key per complete 4-token block -------------------- */
/*
 * keys points at the raw key of token 4*first_block; token 4*first_block + t
 * is at keys + t*key_stride.  Block b = first_block + i is written to
 * block_keys + b*128 and rotated at its first token, position 4b.
 */
int orc_pool_blocks(const uint16_t *keys, int64_t key_stride, int32_t first_block,
                    int32_t n_blocks, const uint16_t *k_norm_w, const uint16_t *cos_t,
                    const uint16_t *sin_t, float eps, uint16_t *block_keys)
{
    if (n_blocks < 0 || first_block < 0 || key_stride < ORC_HD)
        return ORC_ERR_INVALID_VALUE;
    for (int32_t i = 0; i < n_blocks; ++i) {
        int64_t b = (int64_t)first_block + i;
        const uint16_t *k0 = keys + (int64_t)ORC_RATIO * i * key_stride;
        float m[ORC_HD];
        for (int d = 0; d < ORC_HD; ++d) {
            double acc = 0.0;
            for (int t = 0; t < ORC_RATIO; ++t)
                acc += (double)orc_widen(k0[(int64_t)t * key_stride + d]);
            float mean = (float)acc * 0.25f;     /* float32 average ... */
            m[d] = orc_round_bf16(mean);         /* ... cast back to bf16 */
        }
        orc_norm_rope(m, k_norm_w, (int64_t)ORC_RATIO * b, cos_t, sin_t, eps,
                      block_keys + b * ORC_HD);
    }
    return ORC_OK;
}

/* ---- R5: query heads of one row ------------------------------------------ */

int orc_qprep(const uint16_t *q_row, int32_t pos, const uint16_t *q_norm_w,
              const uint16_t *cos_t, const uint16_t *sin_t, float eps, uint16_t *q_out)
{
    if (pos < 0)
        return ORC_ERR_ROW_RANGE;
    for (int h = 0; h < ORC_HEADS; ++h) {
        float x[ORC_HD];
        for (int d = 0; d < ORC_HD; ++d)
            x[d] = orc_widen(q_row[h * ORC_HD + d]);
        orc_norm_rope(x, q_norm_w, pos, cos_t, sin_t, eps, q_out + h * ORC_HD);
    }
    return ORC_OK;
}

/* ---- R6: one row's block scores ------------------------------------------ */

static float orc_relu(float d) { return (d < 0.0f) ? 0.0f : d; }

void orc_score_row(const uint16_t *q_prepped, const uint16_t *block_keys, int32_t n_blocks,
                   float *out)
{
    const double root = sqrt((double)ORC_HD);
    for (int32_t b = 0; b < n_blocks; ++b) {
        const uint16_t *k = block_keys + (int64_t)b * ORC_HD;
        float rl[ORC_HEADS];
        for (int h = 0; h < ORC_HEADS; ++h) {
            double acc = 0.0;
            for (int d = 0; d < ORC_HD; ++d)
                acc += (double)orc_widen(q_prepped[h * ORC_HD + d]) * (double)orc_widen(k[d]);
            rl[h] = orc_relu((float)acc);
        }
        float s = ((rl[0] + rl[1]) + rl[2]) + rl[3];
        out[b] = (float)((double)s / root);
    }
}

/*
 * Score rows: row i reads its 4 query heads at q + i*q_stride (512 bf16),
 * sits at position pos[i], sees visible_len[i] tokens (pos[i] + 1 when the
 * array is NULL) and the block keys at block_keys + key_base[i]*128 (offset 0
 * when NULL).  It writes scores[i*score_cols + b] for b < visible/4 and
 * nothing past that.  Returns the first error; *err_row gets its row.
 */
int orc_score_rows(const uint16_t *q, int64_t q_stride, const int32_t *pos,
                   const int32_t *visible_len, int32_t n_rows, int32_t tokens,
                   const uint16_t *q_norm_w, const uint16_t *cos_t, const uint16_t *sin_t,
                   float eps, const uint16_t *block_keys, const int64_t *key_base,
                   float *scores, int64_t score_cols, int32_t *err_row)
{
    int first = ORC_OK;
    for (int32_t i = 0; i < n_rows; ++i) {
        int32_t p = pos[i];
        int32_t vis = visible_len ? visible_len[i] : p + 1;
        if (p < 0 || p >= tokens || vis < 0 || vis > p + 1) {
            if (first == ORC_OK) {
                first = ORC_ERR_ROW_RANGE;
                if (err_row)
                    *err_row = i;
            }
            continue;
        }
        uint16_t qp[ORC_HEADS * ORC_HD];
        orc_qprep(q + (int64_t)i * q_stride, p, q_norm_w, cos_t, sin_t, eps, qp);
        const uint16_t *keys_row = block_keys + (key_base ? key_base[i] : 0) * ORC_HD;
        orc_score_row(qp, keys_row, vis / ORC_RATIO, scores + (int64_t)i * score_cols);
    }
    return first;
}

/* ---- R7: exact selection and the visibility mask ------------------------- */

typedef struct {
    float v;
    int32_t b;
} orc_item;

static int orc_canonical(const void *pa, const void *pb)
{
    const orc_item *a = (const orc_item *)pa;
    const orc_item *b = (const orc_item *)pb;
    if (a->v > b->v)
        return -1;                 /* higher score first */
    if (a->v < b->v)
        return 1;
    return (a->b < b->b) ? -1 : (a->b > b->b);   /* then lower block index */
}

/*
 * One query row at position p over a mask row of `tokens` bytes.  blocks =
 * (p+1)/4, tail = (p+1)%4, keep = min(budget/4, blocks).  The mask is 1 on the
 * four tokens of every kept block and on the tail [4*blocks, p], 0 elsewhere.
 */
int orc_select_row(const float *s, int32_t p, int32_t tokens, int32_t budget, uint8_t *mask_row)
{
    if (budget <= 0 || budget % ORC_RATIO != 0 || budget / ORC_RATIO > 512)
        return ORC_ERR_INVALID_VALUE;
    if (p < 0 || p >= tokens)
        return ORC_ERR_ROW_RANGE;
    int32_t blocks = (p + 1) / ORC_RATIO;
    int32_t keep = budget / ORC_RATIO;
    for (int32_t b = 0; b < blocks; ++b)   /* finiteness is checked on truncating rows only */
        if (blocks > keep && !isfinite(s[b]))
            return ORC_ERR_NONFINITE;
    memset(mask_row, 0, (size_t)tokens);
    if (blocks <= keep) {                  /* every block kept: the visible prefix */
        memset(mask_row, 1, (size_t)p + 1);
        return ORC_OK;
    }
    orc_item *items = (orc_item *)malloc(sizeof(orc_item) * (size_t)blocks);
    if (!items)
        return ORC_ERR_INVALID_VALUE;
    for (int32_t b = 0; b < blocks; ++b) {
        items[b].v = (s[b] == 0.0f) ? 0.0f : s[b];   /* -0.0 ties +0.0 */
        items[b].b = b;
    }
    qsort(items, (size_t)blocks, sizeof(orc_item), orc_canonical);
    for (int32_t i = 0; i < keep; ++i)
        memset(mask_row + (int64_t)ORC_RATIO * items[i].b, 1, ORC_RATIO);
    free(items);
    for (int32_t t = ORC_RATIO * blocks; t <= p; ++t)
        mask_row[t] = 1;
    return ORC_OK;
}

int orc_select_rows(const float *scores, int64_t score_cols, const int32_t *pos, int32_t n_rows,
                    int32_t tokens, int32_t budget, uint8_t *mask, int32_t *err_row)
{
    int first = ORC_OK;
    for (int32_t i = 0; i < n_rows; ++i) {
        int rc = orc_select_row(scores + (int64_t)i * score_cols, pos[i], tokens, budget,
                                mask + (int64_t)i * tokens);
        if (rc != ORC_OK && first == ORC_OK) {
            first = rc;
            if (err_row)
                *err_row = i;
        }
    }
    return first;
}

/*
 * [LAYER] metrale layers/qsa.rs decode_select, after the top-k: the selected
 * token list is every kept block's `ratio` tokens, blocks ascending, then the
 * tail tokens -- i.e. every token whose mask byte is 1, in ascending order.
 * Here: the tokens t < tokens with mask_row[t] != 0, ascending; at most `cap`
 * are written to out; the return value is how many there are.
 */
int32_t orc_mask_tokens(const uint8_t *mask_row, int32_t tokens, int32_t *out, int32_t cap)
{
    int32_t n = 0;
    for (int32_t t = 0; t < tokens; ++t) {
        if (mask_row[t] != 0) {
            if (n < cap)
                out[n] = t;
            ++n;
        }
    }
    return n;
}

/*
 * [LAYER] metrale layers/qsa.rs decode_select's gather (QsaSelection: a
 * contiguous NHD k/v scratch read as a paged cache through an identity table).
 * The paged pool holds `width` = kv_heads * head_dim bf16 values per token,
 * pages of page_size tokens: token t of the sequence lives in physical page
 * table[t / page_size], slot t % page_size.  Output row i is the pool row of
 * token sel[i], for i < n_sel.  Returns ORC_ERR_INVALID_VALUE (and copies
 * nothing more) at the first token outside [0, table_len * page_size).
 */
int orc_gather(const uint16_t *pool, const int32_t *table, int32_t table_len, int32_t page_size,
               int32_t width, const int32_t *sel, int32_t n_sel, uint16_t *out)
{
    for (int32_t i = 0; i < n_sel; ++i) {
        const int32_t t = sel[i];
        if (t < 0 || t / page_size >= table_len)
            return ORC_ERR_INVALID_VALUE;
        const int64_t slot = (int64_t)table[t / page_size] * page_size + t % page_size;
        memcpy(out + (int64_t)i * width, pool + slot * width, (size_t)width * sizeof(uint16_t));
    }
    return ORC_OK;
}

/* The pool slot of token t: its page's physical index, then its place in the page. */
static int64_t orc_attn_slot(const int32_t *table, int32_t page_size, int32_t t)
{
    const int32_t page = t / page_size;
    return (int64_t)table[page] * page_size + (t - page * page_size);
}

/*
 * [PREFILL] + R8: one query row's sparse attention.  q holds nq heads of hd
 * bf16 values; the pools hold [slots, nkv, hd] bf16 (slot = page * page_size +
 * t % page_size, page = table[t / page_size]); out receives nq * hd bf16.
 * Returns ORC_ERR_INVALID_VALUE (out unspecified) at a token outside
 * [0, table_len * page_size).
 */
int orc_sparse_attn(const uint16_t *q, int32_t nq, int32_t nkv, int32_t hd, const uint16_t *k_pool,
                    const uint16_t *v_pool, const int32_t *table, int32_t table_len,
                    int32_t page_size, const int32_t *sel, int32_t n_sel, double scale,
                    uint16_t *out)
{
    if (nq <= 0 || nkv <= 0 || nq % nkv != 0 || hd <= 0)
        return ORC_ERR_INVALID_VALUE;
    for (int32_t j = 0; j < n_sel; ++j)
        if (sel[j] < 0 || sel[j] / page_size >= table_len)
            return ORC_ERR_INVALID_VALUE;
    const int32_t group = nq / nkv;
    double *w = (double *)malloc(sizeof(double) * (n_sel > 0 ? n_sel : 1));
    double *acc = (double *)malloc(sizeof(double) * hd);
    if (!w || !acc) {
        free(w);
        free(acc);
        return ORC_ERR_INVALID_VALUE;
    }
    for (int32_t h = 0; h < nq; ++h) {
        const int32_t g = h / group;
        const uint16_t *qh = q + (int64_t)h * hd;
        double mx = -INFINITY;
        for (int32_t j = 0; j < n_sel; ++j) {
            const int32_t t = sel[j];
            const uint16_t *k = k_pool + (orc_attn_slot(table, page_size, t) * nkv + g) * hd;
            double d = 0.0;
            for (int32_t e = 0; e < hd; ++e)
                d += (double)orc_widen(qh[e]) * (double)orc_widen(k[e]);
            w[j] = d * scale;
            if (w[j] > mx)
                mx = w[j];
        }
        double den = 0.0;
        for (int32_t e = 0; e < hd; ++e)
            acc[e] = 0.0;
        for (int32_t j = 0; j < n_sel; ++j) {
            const int32_t t = sel[j];
            const uint16_t *v = v_pool + (orc_attn_slot(table, page_size, t) * nkv + g) * hd;
            const double wj = exp(w[j] - mx);
            den += wj;
            for (int32_t e = 0; e < hd; ++e)
                acc[e] += wj * (double)orc_widen(v[e]);
        }
        for (int32_t e = 0; e < hd; ++e)
            out[(int64_t)h * hd + e] = n_sel > 0 ? orc_narrow((float)(acc[e] / den)) : 0;
    }
    free(w);
    free(acc);
    return ORC_OK;
}

/*
 * [PREFILL] + R9: the index_qk_proj projection of one slab.  x holds n_rows
 * rows of `hidden` bf16 at row stride x_stride; w holds out_cols rows of
 * `hidden` bf16 (a linear layer's [out, in] weight); y receives n_rows rows of
 * out_cols bf16 at row stride y_stride.
 */
int orc_proj(const uint16_t *x, int64_t x_stride, const uint16_t *w, int32_t n_rows,
             int32_t hidden, int32_t out_cols, uint16_t *y, int64_t y_stride)
{
    if (n_rows < 0 || hidden <= 0 || out_cols <= 0)
        return ORC_ERR_INVALID_VALUE;
    for (int32_t r = 0; r < n_rows; ++r) {
        const uint16_t *xr = x + (int64_t)r * x_stride;
        for (int32_t n = 0; n < out_cols; ++n) {
            const uint16_t *wn = w + (int64_t)n * hidden;
            double acc = 0.0;
            for (int32_t k = 0; k < hidden; ++k)
                acc += (double)orc_widen(xr[k]) * (double)orc_widen(wn[k]);
            y[(int64_t)r * y_stride + n] = orc_narrow((float)acc);
        }
    }
    return ORC_OK;
}

