/*
 * sa_oracle.c -- fp64 CPU oracle for grouped-query attention with per-head
 * attention sinks.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the CPU
 * baseline leg of bench.py load this file's library.  It shares no code, no
 * header and no table with the CUDA library: it has its own bf16 and E4M3
 * decoders, its own page-table walk and its own mask.
 *
 * What it computes (the plain definition; the method reaches exactly this
 * result up to rounding order, so this file does not follow the online
 * algorithm).  For one query row at position p of sequence b and query head h,
 * with G = Hq / Hkv query heads per kv head and g = floor(h / G):
 *
 *   J     = { j : 0 <= j <= p, j < L_b, and (w == 0 or j > p - w) }
 *   s_j   = sm_scale * sum_d q[h,d] * k[b,g,j,d]           (fp64)
 *   sigma = sinks[h]          (-inf when the caller passes no sinks)
 *   M     = max(sigma, max_{j in J} s_j)
 *   Z     = exp(sigma - M) + sum_{j in J} exp(s_j - M)
 *   o     = sum_{j in J} exp(s_j - M) v[b,g,j,:] / Z
 *   lse   = M + log(Z)                                      (natural log)
 *   J empty and sigma = -inf:  o = 0, lse = -inf
 *
 * Sources:
 *  - "GPT-OSS on day 0" (Perplexity), section "Attention: GQA with attention
 *    sinks": every attention head owns one pretrained sink parameter that
 *    takes part in the softmax.
 *  - same page, section "GPT-OSS kernels / Sink Attention": the sink is an
 *    extra term that enters the softmax beside the Q.K products (the printed
 *    formula is lost in the extracted text; the reading taken here is a softmax
 *    over the row [s_j..., sigma] whose sigma column has no value vector), and
 *    the online form seeds its running max with the sink and counts the sink
 *    in the first sequence chunk only.
 *  - NVIDIA gpt-oss launch article, introduction: attention layers alternate
 *    full context with a 128-token sliding window (read as the 128 keys
 *    j in (p-128, p]).
 *
 * The split mode (sao_attend_split + sao_merge) restates the chunked form of
 * the same page: per-chunk partial states without the sink, merged with the
 * sink counted once.  It exists to check that algebra; it is not used to
 * produce reference values for the kernels' unsplit outputs.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* Element decoders, written from the format definitions.                   */
/* ------------------------------------------------------------------------ */

/* bfloat16: the upper 16 bits of an IEEE-754 binary32. */
double sao_bf16_to_f64(uint16_t bits)
{
    uint32_t w = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* FP8 E4M3 (OCP 8-bit floating point, "E4M3"): 1 sign bit, 4 exponent bits
 * with bias 7, 3 mantissa bits.  Exponent field 0 holds subnormals
 * (m/8) * 2^(1-7).  Exponent 15 with mantissa 7 is NaN; there is no infinity,
 * so exponent 15 with mantissa 0..6 is an ordinary normal (largest 448). */
double sao_e4m3_to_f64(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double mag;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, 1 - 7);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/* ------------------------------------------------------------------------ */
/* KV cache description (the oracle's own; not the library's struct).       */
/* ------------------------------------------------------------------------ */
typedef struct {
    const void *k;               /* bf16 bit patterns (uint16) or E4M3 codes (uint8) */
    const void *v;
    int32_t dtype;               /* 0 = bf16, 1 = E4M3 */
    int32_t num_pages;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t page_size;
    int64_t stride_page;         /* elements */
    int64_t stride_head;
    int64_t stride_token;
    const int32_t *page_table;   /* [B, page_table_stride]; NULL: sequence b lives in page b */
    int32_t page_table_stride;
    double k_scale;              /* real value = decoded code * scale (1.0 for bf16) */
    double v_scale;
} sao_kv_t;

/* Offset (in elements) of token t of sequence b, kv head g, dim 0.  Returns
 * -1 when the page table points outside the pool, so that a malformed case
 * shows up as an error instead of an out-of-bounds read. */
static int64_t kv_offset(const sao_kv_t *kv, int b, int g, int t)
{
    int64_t page;
    int64_t slot = t % kv->page_size;
    if (kv->page_table)
        page = kv->page_table[(int64_t)b * kv->page_table_stride + t / kv->page_size];
    else
        page = b;
    if (page < 0 || page >= kv->num_pages)
        return -1;
    return page * kv->stride_page + (int64_t)g * kv->stride_head + slot * kv->stride_token;
}

static double kv_elem(const sao_kv_t *kv, const void *base, double scale, int64_t off, int d)
{
    if (kv->dtype == 0)
        return sao_bf16_to_f64(((const uint16_t *)base)[off + d]) * scale;
    return sao_e4m3_to_f64(((const uint8_t *)base)[off + d]) * scale;
}

/* Is key j visible to a query at position p of a sequence holding L keys? */
static int key_visible(int j, int p, int L, int window)
{
    if (j < 0 || j > p || j >= L)
        return 0;
    if (window > 0 && j <= p - window)
        return 0;
    return 1;
}

/* One query element: bf16 bits (q_fmt 0) or an E4M3 code times q_scale (q_fmt 1). */
typedef struct {
    const void *row;
    int fmt;
    double scale;
} sao_qrow_t;

static double q_elem(const sao_qrow_t *q, int d)
{
    if (q->fmt == 0)
        return sao_bf16_to_f64(((const uint16_t *)q->row)[d]);
    return sao_e4m3_to_f64(((const uint8_t *)q->row)[d]) * q->scale;
}

/* Score s_j for one (row, head): sm_scale * q . k_j, in fp64. */
static double score(const sao_qrow_t *qrow, const sao_kv_t *kv, int b, int g, int j,
                    double sm_scale, int *err)
{
    int64_t off = kv_offset(kv, b, g, j);
    double acc = 0.0;
    int d;
    if (off < 0) {
        *err = 1;
        return 0.0;
    }
    for (d = 0; d < kv->head_dim; ++d)
        acc += q_elem(qrow, d) * kv_elem(kv, kv->k, kv->k_scale, off, d);
    return sm_scale * acc;
}

/*
 * One (row, head) of the definition, restricted to keys in [j_lo, j_hi) on top
 * of the causal/window set J.  with_sink selects whether sigma takes part.
 * Writes o[0..D) and *lse.  Two passes: all scores first, then max, then sums.
 */
static int attend_one(const sao_qrow_t *qrow, const sao_kv_t *kv, int b, int g, int p, int L,
                      int window, double sm_scale, double sigma, int with_sink,
                      int j_lo, int j_hi, double *o, double *lse)
{
    const int D = kv->head_dim;
    int n = 0, j, d, err = 0;
    int lo = j_lo < 0 ? 0 : j_lo;
    int hi = j_hi;
    double *s, M, Z;
    int *idx;
    if (hi > p + 1)
        hi = p + 1;
    if (hi > L)
        hi = L;
    for (d = 0; d < D; ++d)
        o[d] = 0.0;
    if (!with_sink)
        sigma = -INFINITY;

    s = (double *)malloc(sizeof(double) * (size_t)(hi > lo ? hi - lo : 1));
    idx = (int *)malloc(sizeof(int) * (size_t)(hi > lo ? hi - lo : 1));
    if (!s || !idx) {
        free(s);
        free(idx);
        return 2;
    }
    /* pass 1: scores of the visible keys */
    for (j = lo; j < hi; ++j) {
        if (!key_visible(j, p, L, window))
            continue;
        s[n] = score(qrow, kv, b, g, j, sm_scale, &err);
        idx[n] = j;
        ++n;
    }
    if (err) {
        free(s);
        free(idx);
        return 1;
    }
    /* max over the sink and the scores */
    M = sigma;
    for (j = 0; j < n; ++j)
        if (s[j] > M)
            M = s[j];
    if (M == -INFINITY) { /* no key and no sink: empty softmax */
        *lse = -INFINITY;
        free(s);
        free(idx);
        return 0;
    }
    /* pass 2: denominator and weighted sum of values */
    Z = (sigma == -INFINITY) ? 0.0 : exp(sigma - M);
    for (j = 0; j < n; ++j) {
        double e = exp(s[j] - M);
        int64_t off = kv_offset(kv, b, g, idx[j]);
        Z += e;
        for (d = 0; d < D; ++d)
            o[d] += e * kv_elem(kv, kv->v, kv->v_scale, off, d);
    }
    for (d = 0; d < D; ++d)
        o[d] /= Z;
    *lse = M + log(Z);
    free(s);
    free(idx);
    return 0;
}

/*
 * Full definition for a list of (row, head) selections.
 *   q         bf16 bits [n_rows, num_qo_heads, head_dim] (row-major)
 *   row_seq   [n_rows] sequence of each query row
 *   row_pos   [n_rows] position p of each query row
 *   seqlens   [B] keys held by each sequence
 *   sinks     [num_qo_heads] or NULL (no sink: sigma = -inf)
 *   sel_row, sel_head [n_sel]; out [n_sel, head_dim] fp64; lse [n_sel] fp64
 * Returns 0, or nonzero on a page table that points outside the pool.
 */
static int attend_sel(const void *q, int q_fmt, double q_scale, int32_t num_qo_heads,
                      const int32_t *row_seq, const int32_t *row_pos, const sao_kv_t *kv,
                      const int32_t *seqlens, const float *sinks, int32_t window, double sm_scale,
                      const int32_t *sel_row, const int32_t *sel_head, int64_t n_sel,
                      int32_t j_lo, int32_t j_hi, double *out, double *lse)
{
    const int D = kv->head_dim;
    const int G = num_qo_heads / kv->num_kv_heads;
    int64_t i;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (i = 0; i < n_sel; ++i) {
        int r = sel_row[i], h = sel_head[i];
        int b = row_seq[r];
        double sigma = sinks ? (double)sinks[h] : -INFINITY;
        const int64_t qoff = ((int64_t)r * num_qo_heads + h) * D;
        sao_qrow_t qrow;
        qrow.row = q_fmt == 0 ? (const void *)((const uint16_t *)q + qoff) : (const void *)((const uint8_t *)q + qoff);
        qrow.fmt = q_fmt;
        qrow.scale = q_scale;
        bad |= attend_one(&qrow, kv, b, h / G, row_pos[r], seqlens[b], window, sm_scale,
                          sigma, sinks != NULL, j_lo, j_hi, out + i * D, lse + i);
    }
    return bad;
}

int sao_attend(const uint16_t *q, int32_t n_rows, int32_t num_qo_heads,
               const int32_t *row_seq, const int32_t *row_pos,
               const sao_kv_t *kv, const int32_t *seqlens,
               const float *sinks, int32_t window, double sm_scale,
               const int32_t *sel_row, const int32_t *sel_head, int64_t n_sel,
               double *out, double *lse)
{
    (void)n_rows;
    return attend_sel(q, 0, 1.0, num_qo_heads, row_seq, row_pos, kv, seqlens, sinks, window, sm_scale,
                      sel_row, sel_head, n_sel, 0, 0x7fffffff, out, lse);
}

/*
 * sao_attend with the query given as E4M3 codes: element value = code *
 * q_scale (vLLM "GPT-OSS optimisations on NVIDIA Blackwell": part of the
 * attention runs in FP8).  Everything else is sao_attend.
 */
int sao_attend_q8(const uint8_t *q, double q_scale, int32_t n_rows, int32_t num_qo_heads,
                  const int32_t *row_seq, const int32_t *row_pos,
                  const sao_kv_t *kv, const int32_t *seqlens,
                  const float *sinks, int32_t window, double sm_scale,
                  const int32_t *sel_row, const int32_t *sel_head, int64_t n_sel,
                  double *out, double *lse)
{
    (void)n_rows;
    return attend_sel(q, 1, q_scale, num_qo_heads, row_seq, row_pos, kv, seqlens, sinks, window, sm_scale,
                      sel_row, sel_head, n_sel, 0, 0x7fffffff, out, lse);
}

/*
 * The same definition restricted to keys j in [j_lo, j_hi) (on top of the
 * causal/window set), with the sink only when `sinks` is given: the partial
 * state of one sequence chunk.  With sinks == NULL it is the sink-free state
 * (o, lse) that a chunk contributes to the merge.
 */
int sao_attend_range(const uint16_t *q, int32_t n_rows, int32_t num_qo_heads,
                     const int32_t *row_seq, const int32_t *row_pos,
                     const sao_kv_t *kv, const int32_t *seqlens,
                     const float *sinks, int32_t window, double sm_scale,
                     const int32_t *sel_row, const int32_t *sel_head, int64_t n_sel,
                     int32_t j_lo, int32_t j_hi, double *out, double *lse)
{
    (void)n_rows;
    return attend_sel(q, 0, 1.0, num_qo_heads, row_seq, row_pos, kv, seqlens, sinks, window, sm_scale,
                      sel_row, sel_head, n_sel, j_lo, j_hi, out, lse);
}

/*
 * Merge of partial states (o_s, lse_s), s = 0..S-1, with the sink counted once:
 *   M   = max(sigma, max_s lse_s)
 *   Z   = exp(sigma - M) + sum_s exp(lse_s - M)
 *   out = sum_s exp(lse_s - M) o_s / Z
 *   lse = M + log(Z)
 * o_part [S, N, H, D], lse_part [S, N, H] (fp64); sinks [H] or NULL;
 * out [N, H, D]; lse_out [N, H].  A partial with lse = -inf carries no weight.
 * Source: "GPT-OSS on day 0", "Sink Attention": with the softmax split into
 * chunks along the sequence, the sink enters once.
 */
void sao_merge(const double *o_part, const double *lse_part, int32_t S, int64_t N,
               int32_t H, int32_t D, const float *sinks, double *out, double *lse_out)
{
    int64_t nh;
#pragma omp parallel for schedule(static)
    for (nh = 0; nh < N * H; ++nh) {
        int h = (int)(nh % H);
        double sigma = sinks ? (double)sinks[h] : -INFINITY;
        double M = sigma, Z;
        int s, d;
        double *o = out + nh * D;
        for (s = 0; s < S; ++s) {
            double l = lse_part[(int64_t)s * N * H + nh];
            if (l > M)
                M = l;
        }
        for (d = 0; d < D; ++d)
            o[d] = 0.0;
        if (M == -INFINITY) {
            lse_out[nh] = -INFINITY;
            continue;
        }
        Z = (sigma == -INFINITY) ? 0.0 : exp(sigma - M);
        for (s = 0; s < S; ++s) {
            double l = lse_part[(int64_t)s * N * H + nh];
            double w;
            if (l == -INFINITY)
                continue;
            w = exp(l - M);
            Z += w;
            for (d = 0; d < D; ++d)
                o[d] += w * o_part[((int64_t)s * N * H + nh) * D + d];
        }
        for (d = 0; d < D; ++d)
            o[d] /= Z;
        lse_out[nh] = M + log(Z);
    }
}

/*
 * Chunked form: the visible keys of each selection are cut into chunks
 * [c0 + s*chunk, c0 + (s+1)*chunk), s = 0..S-1, where c0 is the first visible
 * key; every chunk gives a sink-free partial state (o_s, lse_s) and sao_merge
 * adds the sink once.  Must equal sao_attend for every chunk size.
 * part_o [S, n_sel, D] and part_lse [S, n_sel] are caller scratch.
 */
int sao_attend_split(const uint16_t *q, int32_t n_rows, int32_t num_qo_heads,
                     const int32_t *row_seq, const int32_t *row_pos,
                     const sao_kv_t *kv, const int32_t *seqlens,
                     const float *sinks, int32_t window, double sm_scale,
                     const int32_t *sel_row, const int32_t *sel_head, int64_t n_sel,
                     int32_t num_chunks, int32_t chunk,
                     double *part_o, double *part_lse, double *out, double *lse)
{
    const int D = kv->head_dim;
    const int G = num_qo_heads / kv->num_kv_heads;
    int64_t i;
    int bad = 0;
    float *sel_sinks = NULL;
    (void)n_rows;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (i = 0; i < n_sel; ++i) {
        int r = sel_row[i], h = sel_head[i];
        int b = row_seq[r], p = row_pos[r], L = seqlens[b];
        int first = window > 0 ? p - window + 1 : 0;
        int s;
        sao_qrow_t qrow;
        qrow.row = q + ((int64_t)r * num_qo_heads + h) * D;
        qrow.fmt = 0;
        qrow.scale = 1.0;
        if (first < 0)
            first = 0;
        for (s = 0; s < num_chunks; ++s) {
            int lo = first + s * chunk;
            bad |= attend_one(&qrow, kv, b, h / G, p, L, window, sm_scale, 0.0, 0,
                              lo, lo + chunk, part_o + ((int64_t)s * n_sel + i) * D,
                              part_lse + (int64_t)s * n_sel + i);
        }
    }
    if (bad)
        return bad;
    /* merge row by row: an [N = 1, H = 1] grid whose sink is the row's own */
    if (sinks) {
        sel_sinks = (float *)malloc(sizeof(float) * (size_t)(n_sel > 0 ? n_sel : 1));
        if (!sel_sinks)
            return 2;
        for (i = 0; i < n_sel; ++i)
            sel_sinks[i] = sinks[sel_head[i]];
    }
    for (i = 0; i < n_sel; ++i) {
        double *po = (double *)malloc(sizeof(double) * (size_t)num_chunks * D);
        double *pl = (double *)malloc(sizeof(double) * (size_t)num_chunks);
        int s;
        if (!po || !pl) {
            free(po);
            free(pl);
            free(sel_sinks);
            return 2;
        }
        for (s = 0; s < num_chunks; ++s) {
            memcpy(po + (int64_t)s * D, part_o + ((int64_t)s * n_sel + i) * D, sizeof(double) * D);
            pl[s] = part_lse[(int64_t)s * n_sel + i];
        }
        sao_merge(po, pl, num_chunks, 1, 1, D, sinks ? sel_sinks + i : NULL, out + i * D, lse + i);
        free(po);
        free(pl);
    }
    free(sel_sinks);
    return 0;
}

/* Array forms of the two decoders, for the decoder pins. */
void sao_bf16_array(const uint16_t *bits, int64_t n, double *out)
{
    int64_t i;
    for (i = 0; i < n; ++i)
        out[i] = sao_bf16_to_f64(bits[i]);
}

void sao_e4m3_array(const uint8_t *codes, int64_t n, double *out)
{
    int64_t i;
    for (i = 0; i < n; ++i)
        out[i] = sao_e4m3_to_f64(codes[i]);
}

int sao_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads the next parallel loops use (timing only; results do not depend on it). */
void sao_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}
