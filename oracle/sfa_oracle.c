/*
 * sfa_oracle.c -- the parity oracle for indexer-selected block-sparse attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls this file:
 * only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg do.  It shares no
 * code, header, table or helper with the CUDA library.
 *
 * Plain, slow and obviously correct: every quantity is computed in double precision from
 * the (exactly representable) input values, straight from the definition, with no
 * blocking, fusion or reordering beyond what the definition states.
 *
 * Sources (the pages this restates):
 *  [QSA]  llama.cpp commit "model: add Qwen3.8-Flash-Next (qwen4exp)", the paragraphs on
 *         the QSA indexer: one mean-pooled key per block of compress_ratio tokens is scored,
 *         the best blocks within a budget are kept together with the tail that does not
 *         fill a block; the indexer key cache holds raw keys (pooling precedes norm and
 *         rotation); each head's dot product is rectified before the sum over heads; the
 *         graph expands block scores to tokens so the cut lands on a block boundary.
 *  [SFA]  llama.cpp PR #27970 "CUDA + ggml: add sparse-fa for DSV4/GLM": attention over a
 *         sparse K/V set with V a view of the first DV dims of K, no ALiBi, no softcap,
 *         index rows padded with -1.
 *
 * Readings where the pages are silent (each one is listed with its reason in the design
 * notes): indexer_top_k counts blocks; a block counts for query i only when all of its
 * tokens are at positions <= p_i; the tail is [B_i*cr, p_i]; ties at the cut go to the
 * lower block index; the indexer has no extra scale; head h reads KV head h / (H_q/H_kv).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------------------ */
/* Step 1 -- block mean pooling of the raw index keys [QSA, indexer paragraph].
 *   kbar_b[d] = (1/cr) * sum_{t = b*cr}^{b*cr + cr - 1} X[t][d],   b = 0 .. n_blk-1
 * X is one sequence's index-key cache, row-major [n_tok][d_idx]; n_blk*cr <= n_tok.     */
void sfa_oracle_pool(const float *X, int64_t n_blk, int d_idx, int cr, double *kbar)
{
    for (int64_t b = 0; b < n_blk; ++b) {
        for (int d = 0; d < d_idx; ++d) {
            double sum = 0.0;
            for (int t = 0; t < cr; ++t)
                sum += (double)X[(b * cr + t) * (int64_t)d_idx + d];
            kbar[b * d_idx + d] = sum / (double)cr;
        }
    }
}

/* ------------------------------------------------------------------------------------ */
/* Step 1, paged cell layout [QSA paragraph that computes every layout-dependent input on the
 * host and cuts blocks on positions, so nothing assumes a contiguous cache; "support a
 * non-unified KV cache in QSA": a cell means a different token in each stream, so the maps
 * are kept per stream].  Position t's raw key is row cell_of[t] of the flat cell array
 * X[n_cells][d_idx] (cell_of is one stream's map); blocks are still cuts of the positions:
 *   kbar_b[d] = (1/cr) * sum_{t = b*cr}^{b*cr + cr - 1} X[cell_of[t]][d]
 * Returns 0, or -1 when a map entry read lies outside [0, n_cells).                       */
int sfa_oracle_pool_cells(const float *X, int64_t n_cells, const int32_t *cell_of,
                          int64_t n_blk, int d_idx, int cr, double *kbar)
{
    for (int64_t t = 0; t < n_blk * cr; ++t)
        if (cell_of[t] < 0 || cell_of[t] >= n_cells) return -1;
    for (int64_t b = 0; b < n_blk; ++b) {
        for (int d = 0; d < d_idx; ++d) {
            double sum = 0.0;
            for (int t = 0; t < cr; ++t)
                sum += (double)X[(int64_t)cell_of[b * cr + t] * d_idx + d];
            kbar[b * d_idx + d] = sum / (double)cr;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------------------ */
/* Step 1b -- the norm and the rotation of the pooled keys [QSA, indexer key cache paragraph:
 * the cache holds raw keys because pooling precedes the norm and the rotation; the indexer
 * ropes with the main attention's rotary width].  In place on kbar[n_blk][d_idx]; the pages
 * name neither the norm nor the rotary pairing nor a block's position, so each is a choice
 * (the readings are listed in the design notes):
 *   norm_kind 0: none;  1: RMS norm   y_d = x_d / sqrt(mean_e x_e^2 + eps) * gamma_d;
 *              2: layer norm         y_d = (x_d - mu) / sqrt(mean_e (x_e - mu)^2 + eps) * gamma_d + beta_d
 *   rotation of the first n_rot dims at position p = b * cr + pos_offset, pair j
 *   (0 <= j < n_rot/2) turned by theta_j = p * rope_base^(-2j / n_rot):
 *     rope_neox 1: the pair (j, j + n_rot/2);  0: the pair (2j, 2j + 1)
 *     (x_a, x_b) -> (x_a cos theta - x_b sin theta, x_a sin theta + x_b cos theta)        */
void sfa_oracle_key_transform(double *kbar, int64_t n_blk, int d_idx, int cr, int norm_kind,
                              const float *gamma, const float *beta, double eps, int n_rot,
                              double rope_base, int rope_neox, int64_t pos_offset)
{
    for (int64_t b = 0; b < n_blk; ++b) {
        double *x = kbar + b * d_idx;
        if (norm_kind == 1) {
            double ss = 0.0;
            for (int d = 0; d < d_idx; ++d) ss += x[d] * x[d];
            const double r = sqrt(ss / d_idx + eps);
            for (int d = 0; d < d_idx; ++d) x[d] = x[d] / r * (double)gamma[d];
        } else if (norm_kind == 2) {
            double mu = 0.0;
            for (int d = 0; d < d_idx; ++d) mu += x[d];
            mu /= d_idx;
            double var = 0.0;
            for (int d = 0; d < d_idx; ++d) var += (x[d] - mu) * (x[d] - mu);
            const double r = sqrt(var / d_idx + eps);
            for (int d = 0; d < d_idx; ++d) x[d] = (x[d] - mu) / r * (double)gamma[d] + (double)beta[d];
        }
        const double p = (double)(b * cr + pos_offset);
        for (int j = 0; j < n_rot / 2; ++j) {
            const double theta = p * pow(rope_base, -2.0 * j / n_rot);
            const int ia = rope_neox ? j : 2 * j, ib = rope_neox ? j + n_rot / 2 : 2 * j + 1;
            const double xa = x[ia], xb = x[ib];
            x[ia] = xa * cos(theta) - xb * sin(theta);
            x[ib] = xa * sin(theta) + xb * cos(theta);
        }
    }
}

/* ------------------------------------------------------------------------------------ */
/* KV cache quantization, q8_0 [qwen4exp commit: the QSA attention path takes a quantized KV
 * cache; the pages do not spell the format out, and q8_0 is the 8-bit block format of the
 * llama.cpp caches they describe].  Each row of d elements (d a multiple of 32) is cut into
 * blocks of 32 consecutive elements.  Per block:
 *   amax = max_j |x_j|,  delta = amax / 127                        (binary32 division)
 *   q_j  = x_j / delta rounded half away from zero, or 0 when delta = 0   (binary32)
 *   the stored scale s = delta rounded to binary16 (nearest, ties to even)
 * and the value a quantized element stands for is s * q_j.  The codes are taken with the
 * unrounded delta; only the stored scale is binary16.                                     */

/* binary16 bits of a finite or infinite float, rounded to nearest with ties to even (IEEE
 * 754): subnormals in units of 2^-24, normals with a 10-bit fraction, overflow to infinity. */
static uint16_t fp16_bits(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    const uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)(sign | 0x7E00u);   /* NaN */
    const double a = fabs((double)f);
    if (a < 6.103515625e-05) {                       /* below 2^-14: subnormal or zero */
        const double units = nearbyint(a * 16777216.0);   /* a / 2^-24, exact, then RNE */
        return (uint16_t)(sign | (uint16_t)units);        /* 1024 units is 2^-14: 0x0400 */
    }
    int e;
    const double m = frexp(a, &e);                   /* a = m * 2^e, 0.5 <= m < 1 */
    double frac = nearbyint(ldexp(m, 11));           /* 1024 .. 2048 after rounding */
    int E = e - 1 + 15;                              /* biased binary16 exponent */
    if (frac == 2048.0) {
        frac = 1024.0;
        E += 1;
    }
    if (E >= 31) return (uint16_t)(sign | 0x7C00u);  /* infinity */
    return (uint16_t)(sign | (uint16_t)(E << 10) | (uint16_t)((int)frac - 1024));
}

/* The value of binary16 bits (IEEE 754). */
static float fp16_value(uint16_t h)
{
    const int E = (h >> 10) & 0x1F, M = h & 0x3FF;
    double v;
    if (E == 0) v = ldexp((double)M, -24);
    else if (E == 31) v = M ? NAN : INFINITY;
    else v = ldexp((double)(M | 0x400), E - 25);
    return (float)((h & 0x8000u) ? -v : v);
}

/* x[n_rows][d] -> codes q[n_rows][d] and scale bits[n_rows][d/32].  Returns -1 when a scale
 * overflows binary16 (amax above ~8.3e6), else 0.                                          */
int sfa_oracle_quantize_q8_0(const float *x, int64_t n_rows, int d, int8_t *q, uint16_t *scale)
{
    int rc = 0;
    for (int64_t i = 0; i < n_rows; ++i) {
        for (int b = 0; b < d / 32; ++b) {
            const float *xb = x + i * d + b * 32;
            int8_t *qb = q + i * d + b * 32;
            float amax = 0.0f;
            for (int j = 0; j < 32; ++j)
                if (fabsf(xb[j]) > amax) amax = fabsf(xb[j]);
            const float delta = amax / 127.0f;
            for (int j = 0; j < 32; ++j)
                qb[j] = delta == 0.0f ? 0 : (int8_t)roundf(xb[j] / delta);
            const uint16_t sb = fp16_bits(delta);
            scale[i * (d / 32) + b] = sb;
            if ((sb & 0x7FFFu) == 0x7C00u) rc = -1;
        }
    }
    return rc;
}

/* The values the codes stand for: out[i][j] = s(i, j / 32) * q[i][j] (exact in binary32).  */
void sfa_oracle_dequantize_q8_0(const int8_t *q, const uint16_t *scale, int64_t n_rows, int d,
                                float *out)
{
    for (int64_t i = 0; i < n_rows; ++i)
        for (int j = 0; j < d; ++j)
            out[i * d + j] = fp16_value(scale[i * (d / 32) + j / 32]) * (float)q[i * d + j];
}

/* binary16 bits of each float (exposed so the conversion can be checked on its own).       */
void sfa_oracle_fp16_bits(const float *x, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = fp16_bits(x[i]);
}

/* ------------------------------------------------------------------------------------ */
/* Step 2 -- indexer score of every complete block [QSA, ReLU paragraph].
 *   s_b = sum_j w_j * max(0, q_j . kbar_b)
 * q_idx is [h_idx][d_idx] for one query token, w is [h_idx].                              */
void sfa_oracle_index_scores(const float *q_idx, const float *w, int h_idx, int d_idx,
                             const double *kbar, int64_t n_blk, double *score)
{
    for (int64_t b = 0; b < n_blk; ++b) {
        double s = 0.0;
        for (int j = 0; j < h_idx; ++j) {
            double dot = 0.0;
            for (int d = 0; d < d_idx; ++d)
                dot += (double)q_idx[j * d_idx + d] * kbar[b * d_idx + d];
            double relu = dot > 0.0 ? dot : 0.0;
            s += (double)w[j] * relu;
        }
        score[b] = s;
    }
}

/* ------------------------------------------------------------------------------------ */
/* Step 3 -- the budget rule [QSA, budget paragraph].
 * If every block fits the budget (n_blk <= top_k) all blocks are kept.  Otherwise all
 * blocks are fully sorted by (score descending, block index ascending) and the first
 * top_k are kept.  The kept ids are written ascending and the row is padded with -1
 * (the padding convention of [SFA]).  Returns the number kept.                           */
struct scored_block { double s; int64_t b; };

static int by_score_then_index(const void *pa, const void *pb)
{
    const struct scored_block *a = pa, *b = pb;
    if (a->s > b->s) return -1;
    if (a->s < b->s) return 1;
    return (a->b < b->b) ? -1 : (a->b > b->b);
}

static int ascending_i32(const void *pa, const void *pb)
{
    int32_t a = *(const int32_t *)pa, b = *(const int32_t *)pb;
    return (a > b) - (a < b);
}

int sfa_oracle_select(const double *score, int64_t n_blk, int top_k, int32_t *sel)
{
    int n_sel;
    if (n_blk <= top_k) {
        n_sel = (int)n_blk;
        for (int i = 0; i < n_sel; ++i) sel[i] = i;
    } else {
        struct scored_block *all = malloc(sizeof(*all) * (size_t)n_blk);
        for (int64_t b = 0; b < n_blk; ++b) { all[b].s = score[b]; all[b].b = b; }
        qsort(all, (size_t)n_blk, sizeof(*all), by_score_then_index);
        n_sel = top_k;
        for (int i = 0; i < n_sel; ++i) sel[i] = (int32_t)all[i].b;
        free(all);
        qsort(sel, (size_t)n_sel, sizeof(int32_t), ascending_i32);
    }
    for (int i = n_sel; i < top_k; ++i) sel[i] = -1;
    return n_sel;
}

/* ------------------------------------------------------------------------------------ */
/* Step 4 -- the attended set as an explicit mask over positions 0..p [QSA, budget
 * paragraph]: every token of a kept block, plus the tail [B*cr, p] of tokens that do not
 * form a complete block, B = floor((p+1)/cr).  top_k <= 0 means dense: all of 0..p.      */
void sfa_oracle_mask(int64_t p, int cr, const int32_t *sel, int n_sel, int dense,
                     uint8_t *mask)
{
    const int64_t n_vis = p + 1;
    if (dense) {
        for (int64_t t = 0; t < n_vis; ++t) mask[t] = 1;
        return;
    }
    const int64_t n_blk = n_vis / cr;
    for (int64_t t = 0; t < n_vis; ++t) mask[t] = 0;
    for (int i = 0; i < n_sel; ++i)
        for (int64_t t = (int64_t)sel[i] * cr; t < (int64_t)sel[i] * cr + cr; ++t) mask[t] = 1;
    for (int64_t t = n_blk * cr; t < n_vis; ++t) mask[t] = 1;
}

/* ------------------------------------------------------------------------------------ */
/* Step 4, windowed -- the attended set when a contiguous run of the most recent keys is
 * attended densely beside the selected blocks [PR #27970 review discussion: dense attention
 * over the continuous block of keys, sparse attention over the selected keys, the two
 * results combined].  Reading: the run is the window of the `window` most recent positions
 * p - window + 1 .. p (clipped at 0); the attended set is its union with the kept blocks and
 * the tail.  window = 0 gives the plain set above; window >= p + 1 gives every position.    */
void sfa_oracle_mask_window(int64_t p, int cr, const int32_t *sel, int n_sel, int64_t window,
                            uint8_t *mask)
{
    sfa_oracle_mask(p, cr, sel, n_sel, 0, mask);
    int64_t first = p - window + 1;
    if (first < 0) first = 0;
    for (int64_t t = first; t <= p; ++t) mask[t] = 1;
}

/* ------------------------------------------------------------------------------------ */
/* Step 5 -- exact softmax attention over the masked tokens [SFA].
 * For head h (KV head g = h / (h_q / h_kv)):
 *   l_t = scale * q_h . K[t][g],   O_h = sum_t exp(l_t - m) V[t][g] / sum_t exp(l_t - m),
 *   lse_h = m + log(sum_t exp(l_t - m)),   m = max over masked t of l_t.
 * Token t's K row is K + row(t)*k_row_stride + g*dkq where row(t) = t, or tok_row[t] when
 * tok_row is given (so callers may pass only the rows that the mask touches).  V == NULL
 * means V[t][g] is the first dv entries of K[t][g].                                      */
void sfa_oracle_attend(const float *q, int h_q, int h_kv, int dkq, int dv, double scale,
                       const float *K, int64_t k_row_stride, const float *V,
                       int64_t v_row_stride, const int64_t *tok_row, const uint8_t *mask,
                       int64_t n_vis, double *out, double *lse)
{
    const int group = h_q / h_kv;
    double *logit = malloc(sizeof(double) * (size_t)(n_vis > 0 ? n_vis : 1));
    for (int h = 0; h < h_q; ++h) {
        const int g = h / group;
        const float *qh = q + (int64_t)h * dkq;
        double m = -INFINITY;
        for (int64_t t = 0; t < n_vis; ++t) {
            if (!mask[t]) continue;
            const int64_t r = tok_row ? tok_row[t] : t;
            const float *kt = K + r * k_row_stride + (int64_t)g * dkq;
            double dot = 0.0;
            for (int d = 0; d < dkq; ++d) dot += (double)qh[d] * (double)kt[d];
            logit[t] = scale * dot;
            if (logit[t] > m) m = logit[t];
        }
        double denom = 0.0;
        double *oh = out + (int64_t)h * dv;
        for (int d = 0; d < dv; ++d) oh[d] = 0.0;
        for (int64_t t = 0; t < n_vis; ++t) {
            if (!mask[t]) continue;
            const int64_t r = tok_row ? tok_row[t] : t;
            const float *vt = V ? V + r * v_row_stride + (int64_t)g * dv
                                : K + r * k_row_stride + (int64_t)g * dkq;
            const double e = exp(logit[t] - m);
            denom += e;
            for (int d = 0; d < dv; ++d) oh[d] += e * (double)vt[d];
        }
        for (int d = 0; d < dv; ++d) oh[d] /= denom;
        if (lse) lse[h] = m + log(denom);
    }
    free(logit);
}

/* ------------------------------------------------------------------------------------ */
/* The whole method for a batch of query tokens, one query per task over n_threads
 * host threads.  Each query i belongs to sequence q_seq[i] at position q_pos[i] and sees
 * that sequence's tokens 0..q_pos[i] only.
 *
 * Layouts (row-major, contiguous):
 *   X     [n_seq][n_tok][d_idx]         raw index keys
 *   q_idx [n_q][h_idx][d_idx], w [n_q][h_idx]
 *   Q     [n_q][h_q][dkq]
 *   K     [n_seq][n_tok][h_kv][dkq],  V [n_seq][n_tok][h_kv][dv] or NULL
 * Outputs: sel [n_q][top_k] (-1 padded), n_sel [n_q], O [n_q][h_q][dv], lse [n_q][h_q],
 *   and, when score != NULL, score [n_q][score_stride] (entries b >= B_i untouched).
 * top_k <= 0 runs dense attention (sel / n_sel / score are then not written).            */
struct run_args {
    const float *X, *q_idx, *w, *Q, *K, *V;
    const int32_t *q_seq, *q_pos;
    int n_q, n_tok, h_idx, d_idx, cr, top_k, h_q, h_kv, dkq, dv;
    double scale;
    int32_t *sel, *n_sel;
    double *score;
    int64_t score_stride;
    double *O, *lse;
    int next;
    pthread_mutex_t lock;
};

static void run_one_query(struct run_args *a, int i)
{
    const int64_t s = a->q_seq[i], p = a->q_pos[i], n_vis = p + 1;
    const int dense = a->top_k <= 0;
    uint8_t *mask = malloc((size_t)n_vis);
    const float *Ks = a->K + s * (int64_t)a->n_tok * a->h_kv * a->dkq;
    const float *Vs = a->V ? a->V + s * (int64_t)a->n_tok * a->h_kv * a->dv : NULL;
    if (dense) {
        sfa_oracle_mask(p, a->cr, NULL, 0, 1, mask);
    } else {
        const int64_t n_blk = n_vis / a->cr;
        double *kbar = malloc(sizeof(double) * (size_t)(n_blk > 0 ? n_blk : 1) * a->d_idx);
        double *score = malloc(sizeof(double) * (size_t)(n_blk > 0 ? n_blk : 1));
        sfa_oracle_pool(a->X + s * (int64_t)a->n_tok * a->d_idx, n_blk, a->d_idx, a->cr, kbar);
        sfa_oracle_index_scores(a->q_idx + (int64_t)i * a->h_idx * a->d_idx,
                                a->w + (int64_t)i * a->h_idx, a->h_idx, a->d_idx, kbar, n_blk,
                                score);
        int32_t *sel = a->sel + (int64_t)i * a->top_k;
        a->n_sel[i] = sfa_oracle_select(score, n_blk, a->top_k, sel);
        if (a->score)
            for (int64_t b = 0; b < n_blk; ++b) a->score[i * a->score_stride + b] = score[b];
        sfa_oracle_mask(p, a->cr, sel, a->n_sel[i], 0, mask);
        free(kbar);
        free(score);
    }
    sfa_oracle_attend(a->Q + (int64_t)i * a->h_q * a->dkq, a->h_q, a->h_kv, a->dkq, a->dv,
                      a->scale, Ks, (int64_t)a->h_kv * a->dkq, Vs, (int64_t)a->h_kv * a->dv,
                      NULL, mask, n_vis, a->O + (int64_t)i * a->h_q * a->dv,
                      a->lse + (int64_t)i * a->h_q);
    free(mask);
}

static void *run_worker(void *p)
{
    struct run_args *a = p;
    for (;;) {
        pthread_mutex_lock(&a->lock);
        const int i = a->next++;
        pthread_mutex_unlock(&a->lock);
        if (i >= a->n_q) return NULL;
        run_one_query(a, i);
    }
}

void sfa_oracle_run(const float *X, const float *q_idx, const float *w, const float *Q,
                    const float *K, const float *V, const int32_t *q_seq, const int32_t *q_pos,
                    int n_q, int n_tok, int h_idx, int d_idx, int cr, int top_k, int h_q,
                    int h_kv, int dkq, int dv, double scale, int32_t *sel, int32_t *n_sel,
                    double *score, int64_t score_stride, double *O, double *lse, int n_threads)
{
    struct run_args a = {X, q_idx, w, Q, K, V, q_seq, q_pos, n_q, n_tok, h_idx, d_idx, cr,
                         top_k, h_q, h_kv, dkq, dv, scale, sel, n_sel, score, score_stride,
                         O, lse, 0, PTHREAD_MUTEX_INITIALIZER};
    if (n_threads < 1) n_threads = 1;
    if (n_threads > n_q) n_threads = n_q > 0 ? n_q : 1;
    pthread_t *tid = malloc(sizeof(pthread_t) * (size_t)n_threads);
    for (int t = 0; t < n_threads; ++t) pthread_create(&tid[t], NULL, run_worker, &a);
    for (int t = 0; t < n_threads; ++t) pthread_join(tid[t], NULL);
    free(tid);
}
