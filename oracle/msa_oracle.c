/*
 * msa_oracle.c -- plain, slow, obviously-correct CPU definition of the
 * MiniMax Sparse Attention (MSA) hot path.  TEST INFRASTRUCTURE ONLY: it is
 * the parity oracle for the CUDA library and is never on the product path.
 *
 * Everything here follows the definition written in "Sparse Attention ·
 * Part II" (mtreviso.github.io/blog/sparse-attention-2.html), section 3.2
 * "MiniMax's MSA", and the loss equation in that section.  Arithmetic is
 * fp64 throughout.  Inputs are bf16 bit patterns (uint16) widened exactly,
 * or, when compiled with -DORC_F64, fp64 values (used by the finite-
 * difference checks, which must perturb inputs by amounts bf16 cannot hold).
 * Block scores are rounded to fp32 once, and selection compares those fp32
 * values, so that selection ties and near-ties are decided the same way a
 * fp32 implementation decides them.
 *
 * Also here: the index projections of the detached hidden states and their
 * weight gradient (the detachment equation of section 3.2), and the dense
 * indexer warm-up loss of section 3.1 with its gradient.
 *
 * No blocking, fusion or reordering beyond the definition: every function
 * walks queries, heads and tokens in the obvious order.  Parallelism is an
 * OpenMP loop over independent (row, group) or (batch, group, chunk) items.
 *
 * Layouts (row-major, contiguous, "kv_rows" rows per batch entry in the
 * key-side tensors, kv_rows >= Nk):
 *   q      [B, Nq, Hq,  d]          k, v   [B, kv_rows, Hkv, d]
 *   q_idx  [B, Nq, Hkv, d_idx]      k_idx  [B, kv_rows, d_idx]
 *   d_o    like q
 * Query row i of batch b sits at absolute position pos = q_offset + i and
 * sees key j iff j <= pos.  Head h belongs to group r = h / (Hq/Hkv).
 * A "row id" is b*Nq + i.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int B, Nq, Nk, q_offset, Hq, Hkv, d, d_idx, block, topk;
    long long kv_rows;
    double scale, scale_idx;
} orc_shape;

#ifdef ORC_F64
typedef double orc_in;
static double bfv(orc_in x) { return x; }
#else
typedef uint16_t orc_in;
/* bf16 bit pattern -> exact double. */
static double bfv(orc_in x)
{
    uint32_t u = ((uint32_t)x) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}
#endif

static long long kvrows(const orc_shape *s) { return s->kv_rows > 0 ? s->kv_rows : s->Nk; }
static int nblocks(const orc_shape *s) { return (s->Nk + s->block - 1) / s->block; }

/* dot of a bf16 row with a bf16 row, in fp64 */
static double dot_bf(const orc_in *a, const orc_in *b, int n)
{
    double acc = 0.0;
    for (int e = 0; e < n; ++e) acc += bfv(a[e]) * bfv(b[e]);
    return acc;
}

/* ------------------------------------------------------------------------ */
/* Index branch: token scores and block max-pool (section 3.2).  Per query
 * and GQA group, the group's index query is dotted with the one index key
 * head that all groups share, over every causally visible token; a block's
 * score is the largest of its visible tokens' scores.
 * out_bs: [n_rows, Hkv, nb] fp32; blocks after the query's local block are
 * not visible and are written as -INFINITY.                                 */
int orc_block_scores(const orc_shape *s, const orc_in *q_idx, const orc_in *k_idx,
                     int n_rows, const long long *rows, float *out_bs)
{
    const int nb = nblocks(s);
    const long long KR = kvrows(s);
    #pragma omp parallel for schedule(dynamic, 1)
    for (long long t = 0; t < (long long)n_rows * s->Hkv; ++t) {
        const long long row = rows[t / s->Hkv];
        const int r = (int)(t % s->Hkv);
        const int b = (int)(row / s->Nq), i = (int)(row % s->Nq);
        const long long pos = (long long)s->q_offset + i;
        const orc_in *qi = q_idx + (((long long)b * s->Nq + i) * s->Hkv + r) * s->d_idx;
        float *bs = out_bs + t * nb;
        for (int c = 0; c < nb; ++c) {
            double best = -INFINITY;
            int any = 0;
            for (long long j = (long long)c * s->block; j < (long long)(c + 1) * s->block && j < s->Nk; ++j) {
                if (j > pos) break;
                const double sc = s->scale_idx * dot_bf(qi, k_idx + ((long long)b * KR + j) * s->d_idx, s->d_idx);
                if (!any || sc > best) best = sc;
                any = 1;
            }
            bs[c] = any ? (float)best : -INFINITY;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Top-k block selection (section 3.2).  The block holding the query always
 * takes one of the k slots; the remaining k-1 go to the best-scoring earlier
 * blocks.  Ranking is by fp32 block score, descending, ties to the lower
 * block index.  When the query sees at most k blocks, all of
 * them are kept.  Output per (row, group): block ids ascending, then -1.   */
typedef struct { float score; int c; } orc_cand;

static int cand_cmp(const void *pa, const void *pb)
{
    const orc_cand *a = (const orc_cand *)pa, *b = (const orc_cand *)pb;
    if (a->score > b->score) return -1;
    if (a->score < b->score) return 1;
    return (a->c < b->c) ? -1 : (a->c > b->c);
}

static int int_cmp(const void *pa, const void *pb)
{
    const int a = *(const int *)pa, b = *(const int *)pb;
    return (a > b) - (a < b);
}

int orc_select(const orc_shape *s, const float *bs, int n_rows, const long long *rows, int32_t *out_sel)
{
    const int nb = nblocks(s);
    const int k = s->topk;
    int err = 0;
    #pragma omp parallel for schedule(dynamic, 16)
    for (long long t = 0; t < (long long)n_rows * s->Hkv; ++t) {
        const long long row = rows[t / s->Hkv];
        const int i = (int)(row % s->Nq);
        const long long pos = (long long)s->q_offset + i;
        const int c0 = (int)(pos / s->block);
        int32_t *sel = out_sel + t * k;
        int chosen[64];
        int n = 0;
        if (k > 64) { err = 1; continue; }
        if (c0 + 1 <= k) {
            for (int c = 0; c <= c0; ++c) chosen[n++] = c;
        } else {
            orc_cand *cands = (orc_cand *)malloc(sizeof(orc_cand) * (size_t)c0);
            for (int c = 0; c < c0; ++c) { cands[c].score = bs[t * nb + c]; cands[c].c = c; }
            qsort(cands, (size_t)c0, sizeof(orc_cand), cand_cmp);
            chosen[n++] = c0;
            for (int m = 0; m < k - 1; ++m) chosen[n++] = cands[m].c;
            free(cands);
        }
        qsort(chosen, (size_t)n, sizeof(int), int_cmp);
        for (int m = 0; m < k; ++m) sel[m] = m < n ? chosen[m] : -1;
    }
    return err ? -1 : 0;
}

/* ------------------------------------------------------------------------ */
/* Token set T(i, r): all j <= pos whose block is among the selected ones.  */
static int token_set(const orc_shape *s, const int32_t *sel, long long pos, long long *tok)
{
    int n = 0;
    for (int m = 0; m < s->topk; ++m) {
        const int c = sel[m];
        if (c < 0) continue;
        for (long long j = (long long)c * s->block; j < (long long)(c + 1) * s->block && j < s->Nk; ++j) {
            if (j > pos) break;
            tok[n++] = j;
        }
    }
    return n;
}

/* Softmax of x[0..n) into p, returns the log-sum-exp (two passes: max, sum). */
static double softmax_lse(const double *x, int n, double *p)
{
    double m = -INFINITY;
    for (int t = 0; t < n; ++t) if (x[t] > m) m = x[t];
    double z = 0.0;
    for (int t = 0; t < n; ++t) z += exp(x[t] - m);
    for (int t = 0; t < n; ++t) p[t] = exp(x[t] - m) / z;
    return m + log(z);
}

/* ------------------------------------------------------------------------ */
/* Main branch (section 3.2).  Each query head of the group runs ordinary
 * softmax attention with its own logits over the visible tokens of the
 * selected blocks only, so the weights sum to one over that set (section 2
 * states that DSA and MSA normalise within the selection).
 * sel: [n_rows, Hkv, topk] for the listed rows.
 * out_o [n_rows, Hq, d], out_lse [n_rows, Hq] (natural log of the sum of
 * exp of the scaled logits).                                               */
int orc_sparse_fwd(const orc_shape *s, const orc_in *q, const orc_in *k, const orc_in *v,
                   const int32_t *sel, int n_rows, const long long *rows, double *out_o, double *out_lse)
{
    const int G = s->Hq / s->Hkv;
    const long long KR = kvrows(s);
    const int tmax = s->topk * s->block;
    #pragma omp parallel
    {
        long long *tok = (long long *)malloc(sizeof(long long) * (size_t)tmax);
        double *lg = (double *)malloc(sizeof(double) * (size_t)tmax);
        double *p = (double *)malloc(sizeof(double) * (size_t)tmax);
        #pragma omp for schedule(dynamic, 1)
        for (long long t = 0; t < (long long)n_rows * s->Hq; ++t) {
            const long long ri = t / s->Hq;
            const int h = (int)(t % s->Hq), r = h / G;
            const long long row = rows[ri];
            const int b = (int)(row / s->Nq), i = (int)(row % s->Nq);
            const long long pos = (long long)s->q_offset + i;
            const int n = token_set(s, sel + (ri * s->Hkv + r) * s->topk, pos, tok);
            const orc_in *qh = q + (((long long)b * s->Nq + i) * s->Hq + h) * s->d;
            for (int u = 0; u < n; ++u)
                lg[u] = s->scale * dot_bf(qh, k + (((long long)b * KR + tok[u]) * s->Hkv + r) * s->d, s->d);
            out_lse[t] = softmax_lse(lg, n, p);
            double *o = out_o + t * s->d;
            for (int e = 0; e < s->d; ++e) o[e] = 0.0;
            for (int u = 0; u < n; ++u) {
                const orc_in *vj = v + (((long long)b * KR + tok[u]) * s->Hkv + r) * s->d;
                for (int e = 0; e < s->d; ++e) o[e] += p[u] * bfv(vj[e]);
            }
        }
        free(tok); free(lg); free(p);
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* KL alignment loss (section 3.2, the L_KL equation).  For query i, group r:
 * teacher P = mean over the group's heads of each head's softmax over the
 * selected token set; student P_idx = softmax of the index scores on the
 * same set; KL(P || P_idx) = sum_j P_j (log P_j - log P_idx_j), 0 log 0 = 0.
 * out_lse_idx [n_rows, Hkv] = log sum_j exp(s_j); out_kl [n_rows, Hkv].
 * The scalar loss is kl_coef / (B Nq Hkv) times the sum of out_kl over all
 * rows (the caller sums when it passes every row).                         */
int orc_kl(const orc_shape *s, const orc_in *q, const orc_in *k, const orc_in *q_idx,
           const orc_in *k_idx, const int32_t *sel, int n_rows, const long long *rows,
           double *out_lse_idx, double *out_kl)
{
    const int G = s->Hq / s->Hkv;
    const long long KR = kvrows(s);
    const int tmax = s->topk * s->block;
    #pragma omp parallel
    {
        long long *tok = (long long *)malloc(sizeof(long long) * (size_t)tmax);
        double *lg = (double *)malloc(sizeof(double) * (size_t)tmax);
        double *p = (double *)malloc(sizeof(double) * (size_t)tmax);
        double *pt = (double *)malloc(sizeof(double) * (size_t)tmax);
        double *ps = (double *)malloc(sizeof(double) * (size_t)tmax);
        #pragma omp for schedule(dynamic, 1)
        for (long long t = 0; t < (long long)n_rows * s->Hkv; ++t) {
            const long long ri = t / s->Hkv;
            const int r = (int)(t % s->Hkv);
            const long long row = rows[ri];
            const int b = (int)(row / s->Nq), i = (int)(row % s->Nq);
            const long long pos = (long long)s->q_offset + i;
            const int n = token_set(s, sel + t * s->topk, pos, tok);
            for (int u = 0; u < n; ++u) pt[u] = 0.0;
            for (int g = 0; g < G; ++g) {
                const int h = r * G + g;
                const orc_in *qh = q + (((long long)b * s->Nq + i) * s->Hq + h) * s->d;
                for (int u = 0; u < n; ++u)
                    lg[u] = s->scale * dot_bf(qh, k + (((long long)b * KR + tok[u]) * s->Hkv + r) * s->d, s->d);
                softmax_lse(lg, n, p);
                for (int u = 0; u < n; ++u) pt[u] += p[u] / G;
            }
            const orc_in *qi = q_idx + (((long long)b * s->Nq + i) * s->Hkv + r) * s->d_idx;
            for (int u = 0; u < n; ++u)
                lg[u] = s->scale_idx * dot_bf(qi, k_idx + ((long long)b * KR + tok[u]) * s->d_idx, s->d_idx);
            out_lse_idx[t] = softmax_lse(lg, n, ps);
            double kl = 0.0;
            for (int u = 0; u < n; ++u)
                if (pt[u] > 0.0) kl += pt[u] * (log(pt[u]) - log(ps[u]));
            out_kl[t] = kl;
        }
        free(tok); free(lg); free(p); free(pt); free(ps);
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Backward.  Loss = sum(d_o . O) + L_KL.  Main gradients: the textbook
 * softmax-attention backward over the selected set, per head.  Index
 * gradients: the direct derivative of KL(P || softmax(s)) in s, which is
 * softmax(s) - P, times kl_coef/(B Nq Hkv), chained through
 * s = scale_idx q_idx . k_idx.  The teacher is a constant (stopgrad) and the
 * selection is piecewise constant, so neither carries gradient (section
 * 3.2, on the two detachments).
 *
 * Work for one (row, group): it fills, per head, P and dS on the token set,
 * and the index-side dsigma.  Two drivers use it:
 *   orc_bwd_rows: dq, dq_idx for listed rows  (query-side gradients)
 *   orc_bwd_keys: dk, dv, dk_idx for listed key blocks (key-side)          */
typedef struct {
    long long *tok;
    double *lg, *p, *dsc, *pt, *ps, *dsig;   /* p, dsc: [G][tmax] */
} orc_bwd_scratch;

static void bwd_scratch_alloc(orc_bwd_scratch *w, int G, int tmax)
{
    w->tok = (long long *)malloc(sizeof(long long) * (size_t)tmax);
    w->lg = (double *)malloc(sizeof(double) * (size_t)tmax);
    w->p = (double *)malloc(sizeof(double) * (size_t)tmax * G);
    w->dsc = (double *)malloc(sizeof(double) * (size_t)tmax * G);
    w->pt = (double *)malloc(sizeof(double) * (size_t)tmax);
    w->ps = (double *)malloc(sizeof(double) * (size_t)tmax);
    w->dsig = (double *)malloc(sizeof(double) * (size_t)tmax);
}

static void bwd_scratch_free(orc_bwd_scratch *w)
{
    free(w->tok); free(w->lg); free(w->p); free(w->dsc); free(w->pt); free(w->ps); free(w->dsig);
}

/* Returns n = |T|.  After the call, for head g of the group and token u:
 *   p[g*tmax+u]   = main softmax weight,
 *   dsc[g*tmax+u] = dL/dlogit (before the 'scale' chain factor),
 *   dsig[u]       = dL_KL/ds_u.                                            */
static int bwd_row_group(const orc_shape *s, const orc_in *q, const orc_in *k, const orc_in *v,
                         const orc_in *d_o, const orc_in *q_idx, const orc_in *k_idx,
                         const int32_t *sel_rg, double kl_coef, int b, int i, int r, orc_bwd_scratch *w)
{
    const int G = s->Hq / s->Hkv;
    const long long KR = kvrows(s);
    const int tmax = s->topk * s->block;
    const long long pos = (long long)s->q_offset + i;
    const int n = token_set(s, sel_rg, pos, w->tok);
    for (int u = 0; u < n; ++u) w->pt[u] = 0.0;
    for (int g = 0; g < G; ++g) {
        const int h = r * G + g;
        const orc_in *qh = q + (((long long)b * s->Nq + i) * s->Hq + h) * s->d;
        const orc_in *doh = d_o + (((long long)b * s->Nq + i) * s->Hq + h) * s->d;
        double *p = w->p + (size_t)g * tmax, *ds = w->dsc + (size_t)g * tmax;
        for (int u = 0; u < n; ++u)
            w->lg[u] = s->scale * dot_bf(qh, k + (((long long)b * KR + w->tok[u]) * s->Hkv + r) * s->d, s->d);
        softmax_lse(w->lg, n, p);
        /* dP_u = dO . v_u ; D = sum_u P_u dP_u ; dS_u = P_u (dP_u - D) */
        double D = 0.0;
        for (int u = 0; u < n; ++u) {
            ds[u] = dot_bf(doh, v + (((long long)b * KR + w->tok[u]) * s->Hkv + r) * s->d, s->d);
            D += p[u] * ds[u];
        }
        for (int u = 0; u < n; ++u) ds[u] = p[u] * (ds[u] - D);
        for (int u = 0; u < n; ++u) w->pt[u] += p[u] / G;
    }
    const orc_in *qi = q_idx + (((long long)b * s->Nq + i) * s->Hkv + r) * s->d_idx;
    for (int u = 0; u < n; ++u)
        w->lg[u] = s->scale_idx * dot_bf(qi, k_idx + ((long long)b * KR + w->tok[u]) * s->d_idx, s->d_idx);
    softmax_lse(w->lg, n, w->ps);
    const double coef = kl_coef / ((double)s->B * s->Nq * s->Hkv);
    for (int u = 0; u < n; ++u) w->dsig[u] = coef * (w->ps[u] - w->pt[u]);
    return n;
}

/* dq [n_rows, Hq, d], dq_idx [n_rows, Hkv, d_idx]; sel covers every row of
 * the problem: [B, Hkv, Nq, topk] (the library's layout).                  */
int orc_bwd_rows(const orc_shape *s, const orc_in *q, const orc_in *k, const orc_in *v,
                 const orc_in *d_o, const orc_in *q_idx, const orc_in *k_idx,
                 const int32_t *sel, double kl_coef, int n_rows, const long long *rows,
                 double *dq, double *dq_idx)
{
    const int G = s->Hq / s->Hkv;
    const long long KR = kvrows(s);
    const int tmax = s->topk * s->block;
    #pragma omp parallel
    {
        orc_bwd_scratch w;
        bwd_scratch_alloc(&w, G, tmax);
        #pragma omp for schedule(dynamic, 1)
        for (long long t = 0; t < (long long)n_rows * s->Hkv; ++t) {
            const long long ri = t / s->Hkv;
            const int r = (int)(t % s->Hkv);
            const long long row = rows[ri];
            const int b = (int)(row / s->Nq), i = (int)(row % s->Nq);
            const int32_t *sr = sel + (((long long)b * s->Hkv + r) * s->Nq + i) * s->topk;
            const int n = bwd_row_group(s, q, k, v, d_o, q_idx, k_idx, sr, kl_coef, b, i, r, &w);
            for (int g = 0; g < G; ++g) {
                double *out = dq + (ri * s->Hq + r * G + g) * s->d;
                const double *ds = w.dsc + (size_t)g * tmax;
                for (int e = 0; e < s->d; ++e) out[e] = 0.0;
                for (int u = 0; u < n; ++u) {
                    const orc_in *kj = k + (((long long)b * KR + w.tok[u]) * s->Hkv + r) * s->d;
                    for (int e = 0; e < s->d; ++e) out[e] += s->scale * ds[u] * bfv(kj[e]);
                }
            }
            double *oi = dq_idx + (ri * s->Hkv + r) * s->d_idx;
            for (int e = 0; e < s->d_idx; ++e) oi[e] = 0.0;
            for (int u = 0; u < n; ++u) {
                const orc_in *kj = k_idx + ((long long)b * KR + w.tok[u]) * s->d_idx;
                for (int e = 0; e < s->d_idx; ++e) oi[e] += s->scale_idx * w.dsig[u] * bfv(kj[e]);
            }
        }
        bwd_scratch_free(&w);
    }
    return 0;
}

/* Key-side gradients for the listed key blocks (of every batch entry):
 *   dk, dv   [B, n_kb*block, Hkv, d]   dk_idx [B, n_kb*block, d_idx]
 * (token j of listed block m, at local row m*block + (j mod block); rows of
 * a partial last block beyond Nk stay zero).  Work items are (b, r, chunk of
 * queries); each item accumulates into its own buffers, summed at the end. */
int orc_bwd_keys(const orc_shape *s, const orc_in *q, const orc_in *k, const orc_in *v,
                 const orc_in *d_o, const orc_in *q_idx, const orc_in *k_idx,
                 const int32_t *sel, double kl_coef, int n_kb, const int32_t *kblocks,
                 double *dk, double *dv, double *dk_idx)
{
    const int G = s->Hq / s->Hkv;
    const int nb = nblocks(s);
    const int tmax = s->topk * s->block;
    const long long rows_kb = (long long)n_kb * s->block;
    const size_t per_item = (size_t)rows_kb * (2 * (size_t)s->d + (size_t)s->d_idx);
    /* query chunks per (b, r): up to 16, fewer if the partial buffers would
     * exceed about 1 GiB in total */
    long long CH = (1LL << 27) / ((long long)s->B * s->Hkv * (long long)per_item + 1);
    if (CH > 16) CH = 16;
    if (CH < 1) CH = 1;
    const long long n_items = (long long)s->B * s->Hkv * CH;
    int *slot = (int *)malloc(sizeof(int) * (size_t)nb);   /* block -> listed index or -1 */
    for (int c = 0; c < nb; ++c) slot[c] = -1;
    for (int m = 0; m < n_kb; ++m) slot[kblocks[m]] = m;
    double *part = (double *)calloc((size_t)n_items * per_item, sizeof(double));
    if (!part) { free(slot); return -1; }
    #pragma omp parallel
    {
        orc_bwd_scratch w;
        bwd_scratch_alloc(&w, G, tmax);
        #pragma omp for schedule(dynamic, 1)
        for (long long it = 0; it < n_items; ++it) {
            const int b = (int)(it / ((long long)s->Hkv * CH));
            const int r = (int)((it / CH) % s->Hkv);
            const int ch = (int)(it % CH);
            double *pk = part + (size_t)it * per_item;
            double *pv = pk + (size_t)rows_kb * s->d;
            double *pki = pv + (size_t)rows_kb * s->d;
            const long long i0 = (long long)s->Nq * ch / CH, i1 = (long long)s->Nq * (ch + 1) / CH;
            for (long long i = i0; i < i1; ++i) {
                const int32_t *sr = sel + (((long long)b * s->Hkv + r) * s->Nq + i) * s->topk;
                int hit = 0;
                for (int m = 0; m < s->topk; ++m) if (sr[m] >= 0 && slot[sr[m]] >= 0) hit = 1;
                if (!hit) continue;
                const int n = bwd_row_group(s, q, k, v, d_o, q_idx, k_idx, sr, kl_coef, b, (int)i, r, &w);
                for (int u = 0; u < n; ++u) {
                    const long long j = w.tok[u];
                    const int m = slot[j / s->block];
                    if (m < 0) continue;
                    const long long lr = (long long)m * s->block + j % s->block;
                    for (int g = 0; g < G; ++g) {
                        const int h = r * G + g;
                        const orc_in *qh = q + (((long long)b * s->Nq + i) * s->Hq + h) * s->d;
                        const orc_in *doh = d_o + (((long long)b * s->Nq + i) * s->Hq + h) * s->d;
                        const double pgu = w.p[(size_t)g * tmax + u], dsu = w.dsc[(size_t)g * tmax + u];
                        for (int e = 0; e < s->d; ++e) {
                            pk[lr * s->d + e] += s->scale * dsu * bfv(qh[e]);
                            pv[lr * s->d + e] += pgu * bfv(doh[e]);
                        }
                    }
                    const orc_in *qi = q_idx + ((((long long)b * s->Nq + i) * s->Hkv + r) * s->d_idx);
                    for (int e = 0; e < s->d_idx; ++e) pki[lr * s->d_idx + e] += s->scale_idx * w.dsig[u] * bfv(qi[e]);
                }
            }
        }
        bwd_scratch_free(&w);
    }
    /* sum the per-item partials into the outputs */
    const size_t nk_out = (size_t)s->B * rows_kb * s->Hkv * s->d;
    const size_t nki_out = (size_t)s->B * rows_kb * s->d_idx;
    memset(dk, 0, nk_out * sizeof(double));
    memset(dv, 0, nk_out * sizeof(double));
    memset(dk_idx, 0, nki_out * sizeof(double));
    for (long long it = 0; it < n_items; ++it) {
        const int b = (int)(it / ((long long)s->Hkv * CH));
        const int r = (int)((it / CH) % s->Hkv);
        const double *pk = part + (size_t)it * per_item;
        const double *pv = pk + (size_t)rows_kb * s->d;
        const double *pki = pv + (size_t)rows_kb * s->d;
        for (long long lr = 0; lr < rows_kb; ++lr) {
            for (int e = 0; e < s->d; ++e) {
                dk[(((size_t)b * rows_kb + lr) * s->Hkv + r) * s->d + e] += pk[lr * s->d + e];
                dv[(((size_t)b * rows_kb + lr) * s->Hkv + r) * s->d + e] += pv[lr * s->d + e];
            }
            for (int e = 0; e < s->d_idx; ++e)
                dk_idx[((size_t)b * rows_kb + lr) * s->d_idx + e] += pki[lr * s->d_idx + e];
        }
    }
    free(part);
    free(slot);
    return 0;
}

/* Number of OpenMP threads the oracle runs with (for reporting). */
/* ------------------------------------------------------------------------ */
/* Block mask of a selection ("Sparse Attention · Part II", section 4.3,
 * "Turn support into a block mask").  A query tile is 128 consecutive query
 * rows i of one (batch, group); the tile's bit for key block c is set when
 * some query of the tile selected c.  Flags are packed 32 to an unsigned
 * word: block c lives in word c/32 at bit c%32, set by OR-ing 1 << (c%32).
 * Bits of blocks >= nb (the tail of the last word) stay zero; -1 entries of
 * the selection (padding) set nothing.
 * sel  [B, Hkv, Nq, topk]  ->  mask [B, Hkv, ceil(Nq/128), ceil(nb/32)]      */
int orc_block_mask(const orc_shape *s, const int32_t *sel, uint32_t *mask)
{
    const int nb = nblocks(s);
    const int W = (nb + 31) / 32;
    const int T = (s->Nq + 127) / 128;
    memset(mask, 0, sizeof(uint32_t) * (size_t)s->B * s->Hkv * T * W);
    for (int b = 0; b < s->B; ++b)
        for (int r = 0; r < s->Hkv; ++r)
            for (int i = 0; i < s->Nq; ++i) {
                const int32_t *row = sel + (((long long)b * s->Hkv + r) * s->Nq + i) * s->topk;
                uint32_t *words = mask + (((long long)b * s->Hkv + r) * T + i / 128) * W;
                for (int m = 0; m < s->topk; ++m) {
                    const int c = row[m];
                    if (c < 0 || c >= nb) continue;
                    words[c / 32] |= 1u << (c % 32);
                }
            }
    return 0;
}

/* The traversal of the same section: for each word, count its set bits and
 * visit them by rank, the n-th set bit found by scanning the word from bit
 * 0; the visited block is 32*w + bit.  Writes the active blocks in visiting
 * (ascending) order to out and returns how many there are.                  */
static int popcount32(uint32_t x)
{
    int n = 0;
    for (int bit = 0; bit < 32; ++bit) n += (int)((x >> bit) & 1u);
    return n;
}

static int nth_set_bit(uint32_t x, int rank)
{
    int seen = 0;
    for (int bit = 0; bit < 32; ++bit)
        if ((x >> bit) & 1u) {
            if (seen == rank) return bit;
            ++seen;
        }
    return -1;
}

int orc_mask_walk(const uint32_t *words, int n_words, int32_t *out)
{
    int n = 0;
    for (int w = 0; w < n_words; ++w) {
        const int count = popcount32(words[w]);
        for (int rank = 0; rank < count; ++rank) out[n++] = 32 * w + nth_set_bit(words[w], rank);
    }
    return n;
}

/* ------------------------------------------------------------------------ */
/* Index projections (section 3.2, the detachment equation): the index
 * queries and keys are linear maps of the detached hidden states X,
 *   q_idx[t, r, e] = sum_m X[t, m] Wq[m, r*d_idx + e]
 *   k_idx[t, e]    = sum_m X[t, m] Wk[m, e]
 * X [T, Dm] (T = B*N tokens), Wq [Dm, Hkv*d_idx], Wk [Dm, d_idx]; outputs
 * fp64, q_idx [T, Hkv*d_idx], k_idx [T, d_idx].                            */
int orc_index_proj(int T, int Dm, int Hkv, int d_idx, const orc_in *X, const orc_in *Wq, const orc_in *Wk,
                   double *q_idx, double *k_idx)
{
    const int nq = Hkv * d_idx;
    #pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        for (int c = 0; c < nq; ++c) {
            double acc = 0.0;
            for (int m = 0; m < Dm; ++m) acc += bfv(X[(long long)t * Dm + m]) * bfv(Wq[(long long)m * nq + c]);
            q_idx[(long long)t * nq + c] = acc;
        }
        for (int e = 0; e < d_idx; ++e) {
            double acc = 0.0;
            for (int m = 0; m < Dm; ++m) acc += bfv(X[(long long)t * Dm + m]) * bfv(Wk[(long long)m * d_idx + e]);
            k_idx[(long long)t * d_idx + e] = acc;
        }
    }
    return 0;
}

/* Gradient of the projections in their weights.  X is detached (stopgrad),
 * so nothing flows into it; the weights collect
 *   dWq[m, c] = sum_t X[t, m] dq_idx[t, c],   dWk[m, e] = sum_t X[t, m] dk_idx[t, e].
 * dq_idx [T, Hkv*d_idx], dk_idx [T, d_idx] (inputs); dWq [Dm, Hkv*d_idx],
 * dWk [Dm, d_idx] fp64.                                                     */
int orc_index_proj_bwd(int T, int Dm, int Hkv, int d_idx, const orc_in *X, const orc_in *dq_idx,
                       const orc_in *dk_idx, double *dWq, double *dWk)
{
    const int nq = Hkv * d_idx;
    #pragma omp parallel for schedule(static)
    for (int m = 0; m < Dm; ++m) {
        for (int c = 0; c < nq; ++c) {
            double acc = 0.0;
            for (int t = 0; t < T; ++t) acc += bfv(X[(long long)t * Dm + m]) * bfv(dq_idx[(long long)t * nq + c]);
            dWq[(long long)m * nq + c] = acc;
        }
        for (int e = 0; e < d_idx; ++e) {
            double acc = 0.0;
            for (int t = 0; t < T; ++t) acc += bfv(X[(long long)t * Dm + m]) * bfv(dk_idx[(long long)t * d_idx + e]);
            dWk[(long long)m * d_idx + e] = acc;
        }
    }
    return 0;
}

/* Dense indexer warm-up (section 3.1, the warm-up loss, in MSA's per-group
 * form of section 3.2): for query i and group r over EVERY causally visible
 * key j <= pos (no blocks, no selection),
 *   teacher  p_j = (1/G) sum over the group's heads h of softmax_j(scale q_h . k_j)
 *   student  s_j = softmax_j(scale_idx q_idx . k_idx_j)
 *   kl = sum_j p_j (log p_j - log s_j),  lse_idx = log sum_j exp(scale_idx q_idx . k_idx_j).
 * Requires q_offset == 0 and Nq == Nk (a training sequence).              */
int orc_warmup_kl(const orc_shape *s, const orc_in *q, const orc_in *k, const orc_in *q_idx, const orc_in *k_idx,
                  int n_rows, const long long *rows, double *out_lse_idx, double *out_kl)
{
    const int G = s->Hq / s->Hkv;
    const long long KR = kvrows(s);
    #pragma omp parallel
    {
        double *lg = (double *)malloc(sizeof(double) * (size_t)s->Nk);
        double *p = (double *)malloc(sizeof(double) * (size_t)s->Nk);
        double *pt = (double *)malloc(sizeof(double) * (size_t)s->Nk);
        double *ps = (double *)malloc(sizeof(double) * (size_t)s->Nk);
        #pragma omp for schedule(dynamic, 1)
        for (long long t = 0; t < (long long)n_rows * s->Hkv; ++t) {
            const long long row = rows[t / s->Hkv];
            const int r = (int)(t % s->Hkv);
            const int b = (int)(row / s->Nq), i = (int)(row % s->Nq);
            const int n = i + 1;                         /* keys 0 .. i */
            for (int j = 0; j < n; ++j) pt[j] = 0.0;
            for (int g = 0; g < G; ++g) {
                const orc_in *qh = q + (((long long)b * s->Nq + i) * s->Hq + r * G + g) * s->d;
                for (int j = 0; j < n; ++j)
                    lg[j] = s->scale * dot_bf(qh, k + (((long long)b * KR + j) * s->Hkv + r) * s->d, s->d);
                softmax_lse(lg, n, p);
                for (int j = 0; j < n; ++j) pt[j] += p[j] / G;
            }
            const orc_in *qi = q_idx + (((long long)b * s->Nq + i) * s->Hkv + r) * s->d_idx;
            for (int j = 0; j < n; ++j)
                lg[j] = s->scale_idx * dot_bf(qi, k_idx + ((long long)b * KR + j) * s->d_idx, s->d_idx);
            out_lse_idx[t] = softmax_lse(lg, n, ps);
            double kl = 0.0;
            for (int j = 0; j < n; ++j)
                if (pt[j] > 0.0) kl += pt[j] * (log(pt[j]) - log(ps[j]));
            out_kl[t] = kl;
        }
        free(lg); free(p); free(pt); free(ps);
    }
    return 0;
}

/* Gradient of L_warm = kl_coef / (B Nq Hkv) * sum of the rows' kl in the
 * index inputs (the teacher is detached): with dsig_j = coef (s_j - p_j),
 *   dq_idx[b, i, r, :] = scale_idx sum_j dsig_j k_idx[b, j, :]
 *   dk_idx[b, j, :]   += scale_idx dsig_j q_idx[b, i, r, :]
 * dq_idx [B, Nq, Hkv, d_idx], dk_idx [B, Nk, d_idx] fp64 (overwritten).
 * Rows are taken one (b, group) at a time so the dk_idx sums are formed in
 * a fixed order per thread and added under a lock.                         */
int orc_warmup_grad(const orc_shape *s, const orc_in *q, const orc_in *k, const orc_in *q_idx,
                    const orc_in *k_idx, double kl_coef, double *dq_idx, double *dk_idx)
{
    const int G = s->Hq / s->Hkv;
    const long long KR = kvrows(s);
    const double coef = kl_coef / ((double)s->B * s->Nq * s->Hkv);
    memset(dk_idx, 0, sizeof(double) * (size_t)s->B * s->Nk * s->d_idx);
    #pragma omp parallel
    {
        double *lg = (double *)malloc(sizeof(double) * (size_t)s->Nk);
        double *p = (double *)malloc(sizeof(double) * (size_t)s->Nk);
        double *pt = (double *)malloc(sizeof(double) * (size_t)s->Nk);
        double *ps = (double *)malloc(sizeof(double) * (size_t)s->Nk);
        double *dki = (double *)malloc(sizeof(double) * (size_t)s->Nk * s->d_idx);
        #pragma omp for schedule(dynamic, 1)
        for (int br = 0; br < s->B * s->Hkv; ++br) {
            const int b = br / s->Hkv, r = br % s->Hkv;
            memset(dki, 0, sizeof(double) * (size_t)s->Nk * s->d_idx);
            for (int i = 0; i < s->Nq; ++i) {
                const int n = i + 1;
                for (int j = 0; j < n; ++j) pt[j] = 0.0;
                for (int g = 0; g < G; ++g) {
                    const orc_in *qh = q + (((long long)b * s->Nq + i) * s->Hq + r * G + g) * s->d;
                    for (int j = 0; j < n; ++j)
                        lg[j] = s->scale * dot_bf(qh, k + (((long long)b * KR + j) * s->Hkv + r) * s->d, s->d);
                    softmax_lse(lg, n, p);
                    for (int j = 0; j < n; ++j) pt[j] += p[j] / G;
                }
                const orc_in *qi = q_idx + (((long long)b * s->Nq + i) * s->Hkv + r) * s->d_idx;
                for (int j = 0; j < n; ++j)
                    lg[j] = s->scale_idx * dot_bf(qi, k_idx + ((long long)b * KR + j) * s->d_idx, s->d_idx);
                softmax_lse(lg, n, ps);
                double *dq = dq_idx + (((long long)b * s->Nq + i) * s->Hkv + r) * s->d_idx;
                for (int e = 0; e < s->d_idx; ++e) dq[e] = 0.0;
                for (int j = 0; j < n; ++j) {
                    const double dsig = coef * (ps[j] - pt[j]);
                    const orc_in *kj = k_idx + ((long long)b * KR + j) * s->d_idx;
                    for (int e = 0; e < s->d_idx; ++e) {
                        dq[e] += s->scale_idx * dsig * bfv(kj[e]);
                        dki[(long long)j * s->d_idx + e] += s->scale_idx * dsig * bfv(qi[e]);
                    }
                }
            }
            #pragma omp critical
            {
                double *out = dk_idx + (long long)b * s->Nk * s->d_idx;
                for (long long x = 0; x < (long long)s->Nk * s->d_idx; ++x) out[x] += dki[x];
            }
        }
        free(lg); free(p); free(pt); free(ps); free(dki);
    }
    return 0;
}

int orc_num_threads(void)
{
    int n = 1;
    #pragma omp parallel
    {
        #pragma omp single
        {
#ifdef _OPENMP
            n = omp_get_num_threads();
#endif
        }
    }
    return n;
}
