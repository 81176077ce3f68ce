/*
 * llsa_oracle.c -- plain, slow CPU oracle for Log-linear Sparse Attention (LLSA).
 *
 * TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT. Only the test suite, the smoke
 * check and the CPU-baseline leg of the benchmark may load this library. It
 * shares no source, header, table or helper with the CUDA library.
 *
 * What it follows: "Trainable Log-linear Sparse Attention for Efficient
 * Diffusion Transformers" (arXiv 2512.16615), as described on its Pith review
 * page (pith.science/paper/2512.16615):
 *   - "Core claim": Q, K, V are mean-pooled over log-many levels; the coarsest
 *     level scores every token, keeps the K best per query; each finer level
 *     scores only the K*B children of the blocks kept above; one coarse K/V
 *     token per level is appended to every query's key set with weight B^l.
 *   - "What carries the argument": L = floor(log_B N - 1) levels; the sparse
 *     index transpose (CSR to CSC) that gives each key block its query blocks.
 *   - Referee report, major comment 1 (Algorithm 1): the parent-to-child map is
 *     left undefined; read here as contiguous (children of j are jB..jB+B-1).
 *   - Referee report, minor comment 2 (KV Reweighting): W^(l) = B^l.
 *   - Figure 1: N = 8, B = 2, K = 1 worked layout.
 *
 * Readings where the page is silent (each is listed in the design notes):
 *   - The coarsest full scoring runs over the n_L level-L tokens.
 *   - Selection score: raw dot product of the mean-pooled query and key.
 *   - Ranking: higher score first; equal scores go to the lower index. The
 *     stored index rows are sorted ascending.
 *   - K at a level is clamped to the number of candidates there.
 *   - Enrichment token of level l for query block i: the rank-1 selection of
 *     level l for i's level-l ancestor (TOP1 rule, the default), or that
 *     ancestor itself (ANCESTOR rule).
 *   - Reweighting adds ln(B^l) to the coarse token's logit; softmax scale is
 *     1/sqrt(d) unless the caller gives one.
 *
 * Arithmetic: inputs arrive as float (they hold bf16- or fp32-exact values);
 * every sum, dot product, exponential and logarithm runs in double. Compile
 * without fast-math and without FP contraction so that x86 and Arm agree.
 *
 * Every function works on ONE (batch, head) slice; the Python wrapper loops
 * over slices (ctypes releases the GIL, so slices may run on threads).
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_ERR_ARG (-1)
#define ORC_ERR_MEM (-2)
#define ORC_MAX_COARSE 512 /* coarse columns per query block */

/* ------------------------------------------------------------------------ */
/* Level bookkeeping ("What carries the argument": L = floor(log_B N - 1)).  */
/* ------------------------------------------------------------------------ */

/* L = floor(log_B n - 1) = (largest e with B^e <= n) - 1, in integers. */
int orc_num_levels(long long n, int B)
{
    if (n < 1 || B < 2) return -1;
    long long p = 1;
    int e = 0;
    while (p * B <= n) { p *= B; e++; }
    return e - 1;
}

/* n_l = n / B^l for l = 0..L; returns 0 when every level divides evenly. */
int orc_level_sizes(long long n, int B, int L, long long *n_level)
{
    n_level[0] = n;
    for (int l = 1; l <= L; l++) {
        if (n_level[l - 1] % B != 0) return ORC_ERR_ARG;
        n_level[l] = n_level[l - 1] / B;
    }
    return ORC_OK;
}

/* Per-level Top-K after clamping to the candidate count:
 * K_L = min(K, n_L) at the coarsest level, K_l = min(K, K_{l+1} * B) below.
 * topk_level[l] for l = 1..L. */
int orc_level_topk(long long n, int B, int L, int K, int *topk_level)
{
    long long nl[64];
    if (L < 1 || L > 60 || K < 1) return ORC_ERR_ARG;
    if (orc_level_sizes(n, B, L, nl) != ORC_OK) return ORC_ERR_ARG;
    long long c = nl[L];
    topk_level[L] = (int)(K < c ? K : c);
    for (int l = L - 1; l >= 1; l--) {
        c = (long long)topk_level[l + 1] * B;
        topk_level[l] = (int)(K < c ? K : c);
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Hierarchical compression ("Core claim": mean pooling of Q, K, V).          */
/* ------------------------------------------------------------------------ */

/* pyr holds levels 1..L one after another: level l has n_l rows of d values.
 * P^(l)[j] = (1/B) * sum_{c<B} P^(l-1)[j*B + c], with P^(0) = x. */
int orc_pool(const float *x, long long n, int d, int B, int L, double *pyr)
{
    long long nl[64];
    if (L < 1 || L > 60 || orc_level_sizes(n, B, L, nl) != ORC_OK) return ORC_ERR_ARG;
    double *out = pyr;
    const double *prev = NULL;
    for (int l = 1; l <= L; l++) {
        for (long long j = 0; j < nl[l]; j++) {
            for (int c = 0; c < d; c++) {
                double s = 0.0;
                for (int r = 0; r < B; r++) {
                    long long row = j * B + r;
                    s += (l == 1) ? (double)x[row * d + c] : prev[row * d + c];
                }
                out[j * d + c] = s / (double)B;
            }
        }
        prev = out;
        out += nl[l] * d;
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Hierarchical Top-K selection ("Core claim"; referee major comment 1).      */
/* ------------------------------------------------------------------------ */

static double dot_dd(const double *a, const double *b, int d)
{
    double s = 0.0;
    for (int c = 0; c < d; c++) s += a[c] * b[c];
    return s;
}

/* Ranking order: a precedes b when its score is higher, or equal with a lower
 * index. */
static int precedes(double sa, long long ia, double sb, long long ib)
{
    return sa > sb || (sa == sb && ia < ib);
}

static int cmp_ll(const void *a, const void *b)
{
    long long x = *(const long long *)a, y = *(const long long *)b;
    return (x > y) - (x < y);
}

/* Selection for every query token of one level.
 *   qpyr_l, kpyr_l : level-l pooled Q and K, n_l rows of d doubles.
 *   parent_sel     : NULL at the coarsest level (every token is a candidate);
 *                    otherwise level-(l+1) selection, (n_l/B) rows of Kp
 *                    indices; the candidates of row i are the B children
 *                    j*B..j*B+B-1 of each j in row floor(i/B).
 *   K              : requested Top-K; the kept count is min(K, #candidates).
 *   sel_out        : n_l rows of Kl indices, ascending.
 *   top1_out       : n_l rank-1 indices (may be NULL).
 *   work_out       : incremented by the number of scored (query, key) pairs.
 * Returns Kl (>0) or an error. */
int orc_select_level(const double *qpyr_l, const double *kpyr_l, long long n_l, int d, int B,
                     const int *parent_sel, int Kp, int K,
                     int *sel_out, int *top1_out, long long *work_out)
{
    long long C = parent_sel ? (long long)Kp * B : n_l;
    if (C < 1 || K < 1) return ORC_ERR_ARG;
    int Kl = (int)(K < C ? K : C);
    long long *cand = (long long *)malloc(sizeof(long long) * C);
    double *score = (double *)malloc(sizeof(double) * C);
    char *taken = (char *)malloc((size_t)C);
    long long *kept = (long long *)malloc(sizeof(long long) * Kl);
    if (!cand || !score || !taken || !kept) {
        free(cand); free(score); free(taken); free(kept);
        return ORC_ERR_MEM;
    }
    for (long long i = 0; i < n_l; i++) {
        /* candidate set */
        if (parent_sel) {
            const int *prow = parent_sel + (i / B) * Kp;
            for (int m = 0; m < Kp; m++)
                for (int c = 0; c < B; c++) cand[(long long)m * B + c] = (long long)prow[m] * B + c;
        } else {
            for (long long c = 0; c < C; c++) cand[c] = c;
        }
        /* full similarity with each candidate */
        for (long long c = 0; c < C; c++)
            score[c] = dot_dd(qpyr_l + i * d, kpyr_l + cand[c] * d, d);
        if (work_out) *work_out += C;
        /* Top-K by repeated choice of the best remaining candidate */
        memset(taken, 0, (size_t)C);
        for (int k = 0; k < Kl; k++) {
            long long best = -1;
            for (long long c = 0; c < C; c++) {
                if (taken[c]) continue;
                if (best < 0 || precedes(score[c], cand[c], score[best], cand[best])) best = c;
            }
            taken[best] = 1;
            kept[k] = cand[best];
        }
        if (top1_out) top1_out[i] = (int)kept[0];
        qsort(kept, (size_t)Kl, sizeof(long long), cmp_ll);
        for (int k = 0; k < Kl; k++) sel_out[i * Kl + k] = (int)kept[k];
    }
    free(cand); free(score); free(taken); free(kept);
    return Kl;
}

/* Score of arbitrary (level-l query, level-l key) pairs: the same raw dot
 * product the selection uses. Lets a test judge whether a selection is a
 * legal Top-K of its candidates. */
int orc_pair_scores(const double *qpyr_l, const double *kpyr_l, int d,
                    const long long *rows, const long long *cols, long long npairs, double *out)
{
    for (long long p = 0; p < npairs; p++)
        out[p] = dot_dd(qpyr_l + rows[p] * d, kpyr_l + cols[p] * d, d);
    return ORC_OK;
}

/* The coarse-token columns of a query block's enrichment row, levels 1..L
 * in order: one column per level for TOP1 (rule 0) and ANCESTOR (rule 1), K_l
 * columns for level l under ALLK (rule 2: every token level l keeps for the
 * block's ancestor). Fills clev[c] = level of column c (when clev is not
 * NULL) and returns the column count, or a negative error. */
int orc_coarse_cols(long long n, int B, int L, int K, int rule, int *clev)
{
    int kl[64];
    if (L < 1 || L > 60 || orc_level_topk(n, B, L, K, kl) != ORC_OK) return ORC_ERR_ARG;
    if (rule < 0 || rule > 2) return ORC_ERR_ARG;
    int c = 0;
    for (int l = 1; l <= L; l++) {
        int cnt = rule == 2 ? kl[l] : 1;
        for (int r = 0; r < cnt; r++) {
            if (c >= ORC_MAX_COARSE) return ORC_ERR_ARG;
            if (clev) clev[c] = l;
            c++;
        }
    }
    return c;
}

/* All levels, coarsest first, plus the enrichment index.
 *   qpyr, kpyr : pyramids (levels 1..L one after another).
 *   rule       : 0 (TOP1), 1 (ANCESTOR) or 2 (ALLK), see coarse.
 *   idx_all    : level 1 first: n_1*K_1 ints, then n_2*K_2, ... n_L*K_L.
 *   top1_all   : n_1 + ... + n_L rank-1 indices, level 1 first.
 *   coarse     : n_1 rows of orc_coarse_cols(...) entries. The level-l columns
 *                of query block i hold its level-l enrichment tokens: for TOP1
 *                the rank-1 selection of level l for i's ancestor
 *                floor(i / B^(l-1)), for ANCESTOR that ancestor itself, for
 *                ALLK all K_l selections of level l for that ancestor
 *                (ascending, as the level's row is stored).
 *   work_out   : number of scored candidate pairs over all levels. */
int orc_select_all(const double *qpyr, const double *kpyr, long long n, int d, int B, int L, int K, int rule,
                   int *idx_all, int *top1_all, int *coarse, long long *work_out)
{
    long long nl[64];
    int kl[64];
    if (L < 1 || L > 60 || orc_level_sizes(n, B, L, nl) != ORC_OK) return ORC_ERR_ARG;
    if (orc_level_topk(n, B, L, K, kl) != ORC_OK) return ORC_ERR_ARG;
    const int ncol = orc_coarse_cols(n, B, L, K, rule, NULL);
    if (ncol < 0) return ORC_ERR_ARG;
    long long row_off[64], idx_off[64], t1_off[64];
    row_off[1] = 0; idx_off[1] = 0; t1_off[1] = 0;
    for (int l = 2; l <= L; l++) {
        row_off[l] = row_off[l - 1] + nl[l - 1];
        idx_off[l] = idx_off[l - 1] + nl[l - 1] * kl[l - 1];
        t1_off[l] = t1_off[l - 1] + nl[l - 1];
    }
    if (work_out) *work_out = 0;
    for (int l = L; l >= 1; l--) {
        const int *parent = (l == L) ? NULL : idx_all + idx_off[l + 1];
        int Kp = (l == L) ? 0 : kl[l + 1];
        int r = orc_select_level(qpyr + row_off[l] * d, kpyr + row_off[l] * d, nl[l], d, B,
                                 parent, Kp, K, idx_all + idx_off[l], top1_all + t1_off[l], work_out);
        if (r != kl[l]) return r < 0 ? r : ORC_ERR_ARG;
    }
    long long span = 1;
    int c0 = 0;
    for (int l = 1; l <= L; l++) {
        int cnt = rule == 2 ? kl[l] : 1;
        for (long long i = 0; i < nl[1]; i++) {
            long long anc = i / span;
            for (int r = 0; r < cnt; r++)
                coarse[i * ncol + c0 + r] = rule == 0 ? top1_all[t1_off[l] + anc]
                                            : rule == 1 ? (int)anc
                                                        : idx_all[idx_off[l] + anc * kl[l] + r];
        }
        c0 += cnt;
        span *= B;
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Block-sparse attention with KV enrichment ("Core claim").                  */
/* ------------------------------------------------------------------------ */

/* The key set of query block i: the B fine tokens of each selected level-1
 * block (kf, vf), then the coarse tokens of the enrichment levels 1..Le:
 * every column c of i's coarse row with clev[c] <= Le, with logit offset
 * ln(B^l), l = clev[c] (kc, vc, bias_c; crow[m] = its pyramid row). Returns
 * the number of coarse keys. */
static int key_set(const float *k, const float *v, const double *kpyr, const double *vpyr,
                   const long long *row_off, int d, int B, int Le, int K1,
                   const int *sel, const int *coarse, int ncol, const int *clev, long long i,
                   const float **kf, const float **vf, const double **kc, const double **vc,
                   double *bias_c, long long *crow)
{
    int nf = 0;
    for (int m = 0; m < K1; m++) {
        long long j = sel[i * K1 + m];
        for (int c = 0; c < B; c++) {
            kf[nf] = k + (j * B + c) * d;
            vf[nf] = v + (j * B + c) * d;
            nf++;
        }
    }
    int nc = 0;
    for (int c = 0; c < ncol; c++) {
        int l = clev[c];
        if (l > Le) continue;
        long long row = row_off[l] + coarse[i * ncol + c];
        kc[nc] = kpyr + row * d;
        vc[nc] = vpyr + row * d;
        bias_c[nc] = (double)l * log((double)B);
        crow[nc] = row;
        nc++;
    }
    return nc;
}

/* A coarse row description is valid: ncol columns, levels nondecreasing in
 * 1..L (columns of the levels 1..Le come first). */
static int coarse_ok(int ncol, const int *clev, int L)
{
    if (ncol < 0 || ncol > ORC_MAX_COARSE) return 0;
    for (int c = 0; c < ncol; c++) {
        if (clev[c] < 1 || clev[c] > L) return 0;
        if (c > 0 && clev[c] < clev[c - 1]) return 0;
    }
    return 1;
}

static double dot_fd(const float *a, const float *b, int d)
{
    double s = 0.0;
    for (int c = 0; c < d; c++) s += (double)a[c] * (double)b[c];
    return s;
}

static double dot_fD(const float *a, const double *b, int d)
{
    double s = 0.0;
    for (int c = 0; c < d; c++) s += (double)a[c] * b[c];
    return s;
}

/* Forward for the query tokens in qlist (all n tokens when qlist is NULL).
 * For token t in block i = t/B:
 *   s_j = scale * q_t . k_j            for the fine keys j,
 *   s_x = scale * q_t . K^(l)[e] + ln(B^l)   for each coarse key x = (l, e) of
 *                                             the enrichment levels l = 1..Le,
 *   lse_t = ln(sum_j e^{s_j} + sum_x e^{s_x}),
 *   o_t = sum_j e^{s_j - lse_t} v_j + sum_x e^{s_x - lse_t} V^(l)[e].
 * coarse: n_1 rows of ncol columns, clev[c] the level of column c.
 * Outputs are compacted: o[r*d..], lse[r] for the r-th listed token. */
int orc_fwd(const float *q, const float *k, const float *v, const double *kpyr, const double *vpyr,
            long long n, int d, int B, int L, int Le, int K1, const int *sel, const int *coarse,
            int ncol, const int *clev, double scale, const long long *qlist, long long nq, double *o, double *lse)
{
    long long nl[64], row_off[64];
    if (L < 1 || L > 60 || Le < 0 || Le > L || orc_level_sizes(n, B, L, nl) != ORC_OK) return ORC_ERR_ARG;
    if (!coarse_ok(ncol, clev, L)) return ORC_ERR_ARG;
    row_off[1] = 0;
    for (int l = 2; l <= L; l++) row_off[l] = row_off[l - 1] + nl[l - 1];
    int nkf = K1 * B;
    const float **kf = (const float **)malloc(sizeof(void *) * nkf);
    const float **vf = (const float **)malloc(sizeof(void *) * nkf);
    const double *kc[ORC_MAX_COARSE], *vc[ORC_MAX_COARSE];
    double bias[ORC_MAX_COARSE];
    long long crow[ORC_MAX_COARSE];
    double *s = (double *)malloc(sizeof(double) * (nkf + ncol + 1));
    if (!kf || !vf || !s) { free(kf); free(vf); free(s); return ORC_ERR_MEM; }
    long long count = qlist ? nq : n;
    for (long long r = 0; r < count; r++) {
        long long t = qlist ? qlist[r] : r;
        long long i = t / B;
        int nc = key_set(k, v, kpyr, vpyr, row_off, d, B, Le, K1, sel, coarse, ncol, clev, i, kf, vf, kc, vc, bias, crow);
        const float *qt = q + t * d;
        double m = -INFINITY;
        for (int j = 0; j < nkf; j++) { s[j] = scale * dot_fd(qt, kf[j], d); if (s[j] > m) m = s[j]; }
        for (int x = 0; x < nc; x++) { s[nkf + x] = scale * dot_fD(qt, kc[x], d) + bias[x]; if (s[nkf + x] > m) m = s[nkf + x]; }
        double z = 0.0;
        for (int j = 0; j < nkf + nc; j++) z += exp(s[j] - m);
        double lt = m + log(z);
        lse[r] = lt;
        double *ot = o + r * d;
        for (int c = 0; c < d; c++) ot[c] = 0.0;
        for (int j = 0; j < nkf; j++) {
            double p = exp(s[j] - lt);
            for (int c = 0; c < d; c++) ot[c] += p * (double)vf[j][c];
        }
        for (int x = 0; x < nc; x++) {
            double p = exp(s[nkf + x] - lt);
            for (int c = 0; c < d; c++) ot[c] += p * vc[x][c];
        }
    }
    free(kf); free(vf); free(s);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Sparse index transpose ("What carries the argument": CSR to CSC scan).     */
/* ------------------------------------------------------------------------ */

/* sel: T rows of K column indices in [0, ncols). Column j of the result lists
 * every row i whose selection contains j, in ascending i; col_ptr is the
 * exclusive prefix sum of the column counts (ncols + 1 entries). */
int orc_transpose(const int *sel, long long T, int K, long long ncols, int *col_ptr, int *row_idx)
{
    long long *cursor = (long long *)calloc((size_t)ncols, sizeof(long long));
    if (!cursor) return ORC_ERR_MEM;
    for (long long j = 0; j <= ncols; j++) col_ptr[j] = 0;
    for (long long e = 0; e < T * K; e++) {
        if (sel[e] < 0 || sel[e] >= ncols) { free(cursor); return ORC_ERR_ARG; }
        col_ptr[sel[e] + 1]++;
    }
    for (long long j = 0; j < ncols; j++) col_ptr[j + 1] += col_ptr[j];
    for (long long i = 0; i < T; i++)
        for (int m = 0; m < K; m++) {
            long long j = sel[i * K + m];
            row_idx[col_ptr[j] + cursor[j]] = (int)i;
            cursor[j]++;
        }
    free(cursor);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Backward with gradients through the pooled levels.                        */
/* ------------------------------------------------------------------------ */

/* Gradients of sum_t dO_t . o_t with the selection held fixed (Top-K is not
 * differentiable; pooled Q feeds only the selection, so it gets none).
 * For every (query t, key x) pair of the forward:
 *   P = e^{s - lse_t}, dP = dO_t . v_x, D_t = dO_t . o_t, dS = P (dP - D_t),
 *   dq_t += scale dS k_x,  dk_x += scale dS q_t,  dv_x += P dO_t,
 * where a coarse key x = K^(l)[e] accumulates into dK^(l)[e], dV^(l)[e].
 * Then, since K^(l)[e] is the mean of the B^l fine rows it covers,
 *   dk_t += sum_l dK^(l)[t / B^l] / B^l   (same for dv), l = 1..Le.
 * o and lse are this oracle's own forward results for all n tokens. */
int orc_bwd(const float *q, const float *k, const float *v, const double *kpyr, const double *vpyr,
            const double *o, const double *lse, const float *dout,
            long long n, int d, int B, int L, int Le, int K1, const int *sel, const int *coarse,
            int ncol, const int *clev, double scale, double *dq, double *dk, double *dv)
{
    long long nl[64], row_off[64];
    if (L < 1 || L > 60 || Le < 0 || Le > L || orc_level_sizes(n, B, L, nl) != ORC_OK) return ORC_ERR_ARG;
    if (!coarse_ok(ncol, clev, L)) return ORC_ERR_ARG;
    row_off[1] = 0;
    long long P = nl[1];
    for (int l = 2; l <= L; l++) { row_off[l] = row_off[l - 1] + nl[l - 1]; P += nl[l]; }
    int nkf = K1 * B;
    const float **kf = (const float **)malloc(sizeof(void *) * nkf);
    const float **vf = (const float **)malloc(sizeof(void *) * nkf);
    long long *kfi = (long long *)malloc(sizeof(long long) * nkf);
    double *dkc = (double *)calloc((size_t)(P * d), sizeof(double));
    double *dvc = (double *)calloc((size_t)(P * d), sizeof(double));
    const double *kc[ORC_MAX_COARSE], *vc[ORC_MAX_COARSE];
    double bias[ORC_MAX_COARSE];
    long long crow[ORC_MAX_COARSE];
    if (!kf || !vf || !kfi || !dkc || !dvc) {
        free(kf); free(vf); free(kfi); free(dkc); free(dvc);
        return ORC_ERR_MEM;
    }
    memset(dq, 0, sizeof(double) * n * d);
    memset(dk, 0, sizeof(double) * n * d);
    memset(dv, 0, sizeof(double) * n * d);
    for (long long t = 0; t < n; t++) {
        long long i = t / B;
        int nc = key_set(k, v, kpyr, vpyr, row_off, d, B, Le, K1, sel, coarse, ncol, clev, i, kf, vf, kc, vc, bias, crow);
        for (int m = 0; m < K1; m++)
            for (int c = 0; c < B; c++) kfi[m * B + c] = (long long)sel[i * K1 + m] * B + c;
        const float *qt = q + t * d;
        const float *gt = dout + t * d;
        double Dt = 0.0;
        for (int c = 0; c < d; c++) Dt += (double)gt[c] * o[t * d + c];
        for (int j = 0; j < nkf; j++) {
            double s = scale * dot_fd(qt, kf[j], d);
            double p = exp(s - lse[t]);
            double dp = dot_fd(gt, vf[j], d);
            double ds = p * (dp - Dt);
            long long x = kfi[j];
            for (int c = 0; c < d; c++) {
                dq[t * d + c] += scale * ds * (double)kf[j][c];
                dk[x * d + c] += scale * ds * (double)qt[c];
                dv[x * d + c] += p * (double)gt[c];
            }
        }
        for (int x = 0; x < nc; x++) {
            double s = scale * dot_fD(qt, kc[x], d) + bias[x];
            double p = exp(s - lse[t]);
            double dp = 0.0;
            for (int c = 0; c < d; c++) dp += (double)gt[c] * vc[x][c];
            double ds = p * (dp - Dt);
            double *gk = dkc + crow[x] * d;
            double *gv = dvc + crow[x] * d;
            for (int c = 0; c < d; c++) {
                dq[t * d + c] += scale * ds * kc[x][c];
                gk[c] += scale * ds * (double)qt[c];
                gv[c] += p * (double)gt[c];
            }
        }
    }
    /* through the means: every fine row of a pooled token gets 1/B^l of it */
    for (long long t = 0; t < n; t++) {
        long long span = 1;
        for (int l = 1; l <= Le; l++) {
            span *= B;
            long long e = t / span;
            for (int c = 0; c < d; c++) {
                dk[t * d + c] += dkc[(row_off[l] + e) * d + c] / (double)span;
                dv[t * d + c] += dvc[(row_off[l] + e) * d + c] / (double)span;
            }
        }
    }
    free(kf); free(vf); free(kfi); free(dkc); free(dvc);
    return ORC_OK;
}

/* dq for the listed query tokens only (same formula as orc_bwd, restricted to
 * the rows asked for). o_rows and lse_rows are the forward results for the
 * listed tokens, in list order. */
int orc_bwd_dq_rows(const float *q, const float *k, const float *v, const double *kpyr, const double *vpyr,
                    const double *o_rows, const double *lse_rows, const float *dout,
                    long long n, int d, int B, int L, int Le, int K1, const int *sel, const int *coarse,
                    int ncol, const int *clev, double scale, const long long *qlist, long long nq, double *dq_rows)
{
    long long nl[64], row_off[64];
    if (L < 1 || L > 60 || Le < 0 || Le > L || orc_level_sizes(n, B, L, nl) != ORC_OK) return ORC_ERR_ARG;
    if (!coarse_ok(ncol, clev, L)) return ORC_ERR_ARG;
    row_off[1] = 0;
    for (int l = 2; l <= L; l++) row_off[l] = row_off[l - 1] + nl[l - 1];
    int nkf = K1 * B;
    const float **kf = (const float **)malloc(sizeof(void *) * nkf);
    const float **vf = (const float **)malloc(sizeof(void *) * nkf);
    const double *kc[ORC_MAX_COARSE], *vc[ORC_MAX_COARSE];
    double bias[ORC_MAX_COARSE];
    long long crow[ORC_MAX_COARSE];
    if (!kf || !vf) { free(kf); free(vf); return ORC_ERR_MEM; }
    for (long long r = 0; r < nq; r++) {
        long long t = qlist[r];
        long long i = t / B;
        int nc = key_set(k, v, kpyr, vpyr, row_off, d, B, Le, K1, sel, coarse, ncol, clev, i, kf, vf, kc, vc, bias, crow);
        const float *qt = q + t * d;
        const float *gt = dout + t * d;
        double *g = dq_rows + r * d;
        double Dt = 0.0;
        for (int c = 0; c < d; c++) { Dt += (double)gt[c] * o_rows[r * d + c]; g[c] = 0.0; }
        for (int j = 0; j < nkf; j++) {
            double p = exp(scale * dot_fd(qt, kf[j], d) - lse_rows[r]);
            double ds = p * (dot_fd(gt, vf[j], d) - Dt);
            for (int c = 0; c < d; c++) g[c] += scale * ds * (double)kf[j][c];
        }
        for (int x = 0; x < nc; x++) {
            double p = exp(scale * dot_fD(qt, kc[x], d) + bias[x] - lse_rows[r]);
            double dp = 0.0;
            for (int c = 0; c < d; c++) dp += (double)gt[c] * vc[x][c];
            double ds = p * (dp - Dt);
            for (int c = 0; c < d; c++) g[c] += scale * ds * kc[x][c];
        }
    }
    free(kf); free(vf);
    return ORC_OK;
}

/* dk, dv for the fine tokens of the listed key blocks (block j covers tokens
 * jB..jB+B-1). Every query block whose selection contains j contributes its
 * fine pairs; every query block with the level-l ancestor of j among its
 * level-l enrichment tokens contributes through the mean, divided by B^l. o
 * and lse are the forward results for ALL n tokens. Output rows: nkb*B rows
 * of d. */
int orc_bwd_dkv_blocks(const float *q, const float *k, const float *v, const double *kpyr, const double *vpyr,
                       const double *o, const double *lse, const float *dout,
                       long long n, int d, int B, int L, int Le, int K1, const int *sel, const int *coarse,
                       int ncol, const int *clev, double scale, const long long *kblocks, long long nkb,
                       double *dk_rows, double *dv_rows)
{
    long long nl[64], row_off[64];
    if (L < 1 || L > 60 || Le < 0 || Le > L || orc_level_sizes(n, B, L, nl) != ORC_OK) return ORC_ERR_ARG;
    if (!coarse_ok(ncol, clev, L)) return ORC_ERR_ARG;
    row_off[1] = 0;
    for (int l = 2; l <= L; l++) row_off[l] = row_off[l - 1] + nl[l - 1];
    long long T = nl[1];
    double *gk = (double *)malloc(sizeof(double) * d);
    double *gv = (double *)malloc(sizeof(double) * d);
    if (!gk || !gv) { free(gk); free(gv); return ORC_ERR_MEM; }
    for (long long b = 0; b < nkb; b++) {
        long long j = kblocks[b];
        double *dkb = dk_rows + b * B * d;
        double *dvb = dv_rows + b * B * d;
        memset(dkb, 0, sizeof(double) * B * d);
        memset(dvb, 0, sizeof(double) * B * d);
        for (long long i = 0; i < T; i++) {
            int hit = 0;
            for (int m = 0; m < K1; m++) if (sel[i * K1 + m] == j) hit = 1;
            if (!hit) continue;
            for (int r = 0; r < B; r++) {
                long long t = i * B + r;
                const float *qt = q + t * d;
                const float *gt = dout + t * d;
                double Dt = 0.0;
                for (int c = 0; c < d; c++) Dt += (double)gt[c] * o[t * d + c];
                for (int c2 = 0; c2 < B; c2++) {
                    long long x = j * B + c2;
                    double p = exp(scale * dot_fd(qt, k + x * d, d) - lse[t]);
                    double ds = p * (dot_fd(gt, v + x * d, d) - Dt);
                    for (int c = 0; c < d; c++) {
                        dkb[c2 * d + c] += scale * ds * (double)qt[c];
                        dvb[c2 * d + c] += p * (double)gt[c];
                    }
                }
            }
        }
        long long span = 1;
        for (int l = 1; l <= Le; l++) {
            span *= B;
            long long e = (j * B) / span;           /* level-l ancestor of block j */
            const double *kcl = kpyr + (row_off[l] + e) * d;
            const double *vcl = vpyr + (row_off[l] + e) * d;
            double bias = (double)l * log((double)B);
            for (int c = 0; c < d; c++) { gk[c] = 0.0; gv[c] = 0.0; }
            for (long long i = 0; i < T; i++) {
                int has = 0;
                for (int c = 0; c < ncol; c++)
                    if (clev[c] == l && coarse[i * ncol + c] == e) has = 1;
                if (!has) continue;
                for (int r = 0; r < B; r++) {
                    long long t = i * B + r;
                    const float *qt = q + t * d;
                    const float *gt = dout + t * d;
                    double Dt = 0.0, dp = 0.0;
                    for (int c = 0; c < d; c++) { Dt += (double)gt[c] * o[t * d + c]; dp += (double)gt[c] * vcl[c]; }
                    double p = exp(scale * dot_fD(qt, kcl, d) + bias - lse[t]);
                    double ds = p * (dp - Dt);
                    for (int c = 0; c < d; c++) {
                        gk[c] += scale * ds * (double)qt[c];
                        gv[c] += p * (double)gt[c];
                    }
                }
            }
            for (int c2 = 0; c2 < B; c2++)
                for (int c = 0; c < d; c++) {
                    dkb[c2 * d + c] += gk[c] / (double)span;
                    dvb[c2 * d + c] += gv[c] / (double)span;
                }
        }
    }
    free(gk); free(gv);
    return ORC_OK;
}
