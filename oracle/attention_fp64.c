/*
 * Exact softmax attention in fp64 on the CPU: the oracle for ring attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the tests, the package's smoke check and the bench's
 * CPU-baseline leg use it.  It shares no code with the CUDA library.
 *
 * What it computes is the plain definition of attention over the WHOLE,
 * unsharded sequence.  Ring attention (context parallelism) is an exact
 * re-ordering of this sum: the sequence is split into shards, each shard's
 * queries visit every key/value shard in ring order and the partial results
 * are aggregated (axolotl "Sequence Parallelism" page, introduction and
 * "Implementation Details"; aicassindra "tm_sp_math", section "Context
 * parallelism is the axis that is independent": every query must see every
 * key, and the ring rotates K/V blocks so no device holds the full
 * sequence).  The pages give no formula, so the oracle is the textbook
 * definition, written out step by step:
 *
 *   visible set   V(i) = { j : doc(j) = doc(i) and (not causal or j <= i) }
 *                 doc() comes from cu_seqlens (packed samples, positions
 *                 reset per sample: axolotl page, "Sample Packing with
 *                 Sequence Parallelism"); no cu_seqlens = one document.
 *   scores        s_ij = scale * sum_d q[i,h,d] k[j,g,d],  g = h / (Hq/Hkv)
 *   log-sum-exp   m_i = max_j s_ij, lse_i = m_i + ln sum_j exp(s_ij - m_i)
 *   output        O[i,h,:] = sum_j exp(s_ij - lse_i) v[j,g,:]
 *   backward      P_ij = exp(s_ij - lse_i), dP_ij = dO_i . v_j,
 *                 D_i = sum_j P_ij dP_ij, dS_ij = P_ij (dP_ij - D_i),
 *                 dQ_i = scale sum_j dS_ij k_j,
 *                 dK_j = scale sum_{h in group} sum_i dS_ij q_i,
 *                 dV_j = sum_{h in group} sum_i P_ij dO_i
 *   merge         the log-sum-exp merge of two partial results over
 *                 disjoint key sets (how ring steps are aggregated).
 *
 * Layouts: q/o/dq [T, Hq, D], k/v/dk/dv [T, Hkv, D], row-major doubles.
 * Rows with an empty visible set get O = 0 and lse = -inf (only possible
 * when a key subset is imposed through key_allowed).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Document index of every token, from cu_seqlens (NULL: one document). */
static int *doc_ids(int T, const int32_t *cu_seqlens, int num_seqs)
{
    int *doc = (int *)malloc(sizeof(int) * (size_t)(T > 0 ? T : 1));
    if (!doc) return NULL;
    for (int t = 0; t < T; ++t) {
        int d = 0;
        if (cu_seqlens) {
            /* the document whose range [cu[d], cu[d+1]) holds t */
            for (d = 0; d < num_seqs; ++d)
                if (t >= cu_seqlens[d] && t < cu_seqlens[d + 1]) break;
        }
        doc[t] = d;
    }
    return doc;
}

/* Key j is visible to query i: same document, and j <= i when causal. */
static int visible(const int *doc, int causal, int i, int j)
{
    if (doc[i] != doc[j]) return 0;
    if (causal && j > i) return 0;
    return 1;
}

static double dot(const double *a, const double *b, int n)
{
    double s = 0.0;
    for (int d = 0; d < n; ++d) s += a[d] * b[d];
    return s;
}

typedef struct {
    const double *q, *k, *v;
    int T, hq, hkv, d;
    const int *doc;
    int causal;
    double scale;
    const uint8_t *key_allowed;
} problem;

/* Scores of row (h, i) against every key it may see; returns the count of
 * visible keys and fills s[j] (only meaningful where vis[j] is set). */
static int row_scores(const problem *p, int h, int i, double *s, uint8_t *vis)
{
    int group = p->hq / p->hkv;
    int g = h / group;
    const double *qi = p->q + ((size_t)i * p->hq + h) * p->d;
    int n = 0;
    for (int j = 0; j < p->T; ++j) {
        int ok = visible(p->doc, p->causal, i, j);
        if (ok && p->key_allowed && !p->key_allowed[j]) ok = 0;
        vis[j] = (uint8_t)ok;
        if (!ok) continue;
        const double *kj = p->k + ((size_t)j * p->hkv + g) * p->d;
        s[j] = p->scale * dot(qi, kj, p->d);
        ++n;
    }
    return n;
}

/* lse of row (h, i) from its scores: max first, then the shifted sum. */
static double row_lse(const problem *p, const double *s, const uint8_t *vis)
{
    double m = -INFINITY;
    for (int j = 0; j < p->T; ++j)
        if (vis[j] && s[j] > m) m = s[j];
    if (m == -INFINITY) return -INFINITY;
    double z = 0.0;
    for (int j = 0; j < p->T; ++j)
        if (vis[j]) z += exp(s[j] - m);
    return m + log(z);
}

/*
 * Forward for n chosen (head, row) pairs: o[n*d], lse[n].
 * key_allowed (length T, or NULL) restricts the visible set further; it is
 * how a test computes one ring step's partial result.
 */
int oracle_fwd_rows(const double *q, const double *k, const double *v,
                    int T, int hq, int hkv, int d,
                    const int32_t *cu_seqlens, int num_seqs, int causal,
                    double scale, const uint8_t *key_allowed,
                    int n, const int32_t *hs, const int32_t *is,
                    double *o, double *lse)
{
    if (T <= 0 || hq <= 0 || hkv <= 0 || d <= 0 || hq % hkv) return -1;
    int *doc = doc_ids(T, cu_seqlens, num_seqs);
    if (!doc) return -2;
    problem p = {q, k, v, T, hq, hkv, d, doc, causal, scale, key_allowed};
    int group = hq / hkv;
    int err = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)T);
        uint8_t *vis = (uint8_t *)malloc((size_t)T);
        if (!s || !vis) {
#pragma omp atomic write
            err = -2;
        }
#pragma omp for schedule(dynamic, 4)
        for (int r = 0; r < n; ++r) {
            if (!s || !vis) continue;
            int h = hs[r], i = is[r];
            double *orow = o + (size_t)r * d;
            row_scores(&p, h, i, s, vis);
            double L = row_lse(&p, s, vis);
            lse[r] = L;
            for (int c = 0; c < d; ++c) orow[c] = 0.0;
            if (L == -INFINITY) continue;
            int g = h / group;
            for (int j = 0; j < T; ++j) {
                if (!vis[j]) continue;
                double w = exp(s[j] - L);
                const double *vj = v + ((size_t)j * hkv + g) * d;
                for (int c = 0; c < d; ++c) orow[c] += w * vj[c];
            }
        }
        free(s);
        free(vis);
    }
    free(doc);
    return err;
}

/* Row statistics of the backward: lse_i and D_i = sum_j P_ij dP_ij, and
 * dQ_i = scale sum_j dS_ij k_j, for one (head, row). */
static void bwd_row(const problem *p, const double *dout, int h, int i,
                    double *s, uint8_t *vis, double *lse_out, double *D_out,
                    double *dq_row)
{
    int group = p->hq / p->hkv, g = h / group, d = p->d;
    const double *doi = dout + ((size_t)i * p->hq + h) * d;
    row_scores(p, h, i, s, vis);
    double L = row_lse(p, s, vis);
    double D = 0.0;
    for (int j = 0; j < p->T; ++j) {
        if (!vis[j]) continue;
        const double *vj = p->v + ((size_t)j * p->hkv + g) * d;
        D += exp(s[j] - L) * dot(doi, vj, d);
    }
    if (dq_row) {
        for (int c = 0; c < d; ++c) dq_row[c] = 0.0;
        for (int j = 0; j < p->T; ++j) {
            if (!vis[j]) continue;
            const double *vj = p->v + ((size_t)j * p->hkv + g) * d;
            const double *kj = p->k + ((size_t)j * p->hkv + g) * d;
            double P = exp(s[j] - L);
            double dS = P * (dot(doi, vj, d) - D);
            for (int c = 0; c < d; ++c) dq_row[c] += p->scale * dS * kj[c];
        }
    }
    *lse_out = L;
    *D_out = D;
}

/*
 * Backward, query side, for n chosen (head, row) pairs:
 * dq[n*d], D[n] (= sum_j P_ij dP_ij from the definition), lse[n].
 */
int oracle_bwd_rows(const double *q, const double *k, const double *v,
                    const double *dout, int T, int hq, int hkv, int d,
                    const int32_t *cu_seqlens, int num_seqs, int causal,
                    double scale, int n, const int32_t *hs, const int32_t *is,
                    double *dq, double *Dvec, double *lse)
{
    if (T <= 0 || hq <= 0 || hkv <= 0 || d <= 0 || hq % hkv) return -1;
    int *doc = doc_ids(T, cu_seqlens, num_seqs);
    if (!doc) return -2;
    problem p = {q, k, v, T, hq, hkv, d, doc, causal, scale, NULL};
    int err = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)T);
        uint8_t *vis = (uint8_t *)malloc((size_t)T);
        if (!s || !vis) {
#pragma omp atomic write
            err = -2;
        }
#pragma omp for schedule(dynamic, 4)
        for (int r = 0; r < n; ++r) {
            if (!s || !vis) continue;
            bwd_row(&p, dout, hs[r], is[r], s, vis, &lse[r], &Dvec[r],
                    dq + (size_t)r * d);
        }
        free(s);
        free(vis);
    }
    free(doc);
    return err;
}

/*
 * Backward, key side, for n chosen (kv head, key row) pairs:
 * dk[n*d] = scale sum_{h in group} sum_i dS_ij q_i,
 * dv[n*d] = sum_{h in group} sum_i P_ij dO_i.
 * The row statistics (lse_i, D_i) of every query that sees one of the keys
 * are computed first, from the definition.
 */
int oracle_bwd_keys(const double *q, const double *k, const double *v,
                    const double *dout, int T, int hq, int hkv, int d,
                    const int32_t *cu_seqlens, int num_seqs, int causal,
                    double scale, int n, const int32_t *gs, const int32_t *js,
                    double *dk, double *dv)
{
    if (T <= 0 || hq <= 0 || hkv <= 0 || d <= 0 || hq % hkv) return -1;
    int *doc = doc_ids(T, cu_seqlens, num_seqs);
    if (!doc) return -2;
    problem p = {q, k, v, T, hq, hkv, d, doc, causal, scale, NULL};
    int group = hq / hkv;
    size_t HT = (size_t)hq * T;
    uint8_t *need = (uint8_t *)calloc(HT, 1);
    double *L = (double *)malloc(sizeof(double) * HT);
    double *Dv = (double *)malloc(sizeof(double) * HT);
    int *list = (int *)malloc(sizeof(int) * HT);
    int err = 0;
    if (!need || !L || !Dv || !list) err = -2;
    size_t nneed = 0;
    if (!err) {
        /* every (h, i) with some requested key j visible to it */
        for (int r = 0; r < n; ++r) {
            int g = gs[r], j = js[r];
            for (int h = g * group; h < (g + 1) * group; ++h)
                for (int i = 0; i < T; ++i)
                    if (visible(doc, causal, i, j)) need[(size_t)h * T + i] = 1;
        }
        for (size_t x = 0; x < HT; ++x)
            if (need[x]) list[nneed++] = (int)x;
    }
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)T);
        uint8_t *vis = (uint8_t *)malloc((size_t)T);
        if (!s || !vis) {
#pragma omp atomic write
            err = -2;
        }
#pragma omp for schedule(dynamic, 4)
        for (long x = 0; x < (long)nneed; ++x) {
            if (err || !s || !vis) continue;
            int h = list[x] / T, i = list[x] % T;
            bwd_row(&p, dout, h, i, s, vis, &L[list[x]], &Dv[list[x]], NULL);
        }
#pragma omp for schedule(dynamic, 4)
        for (int r = 0; r < n; ++r) {
            if (err) continue;
            int g = gs[r], j = js[r];
            const double *kj = k + ((size_t)j * hkv + g) * d;
            const double *vj = v + ((size_t)j * hkv + g) * d;
            double *dkr = dk + (size_t)r * d, *dvr = dv + (size_t)r * d;
            for (int c = 0; c < d; ++c) dkr[c] = dvr[c] = 0.0;
            for (int h = g * group; h < (g + 1) * group; ++h) {
                for (int i = 0; i < T; ++i) {
                    if (!visible(doc, causal, i, j)) continue;
                    const double *qi = q + ((size_t)i * hq + h) * d;
                    const double *doi = dout + ((size_t)i * hq + h) * d;
                    double sij = scale * dot(qi, kj, d);
                    double P = exp(sij - L[(size_t)h * T + i]);
                    double dS = P * (dot(doi, vj, d) - Dv[(size_t)h * T + i]);
                    for (int c = 0; c < d; ++c) {
                        dkr[c] += scale * dS * qi[c];
                        dvr[c] += P * doi[c];
                    }
                }
            }
        }
        free(s);
        free(vis);
    }
    free(need);
    free(L);
    free(Dv);
    free(list);
    free(doc);
    return err;
}

/*
 * Log-sum-exp merge of two partial results over disjoint key sets, in
 * place into (o_a, lse_a); n rows of d values.  This is how the pages'
 * ring steps are "aggregated" (axolotl page, introduction); the formula is
 * the identity  ln(e^a + e^b) = max(a,b) + ln(1 + e^-|a-b|)  with weights
 * e^(lse_x - lse) on each side.  An empty side (lse = -inf) contributes
 * nothing; two empty sides give O = 0, lse = -inf.
 */
void oracle_lse_merge(int n, int d, double *o_a, double *lse_a,
                      const double *o_b, const double *lse_b)
{
    for (int r = 0; r < n; ++r) {
        double a = lse_a[r], b = lse_b[r];
        double *oa = o_a + (size_t)r * d;
        const double *ob = o_b + (size_t)r * d;
        if (b == -INFINITY) continue;
        if (a == -INFINITY) {
            for (int c = 0; c < d; ++c) oa[c] = ob[c];
            lse_a[r] = b;
            continue;
        }
        double mx = a > b ? a : b;
        double L = mx + log1p(exp(-fabs(a - b)));
        double wa = exp(a - L), wb = exp(b - L);
        for (int c = 0; c < d; ++c) oa[c] = wa * oa[c] + wb * ob[c];
        lse_a[r] = L;
    }
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
