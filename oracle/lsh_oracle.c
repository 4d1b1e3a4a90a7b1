/*
 * lsh_oracle.c -- the oracle for multi-round LSH attention (forward pass).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is a plain, slow, obviously-correct CPU
 * restatement of what the method computes, in fp64.  Only the test suite, the
 * smoke check and the benchmark's CPU-baseline leg may load it.  It shares no
 * code, header, table or helper with the CUDA library, and the library never
 * calls it.
 *
 * Sources (all describe Reformer's LSH attention, Kitaev, Kaiser & Levskaya):
 *  [U]  "Reformer" glossary entry, ultralytics.com (es), section "Atencion LSH":
 *       shared query/key projection; angular LSH, bucket = position of the
 *       largest entry of [xR, -xR] for a random matrix R; sort tokens by bucket;
 *       split the sorted sequence into equal chunks; each token attends only to
 *       its own chunk and the previous one; several hash rounds in parallel.
 *       (The Arabic page of the same glossary states the same.)
 *  [M]  Reformer paper notes, modulabs-hub (ko), sections "Locality sensitive
 *       hashing" (R has half as many columns as there are buckets, and the +/-
 *       projections are concatenated), "LSH attention" (keys outside the
 *       query's bucket get -infinity; the token itself is removed because under
 *       shared QK it always scores highest; only keys at earlier positions in
 *       the causal case), "Multi-round LSH attention" (repeat the hashing).
 *  [Z]  Reformer article, ai-scholar.tech (zh), section "LSH attention": sort by
 *       LSH bucket, cut into equal-length chunks, attend within each chunk and
 *       the previous chunk; section "Overview": softmax(QK^T / sqrt(d_k)) V.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - keys are L2-normalised, queries are not; a zero key has inverse norm 0;
 *  - the score is scale * (q_i . k_j) / |k_j|, scale passed in;
 *  - self is a candidate only when no other candidate exists; such a row gets
 *    o = v_i and lse = SELF_LOGIT = -1e5;
 *  - chunk 0 has no previous chunk (no wrap-around); the window of sorted row
 *    s is [(floor(s/c)-1)c, (floor(s/c)+1)c) clipped to [0, L);
 *  - causal means strictly earlier original position;
 *  - argmax ties go to the first index of the concatenated [p, -p] vector;
 *  - the sort key is (bucket, original position), ascending;
 *  - rounds are combined with weights exp(lse_r - logsumexp_r lse_r);
 *  - backward: the gradient of the forward with the buckets held fixed (the
 *    hash is piecewise constant); a self-only row's logit is a constant, and
 *    a zero key (inverse norm 0) receives no gradient through its key role.
 *
 * Parity unpinned: the pages fix neither the value of `scale` (they disagree on the
 * 1/sqrt(d) factor) nor the self logit -1e5, so the tests cannot pin those to anything
 * but this restatement.  The logsumexp weighting of the rounds is a reading as well (the
 * pages only say the hashing is repeated), but its arithmetic is pinned: it must equal
 * one softmax over the multiset union of the rounds' candidate sets.  Everything else in
 * this file is pinned by the tests (closed forms, the pages' worked hashing statistic,
 * brute force on tiny inputs, library SDPA, planted mistakes).
 *
 * Layouts (row-major, all fp64 unless stated):
 *  x/qk, v      [L][d]          (one head)
 *  R            [n_rounds][d][nb/2]
 *  bucket       int32 [n_rounds][L]
 *  perm, inv    int32 [n_rounds][L]   perm: sorted -> original, inv = perm^-1
 *  bstart       int32 [n_rounds][nb+1] first sorted index of each bucket
 *  o_r          [n_rounds][L][d] in SORTED order;  lse_r [n_rounds][L] sorted
 *  out          [L][d];  lse [L]       in original order
 *  g_out, g_lse  like out, lse;  dqk, dv like qk, v  (backward)
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_SELF_LOGIT (-1.0e5)

double oracle_self_logit(void) { return ORACLE_SELF_LOGIT; }

/* ------------------------------------------------------------------------ */
/* Step 1: angular LSH.  p = x . R_r (nb/2 values); the bucket is the first   */
/* index of the maximum of the concatenation [p, -p]  ([U], [M]).  margin is  */
/* the gap between the largest and second-largest entry of that vector.      */
/* ------------------------------------------------------------------------ */
void oracle_hash(const double *x, long n, int d, const double *Rr, int nb,
                 int32_t *bucket, double *margin)
{
    int half = nb / 2;
    double *cat = (double *)malloc(sizeof(double) * (size_t)nb);
    for (long i = 0; i < n; ++i) {
        const double *xi = x + (size_t)i * d;
        for (int j = 0; j < half; ++j) {
            double p = 0.0;
            for (int k = 0; k < d; ++k) p += xi[k] * Rr[(size_t)k * half + j];
            cat[j] = p;
            cat[half + j] = -p;
        }
        int best = 0;
        for (int t = 1; t < nb; ++t)
            if (cat[t] > cat[best]) best = t;
        double second = -INFINITY;
        for (int t = 0; t < nb; ++t)
            if (t != best && cat[t] > second) second = cat[t];
        bucket[i] = best;
        if (margin) margin[i] = (nb > 1) ? cat[best] - second : INFINITY;
    }
    free(cat);
}

/* ------------------------------------------------------------------------ */
/* Step 2: sort the positions of one (batch, head, round) by (bucket,        */
/* position) ([Z] "sort each LSH bucket", [M] "order to solve it").  The key  */
/* is unique, so any correct sort gives the one permutation; qsort is used.  */
/* ------------------------------------------------------------------------ */
typedef struct { int32_t bucket, pos; } sort_key_t;

static int sort_key_cmp(const void *a, const void *b)
{
    const sort_key_t *x = (const sort_key_t *)a, *y = (const sort_key_t *)b;
    if (x->bucket != y->bucket) return x->bucket < y->bucket ? -1 : 1;
    if (x->pos != y->pos) return x->pos < y->pos ? -1 : 1;
    return 0;
}

void oracle_sort(const int32_t *bucket, int L, int nb, int32_t *perm,
                 int32_t *inv, int32_t *bstart)
{
    sort_key_t *keys = (sort_key_t *)malloc(sizeof(sort_key_t) * (size_t)L);
    for (int i = 0; i < L; ++i) { keys[i].bucket = bucket[i]; keys[i].pos = i; }
    qsort(keys, (size_t)L, sizeof(sort_key_t), sort_key_cmp);
    for (int s = 0; s < L; ++s) {
        perm[s] = keys[s].pos;
        if (inv) inv[keys[s].pos] = s;
    }
    if (bstart) {
        /* bstart[b] = number of tokens whose bucket is below b */
        for (int b = 0; b <= nb; ++b) bstart[b] = 0;
        for (int i = 0; i < L; ++i) bstart[bucket[i] + 1] += 1;
        for (int b = 0; b < nb; ++b) bstart[b + 1] += bstart[b];
    }
    free(keys);
}

/* Inverse L2 norm of each key row (0 for a zero row). */
void oracle_inv_norm(const double *qk, int L, int d, double *inv_norm)
{
    for (int j = 0; j < L; ++j) {
        double s = 0.0;
        for (int k = 0; k < d; ++k) s += qk[(size_t)j * d + k] * qk[(size_t)j * d + k];
        inv_norm[j] = s > 0.0 ? 1.0 / sqrt(s) : 0.0;
    }
}

/* ------------------------------------------------------------------------ */
/* The candidate set of sorted row s of one round, built straight from the   */
/* definition: every sorted position t of the own chunk or the previous      */
/* chunk ([U], [Z]), t != s, whose token has the query's bucket ([M]), and,  */
/* if causal, an earlier original position ([M]).  Writes the candidates'    */
/* original positions to cand (room for 2*chunk) and returns their number.   */
/* ------------------------------------------------------------------------ */
static int oracle_candidates(const int32_t *bucket, const int32_t *perm, int L,
                             int chunk, int causal, int s, int32_t *cand)
{
    int i = perm[s];
    int k = s / chunk;
    int lo = (k - 1) * chunk;
    if (lo < 0) lo = 0;
    int hi = (k + 1) * chunk;
    if (hi > L) hi = L;
    int n = 0;
    for (int t = lo; t < hi; ++t) {
        int j = perm[t];
        if (t == s) continue;
        if (bucket[j] != bucket[i]) continue;
        if (causal && !(j < i)) continue;
        cand[n++] = j;
    }
    return n;
}

/* ------------------------------------------------------------------------ */
/* Steps 3-4: chunked attention of one round, for the sorted rows listed in  */
/* `rows` (all rows when rows == NULL).  The self row is used only when the  */
/* candidate set is empty.                                                  */
/* ------------------------------------------------------------------------ */
void oracle_attend(const double *qk, const double *v, const double *inv_norm,
                   const int32_t *bucket, const int32_t *perm, int L, int d,
                   int chunk, int causal, double scale, const int32_t *rows,
                   int n_rows, double *o_sorted, double *lse_sorted)
{
    double *score = (double *)malloc(sizeof(double) * (size_t)(2 * chunk));
    int32_t *cand = (int32_t *)malloc(sizeof(int32_t) * (size_t)(2 * chunk));
    int count = rows ? n_rows : L;
    for (int q = 0; q < count; ++q) {
        int s = rows ? rows[q] : q;
        int i = perm[s];
        int n = oracle_candidates(bucket, perm, L, chunk, causal, s, cand);
        double *o = o_sorted + (size_t)s * d;
        if (n == 0) {
            for (int c = 0; c < d; ++c) o[c] = v[(size_t)i * d + c];
            lse_sorted[s] = ORACLE_SELF_LOGIT;
            continue;
        }
        double mx = -INFINITY;
        for (int a = 0; a < n; ++a) {
            int j = cand[a];
            double dot = 0.0;
            for (int c = 0; c < d; ++c) dot += qk[(size_t)i * d + c] * qk[(size_t)j * d + c];
            score[a] = scale * dot * inv_norm[j];
            if (score[a] > mx) mx = score[a];
        }
        double sum = 0.0;
        for (int a = 0; a < n; ++a) sum += exp(score[a] - mx);
        for (int c = 0; c < d; ++c) o[c] = 0.0;
        for (int a = 0; a < n; ++a) {
            double w = exp(score[a] - mx) / sum;
            const double *vj = v + (size_t)cand[a] * d;
            for (int c = 0; c < d; ++c) o[c] += w * vj[c];
        }
        lse_sorted[s] = mx + log(sum);
    }
    free(score);
    free(cand);
}

/* ------------------------------------------------------------------------ */
/* LSH bucketing as approximate nearest-neighbour search ([U], the paragraph */
/* after the algorithm: LSH finds most of a query's nearest neighbours at a  */
/* small fraction of the cost of an exhaustive search).  The candidates of   */
/* token i are the union over the rounds of its attention candidates without */
/* causality (same bucket, own chunk or previous chunk, i itself left out).  */
/* They are ranked by cosine similarity x_i.x_j / (|x_i| |x_j|) (0 when      */
/* either vector is zero), ties to the smaller j, and the first k are        */
/* written, a shorter list padded with index -1 and similarity -2.           */
/* ------------------------------------------------------------------------ */
static void oracle_top_k(const double *sim, const int32_t *idx, int n, int k,
                         int32_t *out_idx, double *out_sim)
{
    char *taken = (char *)calloc((size_t)(n > 0 ? n : 1), 1);
    for (int a = 0; a < k; ++a) {
        int b = -1;
        for (int t = 0; t < n; ++t) {
            if (taken[t]) continue;
            if (b < 0 || sim[t] > sim[b] || (sim[t] == sim[b] && idx[t] < idx[b])) b = t;
        }
        if (b < 0) {
            out_idx[a] = -1;
            out_sim[a] = -2.0;
            continue;
        }
        taken[b] = 1;
        out_idx[a] = idx[b];
        out_sim[a] = sim[b];
    }
    free(taken);
}

static double oracle_cosine(const double *x, const double *inv_norm, int d, int i, int j)
{
    double dot = 0.0;
    for (int c = 0; c < d; ++c) dot += x[(size_t)i * d + c] * x[(size_t)j * d + c];
    return dot * inv_norm[i] * inv_norm[j];
}

/* bucket, perm, inv: [n_rounds][L] of one head; tokens: the queries (all when NULL);  */
/* nn_idx, nn_sim: [count][k]                                                          */
void oracle_knn(const double *x, int L, int d, const int32_t *bucket, const int32_t *perm,
                const int32_t *inv, int n_rounds, int chunk, int k, const int32_t *tokens,
                int n_tokens, int32_t *nn_idx, double *nn_sim)
{
    double *inv_norm = (double *)malloc(sizeof(double) * (size_t)L);
    int32_t *cand = (int32_t *)malloc(sizeof(int32_t) * (size_t)(2 * chunk));
    int32_t *all = (int32_t *)malloc(sizeof(int32_t) * (size_t)(2 * chunk) * (size_t)n_rounds);
    double *sim = (double *)malloc(sizeof(double) * (size_t)(2 * chunk) * (size_t)n_rounds);
    int32_t *seen = (int32_t *)malloc(sizeof(int32_t) * (size_t)L);
    oracle_inv_norm(x, L, d, inv_norm);
    for (int j = 0; j < L; ++j) seen[j] = -1;
    int count = tokens ? n_tokens : L;
    for (int q = 0; q < count; ++q) {
        int i = tokens ? tokens[q] : q;
        int n_all = 0;
        for (int r = 0; r < n_rounds; ++r) {
            int s = inv[(size_t)r * L + i];
            int n = oracle_candidates(bucket + (size_t)r * L, perm + (size_t)r * L, L, chunk, 0,
                                      s, cand);
            for (int a = 0; a < n; ++a) {
                int j = cand[a];
                if (seen[j] != q) { seen[j] = q; all[n_all++] = j; }
            }
        }
        for (int a = 0; a < n_all; ++a) sim[a] = oracle_cosine(x, inv_norm, d, i, all[a]);
        oracle_top_k(sim, all, n_all, k, nn_idx + (size_t)q * k, nn_sim + (size_t)q * k);
    }
    free(inv_norm);
    free(cand);
    free(all);
    free(sim);
    free(seen);
}

/* The exact k nearest neighbours by the same similarity and tie rule, over every j != i */
/* (the reference an approximate search is measured against).                           */
void oracle_exact_knn(const double *x, int L, int d, int k, const int32_t *tokens, int n_tokens,
                      int32_t *nn_idx, double *nn_sim)
{
    double *inv_norm = (double *)malloc(sizeof(double) * (size_t)L);
    int32_t *all = (int32_t *)malloc(sizeof(int32_t) * (size_t)L);
    double *sim = (double *)malloc(sizeof(double) * (size_t)L);
    oracle_inv_norm(x, L, d, inv_norm);
    int count = tokens ? n_tokens : L;
    for (int q = 0; q < count; ++q) {
        int i = tokens ? tokens[q] : q;
        int n = 0;
        for (int j = 0; j < L; ++j) {
            if (j == i) continue;
            all[n] = j;
            sim[n] = oracle_cosine(x, inv_norm, d, i, j);
            ++n;
        }
        oracle_top_k(sim, all, n, k, nn_idx + (size_t)q * k, nn_sim + (size_t)q * k);
    }
    free(inv_norm);
    free(all);
    free(sim);
}

/* ------------------------------------------------------------------------ */
/* Steps 5-6: un-sort each round and combine rounds with logsumexp weights,  */
/* for the tokens listed in `tokens` (all when NULL).                        */
/* ------------------------------------------------------------------------ */
void oracle_combine(const double *o_r, const double *lse_r, const int32_t *inv,
                    int n_rounds, int L, int d, const int32_t *tokens,
                    int n_tokens, double *out, double *lse)
{
    int count = tokens ? n_tokens : L;
    double *l = (double *)malloc(sizeof(double) * (size_t)n_rounds);
    for (int q = 0; q < count; ++q) {
        int i = tokens ? tokens[q] : q;
        double mx = -INFINITY;
        for (int r = 0; r < n_rounds; ++r) {
            int s = inv[(size_t)r * L + i];
            l[r] = lse_r[(size_t)r * L + s];
            if (l[r] > mx) mx = l[r];
        }
        double sum = 0.0;
        for (int r = 0; r < n_rounds; ++r) sum += exp(l[r] - mx);
        double LSE = mx + log(sum);
        double *oi = out + (size_t)q * d;
        for (int c = 0; c < d; ++c) oi[c] = 0.0;
        for (int r = 0; r < n_rounds; ++r) {
            int s = inv[(size_t)r * L + i];
            double w = exp(l[r] - LSE);
            const double *src = o_r + ((size_t)r * L + s) * d;
            for (int c = 0; c < d; ++c) oi[c] += w * src[c];
        }
        lse[q] = LSE;
    }
    free(l);
}

/* ------------------------------------------------------------------------ */
/* Backward pass.  The pages train the model by back-propagation ([M]        */
/* "Introduction": without reversible layers every layer's activations are   */
/* kept for it; [U] on how reversible layers recompute them) but state no    */
/* formula for the attention's gradient.  These functions take the           */
/* derivative of steps 3-6 by the chain rule, in reverse step order, for the */
/* loss  sum_i g_out_i . out_i + sum_i g_lse_i lse_i.  The buckets, and so   */
/* perm and inv, are held fixed: the hash is piecewise constant and is not   */
/* differentiated.  Every gradient is ADDED into the caller's arrays.        */
/* ------------------------------------------------------------------------ */

/* Backward of steps 5-6 for one head.  With w_r = exp(lse_r(i) - LSE_i):
 *   d o_r(i)   = w_r g_out_i
 *   d lse_r(i) = w_r (g_out_i . (o_r(i) - out_i) + g_lse_i)
 * (out_i = sum_r w_r o_r(i) and LSE_i = log sum_r exp lse_r(i) differentiated
 * in lse_r(i)).  Inputs o_r, lse_r in sorted order as the forward leaves them;
 * out, lse, g_out, g_lse in original order; g_o, g_lse_r written in sorted
 * order, [n_rounds][L][d] and [n_rounds][L]. */
void oracle_combine_backward(const double *o_r, const double *lse_r, const int32_t *inv,
                             int n_rounds, int L, int d, const double *out,
                             const double *lse, const double *g_out, const double *g_lse,
                             double *g_o, double *g_lse_r)
{
    for (int i = 0; i < L; ++i) {
        const double *oi = out + (size_t)i * d;
        const double *gi = g_out + (size_t)i * d;
        for (int r = 0; r < n_rounds; ++r) {
            int s = inv[(size_t)r * L + i];
            const double *src = o_r + ((size_t)r * L + s) * d;
            double w = exp(lse_r[(size_t)r * L + s] - lse[i]);
            double *go = g_o + ((size_t)r * L + s) * d;
            double dot = 0.0;
            for (int c = 0; c < d; ++c) {
                go[c] += w * gi[c];
                dot += gi[c] * (src[c] - oi[c]);
            }
            g_lse_r[(size_t)r * L + s] += w * (dot + g_lse[i]);
        }
    }
}

/* Backward of steps 3-4 for one round of one head.  Sorted row s (token i)
 * with candidates j and weights p_j = exp(s_ij - lse_s), s_ij =
 * scale * (qk_i . khat_j), khat_j = qk_j * inv_norm_j:
 *   d v_j      += p_j g_o_s
 *   d s_ij      = p_j (g_o_s . (v_j - o_s) + g_lse_s)
 *   d q_i      += d s_ij * scale * khat_j
 *   d khat_j   += d s_ij * scale * qk_i
 * A row with no candidate copies v_i (d v_i += g_o_s); its logit is a
 * constant.  dq is the gradient through the query role of qk, dkhat through
 * the normalised key; oracle_key_norm_backward folds dkhat into qk. */
void oracle_attend_backward(const double *qk, const double *v, const double *inv_norm,
                            const int32_t *bucket, const int32_t *perm, int L, int d,
                            int chunk, int causal, double scale, const double *o_sorted,
                            const double *lse_sorted, const double *g_o,
                            const double *g_lse_sorted, double *dq, double *dkhat,
                            double *dv)
{
    int32_t *cand = (int32_t *)malloc(sizeof(int32_t) * (size_t)(2 * chunk));
    for (int s = 0; s < L; ++s) {
        int i = perm[s];
        int n = oracle_candidates(bucket, perm, L, chunk, causal, s, cand);
        const double *gs = g_o + (size_t)s * d;
        const double *os = o_sorted + (size_t)s * d;
        if (n == 0) {
            for (int c = 0; c < d; ++c) dv[(size_t)i * d + c] += gs[c];
            continue;
        }
        const double *qi = qk + (size_t)i * d;
        for (int a = 0; a < n; ++a) {
            int j = cand[a];
            const double *kj = qk + (size_t)j * d;
            const double *vj = v + (size_t)j * d;
            double dot = 0.0;
            for (int c = 0; c < d; ++c) dot += qi[c] * kj[c];
            double p = exp(scale * dot * inv_norm[j] - lse_sorted[s]);
            double gv = 0.0;
            for (int c = 0; c < d; ++c) {
                dv[(size_t)j * d + c] += p * gs[c];
                gv += gs[c] * (vj[c] - os[c]);
            }
            double ds = p * (gv + g_lse_sorted[s]);
            for (int c = 0; c < d; ++c) {
                dq[(size_t)i * d + c] += ds * scale * kj[c] * inv_norm[j];
                dkhat[(size_t)j * d + c] += ds * scale * qi[c];
            }
        }
    }
    free(cand);
}

/* d qk_j += inv_norm_j (dkhat_j - khat_j (khat_j . dkhat_j)): the Jacobian of
 * x -> x / |x| at qk_j.  A zero key has inverse norm 0 and a constant score 0
 * (the reading the forward takes), so it receives nothing here. */
void oracle_key_norm_backward(const double *qk, const double *inv_norm, const double *dkhat,
                              int L, int d, double *dqk)
{
    for (int j = 0; j < L; ++j) {
        const double *x = qk + (size_t)j * d;
        const double *g = dkhat + (size_t)j * d;
        double proj = 0.0;
        for (int c = 0; c < d; ++c) proj += x[c] * inv_norm[j] * g[c];
        for (int c = 0; c < d; ++c)
            dqk[(size_t)j * d + c] += inv_norm[j] * (g[c] - x[c] * inv_norm[j] * proj);
    }
}

/* ------------------------------------------------------------------------ */
/* The whole forward pass of one head: hash every round, sort, attend,       */
/* un-sort and combine.  Optional outputs may be NULL.                       */
/* ------------------------------------------------------------------------ */
typedef struct {
    const double *qk, *v, *R;
    int L, d, nb, n_rounds, chunk, causal;
    double scale;
    const double *inv_norm;
    int32_t *bucket, *perm, *inv, *bstart;
    double *margin, *o_r, *lse_r;
    int r;
} round_job_t;

static void run_round(round_job_t *j)
{
    size_t L = (size_t)j->L;
    int half = j->nb / 2;
    int32_t *bucket = j->bucket + j->r * L;
    int32_t *perm = j->perm + j->r * L;
    int32_t *inv = j->inv + j->r * L;
    int32_t *bstart = j->bstart + (size_t)j->r * (j->nb + 1);
    oracle_hash(j->qk, j->L, j->d, j->R + (size_t)j->r * j->d * half, j->nb, bucket,
                j->margin ? j->margin + j->r * L : NULL);
    oracle_sort(bucket, j->L, j->nb, perm, inv, bstart);
    oracle_attend(j->qk, j->v, j->inv_norm, bucket, perm, j->L, j->d, j->chunk,
                  j->causal, j->scale, NULL, 0, j->o_r + j->r * L * j->d,
                  j->lse_r + j->r * L);
}

/* A pool of worker threads pulling (head, round) jobs from a shared counter. */
typedef struct {
    round_job_t *jobs;
    int n_jobs;
    int next;
    pthread_mutex_t lock;
} job_queue_t;

static void *worker(void *arg)
{
    job_queue_t *q = (job_queue_t *)arg;
    for (;;) {
        pthread_mutex_lock(&q->lock);
        int k = q->next++;
        pthread_mutex_unlock(&q->lock);
        if (k >= q->n_jobs) break;
        run_round(&q->jobs[k]);
    }
    return NULL;
}

static void run_jobs(round_job_t *jobs, int n_jobs, int threads)
{
    job_queue_t q;
    q.jobs = jobs; q.n_jobs = n_jobs; q.next = 0;
    pthread_mutex_init(&q.lock, NULL);
    if (threads < 1) threads = 1;
    if (threads > n_jobs) threads = n_jobs;
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)threads);
    for (int t = 1; t < threads; ++t) pthread_create(&tid[t], NULL, worker, &q);
    worker(&q);
    for (int t = 1; t < threads; ++t) pthread_join(tid[t], NULL);
    free(tid);
    pthread_mutex_destroy(&q.lock);
}

/*
 * Forward pass over n_heads independent heads (B*H).  Inputs qk, v are
 * [n_heads][L][d]; R is [n_rounds][d][nb/2] and shared by every head.
 * out [n_heads][L][d], lse [n_heads][L].  Intermediates, when not NULL, are
 * per head: bucket/perm/inv [n_heads][n_rounds][L], bstart
 * [n_heads][n_rounds][nb+1], margin [n_heads][n_rounds][L], o_r
 * [n_heads][n_rounds][L][d] (sorted order), lse_r [n_heads][n_rounds][L].
 * Returns 0, or -1 when memory runs out.
 */
int oracle_forward(const double *qk, const double *v, const double *R, int n_heads,
                   int L, int d, int nb, int n_rounds, int chunk, int causal,
                   double scale, int threads, double *out, double *lse,
                   int32_t *bucket_o, int32_t *perm_o, int32_t *inv_o,
                   int32_t *bstart_o, double *margin_o, double *o_r_o,
                   double *lse_r_o)
{
    size_t HL = (size_t)n_heads * L;
    size_t RL = (size_t)n_rounds * L;
    int32_t *bucket = bucket_o ? bucket_o : (int32_t *)malloc(sizeof(int32_t) * HL * n_rounds);
    int32_t *perm = perm_o ? perm_o : (int32_t *)malloc(sizeof(int32_t) * HL * n_rounds);
    int32_t *inv = inv_o ? inv_o : (int32_t *)malloc(sizeof(int32_t) * HL * n_rounds);
    int32_t *bstart = bstart_o ? bstart_o
                               : (int32_t *)malloc(sizeof(int32_t) * (size_t)n_heads * n_rounds * (nb + 1));
    double *o_r = o_r_o ? o_r_o : (double *)malloc(sizeof(double) * HL * n_rounds * d);
    double *lse_r = lse_r_o ? lse_r_o : (double *)malloc(sizeof(double) * HL * n_rounds);
    double *inv_norm = (double *)malloc(sizeof(double) * HL);
    round_job_t *jobs = (round_job_t *)malloc(sizeof(round_job_t) * (size_t)n_heads * n_rounds);
    int rc = 0;
    if (!bucket || !perm || !inv || !bstart || !o_r || !lse_r || !inv_norm || !jobs) {
        rc = -1;
        goto done;
    }
    for (int h = 0; h < n_heads; ++h)
        oracle_inv_norm(qk + (size_t)h * L * d, L, d, inv_norm + (size_t)h * L);
    for (int h = 0; h < n_heads; ++h)
        for (int r = 0; r < n_rounds; ++r) {
            round_job_t *j = &jobs[h * n_rounds + r];
            j->qk = qk + (size_t)h * L * d;
            j->v = v + (size_t)h * L * d;
            j->R = R;
            j->L = L; j->d = d; j->nb = nb; j->n_rounds = n_rounds;
            j->chunk = chunk; j->causal = causal; j->scale = scale;
            j->inv_norm = inv_norm + (size_t)h * L;
            j->bucket = bucket + h * RL;
            j->perm = perm + h * RL;
            j->inv = inv + h * RL;
            j->bstart = bstart + (size_t)h * n_rounds * (nb + 1);
            j->margin = margin_o ? margin_o + h * RL : NULL;
            j->o_r = o_r + h * RL * d;
            j->lse_r = lse_r + h * RL;
            j->r = r;
        }
    run_jobs(jobs, n_heads * n_rounds, threads);
    for (int h = 0; h < n_heads; ++h)
        oracle_combine(o_r + h * RL * d, lse_r + h * RL, inv + h * RL, n_rounds, L, d,
                       NULL, 0, out + (size_t)h * L * d, lse + (size_t)h * L);
done:
    if (!bucket_o) free(bucket);
    if (!perm_o) free(perm);
    if (!inv_o) free(inv);
    if (!bstart_o) free(bstart);
    if (!o_r_o) free(o_r);
    if (!lse_r_o) free(lse_r);
    free(inv_norm);
    free(jobs);
    return rc;
}

/*
 * Backward pass over n_heads independent heads: recompute the forward of each
 * head (buckets, perm, inv, per-round o_r/lse_r, out, lse), then run the
 * backward steps above in reverse order: combination, every round's
 * attention, key normalisation.  g_out [n_heads][L][d] and g_lse
 * [n_heads][L] are the loss's gradients in out and lse; dqk and dv
 * [n_heads][L][d] are overwritten.  Returns 0, or -1 when memory runs out.
 */
int oracle_backward(const double *qk, const double *v, const double *R, int n_heads,
                    int L, int d, int nb, int n_rounds, int chunk, int causal,
                    double scale, const double *g_out, const double *g_lse,
                    double *dqk, double *dv)
{
    size_t Ld = (size_t)L * d, RL = (size_t)n_rounds * L;
    int32_t *bucket = (int32_t *)malloc(sizeof(int32_t) * RL);
    int32_t *perm = (int32_t *)malloc(sizeof(int32_t) * RL);
    int32_t *inv = (int32_t *)malloc(sizeof(int32_t) * RL);
    int32_t *bstart = (int32_t *)malloc(sizeof(int32_t) * (size_t)n_rounds * (nb + 1));
    double *o_r = (double *)malloc(sizeof(double) * RL * d);
    double *lse_r = (double *)malloc(sizeof(double) * RL);
    double *g_o = (double *)malloc(sizeof(double) * RL * d);
    double *g_lse_r = (double *)malloc(sizeof(double) * RL);
    double *out = (double *)malloc(sizeof(double) * Ld);
    double *lse = (double *)malloc(sizeof(double) * L);
    double *inv_norm = (double *)malloc(sizeof(double) * L);
    double *dkhat = (double *)malloc(sizeof(double) * Ld);
    int rc = 0;
    if (!bucket || !perm || !inv || !bstart || !o_r || !lse_r || !g_o || !g_lse_r || !out ||
        !lse || !inv_norm || !dkhat) {
        rc = -1;
        goto done;
    }
    for (int h = 0; h < n_heads; ++h) {
        const double *qh = qk + h * Ld, *vh = v + h * Ld;
        double *dq = dqk + h * Ld, *dvh = dv + h * Ld;
        rc = oracle_forward(qh, vh, R, 1, L, d, nb, n_rounds, chunk, causal, scale, 1, out,
                            lse, bucket, perm, inv, bstart, NULL, o_r, lse_r);
        if (rc != 0) goto done;
        oracle_inv_norm(qh, L, d, inv_norm);
        memset(g_o, 0, sizeof(double) * RL * d);
        memset(g_lse_r, 0, sizeof(double) * RL);
        memset(dkhat, 0, sizeof(double) * Ld);
        memset(dq, 0, sizeof(double) * Ld);
        memset(dvh, 0, sizeof(double) * Ld);
        oracle_combine_backward(o_r, lse_r, inv, n_rounds, L, d, out, lse, g_out + h * Ld,
                                g_lse + (size_t)h * L, g_o, g_lse_r);
        for (int r = 0; r < n_rounds; ++r)
            oracle_attend_backward(qh, vh, inv_norm, bucket + r * (size_t)L, perm + r * (size_t)L,
                                   L, d, chunk, causal, scale, o_r + r * Ld, lse_r + r * (size_t)L,
                                   g_o + r * Ld, g_lse_r + r * (size_t)L, dq, dkhat, dvh);
        oracle_key_norm_backward(qh, inv_norm, dkhat, L, d, dq);
    }
done:
    free(bucket); free(perm); free(inv); free(bstart); free(o_r); free(lse_r);
    free(g_o); free(g_lse_r); free(out); free(lse); free(inv_norm); free(dkhat);
    return rc;
}
