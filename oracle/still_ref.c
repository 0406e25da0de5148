/*
 * still_ref.c -- plain fp64 CPU oracle for one STILL attention layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file; only tests/, the smoke check and the benchmark's CPU-baseline leg
 * do.  It shares no code, header, table or constant with the CUDA library.
 *
 * What it computes follows "STILL: Content-Aware Intra-Layer Hybrid Attention
 * for Efficient LLM Linearization" (besthub.dev summary) and its companion
 * write-ups (roboind.com news page "STILL: Selecting Tokens for Intra-Layer
 * Hybrid Attention to Linearize LLMs"; shishifenxi.com page "NeurIPS 2026 |
 * 层内混合注意力 ... STILL"):
 *
 *   - Self-Saliency Score (section "Self-Saliency Score: Predicting Future
 *     Utility from Local Context"; roboind "Highlight 2"): the KL sensitivity
 *     between the sliding-window attention distribution with the self term
 *     (a^diag) and without it (a^nodiag).  KL(a^nodiag || a^diag) equals
 *     -log(1 - p_t) exactly, p_t being the self probability in a^diag; the
 *     pages' equation did not survive extraction, and this library fixes the
 *     regularised closed form -log(1 - p_t + 1e-6).
 *   - Fixed-budget routing and delayed chunk-level selection (sections
 *     "Content-Aware Routing with Fixed Budget" and "Delayed Chunk-Level
 *     Selection for Unified Training-Inference Parallelism"; shishifenxi
 *     "固定预算路由" / "延迟选择与分块并行"): W window slots, and each completed
 *     chunk of C tokens keeps its top-lambda tokens for good,
 *     lambda = floor((m - W) / T_max); everything else that left the window is
 *     accumulated into the linear-attention recurrent state.
 *   - NP-Map (section "NP-Map: Norm-Preserving Feature Map"): the learned map
 *     only sets a direction, the input norm is put back, the result is
 *     non-negative.  This library fixes phi(x) = ||x|| u / ||u||, with
 *     u = softmax(x Wf) over the d_f feature columns.
 *   - One shared normalisation of both branches:
 *       y_t = (sum_SA e^{s-c} v + phi(q)^T S) / (sum_SA e^{s-c} + phi(q)^T z),
 *     c = the maximum logit over the softmax keys of the row.
 *   - The gate of the linear branch (section "NP-Map: Norm-Preserving Feature
 *     Map": a gating mechanism raises the rank of the linear branch; its
 *     equation did not survive extraction).  Reading taken by this library: a
 *     per-channel sigmoid gate on the linear branch's numerator,
 *       y_t = (sum_SA e^{s-c} v + g_t * (phi(q)^T S)) / (sum_SA e^{s-c} + phi(q)^T z),
 *     g_t = 1 / (1 + exp(-a_t)) elementwise over the d channels, a_t the
 *     gate pre-activation of the query head at token t (an input of the
 *     layer).  Without a gate (g = 1) this is the layer above.
 *
 * The implementation is the decode recurrence (one token at a time, bounded
 * m-slot cache plus (S, z)), and the prefill is that recurrence run N times
 * from an empty state: the pages state that prefill, training and decode share
 * one routing rule and one memory update.  Each (sequence, kv head) unit is
 * independent; OpenMP spreads units over host threads.
 *
 * Per-unit state (all arrays owned by the caller):
 *   K, V   [m, d]   slots 0..W-1: window ring (token j in slot j % W);
 *                   slots W + c*lambda + r: the r-th kept token of chunk c.
 *                   While chunk c is the current (unfinished) chunk, its slots
 *                   hold "candidates": tokens of chunk c that already left the
 *                   window but may still be among the chunk's top-lambda.
 *   pos    [m]      token position held by the slot, -1 = empty
 *   cnt    [m]      candidates: how many tokens of the chunk seen so far
 *                   outrank the candidate (it is dropped at cnt == lambda)
 *   ssc    [m]      score of the token held by the slot
 *   S, z   [df, d], [df]  sum of phi(k) v^T and of phi(k) over folded tokens
 *   ring   [C]      scores of the current chunk, token j at j % C
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OREF_EPS 1e-6

typedef struct {
    int Hq, Hkv, G, d, df, W, C, m, T_max, lam;
} prm_t;

typedef struct {
    double *K, *V;
    int32_t *pos, *cnt;
    double *ssc, *S, *z, *ring;
} unit_t;

/* Ranking used by the top-lambda selection: a higher score wins, an exact tie
 * goes to the lower position. */
static int outranks(long i, double si, long j, double sj)
{
    return si > sj || (si == sj && i < j);
}

/* lambda = floor((m - W) / T_max); -1 when the budget is not valid. */
int oref_lambda(int m, int W, int T_max)
{
    if (T_max < 1 || W < 0 || m < W) return -1;
    return (m - W) / T_max;
}

/* NP-Map of `rows` rows of x [rows, d] with Wf [d, df] -> phi [rows, df]. */
void oref_npmap(const double *x, long rows, int d, const double *Wf, int df, double *phi)
{
    double *u = (double *)malloc(sizeof(double) * (size_t)df);
    for (long r = 0; r < rows; ++r) {
        const double *xr = x + r * d;
        double nx = 0.0;
        for (int i = 0; i < d; ++i) nx += xr[i] * xr[i];
        nx = sqrt(nx);
        double mx = -INFINITY;
        for (int j = 0; j < df; ++j) {
            double a = 0.0;
            for (int i = 0; i < d; ++i) a += xr[i] * Wf[(long)i * df + j];
            u[j] = a;
            if (a > mx) mx = a;
        }
        double su = 0.0;
        for (int j = 0; j < df; ++j) { u[j] = exp(u[j] - mx); su += u[j]; }
        double nu = 0.0;
        for (int j = 0; j < df; ++j) { u[j] /= su; nu += u[j] * u[j]; }
        nu = sqrt(nu);
        for (int j = 0; j < df; ++j) phi[r * df + j] = nx * u[j] / nu;
    }
    free(u);
}

/* Self-Saliency score of one query row against its window.  keys[0..n-2] are
 * the older window keys, keys[n-1] is the token's own key.  1 - p is formed as
 * the off-diagonal mass over the total mass, so no cancellation occurs. */
static double saliency(const double *qrow, const double *const *keys, int n, int d)
{
    double sc = 1.0 / sqrt((double)d);
    double *s = (double *)malloc(sizeof(double) * (size_t)n);
    double mx = -INFINITY;
    for (int i = 0; i < n; ++i) {
        double a = 0.0;
        for (int e = 0; e < d; ++e) a += qrow[e] * keys[i][e];
        s[i] = a * sc;
        if (s[i] > mx) mx = s[i];
    }
    double tot = 0.0, oth = 0.0;
    for (int i = 0; i < n; ++i) {
        double w = exp(s[i] - mx);
        tot += w;
        if (i < n - 1) oth += w;
    }
    free(s);
    return -log(oth / tot + OREF_EPS);
}

/* Per-kv-head scores of one sequence straight from the definition:
 * q [Hq, N, d], k [Hkv, N, d] -> head_scores [Hq, N] (nullable), scores
 * [Hkv, N] = mean of head_scores over the G query heads of each kv head. */
void oref_scores(const double *q, const double *k, int Hq, int Hkv, int N, int d, int W,
                 double *head_scores, double *scores)
{
    int G = Hq / Hkv;
    const double **keys = (const double **)malloc(sizeof(double *) * (size_t)(W > 0 ? W : 1));
    for (int g = 0; g < Hkv; ++g)
        for (long t = 0; t < N; ++t) scores[(long)g * N + t] = 0.0;
    for (int h = 0; h < Hq; ++h) {
        int g = h / G;
        for (long t = 0; t < N; ++t) {
            long lo = t - W + 1 < 0 ? 0 : t - W + 1;
            int n = (int)(t - lo + 1);
            for (int i = 0; i < n; ++i) keys[i] = k + ((long)g * N + lo + i) * d;
            double s = saliency(q + ((long)h * N + t) * d, keys, n, d);
            if (head_scores) head_scores[(long)h * N + t] = s;
            scores[(long)g * N + t] += s / G;
        }
    }
    free(keys);
}

/* ---- routing metrics of the ablation ("Ablation Studies", routing metric
 * comparison): other per-token scores ranked by the same chunk selection.
 * The pages name them without formulas; each is written out from its plain
 * reading.  1 diagonal: mean over the G heads of the self probability p_t of
 * the window softmax; 2 q.k / sqrt(d), mean over the G heads; 3 ||k_t||;
 * 4 uniform: 1 at the lambda evenly spaced offsets floor((r + 1/2) C / lambda)
 * of each chunk; 5 random: SplitMix64 (Steele, Lea, Flood 2014), the stream
 * that starts at `seed`, draw number i + 1 for the token with flat index
 * i = (unit0 + g) N + t, its top 24 bits over 2^24. */

static uint64_t oref_splitmix64_next(uint64_t *x)
{
    uint64_t z = (*x += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

void oref_metric_scores(const double *q, const double *k, int Hq, int Hkv, int N, int d, int W, int C, int lam,
                        int metric, uint64_t seed, long unit0, double *scores)
{
    int G = Hq / Hkv;
    double sc = 1.0 / sqrt((double)d);
    for (long i = 0; i < (long)Hkv * N; ++i) scores[i] = 0.0;
    if (metric == 5) {
        uint64_t x = seed;
        for (long j = 0; j < unit0 * (long)N; ++j) oref_splitmix64_next(&x);   /* earlier sequences' draws */
        for (long i = 0; i < (long)Hkv * N; ++i) scores[i] = (double)(oref_splitmix64_next(&x) >> 40) / 16777216.0;
        return;
    }
    for (int g = 0; g < Hkv; ++g)
        for (long t = 0; t < N; ++t) {
            const double *kt = k + ((long)g * N + t) * d;
            double v = 0.0;
            if (metric == 3) {
                for (int e = 0; e < d; ++e) v += kt[e] * kt[e];
                v = sqrt(v);
            } else if (metric == 4) {
                long off = t % C;
                if (lam >= C) v = 1.0;
                for (int r = 0; r < lam && r < C; ++r)
                    if (((2L * r + 1) * C) / (2L * lam) == off) v = 1.0;
            } else {
                for (int h = g * G; h < (g + 1) * G; ++h) {
                    const double *qt = q + ((long)h * N + t) * d;
                    if (metric == 2) {
                        double a = 0.0;
                        for (int e = 0; e < d; ++e) a += qt[e] * kt[e];
                        v += a * sc / G;
                    } else { /* 1: softmax over keys [max(0, t-W+1), t], the weight of key t */
                        long lo = t - W + 1 < 0 ? 0 : t - W + 1;
                        double mx = -INFINITY, tot = 0.0, self = 0.0;
                        for (long j = lo; j <= t; ++j) {
                            double a = 0.0;
                            for (int e = 0; e < d; ++e) a += qt[e] * k[((long)g * N + j) * d + e];
                            if (a * sc > mx) mx = a * sc;
                        }
                        for (long j = lo; j <= t; ++j) {
                            double a = 0.0;
                            for (int e = 0; e < d; ++e) a += qt[e] * k[((long)g * N + j) * d + e];
                            double w = exp(a * sc - mx);
                            tot += w;
                            if (j == t) self = w;
                        }
                        v += self / tot / G;
                    }
                }
            }
            scores[(long)g * N + t] = v;
        }
}

/* Top-lambda of each completed chunk c < T_max, ascending positions, -1 pad.
 * scores [Hkv, N] -> sel [Hkv, T_max, lam]. */
void oref_select(const double *scores, int Hkv, int N, int C, int lam, int T_max, int32_t *sel)
{
    int nfull = N / C;
    for (int g = 0; g < Hkv; ++g)
        for (int c = 0; c < T_max; ++c)
            for (int r = 0; r < lam; ++r) sel[((long)g * T_max + c) * lam + r] = -1;
    if (lam <= 0) return;
    char *taken = (char *)malloc((size_t)C);
    for (int g = 0; g < Hkv; ++g) {
        const double *sg = scores + (long)g * N;
        for (int c = 0; c < nfull && c < T_max; ++c) {
            long base = (long)c * C;
            int keep = lam < C ? lam : C;
            memset(taken, 0, (size_t)C);
            /* repeated arg-max: the best not-yet-taken token under outranks() */
            for (int r = 0; r < keep; ++r) {
                int best = -1;
                for (int i = 0; i < C; ++i) {
                    if (taken[i]) continue;
                    if (best < 0 || outranks(base + i, sg[base + i], base + best, sg[base + best])) best = i;
                }
                taken[best] = 1;
            }
            int r = 0;
            for (int i = 0; i < C; ++i)
                if (taken[i]) sel[((long)g * T_max + c) * lam + r++] = (int32_t)(base + i);
        }
    }
    free(taken);
}

/* ---- streaming recurrence --------------------------------------------- */

static void fold(const prm_t *P, unit_t *u, const double *key, const double *val, const double *Wf)
{
    double *phk = (double *)malloc(sizeof(double) * (size_t)P->df);
    oref_npmap(key, 1, P->d, Wf, P->df, phk);
    for (int i = 0; i < P->df; ++i) {
        u->z[i] += phk[i];
        for (int e = 0; e < P->d; ++e) u->S[(long)i * P->d + e] += phk[i] * val[e];
    }
    free(phk);
}

static int free_slot(const prm_t *P, const unit_t *u, long c)
{
    for (int r = 0; r < P->lam; ++r) {
        int s = P->W + (int)c * P->lam + r;
        if (u->pos[s] < 0) return s;
    }
    return -1;
}

static int in_override(const prm_t *P, const int32_t *ovr, long c, long pos)
{
    for (int r = 0; r < P->lam; ++r)
        if (ovr[c * P->lam + r] == pos) return 1;
    return 0;
}

/* One decode step of one (sequence, kv head) unit at token position t (tokens
 * 0..t-1 already absorbed).  q [G, d] holds the G query rows of the group.
 * ovr (nullable) [T_max, lam] replaces the score ranking by a given selection.
 * Returns 0, or a negative code if an internal invariant breaks. */
static int step_unit(const prm_t *P, unit_t *u, long t, const double *q, const double *kt,
                     const double *vt, const double *Wf, const int32_t *ovr, const double *gate,
                     double *y, double *score_out)
{
    const int W = P->W, C = P->C, lam = P->lam, d = P->d, df = P->df, G = P->G;
    const long ct = t / C;
    const int selecting = lam > 0 && ct < P->T_max;
    double st = 0.0;

    /* (1) Self-Saliency score of token t over its window [t-W+1, t] */
    if (W >= 1) {
        int n = t + 1 < W ? (int)(t + 1) : W;
        const double **keys = (const double **)malloc(sizeof(double *) * (size_t)n);
        for (int i = 0; i < n - 1; ++i) keys[i] = u->K + ((t - n + 1 + i) % W) * d;
        keys[n - 1] = kt;
        for (int h = 0; h < G; ++h) st += saliency(q + (long)h * d, keys, n, d);
        st /= G;
        free(keys);
        if (selecting) u->ring[t % C] = st;
    }
    if (score_out) *score_out = st;

    /* (2) token t may push candidates of its own chunk out of the top-lambda */
    if (selecting && !ovr) {
        for (int r = 0; r < lam; ++r) {
            int s = W + (int)ct * lam + r;
            if (u->pos[s] < 0) continue;
            if (outranks(t, st, u->pos[s], u->ssc[s]) && ++u->cnt[s] >= lam) {
                fold(P, u, u->K + (long)s * d, u->V + (long)s * d, Wf);
                u->pos[s] = -1;
                u->cnt[s] = 0;
            }
        }
    }

    /* (3) token e = t - W leaves the window */
    const long e = t - W;
    if (e >= 0) {
        const double *ke = W > 0 ? u->K + (e % W) * d : kt;
        const double *ve = W > 0 ? u->V + (e % W) * d : vt;
        const long ce = e / C;
        if (lam == 0 || ce >= P->T_max) {
            fold(P, u, ke, ve, Wf);
        } else if (ce < ct) {
            /* finished chunk: kept tokens were copied to their slot when the
             * chunk finished; everything else goes to the linear state */
            int kept = 0;
            for (int r = 0; r < lam; ++r)
                if (u->pos[W + ce * lam + r] == e) kept = 1;
            if (!kept) fold(P, u, ke, ve, Wf);
        } else {
            /* current chunk: keep e as a candidate while fewer than lambda
             * tokens of the chunk seen so far outrank it */
            int count = 0, cand;
            double se = u->ring[e % C];
            for (long i = ct * C; i <= t; ++i)
                if (i != e && outranks(i, u->ring[i % C], e, se)) ++count;
            cand = ovr ? in_override(P, ovr, ce, e) : count < lam;
            if (cand) {
                int s = free_slot(P, u, ce);
                if (s < 0) return -1;
                memcpy(u->K + (long)s * d, ke, sizeof(double) * (size_t)d);
                memcpy(u->V + (long)s * d, ve, sizeof(double) * (size_t)d);
                u->pos[s] = (int32_t)e;
                u->cnt[s] = count;
                u->ssc[s] = se;
            } else {
                fold(P, u, ke, ve, Wf);
            }
        }
    }

    /* (4) token t enters the window ring */
    if (W > 0) {
        long s = t % W;
        memcpy(u->K + s * d, kt, sizeof(double) * (size_t)d);
        memcpy(u->V + s * d, vt, sizeof(double) * (size_t)d);
        u->pos[s] = (int32_t)t;
    }

    /* (5) attend: softmax keys = window + kept tokens of finished chunks that
     * left the window; linear keys = (S, z) + current-chunk candidates */
    {
        const double sc = 1.0 / sqrt((double)d);
        int nslot = W + lam * P->T_max;
        double *logit = (double *)malloc(sizeof(double) * (size_t)(nslot > 0 ? nslot : 1));
        char *is_sa = (char *)malloc((size_t)(nslot > 0 ? nslot : 1));
        double *phq = (double *)malloc(sizeof(double) * (size_t)df);
        double *phk = (double *)malloc(sizeof(double) * (size_t)df);
        double *ylin = (double *)malloc(sizeof(double) * (size_t)d);   /* the linear branch's numerator */
        for (int s = 0; s < nslot; ++s) {
            int p = u->pos[s];
            if (s < W) is_sa[s] = p >= 0;
            else is_sa[s] = p >= 0 && p / C < ct && p <= t - W;
        }
        for (int h = 0; h < G; ++h) {
            const double *qh = q + (long)h * d;
            double *yh = y + (long)h * d;
            double mx = -INFINITY, den = 0.0;
            for (int s = 0; s < nslot; ++s) {
                if (!is_sa[s]) continue;
                double a = 0.0;
                for (int e2 = 0; e2 < d; ++e2) a += qh[e2] * u->K[(long)s * d + e2];
                logit[s] = a * sc;
                if (logit[s] > mx) mx = logit[s];
            }
            for (int e2 = 0; e2 < d; ++e2) yh[e2] = 0.0;
            for (int s = 0; s < nslot; ++s) {
                if (!is_sa[s]) continue;
                double w = exp(logit[s] - mx);
                den += w;
                for (int e2 = 0; e2 < d; ++e2) yh[e2] += w * u->V[(long)s * d + e2];
            }
            oref_npmap(qh, 1, d, Wf, df, phq);
            for (int e2 = 0; e2 < d; ++e2) ylin[e2] = 0.0;
            for (int i = 0; i < df; ++i) {
                den += phq[i] * u->z[i];
                for (int e2 = 0; e2 < d; ++e2) ylin[e2] += phq[i] * u->S[(long)i * d + e2];
            }
            for (int s = W; s < nslot; ++s) {
                int p = u->pos[s];
                if (p < 0 || p / C != ct) continue;
                oref_npmap(u->K + (long)s * d, 1, d, Wf, df, phk);
                double a = 0.0;
                for (int i = 0; i < df; ++i) a += phq[i] * phk[i];
                den += a;
                for (int e2 = 0; e2 < d; ++e2) ylin[e2] += a * u->V[(long)s * d + e2];
            }
            for (int e2 = 0; e2 < d; ++e2) {
                const double gch = gate ? 1.0 / (1.0 + exp(-gate[(long)h * d + e2])) : 1.0;
                yh[e2] += gch * ylin[e2];
                yh[e2] = den != 0.0 ? yh[e2] / den : 0.0;
            }
        }
        free(logit);
        free(is_sa);
        free(phq);
        free(phk);
        free(ylin);
    }

    /* (6) chunk ct is complete after token t: its top-lambda are kept for good */
    if (selecting && (t + 1) % C == 0) {
        long base = ct * C;
        int keep = lam < C ? lam : C;
        long *win = (long *)malloc(sizeof(long) * (size_t)keep);
        int nwin = 0;
        if (ovr) {
            for (int r = 0; r < lam; ++r)
                if (ovr[ct * lam + r] >= 0) win[nwin++] = ovr[ct * lam + r];
        } else {
            char *taken = (char *)calloc((size_t)C, 1);
            for (int r = 0; r < keep; ++r) {
                int best = -1;
                for (int i = 0; i < C; ++i) {
                    if (taken[i]) continue;
                    if (best < 0 || outranks(base + i, u->ring[i], base + best, u->ring[best])) best = i;
                }
                taken[best] = 1;
                win[nwin++] = base + best;
            }
            free(taken);
        }
        for (int r = 0; r < nwin; ++r) {
            long w = win[r];
            if (w <= t - W) {
                /* already left the window: must be a live candidate */
                int found = 0;
                for (int q2 = 0; q2 < lam; ++q2)
                    if (u->pos[W + ct * lam + q2] == w) found = 1;
                if (!found) { free(win); return -2; }
            } else {
                int s = free_slot(P, u, ct);
                if (s < 0) { free(win); return -3; }
                memcpy(u->K + (long)s * d, u->K + (w % W) * d, sizeof(double) * (size_t)d);
                memcpy(u->V + (long)s * d, u->V + (w % W) * d, sizeof(double) * (size_t)d);
                u->pos[s] = (int32_t)w;
                u->ssc[s] = u->ring[w % C];
            }
        }
        for (int r = 0; r < lam; ++r) u->cnt[W + ct * lam + r] = 0;
        free(win);
    }
    return 0;
}

static int make_prm(prm_t *P, int Hq, int Hkv, int d, int df, int W, int C, int m, int T_max)
{
    if (Hq < 1 || Hkv < 1 || Hq % Hkv || d < 1 || df < 1 || C < 1) return -10;
    P->Hq = Hq; P->Hkv = Hkv; P->G = Hq / Hkv; P->d = d; P->df = df;
    P->W = W; P->C = C; P->m = m; P->T_max = T_max;
    P->lam = oref_lambda(m, W, T_max);
    if (P->lam < 0) return -11;
    if (W < 1 && P->lam > 0) return -12;
    return 0;
}

static unit_t unit_at(const prm_t *P, long b, int g, double *K, double *V, int32_t *pos,
                      int32_t *cnt, double *ssc, double *S, double *z, double *ring)
{
    long ug = b * P->Hkv + g;
    unit_t u;
    u.K = K + ug * P->m * P->d;
    u.V = V + ug * P->m * P->d;
    u.pos = pos + ug * P->m;
    u.cnt = cnt + ug * P->m;
    u.ssc = ssc + ug * P->m;
    u.S = S + ug * P->df * P->d;
    u.z = z + ug * P->df;
    u.ring = ring + ug * P->C;
    return u;
}

/* Empty state for B sequences (arrays sized as documented at the top). */
void oref_state_init(int B, int Hkv, int d, int df, int C, int m, double *K, double *V,
                     int32_t *pos, int32_t *cnt, double *ssc, double *S, double *z, double *ring)
{
    long nu = (long)B * Hkv;
    memset(K, 0, sizeof(double) * (size_t)(nu * m * d));
    memset(V, 0, sizeof(double) * (size_t)(nu * m * d));
    for (long i = 0; i < nu * m; ++i) { pos[i] = -1; cnt[i] = 0; ssc[i] = 0.0; }
    memset(S, 0, sizeof(double) * (size_t)(nu * df * d));
    memset(z, 0, sizeof(double) * (size_t)(nu * df));
    memset(ring, 0, sizeof(double) * (size_t)(nu * C));
}

/* Prefill of B sequences of N tokens = N streaming steps from an empty state.
 * q [B,Hq,N,d], k,v [B,Hkv,N,d], Wf [d,df] -> y [B,Hq,N,d], scores [B,Hkv,N]
 * (nullable) and the state after N tokens.  sel_override [B,Hkv,T_max,lam] is
 * nullable; gate [B,Hq,N,d] (nullable: no gate) holds the gate pre-activations
 * of the linear branch.  nthreads <= 0 uses the OpenMP default.  Returns 0 or
 * an error. */
int oref_prefill(int B, int Hq, int Hkv, int N, int d, int df, int W, int C, int m, int T_max,
                 const double *q, const double *k, const double *v, const double *Wf,
                 const int32_t *sel_override, const double *gate, double *y, double *scores, double *K, double *V,
                 int32_t *pos, int32_t *cnt, double *ssc, double *S, double *z, double *ring,
                 int nthreads)
{
    prm_t P;
    int rc = make_prm(&P, Hq, Hkv, d, df, W, C, m, T_max);
    if (rc) return rc;
    oref_state_init(B, Hkv, d, df, C, m, K, V, pos, cnt, ssc, S, z, ring);
    long nunits = (long)B * Hkv;
    int err = 0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(min : err)
#endif
    for (long ug = 0; ug < nunits; ++ug) {
        long b = ug / Hkv;
        int g = (int)(ug % Hkv);
        unit_t u = unit_at(&P, b, g, K, V, pos, cnt, ssc, S, z, ring);
        double *qbuf = (double *)malloc(sizeof(double) * (size_t)(P.G * d));
        double *gbuf = gate ? (double *)malloc(sizeof(double) * (size_t)(P.G * d)) : NULL;
        double *ybuf = (double *)malloc(sizeof(double) * (size_t)(P.G * d));
        const int32_t *ovr = sel_override ? sel_override + ug * T_max * (P.lam > 0 ? P.lam : 1) : NULL;
        if (P.lam == 0) ovr = NULL;
        for (long t = 0; t < N; ++t) {
            for (int h = 0; h < P.G; ++h) {
                memcpy(qbuf + (long)h * d, q + (((b * Hq) + g * P.G + h) * (long)N + t) * d,
                       sizeof(double) * (size_t)d);
                if (gbuf)
                    memcpy(gbuf + (long)h * d, gate + (((b * Hq) + g * P.G + h) * (long)N + t) * d,
                           sizeof(double) * (size_t)d);
            }
            const double *kt = k + ((b * Hkv + g) * (long)N + t) * d;
            const double *vt = v + ((b * Hkv + g) * (long)N + t) * d;
            double st;
            int r = step_unit(&P, &u, t, qbuf, kt, vt, Wf, ovr, gbuf, ybuf, &st);
            if (r < err) err = r;
            if (scores) scores[(b * Hkv + g) * (long)N + t] = st;
            for (int h = 0; h < P.G; ++h)
                memcpy(y + (((b * Hq) + g * P.G + h) * (long)N + t) * d, ybuf + (long)h * d,
                       sizeof(double) * (size_t)d);
        }
        free(qbuf);
        free(gbuf);
        free(ybuf);
    }
    return err;
}

/* One decode step for B sequences: token position t[b] of each sequence
 * (t[b] tokens already absorbed).  q_t [B,Hq,d], k_t,v_t [B,Hkv,d] -> y
 * [B,Hq,d]; gate_t [B,Hq,d] (nullable) the gate pre-activations of the
 * linear branch; the state is updated in place.  The caller advances t. */
int oref_decode_step(int B, int Hq, int Hkv, int d, int df, int W, int C, int m, int T_max,
                     const int64_t *t, const double *q_t, const double *k_t, const double *v_t,
                     const double *Wf, const double *gate_t, double *y, double *K, double *V, int32_t *pos,
                     int32_t *cnt, double *ssc, double *S, double *z, double *ring, int nthreads)
{
    prm_t P;
    int rc = make_prm(&P, Hq, Hkv, d, df, W, C, m, T_max);
    if (rc) return rc;
    long nunits = (long)B * Hkv;
    int err = 0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(min : err)
#endif
    for (long ug = 0; ug < nunits; ++ug) {
        long b = ug / Hkv;
        int g = (int)(ug % Hkv);
        unit_t u = unit_at(&P, b, g, K, V, pos, cnt, ssc, S, z, ring);
        int r = step_unit(&P, &u, (long)t[b], q_t + (b * Hq + g * P.G) * (long)d,
                          k_t + (b * Hkv + g) * (long)d, v_t + (b * Hkv + g) * (long)d, Wf, NULL,
                          gate_t ? gate_t + (b * Hq + g * P.G) * (long)d : NULL,
                          y + (b * Hq + g * P.G) * (long)d, NULL);
        if (r < err) err = r;
    }
    return err;
}

int oref_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
