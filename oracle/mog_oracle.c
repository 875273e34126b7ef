/*
 * mog_oracle.c -- plain, slow, fp64 CPU statement of Mixture-of-Gaussians (MoG)
 * decode attention.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * benchmark's CPU-baseline leg are the only callers.  It shares no code, header,
 * table or helper with the CUDA library and never calls it.
 *
 * Sources (web pages, cited by title and section):
 *  [IA]  "Iceberg Attention: Sublinear Long-Context Decoding with Mixture-of-Gaussians",
 *        Abstract.  Sentences are numbered s1..s14 in reading order:
 *          s6  after prefill the keys of each head are split into O(sqrt N) clusters and
 *              O(log N) subclusters per cluster, each group described by a Gaussian;
 *          s7  the query is scored against these summaries, the most relevant clusters
 *              and subclusters are attended exactly;
 *          s8  the rest of the cache is approximated from the groups' means and variances.
 *  [RC]  newx.sg paper page on retrieval-completion attention, Abstract and AI Summary:
 *        exact attention over sink/tail anchors plus the retrieved keys, a prefill-time
 *        summary for the mid region, numerator and denominator of both parts added in the
 *        unnormalised domain, then one normalisation.
 *
 * The residual form used here (fixed by this library's specification, consistent with
 * [IA] s8): for an unselected group s with count n_s, mean mu_s, per-dimension
 * population variance sigma2_s and value mean vbar_s,
 *        e_s   = ln n_s + tau*q.mu_s + 0.5*tau^2 * sum_j q_j^2 sigma2_sj
 *        den_s = exp(e_s - m),   num_s = den_s * vbar_s,   tau = 1/sqrt(d),
 * i.e. n_s times the moment generating function of N(mu_s, diag sigma2_s) at tau*q.
 *
 * Readings of points the pages leave open (each applied below where marked):
 *  R1  sinks [0,S) and recent keys [N_build-R, N) are anchors: never clustered, always
 *      attended exactly; the clustered mid region is [S, N_build-R).
 *  R3  k-means seeding is strided: centroid j starts at member floor(j*n/k), members
 *      taken in ascending position order.
 *  R4  Lloyd iterations: T assignment steps at most, a centroid update between steps,
 *      stopping early when a step changes no assignment.
 *  R5  distance D(x,c) = sum_{j=0}^{d-1} (x_j - c_j)^2, fp64, summed in index order;
 *      the lowest centroid index wins ties.
 *  R6  an empty cluster keeps its centroid; a group that ends empty is ignored by
 *      scoring and residual.
 *  R8  variance is the population (divide by n) per-dimension variance, two-pass.
 *  R9  the value mean is the arithmetic mean of the members' value rows.
 *  R10 selection score = the same log-mass exponent e_s as the residual (score mode 0);
 *      mode 1 scores by tau*q.mu only (the residual always uses e_s).
 *  R11 top-ts subclusters are chosen inside each selected cluster.
 *  R12 an unselected cluster contributes its cluster Gaussian; inside a selected cluster
 *      each unselected non-empty subcluster contributes its own Gaussian.
 *  R13 m is the maximum over exact logits and residual exponents.
 *  R28 k-means++ seeding (a variant of the first level; the pages name no seeding): the
 *      first seed is member floor(u_0 n); seed r >= 1 is member i with probability
 *      D2_i / sum D2, D2_i the squared distance of member i to its nearest seed so far,
 *      drawn by inversion with the given uniform u_r: the first i (in member order) whose
 *      running sum of D2 exceeds u_r sum D2.  D2 is computed in fp32, the precision of
 *      the library's kernel, because it decides an index: each difference x_j - c_j is
 *      rounded to fp32, four partial sums s_m (m = j mod 4) take its square by fused
 *      multiply-add in increasing j, and D2 = (s_0 + s_1) + (s_2 + s_3), each sum
 *      rounded to fp32.  The running sums over the members are fp64.  With sum D2 = 0
 *      (every member on a seed) the pick is floor(u_r n) again.
 *  R29 the feature-map residual (a second estimator, [RC]: a fixed-size feature-map
 *      summary of the mid region, built at prefill, estimates the numerator and
 *      denominator of the keys not retrieved): positive random features of the softmax
 *      kernel, phi_i(x) = m^(-1/2) exp(w_i.x - |x|^2/2) for i < m with w_i drawn N(0, I_d)
 *      (an input), so that E[phi(x).phi(y)] = exp(x.y).  With q~ = sqrt(tau) q and
 *      k~ = sqrt(tau) k, every mid key k that is not attended exactly adds
 *      phi(q~).phi(k~) [v_k, 1] to the numerator and denominator; the exact part is the
 *      same as ora_decode's; one normalisation.
 *  Ranking order everywhere: score descending, then index ascending.
 *
 * Inputs are bf16 bit patterns (uint16) read as exact fp64 values.  Build with
 * -ffp-contract=off so that no multiply-add is fused (the distance must be the plain
 * sum of rounded squares in index order on every host).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORA_OK 0
#define ORA_EINVAL 1
#define ORA_ENOMEM 2

static double bf(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ---------------------------------------------------------------------------------
 * k-means (R3-R6)
 * ------------------------------------------------------------------------------- */

/* D(x,c) of R5: plain sum of squared differences in index order. */
static double sqdist(const uint16_t *x, const double *c, int64_t d)
{
    double acc = 0.0;
    for (int64_t j = 0; j < d; ++j) {
        double diff = bf(x[j]) - c[j];
        double sq = diff * diff;
        acc = acc + sq;
    }
    return acc;
}

/* Assignment step: out[r] = argmin_c D(x_{rows[r]}, cent_c), lowest index on ties. */
int ora_assign(const uint16_t *x, int64_t ld, const int64_t *rows, int64_t n,
               const double *cent, int64_t k, int64_t d, int32_t *out)
{
    if (n < 0 || k <= 0 || d <= 0)
        return ORA_EINVAL;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; ++r) {
        const uint16_t *xr = x + rows[r] * ld;
        int32_t best = 0;
        double bestd = sqdist(xr, cent, d);
        for (int64_t c = 1; c < k; ++c) {
            double dc = sqdist(xr, cent + c * d, d);
            if (dc < bestd) {
                bestd = dc;
                best = (int32_t)c;
            }
        }
        out[r] = best;
    }
    return ORA_OK;
}

/* Update step: centroid = fp64 mean of its members in row order; empty keeps (R6). */
static void update_means(const uint16_t *x, int64_t ld, const int64_t *rows, int64_t n,
                         const int32_t *a, int64_t k, int64_t d, double *cent,
                         double *sum, int64_t *cnt)
{
    memset(sum, 0, (size_t)(k * d) * sizeof(double));
    memset(cnt, 0, (size_t)k * sizeof(int64_t));
    for (int64_t r = 0; r < n; ++r) {
        const uint16_t *xr = x + rows[r] * ld;
        double *s = sum + (int64_t)a[r] * d;
        for (int64_t j = 0; j < d; ++j)
            s[j] = s[j] + bf(xr[j]);
        cnt[a[r]] += 1;
    }
    for (int64_t c = 0; c < k; ++c) {
        if (cnt[c] == 0)
            continue;
        for (int64_t j = 0; j < d; ++j)
            cent[c * d + j] = sum[c * d + j] / (double)cnt[c];
    }
}

/*
 * The update step on its own (R6), for lockstep comparison with another implementation's
 * steps: cent[c] becomes the fp64 mean of the rows r with a[r] == c, summed in row order;
 * a centroid with no rows keeps its value.  cent [k*d] is read and written.
 */
int ora_update(const uint16_t *x, int64_t ld, const int64_t *rows, int64_t n, const int32_t *a,
               int64_t k, int64_t d, double *cent)
{
    if (n < 0 || k <= 0 || d <= 0)
        return ORA_EINVAL;
    for (int64_t r = 0; r < n; ++r)
        if (a[r] < 0 || a[r] >= k)
            return ORA_EINVAL;
    double *sum = malloc((size_t)(k * d) * sizeof(double));
    int64_t *cnt = malloc((size_t)k * sizeof(int64_t));
    if (!sum || !cnt) {
        free(sum); free(cnt);
        return ORA_ENOMEM;
    }
    update_means(x, ld, rows, n, a, k, d, cent, sum, cnt);
    free(sum); free(cnt);
    return ORA_OK;
}

/* ---------------------------------------------------------------------------------
 * k-means++ seeding (R28)
 * ------------------------------------------------------------------------------- */

/* D2 of R28: fp32 squared distance of bf16 rows x and c (d a multiple of 4): four
 * interleaved partial sums by fused multiply-add, then (s0 + s1) + (s2 + s3). */
static float sqdist32(const uint16_t *x, const uint16_t *c, int64_t d)
{
    float s[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    for (int64_t j = 0; j < d; ++j) {
        float diff = (float)bf(x[j]) - (float)bf(c[j]);
        s[j % 4] = fmaf(diff, diff, s[j % 4]);
    }
    float a = s[0] + s[1];
    float b = s[2] + s[3];
    return a + b;
}

/* The inversion pick of R28 over weights w[0..n) with uniform u. */
static int64_t pp_draw(const float *w, int64_t n, double u)
{
    double total = 0.0;
    for (int64_t i = 0; i < n; ++i)
        total = total + (double)w[i];
    if (!(total > 0.0)) {
        int64_t j = (int64_t)floor(u * (double)n);
        return j < n - 1 ? j : n - 1;
    }
    double target = u * total, run = 0.0;
    int64_t last = 0;
    for (int64_t i = 0; i < n; ++i) {
        if (w[i] > 0.0f)
            last = i;
        run = run + (double)w[i];
        if (run > target)
            return i;
    }
    return last; /* u * total rounded up to total: the last member of positive weight */
}

/*
 * One k-means++ step (R28), on its own: given r seeds (member indices seeds[0..r)), the
 * member picked as seed r with the uniform u.  r = 0 picks floor(u n).  For comparison
 * with another implementation's seeding at any round.
 */
int ora_pp_pick(const uint16_t *x, int64_t ld, const int64_t *rows, int64_t n, int64_t d,
                const int64_t *seeds, int64_t r, double u, int64_t *pick)
{
    if (n <= 0 || d <= 0 || r < 0 || !(u >= 0.0 && u < 1.0))
        return ORA_EINVAL;
    for (int64_t i = 0; i < r; ++i)
        if (seeds[i] < 0 || seeds[i] >= n)
            return ORA_EINVAL;
    float *w = malloc((size_t)n * sizeof(float));
    if (!w)
        return ORA_ENOMEM;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        float best = 0.0f;
        for (int64_t s = 0; s < r; ++s) {
            float ds = sqdist32(x + rows[i] * ld, x + rows[seeds[s]] * ld, d);
            if (s == 0 || ds < best)
                best = ds;
        }
        w[i] = best;
    }
    if (r == 0) {
        int64_t j = (int64_t)floor(u * (double)n);
        *pick = j < n - 1 ? j : n - 1;
    } else {
        *pick = pp_draw(w, n, u);
    }
    free(w);
    return ORA_OK;
}

/*
 * k-means++ seeding (R28) of the rows listed in `rows`: seeds_out[r] (r < k) is the member
 * index of seed r, drawn with draws[r].  D2 is kept as the minimum over the seeds so far,
 * which equals its definition.
 */
int ora_kmeanspp(const uint16_t *x, int64_t ld, const int64_t *rows, int64_t n, int64_t k,
                 int64_t d, const double *draws, int64_t *seeds_out)
{
    if (n <= 0 || k <= 0 || d <= 0)
        return ORA_EINVAL;
    for (int64_t r = 0; r < k; ++r)
        if (!(draws[r] >= 0.0 && draws[r] < 1.0))
            return ORA_EINVAL;
    float *w = malloc((size_t)n * sizeof(float));
    if (!w)
        return ORA_ENOMEM;
    int64_t j = (int64_t)floor(draws[0] * (double)n);
    seeds_out[0] = j < n - 1 ? j : n - 1;
    for (int64_t r = 1; r < k; ++r) {
        const uint16_t *c = x + rows[seeds_out[r - 1]] * ld;
#pragma omp parallel for schedule(static)
        for (int64_t i = 0; i < n; ++i) {
            float ds = sqdist32(x + rows[i] * ld, c, d);
            if (r == 1 || ds < w[i])
                w[i] = ds;
        }
        seeds_out[r] = pp_draw(w, n, draws[r]);
    }
    free(w);
    return ORA_OK;
}

/*
 * Lloyd's algorithm over the rows listed in `rows` (ascending positions), k centroids,
 * at most `iters` assignment steps (R3, R4).
 *   cent_out  [k*d]   centroids used by the last assignment step
 *   assign_out[n]     the last assignment
 *   hist      [iters*k*d] or NULL: centroids used by each assignment step
 *   steps_out         number of assignment steps taken
 * With n == 0 nothing is assigned and the centroids are left at zero.
 */
static int lloyd_seeded(const uint16_t *x, int64_t ld, const int64_t *rows, int64_t n,
                        int64_t k, int64_t d, int64_t iters, const int64_t *seeds,
                        double *cent_out, int32_t *assign_out, double *hist, int64_t *steps_out);

int ora_lloyd(const uint16_t *x, int64_t ld, const int64_t *rows, int64_t n, int64_t k,
              int64_t d, int64_t iters, double *cent_out, int32_t *assign_out, double *hist,
              int64_t *steps_out)
{
    return lloyd_seeded(x, ld, rows, n, k, d, iters, NULL, cent_out, assign_out, hist, steps_out);
}

/* Lloyd's algorithm from the seeds seeds[0..k) (member indices), or strided (R3) when
 * seeds is NULL. */
static int lloyd_seeded(const uint16_t *x, int64_t ld, const int64_t *rows, int64_t n,
                        int64_t k, int64_t d, int64_t iters, const int64_t *seeds,
                        double *cent_out, int32_t *assign_out, double *hist, int64_t *steps_out)
{
    if (n < 0 || k <= 0 || d <= 0 || iters <= 0)
        return ORA_EINVAL;
    *steps_out = 0;
    memset(cent_out, 0, (size_t)(k * d) * sizeof(double));
    if (n == 0)
        return ORA_OK;
    double *sum = malloc((size_t)(k * d) * sizeof(double));
    int64_t *cnt = malloc((size_t)k * sizeof(int64_t));
    int32_t *prev = malloc((size_t)n * sizeof(int32_t));
    if (!sum || !cnt || !prev) {
        free(sum); free(cnt); free(prev);
        return ORA_ENOMEM;
    }
    /* R3: strided seeding in position order (R28: the k-means++ seeds instead) */
    for (int64_t c = 0; c < k; ++c) {
        const uint16_t *xr = x + rows[seeds ? seeds[c] : (c * n) / k] * ld;
        for (int64_t j = 0; j < d; ++j)
            cent_out[c * d + j] = bf(xr[j]);
    }
    for (int64_t t = 0; t < iters; ++t) {
        if (hist)
            memcpy(hist + t * k * d, cent_out, (size_t)(k * d) * sizeof(double));
        ora_assign(x, ld, rows, n, cent_out, k, d, assign_out);
        *steps_out = t + 1;
        if (t > 0 && memcmp(prev, assign_out, (size_t)n * sizeof(int32_t)) == 0)
            break; /* R4: no assignment changed */
        if (t + 1 < iters)
            update_means(x, ld, rows, n, assign_out, k, d, cent_out, sum, cnt);
        memcpy(prev, assign_out, (size_t)n * sizeof(int32_t));
    }
    free(sum); free(cnt); free(prev);
    return ORA_OK;
}

/* ---------------------------------------------------------------------------------
 * Gaussian summaries ([IA] s6, s8; R8, R9)
 * ------------------------------------------------------------------------------- */

/* Count, mean, population variance (two-pass) and value mean of the rows
 * perm[lo..hi).  An empty group gets zeros. */
static void group_stats(const uint16_t *K, const uint16_t *V, int64_t ld, int64_t d,
                        const int32_t *perm, int64_t lo, int64_t hi, int32_t *n_out,
                        double *mu, double *var, double *vbar)
{
    int64_t n = hi - lo;
    *n_out = (int32_t)n;
    for (int64_t j = 0; j < d; ++j)
        mu[j] = var[j] = vbar[j] = 0.0;
    if (n == 0)
        return;
    for (int64_t i = lo; i < hi; ++i) {
        const uint16_t *kr = K + (int64_t)perm[i] * ld;
        const uint16_t *vr = V + (int64_t)perm[i] * ld;
        for (int64_t j = 0; j < d; ++j) {
            mu[j] = mu[j] + bf(kr[j]);
            vbar[j] = vbar[j] + bf(vr[j]);
        }
    }
    for (int64_t j = 0; j < d; ++j) {
        mu[j] = mu[j] / (double)n;
        vbar[j] = vbar[j] / (double)n;
    }
    for (int64_t i = lo; i < hi; ++i) {
        const uint16_t *kr = K + (int64_t)perm[i] * ld;
        for (int64_t j = 0; j < d; ++j) {
            double diff = bf(kr[j]) - mu[j];
            var[j] = var[j] + diff * diff;
        }
    }
    for (int64_t j = 0; j < d; ++j)
        var[j] = var[j] / (double)n;
}

/*
 * Summaries of a given two-level partition.  perm lists positions ordered by
 * (cluster, subcluster); the members of subcluster g = c*L + l are
 * perm[sub_off[g] .. sub_off[g+1]), and those of cluster c are
 * perm[sub_off[c*L] .. sub_off[(c+1)*L]).  Outputs: cl_* [C], [C*d]; sub_* [C*L], [C*L*d].
 */
int ora_stats(const uint16_t *K, const uint16_t *V, int64_t ld, int64_t d, const int32_t *perm,
              const int32_t *sub_off, int64_t C, int64_t L, int32_t *cl_n, double *cl_mu,
              double *cl_var, double *cl_vbar, int32_t *sub_n, double *sub_mu, double *sub_var,
              double *sub_vbar)
{
    if (C < 0 || L <= 0 || d <= 0)
        return ORA_EINVAL;
#pragma omp parallel for schedule(dynamic)
    for (int64_t c = 0; c < C; ++c) {
        group_stats(K, V, ld, d, perm, sub_off[c * L], sub_off[(c + 1) * L], cl_n + c,
                    cl_mu + c * d, cl_var + c * d, cl_vbar + c * d);
        for (int64_t l = 0; l < L; ++l) {
            int64_t g = c * L + l;
            group_stats(K, V, ld, d, perm, sub_off[g], sub_off[g + 1], sub_n + g,
                        sub_mu + g * d, sub_var + g * d, sub_vbar + g * d);
        }
    }
    return ORA_OK;
}

/*
 * The MoG build for one KV head ([IA] s6): cluster the mid region (R1) into C clusters
 * with Lloyd's algorithm (T1 steps), then each cluster's members (ascending positions)
 * into L subclusters (T2 steps), then summarise every group.
 * Outputs: perm[N_mid] ordered by (cluster, subcluster, position), sub_off[C*L+1] with
 * offsets into perm, the summaries as in ora_stats, and optionally the first-level
 * assignment l1_assign[N_mid] (indexed by position - S) and l1_steps, l2_steps_max.
 */
int ora_build(const uint16_t *K, const uint16_t *V, int64_t ld, int64_t n_build, int64_t d,
              int64_t S, int64_t R, int64_t C, int64_t L, int64_t T1, int64_t T2,
              const double *draws, int32_t *perm, int32_t *sub_off, int32_t *cl_n,
              double *cl_mu, double *cl_var, double *cl_vbar, int32_t *sub_n, double *sub_mu,
              double *sub_var, double *sub_vbar, int32_t *l1_assign, int64_t *steps)
{
    if (n_build < 0 || d <= 0 || S < 0 || R < 0 || C <= 0 || L <= 0 || T1 <= 0 || T2 <= 0)
        return ORA_EINVAL;
    int64_t mid_lo = S, mid_hi = n_build - R; /* R1 */
    int64_t nm = mid_hi > mid_lo ? mid_hi - mid_lo : 0;
    int64_t *rows = malloc((size_t)(nm > 0 ? nm : 1) * sizeof(int64_t));
    int32_t *a1 = malloc((size_t)(nm > 0 ? nm : 1) * sizeof(int32_t));
    int32_t *a2 = malloc((size_t)(nm > 0 ? nm : 1) * sizeof(int32_t));
    int64_t *coff = calloc((size_t)(C + 1), sizeof(int64_t));
    double *cent1 = malloc((size_t)(C * d) * sizeof(double));
    double *cent2 = malloc((size_t)(L * d) * sizeof(double));
    int64_t *mem = malloc((size_t)(nm > 0 ? nm : 1) * sizeof(int64_t));
    int64_t *scount = malloc((size_t)L * sizeof(int64_t));
    if (!rows || !a1 || !a2 || !coff || !cent1 || !cent2 || !mem || !scount) {
        free(rows); free(a1); free(a2); free(coff); free(cent1); free(cent2); free(mem);
        free(scount);
        return ORA_ENOMEM;
    }
    for (int64_t i = 0; i < nm; ++i)
        rows[i] = mid_lo + i;
    int64_t st1 = 0, st2max = 0;
    if (nm > 0) {
        int64_t *seeds = NULL;
        if (draws) { /* R28: k-means++ seeds for the first level */
            seeds = malloc((size_t)C * sizeof(int64_t));
            if (!seeds || ora_kmeanspp(K, ld, rows, nm, C, d, draws, seeds) != ORA_OK) {
                free(seeds); free(rows); free(a1); free(a2); free(coff); free(cent1);
                free(cent2); free(mem); free(scount);
                return ORA_EINVAL;
            }
        }
        lloyd_seeded(K, ld, rows, nm, C, d, T1, seeds, cent1, a1, NULL, &st1);
        free(seeds);
    }
    if (l1_assign)
        for (int64_t i = 0; i < nm; ++i)
            l1_assign[i] = a1[i];
    /* members of each cluster in ascending position order */
    for (int64_t i = 0; i < nm; ++i)
        coff[a1[i] + 1] += 1;
    for (int64_t c = 0; c < C; ++c)
        coff[c + 1] += coff[c];
    {
        int64_t *fill = malloc((size_t)C * sizeof(int64_t));
        if (!fill) {
            free(rows); free(a1); free(a2); free(coff); free(cent1); free(cent2); free(mem);
            free(scount);
            return ORA_ENOMEM;
        }
        memcpy(fill, coff, (size_t)C * sizeof(int64_t));
        for (int64_t i = 0; i < nm; ++i)
            mem[fill[a1[i]]++] = rows[i];
        free(fill);
    }
    /* second level, cluster by cluster, then order members by (subcluster, position) */
    sub_off[0] = 0;
    for (int64_t c = 0; c < C; ++c) {
        int64_t lo = coff[c], n = coff[c + 1] - lo;
        int64_t st2 = 0;
        if (n > 0)
            ora_lloyd(K, ld, mem + lo, n, L, d, T2, cent2, a2 + lo, NULL, &st2);
        if (st2 > st2max)
            st2max = st2;
        for (int64_t l = 0; l < L; ++l)
            scount[l] = 0;
        for (int64_t i = 0; i < n; ++i)
            scount[a2[lo + i]] += 1;
        int64_t base = lo;
        for (int64_t l = 0; l < L; ++l) {
            int64_t w = base;
            for (int64_t i = 0; i < n; ++i)
                if (a2[lo + i] == l)
                    perm[w++] = (int32_t)mem[lo + i];
            base += scount[l];
            sub_off[c * L + l + 1] = (int32_t)base;
        }
    }
    if (steps) {
        steps[0] = st1;
        steps[1] = st2max;
    }
    free(rows); free(a1); free(a2); free(coff); free(cent1); free(cent2); free(mem);
    free(scount);
    return ora_stats(K, V, ld, d, perm, sub_off, C, L, cl_n, cl_mu, cl_var, cl_vbar, sub_n,
                     sub_mu, sub_var, sub_vbar);
}

/* ---------------------------------------------------------------------------------
 * Decode: scoring and selection ([IA] s7; R10, R11)
 * ------------------------------------------------------------------------------- */

/* log-mass exponent of a Gaussian group: ln n + tau q.mu + 0.5 tau^2 sum q_j^2 var_j */
static double log_mass(const double *q, int64_t d, double tau, int32_t n, const double *mu,
                       const double *var)
{
    double dot = 0.0, quad = 0.0;
    for (int64_t j = 0; j < d; ++j) {
        dot = dot + q[j] * mu[j];
        quad = quad + q[j] * q[j] * var[j];
    }
    return log((double)n) + tau * dot + 0.5 * tau * tau * quad;
}

static double score_of(int mode, const double *q, int64_t d, double tau, int32_t n,
                       const double *mu, const double *var)
{
    if (mode == 1) {
        double dot = 0.0;
        for (int64_t j = 0; j < d; ++j)
            dot = dot + q[j] * mu[j];
        return tau * dot;
    }
    return log_mass(q, d, tau, n, mu, var);
}

/* top-k of scores[0..n) among eligible[i] != 0, order (score desc, index asc);
 * out[0..k) gets the indices, -1 where fewer than k are eligible. */
static void top_k(const double *scores, const int *eligible, int64_t n, int64_t k, int32_t *out)
{
    char *taken = calloc((size_t)(n > 0 ? n : 1), 1);
    for (int64_t r = 0; r < k; ++r) {
        int64_t best = -1;
        for (int64_t i = 0; i < n; ++i) {
            if (!eligible[i] || taken[i])
                continue;
            if (best < 0 || scores[i] > scores[best])
                best = i;
        }
        out[r] = (int32_t)best;
        if (best >= 0)
            taken[best] = 1;
    }
    free(taken);
}

static void bf_vec(const uint16_t *src, int64_t d, double *dst)
{
    for (int64_t j = 0; j < d; ++j)
        dst[j] = bf(src[j]);
}

/*
 * Selection for one query head: cluster scores cscore[C] (empty clusters: -inf), the
 * top-tc clusters sel_c[tc], and inside the i-th selected cluster the top-ts
 * subclusters sel_s[i*ts + r] (subcluster index within the cluster), -1 padded;
 * sscore[tc*L] holds the subcluster scores of the selected clusters (-inf if empty).
 */
int ora_select(const uint16_t *q_bf16, int64_t d, double tau, int64_t C, int64_t L,
               const int32_t *cl_n, const double *cl_mu, const double *cl_var,
               const int32_t *sub_n, const double *sub_mu, const double *sub_var, int64_t tc,
               int64_t ts, int score_mode, int32_t *sel_c, int32_t *sel_s, double *cscore,
               double *sscore)
{
    if (C < 0 || L <= 0 || tc < 0 || ts < 0 || d <= 0)
        return ORA_EINVAL;
    double *q = malloc((size_t)d * sizeof(double));
    int *elig = malloc((size_t)((C > L ? C : L) + 1) * sizeof(int));
    double *ls = malloc((size_t)L * sizeof(double));
    if (!q || !elig || !ls) {
        free(q); free(elig); free(ls);
        return ORA_ENOMEM;
    }
    bf_vec(q_bf16, d, q);
    for (int64_t c = 0; c < C; ++c) {
        elig[c] = cl_n[c] > 0;
        cscore[c] = elig[c] ? score_of(score_mode, q, d, tau, cl_n[c], cl_mu + c * d,
                                       cl_var + c * d)
                            : -INFINITY;
    }
    top_k(cscore, elig, C, tc, sel_c);
    for (int64_t i = 0; i < tc; ++i) {
        for (int64_t l = 0; l < L; ++l)
            sscore[i * L + l] = -INFINITY;
        for (int64_t r = 0; r < ts; ++r)
            sel_s[i * ts + r] = -1;
        if (sel_c[i] < 0)
            continue;
        int64_t c = sel_c[i];
        for (int64_t l = 0; l < L; ++l) {
            int64_t g = c * L + l;
            elig[l] = sub_n[g] > 0;
            ls[l] = elig[l] ? score_of(score_mode, q, d, tau, sub_n[g], sub_mu + g * d,
                                       sub_var + g * d)
                            : -INFINITY;
            sscore[i * L + l] = ls[l];
        }
        top_k(ls, elig, L, ts, sel_s + i * ts);
    }
    free(q); free(elig); free(ls);
    return ORA_OK;
}

/* ---------------------------------------------------------------------------------
 * Decode: exact part + Gaussian residual + one normalisation ([IA] s7, s8; [RC])
 * ------------------------------------------------------------------------------- */

/*
 * Output for one query head given a selection (sel_c[tc], sel_s[tc*ts] as produced by
 * ora_select).  n_now >= n_build is the current length (keys appended after the build
 * join the recent anchors).  residual = 0 drops the Gaussian terms (top-only ablation).
 * out[d]; diag[3] = {m, den, number of exactly attended keys}.
 */
int ora_decode(const uint16_t *K, const uint16_t *V, int64_t ld, int64_t d, int64_t n_now,
               int64_t n_build, int64_t S, int64_t R, const uint16_t *q_bf16, double tau,
               int64_t C, int64_t L, const int32_t *perm, const int32_t *sub_off,
               const int32_t *cl_n, const double *cl_mu, const double *cl_var,
               const double *cl_vbar, const int32_t *sub_n, const double *sub_mu,
               const double *sub_var, const double *sub_vbar, const int32_t *sel_c,
               const int32_t *sel_s, int64_t tc, int64_t ts, int residual, double *out,
               double *diag)
{
    if (d <= 0 || n_now < n_build || L <= 0 || C < 0)
        return ORA_EINVAL;
    double *q = malloc((size_t)d * sizeof(double));
    char *csel = calloc((size_t)(C > 0 ? C : 1), 1);
    char *ssel = calloc((size_t)(C * L > 0 ? C * L : 1), 1);
    int64_t cap = n_now + C + C * L + 1;
    int64_t *epos = malloc((size_t)cap * sizeof(int64_t)); /* exact positions */
    double *elog = malloc((size_t)cap * sizeof(double));   /* their logits */
    int64_t *rgrp = malloc((size_t)cap * sizeof(int64_t)); /* residual groups (<0: cluster) */
    double *rexp = malloc((size_t)cap * sizeof(double));
    if (!q || !csel || !ssel || !epos || !elog || !rgrp || !rexp) {
        free(q); free(csel); free(ssel); free(epos); free(elog); free(rgrp); free(rexp);
        return ORA_ENOMEM;
    }
    bf_vec(q_bf16, d, q);
    int64_t ne = 0, nr = 0;
    /* R1: anchors */
    int64_t s_hi = S < n_now ? S : n_now;
    for (int64_t p = 0; p < s_hi; ++p)
        epos[ne++] = p;
    int64_t r_lo = n_build - R > S ? n_build - R : S;
    for (int64_t p = r_lo; p < n_now; ++p)
        epos[ne++] = p;
    /* members of the selected subclusters */
    for (int64_t i = 0; i < tc; ++i) {
        if (sel_c[i] < 0)
            continue;
        int64_t c = sel_c[i];
        csel[c] = 1;
        for (int64_t r = 0; r < ts; ++r) {
            if (sel_s[i * ts + r] < 0)
                continue;
            int64_t g = c * L + sel_s[i * ts + r];
            ssel[g] = 1;
            for (int64_t t = sub_off[g]; t < sub_off[g + 1]; ++t)
                epos[ne++] = perm[t];
        }
    }
    for (int64_t e = 0; e < ne; ++e) {
        const uint16_t *kr = K + epos[e] * ld;
        double dot = 0.0;
        for (int64_t j = 0; j < d; ++j)
            dot = dot + q[j] * bf(kr[j]);
        elog[e] = tau * dot;
    }
    /* R12: residual groups */
    if (residual) {
        for (int64_t c = 0; c < C; ++c) {
            if (cl_n[c] <= 0)
                continue;
            if (!csel[c]) {
                rgrp[nr] = -1 - c;
                rexp[nr++] = log_mass(q, d, tau, cl_n[c], cl_mu + c * d, cl_var + c * d);
                continue;
            }
            for (int64_t l = 0; l < L; ++l) {
                int64_t g = c * L + l;
                if (sub_n[g] <= 0 || ssel[g])
                    continue;
                rgrp[nr] = g;
                rexp[nr++] = log_mass(q, d, tau, sub_n[g], sub_mu + g * d, sub_var + g * d);
            }
        }
    }
    /* R13: one max over everything, then a single normalisation */
    double m = -INFINITY;
    for (int64_t e = 0; e < ne; ++e)
        if (elog[e] > m)
            m = elog[e];
    for (int64_t r = 0; r < nr; ++r)
        if (rexp[r] > m)
            m = rexp[r];
    double den = 0.0;
    for (int64_t j = 0; j < d; ++j)
        out[j] = 0.0;
    for (int64_t e = 0; e < ne; ++e) {
        double w = exp(elog[e] - m);
        const uint16_t *vr = V + epos[e] * ld;
        den = den + w;
        for (int64_t j = 0; j < d; ++j)
            out[j] = out[j] + w * bf(vr[j]);
    }
    for (int64_t r = 0; r < nr; ++r) {
        double w = exp(rexp[r] - m);
        const double *vb = rgrp[r] < 0 ? cl_vbar + (-1 - rgrp[r]) * d : sub_vbar + rgrp[r] * d;
        den = den + w;
        for (int64_t j = 0; j < d; ++j)
            out[j] = out[j] + w * vb[j];
    }
    for (int64_t j = 0; j < d; ++j)
        out[j] = den > 0.0 ? out[j] / den : 0.0;
    if (diag) {
        diag[0] = m;
        diag[1] = den;
        diag[2] = (double)ne;
    }
    free(q); free(csel); free(ssel); free(epos); free(elog); free(rgrp); free(rexp);
    return ORA_OK;
}

/* ---------------------------------------------------------------------------------
 * The feature-map residual (R29, [RC])
 * ------------------------------------------------------------------------------- */

/* log(phi(q~).phi(k~)): log of (1/m) sum_i exp(w_i.q~ - |q~|^2/2 + w_i.k~ - |k~|^2/2),
 * summed with the largest term factored out. */
static double log_feature_kernel(const double *qt, const double *kt, const double *omega,
                                 int64_t m, int64_t d, double *tmp)
{
    double qq = 0.0, kk = 0.0;
    for (int64_t j = 0; j < d; ++j) {
        qq = qq + qt[j] * qt[j];
        kk = kk + kt[j] * kt[j];
    }
    double mx = -INFINITY;
    for (int64_t i = 0; i < m; ++i) {
        double a = 0.0, b = 0.0;
        for (int64_t j = 0; j < d; ++j) {
            a = a + omega[i * d + j] * qt[j];
            b = b + omega[i * d + j] * kt[j];
        }
        tmp[i] = a - 0.5 * qq + b - 0.5 * kk;
        if (tmp[i] > mx)
            mx = tmp[i];
    }
    double acc = 0.0;
    for (int64_t i = 0; i < m; ++i)
        acc = acc + exp(tmp[i] - mx);
    return mx + log(acc) - log((double)m);
}

/*
 * Decode of one query head with the feature-map residual (R29): the exact part over the
 * anchors and the members of the selected subclusters (sel_c, sel_s as ora_decode), and
 * the estimate phi(q~).phi(k~) for every other mid key; omega [m][d].
 *   out[d]; diag (or NULL): [max log-weight, denominator, exact rows, estimated keys]
 */
int ora_decode_fm(const uint16_t *K, const uint16_t *V, int64_t ld, int64_t d, int64_t n_now,
                  int64_t n_build, int64_t S, int64_t R, const uint16_t *q_bf16, double tau,
                  int64_t C, int64_t L, const int32_t *perm, const int32_t *sub_off,
                  const int32_t *sel_c, const int32_t *sel_s, int64_t tc, int64_t ts,
                  const double *omega, int64_t m, double *out, double *diag)
{
    if (d <= 0 || n_now < n_build || L <= 0 || C < 0 || m <= 0)
        return ORA_EINVAL;
    int64_t mid_lo = S, mid_hi = n_build - R > S ? n_build - R : S;
    double *q = malloc((size_t)d * sizeof(double));
    double *qt = malloc((size_t)d * sizeof(double));
    double *kt = malloc((size_t)d * sizeof(double));
    double *tmp = malloc((size_t)m * sizeof(double));
    char *exact = calloc((size_t)(n_now > 0 ? n_now : 1), 1);
    double *lw = malloc((size_t)(n_now > 0 ? n_now : 1) * sizeof(double)); /* log-weights */
    if (!q || !qt || !kt || !tmp || !exact || !lw) {
        free(q); free(qt); free(kt); free(tmp); free(exact); free(lw);
        return ORA_ENOMEM;
    }
    bf_vec(q_bf16, d, q);
    double st = sqrt(tau);
    for (int64_t j = 0; j < d; ++j)
        qt[j] = st * q[j];
    /* R1: anchors; then the members of the selected subclusters */
    for (int64_t p = 0; p < (S < n_now ? S : n_now); ++p)
        exact[p] = 1;
    for (int64_t p = mid_hi; p < n_now; ++p)
        exact[p] = 1;
    for (int64_t i = 0; i < tc; ++i) {
        if (sel_c[i] < 0)
            continue;
        for (int64_t r = 0; r < ts; ++r) {
            if (sel_s[i * ts + r] < 0)
                continue;
            int64_t g = sel_c[i] * L + sel_s[i * ts + r];
            for (int64_t t = sub_off[g]; t < sub_off[g + 1]; ++t)
                exact[perm[t]] = 1;
        }
    }
    int64_t ne = 0, nf = 0;
    double mx = -INFINITY;
    for (int64_t p = 0; p < n_now; ++p) {
        const uint16_t *kr = K + p * ld;
        if (exact[p]) {
            double dot = 0.0;
            for (int64_t j = 0; j < d; ++j)
                dot = dot + q[j] * bf(kr[j]);
            lw[p] = tau * dot;
            ++ne;
        } else if (p >= mid_lo && p < mid_hi) {
            for (int64_t j = 0; j < d; ++j)
                kt[j] = st * bf(kr[j]);
            lw[p] = log_feature_kernel(qt, kt, omega, m, d, tmp);
            ++nf;
        } else {
            lw[p] = -INFINITY; /* beyond the build's mid region and not an anchor: none */
        }
        if (lw[p] > mx)
            mx = lw[p];
    }
    double den = 0.0;
    for (int64_t j = 0; j < d; ++j)
        out[j] = 0.0;
    for (int64_t p = 0; p < n_now; ++p) {
        if (lw[p] == -INFINITY)
            continue;
        double w = exp(lw[p] - mx);
        const uint16_t *vr = V + p * ld;
        den = den + w;
        for (int64_t j = 0; j < d; ++j)
            out[j] = out[j] + w * bf(vr[j]);
    }
    for (int64_t j = 0; j < d; ++j)
        out[j] = den > 0.0 ? out[j] / den : 0.0;
    if (diag) {
        diag[0] = mx;
        diag[1] = den;
        diag[2] = (double)ne;
        diag[3] = (double)nf;
    }
    free(q); free(qt); free(kt); free(tmp); free(exact); free(lw);
    return ORA_OK;
}

/*
 * The feature sums of every subcluster (R29), unscaled: for subcluster g and feature i,
 * z[(g*m + i)*(d+1) + j] = sum over its members k of exp(w_i.k~ - |k~|^2/2) v_kj for j < d,
 * and the same sum of exp(...) alone at j = d.
 */
int ora_fm_sums(const uint16_t *K, const uint16_t *V, int64_t ld, int64_t d, const int32_t *perm,
                const int32_t *sub_off, int64_t C, int64_t L, double tau, const double *omega,
                int64_t m, double *z)
{
    if (d <= 0 || C < 0 || L <= 0 || m <= 0)
        return ORA_EINVAL;
    double *kt = malloc((size_t)d * sizeof(double));
    if (!kt)
        return ORA_ENOMEM;
    double st = sqrt(tau);
    memset(z, 0, (size_t)(C * L * m * (d + 1)) * sizeof(double));
    for (int64_t g = 0; g < C * L; ++g) {
        for (int64_t t = sub_off[g]; t < sub_off[g + 1]; ++t) {
            const uint16_t *kr = K + (int64_t)perm[t] * ld, *vr = V + (int64_t)perm[t] * ld;
            double kk = 0.0;
            for (int64_t j = 0; j < d; ++j) {
                kt[j] = st * bf(kr[j]);
                kk = kk + kt[j] * kt[j];
            }
            for (int64_t i = 0; i < m; ++i) {
                double a = 0.0;
                for (int64_t j = 0; j < d; ++j)
                    a = a + omega[i * d + j] * kt[j];
                double f = exp(a - 0.5 * kk);
                double *zr = z + (g * m + i) * (d + 1);
                for (int64_t j = 0; j < d; ++j)
                    zr[j] = zr[j] + f * bf(vr[j]);
                zr[d] = zr[d] + f;
            }
        }
    }
    free(kt);
    return ORA_OK;
}

/* Exact softmax attention of one query over keys [0, n): the full-scan comparison. */
int ora_dense(const uint16_t *K, const uint16_t *V, int64_t ld, int64_t d, int64_t n,
              const uint16_t *q_bf16, double tau, double *out)
{
    if (d <= 0 || n < 0)
        return ORA_EINVAL;
    double *q = malloc((size_t)d * sizeof(double));
    double *lg = malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
    if (!q || !lg) {
        free(q); free(lg);
        return ORA_ENOMEM;
    }
    bf_vec(q_bf16, d, q);
    double m = -INFINITY;
    for (int64_t i = 0; i < n; ++i) {
        const uint16_t *kr = K + i * ld;
        double dot = 0.0;
        for (int64_t j = 0; j < d; ++j)
            dot = dot + q[j] * bf(kr[j]);
        lg[i] = tau * dot;
        if (lg[i] > m)
            m = lg[i];
    }
    double den = 0.0;
    for (int64_t j = 0; j < d; ++j)
        out[j] = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        double w = exp(lg[i] - m);
        const uint16_t *vr = V + i * ld;
        den = den + w;
        for (int64_t j = 0; j < d; ++j)
            out[j] = out[j] + w * bf(vr[j]);
    }
    for (int64_t j = 0; j < d; ++j)
        out[j] = den > 0.0 ? out[j] / den : 0.0;
    free(q); free(lg);
    return ORA_OK;
}
