/*
 * fp64 CPU oracle for the row-wise log-softmax / token cross-entropy path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this code; the product path never
 * does, and it shares no code, header or constant with the CUDA library.
 *
 * It is deliberately plain: one row at a time, every sum in fp64 with
 * Neumaier compensation, no blocking, no fusion, no reordering beyond what
 * the definitions below state.  Rows are spread over OpenMP threads only so
 * that the full-size workloads finish; each row's arithmetic is serial.
 *
 * Definitions (z_j = x_j / T, T the exact value of the fp32 temperature):
 *
 *   others(t)      = { j in [0,V) : j != t }
 *   lse_others(t)  = max_{j in others(t)} z_j
 *                    + log sum_{j in others(t)} exp(z_j - max)
 *   log p_t        = -softplus(lse_others(t) - z_t)
 *   softplus(a)    = max(a, 0) + log1p(exp(-|a|))
 *
 * This is the fp64 reference written as softplus(lse_others - x_y) that
 * "Fix softmax collapse in CE, GRPO, KL/JSD and softmax" (Liger-Kernel PR
 * #1555, section "Details") compares against, because a plain fp64
 * x_y - logsumexp(x) itself collapses once the target leads the rest by
 * more than about 36.7.  Mathematically it equals z_t - logsumexp_j z_j.
 *
 * Cross-entropy (same page, "Summary", first bullet; ms-swift PR #10353
 * "PR information", second bullet):
 *   loss_r  = -log p_{y_r}  for rows whose label is not ignore_index, else 0
 *   sum     = sum_r loss_r;  mean = sum / n_items, n_items = #non-ignored
 *             rows, and mean = 0 when n_items = 0 (all rows ignored)
 *   dlogits = g_r * d(loss)/dx = (g_r/T) * (softmax(z) - onehot(y)):
 *     j != y : (g_r/T) * exp(z_j - z_y + log p_y)
 *     j == y : (g_r/T) * expm1(log p_y)
 *   where the target term is the "-expm1(log p_t)" form of the unsloth-zoo
 *   fix quoted on the same page (commit #2080, section "Fix", backward
 *   bullet), so it never rounds to zero; ignored rows get a zero row
 *   (ms-swift PR #10353: zero upstream weight for ignored labels).
 *   g_r = grad_out[r] (reduction none), grad_out[0] (sum),
 *         grad_out[0] / n_items (mean).
 *
 * Selective log-softmax ("perf(rlhf): chunk selective_log_softmax instead
 * of looping per token", ms-swift PR #10337, "PR information": the naive
 * gather(logits.log_softmax(-1)) with top-K indices, temperature and a row
 * mask): out[r,k] = log p_{idx[r,k]} for rows with row_mask[r] != 0, and 0
 * for masked-out rows, which are not read.
 *
 * Selective log-softmax backward (the gradient a GRPO-style loss sends
 * through the gathered log-probs; "Fix softmax collapse ..." page, "Summary",
 * second bullet, and the unsloth-zoo #2080 "Fix" section's -expm1(log p_t)):
 * with upstream g_k = dL/d out[r,k] and G = sum_k g_k,
 *   dL/dx_j = (1/T) * ( sum_{k : idx[r,k] = j} g_k  -  G * p_j ),
 * written at a gathered column t (g_t = sum of g_k over the k that gather t)
 * as (1/T) * ( -g_t * expm1(log p_t) - (G - g_t) * exp(log p_t) ), which
 * keeps 1 - p_t exact when p_t rounds to 1; masked-out rows get a zero row.
 *
 * Entropy of a row's softmax (the per-token entropy the unsloth-zoo #2080
 * commit computes beside the log-probs, "Fix"): H = -sum_j p_j log p_j.  The
 * reference column t (the label, or a row's first gathered index) enters
 * with its collapse-safe log p_t, every other column with
 * log p_j = z_j - lse, lse = z_t - log p_t; so a row whose t holds almost all
 * of the mass keeps its small positive entropy instead of rounding to 0.
 *
 * An index or label outside [0,V) (and, for labels, not ignore_index)
 * makes that row's outputs NaN and is counted in the return value.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Neumaier (Kahan-Babuska) compensated running sum. */
typedef struct {
    double sum;
    double comp;
} oracle_sum;

static void sum_add(oracle_sum *acc, double v)
{
    double t = acc->sum + v;
    if (fabs(acc->sum) >= fabs(v))
        acc->comp += (acc->sum - t) + v;
    else
        acc->comp += (v - t) + acc->sum;
    acc->sum = t;
}

static double sum_value(const oracle_sum *acc) { return acc->sum + acc->comp; }

/* log sum_{j != skip} exp(x_j / T); -inf when the set is empty. */
static double lse_excluding(const double *x, int64_t V, int64_t skip, double T)
{
    double m = -INFINITY;
    for (int64_t j = 0; j < V; ++j) {
        if (j == skip)
            continue;
        double z = x[j] / T;
        if (z > m)
            m = z;
    }
    if (m == -INFINITY)
        return -INFINITY;
    oracle_sum s = {0.0, 0.0};
    for (int64_t j = 0; j < V; ++j) {
        if (j == skip)
            continue;
        sum_add(&s, exp(x[j] / T - m));
    }
    return m + log(sum_value(&s));
}

static double softplus(double a)
{
    if (a == -INFINITY)
        return 0.0;
    return fmax(a, 0.0) + log1p(exp(-fabs(a)));
}

/* log p_t of one row: -softplus(lse_others(t) - z_t). */
static double row_logp(const double *x, int64_t V, int64_t t, double T)
{
    return -softplus(lse_excluding(x, V, t, T) - x[t] / T);
}

/* -p log p for p = e^lp, with 0 log 0 = 0. */
static double neg_plogp(double lp)
{
    const double p = exp(lp);
    return p == 0.0 ? 0.0 : -p * lp;
}

/* The first column holding a row's largest logit (its dominant column). */
static int64_t row_argmax(const double *x, int64_t V)
{
    int64_t d = 0;
    for (int64_t j = 1; j < V; ++j)
        if (x[j] > x[d])
            d = j;
    return d;
}

/*
 * -sum_j p_j log p_j of one row.  The dominant column d enters with its
 * accurate log p (the collapse-safe form), every other column with
 * z_j - lse, lse = z_d - log p_d.  A row whose mass sits almost all on one
 * column thus keeps its small entropy, whichever column that is: the value
 * depends on the row alone.
 */
static double row_entropy(const double *x, int64_t V, double T)
{
    const int64_t d = row_argmax(x, V);
    const double lp_d = row_logp(x, V, d, T);
    /* logsumexp of all columns; the others' alone when p_d is exactly 0 */
    const double lse = lp_d == -INFINITY ? lse_excluding(x, V, d, T) : x[d] / T - lp_d;
    oracle_sum h = {0.0, 0.0};
    sum_add(&h, neg_plogp(lp_d));
    for (int64_t j = 0; j < V; ++j) {
        if (j == d)
            continue;
        sum_add(&h, neg_plogp(x[j] / T - lse));
    }
    return sum_value(&h);
}

/*
 * Row entropy.
 *   x        [rows, ld] fp64
 *   ref      [rows] int64: a column of each row (the sampled token); the
 *            entropy does not depend on it, but a row whose column is out
 *            of range gets NaN, as its log-prob does
 *   live     [rows] uint8 or NULL: rows with 0 are skipped (entropy 0)
 *   out      [rows] fp64
 * Returns the number of live rows whose reference column is out of range.
 */
int64_t oracle_entropy(const double *x, int64_t rows, int64_t V, int64_t ld, const int64_t *ref,
                       double T, const uint8_t *live, double *out)
{
    int64_t bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : bad)
    for (int64_t r = 0; r < rows; ++r) {
        if (live && live[r] == 0) {
            out[r] = 0.0;
            continue;
        }
        const int64_t t = ref[r];
        if (t < 0 || t >= V) {
            out[r] = NAN;
            ++bad;
            continue;
        }
        out[r] = row_entropy(x + r * ld, V, T);
    }
    return bad;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/*
 * Selective log-softmax.
 *   x        [rows, ld] fp64, row r at x + r*ld, first V entries used
 *   idx      [rows, K] int64
 *   row_mask [rows] uint8 or NULL (all rows live)
 *   out      [rows, K] fp64
 * Returns the number of out-of-range indices met in live rows.
 */
int64_t oracle_selective_logsoftmax(const double *x, int64_t rows, int64_t V, int64_t ld,
                                    const int64_t *idx, int64_t K, double T,
                                    const uint8_t *row_mask, double *out)
{
    int64_t bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : bad)
    for (int64_t r = 0; r < rows; ++r) {
        const double *xr = x + r * ld;
        for (int64_t k = 0; k < K; ++k) {
            double *o = out + r * K + k;
            if (row_mask && row_mask[r] == 0) {
                *o = 0.0;
                continue;
            }
            int64_t t = idx[r * K + k];
            if (t < 0 || t >= V) {
                *o = NAN;
                ++bad;
                continue;
            }
            *o = row_logp(xr, V, t, T);
        }
    }
    return bad;
}

/*
 * Token cross-entropy, forward and (when dx != NULL) backward, with optional
 * label smoothing and DFT weighting.  For a kept row with label y,
 *   loss_r = w_r * ((1 - eps) * (-log p_y) + eps * mean_j(-log p_j))
 * (the smoothed target puts 1 - eps on y and eps / V on every class), and
 *   dz_j = g_r * w_r * (p_j - (1 - eps) [j == y] - eps / V),  dx = dz / T,
 * where w_r = p_y, held constant (the detached DFT weight), when dft != 0,
 * else 1.  The label column of the gradient is written with expm1(log p_y)
 * for p_y - 1.
 *   x          [rows, ld] fp64
 *   labels     [rows] int64, ignore_index marks rows to skip
 *   reduction  0 = none, 1 = sum, 2 = mean
 *   eps        label smoothing in [0, 1]
 *   dft        nonzero: weight each row by its detached p_y
 *   grad_out   [rows] for none, [1] otherwise; may be NULL when dx == NULL
 *   logp_y     [rows] out: log p of the label (0 for ignored rows)
 *   loss_rows  [rows] out: the row's loss above (0 for ignored rows)
 *   loss       [1] out: the reduced loss (sum for none, for reference)
 *   n_items    [1] out: number of rows whose label is not ignore_index
 *   dx         [rows, ldx] out or NULL
 * Returns the number of rows whose label is out of range.
 */
static int64_t ce_core(const double *x, int64_t rows, int64_t V, int64_t ld,
                       const int64_t *labels, int64_t ignore_index, double T, int reduction,
                       double eps, int dft, const double *grad_out, double *logp_y,
                       double *loss_rows, double *loss, int64_t *n_items, double *dx,
                       int64_t ldx)
{
    int64_t count = 0;
    for (int64_t r = 0; r < rows; ++r)
        if (labels[r] != ignore_index)
            ++count;
    *n_items = count;

    int64_t bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : bad)
    for (int64_t r = 0; r < rows; ++r) {
        const double *xr = x + r * ld;
        int64_t y = labels[r];
        if (y == ignore_index) {
            logp_y[r] = 0.0;
            loss_rows[r] = 0.0;
        } else if (y < 0 || y >= V) {
            logp_y[r] = NAN;
            loss_rows[r] = NAN;
            ++bad;
        } else {
            const double lp = row_logp(xr, V, y, T);
            logp_y[r] = lp;
            double loss_r = -lp;
            if (eps != 0.0) {
                /* mean over all classes of -log p_j, -log p_j = lse - z_j */
                const double lse = xr[y] / T - lp;
                oracle_sum nl = {0.0, 0.0};
                sum_add(&nl, -lp);
                for (int64_t j = 0; j < V; ++j)
                    if (j != y)
                        sum_add(&nl, lse - xr[j] / T);
                loss_r = (1.0 - eps) * (-lp) + eps * (sum_value(&nl) / (double)V);
            }
            loss_rows[r] = dft ? exp(lp) * loss_r : loss_r;
        }
    }

    oracle_sum total = {0.0, 0.0};
    for (int64_t r = 0; r < rows; ++r)
        sum_add(&total, loss_rows[r]);
    if (reduction == 2)
        *loss = count > 0 ? sum_value(&total) / (double)count : 0.0;
    else
        *loss = sum_value(&total);

    if (dx == NULL)
        return bad;

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < rows; ++r) {
        const double *xr = x + r * ld;
        double *dr = dx + r * ldx;
        int64_t y = labels[r];
        if (y == ignore_index) {
            for (int64_t j = 0; j < V; ++j)
                dr[j] = 0.0;
            continue;
        }
        if (y < 0 || y >= V) {
            for (int64_t j = 0; j < V; ++j)
                dr[j] = NAN;
            continue;
        }
        double g;
        if (reduction == 0)
            g = grad_out[r];
        else if (reduction == 1)
            g = grad_out[0];
        else
            g = count > 0 ? grad_out[0] / (double)count : 0.0;
        double lp = logp_y[r];
        double scale = (dft ? exp(lp) * g : g) / T;
        double zy = xr[y] / T;
        const double u = eps / (double)V;
        for (int64_t j = 0; j < V; ++j) {
            if (j == y)
                dr[j] = scale * (expm1(lp) + (eps - u));
            else
                dr[j] = scale * (exp(xr[j] / T - zy + lp) - u);
        }
    }
    return bad;
}

/*
 * The exported cross-entropy: ce_core above, with optional logit soft-capping.
 * softcap > 0 replaces every logit x by cap * tanh(x / cap) before the
 * temperature and the softmax (a per-element transform of the logits), and
 * the gradient with respect to x takes the chain factor
 * d/dx [cap tanh(x / cap)] = sech^2(x / cap), written as 1 / cosh^2: the
 * equal form 1 - tanh^2 loses its digits once tanh rounds to +-1 (|x / cap|
 * of about 19 in fp64), where the factor is still far above fp64's range.
 */
int64_t oracle_cross_entropy(const double *x, int64_t rows, int64_t V, int64_t ld,
                             const int64_t *labels, int64_t ignore_index, double T,
                             int reduction, double eps, int dft, double softcap,
                             const double *grad_out, double *logp_y, double *loss_rows,
                             double *loss, int64_t *n_items, double *dx, int64_t ldx)
{
    if (!(softcap > 0.0))
        return ce_core(x, rows, V, ld, labels, ignore_index, T, reduction, eps, dft, grad_out,
                       logp_y, loss_rows, loss, n_items, dx, ldx);
    double *z = (double *)malloc((size_t)rows * (size_t)V * sizeof(double));
    if (z == NULL)
        return -1;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t j = 0; j < V; ++j)
            z[r * V + j] = softcap * tanh(x[r * ld + j] / softcap);
    const int64_t bad = ce_core(z, rows, V, V, labels, ignore_index, T, reduction, eps, dft,
                                grad_out, logp_y, loss_rows, loss, n_items, dx, ldx);
    if (dx != NULL) {
#pragma omp parallel for schedule(static)
        for (int64_t r = 0; r < rows; ++r)
            for (int64_t j = 0; j < V; ++j) {
                const double sech = 1.0 / cosh(x[r * ld + j] / softcap);
                dx[r * ldx + j] *= sech * sech;
            }
    }
    free(z);
    return bad;
}

/* Forward declarations: the entropy term of the backward below uses them. */
static double row_entropy(const double *x, int64_t V, double T);
static int64_t row_argmax(const double *x, int64_t V);

/*
 * Selective log-softmax backward, optionally with an entropy term.
 *   x         [rows, ld] fp64
 *   idx       [rows, K] int64
 *   row_mask  [rows] uint8 or NULL
 *   grad      [rows, K] fp64: dL/d out[r, k]
 *   grad_ent  [rows] fp64 or NULL: dL/d H_r, H_r = -sum_j p_j log p_j; it
 *             adds -(grad_ent / T) p_j (log p_j + H_r) to column j (the
 *             derivative of the entropy, written out), 0 where p_j = 0.
 *             For the row's dominant column d, log p_d + H_r is taken as
 *             sum_{j != d} p_j (z_d - z_j), the same number (H_r = lse -
 *             sum_j p_j z_j) as a sum of non-negative terms: the difference
 *             itself cancels when p_d is near 1.
 *   dx        [rows, ldx] out
 * Returns the number of rows with an out-of-range index (their rows NaN).
 */
int64_t oracle_selective_logsoftmax_backward(const double *x, int64_t rows, int64_t V,
                                             int64_t ld, const int64_t *idx, int64_t K, double T,
                                             const uint8_t *row_mask, const double *grad,
                                             const double *grad_ent, double *dx, int64_t ldx)
{
    int64_t bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : bad)
    for (int64_t r = 0; r < rows; ++r) {
        const double *xr = x + r * ld;
        double *dr = dx + r * ldx;
        if (row_mask && row_mask[r] == 0) {
            for (int64_t j = 0; j < V; ++j)
                dr[j] = 0.0;
            continue;
        }
        int row_bad = 0;
        for (int64_t k = 0; k < K; ++k)
            if (idx[r * K + k] < 0 || idx[r * K + k] >= V)
                row_bad = 1;
        if (row_bad) {
            for (int64_t j = 0; j < V; ++j)
                dr[j] = NAN;
            ++bad;
            continue;
        }
        /* log-sum-exp of the whole row, then p_j = exp(z_j - lse) */
        double m = -INFINITY;
        for (int64_t j = 0; j < V; ++j)
            if (xr[j] / T > m)
                m = xr[j] / T;
        oracle_sum s = {0.0, 0.0};
        for (int64_t j = 0; j < V; ++j)
            sum_add(&s, exp(xr[j] / T - m));
        const double lse = m + log(sum_value(&s));
        oracle_sum G = {0.0, 0.0};
        for (int64_t k = 0; k < K; ++k)
            sum_add(&G, grad[r * K + k]);
        const double Gv = sum_value(&G);
        const double gH = grad_ent ? grad_ent[r] : 0.0;
        const double H = grad_ent ? row_entropy(xr, V, T) : 0.0;
        const int64_t d = row_argmax(xr, V);
        oracle_sum q = {0.0, 0.0};
        if (gH != 0.0)
            for (int64_t j = 0; j < V; ++j) {
                const double pj = exp(xr[j] / T - lse);
                if (j != d && pj != 0.0)
                    sum_add(&q, pj * ((xr[d] - xr[j]) / T));
            }
        const double Hd = sum_value(&q); /* log p_d + H */
        for (int64_t j = 0; j < V; ++j) {
            const double lpj = xr[j] / T - lse;
            const double pj = exp(lpj);
            dr[j] = -(Gv / T) * pj;
            if (gH != 0.0 && pj != 0.0)
                dr[j] -= (gH / T) * pj * (j == d ? Hd : lpj + H);
        }
        /* gathered columns, each once, in the collapse-safe form */
        for (int64_t k = 0; k < K; ++k) {
            const int64_t t = idx[r * K + k];
            int seen = 0;
            for (int64_t i = 0; i < k; ++i)
                if (idx[r * K + i] == t)
                    seen = 1;
            if (seen)
                continue;
            oracle_sum gt = {0.0, 0.0};
            for (int64_t i = 0; i < K; ++i)
                if (idx[r * K + i] == t)
                    sum_add(&gt, grad[r * K + i]);
            const double g_t = sum_value(&gt);
            const double lp = row_logp(xr, V, t, T);
            dr[t] = (-g_t * expm1(lp) - (Gv - g_t) * exp(lp)) / T;
            if (gH != 0.0 && exp(lp) != 0.0)
                dr[t] -= (gH / T) * exp(lp) * (t == d ? Hd : lp + H);
        }
    }
    return bad;
}
