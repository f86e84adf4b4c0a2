/*
 * oracle.c -- plain, slow, fp64 CPU reference for the symbolic kernel reductions.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or load
 * this file: only the test suite, the smoke check and the CPU-baseline leg of the
 * benchmark use it.  It shares no code, header, table or helper with the CUDA
 * library; it is written from the definitions, in the order the definitions give,
 * with no blocking, fusion or reordering, so that it can be checked by eye.
 *
 * Every input array arrives as double (the caller converts the fp32 arrays the GPU
 * sees, which is exact).  Layouts are row-major and contiguous:
 *   x : M x D      y : N x D      b, w : N x E      g : M x E
 * Rows i are independent, so a caller may pass any subset of the rows of x (and
 * of g) and get exactly those rows of the result.
 *
 * Sources (the pages this follows):
 *  - "Kernel Operations on the GPU, with Autodiff, without Memory Overflows",
 *    §1 Introduction, "Target operation": a_i = sum_j k(x_i, y_j) b_j with a
 *    Gaussian k of deviation sigma; §2 "Generic reduction framework" and
 *    "Performance and differentiation": sum, logsumexp, min, argmin, argKmin
 *    reductions and gradients through autodiff.
 *  - KeOps README, PyTorch usage example: D_ij = sum_d (x_id - y_jd)^2,
 *    K_ij = exp(-D_ij), a_i = sum_j K_ij, and the gradient of sum_i a_i^2 wrt x;
 *    feature list: Sum, LogSumExp, ArgMin and K-min reductions.
 *  Readings where the pages leave a step open (all listed in the design notes):
 *  - the Gaussian is exp(-|x - y|^2 / sigma^2) (the example has sigma = 1);
 *  - LogSumExp takes an additive log-weight w_je per column: log sum_j exp(t_ij + w_je)
 *    with t_ij = -|x_i - y_j|^2 / sigma^2, one independent reduction per column e;
 *  - K-min orders candidates by the pair (distance, index), so ties keep the lowest
 *    index; slots beyond N get index -1 and distance +inf;
 *  - N = 0: the sum is 0 and the LogSumExp is -inf.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Number of threads the OpenMP loops below use. */
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
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Squared Euclidean distance between row i of x and row j of y (KeOps README,
 * usage example: D_ij = ((x_i - y_j)**2).sum over the coordinate axis). */
static double sq_dist(const double *xi, const double *yj, int D)
{
    double s = 0.0;
    for (int d = 0; d < D; ++d) {
        double diff = xi[d] - yj[d];
        s += diff * diff;
    }
    return s;
}

/* Gaussian kernel value k(x_i, y_j) = exp(-|x_i - y_j|^2 / sigma^2)
 * ("Kernel Operations on the GPU...", §1, target operation; sigma > 0). */
static double gauss(const double *xi, const double *yj, int D, double sigma)
{
    return exp(-sq_dist(xi, yj, D) / (sigma * sigma));
}

/* Neumaier's compensated summation: adds v to the running (sum, comp) pair. */
static void neumaier_add(double *sum, double *comp, double v)
{
    double t = *sum + v;
    if (fabs(*sum) >= fabs(v))
        *comp += (*sum - t) + v;
    else
        *comp += (v - t) + *sum;
    *sum = t;
}

/*
 * Sum reduction: a_ie = sum_j k(x_i, y_j) b_je, summed in increasing j.
 * Also writes the tolerance scale S_ie = sum_j |k(x_i, y_j) b_je|.
 * ("Kernel Operations on the GPU...", §1 target operation; KeOps README,
 * a_i = K_ij.sum(dim=1).)
 */
void oracle_gauss_sum(const double *x, const double *y, const double *b,
                      int64_t M, int64_t N, int D, int E, double sigma,
                      double *a, double *scale)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < M; ++i) {
        for (int e = 0; e < E; ++e) {
            double s = 0.0, c = 0.0, sa = 0.0, ca = 0.0;
            for (int64_t j = 0; j < N; ++j) {
                double k = gauss(x + i * D, y + j * D, D, sigma);
                double term = k * b[j * E + e];
                neumaier_add(&s, &c, term);
                neumaier_add(&sa, &ca, fabs(term));
            }
            a[i * E + e] = s + c;
            if (scale) scale[i * E + e] = sa + ca;
        }
    }
}

/*
 * LogSumExp reduction: L_ie = log sum_j exp(t_ij + w_je), t_ij = -|x_i - y_j|^2 / sigma^2.
 * Computed the textbook stable way in two passes: m = max_j (t_ij + w_je), then
 * L = m + log sum_j exp(t_ij + w_je - m).  N = 0 gives -inf.
 * (KeOps README, reductions .logsumexp(); feature list "LogSumExp".)
 */
void oracle_gauss_lse(const double *x, const double *y, const double *w,
                      int64_t M, int64_t N, int D, int E, double sigma,
                      double *L)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < M; ++i) {
        for (int e = 0; e < E; ++e) {
            if (N == 0) { L[i * E + e] = -INFINITY; continue; }
            double m = -INFINITY;
            for (int64_t j = 0; j < N; ++j) {
                double t = -sq_dist(x + i * D, y + j * D, D) / (sigma * sigma) + w[j * E + e];
                if (t > m) m = t;
            }
            double s = 0.0, c = 0.0;
            for (int64_t j = 0; j < N; ++j) {
                double t = -sq_dist(x + i * D, y + j * D, D) / (sigma * sigma) + w[j * E + e];
                neumaier_add(&s, &c, exp(t - m));
            }
            L[i * E + e] = m + log(s + c);
        }
    }
}

/*
 * Gradient wrt x of the scalar sum_{i,e} g_ie a_ie, where a is the Sum reduction:
 *   d/dx_id exp(-|x_i - y_j|^2 / sigma^2) = -(2 / sigma^2) (x_id - y_jd) k(x_i, y_j),
 * so  gx_id = -(2 / sigma^2) sum_j k(x_i, y_j) (sum_e g_ie b_je) (x_id - y_jd).
 * With g = 2a this is the gradient of sum_i |a_i|^2 (KeOps README,
 * torch.autograd.grad((a_i ** 2).sum(), [x])).
 * Also writes the tolerance scale
 *   G_id = (2 / sigma^2) sum_j k(x_i, y_j) |sum_e g_ie b_je| |x_id - y_jd|.
 */
void oracle_gauss_grad_x(const double *x, const double *y, const double *b,
                         const double *g, int64_t M, int64_t N, int D, int E,
                         double sigma, double *gx, double *G)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < M; ++i) {
        for (int d = 0; d < D; ++d) {
            double s = 0.0, c = 0.0, sa = 0.0, ca = 0.0;
            for (int64_t j = 0; j < N; ++j) {
                double k = gauss(x + i * D, y + j * D, D, sigma);
                double beta = 0.0;
                for (int e = 0; e < E; ++e) beta += g[i * E + e] * b[j * E + e];
                double diff = x[i * D + d] - y[j * D + d];
                double term = -(2.0 / (sigma * sigma)) * k * beta * diff;
                neumaier_add(&s, &c, term);
                neumaier_add(&sa, &ca, fabs(term));
            }
            gx[i * D + d] = s + c;
            if (G) G[i * D + d] = sa + ca;
        }
    }
}

/*
 * Gradient wrt y of the same scalar sum_{i,e} g_ie a_ie.  The kernel depends on
 * y_j through |x_i - y_j|^2, and d/dy_jd exp(-|x_i - y_j|^2 / sigma^2)
 *   = (2 / sigma^2) (x_id - y_jd) k(x_i, y_j), so
 *   gy_jd = (2 / sigma^2) sum_i k(x_i, y_j) (sum_e g_ie b_je) (x_id - y_jd),
 * summed in increasing i.  Rows j are independent: pass any subset of the rows
 * of y (with the matching rows of b) to get those rows of gy.
 * Also writes the tolerance scale
 *   G_jd = (2 / sigma^2) sum_i k(x_i, y_j) |sum_e g_ie b_je| |x_id - y_jd|.
 * ("Kernel Operations on the GPU...", §2 "Performance and differentiation":
 * gradients through torch.autograd with respect to every input.)
 */
void oracle_gauss_grad_y(const double *x, const double *y, const double *b,
                         const double *g, int64_t M, int64_t N, int D, int E,
                         double sigma, double *gy, double *G)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t j = 0; j < N; ++j) {
        for (int d = 0; d < D; ++d) {
            double s = 0.0, c = 0.0, sa = 0.0, ca = 0.0;
            for (int64_t i = 0; i < M; ++i) {
                double k = gauss(x + i * D, y + j * D, D, sigma);
                double beta = 0.0;
                for (int e = 0; e < E; ++e) beta += g[i * E + e] * b[j * E + e];
                double diff = x[i * D + d] - y[j * D + d];
                double term = (2.0 / (sigma * sigma)) * k * beta * diff;
                neumaier_add(&s, &c, term);
                neumaier_add(&sa, &ca, fabs(term));
            }
            gy[j * D + d] = s + c;
            if (G) G[j * D + d] = sa + ca;
        }
    }
}

/*
 * Gradient wrt b of sum_{i,e} g_ie a_ie.  a is linear in b, so
 *   gb_je = sum_i k(x_i, y_j) g_ie,
 * the transposed kernel product, summed in increasing i.  Rows j are independent.
 * Also writes the tolerance scale S_je = sum_i |k(x_i, y_j) g_ie|.
 * ("Kernel Operations on the GPU...", §2 "Performance and differentiation".)
 */
void oracle_gauss_grad_b(const double *x, const double *y, const double *g,
                         int64_t M, int64_t N, int D, int E, double sigma,
                         double *gb, double *scale)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t j = 0; j < N; ++j) {
        for (int e = 0; e < E; ++e) {
            double s = 0.0, c = 0.0, sa = 0.0, ca = 0.0;
            for (int64_t i = 0; i < M; ++i) {
                double term = gauss(x + i * D, y + j * D, D, sigma) * g[i * E + e];
                neumaier_add(&s, &c, term);
                neumaier_add(&sa, &ca, fabs(term));
            }
            gb[j * E + e] = s + c;
            if (scale) scale[j * E + e] = sa + ca;
        }
    }
}

/*
 * Other radial kernels of the squared distance q = |x - y|^2 and width sigma
 * ("Kernel Operations on the GPU...", §2: reductions of generic formulas F(x_i, y_j);
 * KeOps README: "support for a wide range of mathematical formulas").  kind:
 *   0 Gaussian               exp(-q / sigma^2)
 *   1 Laplace (exponential)  exp(-sqrt(q) / sigma)
 *   2 Cauchy                 1 / (1 + q / sigma^2)
 *   3 inverse multiquadric   1 / sqrt(1 + q / sigma^2)
 * Each is 1 at q = 0 and decreases to 0 as q grows.
 */
static double radial_kernel(int kind, double q, double sigma)
{
    switch (kind) {
    case 0: return exp(-q / (sigma * sigma));
    case 1: return exp(-sqrt(q) / sigma);
    case 2: return 1.0 / (1.0 + q / (sigma * sigma));
    case 3: return 1.0 / sqrt(1.0 + q / (sigma * sigma));
    default: return NAN;
    }
}

/*
 * Sum reduction with any of the radial kernels above:
 *   a_ie = sum_j k(x_i, y_j) b_je, summed in increasing j, with the scale
 *   S_ie = sum_j |k(x_i, y_j) b_je|.
 */
void oracle_kernel_sum(const double *x, const double *y, const double *b,
                       int64_t M, int64_t N, int D, int E, double sigma, int kind,
                       double *a, double *scale)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < M; ++i) {
        for (int e = 0; e < E; ++e) {
            double s = 0.0, c = 0.0, sa = 0.0, ca = 0.0;
            for (int64_t j = 0; j < N; ++j) {
                double k = radial_kernel(kind, sq_dist(x + i * D, y + j * D, D), sigma);
                double term = k * b[j * E + e];
                neumaier_add(&s, &c, term);
                neumaier_add(&sa, &ca, fabs(term));
            }
            a[i * E + e] = s + c;
            if (scale) scale[i * E + e] = sa + ca;
        }
    }
}

/*
 * Max (sense = +1) or Min (sense = -1) reduction of the formula F_ije = k(x_i, y_j) b_je
 * over j, with its Arg: val[i*E+e] = the extreme value, idx[i*E+e] = the lowest j
 * that attains it ("Kernel Operations on the GPU...", §2: max, min and argmin
 * reductions; KeOps README feature list: Min, Max, ArgMin, ArgMax).  N = 0 gives
 * -inf (Max) / +inf (Min) and index -1.
 * second[i*E+e] (if not NULL) is the best value over the other j (the runner-up,
 * equal to val when the extreme is attained twice); the parity tests use it to
 * find near-ties.  A plain scan in increasing j that replaces the best only on a
 * strictly better value.
 */
void oracle_kernel_maxmin(const double *x, const double *y, const double *b,
                          int64_t M, int64_t N, int D, int E, double sigma, int kind,
                          int sense, double *val, int64_t *idx, double *second)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < M; ++i) {
        for (int e = 0; e < E; ++e) {
            double best = sense > 0 ? -INFINITY : INFINITY, runner = best;
            int64_t bj = -1;
            for (int64_t j = 0; j < N; ++j) {
                double f = radial_kernel(kind, sq_dist(x + i * D, y + j * D, D), sigma) * b[j * E + e];
                int better = sense > 0 ? f > best : f < best;
                if (better) {
                    runner = best;
                    best = f;
                    bj = j;
                } else {
                    int beats_runner = sense > 0 ? f > runner : f < runner;
                    if (beats_runner || f == best) runner = f;
                }
            }
            val[i * E + e] = best;
            idx[i * E + e] = bj;
            if (second) second[i * E + e] = runner;
        }
    }
}

/*
 * Block-sparse (cluster-wise truncated) Sum, Max and Min ("Kernel Operations on the
 * GPU...", §3 "Applications": cluster-wise block-sparsity for large kernel systems;
 * §4: the block-sparse truncation rule; KeOps README: an interface for block-sparse
 * strategies).  The rows are grouped in clusters c = 0..nc-1, cluster c owning rows
 * [ranges_i[2c], ranges_i[2c+1]); cluster c reduces over the j-ranges
 * redranges_j[2r] <= j < redranges_j[2r+1] for r from slices_i[c-1] (0 for c = 0) to
 * slices_i[c] - 1.  A point listed in two ranges of a cluster counts twice in the Sum.
 *   red = 0: a_ie = sum over the cluster's ranges of k(x_i, y_j) b_je (+ scale S_ie)
 *   red = +1 / -1: the Max / Min of k(x_i, y_j) b_je over those j with the lowest j
 *   attaining it (val, idx, runner-up in second).
 * Rows in no cluster reduce over nothing: Sum 0, Max -inf, Min +inf, index -1.
 */
void oracle_kernel_ranges(const double *x, const double *y, const double *b,
                          int64_t M, int64_t N, int D, int E, double sigma, int kind, int red,
                          int64_t nc, const int64_t *ranges_i, const int64_t *slices_i,
                          const int64_t *redranges_j,
                          double *val, double *scale, int64_t *idx, double *second)
{
    (void)N;
    for (int64_t i = 0; i < M * E; ++i) {
        val[i] = red == 0 ? 0.0 : (red > 0 ? -INFINITY : INFINITY);
        if (scale) scale[i] = 0.0;
        if (idx) idx[i] = -1;
        if (second) second[i] = val[i];
    }
    for (int64_t c = 0; c < nc; ++c) {
        int64_t r0 = c == 0 ? 0 : slices_i[c - 1], r1 = slices_i[c];
#pragma omp parallel for schedule(dynamic, 1)
        for (int64_t i = ranges_i[2 * c]; i < ranges_i[2 * c + 1]; ++i) {
            for (int e = 0; e < E; ++e) {
                double s = 0.0, cs = 0.0, sa = 0.0, ca = 0.0;
                double best = red > 0 ? -INFINITY : INFINITY, runner = best;
                int64_t bj = -1;
                for (int64_t r = r0; r < r1; ++r) {
                    for (int64_t j = redranges_j[2 * r]; j < redranges_j[2 * r + 1]; ++j) {
                        double f = radial_kernel(kind, sq_dist(x + i * D, y + j * D, D), sigma) * b[j * E + e];
                        if (red == 0) {
                            neumaier_add(&s, &cs, f);
                            neumaier_add(&sa, &ca, fabs(f));
                            continue;
                        }
                        int better = red > 0 ? f > best : f < best;
                        int same_lower = f == best && bj >= 0 && j < bj;
                        if (better || same_lower) {
                            runner = best;  /* the displaced value (equal to f on a tie) */
                            best = f;
                            bj = j;
                        } else {
                            int beats_runner = red > 0 ? f > runner : f < runner;
                            if (beats_runner || (f == best && j != bj)) runner = f;
                        }
                    }
                }
                if (red == 0) {
                    val[i * E + e] = s + cs;
                    if (scale) scale[i * E + e] = sa + ca;
                } else {
                    val[i * E + e] = best;
                    if (idx) idx[i * E + e] = bj;
                    if (second) second[i * E + e] = runner;
                }
            }
        }
    }
}

/* (d1, j1) < (d2, j2) in lexicographic order: smaller distance first, then the
 * lower index. */
static int lex_less(double d1, int64_t j1, double d2, int64_t j2)
{
    return d1 < d2 || (d1 == d2 && j1 < j2);
}

/*
 * K-min / ArgMin reduction over squared Euclidean distance.
 * For each row i, the K smallest pairs (d_ij, j) in lexicographic order, sorted
 * ascending: idx[i*K + k] = j, dist[i*K + k] = d_ij.  Slots past N hold -1 / +inf.
 * next[i] (if not NULL) is the distance of the (K+1)-th pair, +inf if N <= K; the
 * parity tests use it to find near-ties.
 * The selection keeps a sorted list of the K+1 best pairs seen so far and inserts
 * each new pair at its lexicographic place (plain insertion).
 * (KeOps README, feature list: ArgMin and K-min reductions; "Kernel Operations on
 * the GPU...", §2: argmin and argKmin.)
 */
void oracle_knn(const double *x, const double *y, int64_t M, int64_t N, int D,
                int K, int64_t *idx, double *dist, double *next)
{
#pragma omp parallel
    {
        int cap = K + 1;
        double *bd = (double *)malloc(sizeof(double) * (size_t)cap);
        int64_t *bj = (int64_t *)malloc(sizeof(int64_t) * (size_t)cap);
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < M; ++i) {
            int n = 0; /* entries held, n <= cap */
            for (int64_t j = 0; j < N; ++j) {
                double d = sq_dist(x + i * D, y + j * D, D);
                if (n == cap && !lex_less(d, j, bd[cap - 1], bj[cap - 1]))
                    continue;
                int p = (n < cap) ? n : cap - 1; /* slot freed for the new pair */
                while (p > 0 && lex_less(d, j, bd[p - 1], bj[p - 1])) {
                    bd[p] = bd[p - 1];
                    bj[p] = bj[p - 1];
                    --p;
                }
                bd[p] = d;
                bj[p] = j;
                if (n < cap) ++n;
            }
            for (int k = 0; k < K; ++k) {
                idx[i * K + k] = (k < n) ? bj[k] : -1;
                dist[i * K + k] = (k < n) ? bd[k] : INFINITY;
            }
            if (next) next[i] = (K < n) ? bd[K] : INFINITY;
        }
        free(bd);
        free(bj);
    }
}
