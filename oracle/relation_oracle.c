/*
 * Full Relation oracle: plain, slow, float64, row-materialised.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header, table or constant with the CUDA
 * path.
 *
 * Source: "Ask Self, Ask Others: Relation Is All You Need" (arXiv:2608.20172),
 *   Sec. 3.1 eq.(1)-(3) and Appendix A.1 (A.1.1 construction, A.1.2 normaliser,
 *   A.1.7 boundary case); FlashRelation path: Sec. 5.1 eq.(12)-(14) and
 *   Appendix A.3.  The author's blog "Attention -> Relation" (qingkeai.online),
 *   sections 2.3-2.7, gives the same construction with the count correction.
 *
 * For one head with P1, P2, V in R^{T x d} (V is the Givens-mixed information
 * state I~) and one-based row index i:
 *   U_ij = p1_i . p2_j / sqrt(d)                                  eq.(1)
 *   R_ii = sigmoid(U_ii / tau_S)                                  eq.(2), Self
 *   R_ij = SiLU(U_ij) - lambda * log(c_i),  j in history          eq.(2), Exchange
 *   R_ij = -inf,  j > i (causal)                                  eq.(2), mask
 *   F_i  = Softmax(R_i),  Y_i = sum_j F_ij V_j                    eq.(3)
 * c_i is the number of visible candidates: i when causal (the pages' log i);
 * T when non-causal (a reading: the pages define only the causal operator).
 * L_i = log sum_j exp(R_ij) (natural log, the pages' R, correction included).
 *
 * Backward (not on the pages; the chain rule applied to the definition above):
 *   D_i = sum_j F_ij dF_ij = dY_i . Y_i,   dF_ij = dY_i . V_j
 *   dR_ij = F_ij (dF_ij - D_i)
 *   dU_ii = dR_ii * S_i (1 - S_i) / tau_S
 *   dU_ij = dR_ij * s(U_ij) (1 + U_ij (1 - s(U_ij))),  s = logistic sigmoid
 *   dP1_i += dU_ij p2_j / sqrt(d),  dP2_j += dU_ij p1_i / sqrt(d),  dV_j += F_ij dY_i
 *   dlambda = sum_{rows} sum_{j != i} dR_ij * (-log c_i)
 *
 * Parallelism: heads (b,h) are independent (Multi-Head Relation, Sec. 3.2 /
 * Appendix A.2.1: construction is head-local), so OpenMP runs over heads, or
 * over rows where only rows are asked for.  No blocking, fusion or
 * reordering of the per-row arithmetic beyond the definition.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int64_t B, H, T, d;
    double tau_S;
    double lambda;
    int causal;
} oracle_problem_t;

enum { ORACLE_OK = 0, ORACLE_BAD_ARG = 1, ORACLE_NO_MEMORY = 2 };

int relation_oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Logistic sigmoid, evaluated so that neither branch overflows. */
static double sigmoid(double x) {
    if (x >= 0.0) return 1.0 / (1.0 + exp(-x));
    double e = exp(x);
    return e / (1.0 + e);
}

/* SiLU(x) = x * sigmoid(x) (the Exchange mapping of eq.(2)). */
static double silu(double x) { return x * sigmoid(x); }

static int check_problem(const oracle_problem_t* p) {
    if (!p) return ORACLE_BAD_ARG;
    if (p->B < 1 || p->H < 1 || p->T < 1 || p->d < 1) return ORACLE_BAD_ARG;
    if (!(p->tau_S > 0.0) || !isfinite(p->tau_S) || !isfinite(p->lambda)) return ORACLE_BAD_ARG;
    return ORACLE_OK;
}

/* Number of visible candidates c_i for zero-based row ii. */
static int64_t candidate_count(const oracle_problem_t* p, int64_t ii) {
    return p->causal ? ii + 1 : p->T;
}

/* Last visible column (inclusive) for zero-based row ii. */
static int64_t last_visible(const oracle_problem_t* p, int64_t ii) {
    return p->causal ? ii : p->T - 1;
}

/* Evidence U_ij for one head (eq.(1)). */
static double evidence(const double* P1h, const double* P2h, int64_t d, int64_t ii, int64_t j) {
    const double* a = P1h + ii * d;
    const double* b = P2h + j * d;
    double acc = 0.0;
    for (int64_t c = 0; c < d; ++c) acc += a[c] * b[c];
    return acc / sqrt((double)d);
}

/* Relation row R_i over the visible columns 0..last (eq.(2)); also returns U. */
static void relation_row(const oracle_problem_t* p, const double* P1h, const double* P2h,
                         int64_t ii, double* u, double* r) {
    const int64_t last = last_visible(p, ii);
    const double corr = p->lambda * log((double)candidate_count(p, ii));
    for (int64_t j = 0; j <= last; ++j) {
        u[j] = evidence(P1h, P2h, p->d, ii, j);
        if (j == ii)
            r[j] = sigmoid(u[j] / p->tau_S);
        else
            r[j] = silu(u[j]) - corr;
    }
}

/* Softmax of a relation row (eq.(3)): F in place of w, returns L = M + log Z~. */
static double flow_row(int64_t n, const double* r, double* f) {
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j)
        if (r[j] > m) m = r[j];
    double z = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        f[j] = exp(r[j] - m);
        z += f[j];
    }
    for (int64_t j = 0; j < n; ++j) f[j] /= z;
    return m + log(z);
}

/* Forward of one row ii of one head: Y_i (d values) and L_i. */
static void forward_row(const oracle_problem_t* p, const double* P1h, const double* P2h,
                        const double* Vh, int64_t ii, double* u, double* r, double* f,
                        double* y, double* L) {
    const int64_t n = last_visible(p, ii) + 1;
    relation_row(p, P1h, P2h, ii, u, r);
    double Li = flow_row(n, r, f);
    for (int64_t c = 0; c < p->d; ++c) y[c] = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        const double* v = Vh + j * p->d;
        for (int64_t c = 0; c < p->d; ++c) y[c] += f[j] * v[c];
    }
    if (L) *L = Li;
}

/* Forward over all heads and rows.  Y: [B,H,T,d]; L: [B,H,T] or NULL. */
int relation_oracle_fwd(const oracle_problem_t* p, const double* P1, const double* P2,
                        const double* V, double* Y, double* L) {
    int rc = check_problem(p);
    if (rc) return rc;
    if (!P1 || !P2 || !V || !Y) return ORACLE_BAD_ARG;
    const int64_t T = p->T, d = p->d, BH = p->B * p->H;
    int failed = 0;
#pragma omp parallel
    {
        double* u = (double*)malloc(sizeof(double) * (size_t)T);
        double* r = (double*)malloc(sizeof(double) * (size_t)T);
        double* f = (double*)malloc(sizeof(double) * (size_t)T);
        if (!u || !r || !f) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 1) collapse(2)
            for (int64_t bh = 0; bh < BH; ++bh)
                for (int64_t ii = 0; ii < T; ++ii) {
                    const size_t off = (size_t)bh * (size_t)T * (size_t)d;
                    forward_row(p, P1 + off, P2 + off, V + off, ii, u, r, f,
                                Y + off + (size_t)ii * d, L ? L + (size_t)bh * T + ii : NULL);
                }
        }
        free(u);
        free(r);
        free(f);
    }
    return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/* Forward of selected (head, row) pairs only.  Y: [n,d]; L: [n] or NULL. */
int relation_oracle_fwd_rows(const oracle_problem_t* p, const double* P1, const double* P2,
                             const double* V, int64_t n, const int64_t* heads,
                             const int64_t* rows, double* Y, double* L) {
    int rc = check_problem(p);
    if (rc) return rc;
    if (!P1 || !P2 || !V || !Y || n < 0 || (n > 0 && (!heads || !rows))) return ORACLE_BAD_ARG;
    for (int64_t k = 0; k < n; ++k)
        if (heads[k] < 0 || heads[k] >= p->B * p->H || rows[k] < 0 || rows[k] >= p->T)
            return ORACLE_BAD_ARG;
    const int64_t T = p->T, d = p->d;
    int failed = 0;
#pragma omp parallel
    {
        double* u = (double*)malloc(sizeof(double) * (size_t)T);
        double* r = (double*)malloc(sizeof(double) * (size_t)T);
        double* f = (double*)malloc(sizeof(double) * (size_t)T);
        if (!u || !r || !f) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t k = 0; k < n; ++k) {
                const size_t off = (size_t)heads[k] * (size_t)T * (size_t)d;
                forward_row(p, P1 + off, P2 + off, V + off, rows[k], u, r, f,
                            Y + (size_t)k * d, L ? L + k : NULL);
            }
        }
        free(u);
        free(r);
        free(f);
    }
    return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/* Derivative of the row's relation entry with respect to U_ij. */
static double relation_slope(const oracle_problem_t* p, int64_t ii, int64_t j, double u) {
    if (j == ii) {
        double s = sigmoid(u / p->tau_S);
        return s * (1.0 - s) / p->tau_S;
    }
    double s = sigmoid(u);
    return s * (1.0 + u * (1.0 - s));
}

/* Backward over all heads: dP1, dP2, dV [B,H,T,d]; dlambda scalar (may be NULL). */
int relation_oracle_bwd(const oracle_problem_t* p, const double* P1, const double* P2,
                        const double* V, const double* dY, double* dP1, double* dP2, double* dV,
                        double* dlambda) {
    int rc = check_problem(p);
    if (rc) return rc;
    if (!P1 || !P2 || !V || !dY || !dP1 || !dP2 || !dV) return ORACLE_BAD_ARG;
    const int64_t T = p->T, d = p->d, BH = p->B * p->H;
    const double inv_sqrt_d = 1.0 / sqrt((double)d);
    const size_t total = (size_t)BH * (size_t)T * (size_t)d;
    memset(dP1, 0, sizeof(double) * total);
    memset(dP2, 0, sizeof(double) * total);
    memset(dV, 0, sizeof(double) * total);
    double dlam = 0.0;
    int failed = 0;
#pragma omp parallel reduction(+ : dlam)
    {
        double* u = (double*)malloc(sizeof(double) * (size_t)T);
        double* r = (double*)malloc(sizeof(double) * (size_t)T);
        double* f = (double*)malloc(sizeof(double) * (size_t)T);
        double* y = (double*)malloc(sizeof(double) * (size_t)d);
        if (!u || !r || !f || !y) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t bh = 0; bh < BH; ++bh) {
                const size_t off = (size_t)bh * (size_t)T * (size_t)d;
                const double *P1h = P1 + off, *P2h = P2 + off, *Vh = V + off, *dYh = dY + off;
                double *dP1h = dP1 + off, *dP2h = dP2 + off, *dVh = dV + off;
                for (int64_t ii = 0; ii < T; ++ii) {
                    const int64_t n = last_visible(p, ii) + 1;
                    forward_row(p, P1h, P2h, Vh, ii, u, r, f, y, NULL);
                    const double* dy = dYh + ii * d;
                    double D = 0.0;
                    for (int64_t c = 0; c < d; ++c) D += dy[c] * y[c];
                    const double logc = log((double)candidate_count(p, ii));
                    for (int64_t j = 0; j < n; ++j) {
                        const double* v = Vh + j * d;
                        double dF = 0.0;
                        for (int64_t c = 0; c < d; ++c) dF += dy[c] * v[c];
                        const double dR = f[j] * (dF - D);
                        if (j != ii) dlam += -logc * dR;
                        const double dU = dR * relation_slope(p, ii, j, u[j]);
                        double* dv = dVh + j * d;
                        double* dp1 = dP1h + ii * d;
                        double* dp2 = dP2h + j * d;
                        const double* p1 = P1h + ii * d;
                        const double* p2 = P2h + j * d;
                        for (int64_t c = 0; c < d; ++c) {
                            dv[c] += f[j] * dy[c];
                            dp1[c] += dU * p2[c] * inv_sqrt_d;
                            dp2[c] += dU * p1[c] * inv_sqrt_d;
                        }
                    }
                }
            }
        }
        free(u);
        free(r);
        free(f);
        free(y);
    }
    if (dlambda) *dlambda = dlam;
    return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/* Per-row statistics of one head: L_i and D_i = dY_i . Y_i for all rows. */
int relation_oracle_row_stats(const oracle_problem_t* p, const double* P1, const double* P2,
                              const double* V, const double* dY, int64_t head, double* L,
                              double* D) {
    int rc = check_problem(p);
    if (rc) return rc;
    if (!P1 || !P2 || !V || !dY || !L || !D || head < 0 || head >= p->B * p->H)
        return ORACLE_BAD_ARG;
    const int64_t T = p->T, d = p->d;
    const size_t off = (size_t)head * (size_t)T * (size_t)d;
    int failed = 0;
#pragma omp parallel
    {
        double* u = (double*)malloc(sizeof(double) * (size_t)T);
        double* r = (double*)malloc(sizeof(double) * (size_t)T);
        double* f = (double*)malloc(sizeof(double) * (size_t)T);
        double* y = (double*)malloc(sizeof(double) * (size_t)d);
        if (!u || !r || !f || !y) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 16)
            for (int64_t ii = 0; ii < T; ++ii) {
                forward_row(p, P1 + off, P2 + off, V + off, ii, u, r, f, y, L + ii);
                const double* dy = dY + off + ii * d;
                double acc = 0.0;
                for (int64_t c = 0; c < d; ++c) acc += dy[c] * y[c];
                D[ii] = acc;
            }
        }
        free(u);
        free(r);
        free(f);
        free(y);
    }
    return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/*
 * Column gradients dP2_j and dV_j of one head for selected columns j, given
 * that head's L and D from relation_oracle_row_stats.  F_ij = exp(R_ij - L_i)
 * is the softmax entry of eq.(3) written with the row's log-normaliser.
 */
int relation_oracle_bwd_cols(const oracle_problem_t* p, const double* P1, const double* P2,
                             const double* V, const double* dY, int64_t head, const double* L,
                             const double* D, int64_t n, const int64_t* cols, double* dP2,
                             double* dV) {
    int rc = check_problem(p);
    if (rc) return rc;
    if (!P1 || !P2 || !V || !dY || !L || !D || !dP2 || !dV || n < 0 || (n > 0 && !cols) ||
        head < 0 || head >= p->B * p->H)
        return ORACLE_BAD_ARG;
    for (int64_t k = 0; k < n; ++k)
        if (cols[k] < 0 || cols[k] >= p->T) return ORACLE_BAD_ARG;
    const int64_t T = p->T, d = p->d;
    const double inv_sqrt_d = 1.0 / sqrt((double)d);
    const size_t off = (size_t)head * (size_t)T * (size_t)d;
    const double *P1h = P1 + off, *P2h = P2 + off, *Vh = V + off, *dYh = dY + off;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t k = 0; k < n; ++k) {
        const int64_t j = cols[k];
        double* dp2 = dP2 + k * d;
        double* dv = dV + k * d;
        for (int64_t c = 0; c < d; ++c) dp2[c] = dv[c] = 0.0;
        const int64_t first = p->causal ? j : 0;
        for (int64_t ii = first; ii < T; ++ii) {
            const double u = evidence(P1h, P2h, d, ii, j);
            double r;
            if (j == ii)
                r = sigmoid(u / p->tau_S);
            else
                r = silu(u) - p->lambda * log((double)candidate_count(p, ii));
            const double f = exp(r - L[ii]);
            const double* dy = dYh + ii * d;
            const double* v = Vh + j * d;
            double dF = 0.0;
            for (int64_t c = 0; c < d; ++c) dF += dy[c] * v[c];
            const double dR = f * (dF - D[ii]);
            const double dU = dR * relation_slope(p, ii, j, u);
            const double* p1 = P1h + ii * d;
            for (int64_t c = 0; c < d; ++c) {
                dv[c] += f * dy[c];
                dp2[c] += dU * p1[c] * inv_sqrt_d;
            }
        }
    }
    return ORACLE_OK;
}

/* Row gradients dP1_i of one head for selected rows i. */
int relation_oracle_bwd_rows(const oracle_problem_t* p, const double* P1, const double* P2,
                             const double* V, const double* dY, int64_t head, int64_t n,
                             const int64_t* rows, double* dP1) {
    int rc = check_problem(p);
    if (rc) return rc;
    if (!P1 || !P2 || !V || !dY || !dP1 || n < 0 || (n > 0 && !rows) || head < 0 ||
        head >= p->B * p->H)
        return ORACLE_BAD_ARG;
    for (int64_t k = 0; k < n; ++k)
        if (rows[k] < 0 || rows[k] >= p->T) return ORACLE_BAD_ARG;
    const int64_t T = p->T, d = p->d;
    const double inv_sqrt_d = 1.0 / sqrt((double)d);
    const size_t off = (size_t)head * (size_t)T * (size_t)d;
    const double *P1h = P1 + off, *P2h = P2 + off, *Vh = V + off, *dYh = dY + off;
    int failed = 0;
#pragma omp parallel
    {
        double* u = (double*)malloc(sizeof(double) * (size_t)T);
        double* r = (double*)malloc(sizeof(double) * (size_t)T);
        double* f = (double*)malloc(sizeof(double) * (size_t)T);
        double* y = (double*)malloc(sizeof(double) * (size_t)d);
        if (!u || !r || !f || !y) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t k = 0; k < n; ++k) {
                const int64_t ii = rows[k];
                const int64_t nv = last_visible(p, ii) + 1;
                forward_row(p, P1h, P2h, Vh, ii, u, r, f, y, NULL);
                const double* dy = dYh + ii * d;
                double D = 0.0;
                for (int64_t c = 0; c < d; ++c) D += dy[c] * y[c];
                double* dp1 = dP1 + k * d;
                for (int64_t c = 0; c < d; ++c) dp1[c] = 0.0;
                for (int64_t j = 0; j < nv; ++j) {
                    const double* v = Vh + j * d;
                    double dF = 0.0;
                    for (int64_t c = 0; c < d; ++c) dF += dy[c] * v[c];
                    const double dU = f[j] * (dF - D) * relation_slope(p, ii, j, u[j]);
                    const double* p2 = P2h + j * d;
                    for (int64_t c = 0; c < d; ++c) dp1[c] += dU * p2[c] * inv_sqrt_d;
                }
            }
        }
        free(u);
        free(r);
        free(f);
        free(y);
    }
    return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/*
 * Second path, for cross-checks only: FlashRelation (Sec. 5.1 eq.(12)-(14),
 * Appendix A.3).  Causal only, as on the pages.  For row i the historical
 * Exchange entries j < i are scanned in tiles whose sizes are given by
 * tile_sizes[0..n_tiles) (cycled); the running (m, l, z) start empty
 * (m = -inf, l = 0, z = 0, A.3.1).  Then L^E = m + log l,
 * A = L^E - lambda log i, g = sigmoid(A - S), Y = (1 - g) V_i + g z / l
 * (A.3.5); the empty history of the first row gives g = 0 (A.1.7).
 * L_i = log(e^{S_i} + e^{A_i}) (A.1.2).
 */
int relation_oracle_flash_fwd(const oracle_problem_t* p, const double* P1, const double* P2,
                              const double* V, int64_t n_tiles, const int64_t* tile_sizes,
                              double* Y, double* L) {
    int rc = check_problem(p);
    if (rc) return rc;
    if (!p->causal || !P1 || !P2 || !V || !Y || n_tiles < 1 || !tile_sizes) return ORACLE_BAD_ARG;
    for (int64_t k = 0; k < n_tiles; ++k)
        if (tile_sizes[k] < 1) return ORACLE_BAD_ARG;
    const int64_t T = p->T, d = p->d, BH = p->B * p->H;
    int failed = 0;
#pragma omp parallel
    {
        double* z = (double*)malloc(sizeof(double) * (size_t)d);
        double* e = (double*)malloc(sizeof(double) * (size_t)T);
        if (!z || !e) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 1) collapse(2)
            for (int64_t bh = 0; bh < BH; ++bh)
                for (int64_t ii = 0; ii < T; ++ii) {
                    const size_t off = (size_t)bh * (size_t)T * (size_t)d;
                    const double *P1h = P1 + off, *P2h = P2 + off, *Vh = V + off;
                    double m = -INFINITY, l = 0.0;
                    for (int64_t c = 0; c < d; ++c) z[c] = 0.0;
                    int64_t j0 = 0, t = 0;
                    while (j0 < ii) {
                        int64_t j1 = j0 + tile_sizes[t % n_tiles];
                        if (j1 > ii) j1 = ii;
                        double mb = -INFINITY;
                        for (int64_t j = j0; j < j1; ++j) {
                            e[j] = silu(evidence(P1h, P2h, d, ii, j));
                            if (e[j] > mb) mb = e[j];
                        }
                        const double mn = mb > m ? mb : m;
                        const double scale = (m == -INFINITY) ? 0.0 : exp(m - mn);
                        l *= scale;
                        for (int64_t c = 0; c < d; ++c) z[c] *= scale;
                        for (int64_t j = j0; j < j1; ++j) {
                            const double w = exp(e[j] - mn);
                            l += w;
                            const double* v = Vh + j * d;
                            for (int64_t c = 0; c < d; ++c) z[c] += w * v[c];
                        }
                        m = mn;
                        j0 = j1;
                        ++t;
                    }
                    const double S = sigmoid(evidence(P1h, P2h, d, ii, ii) / p->tau_S);
                    double* y = Y + off + ii * d;
                    const double* vi = Vh + ii * d;
                    if (ii == 0) {
                        for (int64_t c = 0; c < d; ++c) y[c] = vi[c];
                        if (L) L[bh * T + ii] = S;
                    } else {
                        const double A = m + log(l) - p->lambda * log((double)(ii + 1));
                        const double g = sigmoid(A - S);
                        for (int64_t c = 0; c < d; ++c) y[c] = (1.0 - g) * vi[c] + g * z[c] / l;
                        if (L) {
                            const double hi = S > A ? S : A, lo = S > A ? A : S;
                            L[bh * T + ii] = hi + log1p(exp(lo - hi));
                        }
                    }
                }
        }
        free(z);
        free(e);
    }
    return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}
