/*
 * fibatt_oracle.c -- plain, slow fp64 CPU oracle for Fibottention's per-head
 * sparse self-attention (forward and backward).
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * CPU-baseline leg of bench.py may load this file.  It shares no code, header,
 * table or constant generator with the CUDA library; the library never loads
 * it, and it never loads the library.
 *
 * What it follows (page, section):
 *   [P1] "Fibottention: Inceptive Visual Representation Learning with Diverse
 *        Attention Across Heads" (arXiv 2406.19391), Sec. 3:
 *          - support set Omega_w^{Fib(a,b)} = {(j,k) : |j-k| in Fib(a,b), |j-k| <= w}
 *          - Wythoff row i: a_i, b_i ("no overlap, each integer exactly once")
 *          - window schedule w_i = w_min + floor((w_max-w_min)(i-1)/(h-1))
 *          - "compute only the dot products whose indices are supported on Omega"
 *   [P2] Fibottention project README, Algorithm 1 (generalised Fibonacci list,
 *        extended while its last term is below w) and Algorithm 3 (scores,
 *        mask, row softmax, weighted sum of V).
 *
 * Readings taken where the pages are silent or garbled (each also listed in
 * the design notes):
 *   - Wythoff row i is (a_i, b_i) = (floor(r*phi), floor(r*phi^2)) with
 *     r = floor(i*phi); the only reading that gives rows that are disjoint and
 *     cover every positive integer.  Computed with exact integer square roots.
 *   - Entries outside Omega are excluded from the softmax (weight exactly 0).
 *   - Offsets are a set: duplicates in Fib(a,b) count once.
 *   - The main diagonal is in Omega iff the caller asks for it, or 0 is in
 *     the distance set.
 *   - A row with no support has output 0 and log-sum-exp -inf, and
 *     contributes nothing to any gradient.
 *   - The backward pass is the exact derivative of the forward pass with
 *     respect to Q, K and V for the loss L = sum(dO * O); the pages print no
 *     backward, so it is derived here from the softmax Jacobian.
 *   - Global first token ([P2] Algorithm 2 leaves row 0 and column 0 of its
 *     mask all ones: the class token attends every key and every query
 *     attends it).  Optional, selected by bit 1 of the flags argument (bit 0
 *     is the diagonal): (j,k) with j == 0 or k == 0 is then in Omega too.
 *     The signed-offset table describes the banded part only.
 *
 * Every loop below visits (j,k) pairs by brute force over the whole N x N
 * index square and tests membership from the definition; nothing is tiled,
 * fused or reordered.  Arithmetic is fp64 throughout.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

static int g_threads = 1;

/* Number of host threads the row loops below may use (1 = serial). */
int orc_set_threads(int n)
{
    g_threads = n < 1 ? 1 : n;
#ifdef _OPENMP
    return g_threads;
#else
    return 1;
#endif
}

int orc_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_num_procs();
#else
    return 1;
#endif
}

/* ---------------------------------------------------------------- integers */

/* floor(sqrt(n)) for 0 <= n < 2^62, exact (Newton iteration on integers). */
int64_t orc_isqrt(int64_t n)
{
    if (n < 2) return n < 0 ? -1 : n;
    int64_t x = (int64_t)sqrt((double)n);
    while (x > 0 && x > n / x) --x;                 /* x*x > n  -> step down */
    while ((x + 1) <= n / (x + 1)) ++x;             /* (x+1)^2 <= n -> up    */
    return x;
}

/* floor(n*phi) with phi = (1+sqrt 5)/2, exact for n >= 0:
 * n*phi = (n + sqrt(5 n^2)) / 2 and sqrt(5 n^2) is irrational for n >= 1,
 * so the floor equals (n + floor(sqrt(5 n^2))) div 2. */
int64_t orc_floor_mul_phi(int64_t n)
{
    if (n <= 0) return 0;
    return (n + orc_isqrt(5 * n * n)) / 2;
}

/* [P1] Sec. 3.2: row i (i >= 1) of the Wythoff array starts with
 * a_i = floor(floor(i*phi)*phi) and b_i = floor(floor(i*phi)*phi^2);
 * phi^2 = phi + 1 gives b_i = a_i + floor(i*phi). */
int orc_wythoff_row(int64_t i, int64_t *a, int64_t *b)
{
    if (i < 1 || i > 100000000) return -1;
    int64_t r = orc_floor_mul_phi(i);
    *a = orc_floor_mul_phi(r);
    *b = *a + r;
    return 0;
}

/* [P2] Algorithm 1: start from [a, b] and append the sum of the last two
 * terms while the last term is below w.  Writes at most cap terms and
 * returns how many the full list has (-1 if a = b = 0, which never ends). */
int orc_fib_list(int64_t a, int64_t b, int64_t w, int64_t *out, int cap)
{
    if (a < 0 || b < 0) return -1;
    if (a == 0 && b == 0) return -1;
    int64_t x = a, y = b;
    int n = 0;
    if (n < cap) out[n] = x;
    ++n;
    if (n < cap) out[n] = y;
    ++n;
    while (y < w) {
        int64_t z = x + y;
        x = y;
        y = z;
        if (n < cap) out[n] = y;
        ++n;
        if (n > 4096) return -1;
    }
    return n;
}

/* [P1] Sec. 3.2 window of head i (1-based) out of h heads.  With h = 1 the
 * interpolation has no spread and the single head takes w_min. */
int64_t orc_window(int64_t i, int64_t h, int64_t w_min, int64_t w_max)
{
    if (h <= 1) return w_min;
    return w_min + ((w_max - w_min) * (i - 1)) / (h - 1);
}

/* ----------------------------------------------------------------- support */

/* [P1] Sec. 3: (j,k) is in Omega_w^{S} iff |j-k| is one of the distances in S
 * and |j-k| <= w; the main diagonal is added when bit 0 of flags is set, and
 * row 0 and column 0 ([P2] Algorithm 2) when bit 1 is set. */
int orc_in_support(int64_t j, int64_t k, const int64_t *S, int nS, int64_t w, int flags)
{
    int64_t d = j > k ? j - k : k - j;
    if ((flags & 2) && (j == 0 || k == 0)) return 1;
    if ((flags & 1) && d == 0) return 1;
    if (d > w) return 0;
    for (int t = 0; t < nS; ++t)
        if (S[t] == d) return 1;
    return 0;
}

/* Dense N x N 0/1 mask of Omega, by testing every pair.  Returns |Omega|. */
int64_t orc_support_mask(int64_t N, const int64_t *S, int nS, int64_t w, int flags, uint8_t *mask)
{
    int64_t count = 0;
    for (int64_t j = 0; j < N; ++j)
        for (int64_t k = 0; k < N; ++k) {
            int in = orc_in_support(j, k, S, nS, w, flags);
            if (mask) mask[j * N + k] = (uint8_t)in;
            count += in;
        }
    return count;
}

/* Signed offsets delta = k - j present in Omega, ascending, read off the
 * first row (j = 0, delta = k >= 0) and first column (k = 0, delta = -j <= 0)
 * of Omega.  Writes at most cap entries, returns the number present. */
int orc_signed_table(int64_t N, const int64_t *S, int nS, int64_t w, int flags, int32_t *out, int cap)
{
    const int diag = flags & 1;   /* the banded part: no global first token */
    int n = 0;
    for (int64_t j = N - 1; j >= 1; --j)            /* column 0: delta = -j */
        if (orc_in_support(j, 0, S, nS, w, diag)) {
            if (n < cap) out[n] = (int32_t)(-j);
            ++n;
        }
    for (int64_t k = 0; k < N; ++k)                 /* row 0: delta = k      */
        if (orc_in_support(0, k, S, nS, w, diag)) {
            if (n < cap) out[n] = (int32_t)k;
            ++n;
        }
    return n;
}

/* ----------------------------------------------------------------- forward */

/* Row j of the masked softmax ([P2] Algorithm 3; [P1] Sec. 3):
 * s_k = scale * <Q_j, K_k> for every k with (j,k) in Omega, P_jk = e^{s_k} /
 * sum_l e^{s_l}.  The maximum is subtracted before exponentiating, which
 * leaves every quotient unchanged.  Fills kidx/p with the support of the row,
 * returns its size and writes log(sum_l e^{s_l}) to *lse (-inf if empty). */
static int64_t row_softmax(int64_t N, int64_t Dh, const double *Q, const double *K,
                           const int64_t *S, int nS, int64_t w, int flags, double scale,
                           int64_t j, int64_t *kidx, double *p, double *lse)
{
    int64_t n = 0;
    double m = -INFINITY;
    for (int64_t k = 0; k < N; ++k) {
        if (!orc_in_support(j, k, S, nS, w, flags)) continue;
        double s = 0.0;
        for (int64_t d = 0; d < Dh; ++d) s += Q[j * Dh + d] * K[k * Dh + d];
        s *= scale;
        kidx[n] = k;
        p[n] = s;
        if (s > m) m = s;
        ++n;
    }
    if (n == 0) {
        *lse = -INFINITY;
        return 0;
    }
    double l = 0.0;
    for (int64_t t = 0; t < n; ++t) l += exp(p[t] - m);
    *lse = m + log(l);
    for (int64_t t = 0; t < n; ++t) p[t] = exp(p[t] - *lse);
    return n;
}

/* Forward pass of one head: O_j = sum_k P_jk V_k and LSE_j, for the query
 * rows listed in rows (all N rows when rows is NULL).  Q, K, V are N x Dh
 * row-major; O is nrows x Dh and LSE has nrows entries, in the order of
 * rows. */
void orc_fwd_rows(int64_t N, int64_t Dh, const double *Q, const double *K, const double *V,
                  const int64_t *S, int nS, int64_t w, int flags, double scale,
                  const int64_t *rows, int64_t nrows, double *O, double *LSE)
{
    if (!rows) nrows = N;
#pragma omp parallel num_threads(g_threads)
    {
        int64_t *kidx = (int64_t *)malloc(sizeof(int64_t) * (size_t)(N > 0 ? N : 1));
        double *p = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < nrows; ++r) {
            int64_t j = rows ? rows[r] : r;
            double lse;
            int64_t n = row_softmax(N, Dh, Q, K, S, nS, w, flags, scale, j, kidx, p, &lse);
            LSE[r] = lse;
            for (int64_t d = 0; d < Dh; ++d) {
                double o = 0.0;
                for (int64_t t = 0; t < n; ++t) o += p[t] * V[kidx[t] * Dh + d];
                O[r * Dh + d] = o;
            }
        }
        free(kidx);
        free(p);
    }
}

/* ---------------------------------------------------------------- backward */

/* Softmax-Jacobian quantities of row j for the loss L = sum(dO * O):
 * dP_jk = <dO_j, V_k>, D_j = sum_l P_jl dP_jl, dS_jk = P_jk (dP_jk - D_j).
 * Fills kidx, p and ds with the row's support; returns its size. */
static int64_t row_ds(int64_t N, int64_t Dh, const double *Q, const double *K, const double *V,
                      const double *dO, const int64_t *S, int nS, int64_t w, int flags,
                      double scale, int64_t j, int64_t *kidx, double *p, double *ds)
{
    double lse;
    int64_t n = row_softmax(N, Dh, Q, K, S, nS, w, flags, scale, j, kidx, p, &lse);
    double Dj = 0.0;
    for (int64_t t = 0; t < n; ++t) {
        double dp = 0.0;
        for (int64_t d = 0; d < Dh; ++d) dp += dO[j * Dh + d] * V[kidx[t] * Dh + d];
        ds[t] = dp;
        Dj += p[t] * dp;
    }
    for (int64_t t = 0; t < n; ++t) ds[t] = p[t] * (ds[t] - Dj);
    return n;
}

/* Backward pass of one head (chain rule through S = scale Q K^T restricted to
 * Omega, the row softmax and O = P V):
 *   dQ_j = scale * sum_k dS_jk K_k
 *   dK_k = scale * sum_j dS_jk Q_j
 *   dV_k = sum_j P_jk dO_j
 * dQ is computed for the query rows in qrows and dK, dV for the key rows in
 * krows (all rows when the list is NULL); outputs are packed in list order.
 * Pass dQ = NULL or dK = dV = NULL to skip that part. */
void orc_bwd_rows(int64_t N, int64_t Dh, const double *Q, const double *K, const double *V,
                  const double *dO, const int64_t *S, int nS, int64_t w, int flags, double scale,
                  const int64_t *qrows, int64_t nq, const int64_t *krows, int64_t nk,
                  double *dQ, double *dK, double *dV)
{
    if (!qrows) nq = N;
    if (!krows) nk = N;
#pragma omp parallel num_threads(g_threads)
    {
        size_t cap = (size_t)(N > 0 ? N : 1);
        int64_t *kidx = (int64_t *)malloc(sizeof(int64_t) * cap);
        double *p = (double *)malloc(sizeof(double) * cap);
        double *ds = (double *)malloc(sizeof(double) * cap);
        if (dQ) {
#pragma omp for schedule(dynamic, 4)
            for (int64_t r = 0; r < nq; ++r) {
                int64_t j = qrows ? qrows[r] : r;
                int64_t n = row_ds(N, Dh, Q, K, V, dO, S, nS, w, flags, scale, j, kidx, p, ds);
                for (int64_t d = 0; d < Dh; ++d) {
                    double g = 0.0;
                    for (int64_t t = 0; t < n; ++t) g += ds[t] * K[kidx[t] * Dh + d];
                    dQ[r * Dh + d] = scale * g;
                }
            }
        }
        if (dK || dV) {
#pragma omp for schedule(dynamic, 4)
            for (int64_t r = 0; r < nk; ++r) {
                int64_t k = krows ? krows[r] : r;
                for (int64_t d = 0; d < Dh; ++d) {
                    if (dK) dK[r * Dh + d] = 0.0;
                    if (dV) dV[r * Dh + d] = 0.0;
                }
                /* every query row j whose support contains key k */
                for (int64_t j = 0; j < N; ++j) {
                    if (!orc_in_support(j, k, S, nS, w, flags)) continue;
                    int64_t n = row_ds(N, Dh, Q, K, V, dO, S, nS, w, flags, scale, j, kidx, p, ds);
                    for (int64_t t = 0; t < n; ++t) {
                        if (kidx[t] != k) continue;
                        for (int64_t d = 0; d < Dh; ++d) {
                            if (dK) dK[r * Dh + d] += scale * ds[t] * Q[j * Dh + d];
                            if (dV) dV[r * Dh + d] += p[t] * dO[j * Dh + d];
                        }
                    }
                }
            }
        }
        free(kidx);
        free(p);
        free(ds);
    }
}
