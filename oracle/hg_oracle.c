/*
 * hg_oracle.c -- TEST INFRASTRUCTURE, not part of the product path.
 *
 * A plain, slow, obviously-correct fp64 CPU evaluation of the multiresolution
 * hash-grid encoding: the gradient-augmented cubic-Hermite variant
 * (Hermite-NGP) and its degenerate d-linear case (Instant-NGP).  Only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg may load this
 * file's shared library.  It shares no code with the CUDA library.
 *
 * Sources (page title, section; the DInf-Grid page for the RBF grid):
 *  - "Hermite-NGP: Gradient-Augmented Hash Encoding for Learning PDEs",
 *    section "整体框架" (pipeline: per-level hash lookup of Hermite
 *    coefficients bucketed by derivative order, tensor-product Hermite
 *    reconstruction of gamma, grad gamma and the Laplacian in one pass);
 *    section "关键设计 1" (the encoding equation
 *        gamma^l(x) = sum_g sum_alpha theta^(alpha)_{l,h(g)}
 *                     H^(alpha)((x - x_g)/dx_l) dx_l^{|alpha|},
 *     H^(alpha) = prod_i h^(alpha_i), the value basis h^(0) = -2t^3 + 3t^2
 *     and the derivative basis h^(1) = t^3 - t^2, and the order-bucketed
 *     tables);
 *    section "关键设计 2" (the factorised derivative
 *        d/dx_i H^(alpha) = d/dx_i h^(alpha_i)(y_i) prod_{k!=i} h^(alpha_k)(y_k)
 *     and the second derivative of the bases).
 *  - "SIGGRAPH 2022｜InstantNGP 与多分辨率哈希编码", section
 *    "InstantNGP 与多分辨率哈希编码流程与原理" (steps 1-3: the cell's corner
 *    features, hashed lookup, d-linear interpolation; one-to-one indexing when
 *    a level's vertices fit the table, hashing otherwise).
 *
 * Readings where the pages are silent (each one is listed in the design
 * notes of the repository):
 *  - Only the bases of the cell's high-side vertex are printed.  The oracle
 *    uses the standard cubic Hermite pair as functions of the signed offset
 *    s = (x - x_g)/dx from the vertex: phi0(s) = (1-|s|)^2 (1+2|s|),
 *    phi1(s) = s (1-|s|)^2.  For the high-side vertex (s = t - 1) these are the
 *    printed h^(0)(t), h^(1)(t).  Derivatives are the one-sided ones from inside
 *    the cell that contains x.
 *  - The hash is the XOR of g_i * pi_i (mod 2^32), pi = (1, 2654435761,
 *    805459861, 3674653429), then mod T.  The pages print no hash formula;
 *    the first three primes are the spatial-hash primes of Instant-NGP, and
 *    the fourth, for the 4D (space-time) grid, the next prime of the same
 *    published list.  A level whose (N+1)^d vertices fit in T is indexed
 *    one-to-one as sum_i g_i (N+1)^i.
 *  - x is clamped to [0,1] (NaN to 0); pos = fl32(x * N) (one fp32 multiply,
 *    rounded to nearest); c = min(floor(pos), N-1); t = pos - c.  Everything
 *    after that is fp64.
 *  - Tables are bucketed by derivative order k = |alpha| (d+1 tables); table k
 *    holds C(d,k) * F values per entry, alpha in lexicographic axis order
 *    (k=1: x,y,z[,w]; k=2: xy,xz,[xw,]yz[,yw,zw]; k=3: xyz[,xyw,xzw,yzw];
 *    k=4: xyzw), then the feature index.
 *  - d = 2, 3 or 4.  The 4D (space-time) grid is the extension the
 *    Hermite-NGP page names as the method's main storage cost (16
 *    coefficients per vertex and feature); it follows the same equation.
 *  - "grad^2 gamma" is the Laplacian (trace of the Hessian), one value per
 *    (level, feature).
 *  - Inactive levels (bit l of the mask clear) output zero and receive no
 *    gradient.
 *  - The Gaussian-RBF grid of the DInf-Grid page: distances in grid units,
 *    ring-R box neighbourhoods clipped to the grid (see its section below).
 *  - INGP-FD (the page's finite-difference baseline): stencil points
 *    x +- eps e_i with the shifted coordinate computed as one fp32 add, and
 *    the textbook central differences (see the INGP-FD section below).
 *
 * Each floating output is returned together with its condition magnitude:
 * the same sum with every factor replaced by its absolute value.  Tests use
 * it to scale the tolerance.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -fPIC -shared
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_MAXD 4
#define OR_MAXP (OR_MAXD * (OR_MAXD + 1) / 2)   /* Hessian entries in OR_MAXD dimensions */

static const uint32_t OR_PRIMES[OR_MAXD] = {1u, 2654435761u, 805459861u, 3674653429u};

/* ------------------------------------------------------------------ */
/* small combinatorics                                                  */
/* ------------------------------------------------------------------ */

static int popcount_small(int m) {
    int c = 0;
    while (m) { c += m & 1; m >>= 1; }
    return c;
}

static int binom(int n, int k) {
    int r = 1;
    for (int i = 0; i < k; ++i) r = r * (n - i) / (i + 1);
    return r;
}

/* Position of the multi-index alpha (bit i set = derivative along axis i)
 * inside its order bucket |alpha|, counting the same-order multi-indices in
 * lexicographic axis order: in 3D k=1 -> x,y,z; k=2 -> xy,xz,yz; k=3 -> xyz;
 * in 4D k=2 -> xy,xz,xw,yz,yw,zw and k=3 -> xyz,xyw,xzw,yzw.               */
static int slot_in_bucket(int d, int alpha) {
    int k = popcount_small(alpha), slot = 0;
    /* enumerate same-order masks in lexicographic order of their axis lists */
    int lists[1 << OR_MAXD][OR_MAXD], nl = 0;
    for (int m = 0; m < (1 << d); ++m) {
        if (popcount_small(m) != k) continue;
        int p = 0;
        for (int i = 0; i < d; ++i) if (m >> i & 1) lists[nl][p++] = i;
        for (int q = p; q < OR_MAXD; ++q) lists[nl][q] = 99;
        nl++;
    }
    /* rank of alpha's axis list among them */
    int mine[OR_MAXD], p = 0;
    for (int i = 0; i < d; ++i) if (alpha >> i & 1) mine[p++] = i;
    for (int q = p; q < OR_MAXD; ++q) mine[q] = 99;
    for (int j = 0; j < nl; ++j) {
        int less = 0;
        for (int q = 0; q < OR_MAXD; ++q) {
            if (lists[j][q] != mine[q]) { less = lists[j][q] < mine[q]; break; }
        }
        if (less) slot++;
    }
    return slot;
}

/* ------------------------------------------------------------------ */
/* cell location and vertex indexing                                    */
/* ------------------------------------------------------------------ */

/* Clamp to [0,1] (NaN -> 0), scale by N in one fp32 multiply, split into the
 * cell index and the local coordinate.                                     */
static void locate(float x, int32_t N, int64_t* c, double* t) {
    float xc = x;
    if (!(xc >= 0.0f)) xc = 0.0f;
    if (xc > 1.0f) xc = 1.0f;
    volatile float pos = xc * (float)N;
    float pf = pos;
    int64_t ci = (int64_t)floorf(pf);
    if (ci > (int64_t)N - 1) ci = (int64_t)N - 1;
    *c = ci;
    *t = (double)pf - (double)ci;
}

/* Index of grid vertex g in an order table of 2^log2T entries at resolution N. */
static uint32_t vertex_index(int d, const int64_t* g, int32_t N, int log2T) {
    uint64_t T = (uint64_t)1 << log2T;
    uint64_t side = (uint64_t)N + 1, nvert = 1;
    for (int i = 0; i < d; ++i) nvert *= side;
    if (nvert <= T) {
        uint64_t idx = 0, mul = 1;
        for (int i = 0; i < d; ++i) { idx += (uint64_t)g[i] * mul; mul *= side; }
        return (uint32_t)idx;
    }
    uint32_t h = 0;
    for (int i = 0; i < d; ++i) h ^= (uint32_t)(((uint64_t)g[i] * OR_PRIMES[i]) & 0xffffffffu);
    return (uint32_t)((uint64_t)h % T);
}

/* ------------------------------------------------------------------ */
/* 1D cubic Hermite bases of a vertex, as functions of the signed offset     */
/* s = (x - x_g)/dx.  sigma = +1 for the cell's low-side vertex and -1 for   */
/* its high-side vertex, so that a = sigma*s = |s| and the derivatives are   */
/* the one-sided ones from inside the cell.  out = {phi, dphi/ds, d2phi/ds2}. */
/* ------------------------------------------------------------------ */
static void hermite_1d(int order, double s, double sigma, double out[3]) {
    double a = sigma * s;
    if (order == 0) {
        out[0] = (1.0 - a) * (1.0 - a) * (1.0 + 2.0 * a);
        out[1] = sigma * (-6.0 * a * (1.0 - a));
        out[2] = -6.0 + 12.0 * a;
    } else {
        out[0] = s * (1.0 - a) * (1.0 - a);
        out[1] = (1.0 - a) * (1.0 - 3.0 * a);
        out[2] = sigma * (6.0 * a - 4.0);
    }
}

/* Exposed for the basis pins: the basis of the vertex on side v (0 = low,
 * 1 = high) of a cell, at local coordinate t.                              */
void oracle_basis_1d(int v, int order, double t, double out[3]) {
    double s = t - (double)v;
    double sigma = v ? -1.0 : 1.0;
    hermite_1d(order, s, sigma, out);
}

/* ------------------------------------------------------------------ */
/* Hermite: one cell of one level                                       */
/* ------------------------------------------------------------------ */

typedef struct {
    int d, F;
    int32_t N;
    const int32_t* log2T;         /* [d+1] */
    const double* const* tab;     /* [d+1]: this level's table k, [T_k][C(d,k)][F] */
} or_level;

/* Evaluate the cell with corner c at local coordinate t (fp64), writing
 * gamma[F], dgamma[d][F] (d/dx), lap[F], and the condition magnitudes.
 * Any output pointer may be NULL.                                           */
/* Number of entries of the upper triangle of a d x d Hessian (i <= j, row-major:
 * 2D xx, xy, yy; 3D xx, xy, xz, yy, yz, zz; 4D xx, xy, xz, xw, yy, yz, yw,
 * zz, zw, ww) and the position of (i, j).                                  */
static int hess_entries(int d) { return d * (d + 1) / 2; }
static int hess_pos(int d, int i, int j) {
    int p = 0;
    for (int a = 0; a < d; ++a)
        for (int b = a; b < d; ++b) {
            if (a == i && b == j) return p;
            ++p;
        }
    return -1;
}

static void hermite_cell_h(const or_level* lv, const int64_t* c, const double* t,
                           double* gamma, double* dgamma, double* lap,
                           double* mg, double* md, double* ml, double* hess, double* mh);

static void hermite_cell(const or_level* lv, const int64_t* c, const double* t,
                         double* gamma, double* dgamma, double* lap,
                         double* mg, double* md, double* ml) {
    hermite_cell_h(lv, c, t, gamma, dgamma, lap, mg, md, ml, NULL, NULL);
}

/* As hermite_cell, plus (when hess != NULL) the Hessian hess[P][F], P the
 * upper-triangle entries: d2/dx_i dx_j = N^2 d2/dy_i dy_j, where the mixed
 * derivative of H replaces factors i and j by their first derivatives and
 * the pure one factor i by its second derivative.  mh: magnitudes.        */
static void hermite_cell_h(const or_level* lv, const int64_t* c, const double* t,
                           double* gamma, double* dgamma, double* lap,
                           double* mg, double* md, double* ml, double* hess, double* mh) {
    const int d = lv->d, F = lv->F;
    const double N = (double)lv->N;
    const double dx = 1.0 / N;
    for (int f = 0; f < F; ++f) {
        if (gamma) gamma[f] = 0.0;
        if (mg) mg[f] = 0.0;
        if (lap) lap[f] = 0.0;
        if (ml) ml[f] = 0.0;
        for (int j = 0; j < d; ++j) {
            if (dgamma) dgamma[j * F + f] = 0.0;
            if (md) md[j * F + f] = 0.0;
        }
        for (int q = 0; q < hess_entries(d); ++q) {
            if (hess) hess[q * F + f] = 0.0;
            if (mh) mh[q * F + f] = 0.0;
        }
    }
    double scale[OR_MAXD + 1];
    for (int k = 0; k <= d; ++k) scale[k] = pow(dx, (double)k);   /* dx^{|alpha|} */
    /* bases of axis i for the corner on side vi, basis order a: {phi, phi', phi''} in y */
    double hb[OR_MAXD][2][2][3];
    for (int i = 0; i < d; ++i)
        for (int vi = 0; vi < 2; ++vi)
            for (int a = 0; a < 2; ++a)
                hermite_1d(a, t[i] - (double)vi, vi ? -1.0 : 1.0, hb[i][vi][a]);
    for (int v = 0; v < (1 << d); ++v) {
        int64_t g[OR_MAXD];
        for (int i = 0; i < d; ++i) g[i] = c[i] + (v >> i & 1);     /* corner vertex */
        uint32_t idx[OR_MAXD + 1];
        for (int k = 0; k <= d; ++k) idx[k] = vertex_index(d, g, lv->N, lv->log2T[k]);
        for (int alpha = 0; alpha < (1 << d); ++alpha) {
            int k = popcount_small(alpha);
            int slot = slot_in_bucket(d, alpha);
            const double* theta = lv->tab[k] + ((size_t)idx[k] * binom(d, k) + slot) * F;
            const double (*h[OR_MAXD])[3];
            for (int i = 0; i < d; ++i) h[i] = &hb[i][v >> i & 1][alpha >> i & 1];
            /* H, dH/dy_j, d2H/dy_j^2 */
            double H = 1.0;
            for (int i = 0; i < d; ++i) H *= (*h[i])[0];
            double dH[OR_MAXD], d2H[OR_MAXD];
            for (int j = 0; j < d; ++j) {
                dH[j] = 1.0; d2H[j] = 1.0;
                for (int i = 0; i < d; ++i) {
                    dH[j] *= (i == j) ? (*h[i])[1] : (*h[i])[0];
                    d2H[j] *= (i == j) ? (*h[i])[2] : (*h[i])[0];
                }
            }
            for (int f = 0; f < F; ++f) {
                double th = theta[f];
                if (gamma) gamma[f] += th * H * scale[k];
                if (mg) mg[f] += fabs(th) * fabs(H) * scale[k];
                for (int j = 0; j < d; ++j) {
                    /* d/dx_j = N d/dy_j */
                    if (dgamma) dgamma[j * F + f] += th * scale[k] * N * dH[j];
                    if (md) md[j * F + f] += fabs(th) * scale[k] * N * fabs(dH[j]);
                    if (lap) lap[f] += th * scale[k] * N * N * d2H[j];
                    if (ml) ml[f] += fabs(th) * scale[k] * N * N * fabs(d2H[j]);
                }
                if (hess) {
                    for (int i = 0; i < d; ++i)
                        for (int j = i; j < d; ++j) {
                            double hij = 1.0;
                            for (int m = 0; m < d; ++m) {
                                if (i == j) hij *= (m == i) ? (*h[m])[2] : (*h[m])[0];
                                else hij *= (m == i || m == j) ? (*h[m])[1] : (*h[m])[0];
                            }
                            const int q = hess_pos(d, i, j);
                            hess[q * F + f] += th * scale[k] * N * N * hij;
                            if (mh) mh[q * F + f] += fabs(th) * scale[k] * N * N * fabs(hij);
                        }
                }
            }
        }
    }
}

/* Exposed for the continuity and finite-difference pins: evaluate one cell
 * of one level at an arbitrary fp64 local coordinate.                      */
int oracle_eval_cell(int d, int F, int32_t N, const int32_t* log2T,
                     const double* const* tables, const int64_t* c, const double* t,
                     double* gamma, double* dgamma, double* lap) {
    if (d < 1 || d > OR_MAXD) return 1;
    or_level lv = {d, F, N, log2T, tables};
    hermite_cell(&lv, c, t, gamma, dgamma, lap, NULL, NULL, NULL);
    return 0;
}

/* ------------------------------------------------------------------ */
/* Public oracle entry points                                            */
/* ------------------------------------------------------------------ */

static void set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

/* idx[N][L][d+1][2^d]: vertex index of corner v (bit i = axis i) in order
 * table k, for every level (the mask does not apply).                       */
int oracle_hash_indices(int d, int L, const int32_t* res, const int32_t* log2T,
                        int64_t n_pts, const float* coords, uint32_t* idx, int nthreads) {
    if (d < 1 || d > OR_MAXD) return 1;
    set_threads(nthreads);
    const int V = 1 << d;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < n_pts; ++n) {
        for (int l = 0; l < L; ++l) {
            int64_t c[OR_MAXD];
            double t[OR_MAXD];
            for (int i = 0; i < d; ++i) locate(coords[n * d + i], res[l], &c[i], &t[i]);
            for (int k = 0; k <= d; ++k) {
                for (int v = 0; v < V; ++v) {
                    int64_t g[OR_MAXD];
                    for (int i = 0; i < d; ++i) g[i] = c[i] + (v >> i & 1);
                    idx[((n * L + l) * (d + 1) + k) * V + v] = vertex_index(d, g, res[l], log2T[k]);
                }
            }
        }
    }
    return 0;
}

/* Forward.  tables[k] is table k for all levels, [L][T_k][C(d,k)][F]
 * contiguous.  Outputs are point-major: gamma[N][L][F], dgamma[N][d][L][F],
 * lap[N][L][F], with magnitudes in the same shapes.  dgamma/lap and the
 * magnitude arrays may be NULL.                                           */
int oracle_encode_fwd(int d, int L, int F, const int32_t* res, const int32_t* log2T,
                      uint32_t level_mask, const double* const* tables,
                      int64_t n_pts, const float* coords,
                      double* gamma, double* dgamma, double* lap,
                      double* mgamma, double* mdgamma, double* mlap, int nthreads) {
    if (d < 1 || d > OR_MAXD || L < 1 || F < 1 || F > 8) return 1;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 256)
    for (int64_t n = 0; n < n_pts; ++n) {
        double g_[8], dg_[OR_MAXD * 8], lp_[8], mg_[8], md_[OR_MAXD * 8], ml_[8];
        for (int l = 0; l < L; ++l) {
            const int active = (level_mask >> l) & 1u;
            if (active) {
                const double* tab_l[OR_MAXD + 1];
                for (int k = 0; k <= d; ++k)
                    tab_l[k] = tables[k] + (size_t)l * ((size_t)1 << log2T[k]) * binom(d, k) * F;
                or_level lv = {d, F, res[l], log2T, tab_l};
                int64_t c[OR_MAXD];
                double t[OR_MAXD];
                for (int i = 0; i < d; ++i) locate(coords[n * d + i], res[l], &c[i], &t[i]);
                hermite_cell(&lv, c, t, g_, dg_, lp_, mg_, md_, ml_);
            } else {
                for (int f = 0; f < F; ++f) {
                    g_[f] = lp_[f] = mg_[f] = ml_[f] = 0.0;
                    for (int j = 0; j < d; ++j) dg_[j * F + f] = md_[j * F + f] = 0.0;
                }
            }
            for (int f = 0; f < F; ++f) {
                size_t o = ((size_t)n * L + l) * F + f;
                gamma[o] = g_[f];
                if (mgamma) mgamma[o] = mg_[f];
                if (lap) lap[o] = lp_[f];
                if (mlap) mlap[o] = ml_[f];
                for (int j = 0; j < d; ++j) {
                    size_t od = (((size_t)n * d + j) * L + l) * F + f;
                    if (dgamma) dgamma[od] = dg_[j * F + f];
                    if (mdgamma) mdgamma[od] = md_[j * F + f];
                }
            }
        }
    }
    return 0;
}

/* Backward for ONE level l: accumulate into grads[k] ([T_k][C(d,k)][F],
 * this level only, caller-zeroed) the transpose of the forward applied to
 * the upstream gradients (float32 inputs, widened exactly; point-major
 * layouts as in the forward; any of them may be NULL).  mags[k] receives the condition magnitudes.
 * Colliding vertices sum their contributions.  Serial over points.         */
int oracle_encode_bwd_level(int d, int L, int F, int l, const int32_t* res, const int32_t* log2T,
                            int64_t n_pts, const float* coords,
                            const float* g_gamma, const float* g_dgamma, const float* g_lap,
                            double* const* grads, double* const* mags) {
    if (d < 1 || d > OR_MAXD || l < 0 || l >= L) return 1;
    const double N = (double)res[l];
    const double dx = 1.0 / N;
    double scale[OR_MAXD + 1];
    for (int k = 0; k <= d; ++k) scale[k] = pow(dx, (double)k);   /* dx^{|alpha|} */
    int slot_of[1 << OR_MAXD], order_of[1 << OR_MAXD];
    for (int alpha = 0; alpha < (1 << d); ++alpha) {
        slot_of[alpha] = slot_in_bucket(d, alpha);
        order_of[alpha] = popcount_small(alpha);
    }
    for (int64_t n = 0; n < n_pts; ++n) {
        int64_t c[OR_MAXD];
        double t[OR_MAXD];
        for (int i = 0; i < d; ++i) locate(coords[n * d + i], res[l], &c[i], &t[i]);
        double hb[OR_MAXD][2][2][3];
        for (int i = 0; i < d; ++i)
            for (int vi = 0; vi < 2; ++vi)
                for (int a = 0; a < 2; ++a)
                    hermite_1d(a, t[i] - (double)vi, vi ? -1.0 : 1.0, hb[i][vi][a]);
        for (int v = 0; v < (1 << d); ++v) {
            int64_t g[OR_MAXD];
            for (int i = 0; i < d; ++i) g[i] = c[i] + (v >> i & 1);
            uint32_t idx[OR_MAXD + 1];
            for (int k = 0; k <= d; ++k) idx[k] = vertex_index(d, g, res[l], log2T[k]);
            for (int alpha = 0; alpha < (1 << d); ++alpha) {
                int k = order_of[alpha];
                const double (*h[OR_MAXD])[3];
                for (int i = 0; i < d; ++i) h[i] = &hb[i][v >> i & 1][alpha >> i & 1];
                double H = 1.0;
                for (int i = 0; i < d; ++i) H *= (*h[i])[0];
                double dH[OR_MAXD], d2H[OR_MAXD];
                for (int j = 0; j < d; ++j) {
                    dH[j] = 1.0; d2H[j] = 1.0;
                    for (int i = 0; i < d; ++i) {
                        dH[j] *= (i == j) ? (*h[i])[1] : (*h[i])[0];
                        d2H[j] *= (i == j) ? (*h[i])[2] : (*h[i])[0];
                    }
                }
                size_t off = ((size_t)idx[k] * binom(d, k) + slot_of[alpha]) * F;
                double* gk = grads[k] + off;
                double* mk = mags ? mags[k] + off : NULL;
                for (int f = 0; f < F; ++f) {
                    double up = g_gamma ? (double)g_gamma[((size_t)n * L + l) * F + f] : 0.0;
                    double w = up * H * scale[k];
                    double m = fabs(up) * fabs(H) * scale[k];
                    for (int j = 0; j < d; ++j) {
                        if (g_dgamma) {
                            double ud = (double)g_dgamma[(((size_t)n * d + j) * L + l) * F + f];
                            w += ud * scale[k] * N * dH[j];
                            m += fabs(ud) * scale[k] * N * fabs(dH[j]);
                        }
                        if (g_lap) {
                            double ul = (double)g_lap[((size_t)n * L + l) * F + f];
                            w += ul * scale[k] * N * N * d2H[j];
                            m += fabs(ul) * scale[k] * N * N * fabs(d2H[j]);
                        }
                    }
                    gk[f] += w;
                    if (mk) mk[f] += m;
                }
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* d-linear (Instant-NGP)                                                */
/* ------------------------------------------------------------------ */

/* gamma[N][L][F] = sum over the cell's corners of w_v * table[l][idx][f],
 * w_v = prod_i (v_i ? t_i : 1 - t_i); table is [L][T][F] contiguous.        */
int oracle_linear_fwd(int d, int L, int F, const int32_t* res, int log2T, uint32_t level_mask,
                      const double* table, int64_t n_pts, const float* coords,
                      double* gamma, double* mgamma, int nthreads) {
    if (d < 1 || d > OR_MAXD) return 1;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 256)
    for (int64_t n = 0; n < n_pts; ++n) {
        for (int l = 0; l < L; ++l) {
            for (int f = 0; f < F; ++f) {
                gamma[((size_t)n * L + l) * F + f] = 0.0;
                if (mgamma) mgamma[((size_t)n * L + l) * F + f] = 0.0;
            }
            if (!((level_mask >> l) & 1u)) continue;
            int64_t c[OR_MAXD];
            double t[OR_MAXD];
            for (int i = 0; i < d; ++i) locate(coords[n * d + i], res[l], &c[i], &t[i]);
            for (int v = 0; v < (1 << d); ++v) {
                int64_t g[OR_MAXD];
                double w = 1.0;
                for (int i = 0; i < d; ++i) {
                    int vi = v >> i & 1;
                    g[i] = c[i] + vi;
                    w *= vi ? t[i] : 1.0 - t[i];
                }
                uint32_t idx = vertex_index(d, g, res[l], log2T);
                const double* th = table + ((size_t)l * ((size_t)1 << log2T) + idx) * F;
                for (int f = 0; f < F; ++f) {
                    gamma[((size_t)n * L + l) * F + f] += w * th[f];
                    if (mgamma) mgamma[((size_t)n * L + l) * F + f] += fabs(w) * fabs(th[f]);
                }
            }
        }
    }
    return 0;
}

/* Backward of the d-linear forward for ONE level l into grad[T][F] (this
 * level only, caller-zeroed); mag may be NULL.  Serial over points.        */
int oracle_linear_bwd_level(int d, int L, int F, int l, const int32_t* res, int log2T,
                            int64_t n_pts, const float* coords, const float* g_gamma,
                            double* grad, double* mag) {
    if (d < 1 || d > OR_MAXD || l < 0 || l >= L) return 1;
    for (int64_t n = 0; n < n_pts; ++n) {
        int64_t c[OR_MAXD];
        double t[OR_MAXD];
        for (int i = 0; i < d; ++i) locate(coords[n * d + i], res[l], &c[i], &t[i]);
        for (int v = 0; v < (1 << d); ++v) {
            int64_t g[OR_MAXD];
            double w = 1.0;
            for (int i = 0; i < d; ++i) {
                int vi = v >> i & 1;
                g[i] = c[i] + vi;
                w *= vi ? t[i] : 1.0 - t[i];
            }
            uint32_t idx = vertex_index(d, g, res[l], log2T);
            for (int f = 0; f < F; ++f) {
                double up = (double)g_gamma[((size_t)n * L + l) * F + f];
                grad[(size_t)idx * F + f] += w * up;
                if (mag) mag[(size_t)idx * F + f] += fabs(w) * fabs(up);
            }
        }
    }
    return 0;
}

/* The bucket slot of alpha, exposed so tests can check the ordering rule. */
int oracle_slot_in_bucket(int d, int alpha) { return slot_in_bucket(d, alpha); }

/* ------------------------------------------------------------------ */
/* Full Hessian (the upper triangle of d2 gamma / dx_i dx_j)            */
/* ------------------------------------------------------------------ */

int oracle_hess_entries(int d) { return hess_entries(d); }

/* One cell at an fp64 local coordinate: gamma[F], dgamma[d][F], hess[P][F]. */
int oracle_eval_cell_hessian(int d, int F, int32_t N, const int32_t* log2T,
                             const double* const* tables, const int64_t* c, const double* t,
                             double* gamma, double* dgamma, double* hess) {
    if (d < 1 || d > OR_MAXD) return 1;
    or_level lv = {d, F, N, log2T, tables};
    hermite_cell_h(&lv, c, t, gamma, dgamma, NULL, NULL, NULL, NULL, hess, NULL);
    return 0;
}

/* Forward with the Hessian: point-major gamma[N][L][F], dgamma[N][d][L][F],
 * hess[N][P][L][F] and their magnitudes (any magnitude array may be NULL). */
int oracle_encode_fwd_hessian(int d, int L, int F, const int32_t* res, const int32_t* log2T,
                              uint32_t level_mask, const double* const* tables,
                              int64_t n_pts, const float* coords,
                              double* gamma, double* dgamma, double* hess,
                              double* mgamma, double* mdgamma, double* mhess, int nthreads) {
    if (d < 1 || d > OR_MAXD || L < 1 || F < 1 || F > 8) return 1;
    set_threads(nthreads);
    const int P = hess_entries(d);
#pragma omp parallel for schedule(dynamic, 256)
    for (int64_t n = 0; n < n_pts; ++n) {
        double g_[8], dg_[OR_MAXD * 8], h_[OR_MAXP * 8], mg_[8], md_[OR_MAXD * 8], mh_[OR_MAXP * 8];
        for (int l = 0; l < L; ++l) {
            if ((level_mask >> l) & 1u) {
                const double* tab_l[OR_MAXD + 1];
                for (int k = 0; k <= d; ++k)
                    tab_l[k] = tables[k] + (size_t)l * ((size_t)1 << log2T[k]) * binom(d, k) * F;
                or_level lv = {d, F, res[l], log2T, tab_l};
                int64_t c[OR_MAXD];
                double t[OR_MAXD];
                for (int i = 0; i < d; ++i) locate(coords[n * d + i], res[l], &c[i], &t[i]);
                hermite_cell_h(&lv, c, t, g_, dg_, NULL, mg_, md_, NULL, h_, mh_);
            } else {
                for (int f = 0; f < F; ++f) {
                    g_[f] = mg_[f] = 0.0;
                    for (int j = 0; j < d; ++j) dg_[j * F + f] = md_[j * F + f] = 0.0;
                    for (int q = 0; q < P; ++q) h_[q * F + f] = mh_[q * F + f] = 0.0;
                }
            }
            for (int f = 0; f < F; ++f) {
                size_t o = ((size_t)n * L + l) * F + f;
                gamma[o] = g_[f];
                if (mgamma) mgamma[o] = mg_[f];
                for (int j = 0; j < d; ++j) {
                    size_t od = (((size_t)n * d + j) * L + l) * F + f;
                    if (dgamma) dgamma[od] = dg_[j * F + f];
                    if (mdgamma) mdgamma[od] = md_[j * F + f];
                }
                for (int q = 0; q < P; ++q) {
                    size_t oh = (((size_t)n * P + q) * L + l) * F + f;
                    if (hess) hess[oh] = h_[q * F + f];
                    if (mhess) mhess[oh] = mh_[q * F + f];
                }
            }
        }
    }
    return 0;
}

/* Backward of the Hessian forward for ONE level l: grads[k] ([T_k][C][F],
 * caller-zeroed) += the transpose applied to g_gamma [N][L][F],
 * g_dgamma [N][d][L][F], g_hess [N][P][L][F] (float32, any may be NULL);
 * mags[k] the condition magnitudes (may be NULL).  Serial over points.    */
int oracle_encode_bwd_hessian_level(int d, int L, int F, int l, const int32_t* res, const int32_t* log2T,
                                    int64_t n_pts, const float* coords,
                                    const float* g_gamma, const float* g_dgamma, const float* g_hess,
                                    double* const* grads, double* const* mags) {
    if (d < 1 || d > OR_MAXD || l < 0 || l >= L) return 1;
    const int P = hess_entries(d);
    const double N = (double)res[l];
    const double dx = 1.0 / N;
    double scale[OR_MAXD + 1];
    for (int k = 0; k <= d; ++k) scale[k] = pow(dx, (double)k);
    for (int64_t n = 0; n < n_pts; ++n) {
        int64_t c[OR_MAXD];
        double t[OR_MAXD];
        for (int i = 0; i < d; ++i) locate(coords[n * d + i], res[l], &c[i], &t[i]);
        double hb[OR_MAXD][2][2][3];
        for (int i = 0; i < d; ++i)
            for (int vi = 0; vi < 2; ++vi)
                for (int a = 0; a < 2; ++a)
                    hermite_1d(a, t[i] - (double)vi, vi ? -1.0 : 1.0, hb[i][vi][a]);
        for (int v = 0; v < (1 << d); ++v) {
            int64_t g[OR_MAXD];
            for (int i = 0; i < d; ++i) g[i] = c[i] + (v >> i & 1);
            for (int alpha = 0; alpha < (1 << d); ++alpha) {
                const int k = popcount_small(alpha);
                const uint32_t idx = vertex_index(d, g, res[l], log2T[k]);
                const double (*h[OR_MAXD])[3];
                for (int i = 0; i < d; ++i) h[i] = &hb[i][v >> i & 1][alpha >> i & 1];
                double H = 1.0;
                for (int i = 0; i < d; ++i) H *= (*h[i])[0];
                double dH[OR_MAXD], hij[OR_MAXP];
                for (int j = 0; j < d; ++j) {
                    dH[j] = 1.0;
                    for (int i = 0; i < d; ++i) dH[j] *= (i == j) ? (*h[i])[1] : (*h[i])[0];
                }
                for (int i = 0; i < d; ++i)
                    for (int j = i; j < d; ++j) {
                        double x = 1.0;
                        for (int m = 0; m < d; ++m) {
                            if (i == j) x *= (m == i) ? (*h[m])[2] : (*h[m])[0];
                            else x *= (m == i || m == j) ? (*h[m])[1] : (*h[m])[0];
                        }
                        hij[hess_pos(d, i, j)] = x;
                    }
                const size_t off = ((size_t)idx * binom(d, k) + slot_in_bucket(d, alpha)) * F;
                for (int f = 0; f < F; ++f) {
                    double w = 0.0, m = 0.0;
                    if (g_gamma) {
                        double up = (double)g_gamma[((size_t)n * L + l) * F + f];
                        w += up * H * scale[k];
                        m += fabs(up) * fabs(H) * scale[k];
                    }
                    for (int j = 0; j < d && g_dgamma; ++j) {
                        double ud = (double)g_dgamma[(((size_t)n * d + j) * L + l) * F + f];
                        w += ud * scale[k] * N * dH[j];
                        m += fabs(ud) * scale[k] * N * fabs(dH[j]);
                    }
                    for (int q = 0; q < P && g_hess; ++q) {
                        double uh = (double)g_hess[(((size_t)n * P + q) * L + l) * F + f];
                        w += uh * scale[k] * N * N * hij[q];
                        m += fabs(uh) * scale[k] * N * N * fabs(hij[q]);
                    }
                    grads[k][off + f] += w;
                    if (mags) mags[k][off + f] += m;
                }
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* INGP-FD: the d-linear encoding with central finite differences       */
/* ------------------------------------------------------------------ */
/* "Hermite-NGP: Gradient-Augmented Hash Encoding for Learning PDEs",
 * sections 研究背景与动机 and 关键设计 2: the INGP-FD baseline takes the
 * Laplacian by central differences from 2d+1 forward passes, at x and at
 * x +- eps e_i.  Readings: the shifted coordinate is one fp32 add
 * (x_i + eps, x_i - eps) and is then located like any coordinate (clamped
 * to [0,1]); the differences are the textbook central ones,
 *   d gamma / dx_i ~ (gamma(x + eps e_i) - gamma(x - eps e_i)) / (2 eps),
 *   lap gamma      ~ sum_i (gamma(x + eps e_i) - 2 gamma(x) + gamma(x - eps e_i)) / eps^2.
 * Stencil output j = 2i is x + eps e_i, j = 2i + 1 is x - eps e_i.          */

/* d-linear encoding of one point at one level (table_l = [T][F]). */
static void linear_point(int d, int F, int32_t N, int log2T, const double* table_l, const float* x,
                         double* out, double* mag) {
    int64_t c[OR_MAXD];
    double t[OR_MAXD];
    for (int i = 0; i < d; ++i) locate(x[i], N, &c[i], &t[i]);
    for (int f = 0; f < F; ++f) out[f] = mag[f] = 0.0;
    for (int v = 0; v < (1 << d); ++v) {
        int64_t g[OR_MAXD];
        double w = 1.0;
        for (int i = 0; i < d; ++i) {
            const int vi = v >> i & 1;
            g[i] = c[i] + vi;
            w *= vi ? t[i] : 1.0 - t[i];
        }
        const double* th = table_l + (size_t)vertex_index(d, g, N, log2T) * F;
        for (int f = 0; f < F; ++f) {
            out[f] += w * th[f];
            mag[f] += fabs(w) * fabs(th[f]);
        }
    }
}

/* The coordinates of stencil point s of x: s = 0 is x, s = 1 + j is stencil
 * output j (j = 2i: x + eps e_i; j = 2i + 1: x - eps e_i). */
static void stencil_coords(int d, const float* x, float eps, int s, float* xs) {
    for (int i = 0; i < d; ++i) xs[i] = x[i];
    if (s > 0) {
        const int j = s - 1, i = j / 2;
        volatile float shifted = (j % 2 == 0) ? x[i] + eps : x[i] - eps;
        xs[i] = shifted;
    }
}

/* Forward: gamma[N][L][F] (at x), dgamma[N][d][L][F], lap[N][L][F] and the
 * stencil encodings stencil[N][2d][L][F]; table [L][T][F].  Any output but
 * gamma, and every magnitude array, may be NULL. */
int oracle_linear_fd_fwd(int d, int L, int F, const int32_t* res, int log2T, uint32_t level_mask,
                         const double* table, int64_t n_pts, const float* coords, float eps,
                         double* gamma, double* dgamma, double* lap, double* stencil,
                         double* mgamma, double* mdgamma, double* mlap, double* mstencil, int nthreads) {
    if (d < 1 || d > OR_MAXD || L < 1 || F < 1 || F > 8 || !(eps > 0.0f)) return 1;
    set_threads(nthreads);
    const int S = 2 * d + 1;
    const double e = (double)eps;
#pragma omp parallel for schedule(dynamic, 256)
    for (int64_t n = 0; n < n_pts; ++n) {
        double gs[2 * OR_MAXD + 1][8], ms[2 * OR_MAXD + 1][8];
        for (int l = 0; l < L; ++l) {
            const int active = (level_mask >> l) & 1u;
            for (int s = 0; s < S; ++s) {
                if (active) {
                    float xs[OR_MAXD];
                    stencil_coords(d, coords + n * d, eps, s, xs);
                    linear_point(d, F, res[l], log2T, table + (size_t)l * ((size_t)1 << log2T) * F, xs, gs[s], ms[s]);
                } else {
                    for (int f = 0; f < F; ++f) gs[s][f] = ms[s][f] = 0.0;
                }
            }
            for (int f = 0; f < F; ++f) {
                const size_t o = ((size_t)n * L + l) * F + f;
                gamma[o] = gs[0][f];
                if (mgamma) mgamma[o] = ms[0][f];
                double lp = 0.0, ml = 0.0;
                for (int i = 0; i < d; ++i) {
                    const double gp = gs[1 + 2 * i][f], gm = gs[2 + 2 * i][f];
                    const double mp = ms[1 + 2 * i][f], mm = ms[2 + 2 * i][f];
                    const size_t od = (((size_t)n * d + i) * L + l) * F + f;
                    if (dgamma) dgamma[od] = (gp - gm) / (2.0 * e);
                    if (mdgamma) mdgamma[od] = (mp + mm) / (2.0 * e);
                    lp += (gp - 2.0 * gs[0][f] + gm) / (e * e);
                    ml += (mp + 2.0 * ms[0][f] + mm) / (e * e);
                }
                if (lap) lap[o] = lp;
                if (mlap) mlap[o] = ml;
                for (int j = 0; j < 2 * d; ++j) {
                    const size_t os = (((size_t)n * 2 * d + j) * L + l) * F + f;
                    if (stencil) stencil[os] = gs[1 + j][f];
                    if (mstencil) mstencil[os] = ms[1 + j][f];
                }
            }
        }
    }
    return 0;
}

/* Backward of oracle_linear_fd_fwd for ONE level l into grad[T][F] (this
 * level only, caller-zeroed; mag may be NULL).  Upstream gradients are
 * float32, point-major as the forward's outputs; any may be NULL.  Each
 * stencil point s receives the upstream weight of its value in the outputs:
 *   s = x:          g_gamma - (2d / eps^2) g_lap
 *   s = x + eps e_i:  g_dgamma_i / (2 eps) + g_lap / eps^2 + g_stencil_2i
 *   s = x - eps e_i: -g_dgamma_i / (2 eps) + g_lap / eps^2 + g_stencil_2i+1
 * and scatters it with its d-linear corner weights.  Serial over points. */
int oracle_linear_fd_bwd_level(int d, int L, int F, int l, const int32_t* res, int log2T, int64_t n_pts,
                               const float* coords, float eps, const float* g_gamma, const float* g_dgamma,
                               const float* g_lap, const float* g_stencil, double* grad, double* mag) {
    if (d < 1 || d > OR_MAXD || l < 0 || l >= L || F < 1 || F > 8 || !(eps > 0.0f)) return 1;
    const int S = 2 * d + 1;
    const double e = (double)eps;
    for (int64_t n = 0; n < n_pts; ++n) {
        double u[2 * OR_MAXD + 1][8], mu[2 * OR_MAXD + 1][8];
        for (int f = 0; f < F; ++f) {
            const size_t o = ((size_t)n * L + l) * F + f;
            const double gg = g_gamma ? (double)g_gamma[o] : 0.0;
            const double gl = g_lap ? (double)g_lap[o] : 0.0;
            u[0][f] = gg - 2.0 * d * gl / (e * e);
            mu[0][f] = fabs(gg) + 2.0 * d * fabs(gl) / (e * e);
            for (int i = 0; i < d; ++i) {
                const double gd = g_dgamma ? (double)g_dgamma[(((size_t)n * d + i) * L + l) * F + f] : 0.0;
                for (int sgn = 0; sgn < 2; ++sgn) {
                    const int j = 2 * i + sgn;
                    const double gs = g_stencil ? (double)g_stencil[(((size_t)n * 2 * d + j) * L + l) * F + f] : 0.0;
                    const double dir = sgn ? -1.0 : 1.0;
                    u[1 + j][f] = dir * gd / (2.0 * e) + gl / (e * e) + gs;
                    mu[1 + j][f] = fabs(gd) / (2.0 * e) + fabs(gl) / (e * e) + fabs(gs);
                }
            }
        }
        for (int s = 0; s < S; ++s) {
            float xs[OR_MAXD];
            stencil_coords(d, coords + n * d, eps, s, xs);
            int64_t c[OR_MAXD];
            double t[OR_MAXD];
            for (int i = 0; i < d; ++i) locate(xs[i], res[l], &c[i], &t[i]);
            for (int v = 0; v < (1 << d); ++v) {
                int64_t g[OR_MAXD];
                double w = 1.0;
                for (int i = 0; i < d; ++i) {
                    const int vi = v >> i & 1;
                    g[i] = c[i] + vi;
                    w *= vi ? t[i] : 1.0 - t[i];
                }
                const size_t idx = vertex_index(d, g, res[l], log2T);
                for (int f = 0; f < F; ++f) {
                    grad[idx * F + f] += w * u[s][f];
                    if (mag) mag[idx * F + f] += fabs(w) * mu[s][f];
                }
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* Gaussian-RBF multi-resolution grid (DInf-Grid)                        */
/* ------------------------------------------------------------------ */
/* "DInf-Grid：一种基于可微特征网格的神经微分方程求解器", sections 可微的径向基函数
 * 插值 and 多分辨率特征网格: per grid (level), the feature at x is
 *   f(x) = sum_{i in N(x)} w(x, x_i) F_i,
 *   w(x, x_i) = phi(|x - x_i|) / sum_{j in N(x)} phi(|x - x_j|),
 *   phi(r) = exp(-(eps r)^2),
 * over a precomputed ring neighbourhood N(x) of the point's cell, and the
 * levels' features are concatenated.  Readings: r is measured in the
 * level's grid units (y = N_l x, vertex g at y = g), so eps = 1 with 3 rings
 * covers the kernel's effective support; ring R holds the vertices g with
 * c_i - R + 1 <= g_i <= c_i + R on every axis, clipped to the grid
 * (0 <= g_i <= N_l); the cell c and y = c + t come from the same location
 * as the hash grid (pos = fl32(x N_l)); vertices are indexed like the hash
 * grid's (one-to-one when the level fits T, so the page's dense grids are
 * that case).  Derivatives are exact: with S = sum_j phi_j,
 *   d w_i / dy = (d phi_i - w_i dS) / S,
 *   lap w_i    = (lap phi_i - 2 grad w_i . grad S - w_i lap S) / S,
 *   d phi / dy_k = -2 eps^2 (y_k - g_k) phi,  lap phi = (4 eps^4 |y - g|^2 - 2 d eps^2) phi,
 * and d/dx = N_l d/dy.                                                   */

#define OR_MAX_RINGS 4

/* Neighbourhood of one point at one level: vertex list, normalised weights
 * w, their x-derivatives dw[k] and Laplacian lw, and the condition
 * magnitudes of each (every term of the quotient rule in absolute value). */
typedef struct {
    int count;
    int64_t g[(2 * OR_MAX_RINGS) * (2 * OR_MAX_RINGS) * (2 * OR_MAX_RINGS) * (2 * OR_MAX_RINGS)][OR_MAXD];
    double w[4096], dw[4096][OR_MAXD], lw[4096];
    double mw[4096], mdw[4096][OR_MAXD], mlw[4096];
} rbf_nbhd;

static void rbf_weights(int d, int32_t N, const float* x_in, double eps, int rings, rbf_nbhd* nb) {
    int64_t c[OR_MAXD];
    double t[OR_MAXD], y[OR_MAXD];
    for (int i = 0; i < d; ++i) {
        locate(x_in[i], N, &c[i], &t[i]);
        y[i] = (double)c[i] + t[i];
    }
    const int side = 2 * rings;
    int64_t total = 1;
    for (int i = 0; i < d; ++i) total *= side;
    const double e2 = eps * eps;
    double phi[4096], dphi[4096][OR_MAXD], lphi[4096];
    double S = 0.0, dS[OR_MAXD] = {0}, lS = 0.0, mdS[OR_MAXD] = {0}, mlS = 0.0;
    nb->count = 0;
    for (int64_t m = 0; m < total; ++m) {
        int64_t g[OR_MAXD], rem = m;
        int inside = 1;
        for (int i = 0; i < d; ++i) {
            g[i] = c[i] - rings + 1 + rem % side;
            rem /= side;
            if (g[i] < 0 || g[i] > N) inside = 0;
        }
        if (!inside) continue;
        const int q = nb->count++;
        double r2 = 0.0;
        for (int i = 0; i < d; ++i) {
            nb->g[q][i] = g[i];
            r2 += (y[i] - (double)g[i]) * (y[i] - (double)g[i]);
        }
        phi[q] = exp(-e2 * r2);
        for (int i = 0; i < d; ++i) dphi[q][i] = -2.0 * e2 * (y[i] - (double)g[i]) * phi[q];
        lphi[q] = (4.0 * e2 * e2 * r2 - 2.0 * d * e2) * phi[q];
        S += phi[q];
        for (int i = 0; i < d; ++i) {
            dS[i] += dphi[q][i];
            mdS[i] += fabs(dphi[q][i]);
        }
        lS += lphi[q];
        mlS += fabs(lphi[q]);
    }
    const double Nd = (double)N;
    for (int q = 0; q < nb->count; ++q) {
        const double w = phi[q] / S;
        nb->w[q] = w;
        nb->mw[q] = w;
        double dot = 0.0, mdot = 0.0;
        double dwy[OR_MAXD], mdwy[OR_MAXD];
        for (int i = 0; i < d; ++i) {
            dwy[i] = (dphi[q][i] - w * dS[i]) / S;
            mdwy[i] = (fabs(dphi[q][i]) + w * mdS[i]) / S;
            dot += dwy[i] * dS[i];
            mdot += mdwy[i] * mdS[i];
            nb->dw[q][i] = Nd * dwy[i];
            nb->mdw[q][i] = Nd * mdwy[i];
        }
        nb->lw[q] = Nd * Nd * (lphi[q] - 2.0 * dot - w * lS) / S;
        nb->mlw[q] = Nd * Nd * (fabs(lphi[q]) + 2.0 * mdot + w * mlS) / S;
    }
}

static int rbf_args_ok(int d, int L, int F, float eps, int rings) {
    return d >= 1 && d <= OR_MAXD && L >= 1 && F >= 1 && F <= 8 && eps > 0.0f && rings >= 1 &&
           rings <= OR_MAX_RINGS;
}

/* Forward: gamma[N][L][F], dgamma[N][d][L][F], lap[N][L][F] and magnitudes
 * (any but gamma may be NULL); table [L][T][F]. */
int oracle_rbf_fwd(int d, int L, int F, const int32_t* res, int log2T, uint32_t level_mask, const double* table,
                   int64_t n_pts, const float* coords, float eps, int rings, double* gamma, double* dgamma, double* lap,
                   double* mgamma, double* mdgamma, double* mlap, int nthreads) {
    if (!rbf_args_ok(d, L, F, eps, rings)) return 1;
    set_threads(nthreads);
#pragma omp parallel
    {
        rbf_nbhd* nb = (rbf_nbhd*)malloc(sizeof(rbf_nbhd));
#pragma omp for schedule(dynamic, 64)
        for (int64_t n = 0; n < n_pts; ++n) {
            for (int l = 0; l < L; ++l) {
                const int active = (level_mask >> l) & 1u;
                if (active && nb) rbf_weights(d, res[l], coords + n * d, (double)eps, rings, nb);
                for (int f = 0; f < F; ++f) {
                    double g = 0, mg = 0, dg[OR_MAXD] = {0}, md[OR_MAXD] = {0}, lp = 0, ml = 0;
                    if (active && nb) {
                        for (int q = 0; q < nb->count; ++q) {
                            const uint32_t idx = vertex_index(d, nb->g[q], res[l], log2T);
                            const double th = table[((size_t)l * ((size_t)1 << log2T) + idx) * F + f];
                            g += nb->w[q] * th;
                            mg += nb->mw[q] * fabs(th);
                            for (int i = 0; i < d; ++i) {
                                dg[i] += nb->dw[q][i] * th;
                                md[i] += nb->mdw[q][i] * fabs(th);
                            }
                            lp += nb->lw[q] * th;
                            ml += nb->mlw[q] * fabs(th);
                        }
                    }
                    const size_t o = ((size_t)n * L + l) * F + f;
                    gamma[o] = g;
                    if (mgamma) mgamma[o] = mg;
                    if (lap) lap[o] = lp;
                    if (mlap) mlap[o] = ml;
                    for (int i = 0; i < d; ++i) {
                        const size_t od = (((size_t)n * d + i) * L + l) * F + f;
                        if (dgamma) dgamma[od] = dg[i];
                        if (mdgamma) mdgamma[od] = md[i];
                    }
                }
            }
        }
        free(nb);
    }
    return 0;
}

/* Backward for ONE level l into grad[T][F] (caller-zeroed; mag may be NULL):
 * grad[idx(g)] += g_gamma w + sum_i g_dgamma_i dw_i + g_lap lw.  Serial. */
int oracle_rbf_bwd_level(int d, int L, int F, int l, const int32_t* res, int log2T, int64_t n_pts,
                         const float* coords, float eps, int rings, const float* g_gamma, const float* g_dgamma,
                         const float* g_lap, double* grad, double* mag) {
    if (!rbf_args_ok(d, L, F, eps, rings) || l < 0 || l >= L) return 1;
    rbf_nbhd* nb = (rbf_nbhd*)malloc(sizeof(rbf_nbhd));
    if (!nb) return 2;
    for (int64_t n = 0; n < n_pts; ++n) {
        rbf_weights(d, res[l], coords + n * d, (double)eps, rings, nb);
        for (int q = 0; q < nb->count; ++q) {
            const size_t idx = vertex_index(d, nb->g[q], res[l], log2T);
            for (int f = 0; f < F; ++f) {
                const size_t o = ((size_t)n * L + l) * F + f;
                double w = 0.0, m = 0.0;
                if (g_gamma) {
                    w += (double)g_gamma[o] * nb->w[q];
                    m += fabs((double)g_gamma[o]) * nb->mw[q];
                }
                for (int i = 0; i < d && g_dgamma; ++i) {
                    const double u = (double)g_dgamma[(((size_t)n * d + i) * L + l) * F + f];
                    w += u * nb->dw[q][i];
                    m += fabs(u) * nb->mdw[q][i];
                }
                if (g_lap) {
                    w += (double)g_lap[o] * nb->lw[q];
                    m += fabs((double)g_lap[o]) * nb->mlw[q];
                }
                grad[idx * F + f] += w;
                if (mag) mag[idx * F + f] += m;
            }
        }
    }
    free(nb);
    return 0;
}
