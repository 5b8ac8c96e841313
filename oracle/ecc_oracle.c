/*
 * ecc_oracle.c -- plain, slow, CPU reference for the Euler characteristic curve (ECC) of a dense
 * cubical grid and for its sigmoid-relaxed ("soft") form with analytic gradients.
 *
 * TEST INFRASTRUCTURE ONLY. The test-suite, the smoke check and the benchmark's CPU-baseline leg
 * are the only callers. The product (the CUDA library behind include/ecc.h and its Python binding)
 * never loads, links or calls this file, and this file shares no code, header, table or constant
 * with it.
 *
 * Method source: the paper notes "Scalable GPU-Accelerated Euler Characteristic Curves:
 * Optimization and Differentiable Learning for PyTorch" (NeurIPS 2025 NeurReps workshop,
 * arXiv 2510.20271), cited below as [ECC notes] with the section name.
 *
 * What is computed, written as the plain definition rather than the fast per-voxel method:
 *
 *  Hard ECC ([ECC notes], "Research background" and "Key designs -- local computation of the Euler
 *  characteristic coefficient"). The grid is the V-construction cubical complex: every voxel is a
 *  vertex, and every axis-aligned box of side 0 or 1 per axis whose 2^dim corners lie in the grid is
 *  a cell of dimension dim (edges, squares, cubes). A cell belongs to the sublevel set at threshold
 *  t exactly when every one of its vertices has value <= t. The curve is
 *        ECC(t_k) = sum over cells in the sublevel set at t_k of (-1)^dim.
 *  Thresholds: H = nbins values, t_0 = vmin, t_{H-1} = vmax, and for 0 < k < H-1
 *        t_k = vmin + ((vmax - vmin) * k) / (H - 1)            (fp64, in that order);
 *  for H = 1 the single threshold is vmax. Voxel values (uint8 or fp32) are promoted exactly to
 *  fp64. NaN never satisfies v <= t, so a NaN voxel and every cell touching it never enter.
 *
 *  Soft ECC ([ECC notes], "Key designs -- differentiable ECC layer (sigmoid relaxation)"). The
 *  indicator 1[X <= t] is replaced by sigma(lambda (t - X)), sigma(z) = 1 / (1 + exp(-z)), with the
 *  single-direction filtration X(p) = alpha f(p) + u . x_p. A cell's filtration value is the max of
 *  X over its vertices, so
 *        S(t_k) = sum over cells of (-1)^dim sigma(lambda (t_k - max_{v in cell} X(v))).
 *  x_p are the voxel's coordinates, centred and scaled to [-1, 1] per axis:
 *        x_{p,d} = (2 i_d - (n_d - 1)) / (n_d - 1)   (0 when n_d = 1).
 *  X is evaluated in fp64 as ((alpha * f) + u_0 x_0) + u_1 x_1 (+ u_2 x_2), each product and sum
 *  rounded separately (this file must be compiled with -ffp-contract=off).
 *  Gradients follow the chain rule through each cell's argmax vertex; when several vertices share
 *  the max, the vertex with the larger linear index owns the cell.
 *  tau, alpha and u are shared across the batch, so their gradients sum over images.
 *
 * Every array is C-contiguous with the last axis fastest: image b, voxel (i_0, ..., i_{ndim-1}) is
 * element b * N + linear index, N = product of dims.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL (-1)
#define ORACLE_ENOMEM (-2)

/* ------------------------------------------------------------------------------------------ */
/* Thresholds                                                                                  */
/* ------------------------------------------------------------------------------------------ */

/* The H thresholds of the hard ECC, in fp64 (see the header comment). */
int oracle_thresholds(int nbins, double vmin, double vmax, double *tau)
{
    if (nbins < 1 || !tau || !(vmin <= vmax)) return ORACLE_EINVAL;
    if (nbins == 1) {
        tau[0] = vmax;
        return ORACLE_OK;
    }
    for (int k = 0; k < nbins; ++k) {
        if (k == 0)
            tau[k] = vmin;
        else if (k == nbins - 1)
            tau[k] = vmax;
        else
            tau[k] = vmin + ((vmax - vmin) * (double)k) / (double)(nbins - 1);
    }
    return ORACLE_OK;
}

/* Smallest k with v <= tau[k]; nbins when no threshold admits v (v above vmax, or NaN).
 * tau is non-decreasing, so this is a plain binary search on the predicate v <= tau[k]. */
static int first_threshold(double v, const double *tau, int nbins)
{
    int lo = 0, hi = nbins; /* answer in [lo, hi] */
    while (lo < hi) {
        int mid = lo + (hi - lo) / 2;
        if (v <= tau[mid])
            hi = mid;
        else
            lo = mid + 1;
    }
    return lo;
}

static double voxel_value(const void *img, int dtype, int64_t i)
{
    if (dtype == 0) return (double)((const uint8_t *)img)[i];
    return (double)((const float *)img)[i];
}

/* ------------------------------------------------------------------------------------------ */
/* Cell enumeration helpers                                                                     */
/* ------------------------------------------------------------------------------------------ */

typedef struct {
    int ndim;
    int64_t n[3];      /* extent per axis, slowest first */
    int64_t stride[3]; /* linear stride per axis */
    int64_t N;         /* voxels per image */
} grid_t;

static int make_grid(int ndim, const int64_t *dims, grid_t *g)
{
    if (ndim < 1 || ndim > 3 || !dims) return ORACLE_EINVAL;
    g->ndim = ndim;
    g->N = 1;
    for (int d = 0; d < ndim; ++d) {
        if (dims[d] < 1) return ORACLE_EINVAL;
        g->n[d] = dims[d];
        g->N *= dims[d];
    }
    int64_t s = 1;
    for (int d = ndim - 1; d >= 0; --d) {
        g->stride[d] = s;
        s *= g->n[d];
    }
    return ORACLE_OK;
}

/* Coordinates of a linear index. */
static void unravel(const grid_t *g, int64_t lin, int64_t *idx)
{
    for (int d = 0; d < g->ndim; ++d) {
        idx[d] = lin / g->stride[d];
        lin -= idx[d] * g->stride[d];
    }
}

/* The cell with lower corner p spanning the axes in bitmask S exists when p + e_d is inside the
 * grid for every d in S. Its vertices are p + sum_{d in T} e_d for every subset T of S. */
static int cell_exists(const grid_t *g, const int64_t *idx, int S)
{
    for (int d = 0; d < g->ndim; ++d)
        if ((S >> d & 1) && idx[d] + 1 >= g->n[d]) return 0;
    return 1;
}

static int popcount_small(int S)
{
    int c = 0;
    while (S) {
        c += S & 1;
        S >>= 1;
    }
    return c;
}

/* Linear offset of vertex T (a subset of the cell's axes) from the lower corner. */
static int64_t vertex_offset(const grid_t *g, int T)
{
    int64_t off = 0;
    for (int d = 0; d < g->ndim; ++d)
        if (T >> d & 1) off += g->stride[d];
    return off;
}

/* ------------------------------------------------------------------------------------------ */
/* Hard ECC                                                                                     */
/* ------------------------------------------------------------------------------------------ */

/*
 * out[b * nbins + k] = ECC of image b at threshold t_k (int64). dtype 0 = uint8, 1 = float32.
 * Each cell enters at the first threshold that admits all of its vertices, which is the largest
 * of its vertices' first thresholds (v <= t is monotone in t); cells that never enter are skipped.
 * The per-threshold count is then the running sum of the cells entering at or below it.
 */
int oracle_ecc_hard(const void *img, int dtype, int ndim, const int64_t *dims, int64_t batch,
                    int nbins, double vmin, double vmax, int64_t *out)
{
    grid_t g;
    if (!img || !out || batch < 0 || (dtype != 0 && dtype != 1)) return ORACLE_EINVAL;
    if (make_grid(ndim, dims, &g) != ORACLE_OK) return ORACLE_EINVAL;
    double *tau = (double *)malloc(sizeof(double) * (size_t)nbins);
    int *first = (int *)malloc(sizeof(int) * (size_t)g.N);
    int64_t *entering = (int64_t *)malloc(sizeof(int64_t) * (size_t)nbins);
    if (!tau || !first || !entering) {
        free(tau);
        free(first);
        free(entering);
        return ORACLE_ENOMEM;
    }
    if (oracle_thresholds(nbins, vmin, vmax, tau) != ORACLE_OK) {
        free(tau);
        free(first);
        free(entering);
        return ORACLE_EINVAL;
    }
    int ncell_types = 1 << ndim;
    int64_t voff[8];
    for (int T = 0; T < ncell_types; ++T) voff[T] = vertex_offset(&g, T);

    for (int64_t b = 0; b < batch; ++b) {
        const int64_t base = b * g.N;
        for (int64_t i = 0; i < g.N; ++i)
            first[i] = first_threshold(voxel_value(img, dtype, base + i), tau, nbins);
        memset(entering, 0, sizeof(int64_t) * (size_t)nbins);
        int64_t idx[3];
        for (int64_t p = 0; p < g.N; ++p) {
            unravel(&g, p, idx);
            for (int S = 0; S < ncell_types; ++S) {
                if (!cell_exists(&g, idx, S)) continue;
                int k = 0;
                for (int T = 0; T < ncell_types; ++T) {
                    if ((T & ~S) != 0) continue; /* T must be a subset of S */
                    int kv = first[p + voff[T]];
                    if (kv > k) k = kv;
                }
                if (k < nbins) entering[k] += (popcount_small(S) & 1) ? -1 : 1;
            }
        }
        int64_t run = 0;
        for (int k = 0; k < nbins; ++k) {
            run += entering[k];
            out[b * nbins + k] = run;
        }
    }
    free(tau);
    free(first);
    free(entering);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------------------------ */
/* Soft ECC                                                                                     */
/* ------------------------------------------------------------------------------------------ */

static double sigmoid(double z)
{
    if (z >= 0) return 1.0 / (1.0 + exp(-z));
    double e = exp(z);
    return e / (1.0 + e);
}

/* Coordinate of index i on an axis of n voxels, centred and scaled to [-1, 1]. */
static double axis_coord(int64_t i, int64_t n)
{
    if (n == 1) return 0.0;
    return (2.0 * (double)i - (double)(n - 1)) / (double)(n - 1);
}

/* X for every voxel of one image, in fp64, in the order stated in the header. */
static void filtration(const grid_t *g, const float *f, double alpha, const double *u, double *X)
{
    int64_t idx[3];
    for (int64_t p = 0; p < g->N; ++p) {
        unravel(g, p, idx);
        double x = alpha * (double)f[p];
        for (int d = 0; d < g->ndim; ++d) x = x + u[d] * axis_coord(idx[d], g->n[d]);
        X[p] = x;
    }
}

/* Owner (argmax of X, ties to the larger linear index) of the cell with lower corner p, axes S. */
static int64_t cell_owner(const double *X, int64_t p, int S, int ncell_types, const int64_t *voff)
{
    int64_t best = p;
    for (int T = 1; T < ncell_types; ++T) {
        if ((T & ~S) != 0) continue;
        int64_t q = p + voff[T];
        if (X[q] > X[best] || (X[q] == X[best] && q > best)) best = q;
    }
    return best;
}

/*
 * out[b * K + k] = S(t_k) for image b (fp64). f: float32 images; tau: K thresholds; u: ndim values.
 */
int oracle_ecc_soft_fwd(const float *img, int ndim, const int64_t *dims, int64_t batch,
                        const float *tau, int K, double lambda, double alpha, const double *u,
                        double *out)
{
    grid_t g;
    if (!img || !tau || !u || !out || K < 1 || batch < 0) return ORACLE_EINVAL;
    if (make_grid(ndim, dims, &g) != ORACLE_OK) return ORACLE_EINVAL;
    double *X = (double *)malloc(sizeof(double) * (size_t)g.N);
    if (!X) return ORACLE_ENOMEM;
    int ncell_types = 1 << ndim;
    int64_t voff[8];
    for (int T = 0; T < ncell_types; ++T) voff[T] = vertex_offset(&g, T);

    for (int64_t b = 0; b < batch; ++b) {
        filtration(&g, img + b * g.N, alpha, u, X);
        double *o = out + b * K;
        for (int k = 0; k < K; ++k) o[k] = 0.0;
        int64_t idx[3];
        for (int64_t p = 0; p < g.N; ++p) {
            unravel(&g, p, idx);
            for (int S = 0; S < ncell_types; ++S) {
                if (!cell_exists(&g, idx, S)) continue;
                double xmax = X[cell_owner(X, p, S, ncell_types, voff)];
                double sign = (popcount_small(S) & 1) ? -1.0 : 1.0;
                for (int k = 0; k < K; ++k) o[k] += sign * sigmoid(lambda * ((double)tau[k] - xmax));
            }
        }
    }
    free(X);
    return ORACLE_OK;
}

/*
 * Analytic gradients of L = sum_{b,k} grad_out[b,k] * S_b(t_k).
 *   grad_tau[k]   = sum_b sum_cells grad_out[b,k] (-1)^dim lambda s (1 - s)
 *   dX[b,owner]  -= the same term, for every cell and k
 *   grad_alpha    = sum_{b,p} dX[b,p] f[b,p]
 *   grad_u[d]     = sum_{b,p} dX[b,p] x_{p,d}
 *   grad_img[b,p] = alpha dX[b,p]                      (only when grad_img is not NULL)
 * with s = sigma(lambda (t_k - max X over the cell)). grad_img_absterms (nullable) receives
 * alpha * (sum over the contributing terms of |term|), the scale of the cancellation in grad_img;
 * grad_tau_absterms (nullable) receives sum_b sum_cells |term| for each k, the same scale for
 * grad_tau.
 */
int oracle_ecc_soft_bwd(const float *img, int ndim, const int64_t *dims, int64_t batch,
                        const float *tau, int K, double lambda, double alpha, const double *u,
                        const double *grad_out, double *grad_tau, double *grad_alpha,
                        double *grad_u, double *grad_img, double *grad_img_absterms,
                        double *grad_tau_absterms)
{
    grid_t g;
    if (!img || !tau || !u || !grad_out || !grad_tau || !grad_alpha || !grad_u || K < 1 ||
        batch < 0)
        return ORACLE_EINVAL;
    if (make_grid(ndim, dims, &g) != ORACLE_OK) return ORACLE_EINVAL;
    double *X = (double *)malloc(sizeof(double) * (size_t)g.N);
    double *dX = (double *)malloc(sizeof(double) * (size_t)g.N);
    double *dXabs = (double *)malloc(sizeof(double) * (size_t)g.N);
    if (!X || !dX || !dXabs) {
        free(X);
        free(dX);
        free(dXabs);
        return ORACLE_ENOMEM;
    }
    int ncell_types = 1 << ndim;
    int64_t voff[8];
    for (int T = 0; T < ncell_types; ++T) voff[T] = vertex_offset(&g, T);
    for (int k = 0; k < K; ++k) grad_tau[k] = 0.0;
    if (grad_tau_absterms)
        for (int k = 0; k < K; ++k) grad_tau_absterms[k] = 0.0;
    *grad_alpha = 0.0;
    for (int d = 0; d < ndim; ++d) grad_u[d] = 0.0;

    for (int64_t b = 0; b < batch; ++b) {
        const float *f = img + b * g.N;
        const double *go = grad_out + b * K;
        filtration(&g, f, alpha, u, X);
        for (int64_t p = 0; p < g.N; ++p) dX[p] = dXabs[p] = 0.0;
        int64_t idx[3];
        for (int64_t p = 0; p < g.N; ++p) {
            unravel(&g, p, idx);
            for (int S = 0; S < ncell_types; ++S) {
                if (!cell_exists(&g, idx, S)) continue;
                int64_t owner = cell_owner(X, p, S, ncell_types, voff);
                double sign = (popcount_small(S) & 1) ? -1.0 : 1.0;
                for (int k = 0; k < K; ++k) {
                    double s = sigmoid(lambda * ((double)tau[k] - X[owner]));
                    double term = go[k] * sign * lambda * s * (1.0 - s);
                    grad_tau[k] += term;
                    if (grad_tau_absterms) grad_tau_absterms[k] += fabs(term);
                    dX[owner] -= term;
                    dXabs[owner] += fabs(term);
                }
            }
        }
        for (int64_t p = 0; p < g.N; ++p) {
            unravel(&g, p, idx);
            *grad_alpha += dX[p] * (double)f[p];
            for (int d = 0; d < ndim; ++d) grad_u[d] += dX[p] * axis_coord(idx[d], g.n[d]);
            if (grad_img) grad_img[b * g.N + p] = alpha * dX[p];
            if (grad_img_absterms) grad_img_absterms[b * g.N + p] = fabs(alpha) * dXabs[p];
        }
    }
    free(X);
    free(dX);
    free(dXabs);
    return ORACLE_OK;
}
