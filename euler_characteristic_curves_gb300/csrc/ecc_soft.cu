// ecc_soft.cu -- sigmoid-relaxed ("soft") ECC of 2-D images with analytic gradients (sm_103a).
//
// Paper notes "Scalable GPU-Accelerated Euler Characteristic Curves: Optimization and
// Differentiable Learning for PyTorch", "Key designs -- differentiable ECC layer (sigmoid
// relaxation)": the indicator 1[X(p) <= t] becomes sigma(lambda (t - X(p))); the single-direction
// filtration is X(p) = alpha f(p) + u . x_p; custom forward and backward kernels give analytic
// gradients for the thresholds, the direction and the scale.
//
// Per-voxel form. As in the hard path, every cell goes to its latest vertex under the order of X
// (ties: the larger linear index is later), so with c_X(p) the local Euler contribution under X,
//     S[b,k] = sum_cells (-1)^dim sigma(lambda (tau_k - max_cell X)) = sum_p c_X(p) s_pk,
//     s_pk = sigma(lambda (tau_k - X_p)).
// Only voxels with c_X(p) != 0 contribute, so a prep kernel computes X and c_X once per call and
// compacts the contributing voxels ("critical list"); the forward and backward kernels then read
// each voxel once for all K thresholds (threads own thresholds, the list is broadcast).
//
// Numerics (fp32 arithmetic unless noted):
//  * X is carried as an unevaluated sum hi + lo of two floats (alpha f and u x by exact products,
//    summed with error-free transformations); the critical-voxel order compares (hi, lo).
//  * e_pk = exp(lambda (X_p - tau_k)) = E_p F_k, E_p = 2^(l2 (X_p - m)), F_k = 2^(l2 (m - tau_k)),
//    with l2 = lambda log2(e) rounded once to fp32 and shared by both factors and m the midpoint
//    of the thresholds. Both exponents are formed in double-float and each factor is within a
//    few ulp, so e_pk is accurate to a few ulp however large the exponents (one reciprocal per
//    term). A block whose exponents exceed +-100 uses the direct form a = 2^(-l2 |tau - X|)
//    (two special-function operations per term).
//  * s is split as  s = [X <= tau] - sign r,  r = sigma(-lambda |tau - X|) = min(e, 1) / (1 + e):
//    the integer part is summed exactly, only the small part r (<= 1/2) carries rounding error.
//  * Per-thread sums use Kahan compensation; block partials go to fp64 and are reduced over the
//    tiles in a fixed order (deterministic results).
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "ecc_internal.cuh"

namespace ecc {

// ---------------------------------------------------------------------------------------------
// Workspace layout
// ---------------------------------------------------------------------------------------------

constexpr int kTileX = 64;
constexpr int kTileY = 32;
constexpr int kTileCap = kTileX * kTileY;  // entries per tile: every pixel may contribute
constexpr int kPrepThreads = 256;
constexpr int kSoftThreads = 64;           // each thread owns two thresholds per pass
constexpr int kKPerPass = 2 * kSoftThreads;
constexpr int kChunk = 256;                // entries staged in shared memory at a time
constexpr int kGroup = 8;                  // entries per backward transpose-reduce
constexpr int kTileFlagDirect = 1 << 30;   // count flag: an exponent of this tile is out of range
constexpr float kExpLimit = 100.0f;

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

bool soft_layout(int ndim, const int64_t *dims, int64_t batch, int K, SoftLayout &L)
{
    if (ndim != 2 || !dims || batch < 1 || K < 1 || K > ECC_MAX_K) return false;
    if (dims[0] < 1 || dims[1] < 1) return false;
    L.Hy = dims[0];
    L.W = dims[1];
    L.batch = batch;
    L.K = K;
    if (L.Hy * L.W >= ((int64_t)1 << 28)) return false;  // entry indices use 28 bits
    L.tiles_x = (L.W + kTileX - 1) / kTileX;
    L.tiles_y = (L.Hy + kTileY - 1) / kTileY;
    L.tiles = L.tiles_x * L.tiles_y;
    const int64_t units = batch * L.tiles;
    if (units > ((int64_t)1 << 40) / kTileCap) return false;
    size_t off = 0;
    L.off_coords = off;
    off = align256(off + sizeof(float2) * (size_t)(L.Hy + L.W));
    L.off_counts = off;
    off = align256(off + sizeof(int) * (size_t)units);
    L.off_entries = off;
    off = align256(off + sizeof(float4) * (size_t)units * kTileCap);
    L.off_part = off;
    off = align256(off + sizeof(double) * (size_t)units * (size_t)K);
    L.off_scal = off;
    off = align256(off + sizeof(double) * (size_t)units * 3);
    L.total = off;
    return true;
}

// ---------------------------------------------------------------------------------------------
// Error-free float transformations (Knuth two-sum, FMA two-product)
// ---------------------------------------------------------------------------------------------

__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e)
{
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

__device__ __forceinline__ void two_prod(float a, float b, float &p, float &e)
{
    p = __fmul_rn(a, b);
    e = fmaf(a, b, -p);
}

// X = alpha f + u0 x0 + u1 x1 as a normalised (hi, lo) pair.
__device__ __forceinline__ float2 filtration_df(float alpha, float f, float u0, float2 x0, float u1,
                                                float2 x1)
{
    float p1, e1, p2, e2, p3, e3;
    two_prod(alpha, f, p1, e1);
    two_prod(u0, x0.x, p2, e2);
    two_prod(u1, x1.x, p3, e3);
    e2 = fmaf(u0, x0.y, e2);
    e3 = fmaf(u1, x1.y, e3);
    float s1, t1, s2, t2;
    two_sum(p1, p2, s1, t1);
    two_sum(s1, p3, s2, t2);
    const float lo = __fadd_rn(__fadd_rn(t1, t2), __fadd_rn(e1, __fadd_rn(e2, e3)));
    const float hi = __fadd_rn(s2, lo);
    return make_float2(hi, __fsub_rn(lo, __fsub_rn(hi, s2)));
}

// q is earlier than p under (X, linear index): X_q < X_p, or equal with q's index smaller.
__device__ __forceinline__ bool df_lt(float2 q, float2 p)
{
    return q.x < p.x || (q.x == p.x && q.y < p.y);
}
__device__ __forceinline__ bool df_le(float2 q, float2 p)
{
    return q.x < p.x || (q.x == p.x && q.y <= p.y);
}

__device__ __forceinline__ float ex2_approx(float x)
{
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ float rcp_approx(float x)
{
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// 2^(l2 (a + b)) for a double-float a + b: the exponent is formed exactly as (p, pe) and the
// power as exp2f(p) (1 + ln2 pe). Returns the exponent's high part in `ex` for range checks.
__device__ __forceinline__ float pow2_scaled(float l2, float a, float b, float &ex)
{
    float s, e, p, pe;
    two_sum(a, b, s, e);
    two_prod(l2, s, p, pe);
    pe = fmaf(l2, e, pe);
    ex = p;
    const float base = exp2f(p);
    return fmaf(base, 0.69314718055994531f * pe, base);
}

// Midpoint of the thresholds (identical in every kernel: exact min / max, one rounding).
__device__ float tau_midpoint(const float *__restrict__ tau, int K)
{
    __shared__ float smin[32], smax[32];
    float lo = INFINITY, hi = -INFINITY;
    for (int k = threadIdx.x; k < K; k += blockDim.x) {
        const float t = __ldg(tau + k);
        lo = fminf(lo, t);
        hi = fmaxf(hi, t);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        lo = fminf(lo, __shfl_xor_sync(kFull, lo, o));
        hi = fmaxf(hi, __shfl_xor_sync(kFull, hi, o));
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) {
        smin[warp] = lo;
        smax[warp] = hi;
    }
    __syncthreads();
    lo = INFINITY;
    hi = -INFINITY;
    for (int w = 0; w < (int)(blockDim.x + 31) / 32; ++w) {
        lo = fminf(lo, smin[w]);
        hi = fmaxf(hi, smax[w]);
    }
    __syncthreads();
    return 0.5f * lo + 0.5f * hi;
}

// Entry: {E_p, X_hi, X_lo, (index << 3) | (c + 4)}.
__device__ __forceinline__ int entry_c(const float4 &en) { return (__float_as_int(en.w) & 7) - 4; }
__device__ __forceinline__ int entry_idx(const float4 &en) { return __float_as_int(en.w) >> 3; }

// ---------------------------------------------------------------------------------------------
// Kernels
// ---------------------------------------------------------------------------------------------

// Coordinates x_d(i) = (2 i - (n - 1)) / (n - 1) in fp64, stored as (hi, lo) float pairs:
// axis 0 (rows) first, then axis 1 (columns).
__global__ void soft_coords_kernel(float2 *coords, int64_t Hy, int64_t W)
{
    const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (i >= Hy + W) return;
    const int64_t n = (i < Hy) ? Hy : W;
    const int64_t j = (i < Hy) ? i : i - Hy;
    double x = 0.0;
    if (n > 1) x = (2.0 * (double)j - (double)(n - 1)) / (double)(n - 1);
    const float hi = (float)x;
    coords[i] = make_float2(hi, (float)(x - (double)hi));
}

// One block per (tile, image). Computes X on the tile plus a one-pixel halo, c_X per pixel, and
// writes the contributing pixels of the tile, in pixel order, to the tile's slot of the list.
__global__ void __launch_bounds__(kPrepThreads) soft_prep_kernel(
    const float *__restrict__ img, const float *__restrict__ alpha_p, const float *__restrict__ u_p,
    const float *__restrict__ tau, int K, float l2, const float2 *__restrict__ coords,
    int *__restrict__ counts, float4 *__restrict__ entries, int64_t Hy, int64_t W,
    int64_t tiles_x, int64_t tiles)
{
    constexpr int HX = kTileX + 2, HY = kTileY + 2;
    __shared__ float2 X[HY][HX];
    __shared__ int warp_tot[kPrepThreads / kWarp];
    __shared__ int running;

    const int64_t b = blockIdx.y;
    const int64_t tile = blockIdx.x;
    const int64_t x0 = (tile % tiles_x) * kTileX;
    const int64_t y0 = (tile / tiles_x) * kTileY;
    const float *__restrict__ f = img + b * Hy * W;
    const float alpha = __ldg(alpha_p), u0 = __ldg(u_p), u1 = __ldg(u_p + 1);
    const float2 *__restrict__ cy = coords;
    const float2 *__restrict__ cx = coords + Hy;
    const float inf = __int_as_float(0x7f800000);
    const float m = tau_midpoint(tau, K);

    for (int i = threadIdx.x; i < HX * HY; i += kPrepThreads) {
        const int iy = i / HX, ix = i % HX;
        const int64_t gy = y0 - 1 + iy, gx = x0 - 1 + ix;
        float2 v = make_float2(inf, 0.0f);  // outside the grid: never earlier
        if (gy >= 0 && gy < Hy && gx >= 0 && gx < W)
            v = filtration_df(alpha, __ldg(f + gy * W + gx), u0, __ldg(cy + gy), u1, __ldg(cx + gx));
        X[iy][ix] = v;
    }
    if (threadIdx.x == 0) running = 0;
    __syncthreads();

    const int lane = threadIdx.x & (kWarp - 1), warp = threadIdx.x >> 5;
    float4 *__restrict__ out = entries + (b * tiles + tile) * (int64_t)kTileCap;
    bool direct = false;
    for (int r = 0; r < kTileCap / kPrepThreads; ++r) {
        const int i = r * kPrepThreads + threadIdx.x;
        const int ly = i / kTileX, lx = i % kTileX;
        const int64_t gy = y0 + ly, gx = x0 + lx;
        int c = 0;
        const float2 p = X[ly + 1][lx + 1];
        if (gy < Hy && gx < W) {
            const float2 n = X[ly][lx + 1], s = X[ly + 2][lx + 1];
            const float2 w = X[ly + 1][lx], e = X[ly + 1][lx + 2];
            const bool N = df_le(n, p), Wf = df_le(w, p), S = df_lt(s, p), E = df_lt(e, p);
            const bool NW = df_le(X[ly][lx], p), NE = df_le(X[ly][lx + 2], p);
            const bool SW = df_lt(X[ly + 2][lx], p), SE = df_lt(X[ly + 2][lx + 2], p);
            c = 1 - (int)N - (int)Wf - (int)S - (int)E + (int)(N && Wf && NW) +
                (int)(N && E && NE) + (int)(S && Wf && SW) + (int)(S && E && SE);
        }
        const unsigned mask = __ballot_sync(kFull, c != 0);
        if (lane == 0) warp_tot[warp] = __popc(mask);
        __syncthreads();
        int before = running;
        for (int w2 = 0; w2 < warp; ++w2) before += warp_tot[w2];
        before += __popc(mask & ((1u << lane) - 1u));
        if (c != 0) {
            float s, e, ex;
            two_sum(p.x, -m, s, e);  // X - m, exactly, as s + (e + lo)
            const float E = pow2_scaled(l2, s, e + p.y, ex);
            direct |= !(fabsf(ex) <= kExpLimit);
            const int packed = ((int)(gy * W + gx) << 3) | (c + 4);
            out[before] = make_float4(E, p.x, p.y, __int_as_float(packed));
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            int tot = 0;
            for (int w2 = 0; w2 < kPrepThreads / kWarp; ++w2) tot += warp_tot[w2];
            running += tot;
        }
        __syncthreads();
    }
    direct = __syncthreads_or(direct);
    if (threadIdx.x == 0) counts[b * tiles + tile] = running | (direct ? kTileFlagDirect : 0);
}

// Per-thread threshold state: tau_k, F_k (factorised path) and whether its exponent is in range.
struct KState {
    float tau, F;
    bool ok;
};

__device__ __forceinline__ KState k_state(const float *__restrict__ tau, int k, int K, float l2,
                                          float m)
{
    KState s;
    s.tau = (k < K) ? __ldg(tau + k) : m;
    float ex;
    s.F = pow2_scaled(l2, m, -s.tau, ex);
    s.ok = fabsf(ex) <= kExpLimit;
    return s;
}

// r = sigma(-lambda |tau - X|) and below = [X <= tau], by the factorised or the direct form.
__device__ __forceinline__ float small_sigma_fact(float E, float F, bool &below)
{
    const float e = E * F;  // exp(lambda (X - tau))
    below = e <= 1.0f;
    const float rc = rcp_approx(1.0f + e);
    return (below ? e : 1.0f) * rc;
}
__device__ __forceinline__ float small_sigma_direct(const float4 &en, float t, float l2,
                                                    bool &below)
{
    const float d = __fsub_rn(__fsub_rn(t, en.y), en.z);  // tau - X
    below = d >= 0.0f;
    const float a = ex2_approx(-l2 * fabsf(d));
    return a * rcp_approx(1.0f + a);
}

__device__ __forceinline__ void kahan_add(float &s, float &comp, float x)
{
    const float y = x - comp;
    const float t = s + y;
    comp = (t - s) - y;
    s = t;
}

// Forward inner loop over staged entries for the thread's two thresholds.
template <bool FACT>
__device__ __forceinline__ void fwd_loop(const float4 *sh, int m_ent, const KState &s0,
                                         const KState &s1, float l2, int &w0, int &w1, float &a0,
                                         float &c0, float &a1, float &c1)
{
    for (int i = 0; i < m_ent; ++i) {
        const float4 en = sh[i];
        const int c = entry_c(en);
        const float cf = (float)c;
        bool b0, b1;
        const float r0 =
            FACT ? small_sigma_fact(en.x, s0.F, b0) : small_sigma_direct(en, s0.tau, l2, b0);
        const float r1 =
            FACT ? small_sigma_fact(en.x, s1.F, b1) : small_sigma_direct(en, s1.tau, l2, b1);
        w0 += b0 ? c : 0;
        w1 += b1 ? c : 0;
        kahan_add(a0, c0, (b0 ? -cf : cf) * r0);
        kahan_add(a1, c1, (b1 ? -cf : cf) * r1);
    }
}

// Forward: one block per (tile, image); thread t owns thresholds k = kb + t and kb + t + 64.
__global__ void __launch_bounds__(kSoftThreads) soft_fwd_kernel(
    const float *__restrict__ tau, int K, float l2, const int *__restrict__ counts,
    const float4 *__restrict__ entries, double *__restrict__ part, int64_t tiles)
{
    __shared__ float4 sh[kChunk];
    const int64_t unit = blockIdx.y * tiles + blockIdx.x;
    const int cnt = counts[unit];
    const int n = cnt & (kTileFlagDirect - 1);
    const float4 *__restrict__ list = entries + unit * (int64_t)kTileCap;
    const float m = tau_midpoint(tau, K);
    for (int kb = 0; kb < K; kb += kKPerPass) {
        const int k0 = kb + threadIdx.x, k1 = k0 + kSoftThreads;
        const KState s0 = k_state(tau, k0, K, l2, m), s1 = k_state(tau, k1, K, l2, m);
        const bool fact = __syncthreads_and(s0.ok && s1.ok && !(cnt & kTileFlagDirect));
        int w0 = 0, w1 = 0;
        float a0 = 0.f, c0 = 0.f, a1 = 0.f, c1 = 0.f;
        for (int e0 = 0; e0 < n; e0 += kChunk) {
            const int m_ent = min(kChunk, n - e0);
            __syncthreads();
            for (int i = threadIdx.x; i < m_ent; i += kSoftThreads) sh[i] = list[e0 + i];
            __syncthreads();
            if (fact)
                fwd_loop<true>(sh, m_ent, s0, s1, l2, w0, w1, a0, c0, a1, c1);
            else
                fwd_loop<false>(sh, m_ent, s0, s1, l2, w0, w1, a0, c0, a1, c1);
        }
        if (k0 < K) part[unit * K + k0] = (double)w0 + ((double)a0 - (double)c0);
        if (k1 < K) part[unit * K + k1] = (double)w1 + ((double)a1 - (double)c1);
    }
}

// out[b][k] = sum over the image's tiles of the partial sums, in tile order.
__global__ void soft_fwd_reduce_kernel(const double *__restrict__ part, float *__restrict__ out,
                                       int K, int64_t tiles, int64_t batch)
{
    const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (i >= batch * K) return;
    const int64_t b = i / K, k = i % K;
    double acc = 0.0;
    for (int64_t t = 0; t < tiles; ++t) acc += part[(b * tiles + t) * K + k];
    out[i] = (float)acc;
}

// Backward group of eight staged entries for the thread's two thresholds:
//   dtau partial[k] += c_p w_pk,   w = s (1 - s) = r (1 - r)      (times lambda g_k at the end)
//   row sum (per entry, over the warp's thresholds) of g_k w_pk   (for dX_p)
// Each lane writes its eight values to a shared 8 x 32 block; lane l sums eight entries of row
// l / 4, and two xor shuffles combine the four lanes of the row.
template <bool FACT>
__device__ __forceinline__ void bwd_group(const float4 *en8, const KState &s0, const KState &s1,
                                          float g0, float g1, float l2, float &a0, float &c0,
                                          float &a1, float &c1, float (*qw)[kWarp], int lane,
                                          float &row_sum)
{
#pragma unroll
    for (int j = 0; j < kGroup; ++j) {
        const float4 en = en8[j];
        const float cf = (float)entry_c(en);
        bool b0, b1;
        const float r0 =
            FACT ? small_sigma_fact(en.x, s0.F, b0) : small_sigma_direct(en, s0.tau, l2, b0);
        const float r1 =
            FACT ? small_sigma_fact(en.x, s1.F, b1) : small_sigma_direct(en, s1.tau, l2, b1);
        const float w0 = fmaf(-r0, r0, r0), w1 = fmaf(-r1, r1, r1);
        kahan_add(a0, c0, cf * w0);
        kahan_add(a1, c1, cf * w1);
        qw[j][lane] = fmaf(g0, w0, g1 * w1);
    }
    __syncwarp();
    const float4 *rowp = reinterpret_cast<const float4 *>(&qw[lane >> 2][(lane & 3) * 8]);
    const float4 x = rowp[0], y = rowp[1];
    float s = ((x.x + x.y) + (x.z + x.w)) + ((y.x + y.y) + (y.z + y.w));
    s += __shfl_xor_sync(kFull, s, 1);
    s += __shfl_xor_sync(kFull, s, 2);
    row_sum = s;  // the warp's partial of sum_k g_k w for entry lane / 4 of the group
    __syncwarp();
}

// Backward: one block per (tile, image); thread t owns thresholds k = kb + t and kb + t + 64.
__global__ void __launch_bounds__(kSoftThreads) soft_bwd_kernel(
    const float *__restrict__ img, const float *__restrict__ tau, int K, float lambda, float l2,
    const float *__restrict__ alpha_p, const float *__restrict__ grad_out,
    const int *__restrict__ counts, const float4 *__restrict__ entries,
    const float2 *__restrict__ coords, double *__restrict__ part, double *__restrict__ scal,
    float *__restrict__ grad_img, int64_t Hy, int64_t W, int64_t tiles)
{
    constexpr int NW = kSoftThreads / kWarp;
    __shared__ __align__(16) float4 sh[kChunk];
    __shared__ __align__(16) float qbuf[NW][kGroup][kWarp];
    __shared__ float red[NW][kChunk];
    __shared__ float dxs[kTileCap];
    __shared__ double scal_red[NW][3];

    const int64_t b = blockIdx.y;
    const int64_t unit = b * tiles + blockIdx.x;
    const int cnt = counts[unit];
    const int n = cnt & (kTileFlagDirect - 1);
    const float4 *__restrict__ list = entries + unit * (int64_t)kTileCap;
    const int lane = threadIdx.x & (kWarp - 1), warp = threadIdx.x >> 5;
    const float m = tau_midpoint(tau, K);
    for (int i = threadIdx.x; i < n; i += kSoftThreads) dxs[i] = 0.0f;

    for (int kb = 0; kb < K; kb += kKPerPass) {
        const int k0 = kb + threadIdx.x, k1 = k0 + kSoftThreads;
        const KState s0 = k_state(tau, k0, K, l2, m), s1 = k_state(tau, k1, K, l2, m);
        const float g0 = (k0 < K) ? __ldg(grad_out + b * K + k0) : 0.0f;
        const float g1 = (k1 < K) ? __ldg(grad_out + b * K + k1) : 0.0f;
        const bool fact = __syncthreads_and(s0.ok && s1.ok && !(cnt & kTileFlagDirect));
        float a0 = 0.f, c0 = 0.f, a1 = 0.f, c1 = 0.f;
        for (int e0 = 0; e0 < n; e0 += kChunk) {
            const int m_ent = min(kChunk, n - e0);
            __syncthreads();
            // stage the chunk; pad the last group with c = 0 entries
            for (int i = threadIdx.x; i < kChunk; i += kSoftThreads)
                sh[i] = (i < m_ent) ? list[e0 + i] : make_float4(0.f, 0.f, 0.f, __int_as_float(4));
            __syncthreads();
            for (int g = 0; g * kGroup < m_ent; ++g) {
                float rs;
                if (fact)
                    bwd_group<true>(sh + g * kGroup, s0, s1, g0, g1, l2, a0, c0, a1, c1,
                                    qbuf[warp], lane, rs);
                else
                    bwd_group<false>(sh + g * kGroup, s0, s1, g0, g1, l2, a0, c0, a1, c1,
                                     qbuf[warp], lane, rs);
                if ((lane & 3) == 0) red[warp][g * kGroup + (lane >> 2)] = rs;
            }
            __syncthreads();
            for (int i = threadIdx.x; i < m_ent; i += kSoftThreads) {
                float q = 0.0f;
#pragma unroll
                for (int w2 = 0; w2 < NW; ++w2) q += red[w2][i];
                dxs[e0 + i] += q;
            }
        }
        if (k0 < K) part[unit * K + k0] = (double)lambda * (double)g0 * ((double)a0 - (double)c0);
        if (k1 < K) part[unit * K + k1] = (double)lambda * (double)g1 * ((double)a1 - (double)c1);
    }
    __syncthreads();

    // per-voxel gradient: dX = -lambda c sum_k g w; grad_img = alpha dX; dalpha, du partials
    const float alpha = __ldg(alpha_p);
    const float *__restrict__ f = img + b * Hy * W;
    float sa = 0.f, ca = 0.f, sy = 0.f, cy = 0.f, sx = 0.f, cx = 0.f;
    for (int i = threadIdx.x; i < n; i += kSoftThreads) {
        const float4 en = list[i];
        const int idx = entry_idx(en);
        const float dX = -lambda * (float)entry_c(en) * dxs[i];
        if (grad_img) grad_img[b * Hy * W + idx] = alpha * dX;
        const int64_t iy = idx / W, ix = idx % W;
        const float2 xy = __ldg(coords + iy), xx = __ldg(coords + Hy + ix);
        kahan_add(sa, ca, dX * __ldg(f + idx));
        kahan_add(sy, cy, dX * (xy.x + xy.y));
        kahan_add(sx, cx, dX * (xx.x + xx.y));
    }
    double v[3] = {(double)sa - (double)ca, (double)sy - (double)cy, (double)sx - (double)cx};
#pragma unroll
    for (int j = 0; j < 3; ++j) {
#pragma unroll
        for (int o = kWarp / 2; o > 0; o >>= 1) v[j] += __shfl_xor_sync(kFull, v[j], o);
    }
    if (lane == 0) {
        scal_red[warp][0] = v[0];
        scal_red[warp][1] = v[1];
        scal_red[warp][2] = v[2];
    }
    __syncthreads();
    if (threadIdx.x < 3) {
        double acc = 0.0;
        for (int w2 = 0; w2 < NW; ++w2) acc += scal_red[w2][threadIdx.x];
        scal[unit * 3 + threadIdx.x] = acc;
    }
}

// grad_tau[k] = sum over (image, tile) of the partials; grad_alpha, grad_u likewise. One block per
// output: threads take strided partials in fp64, then a fixed-order tree (deterministic).
constexpr int kReduceThreads = 256;

__global__ void __launch_bounds__(kReduceThreads) soft_bwd_reduce_kernel(
    const double *__restrict__ part, const double *__restrict__ scal, int K, int64_t units,
    float *__restrict__ grad_tau, float *__restrict__ grad_alpha, float *__restrict__ grad_u)
{
    __shared__ double red[kReduceThreads];
    const int o = blockIdx.x;  // 0..K-1: grad_tau[o]; K: grad_alpha; K+1..: grad_u
    double acc = 0.0;
    if (o < K) {
        for (int64_t u = threadIdx.x; u < units; u += kReduceThreads) acc += part[u * K + o];
    } else {
        const int j = o - K;
        for (int64_t u = threadIdx.x; u < units; u += kReduceThreads) acc += scal[u * 3 + j];
    }
    red[threadIdx.x] = acc;
    __syncthreads();
    for (int s = kReduceThreads / 2; s > 0; s >>= 1) {
        if (threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        const float v = (float)red[0];
        if (o < K)
            grad_tau[o] = v;
        else if (o == K)
            grad_alpha[0] = v;
        else
            grad_u[o - K - 1] = v;
    }
}

// ---------------------------------------------------------------------------------------------
// Host launchers (called from the C ABI after validation)
// ---------------------------------------------------------------------------------------------

static inline float lambda_log2e(float lambda)
{
    return (float)((double)lambda * 1.4426950408889634);
}

cudaError_t soft_run_fwd(const SoftLayout &L, const float *img, const float *tau, float lambda,
                         const float *alpha, const float *u, float *out, void *ws, cudaStream_t s)
{
    char *base = static_cast<char *>(ws);
    float2 *coords = reinterpret_cast<float2 *>(base + L.off_coords);
    int *counts = reinterpret_cast<int *>(base + L.off_counts);
    float4 *entries = reinterpret_cast<float4 *>(base + L.off_entries);
    double *part = reinterpret_cast<double *>(base + L.off_part);
    const float l2 = lambda_log2e(lambda);
    const int64_t ncoord = L.Hy + L.W;
    soft_coords_kernel<<<(unsigned)((ncoord + 255) / 256), 256, 0, s>>>(coords, L.Hy, L.W);
    dim3 grid((unsigned)L.tiles, (unsigned)L.batch);
    soft_prep_kernel<<<grid, kPrepThreads, 0, s>>>(img, alpha, u, tau, L.K, l2, coords, counts,
                                                   entries, L.Hy, L.W, L.tiles_x, L.tiles);
    soft_fwd_kernel<<<grid, kSoftThreads, 0, s>>>(tau, L.K, l2, counts, entries, part, L.tiles);
    const int64_t nout = L.batch * L.K;
    soft_fwd_reduce_kernel<<<(unsigned)((nout + 255) / 256), 256, 0, s>>>(part, out, L.K, L.tiles,
                                                                          L.batch);
    return cudaGetLastError();
}

cudaError_t soft_run_bwd(const SoftLayout &L, const float *img, const float *tau, float lambda,
                         const float *alpha, const float *grad_out, float *grad_tau,
                         float *grad_alpha, float *grad_u, float *grad_img, void *ws,
                         cudaStream_t s)
{
    char *base = static_cast<char *>(ws);
    const float2 *coords = reinterpret_cast<const float2 *>(base + L.off_coords);
    const int *counts = reinterpret_cast<const int *>(base + L.off_counts);
    const float4 *entries = reinterpret_cast<const float4 *>(base + L.off_entries);
    double *part = reinterpret_cast<double *>(base + L.off_part);
    double *scal = reinterpret_cast<double *>(base + L.off_scal);
    if (grad_img) {
        cudaError_t e =
            cudaMemsetAsync(grad_img, 0, sizeof(float) * (size_t)(L.batch * L.Hy * L.W), s);
        if (e != cudaSuccess) return e;
    }
    dim3 grid((unsigned)L.tiles, (unsigned)L.batch);
    soft_bwd_kernel<<<grid, kSoftThreads, 0, s>>>(img, tau, L.K, lambda, lambda_log2e(lambda),
                                                  alpha, grad_out, counts, entries, coords, part,
                                                  scal, grad_img, L.Hy, L.W, L.tiles);
    const int64_t units = L.batch * L.tiles;
    soft_bwd_reduce_kernel<<<(unsigned)(L.K + 3), kReduceThreads, 0, s>>>(
        part, scal, L.K, units, grad_tau, grad_alpha, grad_u);
    return cudaGetLastError();
}

}  // namespace ecc
