// ecc_soft.cu -- sigmoid-relaxed ("soft") ECC of 2-D images and 3-D volumes with analytic
// gradients (sm_103a).
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
// each voxel once for all K thresholds (threads own thresholds, the list is broadcast). In 2-D,
// c_X reads the 8 neighbours; in 3-D the 26 neighbours, with c_X = sum over the 27 cells that
// contain p and whose other vertices are all earlier of (-1)^dim (range [-5, 7]).
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

#include <algorithm>

#include "ecc_internal.cuh"

namespace ecc {

__device__ unsigned g_soft_error;  // device error word of the soft kernels (DeviceErrorBit)

cudaError_t soft_error_word(unsigned **p)
{
    return cudaGetSymbolAddress(reinterpret_cast<void **>(p), g_soft_error);
}

// ---------------------------------------------------------------------------------------------
// Workspace layout
// ---------------------------------------------------------------------------------------------

// Tiles: 64 x 32 pixels (2-D), 32 x 8 x 8 voxels (3-D); both 2048 = kTileCap cells.
template <int NDIM> struct SoftTile;
template <> struct SoftTile<2> {
    static constexpr int X = 64, Y = 32, Z = 1;
};
template <> struct SoftTile<3> {
    static constexpr int X = 32, Y = 8, Z = 8;
};
constexpr int kTileCap = 2048;  // entries per tile: every voxel may contribute
static_assert(SoftTile<2>::X * SoftTile<2>::Y == kTileCap, "2-D tile size");
static_assert(SoftTile<3>::X * SoftTile<3>::Y * SoftTile<3>::Z == kTileCap, "3-D tile size");
constexpr int kPrepThreads = 256;
constexpr int64_t kPrepBlocks = 4096;      // prep grid size aimed at when directions are grouped
constexpr int kSoftThreads = 64;           // two warps per block
constexpr int kTailBatch = 4;              // backward per-voxel loop: entries in flight per thread
constexpr int kChunk = 256;                // entries staged in shared memory at a time
// The backward kernel stages half as many, so that its shared memory (and registers) let a
// full wave of blocks be resident on a 64-image batch of 256^2 images.
constexpr int kBwdChunk = 128;
constexpr int kGroup = 8;                  // entries per backward transpose-reduce
constexpr int kTileFlagDirect = 1 << 30;   // count flag: an exponent of this tile is out of range
constexpr float kExpLimit = 100.0f;
constexpr int kScal = 4;                   // backward scalar partials per tile: alpha, u_0..u_2

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

bool soft_layout(int ndim, const int64_t *dims, int64_t batch, int K, int ndirs, SoftLayout &L)
{
    if ((ndim != 2 && ndim != 3) || !dims || batch < 1 || K < 1 || K > ECC_MAX_K) return false;
    for (int d = 0; d < ndim; ++d)
        if (dims[d] < 1 || dims[d] > ECC_MAX_EXTENT) return false;
    if (ndirs < 1 || ndirs > ECC_MAX_DIRS) return false;
    if (batch * ndirs > 65535) return false;  // (image, direction) pairs run along gridDim.y
    L.ndirs = ndirs;
    L.ndim = ndim;
    L.D = ndim == 3 ? dims[0] : 1;
    L.Hy = dims[ndim - 2];
    L.W = dims[ndim - 1];
    L.batch = batch;
    L.K = K;
    if (L.D * L.Hy > ((int64_t)1 << 40) / L.W) return false;
    const int tx = ndim == 3 ? SoftTile<3>::X : SoftTile<2>::X;
    const int ty = ndim == 3 ? SoftTile<3>::Y : SoftTile<2>::Y;
    const int tz = ndim == 3 ? SoftTile<3>::Z : SoftTile<2>::Z;
    L.tiles_x = (L.W + tx - 1) / tx;
    L.tiles_y = (L.Hy + ty - 1) / ty;
    L.tiles_z = (L.D + tz - 1) / tz;
    L.tiles = L.tiles_x * L.tiles_y * L.tiles_z;
    if (L.tiles >= ((int64_t)1 << 31)) return false;  // tiles run along gridDim.x
    const int64_t units = batch * ndirs * L.tiles;
    if (units > ((int64_t)1 << 40) / kTileCap) return false;
    const int64_t ncoord = (ndim == 3 ? L.D : 0) + L.Hy + L.W;
    size_t off = 0;
    L.off_coords = off;
    off = align256(off + sizeof(float2) * (size_t)ncoord);
    L.off_counts = off;
    off = align256(off + sizeof(int) * (size_t)units);
    L.off_entries = off;
    off = align256(off + sizeof(float4) * (size_t)units * kTileCap);
    L.off_part = off;
    off = align256(off + sizeof(double) * (size_t)units * (size_t)K);
    L.off_scal = off;
    off = align256(off + sizeof(double) * (size_t)units * kScal);
    L.total = off;
    return true;
}

// Geometry handed to the kernels. Coordinate tables: axis 0 first (the z axis of a volume, the
// row axis of an image), then the following axes; nz = D for volumes and 0 for images.
struct SoftGeom {
    int64_t D, Hy, W, nz;
    int64_t tiles_x, tiles_y, tiles;
};

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

// X = alpha f + u0 x0 + u1 x1 + u2 x2 as a normalised (hi, lo) pair.
__device__ __forceinline__ float2 filtration_df3(float alpha, float f, float u0, float2 x0, float u1,
                                                 float2 x1, float u2, float2 x2)
{
    float p1, e1, p2, e2, p3, e3, p4, e4;
    two_prod(alpha, f, p1, e1);
    two_prod(u0, x0.x, p2, e2);
    two_prod(u1, x1.x, p3, e3);
    two_prod(u2, x2.x, p4, e4);
    e2 = fmaf(u0, x0.y, e2);
    e3 = fmaf(u1, x1.y, e3);
    e4 = fmaf(u2, x2.y, e4);
    float s1, t1, s2, t2, s3, t3;
    two_sum(p1, p2, s1, t1);
    two_sum(s1, p3, s2, t2);
    two_sum(s2, p4, s3, t3);
    const float lo = __fadd_rn(__fadd_rn(__fadd_rn(t1, t2), t3),
                               __fadd_rn(e1, __fadd_rn(__fadd_rn(e2, e3), e4)));
    const float hi = __fadd_rn(s3, lo);
    return make_float2(hi, __fsub_rn(lo, __fsub_rn(hi, s3)));
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

// Entry: {E_p, X_hi, X_lo, (index in the tile << 4) | (c + 8)}, c in [-8, 7].
constexpr int kPadWord = 8;  // c = 0 at index 0: a padding entry that contributes nothing
// c as a float without a conversion instruction: 2^23 + (c + 8) is exact in fp32.
__device__ __forceinline__ float entry_cf(const float4 &en)
{
    return __int_as_float(0x4B000000 | (__float_as_int(en.w) & 15)) - 8388616.0f;
}
__device__ __forceinline__ int entry_loc(const float4 &en) { return __float_as_int(en.w) >> 4; }

// The 3-D local contribution by the slice fold, in bits. The cells of the V-construction that
// contain a voxel p split into those of its plane z and those reaching plane z - 1 or z + 1; a
// cell reaching z - 1 is an in-plane cell sigma times [z - 1, z], of sign -(-1)^dim(sigma), and
// counts when p is the latest vertex of sigma in plane z, the voxel straight below is earlier,
// and so are sigma's vertices in plane z - 1. With m_z, m_b, m_a the 8 neighbour bits of planes
// z, z - 1, z + 1 and e_b, e_a the voxels below and above,
//     c3 = T2[m_z] - e_b T2[m_z & m_b] - e_a T2[m_z & m_a],
// T2[m] the signed count of the in-plane cells around a centre whose other vertices are in m
// (checked against the 27 cells for every mask in tests/test_kernel_algebra.py).
// Neighbour bit order in a plane: (dy, dx) = (-1,-1), (-1,0), (-1,1), (0,-1), (0,1), (1,-1),
// (1,0), (1,1).
struct C2Table {
    int8_t v[256];
};
__host__ __device__ constexpr int plane_bit(int dy, int dx)
{
    return (dy + 1) * 3 + (dx + 1) < 4 ? (dy + 1) * 3 + (dx + 1) : (dy + 1) * 3 + (dx + 1) - 1;
}
__host__ __device__ constexpr C2Table make_c2_table()
{
    C2Table t{};
    for (int m = 0; m < 256; ++m) {
        int v = 0;
        for (int sy = -1; sy <= 1; ++sy)
            for (int sx = -1; sx <= 1; ++sx) {
                int need = 0;
                for (int a = 0; a <= (sy != 0); ++a)
                    for (int b = 0; b <= (sx != 0); ++b)
                        if (a * sy != 0 || b * sx != 0) need |= 1 << plane_bit(a * sy, b * sx);
                if ((m & need) == need) v += ((sy != 0) + (sx != 0)) & 1 ? -1 : 1;
            }
        t.v[m] = (int8_t)v;
    }
    return t;
}

__constant__ C2Table kC2Table = make_c2_table();

// ---------------------------------------------------------------------------------------------
// Kernels
// ---------------------------------------------------------------------------------------------

// Coordinates x_d(i) = (2 i - (n - 1)) / (n - 1) in fp64, stored as (hi, lo) float pairs, one
// table per axis, axis 0 first: [nz z-coordinates][Hy row coordinates][W column coordinates].
__global__ void soft_coords_kernel(float2 *coords, int64_t nz, int64_t Hy, int64_t W)
{
    const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (i >= nz + Hy + W) return;
    int64_t n, j;
    if (i < nz) {
        n = nz;
        j = i;
    } else if (i < nz + Hy) {
        n = Hy;
        j = i - nz;
    } else {
        n = W;
        j = i - nz - Hy;
    }
    double x = 0.0;
    if (n > 1) x = (2.0 * (double)j - (double)(n - 1)) / (double)(n - 1);
    const float hi = (float)x;
    coords[i] = make_float2(hi, (float)(x - (double)hi));
}

// Local Euler contribution c_X(p) of a 2-D pixel from its 3 x 3 neighbourhood in X (row pitch HX,
// `c` points at p). Earlier = `<=` for the neighbours with a smaller linear index, `<` otherwise.
template <int HX>
__device__ __forceinline__ int local_c2(const float2 *c)
{
    const float2 p = c[0];
    const bool N = df_le(c[-HX], p), Wf = df_le(c[-1], p), S = df_lt(c[HX], p), E = df_lt(c[1], p);
    const bool NW = df_le(c[-HX - 1], p), NE = df_le(c[-HX + 1], p);
    const bool SW = df_lt(c[HX - 1], p), SE = df_lt(c[HX + 1], p);
    return 1 - (int)N - (int)Wf - (int)S - (int)E + (int)(N && Wf && NW) + (int)(N && E && NE) +
           (int)(S && Wf && SW) + (int)(S && E && SE);
}

// Local Euler contribution of a 3-D voxel from its 3 x 3 x 3 neighbourhood (row pitch HX, plane
// pitch HP) by the bit slice fold above; c2tab is the table T2 in shared memory. Neighbours with
// a smaller linear index are earlier when `<=`, those after it when `<`.
template <int HX, int HP>
__device__ __forceinline__ int local_c3(const float2 *c, const int8_t *c2tab)
{
    const float2 p = c[0];
    uint32_t mb = 0, mz = 0, ma = 0;  // neighbour bits of planes z - 1, z, z + 1
#pragma unroll
    for (int dy = -1; dy <= 1; ++dy)
#pragma unroll
        for (int dx = -1; dx <= 1; ++dx) {
            if (dy == 0 && dx == 0) continue;
            const int bit = plane_bit(dy, dx);
            const int off = dy * HX + dx;
            mb |= (uint32_t)df_le(c[off - HP], p) << bit;  // plane z - 1: smaller index
            mz |= (uint32_t)(off < 0 ? df_le(c[off], p) : df_lt(c[off], p)) << bit;
            ma |= (uint32_t)df_lt(c[off + HP], p) << bit;  // plane z + 1: larger index
        }
    const bool eb = df_le(c[-HP], p), ea = df_lt(c[HP], p);
    int v = c2tab[mz];
    if (eb) v -= c2tab[mz & mb];
    if (ea) v -= c2tab[mz & ma];
    return v;
}

// Position (iz, iy, ix) of element i of a halo box with rows of HX, planes of HP = HX HY
// elements, advanced by kPrepThreads elements at a time (one carry at most per axis).
template <int HX, int HY, int HP>
struct HaloPos {
    static constexpr int dX = kPrepThreads % HX, dY = (kPrepThreads / HX) % HY,
                         dZ = kPrepThreads / HP;
    int ix, iy, iz;
    __device__ __forceinline__ explicit HaloPos(int i) : ix(i % HX), iy((i / HX) % HY), iz(i / HP)
    {
    }
    __device__ __forceinline__ void advance()
    {
        ix += dX;
        const int cx = ix >= HX;
        ix -= cx ? HX : 0;
        iy += dY + cx;
        const int cy = iy >= HY;
        iy -= cy ? HY : 0;
        iz += dZ + cy;
    }
};

// One block per (tile, image). Reads f on the tile plus a one-voxel halo once, then for each
// direction u_j computes X_j = alpha f + u_j . x there, c_X per voxel, and writes the contributing
// voxels of the tile, in the tile's own raster order, to the slot of unit (image, direction,
// tile).
template <int NDIM>
__global__ void __launch_bounds__(kPrepThreads) soft_prep_kernel(
    const float *__restrict__ img, const float *__restrict__ alpha_p, const float *__restrict__ u_p,
    int ndirs, int dirs_per_block, const float *__restrict__ tau, int K, float l2,
    const float2 *__restrict__ coords, int *__restrict__ counts, float4 *__restrict__ entries,
    SoftGeom g)
{
    using T = SoftTile<NDIM>;
    constexpr int HX = T::X + 2, HY = T::Y + 2, HZ = NDIM == 3 ? T::Z + 2 : 1;
    constexpr int HP = HX * HY;
    constexpr int ZO = NDIM == 3 ? 1 : 0;  // halo offset along z
    __shared__ float Fv[HZ * HP];  // f on the tile and its halo; NaN outside the grid
    __shared__ float2 X[HZ * HP];
    __shared__ float2 ctile[HX + HY + HZ];  // coordinates of the tile's columns, rows, planes
    constexpr int kRounds = kTileCap / kPrepThreads;  // pixels per thread
    constexpr int kPrepWarps = kPrepThreads / kWarp;
    static_assert(kRounds * kPrepWarps == 2 * kWarp, "one warp scans the (round, warp) counts");
    __shared__ int wcount[kRounds * kPrepWarps];  // contributing pixels per (round, warp)
    __shared__ int running;                       // the tile's list length
    __shared__ int8_t c2tab[256];                 // T2 of the 3-D slice fold

    // blockIdx.y = b groups + group: the block's directions are one group of dirs_per_block
    const int groups = (ndirs + dirs_per_block - 1) / dirs_per_block;
    const int64_t b = blockIdx.y / groups;
    const int jbeg = (int)(blockIdx.y % groups) * dirs_per_block;
    const int jend = min(jbeg + dirs_per_block, ndirs);
    const int64_t tile = blockIdx.x;
    const int64_t x0 = (tile % g.tiles_x) * T::X;
    const int64_t y0 = ((tile / g.tiles_x) % g.tiles_y) * T::Y;
    const int64_t z0 = (tile / (g.tiles_x * g.tiles_y)) * T::Z;
    const float *__restrict__ f = img + b * g.D * g.Hy * g.W;
    const float alpha = __ldg(alpha_p);
    const float2 *__restrict__ cz = coords;
    const float2 *__restrict__ cy = coords + g.nz;
    const float2 *__restrict__ cx = coords + g.nz + g.Hy;
    const float inf = __int_as_float(0x7f800000);
    const float m = tau_midpoint(tau, K);
    const int lane = threadIdx.x & (kWarp - 1), warp = threadIdx.x >> 5;

    if (NDIM == 3)
        for (int i = threadIdx.x; i < 256; i += kPrepThreads) c2tab[i] = kC2Table.v[i];
    // the tile's coordinates (its halo included) once, then f on the tile and its halo
    for (int i = threadIdx.x; i < HX + HY + HZ; i += kPrepThreads) {
        float2 cv = make_float2(0.0f, 0.0f);  // outside the grid: unused (f reads as NaN there)
        if (i < HX) {
            const int64_t gx = x0 - 1 + i;
            if (gx >= 0 && gx < g.W) cv = __ldg(cx + gx);
        } else if (i < HX + HY) {
            const int64_t gy = y0 - 1 + (i - HX);
            if (gy >= 0 && gy < g.Hy) cv = __ldg(cy + gy);
        } else if (NDIM == 3) {
            const int64_t gz = z0 - ZO + (i - HX - HY);
            if (gz >= 0 && gz < g.D) cv = __ldg(cz + gz);
        }
        ctile[i] = cv;
    }
    // all of a thread's loads are issued before any of them is stored, so their latencies overlap
    // (one load per iteration, stored before the next, waited on each in turn). The element
    // i = thread + r kPrepThreads of the halo box advances by kPrepThreads each round, its
    // position (iz, iy, ix) by carries instead of divisions; grid coordinates fit in 32 bits
    // (extents are at most 2^30) and one unsigned compare tests both ends of an axis.
    constexpr int kLoads = (HZ * HP + kPrepThreads - 1) / kPrepThreads;
    const int tx0 = (int)x0 - 1, ty0 = (int)y0 - 1, tz0 = (int)z0 - ZO;
    const unsigned uW = (unsigned)g.W, uH = (unsigned)g.Hy, uD = (unsigned)g.D;
    float fl[kLoads];
    {
        HaloPos<HX, HY, HP> hp(threadIdx.x);
#pragma unroll
        for (int r = 0; r < kLoads; ++r) {
            const int i = threadIdx.x + r * kPrepThreads;
            const int gz = tz0 + hp.iz, gy = ty0 + hp.iy, gx = tx0 + hp.ix;
            fl[r] = qnan();
            if (i < HZ * HP && (unsigned)gz < uD && (unsigned)gy < uH && (unsigned)gx < uW)
                fl[r] = __ldg(f + ((int64_t)gz * g.Hy + gy) * g.W + gx);
            hp.advance();
        }
    }
#pragma unroll
    for (int r = 0; r < kLoads; ++r) {
        const int i = threadIdx.x + r * kPrepThreads;
        if (i < HZ * HP) Fv[i] = fl[r];
    }

    for (int j = jbeg; j < jend; ++j) {
        const float *u = u_p + j * NDIM;
        const float u0 = __ldg(u), u1 = __ldg(u + 1), u2 = NDIM == 3 ? __ldg(u + 2) : 0.0f;
        __syncthreads();  // Fv is complete; the previous direction is done with X and running
        HaloPos<HX, HY, HP> hp(threadIdx.x);
        for (int i = threadIdx.x; i < HZ * HP; i += kPrepThreads, hp.advance()) {
            const int iz = hp.iz, iy = hp.iy, ix = hp.ix;
            const float fv = Fv[i];
            float2 v = make_float2(inf, 0.0f);  // outside the grid: never earlier
            if (fv == fv) {  // inside the grid (NaN marks outside; inputs are finite)
                if (NDIM == 3)
                    v = filtration_df3(alpha, fv, u0, ctile[HX + HY + iz], u1, ctile[HX + iy],
                                       u2, ctile[ix]);
                else
                    v = filtration_df(alpha, fv, u0, ctile[HX + iy], u1, ctile[ix]);
            }
            X[i] = v;
        }
        __syncthreads();

        const int64_t unit = ((int64_t)b * ndirs + j) * g.tiles + tile;
        float4 *__restrict__ out = entries + unit * (int64_t)kTileCap;
        // Pixel i = r kPrepThreads + thread (round r). A pixel's slot in the list is the number of
        // contributing pixels before it in raster order: those of earlier rounds, of earlier
        // warps in its round and of earlier lanes in its warp. The (round, warp) counts are
        // scanned once for the whole tile.
        int cr[kRounds];
        unsigned bal[kRounds];
#pragma unroll
        for (int r = 0; r < kRounds; ++r) {
            const int i = r * kPrepThreads + threadIdx.x;
            const int lx = i % T::X, ly = (i / T::X) % T::Y, lz = i / (T::X * T::Y);
            const float2 *cp = &X[(lz + ZO) * HP + (ly + 1) * HX + lx + 1];
            int c = 0;
            if (tz0 + ZO + lz < (int)uD && ty0 + 1 + ly < (int)uH && tx0 + 1 + lx < (int)uW)
                c = NDIM == 3 ? local_c3<HX, HP>(cp, c2tab) : local_c2<HX>(cp);
            cr[r] = c;
            bal[r] = __ballot_sync(kFull, c != 0);
            if (lane == 0) wcount[r * kPrepWarps + warp] = __popc(bal[r]);
        }
        __syncthreads();
        if (warp == 0) {  // exclusive scan of the 64 counts in (round, warp) order, two per lane
            const int a = wcount[2 * lane], b2 = wcount[2 * lane + 1];
            int incl = a + b2;
#pragma unroll
            for (int o = 1; o < kWarp; o <<= 1) {
                const int t = __shfl_up_sync(kFull, incl, o);
                if (lane >= o) incl += t;
            }
            const int excl = incl - (a + b2);
            __syncwarp();
            wcount[2 * lane] = excl;
            wcount[2 * lane + 1] = excl + a;
            if (lane == kWarp - 1) running = incl;
        }
        __syncthreads();
        bool direct = false;
#pragma unroll
        for (int r = 0; r < kRounds; ++r) {
            if (cr[r] != 0) {
                const int i = r * kPrepThreads + threadIdx.x;
                const int lx = i % T::X, ly = (i / T::X) % T::Y, lz = i / (T::X * T::Y);
                const float2 p = X[(lz + ZO) * HP + (ly + 1) * HX + lx + 1];
                const int slot =
                    wcount[r * kPrepWarps + warp] + __popc(bal[r] & ((1u << lane) - 1u));
                float s, e, ex;
                two_sum(p.x, -m, s, e);  // X - m, exactly, as s + (e + lo)
                const float E = pow2_scaled(l2, s, e + p.y, ex);
                direct |= !(fabsf(ex) <= kExpLimit);
                const int packed = (i << 4) | (cr[r] + 8);
                if (bounds_ok(&g_soft_error, slot >= 0 && slot < kTileCap, kErrSoftSlot))
                    out[slot] = make_float4(E, p.x, p.y, __int_as_float(packed));
            }
        }
        direct = __syncthreads_or(direct);
        if (threadIdx.x == 0) counts[unit] = running | (direct ? kTileFlagDirect : 0);
    }
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

// r = sigma(-lambda |tau - X|) and below = [X <= tau] by the direct form (the factorised form,
// for both thresholds at once, is written out in the packed loops below).
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
// Kahan step for the term a b, the product entering through one fused multiply-add.
__device__ __forceinline__ void kahan_fma(float &s, float &comp, float a, float b)
{
    const float y = fmaf(a, b, -comp);
    const float t = s + y;
    comp = (t - s) - y;
    s = t;
}

// Packed fp32 pairs: a thread's two thresholds in one 64-bit register pair, so that one
// instruction does both. Each element is rounded exactly as the scalar operation would round it,
// so the packed loops below give the same bits as their scalar forms.
typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 pk2(float a, float b)
{
    f32x2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void upk2(f32x2 r, float &a, float &b)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b)
{
    f32x2 r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f32x2 sub2(f32x2 a, f32x2 b)
{
    f32x2 r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b)
{
    f32x2 r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c)
{
    f32x2 r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

// Kahan step for both thresholds with the compensation carried negated (nc = -comp), which
// makes every step one packed add, subtract or fused multiply-add; same bits as kahan_fma.
__device__ __forceinline__ void kahan_fma2(f32x2 &s, f32x2 &nc, f32x2 a, f32x2 b)
{
    const f32x2 y = fma2(a, b, nc);
    const f32x2 t = add2(s, y);
    nc = sub2(y, sub2(t, s));
    s = t;
}

// Threshold passes of the forward and backward kernels: lane l of a warp owns thresholds
// k = kb + l + 32 j, j = 0 .. 3 (two packed pairs: j = 0, 1 and j = 2, 3), so one warp covers
// a pass of kWarpK thresholds and reads each staged entry once for four of them; the block's
// warps share the entries of a tile out between them.
constexpr int kLaneK = 4;
constexpr int kWarpK = kLaneK * kWarp;  // 128
constexpr int kSoftWarps = kSoftThreads / kWarp;

struct Lane4 {
    KState s[kLaneK];
    bool ok;  // all four in the factorised range
};
__device__ __forceinline__ Lane4 lane_thresholds(const float *__restrict__ tau, int kb, int lane,
                                                 int K, float l2, float m)
{
    Lane4 t;
    t.ok = true;
#pragma unroll
    for (int j = 0; j < kLaneK; ++j) {
        t.s[j] = k_state(tau, kb + lane + kWarp * j, K, l2, m);
        t.ok = t.ok && t.s[j].ok;
    }
    return t;
}

// Sums of the forward for a lane's four thresholds: integer parts w, Kahan sums a (compensation
// carried negated in nc) of the small parts; pairs (j = 0, 1) and (j = 2, 3).
struct FwdAcc {
    f32x2 w[2], a[2], nc[2];
};

// Forward over the staged entries i = first, first + step, ... < m_ent, factorised form (the same
// per-term arithmetic as the scalar form: e = E F_k, r = min(e, 1) / (1 + e), w += [e <= 1] c,
// Kahan over -+c r). The entries are staged as the pairs (E, E), (c, c).
// The below-threshold flag enters as a float b (1.0 / 0.0, one set instruction on the ALU pipe)
// through packed fused multiply-adds on the FMA pipe, w += b c and the small part's coefficient
// c (1 - 2 b) = fma(b, -2 c, c), instead of a compare and two selects on the ALU pipe, which
// this loop saturates. Each value is exact (c, 2c and their sums are small integers), so the
// sums are the same bits as the select form.
__device__ __forceinline__ void fwd_loop4_packed(const float4 *sh, int first, int step,
                                                 int m_ent, const f32x2 *F, FwdAcc &acc)
{
    const f32x2 minus2 = pk2(-2.0f, -2.0f);
#pragma unroll 3
    for (int i = first; i < m_ent; i += step) {
        const ulonglong2 en = *reinterpret_cast<const ulonglong2 *>(sh + i);  // (E, E), (c, c)
        const f32x2 E = en.x, c2 = en.y, m2c2 = mul2(c2, minus2);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float e0, e1, d0, d1;
            const f32x2 e = mul2(E, F[h]);
            upk2(e, e0, e1);
            upk2(add2(e, pk2(1.0f, 1.0f)), d0, d1);
            const f32x2 b = pk2(e0 <= 1.0f ? 1.0f : 0.0f, e1 <= 1.0f ? 1.0f : 0.0f);
            const f32x2 r =
                mul2(pk2(fminf(e0, 1.0f), fminf(e1, 1.0f)), pk2(rcp_approx(d0), rcp_approx(d1)));
            acc.w[h] = fma2(b, c2, acc.w[h]);
            kahan_fma2(acc.a[h], acc.nc[h], fma2(b, m2c2, c2), r);
        }
    }
}

// The same, direct form (tiles whose exponents leave the factorised range).
__device__ __forceinline__ void fwd_loop4_direct(const float4 *sh, int first, int step,
                                                 int m_ent, const Lane4 &t, float l2,
                                                 float *w, float *a, float *c)
{
#pragma unroll 2
    for (int i = first; i < m_ent; i += step) {
        const float4 en = sh[i];
        const float cf = entry_cf(en);
#pragma unroll
        for (int j = 0; j < kLaneK; ++j) {
            bool bj;
            const float r = small_sigma_direct(en, t.s[j].tau, l2, bj);
            w[j] += bj ? cf : 0.0f;
            kahan_fma(a[j], c[j], bj ? -cf : cf, r);
        }
    }
}

// Forward: one block per unit (tile, image x direction). Each warp runs a pass of kWarpK
// thresholds over every other staged entry (warp w: entries w, w + kSoftWarps, ...); the warps'
// sums meet in shared memory, in a fixed order, as fp64 partials per (unit, threshold).
__global__ void __launch_bounds__(kSoftThreads) soft_fwd_kernel(
    const float *__restrict__ tau, int K, float l2, const int *__restrict__ counts,
    const float4 *__restrict__ entries, double *__restrict__ part, int64_t tiles)
{
    __shared__ float4 sh[kChunk];
    __shared__ double wsum[kSoftWarps][kWarpK];
    const int64_t unit = blockIdx.y * tiles + blockIdx.x;
    const int cnt = counts[unit];
    const int n = cnt & (kTileFlagDirect - 1);
    const float4 *__restrict__ list = entries + unit * (int64_t)kTileCap;
    const float m = tau_midpoint(tau, K);
    const int lane = threadIdx.x & (kWarp - 1), warp = threadIdx.x >> 5;
    for (int kb = 0; kb < K; kb += kWarpK) {
        const Lane4 t = lane_thresholds(tau, kb, lane, K, l2, m);
        const bool fact = __syncthreads_and(t.ok && !(cnt & kTileFlagDirect));
        float w[kLaneK] = {0.f, 0.f, 0.f, 0.f}, a[kLaneK] = {0.f, 0.f, 0.f, 0.f};
        float c[kLaneK] = {0.f, 0.f, 0.f, 0.f};
        FwdAcc acc;
        const f32x2 F[2] = {pk2(t.s[0].F, t.s[1].F), pk2(t.s[2].F, t.s[3].F)};
#pragma unroll
        for (int h = 0; h < 2; ++h) acc.w[h] = acc.a[h] = acc.nc[h] = 0ull;
        for (int e0 = 0; e0 < n; e0 += kChunk) {
            const int m_ent = min(kChunk, n - e0);
            __syncthreads();
            // factorised form: each entry staged as the pairs (E, E), (c, c) the packed loop uses
            for (int i = threadIdx.x; i < m_ent; i += kSoftThreads) {
                const float4 en = list[e0 + i];
                sh[i] = fact ? make_float4(en.x, en.x, entry_cf(en), entry_cf(en)) : en;
            }
            __syncthreads();
            if (fact)
                fwd_loop4_packed(sh, warp, kSoftWarps, m_ent, F, acc);
            else
                fwd_loop4_direct(sh, warp, kSoftWarps, m_ent, t, l2, w, a, c);
        }
        if (fact) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float n0, n1;
                upk2(acc.w[h], w[2 * h], w[2 * h + 1]);
                upk2(acc.a[h], a[2 * h], a[2 * h + 1]);
                upk2(acc.nc[h], n0, n1);
                c[2 * h] = -n0;
                c[2 * h + 1] = -n1;
            }
        }
#pragma unroll
        for (int j = 0; j < kLaneK; ++j)
            wsum[warp][lane + kWarp * j] = (double)w[j] + ((double)a[j] - (double)c[j]);
        __syncthreads();
        for (int k = threadIdx.x; k < kWarpK; k += kSoftThreads) {
            double v = 0.0;
#pragma unroll
            for (int ww = 0; ww < kSoftWarps; ++ww) v += wsum[ww][k];
            if (kb + k < K) part[unit * K + kb + k] = v;
        }
        __syncthreads();  // wsum is read before the next pass writes it
    }
}

// out[b][k] = sum over the image's tiles of the partial sums, in tile order.
constexpr int kFwdRedMaxWarps = 32;  // forward-reduction block: up to 32 warps share the tiles

// Block (threshold group, image row bj) of nw = blockDim.x / 32 warps: lane l of warp w adds the
// partials of threshold 32 blockIdx.x + l over tiles w, w + nw, ... in order (each load a
// 256-byte row of 32 thresholds), then the nw warp sums are added in warp order: deterministic
// for a given shape (the host picks nw from the tile count).
__global__ void __launch_bounds__(kFwdRedMaxWarps * kWarp) soft_fwd_reduce_kernel(
    const double *__restrict__ part, float *__restrict__ out, int K, int64_t tiles,
    int64_t batch)
{
    __shared__ double red[kFwdRedMaxWarps][kWarp + 1];
    const int lane = threadIdx.x & (kWarp - 1), warp = threadIdx.x >> 5;
    const int nw = blockDim.x >> 5;
    const int k = blockIdx.x * kWarp + lane;
    const int64_t bj = blockIdx.y;
    double acc = 0.0;
    if (k < K) {
        const double *__restrict__ p = part + bj * tiles * K + k;
        int64_t t = warp;
        for (; t + 3 * nw < tiles; t += 4 * nw) {  // four loads in flight, added in order
            const double v0 = p[t * K], v1 = p[(t + nw) * K];
            const double v2 = p[(t + 2 * nw) * K], v3 = p[(t + 3 * nw) * K];
            acc += v0;
            acc += v1;
            acc += v2;
            acc += v3;
        }
        for (; t < tiles; t += nw) acc += p[t * K];
    }
    red[warp][lane] = acc;
    __syncthreads();
    if (warp == 0 && k < K) {
        double sum = 0.0;
        for (int w = 0; w < nw; ++w) sum += red[w][lane];
        out[bj * K + k] = (float)sum;
    }
}

// Backward over one group of kGroup staged entries for a lane's four thresholds: w = r - r^2
// per term, the dtau Kahan sums over c w, and the entry's sum over the warp's thresholds of
// g_k w (qw: this warp's [kGroup][32] transpose buffer). Returns, in lanes 4e .. 4e + 3, the sum
// over all kWarpK thresholds of the pass for entry e of the group.
__device__ __forceinline__ float group_row_sum(float (*qw)[kWarp], int lane)
{
    __syncwarp();
    const float4 *rowp = reinterpret_cast<const float4 *>(&qw[lane >> 2][(lane & 3) * 8]);
    const float4 x = rowp[0], y = rowp[1];
    float s = ((x.x + x.y) + (x.z + x.w)) + ((y.x + y.y) + (y.z + y.w));
    s += __shfl_xor_sync(kFull, s, 1);
    s += __shfl_xor_sync(kFull, s, 2);
    __syncwarp();
    return s;
}

// The factorised small part for both thresholds, negated: e = E F_k = exp(lambda (X - tau_k)),
// -r = max(-e, -1) / (1 + e) = -min(e, 1) / (1 + e); e may overflow to +inf (-r = -1 * 0) or
// underflow to 0. The backward's terms carry -r and -w: -w = r^2 - r = fma(-r, -r, -r) is one
// packed FMA, where w = fma(-r, r, r) needed a negation first. With -c and -g as the other
// factors every product, and so every sum, keeps its bits.
__device__ __forceinline__ f32x2 neg_small_sigma_fact2(f32x2 E2, f32x2 F)
{
    float e0, e1, d0, d1;
    const f32x2 e = mul2(E2, F);
    upk2(e, e0, e1);
    upk2(add2(e, pk2(1.0f, 1.0f)), d0, d1);
    return mul2(pk2(fmaxf(-e0, -1.0f), fmaxf(-e1, -1.0f)), pk2(rcp_approx(d0), rcp_approx(d1)));
}
__device__ __forceinline__ float entry_neg_cf(const float4 &en)
{
    return 8388616.0f - __int_as_float(0x4B000000 | (__float_as_int(en.w) & 15));
}

// ng: the lane's upstream gradients negated, as pairs; en8: entries staged as (E, E), (-c, -c).
__device__ __forceinline__ float bwd_group4_packed(const float4 *en8, const f32x2 *F,
                                                   const f32x2 *ng, f32x2 *a, f32x2 *nc,
                                                   float (*qw)[kWarp], int lane)
{
#pragma unroll
    for (int j = 0; j < kGroup; ++j) {
        const ulonglong2 en = *reinterpret_cast<const ulonglong2 *>(en8 + j);  // (E, E), (-c, -c)
        f32x2 gw = 0ull;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const f32x2 rn = neg_small_sigma_fact2(en.x, F[h]);  // -r
            const f32x2 wn = fma2(rn, rn, rn);                   // -w = r^2 - r
            kahan_fma2(a[h], nc[h], en.y, wn);                   // (-c)(-w) = c w
            gw = fma2(ng[h], wn, gw);                            // (-g)(-w) = g w
        }
        float q0, q1;
        upk2(gw, q0, q1);
        qw[j][lane] = q0 + q1;
    }
    return group_row_sum(qw, lane);
}

__device__ __forceinline__ float bwd_group4_direct(const float4 *en8, const Lane4 &t,
                                                   const float *g, float l2, float *a, float *c,
                                                   float (*qw)[kWarp], int lane)
{
#pragma unroll
    for (int j = 0; j < kGroup; ++j) {
        const float4 en = en8[j];
        const float cf = entry_cf(en);
        float q = 0.0f;
#pragma unroll
        for (int k = 0; k < kLaneK; ++k) {
            bool bk;
            const float r = small_sigma_direct(en, t.s[k].tau, l2, bk);
            const float w = fmaf(-r, r, r);
            kahan_fma(a[k], c[k], cf, w);
            q = fmaf(g[k], w, q);
        }
        qw[j][lane] = q;
    }
    return group_row_sum(qw, lane);
}

// Backward: one block per (tile, image, direction), or, when the image gradient is wanted, one
// per (tile, image) looping over the directions; thread t owns thresholds k = kb + t and
// kb + t + 64. The image gradient of the tile collects alpha dX over the directions in shared
// memory in a fixed order and is written once, for every voxel of the tile.
template <int NDIM>
__global__ void __launch_bounds__(kSoftThreads) soft_bwd_kernel(
    const float *__restrict__ img, const float *__restrict__ tau, int K, int ndirs, float lambda,
    float l2, const float *__restrict__ alpha_p, const float *__restrict__ grad_out,
    const int *__restrict__ counts, const float4 *__restrict__ entries,
    const float2 *__restrict__ coords, double *__restrict__ part, double *__restrict__ scal,
    float *__restrict__ grad_img, SoftGeom g)
{
    using T = SoftTile<NDIM>;
    constexpr int NW = kSoftThreads / kWarp;
    __shared__ __align__(16) float4 sh[kBwdChunk];
    __shared__ __align__(16) float qbuf[NW][kGroup][kWarp];
    __shared__ double tsum[NW][kWarpK];
    __shared__ float dxs[kTileCap];
    extern __shared__ float gacc[];  // kTileCap floats, present only when grad_img is wanted
    __shared__ double scal_red[NW][kScal];

    // Without an image gradient every (image, direction) pair is a block of its own
    // (blockIdx.y = b ndirs + j); with one, a block walks all directions of its image so that the
    // gradient collects them in a fixed order in shared memory (blockIdx.y = b).
    const bool per_dir = grad_img == nullptr;
    const int64_t b = per_dir ? blockIdx.y / ndirs : blockIdx.y;
    const int jbeg = per_dir ? (int)(blockIdx.y % ndirs) : 0;
    const int jend = per_dir ? jbeg + 1 : ndirs;
    const int64_t tile = blockIdx.x;
    const int64_t units = (int64_t)(per_dir ? gridDim.y : gridDim.y * ndirs) * g.tiles;
    const int lane = threadIdx.x & (kWarp - 1), warp = threadIdx.x >> 5;
    const float m = tau_midpoint(tau, K);
    const float alpha = __ldg(alpha_p);
    const int64_t image = g.D * g.Hy * g.W;
    const float *__restrict__ f = img + b * image;
    const int64_t x0 = (tile % g.tiles_x) * T::X;
    const int64_t y0 = ((tile / g.tiles_x) % g.tiles_y) * T::Y;
    const int64_t z0 = (tile / (g.tiles_x * g.tiles_y)) * T::Z;
    const float2 *__restrict__ cz = coords;
    const float2 *__restrict__ cy = coords + g.nz;
    const float2 *__restrict__ cx = coords + g.nz + g.Hy;
    if (grad_img)
        for (int i = threadIdx.x; i < kTileCap; i += kSoftThreads) gacc[i] = 0.0f;

    for (int j = jbeg; j < jend; ++j) {
        const int64_t bj = b * ndirs + j;
        const int64_t unit = bj * g.tiles + tile;
        const int cnt = counts[unit];
        const int n = cnt & (kTileFlagDirect - 1);
        const float4 *__restrict__ list = entries + unit * (int64_t)kTileCap;
        __syncthreads();  // the previous direction is done with dxs
        for (int i = threadIdx.x; i < n; i += kSoftThreads) dxs[i] = 0.0f;

        for (int kb = 0; kb < K; kb += kWarpK) {
            // lane l: thresholds kb + l + 32 j; warp w: groups w, w + NW, ... of each chunk, so
            // every entry's sum over the pass's thresholds is one warp's (no cross-warp sum)
            const Lane4 t = lane_thresholds(tau, kb, lane, K, l2, m);
            float g[kLaneK];
#pragma unroll
            for (int k = 0; k < kLaneK; ++k) {
                const int kk = kb + lane + kWarp * k;
                g[k] = kk < K ? __ldg(grad_out + bj * K + kk) : 0.0f;
            }
            const bool fact = __syncthreads_and(t.ok && !(cnt & kTileFlagDirect));
            float a[kLaneK] = {0.f, 0.f, 0.f, 0.f}, c[kLaneK] = {0.f, 0.f, 0.f, 0.f};
            const f32x2 F[2] = {pk2(t.s[0].F, t.s[1].F), pk2(t.s[2].F, t.s[3].F)};
            const f32x2 ngp[2] = {pk2(-g[0], -g[1]), pk2(-g[2], -g[3])};
            f32x2 ap[2] = {0ull, 0ull}, ncp[2] = {0ull, 0ull};  // packed dtau sums (factorised)
            for (int e0 = 0; e0 < n; e0 += kBwdChunk) {
                const int m_ent = min(kBwdChunk, n - e0);
                __syncthreads();
                // stage the chunk; pad the last group with c = 0 entries
                // factorised form: each entry staged as the pairs (E, E), (-c, -c)
                for (int i = threadIdx.x; i < kBwdChunk; i += kSoftThreads) {
                    const float4 en = (i < m_ent)
                                          ? list[e0 + i]
                                          : make_float4(0.f, 0.f, 0.f, __int_as_float(kPadWord));
                    sh[i] = fact ? make_float4(en.x, en.x, entry_neg_cf(en), entry_neg_cf(en))
                                 : en;
                }
                __syncthreads();
                for (int gi = warp; gi * kGroup < m_ent; gi += NW) {
                    const float rs =
                        fact ? bwd_group4_packed(sh + gi * kGroup, F, ngp, ap, ncp, qbuf[warp],
                                                 lane)
                             : bwd_group4_direct(sh + gi * kGroup, t, g, l2, a, c, qbuf[warp],
                                                 lane);
                    // padding entries (index n and above) add 0 to unused slots
                    if ((lane & 3) == 0) dxs[e0 + gi * kGroup + (lane >> 2)] += rs;
                }
            }
            if (fact) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float n0, n1;
                    upk2(ap[h], a[2 * h], a[2 * h + 1]);
                    upk2(ncp[h], n0, n1);
                    c[2 * h] = -n0;
                    c[2 * h + 1] = -n1;
                }
            }
#pragma unroll
            for (int k = 0; k < kLaneK; ++k)
                tsum[warp][lane + kWarp * k] = (double)a[k] - (double)c[k];
            __syncthreads();
            for (int k = threadIdx.x; k < kWarpK; k += kSoftThreads) {
                if (kb + k >= K) continue;
                double v = 0.0;
#pragma unroll
                for (int ww = 0; ww < NW; ++ww) v += tsum[ww][k];
                const double gk = (double)__ldg(grad_out + bj * K + kb + k);
                part[(kb + k) * units + unit] = (double)lambda * gk * v;
            }
            __syncthreads();  // tsum and dxs are read before the next pass writes them
        }
        __syncthreads();

        // per-voxel gradient: dX = -lambda c sum_k g w; grad_img += alpha dX; dalpha, du partials
        // A thread takes its entries i = tid, tid + 64, ... in that order, kTailBatch at a time:
        // the batch's loads (entry, then image value and coordinates) are all issued before any
        // is used, so their latencies overlap; the sums see the entries in the same order.
        float sum[kScal] = {0.f, 0.f, 0.f, 0.f}, comp[kScal] = {0.f, 0.f, 0.f, 0.f};
        for (int i0 = threadIdx.x; i0 < n; i0 += kTailBatch * kSoftThreads) {
            float4 en[kTailBatch];
            bool ok[kTailBatch];
#pragma unroll
            for (int u = 0; u < kTailBatch; ++u) {
                const int i = i0 + u * kSoftThreads;
                ok[u] = i < n;
                en[u] = ok[u] ? list[i] : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            int loc[kTailBatch];
            float fv[kTailBatch];
            float2 xy[kTailBatch], xx[kTailBatch], xz[kTailBatch];
#pragma unroll
            for (int u = 0; u < kTailBatch; ++u) {
                loc[u] = entry_loc(en[u]);
                ok[u] = ok[u] && bounds_ok(&g_soft_error, loc[u] >= 0 && loc[u] < kTileCap,
                                           kErrSoftLoc);
                const int l = ok[u] ? loc[u] : 0;
                const int64_t gx = x0 + l % T::X, gy = y0 + (l / T::X) % T::Y,
                              gz = z0 + l / (T::X * T::Y);
                ok[u] = ok[u] && bounds_ok(&g_soft_error, gx < g.W && gy < g.Hy && gz < g.D,
                                           kErrSoftIndex);
                fv[u] = 0.f;
                xy[u] = xx[u] = xz[u] = make_float2(0.f, 0.f);
                if (ok[u]) {
                    fv[u] = __ldg(f + (gz * g.Hy + gy) * g.W + gx);
                    xy[u] = __ldg(cy + gy);
                    xx[u] = __ldg(cx + gx);
                    if (NDIM == 3) xz[u] = __ldg(cz + gz);
                }
            }
#pragma unroll
            for (int u = 0; u < kTailBatch; ++u) {
                if (!ok[u]) continue;
                const float dX = -lambda * entry_cf(en[u]) * dxs[i0 + u * kSoftThreads];
                if (grad_img) gacc[loc[u]] += alpha * dX;  // one entry per voxel and direction
                kahan_add(sum[0], comp[0], dX * fv[u]);
                if (NDIM == 3) kahan_add(sum[1], comp[1], dX * (xz[u].x + xz[u].y));
                kahan_add(sum[NDIM - 1], comp[NDIM - 1], dX * (xy[u].x + xy[u].y));
                kahan_add(sum[NDIM], comp[NDIM], dX * (xx[u].x + xx[u].y));
            }
        }
        double v[kScal];
#pragma unroll
        for (int q = 0; q < kScal; ++q) {
            v[q] = (double)sum[q] - (double)comp[q];
#pragma unroll
            for (int o = kWarp / 2; o > 0; o >>= 1) v[q] += __shfl_xor_sync(kFull, v[q], o);
        }
        if (lane == 0) {
#pragma unroll
            for (int q = 0; q < kScal; ++q) scal_red[warp][q] = v[q];
        }
        __syncthreads();
        if (threadIdx.x < kScal) {
            double acc = 0.0;
            for (int w2 = 0; w2 < NW; ++w2) acc += scal_red[w2][threadIdx.x];
            scal[unit * kScal + threadIdx.x] = acc;
        }
    }
    if (!grad_img) return;
    __syncthreads();
    for (int i = threadIdx.x; i < kTileCap; i += kSoftThreads) {
        const int64_t gx = x0 + i % T::X, gy = y0 + (i / T::X) % T::Y, gz = z0 + i / (T::X * T::Y);
        if (gz < g.D && gy < g.Hy && gx < g.W)
            grad_img[b * image + (gz * g.Hy + gy) * g.W + gx] = gacc[i];
    }
}

// grad_tau[k] = sum over (image, tile) of the partials; grad_alpha, grad_u likewise. One block per
// output: threads take strided partials in fp64, then a fixed-order tree (deterministic).
constexpr int kReduceThreads = 256;

// One block per output: o < K grad_tau[o] (the backward kernel stores its threshold partials
// threshold-major, so a block reads one contiguous row), o = K grad_alpha, o = K + 1 + j ndim + d
// grad_u[j][d]. Threads take strided partials (four loads in flight, added in order), then a
// fixed-order tree: results are deterministic.
__global__ void __launch_bounds__(kReduceThreads) soft_bwd_reduce_kernel(
    const double *__restrict__ part, const double *__restrict__ scal, int K, int ndim, int ndirs,
    int64_t images, int64_t tiles, float *__restrict__ grad_tau, float *__restrict__ grad_alpha,
    float *__restrict__ grad_u)
{
    __shared__ double red[kReduceThreads];
    const int64_t units = images * ndirs * tiles;
    const int o = blockIdx.x;
    double acc = 0.0;
    if (o < K) {
        const double *__restrict__ row = part + (int64_t)o * units;
        int64_t u = threadIdx.x;
        for (; u + 3 * kReduceThreads < units; u += 4 * kReduceThreads) {
            const double v0 = row[u], v1 = row[u + kReduceThreads];
            const double v2 = row[u + 2 * kReduceThreads], v3 = row[u + 3 * kReduceThreads];
            acc += v0;
            acc += v1;
            acc += v2;
            acc += v3;
        }
        for (; u < units; u += kReduceThreads) acc += row[u];
    } else if (o == K) {
        for (int64_t u = threadIdx.x; u < units; u += kReduceThreads) acc += scal[u * kScal];
    } else {
        const int j = (o - K - 1) / ndim, d = (o - K - 1) % ndim;
        // the units of direction j: (image b, tile t) -> ((b ndirs + j) tiles + t)
        for (int64_t i = threadIdx.x; i < images * tiles; i += kReduceThreads) {
            const int64_t b = i / tiles, t = i % tiles;
            acc += scal[((b * ndirs + j) * tiles + t) * kScal + 1 + d];
        }
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

// stats = {listed voxels, tiles on the direct path, tiles}: one block, fixed-order tree.
__global__ void __launch_bounds__(kReduceThreads) soft_stats_kernel(const int *__restrict__ counts,
                                                                    int64_t units,
                                                                    int64_t *__restrict__ stats)
{
    __shared__ long long red[2][kReduceThreads];
    long long n = 0, direct = 0;
    for (int64_t i = threadIdx.x; i < units; i += kReduceThreads) {
        const int c = counts[i];
        n += c & (kTileFlagDirect - 1);
        direct += (c & kTileFlagDirect) ? 1 : 0;
    }
    red[0][threadIdx.x] = n;
    red[1][threadIdx.x] = direct;
    __syncthreads();
    for (int st = kReduceThreads / 2; st > 0; st >>= 1) {
        if (threadIdx.x < st) {
            red[0][threadIdx.x] += red[0][threadIdx.x + st];
            red[1][threadIdx.x] += red[1][threadIdx.x + st];
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        stats[0] = red[0][0];
        stats[1] = red[1][0];
        stats[2] = units;
    }
}

static SoftGeom soft_geom(const SoftLayout &L)
{
    SoftGeom g;
    g.D = L.D;
    g.Hy = L.Hy;
    g.W = L.W;
    g.nz = L.ndim == 3 ? L.D : 0;
    g.tiles_x = L.tiles_x;
    g.tiles_y = L.tiles_y;
    g.tiles = L.tiles;
    return g;
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
    const SoftGeom g = soft_geom(L);
    const int64_t ncoord = g.nz + L.Hy + L.W;
    soft_coords_kernel<<<(unsigned)((ncoord + 255) / 256), 256, 0, s>>>(coords, g.nz, L.Hy, L.W);
    // Directions in groups, each prep block reading its tile of f once for a whole group: as
    // many groups as give about kPrepBlocks blocks (the tile list of a single direction and of
    // a small transform stays one group).
    const int64_t tile_images = L.tiles * L.batch;
    const int groups = (int)std::min<int64_t>(
        L.ndirs, std::max<int64_t>(1, (kPrepBlocks + tile_images - 1) / tile_images));
    const int dpb = (L.ndirs + groups - 1) / groups;
    const int ngroups = (L.ndirs + dpb - 1) / dpb;
    const dim3 grid((unsigned)L.tiles, (unsigned)(L.batch * ngroups));
    if (L.ndim == 3)
        soft_prep_kernel<3><<<grid, kPrepThreads, 0, s>>>(img, alpha, u, L.ndirs, dpb, tau, L.K,
                                                          l2, coords, counts, entries, g);
    else
        soft_prep_kernel<2><<<grid, kPrepThreads, 0, s>>>(img, alpha, u, L.ndirs, dpb, tau, L.K,
                                                          l2, coords, counts, entries, g);
    // one block per unit (tile, image x direction)
    const dim3 ugrid((unsigned)L.tiles, (unsigned)(L.batch * L.ndirs));
    soft_fwd_kernel<<<ugrid, kSoftThreads, 0, s>>>(tau, L.K, l2, counts, entries, part, L.tiles);
    // about eight tiles per warp, 1 to 32 warps
    const int rwarps =
        (int)std::min<int64_t>(kFwdRedMaxWarps, std::max<int64_t>(1, (L.tiles + 7) / 8));
    const dim3 rgrid((unsigned)((L.K + kWarp - 1) / kWarp), (unsigned)(L.batch * L.ndirs));
    soft_fwd_reduce_kernel<<<rgrid, rwarps * kWarp, 0, s>>>(part, out, L.K, L.tiles,
                                                            L.batch * L.ndirs);
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
    const SoftGeom g = soft_geom(L);
    // one block per (tile, image, direction) unless the image gradient is asked for: then one per
    // (tile, image), walking the directions (see soft_bwd_kernel)
    const dim3 grid((unsigned)L.tiles, (unsigned)(grad_img ? L.batch : L.batch * L.ndirs));
    const float l2 = lambda_log2e(lambda);
    // the image-gradient accumulator costs shared memory (and so resident blocks) only when asked
    const size_t dyn = grad_img ? sizeof(float) * kTileCap : 0;
    if (L.ndim == 3)
        soft_bwd_kernel<3><<<grid, kSoftThreads, dyn, s>>>(img, tau, L.K, L.ndirs, lambda, l2,
                                                           alpha, grad_out, counts, entries,
                                                           coords, part, scal, grad_img, g);
    else
        soft_bwd_kernel<2><<<grid, kSoftThreads, dyn, s>>>(img, tau, L.K, L.ndirs, lambda, l2,
                                                           alpha, grad_out, counts, entries,
                                                           coords, part, scal, grad_img, g);
    const unsigned rblocks = (unsigned)(L.K + 1 + L.ndirs * L.ndim);
    soft_bwd_reduce_kernel<<<rblocks, kReduceThreads, 0, s>>>(
        part, scal, L.K, L.ndim, L.ndirs, L.batch, L.tiles, grad_tau, grad_alpha, grad_u);
    return cudaGetLastError();
}

cudaError_t soft_run_stats(const SoftLayout &L, const void *ws, int64_t *stats, cudaStream_t s)
{
    const int *counts = reinterpret_cast<const int *>(static_cast<const char *>(ws) + L.off_counts);
    soft_stats_kernel<<<1, kReduceThreads, 0, s>>>(counts, L.batch * L.ndirs * L.tiles, stats);
    return cudaGetLastError();
}

}  // namespace ecc
