// ecc_hard.cu -- hard Euler characteristic curve of dense 2-D / 3-D grids (sm_103a).
//
// Paper notes "Scalable GPU-Accelerated Euler Characteristic Curves: Optimization and
// Differentiable Learning for PyTorch":
//   "Key designs -- full-scan CUDA kernel": one pass over the whole grid with no chunked
//   re-launches; each thread block keeps a private shared-memory histogram of H bins and flushes
//   it once, with one global atomic per non-empty bin.
//   "Key designs -- local computation of the Euler characteristic coefficient": c(p) from the
//   3x3 / 3x3x3 neighbourhood, accumulated at p's threshold bin.
// The running sum of the histogram over bins is the curve (ecc_bin_scan_kernel).
//
// Both kernels first turn every voxel into its exact threshold key (ecc_keys.cuh) and then work
// on fp16 key patterns, two pixels per instruction. Every position outside the grid reads as NaN
// (key H, "never"), so the steady state has no boundary branches.
//
// 2-D: a warp owns a strip of 128 columns (four per lane, one 16-byte load per lane per row) and
// walks down a band of rows; raw rows are prefetched four rows ahead in registers, and the
// comparisons with the row below are reused as the "above" comparisons of the next row. The
// keys just left and right of the strip ride on the rotated row shuffles.
//
// 3-D: the complex of a volume splits into the cells of each plane z and the vertical cells
// sigma x [z, z+1]; a vertical cell's value is the max over sigma of M_z = max(S_z, S_{z+1}) and
// its dimension is dim(sigma) + 1, so ECC_3D = sum_z ECC_2D(S_z) - sum_z ECC_2D(M_z). Folding
// each max-pixel into the voxel that carries it gives one contribution per voxel p = (x, y, z):
//     c(p) = c2(S_z; p) - [k_{z+1} < k_z] c2(M_z; x,y) - [k_{z-1} <= k_z] c2(M_{z-1}; x,y)
// (the later voxel wins ties; the max of two keys is the key of the max). A block owns a tile of
// 128 columns x 8 rows and walks z; each plane's keys are computed once into a shared tile with a
// one-pixel halo, from which every warp builds the three rows around its own row. The raw values
// of the next plane are loaded into registers one plane ahead.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ecc_internal.cuh"
#include "ecc_keys.cuh"

namespace ecc {

constexpr int kHardThreads = 256;
constexpr int kHardWarps = kHardThreads / kWarp;
constexpr int kStrip = 128;  // columns per warp strip / block tile
// Tables of at most this many bins take the stencil's flags from the FMA pipe (exact for keys
// up to 1024; see flag_lt / flag_le), larger ones from fp16 compares.
constexpr int kSatMaxBins = 1024;

// Resident blocks per SM the kernels are compiled for (register budget 65536 / (256 * blocks)).
#ifndef ECC_2D_MIN_BLOCKS
#define ECC_2D_MIN_BLOCKS 3
#endif
#ifndef ECC_3D_MIN_BLOCKS
#define ECC_3D_MIN_BLOCKS 3
#endif

// ----------------------------------------------------------------------------------------------
// Block setup, keys and histogram
// ----------------------------------------------------------------------------------------------

// Shared layout: int hist[H + 1] (bin H collects the discarded "never" contributions), then the
// table: f32 thresholds T[0..H+1], or for uint8 inputs the fp16 key pattern of each byte value.
__host__ __device__ constexpr int hist_words(int H) { return (H + 2) & ~1; }  // keeps 8-byte align

template <int CAP>
__device__ __forceinline__ void block_setup(const HardParams<CAP> &P, int *hist, float *table)
{
    for (int i = threadIdx.x; i <= P.H; i += blockDim.x) hist[i] = 0;
    for (int i = threadIdx.x; i < P.table_len; i += blockDim.x) table[i] = P.table[i];
    __syncthreads();
}

template <int CAP>
__device__ __forceinline__ void block_flush(const HardParams<CAP> &P, const int *hist, int64_t b)
{
    __syncthreads();
    unsigned long long *dst = reinterpret_cast<unsigned long long *>(P.out + b * (int64_t)P.H);
    for (int i = threadIdx.x; i < P.H; i += blockDim.x) {
        const int v = hist[i];
        if (v != 0) atomicAdd(dst + i, (unsigned long long)(long long)(P.sign * v));
    }
}

template <int CAP>
__device__ __forceinline__ KeyConsts key_consts(const HardParams<CAP> &P)
{
    KeyConsts K;
    K.a = P.key_a;
    K.b = P.key_b;
    K.nH = -(float)P.H;
    K.clo = P.key_clo;
    K.chi = P.key_chi;
    K.H = P.H;
    return K;
}

__device__ __forceinline__ float qnan_f() { return __int_as_float(0x7fffffff); }

// Raw values one lane needs from one row: its four columns and one side value (lane 0: the
// column right of the strip, lane 31: the column left of it; NaN where the grid has none).
template <typename T>
struct Raw;

template <>
struct Raw<float> {
    float v[4];
    float side;
};

template <>
struct Raw<uint8_t> {
    uint32_t bytes;  // four values, first column in the low byte
    uint32_t side;   // the side value, or 256 for "none"
    uint32_t own_ok; // bit j: column j of the lane is inside the grid (and the row exists)
};

// Columns of a lane within the strip starting at x0 (fixed for a whole task).
struct Cols {
    int x;        // first own column
    int sx;       // side column, clamped into the grid
    uint32_t own_ok;  // bit j: x + j < W
    bool side_ok;     // the side column exists
    bool full;        // all four own columns exist and the 16-byte (4-byte for u8) load is legal
};

__device__ __forceinline__ Cols strip_cols(int x0, int W, int lane, bool vec_ok)
{
    Cols c;
    c.x = x0 + 4 * lane;
    const int sx = (lane == 0) ? x0 + kStrip : (lane == kWarp - 1 ? x0 - 1 : c.x);
    c.side_ok = (lane == 0 || lane == kWarp - 1) && sx >= 0 && sx < W;
    c.sx = min(max(sx, 0), W - 1);
    c.own_ok = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) c.own_ok |= (c.x + j < W) ? (1u << j) : 0u;
    c.full = vec_ok && (x0 + kStrip <= W);
    return c;
}

// Keys of a raw row: own pairs (k0 | k1 << 16, k2 | k3 << 16) and the side key (low half).
template <bool SEARCH>
__device__ __forceinline__ void row_keys(const Raw<float> &r, const KeyConsts &K,
                                         const float *__restrict__ T, uint32_t &own0,
                                         uint32_t &own1, uint32_t &side)
{
    uint32_t k[5];
    if (SEARCH) {
#pragma unroll
        for (int j = 0; j < 4; ++j) k[j] = key_search_pattern(r.v[j], K.H, T);
        k[4] = key_search_pattern(r.side, K.H, T);
    } else {
        uint32_t amb = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) k[j] = key_fast(r.v[j], K, amb);
        k[4] = key_fast(r.side, K, amb);
        if (__any_sync(kFull, amb != 0)) {  // rare: a value within E of a threshold
            if (amb != 0) {
#pragma unroll
                for (int j = 0; j < 4; ++j) k[j] = key_fix(r.v[j], k[j], K.H, T);
                k[4] = key_fix(r.side, k[4], K.H, T);
            }
        }
    }
    own0 = prmt(k[0], k[1], 0x5410);
    own1 = prmt(k[2], k[3], 0x5410);
    side = k[4];
}

template <bool SEARCH>
__device__ __forceinline__ void row_keys(const Raw<uint8_t> &r, const KeyConsts &K,
                                         const float *__restrict__ T, uint32_t &own0,
                                         uint32_t &own1, uint32_t &side)
{
    const uint16_t *lut = reinterpret_cast<const uint16_t *>(T);
    const uint32_t never = kKeyBase + (uint32_t)K.H;
    uint32_t k[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t v = lut[(r.bytes >> (8 * j)) & 0xffu];
        k[j] = ((r.own_ok >> j) & 1u) ? v : never;
    }
    own0 = prmt(k[0], k[1], 0x5410);
    own1 = prmt(k[2], k[3], 0x5410);
    side = (r.side < 256u) ? (uint32_t)lut[r.side & 0xffu] : never;
}

// ----------------------------------------------------------------------------------------------
// 2-D kernel
// ----------------------------------------------------------------------------------------------
//
// Work: the rows of an image's 128-column strips, strip-major ("strip-rows", N = strips * Hy),
// are split into equal contiguous ranges, one per warp of the image's blocks (blockIdx.y =
// image). A warp walks its range as one band per strip it touches, so the only repeated work is
// the two rows around each band, and warps that run side by side read neighbouring rows.

template <typename T, bool SEARCH>
__device__ __forceinline__ KeyRow key_row(const Raw<T> &r, const KeyConsts &K,
                                          const float *__restrict__ table, const LaneShuffle &q)
{
    uint32_t own0, own1, side;
    row_keys<SEARCH>(r, K, table, own0, own1, side);
    return make_key_row(own0, own1, side, q);
}

// Predicated loads (no branch): the value at p when ok, else the given default.
__device__ __forceinline__ float ldg_if(const float *p, bool ok, float dflt)
{
    float v = dflt;
    asm("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %2, 0;\n\t@q ld.global.nc.f32 %0, [%1];\n\t}"
        : "+f"(v)
        : "l"(p), "r"((unsigned)ok));
    return v;
}
__device__ __forceinline__ uint32_t ldg_if(const uint8_t *p, bool ok, uint32_t dflt)
{
    uint32_t v = dflt;
    asm("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %2, 0;\n\t@q ld.global.nc.u8 %0, [%1];\n\t}"
        : "+r"(v)
        : "l"(p), "r"((unsigned)ok));
    return v;
}

// Rows of one band as a lane reads them: its own columns and its side column, one row after
// the other; rows before 0 and from `rlim` on read as absent.
template <typename T>
struct RowCursor {
    const T *own;   // the lane's first column in row r
    const T *side;  // the lane's side column in row r
    int r, rlim;
    int W;
};

template <typename T>
__device__ __forceinline__ RowCursor<T> row_cursor(const T *__restrict__ img, const Cols &c, int r0,
                                                   int rlim, int W)
{
    RowCursor<T> rc;
    rc.own = img + (int64_t)r0 * W + c.x;
    rc.side = img + (int64_t)r0 * W + c.sx;
    rc.r = r0;
    rc.rlim = rlim;
    rc.W = W;
    return rc;
}

template <bool FULL>
__device__ __forceinline__ Raw<float> next_row(RowCursor<float> &rc, const Cols &c)
{
    Raw<float> out;
    if ((unsigned)rc.r < (unsigned)rc.rlim) {  // warp-uniform
        if (FULL) {
            const float4 q = __ldg(reinterpret_cast<const float4 *>(rc.own));
            out.v[0] = q.x;
            out.v[1] = q.y;
            out.v[2] = q.z;
            out.v[3] = q.w;
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                out.v[j] = ldg_if(rc.own + j, (c.own_ok >> j) & 1u, qnan_f());
        }
        out.side = ldg_if(rc.side, c.side_ok, qnan_f());
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) out.v[j] = qnan_f();
        out.side = qnan_f();
    }
    rc.own += rc.W;
    rc.side += rc.W;
    ++rc.r;
    return out;
}

template <bool FULL>
__device__ __forceinline__ Raw<uint8_t> next_row(RowCursor<uint8_t> &rc, const Cols &c)
{
    Raw<uint8_t> out;
    if ((unsigned)rc.r < (unsigned)rc.rlim) {  // warp-uniform
        if (FULL) {
            out.bytes = __ldg(reinterpret_cast<const unsigned int *>(rc.own));
        } else {
            out.bytes = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                out.bytes |= ldg_if(rc.own + j, (c.own_ok >> j) & 1u, 0u) << (8 * j);
        }
        out.own_ok = c.own_ok;
        out.side = ldg_if(rc.side, c.side_ok, 256u);
    } else {
        out.bytes = 0;
        out.own_ok = 0;
        out.side = 256u;
    }
    rc.own += rc.W;
    rc.side += rc.W;
    ++rc.r;
    return out;
}

// One band: rows y0 .. y1 - 1 of the strip at x0 (FULL: all 128 columns exist and rows are
// 16-byte / 4-byte aligned, so each lane reads its four values with one load).
template <typename T, bool SEARCH, bool FULL, bool SAT>
__device__ __forceinline__ void band2d(const T *__restrict__ img, int Hy, int W, const Cols &c,
                                       int y0, int y1, const LaneShuffle &q, const KeyConsts &K,
                                       const float *__restrict__ table, uint32_t hist_s)
{
    // rows y0 - 1 .. y1 exist-or-absent; later rows (prefetch overshoot) read as absent
    RowCursor<T> rc = row_cursor(img, c, y0 - 1, min(y1 + 1, Hy), W);
    KeyRow ka = key_row<T, SEARCH>(next_row<FULL>(rc, c), K, table, q);
    KeyRow kb = key_row<T, SEARCH>(next_row<FULL>(rc, c), K, table, q);
    // raw-row ring: at the start of step y, q0 .. q3 (in rotation) hold rows y+1 .. y+4
    Raw<T> q0 = next_row<FULL>(rc, c);
    Raw<T> q1 = next_row<FULL>(rc, c);
    Raw<T> q2 = next_row<FULL>(rc, c);
    Raw<T> q3 = next_row<FULL>(rc, c);
    uint32_t Sp0, Sp1;
    sp_init<SAT>(ka, kb, Sp0, Sp1);

#define ECC_2D_STEP(QS)                                                                     \
    {                                                                                       \
        if (y >= y1) break;                                                                 \
        const KeyRow kd = key_row<T, SEARCH>(QS, K, table, q);                              \
        QS = next_row<FULL>(rc, c);                                                         \
        uint32_t c0, c1;                                                                    \
        c2_quad<SAT>(ka, kb, kd, kBias, Sp0, Sp1, c0, c1);                                  \
        hist_pair(kb.own0, c0, hist_s);                                            \
        hist_pair(kb.own1, c1, hist_s);                                            \
        ka = kb;                                                                            \
        kb = kd;                                                                            \
        ++y;                                                                                \
    }
    for (int y = y0; y < y1;) {
        ECC_2D_STEP(q0)
        ECC_2D_STEP(q1)
        ECC_2D_STEP(q2)
        ECC_2D_STEP(q3)
    }
#undef ECC_2D_STEP
}

template <typename T, int CAP, bool SEARCH>
__global__ void __launch_bounds__(kHardThreads, ECC_2D_MIN_BLOCKS) ecc_hard2d_kernel(const __grid_constant__
                                                                  HardParams<CAP> P)
{
    extern __shared__ int smem[];
    int *hist = smem;
    float *table = reinterpret_cast<float *>(smem + hist_words(P.H));
    block_setup(P, hist, table);

    const int64_t b = blockIdx.y;
    const T *__restrict__ img = static_cast<const T *>(P.img) + b * P.image_elems;
    const int lane = threadIdx.x & (kWarp - 1);
    const int warp = threadIdx.x >> 5;
    const KeyConsts K = key_consts(P);
    const LaneShuffle q = lane_shuffle(lane);
    const int Hy = (int)P.Hy, W = (int)P.W;
    const bool vec_ok = P.vec_ok != 0;
    const uint32_t hist_s = (uint32_t)__cvta_generic_to_shared(hist) - 4u * kKeyBase;

    // this warp's strip-rows [i, iend): warp g gets rows_per_task consecutive strip-rows
    // (strip-major), one more for the first rows_extra warps
    const uint32_t g = blockIdx.x * kHardWarps + warp;
    const uint32_t per = (uint32_t)P.rows_per_task, extra = (uint32_t)P.rows_extra;
    uint32_t i = g * per + min(g, extra);
    const uint32_t iend = i + per + (g < extra ? 1u : 0u);
    while (i < iend) {
        const int strip = (int)(i / (uint32_t)Hy);
        const int y0 = (int)(i - (uint32_t)strip * (uint32_t)Hy);
        const int y1 = min(Hy, y0 + (int)(iend - i));
        const Cols c = strip_cols(strip * kStrip, W, lane, vec_ok);
        constexpr bool SAT = CAP <= kSatMaxBins;
        if (c.full)  // warp-uniform
            band2d<T, SEARCH, true, SAT>(img, Hy, W, c, y0, y1, q, K, table, hist_s);
        else
            band2d<T, SEARCH, false, SAT>(img, Hy, W, c, y0, y1, q, K, table, hist_s);
        i += (uint32_t)(y1 - y0);
    }
    block_flush(P, hist, b);
}

// ----------------------------------------------------------------------------------------------
// 3-D kernel
// ----------------------------------------------------------------------------------------------
//
// Work: block task = (tile of 128 columns x 8 rows) x (chunk of rows_per_task planes), tile x
// fastest, then tile y, then chunk; block g of an image takes tasks g, g + G, ... Warp w owns row
// y0 + w, lane l columns x0 + 4l .. x0 + 4l + 3.

constexpr int kTileRows = kHardWarps;                // 8
constexpr int kKeyPitch = 136;                       // halves per shared row (272 bytes)
constexpr int kKeyRowsHalo = kTileRows + 2;          // rows y0-1 .. y0+8
constexpr int kKeyPlane = kKeyRowsHalo * kKeyPitch;  // halves per plane buffer
// Tile column c (-1 .. 128) sits at half index 4 + c of a shared row, so a lane's own four keys
// form one 8-byte-aligned word pair and its outer neighbours sit in the 4-byte words before and
// after it.

// The raw values one thread needs for one plane of the tile: its warp's row (four columns), one
// value of the two halo rows (thread t: row y0 - 1 or y0 + 8 by t >> 7, column x0 - 1 + (t & 127)),
// and for warp 0 one "extra" value: lanes 0..7 the column left of rows y0 .. y0+7, lanes 8..15
// the column right of them, lanes 16..19 the halo-row columns x0 + 127 and x0 + 128. Positions
// outside the grid read as NaN (f32) or 256 (u8), both meaning "never".
template <typename T>
struct HaloVal;
template <>
struct HaloVal<float> {
    using type = float;
    static __device__ __forceinline__ float none() { return qnan_f(); }
};
template <>
struct HaloVal<uint8_t> {
    using type = uint32_t;
    static __device__ __forceinline__ uint32_t none() { return 256u; }
};

template <typename T>
struct PlaneRaw {
    Raw<T> own;  // own.side unused
    typename HaloVal<T>::type hrow, extra;
};

struct PlaneCols {
    Cols own;    // own.own_ok also clears every column when the warp's row is outside the grid
    bool full;   // the warp's row exists and its four values load with one aligned load
    int hy, hx;  // halo-row position of this thread (clamped)
    bool h_ok;
    int ey, ex;  // extra position (warp 0, clamped)
    bool e_ok;
    int hrow_half;   // shared index of the halo-row key
    int extra_half;  // shared index of the extra key (or -1)
};

__device__ __forceinline__ PlaneCols plane_cols(int x0, int y0, int Hy, int W, int warp, int lane,
                                                bool vec_ok)
{
    PlaneCols pc;
    pc.own = strip_cols(x0, W, lane, vec_ok);
    const bool row_in = y0 + warp < Hy;
    if (!row_in) pc.own.own_ok = 0;
    pc.full = pc.own.full && row_in;
    const int t = threadIdx.x;
    const int hr = t >> 7;  // 0: row y0 - 1, 1: row y0 + 8
    const int hy = hr ? y0 + kTileRows : y0 - 1;
    const int hx = x0 - 1 + (t & 127);
    pc.h_ok = hy >= 0 && hy < Hy && hx >= 0 && hx < W;
    pc.hy = min(max(hy, 0), Hy - 1);
    pc.hx = min(max(hx, 0), W - 1);
    pc.hrow_half = (hr ? kKeyRowsHalo - 1 : 0) * kKeyPitch + 4 + (t & 127) - 1;
    int ey = 0, ex = 0, eh = -1;
    if (warp == 0 && lane < 20) {
        if (lane < 16) {
            ey = y0 + (lane & 7);
            ex = (lane < 8) ? x0 - 1 : x0 + kStrip;
            eh = (1 + (lane & 7)) * kKeyPitch + ((lane < 8) ? 3 : 4 + kStrip);
        } else {
            const int j = lane - 16;  // (row, column): (y0-1, x0+127), (y0-1, x0+128), ...
            ey = (j & 2) ? y0 + kTileRows : y0 - 1;
            ex = x0 + kStrip - 1 + (j & 1);
            eh = ((j & 2) ? kKeyRowsHalo - 1 : 0) * kKeyPitch + 4 + kStrip - 1 + (j & 1);
        }
    }
    pc.e_ok = eh >= 0 && ey >= 0 && ey < Hy && ex >= 0 && ex < W;
    pc.ey = min(max(ey, 0), Hy - 1);
    pc.ex = min(max(ex, 0), W - 1);
    pc.extra_half = eh;
    return pc;
}

// A thread's plane-by-plane reader: pointers into plane z that advance one plane per read;
// planes outside [0, D) read as absent.
template <typename T>
struct PlaneCursor {
    const T *own, *hrow, *extra;
    int64_t stride;
    int64_t z, D;
};

template <typename T>
__device__ __forceinline__ PlaneCursor<T> plane_cursor(const T *__restrict__ img,
                                                       const PlaneCols &pc, int y, int64_t z,
                                                       int64_t D, int Hy, int W)
{
    PlaneCursor<T> cur;
    cur.stride = (int64_t)Hy * W;
    const T *plane = img + z * cur.stride;
    cur.own = plane + (int64_t)min(y, Hy - 1) * W + pc.own.x;
    cur.hrow = plane + (int64_t)pc.hy * W + pc.hx;
    cur.extra = plane + (int64_t)pc.ey * W + pc.ex;
    cur.z = z;
    cur.D = D;
    return cur;
}

__device__ __forceinline__ void load_own4(const float *p, const PlaneCols &pc, Raw<float> &r)
{
    if (pc.full) {  // warp-uniform
        const float4 q = __ldg(reinterpret_cast<const float4 *>(p));
        r.v[0] = q.x;
        r.v[1] = q.y;
        r.v[2] = q.z;
        r.v[3] = q.w;
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) r.v[j] = ldg_if(p + j, (pc.own.own_ok >> j) & 1u, qnan_f());
    }
}

__device__ __forceinline__ void load_own4(const uint8_t *p, const PlaneCols &pc, Raw<uint8_t> &r)
{
    if (pc.full) {  // warp-uniform
        r.bytes = __ldg(reinterpret_cast<const unsigned int *>(p));
    } else {
        r.bytes = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            r.bytes |= ldg_if(p + j, (pc.own.own_ok >> j) & 1u, 0u) << (8 * j);
    }
    r.own_ok = pc.own.own_ok;
}

__device__ __forceinline__ void absent_own(Raw<float> &r)
{
#pragma unroll
    for (int j = 0; j < 4; ++j) r.v[j] = qnan_f();
}
__device__ __forceinline__ void absent_own(Raw<uint8_t> &r)
{
    r.bytes = 0;
    r.own_ok = 0;
}

template <typename T>
__device__ __forceinline__ PlaneRaw<T> next_plane(PlaneCursor<T> &cur, const PlaneCols &pc,
                                                  bool with_extra)
{
    using V = HaloVal<T>;
    PlaneRaw<T> p;
    p.extra = V::none();
    if ((uint64_t)cur.z < (uint64_t)cur.D) {  // block-uniform
        load_own4(cur.own, pc, p.own);
        p.hrow = ldg_if(cur.hrow, pc.h_ok, V::none());
        if (with_extra) p.extra = ldg_if(cur.extra, pc.e_ok, V::none());  // warp-uniform
    } else {
        absent_own(p.own);
        p.hrow = V::none();
    }
    cur.own += cur.stride;
    cur.hrow += cur.stride;
    cur.extra += cur.stride;
    ++cur.z;
    return p;
}

// Keys of a loaded plane into the shared buffer `dst`.
template <bool SEARCH>
__device__ __forceinline__ void store_plane_keys(const PlaneRaw<float> &p, const PlaneCols &pc,
                                                 const KeyConsts &K, const float *__restrict__ T,
                                                 int warp, int lane, bool with_extra,
                                                 uint16_t *dst)
{
    uint32_t k[6];
    if (SEARCH) {
#pragma unroll
        for (int j = 0; j < 4; ++j) k[j] = key_search_pattern(p.own.v[j], K.H, T);
        k[4] = key_search_pattern(p.hrow, K.H, T);
        k[5] = with_extra ? key_search_pattern(p.extra, K.H, T) : 0u;
    } else {
        uint32_t amb = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) k[j] = key_fast(p.own.v[j], K, amb);
        k[4] = key_fast(p.hrow, K, amb);
        k[5] = key_fast(p.extra, K, amb);  // NaN (key H) outside warp 0
        if (__any_sync(kFull, amb != 0)) {  // rare: a value within E of a threshold
            if (amb != 0) {
#pragma unroll
                for (int j = 0; j < 4; ++j) k[j] = key_fix(p.own.v[j], k[j], K.H, T);
                k[4] = key_fix(p.hrow, k[4], K.H, T);
                k[5] = key_fix(p.extra, k[5], K.H, T);
            }
        }
    }
    uint16_t *row = dst + (1 + warp) * kKeyPitch;
    *reinterpret_cast<uint2 *>(row + 4 + 4 * lane) =
        make_uint2(prmt(k[0], k[1], 0x5410), prmt(k[2], k[3], 0x5410));
    dst[pc.hrow_half] = (uint16_t)k[4];
    if (with_extra && pc.extra_half >= 0) dst[pc.extra_half] = (uint16_t)k[5];
}

template <bool SEARCH>
__device__ __forceinline__ void store_plane_keys(const PlaneRaw<uint8_t> &p, const PlaneCols &pc,
                                                 const KeyConsts &K, const float *__restrict__ T,
                                                 int warp, int lane, bool with_extra,
                                                 uint16_t *dst)
{
    const uint16_t *lut = reinterpret_cast<const uint16_t *>(T);
    const uint32_t never = kKeyBase + (uint32_t)K.H;
    Raw<uint8_t> r = p.own;
    r.side = 256u;  // no side value in the plane loads
    uint32_t own0, own1, unused;
    row_keys<SEARCH>(r, K, T, own0, own1, unused);
    uint16_t *row = dst + (1 + warp) * kKeyPitch;
    *reinterpret_cast<uint2 *>(row + 4 + 4 * lane) = make_uint2(own0, own1);
    dst[pc.hrow_half] = (uint16_t)(p.hrow < 256u ? (uint32_t)lut[p.hrow] : never);
    if (with_extra && pc.extra_half >= 0)
        dst[pc.extra_half] = (uint16_t)(p.extra < 256u ? (uint32_t)lut[p.extra] : never);
}

// The 3-D fold for one pair: c = cS - [k_{z+1} < k_z] c2(M_z) - [k_{z-1} <= k_z] c2(M_{z-1}),
// from cs = 1280 + c2(S_z), cn = c2(M_z), cm = c2(M_{z-1}) (plain fp16 values) and the keys of the
// voxel (k), of the voxel above (up_k) and below (dn_k). SAT: flags and products on the FMA pipe.
template <bool SAT>
__device__ __forceinline__ uint32_t fold3(uint32_t cs, uint32_t cn, uint32_t cm, uint32_t up_k,
                                          uint32_t dn_k, uint32_t k)
{
    if (SAT) {
        const uint32_t up = h2_sub_sat(k, up_k);                     // [k_{z+1} < k_z]
        const uint32_t dn = h2_sub_sat(h2_add(k, kOnePair), dn_k);  // [k_{z-1} <= k_z]
        uint32_t t;
        asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(t) : "r"(cm), "r"(dn));
        asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(t) : "r"(cn), "r"(up), "r"(t));
        return h2_sub(cs, t);
    }
    const uint32_t up = h2_lt_mask(up_k, k), dn = h2_le_mask(dn_k, k);
    return h2_sub(h2_sub(cs, cn & up), cm & dn);
}

// Buffer row r (= tile row r - 1, r = 0 .. 9) around the lane's four columns.
__device__ __forceinline__ KeyRow smem_key_row(const uint16_t *buf, int r, int lane)
{
    const uint16_t *row = buf + r * kKeyPitch;
    const uint2 own = *reinterpret_cast<const uint2 *>(row + 4 + 4 * lane);
    const uint32_t left = *reinterpret_cast<const uint32_t *>(row + 2 + 4 * lane);   // (x-2, x-1)
    const uint32_t right = *reinterpret_cast<const uint32_t *>(row + 8 + 4 * lane);  // (x+4, x+5)
    KeyRow k;
    k.own0 = own.x;
    k.own1 = own.y;
    k.L0 = prmt(left, own.x, 0x5432);
    k.R0 = prmt(own.x, own.y, 0x5432);
    k.R1 = prmt(own.y, right, 0x5432);
    return k;
}

template <typename T, int CAP, bool SEARCH>
__global__ void __launch_bounds__(kHardThreads, ECC_3D_MIN_BLOCKS) ecc_hard3d_kernel(const __grid_constant__
                                                                  HardParams<CAP> P)
{
    extern __shared__ int smem[];
    int *hist = smem;
    float *table = reinterpret_cast<float *>(smem + hist_words(P.H));
    __shared__ __align__(16) uint16_t keybuf[2][kKeyPlane];
    block_setup(P, hist, table);

    const int64_t b = blockIdx.y;
    const T *__restrict__ img = static_cast<const T *>(P.img) + b * P.image_elems;
    const int lane = threadIdx.x & (kWarp - 1);
    const int warp = threadIdx.x >> 5;
    const bool with_extra = (warp == 0);
    const int64_t Tn = P.tasks_per_image;
    const int64_t G = P.ctas_per_image;
    const KeyConsts K = key_consts(P);
    const bool vec_ok = P.vec_ok != 0;
    const int64_t D = P.D;
    const int Hy = (int)P.Hy, W = (int)P.W;
    const uint32_t kPlain = 0u;  // bias of the M stencil: plain c values
    constexpr bool SAT = CAP <= kSatMaxBins;
    const uint32_t hist_s = (uint32_t)__cvta_generic_to_shared(hist) - 4u * kKeyBase;

    for (int64_t t = blockIdx.x; t < Tn; t += G) {
        const int tx = (int)(t % P.tasks_x);
        const int64_t rest = t / P.tasks_x;
        const int ty = (int)(rest % P.tasks_y);
        const int64_t tz = rest / P.tasks_y;
        const int x0 = tx * kStrip;
        const int y0 = ty * kTileRows;
        const int64_t z0 = tz * P.rows_per_task;
        const int64_t z1 = min(z0 + (int64_t)P.rows_per_task, D);
        const PlaneCols pc = plane_cols(x0, y0, Hy, W, warp, lane, vec_ok);
        PlaneCursor<T> cur = plane_cursor(img, pc, y0 + warp, z0 - 1, D, Hy, W);

        // prologue: keys of planes z0 - 1 (buffer 0) and z0 (buffer 1); raw plane z0 + 1 in flight
        __syncthreads();  // the previous task's readers are done with both buffers
        {
            const PlaneRaw<T> pm = next_plane(cur, pc, with_extra);
            const PlaneRaw<T> p0 = next_plane(cur, pc, with_extra);
            store_plane_keys<SEARCH>(pm, pc, K, table, warp, lane, with_extra, keybuf[0]);
            store_plane_keys<SEARCH>(p0, pc, K, table, warp, lane, with_extra, keybuf[1]);
        }
        PlaneRaw<T> pnext = next_plane(cur, pc, with_extra);
        __syncthreads();
        uint32_t cm0, cm1;        // c2(M_{z-1}) at the lane's pixels (plain values)
        uint32_t below0, below1;  // keys of plane z - 1 at the lane's pixels
        KeyRow ca = smem_key_row(keybuf[1], warp, lane);
        KeyRow cb = smem_key_row(keybuf[1], warp + 1, lane);
        KeyRow cd = smem_key_row(keybuf[1], warp + 2, lane);
        {
            const KeyRow pa = smem_key_row(keybuf[0], warp, lane);
            const KeyRow pb = smem_key_row(keybuf[0], warp + 1, lane);
            const KeyRow pd = smem_key_row(keybuf[0], warp + 2, lane);
            const KeyRow ma = max_rows(pa, ca), mb = max_rows(pb, cb), md = max_rows(pd, cd);
            uint32_t s0, s1;
            sp_init<SAT>(ma, mb, s0, s1);
            c2_quad<SAT>(ma, mb, md, kPlain, s0, s1, cm0, cm1);
            below0 = pb.own0;
            below1 = pb.own1;
        }
        __syncthreads();  // buffer 0 is read; plane z0 + 1 may replace it

        // One barrier per plane: plane z + 1 goes to buffer (z - z0) & 1, which was last read
        // two steps before, and every warp has passed the previous step's barrier since. The loop
        // is unrolled by two so that the buffer and the carried rows need no register moves.
#define ECC_3D_STEP(NBUF, ZZ)                                                               \
    {                                                                                       \
        store_plane_keys<SEARCH>(pnext, pc, K, table, warp, lane, with_extra, NBUF);        \
        if ((ZZ) + 2 <= z1) pnext = next_plane(cur, pc, with_extra); /* block-uniform */    \
        __syncthreads();                                                                    \
        const KeyRow na = smem_key_row(NBUF, warp, lane);                                   \
        const KeyRow nb = smem_key_row(NBUF, warp + 1, lane);                               \
        const KeyRow nd = smem_key_row(NBUF, warp + 2, lane);                               \
        uint32_t s0, s1, cs0, cs1, cn0, cn1;                                                \
        sp_init<SAT>(ca, cb, s0, s1);                                                       \
        c2_quad<SAT>(ca, cb, cd, kBias, s0, s1, cs0, cs1);                                  \
        const KeyRow ma = max_rows(ca, na), mb = max_rows(cb, nb), md = max_rows(cd, nd);   \
        sp_init<SAT>(ma, mb, s0, s1);                                                       \
        c2_quad<SAT>(ma, mb, md, kPlain, s0, s1, cn0, cn1);                                 \
        /* c = cS - [k_{z+1} < k_z] c2(M_z) - [k_{z-1} <= k_z] c2(M_{z-1}) */                \
        hist_pair(cb.own0, fold3<SAT>(cs0, cn0, cm0, nb.own0, below0, cb.own0), hist_s);   \
        hist_pair(cb.own1, fold3<SAT>(cs1, cn1, cm1, nb.own1, below1, cb.own1), hist_s);   \
        cm0 = cn0;                                                                          \
        cm1 = cn1;                                                                          \
        below0 = cb.own0;                                                                   \
        below1 = cb.own1;                                                                   \
        ca = na;                                                                            \
        cb = nb;                                                                            \
        cd = nd;                                                                            \
    }
        for (int64_t z = z0; z < z1; z += 2) {
            ECC_3D_STEP(keybuf[0], z)
            if (z + 1 >= z1) break;
            ECC_3D_STEP(keybuf[1], z + 1)
        }
#undef ECC_3D_STEP
    }
    block_flush(P, hist, b);
}

// ----------------------------------------------------------------------------------------------
// Running sum over bins: out[b][k] = sum_{j <= k} hist[b][j]  (one block per image)
// ----------------------------------------------------------------------------------------------
constexpr int kScanThreads = 1024;

__global__ void __launch_bounds__(kScanThreads) ecc_bin_scan_kernel(int64_t *out, int H)
{
    __shared__ long long warp_sums[kScanThreads / kWarp];
    __shared__ long long carry;
    int64_t *row = out + (int64_t)blockIdx.x * H;
    const int lane = threadIdx.x & (kWarp - 1);
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    for (int base = 0; base < H; base += kScanThreads) {
        const int i = base + threadIdx.x;
        long long v = (i < H) ? (long long)row[i] : 0;
#pragma unroll
        for (int o = 1; o < kWarp; o <<= 1) {
            long long n = __shfl_up_sync(kFull, v, o);
            if (lane >= o) v += n;
        }
        if (lane == kWarp - 1) warp_sums[warp] = v;
        __syncthreads();
        if (warp == 0) {
            long long s = warp_sums[lane];
#pragma unroll
            for (int o = 1; o < kWarp; o <<= 1) {
                long long n = __shfl_up_sync(kFull, s, o);
                if (lane >= o) s += n;
            }
            warp_sums[lane] = s;
        }
        __syncthreads();
        const long long before = carry + (warp > 0 ? warp_sums[warp - 1] : 0);
        if (i < H) row[i] = (int64_t)(before + v);
        __syncthreads();
        if (threadIdx.x == kScanThreads - 1) carry = before + v;
        __syncthreads();
    }
}

// ----------------------------------------------------------------------------------------------
// Host-side launch (called from the C ABI after validation)
// ----------------------------------------------------------------------------------------------

static int num_sms()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) n = 148;
    return n;
}

// Planes per 3-D block task: the power of two from 32 up that maximises the useful fraction of
// the block time -- tasks shared evenly over the blocks (the busiest block sets the time) times
// R / (R + 2) for the two prologue planes of each task.
static int64_t pick_chunk(int64_t D, int64_t tiles, int64_t blocks)
{
    int64_t best = 32;
    double best_eff = -1.0;
    for (int64_t R = 32;; R *= 2) {
        const int64_t tasks = tiles * ((D + R - 1) / R);
        const double per = (double)tasks / (double)blocks;
        const double busiest = (double)((tasks + blocks - 1) / blocks);
        const double eff = (per / busiest) * ((double)R / (double)(R + 2));
        if (eff > best_eff + 1e-9) {
            best_eff = eff;
            best = R;
        }
        if (R >= D) break;
    }
    return best;
}

template <typename T, int CAP, bool SEARCH>
static cudaError_t launch_hard(const HardPlan &pl, cudaStream_t s)
{
    HardParams<CAP> P;
    P.img = pl.img;
    P.out = pl.out;
    P.D = pl.D;
    P.Hy = pl.Hy;
    P.W = pl.W;
    P.image_elems = pl.D * pl.Hy * pl.W;
    P.H = pl.H;
    P.key_mode = pl.key_mode;
    P.key_a = pl.key_a;
    P.key_b = pl.key_b;
    P.key_clo = pl.key_clo;
    P.key_chi = pl.key_chi;
    P.vec_ok = pl.vec_ok;
    P.sign = pl.sign;
    const int ntab = (pl.dtype == ECC_U8) ? 128 : pl.H + 2;  // u8: 256 uint16 in 128 floats
    P.table_len = ntab;
    for (int i = 0; i < ntab; ++i) P.table[i] = pl.table[i];
    for (int i = ntab; i < CAP + 2; ++i) P.table[i] = 0.0f;

    const int sms = num_sms();
    const int64_t strips = (pl.W + kStrip - 1) / kStrip;
    const int per_sm = pl.ndim == 2 ? ECC_2D_MIN_BLOCKS : ECC_3D_MIN_BLOCKS;
    const int64_t resident = (int64_t)sms * per_sm;  // blocks that fit at once
    // blocks per image: the resident blocks shared out over the batch
    int64_t per_image = (resident + pl.batch - 1) / pl.batch;
    if (pl.ndim == 2) {
        // contiguous strip-row ranges, at least 32 rows per warp
        const int64_t N = strips * pl.Hy;
        if (N >= ((int64_t)1 << 31)) return cudaErrorInvalidValue;  // 32-bit row arithmetic
        const int64_t need = (N + 32 * kHardWarps - 1) / (32 * kHardWarps);
        if (per_image > need) per_image = need;
        if (per_image < 1) per_image = 1;
        const int64_t G = per_image * kHardWarps;
        P.rows_per_task = (int)(N / G);
        P.rows_extra = (int)(N % G);
        P.tasks_x = (int)strips;
        P.tasks_y = (int)pl.Hy;
        P.tasks_z = 1;
        P.tasks_per_image = N;
    } else {
        const int64_t tiles_y = (pl.Hy + kTileRows - 1) / kTileRows;
        const int64_t tiles = strips * tiles_y;
        if (per_image > tiles * pl.D) per_image = tiles * pl.D;
        const int64_t R = pick_chunk(pl.D, tiles, per_image);
        P.rows_per_task = (int)R;
        P.tasks_x = (int)strips;
        P.tasks_y = (int)tiles_y;
        P.tasks_z = (int)((pl.D + R - 1) / R);
        P.tasks_per_image = (int64_t)P.tasks_x * P.tasks_y * P.tasks_z;
        if (per_image > P.tasks_per_image) per_image = P.tasks_per_image;
    }
    if (per_image < 1) per_image = 1;
    P.ctas_per_image = (int)per_image;

    const size_t smem =
        (size_t)hist_words(pl.H) * sizeof(int) + (size_t)(CAP + 2) * sizeof(float);
    dim3 grid((unsigned)per_image, (unsigned)pl.batch);
    if (pl.ndim == 2) {
        ecc_hard2d_kernel<T, CAP, SEARCH><<<grid, kHardThreads, smem, s>>>(P);
    } else {
        ecc_hard3d_kernel<T, CAP, SEARCH><<<grid, kHardThreads, smem, s>>>(P);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || !pl.scan) return e;
    return hard_scan(pl.out, pl.H, pl.batch, s);
}

cudaError_t hard_scan(int64_t *out, int H, int64_t batch, cudaStream_t s)
{
    ecc_bin_scan_kernel<<<(unsigned)batch, kScanThreads, 0, s>>>(out, H);
    return cudaGetLastError();
}

cudaError_t hard_run(const HardPlan &pl, cudaStream_t s)
{
    if (pl.dtype == ECC_U8) {
        if (pl.H <= 256) return launch_hard<uint8_t, 256, false>(pl, s);
        if (pl.H <= 1024) return launch_hard<uint8_t, 1024, false>(pl, s);
        return launch_hard<uint8_t, ECC_MAX_NBINS, false>(pl, s);
    }
    if (pl.key_mode == kKeySearch) return launch_hard<float, ECC_MAX_NBINS, true>(pl, s);
    if (pl.H <= 256) return launch_hard<float, 256, false>(pl, s);
    if (pl.H <= 1024) return launch_hard<float, 1024, false>(pl, s);
    return launch_hard<float, ECC_MAX_NBINS, false>(pl, s);
}

}  // namespace ecc
