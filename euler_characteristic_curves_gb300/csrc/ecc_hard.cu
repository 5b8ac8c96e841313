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
// 128 columns x 32 rows and walks z; each plane's keys are computed once into a shared tile with a
// one-pixel halo. A warp owns eight consecutive rows: it builds the rows around them from the
// shared keys of planes z and z + 1 once per plane and reuses them down its rows, so the row
// building, the max rows and the first-row flags are paid once per eight rows. The raw values of
// the next plane are loaded into registers one plane ahead.
#include <cuda.h>  // CUtensorMap and its enums (the encoder is fetched through the runtime)
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ecc_internal.cuh"
#include "ecc_keys.cuh"

namespace ecc {

__device__ unsigned g_hard_error;  // device error word of the hard kernels (DeviceErrorBit)

// A pair of key patterns (0x6400 + k each) and its contributions into the block histogram; the
// debug build first checks both bins against [0, H].
__device__ __forceinline__ void hist_pair_h(uint32_t keys, uint32_t cv, uint32_t hist_s, int H)
{
    const int lo = (int)(keys & 0xffffu) - (int)kKeyBase, hi = (int)(keys >> 16) - (int)kKeyBase;
    if (bounds_ok(&g_hard_error, lo >= 0 && lo <= H && hi >= 0 && hi <= H, kErrHardBin))
        hist_pair(keys, cv, hist_s);
}

constexpr int kHardThreads = 256;
constexpr int kHardWarps = kHardThreads / kWarp;
constexpr int kStrip = 128;  // columns per warp strip / block tile
// Tables of at most this many bins take the stencil's flags from the FMA pipe (exact for keys
// up to 1024; see flag_lt / flag_le), larger ones from fp16 compares.
constexpr int kSatMaxBins = 1024;

// Resident blocks per SM the kernels are compiled for (register budget 65536 / (threads * blocks);
// 2-D blocks have 256 threads, 3-D blocks k3Threads).
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

// The image's only block (P.direct) writes the curve itself: warp w of the nw warps takes the
// contiguous bins [w per, (w + 1) per), adds the totals of the warps before it, and walks its
// bins 32 at a time with a shuffle scan and a running carry.
__device__ __forceinline__ void block_store_curve(const int *hist, int H, int64_t *dst)
{
    __shared__ long long warp_total[32];
    const int lane = threadIdx.x & (kWarp - 1), warp = threadIdx.x >> 5;
    const int nw = blockDim.x >> 5;
    const int per = (H + nw - 1) / nw;
    const int lo = min(H, warp * per), hi = min(H, lo + per);
    long long t = 0;
    for (int i = lo + lane; i < hi; i += kWarp) t += hist[i];
#pragma unroll
    for (int o = kWarp / 2; o > 0; o >>= 1) t += __shfl_xor_sync(kFull, t, o);
    if (lane == 0) warp_total[warp] = t;
    __syncthreads();
    long long carry = 0;
    for (int w = 0; w < warp; ++w) carry += warp_total[w];
    for (int c = lo; c < hi; c += kWarp) {  // warp-uniform bounds
        const int i = c + lane;
        long long v = i < hi ? (long long)hist[i] : 0;
#pragma unroll
        for (int o = 1; o < kWarp; o <<= 1) {
            const long long n = __shfl_up_sync(kFull, v, o);
            if (lane >= o) v += n;
        }
        if (i < hi) dst[i] = (int64_t)(carry + v);
        carry += __shfl_sync(kFull, v, kWarp - 1);
    }
}

// The block adds the running sum of its histogram into the curve dst (zeroed before the launch):
// the running sum is linear, so the blocks' running sums add up to the running sum of the
// image's histogram, and no scan launch follows. Warp w takes the contiguous bins
// [w per, (w + 1) per) as in block_store_curve; bins whose running sum is 0 add nothing.
__device__ __forceinline__ void block_add_curve(const int *hist, int H, int64_t *dst)
{
    __shared__ long long warp_total[32];
    const int lane = threadIdx.x & (kWarp - 1), warp = threadIdx.x >> 5;
    const int nw = blockDim.x >> 5;
    const int per = (H + nw - 1) / nw;
    const int lo = min(H, warp * per), hi = min(H, lo + per);
    long long t = 0;
    for (int i = lo + lane; i < hi; i += kWarp) t += hist[i];
#pragma unroll
    for (int o = kWarp / 2; o > 0; o >>= 1) t += __shfl_xor_sync(kFull, t, o);
    if (lane == 0) warp_total[warp] = t;
    __syncthreads();
    long long carry = 0;
    for (int w = 0; w < warp; ++w) carry += warp_total[w];
    unsigned long long *d = reinterpret_cast<unsigned long long *>(dst);
    for (int c = lo; c < hi; c += kWarp) {  // warp-uniform bounds
        const int i = c + lane;
        long long v = i < hi ? (long long)hist[i] : 0;
#pragma unroll
        for (int o = 1; o < kWarp; o <<= 1) {
            const long long n = __shfl_up_sync(kFull, v, o);
            if (lane >= o) v += n;
        }
        if (i < hi && carry + v != 0) atomicAdd(d + i, (unsigned long long)(carry + v));
        carry += __shfl_sync(kFull, v, kWarp - 1);
    }
}

// DIRECT_OK: the kernel may run with P.direct or P.prefix (the 2-D kernels; the 3-D kernel
// always flushes its histogram).
template <bool DIRECT_OK, int CAP>
__device__ __forceinline__ void block_flush(const HardParams<CAP> &P, const int *hist, int64_t b)
{
    __syncthreads();
    if (DIRECT_OK && P.direct) {  // grid-uniform
        block_store_curve(hist, P.H, P.out + b * (int64_t)P.H);
        return;
    }
    if (DIRECT_OK && P.prefix) {  // grid-uniform
        block_add_curve(hist, P.H, P.out + b * (int64_t)P.H);
        return;
    }
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
    key_pairs(K);
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
// Work: an image's rows are split into R equal row ranges, and warp g of the image's blocks
// (blockIdx.y = image) walks strip g % strips over row range g / strips as one band, so the only
// repeated work is the two rows around each band. Consecutive warps of a block take adjacent
// strips of the same rows at the same time, so the column a warp reads just left or right of its
// strip was fetched by its neighbour moments before and comes from L1: only the block's outer
// strip edges reach L2 (with strip-major ranges per warp, these side columns cost 14% extra DRAM
// reads on 8192^2).

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
    if ((unsigned)rc.r < (unsigned)rc.rlim &&  // warp-uniform
        bounds_ok(&g_hard_error, !FULL || c.x + 4 <= rc.W, kErrHardRow)) {
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
    if ((unsigned)rc.r < (unsigned)rc.rlim &&  // warp-uniform
        bounds_ok(&g_hard_error, !FULL || c.x + 4 <= rc.W, kErrHardRow)) {
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
        hist_pair_h(kb.own0, c0, hist_s, K.H);                                     \
        hist_pair_h(kb.own1, c1, hist_s, K.H);                                     \
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

    // this warp's band: strip g % strips, rows [r Hy / R, (r + 1) Hy / R) with r = g / strips
    const uint32_t g = blockIdx.x * kHardWarps + warp;
    const uint32_t strips = (uint32_t)P.tasks_x, R = (uint32_t)P.rows_per_task;
    if (g < strips * R) {  // warp-uniform; fewer than `strips` warps of the grid stay idle
        const uint32_t strip = g % strips, r = g / strips;
        const int y0 = (int)((uint64_t)r * (uint32_t)Hy / R);
        const int y1 = (int)((uint64_t)(r + 1) * (uint32_t)Hy / R);
        const Cols c = strip_cols((int)strip * kStrip, W, lane, vec_ok);
        constexpr bool SAT = CAP <= kSatMaxBins;
        if (c.full)  // warp-uniform
            band2d<T, SEARCH, true, SAT>(img, Hy, W, c, y0, y1, q, K, table, hist_s);
        else
            band2d<T, SEARCH, false, SAT>(img, Hy, W, c, y0, y1, q, K, table, hist_s);
    }
    block_flush<true>(P, hist, b);
}

// ----------------------------------------------------------------------------------------------
// 3-D kernel
// ----------------------------------------------------------------------------------------------
//
// Work: block task = (tile of 128 columns x kTileRows rows) x (chunk of rows_per_task planes),
// tile x fastest, then tile y, then chunk; block g of an image takes tasks g, g + G, ... Warp w
// owns the k3Rows rows y0 + w k3Rows .. y0 + (w + 1) k3Rows - 1 of the tile, lane l columns
// x0 + 4l .. x0 + 4l + 3 of each. A warp builds the rows around its own rows once per plane and
// reuses them down its rows, like the 2-D bands. Of the shapes measured (one to eight rows per
// warp, two to eight warps per block), eight rows in four-warp blocks, three blocks per SM, was
// the fastest.

#ifndef ECC_3D_ROWS
#define ECC_3D_ROWS 8
#endif
#ifndef ECC_3D_WARPS
#define ECC_3D_WARPS 4
#endif
constexpr int k3Rows = ECC_3D_ROWS;    // rows per warp
constexpr int k3Warps = ECC_3D_WARPS;  // warps per block
constexpr int k3Threads = k3Warps * kWarp;
constexpr int kTileRows = k3Warps * k3Rows;
constexpr int kKeyPitch = 136;                       // halves per shared row (272 bytes)
constexpr int kKeyRowsHalo = kTileRows + 2;          // rows y0 - 1 .. y0 + kTileRows
constexpr int kKeyPlane = kKeyRowsHalo * kKeyPitch;  // halves per plane buffer
// Tile column c (-1 .. 128) sits at half index 4 + c of a shared row, so a lane's own four keys
// form one 8-byte-aligned word pair and its outer neighbours sit in the 4-byte words before and
// after it.
static_assert(kKeyPitch >= 4 + kStrip + 1 && kKeyPitch % 4 == 0, "shared key row layout");

// The halo of a plane: the rows above and below the tile (130 columns each, x0 - 1 .. x0 + 128),
// then the columns left and right of the tile (kTileRows rows each). Thread t loads halo items
// t, t + k3Threads, ... ("slots"); only the last slot is partly empty.
constexpr int kHaloRowItems = kStrip + 2;
constexpr int kHaloItems = 2 * kHaloRowItems + 2 * kTileRows;
constexpr int kHaloSlots = (kHaloItems + k3Threads - 1) / k3Threads;

__device__ __forceinline__ void halo_item(int i, int x0, int y0, int &y, int &x, int &half)
{
    if (i < 2 * kHaloRowItems) {
        const int below = i >= kHaloRowItems;
        const int c = i - below * kHaloRowItems - 1;  // -1 .. 128
        y = below ? y0 + kTileRows : y0 - 1;
        x = x0 + c;
        half = (below ? kKeyRowsHalo - 1 : 0) * kKeyPitch + 4 + c;
    } else {
        const int j = i - 2 * kHaloRowItems;
        const int right = j >= kTileRows;
        const int r = j - right * kTileRows;
        y = y0 + r;
        x = right ? x0 + kStrip : x0 - 1;
        half = (1 + r) * kKeyPitch + (right ? 4 + kStrip : 3);
    }
}

// Whether some lane of `warp` has an item in halo slot s (warp-uniform): every lane has one in
// all but the last slot, which the compiler sees as a constant.
__device__ __forceinline__ bool slot_active(int s, int warp)
{
    return s + 1 < kHaloSlots || s * k3Threads + warp * kWarp < kHaloItems;
}
// Whether this thread has an item in halo slot s.
__device__ __forceinline__ bool slot_item(int s, const int *h_half)
{
    return s + 1 < kHaloSlots || h_half[s] >= 0;
}

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

// The raw values one thread loads from one plane: its warp's rows (four columns each; side
// unused) and its halo items. Absent slots and positions outside the grid read as NaN (f32) or
// 256 (u8), both meaning "never".
template <typename T>
struct PlaneRaw {
    Raw<T> own[k3Rows];
    typename HaloVal<T>::type halo[kHaloSlots];
};

// A thread's positions within a task's tile (fixed for the task).
struct TileCols {
    Cols own;          // own.own_ok: the lane's columns inside the grid
    uint32_t rows_in;  // bit i: the warp's row i exists
    int hy[kHaloSlots], hx[kHaloSlots];  // halo item positions, clamped into the grid
    bool h_ok[kHaloSlots];               // the item exists and lies inside the grid
    int h_half[kHaloSlots];              // shared index of the item (-1: no item)
};

__device__ __forceinline__ TileCols tile_cols(int x0, int y0, int Hy, int W, int warp, int lane,
                                              bool vec_ok)
{
    TileCols tc;
    tc.own = strip_cols(x0, W, lane, vec_ok);
    tc.rows_in = 0;
#pragma unroll
    for (int i = 0; i < k3Rows; ++i)
        if (y0 + warp * k3Rows + i < Hy) tc.rows_in |= 1u << i;
#pragma unroll
    for (int s = 0; s < kHaloSlots; ++s) {
        const int i = (int)threadIdx.x + s * k3Threads;
        int y = -1, x = -1, half = -1;
        if (i < kHaloItems) halo_item(i, x0, y0, y, x, half);
        tc.h_ok[s] = half >= 0 && y >= 0 && y < Hy && x >= 0 && x < W;
        tc.hy[s] = min(max(y, 0), Hy - 1);
        tc.hx[s] = min(max(x, 0), W - 1);
        tc.h_half[s] = half;
    }
    return tc;
}

// A thread's plane-by-plane reader: pointers into plane z that advance one plane per read;
// planes outside [0, D) read as absent.
template <typename T>
struct TileCursor {
    const T *own;  // the lane's first column in the warp's first row (row clamped into the grid)
    const T *halo[kHaloSlots];
    int64_t stride, z, D;
    int W;
};

template <typename T>
__device__ __forceinline__ TileCursor<T> tile_cursor(const T *__restrict__ img, const TileCols &tc,
                                                     int y, int64_t z, int64_t D, int Hy, int W)
{
    TileCursor<T> cur;
    cur.stride = (int64_t)Hy * W;
    const T *plane = img + z * cur.stride;
    cur.own = plane + (int64_t)min(y, Hy - 1) * W + tc.own.x;
#pragma unroll
    for (int s = 0; s < kHaloSlots; ++s) cur.halo[s] = plane + (int64_t)tc.hy[s] * W + tc.hx[s];
    cur.z = z;
    cur.D = D;
    cur.W = W;
    return cur;
}

// Four values of one row (`full`: one aligned load; else per-column predicated loads).
__device__ __forceinline__ void load_own4(const float *p, const Cols &c, bool full,
                                          Raw<float> &r)
{
    if (full) {  // warp-uniform
        const float4 q = __ldg(reinterpret_cast<const float4 *>(p));
        r.v[0] = q.x;
        r.v[1] = q.y;
        r.v[2] = q.z;
        r.v[3] = q.w;
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) r.v[j] = ldg_if(p + j, (c.own_ok >> j) & 1u, qnan_f());
    }
}

__device__ __forceinline__ void load_own4(const uint8_t *p, const Cols &c, bool full,
                                          Raw<uint8_t> &r)
{
    if (full) {  // warp-uniform
        r.bytes = __ldg(reinterpret_cast<const unsigned int *>(p));
    } else {
        r.bytes = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            r.bytes |= ldg_if(p + j, (c.own_ok >> j) & 1u, 0u) << (8 * j);
    }
    r.own_ok = c.own_ok;
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
__device__ __forceinline__ PlaneRaw<T> next_plane(TileCursor<T> &cur, const TileCols &tc,
                                                  int warp)
{
    using V = HaloVal<T>;
    PlaneRaw<T> p;
    const bool in = (uint64_t)cur.z < (uint64_t)cur.D;  // block-uniform
    if (in && tc.own.full && tc.rows_in == (1u << k3Rows) - 1u) {  // warp-uniform common case
#pragma unroll
        for (int i = 0; i < k3Rows; ++i)
            load_own4(cur.own + (int64_t)i * cur.W, tc.own, true, p.own[i]);
    } else {
#pragma unroll
        for (int i = 0; i < k3Rows; ++i) {
            if (in && ((tc.rows_in >> i) & 1u))  // warp-uniform
                load_own4(cur.own + (int64_t)i * cur.W, tc.own, tc.own.full, p.own[i]);
            else
                absent_own(p.own[i]);
        }
    }
#pragma unroll
    for (int s = 0; s < kHaloSlots; ++s) {
        p.halo[s] = V::none();
        if (slot_active(s, warp)) p.halo[s] = ldg_if(cur.halo[s], in && tc.h_ok[s], V::none());
    }
    cur.own += cur.stride;
#pragma unroll
    for (int s = 0; s < kHaloSlots; ++s) cur.halo[s] += cur.stride;
    ++cur.z;
    return p;
}

// Keys of a loaded plane into the shared buffer `dst`.
template <bool SEARCH>
__device__ __forceinline__ void store_plane_keys(const PlaneRaw<float> &p, const TileCols &tc,
                                                 const KeyConsts &K, const float *__restrict__ T,
                                                 int warp, int lane, uint16_t *dst)
{
    uint32_t k[k3Rows][4], h[kHaloSlots];
    if (SEARCH) {
#pragma unroll
        for (int i = 0; i < k3Rows; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) k[i][j] = key_search_pattern(p.own[i].v[j], K.H, T);
#pragma unroll
        for (int s = 0; s < kHaloSlots; ++s)
            h[s] = slot_active(s, warp) ? key_search_pattern(p.halo[s], K.H, T) : 0u;
    } else {
        // ambiguity flags per group of kFixRows rows (the halo items join the first group), so
        // that the rare fix-up only revisits the groups that need it
        constexpr int kFixRows = k3Rows >= 2 ? 2 : 1;
        constexpr int kGroups = k3Rows / kFixRows;
        uint32_t amb[kGroups];
#pragma unroll
        for (int q = 0; q < kGroups; ++q) amb[q] = 0;
#pragma unroll
        for (int i = 0; i < k3Rows; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) k[i][j] = key_fast(p.own[i].v[j], K, amb[i / kFixRows]);
#pragma unroll
        for (int s = 0; s < kHaloSlots; ++s) {
            h[s] = kKeyBase + (uint32_t)K.H;  // "never" in warps without an item in slot s
            if (slot_active(s, warp)) h[s] = key_fast(p.halo[s], K, amb[0]);
        }
        uint32_t any = 0;
#pragma unroll
        for (int q = 0; q < kGroups; ++q) any |= amb[q];
        if (__any_sync(kFull, any != 0)) {  // rare: a value within E of a threshold
#pragma unroll
            for (int q = 0; q < kGroups; ++q) {
                if (amb[q] != 0) {
#pragma unroll
                    for (int i = q * kFixRows; i < (q + 1) * kFixRows; ++i)
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            k[i][j] = key_fix(p.own[i].v[j], k[i][j], K.H, T);
                    if (q == 0) {
#pragma unroll
                        for (int s = 0; s < kHaloSlots; ++s)
                            if (slot_active(s, warp)) h[s] = key_fix(p.halo[s], h[s], K.H, T);
                    }
                }
            }
        }
    }
    uint16_t *row = dst + (1 + warp * k3Rows) * kKeyPitch + 4 + 4 * lane;
#pragma unroll
    for (int i = 0; i < k3Rows; ++i)
        *reinterpret_cast<uint2 *>(row + i * kKeyPitch) =
            make_uint2(prmt(k[i][0], k[i][1], 0x5410), prmt(k[i][2], k[i][3], 0x5410));
#pragma unroll
    for (int s = 0; s < kHaloSlots; ++s)
        if (slot_item(s, tc.h_half)) dst[tc.h_half[s]] = (uint16_t)h[s];
}

template <bool SEARCH>
__device__ __forceinline__ void store_plane_keys(const PlaneRaw<uint8_t> &p, const TileCols &tc,
                                                 const KeyConsts &K, const float *__restrict__ T,
                                                 int warp, int lane, uint16_t *dst)
{
    const uint16_t *lut = reinterpret_cast<const uint16_t *>(T);
    const uint32_t never = kKeyBase + (uint32_t)K.H;
    uint16_t *row = dst + (1 + warp * k3Rows) * kKeyPitch + 4 + 4 * lane;
#pragma unroll
    for (int i = 0; i < k3Rows; ++i) {
        Raw<uint8_t> r = p.own[i];
        r.side = 256u;  // no side value in the plane loads
        uint32_t own0, own1, unused;
        row_keys<SEARCH>(r, K, T, own0, own1, unused);
        *reinterpret_cast<uint2 *>(row + i * kKeyPitch) = make_uint2(own0, own1);
    }
#pragma unroll
    for (int s = 0; s < kHaloSlots; ++s)
        if (slot_item(s, tc.h_half))
            dst[tc.h_half[s]] =
                (uint16_t)(p.halo[s] < 256u ? (uint32_t)lut[p.halo[s]] : never);
}

// The 3-D fold for one pair: 1280 + c with c = cS - [k_{z+1} < k_z] c2(M_z) - [k_{z-1} <= k_z]
// c2(M_{z-1}), from cn = c2(M_z), cm = c2(M_{z-1}) (plain fp16 values), cs = c2(S_z) (SAT: plain;
// else 1280 + c2(S_z)) and the keys of the voxel (k), of the voxel above (up_k) and below (dn_k).
// SAT: flags and products on the FMA pipe, the bias entering through the first product (every
// value is an integer below 2048 in magnitude, so each fp16 step is exact).
constexpr uint32_t kNegBias = 0xE500E500u;  // (-1280, -1280)
template <bool SAT>
__device__ __forceinline__ uint32_t fold3(uint32_t cs, uint32_t cn, uint32_t cm, uint32_t up_k,
                                          uint32_t dn_k, uint32_t k)
{
    if (SAT) {
        const uint32_t up = h2_sub_sat(k, up_k);                     // [k_{z+1} < k_z]
        const uint32_t dn = h2_sub_sat(h2_add(k, kOnePair), dn_k);  // [k_{z-1} <= k_z]
        uint32_t t;
        asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(t) : "r"(cm), "r"(dn), "r"(kNegBias));
        asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(t) : "r"(cn), "r"(up), "r"(t));
        return h2_sub(cs, t);
    }
    const uint32_t up = h2_lt_mask(up_k, k), dn = h2_le_mask(dn_k, k);
    return h2_sub(h2_sub(cs, cn & up), cm & dn);
}

// Buffer row r (= tile row r - 1, r = 0 .. kTileRows + 1) around the lane's four columns.
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
__global__ void __launch_bounds__(k3Threads, ECC_3D_MIN_BLOCKS) ecc_hard3d_kernel(const __grid_constant__
                                                                  HardParams<CAP> P)
{
    extern __shared__ int smem[];
    int *hist = smem;
    float *table = reinterpret_cast<float *>(smem + hist_words(P.H));
    __shared__ __align__(16) uint16_t keybuf[3][kKeyPlane];
    block_setup(P, hist, table);

    const int64_t b = blockIdx.y;
    const T *__restrict__ img = static_cast<const T *>(P.img) + b * P.image_elems;
    const int lane = threadIdx.x & (kWarp - 1);
    const int warp = threadIdx.x >> 5;
    const int r0 = warp * k3Rows;  // buffer row of the row above the warp's first row
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
        const TileCols tc = tile_cols(x0, y0, Hy, W, warp, lane, vec_ok);
        TileCursor<T> cur = tile_cursor(img, tc, y0 + r0, z0 - 1, D, Hy, W);

        // prologue: keys of planes z0 - 1 (buffer 0) and z0 (buffer 1); raw plane z0 + 1 in flight
        __syncthreads();  // the previous task's readers are done with both buffers
        {
            const PlaneRaw<T> pm = next_plane(cur, tc, warp);
            const PlaneRaw<T> p0 = next_plane(cur, tc, warp);
            store_plane_keys<SEARCH>(pm, tc, K, table, warp, lane, keybuf[0]);
            store_plane_keys<SEARCH>(p0, tc, K, table, warp, lane, keybuf[1]);
        }
        PlaneRaw<T> pnext = next_plane(cur, tc, warp);
        __syncthreads();
        // cm: c2(M_{z-1}) and below: the keys of plane z - 1, at the warp's own pixels.
        uint32_t cm[k3Rows][2], below[k3Rows][2];
        {
            KeyRow M[k3Rows + 2];
#pragma unroll
            for (int j = 0; j < k3Rows + 2; ++j) {
                const KeyRow pj = smem_key_row(keybuf[0], r0 + j, lane);
                M[j] = max_rows(pj, smem_key_row(keybuf[1], r0 + j, lane));
                if (j >= 1 && j <= k3Rows) {
                    below[j - 1][0] = pj.own0;
                    below[j - 1][1] = pj.own1;
                }
            }
            uint32_t s0, s1;
            sp_init<SAT>(M[0], M[1], s0, s1);
#pragma unroll
            for (int i = 0; i < k3Rows; ++i)
                c2_quad<SAT, false>(M[i], M[i + 1], M[i + 2], kPlain, s0, s1, cm[i][0], cm[i][1]);
        }

        // Three buffers in a ring: at step z plane z + 1 goes to the buffer of plane z - 2, read
        // last at step z - 1, before the barrier of step z - 1 that every warp has passed. Both
        // planes z and z + 1 are read from shared memory, so no rows are carried in registers.
        const uint16_t *bc = keybuf[1];
        uint16_t *bn = keybuf[2], *bo = keybuf[0];
        for (int64_t z = z0; z < z1; ++z) {
            store_plane_keys<SEARCH>(pnext, tc, K, table, warp, lane, bn);
            if (z + 2 <= z1) pnext = next_plane(cur, tc, warp);  // block-uniform
            __syncthreads();
            KeyRow c0 = smem_key_row(bc, r0, lane), c1 = smem_key_row(bc, r0 + 1, lane);
            KeyRow n1 = smem_key_row(bn, r0 + 1, lane);
            KeyRow Ma = max_rows(c0, smem_key_row(bn, r0, lane)), Mb = max_rows(c1, n1);
            uint32_t ss0, ss1, sm0, sm1;
            sp_init<SAT>(c0, c1, ss0, ss1);
            sp_init<SAT>(Ma, Mb, sm0, sm1);
#pragma unroll
            for (int i = 0; i < k3Rows; ++i) {
                const KeyRow c2 = smem_key_row(bc, r0 + i + 2, lane);
                const KeyRow n2 = smem_key_row(bn, r0 + i + 2, lane);
                uint32_t cs0, cs1, cn0, cn1;
                c2_quad<SAT, !SAT>(c0, c1, c2, kBias, ss0, ss1, cs0, cs1);
                const KeyRow Md = max_rows(c2, n2);
                c2_quad<SAT, false>(Ma, Mb, Md, kPlain, sm0, sm1, cn0, cn1);
                hist_pair_h(c1.own0,
                            fold3<SAT>(cs0, cn0, cm[i][0], n1.own0, below[i][0], c1.own0),
                            hist_s, K.H);
                hist_pair_h(c1.own1,
                            fold3<SAT>(cs1, cn1, cm[i][1], n1.own1, below[i][1], c1.own1),
                            hist_s, K.H);
                cm[i][0] = cn0;
                cm[i][1] = cn1;
                below[i][0] = c1.own0;
                below[i][1] = c1.own1;
                c0 = c1;
                c1 = c2;
                n1 = n2;
                Ma = Mb;
                Mb = Md;
            }
            const uint16_t *t = bc;
            bc = bn;
            bn = bo;
            bo = const_cast<uint16_t *>(t);
        }
    }
    block_flush<false>(P, hist, b);
}

// ----------------------------------------------------------------------------------------------
// 3-D kernel with TMA-staged planes (float32 volumes whose rows hold a multiple of 4 values on a
// 16-byte-aligned base; tables of at most 256 bins; estimated keys)
// ----------------------------------------------------------------------------------------------
//
// Same tiles, tasks, slice fold and shared key ring as ecc_hard3d_kernel, with three changes.
//
// * Staging. One thread copies each plane's tile plus its one-voxel halo (136 x 34 floats,
//   columns x0 - 4 .. x0 + 131, rows y0 - 1 .. y0 + 32) into one of two shared staging buffers
//   with one cp.async.bulk.tensor copy that completes on the buffer's mbarrier, two planes ahead
//   of its use. The copy fills every position outside the volume (columns, rows and planes) with
//   NaN, whose key is "never", so no thread computes a grid bound and no raw value waits in
//   registers.
// * Coded keys. A voxel's key k is carried as the fp16 value 1024 + 4k + (x & 1) + 2 (y & 1).
//   Ordering voxels by (k, x & 1, y & 1, z) still refines the threshold order, and two vertices of
//   one cell differ in x & 1 or y & 1 unless they are vertical neighbours, so every in-plane
//   comparison is strict, [a earlier than p] = sat(p - a), with no p + 1 term; vertical
//   neighbours break ties by z as before. The bin is (pattern - 0x6400) >> 2. "Never" is
//   1024 + 4H + code, above every valid key (for H = 256 it rounds to 2048 or more, an even
//   integer, so differences with it stay integers and the flags stay 0 or 1).
// * Carried fold. up = [k_{z+1} < k_z] decides which of the two voxels of a pixel takes the
//   vertical cells above it: voxel z takes up c2(M_z), voxel z + 1 takes (1 - up) c2(M_z). Each
//   plane computes up once per voxel and carries q = -(1 - up) c2(M_z) to the next plane instead
//   of the keys and M contributions of the plane below:
//       1280 + c(p) = (1280 + c2(S_z; p)) - up c2(M_z) + q_{z-1}.
//
// Every mbarrier wait gives up after kWaitNs; the block then records the failure in the device
// error word, waits (bounded again) for its copy in flight and leaves without flushing.
// ecc_device_status() reports and clears the word.

// Three blocks per SM: with four, the 128-register cap made the compiler spill and serialise
// (1.355 against 1.338 ms on 1024^3).
#ifndef ECC_3D_TMA_BLOCKS
#define ECC_3D_TMA_BLOCKS 3
#endif
constexpr int kT3Blocks = ECC_3D_TMA_BLOCKS;  // resident blocks per SM the TMA kernel is built for
constexpr int kRawPitch = kKeyPitch;    // floats per staged row (columns x0 - 4 .. x0 + 131)
constexpr int kRawRows = kKeyRowsHalo;  // rows y0 - 1 .. y0 + 32
constexpr int kRawBytes = kRawPitch * kRawRows * 4;
constexpr int kRawStride = (kRawBytes + 127) & ~127;  // staging buffers on 128-byte boundaries
#ifndef ECC_3D_TMA_STAGES
#define ECC_3D_TMA_STAGES 2
#endif
constexpr int kT3Stages = ECC_3D_TMA_STAGES;  // staging buffers: copies run this many planes ahead
constexpr int kKeyRingBytes = 3 * kKeyPlane * 2;
constexpr int kCodedMaxBins = 256;  // 1024 + 4 (H - 1) + 3 < 2048
constexpr unsigned long long kWaitNs = ECC_WAIT_LIMIT_NS;  // 2 s per mbarrier wait
static_assert(kRawBytes % 16 == 0 && kKeyRingBytes % 16 == 0, "shared layout");
static_assert(kStrip + 8 == kRawPitch, "a staged row starts 4 columns left of the tile");


// Block g's segment [a, b) of the W tile-planes of an image shared out over G blocks: lengths
// W / G, the first W % G blocks one more.
__host__ __device__ __forceinline__ void tma3d_segment(int64_t W, int64_t G, int64_t g,
                                                       int64_t &a, int64_t &b)
{
    const int64_t q = W / G, r = W % G;
    a = g * q + (g < r ? g : r);
    b = a + q + (g < r ? 1 : 0);
}

struct Hard3TmaParams {
    CUtensorMap map;  // [batch][D][Hy][W] float32; box 136 x 34 x 1 x 1; NaN outside
    int64_t *out;
    int64_t tasks_per_image;
    int D, Hy, W, H, sign;
    int rows_per_task, tasks_x, tasks_y, ctas_per_image;
    int group;  // blocks per group: tasks_x (a row of tiles side by side) or 1
    float key_a, key_b, key_clo, key_chi;
    float table[kCodedMaxBins + 2];
};

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits for the completion of the phase of parity `parity`; false if it has not come in
// limit_ns (kWaitNs in the kernels).
__device__ __forceinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity,
                                               unsigned long long limit_ns = kWaitNs)
{
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > limit_ns) return false;
    return true;
}
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity)
{
    return mbar_try_wait(bar, parity) || mbar_wait_slow(bar, parity);
}

// One thread: plane z of image b's tile at (x0, y0) into the staging buffer.
__device__ __forceinline__ void stage_plane(const Hard3TmaParams &P, uint32_t raw_s, uint32_t bar,
                                            int x0, int y0, int z, int b)
{
    // (debug build) the tile starts inside the volume; planes -1 and D are the fill planes
    bounds_ok(&g_hard_error, x0 < P.W && y0 < P.Hy && z >= -1 && z <= P.D, kErrTmaTile);
    // the block's earlier reads of the buffer (generic proxy) before the copy's writes
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                 "r"((uint32_t)kRawBytes)
                 : "memory");
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(raw_s),
        "l"(reinterpret_cast<uint64_t>(&P.map)), "r"(x0 - 4), "r"(y0 - 1), "r"(z), "r"(b),
        "r"(bar)
        : "memory");
}

// Coding of a key pair: patterns 0x6400 + k -> 0x6400 + 4k + code, in each half at once. As a
// 32-bit integer, 4 * pair + C with C = c0 + (c1 << 16) - 3 * 0x64006400 (mod 2^32) gives
// (0x6400 + 4 k0 + c0) + (0x6400 + 4 k1 + c1) << 16: each half stays below 2^16 (at most 0x6803
// for k = 256), so no carry crosses into the other half.
__device__ __forceinline__ uint32_t code_pair_const(int yodd)
{
    // codes (x & 1) + 2 (y & 1) of the pair's two columns (the first column is even)
    const uint32_t c0 = 2u * (uint32_t)yodd, c1 = c0 + 1u;
    return c0 + (c1 << 16) - 3u * 0x64006400u;
}
__device__ __forceinline__ uint32_t code_pair(uint32_t pair, uint32_t C) { return 4u * pair + C; }

// A halo item of the staged plane: its index (the same in the raw and the key buffers) and its
// code. Items: rows y0 - 1 and y0 + 32 over columns x0 - 1 .. x0 + 128, then columns x0 - 1 and
// x0 + 128 over the tile's rows.
__device__ __forceinline__ void halo_item_coded(int i, int &off, uint32_t &code)
{
    int row, c;
    if (i < 2 * kHaloRowItems) {
        const int below = i >= kHaloRowItems;
        c = i - below * kHaloRowItems - 1;  // -1 .. 128
        row = below ? kKeyRowsHalo - 1 : 0;
    } else {
        const int j = i - 2 * kHaloRowItems;
        const int right = j >= kTileRows;
        row = 1 + j - right * kTileRows;
        c = right ? kStrip : -1;
    }
    off = row * kKeyPitch + 4 + c;
    // x0 and y0 are even: x & 1 = c & 1, and buffer row `row` is y = y0 - 1 + row
    code = (uint32_t)(c & 1) + 2u * (uint32_t)((row + 1) & 1);
}

// Keys of the staged plane into the key buffer `dst` (coded patterns). Each thread takes its
// warp's eight rows (four columns each) and its halo items; the rare exact fix-up revisits a
// group of two rows (the halo items join the first).
__device__ __forceinline__ void plane_keys_coded(const float *raw, uint16_t *dst,
                                                 const KeyConsts &K, const float *__restrict__ T,
                                                 int r0, int lane, const int *h_off,
                                                 const uint32_t *h_code)
{
    constexpr int kFixRows = 2, kGroups = k3Rows / kFixRows;
    uint32_t amb[kGroups];
#pragma unroll
    for (int q = 0; q < kGroups; ++q) amb[q] = 0;
    const int base = (1 + r0) * kKeyPitch + 4 + 4 * lane;
#pragma unroll
    for (int i = 0; i < k3Rows; ++i) {
        const float4 v = *reinterpret_cast<const float4 *>(raw + base + i * kKeyPitch);
        uint32_t k0, k1, k2, k3;
        key_fast2(v.x, v.y, K, k0, k1, amb[i / kFixRows]);
        key_fast2(v.z, v.w, K, k2, k3, amb[i / kFixRows]);
        const uint32_t cc = code_pair_const(i & 1);
        *reinterpret_cast<uint2 *>(dst + base + i * kKeyPitch) =
            make_uint2(code_pair(prmt(k0, k1, 0x5410), cc), code_pair(prmt(k2, k3, 0x5410), cc));
    }
    uint32_t hk[kHaloSlots];
#pragma unroll
    for (int s = 0; s < kHaloSlots; ++s) {
        hk[s] = 0;
        if (s + 1 < kHaloSlots || h_off[s] >= 0) hk[s] = key_fast(raw[h_off[s]], K, amb[0]);
    }
    uint32_t any = 0;
#pragma unroll
    for (int q = 0; q < kGroups; ++q) any |= amb[q];
    if (__any_sync(kFull, any != 0)) {  // rare: a value within E of a threshold
#pragma unroll
        for (int q = 0; q < kGroups; ++q) {
            if (amb[q] != 0) {
#pragma unroll
                for (int i = q * kFixRows; i < (q + 1) * kFixRows; ++i) {
                    const float4 v =
                        *reinterpret_cast<const float4 *>(raw + base + i * kKeyPitch);
                    uint32_t scratch = 0;
                    const uint32_t k0 = key_fix(v.x, key_fast(v.x, K, scratch), K.H, T);
                    const uint32_t k1 = key_fix(v.y, key_fast(v.y, K, scratch), K.H, T);
                    const uint32_t k2 = key_fix(v.z, key_fast(v.z, K, scratch), K.H, T);
                    const uint32_t k3 = key_fix(v.w, key_fast(v.w, K, scratch), K.H, T);
                    const uint32_t cc = code_pair_const(i & 1);
                    *reinterpret_cast<uint2 *>(dst + base + i * kKeyPitch) =
                        make_uint2(code_pair(prmt(k0, k1, 0x5410), cc),
                                   code_pair(prmt(k2, k3, 0x5410), cc));
                }
                if (q == 0) {
#pragma unroll
                    for (int s = 0; s < kHaloSlots; ++s)
                        if (s + 1 < kHaloSlots || h_off[s] >= 0)
                            hk[s] = key_fix(raw[h_off[s]], hk[s], K.H, T);
                }
            }
        }
    }
    // a halo key: pattern 0x6400 + k -> 0x6400 + 4k + code (k = 256: 0x6800 + code, >= 2048)
#pragma unroll
    for (int s = 0; s < kHaloSlots; ++s)
        if (s + 1 < kHaloSlots || h_off[s] >= 0)
            dst[h_off[s]] = (uint16_t)(4u * (hk[s] & 0xffffu) - 3u * kKeyBase + h_code[s]);
}

// The local Euler contribution of a pixel pair on coded keys (every flag strict:
// [a earlier than p] = sat(p - a)). NEG: return -c2 (plain); otherwise 1280 + c2.
template <bool NEG>
__device__ __forceinline__ uint32_t c2_pair_coded(uint32_t p, uint32_t L, uint32_t R, uint32_t aL,
                                                  uint32_t aR, uint32_t d, uint32_t dL,
                                                  uint32_t dR, uint32_t Sp, uint32_t &S_out)
{
    // five flags from saturating differences (FMA pipe), two from compares (ALU pipe): the same
    // 1.0 / 0.0 values, split so that neither pipe waits on the other (measured on 1024^3: no
    // compares 1.374 ms, one 1.346, two 1.338, three 1.366)
    const uint32_t W = h2_sub_sat(p, L), E = h2_sub_sat(p, R), S = h2_sub_sat(p, d);
    const uint32_t NE = h2_sub_sat(p, aR), SE = h2_sub_sat(p, dR);
    const uint32_t NW = h2_lt(aL, p), SW = h2_lt(dL, p);
    const uint32_t A = lop_or_and(Sp, E, NE);
    const uint32_t B = E & ~(S & SE);
    const uint32_t C = S & ~(W & SW);
    const uint32_t D = W & (Sp | ~NW);
    S_out = S;
    if (NEG) return h2_sub(h2_add(C, D), h2_sub(A, B));
    return h2_sub(h2_sub(h2_add(kBias, A), B), h2_add(C, D));
}

template <bool NEG>
__device__ __forceinline__ void c2_quad_coded(const KeyRow &a, const KeyRow &b, const KeyRow &d,
                                              uint32_t &Sp0, uint32_t &Sp1, uint32_t &c0,
                                              uint32_t &c1)
{
    uint32_t S0, S1;
    c0 = c2_pair_coded<NEG>(b.own0, b.L0, b.R0, a.L0, a.R0, d.own0, d.L0, d.R0, Sp0, S0);
    c1 = c2_pair_coded<NEG>(b.own1, b.R0, b.R1, a.R0, a.R1, d.own1, d.R0, d.R1, Sp1, S1);
    Sp0 = S0;
    Sp1 = S1;
}

// Histogram update for a pair of coded keys: bin (pattern - 0x6400) >> 2, i.e. the byte offset
// (pattern & 0xfffc) from hist_c = (shared address of the histogram) - 0x6400.
__device__ __forceinline__ void hist_pair_coded(uint32_t keys, uint32_t cv, uint32_t hist_c,
                                                int H)
{
    const int lo = ((int)(keys & 0xffffu) - (int)kKeyBase) >> 2;
    const int hi = ((int)(keys >> 16) - (int)kKeyBase) >> 2;
    if (!bounds_ok(&g_hard_error, lo >= 0 && lo <= H && hi >= 0 && hi <= H, kErrHardBin)) return;
    red_shared_add(hist_c + (keys & 0xfffcu), sext_byte0(cv));
    red_shared_add(hist_c + ((keys >> 16) & 0xfffcu), sext_byte2(cv));
}

// One vertical fold step of a pair: returns 1280 + c and updates the carry q for the plane above.
// cs_b = 1280 + c2(S_z), ncn = -c2(M_z), k / k_up: the keys of planes z and z + 1.
__device__ __forceinline__ uint32_t fold_carry(uint32_t cs_b, uint32_t ncn, uint32_t k,
                                               uint32_t k_up, uint32_t &q)
{
    const uint32_t up = h2_sub_sat(k, k_up);  // [k_{z+1} < k_z]
    const uint32_t cv = h2_add(cs_b, h2_fma(up, ncn, q));
    q = h2_fma(h2_neg(up), ncn, ncn);  // -(1 - up) c2(M_z)
    return cv;
}

__global__ void __launch_bounds__(k3Threads, kT3Blocks)
    ecc_hard3d_tma_kernel(const __grid_constant__ Hard3TmaParams P)
{
    extern __shared__ __align__(128) unsigned char smem_t3[];
    // the staging buffers start on 128-byte boundaries (the launch adds 128 bytes of slack)
    unsigned char *base = smem_t3 + ((128u - (smem_u32(smem_t3) & 127u)) & 127u);
    uint16_t *kb = reinterpret_cast<uint16_t *>(base + kT3Stages * kRawStride);
    int *hist = reinterpret_cast<int *>(base + kT3Stages * kRawStride + kKeyRingBytes);
    float *table = reinterpret_cast<float *>(hist + hist_words(P.H));
    __shared__ __align__(8) unsigned long long mbar[kT3Stages];

    const int tid = threadIdx.x, lane = tid & (kWarp - 1), warp = tid >> 5;
    for (int i = tid; i <= P.H; i += k3Threads) hist[i] = 0;
    for (int i = tid; i < P.H + 2; i += k3Threads) table[i] = P.table[i];
    const uint32_t bar0 = smem_u32(&mbar[0]), raw0 = smem_u32(base);
    if (tid == 0) {
        for (int s = 0; s < kT3Stages; ++s)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar0 + 8u * s) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    int h_off[kHaloSlots];
    uint32_t h_code[kHaloSlots];
#pragma unroll
    for (int s = 0; s < kHaloSlots; ++s) {
        const int i = tid + s * k3Threads;
        h_off[s] = -1;
        h_code[s] = 0;
        if (i < kHaloItems) halo_item_coded(i, h_off[s], h_code[s]);
    }
    KeyConsts K;
    K.a = P.key_a;
    K.b = P.key_b;
    K.nH = -(float)P.H;
    K.clo = P.key_clo;
    K.chi = P.key_chi;
    K.H = P.H;
    key_pairs(K);
    const int r0 = warp * k3Rows;  // buffer row of the row above the warp's first row
    const int b = blockIdx.y;
    const uint32_t hist_c = smem_u32(hist) - kKeyBase;
    const int64_t G = P.ctas_per_image;
    // The block's plane copies in issue order: copy n goes to staging buffer n % kT3Stages and
    // completes phase (n / kT3Stages) & 1 of that buffer's mbarrier; copies are waited for in
    // the same order. nq: copies issued, nw: copies waited for.
    uint32_t nq = 0, nw = 0;
    bool failed = false;

    // Blocks work in groups of P.group blocks: a whole row of tiles (one block per strip) when
    // the image has blocks enough, else single tiles. Group h takes a contiguous segment of the
    // image's (row of tiles or tile) x planes, numbered row by row, and its blocks walk the same
    // rows and planes side by side, so the halo columns that neighbouring tiles share are read
    // once into L2 for both. The segment is cut into pieces where a row ends: each piece is one
    // task, planes z0 .. z1 - 1 of this block's tile of the row.
    const int gsz = P.group;
    const int64_t groups = G / gsz, h = blockIdx.x / gsz;
    const int64_t rows = (int64_t)P.tasks_x * P.tasks_y / gsz;
    int64_t s0, s1;
    tma3d_segment(rows * P.D, groups, h, s0, s1);
    while (s0 < s1 && !failed) {
        const int64_t row = s0 / P.D;
        const int z0 = (int)(s0 % P.D);
        const int z1 = (int)min((int64_t)P.D, (int64_t)z0 + (s1 - s0));
        s0 += z1 - z0;
        const int64_t tile = row * gsz + blockIdx.x % gsz;
        const int tx = (int)(tile % P.tasks_x), ty = (int)(tile / P.tasks_x);
        const int x0 = tx * kStrip, y0 = ty * kTileRows;

        // The task reads planes z0 - 1 .. z1 (n_planes of them; planes -1 and D are filled with
        // NaN by the copies). Plane j of the task (z = z0 - 1 + j) is copied kT3Stages planes
        // ahead: its copy is issued once the keys of plane j - kT3Stages are in the key ring,
        // into the staging buffer that plane has just left.
        const int n_planes = z1 - z0 + 2;
        auto issue = [&](int j) {
            if (tid == 0)
                stage_plane(P, raw0 + (uint32_t)((nq % kT3Stages) * kRawStride),
                            bar0 + 8u * (nq % kT3Stages), x0, y0, z0 - 1 + j, b);
            ++nq;
        };
        auto wait = [&](bool &late) {
            const uint32_t s = nw % kT3Stages;
            late = !mbar_wait_bounded(bar0 + 8u * s, (nw / kT3Stages) & 1u);
            ++nw;
            return reinterpret_cast<const float *>(base + s * kRawStride);
        };

        // prologue: keys of planes z0 - 1 (key buffer 0) and z0 (key buffer 1)
        __syncthreads();  // the previous task's readers are done with every buffer
        for (int j = 0; j < kT3Stages && j < n_planes; ++j) issue(j);
        for (int j = 0; j < 2; ++j) {
            bool late;
            const float *raw = wait(late);
            plane_keys_coded(raw, kb + j * kKeyPlane, K, table, r0, lane, h_off, h_code);
            if (__syncthreads_or(late)) {  // block-uniform
                failed = true;
                break;
            }
            if (j + kT3Stages < n_planes) issue(j + kT3Stages);
        }
        if (failed) break;

        // q: -(1 - up) c2(M_{z0-1}) at the warp's pixels, up = [k_{z0} < k_{z0-1}]
        uint32_t q[k3Rows][2];
        {
            const uint16_t *bp = kb, *bq = kb + kKeyPlane;
            KeyRow pb = smem_key_row(bp, r0 + 1, lane), cb = smem_key_row(bq, r0 + 1, lane);
            KeyRow Ma = max_rows(smem_key_row(bp, r0, lane), smem_key_row(bq, r0, lane));
            KeyRow Mb = max_rows(pb, cb);
            uint32_t s0, s1;
            sp_init<true>(Ma, Mb, s0, s1);
#pragma unroll
            for (int i = 0; i < k3Rows; ++i) {
                const KeyRow pd = smem_key_row(bp, r0 + i + 2, lane);
                const KeyRow cd = smem_key_row(bq, r0 + i + 2, lane);
                const KeyRow Md = max_rows(pd, cd);
                uint32_t n0, n1;
                c2_quad_coded<true>(Ma, Mb, Md, s0, s1, n0, n1);
                q[i][0] = h2_fma(h2_neg(h2_sub_sat(pb.own0, cb.own0)), n0, n0);
                q[i][1] = h2_fma(h2_neg(h2_sub_sat(pb.own1, cb.own1)), n1, n1);
                pb = pd;
                cb = cd;
                Ma = Mb;
                Mb = Md;
            }
        }

        // Three key buffers in a ring: at step z plane z + 1 goes to the buffer of plane z - 1,
        // read last at step z - 1, before that step's barrier.
        const uint16_t *bc = kb + kKeyPlane;
        uint16_t *bn = kb + 2 * kKeyPlane, *bo = kb;
        for (int z = z0; z < z1; ++z) {
            const int j = z - z0 + 2;  // the task's plane z + 1
            bool late;
            const float *raw = wait(late);
            plane_keys_coded(raw, bn, K, table, r0, lane, h_off, h_code);
            if (__syncthreads_or(late)) {  // block-uniform
                failed = true;
                break;
            }
            if (j + kT3Stages < n_planes) issue(j + kT3Stages);
            KeyRow c0 = smem_key_row(bc, r0, lane), c1 = smem_key_row(bc, r0 + 1, lane);
            KeyRow n1 = smem_key_row(bn, r0 + 1, lane);
            KeyRow Ma = max_rows(c0, smem_key_row(bn, r0, lane)), Mb = max_rows(c1, n1);
            uint32_t ss0, ss1, sm0, sm1;
            sp_init<true>(c0, c1, ss0, ss1);
            sp_init<true>(Ma, Mb, sm0, sm1);
#pragma unroll
            for (int i = 0; i < k3Rows; ++i) {
                const KeyRow c2 = smem_key_row(bc, r0 + i + 2, lane);
                const KeyRow n2 = smem_key_row(bn, r0 + i + 2, lane);
                uint32_t cs0, cs1, nc0, nc1;
                c2_quad_coded<false>(c0, c1, c2, ss0, ss1, cs0, cs1);
                const KeyRow Md = max_rows(c2, n2);
                c2_quad_coded<true>(Ma, Mb, Md, sm0, sm1, nc0, nc1);
                hist_pair_coded(c1.own0, fold_carry(cs0, nc0, c1.own0, n1.own0, q[i][0]),
                                hist_c, P.H);
                hist_pair_coded(c1.own1, fold_carry(cs1, nc1, c1.own1, n1.own1, q[i][1]),
                                hist_c, P.H);
                c0 = c1;
                c1 = c2;
                n1 = n2;
                Ma = Mb;
                Mb = Md;
            }
            const uint16_t *tmp = bc;
            bc = bn;
            bn = bo;
            bo = const_cast<uint16_t *>(tmp);
        }
    }
    if (failed) {  // block-uniform: a copy did not arrive in time
        if (tid == 0) {
            // the copy that timed out and those issued after it, if they still land
            for (uint32_t n = nw - 1; n < nq; ++n)
                mbar_wait_bounded(bar0 + 8u * (n % kT3Stages), (n / kT3Stages) & 1u);
            atomicOr(&g_hard_error, kErrWaitTimeout);
        }
        return;
    }
    __syncthreads();
    unsigned long long *dst = reinterpret_cast<unsigned long long *>(P.out + b * (int64_t)P.H);
    for (int i = tid; i < P.H; i += k3Threads) {
        const int v = hist[i];
        if (v != 0) atomicAdd(dst + i, (unsigned long long)(long long)(P.sign * v));
    }
}

// ----------------------------------------------------------------------------------------------
// Probe of the wait-timeout path: one thread waits, with the kernels' bounded wait cut to
// limit_ns, for a phase of an mbarrier that nothing arrives at, then records the timeout in the
// device error word as the TMA kernel does. No copy is in flight, so the block may leave.
// ----------------------------------------------------------------------------------------------

__global__ void __launch_bounds__(1) ecc_wait_probe_kernel(unsigned long long limit_ns)
{
    __shared__ __align__(8) unsigned long long mbar;
    const uint32_t bar = smem_u32(&mbar);
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (!(mbar_try_wait(bar, 0) || mbar_wait_slow(bar, 0, limit_ns)))
        atomicOr(&g_hard_error, kErrWaitTimeout);
}

cudaError_t wait_probe(unsigned long long limit_ns, cudaStream_t s)
{
    ecc_wait_probe_kernel<<<1, 1, 0, s>>>(limit_ns);
    return cudaGetLastError();
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

int num_sms()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) n = 148;
    return n;
}

// Planes per 3-D block task. Cutting D planes into k chunks of R = ceil(D / k) planes gives
// tiles * ceil(D / R) tasks; with G blocks taking tasks g, g + G, ..., the busiest block runs
// ceil(tasks / G) of them, each R + 2 planes long (two prologue planes). R minimises that block
// time over k = 1, 2, ... (chunks of at least 8 planes, the prologue then at most a fifth), the
// first k winning ties; more than 64 rounds of tasks cannot gain more than a sixty-fourth.
static int64_t pick_chunk(int64_t D, int64_t tiles, int64_t blocks)
{
    const int64_t rmin = D < 8 ? D : 8;
    int64_t best = D, prev = -1;
    double best_time = -1.0;
    for (int64_t k = 1; k <= D; ++k) {
        const int64_t R = (D + k - 1) / k;
        if (R < rmin) break;
        if (R == prev) continue;
        prev = R;
        const int64_t tasks = tiles * ((D + R - 1) / R);
        const int64_t rounds = (tasks + blocks - 1) / blocks;
        const double t = (double)rounds * (double)(R + 2);
        if (best_time < 0.0 || t < best_time - 1e-9) {
            best_time = t;
            best = R;
        }
        if (rounds > 64) break;
    }
    return best;
}

HardShape plan_hard(const HardPlan &pl, int sms)
{
    HardShape sh;
    const int64_t strips = (pl.W + kStrip - 1) / kStrip;
    const int per_sm = pl.ndim == 2 ? ECC_2D_MIN_BLOCKS : (pl.tma ? kT3Blocks : ECC_3D_MIN_BLOCKS);
    const int64_t resident = (int64_t)sms * per_sm;  // blocks that fit at once
    // blocks per image: the resident blocks shared out over the batch, rounded down so that the
    // whole grid is one wave (rounding up left a few blocks to run alone in a second wave)
    int64_t per_image = resident / pl.batch;
    if (per_image < 1) per_image = 1;  // batches larger than a wave run in several waves
    if (pl.ndim == 2) {
        // R row ranges per strip, one warp per (strip, range), at least 32 rows per warp
        const int64_t N = strips * pl.Hy;
        const int64_t need = (N + 32 * kHardWarps - 1) / (32 * kHardWarps);
        if (per_image > need) per_image = need;
        if (per_image < 1) per_image = 1;
        int64_t R = per_image * kHardWarps / strips;
        if (R < 1) R = 1;
        if (R > pl.Hy) R = pl.Hy;
        per_image = (strips * R + kHardWarps - 1) / kHardWarps;  // every (strip, range) a warp
        sh.rows_per_task = R;
        sh.tasks_x = strips;
        sh.tasks_y = pl.Hy;
        sh.tasks_z = 1;
        sh.tasks_per_image = strips * R;  // warps with a band
    } else if (pl.tma) {
        // segments: groups of blocks (a row of tiles side by side when there are blocks enough,
        // else single tiles) take contiguous shares of the image's (row or tile) x planes,
        // numbered row by row, cut into pieces where a row ends
        const int64_t tiles_y = (pl.Hy + kTileRows - 1) / kTileRows;
        const int64_t group = per_image >= strips ? strips : 1;
        const int64_t units = strips * tiles_y / group * pl.D;
        int64_t groups = per_image / group;
        if (groups > units) groups = units;
        if (groups < 1) groups = 1;
        int64_t pieces = 0, most = 0;
        for (int64_t h = 0; h < groups; ++h) {
            int64_t a, b;
            tma3d_segment(units, groups, h, a, b);
            const int64_t n = (b - 1) / pl.D - a / pl.D + 1;
            pieces += n * group;
            if (n > most) most = n;
        }
        sh.tasks_x = strips;
        sh.tasks_y = tiles_y;
        sh.tasks_z = group;  // blocks per group
        sh.rows_per_task = (units + groups - 1) / groups;  // (row or tile)-planes per group
        sh.tasks_per_image = pieces;
        sh.blocks_per_image = groups * group;
        sh.rounds = most;
        sh.direct = false;
        return sh;
    } else {
        const int64_t tiles_y = (pl.Hy + kTileRows - 1) / kTileRows;
        const int64_t tiles = strips * tiles_y;
        if (per_image > tiles * pl.D) per_image = tiles * pl.D;
        const int64_t R = pick_chunk(pl.D, tiles, per_image);
        sh.rows_per_task = R;
        sh.tasks_x = strips;
        sh.tasks_y = tiles_y;
        sh.tasks_z = (pl.D + R - 1) / R;
        sh.tasks_per_image = sh.tasks_x * sh.tasks_y * sh.tasks_z;
        if (per_image > sh.tasks_per_image) per_image = sh.tasks_per_image;
    }
    if (per_image < 1) per_image = 1;
    sh.blocks_per_image = per_image;
    // 3-D: block g takes tasks g, g + G, ...; 2-D: one band per warp
    sh.rounds = pl.ndim == 2 ? 1 : (sh.tasks_per_image + per_image - 1) / per_image;
    // 2-D, one block per image: it holds the whole histogram and stores the curve itself
    sh.direct = pl.ndim == 2 && per_image == 1 && pl.scan && pl.sign == 1;
    return sh;
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

    const HardShape sh = plan_hard(pl, num_sms());
    if (pl.ndim == 2 && sh.tasks_x * sh.tasks_y >= ((int64_t)1 << 31))
        return cudaErrorInvalidValue;  // 32-bit row arithmetic (the C ABI rejects such sizes)
    P.rows_per_task = (int)sh.rows_per_task;
    P.rows_extra = 0;
    P.tasks_x = (int)sh.tasks_x;
    P.tasks_y = (int)sh.tasks_y;
    P.tasks_z = (int)sh.tasks_z;
    P.tasks_per_image = pl.ndim == 2 ? sh.tasks_x * sh.tasks_y : sh.tasks_per_image;
    P.ctas_per_image = (int)sh.blocks_per_image;
    P.direct = sh.direct ? 1 : 0;
    // 2-D images of several blocks: each block adds the running sum of its histogram, so the
    // call needs no scan launch
    P.prefix = (pl.ndim == 2 && !P.direct && pl.scan && pl.sign == 1) ? 1 : 0;
    if (!P.direct && pl.zero_out) {
        const cudaError_t m =
            cudaMemsetAsync(pl.out, 0, sizeof(int64_t) * (size_t)(pl.batch * pl.H), s);
        if (m != cudaSuccess) return m;
    }

    const size_t smem =
        (size_t)hist_words(pl.H) * sizeof(int) + (size_t)(CAP + 2) * sizeof(float);
    dim3 grid((unsigned)sh.blocks_per_image, (unsigned)pl.batch);
    if (pl.ndim == 2) {
        ecc_hard2d_kernel<T, CAP, SEARCH><<<grid, kHardThreads, smem, s>>>(P);
    } else {
        // the key buffers are static shared memory; past 48 KB in all the launch must opt in
        if (smem + sizeof(uint16_t) * 3 * kKeyPlane > 48 * 1024) {
            const cudaError_t e = cudaFuncSetAttribute(
                ecc_hard3d_kernel<T, CAP, SEARCH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                (int)smem);
            if (e != cudaSuccess) return e;
        }
        ecc_hard3d_kernel<T, CAP, SEARCH><<<grid, k3Threads, smem, s>>>(P);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || !pl.scan || P.direct || P.prefix) return e;
    return hard_scan(pl.out, pl.H, pl.batch, s);
}

// The tensor-map encoder of the driver, fetched through the runtime (no link against libcuda).
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_tiled()
{
    static const EncodeTiledFn fn = []() -> EncodeTiledFn {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

bool tma3d_shape_ok(const HardPlan &pl)
{
    // float32 volumes with rows of a multiple of 4 values (16-byte row strides), estimated keys,
    // at most 256 bins; every tensor-map stride below 2^40 bytes
    return pl.ndim == 3 && pl.dtype == ECC_F32 && pl.key_mode == kKeyEstimate &&
           pl.H <= kCodedMaxBins && pl.W % 4 == 0 &&
           (double)pl.D * (double)pl.Hy * (double)pl.W * 4.0 < (double)((int64_t)1 << 40);
}

// 3-D hard ECC through ecc_hard3d_tma_kernel; cudaErrorNotSupported when the tensor map cannot be
// built (the caller then takes ecc_hard3d_kernel).
static cudaError_t launch_hard3d_tma(const HardPlan &pl, cudaStream_t s)
{
    const EncodeTiledFn encode = encode_tiled();
    if (!encode) return cudaErrorNotSupported;
    Hard3TmaParams P;
    const cuuint64_t gdim[4] = {(cuuint64_t)pl.W, (cuuint64_t)pl.Hy, (cuuint64_t)pl.D,
                                (cuuint64_t)pl.batch};
    const cuuint64_t gstride[3] = {(cuuint64_t)pl.W * 4, (cuuint64_t)(pl.Hy * pl.W) * 4,
                                   (cuuint64_t)(pl.D * pl.Hy * pl.W) * 4};
    const cuuint32_t box[4] = {(cuuint32_t)kRawPitch, (cuuint32_t)kRawRows, 1, 1};
    const cuuint32_t estride[4] = {1, 1, 1, 1};
    if (encode(&P.map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void *>(pl.img), gdim,
               gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NAN_REQUEST_ZERO_FMA) != CUDA_SUCCESS)
        return cudaErrorNotSupported;
    HardPlan tp = pl;
    tp.tma = true;
    const HardShape sh = plan_hard(tp, num_sms());
    P.out = pl.out;
    P.tasks_per_image = sh.tasks_per_image;
    P.D = (int)pl.D;
    P.Hy = (int)pl.Hy;
    P.W = (int)pl.W;
    P.H = pl.H;
    P.sign = pl.sign;
    P.rows_per_task = (int)sh.rows_per_task;
    P.tasks_x = (int)sh.tasks_x;
    P.tasks_y = (int)sh.tasks_y;
    P.ctas_per_image = (int)sh.blocks_per_image;
    P.group = (int)sh.tasks_z;
    P.key_a = pl.key_a;
    P.key_b = pl.key_b;
    P.key_clo = pl.key_clo;
    P.key_chi = pl.key_chi;
    for (int i = 0; i < pl.H + 2; ++i) P.table[i] = pl.table[i];
    for (int i = pl.H + 2; i < kCodedMaxBins + 2; ++i) P.table[i] = 0.0f;
    if (pl.zero_out) {
        const cudaError_t m =
            cudaMemsetAsync(pl.out, 0, sizeof(int64_t) * (size_t)(pl.batch * pl.H), s);
        if (m != cudaSuccess) return m;
    }
    const size_t smem = 128 + (size_t)kT3Stages * kRawStride + kKeyRingBytes +
                        (size_t)hist_words(pl.H) * 4 + (size_t)(pl.H + 2) * 4;
    const cudaError_t a = cudaFuncSetAttribute(
        ecc_hard3d_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (a != cudaSuccess) return a;
    const dim3 grid((unsigned)sh.blocks_per_image, (unsigned)pl.batch);
    ecc_hard3d_tma_kernel<<<grid, k3Threads, smem, s>>>(P);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || !pl.scan) return e;
    return hard_scan(pl.out, pl.H, pl.batch, s);
}

cudaError_t hard_error_word(unsigned **p)
{
    return cudaGetSymbolAddress(reinterpret_cast<void **>(p), g_hard_error);
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
    if (pl.vec_ok && tma3d_shape_ok(pl)) {  // 16-byte-aligned rows: the TMA-staged kernel
        const cudaError_t e = launch_hard3d_tma(pl, s);
        if (e != cudaErrorNotSupported) return e;
    }
    if (pl.H <= 256) return launch_hard<float, 256, false>(pl, s);
    if (pl.H <= 1024) return launch_hard<float, 1024, false>(pl, s);
    return launch_hard<float, ECC_MAX_NBINS, false>(pl, s);
}

}  // namespace ecc
