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
// on fp16 key patterns, two pixels per instruction.
//
// 2-D: a warp owns a strip of 128 columns (four per lane, one 16-byte load per lane per row) and
// walks down a band of rows; raw rows are prefetched three rows ahead in registers, and the
// comparisons with the row below are reused as the "above" comparisons of the next row.
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

// Shared layout: int hist[H], then the table: f32 thresholds T[0..H+1], or for uint8 inputs the
// fp16 key pattern of each byte value (uint16[256]).
template <int CAP>
__device__ __forceinline__ void block_setup(const HardParams<CAP> &P, int *hist, float *table)
{
    for (int i = threadIdx.x; i < P.H; i += blockDim.x) hist[i] = 0;
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
        if (v != 0) atomicAdd(dst + i, (unsigned long long)(long long)v);
    }
}

template <int CAP>
__device__ __forceinline__ KeyConsts key_consts(const HardParams<CAP> &P)
{
    KeyConsts K;
    K.sH = P.scale;
    K.oH = P.offset;
    K.Hf = (float)P.H;
    K.E = P.key_err;
    K.H = P.H;
    K.search = P.key_mode == kKeySearch;
    return K;
}

// Key pattern of one float value (any value; NaN -> H). SEARCH: binary-search every value (the
// estimator is not usable for this threshold range).
template <bool SEARCH>
__device__ __forceinline__ uint32_t key_one(float v, const KeyConsts &K, const float *__restrict__ T)
{
    if (SEARCH) return key_search_pattern(v, K.H, T);
    float amb = 0.0f;
    const uint32_t k = key_fast(v, K, amb);
    return (amb != 0.0f) ? key_fix(v, k, K, T) : k;
}

template <bool SEARCH>
__device__ __forceinline__ uint32_t key_one(uint8_t v, const KeyConsts &, const float *__restrict__ T)
{
    return reinterpret_cast<const uint16_t *>(T)[v];
}

// Raw values of one row around a lane's four columns, plus (lanes 0 / 31 only) the value just
// left of column x0 / right of column x0 + 127. `valid` has bit j set when column x + j is inside
// the grid; `halo_in` says whether the lane's halo column exists.
template <typename T>
struct RawRow;

template <>
struct RawRow<float> {
    float v[4];
    float halo;
    uint32_t valid;
    bool present;  // row inside the grid (warp-uniform)
    bool halo_in;
};

template <>
struct RawRow<uint8_t> {
    uint32_t bytes;
    uint8_t halo;
    uint32_t valid;
    bool present;
    bool halo_in;
};

template <typename T>
__device__ __forceinline__ void load_own(const T *__restrict__ row, int xs, int W, bool vec,
                                         RawRow<T> &r);

template <>
__device__ __forceinline__ void load_own<float>(const float *__restrict__ row, int xs, int W,
                                                bool vec, RawRow<float> &r)
{
    if (vec) {
        const float4 q = __ldg(reinterpret_cast<const float4 *>(row + xs));
        r.v[0] = q.x;
        r.v[1] = q.y;
        r.v[2] = q.z;
        r.v[3] = q.w;
        r.valid = 0xfu;
    } else {
        r.valid = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const bool in = xs + j < W;
            r.v[j] = in ? __ldg(row + xs + j) : 0.0f;
            r.valid |= in ? (1u << j) : 0u;
        }
    }
}

template <>
__device__ __forceinline__ void load_own<uint8_t>(const uint8_t *__restrict__ row, int xs, int W,
                                                  bool vec, RawRow<uint8_t> &r)
{
    if (vec) {
        r.bytes = __ldg(reinterpret_cast<const unsigned int *>(row + xs));
        r.valid = 0xfu;
    } else {
        r.valid = 0;
        r.bytes = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const bool in = xs + j < W;
            r.bytes |= in ? ((uint32_t)__ldg(row + xs + j) << (8 * j)) : 0u;
            r.valid |= in ? (1u << j) : 0u;
        }
    }
}

template <typename T>
__device__ __forceinline__ RawRow<T> load_raw(const T *__restrict__ plane, int Hy, int W, int y,
                                              int x0, int lane, bool vec)
{
    RawRow<T> r;
    r.present = (y >= 0 && y < Hy);
    r.halo_in = false;
    if (!r.present) {
        r.valid = 0;
        return r;
    }
    const T *__restrict__ row = plane + (int64_t)y * W;
    load_own<T>(row, x0 + 4 * lane, W, vec, r);
    const int hx = (lane == 0) ? x0 - 1 : x0 + 128;
    r.halo_in = (lane == 0 || lane == kWarp - 1) && hx >= 0 && hx < W;
    r.halo = r.halo_in ? __ldg(row + hx) : (T)0;
    return r;
}

// fp16 key patterns of the lane's four values as pairs (k0 | k1 << 16, k2 | k3 << 16), and of
// its halo value (absent when there is none). Whole-warp call.
template <bool SEARCH>
__device__ __forceinline__ void raw_keys(const RawRow<float> &r, const KeyConsts &K,
                                         const float *__restrict__ T, uint32_t &own0,
                                         uint32_t &own1, uint32_t &halo_key)
{
    uint32_t k[4];
    if (SEARCH) {
#pragma unroll
        for (int j = 0; j < 4; ++j) k[j] = key_search_pattern(r.v[j], K.H, T);
    } else {
        float amb = 0.0f;
#pragma unroll
        for (int j = 0; j < 4; ++j) k[j] = key_fast(r.v[j], K, amb);
        if (__any_sync(kFull, amb != 0.0f)) {
            if (amb != 0.0f) {
#pragma unroll
                for (int j = 0; j < 4; ++j) k[j] = key_fix(r.v[j], k[j], K, T);
            }
        }
    }
    if (r.valid != 0xfu) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (!(r.valid >> j & 1u)) k[j] = kAbsentHalf;
    }
    own0 = prmt(k[0], k[1], 0x5410);
    own1 = prmt(k[2], k[3], 0x5410);
    halo_key = kAbsentHalf;
    if (r.halo_in) halo_key = key_one<SEARCH>(r.halo, K, T);
}

template <bool SEARCH>
__device__ __forceinline__ void raw_keys(const RawRow<uint8_t> &r, const KeyConsts &K,
                                         const float *__restrict__ T, uint32_t &own0,
                                         uint32_t &own1, uint32_t &halo_key)
{
    const uint16_t *lut = reinterpret_cast<const uint16_t *>(T);
    uint32_t k[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        k[j] = (r.valid >> j & 1u) ? (uint32_t)lut[(r.bytes >> (8 * j)) & 0xffu] : kAbsentHalf;
    own0 = prmt(k[0], k[1], 0x5410);
    own1 = prmt(k[2], k[3], 0x5410);
    halo_key = r.halo_in ? (uint32_t)lut[r.halo] : kAbsentHalf;
}

template <bool SEARCH, typename T>
__device__ __forceinline__ KeyRow key_row(const RawRow<T> &r, const KeyConsts &K,
                                          const float *__restrict__ table, int lane)
{
    if (!r.present) return absent_row();  // warp-uniform
    uint32_t own0, own1, hk;
    raw_keys<SEARCH>(r, K, table, own0, own1, hk);
    return make_key_row(own0, own1, lane, hk, hk);
}

// ----------------------------------------------------------------------------------------------
// 2-D kernel
// ----------------------------------------------------------------------------------------------
//
// Work: an image is cut into warp tasks (strip of 128 columns) x (band of rows_per_task rows),
// strip index fastest. blockIdx.y = image; block g of the image takes the task range
// [g * T / G, (g + 1) * T / G) and its warps take those tasks round-robin.
template <typename T, int CAP, bool SEARCH>
__global__ void __launch_bounds__(kHardThreads, ECC_2D_MIN_BLOCKS) ecc_hard2d_kernel(const __grid_constant__
                                                                  HardParams<CAP> P)
{
    extern __shared__ int smem[];
    int *hist = smem;
    float *table = reinterpret_cast<float *>(smem + P.H);
    block_setup(P, hist, table);

    const int64_t b = blockIdx.y;
    const T *__restrict__ img = static_cast<const T *>(P.img) + b * P.image_elems;
    const int lane = threadIdx.x & (kWarp - 1);
    const int warp = threadIdx.x >> 5;
    const int64_t Tn = P.tasks_per_image;
    const int t_begin = (int)(Tn * blockIdx.x / P.ctas_per_image);
    const int t_end = (int)(Tn * (blockIdx.x + 1) / P.ctas_per_image);
    const KeyConsts K = key_consts(P);
    const int Hy = (int)P.Hy, W = (int)P.W;
    const int R = P.rows_per_task, TX = P.tasks_x;
    const uint32_t limit = (kKeyBase + (uint32_t)P.H) * 0x10001u;

    for (int t = t_begin + warp; t < t_end; t += kHardWarps) {
        const int x0 = (t % TX) * 128;
        const int y0 = (t / TX) * R;
        const int y1 = min(y0 + R, Hy);
        const bool vec = P.vec_ok && (x0 + 128 <= W);

        // raw-row ring: at the start of step y, q0 / q1 / q2 (in rotation) hold rows y+1 .. y+3
        RawRow<T> q0 = load_raw(img, Hy, W, y0 + 1, x0, lane, vec);
        RawRow<T> q1 = load_raw(img, Hy, W, y0 + 2, x0, lane, vec);
        RawRow<T> q2 = load_raw(img, Hy, W, y0 + 3, x0, lane, vec);
        KeyRow ka = key_row<SEARCH>(load_raw(img, Hy, W, y0 - 1, x0, lane, vec), K, table, lane);
        KeyRow kb = key_row<SEARCH>(load_raw(img, Hy, W, y0, x0, lane, vec), K, table, lane);
        uint32_t Sp0, Sp1;
        sp_init(ka, kb, Sp0, Sp1);

#define ECC_2D_STEP(QS)                                                                     \
    {                                                                                       \
        if (y >= y1) break;                                                                 \
        const KeyRow kd = key_row<SEARCH>(QS, K, table, lane);                                    \
        QS = load_raw(img, Hy, W, y + 4, x0, lane, vec);                                    \
        uint32_t c0, c1;                                                                    \
        c2_quad(ka, kb, kd, kBias, Sp0, Sp1, c0, c1);                                       \
        hist_pair(kb.own0, c0, limit, hist);                                                \
        hist_pair(kb.own1, c1, limit, hist);                                                \
        ka = kb;                                                                            \
        kb = kd;                                                                            \
        ++y;                                                                                \
    }
        for (int y = y0; y < y1;) {
            ECC_2D_STEP(q0)
            ECC_2D_STEP(q1)
            ECC_2D_STEP(q2)
        }
#undef ECC_2D_STEP
    }
    block_flush(P, hist, b);
}

// ----------------------------------------------------------------------------------------------
// 3-D kernel
// ----------------------------------------------------------------------------------------------
//
// Work: block task = (tile of 128 columns x 8 rows) x (chunk of rows_per_task planes), tile x
// fastest, then tile y, then chunk. Warp w owns row y0 + w, lane l columns x0 + 4l .. x0 + 4l + 3.

constexpr int kTileRows = kHardWarps;                // 8
constexpr int kKeyPitch = 136;                       // halves per shared row (272 bytes)
constexpr int kKeyRowsHalo = kTileRows + 2;          // rows y0-1 .. y0+8
constexpr int kKeyPlane = kKeyRowsHalo * kKeyPitch;  // halves per plane buffer
// Tile column c (-1 .. 128) sits at half index 4 + c of a shared row, so a lane's own four keys
// form one 8-byte-aligned word pair.

// The raw values one thread needs for one plane of the tile: its warp's row around its columns
// (with the two halo columns on lanes 0 / 31) and one value of the two halo rows (thread t: row
// y0 - 1 or y0 + 8 by t >> 7, column x0 + (t & 127)); threads 0..3 also take the halo corners.
template <typename T>
struct PlaneRaw {
    RawRow<T> own;
    T hrow, corner;
    bool hrow_in, corner_in;
};

template <typename T>
__device__ __forceinline__ PlaneRaw<T> load_plane(const T *__restrict__ img, int64_t D, int Hy,
                                                  int W, int64_t z, int x0, int y0, bool vec_ok,
                                                  int warp, int lane)
{
    PlaneRaw<T> p;
    const bool zin = (z >= 0 && z < D);  // block-uniform
    const T *__restrict__ plane = img + (zin ? z : 0) * (int64_t)Hy * W;
    const bool vec = vec_ok && (x0 + 128 <= W);
    if (zin) {
        p.own = load_raw(plane, Hy, W, y0 + warp, x0, lane, vec);
    } else {
        p.own.present = false;
        p.own.halo_in = false;
        p.own.valid = 0;
    }
    const int t = threadIdx.x;
    const int hy = (t >> 7) ? y0 + kTileRows : y0 - 1;
    const int hx = x0 + (t & 127);
    p.hrow_in = zin && hy >= 0 && hy < Hy && hx < W;
    p.hrow = p.hrow_in ? plane[(int64_t)hy * W + hx] : (T)0;
    const int cy = (t & 2) ? y0 + kTileRows : y0 - 1;
    const int cx = (t & 1) ? x0 + 128 : x0 - 1;
    p.corner_in = zin && t < 4 && cy >= 0 && cy < Hy && cx >= 0 && cx < W;
    p.corner = p.corner_in ? plane[(int64_t)cy * W + cx] : (T)0;
    return p;
}

// Keys of a loaded plane into the shared buffer `dst` (uint16 patterns; absent outside the grid).
template <bool SEARCH, typename T>
__device__ __forceinline__ void store_plane_keys(const PlaneRaw<T> &p, const KeyConsts &K,
                                                 const float *__restrict__ table, int warp,
                                                 int lane, uint16_t *dst)
{
    uint32_t own0 = kAbsentPair, own1 = kAbsentPair, hk = kAbsentHalf;
    if (p.own.present) raw_keys<SEARCH>(p.own, K, table, own0, own1, hk);  // warp-uniform branch
    uint16_t *row = dst + (1 + warp) * kKeyPitch;
    *reinterpret_cast<uint2 *>(row + 4 + 4 * lane) = make_uint2(own0, own1);
    if (lane == 0) row[3] = (uint16_t)hk;
    if (lane == kWarp - 1) row[4 + 128] = (uint16_t)hk;
    const int t = threadIdx.x;
    const uint32_t hkey = p.hrow_in ? key_one<SEARCH>(p.hrow, K, table) : kAbsentHalf;
    dst[((t >> 7) ? kKeyRowsHalo - 1 : 0) * kKeyPitch + 4 + (t & 127)] = (uint16_t)hkey;
    if (t < 4) {
        const uint32_t ck = p.corner_in ? key_one<SEARCH>(p.corner, K, table) : kAbsentHalf;
        dst[((t & 2) ? kKeyRowsHalo - 1 : 0) * kKeyPitch + ((t & 1) ? 4 + 128 : 3)] = (uint16_t)ck;
    }
}

// Buffer row r (= tile row r - 1, r = 0 .. 9) around the lane's four columns.
__device__ __forceinline__ KeyRow smem_key_row(const uint16_t *buf, int r, int lane)
{
    const uint16_t *row = buf + r * kKeyPitch;
    const uint2 own = *reinterpret_cast<const uint2 *>(row + 4 + 4 * lane);
    const uint32_t left = row[3 + 4 * lane];
    const uint32_t right = row[8 + 4 * lane];
    KeyRow k;
    k.own0 = own.x;
    k.own1 = own.y;
    k.L0 = prmt(left, own.x, 0x5410);
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
    float *table = reinterpret_cast<float *>(smem + P.H);
    __shared__ __align__(16) uint16_t keybuf[2][kKeyPlane];
    block_setup(P, hist, table);

    const int64_t b = blockIdx.y;
    const T *__restrict__ img = static_cast<const T *>(P.img) + b * P.image_elems;
    const int lane = threadIdx.x & (kWarp - 1);
    const int warp = threadIdx.x >> 5;
    const int64_t Tn = P.tasks_per_image;
    const int64_t t_begin = Tn * blockIdx.x / P.ctas_per_image;
    const int64_t t_end = Tn * (blockIdx.x + 1) / P.ctas_per_image;
    const KeyConsts K = key_consts(P);
    const bool vec_ok = P.vec_ok != 0;
    const int64_t D = P.D;
    const int Hy = (int)P.Hy, W = (int)P.W;
    const uint32_t limit = (kKeyBase + (uint32_t)P.H) * 0x10001u;
    const uint32_t kPlain = 0u;  // bias of the M stencil: plain c values

    for (int64_t t = t_begin; t < t_end; ++t) {
        const int tx = (int)(t % P.tasks_x);
        const int64_t rest = t / P.tasks_x;
        const int ty = (int)(rest % P.tasks_y);
        const int64_t tz = rest / P.tasks_y;
        const int x0 = tx * 128;
        const int y0 = ty * kTileRows;
        const int64_t z0 = tz * P.rows_per_task;
        const int64_t z1 = min(z0 + (int64_t)P.rows_per_task, D);
        const bool row_in = (y0 + warp) < Hy;  // warp-uniform

        // prologue: keys of planes z0 - 1 (buffer 0) and z0 (buffer 1); raw plane z0 + 1 in flight
        __syncthreads();  // the previous task's readers are done with both buffers
        {
            const PlaneRaw<T> pm = load_plane<T>(img, D, Hy, W, z0 - 1, x0, y0, vec_ok, warp, lane);
            const PlaneRaw<T> p0 = load_plane<T>(img, D, Hy, W, z0, x0, y0, vec_ok, warp, lane);
            store_plane_keys<SEARCH>(pm, K, table, warp, lane, keybuf[0]);
            store_plane_keys<SEARCH>(p0, K, table, warp, lane, keybuf[1]);
        }
        PlaneRaw<T> pnext = load_plane<T>(img, D, Hy, W, z0 + 1, x0, y0, vec_ok, warp, lane);
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
            sp_init(ma, mb, s0, s1);
            c2_quad(ma, mb, md, kPlain, s0, s1, cm0, cm1);
            below0 = pb.own0;
            below1 = pb.own1;
        }

        for (int64_t z = z0; z < z1; ++z) {
            uint16_t *nbuf = keybuf[(z - z0) & 1];  // plane z + 1 replaces plane z - 1
            // One barrier per plane: the buffer written here was last read in the step before
            // the previous one, and every warp has passed the previous step's barrier since.
            if (z == z0) __syncthreads();  // the prologue read buffer 0
            store_plane_keys<SEARCH>(pnext, K, table, warp, lane, nbuf);
            if (z + 2 <= z1) pnext = load_plane<T>(img, D, Hy, W, z + 2, x0, y0, vec_ok, warp, lane);
            __syncthreads();
            const KeyRow na = smem_key_row(nbuf, warp, lane);
            const KeyRow nb = smem_key_row(nbuf, warp + 1, lane);
            const KeyRow nd = smem_key_row(nbuf, warp + 2, lane);
            if (row_in) {
                uint32_t s0, s1, cs0, cs1, cn0, cn1;
                sp_init(ca, cb, s0, s1);
                c2_quad(ca, cb, cd, kBias, s0, s1, cs0, cs1);
                const KeyRow ma = max_rows(ca, na), mb = max_rows(cb, nb), md = max_rows(cd, nd);
                sp_init(ma, mb, s0, s1);
                c2_quad(ma, mb, md, kPlain, s0, s1, cn0, cn1);
                // c = cS - [k_{z+1} < k_z] c2(M_z) - [k_{z-1} <= k_z] c2(M_{z-1})
                const uint32_t up0 = h2_lt_mask(nb.own0, cb.own0);
                const uint32_t up1 = h2_lt_mask(nb.own1, cb.own1);
                const uint32_t dn0 = h2_le_mask(below0, cb.own0);
                const uint32_t dn1 = h2_le_mask(below1, cb.own1);
                const uint32_t c0 = h2_sub(h2_sub(cs0, cn0 & up0), cm0 & dn0);
                const uint32_t c1 = h2_sub(h2_sub(cs1, cn1 & up1), cm1 & dn1);
                hist_pair(cb.own0, c0, limit, hist);
                hist_pair(cb.own1, c1, limit, hist);
                cm0 = cn0;
                cm1 = cn1;
            }
            below0 = cb.own0;
            below1 = cb.own1;
            ca = na;
            cb = nb;
            cd = nd;
        }
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
    P.scale = pl.scale;
    P.offset = pl.offset;
    P.key_err = pl.key_err;
    P.vec_ok = pl.vec_ok;
    const int ntab = (pl.dtype == ECC_U8) ? 128 : pl.H + 2;  // u8: 256 uint16 in 128 floats
    P.table_len = ntab;
    for (int i = 0; i < ntab; ++i) P.table[i] = pl.table[i];
    for (int i = ntab; i < CAP + 2; ++i) P.table[i] = 0.0f;

    const int sms = num_sms();
    const int64_t strips = (pl.W + 127) / 128;
    const int per_sm = pl.ndim == 2 ? ECC_2D_MIN_BLOCKS : ECC_3D_MIN_BLOCKS;
    const int64_t resident = (int64_t)sms * per_sm;
    if (pl.ndim == 2) {
        // rows per warp task: 8, or more for very large batches (at most ~64 K tasks per warp
        // slot keeps the task loop short); small tasks keep the warps of a block balanced
        int64_t R = 8;
        while (R < 256 && pl.Hy * strips * pl.batch / R > resident * kHardWarps * 64) R *= 2;
        P.rows_per_task = (int)R;
        P.tasks_x = (int)strips;
        P.tasks_y = (int)((pl.Hy + R - 1) / R);
        P.tasks_z = 1;
    } else {
        // planes per block task: aim at ~8 tasks per resident block, at least 16 planes each
        const int64_t tiles_y = (pl.Hy + kTileRows - 1) / kTileRows;
        const int64_t tiles = strips * tiles_y * pl.batch;
        const int64_t want = (pl.D * tiles + resident * 8 - 1) / (resident * 8);
        const int64_t R = want < 16 ? 16 : (want > 256 ? 256 : want);
        P.rows_per_task = (int)R;
        P.tasks_x = (int)strips;
        P.tasks_y = (int)tiles_y;
        P.tasks_z = (int)((pl.D + R - 1) / R);
    }
    P.tasks_per_image = (int64_t)P.tasks_x * P.tasks_y * P.tasks_z;
    int64_t per_image_ctas = (resident + pl.batch - 1) / pl.batch;
    const int64_t max_ctas = pl.ndim == 2 ? (P.tasks_per_image + kHardWarps - 1) / kHardWarps
                                          : P.tasks_per_image;
    if (per_image_ctas > max_ctas) per_image_ctas = max_ctas;
    if (per_image_ctas < 1) per_image_ctas = 1;
    P.ctas_per_image = (int)per_image_ctas;

    const size_t smem = (size_t)pl.H * sizeof(int) + (size_t)(CAP + 2) * sizeof(float);
    dim3 grid((unsigned)per_image_ctas, (unsigned)pl.batch);
    if (pl.ndim == 2) {
        ecc_hard2d_kernel<T, CAP, SEARCH><<<grid, kHardThreads, smem, s>>>(P);
    } else {
        ecc_hard3d_kernel<T, CAP, SEARCH><<<grid, kHardThreads, smem, s>>>(P);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    ecc_bin_scan_kernel<<<(unsigned)pl.batch, kScanThreads, 0, s>>>(pl.out, pl.H);
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
