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
// one-pixel halo, from which every warp builds the three rows around its own row.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ecc_internal.cuh"
#include "ecc_keys.cuh"

namespace ecc {

constexpr int kHardThreads = 256;
constexpr int kHardWarps = kHardThreads / kWarp;

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

// Raw values of one row around a lane's four columns, plus (lanes 0 / 31) the value just left of
// column x0 / right of column x0 + 127. `valid` has bit j set when column x + j is inside the grid.
template <typename T>
struct RawRow;

template <>
struct RawRow<float> {
    float v[4];
    float halo;
    uint32_t valid;
    bool present;  // row inside the grid (warp-uniform)
};

template <>
struct RawRow<uint8_t> {
    uint32_t bytes;
    uint32_t halo;
    uint32_t valid;
    bool present;
};

__device__ __forceinline__ RawRow<float> load_raw(const float *__restrict__ plane, int64_t Hy,
                                                  int64_t W, int64_t y, int64_t x0, int lane,
                                                  bool vec)
{
    RawRow<float> r;
    r.present = (y >= 0 && y < Hy);
    r.valid = 0xfu;
    r.halo = 0.0f;
    r.v[0] = r.v[1] = r.v[2] = r.v[3] = 0.0f;
    if (!r.present) return r;
    const float *__restrict__ row = plane + y * W;
    const int64_t xs = x0 + 4 * lane;
    if (vec) {
        const float4 q = __ldg(reinterpret_cast<const float4 *>(row + xs));
        r.v[0] = q.x;
        r.v[1] = q.y;
        r.v[2] = q.z;
        r.v[3] = q.w;
    } else {
        r.valid = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const bool in = xs + j < W;
            r.v[j] = in ? __ldg(row + xs + j) : 0.0f;
            r.valid |= in ? (1u << j) : 0u;
        }
    }
    if (lane == 0 && x0 > 0) r.halo = __ldg(row + x0 - 1);
    if (lane == kWarp - 1 && x0 + 128 < W) r.halo = __ldg(row + x0 + 128);
    return r;
}

__device__ __forceinline__ RawRow<uint8_t> load_raw(const uint8_t *__restrict__ plane, int64_t Hy,
                                                    int64_t W, int64_t y, int64_t x0, int lane,
                                                    bool vec)
{
    RawRow<uint8_t> r;
    r.present = (y >= 0 && y < Hy);
    r.valid = 0xfu;
    r.halo = 0;
    r.bytes = 0;
    if (!r.present) return r;
    const uint8_t *__restrict__ row = plane + y * W;
    const int64_t xs = x0 + 4 * lane;
    if (vec) {
        r.bytes = __ldg(reinterpret_cast<const unsigned int *>(row + xs));
    } else {
        r.valid = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const bool in = xs + j < W;
            r.bytes |= in ? ((uint32_t)__ldg(row + xs + j) << (8 * j)) : 0u;
            r.valid |= in ? (1u << j) : 0u;
        }
    }
    if (lane == 0 && x0 > 0) r.halo = __ldg(row + x0 - 1);
    if (lane == kWarp - 1 && x0 + 128 < W) r.halo = __ldg(row + x0 + 128);
    return r;
}

// Key pattern of one float value (any value, NaN -> H).
__device__ __forceinline__ uint32_t key_one(float v, const KeyConsts &K, const float *__restrict__ T)
{
    if (K.search) return key_search_pattern(v, K.H, T);
    float amb = 0.0f;
    const uint32_t k = key_fast(v, K, amb);
    return (amb != 0.0f) ? key_fix(v, k, K, T) : k;
}

// fp16 key patterns of the lane's four values (pairs k0 | k1 << 16, k2 | k3 << 16) and of its
// halo value (lanes 0 and 31; absent when the halo column is outside the grid). Whole-warp call.
__device__ __forceinline__ void raw_keys(const RawRow<float> &r, const KeyConsts &K,
                                         const float *__restrict__ T, int lane, int64_t x0,
                                         int64_t W, uint32_t &own0, uint32_t &own1,
                                         uint32_t &halo_key)
{
    uint32_t k[4];
    if (K.search) {
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
    if (lane == 0 && x0 > 0) halo_key = key_one(r.halo, K, T);
    if (lane == kWarp - 1 && x0 + 128 < W) halo_key = key_one(r.halo, K, T);
}

__device__ __forceinline__ void raw_keys(const RawRow<uint8_t> &r, const KeyConsts &,
                                         const float *__restrict__ T, int lane, int64_t x0,
                                         int64_t W, uint32_t &own0, uint32_t &own1,
                                         uint32_t &halo_key)
{
    const uint16_t *lut = reinterpret_cast<const uint16_t *>(T);
    uint32_t k[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        k[j] = (r.valid >> j & 1u) ? (uint32_t)lut[(r.bytes >> (8 * j)) & 0xffu] : kAbsentHalf;
    own0 = prmt(k[0], k[1], 0x5410);
    own1 = prmt(k[2], k[3], 0x5410);
    halo_key = kAbsentHalf;
    if (lane == 0 && x0 > 0) halo_key = lut[r.halo & 0xffu];
    if (lane == kWarp - 1 && x0 + 128 < W) halo_key = lut[r.halo & 0xffu];
}

template <typename T>
__device__ __forceinline__ KeyRow key_row(const RawRow<T> &r, const KeyConsts &K,
                                          const float *__restrict__ table, int lane, int64_t x0,
                                          int64_t W)
{
    if (!r.present) return absent_row();  // warp-uniform
    uint32_t own0, own1, hk;
    raw_keys(r, K, table, lane, x0, W, own0, own1, hk);
    return make_key_row(own0, own1, lane, hk, hk);
}

// ----------------------------------------------------------------------------------------------
// 2-D kernel
// ----------------------------------------------------------------------------------------------
//
// Work: an image is cut into warp tasks (strip of 128 columns) x (band of rows_per_task rows),
// strip index fastest. blockIdx.y = image; block g of the image takes the task range
// [g * T / G, (g + 1) * T / G) and its warps take those tasks round-robin.
template <typename T, int CAP>
__global__ void __launch_bounds__(kHardThreads) ecc_hard2d_kernel(const __grid_constant__
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
    const int64_t t_begin = Tn * blockIdx.x / P.ctas_per_image;
    const int64_t t_end = Tn * (blockIdx.x + 1) / P.ctas_per_image;
    const KeyConsts K = key_consts(P);
    const int64_t Hy = P.Hy, W = P.W;
    const uint32_t limit = (kKeyBase + (uint32_t)P.H) * 0x10001u;

    for (int64_t t = t_begin + warp; t < t_end; t += kHardWarps) {
        const int64_t x0 = (t % P.tasks_x) * 128;
        const int64_t y0 = (t / P.tasks_x) * P.rows_per_task;
        const int64_t y1 = min(y0 + (int64_t)P.rows_per_task, Hy);
        const bool vec = P.vec_ok && (x0 + 128 <= W);

        // raw-row ring: at the start of step y, q0 / q1 / q2 (in rotation) hold rows y+1 .. y+3
        RawRow<T> q0 = load_raw(img, Hy, W, y0 + 1, x0, lane, vec);
        RawRow<T> q1 = load_raw(img, Hy, W, y0 + 2, x0, lane, vec);
        RawRow<T> q2 = load_raw(img, Hy, W, y0 + 3, x0, lane, vec);
        KeyRow ka = key_row(load_raw(img, Hy, W, y0 - 1, x0, lane, vec), K, table, lane, x0, W);
        KeyRow kb = key_row(load_raw(img, Hy, W, y0, x0, lane, vec), K, table, lane, x0, W);
        uint32_t Sp0, Sp1;
        sp_init(ka, kb, Sp0, Sp1);

#define ECC_2D_STEP(QS)                                                                     \
    {                                                                                       \
        if (y >= y1) break;                                                                 \
        const KeyRow kd = key_row(QS, K, table, lane, x0, W);                               \
        QS = load_raw(img, Hy, W, y + 4, x0, lane, vec);                                    \
        uint32_t c0, c1;                                                                    \
        c2_quad(ka, kb, kd, kBias, Sp0, Sp1, c0, c1);                                       \
        hist_pair(kb.own0, c0, limit, hist);                                                \
        hist_pair(kb.own1, c1, limit, hist);                                                \
        ka = kb;                                                                            \
        kb = kd;                                                                            \
        ++y;                                                                                \
    }
        for (int64_t y = y0; y < y1;) {
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

// Keys of plane z of the tile plus halo into `dst` (uint16 patterns; absent outside the grid).
template <typename T>
__device__ __forceinline__ void plane_keys(const T *__restrict__ img, int64_t D, int64_t Hy,
                                           int64_t W, int64_t z, int64_t x0, int64_t y0,
                                           bool vec_ok, const KeyConsts &K,
                                           const float *__restrict__ table, uint16_t *dst)
{
    const int lane = threadIdx.x & (kWarp - 1);
    const int warp = threadIdx.x >> 5;
    const bool zin = (z >= 0 && z < D);  // block-uniform
    const T *__restrict__ plane = img + (zin ? z : 0) * Hy * W;
    const bool vec = vec_ok && (x0 + 128 <= W);
    // each warp: its own row (buffer rows 1 .. 8) with the two halo columns
    {
        const int64_t y = y0 + warp;
        uint32_t own0 = kAbsentPair, own1 = kAbsentPair, hk = kAbsentHalf;
        if (zin) {
            const RawRow<T> r = load_raw(plane, Hy, W, y, x0, lane, vec);
            if (r.present) raw_keys(r, K, table, lane, x0, W, own0, own1, hk);
        }
        uint16_t *row = dst + (1 + warp) * kKeyPitch;
        *reinterpret_cast<uint2 *>(row + 4 + 4 * lane) = make_uint2(own0, own1);
        if (lane == 0) row[3] = (uint16_t)hk;
        if (lane == kWarp - 1) row[4 + 128] = (uint16_t)hk;
    }
    // halo rows y0 - 1 (buffer row 0) and y0 + 8 (buffer row 9): 2 x 130 keys
    for (int i = threadIdx.x; i < 2 * 130; i += kHardThreads) {
        const int hr = i / 130;
        const int c = i % 130 - 1;  // tile column -1 .. 128
        const int64_t y = (hr == 0) ? y0 - 1 : y0 + kTileRows;
        const int64_t x = x0 + c;
        uint32_t key = kAbsentHalf;
        if (zin && y >= 0 && y < Hy && x >= 0 && x < W) {
            if constexpr (sizeof(T) == 1) {
                key = reinterpret_cast<const uint16_t *>(table)[(uint32_t)plane[y * W + x]];
            } else {
                key = key_one((float)plane[y * W + x], K, table);
            }
        }
        dst[(hr == 0 ? 0 : kKeyRowsHalo - 1) * kKeyPitch + 4 + c] = (uint16_t)key;
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

template <typename T, int CAP>
__global__ void __launch_bounds__(kHardThreads) ecc_hard3d_kernel(const __grid_constant__
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
    const int64_t D = P.D, Hy = P.Hy, W = P.W;
    const uint32_t limit = (kKeyBase + (uint32_t)P.H) * 0x10001u;
    const uint32_t kPlain = 0u;  // bias of the M stencil: plain c values

    for (int64_t t = t_begin; t < t_end; ++t) {
        const int64_t tx = t % P.tasks_x;
        const int64_t rest = t / P.tasks_x;
        const int64_t ty = rest % P.tasks_y;
        const int64_t tz = rest / P.tasks_y;
        const int64_t x0 = tx * 128;
        const int64_t y0 = ty * kTileRows;
        const int64_t z0 = tz * P.rows_per_task;
        const int64_t z1 = min(z0 + (int64_t)P.rows_per_task, D);
        const bool row_in = (y0 + warp) < Hy;  // warp-uniform

        // prologue: planes z0 - 1 (buffer 0) and z0 (buffer 1)
        __syncthreads();  // the previous task's readers are done with both buffers
        plane_keys<T>(img, D, Hy, W, z0 - 1, x0, y0, vec_ok, K, table, keybuf[0]);
        plane_keys<T>(img, D, Hy, W, z0, x0, y0, vec_ok, K, table, keybuf[1]);
        __syncthreads();
        uint32_t cm0, cm1;  // c2(M_{z-1}) at the lane's pixels (plain values)
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
            __syncthreads();
            plane_keys<T>(img, D, Hy, W, z + 1, x0, y0, vec_ok, K, table, nbuf);
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

template <typename T, int CAP>
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
    const int per_sm = pl.ndim == 2 ? 4 : 3;
    const int64_t resident = (int64_t)sms * per_sm;
    if (pl.ndim == 2) {
        // rows per warp task: aim at ~16 K warp tasks in total, at least 8 rows each
        int64_t want = (pl.Hy * strips * pl.batch + 16383) / 16384;
        int64_t R = ((want + 7) / 8) * 8;
        R = R < 8 ? 8 : (R > 256 ? 256 : R);
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
        ecc_hard2d_kernel<T, CAP><<<grid, kHardThreads, smem, s>>>(P);
    } else {
        ecc_hard3d_kernel<T, CAP><<<grid, kHardThreads, smem, s>>>(P);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    ecc_bin_scan_kernel<<<(unsigned)pl.batch, kScanThreads, 0, s>>>(pl.out, pl.H);
    return cudaGetLastError();
}

cudaError_t hard_run(const HardPlan &pl, cudaStream_t s)
{
    if (pl.dtype == ECC_U8) {
        if (pl.H <= 256) return launch_hard<uint8_t, 256>(pl, s);
        if (pl.H <= 1024) return launch_hard<uint8_t, 1024>(pl, s);
        return launch_hard<uint8_t, ECC_MAX_NBINS>(pl, s);
    }
    if (pl.H <= 256) return launch_hard<float, 256>(pl, s);
    if (pl.H <= 1024) return launch_hard<float, 1024>(pl, s);
    return launch_hard<float, ECC_MAX_NBINS>(pl, s);
}

}  // namespace ecc
