// ecc_hard.cu -- hard Euler characteristic curve of dense 2-D / 3-D grids (sm_103a).
//
// Paper notes "Scalable GPU-Accelerated Euler Characteristic Curves: Optimization and
// Differentiable Learning for PyTorch":
//   "Key designs -- full-scan CUDA kernel": one pass over the whole grid with no chunked
//   re-launches; each thread block keeps a private shared-memory histogram of H bins, and only
//   after all of its voxels does it flush, once, to global memory with atomics.
//   "Key designs -- local computation of the Euler characteristic coefficient": c(p) from the
//   3x3 / 3x3x3 neighbourhood, accumulated at p's threshold bin.
// The histogram's running sum over bins is the curve (second kernel).
//
// 2-D kernel: a warp owns a strip of 128 columns (4 per lane, one 16-byte load per lane per row)
// and walks down a band of rows holding rows y-1, y, y+1 in registers; the columns left and right
// of a lane's four come from its neighbours by shuffle, and the strip's two halo columns from
// one extra scalar load each.
//
// 3-D kernel: the V-construction complex of a volume splits into the cells lying in one plane z
// and the "vertical" cells sigma x [z, z+1], sigma a cell of the plane. A vertical cell's value is
// the max over sigma of M_z = max(S_z, S_{z+1}) and its dimension is dim(sigma) + 1, so
//     ECC_3D = sum_z ECC_2D(S_z) - sum_z ECC_2D(M_z).
// Per voxel p at (x, y, z) this gives one contribution at p's bin:
//     c(p) = c2(S_z; p) - [p owns M_z(x,y)] c2(M_z; x,y) - [p owns M_{z-1}(x,y)] c2(M_{z-1}; x,y)
// where p owns M_z(x,y) when S_{z+1}(x,y) < S_z(x,y) (the later voxel wins ties) and owns
// M_{z-1}(x,y) when S_{z-1}(x,y) <= S_z(x,y). With NaN for "absent / never", both ownership tests
// fail when either value is NaN, and M propagates NaN, so such max-pixels are dropped as they
// must be. A warp owns a 128-column row segment of a 128 x 8 tile and walks z.
#include <cuda_runtime.h>
#include <stdint.h>

#include "ecc_internal.cuh"

namespace ecc {

// ----------------------------------------------------------------------------------------------
// Row loads: six values (x-1 .. x+4) of one row for a lane owning columns x .. x+3, x = x0 + 4 lane
// ----------------------------------------------------------------------------------------------

template <typename T>
struct RowLoader;

template <>
struct RowLoader<float> {
    static __device__ __forceinline__ float at(const float *__restrict__ row, int64_t x)
    {
        return __ldg(row + x);
    }
    static __device__ __forceinline__ void own4(const float *__restrict__ row, int64_t xs,
                                                int64_t W, bool vec, float v[6])
    {
        if (vec) {
            const float4 q = __ldg(reinterpret_cast<const float4 *>(row + xs));
            v[1] = q.x;
            v[2] = q.y;
            v[3] = q.z;
            v[4] = q.w;
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) v[1 + j] = (xs + j < W) ? __ldg(row + xs + j) : qnan();
        }
    }
};

template <>
struct RowLoader<uint8_t> {
    static __device__ __forceinline__ float at(const uint8_t *__restrict__ row, int64_t x)
    {
        return u8_as_ordered_float((uint32_t)__ldg(row + x), 0);
    }
    static __device__ __forceinline__ void own4(const uint8_t *__restrict__ row, int64_t xs,
                                                int64_t W, bool vec, float v[6])
    {
        if (vec) {
            const uint32_t w = __ldg(reinterpret_cast<const unsigned int *>(row + xs));
#pragma unroll
            for (int j = 0; j < 4; ++j) v[1 + j] = u8_as_ordered_float(w, j);
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                v[1 + j] = (xs + j < W) ? u8_as_ordered_float((uint32_t)__ldg(row + xs + j), 0)
                                        : qnan();
        }
    }
};

// Whole-warp call (shuffles): every lane of the warp must take part with the same row/x0.
template <typename T>
__device__ __forceinline__ void load_row(const T *__restrict__ plane, int64_t Hy, int64_t W,
                                         int64_t y, int64_t x0, int lane, bool vec_ok, float v[6])
{
    if (y < 0 || y >= Hy) {
#pragma unroll
        for (int j = 0; j < 6; ++j) v[j] = qnan();
        return;
    }
    const T *__restrict__ row = plane + y * W;
    const int64_t xs = x0 + 4 * lane;
    const bool vec = vec_ok && (x0 + 128 <= W);
    RowLoader<T>::own4(row, xs, W, vec, v);
    float left = __shfl_up_sync(kFull, v[4], 1);
    float right = __shfl_down_sync(kFull, v[1], 1);
    if (lane == 0) left = (x0 > 0) ? RowLoader<T>::at(row, x0 - 1) : qnan();
    if (lane == kWarp - 1) right = (x0 + 128 < W) ? RowLoader<T>::at(row, x0 + 128) : qnan();
    v[0] = left;
    v[5] = right;
}

// ----------------------------------------------------------------------------------------------
// Keys and the block histogram
// ----------------------------------------------------------------------------------------------

template <typename T>
struct KeyOf;

template <>
struct KeyOf<float> {
    template <int CAP>
    static __device__ __forceinline__ int get(float v, const HardParams<CAP> &P,
                                              const float *__restrict__ T)
    {
        if (P.key_mode == kKeyEstimate)
            return key_estimate(v, P.scale, P.offset, (float)(P.H + 1), T);
        return key_search(v, P.H, T);
    }
};

template <>
struct KeyOf<uint8_t> {
    template <int CAP>
    static __device__ __forceinline__ int get(float v, const HardParams<CAP> &P,
                                              const float *__restrict__ T)
    {
        if (v != v) return P.H;  // absent
        return (int)T[__float_as_int(v) & 0xff];
    }
};

// c[j] belongs to the pixel whose value is row[1 + j].
template <typename T, int CAP>
__device__ __forceinline__ void accumulate4(const int c[4], const float row[6],
                                            const HardParams<CAP> &P,
                                            const float *__restrict__ table, int *hist)
{
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if (c[j] != 0) {
            const int k = KeyOf<T>::template get<CAP>(row[1 + j], P, table);
            if (k < P.H) atomicAdd(hist + k, c[j]);
        }
    }
}

template <int CAP>
__device__ __forceinline__ void block_setup(const HardParams<CAP> &P, int *hist, float *table)
{
    for (int i = threadIdx.x; i < P.H; i += blockDim.x) hist[i] = 0;
    for (int i = threadIdx.x; i < P.table_len; i += blockDim.x) table[i] = P.table[i];
    __syncthreads();
}

// One global atomic per non-empty bin per block ("one global atomic flush per block").
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

constexpr int kHardThreads = 256;
constexpr int kHardWarps = kHardThreads / kWarp;

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
    const bool vec_ok = P.vec_ok != 0;

    for (int64_t t = t_begin + warp; t < t_end; t += kHardWarps) {
        const int64_t strip = t % P.tasks_x;
        const int64_t band = t / P.tasks_x;
        const int64_t x0 = strip * 128;
        const int64_t y0 = band * P.rows_per_task;
        const int64_t y1 = min(y0 + (int64_t)P.rows_per_task, P.Hy);
        float a[6], bb[6], d[6];
        load_row<T>(img, P.Hy, P.W, y0 - 1, x0, lane, vec_ok, a);
        load_row<T>(img, P.Hy, P.W, y0, x0, lane, vec_ok, bb);
        for (int64_t y = y0; y < y1; ++y) {
            load_row<T>(img, P.Hy, P.W, y + 1, x0, lane, vec_ok, d);
            int c[4];
            quad_c2d(a, bb, d, c);
            accumulate4<T, CAP>(c, bb, P, table, hist);
#pragma unroll
            for (int j = 0; j < 6; ++j) {
                a[j] = bb[j];
                bb[j] = d[j];
            }
        }
    }
    block_flush(P, hist, b);
}

// ----------------------------------------------------------------------------------------------
// 3-D kernel
// ----------------------------------------------------------------------------------------------
//
// Work: CTA task = (tile of 128 columns x 8 rows) x (chunk of rows_per_task planes), tile x
// fastest, then tile y, then chunk. Warp w owns row y0 + w of the tile; lane l columns x0+4l..+3.

struct Plane3 {  // rows y-1, y, y+1 of one plane around a lane's four columns
    float r[3][6];
};

template <typename T>
__device__ __forceinline__ void load_plane(const T *__restrict__ img, int64_t D, int64_t Hy, int64_t W, int64_t z,
                                           int64_t y, int64_t x0, int lane, bool vec_ok,
                                           Plane3 &p)
{
    if (z < 0 || z >= D) {
#pragma unroll
        for (int i = 0; i < 3; ++i)
#pragma unroll
            for (int j = 0; j < 6; ++j) p.r[i][j] = qnan();
        return;
    }
    const T *__restrict__ plane = img + z * Hy * W;
#pragma unroll
    for (int i = 0; i < 3; ++i) load_row<T>(plane, Hy, W, y - 1 + i, x0, lane, vec_ok, p.r[i]);
}

__device__ __forceinline__ void plane_max(const Plane3 &s, const Plane3 &u, Plane3 &m)
{
#pragma unroll
    for (int i = 0; i < 3; ++i)
#pragma unroll
        for (int j = 0; j < 6; ++j) m.r[i][j] = max_nan(s.r[i][j], u.r[i][j]);
}

template <typename T, int CAP>
__global__ void __launch_bounds__(kHardThreads) ecc_hard3d_kernel(const __grid_constant__
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
    const bool vec_ok = P.vec_ok != 0;
    const int64_t D = P.D, Hy = P.Hy, W = P.W;

    for (int64_t t = t_begin; t < t_end; ++t) {
        const int64_t tx = t % P.tasks_x;
        const int64_t rest = t / P.tasks_x;
        const int64_t ty = rest % P.tasks_y;
        const int64_t tz = rest / P.tasks_y;
        const int64_t x0 = tx * 128;
        const int64_t y = ty * kHardWarps + warp;
        if (y >= Hy) continue;  // warp-uniform; no block-wide barrier inside the task loop
        const int64_t z0 = tz * P.rows_per_task;
        const int64_t z1 = min(z0 + (int64_t)P.rows_per_task, D);

        Plane3 prev, cur, next, m;
        load_plane<T>(img, D, Hy, W, z0 - 1, y, x0, lane, vec_ok, prev);
        load_plane<T>(img, D, Hy, W, z0, y, x0, lane, vec_ok, cur);
        int cm_prev[4];
        plane_max(prev, cur, m);
        quad_c2d(m.r[0], m.r[1], m.r[2], cm_prev);
        float below[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) below[j] = prev.r[1][1 + j];

        for (int64_t z = z0; z < z1; ++z) {
            load_plane<T>(img, D, Hy, W, z + 1, y, x0, lane, vec_ok, next);
            int cs[4], cm[4], c[4];
            quad_c2d(cur.r[0], cur.r[1], cur.r[2], cs);
            plane_max(cur, next, m);
            quad_c2d(m.r[0], m.r[1], m.r[2], cm);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float v = cur.r[1][1 + j];
                const bool own_up = next.r[1][1 + j] < v;
                const bool own_dn = below[j] <= v;
                c[j] = cs[j] - (own_up ? cm[j] : 0) - (own_dn ? cm_prev[j] : 0);
                cm_prev[j] = cm[j];
                below[j] = v;
            }
            accumulate4<T, CAP>(c, cur.r[1], P, table, hist);
            cur = next;
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
        // inclusive warp scan
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
            warp_sums[lane] = s;  // inclusive prefix of warp totals
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

static int g_num_sms = 0;

static int num_sms()
{
    if (g_num_sms > 0) return g_num_sms;
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) n = 148;
    g_num_sms = n;
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
    P.vec_ok = pl.vec_ok;
    const int ntab = (pl.dtype == ECC_U8) ? 256 : pl.H + 2;
    P.table_len = ntab;
    for (int i = 0; i < ntab; ++i) P.table[i] = pl.table[i];
    for (int i = ntab; i < CAP + 2; ++i) P.table[i] = 0.0f;

    const int sms = num_sms();
    const int64_t resident = (int64_t)sms * 4;  // 4 blocks of 256 threads per SM
    const int64_t strips = (pl.W + 127) / 128;
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
        const int64_t tiles_y = (pl.Hy + kHardWarps - 1) / kHardWarps;
        // planes per task: aim at ~8 tasks per resident block, at least 8 planes each
        int64_t tiles = strips * tiles_y * pl.batch;
        int64_t want = (pl.D * tiles + resident * 8 - 1) / (resident * 8);
        int64_t R = want < 8 ? 8 : (want > 128 ? 128 : want);
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
    if (pl.dtype == ECC_U8) return launch_hard<uint8_t, 256>(pl, s);
    if (pl.H <= 256) return launch_hard<float, 256>(pl, s);
    if (pl.H <= 1024) return launch_hard<float, 1024>(pl, s);
    return launch_hard<float, ECC_MAX_NBINS>(pl, s);
}

}  // namespace ecc
