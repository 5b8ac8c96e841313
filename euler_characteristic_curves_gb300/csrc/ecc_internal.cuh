// ecc_internal.cuh -- shared device helpers of the GB300 ECC library (not part of the ABI).
//
// Method: the paper notes "Scalable GPU-Accelerated Euler Characteristic Curves: Optimization and
// Differentiable Learning for PyTorch" (NeurIPS 2025 NeurReps), "Key designs -- local computation
// of the Euler characteristic coefficient": the ECC is a sum of per-voxel contributions c(p) read
// off the voxel's neighbourhood, accumulated into a threshold histogram.
//
// Vertex-centric decomposition used by every kernel here. Order the voxels by (value, linear
// index); a neighbour q is "earlier" than p when value(q) < value(p), or the values are equal and
// q has the smaller linear index. Every cell of the V-construction is assigned to its latest
// vertex (the max under that order), and c(p) = sum over the cells assigned to p of (-1)^dim.
// The latest vertex of a cell carries the cell's max value, hence the cell's threshold bin, so
//     ECC(t_k) = sum over voxels p with bin(p) <= k of c(p)
// for ANY order that refines the bin order -- raw values with the index tie-break do. Keys (bins)
// are therefore computed only where c(p) != 0.
//
// In a row-major scan, the neighbours with a smaller linear index are exactly those in earlier
// rows/planes or to the left in the same row, so "earlier" is `<=` for them and `<` otherwise.
// NaN stands for "absent" (outside the grid) and "never enters": every comparison with NaN is
// false, so a NaN neighbour is never earlier, and a NaN voxel gets bin nbins (dropped).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "ecc.h"

namespace ecc {

constexpr int kWarp = 32;
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float qnan() { return __int_as_float(0x7fffffff); }

// max that propagates NaN ("never enters" wins), sm_80+ PTX max.NaN.
__device__ __forceinline__ float max_nan(float a, float b)
{
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

// ------------------------------------------------------------------------------------------
// Threshold bins ("key" of a value): key(v) = #{k : t_k < v} = min{k : v <= t_k} (nbins if none)
// ------------------------------------------------------------------------------------------
//
// The host rounds every fp64 threshold t_k DOWN to fp32 (T_k = largest float <= t_k), so for any
// float v:  v <= t_k  <=>  v <= T_k. Table layout: T[0..H-1], then T[H] = T[H+1] = +inf.
//
// Estimator mode (uniform thresholds, well conditioned): t = v * scale + offset approximates the
// fractional bin; the host guarantees |t - exact| < 0.25 bin, so k0 = ceil(clamp(t, 1, H+1)) is
// within one of the key and two table comparisons make it exact. NaN clamps to H+1 -> key H.
__device__ __forceinline__ int key_estimate(float v, float scale, float offset, float Hp1,
                                            const float *__restrict__ T)
{
    float t = fmaf(v, scale, offset);
    t = fmaxf(fminf(t, Hp1), 1.0f);
    int k0 = __float2int_ru(t);
    return k0 - 1 + (v > T[k0 - 1] ? 1 : 0) + (v > T[k0] ? 1 : 0);
}

// Binary-search mode (any nbins, degenerate or badly conditioned ranges): first k with v <= T_k.
__device__ __forceinline__ int key_search(float v, int H, const float *__restrict__ T)
{
    int lo = 0, hi = H;
    while (lo < hi) {
        int mid = (lo + hi) >> 1;
        if (v <= T[mid])
            hi = mid;
        else
            lo = mid + 1;
    }
    return lo;
}

// uint8 inputs are carried as the float 2^23 + byte (exact, order preserving), so the byte is the
// low 8 bits of the float's pattern and the key comes from a 256-entry table.
__device__ __forceinline__ float u8_as_ordered_float(uint32_t word, int byte_index)
{
    return __int_as_float((int)__byte_perm(word, 0x4B000000u, 0x7540u + (unsigned)byte_index));
}

// ------------------------------------------------------------------------------------------
// 2-D local Euler contribution of four horizontally adjacent pixels
// ------------------------------------------------------------------------------------------
//
// a, b, d: rows y-1, y, y+1, six columns each (index 0 = x-1, 1..4 = x..x+3, 5 = x+4).
// For pixel j (1..4) with value v = b[j]:
//   earlier flags  W = b[j-1] <= v, E = b[j+1] < v, N = a[j] <= v, S = d[j] < v,
//                  NW = a[j-1] <= v, NE = a[j+1] <= v, SW = d[j-1] < v, SE = d[j+1] < v
//   c = 1 - (W + E + N + S)                  (the vertex, minus its four edges when owned)
//       + [N W NW] + [N E NE] + [S W SW] + [S E SE]   (each of its four squares when owned)
// A square is owned when its three other corners are earlier; an edge when the other end is.
__device__ __forceinline__ void quad_c2d(const float a[6], const float b[6], const float d[6],
                                         int c[4])
{
#pragma unroll
    for (int j = 1; j <= 4; ++j) {
        const float v = b[j];
        const bool W = b[j - 1] <= v, E = b[j + 1] < v;
        const bool N = a[j] <= v, S = d[j] < v;
        const bool NW = a[j - 1] <= v, NE = a[j + 1] <= v;
        const bool SW = d[j - 1] < v, SE = d[j + 1] < v;
        int r = 1 - (int)W - (int)E - (int)N - (int)S;
        r += (int)(N && W && NW) + (int)(N && E && NE) + (int)(S && W && SW) + (int)(S && E && SE);
        c[j - 1] = r;
    }
}

// ------------------------------------------------------------------------------------------
// Kernel parameters
// ------------------------------------------------------------------------------------------

enum KeyMode : int { kKeyEstimate = 0, kKeySearch = 1, kKeyLut = 2 };

// Passed by value as a __grid_constant__ kernel parameter, so concurrent calls on different
// streams each carry their own table. CAP is the table capacity (nbins <= CAP).
template <int CAP>
struct HardParams {
    const void *img;
    int64_t *out;      // [batch][H] int64, zeroed before the launch
    int64_t D, Hy, W;  // extents (D = 1 for 2-D)
    int64_t image_elems;
    int H;
    int table_len;  // entries of table[] in use
    int key_mode;
    float scale, offset;  // estimator
    int vec_ok;           // rows 16-byte (f32) / 4-byte (u8) aligned and W % 4 == 0
    // work decomposition
    int rows_per_task;    // 2-D: rows per warp task; 3-D: planes per CTA task
    int tasks_x, tasks_y, tasks_z;
    int64_t tasks_per_image;
    int ctas_per_image;
    float table[CAP + 2];  // f32: T_0..T_{H-1}, +inf, +inf;  u8: key of byte b stored as float
};

// ------------------------------------------------------------------------------------------
// Host-side plans shared by the C ABI and the launchers
// ------------------------------------------------------------------------------------------

struct HardPlan {
    int ndim;
    int dtype;
    int64_t D, Hy, W, batch;
    int H;
    int key_mode;
    float scale, offset;
    int vec_ok;
    const void *img;
    int64_t *out;
    const float *table;  // H + 2 entries (f32) or 256 keys (u8)
};
cudaError_t hard_run(const HardPlan &pl, cudaStream_t s);

struct SoftLayout {
    int64_t Hy, W, batch;
    int K;
    int64_t tiles_x, tiles_y, tiles;  // tiles per image
    size_t off_coords, off_counts, off_entries, off_part, off_scal, total;
};
bool soft_layout(int ndim, const int64_t *dims, int64_t batch, int K, SoftLayout &L);
cudaError_t soft_run_fwd(const SoftLayout &L, const float *img, const float *tau, float lambda,
                         const float *alpha, const float *u, float *out, void *ws, cudaStream_t s);
cudaError_t soft_run_bwd(const SoftLayout &L, const float *img, const float *tau, float lambda,
                         const float *alpha, const float *grad_out, float *grad_tau,
                         float *grad_alpha, float *grad_u, float *grad_img, void *ws,
                         cudaStream_t s);

}  // namespace ecc
