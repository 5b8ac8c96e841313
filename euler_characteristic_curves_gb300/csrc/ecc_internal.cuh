// ecc_internal.cuh -- shared device helpers of the GB300 ECC library (not part of the ABI).
//
// Method: the paper notes "Scalable GPU-Accelerated Euler Characteristic Curves: Optimization and
// Differentiable Learning for PyTorch" (NeurIPS 2025 NeurReps), "Key designs -- local computation
// of the Euler characteristic coefficient": the ECC is a sum of per-voxel contributions c(p) read
// off the voxel's neighbourhood, accumulated into a threshold histogram.
//
// Vertex-centric decomposition used by every kernel here. Order the voxels by (key, linear
// index), key = threshold bin; a neighbour q is "earlier" than p when key(q) < key(p), or the keys
// are equal and q has the smaller linear index. Every cell of the V-construction is assigned to
// its latest vertex (the max under that order), and c(p) = sum over the cells assigned to p of
// (-1)^dim. The latest vertex of a cell carries the cell's max key, i.e. the cell's bin, so
//     ECC(t_k) = sum over voxels p with key(p) <= k of c(p).
// In a row-major scan, the neighbours with a smaller linear index are exactly those in earlier
// rows/planes or to the left in the same row, so "earlier" is `<=` for them and `<` otherwise.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "ecc.h"

namespace ecc {

constexpr int kWarp = 32;
constexpr unsigned kFull = 0xffffffffu;

// Device error word bits. Bit 0: a kernel gave up waiting for its own staged copy (every build).
// The others are set only by the debug build (ECC_DEBUG_BOUNDS = 1, the library's debug variant),
// which checks data-dependent indices before it uses them and skips the access when a check
// fails (no trap): a histogram bin outside [0, H], a global row or column outside the grid, a
// staged plane's tile outside the volume, a soft-list slot or location outside its tile, a soft
// global index outside the image. Each translation unit keeps its own word; ecc_device_status()
// reads them all.
#ifndef ECC_DEBUG_BOUNDS
#define ECC_DEBUG_BOUNDS 0
#endif
enum DeviceErrorBit : unsigned {
    kErrWaitTimeout = 1u << 0,
    kErrHardBin = 1u << 1,
    kErrHardRow = 1u << 2,
    kErrTmaTile = 1u << 3,
    kErrSoftSlot = 1u << 8,
    kErrSoftLoc = 1u << 9,
    kErrSoftIndex = 1u << 10,
};
// In the debug build: records `bit` in *word when `ok` is false and returns ok; otherwise true.
__device__ __forceinline__ bool bounds_ok(unsigned *word, bool ok, unsigned bit)
{
    if (ECC_DEBUG_BOUNDS && !ok) {
        atomicOr(word, bit);
        return false;
    }
    return true;
}

__device__ __forceinline__ float qnan() { return __int_as_float(0x7fffffff); }

// ------------------------------------------------------------------------------------------
// Kernel parameters
// ------------------------------------------------------------------------------------------

enum KeyMode : int { kKeyEstimate = 0, kKeySearch = 1, kKeyLut = 2 };

// Passed by value as a __grid_constant__ kernel parameter, so concurrent calls on different
// streams each carry their own table. CAP is the table capacity (nbins <= CAP).
template <int CAP>
struct HardParams {
    const void *img;
    int64_t *out;      // [batch][H] int64: zeroed before the launch, unless direct
    int64_t D, Hy, W;  // extents (D = 1 for 2-D)
    int64_t image_elems;
    int H;
    int table_len;  // entries of table[] in use
    int key_mode;
    float key_a, key_b;      // estimator u = sat(v a + b), t = (H - 1/2) - H u
    float key_clo, key_chi;  // (H - 1/2) -+ E, E bounding |t - exact fractional bin|
    int vec_ok;              // rows 16-byte (f32) / 4-byte (u8) aligned and W % 4 == 0
    int sign;                // +1, or -1 to subtract this launch's histogram from out
    // work decomposition. 2-D: warp g of an image takes rows_per_task consecutive strip-rows
    // (one more for the first rows_extra warps); 3-D: tasks are numbered tile-major and block g
    // takes tasks g, g + G, g + 2G, ...
    int rows_per_task;  // 2-D: strip-rows per warp; 3-D: planes per block task
    int rows_extra;
    int tasks_x, tasks_y, tasks_z;
    int64_t tasks_per_image;
    int ctas_per_image;
    int direct;  // 1: one block per image, which stores the running sum itself (no memset, scan)
    int prefix;  // 1: each block adds the running sum of its histogram (no scan launch)
    float table[CAP + 2];  // f32: T_0..T_{H-1}, +inf, +inf;  u8: uint16 key pattern per byte
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
    float key_a, key_b, key_clo, key_chi;
    int vec_ok;
    const void *img;
    int64_t *out;
    const float *table;  // H + 2 thresholds (f32), or 256 uint16 key patterns (u8) in 128 floats
    int sign = 1;        // -1: subtract the histogram from out
    bool scan = true;    // false: leave out as a histogram (the caller scans once at the end)
    bool zero_out = false;  // true: the launcher zeroes out first (when it needs zeroing)
    bool tma = false;       // planned for the TMA-staged 3-D kernel (three blocks per SM)
};
// Launch shape of a hard-ECC call on a device of `sms` SMs (shared by the launcher and
// ecc_hard_launch_info). 2-D: one warp per (strip, row range); TMA-staged 3-D: block g takes a
// contiguous segment of the image's tiles x planes (tile-major), in pieces cut where a tile
// ends; register 3-D: tasks (tile, chunk of planes) taken by the blocks of an image in rounds,
// block g taking tasks g, g + G, ...
struct HardShape {
    int64_t blocks_per_image;
    int64_t tasks_per_image;  // 2-D: (strip, row range) bands; staged 3-D: pieces; 3-D: tasks
    int64_t rows_per_task;    // 2-D: row ranges per strip; staged 3-D: tile-planes per block;
                              // 3-D: planes per chunk
    int64_t tasks_x, tasks_y, tasks_z;
    int64_t rounds;  // staged 3-D: most pieces of a block; 3-D: most tasks of a block; 2-D: 1
    bool direct;     // 2-D: the image's only block stores the curve itself
};
HardShape plan_hard(const HardPlan &pl, int sms);
int num_sms();  // of the current device (148 when the query fails)
// Whether a 3-D call of these sizes and keys takes the TMA-staged kernel when its volume is
// 16-byte aligned.
bool tma3d_shape_ok(const HardPlan &pl);
// Launches the probe of the wait-timeout path (ecc_wait_probe).
cudaError_t wait_probe(unsigned long long limit_ns, cudaStream_t s);
// Device addresses of the error words of the hard and soft kernels (bits above).
cudaError_t hard_error_word(unsigned **p);
cudaError_t soft_error_word(unsigned **p);
cudaError_t hard_run(const HardPlan &pl, cudaStream_t s);
// out[b][k] = running sum over k of out[b][k], for batch rows of H bins
cudaError_t hard_scan(int64_t *out, int H, int64_t batch, cudaStream_t s);
// key constants and threshold table of a hard ECC call (table: ECC_MAX_NBINS + 2 floats)
void hard_keys(int dtype, int nbins, double vmin, double vmax, HardPlan &pl, float *table);

struct SoftLayout {
    int ndim;
    int64_t D, Hy, W, batch;  // D = 1 for 2-D
    int K;
    int ndirs;  // directions u_j (1 for the soft ECC, more for the transform)
    int64_t tiles_x, tiles_y, tiles_z, tiles;  // tiles per image
    size_t off_coords, off_counts, off_entries, off_part, off_scal, total;
};
bool soft_layout(int ndim, const int64_t *dims, int64_t batch, int K, int ndirs, SoftLayout &L);
cudaError_t soft_run_fwd(const SoftLayout &L, const float *img, const float *tau, float lambda,
                         const float *alpha, const float *u, float *out, void *ws, cudaStream_t s);
cudaError_t soft_run_stats(const SoftLayout &L, const void *ws, int64_t *stats, cudaStream_t s);
cudaError_t soft_run_bwd(const SoftLayout &L, const float *img, const float *tau, float lambda,
                         const float *alpha, const float *grad_out, float *grad_tau,
                         float *grad_alpha, float *grad_u, float *grad_img, void *ws,
                         cudaStream_t s);

}  // namespace ecc
