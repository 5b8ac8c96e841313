/*
 * ecc.h -- C ABI of the GB300 (sm_103a) Euler-characteristic-curve library.
 *
 * Method: the paper notes "Scalable GPU-Accelerated Euler Characteristic Curves: Optimization and
 * Differentiable Learning for PyTorch" (NeurIPS 2025 NeurReps workshop, arXiv 2510.20271):
 *   - "Key designs -- full-scan CUDA kernel": one pass over the whole grid, a privatised histogram
 *     of local Euler contributions per thread block, one global flush per block;
 *   - "Key designs -- local computation of the Euler characteristic coefficient": the ECC is a sum
 *     of per-voxel contributions c(p), each read off the 3x3 (2-D) or 3x3x3 (3-D) neighbourhood;
 *   - "Key designs -- differentiable ECC layer (sigmoid relaxation)": 1[X <= t] becomes
 *     sigma(lambda (t - X)) with X(p) = alpha f(p) + u . x_p; custom forward and backward kernels
 *     return analytic gradients for the thresholds, alpha and u.
 *
 * Conventions shared by every entry point
 *   - Images are C-contiguous, last axis fastest: a batch of 2-D images is [batch][H][W], of 3-D
 *     volumes [batch][D][H][W]. `dims` is a HOST array of `ndim` extents, slowest axis first.
 *   - Pointers named img, out, tau, alpha, u, grad_*, ws are DEVICE pointers owned by the caller;
 *     the library never allocates, frees or retains them, and no call allocates device memory
 *     (ecc_soft_fwd_noalloc uses a fixed array that the loaded library image holds).
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL means the legacy default
 *     stream). Arguments are validated on the host before anything is launched; an invalid call
 *     returns a negative status and touches no memory. A failed launch returns ECC_ECUDA; errors
 *     raised later by a kernel surface at the caller's next synchronisation.
 *   - Apart from that array, the library holds no state between calls; it may be called from
 *     several host threads.
 *   - Cell complex: the V-construction. Voxels are vertices; axis-aligned boxes of side 0 or 1 in
 *     each axis whose corners all lie in the grid are cells (edges, squares, cubes); a cell's value
 *     is the max of its vertices. Voxels outside the grid do not exist.
 */
#ifndef ECC_GB300_ECC_H
#define ECC_GB300_ECC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared here so this header needs no CUDA headers. */
struct CUstream_st;
typedef struct CUstream_st *ecc_stream_t;

/* Element types of the hard-ECC input. */
enum ecc_dtype { ECC_U8 = 0, ECC_F32 = 1 };

/* Status codes. */
enum ecc_status {
    ECC_OK = 0,
    ECC_EINVAL = -1,  /* a NULL pointer, a non-positive size, vmin > vmax, a non-finite bound... */
    ECC_EDTYPE = -2,  /* dtype is not ECC_U8 or ECC_F32 */
    ECC_EDIM = -3,    /* ndim outside the supported set, or an extent < 1 */
    ECC_EWS = -4,     /* workspace NULL or smaller than ecc_soft_workspace_bytes() */
    ECC_ECUDA = -5,   /* a CUDA call failed (no device, launch failure...) */
    ECC_ERANGE = -6,  /* nbins or K above the library maximum, or a size that overflows */
    ECC_ETIMEOUT = -7, /* a kernel gave up waiting for its own staged copy (ecc_device_status) */
    ECC_EBOUNDS = -8   /* debug build: a bounds check failed and its access was skipped */
};

#define ECC_MAX_NBINS 4096 /* largest nbins accepted by ecc_hard */
#define ECC_MAX_EXTENT (1 << 30) /* largest extent of any one axis (ECC_ERANGE above) */
#define ECC_MAX_K 8192     /* largest number of soft thresholds */
#define ECC_MAX_DIRS 4096  /* largest number of directions of the soft transform */

/*
 * Hard Euler characteristic curve of a batch of 2-D images or 3-D volumes.
 *
 * Section "Key designs -- full-scan CUDA kernel" and "local computation of the Euler
 * characteristic coefficient" of the ECC paper notes.
 *
 *   out[b * nbins + k] = sum over cells sigma of image b with every vertex value <= t_k of
 *                        (-1)^dim(sigma)                                            (int64)
 *   t_0 = vmin, t_{nbins-1} = vmax, t_k = vmin + ((vmax - vmin) * k) / (nbins - 1) in fp64;
 *   nbins == 1 gives the single threshold vmax.
 *
 * img     device pointer, batch * prod(dims) elements of type dtype (uint8 or float32), any
 *         alignment (a 16-byte-aligned base with a row length divisible by 4 takes the
 *         vectorised fast path). Values are compared exactly as fp64 against t_k: NaN and
 *         values above vmax never enter; values below vmin enter at t_0.
 * dtype   ECC_U8 or ECC_F32.
 * ndim    2 ([H][W] per image) or 3 ([D][H][W] per image).
 * dims    host array of ndim extents, each >= 1, slowest first; an extent above ECC_MAX_EXTENT
 *         returns ECC_ERANGE (the kernels index rows and columns with 32-bit integers).
 * batch   number of independent images (>= 1, at most 65535); no cell joins two images.
 * nbins   number of thresholds, 1 <= nbins <= ECC_MAX_NBINS.
 * vmin, vmax  finite, vmin <= vmax.
 * out     device pointer to batch * nbins int64; fully overwritten.
 * Returns ECC_OK, or ECC_EINVAL / ECC_EDTYPE / ECC_EDIM / ECC_ERANGE / ECC_ECUDA.
 */
int ecc_hard(const void *img, int dtype, int ndim, const int64_t *dims, int64_t batch, int nbins,
             double vmin, double vmax, int64_t *out, ecc_stream_t stream);

/*
 * Sharded hard ECC: the partial histogram of one piece of a grid, and the running sum that turns
 * summed partials into the curve.
 *
 * Section "Limitations" of the ECC paper notes: the method runs on one device, without batching
 * or multi-GPU execution. The ECC is a sum over cells, and each cell enters at the bin of its
 * largest vertex, so per-bin counts add over pieces that share no cells:
 *   - a batch splits by images (no cell joins two images);
 *   - one volume splits into slabs of planes in which consecutive slabs share one plane. Every
 *     cell lies in some slab, and two consecutive slabs share exactly the cells of their common
 *     plane, so hist(volume) = sum_i hist_3D(slab i) - sum_{i > 0} hist_2D(first plane of slab i).
 * Each rank (or device) adds the partials of its pieces into one int64 [batch][nbins] histogram,
 * the ranks sum their histograms (one all-reduce of batch * nbins int64), and ecc_hist_to_curve
 * turns the sum into the curve ecc_hard would return.
 *
 * ecc_hard_partial: arguments as for ecc_hard, plus
 *   sign  +1 or -1: hist[b * nbins + k] += sign * (sum over the cells of image b whose largest
 *         vertex value first enters at t_k of (-1)^dim). Cells that never enter add nothing.
 *   hist  device int64 [batch][nbins], accumulated into (not zeroed): the caller zeroes it once.
 * ecc_hist_to_curve: hist[b][k] = sum_{j <= k} hist[b][j], in place, for batch rows of nbins.
 * Both are asynchronous on `stream`; calls on one stream accumulate in order. Returns ECC_OK or a
 * negative status (ECC_EINVAL for a sign other than +1 / -1).
 */
int ecc_hard_partial(const void *img, int dtype, int ndim, const int64_t *dims, int64_t batch,
                     int nbins, double vmin, double vmax, int sign, int64_t *hist,
                     ecc_stream_t stream);
int ecc_hist_to_curve(int64_t *hist, int nbins, int64_t batch, ecc_stream_t stream);

/*
 * Launch shape that ecc_hard takes for these sizes -- a diagnostic with no counterpart in the paper
 * notes, for tests and tuning. It validates the shape arguments as ecc_hard does (same status
 * codes) and launches nothing.
 *
 * sm_count  SMs of the device to plan for; <= 0 means the current device's.
 * info      host array of 6 int64, written on success:
 *   info[0] blocks per image
 *   info[1] work items per image: 2-D, (128-column strip, row range) bands, one per warp;
 *           3-D float32 with W % 4 == 0 and nbins <= 256 (the TMA-staged kernel), pieces:
 *           block g takes a contiguous share of the image's (tile of 128 x 32 columns x rows)
 *           x planes, numbered tile by tile, cut into pieces where a tile ends; other 3-D
 *           calls, (tile, chunk of planes) tasks
 *   info[2] 2-D: row ranges per strip; staged 3-D: tile-planes per block (at most); other 3-D:
 *           planes per chunk
 *   info[3] staged 3-D: the most pieces one block walks; other 3-D: rounds, the most tasks
 *           one block walks (block g takes tasks g, g + G, ...); 2-D: 1
 *   info[4] 1 when a 2-D image's only block stores the running sum itself, else 0
 *   info[5] the SM count planned for
 */
int ecc_hard_launch_info(int dtype, int ndim, const int64_t *dims, int64_t batch, int nbins,
                         int sm_count, int64_t *info);

/*
 * Hard ECC of one 3-D volume read in slabs of planes from memory the device need not hold
 * (host memory, pinned or pageable, or device memory), for volumes larger than device memory.
 *
 * Section "Limitations" of the ECC paper notes: the full scan is limited by device memory on
 * very large 3-D grids. Cut the volume into slabs of planes [a_i, b_i] with b_i = a_{i+1}
 * (consecutive slabs share one plane). Every cell of the volume lies in a slab, and the cells of
 * two consecutive slabs overlap in the cells of their shared plane, so for every threshold
 *   ECC(volume) = sum_i ECC_3D(slab i) - sum_{i > 0} ECC_2D(plane a_i).
 * The call computes exactly ecc_hard(volume) this way: slab i is copied into one of two device
 * buffers on a second stream while slab i - 1 is processed on `stream`, every slab and shared
 * plane adds or subtracts its histogram in `out`, and one running sum ends the call.
 *
 * img          the volume [D][H][W] (batch 1), uint8 or float32, in any memory the device can
 *              copy from; page-locked host memory lets the copies overlap the kernels.
 * dims         host array {D, H, W}, each >= 1.
 * nbins, vmin, vmax   as for ecc_hard.
 * slab_planes  planes per slab, >= 2 (each slab after the first advances slab_planes - 1 planes).
 * dev_buf      device scratch of at least ecc_hard_stream_buffer_bytes(dtype, dims,
 *              slab_planes) bytes, 256-byte aligned, caller-owned; contents are overwritten.
 * out          device int64 [nbins]; fully overwritten.
 * The call creates and destroys one stream and four events of its own; it returns once the
 * work is queued (the copies from pageable host memory wait for the host, as cudaMemcpyAsync
 * does). Returns ECC_OK or a negative status (ECC_EWS for a short or misaligned dev_buf).
 */
size_t ecc_hard_stream_buffer_bytes(int dtype, const int64_t *dims, int slab_planes);
int ecc_hard_stream(const void *img, int dtype, const int64_t *dims, int nbins, double vmin,
                    double vmax, int slab_planes, void *dev_buf, size_t dev_buf_bytes,
                    int64_t *out, ecc_stream_t stream);

/*
 * Workspace bytes that ecc_soft_fwd / ecc_soft_bwd need for these sizes (0 when the sizes are
 * invalid). The workspace holds the per-voxel critical list written by the forward call and read
 * by the backward call, plus per-block partial sums.
 */
size_t ecc_soft_workspace_bytes(int ndim, const int64_t *dims, int64_t batch, int K);

/*
 * Soft (sigmoid-relaxed) ECC, forward.
 *
 * Section "Key designs -- differentiable ECC layer (sigmoid relaxation)" of the ECC paper notes.
 *
 *   X(p)        = alpha * f(p) + sum_d u[d] * x_{p,d},  x_{p,d} = (2 i_d - (n_d - 1)) / (n_d - 1)
 *                 (0 on an axis of extent 1): coordinates centred and scaled to [-1, 1].
 *   out[b * K + k] = sum over cells sigma of image b of
 *                 (-1)^dim(sigma) / (1 + exp(-lambda (tau[k] - max_{v in sigma} X(v))))   (fp32)
 *
 * img     device float32 [batch][dims...]; finite values.
 * ndim    2 ([H][W] per image) or 3 ([D][H][W] per volume); u has ndim entries, axis 0 first.
 * tau     device float32 [K] thresholds, any order.
 * K       1 <= K <= ECC_MAX_K.
 * lambda  sigmoid sharpness, finite and > 0.
 * alpha   device float32 [1]; u: device float32 [ndim]. tau, alpha and u are shared by the batch.
 * out     device float32 [batch][K]; fully overwritten.
 * ws      device workspace of at least ecc_soft_workspace_bytes(ndim, dims, batch, K) bytes,
 *         256-byte aligned. The forward call fills it; keep it unchanged for the backward call.
 * Returns ECC_OK or a negative status (ECC_EWS for a missing or short workspace).
 */
int ecc_soft_fwd(const float *img, int ndim, const int64_t *dims, int64_t batch, const float *tau,
                 int K, float lambda, const float *alpha, const float *u, float *out, void *ws,
                 size_t ws_bytes, ecc_stream_t stream);

/*
 * Soft ECC, backward: analytic gradients of L = sum_{b,k} grad_out[b,k] * out[b,k].
 *
 * Section "Key designs -- differentiable ECC layer (sigmoid relaxation)" of the ECC paper notes:
 * the gradients below are evaluated in closed form by the library's own kernels. With
 * s = sigma(lambda (tau_k - X))
 * evaluated at each cell's argmax vertex o (ties: the larger linear index owns the cell):
 *   grad_tau[k]   = sum_{b, cells} grad_out[b,k] (-1)^dim lambda s (1 - s)
 *   dX[b, o]      = - sum_{k, cells owned by o} grad_out[b,k] (-1)^dim lambda s (1 - s)
 *   grad_alpha[0] = sum_{b,p} dX[b,p] f[b,p];   grad_u[d] = sum_{b,p} dX[b,p] x_{p,d}
 *   grad_img      = alpha dX                    (optional; pass NULL to skip)
 *
 * Arguments as for ecc_soft_fwd, with the same img, tau, K, lambda, alpha, u and the workspace
 * filled by the forward call. grad_out: device float32 [batch][K]. grad_tau [K], grad_alpha [1],
 * grad_u [ndim], grad_img [batch][dims...] (nullable): device float32, fully overwritten.
 */
int ecc_soft_bwd(const float *img, int ndim, const int64_t *dims, int64_t batch, const float *tau,
                 int K, float lambda, const float *alpha, const float *u, const float *grad_out,
                 float *grad_tau, float *grad_alpha, float *grad_u, float *grad_img, void *ws,
                 size_t ws_bytes, ecc_stream_t stream);

/*
 * Soft Euler characteristic transform: the soft ECC along several directions at once.
 *
 * Section "Limitations" of the ECC paper notes: the layer takes one direction, while the Euler
 * characteristic transform integrates the curve over many. For direction j (u_j = u[j * ndim ..])
 * the transform's curve is the soft ECC of the filtration X_j = alpha f + u_j . x, exactly as
 * ecc_soft_fwd defines it:
 *   out[(b * ndirs + j) * K + k] = ecc_soft_fwd(image b, u_j)[k]
 * One pass reads each image tile once for all directions.
 *
 * Arguments as for ecc_soft_fwd, plus:
 * u       device float32 [ndirs][ndim] directions (any length, zero allowed).
 * ndirs   1 <= ndirs <= ECC_MAX_DIRS, and batch * ndirs <= 65535.
 * out     device float32 [batch][ndirs][K]; fully overwritten.
 * ws      at least ecc_soft_ect_workspace_bytes(ndim, dims, batch, K, ndirs) bytes, 256-aligned.
 * With ndirs = 1 the calls compute exactly what ecc_soft_fwd / ecc_soft_bwd compute.
 */
size_t ecc_soft_ect_workspace_bytes(int ndim, const int64_t *dims, int64_t batch, int K,
                                    int ndirs);
int ecc_soft_ect_fwd(const float *img, int ndim, const int64_t *dims, int64_t batch,
                     const float *tau, int K, float lambda, const float *alpha, const float *u,
                     int ndirs, float *out, void *ws, size_t ws_bytes, ecc_stream_t stream);

/*
 * Backward pass of the transform: analytic gradients of
 * L = sum_{b,j,k} grad_out[(b * ndirs + j) * K + k] * out[(b * ndirs + j) * K + k].
 * grad_tau [K] and grad_alpha [1] sum over images and directions; grad_u [ndirs][ndim] holds one
 * gradient per direction; grad_img (nullable, [batch][dims...]) sums over directions. All device
 * float32, fully overwritten. Same arguments and workspace as the forward call.
 */
int ecc_soft_ect_bwd(const float *img, int ndim, const int64_t *dims, int64_t batch,
                     const float *tau, int K, float lambda, const float *alpha, const float *u,
                     int ndirs, const float *grad_out, float *grad_tau, float *grad_alpha,
                     float *grad_u, float *grad_img, void *ws, size_t ws_bytes,
                     ecc_stream_t stream);

/* ecc_soft_stats for a workspace filled by ecc_soft_ect_fwd (stats[0] sums over directions). */
int ecc_soft_ect_stats(int ndim, const int64_t *dims, int64_t batch, int K, int ndirs,
                       const void *ws, size_t ws_bytes, int64_t *stats, ecc_stream_t stream);

/*
 * Size of the soft forward pass's work list -- a diagnostic with no counterpart in the paper
 * notes, for sizing and for rooflines: the soft kernels evaluate one sigmoid per (listed voxel,
 * threshold) pair.
 *
 * ws must hold the result of an ecc_soft_fwd (or ecc_soft_bwd) call with the same ndim, dims,
 * batch and K. Writes, asynchronously on `stream`:
 *   stats[0] = number of voxels with a non-zero local contribution c_X(p), summed over the batch
 *   stats[1] = number of tiles whose exponents left the factorised range (their terms take the
 *              direct form, two special-function operations per term instead of one)
 *   stats[2] = number of tiles
 * stats: device int64 [3], overwritten. Returns ECC_OK or a negative status (ECC_EWS for a short
 * or misaligned workspace).
 */
int ecc_soft_stats(int ndim, const int64_t *dims, int64_t batch, int K, const void *ws,
                   size_t ws_bytes, int64_t *stats, ecc_stream_t stream);

/*
 * Soft ECC forward pass that allocates nothing -- no counterpart in the paper notes.
 *
 * For callers that cannot allocate device memory (for example a plugin inside a host framework
 * that owns all device memory and provides no allocator, or a latency-critical loop that cannot
 * afford cudaMalloc's device-wide synchronisation). For 2-D images (ndim must be 2; anything else
 * returns ECC_EDIM) it computes exactly what ecc_soft_fwd computes, with the same arguments minus
 * the workspace: the workspace lives in a library-owned device array of
 * ECC_NOALLOC_SCRATCH_BYTES bytes, which every GPU that loads the library holds until the process
 * exits. The call allocates nothing (no cudaMalloc / cudaFree, no allocating library routine).
 *
 * The array serves as the forward pass's workspace: the part of ecc_soft_workspace_bytes() that
 * the forward pass uses (all of it except the backward-only scalar partials) must fit in
 * ECC_NOALLOC_SCRATCH_BYTES; larger sizes are rejected with ECC_ERANGE before anything runs. At
 * K = 128, up to 15 images of 256 x 256 fit (16 need about 16.5 MiB). Each call looks up the
 * current device's array address (cudaGetSymbolAddress) with that device current; the first call
 * on a device may also load the library's device code there, so make that first call before any
 * stream capture. All calls on a device share one array, which keeps the last call's contents
 * (each call overwrites whatever it reads before reading it): calls whose executions overlap on
 * the GPU race and must be serialised by the caller, e.g. by issuing them on one stream.
 */
#define ECC_NOALLOC_SCRATCH_BYTES (16u << 20)
int ecc_soft_fwd_noalloc(const float *img, int ndim, const int64_t *dims, int64_t batch,
                         const float *tau, int K, float lambda, const float *alpha,
                         const float *u, float *out, ecc_stream_t stream);

/*
 * Status of the current device's kernels -- a safety net with no counterpart in the paper notes.
 *
 * A kernel that stages data with asynchronous copies waits for each copy with a time limit
 * (2 s); if the limit passes, the kernel sets a device error word, leaves its result incomplete
 * and returns instead of hanging. The debug build of the library (built with ECC_DEBUG_BOUNDS=1
 * and loaded by the Python binding when the environment variable ECC_DEBUG is 1) also checks
 * data-dependent indices before using them -- histogram bins, global rows and columns, staged
 * tiles, soft-list slots and locations -- and on a failed check sets a bit of the same word and
 * skips the access (no trap).
 *
 * ecc_device_status synchronises with the device, reads the word (clearing it when `clear` is
 * non-zero) and returns ECC_ETIMEOUT if a wait gave up, ECC_EBOUNDS if a bounds check failed,
 * else ECC_OK (ECC_ECUDA when the device cannot be read). ecc_device_error_bits returns the raw
 * bits (>= 0: bit 0 wait timeout; bit 1 histogram bin, bit 2 global row or column, bit 3 staged
 * tile, bit 8 soft-list slot, bit 9 soft-list location, bit 10 soft global index) or ECC_ECUDA.
 * ecc_debug_build returns 1 for the debug build, 0 otherwise.
 */
int ecc_device_status(int clear);
int64_t ecc_device_error_bits(int clear);
int ecc_debug_build(void);

/*
 * Probe of the wait-timeout path -- a test hook with no counterpart in the paper notes.
 *
 * Launches, on `stream`, one kernel whose single thread waits for an mbarrier phase that nothing
 * completes, with the kernels' bounded wait cut to limit_ns nanoseconds (the kernels' own
 * limit is ECC_WAIT_LIMIT_NS); when the limit passes it records the timeout in the device error
 * word exactly as a kernel whose staged copy is late does, and returns. No copy is in flight and
 * the context stays usable, so afterwards ecc_device_status() returns ECC_ETIMEOUT (and clears
 * the word when asked). Returns ECC_EINVAL for limit_ns <= 0, ECC_ERANGE above
 * ECC_WAIT_LIMIT_NS, ECC_ECUDA if the launch fails, else ECC_OK.
 */
#define ECC_WAIT_LIMIT_NS 2000000000LL
int ecc_wait_probe(int64_t limit_ns, ecc_stream_t stream);

/* Human-readable name of a status code (static storage, never NULL). */
const char *ecc_status_str(int status);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int ecc_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ECC_GB300_ECC_H */
