// ecc_stream.cu -- hard ECC of a 3-D volume streamed through the device in slabs of planes.
//
// Paper notes "Scalable GPU-Accelerated Euler Characteristic Curves", "Limitations": the full
// scan is limited by device memory capacity on very large 3-D grids. Consecutive slabs share one
// plane; by inclusion-exclusion over the cells,
//     ECC(volume) = sum_i ECC_3D(slab i) - sum_{i > 0} ECC_2D(first plane of slab i),
// so the kernels of the resident path accumulate signed histograms into one output and a single
// running sum ends the call. Copies run on a stream of the call's own, double-buffered against
// the slab kernels on the caller's stream.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "ecc.h"
#include "ecc_internal.cuh"

namespace ecc {

static size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

// Bytes of one slab buffer (0 on invalid sizes).
static size_t slab_bytes(int dtype, const int64_t *dims, int slab_planes)
{
    if (!dims || (dtype != ECC_U8 && dtype != ECC_F32) || slab_planes < 2) return 0;
    for (int d = 0; d < 3; ++d)
        if (dims[d] < 1 || dims[d] > ECC_MAX_EXTENT) return 0;
    const int64_t planes = slab_planes < dims[0] ? slab_planes : dims[0];
    const double bytes = (double)planes * (double)dims[1] * (double)dims[2] *
                         (dtype == ECC_U8 ? 1.0 : 4.0);
    if (bytes > (double)((int64_t)1 << 46)) return 0;
    return round256((size_t)bytes);
}

struct StreamRes {
    cudaStream_t copy = nullptr;
    cudaEvent_t copied[2] = {nullptr, nullptr}, freed[2] = {nullptr, nullptr};
    ~StreamRes()
    {
        for (int i = 0; i < 2; ++i) {
            if (copied[i]) cudaEventDestroy(copied[i]);
            if (freed[i]) cudaEventDestroy(freed[i]);
        }
        if (copy) cudaStreamDestroy(copy);  // released once its queued copies complete
    }
};

}  // namespace ecc

using namespace ecc;

extern "C" {

size_t ecc_hard_stream_buffer_bytes(int dtype, const int64_t *dims, int slab_planes)
{
    return 2 * slab_bytes(dtype, dims, slab_planes);
}

int ecc_hard_stream(const void *img, int dtype, const int64_t *dims, int nbins, double vmin,
                    double vmax, int slab_planes, void *dev_buf, size_t dev_buf_bytes,
                    int64_t *out, ecc_stream_t stream)
{
    if (!img || !out || !dims) return ECC_EINVAL;
    if (dtype != ECC_U8 && dtype != ECC_F32) return ECC_EDTYPE;
    for (int d = 0; d < 3; ++d)
        if (dims[d] < 1) return ECC_EDIM;
    if (slab_planes < 2 || nbins < 1) return ECC_EINVAL;
    if (nbins > ECC_MAX_NBINS) return ECC_ERANGE;
    if (!isfinite(vmin) || !isfinite(vmax) || !(vmin <= vmax) || !isfinite(vmax - vmin))
        return ECC_EINVAL;
    const size_t one = slab_bytes(dtype, dims, slab_planes);
    if (one == 0) return ECC_ERANGE;
    if (!dev_buf || dev_buf_bytes < 2 * one || ((uintptr_t)dev_buf % 256) != 0) return ECC_EWS;

    const int64_t D = dims[0], Hy = dims[1], W = dims[2];
    const size_t elem = dtype == ECC_U8 ? 1 : 4;
    const size_t plane_bytes = (size_t)Hy * (size_t)W * elem;
    HardPlan base;
    float table[ECC_MAX_NBINS + 2];
    hard_keys(dtype, nbins, vmin, vmax, base, table);
    base.dtype = dtype;
    base.Hy = Hy;
    base.W = W;
    base.batch = 1;
    base.H = nbins;
    base.out = out;
    base.vec_ok = (W % 4 == 0);  // the slab buffers are 256-byte aligned
    base.scan = false;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    StreamRes res;
    if (cudaStreamCreateWithFlags(&res.copy, cudaStreamNonBlocking) != cudaSuccess)
        return ECC_ECUDA;
    for (int i = 0; i < 2; ++i)
        if (cudaEventCreateWithFlags(&res.copied[i], cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&res.freed[i], cudaEventDisableTiming) != cudaSuccess)
            return ECC_ECUDA;
    if (cudaMemsetAsync(out, 0, sizeof(int64_t) * (size_t)nbins, s) != cudaSuccess)
        return ECC_ECUDA;
    // the copy stream starts after everything queued on `stream` so far (the caller's producers
    // of img, and the zeroing of out)
    if (cudaEventRecord(res.freed[1], s) != cudaSuccess ||
        cudaStreamWaitEvent(res.copy, res.freed[1], 0) != cudaSuccess)
        return ECC_ECUDA;

    const char *src = static_cast<const char *>(img);
    for (int64_t a = 0, i = 0;; ++i) {
        const int64_t b = (a + slab_planes - 1 < D - 1) ? a + slab_planes - 1 : D - 1;
        const int64_t n = b - a + 1;
        const int k = (int)(i & 1);
        char *buf = static_cast<char *>(dev_buf) + k * one;
        // copy slab i once the kernels that read this buffer (slab i - 2) are done
        if (i >= 2 && cudaStreamWaitEvent(res.copy, res.freed[k], 0) != cudaSuccess)
            return ECC_ECUDA;
        if (cudaMemcpyAsync(buf, src + (size_t)a * plane_bytes, (size_t)n * plane_bytes,
                            cudaMemcpyDefault, res.copy) != cudaSuccess ||
            cudaEventRecord(res.copied[k], res.copy) != cudaSuccess ||
            cudaStreamWaitEvent(s, res.copied[k], 0) != cudaSuccess)
            return ECC_ECUDA;
        HardPlan pl = base;  // + ECC_3D(slab)
        pl.ndim = 3;
        pl.D = n;
        pl.img = buf;
        pl.sign = 1;
        if (hard_run(pl, s) != cudaSuccess) return ECC_ECUDA;
        if (i > 0) {  // - ECC_2D(plane a), shared with the previous slab
            HardPlan pp = base;
            pp.ndim = 2;
            pp.D = 1;
            pp.img = buf;
            pp.sign = -1;
            if (hard_run(pp, s) != cudaSuccess) return ECC_ECUDA;
        }
        if (cudaEventRecord(res.freed[k], s) != cudaSuccess) return ECC_ECUDA;
        if (b == D - 1) break;
        a = b;
    }
    if (hard_scan(out, nbins, 1, s) != cudaSuccess) return ECC_ECUDA;
    return ECC_OK;
}

}  // extern "C"
