// ecc_noalloc.cu -- soft-ECC forward pass that allocates nothing.
//
// For callers that cannot allocate device memory: a plugin embedded in a host framework that owns
// all device memory and gives the plugin no allocator, a latency-critical loop that cannot afford
// cudaMalloc's implicit device-wide synchronisation, or a service that must not grow its memory
// footprint after start-up. They call ecc_soft_fwd_noalloc, which runs the same kernels as
// ecc_soft_fwd but keeps their workspace in a fixed array that the library itself owns.
//
// The array is a file-scope __device__ variable of ECC_NOALLOC_SCRATCH_BYTES bytes: every GPU that
// loads the library holds one until the process exits. Host code cannot use the array's name as
// a device address (on the host it names a stand-in), so every call looks the address up with
// cudaGetSymbolAddress for the current device. The lookup is cheap, and doing it per call keeps
// it right after cudaDeviceReset or a new primary context, where a cached address would be stale.
#include <cuda_runtime.h>
#include <stdint.h>

#include "ecc.h"
#include "ecc_internal.cuh"

namespace ecc {
namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[ECC_NOALLOC_SCRATCH_BYTES];

// Device address of the current device's copy of g_noalloc_scratch.
int scratch_address(void **addr)
{
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
        return ECC_ECUDA;
    *addr = p;
    return ECC_OK;
}

}  // namespace
}  // namespace ecc

using namespace ecc;

extern "C" int ecc_soft_fwd_noalloc(const float *img, int ndim, const int64_t *dims,
                                    int64_t batch, const float *tau, int K, float lambda,
                                    const float *alpha, const float *u, float *out,
                                    ecc_stream_t stream)
{
    if (!img || !dims || !tau || !alpha || !u || !out) return ECC_EINVAL;
    if (ndim != 2) return ECC_EDIM;
    for (int d = 0; d < ndim; ++d)
        if (dims[d] < 1) return ECC_EDIM;
    if (batch < 1 || K < 1) return ECC_EINVAL;
    if (K > ECC_MAX_K || batch > 65535) return ECC_ERANGE;
    if (!(lambda > 0.0f) || !isfinite(lambda)) return ECC_EINVAL;
    SoftLayout L;
    if (!soft_layout(ndim, dims, batch, K, 1, L)) return ECC_ERANGE;
    // the forward pass uses the workspace up to the backward-only scalar partials
    if (L.off_scal > (size_t)ECC_NOALLOC_SCRATCH_BYTES) return ECC_ERANGE;
    void *ws = nullptr;
    const int rc = scratch_address(&ws);
    if (rc != ECC_OK) return rc;
    // Every workspace byte the kernels read is written earlier in the same call (coordinates,
    // per-tile counts, the entries below each count, the partial sums), so the array needs no
    // clearing between calls.
    if (soft_run_fwd(L, img, tau, lambda, alpha, u, out, ws, reinterpret_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return ECC_ECUDA;
    return ECC_OK;
}
