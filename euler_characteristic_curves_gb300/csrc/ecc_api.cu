// ecc_api.cu -- the extern "C" entry points declared in include/ecc.h: argument validation, the
// exact fp32 threshold tables and the dispatch to the hard / soft kernels.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "ecc.h"
#include "ecc_internal.cuh"

namespace ecc {

// Thresholds of the hard ECC in fp64: t_0 = vmin, t_{H-1} = vmax, interior
// vmin + ((vmax - vmin) * k) / (H - 1); a single threshold at vmax when H == 1.
static double threshold(int k, int H, double vmin, double vmax)
{
    if (H == 1 || k == H - 1) return vmax;
    if (k == 0) return vmin;
    return vmin + ((vmax - vmin) * (double)k) / (double)(H - 1);
}

// Largest float <= x.
static float round_down_f32(double x)
{
    float f = (float)x;
    if ((double)f > x) f = nextafterf(f, -INFINITY);
    return f;
}

static bool mul_ok(int64_t a, int64_t b, int64_t &r)
{
    if (a < 0 || b < 0) return false;
    if (a != 0 && b > INT64_MAX / a) return false;
    r = a * b;
    return true;
}

// Key constants and threshold table of a hard ECC call (shared by the resident and the streamed
// entry points): the u8 key table, or the fp32 thresholds and the estimator constants.
void hard_keys(int dtype, int nbins, double vmin, double vmax, HardPlan &pl, float *table)
{
    const int H = nbins;
    pl.key_a = pl.key_b = pl.key_clo = pl.key_chi = 0.0f;
    if (dtype == ECC_U8) {
        // fp16 key pattern of every byte value: 0x6400 + (first k with b <= t_k; H if none)
        uint16_t lut[256];
        for (int v = 0; v < 256; ++v) {
            int lo = 0, hi = H;
            while (lo < hi) {
                const int mid = (lo + hi) / 2;
                if ((double)v <= threshold(mid, H, vmin, vmax))
                    hi = mid;
                else
                    lo = mid + 1;
            }
            lut[v] = (uint16_t)(0x6400 + lo);
        }
        memcpy(table, lut, sizeof(lut));
        pl.key_mode = kKeyLut;
    } else {
        for (int k = 0; k < H; ++k) table[k] = round_down_f32(threshold(k, H, vmin, vmax));
        table[H] = table[H + 1] = INFINITY;
        // Estimator of the fractional bin t* = v s + o, s = (H-1)/(vmax-vmin), o = -vmin s (the
        // key is ceil(t*) clamped to [0, H]): u = sat(v a + b), a = -s/H, b = (H - 1/2 - o)/H,
        // t = (H - 1/2) - H u. For an unsaturated value (|v| <= M + (vmax-vmin)/(H-1),
        // M = max(|vmin|, |vmax|)), |t - t*| collects the rounding of a and b (2^-24 |v| s and
        // 2^-24 |H - 1/2 - o|), of the FMA for u (2^-24, times H), of the FMA for t and of the
        // constants H - 1/2 -+ E (2^-24 H each), and the fp64 rounding of the thresholds:
        //     |t - t*| < dev = 2^-24 (M s + |o| + 5 H + 2).
        // The kernel proves a key when ceil(t - E) == ceil(t + E); E = 1.25 dev must stay
        // below 1/4 (then the saturated ends t = -1/2, H - 1/2 are never ambiguous), else
        // every key is binary-searched.
        pl.key_mode = kKeySearch;
        if (H >= 2 && vmax > vmin) {
            const double sc = (double)(H - 1) / (vmax - vmin);
            const double o = -vmin * sc;
            const double M = fmax(fabs(vmin), fabs(vmax));
            const double E = 1.25 * ldexp(1.0, -24) * (M * sc + fabs(o) + 5.0 * H + 2.0);
            if (isfinite(sc) && sc < 1e30 && E <= 0.25) {
                pl.key_mode = kKeyEstimate;
                pl.key_a = (float)(-sc / H);
                pl.key_b = (float)((H - 0.5 - o) / H);
                pl.key_clo = (float)(H - 0.5 - E);
                pl.key_chi = (float)(H - 0.5 + E);
            }
        }
    }
    pl.table = table;
}

}  // namespace ecc

using namespace ecc;

extern "C" {

const char *ecc_status_str(int status)
{
    switch (status) {
    case ECC_OK: return "ECC_OK";
    case ECC_EINVAL: return "ECC_EINVAL: invalid argument";
    case ECC_EDTYPE: return "ECC_EDTYPE: unsupported dtype";
    case ECC_EDIM: return "ECC_EDIM: unsupported ndim or extent";
    case ECC_EWS: return "ECC_EWS: workspace missing or too small";
    case ECC_ECUDA: return "ECC_ECUDA: CUDA error";
    case ECC_ERANGE: return "ECC_ERANGE: size above the library maximum";
    case ECC_ETIMEOUT: return "ECC_ETIMEOUT: a kernel gave up waiting for its own staged copy";
    case ECC_EBOUNDS: return "ECC_EBOUNDS: a debug-build bounds check failed (access skipped)";
    default: return "ECC: unknown status";
    }
}

int ecc_version(void) { return 10100; }

// The OR of the hard and soft device error words (read, and cleared when asked); -1 on failure.
static int64_t device_error_bits(int clear)
{
    unsigned *words[2] = {nullptr, nullptr};
    if (hard_error_word(&words[0]) != cudaSuccess || soft_error_word(&words[1]) != cudaSuccess)
        return -1;
    unsigned bits = 0;
    for (unsigned *w : words) {
        unsigned v = 0;
        if (cudaMemcpy(&v, w, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return -1;
        if (clear && v != 0 && cudaMemset(w, 0, sizeof v) != cudaSuccess) return -1;
        bits |= v;
    }
    return bits;
}

int ecc_device_status(int clear)
{
    const int64_t bits = device_error_bits(clear);
    if (bits < 0) return ECC_ECUDA;
    if (bits & kErrWaitTimeout) return ECC_ETIMEOUT;
    return bits != 0 ? ECC_EBOUNDS : ECC_OK;
}

int64_t ecc_device_error_bits(int clear)
{
    const int64_t bits = device_error_bits(clear);
    return bits < 0 ? (int64_t)ECC_ECUDA : bits;
}

int ecc_debug_build(void) { return ECC_DEBUG_BOUNDS ? 1 : 0; }

int ecc_wait_probe(int64_t limit_ns, ecc_stream_t stream)
{
    if (limit_ns <= 0) return ECC_EINVAL;
    if (limit_ns > ECC_WAIT_LIMIT_NS) return ECC_ERANGE;
    return wait_probe((unsigned long long)limit_ns, (cudaStream_t)stream) == cudaSuccess
               ? ECC_OK
               : ECC_ECUDA;
}

// Sizes of a hard-ECC call: the checks ecc_hard makes on its shape arguments, and the plan's
// extents on success.
static int hard_shape_check(int dtype, int ndim, const int64_t *dims, int64_t batch, int nbins,
                            HardPlan &pl)
{
    if (!dims) return ECC_EINVAL;
    if (dtype != ECC_U8 && dtype != ECC_F32) return ECC_EDTYPE;
    if (ndim != 2 && ndim != 3) return ECC_EDIM;
    for (int d = 0; d < ndim; ++d)
        if (dims[d] < 1) return ECC_EDIM;
    if (batch < 1) return ECC_EINVAL;
    if (nbins < 1) return ECC_EINVAL;
    if (nbins > ECC_MAX_NBINS) return ECC_ERANGE;
    // the kernels index rows, columns and strips with 32-bit integers
    for (int d = 0; d < ndim; ++d)
        if (dims[d] > ECC_MAX_EXTENT) return ECC_ERANGE;
    const int64_t D = ndim == 3 ? dims[0] : 1;
    const int64_t Hy = dims[ndim - 2], W = dims[ndim - 1];
    int64_t plane, elems, total, outn;
    if (!mul_ok(Hy, W, plane) || !mul_ok(plane, D, elems) || !mul_ok(elems, batch, total) ||
        total > ((int64_t)1 << 50) || !mul_ok(batch, nbins, outn) || batch > 65535)
        return ECC_ERANGE;
    // 2-D: one warp per (128-column strip, row range); their count stays below 2^31
    if (ndim == 2 && ((W + 127) / 128) * Hy >= ((int64_t)1 << 31)) return ECC_ERANGE;
    pl.ndim = ndim;
    pl.dtype = dtype;
    pl.D = D;
    pl.Hy = Hy;
    pl.W = W;
    pl.batch = batch;
    pl.H = nbins;
    return ECC_OK;
}

int ecc_hard(const void *img, int dtype, int ndim, const int64_t *dims, int64_t batch, int nbins,
             double vmin, double vmax, int64_t *out, ecc_stream_t stream)
{
    if (!img || !out || !dims) return ECC_EINVAL;
    HardPlan pl;
    const int rc = hard_shape_check(dtype, ndim, dims, batch, nbins, pl);
    if (rc != ECC_OK) return rc;
    if (!isfinite(vmin) || !isfinite(vmax) || !(vmin <= vmax) || !isfinite(vmax - vmin))
        return ECC_EINVAL;
    pl.img = img;
    pl.out = out;
    float table[ECC_MAX_NBINS + 2];
    hard_keys(dtype, nbins, vmin, vmax, pl, table);
    const size_t align = dtype == ECC_U8 ? 4 : 16;
    pl.vec_ok = ((uintptr_t)img % align == 0) && (pl.W % 4 == 0);
    pl.table = table;
    pl.zero_out = true;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (hard_run(pl, s) != cudaSuccess) return ECC_ECUDA;
    return ECC_OK;
}

int ecc_hard_partial(const void *img, int dtype, int ndim, const int64_t *dims, int64_t batch,
                     int nbins, double vmin, double vmax, int sign, int64_t *hist,
                     ecc_stream_t stream)
{
    if (!img || !hist || !dims) return ECC_EINVAL;
    if (sign != 1 && sign != -1) return ECC_EINVAL;
    HardPlan pl;
    const int rc = hard_shape_check(dtype, ndim, dims, batch, nbins, pl);
    if (rc != ECC_OK) return rc;
    if (!isfinite(vmin) || !isfinite(vmax) || !(vmin <= vmax) || !isfinite(vmax - vmin))
        return ECC_EINVAL;
    pl.img = img;
    pl.out = hist;
    float table[ECC_MAX_NBINS + 2];
    hard_keys(dtype, nbins, vmin, vmax, pl, table);
    const size_t align = dtype == ECC_U8 ? 4 : 16;
    pl.vec_ok = ((uintptr_t)img % align == 0) && (pl.W % 4 == 0);
    pl.table = table;
    pl.sign = sign;
    pl.scan = false;     // a histogram: the caller adds partials, then takes one running sum
    pl.zero_out = false; // added to what hist holds
    if (hard_run(pl, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return ECC_ECUDA;
    return ECC_OK;
}

int ecc_hist_to_curve(int64_t *hist, int nbins, int64_t batch, ecc_stream_t stream)
{
    if (!hist) return ECC_EINVAL;
    if (nbins < 1 || batch < 1) return ECC_EINVAL;
    if (nbins > ECC_MAX_NBINS || batch > 65535) return ECC_ERANGE;
    if (hard_scan(hist, nbins, batch, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return ECC_ECUDA;
    return ECC_OK;
}

int ecc_hard_launch_info(int dtype, int ndim, const int64_t *dims, int64_t batch, int nbins,
                         int sm_count, int64_t *info)
{
    if (!info) return ECC_EINVAL;
    HardPlan pl;
    const int rc = hard_shape_check(dtype, ndim, dims, batch, nbins, pl);
    if (rc != ECC_OK) return rc;
    const int sms = sm_count > 0 ? sm_count : num_sms();
    // float32: the thresholds of an ordinary range are estimated (a degenerate range searches)
    pl.key_mode = dtype == ECC_U8 ? kKeyLut : kKeyEstimate;
    pl.tma = tma3d_shape_ok(pl);
    const HardShape sh = plan_hard(pl, sms);
    info[0] = sh.blocks_per_image;
    info[1] = sh.tasks_per_image;
    info[2] = sh.rows_per_task;
    info[3] = sh.rounds;
    info[4] = sh.direct ? 1 : 0;
    info[5] = sms;
    return ECC_OK;
}

size_t ecc_soft_ect_workspace_bytes(int ndim, const int64_t *dims, int64_t batch, int K,
                                    int ndirs)
{
    SoftLayout L;
    if (!soft_layout(ndim, dims, batch, K, ndirs, L)) return 0;
    return L.total;
}

size_t ecc_soft_workspace_bytes(int ndim, const int64_t *dims, int64_t batch, int K)
{
    return ecc_soft_ect_workspace_bytes(ndim, dims, batch, K, 1);
}

static int soft_check(const float *img, int ndim, const int64_t *dims, int64_t batch,
                      const float *tau, int K, float lambda, const float *alpha, const float *u,
                      int ndirs, void *ws, size_t ws_bytes, SoftLayout &L)
{
    if (!img || !dims || !tau || !alpha || !u) return ECC_EINVAL;
    if (ndim != 2 && ndim != 3) return ECC_EDIM;
    for (int d = 0; d < ndim; ++d)
        if (dims[d] < 1) return ECC_EDIM;
    if (batch < 1 || K < 1 || ndirs < 1) return ECC_EINVAL;
    if (K > ECC_MAX_K || ndirs > ECC_MAX_DIRS || batch * ndirs > 65535) return ECC_ERANGE;
    if (!(lambda > 0.0f) || !isfinite(lambda)) return ECC_EINVAL;
    if (!soft_layout(ndim, dims, batch, K, ndirs, L)) return ECC_ERANGE;
    if (L.tiles > 2147483647) return ECC_ERANGE;
    if (!ws || ws_bytes < L.total || ((uintptr_t)ws % 256) != 0) return ECC_EWS;
    return ECC_OK;
}

int ecc_soft_ect_fwd(const float *img, int ndim, const int64_t *dims, int64_t batch,
                     const float *tau, int K, float lambda, const float *alpha, const float *u,
                     int ndirs, float *out, void *ws, size_t ws_bytes, ecc_stream_t stream)
{
    SoftLayout L;
    const int rc =
        soft_check(img, ndim, dims, batch, tau, K, lambda, alpha, u, ndirs, ws, ws_bytes, L);
    if (rc != ECC_OK) return rc;
    if (!out) return ECC_EINVAL;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (soft_run_fwd(L, img, tau, lambda, alpha, u, out, ws, s) != cudaSuccess) return ECC_ECUDA;
    return ECC_OK;
}

int ecc_soft_fwd(const float *img, int ndim, const int64_t *dims, int64_t batch, const float *tau,
                 int K, float lambda, const float *alpha, const float *u, float *out, void *ws,
                 size_t ws_bytes, ecc_stream_t stream)
{
    return ecc_soft_ect_fwd(img, ndim, dims, batch, tau, K, lambda, alpha, u, 1, out, ws,
                            ws_bytes, stream);
}

int ecc_soft_ect_bwd(const float *img, int ndim, const int64_t *dims, int64_t batch,
                     const float *tau, int K, float lambda, const float *alpha, const float *u,
                     int ndirs, const float *grad_out, float *grad_tau, float *grad_alpha,
                     float *grad_u, float *grad_img, void *ws, size_t ws_bytes,
                     ecc_stream_t stream)
{
    SoftLayout L;
    const int rc =
        soft_check(img, ndim, dims, batch, tau, K, lambda, alpha, u, ndirs, ws, ws_bytes, L);
    if (rc != ECC_OK) return rc;
    if (!grad_out || !grad_tau || !grad_alpha || !grad_u) return ECC_EINVAL;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (soft_run_bwd(L, img, tau, lambda, alpha, grad_out, grad_tau, grad_alpha, grad_u, grad_img,
                     ws, s) != cudaSuccess)
        return ECC_ECUDA;
    return ECC_OK;
}

int ecc_soft_bwd(const float *img, int ndim, const int64_t *dims, int64_t batch, const float *tau,
                 int K, float lambda, const float *alpha, const float *u, const float *grad_out,
                 float *grad_tau, float *grad_alpha, float *grad_u, float *grad_img, void *ws,
                 size_t ws_bytes, ecc_stream_t stream)
{
    return ecc_soft_ect_bwd(img, ndim, dims, batch, tau, K, lambda, alpha, u, 1, grad_out,
                            grad_tau, grad_alpha, grad_u, grad_img, ws, ws_bytes, stream);
}

int ecc_soft_ect_stats(int ndim, const int64_t *dims, int64_t batch, int K, int ndirs,
                       const void *ws, size_t ws_bytes, int64_t *stats, ecc_stream_t stream)
{
    if (!dims || !stats) return ECC_EINVAL;
    if (ndim != 2 && ndim != 3) return ECC_EDIM;
    for (int d = 0; d < ndim; ++d)
        if (dims[d] < 1) return ECC_EDIM;
    if (batch < 1 || K < 1 || ndirs < 1) return ECC_EINVAL;
    SoftLayout L;
    if (!soft_layout(ndim, dims, batch, K, ndirs, L)) return ECC_ERANGE;
    if (!ws || ws_bytes < L.total || ((uintptr_t)ws % 256) != 0) return ECC_EWS;
    if (soft_run_stats(L, ws, stats, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return ECC_ECUDA;
    return ECC_OK;
}

int ecc_soft_stats(int ndim, const int64_t *dims, int64_t batch, int K, const void *ws,
                   size_t ws_bytes, int64_t *stats, ecc_stream_t stream)
{
    return ecc_soft_ect_stats(ndim, dims, batch, K, 1, ws, ws_bytes, stats, stream);
}

}  // extern "C"
