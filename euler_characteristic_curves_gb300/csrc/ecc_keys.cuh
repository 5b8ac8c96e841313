// ecc_keys.cuh -- threshold keys carried as fp16 patterns, and the half2 local-Euler stencil.
//
// Paper notes "Scalable GPU-Accelerated Euler Characteristic Curves: Optimization and
// Differentiable Learning for PyTorch", "Key designs -- local computation of the Euler
// characteristic coefficient": c(p) from the 3x3 neighbourhood, accumulated at p's bin.
//
// Every voxel first gets its exact threshold key k = #{j : t_j < v} (nbins = "never"). The order
// by (key, linear index) refines the bin order, so the vertex-centric decomposition is exact on
// keys. A key is stored as the fp16 bit pattern 0x6400 + k, which is finite, strictly increasing
// in k for k <= 6143, and compares correctly with fp16 comparisons. Two keys share one 32-bit
// register (half2), so each comparison, logic and add instruction below serves two pixels.
//
// Positions outside the grid take the key H ("never enters"), the key of a NaN value: for every
// voxel whose key is below H such a neighbour is never earlier, exactly like a missing vertex
// (the cells through it never enter), and the contributions of voxels with key H are discarded.
// So the kernels read NaN for every position outside the grid and need no boundary branches.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ecc {

constexpr int kWarpLanes = 32;
constexpr uint32_t kKeyBase = 0x6400u;      // fp16 pattern of key 0 (the value 1024.0)
// 1.5 * 2^23 + 0x6400: adding a value t in (-2^22, 2^22) with rounding up gives the float whose
// bit pattern is kMagicKeyBits + ceil(t), so its low 16 bits are the fp16 key pattern of ceil(t).
constexpr float kMagicKey = 12608512.0f;
constexpr uint32_t kMagicKeyBits = 0x4B406400u;

// Estimator constants for float32 keys (host-computed, see ecc_api.cu). With the fractional bin
// t* = (v - vmin) (H - 1) / (vmax - vmin) (key = ceil(t*) clamped to [0, H]) the kernels compute
//     u = sat(v a + b) = sat((H - 1/2 - t*) / H),   t = H - 1/2 - H u,
// so t = t* up to a rounding error below E (E <= 1/4), saturated values land on t = -1/2 (key 0)
// or t = H - 1/2 (key H), and NaN, which saturates to u = 0, gets key H ("never enters").
// ceil(t - E) == ceil(t + E) proves the key; otherwise the threshold table decides.
struct KeyConsts {
    float a, b;      // u = sat(v a + b)
    float nH;        // -H
    float clo, chi;  // H - 1/2 - E, H - 1/2 + E
    int H;
    uint64_t nH2, clo2, chi2, magic2;  // nH, clo, chi and kMagicKey in both halves of a pair
};

// Fast key of one value: returns bits whose low half is the fp16 pattern of ceil(t - E), and ORs
// into `amb` a non-zero value when ceil(t + E) differs (the estimate is then ambiguous).
__device__ __forceinline__ uint32_t key_fast(float v, const KeyConsts &K, uint32_t &amb)
{
    const float u = __saturatef(fmaf(v, K.a, K.b));
    const float lo = __fadd_ru(fmaf(u, K.nH, K.clo), kMagicKey);
    const float hi = __fadd_ru(fmaf(u, K.nH, K.chi), kMagicKey);
    amb |= __float_as_uint(lo) ^ __float_as_uint(hi);
    return __float_as_uint(lo);
}

// Packed fp32 pairs (sm_100-family f32x2 instructions; each element rounds as the scalar op does).
__device__ __forceinline__ uint64_t pk(float a, float b)
{
    return (uint64_t)__float_as_uint(a) | ((uint64_t)__float_as_uint(b) << 32);
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_add_rp(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("add.rp.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint32_t h2_fma(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t h2_neg(uint32_t a)
{
    uint32_t d;
    asm("neg.f16x2 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}

// Fills the packed copies of the estimator constants.
__device__ __forceinline__ void key_pairs(KeyConsts &K)
{
    K.nH2 = pk(K.nH, K.nH);
    K.clo2 = pk(K.clo, K.clo);
    K.chi2 = pk(K.chi, K.chi);
    K.magic2 = pk(kMagicKey, kMagicKey);
}

// Estimated key patterns of two values (low halves 0x6400 + ceil(t - E), as key_fast); ORs into
// `amb` a non-zero value when either estimate is ambiguous. The normalisation saturates value by
// value; the rest runs on packed pairs.
__device__ __forceinline__ void key_fast2(float v0, float v1, const KeyConsts &K, uint32_t &k0,
                                          uint32_t &k1, uint32_t &amb)
{
    const uint64_t u = pk(__saturatef(fmaf(v0, K.a, K.b)), __saturatef(fmaf(v1, K.a, K.b)));
    const uint64_t lo = f2_add_rp(f2_fma(u, K.nH2, K.clo2), K.magic2);
    const uint64_t hi = f2_add_rp(f2_fma(u, K.nH2, K.chi2), K.magic2);
    k0 = (uint32_t)lo;
    k1 = (uint32_t)(lo >> 32);
    amb |= (k0 ^ (uint32_t)hi) | (k1 ^ (uint32_t)(hi >> 32));
}

// Exact key given the fast estimate `lo_bits` (any value whose estimate window holds the key):
// the key is lo or lo + 1, decided by the rounded-down fp32 threshold table T (T[H] = +inf).
// Correct for unambiguous values too (then v <= T[lo]); NaN estimates lo = H and stays there.
__device__ __forceinline__ uint32_t key_fix(float v, uint32_t lo_bits, int H,
                                           const float *__restrict__ T)
{
    const int lo = min((int)(lo_bits & 0xffffu) - (int)kKeyBase, H);
    return kKeyBase + (uint32_t)(lo + (v > T[lo] ? 1 : 0));
}

// Binary search on the table: first k with v <= T[k] (H when none, also for NaN).
__device__ __forceinline__ uint32_t key_search_pattern(float v, int H, const float *__restrict__ T)
{
    int lo = 0, hi = H;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (v <= T[mid])
            hi = mid;
        else
            lo = mid + 1;
    }
    return kKeyBase + (uint32_t)lo;
}

// ------------------------------------------------------------------------------------------
// half2 primitives (inline PTX so that each is exactly one instruction)
// ------------------------------------------------------------------------------------------

// 1.0 / 0.0 per half: a < b, a <= b
__device__ __forceinline__ uint32_t h2_lt(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("set.lt.f16x2.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t h2_le(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("set.le.f16x2.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t h2_add(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t h2_sub(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
// NaN-free max of two key pairs (keys are never NaN)
__device__ __forceinline__ uint32_t h2_max(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("max.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    return __byte_perm(a, b, sel);
}

// A row of keys around a lane's four columns x .. x+3, as half2 pairs:
//   own0 = (k[x], k[x+1]), own1 = (k[x+2], k[x+3]),
//   L0 = (k[x-1], k[x]), R0 = (k[x+1], k[x+2]) (= left pair of own1), R1 = (k[x+3], k[x+4]).
struct KeyRow {
    uint32_t own0, own1, L0, R0, R1;
};

// Lane constants for building rows with two shuffles. The keys just outside a warp's 128-column
// strip travel on the rotated shuffles: lane 31 carries the key left of the strip (column x0 - 1)
// into lane 0, and lane 0 carries the key right of it (column x0 + 128) into lane 31.
struct LaneShuffle {
    int src_l, src_r;    // lane - 1 and lane + 1, modulo 32
    uint32_t sel_l, sel_r;  // byte selectors that splice the side key into the published word
};

__device__ __forceinline__ LaneShuffle lane_shuffle(int lane)
{
    LaneShuffle q;
    q.src_l = (lane + kWarpLanes - 1) & (kWarpLanes - 1);
    q.src_r = (lane + 1) & (kWarpLanes - 1);
    q.sel_l = (lane == kWarpLanes - 1) ? 0x5410u : 0x3210u;  // lane 31: side key in the high half
    q.sel_r = (lane == 0) ? 0x3254u : 0x3210u;               // lane 0: side key in the low half
    return q;
}

// A lane's row from its own pairs and its side key (low half of `side`; lane 0: column x0 + 128,
// lane 31: column x0 - 1, other lanes: ignored). Whole-warp call.
__device__ __forceinline__ KeyRow make_key_row(uint32_t own0, uint32_t own1, uint32_t side,
                                               const LaneShuffle &q)
{
    const uint32_t pub_l = prmt(own1, side, q.sel_l);
    const uint32_t pub_r = prmt(own0, side, q.sel_r);
    const uint32_t left = __shfl_sync(0xffffffffu, pub_l, q.src_l);   // (k[x-2], k[x-1])
    const uint32_t right = __shfl_sync(0xffffffffu, pub_r, q.src_r);  // (k[x+4], k[x+5])
    KeyRow r;
    r.own0 = own0;
    r.own1 = own1;
    r.L0 = prmt(left, own0, 0x5432);
    r.R0 = prmt(own0, own1, 0x5432);
    r.R1 = prmt(own1, right, 0x5432);
    return r;
}

__device__ __forceinline__ KeyRow max_rows(const KeyRow &a, const KeyRow &b)
{
    KeyRow r;
    r.own0 = h2_max(a.own0, b.own0);
    r.own1 = h2_max(a.own1, b.own1);
    r.L0 = h2_max(a.L0, b.L0);
    r.R0 = h2_max(a.R0, b.R0);
    r.R1 = h2_max(a.R1, b.R1);
    return r;
}

// The value bias + c for two pixels at once (c in [-3, 1]; fp16 sums of small integers are
// exact). p: the pixels' keys; L, R: their left and right neighbours; a*, d*: the rows above and
// below, same alignment. Sp = [p < above] (1.0 / 0.0), i.e. "the pixel above is NOT earlier",
// reused from the previous row when marching down.
//   earlier flags:  W = L <= p, E = R < p, N = 1 - Sp, S = d < p, NW = aL <= p, NE = aR <= p,
//                   SW = dL < p, SE = dR < p
//   c = 1 - (W + E + N + S) + N W NW + N E NE + S W SW + S E SE
// Attaching each square to the edge that precedes it around p (N -> E -> S -> W) gives
//   c = 1 - N ~(E NE) - E ~(S SE) - S ~(W SW) - W ~(N NW)
//     = (Sp | E NE) - E ~(S SE) - S ~(W SW) - W (Sp | ~NW),
// four 3-input logic operations on 1.0 patterns (0x3C00): each has a plain (non-negated) flag
// as an AND operand or is an OR of plain flags, so its result is exactly 0 or 1.0.
__device__ __forceinline__ uint32_t lop_or_and(uint32_t a, uint32_t b, uint32_t c)
{
    return a | (b & c);
}
// The same 1.0 / 0.0 flags from the FMA pipe instead of the (half-rate) ALU pipe. Key patterns
// of keys k <= 1024 are the fp16 values 1024 + k, integers below 2048 and so exact, as are their
// differences. Hence [a < p] = sat(p - a), and [a <= p] = sat((p + 1) - a) wherever p + 1 is
// exact, i.e. for every centre with key < 1024. Centres whose key is H ("never") may get a wrong
// flag, but their contributions are discarded. So the forms hold for every table of at most 1024
// bins (checked exhaustively over all key pairs in tests/test_kernel_algebra.py).
__device__ __forceinline__ uint32_t h2_sub_sat(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("sub.rn.sat.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
constexpr uint32_t kOnePair = 0x3C003C00u;  // (1.0, 1.0)
template <bool SAT>
__device__ __forceinline__ uint32_t flag_lt(uint32_t a, uint32_t p)  // [a < p]
{
    return SAT ? h2_sub_sat(p, a) : h2_lt(a, p);
}
template <bool SAT>
__device__ __forceinline__ uint32_t flag_le(uint32_t a, uint32_t p, uint32_t p1)  // [a <= p]
{
    return SAT ? h2_sub_sat(p1, a) : h2_le(a, p);
}

// BIAS: return bias + c; otherwise the plain c (one add fewer).
template <bool SAT, bool BIAS>
__device__ __forceinline__ uint32_t c2_pair(uint32_t p, uint32_t L, uint32_t R, uint32_t aL,
                                            uint32_t aR, uint32_t d, uint32_t dL, uint32_t dR,
                                            uint32_t Sp, uint32_t bias, uint32_t &S_out)
{
    const uint32_t p1 = SAT ? h2_add(p, kOnePair) : p;
    const uint32_t W = flag_le<SAT>(L, p, p1), E = flag_lt<SAT>(R, p);
    const uint32_t S = flag_lt<SAT>(d, p);
    const uint32_t NW = flag_le<SAT>(aL, p, p1), NE = flag_le<SAT>(aR, p, p1);
    const uint32_t SW = flag_lt<SAT>(dL, p), SE = flag_lt<SAT>(dR, p);
    const uint32_t A = lop_or_and(Sp, E, NE);
    const uint32_t B = E & ~(S & SE);
    const uint32_t C = S & ~(W & SW);
    const uint32_t D = W & (Sp | ~NW);
    S_out = S;
    return h2_sub(h2_sub(BIAS ? h2_add(bias, A) : A, B), h2_add(C, D));
}

// Local Euler contributions of the lane's four pixels of row b (rows a above, d below).
// Returns the pairs (bias + c) in c0 (pixels x, x+1) and c1 (x+2, x+3); Sp0/Sp1 carry the
// "pixel above is not earlier" flags in, and the S flags of this row out (for the row below).
template <bool SAT, bool BIAS = true>
__device__ __forceinline__ void c2_quad(const KeyRow &a, const KeyRow &b, const KeyRow &d,
                                        uint32_t bias, uint32_t &Sp0, uint32_t &Sp1, uint32_t &c0,
                                        uint32_t &c1)
{
    uint32_t S0, S1;
    c0 = c2_pair<SAT, BIAS>(b.own0, b.L0, b.R0, a.L0, a.R0, d.own0, d.L0, d.R0, Sp0, bias, S0);
    c1 = c2_pair<SAT, BIAS>(b.own1, b.R0, b.R1, a.R0, a.R1, d.own1, d.R0, d.R1, Sp1, bias, S1);
    Sp0 = S0;
    Sp1 = S1;
}

// Sp for the first row of a band: [b < a] per pixel (the row above is not earlier).
template <bool SAT>
__device__ __forceinline__ void sp_init(const KeyRow &a, const KeyRow &b, uint32_t &Sp0,
                                        uint32_t &Sp1)
{
    Sp0 = flag_lt<SAT>(b.own0, a.own0);
    Sp1 = flag_lt<SAT>(b.own1, a.own1);
}

// 0xFFFF / 0x0000 per half: a < b, a <= b (masks, for selecting with bitwise AND)
__device__ __forceinline__ uint32_t h2_lt_mask(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("set.lt.u32.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t h2_le_mask(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("set.le.u32.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

constexpr uint32_t kBias = 0x65006500u;  // (1280, 1280): contributions carried as 1280 + c
// The pattern of 1280 + c is 0x6500 + c for |c| <= 8, so its low byte is c as a signed byte.

__device__ __forceinline__ int sext_byte0(uint32_t x)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, 0, 0x8880;" : "=r"(d) : "r"(x));
    return (int)d;
}
__device__ __forceinline__ int sext_byte2(uint32_t x)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, 0, 0xAAA2;" : "=r"(d) : "r"(x));
    return (int)d;
}

// Shared-memory reduction without a predicate (the kernels keep histograms in shared memory).
__device__ __forceinline__ void red_shared_add(uint32_t addr, int v)
{
    asm volatile("red.shared.add.s32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Adds the contributions of one pair to the block histogram: pixel key patterns `keys`, values
// `cv` = 1280 + c. `hist_s` is the shared address of the histogram minus 4 * kKeyBase, so a key
// pattern indexes it directly (H + 1 bins: pixels whose key is H, "never", land in the unused bin
// H). Every pixel adds, c = 0 included: that costs fewer issue slots than a predicate or a
// redirect, and measured faster despite the extra same-bin collisions.
__device__ __forceinline__ void hist_pair(uint32_t keys, uint32_t cv, uint32_t hist_s)
{
    red_shared_add(hist_s + ((keys & 0xffffu) << 2), sext_byte0(cv));
    red_shared_add(hist_s + ((keys >> 16) << 2), sext_byte2(cv));
}

}  // namespace ecc
