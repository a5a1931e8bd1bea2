// router.cu -- RMSNorm, fp32 gate and GatingTopK.
//
// "NPU HunyuanImage-3.0模型推理优化实践": "RmsNorm算子优化" (RMSNorm before
// the MoE block), "消除gate计算冗余cast算子" (the gate runs in fp32 on the
// hidden states cast to float, autocast off) and "MoE EP优化" (GatingTopK).
//
// Two gates.  The sequential one (router_kernel, router_small_kernel below)
// reproduces the plain fp32 loop bit for bit; the layer uses it for batches
// of at most 512 tokens and on request.  For larger batches the layer runs
// the tensor-core gate (end of this file): RMSNorm alone (rmsnorm_kernel),
// the exact three-way bf16 split of the gate weight, the grouped GEMM kernel
// for the partial logits, and gate_combine_kernel (the fp32 sum of the
// parts, top-k, weights and the routing histogram).
//
// RMSNorm's sum of squares is the exact sum of the bf16 squares rounded once
// to fp32 (see "sum of squares" below): every kernel here takes it with one
// warp per row, in parallel, and they all give the same bits.
//
// The sequential router: one CTA owns 32 tokens and 64 experts:
//   phase 1 (RMSNorm only): each of the 4 warps takes the sum of squares of
//     every 4th row, reading it from memory;
//   phase 2: 32-wide slices of the normalised rows (bf16-rounded, then fp32)
//     and of the gate weight are staged in shared memory; every thread owns
//     4 tokens x 4 experts and accumulates each logit with one FMA per term
//     in ascending h.  These are the same fp32 operations in the same order
//     as a plain sequential loop, so the logits (and every routing decision
//     taken on them) are bit-identical to it;
//   phase 3 (E <= 64): warp-per-token top-k / softmax, the routing
//     histogram of the 32-token chunk, and the logits row write-out.
// Batches of at most 512 tokens use router_small_kernel instead (one thread
// per expert, one token per CTA up to one CTA per SM, two tokens per CTA
// beyond), which keeps every SM busy; the routing histogram is then counted
// by the scan (routing.cu).
// This gate is plain fp32 FMA work (2*T*H*E flops); the tensor cores' fp32
// input mode (tf32) would round the inputs, hence the exact bf16 split of the
// other gate.
#include <math.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int RT_THREADS = 128;
constexpr int RT_TOK = kChunkTokens;     // 32
constexpr int RT_EXP = kRouterExperts;   // 64
constexpr int G_HC = 32;                 // h per gate slice
constexpr int G_LD = 36;                 // padded fp32 row stride
constexpr int G_STAGES = 3;              // cp.async ring depth of the gate slices

constexpr int WG_STAGE = RT_EXP * G_LD * 4;                                // 9216
constexpr int XR_STAGE = RT_TOK * G_HC * 2;                                // 2048
constexpr int SMEM_XS = 2 * RT_TOK * G_LD * 4;                             // 9216
constexpr int SMEM_G = G_STAGES * (WG_STAGE + XR_STAGE) + SMEM_XS;         // 43008
constexpr int SMEM_LG = RT_TOK * (RT_EXP + 1) * 4;                         // 8320
constexpr int SMEM_MAIN = SMEM_G;
constexpr int SMEM_TOTAL = SMEM_MAIN + SMEM_LG + RT_TOK * 4 + RT_EXP * 4;

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem)),
                 "l"(reinterpret_cast<uint64_t>(gmem)), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
    return va > vb || (va == vb && ia < ib);
}

// Warp-wide top-k over values spread as v[i] = value of expert lane + 32*i
// (-inf where the expert does not exist).  Lane j < k receives slot j's
// expert in *sel_e and its logit in *sel_v.
template <int NV>
__device__ __forceinline__ void warp_topk(const float (&v)[NV], int k, int *sel_e,
                                          float *sel_v) {
    const int lane = threadIdx.x & 31;
    uint32_t taken = 0;
    *sel_e = -1;
    *sel_v = -INFINITY;
    for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int bi = 0x7FFFFFFF;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int e = lane + 32 * i;
            if (!((taken >> i) & 1u) && better(v[i], e, bv, bi)) {
                bv = v[i];
                bi = e;
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
            if (better(ov, oi, bv, bi)) {
                bv = ov;
                bi = oi;
            }
        }
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        if (lane == j) {
            *sel_e = bi;
            *sel_v = bv;
        }
    }
}

__device__ __forceinline__ float warp_sum(float s) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    return s;
}

// Softmax weights of the chosen slots.  Lane j < k holds slot j (sel_v); m is
// slot 0's logit (the row maximum).  renorm: divide by the sum over the k
// chosen; otherwise by the sum over all experts (v[], -inf for absent ones).
template <int NV>
__device__ __forceinline__ float slot_weight(const float (&v)[NV], int k, bool renorm,
                                             float sel_v) {
    const int lane = threadIdx.x & 31;
    const float m = __shfl_sync(0xffffffffu, sel_v, 0);
    const float ej = lane < k ? expf(sel_v - m) : 0.0f;
    float den;
    if (renorm) {
        den = warp_sum(ej);
    } else {
        float s = 0.0f;
#pragma unroll
        for (int i = 0; i < NV; ++i) s += expf(v[i] - m);   // exp(-inf) = 0
        den = warp_sum(s);
    }
    return ej / den;
}

// ---------------------------------------------------------------- sum of squares
// The RMSNorm's sum of squares is the exact sum of the squares of a bf16 row
// rounded once to fp32 (nearest, ties to even), a value that does not depend
// on a summation order, so one warp sums a row in parallel.
//
// Fast path (finite rows whose largest |x| lies in [2^-20, 2^40]), on packed
// fp32 pairs (one instruction for two values).  With ex the exponent of the
// largest |x|, every square v is below 2^(2ex+2) and exact in fp32 (16
// significant bits; see below for |x| < 2^-63).  Per group of at most 64
// squares (one half of the pairs of 16 vectors of a lane) two accumulators
// are kept inside one binade each, so that every addition into them is an
// error-free transformation of round-to-nearest (the accumulator is the
// larger operand):
//   a1 starts at s1 = 2^(2ex+9) and stays below s1 + 2^(2ex+8), on the grid
//      u1 = 2^(2ex-14):  t = a1 + v,  r1 = v - (t - a1) exactly,  a1 = t,
//      so |r1| <= u1 / 2;
//   a2 starts at s2 = 3 2^(2ex-8) and stays within s2 +- 2^(2ex-9), on the
//      grid u2 = 2^(2ex-30):  t = a2 + r1,  e = r1 - (t - a2) exactly,
//      a2 = t, so |e| <= u2 / 2.
// a1 - s1 and a2 - s2 are then exact integers in units u1 and u2 (signed for
// a2), summed across the lanes as integers, giving T = sum(v - e) / u2
// exactly.  The e are summed in fp32 (A, in units of u2 after scaling); a
// value passes through at most m = 4 vpl + 5 roundings (vpl vectors per
// lane: 4 vpl per pair half, the halves, five butterfly steps), so the
// error is at most m 2^-24 (1 + 2^-20) sum|e| <= (4 vpl + 5) vpl 2^-17 u2.
// A nonzero |x| below 2^-63 has an inexact fp32 square (at most 2^-149 off,
// or zero), which moves the sum by at most H 2^-149, below 2^-66 u2 for
// ex >= -20.  The exact sum is thus within E of T + A.  The ends T + A -+ E
// are taken in 64-bit fixed point with 16 fractional bits (T below 2^46,
// else the slow path; A rounded down for the lower end and up for the upper
// one; E rounded up with at least one unit to spare).  Rounded to 24 bits,
// both ends giving the same fp32 value decides the result; otherwise (the
// interval holds a rounding tie, or the sum sits exactly on one) the slow
// path decides.  All of it is fp32 and integer arithmetic: the fp64 rate of
// the part is a small fraction of its fp32 rate.
// Slow path: every square m^2 * 2^(2E-268) (m the 8-bit significand, E the
// biased exponent, at least 1) is added exactly into a fixed-point number of
// 20 32-bit limbs per lane (unit 2^-266), the lanes' numbers are added
// exactly across the warp, and the total is rounded (to 24 significant bits,
// or to a multiple of 2^-149 in fp32's subnormal range; infinity past the
// largest fp32).
constexpr int SQ_LIMBS = 20;

__device__ __forceinline__ uint32_t warp_max_u32(uint32_t v) {
    return __reduce_max_sync(0xffffffffu, v);
}
__device__ __forceinline__ long long warp_sum_ll(long long v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// Slow path: exact fixed-point sum of the squares of the row (nvec vectors of
// 8 bf16, lanes take vectors lane, lane + 32, ...), rounded; every lane
// returns the result.
__device__ __noinline__ float sumsq_row_exact(const uint4 *row, int nvec) {
    const int lane = threadIdx.x & 31;
    uint32_t acc[SQ_LIMBS];
#pragma unroll
    for (int j = 0; j < SQ_LIMBS; ++j) acc[j] = 0u;
    for (int v = lane; v < nvec; v += 32) {
        const uint4 q = row[v];
        const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
        for (int i = 0; i < 8; ++i) {
            const uint32_t b = (i & 1) ? (wd[i >> 1] >> 16) : (wd[i >> 1] & 0xFFFFu);
            const uint32_t e = (b >> 7) & 0xFFu;
            const uint32_t m = (b & 0x7Fu) | (e ? 0x80u : 0u);
            if (m == 0u) continue;
            const uint32_t sh = 2u * (e ? e : 1u) - 2u;     // bit of the square's unit
            const uint64_t val = static_cast<uint64_t>(m * m) << (sh & 31u);   // < 2^47
            uint32_t j = sh >> 5;
            uint64_t carry = (val & 0xFFFFFFFFull);
            carry += acc[j];
            acc[j] = static_cast<uint32_t>(carry);
            carry = (carry >> 32) + (val >> 32);
            for (++j; carry != 0u && j < SQ_LIMBS; ++j) {
                carry += acc[j];
                acc[j] = static_cast<uint32_t>(carry);
                carry >>= 32;
            }
        }
    }
    // add the lanes' numbers: lane 0 ends with the total
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        uint64_t carry = 0;
#pragma unroll
        for (int j = 0; j < SQ_LIMBS; ++j) {
            const uint32_t o = __shfl_down_sync(0xffffffffu, acc[j], off);
            carry += static_cast<uint64_t>(acc[j]) + o;
            acc[j] = static_cast<uint32_t>(carry);
            carry >>= 32;
        }
    }
    float res = 0.0f;
    if (lane == 0) {
        int top = -1;
        for (int j = SQ_LIMBS - 1; j >= 0 && top < 0; --j)
            if (acc[j]) top = 32 * j + 31 - __clz(acc[j]);
        if (top >= 0) {
            auto bit = [&](int i) { return (acc[i >> 5] >> (i & 31)) & 1u; };
            const int lsb = max(top - 23, 117);             // bit 117 = 2^-149
            uint32_t q = 0;
            for (int i = top; i >= lsb; --i) q = (q << 1) | bit(i);
            if (bit(lsb - 1)) {
                bool rest = false;
                for (int i = lsb - 2; i >= 0 && !rest; --i) rest = bit(i) != 0u;
                if (rest || (q & 1u)) ++q;
            }
            // q * 2^(lsb - 266), q <= 2^24: exact in double, and either an exact
            // fp32 value or at least 2^128, which the conversion turns into inf
            res = static_cast<float>(ldexp(static_cast<double>(q), lsb - 266));
        }
    }
    return __shfl_sync(0xffffffffu, res, 0);
}

// v / 2^16 (v > 0 in fixed point with 16 fractional bits, its integer part
// at least 2^29 in units u2) rounded to 24 significant bits, nearest-even:
// the rounded value in units u2, an integer of at most 24 significant bits.
// (At least 2^29: the largest square alone is at least 2^30 u2, the error
// terms below 2^19 u2 for the row lengths taken here.)
__device__ __forceinline__ long long round24_fx16(long long v) {
    const int shift = (63 - __clzll(v)) - 23;       // >= 23: drops the fraction too
    const long long q = v >> shift;
    const long long rem = v & ((1ll << shift) - 1);
    const long long half = 1ll << (shift - 1);
    const bool up = rem > half || (rem == half && (q & 1));
    return (q + (up ? 1 : 0)) << (shift - 16);
}

// Packed fp32 pairs (the two halves of a 64-bit register): one instruction
// works on both values.
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// a bf16 pair word -> the fp32 pair (low value, high value)
__device__ __forceinline__ uint64_t f2_from_bf16x2(uint32_t w) {
    return static_cast<uint64_t>(w << 16) | (static_cast<uint64_t>(w & 0xFFFF0000u) << 32);
}
__device__ __forceinline__ uint64_t f2_splat(float v) {
    const uint64_t u = __float_as_uint(v);
    return u | (u << 32);
}
__device__ __forceinline__ float f2_lo(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v)); }
__device__ __forceinline__ float f2_hi(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v >> 32)); }
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Scales of the fast path for the row's largest exponent ex: s1, s2 and the
// factors that turn multiples of u1 and u2 into integers.
struct SumsqScales {
    float s1, s2, k1, k2;
};
__device__ __forceinline__ float pow2f(int e) {   // 2^e, e in fp32's normal range
    return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
}
__device__ __forceinline__ SumsqScales sumsq_scales(int ex) {
    return SumsqScales{pow2f(2 * ex + 9), 3.0f * pow2f(2 * ex - 8), pow2f(14 - 2 * ex),
                       pow2f(30 - 2 * ex)};
}

// Pass 1 over a vector: the packed maximum of its 16-bit magnitudes.
__device__ __forceinline__ uint32_t sumsq_vmax(uint32_t mx, const uint4 &q) {
    mx = max_u16x2(mx, q.x & 0x7FFF7FFFu);
    mx = max_u16x2(mx, q.y & 0x7FFF7FFFu);
    mx = max_u16x2(mx, q.z & 0x7FFF7FFFu);
    return max_u16x2(mx, q.w & 0x7FFF7FFFu);
}

// Pass 1 across the warp: true = the fast path applies (ex set), else *early
// is the result to return now (+0 for an all-zero row, inf/NaN for a
// non-finite one) or *slow asks for the slow path.
__device__ __forceinline__ bool sumsq_plan(uint32_t mx, int *ex, float *early, bool *slow) {
    const uint32_t amax = warp_max_u32(max(mx & 0xFFFFu, mx >> 16) << 16);
    *slow = false;
    if (amax == 0u) {
        *early = 0.0f;
        return false;
    }
    if (amax >= 0x7F800000u) {
        *early = __uint_as_float(amax);   // inf, or NaN
        return false;
    }
    *ex = static_cast<int>(amax >> 23) - 127;
    if (*ex < -20 || *ex > 40) {
        *slow = true;
        return false;
    }
    return true;
}

// Pass 2 over one word (two bf16 values): the squares added into a1, their
// rounding errors into a2, and those rounding errors into a3.
__device__ __forceinline__ void sumsq_word(uint32_t w, uint64_t &a1, uint64_t &a2, uint64_t &a3) {
    const uint64_t x2 = f2_from_bf16x2(w);
    const uint64_t sq = f2_mul(x2, x2);
    const uint64_t t1 = f2_add(a1, sq);
    const uint64_t r1 = f2_sub(sq, f2_sub(t1, a1));
    a1 = t1;
    const uint64_t t2 = f2_add(a2, r1);
    a3 = f2_add(a3, f2_sub(r1, f2_sub(t2, a2)));
    a2 = t2;
}

// A group's exact accumulator offsets (both halves) as integers in units u1,
// u2 (the subtractions are exact: each accumulator stays within a factor of
// two of its start).
__device__ __forceinline__ void sumsq_group_end(uint64_t a1, uint64_t a2, const SumsqScales &sc,
                                                long long &n1, long long &n2) {
    const uint64_t d1 = f2_sub(a1, f2_splat(sc.s1)), d2 = f2_sub(a2, f2_splat(sc.s2));
    n1 += __float2ll_rn(__fmul_rn(f2_lo(d1), sc.k1)) + __float2ll_rn(__fmul_rn(f2_hi(d1), sc.k1));
    n2 += __float2ll_rn(__fmul_rn(f2_lo(d2), sc.k2)) + __float2ll_rn(__fmul_rn(f2_hi(d2), sc.k2));
}

// The lanes' integer sums and residual sums -> the rounded result, or the
// slow path when the error interval holds a rounding tie.  vpl: vectors per
// lane at most.
__device__ __forceinline__ float sumsq_finish(long long n1, long long n2, uint64_t a3, int ex,
                                              int vpl, const SumsqScales &sc, const uint4 *row,
                                              int nvec) {
    // A lane's |n1| and |n2| are each below ceil(vpl / 16) 2^23 (per group of
    // 16 vectors, two pair halves of 64 terms below 2^22 units each): up to
    // 64 vectors per lane the warp's sums fit 32 bits and take one reduction
    // instruction each.
    if (vpl <= 64) {
        n1 = __reduce_add_sync(0xffffffffu, static_cast<int>(n1));
        n2 = __reduce_add_sync(0xffffffffu, static_cast<int>(n2));
    } else {
        n1 = warp_sum_ll(n1);
        n2 = warp_sum_ll(n2);
    }
    float r = __fadd_rn(f2_lo(a3), f2_hi(a3));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) r = __fadd_rn(r, __shfl_xor_sync(0xffffffffu, r, off));
    const long long T = (n1 << 16) + n2;          // units u2 = 2^(2ex - 30)
    if (T >= (1ll << 46) || nvec > (1 << 17)) return sumsq_row_exact(row, nvec);
    // A = r / u2 exactly in fp32 (a power-of-two scaling), |A| <= H / 2; in
    // fixed point with 16 fractional bits, rounded down and up
    const float a16 = __fmul_rn(__fmul_rn(r, sc.k2), 65536.0f);
    const long long a_lo = __float2ll_rd(a16), a_hi = __float2ll_ru(a16);
    // E = (4 vpl + 5) vpl 2^-17 u2 = (4 vpl + 5) vpl / 2 units, rounded up
    // with more than one unit to spare
    const long long err = (4ll * vpl + 6) * vpl / 2 + 2;
    const long long base = T << 16;
    const long long lo = base + a_lo - err;
    const long long hi = base + a_hi + err;
    const long long res = round24_fx16(lo);
    if (round24_fx16(hi) != res) return sumsq_row_exact(row, nvec);
    // res has at most 24 significant bits: exact in fp32, and so is the
    // power-of-two scaling (the result is normal)
    return __fmul_rn(__ll2float_rn(res), pow2f(2 * ex - 30));
}

// The row's exact sum of squares rounded to fp32, by one warp, from the
// lane's VPL vectors held in registers (vector lane + 32 i of the row; the
// caller passes zeros past the row's nvec vectors).  `row` is the row in
// memory, for the slow path.
template <int VPL>
__device__ __forceinline__ float warp_sumsq_rn_packed(const uint4 (&vec)[VPL], const uint4 *row,
                                                      int nvec) {
    uint32_t mx = 0u;
#pragma unroll
    for (int i = 0; i < VPL; ++i) mx = sumsq_vmax(mx, vec[i]);
    int ex = 0;
    float early = 0.0f;
    bool slow;
    if (!sumsq_plan(mx, &ex, &early, &slow)) return slow ? sumsq_row_exact(row, nvec) : early;
    const SumsqScales sc = sumsq_scales(ex);
    const uint64_t s1 = f2_splat(sc.s1), s2 = f2_splat(sc.s2);   // accumulator starts
    long long n1 = 0, n2 = 0;
    uint64_t a3 = 0;
#pragma unroll
    for (int g = 0; g < VPL; g += 16) {
        uint64_t a1 = s1, a2 = s2;     // 64 squares per half at most
#pragma unroll
        for (int i = g; i < g + 16 && i < VPL; ++i) {
            sumsq_word(vec[i].x, a1, a2, a3);
            sumsq_word(vec[i].y, a1, a2, a3);
            sumsq_word(vec[i].z, a1, a2, a3);
            sumsq_word(vec[i].w, a1, a2, a3);
        }
        sumsq_group_end(a1, a2, sc, n1, n2);
    }
    return sumsq_finish(n1, n2, a3, ex, VPL, sc, row, nvec);
}

// The same, reading the row (global or shared memory) twice instead of
// holding it in registers.
__device__ float warp_sumsq_rn_mem(const uint4 *row, int nvec) {
    const int lane = threadIdx.x & 31;
    uint32_t mx = 0u;
    for (int v = lane; v < nvec; v += 32) mx = sumsq_vmax(mx, row[v]);
    int ex = 0;
    float early = 0.0f;
    bool slow;
    if (!sumsq_plan(mx, &ex, &early, &slow)) return slow ? sumsq_row_exact(row, nvec) : early;
    const SumsqScales sc = sumsq_scales(ex);
    const uint64_t s1 = f2_splat(sc.s1), s2 = f2_splat(sc.s2);   // accumulator starts
    long long n1 = 0, n2 = 0;
    uint64_t a3 = 0;
    for (int v0 = lane; v0 < nvec; v0 += 32 * 16) {
        uint64_t a1 = s1, a2 = s2;     // 64 squares per half at most
#pragma unroll 4
        for (int v = v0; v < v0 + 32 * 16 && v < nvec; v += 32) {
            const uint4 q = row[v];
            sumsq_word(q.x, a1, a2, a3);
            sumsq_word(q.y, a1, a2, a3);
            sumsq_word(q.z, a1, a2, a3);
            sumsq_word(q.w, a1, a2, a3);
        }
        sumsq_group_end(a1, a2, sc, n1, n2);
    }
    return sumsq_finish(n1, n2, a3, ex, (nvec + 31) / 32, sc, row, nvec);
}

__global__ void __launch_bounds__(RT_THREADS)
router_kernel(const uint16_t *__restrict__ x, const uint16_t *__restrict__ gamma,
              const float *__restrict__ wg, const float *__restrict__ gate_bias, int T, int H,
              int E, float eps, int rmsnorm, uint16_t *__restrict__ xn,
              float *__restrict__ logits, int fuse_topk, int k, int renorm,
              int32_t *__restrict__ topk_idx, float *__restrict__ topk_w,
              int32_t *__restrict__ hist, int32_t *dev_status) {
    extern __shared__ __align__(128) uint8_t smem[];
    float *lg = reinterpret_cast<float *>(smem + SMEM_MAIN);       // phase 3
    float *s_r = reinterpret_cast<float *>(smem + SMEM_MAIN + SMEM_LG);
    int *s_cnt = reinterpret_cast<int *>(s_r + RT_TOK);
    (void)dev_status;   // no waits that could time out

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int tok0 = blockIdx.x * RT_TOK;
    const int e0 = blockIdx.y * RT_EXP;
    const int ntok = min(RT_TOK, T - tok0);

    if (tid < RT_EXP) s_cnt[tid] = 0;
    if (tid < RT_TOK) s_r[tid] = 1.0f;
    __syncthreads();

    // ---------------- phase 1: r = 1/sqrt(mean(x^2) + eps) per token, the
    // sum of squares of each row by one warp (rows w, w + 4, ...)
    if (rmsnorm) {
        for (int t = warp; t < ntok; t += RT_THREADS / 32) {
            const float ss = warp_sumsq_rn_mem(
                reinterpret_cast<const uint4 *>(x + static_cast<size_t>(tok0 + t) * H), H / 8);
            if (lane == 0) {
                const float mean = __fdiv_rn(ss, static_cast<float>(H));
                s_r[t] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, eps)));
            }
        }
        __syncthreads();
    }

    // ---------------- phase 2: logits
    // Slices of G_HC columns: the raw x slice (bf16) and the gate-weight slice
    // (fp32, padded rows) arrive through a G_STAGES-deep cp.async ring; each x
    // slice is then normalised once into an fp32 buffer (double-buffered).
    __syncthreads();
    uint8_t *wg_ring = smem;
    uint8_t *xr_ring = smem + G_STAGES * WG_STAGE;
    float *xs = reinterpret_cast<float *>(smem + G_STAGES * (WG_STAGE + XR_STAGE));

    const int ty = tid >> 4, tx = tid & 15;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;

    const int lt = tid >> 2, lg4 = tid & 3;           // x slice: token, 8-column group
    const bool write_xn = rmsnorm && xn != nullptr && blockIdx.y == 0;
    const float r_t = s_r[lt];
    const int nslices = H / G_HC;

    auto issue = [&](int c) {
        const int st = c % G_STAGES;
        const int h0 = c * G_HC;
        const bool okt = lt < ntok;
        const uint16_t *xsrc = okt ? x + static_cast<size_t>(tok0 + lt) * H + h0 + 8 * lg4 : x;
        cp_async16(xr_ring + st * XR_STAGE + lt * (G_HC * 2) + lg4 * 16, xsrc, okt ? 16 : 0);
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const int e = p * 16 + (tid >> 3);
            const bool oke = e0 + e < E;
            const float *wsrc =
                oke ? wg + static_cast<size_t>(e0 + e) * H + h0 + 4 * (tid & 7) : wg;
            cp_async16(wg_ring + st * WG_STAGE + e * (G_LD * 4) + (tid & 7) * 16, wsrc,
                       oke ? 16 : 0);
        }
    };
    auto convert = [&](int c, int buf) {
        const int h0 = c * G_HC;
        const uint4 xq = *reinterpret_cast<const uint4 *>(
            xr_ring + (c % G_STAGES) * XR_STAGE + lt * (G_HC * 2) + lg4 * 16);
        const uint32_t w[4] = {xq.x, xq.y, xq.z, xq.w};
        float f[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
        if (rmsnorm) {
            float gm[8];
            if (gamma) {
                const uint4 gq = *reinterpret_cast<const uint4 *>(gamma + h0 + 8 * lg4);
                const uint32_t gw[4] = {gq.x, gq.y, gq.z, gq.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    gm[2 * i] = __uint_as_float(gw[i] << 16);
                    gm[2 * i + 1] = __uint_as_float(gw[i] & 0xFFFF0000u);
                }
            }
            uint32_t packed[4];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float v = __fmul_rn(f[i], r_t);
                if (gamma) v = __fmul_rn(v, gm[i]);
                const uint16_t b = float_to_bf16_bits(v);
                f[i] = bf16_bits_to_float(b);
                if (i & 1)
                    packed[i >> 1] |= static_cast<uint32_t>(b) << 16;
                else
                    packed[i >> 1] = b;
            }
            if (write_xn && lt < ntok)
                *reinterpret_cast<uint4 *>(xn + static_cast<size_t>(tok0 + lt) * H + h0 +
                                           8 * lg4) =
                    make_uint4(packed[0], packed[1], packed[2], packed[3]);
        }
        float *xd = xs + (buf * RT_TOK + lt) * G_LD + 8 * lg4;
        *reinterpret_cast<float4 *>(xd) = make_float4(f[0], f[1], f[2], f[3]);
        *reinterpret_cast<float4 *>(xd + 4) = make_float4(f[4], f[5], f[6], f[7]);
    };

#pragma unroll
    for (int c = 0; c < G_STAGES - 1; ++c) {
        if (c < nslices) issue(c);
        cp_async_commit();
    }
    cp_async_wait<G_STAGES - 2>();
    __syncthreads();
    convert(0, 0);
    __syncthreads();
    for (int c = 0; c < nslices; ++c) {
        if (c + G_STAGES - 1 < nslices) issue(c + G_STAGES - 1);
        cp_async_commit();
        const float *xb = xs + (c & 1) * RT_TOK * G_LD;
        const float *wb = reinterpret_cast<const float *>(wg_ring + (c % G_STAGES) * WG_STAGE);
#pragma unroll
        for (int hh = 0; hh < G_HC; hh += 4) {
            float4 xv[4], wv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                xv[i] = *reinterpret_cast<const float4 *>(xb + (ty + 8 * i) * G_LD + hh);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                wv[j] = *reinterpret_cast<const float4 *>(wb + (tx + 16 * j) * G_LD + hh);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    acc[i][j] = __fmaf_rn(xv[i].x, wv[j].x, acc[i][j]);
                    acc[i][j] = __fmaf_rn(xv[i].y, wv[j].y, acc[i][j]);
                    acc[i][j] = __fmaf_rn(xv[i].z, wv[j].z, acc[i][j]);
                    acc[i][j] = __fmaf_rn(xv[i].w, wv[j].w, acc[i][j]);
                }
        }
        cp_async_wait<G_STAGES - 2>();
        __syncthreads();
        if (c + 1 < nslices) convert(c + 1, (c + 1) & 1);
        __syncthreads();
    }

    // ---------------- phase 3: bias, logits out, top-k, histogram
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int e = e0 + tx + 16 * j;
            float v = acc[i][j];
            if (gate_bias && e < E) v = __fadd_rn(v, gate_bias[e]);
            lg[(ty + 8 * i) * (RT_EXP + 1) + tx + 16 * j] = v;
        }
    __syncthreads();
    if (logits) {
        const int ne = min(RT_EXP, E - e0);
        for (int idx = tid; idx < ntok * ne; idx += RT_THREADS) {
            const int t = idx / ne, e = idx % ne;
            logits[static_cast<size_t>(tok0 + t) * E + e0 + e] = lg[t * (RT_EXP + 1) + e];
        }
    }
    if (!fuse_topk) return;

    for (int t = warp; t < ntok; t += RT_THREADS / 32) {
        float v[2];
        v[0] = lane < E ? lg[t * (RT_EXP + 1) + lane] : -INFINITY;
        v[1] = lane + 32 < E ? lg[t * (RT_EXP + 1) + lane + 32] : -INFINITY;
        int sel_e;
        float sel_v;
        warp_topk<2>(v, k, &sel_e, &sel_v);
        const float w = slot_weight<2>(v, k, renorm != 0, sel_v);
        if (lane < k) {
            const size_t a = static_cast<size_t>(tok0 + t) * k + lane;
            topk_idx[a] = sel_e;
            topk_w[a] = w;
            atomicAdd(&s_cnt[sel_e], 1);
        }
    }
    if (hist) {
        __syncthreads();
        for (int e = tid; e < E; e += RT_THREADS)
            hist[static_cast<size_t>(blockIdx.x) * E + e] = s_cnt[e];
    }
}

// Few tokens (T <= 512): one CTA per token and one thread per expert, so
// that every logit's sequential FMA chain runs at the same time.  The row is
// kept in shared memory as fp32; thread 0 takes the sum of squares in
// ascending h; the gate weight streams through a SLOTS-deep ring of chunks
// of NB*32 columns, filled while the sum of squares runs.  Every CTA streams
// the whole gate weight from L2: a chunk arrives as NB TMA tensor boxes
// (E rows x 32 fp32 columns, 128-byte swizzle: 16-byte piece q of row e sits
// at piece q ^ (e & 7), so the 32 lanes' reads of one piece are
// conflict-free) completed on the slot's mbarrier.  With at most one CTA per
// SM the ring is as deep as shared memory allows, in 128-column chunks when
// H allows (one barrier test and one release per 128 FMAs of each chain);
// with more tokens it is sized for two CTAs per SM.
// Same arithmetic, in the same order, as the tiled kernel above.
constexpr int SM_BOX = 32;    // columns of one tensor box
constexpr int SM_SMEM_CAP = 220 * 1024;
// bytes of one box of a ring slot: E rows of 128 bytes, rounded to whole
// 1 KB swizzle atoms
__host__ __device__ inline int sm_box_bytes(int E) { return ((E + 7) / 8) * 1024; }
constexpr int SMALL_MAX_T = kGateSmallMaxT;
constexpr int SMALL_MAX_E = 128;
constexpr int SMALL_MAX_H = 8192;

__device__ __forceinline__ void consumer_sync(int nthreads) {
    asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

// Threads [0, nc) are the consumers (one per expert, nc = max(64, E rounded
// up to 32)); the warp after them only streams the gate weight: it refills a
// slot once every consumer warp has arrived on the slot's empty barrier, so
// the consumers' FMA chains never stop at a block-wide barrier.  A CTA takes
// TPC consecutive tokens: every consumer runs one chain per token on the
// same weight operands, so the weight streams through the SM once per TPC
// tokens.
template <int SLOTS, int NB, int TPC>
__global__ void __launch_bounds__(160)
router_small_kernel(const uint16_t *__restrict__ x, const uint16_t *__restrict__ gamma,
                    const float *__restrict__ wg, const float *__restrict__ gate_bias, int T,
                    int H, int E, float eps, int rmsnorm, uint16_t *__restrict__ xn,
                    float *__restrict__ logits, int fuse_topk, int k, int renorm,
                    int32_t *__restrict__ topk_idx, float *__restrict__ topk_w,
                    int32_t *dev_status, const __grid_constant__ CUtensorMap tmw) {
    extern __shared__ uint8_t sm_raw[];
    // 1 KB aligned for the swizzled boxes; offsetting the shared pointer (not
    // an integer copy of it) keeps the loads below in the shared window
    uint8_t *ring = sm_raw + ((1024u - (smem_u32(sm_raw) & 1023u)) & 1023u);
    static_assert(NB >= 2 && NB % 2 == 0, "boxes are consumed in pairs");
    static_assert(TPC >= 1 && TPC <= 2, "one chain-running warp per token among the first two");
    constexpr int HC = NB * SM_BOX;    // columns of one chunk
    const int hb = sm_box_bytes(E);   // ring: [SLOTS][NB boxes][hb]
    float *xf = reinterpret_cast<float *>(ring + SLOTS * NB * hb);   // [TPC][H]
    __shared__ float s_r[TPC];
    __shared__ float s_lg[TPC][SMALL_MAX_E];
    __shared__ __align__(8) uint64_t s_full[SLOTS];
    __shared__ __align__(8) uint64_t s_empty[SLOTS];
    __shared__ int s_abort_v;
    volatile int *s_abort = &s_abort_v;
    const int t0 = blockIdx.x * TPC;
    const int ntok = min(TPC, T - t0);
    const int tid = threadIdx.x;
    const int nc = blockDim.x - 32;      // consumer threads
    const int nvec = H / 8;
    const int nch = H / HC;

    if (tid == 0) {
        *s_abort = 0;
        for (int q = 0; q < SLOTS; ++q) {
            mbar_init(&s_full[q], 1);
            mbar_init(&s_empty[q], nc / 32);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (tid >= nc) {
        // ---- producer warp: chunk c of the gate weight into slot c % SLOTS
        if (tid == nc) {
            int issued = 0;
            for (int c = 0; c < nch; ++c) {
                const int st = c % SLOTS;
                if (c >= SLOTS &&
                    !mbar_wait_bounded(&s_empty[st], static_cast<uint32_t>((c / SLOTS - 1) & 1),
                                       s_abort, dev_status))
                    break;
                mbar_arrive_expect_tx(&s_full[st], static_cast<uint32_t>(E) * HC * 4);
                uint8_t *slot = ring + st * NB * hb;
#pragma unroll
                for (int b = 0; b < NB; ++b)
                    tma_load_2d(slot + b * hb, &tmw, &s_full[st], c * HC + b * SM_BOX, 0);
                issued = c + 1;
            }
            if (*s_abort) {
                // unwinding: let the copies still in flight land
                for (int c = issued - SLOTS; c < issued; ++c)
                    if (c >= 0)
                        mbar_wait_drain(&s_full[c % SLOTS], static_cast<uint32_t>((c / SLOTS) & 1));
            }
        }
        return;
    }

    // ---- consumers: the tokens' rows as fp32 (a missing last token repeats
    // the CTA's first row; nothing of it is written)
#pragma unroll
    for (int tk = 0; tk < TPC; ++tk) {
        const int t = tk < ntok ? t0 + tk : t0;
        const uint4 *xq = reinterpret_cast<const uint4 *>(x + static_cast<size_t>(t) * H);
        float *xr = xf + tk * H;
        for (int v = tid; v < nvec; v += nc) {
            const uint4 q = xq[v];
            const uint32_t w[4] = {q.x, q.y, q.z, q.w};
            float f[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                f[2 * i] = __uint_as_float(w[i] << 16);
                f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
            }
            *reinterpret_cast<float4 *>(xr + 8 * v) = make_float4(f[0], f[1], f[2], f[3]);
            *reinterpret_cast<float4 *>(xr + 8 * v + 4) = make_float4(f[4], f[5], f[6], f[7]);
        }
    }
    consumer_sync(nc);

    if (rmsnorm) {
        // warp tk takes token tk's sum of squares (reading the row from
        // memory); every consumer fetches its gamma groups meanwhile
        // (nvec <= SMALL_MAX_H / 8, nc >= 64: at most 16 each)
        constexpr int GQ = SMALL_MAX_H / 8 / 64;
        uint4 gqs[GQ];
#pragma unroll
        for (int j = 0; j < GQ; ++j) {
            const int v = tid + j * nc;
            gqs[j] = make_uint4(0u, 0u, 0u, 0u);
            if (gamma && v < nvec) gqs[j] = __ldg(reinterpret_cast<const uint4 *>(gamma) + v);
        }
        if ((tid >> 5) < TPC) {
            const int tk = tid >> 5;
            const int t = tk < ntok ? t0 + tk : t0;
            const float ss = warp_sumsq_rn_mem(
                reinterpret_cast<const uint4 *>(x + static_cast<size_t>(t) * H), nvec);
            if ((tid & 31) == 0) {
                const float mean = __fdiv_rn(ss, static_cast<float>(H));
                s_r[tk] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, eps)));
            }
        }
        consumer_sync(nc);
#pragma unroll
        for (int j = 0; j < GQ; ++j) {
            const int v = tid + j * nc;
            if (v >= nvec) break;
            float gm[8];
            if (gamma) {
                const uint4 gq = gqs[j];
                const uint32_t gw[4] = {gq.x, gq.y, gq.z, gq.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    gm[2 * i] = __uint_as_float(gw[i] << 16);
                    gm[2 * i + 1] = __uint_as_float(gw[i] & 0xFFFF0000u);
                }
            }
#pragma unroll
            for (int tk = 0; tk < TPC; ++tk) {
                const float r = s_r[tk];
                float *xr = xf + tk * H;
                uint32_t packed[4];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    float val = __fmul_rn(xr[8 * v + i], r);
                    if (gamma) val = __fmul_rn(val, gm[i]);
                    const uint16_t b = float_to_bf16_bits(val);
                    xr[8 * v + i] = bf16_bits_to_float(b);
                    if (i & 1)
                        packed[i >> 1] |= static_cast<uint32_t>(b) << 16;
                    else
                        packed[i >> 1] = b;
                }
                if (xn && tk < ntok)
                    reinterpret_cast<uint4 *>(xn + static_cast<size_t>(t0 + tk) * H)[v] =
                        make_uint4(packed[0], packed[1], packed[2], packed[3]);
            }
        }
        consumer_sync(nc);
    }

    // The logit's FMA chain is the critical path: its operands are read into
    // registers one box (32 columns) ahead, so the chain never waits on
    // shared memory, and neither on the full barriers while the ring is ahead
    // (their test overlaps the FMAs).  A warp releases a slot (empty barrier)
    // once its loads of the slot's last box have landed.
    const int e = tid;
    const int lane = tid & 31;
    const int er = e < E ? e : 0;             // threads past E follow along on row 0
    constexpr int HQ = SM_BOX / 4;            // float4s per box row
    float acc[TPC];
#pragma unroll
    for (int tk = 0; tk < TPC; ++tk) acc[tk] = 0.0f;
    float4 wa[HQ], xa[TPC][HQ], wb[HQ], xb[TPC][HQ];
    auto load_box = [&](int c, int b, float4 (&w)[HQ], float4 (&xv)[TPC][HQ]) {
        const uint8_t *wr = ring + ((c % SLOTS) * NB + b) * hb + er * 128;
        const float *xc = xf + c * HC + b * SM_BOX;
#pragma unroll
        for (int q = 0; q < HQ; ++q) {
            w[q] = *reinterpret_cast<const float4 *>(wr + ((q ^ (er & 7)) << 4));
#pragma unroll
            for (int tk = 0; tk < TPC; ++tk)
                xv[tk][q] = *reinterpret_cast<const float4 *>(xc + tk * H + 4 * q);
        }
    };
    auto fma_box = [&](const float4 (&w)[HQ], const float4 (&xv)[TPC][HQ]) {
#pragma unroll
        for (int q = 0; q < HQ; ++q) {
#pragma unroll
            for (int tk = 0; tk < TPC; ++tk) {
                acc[tk] = __fmaf_rn(xv[tk][q].x, w[q].x, acc[tk]);
                acc[tk] = __fmaf_rn(xv[tk][q].y, w[q].y, acc[tk]);
                acc[tk] = __fmaf_rn(xv[tk][q].z, w[q].z, acc[tk]);
                acc[tk] = __fmaf_rn(xv[tk][q].w, w[q].w, acc[tk]);
            }
        }
    };
    auto wait_chunk = [&](int c) {
        mbar_wait_bounded(&s_full[c % SLOTS], static_cast<uint32_t>((c / SLOTS) & 1), s_abort,
                          dev_status);
    };
    wait_chunk(0);
    load_box(0, 0, wa, xa);
    for (int c = 0; c < nch; ++c) {
        const bool more = c + 1 < nch;
#pragma unroll
        for (int j = 0; j < NB; j += 2) {
            // box j is in (wa, xa); box j + 1 goes to (wb, xb)
            load_box(c, j + 1, wb, xb);
            if (j + 2 < NB) {
                fma_box(wa, xa);
                load_box(c, j + 2, wa, xa);
                fma_box(wb, xb);
                continue;
            }
            // the test of the next chunk's barrier is in flight while box j's
            // FMAs issue; the release of slot c follows them, when the loads
            // of its last box have landed
            const bool ready = !more || mbar_try_wait(&s_full[(c + 1) % SLOTS],
                                                      static_cast<uint32_t>(((c + 1) / SLOTS) & 1));
            fma_box(wa, xa);
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_empty[c % SLOTS]);
            if (more) {
                if (!ready) wait_chunk(c + 1);
                load_box(c + 1, 0, wa, xa);
            }
            fma_box(wb, xb);
        }
    }
    if (e < E) {
#pragma unroll
        for (int tk = 0; tk < TPC; ++tk) {
            float a = acc[tk];
            if (gate_bias) a = __fadd_rn(a, gate_bias[e]);
            s_lg[tk][e] = a;
            if (logits && tk < ntok) logits[static_cast<size_t>(t0 + tk) * E + e] = a;
        }
    }
    consumer_sync(nc);
    // warp tk: token tk's top-k
    const int tk = tid >> 5;
    if (fuse_topk && tk < ntok) {
        float v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int ee = lane + 32 * i;
            v[i] = ee < E ? s_lg[tk][ee] : -INFINITY;
        }
        int sel_e;
        float sel_v;
        warp_topk<4>(v, k, &sel_e, &sel_v);
        const float w = slot_weight<4>(v, k, renorm != 0, sel_v);
        if (lane < k) {
            topk_idx[static_cast<size_t>(t0 + tk) * k + lane] = sel_e;
            topk_w[static_cast<size_t>(t0 + tk) * k + lane] = w;
        }
    }
}

template <int NV>
__global__ void __launch_bounds__(256)
topk_kernel(const float *__restrict__ logits, int T, int E, int k, int renorm,
            int32_t *__restrict__ topk_idx, float *__restrict__ topk_w) {
    const int lane = threadIdx.x & 31;
    const int warps = blockDim.x >> 5;
    for (int t = blockIdx.x * warps + (threadIdx.x >> 5); t < T; t += gridDim.x * warps) {
        float v[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int e = lane + 32 * i;
            v[i] = e < E ? logits[static_cast<size_t>(t) * E + e] : -INFINITY;
        }
        int sel_e;
        float sel_v;
        warp_topk<NV>(v, k, &sel_e, &sel_v);
        const float w = slot_weight<NV>(v, k, renorm != 0, sel_v);
        if (lane < k) {
            topk_idx[static_cast<size_t>(t) * k + lane] = sel_e;
            topk_w[static_cast<size_t>(t) * k + lane] = w;
        }
    }
}

// ---------------------------------------------------------------- RMSNorm alone
// Used ahead of the tensor-core gate: one warp per row.  The row (at most
// VPL 16-byte vectors per lane) is held in registers; its sum of squares is
// the warp's exact one above; then xn = bf16((x * r) * gamma) leaves as
// 16-byte stores.  gamma is staged in shared memory once per CTA (zeros past
// the row), so the normalisation reads it without a global-load latency per
// vector and without a bound check.  While a row is summed, the warp's next
// row is prefetched into L2.  No waits.
constexpr int RN_THREADS = 256;

template <int VPL>
__global__ void __launch_bounds__(RN_THREADS, 2)
rmsnorm_kernel(const uint16_t *__restrict__ x, const uint16_t *__restrict__ gamma, int T, int H,
               float eps, uint16_t *__restrict__ xn) {
    __shared__ uint4 s_gamma[VPL * 32];
    const int lane = threadIdx.x & 31;
    const int nvec = H / 8;
    const int nwarps = gridDim.x * (RN_THREADS / 32);
    if (gamma) {
        for (int v = threadIdx.x; v < VPL * 32; v += RN_THREADS)
            s_gamma[v] = v < nvec ? __ldg(reinterpret_cast<const uint4 *>(gamma) + v)
                                  : make_uint4(0u, 0u, 0u, 0u);
        __syncthreads();
    }
    for (int t = blockIdx.x * (RN_THREADS / 32) + (threadIdx.x >> 5); t < T; t += nwarps) {
        const uint4 *row = reinterpret_cast<const uint4 *>(x + static_cast<size_t>(t) * H);
        uint4 q[VPL];
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const int v = lane + 32 * i;
            q[i] = v < nvec ? __ldcs(row + v) : make_uint4(0u, 0u, 0u, 0u);
        }
        // the warp's next row into L2 meanwhile (one 128-byte line per lane and step)
        if (t + nwarps < T) {
            const char *nrow = reinterpret_cast<const char *>(x + static_cast<size_t>(t + nwarps) * H);
            for (int off = lane * 128; off < H * 2; off += 32 * 128)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(nrow + off));
        }
        const float ss = warp_sumsq_rn_packed<VPL>(q, row, nvec);
        const float mean = __fdiv_rn(ss, static_cast<float>(H));
        const uint64_t r2 = f2_splat(__fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, eps))));
        uint4 *out = reinterpret_cast<uint4 *>(xn + static_cast<size_t>(t) * H);
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const int v = lane + 32 * i;
            uint4 gq = make_uint4(0u, 0u, 0u, 0u);
            if (gamma) gq = s_gamma[v];
            const uint32_t gw[4] = {gq.x, gq.y, gq.z, gq.w};
            const uint32_t wd[4] = {q[i].x, q[i].y, q[i].z, q[i].w};
            uint32_t packed[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                // (x * r) * gamma, each product rounded, on both values at once
                uint64_t y = f2_mul(f2_from_bf16x2(wd[j]), r2);
                if (gamma) y = f2_mul(y, f2_from_bf16x2(gw[j]));
                const __nv_bfloat162 p2 = __floats2bfloat162_rn(f2_lo(y), f2_hi(y));
                packed[j] = *reinterpret_cast<const uint32_t *>(&p2);
            }
            if (v < nvec) out[v] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
        }
    }
}

// The sum of squares alone, one warp per row (moe_rmsnorm_sumsq).
__global__ void __launch_bounds__(256)
sumsq_kernel(const uint16_t *__restrict__ x, int T, int H, float *__restrict__ ss) {
    const int nwarps = gridDim.x * 8;
    for (int t = blockIdx.x * 8 + (threadIdx.x >> 5); t < T; t += nwarps) {
        const float v = warp_sumsq_rn_mem(
            reinterpret_cast<const uint4 *>(x + static_cast<size_t>(t) * H), H / 8);
        if ((threadIdx.x & 31) == 0) ss[t] = v;
    }
}

// ---------------------------------------------------------------- tensor-core gate
// The gate on the tensor cores at fp32 accuracy: each fp32 weight splits
// exactly into three bf16 parts, w = w1 + w2 + w3 (w1 = bf16(w), w2 =
// bf16(w - w1), w3 = bf16(w - w1 - w2); the two differences are exact in
// fp32 and the last part holds the remaining bits -- for |w| >= 2^-110;
// closer to fp32's underflow the parts are within 2^-134 of w), and every
// product of a bf16 xn value with a part is exact.  The grouped GEMM computes the three
// partial dot products as separate output columns (fp32 accumulation in the
// tensor core) and the combine kernel adds them: logit = (p1 + p2) + p3.
// The sum is fp32-accurate but not in the sequential order of the plain
// definition, so a logit can differ from it in the last bits.
//
// Split: blockIdx.y = output row (part * E + e, zero rows up to NW), four
// columns per thread.
__global__ void __launch_bounds__(256)
gate_split_kernel(const float *__restrict__ wg, int E, int H, uint16_t *__restrict__ ws) {
    const int row = blockIdx.y;
    const int part = row / E, e = row - part * E;
    const int h = 4 * (blockIdx.x * 256 + threadIdx.x);
    if (h >= H) return;
    uint32_t out[2] = {0u, 0u};
    if (part < 3) {
        const float4 wv = __ldg(reinterpret_cast<const float4 *>(wg + static_cast<size_t>(e) * H + h));
        const float w4[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float w = w4[i];
            const uint16_t b1 = float_to_bf16_bits(w);
            const float r1 = __fsub_rn(w, bf16_bits_to_float(b1));
            const uint16_t b2 = float_to_bf16_bits(r1);
            const float r2 = __fsub_rn(r1, bf16_bits_to_float(b2));
            const uint16_t v = part == 0 ? b1 : part == 1 ? b2 : float_to_bf16_bits(r2);
            out[i >> 1] |= static_cast<uint32_t>(v) << (16 * (i & 1));
        }
    }
    *reinterpret_cast<uint2 *>(ws + static_cast<size_t>(row) * H + h) = make_uint2(out[0], out[1]);
}

// Combine: one CTA per 32-token chunk.  All threads form the chunk's logits,
// logit = (p1 + p2) + p3 (+ bias), coalesced over (token, expert); without
// fuse_topk they go to `logits`.  With it (E <= 64) they stay in shared
// memory and a group of 8 lanes takes each token's top-k: per slot every
// lane finds the best untaken expert among its eighth of the row, three
// shuffles pick the group's best (larger logit, equal logits to the lower
// index), then the softmax weights and the chunk's routing histogram.  (One
// lane per token left 7 of 8 warps waiting at the barrier; a warp-wide
// argmax per token spent the time on shuffles.)
constexpr int GC_THREADS = 256;

__device__ __forceinline__ bool better_sel(float va, int ia, float vb, int ib) {
    if (ia < 0) return false;
    if (ib < 0) return true;
    return va > vb || (va == vb && ia < ib);
}

__global__ void __launch_bounds__(GC_THREADS)
gate_combine_kernel(const float *__restrict__ parts, int NW, int T, int E,
                    const float *__restrict__ gate_bias, float *__restrict__ logits,
                    int fuse_topk, int k, int renorm, int32_t *__restrict__ topk_idx,
                    float *__restrict__ topk_w, int32_t *__restrict__ hist) {
    __shared__ float s_lg[RT_TOK][RT_EXP + 1];
    __shared__ int s_cnt[RT_EXP];
    const int tok0 = blockIdx.x * RT_TOK;
    const int ntok = min(RT_TOK, T - tok0);
    if (fuse_topk && threadIdx.x < RT_EXP) s_cnt[threadIdx.x] = 0;
    for (int i = threadIdx.x; i < ntok * E; i += GC_THREADS) {
        const int t = i / E, e = i - t * E;
        const float *pr = parts + static_cast<size_t>(tok0 + t) * NW;
        float v = __fadd_rn(__fadd_rn(__ldg(pr + e), __ldg(pr + E + e)), __ldg(pr + 2 * E + e));
        if (gate_bias) v = __fadd_rn(v, __ldg(gate_bias + e));
        if (fuse_topk)
            s_lg[t][e] = v;
        else
            logits[static_cast<size_t>(tok0 + t) * E + e] = v;
    }
    if (!fuse_topk) return;
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int t = (threadIdx.x >> 5) * 4 + (lane >> 3);    // 8 warps x 4 tokens
    const int sl = lane & 7;                                // this lane's experts: sl + 8i
    if (t < ntok) {                                         // whole 8-lane groups agree
        const float *row = s_lg[t];
        const unsigned gmask = 0xFFu << (lane & 24);
        uint32_t taken = 0;                                 // bit i: expert sl + 8i
        int sel = -1, sel0 = -1;
        for (int j = 0; j < k; ++j) {
            int bi = -1;
            float bv = -INFINITY;
            for (int i = 0, e = sl; e < E; ++i, e += 8) {
                const float v = row[e];
                if (!((taken >> i) & 1u) && (bi < 0 || v > bv)) {
                    bv = v;
                    bi = e;
                }
            }
#pragma unroll
            for (int off = 4; off > 0; off >>= 1) {
                const float ov = __shfl_xor_sync(gmask, bv, off);
                const int oi = __shfl_xor_sync(gmask, bi, off);
                if (better_sel(ov, oi, bv, bi)) {
                    bv = ov;
                    bi = oi;
                }
            }
            if ((bi & 7) == sl) taken |= 1u << (bi >> 3);
            if (j == 0) sel0 = bi;
            if ((j & 7) == sl) sel = bi;                    // lane sl keeps slots sl, sl+8, ...
            if ((j & 7) == 7 || j == k - 1) {
                // flush the (up to) 8 slots gathered so far
                const int j0 = j & ~7;
                if (j0 + sl <= j) {
                    topk_idx[static_cast<size_t>(tok0 + t) * k + j0 + sl] = sel;
                    atomicAdd(&s_cnt[sel], 1);
                }
            }
        }
        // softmax weights over the chosen slots (renorm) or over all experts
        const float m = row[sel0];
        float den = 0.0f;
        if (renorm) {
            for (int j = sl; j < k; j += 8)
                den += expf(row[topk_idx[static_cast<size_t>(tok0 + t) * k + j]] - m);
        } else {
            for (int e = sl; e < E; e += 8) den += expf(row[e] - m);
        }
#pragma unroll
        for (int off = 4; off > 0; off >>= 1) den += __shfl_xor_sync(gmask, den, off);
        for (int j = sl; j < k; j += 8) {
            const int e = topk_idx[static_cast<size_t>(tok0 + t) * k + j];
            topk_w[static_cast<size_t>(tok0 + t) * k + j] = expf(row[e] - m) / den;
        }
    }
    if (hist) {
        __syncthreads();
        for (int e = threadIdx.x; e < E; e += GC_THREADS)
            hist[static_cast<size_t>(blockIdx.x) * E + e] = s_cnt[e];
    }
}

}  // namespace

// The gate weight [E, H] fp32 as 32-column x E-row boxes, 128-byte swizzle.
typedef CUresult (*EncodeTiledFnR)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
bool make_wg_map(CUtensorMap *m, const float *wg, int H, int E) {
    static EncodeTiledFnR fn = [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFnR>(ptr);
        return static_cast<EncodeTiledFnR>(nullptr);
    }();
    if (!fn) return false;
    cuuint64_t gdim[2] = {static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(E)};
    cuuint64_t gstride[1] = {static_cast<cuuint64_t>(H) * 4};
    cuuint32_t box[2] = {SM_BOX, static_cast<cuuint32_t>(E)};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(wg), gdim, gstride, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

cudaError_t launch_router(const uint16_t *x, const uint16_t *gamma, const float *wg,
                          const float *gate_bias, int T, int H, int E, float eps, bool rmsnorm,
                          uint16_t *xn, float *logits, bool fuse_topk, int k, bool renorm,
                          int32_t *topk_idx, float *topk_w, int32_t *hist,
                          int32_t *dev_status, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    if (T <= SMALL_MAX_T && E <= SMALL_MAX_E && H <= SMALL_MAX_H) {
        // consumers (one per expert, at least two warps) + the producer warp
        const int threads = std::max(64, static_cast<int>(ceil_div(E, 32)) * 32) + 32;
        CUtensorMap tmw;
        if (!make_wg_map(&tmw, wg, H, E)) return cudaErrorInvalidValue;
        auto smem_for = [&](int slots, int nb, int tpc) {
            return 1024 + static_cast<size_t>(slots) * nb * sm_box_bytes(E) +
                   static_cast<size_t>(tpc) * H * sizeof(float);
        };
        auto run = [&](auto kernel, int slots, int nb, int tpc) -> cudaError_t {
            const size_t smem = smem_for(slots, nb, tpc);
            if (smem > 48 * 1024) {
                cudaError_t e = cudaFuncSetAttribute(
                    kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
                if (e != cudaSuccess) return e;
            }
            kernel<<<static_cast<unsigned>(ceil_div(T, tpc)), threads, smem, stream>>>(
                x, gamma, wg, gate_bias, T, H, E, eps, rmsnorm ? 1 : 0, xn, logits,
                fuse_topk ? 1 : 0, k, renorm ? 1 : 0, topk_idx, topk_w, dev_status, tmw);
            return cudaSuccess;
        };
        // One CTA per SM: one token per CTA up to a CTA per SM, else two (the
        // weight then streams through each SM once per two tokens; beyond two
        // tokens per SM a second wave), the deepest ring that fits, in
        // 128-column chunks when H allows.
        const int64_t sms = num_sms();
        const bool h128 = H % (4 * SM_BOX) == 0;
        const size_t full = SM_SMEM_CAP, half = SM_SMEM_CAP / 2;
        cudaError_t le;
        if (T <= sms && h128 && smem_for(6, 4, 1) <= full)
            le = run(router_small_kernel<6, 4, 1>, 6, 4, 1);
        else if (T <= sms && smem_for(12, 2, 1) <= full)
            le = run(router_small_kernel<12, 2, 1>, 12, 2, 1);
        else if (T > sms && h128 && smem_for(5, 4, 2) <= full)
            le = run(router_small_kernel<5, 4, 2>, 5, 4, 2);
        else if (T > sms && smem_for(10, 2, 2) <= full)
            le = run(router_small_kernel<10, 2, 2>, 10, 2, 2);
        else if (smem_for(5, 2, 1) <= half)
            le = run(router_small_kernel<5, 2, 1>, 5, 2, 1);
        else
            le = run(router_small_kernel<3, 2, 1>, 3, 2, 1);
        if (le != cudaSuccess) return le;
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess || !fuse_topk || hist == nullptr) return e;
        return launch_route_hist(topk_idx, T, k, E, hist, dev_status, stream);
    }
    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(router_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             SMEM_TOTAL);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    dim3 grid(static_cast<unsigned>(ceil_div(T, RT_TOK)),
              static_cast<unsigned>(ceil_div(E, RT_EXP)));
    router_kernel<<<grid, RT_THREADS, SMEM_TOTAL, stream>>>(
        x, gamma, wg, gate_bias, T, H, E, eps, rmsnorm ? 1 : 0, xn, logits,
        fuse_topk ? 1 : 0, k, renorm ? 1 : 0, topk_idx, topk_w, hist, dev_status);
    return cudaGetLastError();
}

cudaError_t launch_topk(const float *logits, int T, int E, int k, bool renorm,
                        int32_t *topk_idx, float *topk_w, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const int threads = 256;
    const int blocks = static_cast<int>(std::min<int64_t>(ceil_div(T, threads / 32), 152 * 16));
    const int nv = static_cast<int>(ceil_div(E, 32));
    const int rn = renorm ? 1 : 0;
    if (nv <= 1)
        topk_kernel<1><<<blocks, threads, 0, stream>>>(logits, T, E, k, rn, topk_idx, topk_w);
    else if (nv <= 2)
        topk_kernel<2><<<blocks, threads, 0, stream>>>(logits, T, E, k, rn, topk_idx, topk_w);
    else if (nv <= 4)
        topk_kernel<4><<<blocks, threads, 0, stream>>>(logits, T, E, k, rn, topk_idx, topk_w);
    else if (nv <= 8)
        topk_kernel<8><<<blocks, threads, 0, stream>>>(logits, T, E, k, rn, topk_idx, topk_w);
    else if (nv <= 16)
        topk_kernel<16><<<blocks, threads, 0, stream>>>(logits, T, E, k, rn, topk_idx, topk_w);
    else
        topk_kernel<32><<<blocks, threads, 0, stream>>>(logits, T, E, k, rn, topk_idx, topk_w);
    return cudaGetLastError();
}

cudaError_t launch_rmsnorm(const uint16_t *x, const uint16_t *gamma, int T, int H, float eps,
                           uint16_t *xn, int32_t *dev_status, cudaStream_t stream) {
    (void)dev_status;    // the kernel has no waits to time out
    if (T == 0) return cudaSuccess;
    if (H <= 0 || H % 128 != 0) return cudaErrorInvalidValue;
    // one warp per row: enough rows in flight to cover the memory latency
    const int vpl = static_cast<int>(ceil_div(H / 8, 32));
    const int64_t warps = T;
    const int grid = static_cast<int>(std::max<int64_t>(
        1, std::min<int64_t>(ceil_div(warps, RN_THREADS / 32), int64_t{num_sms()} * 4)));
    if (vpl <= 4)
        rmsnorm_kernel<4><<<grid, RN_THREADS, 0, stream>>>(x, gamma, T, H, eps, xn);
    else if (vpl <= 8)
        rmsnorm_kernel<8><<<grid, RN_THREADS, 0, stream>>>(x, gamma, T, H, eps, xn);
    else if (vpl <= 16)
        rmsnorm_kernel<16><<<grid, RN_THREADS, 0, stream>>>(x, gamma, T, H, eps, xn);
    else if (vpl <= 32)
        rmsnorm_kernel<32><<<grid, RN_THREADS, 0, stream>>>(x, gamma, T, H, eps, xn);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

cudaError_t launch_sumsq(const uint16_t *x, int T, int H, float *ss, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    if (H <= 0 || H % 8 != 0) return cudaErrorInvalidValue;
    const int grid = static_cast<int>(
        std::max<int64_t>(1, std::min<int64_t>(ceil_div(T, 8), int64_t{num_sms()} * 8)));
    sumsq_kernel<<<grid, 256, 0, stream>>>(x, T, H, ss);
    return cudaGetLastError();
}

cudaError_t launch_gate_split(const float *wg, int E, int H, uint16_t *wsplit, int NW,
                              cudaStream_t stream) {
    if (H % 4 != 0 || NW < 3 * E) return cudaErrorInvalidValue;
    dim3 grid(static_cast<unsigned>(ceil_div(H / 4, 256)), static_cast<unsigned>(NW));
    gate_split_kernel<<<grid, 256, 0, stream>>>(wg, E, H, wsplit);
    return cudaGetLastError();
}

cudaError_t launch_gate_combine(const float *parts, int NW, int T, int E, const float *gate_bias,
                                float *logits, bool fuse_topk, int k, bool renorm,
                                int32_t *topk_idx, float *topk_w, int32_t *hist,
                                cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const bool fuse = fuse_topk && E <= RT_EXP;
    if (!fuse && !logits) return cudaErrorInvalidValue;
    gate_combine_kernel<<<static_cast<unsigned>(ceil_div(T, RT_TOK)), GC_THREADS, 0, stream>>>(
        parts, NW, T, E, gate_bias, logits, fuse ? 1 : 0, k, renorm ? 1 : 0, topk_idx, topk_w,
        fuse ? hist : nullptr);
    return cudaGetLastError();
}

}  // namespace moe
