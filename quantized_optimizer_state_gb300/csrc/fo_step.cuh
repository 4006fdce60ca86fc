// fo_step.cuh -- the fused compressed optimizer step (FlashAdamW, FlashSGD,
// FlashLion): "FlashOptim: Optimizers for Memory Efficient Training",
// section "融合优化器步骤" (Algorithm 4) -- dequantize m and v, rebuild the
// master weight, apply the standard update, requantize and re-split, in one
// pass so that each byte of state crosses HBM once.
//
// Design (GB300, sm_103a): the work is element-wise plus a 32-wide absmax per
// group, so it is bound by HBM traffic and instruction issue, never by tensor
// cores. A persistent grid (SMs x resident CTAs) walks the tiles of the
// concatenated tensor list in a static round-robin. A tile is 8 (large
// tables), 2 (small ones) or 1 (a few million elements) consecutive
// 4096-element chunks of one tensor, stepped one after the other. In a chunk, a thread owns 16 contiguous
// elements (half a group) and loads them with 128-bit streaming loads; the
// two threads of a group combine their absmax with one shuffle, and the
// results leave with 128-bit streaming stores. Pairs of elements are computed
// with packed FP32 instructions and exact fast division and square root
// (fo_pair.cuh; their hardware-dependent domains are enumerated on the device
// by fo_verify_fast_arithmetic).
// Exact zeros (zero gradients, momenta and second moments, as in rows that
// receive no gradient) stay on this path; a thread whose operands leave the
// validated ranges (a zero theta', a tiny non-zero gradient, extreme
// hyper-parameters) recomputes its 16 elements with IEEE operations. Tensor
// rows travel in the kernel parameters, so a step allocates nothing.
#pragma once

#include <atomic>
#include <utility>

#include "fo_device.cuh"
#include "fo_internal.h"
#include "fo_pair.cuh"

namespace fo {
namespace {

constexpr int kEPT = kElemsPerThread;

// AdamW's packed fast path carries the momentum and its companded value z
// scaled by 2^32 (m' = 2^32 m, z' = 2^32 z): every scaling is exact there and
// keeps the operands of its divisions inside their validated ranges (see
// pair_fast). SGD and Lion are unscaled. The exact path delivers z scaled the
// same way, so the requantization is common.
template <Opt O> struct ZScale {
    static constexpr int kInt = O == Opt::kAdamW ? 2 : 1;   // template tag of phi_m_pair
    static constexpr float up = O == Opt::kAdamW ? 0x1p32f : 1.0f;
    static constexpr float down = O == Opt::kAdamW ? 0x1p-32f : 1.0f;
};



struct Loaded {
    uint32_t g[16];  // 16 gradients: BF16 pairs in g[0..7], or FP32 in g[0..15]
    uint32_t t[8];   // 16 BF16 theta'
    uint32_t r[8];   // 16 rho codes (4 words for 8-bit, 8 for 16-bit)
    uint32_t m[4];   // 16 INT8 momentum codes
    uint32_t v[4];   // 16 UINT8 second-moment codes
    uint16_t ms, vs; // the group's FP16 scales
};

template <int RB, bool WithV, int GB>
__device__ __forceinline__ void load_chunk(const StepRow &row, int64_t i0, int cnt, Loaded &L)
{
    if (cnt == kEPT) {
        uint4 a, b;
        if (GB == 16) {
            const uint16_t *gp = static_cast<const uint16_t *>(row.grad) + i0;
            a = ld_stream(gp);
            b = ld_stream(gp + 8);
            L.g[0] = a.x; L.g[1] = a.y; L.g[2] = a.z; L.g[3] = a.w;
            L.g[4] = b.x; L.g[5] = b.y; L.g[6] = b.z; L.g[7] = b.w;
        } else {
            const float *gp = static_cast<const float *>(row.grad) + i0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                a = ld_stream(gp + 4 * q);
                L.g[4 * q] = a.x; L.g[4 * q + 1] = a.y; L.g[4 * q + 2] = a.z; L.g[4 * q + 3] = a.w;
            }
        }
        a = ld_stream(row.theta + i0);
        b = ld_stream(row.theta + i0 + 8);
        L.t[0] = a.x; L.t[1] = a.y; L.t[2] = a.z; L.t[3] = a.w;
        L.t[4] = b.x; L.t[5] = b.y; L.t[6] = b.z; L.t[7] = b.w;
        if (RB == 8) {
            a = ld_stream(static_cast<const int8_t *>(row.rho) + i0);
            L.r[0] = a.x; L.r[1] = a.y; L.r[2] = a.z; L.r[3] = a.w;
        } else {
            a = ld_stream(static_cast<const int16_t *>(row.rho) + i0);
            b = ld_stream(static_cast<const int16_t *>(row.rho) + i0 + 8);
            L.r[0] = a.x; L.r[1] = a.y; L.r[2] = a.z; L.r[3] = a.w;
            L.r[4] = b.x; L.r[5] = b.y; L.r[6] = b.z; L.r[7] = b.w;
        }
        a = ld_stream(row.mq + i0);
        L.m[0] = a.x; L.m[1] = a.y; L.m[2] = a.z; L.m[3] = a.w;
        if (WithV) {
            a = ld_stream(row.vq + i0);
            L.v[0] = a.x; L.v[1] = a.y; L.v[2] = a.z; L.v[3] = a.w;
        }
        L.ms = __ldcs(row.ms + (i0 >> 5));
        if (WithV)
            L.vs = __ldcs(row.vs + (i0 >> 5));
        return;
    }
    // ragged tail of a tensor: element-wise loads of the first cnt elements,
    // the rest read as 0 (and are masked out of the group absmax)
#pragma unroll
    for (int w = 0; w < 8; ++w) { L.t[w] = 0; L.r[w] = 0; }
    constexpr int kGradWords = GB == 16 ? 8 : 16;
#pragma unroll
    for (int w = 0; w < kGradWords; ++w)
        L.g[w] = 0;
#pragma unroll
    for (int w = 0; w < 4; ++w) { L.m[w] = 0; L.v[w] = 0; }
    // the group's scales, read only while the group exists (a lane whose
    // elements all lie past the end holds zero codes, which decode to zero
    // whatever the scale)
    const bool group_exists = ((i0 >> 5) << 5) < row.numel;
    L.ms = group_exists ? row.ms[i0 >> 5] : (uint16_t)0;
    L.vs = (WithV && group_exists) ? row.vs[i0 >> 5] : (uint16_t)0;
    if (cnt <= 0)
        return;
#pragma unroll
    for (int j = 0; j < kEPT; ++j) {
        if (j >= cnt)
            break;
        const int sh16 = 16 * (j & 1), sh8 = 8 * (j & 3);
        if (GB == 16)
            L.g[j >> 1] |= (uint32_t)static_cast<const uint16_t *>(row.grad)[i0 + j] << sh16;
        else
            L.g[j] = static_cast<const uint32_t *>(row.grad)[i0 + j];
        L.t[j >> 1] |= (uint32_t)row.theta[i0 + j] << sh16;
        if (RB == 8)
            L.r[j >> 2] |= (uint32_t)(uint8_t)static_cast<const int8_t *>(row.rho)[i0 + j] << sh8;
        else
            L.r[j >> 1] |= (uint32_t)(uint16_t)static_cast<const int16_t *>(row.rho)[i0 + j] << sh16;
        L.m[j >> 2] |= (uint32_t)(uint8_t)row.mq[i0 + j] << sh8;
        if (WithV)
            L.v[j >> 2] |= (uint32_t)row.vq[i0 + j] << sh8;
    }
}

// rho of element j as a float (exact).
template <int RB, int J>
__device__ __forceinline__ float rho_at(const uint32_t (&rx)[8])
{
    if (RB == 8)
        return s8_at<J & 3>(rx[J >> 2]);
    else
        return s16_at<J & 1>(rx[J >> 1]);
}

template <int J>
__device__ __forceinline__ uint32_t theta_p_bits(const uint32_t (&t)[8])
{
    return (J & 1) ? bf16_hi_bits(t[J >> 1]) : bf16_lo_bits(t[J >> 1]);
}

// gradient of element j as FP32 (BF16 widened exactly, or FP32 as loaded)
template <int GB, int J>
__device__ __forceinline__ float grad_at(const Loaded &L)
{
    if (GB == 16)
        return __uint_as_float((J & 1) ? (L.g[J >> 1] & 0xFFFF0000u) : (L.g[J >> 1] << 16));
    else
        return __uint_as_float(L.g[J]);
}

// gradients of elements 2w and 2w+1, packed
template <int GB, int W>
__device__ __forceinline__ f2 grad_pair(const Loaded &L)
{
    if (GB == 16)
        return pk(__uint_as_float(L.g[W] << 16), __uint_as_float(L.g[W] & 0xFFFF0000u));
    else
        return pk(__uint_as_float(L.g[2 * W]), __uint_as_float(L.g[2 * W + 1]));
}

// Exact path, element j: decode, update, and the new theta (FP32), the
// companded momentum z and nr = -sqrt(v) (AdamW; 0 otherwise), with the IEEE
// operations of the library's arithmetic contract. It serves the threads
// whose operands fall outside the validated ranges of the packed fast path.
template <Opt O, int RB, int GB, int J>
__device__ __forceinline__ void element_exact(const Loaded &L, const uint32_t (&rx)[8], const uint32_t (&mx)[4],
                                              const StepScalars &s, float coef, float cm, float cv,
                                              float &theta_out, float &z_out, float &nr_out)
{
    const float g = grad_at<GB, J>(L);
    float theta = merge_one<RB>(theta_p_bits<J>(L.t), rho_at<RB, J>(rx));
    const float zq = __fmul_rn(s8_at<J & 3>(mx[J >> 2]), cm);
    float m = phi_m_inv(zq);

    if (O == Opt::kAdamW) {
        const float rq = __fmul_rn(u8_at<J & 3>(L.v[J >> 2]), cv);
        float v = __fmul_rn(rq, rq);
        theta = __fmul_rn(theta, coef);
        m = __fmaf_rn(s.a[0], m, __fmul_rn(s.a[2], g));
        v = __fmaf_rn(s.a[1], v, __fmul_rn(__fmul_rn(s.a[3], g), g));
        const float r = __fsqrt_rn(v);
        const float den = __fmaf_rn(r, s.a[6], s.a[4]);
        theta = __fmaf_rn(s.a[5], __fdiv_rn(m, den), theta);
        nr_out = -r;
    } else if (O == Opt::kSgd) {
        const float gp = __fmaf_rn(coef, theta, g);
        m = __fmaf_rn(s.a[0], m, gp);
        theta = __fmaf_rn(s.a[1], m, theta);
        nr_out = 0.0f;
    } else {
        const float c = __fmaf_rn(s.a[0], m, __fmul_rn(s.a[2], g));
        const float sgn = c > 0.0f ? 1.0f : (c < 0.0f ? -1.0f : 0.0f);
        theta = __fmaf_rn(s.a[4], sgn, __fmul_rn(theta, coef));
        m = __fmaf_rn(s.a[1], m, __fmul_rn(s.a[3], g));
        nr_out = 0.0f;
    }
    theta_out = theta;
    // an infinite momentum (a code byte of -128 decodes to -inf under the
    // scale 127/64) companded is NaN: coded 0 like any NaN, which a zero z
    // gives, and left out of the group maximum (fmaxf ignores NaN and 0 does
    // not raise it)
    const float zz = __fmul_rn(phi_m(m), ZScale<O>::up);
    z_out = zz != zz ? 0.0f : zz;
}

template <Opt O, int RB, int GB, int... J>
__device__ __forceinline__ void all_exact(const Loaded &L, const uint32_t (&rx)[8], const uint32_t (&mx)[4],
                                          const StepScalars &s, float coef, float cm, float cv,
                                          float (&th)[kEPT], float (&z)[kEPT], float (&nr)[kEPT],
                                          std::integer_sequence<int, J...>)
{
    (element_exact<O, RB, GB, J>(L, rx, mx, s, coef, cm, cv, th[J], z[J], nr[J]), ...);
}

// ---------------------------------------------------------------------------
// Packed fast path: elements 2w and 2w+1 in the two lanes of f32x2 operations.
// Every operation rounds exactly as its scalar counterpart in element_exact;
// division and square root use the validated sequences of fo_pair.cuh, and
// `bad` is raised when an operand leaves their validated range.
// ---------------------------------------------------------------------------

// Running extremes of the fast path's range-checked operands; one check per
// thread at the end (three-input min/max instead of a compare per element).
//
// The checked operand x (the gradient for AdamW, the new momentum for SGD and
// Lion) may be an exact zero or lie in a range [lo, hi] of magnitudes. A zero
// is told apart from a tiny value without a compare: c = pattern(x) +
// 0x7FFFFFFF (mod 2^32) is a NaN for x = +-0 and otherwise a float whose
// magnitude is the FP32 value just below |x|. min/max ignore NaNs, so the
// running extremes of |c| see only the non-zero operands.
struct Guard {
    float min_tp;   // smallest |theta'| (0: a zero theta', exact path)
    float min_c;    // smallest |c| over non-zero checked operands
    float max_c;    // largest |c|
    __device__ __forceinline__ void init()
    {
        min_tp = __int_as_float(0x7F800000);
        min_c = __int_as_float(0x7F800000);
        max_c = 0.0f;
    }
    // both bounds (SGD, Lion: the new momentum)
    __device__ __forceinline__ void range(float x0, float x1)
    {
        const float c0 = __uint_as_float(__float_as_uint(x0) + 0x7FFFFFFFu);
        const float c1 = __uint_as_float(__float_as_uint(x1) + 0x7FFFFFFFu);
        min_c = fminf(min_c, fminf(fabsf(c0), fabsf(c1)));
        max_c = fmaxf(max_c, fmaxf(fabsf(c0), fabsf(c1)));
    }
    // the lower bound only (AdamW: the gradient; its upper bound is checked
    // through sqrt(v), see thread_step)
    __device__ __forceinline__ void range_lo(float x0, float x1)
    {
        const float c0 = __uint_as_float(__float_as_uint(x0) + 0x7FFFFFFFu);
        const float c1 = __uint_as_float(__float_as_uint(x1) + 0x7FFFFFFFu);
        min_c = fminf(min_c, fminf(fabsf(c0), fabsf(c1)));
    }
    // lo, hi: the bounds on |c| (the FP32 values just below the bounds on |x|)
    __device__ __forceinline__ bool failed(float lo, float hi) const
    {
        return !(min_tp > 0.0f) | !(min_c >= lo) | !(max_c <= hi);
    }
};

// Per-thread packed constants.
struct PairConsts {
    f2 cm;      // s_m / 127 (both lanes)
    f2 cv;      // s_v / 255
    f2 ncv23;   // -(2^23 * s_v / 255): (2^23 + q) * cv - 2^23 * cv = q * cv exactly
    f2 coef;    // per-row decay (AdamW, Lion) or weight decay (SGD)
};

// theta^ of elements 2w, 2w+1 (see merge_one), packed: the pattern of theta'
// plus sign(theta') * rint(rho*kappa * 2^15), the sign applied through the
// multiplier +-2^15 of the rounding fma. A zero theta' (whose h is 2^-134
// instead) raises `bad` for the exact path.
template <int RB, int W>
__device__ __forceinline__ f2 merge_pair(const Loaded &L, const uint32_t (&rx)[8], Guard &gd)
{
    const uint32_t u0 = L.t[W] << 16, u1 = L.t[W] & 0xFFFF0000u;
    f2 rho;
    if (RB == 8) {
        constexpr int b0 = (2 * W) & 3, b1 = (2 * W + 1) & 3;
        const uint32_t w = rx[(2 * W) >> 2];
        rho = add2(pk(__uint_as_float(__byte_perm(w, 0x4B000000u, 0x7440u | b0)),
                      __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7440u | b1))),
                   splat(-8388736.0f));
    } else {
        const uint32_t w = rx[W];
        rho = add2(pk(__uint_as_float(__byte_perm(w, 0x4B000000u, 0x7410u)),
                      __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7432u))),
                   splat(-8421376.0f));
    }
    f2 nb;   // M + sign(theta') * rint(RN(rho*kappa) * 2^15)
    if (RB == 8) {
        // for every 8-bit rho, rint(rho*kappa*2^15) with the exact product
        // equals rint(RN(rho*kappa)*2^15): one fma with +-kappa*2^15
        const uint32_t kb = __float_as_uint(RhoConst<8>::kappa * 32768.0f);
        nb = fma2(rho, pk(__uint_as_float((u0 & 0x80000000u) | kb), __uint_as_float((u1 & 0x80000000u) | kb)),
                  splat(kRoundMagic));
    } else {
        const f2 t = mul2(rho, splat(RhoConst<RB>::kappa));
        nb = fma2(t, pk(__uint_as_float((u0 & 0x80000000u) | 0x47000000u),       // +-2^15
                        __uint_as_float((u1 & 0x80000000u) | 0x47000000u)),
                  splat(kRoundMagic));
    }
    float n0f, n1f;
    unpk(nb, n0f, n1f);
    gd.min_tp = fminf(gd.min_tp, fminf(fabsf(__uint_as_float(u0)), fabsf(__uint_as_float(u1))));
    return pk(__uint_as_float(u0 + __float_as_uint(n0f) - kRoundMagicBits),
              __uint_as_float(u1 + __float_as_uint(n1f) - kRoundMagicBits));
}

// m^ = phi_m^-1(code * s_m/127) of elements 2w, 2w+1, packed.
template <int W>
__device__ __forceinline__ f2 mhat_pair(const uint32_t (&mx)[4], const PairConsts &k)
{
    constexpr int b0 = (2 * W) & 3, b1 = (2 * W + 1) & 3;
    const uint32_t w = mx[(2 * W) >> 2];
    const f2 q = add2(pk(__uint_as_float(__byte_perm(w, 0x4B000000u, 0x7440u | b0)),
                         __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7440u | b1))),
                      splat(-8388736.0f));
    const f2 zq = mul2(q, k.cm);
    float a0, a1;
    unpk(zq, a0, a1);
    // |zq| - 2 = -(2 - |zq|): |zq| < 2 for every code byte (-128 included)
    // under the fast path's momentum scales (below 127/64, see thread_step)
    return div2_short(zq, pk(__fsub_rn(fabsf(a0), 2.0f), __fsub_rn(fabsf(a1), 2.0f)));   // enumerated domain
}

// z = phi_m(m) = RN(2m / RN(1 + |m|)), packed, as RN(m / (RN(1 + |m|)/2)):
// halving is exact and commutes with rounding (the divisor is at least 1/2),
// so the quotient is the same real number without forming 2m. The halved
// divisor is one fma, RN(-0.5*|m| - 0.5) = -RN(1 + |m|)/2. With ZS = 2^32 the
// argument is m' = 2^32 m and the result 2^32 z (exact scalings: the fast path
// keeps them inside the normal range).
template <int ZS>
__device__ __forceinline__ f2 phi_m_pair(f2 m)
{
    constexpr float kHalfOverZ = ZS == 1 ? -0.5f : -0x1p-33f;
    float m0, m1;
    unpk(m, m0, m1);
    // (the short division: enumerated over every m of the fast path's range)
    return div2_short(m, pk(__fmaf_rn(kHalfOverZ, fabsf(m0), -0.5f), __fmaf_rn(kHalfOverZ, fabsf(m1), -0.5f)));
}

template <Opt O, int RB, int GB, int W>
__device__ __forceinline__ void pair_fast(const Loaded &L, const uint32_t (&rx)[8], const uint32_t (&mx)[4],
                                          const StepScalars &s, const PairConsts &k,
                                          f2 &th_out, float (&z)[kEPT], float (&nr)[kEPT], Guard &gd)
{
    constexpr int j0 = 2 * W, j1 = 2 * W + 1;
    const f2 g = grad_pair<GB, W>(L);
    const f2 theta = merge_pair<RB, W>(L, rx, gd);
    const f2 mhat = mhat_pair<W>(mx, k);
    f2 thn, m, nrv = 0;

    if (O == Opt::kAdamW) {
        // the gradient decides every operand range: g = 0 or |g| >= lo, with
        // the host's preconditions and sqrt(v) <= 2^40 (checked in
        // thread_step), keeps v at 0 or in [2^-100, 2^80] and m at 0 or |m| in
        // [2^-94, 2^53] (see fo_api.cu)
        float g0, g1;
        unpk(g, g0, g1);
        gd.range_lo(g0, g1);
        // (2^23 + q) as floats -> q * s_v/255 in one fma
        constexpr int b0 = j0 & 3, b1 = j1 & 3;
        const uint32_t vw = L.v[j0 >> 2];
        const f2 rq = fma2(pk(__uint_as_float(__byte_perm(vw, 0x4B000000u, 0x7440u | b0)),
                              __uint_as_float(__byte_perm(vw, 0x4B000000u, 0x7440u | b1))),
                           k.cv, k.ncv23);
        const f2 vhat = mul2(rq, rq);
        const f2 thd = mul2(theta, k.coef);
        m = fma2(s.p[0], mhat, mul2(s.p[2], g));                   // m' = 2^32 (b1*m + (1-b1)*g)
        const f2 nv = fma2(s.p[1], vhat, mul2(mul2(s.p[3], g), g)); // -(b2*v + ((1-b2)*g)*g)
        nrv = neg_sqrt2(nv);                                        // -sqrt(v) (+0 for v = 0)
        const f2 nden = fma2(nrv, s.p[4], s.p[5]);                  // -(sqrt(v)/sqrt(bc2) + eps)
        const f2 u = div2(m, nden);                                 // 2^32 m / den
        thn = fma2(s.p[6], u, thd);                                 // theta - lr/bc1 * m/den
    } else if (O == Opt::kSgd) {
        const f2 gp = fma2(k.coef, theta, g);                       // g + wd*theta
        m = fma2(s.p[0], mhat, gp);                                 // mu*m + g'
        thn = fma2(s.p[1], m, theta);                               // theta - lr*m
        float m0, m1;
        unpk(m, m0, m1);
        gd.range(m0, m1);                                           // m = 0 or |m| in [2^-100, 2^100]
    } else {
        const f2 c = fma2(s.p[0], mhat, mul2(s.p[2], g));           // b1*m + (1-b1)*g
        float c0, c1;
        unpk(c, c0, c1);
        const f2 sgn = pk(c0 > 0.0f ? 1.0f : (c0 < 0.0f ? -1.0f : 0.0f),
                          c1 > 0.0f ? 1.0f : (c1 < 0.0f ? -1.0f : 0.0f));
        thn = fma2(s.p[4], sgn, mul2(theta, k.coef));               // theta*(1-lr*wd) - lr*sign(c)
        m = fma2(s.p[1], mhat, mul2(s.p[3], g));                    // b2*m + (1-b2)*g
        float m0, m1;
        unpk(m, m0, m1);
        gd.range(m0, m1);                                           // m = 0 or |m| in [2^-100, 2^100]
    }
    th_out = thn;
    unpk(phi_m_pair<ZScale<O>::kInt>(m), z[j0], z[j1]);
    unpk(nrv, nr[j0], nr[j1]);
}

// Re-split of two new theta values: theta' (BF16, nearest even) as one word
// and their rho codes (8-bit: the low two bytes; 16-bit: two halves). See
// split_code: the magnitude residual is scaled in a packed fma and theta's
// sign is applied to the FP32 value before rounding, as rint is odd.
template <int RB>
__device__ __forceinline__ void split_pair(float th0, float th1, uint32_t &tpw, uint32_t &rw)
{
    tpw = pack_bf16x2(th0, th1);
    const uint32_t t0 = __float_as_uint(th0), t1 = __float_as_uint(th1);
    const f2 x = fma2(pk(__uint_as_float(t0 - bf16_lo_bits(tpw) + kRoundMagicBits),
                         __uint_as_float(t1 - bf16_hi_bits(tpw) + kRoundMagicBits)),
                      splat(RhoConst<RB>::qscale), splat(-RhoConst<RB>::offset));
    float x0, x1;
    unpk(x, x0, x1);
    const f2 c = add2(pk(__uint_as_float(__float_as_uint(x0) ^ (t0 & 0x80000000u)),
                         __uint_as_float(__float_as_uint(x1) ^ (t1 & 0x80000000u))),
                      splat(kRoundMagic));
    float c0f, c1f;
    unpk(c, c0f, c1f);
    const uint32_t c0 = __float_as_uint(c0f), c1 = __float_as_uint(c1f);
    rw = RB == 16 ? pack_halves(c0, c1) : __byte_perm(c0, c1, 0x0040u);
}

// theta', rho of elements 4q .. 4q+3 into tp and ro
template <int RB, int Q>
__device__ __forceinline__ void split_quad(float th0, float th1, float th2, float th3, uint32_t (&tp)[8],
                                           uint32_t (&ro)[8])
{
    uint32_t r0, r1;
    split_pair<RB>(th0, th1, tp[2 * Q], r0);
    split_pair<RB>(th2, th3, tp[2 * Q + 1], r1);
    if (RB == 8) {
        ro[Q] = __byte_perm(r0, r1, 0x5410u);
    } else {
        ro[2 * Q] = r0;
        ro[2 * Q + 1] = r1;
    }
}

template <int RB, int... Q>
__device__ __forceinline__ void split_all(const float (&th)[kEPT], uint32_t (&tp)[8], uint32_t (&ro)[8],
                                          std::integer_sequence<int, Q...>)
{
    (split_quad<RB, Q>(th[4 * Q], th[4 * Q + 1], th[4 * Q + 2], th[4 * Q + 3], tp, ro), ...);
}

// Elements 4q .. 4q+3 (two pairs). ES: re-split the new theta at once into tp
// and ro (AdamW: fewer live registers); otherwise leave it in th.
template <Opt O, int RB, int GB, bool ES, int Q>
__device__ __forceinline__ void quad_fast(const Loaded &L, const uint32_t (&rx)[8], const uint32_t (&mx)[4],
                                          const StepScalars &s, const PairConsts &k, float (&th)[kEPT],
                                          uint32_t (&tp)[8], uint32_t (&ro)[8], float (&z)[kEPT],
                                          float (&nr)[kEPT], Guard &gd)
{
    f2 t0, t1;
    pair_fast<O, RB, GB, 2 * Q>(L, rx, mx, s, k, t0, z, nr, gd);
    pair_fast<O, RB, GB, 2 * Q + 1>(L, rx, mx, s, k, t1, z, nr, gd);
    float a, b, c, d;
    unpk(t0, a, b);
    unpk(t1, c, d);
    if (ES) {
        split_quad<RB, Q>(a, b, c, d, tp, ro);
    } else {
        th[4 * Q] = a;
        th[4 * Q + 1] = b;
        th[4 * Q + 2] = c;
        th[4 * Q + 3] = d;
    }
}

template <Opt O, int RB, int GB, bool ES, int... Q>
__device__ __forceinline__ void all_fast(const Loaded &L, const uint32_t (&rx)[8], const uint32_t (&mx)[4],
                                         const StepScalars &s, const PairConsts &k, float (&th)[kEPT],
                                         uint32_t (&tp)[8], uint32_t (&ro)[8], float (&z)[kEPT],
                                         float (&nr)[kEPT], Guard &gd, std::integer_sequence<int, Q...>)
{
    (quad_fast<O, RB, GB, ES, Q>(L, rx, mx, s, k, th, tp, ro, z, nr, gd), ...);
}

__device__ __forceinline__ int chunk_count(const StepRow &row, int64_t i0)
{
    const int64_t rem = row.numel - i0;
    return rem >= kEPT ? kEPT : (rem > 0 ? (int)rem : 0);
}

// One thread's 16 elements of a tile, from data already loaded into L.
// VNZ (AdamW): requantize v with no code 0 in groups with a non-zero scale.
template <Opt O, int RB, int GB, bool VNZ, int CH>
__device__ __forceinline__ void thread_step(const StepRow &row, const StepScalars &s, int64_t i0, int cnt,
                                            Loaded &L)
{
    constexpr bool WithV = (O == Opt::kAdamW);
    const bool even = (threadIdx.x & 1) == 0;

    // bias the signed codes once per word for the exact byte -> float unpack
    uint32_t rx[8], mx[4];
#pragma unroll
    for (int w = 0; w < 8; ++w)
        rx[w] = L.r[w] ^ (RB == 8 ? 0x80808080u : 0x80008000u);
#pragma unroll
    for (int w = 0; w < 4; ++w)
        mx[w] = L.m[w] ^ 0x80808080u;

    // decode steps s/127 (m) and s/255 (v): correctly rounded divisions by a
    // constant through its correctly rounded reciprocal (s is 0 or an FP16
    // value in [2^-24, 65504], inside the validated range)
    const float cm = div_by_const(scale_value(L.ms), -127.0f, kRcp127);
    const float cv = WithV ? div_by_const(scale_value(L.vs), -255.0f, kRcp255) : 0.0f;

    // AdamW, and SGD on short tiles (5 CTAs per SM), re-split theta on the
    // fast path as soon as a quad is stepped, so that the 16 new theta values
    // are never held (AdamW at 4 CTAs: 5 % faster); SGD on long tiles and Lion
    // re-split after the step (faster for them)
    constexpr bool ES = (O == Opt::kAdamW) || (O == Opt::kSgd && CH != kLongChunks);
    float th[kEPT], z[kEPT], nr[kEPT];
    uint32_t tp[8], ro[8];
    float av = 0.0f;   // the thread's largest sqrt(v) (AdamW)
    // the fast path needs the host's range preconditions and a momentum scale
    // s below 127/64 = 1.984375, where |z| = |q| s/127 < 2 for every code
    // byte q (-128 included, which the quantizer never writes but a caller
    // may pass), so that 2 - |z| stays positive; otherwise every element of
    // this thread goes through the exact path (an FP16 pattern of 0x3FF0 or
    // more is 127/64 or above, infinite, NaN or negative). AdamW and Lion also
    // need a decay factor of at least 2^-8 in magnitude, so that a decayed
    // theta is never zero.
    bool bad = !s.fast || L.ms >= 0x3FF0u || (O != Opt::kSgd && !(fabsf(row.coef) >= 0x1p-8f));
    if (!bad) {
        PairConsts k;
        k.cm = splat(cm);
        k.cv = splat(cv);
        k.ncv23 = splat(__fmul_rn(cv, -8388608.0f));
        k.coef = splat(row.coef);
        Guard gd;
        gd.init();
        all_fast<O, RB, GB, ES>(L, rx, mx, s, k, th, tp, ro, z, nr, gd, std::make_integer_sequence<int, kEPT / 4>{});
        bad = gd.failed(s.lo, s.hi);
        if (WithV) {
            // the largest sqrt(v), with NaNs propagated: sqrt(v) <= 2^40 bounds
            // |g| <= 2^52 (v >= (1-b2) g^2 and 1-b2 >= 2^-24), the upper half
            // of the gradient's range check
#pragma unroll
            for (int j = 0; j < kEPT; j += 2)
                av = max3_nan(av, fabsf(nr[j]), fabsf(nr[j + 1]));
            bad = bad | !(av <= 0x1p40f);
        }
    }
    if (bad) {
        // rare: reload (the data is unchanged) and recompute with IEEE operations
        load_chunk<RB, WithV, GB>(row, i0, cnt, L);
#pragma unroll
        for (int w = 0; w < 8; ++w)
            rx[w] = L.r[w] ^ (RB == 8 ? 0x80808080u : 0x80008000u);
#pragma unroll
        for (int w = 0; w < 4; ++w)
            mx[w] = L.m[w] ^ 0x80808080u;
        all_exact<O, RB, GB>(L, rx, mx, s, row.coef, cm, cv, th, z, nr, std::make_integer_sequence<int, kEPT>{});
        av = 0.0f;
#pragma unroll
        for (int j = 0; j < kEPT; ++j)
            av = fmaxf(av, fabsf(nr[j]));   // sqrt(v); nr is -sqrt(v)
        if (ES)
            split_all<RB>(th, tp, ro, std::make_integer_sequence<int, kEPT / 4>{});
    }

    // re-split theta: theta' (BF16, nearest even) and rho (split_pair)
    if (!ES)
        split_all<RB>(th, tp, ro, std::make_integer_sequence<int, kEPT / 4>{});

    // group absmax over this thread's elements, then over the pair. Lanes past
    // the end of the tensor were loaded as zeros and so hold z = 0 and
    // sqrt(v) = 0 exactly: they leave the maxima unchanged.
    // (av, the second moment's, is already formed: on the fast path nr is
    // -sqrt(v), or +0 for v = 0, and fabs makes both paths agree)
    float am = 0.0f;
#pragma unroll
    for (int j = 0; j < kEPT; ++j)
        am = fmaxf(am, fabsf(z[j]));
    am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 1));
    if (WithV)
        av = fmaxf(av, __shfl_xor_sync(0xFFFFFFFFu, av, 1));

    const uint16_t sm_new = scale_of(__fmul_rn(am, ZScale<O>::down));   // exact: am is 2^32 |z| for AdamW
    const uint16_t sv_new = WithV ? scale_of(av) : (uint16_t)0;
    // code multipliers 127/s (m) and 255/s (v), 0 for a zero scale; s is a
    // positive finite FP16 value there, on which the short division was
    // enumerated
    const float s_m = scale_value(sm_new), s_v = scale_value(sv_new);
    // (for AdamW z holds 2^32 z, so the multiplier is scaled by 2^-32: exact,
    // and the product z * (127/s) is the same real number)
    const float mult_m = s_m > 0.0f ? __fmul_rn(div1_short(127.0f, s_m), ZScale<O>::down) : 0.0f;
    const float mult_v = (WithV && s_v > 0.0f) ? div1_short(255.0f, s_v) : 0.0f;
    // codes: clamp(rint(x)), x = RN(phi * (L/s)). For m with a normal FP16
    // scale below the 65504 cap the group maximum is at most s*(1 + 2^-11),
    // so |x| <= 127.07: no clamp can apply, and rint is the magic-number
    // addition on the FMA pipe (the code in the low byte). Subnormal or
    // capped m scales, and all v codes, take the saturating conversion.
    const bool fadd_m = s_m == 0.0f || (s_m >= 0x1p-14f && s_m < 65504.0f);
    uint32_t mo[4], vo[4];
    if (fadd_m) {
        // The product is formed as fma(z, 127/s, +0) with a zero the compiler
        // cannot prove (127/s * 0 is not 0 for an infinite 127/s), so that the
        // rounding add stays a separate rounding: fusing the two would need
        // four operands.
        const f2 zero_m = splat(__fmul_rn(mult_m, 0.0f));
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            float c0, c1, c2, c3;
            unpk(add2(fma2(pk(z[4 * w], z[4 * w + 1]), splat(mult_m), zero_m), splat(kRoundMagic)), c0, c1);
            unpk(add2(fma2(pk(z[4 * w + 2], z[4 * w + 3]), splat(mult_m), zero_m), splat(kRoundMagic)), c2, c3);
            mo[w] = pack_bytes(__float_as_uint(c0), __float_as_uint(c1), __float_as_uint(c2), __float_as_uint(c3));
        }
    } else {
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            float x0, x1, x2, x3;
            unpk(mul2(pk(z[4 * w], z[4 * w + 1]), splat(mult_m)), x0, x1);
            unpk(mul2(pk(z[4 * w + 2], z[4 * w + 3]), splat(mult_m)), x2, x3);
            mo[w] = pack_bytes(m_code_sat(x0), m_code_sat(x1), m_code_sat(x2), m_code_sat(x3));
        }
    }
    if (WithV) {
        // r * (255/s) = (-r) * (-(255/s)), exactly
        const float nmult_v = -mult_v;
        const float vfloor = mult_v > 0.0f ? 1.0f : 0.0f;   // VNZ: at least code 1 in a live group
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            float x0, x1, x2, x3;
            unpk(mul2(pk(nr[4 * w], nr[4 * w + 1]), splat(nmult_v)), x0, x1);
            unpk(mul2(pk(nr[4 * w + 2], nr[4 * w + 3]), splat(nmult_v)), x2, x3);
            if (VNZ) {
                x0 = fmaxf(x0, vfloor);
                x1 = fmaxf(x1, vfloor);
                x2 = fmaxf(x2, vfloor);
                x3 = fmaxf(x3, vfloor);
            }
            vo[w] = pack_bytes(v_code_sat(x0), v_code_sat(x1), v_code_sat(x2), v_code_sat(x3));
        }
    }

    if (cnt == kEPT) {
        st_stream(row.theta + i0, make_uint4(tp[0], tp[1], tp[2], tp[3]));
        st_stream(row.theta + i0 + 8, make_uint4(tp[4], tp[5], tp[6], tp[7]));
        if (RB == 8) {
            st_stream(static_cast<int8_t *>(row.rho) + i0, make_uint4(ro[0], ro[1], ro[2], ro[3]));
        } else {
            st_stream(static_cast<int16_t *>(row.rho) + i0, make_uint4(ro[0], ro[1], ro[2], ro[3]));
            st_stream(static_cast<int16_t *>(row.rho) + i0 + 8, make_uint4(ro[4], ro[5], ro[6], ro[7]));
        }
        st_stream(row.mq + i0, make_uint4(mo[0], mo[1], mo[2], mo[3]));
        if (WithV)
            st_stream(row.vq + i0, make_uint4(vo[0], vo[1], vo[2], vo[3]));
    } else {
#pragma unroll
        for (int j = 0; j < kEPT; ++j) {
            if (j >= cnt)
                break;
            const int sh16 = 16 * (j & 1), sh8 = 8 * (j & 3);
            row.theta[i0 + j] = (uint16_t)(tp[j >> 1] >> sh16);
            if (RB == 8)
                static_cast<int8_t *>(row.rho)[i0 + j] = (int8_t)(ro[j >> 2] >> sh8);
            else
                static_cast<int16_t *>(row.rho)[i0 + j] = (int16_t)(ro[j >> 1] >> sh16);
            row.mq[i0 + j] = (int8_t)(mo[j >> 2] >> sh8);
            if (WithV)
                row.vq[i0 + j] = (uint8_t)(vo[j >> 2] >> sh8);
        }
    }
    if (even && cnt > 0) {
        __stcs(row.ms + (i0 >> 5), sm_new);
        if (WithV)
            __stcs(row.vs + (i0 >> 5), sv_new);
    }
}

// b^t by repeated squaring in double: the same operations, in the same order,
// as the host's derivation of the step scalars.
__device__ double pow_by_squaring_dev(double b, long long t)
{
    double r = 1.0;
    while (t > 0) {
        if (t & 1)
            r = __dmul_rn(r, b);
        b = __dmul_rn(b, b);
        t >>= 1;
    }
    return r;
}

__device__ unsigned long long lanes_dev(float x)
{
    const unsigned long long u = __float_as_uint(x);
    return (u << 32) | u;
}

// AdamW's step-dependent scalars from the step counter in device memory, with
// the host's expressions (fo_api.cu): bc_i = 1 - b_i^t, a[5] = -(float)(lr/bc1),
// a[6] = (float)(1/sqrt(bc2)), their packed forms, and the fast path's
// t-dependent preconditions. skip is set for t < 1 (nothing is updated).
__device__ void derive_step_scalars(const StepScalars &in, StepScalars &out)
{
    out = in;
    const long long t = *in.step_dev;
    if (t < 1) {
        out.skip = 1;
        return;
    }
    const double bc1 = __dadd_rn(1.0, -pow_by_squaring_dev(in.beta1, t));
    const double bc2 = __dadd_rn(1.0, -pow_by_squaring_dev(in.beta2, t));
    const float step = __double2float_rn(__ddiv_rn(in.lr, bc1));
    const float a6 = __double2float_rn(__ddiv_rn(1.0, __dsqrt_rn(bc2)));
    out.a[5] = -step;
    out.a[6] = a6;
    out.p[4] = lanes_dev(a6);
    out.p[6] = lanes_dev(__fmul_rn(-step, 0x1p-32f));
    out.fast = (in.fast && a6 <= 0x1p8f && (step == 0.0f || step >= 0x1p-80f)) ? 1 : 0;
}

// The tile walk of one CTA, with the step scalars in s.
template <Opt O, int RB, int GB, bool VNZ, int CH>
__device__ __forceinline__ void step_tiles(const StepParams &p, const StepScalars &s)
{
    constexpr bool WithV = (O == Opt::kAdamW);
    // Lion's chunk loop is unrolled by two (13.27 -> 13.06 ms on the
    // Llama-3.1-8B Lion step); AdamW's, unrolled, was 4 % slower
    constexpr int kUnroll = O == Opt::kLion ? 2 : 1;
    int row = 0;
    for (int tile = blockIdx.x; tile < p.total_tiles; tile += gridDim.x) {
        while (tile >= p.tile_end[row])
            ++row;
        const int first = row == 0 ? 0 : p.tile_end[row - 1];
        const StepRow &r = p.rows[row];
        const int64_t t0 = (int64_t)(tile - first) * CH * kStepChunk + (int64_t)threadIdx.x * kEPT;
#pragma unroll kUnroll
        for (int c = 0; c < CH; ++c) {
            const int64_t i0 = t0 + (int64_t)c * kStepChunk;
            const int cnt = chunk_count(r, i0);
            // a warp entirely past the tensor's end has nothing to do (a
            // warp-uniform exit: no lane is left waiting on the group shuffle)
            if (__all_sync(0xFFFFFFFFu, cnt <= 0))
                break;
            Loaded L;
            load_chunk<RB, WithV, GB>(r, i0, cnt, L);
            thread_step<O, RB, GB, VNZ, CH>(r, s, i0, cnt, L);
        }
    }
}

// One launch: rows of one rho width (RB) and gradient width (GB), walked
// tile by tile, CH chunks per tile. DEV (AdamW): the step counter is read
// from device memory when the kernel runs and the step scalars are derived
// from it, once per CTA, into shared memory.
template <Opt O, int RB, int GB, bool VNZ, int CH, bool DEV = false>
__global__ void __launch_bounds__(kStepThreads, step_ctas_per_sm(O, RB, GB, CH))
fo_fused_step_kernel(const __grid_constant__ StepParams p)
{
    if constexpr (DEV) {
        __shared__ StepScalars dev_s;
        if (threadIdx.x == 0)
            derive_step_scalars(p.s, dev_s);
        __syncthreads();
        if (dev_s.skip)
            return;
        step_tiles<O, RB, GB, VNZ, CH>(p, dev_s);
    } else {
        step_tiles<O, RB, GB, VNZ, CH>(p, p.s);
    }
}

template <Opt O, int RB, int GB, bool VNZ, int CH, bool DEV>
int resident_ctas()
{
    // per device (up to 64), cached after the first successful query; a
    // failed query is not cached, and its error is consumed so that the
    // launch reports its own status
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
        (void)cudaGetLastError();
        dev = 0;
    }
    std::atomic<int> &slot = cached[dev & 63];
    int n = slot.load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fo_fused_step_kernel<O, RB, GB, VNZ, CH, DEV>, kStepThreads,
                                                          0) != cudaSuccess ||
            n < 1) {
            (void)cudaGetLastError();
            return 1;
        }
        slot.store(n, std::memory_order_relaxed);
    }
    return n;
}

template <Opt O, int RB, int GB, bool VNZ, int CH, bool DEV>
cudaError_t launch_ch(const StepParams &p, cudaStream_t stream)
{
    const long long want = (long long)sm_count() * resident_ctas<O, RB, GB, VNZ, CH, DEV>();
    const int grid = (int)(want < p.total_tiles ? want : p.total_tiles);
    fo_fused_step_kernel<O, RB, GB, VNZ, CH, DEV><<<grid, kStepThreads, 0, stream>>>(p);
    count_launch();
    return cudaGetLastError();
}

template <Opt O, int RB, int GB, bool VNZ = false, bool DEV = false>
cudaError_t launch(const StepParams &p, cudaStream_t stream)
{
    if (p.chunks == kLongChunks)
        return launch_ch<O, RB, GB, VNZ, kLongChunks, DEV>(p, stream);
    if (p.chunks == kShortChunks)
        return launch_ch<O, RB, GB, VNZ, kShortChunks, DEV>(p, stream);
    return launch_ch<O, RB, GB, VNZ, kTinyChunks, DEV>(p, stream);
}

// Dispatch over the correction width and the gradient type, for one
// optimizer (and, for AdamW, v floor and counter source).
template <Opt O, bool VNZ, bool DEV>
cudaError_t launch_widths(int rho_bits, int grad_bits, const StepParams &p, cudaStream_t stream)
{
    if (grad_bits == 32)
        return rho_bits == 8 ? launch<O, 8, 32, VNZ, DEV>(p, stream) : launch<O, 16, 32, VNZ, DEV>(p, stream);
    return rho_bits == 8 ? launch<O, 8, 16, VNZ, DEV>(p, stream) : launch<O, 16, 16, VNZ, DEV>(p, stream);
}

}  // namespace

// One translation unit per group of instantiations (they compile in parallel).
cudaError_t launch_step_adamw(int rho_bits, int grad_bits, const StepParams &p, cudaStream_t stream);
cudaError_t launch_step_adamw_dev(int rho_bits, int grad_bits, const StepParams &p, cudaStream_t stream);
cudaError_t launch_step_sgd(int rho_bits, int grad_bits, const StepParams &p, cudaStream_t stream);
cudaError_t launch_step_lion(int rho_bits, int grad_bits, const StepParams &p, cudaStream_t stream);

}  // namespace fo
