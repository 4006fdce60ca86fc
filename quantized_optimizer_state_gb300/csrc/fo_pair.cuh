// fo_pair.cuh -- packed two-lane FP32 arithmetic for the fused step's fast
// path (sm_103a add/sub/mul/fma.rn.f32x2: two IEEE round-to-nearest results
// per instruction, bit-identical to the scalar operations), and correctly
// rounded division and square root built from the hardware approximations.
//
// Division (RN(a/b), b > 0): one Newton step on the hardware reciprocal
// approximation y0 of 1/b, y1 = y0 + y0*(1 - b*y0), gives the correctly
// rounded reciprocal RN(1/b); then q0 = RN(a*y1) is within one ulp of a/b,
// the remainder r = a - b*q0 is exact, and RN(q0 + r*y1) = RN(a/b)
// (P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990; see also Muller et
// al., "Handbook of Floating-Point Arithmetic", ch. on FMA-based division).
// Square root (RN(sqrt(v))): s = v*y and h = y/2 from the hardware
// reciprocal-square-root approximation y, the exact remainder d = v - s*s
// and RN(s + d*h) (the same remainder correction, for square roots).
//
// Short division (div2_short, div1_short): the same correction on the
// unrefined approximation y0, RN(q0 + r*y0) with q0 = RN(a*y0). y0 is not
// always RN(1/b) (on GB300 it differs for 13 % of the FP32 values of b in
// [2^-100, 2^100]), and over all 2^46 pairs of significands this sequence
// misses RN(a/b) 79,381 times there, so it
// serves only domains on which it was enumerated exhaustively and found equal
// to the IEEE division: phi_m's divisions (every m in the fast path's range),
// the momentum dequantization (every code byte under every fast-path scale)
// and the code multipliers 127/s and 255/s (every positive finite FP16 s).
//
// Validity: the hardware approximations are facts of the GPU, not of the
// instruction set, so fo_verify_fast_arithmetic (fo_verify.cu) re-enumerates,
// on the device at hand, every one-variable or finite domain the fast path
// relies on: the refined reciprocal equal to RN(1/b) for every b in
// [2^-100, 2^100] (the premise of Markstein's theorem for div2), the short
// division on the domains above, and the square root for every v in
// [2^-100, 2^126] and v = 0. The sequences are used only where the operands
// are inside the ranges listed at each function; callers check the ranges
// and recompute elsewhere with the IEEE operations.
#pragma once

#include <cstdint>

namespace fo {

typedef unsigned long long f2;  // two FP32 lanes in one 64-bit register pair

__device__ __forceinline__ f2 pk(float lo, float hi)
{
    f2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void unpk(f2 v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ f2 add2(f2 a, f2 b)
{
    f2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ f2 mul2(f2 a, f2 b)
{
    f2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c)
{
    f2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ f2 splat(float x) { return pk(x, x); }

// max(a, b, c) with NaN propagated (a NaN operand gives NaN), in one instruction.
__device__ __forceinline__ float max3_nan(float a, float b, float c)
{
    float d;
    asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ float rcp_approx(float x)
{
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float rsqrt_approx(float x)
{
    float y;
    asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// RN(1/b) in both lanes, given nb = -b with b in [2^-100, 2^100]: one
// Newton step y0 + y0*(1 - b*y0) on the hardware approximation y0
// (enumerated over that whole range).
__device__ __forceinline__ f2 rcp2_rn(f2 nb)
{
    float n0, n1;
    unpk(nb, n0, n1);
    const f2 y0 = pk(rcp_approx(-n0), rcp_approx(-n1));
    const f2 e = fma2(nb, y0, splat(1.0f));  // 1 - b*y0
    return fma2(y0, e, y0);
}

// RN(a / b) in both lanes, given nb = -b. Valid when b is in [2^-100, 2^100],
// a is +0 or has |a| >= 2^-100, and the quotient is in [2^-100, 2^100] or 0
// (Markstein's theorem, given the correctly rounded reciprocal).
__device__ __forceinline__ f2 div2(f2 a, f2 nb)
{
    const f2 y1 = rcp2_rn(nb);                // RN(1/b)
    const f2 q0 = mul2(a, y1);
    const f2 r = fma2(nb, q0, a);             // a - b*q0, exact
    return fma2(r, y1, q0);
}

// -RN(sqrt(v)) in both lanes, given nv = -v with v in [2^-100, 2^126]:
// s = v*y and h = y/2 from the hardware reciprocal square root y, then the
// exact remainder d = v - s*s and RN(s + d*h) (enumerated equal to the IEEE
// square root over that whole range). Also v = +0 (nv = -0), for which the
// result is +0: the approximation reads v + 2^-126, which is v itself for
// every v >= 2^-100 (2^-126 is below half an ulp there) and a normal number
// for v = 0, so that y stays finite and s = -0 * y, d and the result are
// zeros.
__device__ __forceinline__ f2 neg_sqrt2(f2 nv)
{
    float v0, v1;
    unpk(add2(nv, splat(-0x1p-126f)), v0, v1);
    const f2 y = pk(rsqrt_approx(-v0), rsqrt_approx(-v1));
    const f2 ns = mul2(nv, y);                // -s
    const f2 h = mul2(splat(0.5f), y);
    const f2 d = fma2(ns, ns, nv);            // s*s - v = -(v - s*s), exact
    return fma2(d, h, ns);                    // -(s + (v - s*s)*h)
}

// RN(a / b) in both lanes, given nb = -b, by the short sequence (no
// refinement of the reciprocal approximation). Exact only on the enumerated
// domains listed at the top of this file; for a = -0 it returns +0 (as div2
// does), where callers rely on the value only.
__device__ __forceinline__ f2 div2_short(f2 a, f2 nb)
{
    float n0, n1;
    unpk(nb, n0, n1);
    const f2 y0 = pk(rcp_approx(-n0), rcp_approx(-n1));
    const f2 q0 = mul2(a, y0);
    const f2 r = fma2(nb, q0, a);             // a - b*q0, exact
    return fma2(r, y0, q0);
}

// RN(a / s) by the short sequence, for a = 127 or 255 and s a positive
// finite FP16 value (enumerated).
__device__ __forceinline__ float div1_short(float a, float s)
{
    const float y0 = rcp_approx(s);
    const float q0 = __fmul_rn(a, y0);
    const float r = __fmaf_rn(-s, q0, a);
    return __fmaf_rn(r, y0, q0);
}

// RN(a / b) for a constant b with its correctly rounded reciprocal y = RN(1/b)
// (Markstein's correction step only), valid for a = 0 or |a/b| in
// [2^-100, 2^100] with a normal.
__device__ __forceinline__ float div_by_const(float a, float nb, float y)
{
    const float q0 = __fmul_rn(a, y);
    const float r = __fmaf_rn(nb, q0, a);   // a - b*q0, exact
    return __fmaf_rn(r, y, q0);
}


}  // namespace fo
