// fo_device.cuh -- device-side number primitives of the fused compressed
// optimizer step ("FlashOptim: Optimizers for Memory Efficient Training").
//
// Every function here is exact IEEE binary32 arithmetic (round to nearest
// even, no flush to zero, no contraction: the library is built with
// -fmad=false and spells each operation as an intrinsic), so that the GPU
// path reproduces the arithmetic contract in include/fo.h bit for bit.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fo_internal.h"

namespace fo {

// x + 1.5*2^23 rounds x to an integer (ties to even) for |x| < 2^22, and the
// low bits of the sum's pattern hold that integer in two's complement.
constexpr float kRoundMagic = 12582912.0f;
constexpr uint32_t kRoundMagicBits = 0x4B400000u;

// 1/Q rounded to FP32 (Q = 127 and 32767), and Q * 2^-15 (exact).
constexpr float kKappa8 = 0x1.020408p-7f;
constexpr float kKappa16 = 0x1.0002p-15f;
constexpr float kQScale8 = 0x1.fcp-9f;       // 127 / 32768
constexpr float kQScale16 = 0x1.fffcp-1f;    // 32767 / 32768
constexpr float kTwoPowMinus134 = 0x1p-134f; // h of a zero theta'
constexpr float kRcp127 = 0x1.020408p-7f;    // RN(1/127)
constexpr float kRcp255 = 0x1.010102p-8f;    // RN(1/255)

template <int RB> struct RhoConst;
template <> struct RhoConst<8> {
    static constexpr float kappa = kKappa8;
    static constexpr float qscale = kQScale8;
    // kRoundMagic * qscale, exact: the offset that fma(M + k, qscale, -offset) removes
    static constexpr float offset = 48768.0f;        // 384 * 127
};
template <> struct RhoConst<16> {
    static constexpr float kappa = kKappa16;
    static constexpr float qscale = kQScale16;
    static constexpr float offset = 12582528.0f;     // 384 * 32767
};

// ---------------------------------------------------------------------------
// Unpacking of stored codes
// ---------------------------------------------------------------------------

// Unsigned byte j of w as a float: 2^23 + byte is exact, then subtract 2^23.
template <int J>
__device__ __forceinline__ float u8_at(uint32_t w)
{
    return __fsub_rn(__uint_as_float(__byte_perm(w, 0x4B000000u, 0x7440u | J)), 8388608.0f);
}

// Signed byte j of w, given wx = w ^ 0x80808080 (bytes biased by 128).
template <int J>
__device__ __forceinline__ float s8_at(uint32_t wx)
{
    return __fsub_rn(__uint_as_float(__byte_perm(wx, 0x4B000000u, 0x7440u | J)), 8388736.0f);
}

// Signed 16-bit half j of w, given wx = w ^ 0x80008000.
template <int J>
__device__ __forceinline__ float s16_at(uint32_t wx)
{
    constexpr uint32_t sel = 0x7400u | ((2u * J + 1u) << 4) | (2u * J);
    return __fsub_rn(__uint_as_float(__byte_perm(wx, 0x4B000000u, sel)), 8421376.0f);
}

// The two BF16 values of a 32-bit word as FP32 bit patterns (low half first).
__device__ __forceinline__ uint32_t bf16_lo_bits(uint32_t w) { return w << 16; }
__device__ __forceinline__ uint32_t bf16_hi_bits(uint32_t w) { return w & 0xFFFF0000u; }

// ---------------------------------------------------------------------------
// Packing of results
// ---------------------------------------------------------------------------

// Round two floats to BF16 (nearest even) and pack: lo in bits 0-15, hi in 16-31.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// Four rounded-code patterns (low byte = code) -> one word of bytes.
__device__ __forceinline__ uint32_t pack_bytes(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3)
{
    uint32_t lo = __byte_perm(c0, c1, 0x0040u);
    uint32_t hi = __byte_perm(c2, c3, 0x0040u);
    return __byte_perm(lo, hi, 0x5410u);
}

// Two rounded-code patterns (low half = code) -> one word of 16-bit halves.
__device__ __forceinline__ uint32_t pack_halves(uint32_t c0, uint32_t c1)
{
    return __byte_perm(c0, c1, 0x5410u);
}

// rint(x) for |x| < 2^22, as the pattern whose low bits hold the integer.
__device__ __forceinline__ uint32_t round_code(float x)
{
    return __float_as_uint(__fadd_rn(x, kRoundMagic));
}

// ---------------------------------------------------------------------------
// Weight splitting (Eq. 1-2)
// ---------------------------------------------------------------------------

// theta^ = theta' + (rho * kappa) * h, h = ULP(theta')/2 on the side of rho's sign.
//
// For theta' != 0 the FP32 values within h of theta' on either side are
// evenly spaced by h * 2^-15 (the FP32 spacing of theta's binade; just below
// a power of two both the FP32 and the BF16 spacings halve), and their bit
// patterns step by one. So rounding theta' + t*h to FP32 moves the magnitude
// pattern of theta' by rint(t * 2^15) (ties to even, as theta' has an even
// pattern). For theta' = +-0, h = 2^-134 and the result is t * 2^-134.
template <int RB>
__device__ __forceinline__ float merge_one(uint32_t tp_bits, float rho_f)
{
    const float t = __fmul_rn(rho_f, RhoConst<RB>::kappa);
    const float nb = __fmaf_rn(t, 32768.0f, kRoundMagic);           // t*2^15 is exact
    const int n = (int)(__float_as_uint(nb) - kRoundMagicBits);
    const int s = (int)tp_bits >> 31;                                // -1 if theta' < 0
    const uint32_t bits = tp_bits + (uint32_t)((n ^ s) - s);
    const float zero_case = __fmul_rn(t, kTwoPowMinus134);
    return __uint_as_float(tp_bits) == 0.0f ? zero_case : __uint_as_float(bits);
}

// rho code pattern for theta given its BF16 rounding theta' (as FP32 bits).
//
// theta and theta' share the sign bit, and theta' is theta's pattern rounded
// to a multiple of 2^16, so k = pattern(theta) - pattern(theta') counts FP32
// steps of h * 2^-15 from theta' toward larger magnitude: the normalised error
// is e = sign(theta) * k * 2^-15 exactly (|k| <= 2^15). Then rho = rint(RN(e*Q)),
// with e*Q evaluated as one FP32 product.
template <int RB>
__device__ __forceinline__ uint32_t split_code(uint32_t theta_bits, uint32_t tp_bits)
{
    const int k = (int)(theta_bits - tp_bits);
    const int s = (int)theta_bits >> 31;
    const int ks = (k ^ s) - s;
    // fma((2^23*1.5 + ks), Q*2^-15, -(2^23*1.5)*Q*2^-15) = RN(ks * Q * 2^-15) exactly
    const float x = __fmaf_rn(__uint_as_float(kRoundMagicBits + (uint32_t)ks), RhoConst<RB>::qscale,
                              -RhoConst<RB>::offset);
    return round_code(x);
}

// ---------------------------------------------------------------------------
// Companding (Algorithms 2-3)
// ---------------------------------------------------------------------------

__device__ __forceinline__ float phi_m(float x)
{
    return __fdiv_rn(__fadd_rn(x, x), __fadd_rn(1.0f, fabsf(x)));
}

__device__ __forceinline__ float phi_m_inv(float z)
{
    return __fdiv_rn(z, __fsub_rn(2.0f, fabsf(z)));
}

// FP16 group scale of an absmax a (round to nearest even, capped at 65504).
__device__ __forceinline__ uint16_t scale_of(float a)
{
    return __half_as_ushort(__float2half_rn(fminf(a, 65504.0f)));
}

__device__ __forceinline__ float scale_value(uint16_t s)
{
    return __half2float(__ushort_as_half(s));
}

// Multiplier taking a companded value to code units: L / s, or 0 when s = 0
// (then every code is 0).
__device__ __forceinline__ float code_multiplier(float s, float levels)
{
    return s > 0.0f ? __fdiv_rn(levels, s) : 0.0f;
}

// Momentum code pattern: clamp(rint(z * mult), -127, 127).
__device__ __forceinline__ uint32_t m_code_of(float x)
{
    return round_code(fminf(fmaxf(x, -127.0f), 127.0f));
}
__device__ __forceinline__ uint32_t m_code(float z, float mult) { return m_code_of(__fmul_rn(z, mult)); }

// Second-moment code pattern: min(rint(r * mult), 255), r >= 0.
__device__ __forceinline__ uint32_t v_code_of(float x)
{
    return round_code(fminf(x, 255.0f));
}
__device__ __forceinline__ uint32_t v_code(float r, float mult) { return v_code_of(__fmul_rn(r, mult)); }
// The same with the opt-in rule: no code 0 in a group whose scale is non-zero
// (mult > 0); a zero scale keeps codes 0.
__device__ __forceinline__ uint32_t v_code_nonzero(float r, float mult)
{
    return v_code_of(fmaxf(__fmul_rn(r, mult), mult > 0.0f ? 1.0f : 0.0f));
}

// The same codes through the saturating round-to-nearest-even conversion
// (one conversion-unit instruction instead of min/max and an add); the low
// byte of the result equals that of m_code_of / v_code_of for every input.
#ifndef FO_CODE_CVT
#define FO_CODE_CVT 1
#endif
__device__ __forceinline__ uint32_t m_code_sat(float x)
{
#if FO_CODE_CVT
    uint32_t c;
    asm("cvt.rni.sat.s8.f32 %0, %1;" : "=r"(c) : "f"(fmaxf(x, -127.0f)));
    return c;
#else
    return m_code_of(x);
#endif
}
__device__ __forceinline__ uint32_t v_code_sat(float x)
{
#if FO_CODE_CVT
    uint32_t c;
    asm("cvt.rni.sat.u8.f32 %0, %1;" : "=r"(c) : "f"(x));
    return c;
#else
    return v_code_of(x);
#endif
}

// ---------------------------------------------------------------------------
// Streaming global memory access (touched once: evict-first)
// ---------------------------------------------------------------------------

#ifndef FO_CACHE_HINT
#define FO_CACHE_HINT 0
#endif
__device__ __forceinline__ uint4 ld_stream(const void *p)
{
#if FO_CACHE_HINT == 0
    return __ldcs(reinterpret_cast<const uint4 *>(p));
#elif FO_CACHE_HINT == 1
    return *reinterpret_cast<const uint4 *>(p);
#else
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
#endif
}

__device__ __forceinline__ void st_stream(void *p, uint4 v)
{
#if FO_CACHE_HINT == 0
    __stcs(reinterpret_cast<uint4 *>(p), v);
#else
    *reinterpret_cast<uint4 *>(p) = v;
#endif
}

}  // namespace fo
