// fo_verify.cu -- on-device enumeration of the fast path's hardware-dependent
// arithmetic (fo_verify_fast_arithmetic).
//
// The fused step ("FlashOptim", section "融合优化器步骤") must leave exactly
// the state that the arithmetic contract's IEEE operations give. Its packed
// fast path builds division and square root from the GPU's reciprocal and
// reciprocal-square-root approximations, whose exact outputs the instruction
// set does not fix. Each sequence is exact on a one-variable or finite operand
// domain when the approximation behaves as on the GPU where the domain was
// first enumerated; these kernels enumerate every such domain again on the
// device at hand, calling the very functions the step kernel inlines, and
// count the operands whose result differs from the IEEE operation.
#include "fo_step.cuh"

namespace fo {
namespace {

enum Check : int {
    kRecip = 0,      // rcp2_rn(b) = RN(1/b), b in [2^-100, 2^100]
    kSqrt = 1,       // neg_sqrt2(-v) = -RN(sqrt(v)), v in [2^-100, 2^126]
    kPhiAdamW = 2,   // phi_m_pair<2>: m' / RN(2^-33 |m'| + 1/2), |m'| in [2^-62, 2^85]
    kPhiOther = 3,   // phi_m_pair<1>: m / RN(|m|/2 + 1/2), |m| in [2^-100, 2^100]
    kDequant = 4,    // mhat_pair: every code byte under every scale 0x0000-0x3FEF
    kScale = 5,      // 127/s, 255/s (short division) and s/127, s/255, every positive finite FP16 s
};

__device__ __forceinline__ uint32_t same(float got, float want) { return __float_as_uint(got) == __float_as_uint(want); }

// mismatches among the element with FP32 pattern `bits` (and, where the
// domain is signed, its negation) for check C
template <int C>
__device__ __forceinline__ uint32_t mismatches(uint32_t bits)
{
    const float x = __uint_as_float(bits);
    if (C == kRecip) {
        float y, y_;
        unpk(rcp2_rn(splat(-x)), y, y_);
        return !same(y, __frcp_rn(x));
    } else if (C == kSqrt) {
        float r, r_;
        unpk(neg_sqrt2(splat(-x)), r, r_);
        return !same(r, -__fsqrt_rn(x));
    } else if (C == kPhiAdamW || C == kPhiOther) {
        const float half = C == kPhiAdamW ? 0x1p-33f : 0.5f;
        const float d = __fmaf_rn(half, x, 0.5f);
        float z0, z1;
        unpk(phi_m_pair<C == kPhiAdamW ? 2 : 1>(pk(x, -x)), z0, z1);
        return !same(z0, __fdiv_rn(x, d)) + !same(z1, __fdiv_rn(-x, d));
    } else if (C == kDequant) {
        // bits: scale pattern * 64 + w; the word holds the biased code bytes
        // 4w .. 4w+3 (code q = byte - 128), as thread_step forms them
        const uint32_t sb = bits >> 6, w = bits & 63u;
        const uint32_t word = (4u * w) | (4u * w + 1u) << 8 | (4u * w + 2u) << 16 | (4u * w + 3u) << 24;
        const uint32_t mx[4] = {word, 0u, 0u, 0u};
        PairConsts k;
        k.cm = splat(div_by_const(scale_value((uint16_t)sb), -127.0f, kRcp127));
        k.cv = k.ncv23 = k.coef = 0;
        float got[4];
        unpk(mhat_pair<0>(mx, k), got[0], got[1]);
        unpk(mhat_pair<1>(mx, k), got[2], got[3]);
        const float cm = __fdiv_rn(scale_value((uint16_t)sb), 127.0f);
        uint32_t bad = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float zq = __fmul_rn((float)((int)(4u * w) + j - 128), cm);
            const float want = __fdiv_rn(zq, __fsub_rn(2.0f, fabsf(zq)));
            // a zero z decodes to a zero of either sign on the fast path (the
            // remainder step adds +0); the step uses the value only
            bad += zq == 0.0f ? !(got[j] == 0.0f) : !same(got[j], want);
        }
        return bad;
    } else {
        const float s = scale_value((uint16_t)bits);
        return !same(div1_short(127.0f, s), __fdiv_rn(127.0f, s)) +
               !same(div1_short(255.0f, s), __fdiv_rn(255.0f, s)) +
               !same(div_by_const(s, -127.0f, kRcp127), __fdiv_rn(s, 127.0f)) +
               !same(div_by_const(s, -255.0f, kRcp255), __fdiv_rn(s, 255.0f));
    }
}

// Patterns lo .. lo+n-1, grid-stride; one atomic per block that saw a mismatch.
template <int C>
__global__ void __launch_bounds__(256) verify_kernel(uint32_t lo, uint32_t n, unsigned long long *count)
{
    uint32_t bad = 0;
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
        bad += mismatches<C>(lo + i);
    if (C == kSqrt && blockIdx.x == 0 && threadIdx.x == 0) {
        float r, r_;
        unpk(neg_sqrt2(splat(-0.0f)), r, r_);
        bad += __float_as_uint(r) != 0u;   // v = 0 gives +0
    }
    bad = __reduce_add_sync(0xFFFFFFFFu, bad);
    if ((threadIdx.x & 31) == 0 && bad)
        atomicAdd(count, (unsigned long long)bad);
}

template <int C>
cudaError_t run(uint32_t lo, uint32_t hi_inclusive, unsigned long long *counts, cudaStream_t stream)
{
    verify_kernel<C><<<sm_count() * 8, 256, 0, stream>>>(lo, hi_inclusive - lo + 1u, counts + C);
    count_launch();
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_verify(unsigned long long *counts, cudaStream_t stream)
{
    cudaError_t e = cudaMemsetAsync(counts, 0, kVerifyCounts * sizeof(unsigned long long), stream);
    if (e == cudaSuccess)
        e = run<kRecip>(0x0D800000u, 0x71800000u, counts, stream);      // 2^-100 .. 2^100
    if (e == cudaSuccess)
        e = run<kSqrt>(0x0D800000u, 0x7E800000u, counts, stream);       // 2^-100 .. 2^126
    if (e == cudaSuccess)
        e = run<kPhiAdamW>(0x20800000u, 0x6A000000u, counts, stream);   // 2^-62 .. 2^85
    if (e == cudaSuccess)
        e = run<kPhiOther>(0x0D800000u, 0x71800000u, counts, stream);   // 2^-100 .. 2^100
    if (e == cudaSuccess)
        e = run<kDequant>(0u, 0x3FF0u * 64u - 1u, counts, stream);
    if (e == cudaSuccess)
        e = run<kScale>(1u, 0x7BFFu, counts, stream);
    return e;
}

}  // namespace fo
