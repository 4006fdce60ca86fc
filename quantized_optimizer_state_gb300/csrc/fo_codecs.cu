// fo_codecs.cu -- stand-alone codecs of "FlashOptim: Optimizers for Memory
// Efficient Training": weight splitting and merging (section "权重复分裂",
// Eq. 1-2) and companded group quantization of the optimizer state (section
// "带压缩扩展的优化器状态量化", Algorithms 2-3). They initialise and export
// the compressed state; the fused step (fo_step.cu) uses the same primitives.
//
// A thread owns 16 contiguous elements; a 32-element group is a pair of
// adjacent lanes. Grid-stride loops run the same number of iterations in
// every thread so that the pair shuffle always has both lanes present.
#include "fo_device.cuh"
#include "fo_internal.h"
#include "fo_pair.cuh"

namespace fo {
namespace {

constexpr int kThreads = 256;
constexpr int kEPT = kElemsPerThread;

struct Chunking {
    int64_t nchunks;  // 16-element chunks
    int64_t stride;   // threads in the grid
    int64_t iters;    // loop trips, the same in every thread
};

Chunking plan(int64_t n, int *grid)
{
    Chunking c;
    c.nchunks = (n + kEPT - 1) / kEPT;
    const int64_t blocks_needed = (c.nchunks + kThreads - 1) / kThreads;
    const int64_t cap = (int64_t)sm_count() * 8;
    *grid = (int)(blocks_needed < cap ? blocks_needed : cap);
    c.stride = (int64_t)(*grid) * kThreads;
    c.iters = (c.nchunks + c.stride - 1) / c.stride;
    return c;
}

__device__ __forceinline__ int valid_count(int64_t i0, int64_t n)
{
    const int64_t rem = n - i0;
    return rem >= kEPT ? kEPT : (rem > 0 ? (int)rem : 0);
}

template <int RB>
__global__ void __launch_bounds__(kThreads) split_kernel(const float *__restrict__ theta,
                                                         uint16_t *__restrict__ tp, void *__restrict__ rho,
                                                         int64_t n, Chunking ck)
{
    for (int64_t it = 0; it < ck.iters; ++it) {
        const int64_t c = (int64_t)blockIdx.x * kThreads + threadIdx.x + it * ck.stride;
        const int64_t i0 = c * kEPT;
        const int cnt = valid_count(i0, n);
        if (cnt == 0)
            continue;
        float x[kEPT];
        if (cnt == kEPT) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint4 a = ld_stream(theta + i0 + 4 * q);
                x[4 * q] = __uint_as_float(a.x); x[4 * q + 1] = __uint_as_float(a.y);
                x[4 * q + 2] = __uint_as_float(a.z); x[4 * q + 3] = __uint_as_float(a.w);
            }
        } else {
#pragma unroll
            for (int j = 0; j < kEPT; ++j)
                x[j] = j < cnt ? theta[i0 + j] : 0.0f;
        }
        uint32_t tw[8], cw[kEPT];
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            tw[w] = pack_bf16x2(x[2 * w], x[2 * w + 1]);
            cw[2 * w] = split_code<RB>(__float_as_uint(x[2 * w]), bf16_lo_bits(tw[w]));
            cw[2 * w + 1] = split_code<RB>(__float_as_uint(x[2 * w + 1]), bf16_hi_bits(tw[w]));
        }
        if (cnt == kEPT) {
            st_stream(tp + i0, make_uint4(tw[0], tw[1], tw[2], tw[3]));
            st_stream(tp + i0 + 8, make_uint4(tw[4], tw[5], tw[6], tw[7]));
            if (RB == 8) {
                uint32_t o[4];
#pragma unroll
                for (int w = 0; w < 4; ++w)
                    o[w] = pack_bytes(cw[4 * w], cw[4 * w + 1], cw[4 * w + 2], cw[4 * w + 3]);
                st_stream(static_cast<int8_t *>(rho) + i0, make_uint4(o[0], o[1], o[2], o[3]));
            } else {
                uint32_t o[8];
#pragma unroll
                for (int w = 0; w < 8; ++w)
                    o[w] = pack_halves(cw[2 * w], cw[2 * w + 1]);
                st_stream(static_cast<int16_t *>(rho) + i0, make_uint4(o[0], o[1], o[2], o[3]));
                st_stream(static_cast<int16_t *>(rho) + i0 + 8, make_uint4(o[4], o[5], o[6], o[7]));
            }
        } else {
#pragma unroll
            for (int j = 0; j < kEPT; ++j) {
                if (j < cnt) {
                    tp[i0 + j] = (uint16_t)(tw[j >> 1] >> (16 * (j & 1)));
                    if (RB == 8)
                        static_cast<int8_t *>(rho)[i0 + j] = (int8_t)cw[j];
                    else
                        static_cast<int16_t *>(rho)[i0 + j] = (int16_t)cw[j];
                }
            }
        }
    }
}

template <int RB>
__global__ void __launch_bounds__(kThreads) merge_kernel(const uint16_t *__restrict__ tp,
                                                         const void *__restrict__ rho,
                                                         float *__restrict__ theta, int64_t n, Chunking ck)
{
    for (int64_t it = 0; it < ck.iters; ++it) {
        const int64_t c = (int64_t)blockIdx.x * kThreads + threadIdx.x + it * ck.stride;
        const int64_t i0 = c * kEPT;
        const int cnt = valid_count(i0, n);
        if (cnt == 0)
            continue;
        uint32_t tw[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        int32_t rv[kEPT];
        if (cnt == kEPT) {
            uint4 a = ld_stream(tp + i0), b = ld_stream(tp + i0 + 8);
            tw[0] = a.x; tw[1] = a.y; tw[2] = a.z; tw[3] = a.w;
            tw[4] = b.x; tw[5] = b.y; tw[6] = b.z; tw[7] = b.w;
        } else {
#pragma unroll
            for (int j = 0; j < kEPT; ++j)
                if (j < cnt)
                    tw[j >> 1] |= (uint32_t)tp[i0 + j] << (16 * (j & 1));
        }
        if (cnt == kEPT) {
            // one 16-byte load of 8-bit rho (two of 16-bit), unpacked with sign extension
            uint32_t rw[8];
            if (RB == 8) {
                const uint4 a = ld_stream(static_cast<const int8_t *>(rho) + i0);
                rw[0] = a.x; rw[1] = a.y; rw[2] = a.z; rw[3] = a.w;
#pragma unroll
                for (int j = 0; j < kEPT; ++j)
                    rv[j] = (int32_t)(int8_t)(rw[j >> 2] >> (8 * (j & 3)));
            } else {
                const uint4 a = ld_stream(static_cast<const int16_t *>(rho) + i0);
                const uint4 b = ld_stream(static_cast<const int16_t *>(rho) + i0 + 8);
                rw[0] = a.x; rw[1] = a.y; rw[2] = a.z; rw[3] = a.w;
                rw[4] = b.x; rw[5] = b.y; rw[6] = b.z; rw[7] = b.w;
#pragma unroll
                for (int j = 0; j < kEPT; ++j)
                    rv[j] = (int32_t)(int16_t)(rw[j >> 1] >> (16 * (j & 1)));
            }
        } else {
#pragma unroll
            for (int j = 0; j < kEPT; ++j) {
                if (RB == 8)
                    rv[j] = j < cnt ? static_cast<const int8_t *>(rho)[i0 + j] : 0;
                else
                    rv[j] = j < cnt ? static_cast<const int16_t *>(rho)[i0 + j] : 0;
            }
        }
        float x[kEPT];
#pragma unroll
        for (int j = 0; j < kEPT; ++j) {
            const uint32_t bits = (j & 1) ? bf16_hi_bits(tw[j >> 1]) : bf16_lo_bits(tw[j >> 1]);
            x[j] = merge_one<RB>(bits, (float)rv[j]);
        }
        if (cnt == kEPT) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
                st_stream(theta + i0 + 4 * q,
                          make_uint4(__float_as_uint(x[4 * q]), __float_as_uint(x[4 * q + 1]),
                                     __float_as_uint(x[4 * q + 2]), __float_as_uint(x[4 * q + 3])));
        } else {
#pragma unroll
            for (int j = 0; j < kEPT; ++j)
                if (j < cnt)
                    theta[i0 + j] = x[j];
        }
    }
}

// kind 0: momentum (INT8, phi_m); kind 1: second moment (UINT8, phi_v);
// kinds 2 and 3: the same group quantization without companding (phi the
// identity), the linear quantizer the page compares against in Fig. 4;
// kind 5: kind 1 with no code 0 in a group whose scale is non-zero.
template <int Kind>
struct KindTraits {
    static constexpr bool kSigned = (Kind & 1) == 0;
    static constexpr bool kCompanded = Kind != 2 && Kind != 3;
    static constexpr bool kNonzero = Kind == 5;
    static constexpr float kLevels = kSigned ? 127.0f : 255.0f;
};

template <int Kind>
__device__ __forceinline__ float compand(float x)
{
    if (!KindTraits<Kind>::kCompanded)
        return x;
    return KindTraits<Kind>::kSigned ? phi_m(x) : __fsqrt_rn(x);
}

template <int Kind>
__device__ __forceinline__ float expand(float d)
{
    if (!KindTraits<Kind>::kCompanded)
        return d;
    return KindTraits<Kind>::kSigned ? phi_m_inv(d) : __fmul_rn(d, d);
}

// phi_m^-1(z) = z / (2 - |z|) for |z| < 2: the divisor lies in [2^-23, 2]
// and the quotient is 0 or at least 2^-33 in magnitude (|z| >= 2^-24/127),
// inside the validated range of div1 (the correctly rounded division of
// fo_pair.cuh)
__device__ __forceinline__ float phi_m_inv_fast(float z)
{
    return div1(z, __fsub_rn(2.0f, fabsf(z)));
}

template <int Kind>
__global__ void __launch_bounds__(kThreads) quant_kernel(const float *__restrict__ xin, void *__restrict__ q,
                                                         uint16_t *__restrict__ scales, int64_t n, Chunking ck)
{
    for (int64_t it = 0; it < ck.iters; ++it) {
        const int64_t c = (int64_t)blockIdx.x * kThreads + threadIdx.x + it * ck.stride;
        const int64_t i0 = c * kEPT;
        const int cnt = valid_count(i0, n);
        float y[kEPT];
        if (cnt == kEPT) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint4 a = ld_stream(xin + i0 + 4 * k);
                y[4 * k] = __uint_as_float(a.x); y[4 * k + 1] = __uint_as_float(a.y);
                y[4 * k + 2] = __uint_as_float(a.z); y[4 * k + 3] = __uint_as_float(a.w);
            }
        } else {
#pragma unroll
            for (int j = 0; j < kEPT; ++j)
                y[j] = j < cnt ? xin[i0 + j] : 0.0f;
        }
        float a = 0.0f;
#pragma unroll
        for (int j = 0; j < kEPT; ++j) {
            y[j] = compand<Kind>(y[j]);
            if (j < cnt)
                a = fmaxf(a, fabsf(y[j]));
        }
        a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
        const uint16_t s = scale_of(a);
        const float mult = code_multiplier(scale_value(s), KindTraits<Kind>::kLevels);
        uint32_t cw[kEPT];
#pragma unroll
        for (int j = 0; j < kEPT; ++j)
            cw[j] = KindTraits<Kind>::kSigned ? m_code(y[j], mult)
                    : KindTraits<Kind>::kNonzero ? v_code_nonzero(y[j], mult)
                                                 : v_code(y[j], mult);
        if (cnt == kEPT) {
            uint32_t o[4];
#pragma unroll
            for (int w = 0; w < 4; ++w)
                o[w] = pack_bytes(cw[4 * w], cw[4 * w + 1], cw[4 * w + 2], cw[4 * w + 3]);
            st_stream(static_cast<uint8_t *>(q) + i0, make_uint4(o[0], o[1], o[2], o[3]));
        } else {
#pragma unroll
            for (int j = 0; j < kEPT; ++j)
                if (j < cnt)
                    static_cast<uint8_t *>(q)[i0 + j] = (uint8_t)cw[j];
        }
        if ((threadIdx.x & 1) == 0 && cnt > 0)
            scales[i0 >> 5] = s;
    }
}

template <int Kind>
__global__ void __launch_bounds__(kThreads) dequant_kernel(const void *__restrict__ q,
                                                           const uint16_t *__restrict__ scales,
                                                           float *__restrict__ xout, int64_t n, Chunking ck)
{
    for (int64_t it = 0; it < ck.iters; ++it) {
        const int64_t c = (int64_t)blockIdx.x * kThreads + threadIdx.x + it * ck.stride;
        const int64_t i0 = c * kEPT;
        const int cnt = valid_count(i0, n);
        if (cnt == 0)
            continue;
        uint32_t w[4] = {0, 0, 0, 0};
        if (cnt == kEPT) {
            const uint4 a = ld_stream(static_cast<const uint8_t *>(q) + i0);
            w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
        } else {
#pragma unroll
            for (int j = 0; j < kEPT; ++j)
                if (j < cnt)
                    w[j >> 2] |= (uint32_t)static_cast<const uint8_t *>(q)[i0 + j] << (8 * (j & 3));
        }
        const uint16_t sbits = scales[i0 >> 5];
        const float step = __fdiv_rn(scale_value(sbits), KindTraits<Kind>::kLevels);
        // 0 < s < 1.984375 (FP16 0x0001..0x3FEF): |z| <= 128 * s/127 < 2 for
        // every byte, -128 included, and z = code * step is never -0 (the fast
        // division would return +0 for it where IEEE division keeps -0)
        const bool small_scale = (uint32_t)sbits - 1u < 0x3FEFu;
        float x[kEPT];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t wx = KindTraits<Kind>::kSigned ? (w[k] ^ 0x80808080u) : w[k];
            float c0, c1, c2, c3;
            if (KindTraits<Kind>::kSigned) {
                c0 = s8_at<0>(wx); c1 = s8_at<1>(wx); c2 = s8_at<2>(wx); c3 = s8_at<3>(wx);
            } else {
                c0 = u8_at<0>(wx); c1 = u8_at<1>(wx); c2 = u8_at<2>(wx); c3 = u8_at<3>(wx);
            }
            const float cc[4] = {c0, c1, c2, c3};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float d = __fmul_rn(cc[e], step);
                x[4 * k + e] = (Kind == 0 && small_scale) ? phi_m_inv_fast(d) : expand<Kind>(d);
            }
        }
        if (cnt == kEPT) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
                st_stream(xout + i0 + 4 * k,
                          make_uint4(__float_as_uint(x[4 * k]), __float_as_uint(x[4 * k + 1]),
                                     __float_as_uint(x[4 * k + 2]), __float_as_uint(x[4 * k + 3])));
        } else {
#pragma unroll
            for (int j = 0; j < kEPT; ++j)
                if (j < cnt)
                    xout[i0 + j] = x[j];
        }
    }
}

}  // namespace

cudaError_t launch_split(const float *theta, uint16_t *tp, void *rho, int64_t n, int rho_bits,
                         cudaStream_t stream)
{
    int grid = 0;
    const Chunking ck = plan(n, &grid);
    if (rho_bits == 8)
        split_kernel<8><<<grid, kThreads, 0, stream>>>(theta, tp, rho, n, ck);
    else
        split_kernel<16><<<grid, kThreads, 0, stream>>>(theta, tp, rho, n, ck);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_merge(const uint16_t *tp, const void *rho, float *theta, int64_t n, int rho_bits,
                         cudaStream_t stream)
{
    int grid = 0;
    const Chunking ck = plan(n, &grid);
    if (rho_bits == 8)
        merge_kernel<8><<<grid, kThreads, 0, stream>>>(tp, rho, theta, n, ck);
    else
        merge_kernel<16><<<grid, kThreads, 0, stream>>>(tp, rho, theta, n, ck);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_quant(const float *x, void *q, uint16_t *scales, int64_t n, int kind,
                         cudaStream_t stream)
{
    int grid = 0;
    const Chunking ck = plan(n, &grid);
    switch (kind) {
    case 0: quant_kernel<0><<<grid, kThreads, 0, stream>>>(x, q, scales, n, ck); break;
    case 1: quant_kernel<1><<<grid, kThreads, 0, stream>>>(x, q, scales, n, ck); break;
    case 2: quant_kernel<2><<<grid, kThreads, 0, stream>>>(x, q, scales, n, ck); break;
    case 3: quant_kernel<3><<<grid, kThreads, 0, stream>>>(x, q, scales, n, ck); break;
    default: quant_kernel<5><<<grid, kThreads, 0, stream>>>(x, q, scales, n, ck); break;
    }
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_dequant(const void *q, const uint16_t *scales, float *x, int64_t n, int kind,
                           cudaStream_t stream)
{
    int grid = 0;
    const Chunking ck = plan(n, &grid);
    switch (kind) {
    case 0: dequant_kernel<0><<<grid, kThreads, 0, stream>>>(q, scales, x, n, ck); break;
    case 1: dequant_kernel<1><<<grid, kThreads, 0, stream>>>(q, scales, x, n, ck); break;
    case 2: dequant_kernel<2><<<grid, kThreads, 0, stream>>>(q, scales, x, n, ck); break;
    case 3: dequant_kernel<3><<<grid, kThreads, 0, stream>>>(q, scales, x, n, ck); break;
    default: dequant_kernel<1><<<grid, kThreads, 0, stream>>>(q, scales, x, n, ck); break;   // kind 5 decodes as 1
    }
    count_launch();
    return cudaGetLastError();
}

}  // namespace fo
