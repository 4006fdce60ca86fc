// fo_codecs.cu -- stand-alone codecs of "FlashOptim: Optimizers for Memory
// Efficient Training": weight splitting and merging (section "权重复分裂",
// Eq. 1-2) and companded group quantization of the optimizer state (section
// "带压缩扩展的优化器状态量化", Algorithms 2-3). They initialise and export
// the compressed state; the fused step (fo_step.cuh) uses the same primitives.
//
// Split and quant: a thread owns 16 contiguous elements, and a 32-element
// group is a pair of adjacent lanes (quant combines their absmax with one
// shuffle). Quant reads its 64 bytes with two 32-byte loads when the input is
// 32-byte aligned (whole sectors per warp access; 4-9 % faster), else four
// 16-byte ones. Merge and dequant, which write 4 bytes per element: a warp owns
// 512 contiguous elements and lane l takes elements 128k + 4l .. 128k + 4l + 3
// (k = 0..3), so that each 16-byte store of the warp covers 512 contiguous
// bytes (a thread's 64 contiguous bytes left every store strided by 64 bytes;
// this layout is 13-30 % faster). Grid-stride loops run the same number of
// iterations in every thread so that the pair shuffle always has both lanes
// present.
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

// 32 contiguous bytes in one streaming load (p must be 32-byte aligned)
__device__ __forceinline__ void ld_stream8(const void *p, uint32_t (&w)[8])
{
    asm volatile("ld.global.cs.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
                 : "l"(p));
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
    // a warp covers 512 consecutive elements; lane l takes elements
    // 128k + 4l .. 128k + 4l + 3 (k = 0..3), so each of the warp's 16-byte
    // stores writes 512 contiguous bytes
    const int lane = threadIdx.x & 31;
    for (int64_t it = 0; it < ck.iters; ++it) {
        const int64_t c = (int64_t)blockIdx.x * kThreads + threadIdx.x + it * ck.stride;
        const int64_t base = (c >> 5) * 512;
        if (base >= n)
            continue;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int64_t i = base + 128 * k + 4 * lane;
            const int64_t rem = n - i;
            const int cnt = rem >= 4 ? 4 : (rem > 0 ? (int)rem : 0);
            if (cnt == 0)
                continue;
            uint32_t tw[2] = {0, 0};
            int32_t rv[4] = {0, 0, 0, 0};
            if (cnt == 4) {
                const uint2 a = __ldcs(reinterpret_cast<const uint2 *>(tp + i));
                tw[0] = a.x; tw[1] = a.y;
                if (RB == 8) {
                    const uint32_t w = __ldcs(reinterpret_cast<const unsigned int *>(static_cast<const int8_t *>(rho) + i));
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        rv[e] = (int32_t)(int8_t)(w >> (8 * e));
                } else {
                    const uint2 w = __ldcs(reinterpret_cast<const uint2 *>(static_cast<const int16_t *>(rho) + i));
                    rv[0] = (int32_t)(int16_t)w.x; rv[1] = (int32_t)(int16_t)(w.x >> 16);
                    rv[2] = (int32_t)(int16_t)w.y; rv[3] = (int32_t)(int16_t)(w.y >> 16);
                }
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (e < cnt) {
                        tw[e >> 1] |= (uint32_t)tp[i + e] << (16 * (e & 1));
                        rv[e] = RB == 8 ? static_cast<const int8_t *>(rho)[i + e]
                                        : static_cast<const int16_t *>(rho)[i + e];
                    }
                }
            }
            float x[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const uint32_t bits = (e & 1) ? bf16_hi_bits(tw[e >> 1]) : bf16_lo_bits(tw[e >> 1]);
                x[e] = merge_one<RB>(bits, (float)rv[e]);
            }
            if (cnt == 4) {
                st_stream(theta + i, make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]),
                                                __float_as_uint(x[3])));
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (e < cnt)
                        theta[i + e] = x[e];
            }
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


template <int Kind>
__global__ void __launch_bounds__(kThreads) quant_kernel(const float *__restrict__ xin, void *__restrict__ q,
                                                         uint16_t *__restrict__ scales, int64_t n, Chunking ck)
{
    // a thread's 64 bytes start 32-byte aligned when the array does
    const bool wide = (reinterpret_cast<uintptr_t>(xin) & 31u) == 0;
    for (int64_t it = 0; it < ck.iters; ++it) {
        const int64_t c = (int64_t)blockIdx.x * kThreads + threadIdx.x + it * ck.stride;
        const int64_t i0 = c * kEPT;
        const int cnt = valid_count(i0, n);
        float y[kEPT];
        if (cnt == kEPT && wide) {
            // two 32-byte loads: each covers whole 32-byte sectors
            uint32_t w[8];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                ld_stream8(xin + i0 + 8 * h, w);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    y[8 * h + e] = __uint_as_float(w[e]);
            }
        } else if (cnt == kEPT) {
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
    // a warp covers 512 consecutive elements; lane l takes elements
    // 128k + 4l .. 128k + 4l + 3 (k = 0..3), so each of the warp's four
    // 16-byte stores writes 512 contiguous bytes
    const int lane = threadIdx.x & 31;
    for (int64_t it = 0; it < ck.iters; ++it) {
        const int64_t c = (int64_t)blockIdx.x * kThreads + threadIdx.x + it * ck.stride;
        const int64_t base = (c >> 5) * 512;
        if (base >= n)
            continue;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int64_t i = base + 128 * k + 4 * lane;
            const int64_t rem = n - i;
            const int cnt = rem >= 4 ? 4 : (rem > 0 ? (int)rem : 0);
            if (cnt == 0)
                continue;
            uint32_t w = 0;
            if (cnt == 4) {
                w = __ldcs(reinterpret_cast<const unsigned int *>(static_cast<const uint8_t *>(q) + i));
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (j < cnt)
                        w |= (uint32_t)static_cast<const uint8_t *>(q)[i + j] << (8 * j);
            }
            const uint16_t sbits = scales[i >> 5];
            // s/L: the validated constant division for positive finite FP16
            // scales (0x0001..0x7BFF), IEEE division for the rest
            const float sv = scale_value(sbits);
            const float step = (uint32_t)sbits - 1u < 0x7BFFu
                                   ? div_by_const(sv, -KindTraits<Kind>::kLevels,
                                                  KindTraits<Kind>::kLevels == 127.0f ? kRcp127 : kRcp255)
                                   : __fdiv_rn(sv, KindTraits<Kind>::kLevels);
            const bool small_scale = (uint32_t)sbits - 1u < 0x3FEFu;
            const uint32_t wx = KindTraits<Kind>::kSigned ? (w ^ 0x80808080u) : w;
            float cc[4];
            if (KindTraits<Kind>::kSigned) {
                cc[0] = s8_at<0>(wx); cc[1] = s8_at<1>(wx); cc[2] = s8_at<2>(wx); cc[3] = s8_at<3>(wx);
            } else {
                cc[0] = u8_at<0>(wx); cc[1] = u8_at<1>(wx); cc[2] = u8_at<2>(wx); cc[3] = u8_at<3>(wx);
            }
            float x[4];
            if (Kind == 0 && small_scale) {
                // phi_m^-1(z) = z / (2 - |z|) on element pairs, |z| < 2: the
                // short division of fo_pair.cuh, enumerated equal to the IEEE
                // division for every code byte under every scale 0x0000-0x3FEF
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const f2 d = mul2(pk(cc[2 * h], cc[2 * h + 1]), splat(step));
                    float d0, d1;
                    unpk(d, d0, d1);
                    unpk(div2_short(d, pk(__fsub_rn(fabsf(d0), 2.0f), __fsub_rn(fabsf(d1), 2.0f))), x[2 * h],
                         x[2 * h + 1]);
                }
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    x[e] = expand<Kind>(__fmul_rn(cc[e], step));
            }
            if (cnt == 4) {
                st_stream(xout + i, make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]),
                                               __float_as_uint(x[3])));
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (j < cnt)
                        xout[i + j] = x[j];
            }
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
