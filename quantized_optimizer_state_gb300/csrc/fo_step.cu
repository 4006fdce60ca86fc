// fo_step.cu -- the fused compressed optimizer step (FlashAdamW, FlashSGD,
// FlashLion): "FlashOptim: Optimizers for Memory Efficient Training",
// section "融合优化器步骤" (Algorithm 4) -- dequantize m and v, rebuild the
// master weight, apply the standard update, requantize and re-split, in one
// pass so that each byte of state crosses HBM once.
//
// Design (GB300, sm_103a): the work is element-wise plus a 32-wide absmax per
// group, so it is bound by HBM traffic and instruction issue, never by tensor
// cores. A persistent grid (SMs x resident CTAs) walks 4096-element tiles of
// the concatenated tensor list in a static round-robin; a thread owns 16
// contiguous elements (half a group) and loads them with 128-bit streaming
// loads, the two threads of a group combine their absmax with one shuffle,
// and the results leave with 128-bit streaming stores. Tensor rows travel in
// the kernel parameters, so a step allocates nothing.
#include <utility>

#include "fo_device.cuh"
#include "fo_internal.h"

namespace fo {
namespace {

constexpr int kEPT = kElemsPerThread;

struct Loaded {
    uint32_t g[8];   // 16 BF16 gradients
    uint32_t t[8];   // 16 BF16 theta'
    uint32_t r[8];   // 16 rho codes (4 words for 8-bit, 8 for 16-bit)
    uint32_t m[4];   // 16 INT8 momentum codes
    uint32_t v[4];   // 16 UINT8 second-moment codes
    uint16_t ms, vs; // the group's FP16 scales
};

template <int RB, bool WithV>
__device__ __forceinline__ void load_full(const StepRow &row, int64_t i0, Loaded &L)
{
    uint4 a = ld_stream(row.grad + i0), b = ld_stream(row.grad + i0 + 8);
    L.g[0] = a.x; L.g[1] = a.y; L.g[2] = a.z; L.g[3] = a.w;
    L.g[4] = b.x; L.g[5] = b.y; L.g[6] = b.z; L.g[7] = b.w;
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
}

// Element-wise loads of the first cnt (< 16) elements; the rest read as 0.
template <int RB, bool WithV>
__device__ __forceinline__ void load_partial(const StepRow &row, int64_t i0, int cnt, Loaded &L)
{
#pragma unroll
    for (int w = 0; w < 8; ++w) { L.g[w] = 0; L.t[w] = 0; L.r[w] = 0; }
#pragma unroll
    for (int w = 0; w < 4; ++w) { L.m[w] = 0; L.v[w] = 0; }
    L.ms = 0;
    L.vs = 0;
    if (cnt <= 0)
        return;
#pragma unroll
    for (int j = 0; j < kEPT; ++j) {
        if (j < cnt) {
            const int sh16 = 16 * (j & 1), sh8 = 8 * (j & 3);
            L.g[j >> 1] |= (uint32_t)row.grad[i0 + j] << sh16;
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
    L.ms = row.ms[i0 >> 5];
    if (WithV)
        L.vs = row.vs[i0 >> 5];
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

// Element j: decode, update, re-split. Writes the new theta (FP32) and the
// companded momentum z (and r = sqrt(v) for AdamW).
template <Opt O, int RB, int J>
__device__ __forceinline__ void element(const Loaded &L, const uint32_t (&rx)[8], const uint32_t (&mx)[4],
                                        const StepScalars &s, float coef, float cm, float cv,
                                        float &theta_out, float &z_out, float &r_out)
{
    const float g = __uint_as_float(theta_p_bits<J>(L.g));
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
        r_out = r;
    } else if (O == Opt::kSgd) {
        const float gp = __fmaf_rn(coef, theta, g);
        m = __fmaf_rn(s.a[0], m, gp);
        theta = __fmaf_rn(s.a[1], m, theta);
        r_out = 0.0f;
    } else {
        const float c = __fmaf_rn(s.a[0], m, __fmul_rn(s.a[2], g));
        const float sgn = c > 0.0f ? 1.0f : (c < 0.0f ? -1.0f : 0.0f);
        theta = __fmaf_rn(s.a[4], sgn, __fmul_rn(theta, coef));
        m = __fmaf_rn(s.a[1], m, __fmul_rn(s.a[3], g));
        r_out = 0.0f;
    }
    theta_out = theta;
    z_out = phi_m(m);
}

template <Opt O, int RB, int... J>
__device__ __forceinline__ void all_elements(const Loaded &L, const uint32_t (&rx)[8], const uint32_t (&mx)[4],
                                             const StepScalars &s, float coef, float cm, float cv,
                                             float (&th)[kEPT], float (&z)[kEPT], float (&r)[kEPT],
                                             std::integer_sequence<int, J...>)
{
    (element<O, RB, J>(L, rx, mx, s, coef, cm, cv, th[J], z[J], r[J]), ...);
}

template <Opt O, int RB, bool Full>
__device__ __forceinline__ void thread_step(const StepRow &row, const StepScalars &s, int64_t i0)
{
    constexpr bool WithV = (O == Opt::kAdamW);
    int cnt = kEPT;
    if (!Full) {
        const int64_t rem = row.numel - i0;
        cnt = rem >= kEPT ? kEPT : (rem > 0 ? (int)rem : 0);
    }

    Loaded L;
    if (Full || cnt == kEPT)
        load_full<RB, WithV>(row, i0, L);
    else
        load_partial<RB, WithV>(row, i0, cnt, L);

    // bias the signed codes once per word for the exact byte -> float unpack
    uint32_t rx[8], mx[4];
#pragma unroll
    for (int w = 0; w < 8; ++w)
        rx[w] = L.r[w] ^ (RB == 8 ? 0x80808080u : 0x80008000u);
#pragma unroll
    for (int w = 0; w < 4; ++w)
        mx[w] = L.m[w] ^ 0x80808080u;

    const float cm = __fdiv_rn(scale_value(L.ms), 127.0f);
    const float cv = WithV ? __fdiv_rn(scale_value(L.vs), 255.0f) : 0.0f;

    float th[kEPT], z[kEPT], r[kEPT];
    all_elements<O, RB>(L, rx, mx, s, row.coef, cm, cv, th, z, r,
                        std::make_integer_sequence<int, kEPT>{});

    // re-split theta: theta' (BF16, nearest even) and rho
    uint32_t tp[8], ro[8];
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        tp[w] = pack_bf16x2(th[2 * w], th[2 * w + 1]);
        const uint32_t c0 = split_code<RB>(__float_as_uint(th[2 * w]), bf16_lo_bits(tp[w]));
        const uint32_t c1 = split_code<RB>(__float_as_uint(th[2 * w + 1]), bf16_hi_bits(tp[w]));
        if (RB == 16) {
            ro[w] = pack_halves(c0, c1);
        } else {
            // bytes 2w, 2w+1 of the rho words; assembled below
            ro[w] = __byte_perm(c0, c1, 0x0040u);
        }
    }
    if (RB == 8) {
#pragma unroll
        for (int w = 0; w < 4; ++w)
            ro[w] = __byte_perm(ro[2 * w], ro[2 * w + 1], 0x5410u);
    }

    // group absmax over this thread's valid elements, then over the pair
    float am = 0.0f, av = 0.0f;
#pragma unroll
    for (int j = 0; j < kEPT; ++j) {
        if (Full || j < cnt) {
            am = fmaxf(am, fabsf(z[j]));
            if (WithV)
                av = fmaxf(av, r[j]);
        }
    }
    am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 1));
    if (WithV)
        av = fmaxf(av, __shfl_xor_sync(0xFFFFFFFFu, av, 1));

    const uint16_t sm_new = scale_of(am);
    const float mult_m = code_multiplier(scale_value(sm_new), 127.0f);
    uint32_t mo[4], vo[4];
#pragma unroll
    for (int w = 0; w < 4; ++w)
        mo[w] = pack_bytes(m_code(z[4 * w], mult_m), m_code(z[4 * w + 1], mult_m),
                           m_code(z[4 * w + 2], mult_m), m_code(z[4 * w + 3], mult_m));
    uint16_t sv_new = 0;
    if (WithV) {
        sv_new = scale_of(av);
        const float mult_v = code_multiplier(scale_value(sv_new), 255.0f);
#pragma unroll
        for (int w = 0; w < 4; ++w)
            vo[w] = pack_bytes(v_code(r[4 * w], mult_v), v_code(r[4 * w + 1], mult_v),
                               v_code(r[4 * w + 2], mult_v), v_code(r[4 * w + 3], mult_v));
    }

    if (Full || cnt == kEPT) {
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
            if (j < cnt) {
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
    }
    if ((threadIdx.x & 1) == 0 && cnt > 0) {
        __stcs(row.ms + (i0 >> 5), sm_new);
        if (WithV)
            __stcs(row.vs + (i0 >> 5), sv_new);
    }
}

template <Opt O>
__global__ void __launch_bounds__(kStepThreads)
fo_fused_step_kernel(const __grid_constant__ StepParams p)
{
    int row = 0;
    for (int tile = blockIdx.x; tile < p.total_tiles; tile += gridDim.x) {
        while (tile >= p.tile_end[row])
            ++row;
        const int first = row == 0 ? 0 : p.tile_end[row - 1];
        const StepRow &r = p.rows[row];
        const int64_t e0 = (int64_t)(tile - first) * kStepTile;
        const int64_t i0 = e0 + (int64_t)threadIdx.x * kEPT;
        const bool full = e0 + kStepTile <= r.numel;
        if (r.rho_bits == 8) {
            if (full)
                thread_step<O, 8, true>(r, p.s, i0);
            else
                thread_step<O, 8, false>(r, p.s, i0);
        } else {
            if (full)
                thread_step<O, 16, true>(r, p.s, i0);
            else
                thread_step<O, 16, false>(r, p.s, i0);
        }
    }
}

template <Opt O>
int resident_ctas()
{
    static int cached = 0;
    if (cached == 0) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fo_fused_step_kernel<O>, kStepThreads, 0) !=
                cudaSuccess || n < 1)
            n = 1;
        cached = n;
    }
    return cached;
}

}  // namespace

cudaError_t launch_step(Opt opt, const StepParams &p, cudaStream_t stream)
{
    int ctas = 0;
    switch (opt) {
    case Opt::kAdamW: ctas = resident_ctas<Opt::kAdamW>(); break;
    case Opt::kSgd: ctas = resident_ctas<Opt::kSgd>(); break;
    default: ctas = resident_ctas<Opt::kLion>(); break;
    }
    const long long want = (long long)sm_count() * ctas;
    const int grid = (int)(want < p.total_tiles ? want : p.total_tiles);
    switch (opt) {
    case Opt::kAdamW: fo_fused_step_kernel<Opt::kAdamW><<<grid, kStepThreads, 0, stream>>>(p); break;
    case Opt::kSgd: fo_fused_step_kernel<Opt::kSgd><<<grid, kStepThreads, 0, stream>>>(p); break;
    default: fo_fused_step_kernel<Opt::kLion><<<grid, kStepThreads, 0, stream>>>(p); break;
    }
    count_launch();
    return cudaGetLastError();
}

}  // namespace fo
