// fo_api.cu -- the C ABI declared in include/fo.h: argument validation,
// per-step scalar derivation and kernel launches. No entry point allocates
// device memory, synchronizes, or falls back to the CPU.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <vector>

#include "fo.h"
#include "fo_internal.h"

namespace fo {

static std::atomic<uint64_t> g_launches{0};
static thread_local int t_last_cuda_error = 0;

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

int sm_count()
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
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) {
            (void)cudaGetLastError();
            return 1;
        }
        slot.store(n, std::memory_order_relaxed);
    }
    return n;
}

}  // namespace fo

namespace {

using fo::Opt;

fo_status_t cuda_status(cudaError_t e)
{
    if (e == cudaSuccess)
        return FO_OK;
    fo::t_last_cuda_error = (int)e;
    return FO_ERR_CUDA;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool is_finite(double x) { return std::isfinite(x); }

// b^t by repeated squaring in double (the contract in fo.h).
double pow_by_squaring(double b, int64_t t)
{
    double r = 1.0;
    while (t > 0) {
        if (t & 1)
            r *= b;
        b *= b;
        t >>= 1;
    }
    return r;
}

fo_status_t check_row(const fo_tensor_t &t, bool with_v)
{
    if (t.numel < 0)
        return FO_ERR_SIZE;
    if (t.rho_bits != 8 && t.rho_bits != 16)
        return FO_ERR_BAD_ARG;
    if ((t.grad_dtype != FO_GRAD_BF16 && t.grad_dtype != FO_GRAD_F32) || !is_finite(t.weight_decay))
        return FO_ERR_BAD_ARG;
    if (t.numel == 0)
        return FO_OK;
    if (t.numel > ((int64_t)1 << 46))
        return FO_ERR_SIZE;
    if (!t.theta || !t.rho || !t.m_q || !t.m_scale || !t.grad || (with_v && (!t.v_q || !t.v_scale)))
        return FO_ERR_NULL;
    if (!aligned16(t.theta) || !aligned16(t.rho) || !aligned16(t.m_q) || !aligned16(t.grad) ||
        (with_v && !aligned16(t.v_q)))
        return FO_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(t.m_scale) & 1u) || (with_v && (reinterpret_cast<uintptr_t>(t.v_scale) & 1u)))
        return FO_ERR_MISALIGNED;
    return FO_OK;
}

// One array of a table row: bytes [lo, hi), and whether the step writes it.
struct Span {
    uintptr_t lo, hi;
    bool written;
};

// No array that a step writes may share a byte with any other array of the
// table (in the same row or another): rows updated by one launch would race,
// and rows of different launches would be stepped twice. Gradients are only
// read, so several rows may share one. The spans are sorted by start address
// (O(n log n)); a per-thread scratch array holds them between calls.
fo_status_t check_disjoint(const fo_tensor_t *table, int32_t ntensors, bool with_v)
{
    static thread_local std::vector<Span> spans;
    try {
        spans.clear();
        spans.reserve((size_t)ntensors * (with_v ? 7 : 5));
    } catch (...) {
        return FO_ERR_SIZE;
    }
    for (int32_t i = 0; i < ntensors; ++i) {
        const fo_tensor_t &t = table[i];
        if (t.numel <= 0)
            continue;
        const int64_t n = t.numel, ng = (n + 31) / 32;
        const void *ptr[7] = {t.grad, t.theta, t.rho, t.m_q, t.m_scale, t.v_q, t.v_scale};
        const int64_t bytes[7] = {(t.grad_dtype == FO_GRAD_F32 ? 4 : 2) * n, 2 * n, n * (t.rho_bits / 8), n,
                                  2 * ng, n, 2 * ng};
        const int count = with_v ? 7 : 5;
        for (int a = 0; a < count; ++a) {
            const uintptr_t lo = reinterpret_cast<uintptr_t>(ptr[a]);
            spans.push_back(Span{lo, lo + (uintptr_t)bytes[a], a != 0});
        }
    }
    std::sort(spans.begin(), spans.end(), [](const Span &x, const Span &y) { return x.lo < y.lo; });
    // a span overlaps an earlier-starting one exactly when it starts below that
    // one's end: track the furthest end among written spans and among all
    uintptr_t end_written = 0, end_any = 0;
    for (const Span &sp : spans) {
        if (sp.lo < end_written || (sp.written && sp.lo < end_any))
            return FO_ERR_ALIAS;
        end_any = std::max(end_any, sp.hi);
        if (sp.written)
            end_written = std::max(end_written, sp.hi);
    }
    return FO_OK;
}

// A CUDA error left pending by earlier work (a non-sticky launch error that
// nobody has read yet) would be reported by the first cudaGetLastError after
// this call's own launch, and the call would look failed after part of its
// work was enqueued. So it is read (and cleared) before anything is launched,
// and reported as this call's FO_ERR_CUDA, with nothing launched.
fo_status_t pending_error()
{
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess)
        return FO_OK;
    fo::t_last_cuda_error = (int)e;
    return FO_ERR_CUDA;
}

// Per-row scalar: decay (AdamW, Lion) or weight decay (SGD), rounded once to FP32.
using RowCoef = float (*)(double lr, double weight_decay);

fo_status_t run_table(Opt opt, const fo_tensor_t *table, int32_t ntensors, const fo::StepScalars &s,
                      double lr, RowCoef coef, fo_stream_t stream)
{
    if (ntensors < 0)
        return FO_ERR_SIZE;
    if (ntensors > FO_MAX_TENSORS)
        return FO_ERR_TOO_MANY_TENSORS;
    if (ntensors == 0)
        return FO_OK;
    if (!table)
        return FO_ERR_NULL;
    const bool with_v = opt == Opt::kAdamW;
    bool any_work = false;
    for (int32_t i = 0; i < ntensors; ++i) {
        const fo_status_t st = check_row(table[i], with_v);
        if (st != FO_OK)
            return st;
        any_work = any_work || table[i].numel > 0;
    }
    if (!any_work)
        return FO_OK;
    fo_status_t st0 = check_disjoint(table, ntensors, with_v);
    if (st0 == FO_OK)
        st0 = pending_error();
    if (st0 != FO_OK)
        return st0;

    // Pack rows into launches of one correction width and one gradient type,
    // at most kRowsPerLaunch rows and 2^31-1 tiles each (a kernel is
    // specialised per width and type).
    static thread_local fo::StepParams p;  // large: kept off the stack
    p.s = s;
    for (int combo = 0; combo < 4; ++combo) {
        const int rb = (combo & 1) ? 16 : 8;
        const int gdt = (combo & 2) ? FO_GRAD_F32 : FO_GRAD_BF16;
        // chunks per tile for this combination's rows: long tiles for large
        // tables, shorter ones while the table would give a resident CTA
        // fewer than kMinTilesPerCta tiles
        int64_t total = 0;
        for (int32_t j = 0; j < ntensors; ++j)
            if (table[j].rho_bits == rb && table[j].grad_dtype == gdt)
                total += table[j].numel;
        if (total == 0)
            continue;
        const int64_t ctas =
            (int64_t)fo::sm_count() * fo::step_ctas_per_sm(opt, rb, gdt == FO_GRAD_F32 ? 32 : 16, fo::kLongChunks);
        const int chunks = total / ((int64_t)fo::kStepChunk * fo::kLongChunks) >= ctas * fo::kMinTilesPerCta
                               ? fo::kLongChunks
                           : total / ((int64_t)fo::kStepChunk * fo::kShortChunks) >= ctas ? fo::kShortChunks
                                                                                           : fo::kTinyChunks;
        p.chunks = chunks;
        const int64_t tile_elems = (int64_t)fo::kStepChunk * chunks;
        int32_t i = 0;
        while (i < ntensors) {
            int nrows = 0;
            int64_t tiles = 0;
            while (i < ntensors && nrows < fo::kRowsPerLaunch) {
                const fo_tensor_t &t = table[i];
                if (t.numel == 0 || t.rho_bits != rb || t.grad_dtype != gdt) {
                    ++i;
                    continue;
                }
                const int64_t rt = (t.numel + tile_elems - 1) / tile_elems;
                if (nrows > 0 && tiles + rt > INT32_MAX)
                    break;
                fo::StepRow &r = p.rows[nrows];
                r.theta = t.theta;
                r.rho = t.rho;
                r.mq = t.m_q;
                r.ms = t.m_scale;
                r.vq = with_v ? t.v_q : nullptr;
                r.vs = with_v ? t.v_scale : nullptr;
                r.grad = t.grad;
                r.numel = t.numel;
                r.coef = coef(lr, t.weight_decay);
                r.rho_bits = t.rho_bits;
                tiles += rt;
                p.tile_end[nrows] = (int32_t)tiles;
                ++nrows;
                ++i;
            }
            if (nrows == 0)
                break;
            p.nrows = nrows;
            p.total_tiles = (int32_t)tiles;
            const fo_status_t st = cuda_status(fo::launch_step(opt, rb, gdt == FO_GRAD_F32 ? 32 : 16, p, static_cast<cudaStream_t>(stream)));
            if (st != FO_OK)
                return st;
        }
    }
    return FO_OK;
}

float decay_coef(double lr, double wd) { return (float)(1.0 - lr * wd); }

// The fast path's range for a checked operand x: x = 0 or lo <= |x| <= hi,
// stored as the FP32 values just below lo and hi (see StepScalars).
void set_range(fo::StepScalars &s, float lo, float hi)
{
    s.lo = std::nextafter(lo, 0.0f);
    s.hi = std::nextafter(hi, 0.0f);
}

// AdamW's packed fast path (fo_step.cuh, pair_fast) divides and takes square
// roots with sequences validated for operands in [2^-100, 2^100] (and zero
// numerators). With the per-element check that the gradient g is 0 or
// T <= |g| <= 2^24, these conditions keep every operand inside:
//  - eps in [2^-40, 2^20] and 1/sqrt(bc2) <= 2^8: den in [2^-40, 2^33];
//  - b1, b2 zero or at least 2^-16 and 1-b1, 1-b2 at least 2^-24: a non-zero
//    v is at least 2^-99 and a non-zero m at least 2^-94 (a decoded non-zero
//    momentum is at least 2^-32 and its second moment 2^-64; a cancellation
//    in b1*m + (1-b1)*g leaves a multiple of the operands' finest ulp);
//  - T is the smallest power of two with (1-b1)*T >= 2^-96 and
//    (1-b2)*T^2 >= 2^-98, so that a gradient alone gives the same bounds;
//  - lr/bc1 zero or at least 2^-80: its 2^-32 scaling stays exact;
//  - per thread, the largest sqrt(v) at most 2^40, which bounds |g| by 2^52
//    and |m| by 2^53 (v >= (1-b2)*g^2).
// Then m' = 2^32 m and m'/den lie in [2^-100, 2^100] or are zero (a large
// gradient also makes den large), and phi_m's quotient too. Calls outside
// these conditions take the IEEE path throughout.
// t_known: the step scalars a[5], a[6] are set (fo_adamw_step); otherwise
// (fo_adamw_step_dev) the kernel adds their conditions on the device.
void adamw_fast_ranges(fo::StepScalars &s, bool t_known)
{
    const float b1 = s.a[0], b2 = s.a[1], c1 = s.a[2], c2 = s.a[3], step = -s.a[5];
    bool fast = s.a[4] >= 0x1p-40f && s.a[4] <= 0x1p20f;
    fast = fast && (b1 == 0.0f || b1 >= 0x1p-16f) && (b2 == 0.0f || b2 >= 0x1p-16f);
    fast = fast && c1 >= 0x1p-24f && c2 >= 0x1p-24f;
    if (t_known)
        fast = fast && s.a[6] <= 0x1p8f && (step == 0.0f || step >= 0x1p-80f);
    double t = 0x1p-100;
    while (t < 0x1p-30 && !((double)c1 * t >= 0x1p-96 && (double)c2 * t * t >= 0x1p-98))
        t *= 2.0;
    s.fast = fast ? 1 : 0;
    set_range(s, (float)t, __builtin_inff());   // the upper bound is checked through sqrt(v)
}

// Both lanes of a packed FP32 pair set to x.
unsigned long long lanes(float x)
{
    uint32_t u;
    std::memcpy(&u, &x, sizeof u);
    return ((unsigned long long)u << 32) | u;
}
float wd_coef(double, double wd) { return (float)wd; }

bool beta_ok(double b) { return is_finite(b) && b >= 0.0 && b < 1.0; }

bool kind_ok(fo_state_kind_t kind)
{
    return kind == FO_STATE_MOMENTUM || kind == FO_STATE_VARIANCE || kind == FO_STATE_MOMENTUM_LINEAR ||
           kind == FO_STATE_VARIANCE_LINEAR || kind == FO_STATE_VARIANCE_NONZERO;
}

fo_status_t check_codec(const void *a, const void *b, const void *c, int64_t n)
{
    if (n < 0)
        return FO_ERR_SIZE;
    if (n == 0)
        return FO_OK;
    if (n > ((int64_t)1 << 46))
        return FO_ERR_SIZE;
    if (!a || !b || !c)
        return FO_ERR_NULL;
    return FO_OK;
}

bool overlap(const void *a, int64_t abytes, const void *b, int64_t bbytes)
{
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + (uintptr_t)bbytes && b0 < a0 + (uintptr_t)abytes;
}

// A codec reads one or two arrays and writes the others: the written arrays
// may share no byte with any other array of the call. Arrays 0..nin-1 are
// read, the rest written.
bool codec_aliases(int nin, const void *const *ptr, const int64_t *bytes, int count)
{
    for (int a = 0; a < count; ++a)
        for (int b = a + 1; b < count; ++b)
            if ((a >= nin || b >= nin) && overlap(ptr[a], bytes[a], ptr[b], bytes[b]))
                return true;
    return false;
}

// The step-independent part of AdamW's per-step scalars (the argument checks
// and everything but the bias corrections), shared by both AdamW entry points.
fo_status_t adamw_scalars(const fo_adamw_hparams_t *hp, fo::StepScalars &s)
{
    if (!hp)
        return FO_ERR_NULL;
    if (!is_finite(hp->lr) || hp->lr < 0.0 || !beta_ok(hp->beta1) || !beta_ok(hp->beta2) || !is_finite(hp->eps) ||
        hp->eps <= 0.0 || (hp->flags & ~FO_ADAMW_V_NONZERO) != 0 || hp->reserved != 0)
        return FO_ERR_BAD_ARG;
    std::memset(&s, 0, sizeof s);
    s.a[0] = (float)hp->beta1;
    s.a[1] = (float)hp->beta2;
    s.a[2] = (float)(1.0 - hp->beta1);
    s.a[3] = (float)(1.0 - hp->beta2);
    s.a[4] = (float)hp->eps;
    // the packed fast path carries m' = 2^32 m (exact scalings of the constants)
    s.p[0] = lanes(s.a[0] * 0x1p32f);
    s.p[1] = lanes(-s.a[1]);
    s.p[2] = lanes(s.a[2] * 0x1p32f);
    s.p[3] = lanes(-s.a[3]);
    s.p[5] = lanes(-s.a[4]);
    s.v_nonzero = (hp->flags & FO_ADAMW_V_NONZERO) ? 1 : 0;
    return FO_OK;
}

}  // namespace

extern "C" {

fo_status_t fo_split(const float *theta_f32, uint16_t *theta_bf16, void *rho, int64_t n, int32_t rho_bits,
                     fo_stream_t stream)
{
    fo_status_t st = check_codec(theta_f32, theta_bf16, rho, n);
    if (st != FO_OK || n == 0)
        return st;
    if (rho_bits != 8 && rho_bits != 16)
        return FO_ERR_BAD_ARG;
    if (!aligned16(theta_f32) || !aligned16(theta_bf16) || !aligned16(rho))
        return FO_ERR_MISALIGNED;
    {
        const void *ptr[3] = {theta_f32, theta_bf16, rho};
        const int64_t bytes[3] = {4 * n, 2 * n, n * (rho_bits / 8)};
        if (codec_aliases(1, ptr, bytes, 3))
            return FO_ERR_ALIAS;
    }
    if ((st = pending_error()) != FO_OK)
        return st;
    return cuda_status(fo::launch_split(theta_f32, theta_bf16, rho, n, rho_bits, static_cast<cudaStream_t>(stream)));
}

fo_status_t fo_merge(const uint16_t *theta_bf16, const void *rho, float *theta_f32, int64_t n, int32_t rho_bits,
                     fo_stream_t stream)
{
    fo_status_t st = check_codec(theta_bf16, rho, theta_f32, n);
    if (st != FO_OK || n == 0)
        return st;
    if (rho_bits != 8 && rho_bits != 16)
        return FO_ERR_BAD_ARG;
    if (!aligned16(theta_f32) || !aligned16(theta_bf16) || !aligned16(rho))
        return FO_ERR_MISALIGNED;
    {
        const void *ptr[3] = {theta_bf16, rho, theta_f32};
        const int64_t bytes[3] = {2 * n, n * (rho_bits / 8), 4 * n};
        if (codec_aliases(2, ptr, bytes, 3))
            return FO_ERR_ALIAS;
    }
    if ((st = pending_error()) != FO_OK)
        return st;
    return cuda_status(fo::launch_merge(theta_bf16, rho, theta_f32, n, rho_bits, static_cast<cudaStream_t>(stream)));
}

fo_status_t fo_quant_state(const float *x, void *q, uint16_t *scales, int64_t n, fo_state_kind_t kind,
                           fo_stream_t stream)
{
    fo_status_t st = check_codec(x, q, scales, n);
    if (st != FO_OK || n == 0)
        return st;
    if (!kind_ok(kind))
        return FO_ERR_BAD_ARG;
    if (!aligned16(x) || !aligned16(q) || (reinterpret_cast<uintptr_t>(scales) & 1u))
        return FO_ERR_MISALIGNED;
    {
        const void *ptr[3] = {x, q, scales};
        const int64_t bytes[3] = {4 * n, n, 2 * ((n + 31) / 32)};
        if (codec_aliases(1, ptr, bytes, 3))
            return FO_ERR_ALIAS;
    }
    if ((st = pending_error()) != FO_OK)
        return st;
    return cuda_status(fo::launch_quant(x, q, scales, n, (int)kind, static_cast<cudaStream_t>(stream)));
}

fo_status_t fo_dequant_state(const void *q, const uint16_t *scales, float *x, int64_t n, fo_state_kind_t kind,
                             fo_stream_t stream)
{
    fo_status_t st = check_codec(q, scales, x, n);
    if (st != FO_OK || n == 0)
        return st;
    if (!kind_ok(kind))
        return FO_ERR_BAD_ARG;
    if (!aligned16(x) || !aligned16(q) || (reinterpret_cast<uintptr_t>(scales) & 1u))
        return FO_ERR_MISALIGNED;
    {
        const void *ptr[3] = {q, scales, x};
        const int64_t bytes[3] = {n, 2 * ((n + 31) / 32), 4 * n};
        if (codec_aliases(2, ptr, bytes, 3))
            return FO_ERR_ALIAS;
    }
    if ((st = pending_error()) != FO_OK)
        return st;
    return cuda_status(fo::launch_dequant(q, scales, x, n, (int)kind, static_cast<cudaStream_t>(stream)));
}

fo_status_t fo_adamw_step(const fo_tensor_t *table, int32_t ntensors, const fo_adamw_hparams_t *hp, int64_t step,
                          fo_stream_t stream)
{
    fo::StepScalars s;
    fo_status_t st = adamw_scalars(hp, s);
    if (st != FO_OK)
        return st;
    if (step < 1)
        return FO_ERR_SIZE;
    const double bc1 = 1.0 - pow_by_squaring(hp->beta1, step);
    const double bc2 = 1.0 - pow_by_squaring(hp->beta2, step);
    s.a[5] = -(float)(hp->lr / bc1);
    s.a[6] = (float)(1.0 / std::sqrt(bc2));
    s.p[4] = lanes(s.a[6]);
    s.p[6] = lanes(s.a[5] * 0x1p-32f);
    adamw_fast_ranges(s, true);
    return run_table(Opt::kAdamW, table, ntensors, s, hp->lr, decay_coef, stream);
}

fo_status_t fo_adamw_step_dev(const fo_tensor_t *table, int32_t ntensors, const fo_adamw_hparams_t *hp,
                              const int64_t *step_dev, fo_stream_t stream)
{
    fo::StepScalars s;
    fo_status_t st = adamw_scalars(hp, s);
    if (st != FO_OK)
        return st;
    if (!step_dev)
        return FO_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(step_dev) & 7u)
        return FO_ERR_MISALIGNED;
    // the kernel reads t and derives the step scalars (with the expressions
    // of fo_adamw_step above) and the t-dependent preconditions itself
    s.step_dev = reinterpret_cast<const long long *>(step_dev);
    s.lr = hp->lr;
    s.beta1 = hp->beta1;
    s.beta2 = hp->beta2;
    adamw_fast_ranges(s, false);
    return run_table(Opt::kAdamW, table, ntensors, s, hp->lr, decay_coef, stream);
}

fo_status_t fo_sgd_step(const fo_tensor_t *table, int32_t ntensors, const fo_sgd_hparams_t *hp, fo_stream_t stream)
{
    if (!hp)
        return FO_ERR_NULL;
    if (!is_finite(hp->lr) || hp->lr < 0.0 || !is_finite(hp->momentum) || hp->momentum < 0.0)
        return FO_ERR_BAD_ARG;
    fo::StepScalars s;
    std::memset(&s, 0, sizeof s);
    s.a[0] = (float)hp->momentum;
    s.a[1] = -(float)hp->lr;
    s.p[0] = lanes(s.a[0]);
    s.p[1] = lanes(s.a[1]);
    s.fast = 1;
    set_range(s, 0x1p-100f, 0x1p100f);   // the new momentum: phi_m's validated range
    return run_table(Opt::kSgd, table, ntensors, s, hp->lr, wd_coef, stream);
}

fo_status_t fo_lion_step(const fo_tensor_t *table, int32_t ntensors, const fo_lion_hparams_t *hp,
                         fo_stream_t stream)
{
    if (!hp)
        return FO_ERR_NULL;
    if (!is_finite(hp->lr) || hp->lr < 0.0 || !beta_ok(hp->beta1) || !beta_ok(hp->beta2))
        return FO_ERR_BAD_ARG;
    fo::StepScalars s;
    std::memset(&s, 0, sizeof s);
    s.a[0] = (float)hp->beta1;
    s.a[1] = (float)hp->beta2;
    s.a[2] = (float)(1.0 - hp->beta1);
    s.a[3] = (float)(1.0 - hp->beta2);
    s.a[4] = -(float)hp->lr;
    for (int i = 0; i < 5; ++i)
        s.p[i] = lanes(s.a[i]);
    s.fast = 1;
    set_range(s, 0x1p-100f, 0x1p100f);   // the new momentum: phi_m's validated range
    return run_table(Opt::kLion, table, ntensors, s, hp->lr, decay_coef, stream);
}

const char *fo_status_string(fo_status_t status)
{
    switch (status) {
    case FO_OK: return "FO_OK";
    case FO_ERR_NULL: return "FO_ERR_NULL: a required pointer is NULL";
    case FO_ERR_MISALIGNED: return "FO_ERR_MISALIGNED: an element array is not 16-byte aligned";
    case FO_ERR_SIZE: return "FO_ERR_SIZE: a count is negative or too large";
    case FO_ERR_BAD_ARG: return "FO_ERR_BAD_ARG: a flag or hyper-parameter is out of range";
    case FO_ERR_TOO_MANY_TENSORS: return "FO_ERR_TOO_MANY_TENSORS: ntensors exceeds FO_MAX_TENSORS";
    case FO_ERR_CUDA: return "FO_ERR_CUDA: a CUDA call failed";
    case FO_ERR_ALIAS: return "FO_ERR_ALIAS: an array the call writes overlaps another array of the call";
    }
    return "unknown fo_status_t";
}

fo_status_t fo_verify_fast_arithmetic(uint64_t *counts, fo_stream_t stream)
{
    if (!counts)
        return FO_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(counts) & 7u) != 0)
        return FO_ERR_MISALIGNED;
    fo_status_t st = pending_error();
    if (st != FO_OK)
        return st;
    return cuda_status(fo::launch_verify(reinterpret_cast<unsigned long long *>(counts),
                                         static_cast<cudaStream_t>(stream)));
}

int fo_last_cuda_error(void) { return fo::t_last_cuda_error; }

uint64_t fo_kernel_launch_count(void) { return fo::g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
