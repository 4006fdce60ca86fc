// fo_api.cu -- the C ABI declared in include/fo.h: argument validation,
// per-step scalar derivation and kernel launches. No entry point allocates
// memory, synchronizes, or falls back to the CPU.
#include <atomic>
#include <cmath>
#include <cstring>

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

bool overlaps(const void *a, int64_t abytes, const void *b, int64_t bbytes)
{
    if (!a || !b || abytes <= 0 || bbytes <= 0)
        return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + (uintptr_t)bbytes && b0 < a0 + (uintptr_t)abytes;
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
    // no two arrays of the row may share a byte: the step reads each one and
    // writes the state arrays in place
    const int64_t n = t.numel, ng = (n + 31) / 32;
    const void *ptr[7] = {t.grad, t.theta, t.rho, t.m_q, t.m_scale, t.v_q, t.v_scale};
    const int64_t bytes[7] = {(t.grad_dtype == FO_GRAD_F32 ? 4 : 2) * n, 2 * n, n * (t.rho_bits / 8), n, 2 * ng,
                              n, 2 * ng};
    const int count = with_v ? 7 : 5;
    for (int a = 0; a < count; ++a)
        for (int b = a + 1; b < count; ++b)
            if (overlaps(ptr[a], bytes[a], ptr[b], bytes[b]))
                return FO_ERR_ALIAS;
    return FO_OK;
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
    for (int32_t i = 0; i < ntensors; ++i) {
        const fo_status_t st = check_row(table[i], with_v);
        if (st != FO_OK)
            return st;
    }

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
        const int64_t want_tiles = (int64_t)fo::sm_count() * fo::step_ctas_per_sm(opt) * fo::kMinTilesPerCta;
        const int chunks = total / ((int64_t)fo::kStepChunk * fo::kLongChunks) >= want_tiles ? fo::kLongChunks
                                                                                            : fo::kShortChunks;
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
    if (!a || !b || !c)
        return FO_ERR_NULL;
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
    return cuda_status(fo::launch_dequant(q, scales, x, n, (int)kind, static_cast<cudaStream_t>(stream)));
}

fo_status_t fo_adamw_step(const fo_tensor_t *table, int32_t ntensors, const fo_adamw_hparams_t *hp, int64_t step,
                          fo_stream_t stream)
{
    if (!hp)
        return FO_ERR_NULL;
    if (step < 1)
        return FO_ERR_SIZE;
    if (!is_finite(hp->lr) || hp->lr < 0.0 || !beta_ok(hp->beta1) || !beta_ok(hp->beta2) || !is_finite(hp->eps) ||
        hp->eps <= 0.0 || (hp->flags & ~FO_ADAMW_V_NONZERO) != 0 || hp->reserved != 0)
        return FO_ERR_BAD_ARG;
    const double bc1 = 1.0 - pow_by_squaring(hp->beta1, step);
    const double bc2 = 1.0 - pow_by_squaring(hp->beta2, step);
    fo::StepScalars s;
    std::memset(&s, 0, sizeof s);
    s.a[0] = (float)hp->beta1;
    s.a[1] = (float)hp->beta2;
    s.a[2] = (float)(1.0 - hp->beta1);
    s.a[3] = (float)(1.0 - hp->beta2);
    s.a[4] = (float)hp->eps;
    s.a[5] = -(float)(hp->lr / bc1);
    s.a[6] = (float)(1.0 / std::sqrt(bc2));
    s.p[0] = lanes(s.a[0]);
    s.p[1] = lanes(-s.a[1]);
    s.p[2] = lanes(s.a[2]);
    s.p[3] = lanes(-s.a[3]);
    s.p[4] = lanes(s.a[6]);
    s.p[5] = lanes(-s.a[4]);
    s.p[6] = lanes(s.a[5]);
    // validated operand ranges of the packed division/square root: den = sqrt(v)
    // /sqrt(bc2) + eps stays in [2^-40, 2^40] when these hold (|g| <= 2^24 is
    // checked per element)
    s.fast = (s.a[4] >= 0x1p-40f && s.a[4] <= 0x1p20f && s.a[6] <= 0x1p8f) ? 1 : 0;
    s.v_nonzero = (hp->flags & FO_ADAMW_V_NONZERO) ? 1 : 0;
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
    case FO_ERR_ALIAS: return "FO_ERR_ALIAS: two arrays of one table row overlap";
    }
    return "unknown fo_status_t";
}

int fo_last_cuda_error(void) { return fo::t_last_cuda_error; }

uint64_t fo_kernel_launch_count(void) { return fo::g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
