/*
 * oracle.c -- CPU oracle for the FlashOptim compressed optimizer step.
 *
 * TEST INFRASTRUCTURE ONLY: a plain, slow, scalar restatement of what the GPU
 * path computes. Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg load it. It shares no code, header, table or constant with
 * the CUDA library, and neither side calls the other.
 *
 * Source: "FlashOptim: Optimizers for Memory Efficient Training"
 * (Gonzalez Ortiz et al., arXiv 2602.23349v1), as summarised on its web page:
 *   - section "权重复分裂" (weight splitting; Eq. 1-2, Algorithm 1):
 *     the FP32 master weight theta is stored as a BF16 weight theta' and an
 *     integer correction rho, the error theta - theta' normalised by
 *     ULP(theta')/2 and quantized uniformly to b bits;
 *   - section "带压缩扩展的优化器状态量化" (companded state quantization;
 *     Algorithms 2-3): phi_m(x) = 2x/(1+|x|), phi_m^-1(z) = z/(2-|z|),
 *     phi_v(x) = sqrt(x), phi_v^-1(z) = z^2, groups of G = 32, one FP16 scale
 *     per group, momentum as INT8, second moment as UINT8;
 *   - section "融合优化器步骤" (fused step; Algorithm 4): dequantize m and v,
 *     rebuild the master weight, apply the standard optimizer update,
 *     requantize the state and re-split the weight.
 * The page prints none of the algorithms; the readings taken where it is
 * silent are stated beside each function.
 *
 * Arithmetic: IEEE-754 binary32, round-to-nearest-even, no flush-to-zero,
 * no implicit contraction (build with -ffp-contract=off). Where the
 * definition below uses a fused multiply-add it is written as fmaf().
 * Hyper-parameters arrive as doubles; each scalar used per element is the
 * hyper-parameter, or a quantity derived from them in double, rounded once to
 * FP32 (as PyTorch's optimizers do with Python-float hyper-parameters).
 * Inputs are assumed finite; NaN or infinite inputs give unspecified codes.
 */
#include "oracle.h"

#include <math.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Bit views                                                                 */
/* ------------------------------------------------------------------------ */

static float f32_from_bits(uint32_t u)
{
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static uint32_t bits_of_f32(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return u;
}

/* ------------------------------------------------------------------------ */
/* BF16 and FP16                                                             */
/* ------------------------------------------------------------------------ */

/* A BF16 value is the upper half of the FP32 with the same bits. */
float oracle_bf16_to_f32(uint16_t b)
{
    return f32_from_bits((uint32_t)b << 16);
}

/* Value of a BF16 pattern for distance comparisons; the pattern past the
 * largest finite magnitude stands for 2^128, as IEEE rounding treats overflow. */
static double bf16_value_unbounded(uint16_t b)
{
    if ((b & 0x7FFFu) == 0x7F80u)
        return (b & 0x8000u) ? -ldexp(1.0, 128) : ldexp(1.0, 128);
    return (double)oracle_bf16_to_f32(b);
}

/*
 * FP32 -> BF16, round to nearest, ties to even. x lies between the BF16
 * value obtained by dropping its low 16 bits (toward zero) and the next BF16
 * value away from zero; the nearer one is returned, and on a tie the one with
 * an even last mantissa bit.
 */
uint16_t oracle_bf16_rne(float x)
{
    uint32_t u = bits_of_f32(x);
    if (isnan(x))
        return (uint16_t)((u >> 16) | 0x0040u);
    uint16_t toward_zero = (uint16_t)(u >> 16);
    if ((u & 0xFFFFu) == 0)
        return toward_zero;
    uint16_t away = (uint16_t)(toward_zero + 1u);
    double d_tz = fabs((double)x - bf16_value_unbounded(toward_zero));
    double d_aw = fabs(bf16_value_unbounded(away) - (double)x);
    if (d_tz < d_aw)
        return toward_zero;
    if (d_aw < d_tz)
        return away;
    return (toward_zero & 1u) ? away : toward_zero;
}

/*
 * FP32 -> FP16 (IEEE binary16), round to nearest, ties to even, with
 * gradual underflow. The FP16 grid in the binade 2^E (E >= -14; below that
 * the subnormal grid continues with the same spacing) has spacing 2^(E-10);
 * |x| is rounded on that grid in double precision, where every step is exact.
 */
uint16_t oracle_fp16_rne(float x)
{
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x))
        return (uint16_t)(sign | 0x7E00u);
    double a = fabs((double)x);
    if (a >= 65520.0) /* 65504 + half a spacing: rounds to infinity */
        return (uint16_t)(sign | 0x7C00u);
    if (a == 0.0)
        return sign;
    int e2;
    (void)frexp(a, &e2); /* a = f * 2^e2, f in [0.5, 1): binade exponent e2-1 */
    int E = e2 - 1;
    if (E < -14)
        E = -14;
    double spacing = ldexp(1.0, E - 10);
    double r = rint(a / spacing) * spacing;
    if (r < ldexp(1.0, -14)) /* subnormal or zero: count of 2^-24 steps */
        return (uint16_t)(sign | (uint16_t)(r / ldexp(1.0, -24)));
    (void)frexp(r, &e2);
    E = e2 - 1;
    double frac = r / ldexp(1.0, E) - 1.0; /* in [0, 1), a multiple of 2^-10 */
    return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)(frac * 1024.0));
}

float oracle_fp16_to_f32(uint16_t h)
{
    int negative = (h & 0x8000u) != 0;
    int E = (h >> 10) & 0x1F;
    int M = h & 0x3FF;
    double v;
    if (E == 31)
        v = M ? NAN : INFINITY;
    else if (E == 0)
        v = ldexp((double)M, -24);
    else
        v = ldexp((double)(1024 + M), E - 25);
    return (float)(negative ? -v : v);
}

/* ------------------------------------------------------------------------ */
/* ULP(theta')/2                                                             */
/* ------------------------------------------------------------------------ */

/* The BF16 pattern adjacent to b on side dir (+1: toward +inf, -1: toward -inf). */
static uint16_t bf16_adjacent(uint16_t b, int dir)
{
    int negative = (b & 0x8000u) != 0;
    if ((b & 0x7FFFu) == 0)
        return dir > 0 ? 0x0001u : 0x8001u;
    int away_from_zero = (dir > 0) != negative;
    return away_from_zero ? (uint16_t)(b + 1u) : (uint16_t)(b - 1u);
}

/*
 * Half the gap between theta' and its BF16 neighbour on side dir.
 *
 * The weight-splitting section bounds theta to
 * [theta' - ULP(theta')/2, theta' + ULP(theta')/2] under round-to-nearest.
 * Reading taken: ULP is the BF16 gap on the side where theta lies. It equals
 * the usual ULP except below an exact power of two, where the gap is half as
 * large; with it the normalised error fills [-1, 1] on both sides, and the
 * 16-bit correction reproduces the page's 99.92 % bit-exact reconstruction
 * (Fig. 3), which the symmetric ULP does not (99.73 %).
 */
float oracle_half_ulp(uint16_t theta_p, int dir)
{
    /* Past the largest finite BF16 the next value is taken as 2^128, as IEEE
     * rounding treats overflow (unbounded exponent), so the gap stays 2^120. */
    double a = bf16_value_unbounded(theta_p);
    double b = bf16_value_unbounded(bf16_adjacent(theta_p, dir));
    return (float)(fabs(b - a) * 0.5); /* neighbours: exact in double, and a power of two */
}

/* ------------------------------------------------------------------------ */
/* Companding (Algorithms 2-3)                                               */
/* ------------------------------------------------------------------------ */

float oracle_phi_m(float x) { return (x + x) / (1.0f + fabsf(x)); }
float oracle_phi_m_inv(float z) { return z / (2.0f - fabsf(z)); }
float oracle_phi_v(float x) { return sqrtf(x); }
float oracle_phi_v_inv(float z) { return z * z; }

/* ------------------------------------------------------------------------ */
/* Weight splitting (Eq. 1-2, Algorithm 1)                                   */
/* ------------------------------------------------------------------------ */

/* Q_rho = 2^(b-1) - 1: symmetric levels, so e = +-1 (a rounding tie) fits. */
static int32_t rho_levels(int rho_bits) { return rho_bits == 16 ? 32767 : 127; }

static int32_t rho_load(const void *rho, int64_t i, int rho_bits)
{
    return rho_bits == 16 ? (int32_t)((const int16_t *)rho)[i] : (int32_t)((const int8_t *)rho)[i];
}

static void rho_store(void *rho, int64_t i, int rho_bits, int32_t r)
{
    if (rho_bits == 16)
        ((int16_t *)rho)[i] = (int16_t)r;
    else
        ((int8_t *)rho)[i] = (int8_t)r;
}

/*
 * Split one FP32 weight: theta' = BF16(theta) (round to nearest even), the
 * error e = (theta - theta') / h with h = ULP(theta')/2 on theta's side
 * (|e| <= 1; the subtraction and the division are exact), and
 * rho = rint(e * Q_rho), clamped to [-Q_rho, Q_rho].
 */
static void split_one(float theta, int rho_bits, uint16_t *theta_p, int32_t *rho)
{
    const float Q = (float)rho_levels(rho_bits);
    uint16_t b = oracle_bf16_rne(theta);
    float base = oracle_bf16_to_f32(b);
    float d = theta - base;
    float h = oracle_half_ulp(b, d < 0.0f ? -1 : +1);
    float e = d / h;
    float r = rintf(e * Q);
    if (r > Q)
        r = Q;
    if (r < -Q)
        r = -Q;
    *theta_p = b;
    *rho = (int32_t)r;
}

/*
 * Rebuild theta^ = theta' + (rho / Q_rho) * h, with h = ULP(theta')/2 on the
 * side that the sign of rho names. rho / Q_rho is evaluated as rho * kappa
 * with kappa = 1/Q_rho rounded to FP32; the product with h and the sum are
 * rounded once (fmaf).
 */
static float merge_one(uint16_t theta_p, int32_t rho, int rho_bits)
{
    const float kappa = 1.0f / (float)rho_levels(rho_bits);
    float base = oracle_bf16_to_f32(theta_p);
    float h = oracle_half_ulp(theta_p, rho < 0 ? -1 : +1);
    float e = (float)rho * kappa;
    return fmaf(e, h, base);
}

void oracle_split(const float *theta, uint16_t *theta_p, void *rho, int64_t n, int rho_bits)
{
    for (int64_t i = 0; i < n; ++i) {
        int32_t r;
        split_one(theta[i], rho_bits, &theta_p[i], &r);
        rho_store(rho, i, rho_bits, r);
    }
}

void oracle_merge(const uint16_t *theta_p, const void *rho, float *theta, int64_t n, int rho_bits)
{
    for (int64_t i = 0; i < n; ++i)
        theta[i] = merge_one(theta_p[i], rho_load(rho, i, rho_bits), rho_bits);
}

/* ------------------------------------------------------------------------ */
/* Group quantization (Algorithms 2-3)                                       */
/* ------------------------------------------------------------------------ */

/*
 * Readings taken where the page is silent:
 *  - the FP16 scale s stored for a group is the largest |phi(x)| in the group
 *    (rounded to nearest even, capped at the largest finite FP16), so a code
 *    q decodes to q * s / Q_state, Q_state = 127 (INT8 momentum) or 255
 *    (UINT8 second moment);
 *  - codes are rint(phi(x) * (Q_state / s)), clamped to [-127, 127] or
 *    [0, 255]; a group whose scale is 0 stores all codes 0;
 *  - groups are 32 consecutive elements of one tensor; the last group of a
 *    tensor holds the remaining numel mod 32 elements.
 * The linear kinds are the same steps with phi the identity (Fig. 4's plain
 * group-wise linear quantization).
 */

/* phi of a state kind (identity for the linear kinds) */
static float compand(float x, int kind)
{
    switch (kind) {
    case ORACLE_MOMENTUM: return oracle_phi_m(x);
    case ORACLE_VARIANCE:
    case ORACLE_VARIANCE_NONZERO: return oracle_phi_v(x);
    default: return x;
    }
}

static float expand(float z, int kind)
{
    switch (kind) {
    case ORACLE_MOMENTUM: return oracle_phi_m_inv(z);
    case ORACLE_VARIANCE:
    case ORACLE_VARIANCE_NONZERO: return oracle_phi_v_inv(z);
    default: return z;
    }
}

static int kind_signed(int kind) { return kind == ORACLE_MOMENTUM || kind == ORACLE_MOMENTUM_LINEAR; }
static void quant_group(const float *x, int len, int kind, void *q, uint16_t *scale)
{
    float c[ORACLE_GROUP];
    float a = 0.0f;
    for (int i = 0; i < len; ++i) {
        c[i] = compand(x[i], kind);
        if (fabsf(c[i]) > a)
            a = fabsf(c[i]);
    }
    uint16_t s = oracle_fp16_rne(fminf(a, 65504.0f));
    float sf = oracle_fp16_to_f32(s);
    *scale = s;
    const float levels = kind_signed(kind) ? 127.0f : 255.0f;
    const float lo = kind_signed(kind) ? -127.0f : 0.0f;
    float inv = sf == 0.0f ? 0.0f : levels / sf;
    for (int i = 0; i < len; ++i) {
        float code = 0.0f;
        if (sf != 0.0f && !isnan(c[i])) {
            code = rintf(c[i] * inv);
            if (code > levels)
                code = levels;
            if (code < lo)
                code = lo;
            /* opt-in safety rule: in a group with a non-zero scale no code is
             * 0, so no second moment there decodes to 0 (v^ >= (s/255)^2) */
            if (kind == ORACLE_VARIANCE_NONZERO && code < 1.0f)
                code = 1.0f;
        }
        if (kind_signed(kind))
            ((int8_t *)q)[i] = (int8_t)code;
        else
            ((uint8_t *)q)[i] = (uint8_t)code;
    }
}

static void dequant_group(const void *q, uint16_t scale, int len, int kind, float *x)
{
    float sf = oracle_fp16_to_f32(scale);
    float step = sf / (kind_signed(kind) ? 127.0f : 255.0f);
    for (int i = 0; i < len; ++i) {
        float code = kind_signed(kind) ? (float)((const int8_t *)q)[i] : (float)((const uint8_t *)q)[i];
        x[i] = expand(code * step, kind);
    }
}

void oracle_quant_state(const float *x, void *q, uint16_t *scales, int64_t n, int kind)
{
    for (int64_t g0 = 0; g0 < n; g0 += ORACLE_GROUP) {
        int len = (int)(n - g0 < ORACLE_GROUP ? n - g0 : ORACLE_GROUP);
        quant_group(x + g0, len, kind, (char *)q + g0, &scales[g0 / ORACLE_GROUP]);
    }
}

void oracle_dequant_state(const void *q, const uint16_t *scales, float *x, int64_t n, int kind)
{
    for (int64_t g0 = 0; g0 < n; g0 += ORACLE_GROUP) {
        int len = (int)(n - g0 < ORACLE_GROUP ? n - g0 : ORACLE_GROUP);
        dequant_group((const char *)q + g0, scales[g0 / ORACLE_GROUP], len, kind,
                      x + g0);
    }
}

/* ------------------------------------------------------------------------ */
/* Optimizer updates ("standard" semantics, fused step section)              */
/* ------------------------------------------------------------------------ */

/* beta^t by repeated squaring in double (deterministic, no libm). */
static double pow_int(double b, int64_t t)
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

static float decay_factor(double lr, double weight_decay)
{
    return (float)(1.0 - lr * weight_decay);
}

typedef struct {
    float beta1, beta2, c1, c2, eps, step_size, inv_sqrt_bc2;
} adamw_consts_t;

/* Bias corrections bc_i = 1 - beta_i^t (t >= 1) of AdamW. */
static adamw_consts_t adamw_consts(const oracle_adamw_hparams_t *hp, int64_t step)
{
    adamw_consts_t k;
    double bc1 = 1.0 - pow_int(hp->beta1, step);
    double bc2 = 1.0 - pow_int(hp->beta2, step);
    k.beta1 = (float)hp->beta1;
    k.beta2 = (float)hp->beta2;
    k.c1 = (float)(1.0 - hp->beta1);
    k.c2 = (float)(1.0 - hp->beta2);
    k.eps = (float)hp->eps;
    k.step_size = (float)(hp->lr / bc1);
    k.inv_sqrt_bc2 = (float)(1.0 / sqrt(bc2));
    return k;
}

/*
 * AdamW (decoupled weight decay, bias-corrected moments, eps added after the
 * bias-corrected square root), one element:
 *   theta <- theta * (1 - lr*wd)
 *   m     <- beta1*m + (1-beta1)*g
 *   v     <- beta2*v + (1-beta2)*g*g
 *   theta <- theta - (lr/bc1) * m / (sqrt(v)/sqrt(bc2) + eps)
 */
static void adamw_element(float *theta, float *m, float *v, float g, const adamw_consts_t *k,
                          float decay)
{
    float th = *theta * decay;
    float mm = fmaf(k->beta1, *m, k->c1 * g);
    float vv = fmaf(k->beta2, *v, (k->c2 * g) * g);
    float den = fmaf(sqrtf(vv), k->inv_sqrt_bc2, k->eps);
    *theta = fmaf(-k->step_size, mm / den, th);
    *m = mm;
    *v = vv;
}

/*
 * SGD with momentum (dampening 0, no Nesterov, L2 weight decay added to the
 * gradient), one element:
 *   g' <- g + wd*theta ;  m <- mu*m + g' ;  theta <- theta - lr*m
 */
static void sgd_element(float *theta, float *m, float g, float lr, float mu, float weight_decay)
{
    float gp = fmaf(weight_decay, *theta, g);
    float mm = fmaf(mu, *m, gp);
    *theta = fmaf(-lr, mm, *theta);
    *m = mm;
}

typedef struct {
    float lr, beta1, beta2, c1, c2;
} lion_consts_t;

static lion_consts_t lion_consts(const oracle_lion_hparams_t *hp)
{
    lion_consts_t k;
    k.lr = (float)hp->lr;
    k.beta1 = (float)hp->beta1;
    k.beta2 = (float)hp->beta2;
    k.c1 = (float)(1.0 - hp->beta1);
    k.c2 = (float)(1.0 - hp->beta2);
    return k;
}

/*
 * Lion (Chen et al., "Symbolic Discovery of Optimization Algorithms"), one
 * element, decoupled weight decay:
 *   c <- beta1*m + (1-beta1)*g
 *   theta <- theta*(1 - lr*wd) - lr*sign(c)      (sign(0) = 0)
 *   m <- beta2*m + (1-beta2)*g
 */
static void lion_element(float *theta, float *m, float g, const lion_consts_t *k, float decay)
{
    float c = fmaf(k->beta1, *m, k->c1 * g);
    float sgn = c > 0.0f ? 1.0f : (c < 0.0f ? -1.0f : 0.0f);
    float th = *theta * decay;
    *theta = fmaf(-k->lr, sgn, th);
    *m = fmaf(k->beta2, *m, k->c2 * g);
}

void oracle_adamw_update_fp32(float *theta, float *m, float *v, const float *g, int64_t n,
                              const oracle_adamw_hparams_t *hp, int64_t step, double weight_decay)
{
    adamw_consts_t k = adamw_consts(hp, step);
    float decay = decay_factor(hp->lr, weight_decay);
    for (int64_t i = 0; i < n; ++i)
        adamw_element(&theta[i], &m[i], &v[i], g[i], &k, decay);
}

void oracle_sgd_update_fp32(float *theta, float *m, const float *g, int64_t n,
                            const oracle_sgd_hparams_t *hp, double weight_decay)
{
    for (int64_t i = 0; i < n; ++i)
        sgd_element(&theta[i], &m[i], g[i], (float)hp->lr, (float)hp->momentum, (float)weight_decay);
}

void oracle_lion_update_fp32(float *theta, float *m, const float *g, int64_t n,
                             const oracle_lion_hparams_t *hp, double weight_decay)
{
    lion_consts_t k = lion_consts(hp);
    float decay = decay_factor(hp->lr, weight_decay);
    for (int64_t i = 0; i < n; ++i)
        lion_element(&theta[i], &m[i], g[i], &k, decay);
}

/* ------------------------------------------------------------------------ */
/* Fused compressed steps (Algorithm 4)                                      */
/* ------------------------------------------------------------------------ */

enum { OPT_ADAMW, OPT_SGD, OPT_LION };

typedef struct {
    int opt;
    int v_kind;   /* ORACLE_VARIANCE, or ORACLE_VARIANCE_NONZERO (AdamW's opt-in rule) */
    adamw_consts_t adamw;
    lion_consts_t lion;
    double lr;
    float lr_f, mu;
} step_consts_t;

static int row_ok(const oracle_tensor_t *t, int opt)
{
    if (t->numel < 0 || (t->rho_bits != 8 && t->rho_bits != 16))
        return 0;
    if (t->grad_is_f32 != 0 && t->grad_is_f32 != 1)
        return 0;
    if (t->numel == 0)
        return 1;
    if (!t->theta || !t->rho || !t->m_q || !t->m_scale || !t->grad)
        return 0;
    if (opt == OPT_ADAMW && (!t->v_q || !t->v_scale))
        return 0;
    return 1;
}

/*
 * One group of one tensor: dequantize m (and v), rebuild theta, update in
 * FP32, re-split theta, requantize m (and v) from the updated FP32 values.
 */
static void step_group(const oracle_tensor_t *t, int64_t g0, int len, const step_consts_t *k)
{
    float theta[ORACLE_GROUP], m[ORACLE_GROUP], v[ORACLE_GROUP];
    int64_t gi = g0 / ORACLE_GROUP;

    for (int i = 0; i < len; ++i)
        theta[i] = merge_one(t->theta[g0 + i], rho_load(t->rho, g0 + i, t->rho_bits), t->rho_bits);
    dequant_group(t->m_q + g0, t->m_scale[gi], len, ORACLE_MOMENTUM, m);
    if (k->opt == OPT_ADAMW)
        dequant_group(t->v_q + g0, t->v_scale[gi], len, ORACLE_VARIANCE, v);

    for (int i = 0; i < len; ++i) {
        /* the update is FP32: a BF16 gradient is widened, an FP32 one taken as is */
        float g = t->grad_is_f32 ? ((const float *)t->grad)[g0 + i]
                                 : oracle_bf16_to_f32(((const uint16_t *)t->grad)[g0 + i]);
        if (k->opt == OPT_ADAMW)
            adamw_element(&theta[i], &m[i], &v[i], g, &k->adamw,
                          decay_factor(k->lr, t->weight_decay));
        else if (k->opt == OPT_SGD)
            sgd_element(&theta[i], &m[i], g, k->lr_f, k->mu, (float)t->weight_decay);
        else
            lion_element(&theta[i], &m[i], g, &k->lion, decay_factor(k->lr, t->weight_decay));
    }

    for (int i = 0; i < len; ++i) {
        int32_t r;
        split_one(theta[i], t->rho_bits, &t->theta[g0 + i], &r);
        rho_store(t->rho, g0 + i, t->rho_bits, r);
    }
    quant_group(m, len, ORACLE_MOMENTUM, t->m_q + g0, &t->m_scale[gi]);
    if (k->opt == OPT_ADAMW)
        quant_group(v, len, k->v_kind, t->v_q + g0, &t->v_scale[gi]);
}

static int run_step(const oracle_tensor_t *table, int32_t ntensors, const step_consts_t *k)
{
    if (ntensors < 0 || (ntensors > 0 && !table))
        return -1;
    for (int32_t j = 0; j < ntensors; ++j)
        if (!row_ok(&table[j], k->opt))
            return -1;
    for (int32_t j = 0; j < ntensors; ++j) {
        const oracle_tensor_t *t = &table[j];
        for (int64_t g0 = 0; g0 < t->numel; g0 += ORACLE_GROUP) {
            int len = (int)(t->numel - g0 < ORACLE_GROUP ? t->numel - g0 : ORACLE_GROUP);
            step_group(t, g0, len, k);
        }
    }
    return 0;
}

int oracle_adamw_step(const oracle_tensor_t *table, int32_t ntensors,
                      const oracle_adamw_hparams_t *hp, int64_t step)
{
    if (!hp || step < 1)
        return -1;
    step_consts_t k;
    memset(&k, 0, sizeof k);
    if (hp->v_nonzero != 0 && hp->v_nonzero != 1)
        return -1;
    k.opt = OPT_ADAMW;
    k.v_kind = hp->v_nonzero ? ORACLE_VARIANCE_NONZERO : ORACLE_VARIANCE;
    k.adamw = adamw_consts(hp, step);
    k.lr = hp->lr;
    return run_step(table, ntensors, &k);
}

int oracle_sgd_step(const oracle_tensor_t *table, int32_t ntensors, const oracle_sgd_hparams_t *hp)
{
    if (!hp)
        return -1;
    step_consts_t k;
    memset(&k, 0, sizeof k);
    k.opt = OPT_SGD;
    k.lr = hp->lr;
    k.lr_f = (float)hp->lr;
    k.mu = (float)hp->momentum;
    return run_step(table, ntensors, &k);
}

int oracle_lion_step(const oracle_tensor_t *table, int32_t ntensors,
                     const oracle_lion_hparams_t *hp)
{
    if (!hp)
        return -1;
    step_consts_t k;
    memset(&k, 0, sizeof k);
    k.opt = OPT_LION;
    k.lion = lion_consts(hp);
    k.lr = hp->lr;
    return run_step(table, ntensors, &k);
}

/* ------------------------------------------------------------------------ */
/* Array forms of the scalar encodings, for exhaustive checks                */
/* ------------------------------------------------------------------------ */

void oracle_bf16_rne_n(const float *x, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_bf16_rne(x[i]);
}

void oracle_fp16_rne_n(const float *x, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_fp16_rne(x[i]);
}

void oracle_fp16_to_f32_n(const uint16_t *h, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_fp16_to_f32(h[i]);
}

void oracle_half_ulp_n(const uint16_t *theta_p, int dir, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_half_ulp(theta_p[i], dir);
}

void oracle_phi_n(const float *x, float *out, int64_t n, int which)
{
    for (int64_t i = 0; i < n; ++i) {
        switch (which) {
        case 0: out[i] = oracle_phi_m(x[i]); break;
        case 1: out[i] = oracle_phi_m_inv(x[i]); break;
        case 2: out[i] = oracle_phi_v(x[i]); break;
        default: out[i] = oracle_phi_v_inv(x[i]); break;
        }
    }
}
