/*
 * fo.h -- C ABI of the GB300 fused compressed-optimizer library (libfo.so).
 *
 * The library implements the optimizer step of "FlashOptim: Optimizers for
 * Memory Efficient Training" (Gonzalez Ortiz et al., arXiv 2602.23349v1):
 *
 *   - weight splitting (page section "权重复分裂", Eq. 1-2, Algorithm 1): the
 *     FP32 master weight theta is held as a BF16 weight theta' plus a b-bit
 *     integer correction rho, the rounding error normalised by ULP(theta')/2;
 *   - companded state quantization (section "带压缩扩展的优化器状态量化",
 *     Algorithms 2-3): momentum m as INT8 codes of phi_m(m) = 2m/(1+|m|),
 *     second moment v as UINT8 codes of phi_v(v) = sqrt(v), in groups of 32
 *     elements with one FP16 scale per group;
 *   - the fused step (section "融合优化器步骤", Algorithm 4): dequantize m
 *     and v, rebuild theta, apply the standard AdamW / SGD / Lion update,
 *     requantize m and v and re-split theta, in one pass over memory.
 *
 * Exact arithmetic contract (what every entry point computes, bit for bit):
 *   theta' = BF16(theta), round to nearest even.
 *   h      = half the BF16 gap between theta' and its neighbour on theta's
 *            side (the usual ULP/2, halved again just below a power of two).
 *   rho    = rint(((theta - theta') / h) * Q), Q = 127 (8-bit) or 32767
 *            (16-bit); FP32 product, round half to even.
 *   theta^ = fma(rho * kappa, h, theta'), kappa = 1/Q rounded to FP32.
 *   group scale s = FP16(max |phi(x)|) (round to nearest even, capped at
 *            65504); code = clamp(rint(phi(x) * (L / s)), ...), L = 127 for m
 *            (codes -127..127) and 255 for v (codes 0..255); s = 0 gives codes 0.
 *   decode: m = z / (2 - |z|), z = code * (s / 127);  v = r * r, r = code * (s / 255).
 *   AdamW:  theta *= (1 - lr*wd); m = fma(b1, m, (1-b1)*g);
 *           v = fma(b2, v, ((1-b2)*g)*g);
 *           theta = fma(-lr/bc1, m / fma(sqrt(v), 1/sqrt(bc2), eps), theta),
 *           bc_i = 1 - b_i^t (t >= 1), b^t by repeated squaring in double.
 *   SGD:    m = fma(mu, m, fma(wd, theta, g)); theta = fma(-lr, m, theta).
 *   Lion:   c = fma(b1, m, (1-b1)*g); theta = fma(-lr, sign(c), theta*(1-lr*wd));
 *           m = fma(b2, m, (1-b2)*g).
 *   g is the row's gradient as FP32 (a BF16 gradient widened exactly).
 *   All arithmetic is IEEE binary32 round-to-nearest-even without flush to
 *   zero. Hyper-parameters are doubles; each per-element scalar is the
 *   hyper-parameter, or a quantity formed from them in double, rounded to FP32.
 *   The contract holds for finite inputs with |theta| below the largest BF16;
 *   NaN and infinity propagate into unspecified codes without a trap.
 *
 * Memory and ownership: every array argument is DEVICE memory owned by the
 * caller (for example torch tensors' data pointers). The library allocates no
 * device memory. Tables and hyper-parameter structs are HOST memory, read
 * only during the call (the table is copied into kernel parameters before the
 * call returns). To check a table for overlapping arrays, a step call sorts
 * the table's address ranges in a per-thread host array (16 bytes per array
 * of the largest table seen), kept until the thread exits; nothing else
 * persists between calls.
 *
 * Layout: element arrays are contiguous, one element per entry; each array
 * must start on a 16-byte boundary. Scale arrays hold ceil(numel/32) FP16
 * values (any 2-byte alignment); group k covers elements [32k, 32k+32) of its
 * tensor and the last group of a tensor may be partial.
 *
 * Streams and errors: all work is enqueued on `stream` (a cudaStream_t; NULL
 * is the legacy default stream) of the CURRENT device, and the calls return
 * without synchronizing. Argument errors are detected on the host before
 * anything is launched and return a non-zero fo_status_t. A CUDA error left
 * pending by earlier, unrelated work is read (and so cleared) before the
 * first launch and returned as FO_ERR_CUDA with nothing launched; a launch
 * that fails returns FO_ERR_CUDA (fo_last_cuda_error gives the cudaError_t).
 * A step table can need several launches (one per correction width and
 * gradient type, and per 384 rows): if one of them fails, the launches
 * before it stay enqueued, so the rows they cover are stepped and the others
 * are not -- do not simply retry such a call. Faults that happen later
 * surface at the caller's next synchronization. Nothing is thrown across the
 * ABI. Calls on distinct streams over disjoint buffers are independent and
 * thread-safe. State buffers are updated in place: an array that a call
 * writes may share no byte with any other array of the call (FO_ERR_ALIAS),
 * in the same table row or another; gradients are only read, so rows may
 * share one gradient array.
 */
#ifndef FO_H
#define FO_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. FO_OK is 0; every error is non-zero. */
typedef enum fo_status {
    FO_OK = 0,
    FO_ERR_NULL = 1,             /* a required pointer is NULL                  */
    FO_ERR_MISALIGNED = 2,       /* an element array is not 16-byte aligned     */
    FO_ERR_SIZE = 3,             /* a count is negative or too large            */
    FO_ERR_BAD_ARG = 4,          /* a flag or hyper-parameter is out of range   */
    FO_ERR_TOO_MANY_TENSORS = 5, /* ntensors exceeds FO_MAX_TENSORS             */
    FO_ERR_CUDA = 6,             /* a CUDA call failed (see fo_last_cuda_error) */
    FO_ERR_ALIAS = 7             /* a written array overlaps another array      */
} fo_status_t;

/* Kind of optimizer state coded by fo_quant_state / fo_dequant_state. */
typedef enum fo_state_kind {
    FO_STATE_MOMENTUM = 0,        /* INT8 codes (int8_t), phi_m companding   */
    FO_STATE_VARIANCE = 1,        /* UINT8 codes (uint8_t), phi_v companding */
    /* The same group quantization with phi the identity: the plain linear
     * quantizer that section "实验结果分析" (Fig. 4, Fig. 5) compares the
     * companded codecs against. For quality studies; the step never uses it. */
    FO_STATE_MOMENTUM_LINEAR = 2, /* INT8 codes of m itself                  */
    FO_STATE_VARIANCE_LINEAR = 3, /* UINT8 codes of v itself                 */
    /* FO_STATE_VARIANCE with an opt-in safety rule that the page does not
     * have (its Algorithm 3 "numerical stability" step is unprinted): in a
     * group with a non-zero scale s the codes are max(rint(.), 1), so every
     * decoded v there is at least (s/255)^2 and none is 0. A group whose
     * largest sqrt(v) rounds to an FP16 scale of 0 still stores codes 0.
     * Decoding is FO_STATE_VARIANCE's. */
    FO_STATE_VARIANCE_NONZERO = 5
} fo_state_kind_t;

#define FO_GROUP 32               /* elements per quantization group            */
#define FO_MAX_TENSORS (1 << 20)  /* rows per step call (split into launches)   */

/* A cudaStream_t passed through the ABI without CUDA headers. */
typedef void *fo_stream_t;

/*
 * Element type of a row's gradient. BF16 is the page's setting (the fused
 * step reads 2 bytes of gradient per parameter). FP32 serves callers whose
 * gradients are FP32 (for example accumulated in FP32): the FP32 value enters
 * the FP32 update as it is, with no rounding to BF16 first, at 2 more bytes
 * of reads per parameter.
 */
typedef enum fo_grad_dtype {
    FO_GRAD_BF16 = 0, /* grad holds uint16_t BF16 bit patterns */
    FO_GRAD_F32 = 1   /* grad holds float                      */
} fo_grad_dtype_t;

/*
 * One row of the multi-tensor parameter table: the compressed state of one
 * tensor of numel elements. All pointers are device memory.
 */
typedef struct fo_tensor {
    uint16_t *theta;       /* theta': BF16 bit patterns, numel, in/out                 */
    void *rho;             /* rho: int8_t (rho_bits 8) or int16_t (16), numel, in/out  */
    int8_t *m_q;           /* momentum codes, numel, in/out                            */
    uint16_t *m_scale;     /* FP16 momentum scales, ceil(numel/32), in/out             */
    uint8_t *v_q;          /* second-moment codes, numel, in/out (AdamW; else NULL)     */
    uint16_t *v_scale;     /* FP16 second-moment scales (AdamW; else NULL)              */
    const void *grad;      /* gradient, numel, read only; element type per grad_dtype  */
    int64_t numel;         /* elements; 0 skips the row                                */
    double weight_decay;   /* this tensor's weight decay (0 disables it)               */
    int32_t rho_bits;      /* 8 or 16                                                  */
    int32_t grad_dtype;    /* fo_grad_dtype_t: FO_GRAD_BF16 (0) or FO_GRAD_F32 (1)     */
} fo_tensor_t;

/* AdamW: lr > 0 finite, 0 <= beta < 1, eps > 0 (weight decay is per row).
 * flags: 0, or FO_ADAMW_V_NONZERO to requantize v with the rule of
 * FO_STATE_VARIANCE_NONZERO. Without it, an element whose sqrt(v) falls below
 * 1/510 of its group's scale decodes to v = 0, and the next step divides its
 * momentum by little more than its newest gradient's share of v (or by eps).
 * reserved must be 0. */
#define FO_ADAMW_V_NONZERO 1u
typedef struct fo_adamw_hparams {
    double lr, beta1, beta2, eps;
    uint32_t flags;
    uint32_t reserved;
} fo_adamw_hparams_t;
/* SGD with momentum, dampening 0, no Nesterov, L2 weight decay added to grad. */
typedef struct fo_sgd_hparams { double lr, momentum; } fo_sgd_hparams_t;
/* Lion (Chen et al. 2023) with decoupled weight decay. */
typedef struct fo_lion_hparams { double lr, beta1, beta2; } fo_lion_hparams_t;

/*
 * fo_split -- weight splitting, section "权重复分裂" (Eq. 1-2): from FP32
 * weights theta_f32[n] write theta'[n] (BF16) and rho[n] (int8_t or int16_t
 * per rho_bits). Used to initialise the compressed weights.
 * Errors: FO_ERR_NULL, FO_ERR_MISALIGNED, FO_ERR_SIZE (n < 0 or n > 2^46),
 * FO_ERR_BAD_ARG (rho_bits not 8 or 16), FO_ERR_ALIAS (an output overlaps
 * another array), FO_ERR_CUDA. n = 0 is a no-op.
 */
fo_status_t fo_split(const float *theta_f32, uint16_t *theta_bf16, void *rho, int64_t n,
                     int32_t rho_bits, fo_stream_t stream);

/*
 * fo_merge -- the inverse of fo_split, section "权重复分裂": rebuild
 * theta^[n] (FP32) from theta'[n] and rho[n]. Used to export FP32 weights.
 * Errors as fo_split.
 */
fo_status_t fo_merge(const uint16_t *theta_bf16, const void *rho, float *theta_f32, int64_t n,
                     int32_t rho_bits, fo_stream_t stream);

/*
 * fo_quant_state -- companded group quantization, section
 * "带压缩扩展的优化器状态量化" (Algorithm 2 for m, Algorithm 3 for v):
 * x[n] (FP32; v must be >= 0) -> codes q[n] (int8_t for the momentum kinds,
 * uint8_t for the variance kinds) and scales[ceil(n/32)] (FP16).
 * Errors: FO_ERR_NULL, FO_ERR_MISALIGNED, FO_ERR_SIZE (n < 0 or n > 2^46),
 * FO_ERR_BAD_ARG (kind), FO_ERR_ALIAS (an output overlaps another array),
 * FO_ERR_CUDA. n = 0 is a no-op.
 */
fo_status_t fo_quant_state(const float *x, void *q, uint16_t *scales, int64_t n,
                           fo_state_kind_t kind, fo_stream_t stream);

/*
 * fo_dequant_state -- the inverse of fo_quant_state (same section): codes and
 * scales -> x[n] (FP32). Errors as fo_quant_state.
 */
fo_status_t fo_dequant_state(const void *q, const uint16_t *scales, float *x, int64_t n,
                             fo_state_kind_t kind, fo_stream_t stream);

/*
 * fo_adamw_step -- one fused FlashAdamW step, section "融合优化器步骤"
 * (Algorithm 4), over `ntensors` rows of `table` (host array), step counter
 * `step` = t >= 1 (owned by the caller; it is the only state outside the
 * buffers, so a checkpoint is the buffers plus t). Every row needs theta, rho,
 * m_q, m_scale, v_q, v_scale and grad. Each byte of the state crosses device
 * memory once per call.
 * Errors: FO_ERR_NULL, FO_ERR_MISALIGNED, FO_ERR_SIZE (numel < 0, step < 1,
 * ntensors < 0), FO_ERR_TOO_MANY_TENSORS, FO_ERR_BAD_ARG (rho_bits,
 * grad_dtype, non-finite or out-of-range hyper-parameters), FO_ERR_ALIAS,
 * FO_ERR_CUDA. ntensors = 0 is a no-op. Rows of both correction widths and
 * both gradient types may be mixed in one table (one launch per combination
 * present).
 */
fo_status_t fo_adamw_step(const fo_tensor_t *table, int32_t ntensors,
                          const fo_adamw_hparams_t *hp, int64_t step, fo_stream_t stream);

/*
 * fo_adamw_step_dev -- fo_adamw_step with the step counter t read from
 * DEVICE memory when the kernel runs: step_dev points to one int64_t
 * (8-byte aligned, caller-owned) on the current device. The bias corrections
 * and the other step-dependent scalars are then derived on the device, with
 * the same double-precision expressions as fo_adamw_step, so the two calls
 * give identical results for the same t. This serves steps captured in a
 * CUDA graph: a replay reads the counter's value at that moment, where
 * fo_adamw_step would repeat the t it was captured with. The call does not
 * advance the counter; the caller does (for example with an increment
 * enqueued, or captured, before the call). If the counter holds a value below
 * 1 when the kernel runs, the launch updates nothing.
 * Errors: those of fo_adamw_step (without the step check), FO_ERR_NULL
 * (step_dev), FO_ERR_MISALIGNED (step_dev not 8-byte aligned).
 */
fo_status_t fo_adamw_step_dev(const fo_tensor_t *table, int32_t ntensors,
                              const fo_adamw_hparams_t *hp, const int64_t *step_dev,
                              fo_stream_t stream);

/*
 * fo_sgd_step -- one fused FlashSGD step (SGD with momentum and the same
 * compression; pages' sections "论文背景和研究动机" and "融合优化器步骤").
 * Rows need theta, rho, m_q, m_scale, grad; v_q and v_scale are ignored.
 * Errors as fo_adamw_step (without the step counter).
 */
fo_status_t fo_sgd_step(const fo_tensor_t *table, int32_t ntensors, const fo_sgd_hparams_t *hp,
                        fo_stream_t stream);

/*
 * fo_lion_step -- one fused FlashLion step (Lion with the same compression;
 * same sections). Rows need theta, rho, m_q, m_scale, grad; v_q and v_scale
 * are ignored. Errors as fo_sgd_step.
 */
fo_status_t fo_lion_step(const fo_tensor_t *table, int32_t ntensors,
                         const fo_lion_hparams_t *hp, fo_stream_t stream);

/*
 * fo_verify_fast_arithmetic -- the fused step (section "融合优化器步骤")
 * must leave exactly the state the IEEE operations of the contract above
 * give. Its fast path builds division and square root from the GPU's
 * reciprocal and reciprocal-square-root approximations, whose exact results
 * the instruction set leaves open; each sequence is exact on a one-variable
 * or finite operand domain given the approximation's behaviour. This call
 * enumerates every such domain on the CURRENT device, running the step's own
 * device functions, and counts the operands whose result differs from the
 * IEEE operation (both signs where the domain is signed):
 *   counts[0]  refined reciprocal vs RN(1/b), every b in [2^-100, 2^100]
 *   counts[1]  square root vs RN(sqrt(v)), every v in [2^-100, 2^126] and 0
 *   counts[2]  phi_m division of AdamW (m scaled by 2^32), every |m'| in
 *              [2^-62, 2^85]
 *   counts[3]  phi_m division of SGD and Lion, every |m| in [2^-100, 2^100]
 *   counts[4]  momentum decoding phi_m^-1(code * s/127), every code byte
 *              under every FP16 scale below 127/64
 *   counts[5]  127/s, 255/s, s/127 and s/255, every positive finite FP16 s
 * All are 0 where the fast path is exact. `counts`: DEVICE memory of
 * FO_VERIFY_COUNTS uint64 entries (8-byte aligned) owned by the caller,
 * overwritten; the work (about 7e9 evaluations) is enqueued on `stream`.
 * Errors: FO_ERR_NULL, FO_ERR_MISALIGNED, FO_ERR_CUDA.
 */
#define FO_VERIFY_COUNTS 6
fo_status_t fo_verify_fast_arithmetic(uint64_t *counts, fo_stream_t stream);

/* A static, human-readable name for a status code (never NULL). */
const char *fo_status_string(fo_status_t status);

/* The cudaError_t (as int) behind the last FO_ERR_CUDA on this thread, or 0. */
int fo_last_cuda_error(void);

/*
 * Launch accounting for measurements: the number of kernels this library has
 * launched in the calling process so far (all threads).
 */
uint64_t fo_kernel_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* FO_H */
