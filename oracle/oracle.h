/*
 * oracle.h -- declarations of the CPU oracle for the FlashOptim compressed
 * optimizer step.
 *
 * TEST INFRASTRUCTURE. The oracle is a plain, slow, scalar restatement of
 * "FlashOptim: Optimizers for Memory Efficient Training" (arXiv 2602.23349v1)
 * used only by the test suite, the smoke check and the benchmark's CPU
 * baseline. The product library never includes this header or links this code.
 *
 * All buffers are host memory owned by the caller. Every function is
 * synchronous and single-threaded. Arithmetic is IEEE-754 binary32 with
 * round-to-nearest-even; see oracle.c for the exact expression order.
 */
#ifndef FO_ORACLE_H
#define FO_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORACLE_GROUP 32 /* quantization group size G ("companded state quantization" section) */

/* state kinds: the companded codecs of the method, and the same group
 * quantization without companding (the ablation the page compares against in
 * Fig. 4 and Fig. 5): odd kinds are unsigned (second moment), even signed */
enum { ORACLE_MOMENTUM = 0, ORACLE_VARIANCE = 1, ORACLE_MOMENTUM_LINEAR = 2, ORACLE_VARIANCE_LINEAR = 3,
       /* the second-moment codec with the opt-in safety rule: in a group
        * with a non-zero scale the codes are max(rint(.), 1), so no v there
        * decodes to 0 */
       ORACLE_VARIANCE_NONZERO = 5 };

/* One row of the parameter table: the compressed state of one tensor. */
typedef struct oracle_tensor {
    uint16_t *theta;        /* theta': BF16 bit patterns, numel, in/out          */
    void *rho;              /* rho: int8 (rho_bits 8) or int16 (16), numel        */
    int8_t *m_q;            /* momentum codes, numel                              */
    uint16_t *m_scale;      /* FP16 momentum group scales, ceil(numel/32)         */
    uint8_t *v_q;           /* second-moment codes, numel (AdamW only)            */
    uint16_t *v_scale;      /* FP16 second-moment group scales (AdamW only)       */
    const void *grad;       /* gradient, numel, read only: BF16 bit patterns
                               (uint16_t), or float when grad_is_f32 is 1      */
    int64_t numel;
    double weight_decay;
    int32_t rho_bits;
    int32_t grad_is_f32;    /* 0: BF16 gradient; 1: FP32 gradient, used as is  */
} oracle_tensor_t;

/* Hyper-parameters are doubles (as Python floats are); the per-element
 * arithmetic uses them rounded to FP32, and derived scalars are formed in
 * double and rounded once. */
/* v_nonzero = 1 requantizes v with ORACLE_VARIANCE_NONZERO (opt-in safety rule) */
typedef struct { double lr, beta1, beta2, eps; int32_t v_nonzero, pad; } oracle_adamw_hparams_t;
typedef struct { double lr, momentum; } oracle_sgd_hparams_t;
typedef struct { double lr, beta1, beta2; } oracle_lion_hparams_t;

/* number encodings */
float oracle_bf16_to_f32(uint16_t b);
uint16_t oracle_bf16_rne(float x);
uint16_t oracle_fp16_rne(float x);
float oracle_fp16_to_f32(uint16_t h);
float oracle_half_ulp(uint16_t theta_p, int dir);

/* array forms of the encodings (which: 0 phi_m, 1 phi_m^-1, 2 phi_v, 3 phi_v^-1) */
void oracle_bf16_rne_n(const float *x, uint16_t *out, int64_t n);
void oracle_fp16_rne_n(const float *x, uint16_t *out, int64_t n);
void oracle_fp16_to_f32_n(const uint16_t *h, float *out, int64_t n);
void oracle_half_ulp_n(const uint16_t *theta_p, int dir, float *out, int64_t n);
void oracle_phi_n(const float *x, float *out, int64_t n, int which);

/* companding functions */
float oracle_phi_m(float x);
float oracle_phi_m_inv(float z);
float oracle_phi_v(float x);
float oracle_phi_v_inv(float z);

/* weight splitting */
void oracle_split(const float *theta, uint16_t *theta_p, void *rho, int64_t n, int rho_bits);
void oracle_merge(const uint16_t *theta_p, const void *rho, float *theta, int64_t n, int rho_bits);

/* group quantization of one state tensor (kind: one of the ORACLE_* state kinds) */
void oracle_quant_state(const float *x, void *q, uint16_t *scales, int64_t n, int kind);
void oracle_dequant_state(const void *q, const uint16_t *scales, float *x, int64_t n, int kind);

/* fused compressed steps over a table; return 0, or -1 on a bad argument */
int oracle_adamw_step(const oracle_tensor_t *table, int32_t ntensors,
                      const oracle_adamw_hparams_t *hp, int64_t step);
int oracle_sgd_step(const oracle_tensor_t *table, int32_t ntensors,
                    const oracle_sgd_hparams_t *hp);
int oracle_lion_step(const oracle_tensor_t *table, int32_t ntensors,
                     const oracle_lion_hparams_t *hp);

/* the same element updates on uncompressed FP32 state (codecs bypassed) */
void oracle_adamw_update_fp32(float *theta, float *m, float *v, const float *g, int64_t n,
                              const oracle_adamw_hparams_t *hp, int64_t step, double weight_decay);
void oracle_sgd_update_fp32(float *theta, float *m, const float *g, int64_t n,
                            const oracle_sgd_hparams_t *hp, double weight_decay);
void oracle_lion_update_fp32(float *theta, float *m, const float *g, int64_t n,
                             const oracle_lion_hparams_t *hp, double weight_decay);

#ifdef __cplusplus
}
#endif
#endif
