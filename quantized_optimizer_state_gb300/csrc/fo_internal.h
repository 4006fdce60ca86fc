// fo_internal.h -- interface between the C-ABI layer (fo_api.cu) and the
// kernels (fo_step.cu, fo_codecs.cu). Not installed; not part of the ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace fo {

constexpr int kGroup = 32;           // quantization group (page: G = 32)
constexpr int kElemsPerThread = 16;  // one thread holds half a group
#ifndef FO_STEP_THREADS
#define FO_STEP_THREADS 256
#endif
constexpr int kStepThreads = FO_STEP_THREADS;
constexpr int kStepChunk = kStepThreads * kElemsPerThread;  // 4096 elements
// A tile is `chunks` consecutive chunks of one row, stepped by one CTA one
// after the other (they share the row lookup and per-row constants). The
// kernel is compiled for kLongChunks, kShortChunks and kTinyChunks chunks per
// tile; the host takes the long tiles when they still give every resident CTA
// at least kMinTilesPerCta tiles (large tables), the short ones otherwise,
// and one-chunk tiles when short ones would leave CTAs without a tile (tables
// of a few million elements, whose step is latency: more CTAs at work).
constexpr int kLongChunks = 8;
constexpr int kShortChunks = 2;
constexpr int kTinyChunks = 1;
constexpr int kMinTilesPerCta = 6;   // 8 and 6 tie on the large tables; GPT-2 small is 1 % faster on long tiles


enum class Opt : int { kAdamW = 0, kSgd = 1, kLion = 2 };

// Resident CTAs per SM each step kernel is built for (256 threads each), by
// measurement. AdamW with 8-bit rho and BF16 gradients runs 4 (64 registers,
// a few bytes of spills: 16.7 against 17.5 ms at 3 on the Llama-3.1-8B
// table); with 16-bit rho or FP32 gradients, which hold 4 or 8 more words a
// thread, 3 on long tiles (80 registers: 18.4 against 18.9 ms at 4 on the 8B
// table) and 4 on the short and one-chunk tiles of small tables, which are
// latency-bound (the 64M-element stress set at 16-bit rho: 0.165 against
// 0.168 ms). Lion runs 4 (6 % faster on the Llama-3.1-8B step than 3; 5 was
// 1 % slower). SGD runs 4 on long tiles and 5 (48 registers) on short and
// one-chunk tiles (ResNet-50: 0.0524 against 0.0533 ms).
constexpr int step_ctas_per_sm(Opt o, int rho_bits, int grad_bits, int chunks)
{
    return o == Opt::kSgd    ? (chunks == kLongChunks ? 4 : 5)
           : o == Opt::kLion ? 4
                             : ((rho_bits == 8 && grad_bits == 16) || chunks != kLongChunks ? 4 : 3);
}

// One table row as the step kernel sees it. `coef` is the per-tensor scalar:
// the decay factor (1 - lr*wd) for AdamW and Lion, the weight decay for SGD.
struct StepRow {
    uint16_t *theta;
    void *rho;
    int8_t *mq;
    uint16_t *ms;
    uint8_t *vq;
    uint16_t *vs;
    const void *grad;   // uint16_t (BF16) or float, per the launch's gradient type
    int64_t numel;
    float coef;
    int32_t rho_bits;
};
static_assert(sizeof(StepRow) == 72, "StepRow layout");

// Per-step FP32 scalars.
//  AdamW: a = {beta1, beta2, 1-beta1, 1-beta2, eps, -lr/bc1, 1/sqrt(bc2)}
//  SGD:   a = {momentum, -lr}
//  Lion:  a = {beta1, beta2, 1-beta1, 1-beta2, -lr}
// and the same values as lane pairs for the packed fast path (p), with the
// signs and scalings that path needs (AdamW carries m scaled by 2^32):
//  AdamW: p = {2^32 b1, -b2, 2^32 (1-b1), -(1-b2), 1/sqrt(bc2), -eps, -2^-32 lr/bc1}
//  SGD:   p = {momentum, -lr}
//  Lion:  p = {b1, b2, 1-b1, 1-b2, -lr}
// fast = 1 when the call's hyper-parameters keep the fast path's operands in
// its validated ranges (conditions in fo_api.cu).
// lo, hi: the fast path's range for its checked operand x (AdamW: the
// gradient; SGD, Lion: the new momentum): x = 0 or lo' <= |x| <= hi', given
// as the FP32 values just below lo' and hi' (the guard compares the float
// below |x|, see Guard in fo_step.cuh).
// v_nonzero (AdamW): requantize v with no code 0 in a group with a non-zero scale.
// step_dev (AdamW, may be null): the step counter t in device memory; when
// set, the kernel derives a[5], a[6], p[4], p[6] and the t-dependent part of
// `fast` from *step_dev, lr, beta1 and beta2 (the host leaves them unset),
// and skips the launch (skip) for t < 1.
struct StepScalars {
    float a[8];
    unsigned long long p[8];
    float lo, hi;
    int32_t fast;
    int32_t v_nonzero;
    const long long *step_dev;
    double lr, beta1, beta2;
    int32_t skip;
    int32_t pad;
};

// Rows per launch: the whole table of one launch travels in the kernel's
// parameter space (at most 32764 bytes on sm_70 and later).
constexpr int kRowsPerLaunch = 384;

struct StepParams {
    StepScalars s;
    int32_t nrows;
    int32_t total_tiles;
    int32_t chunks;                    // chunks per tile: kLongChunks, kShortChunks or kTinyChunks
    int32_t pad;
    int32_t tile_end[kRowsPerLaunch];  // inclusive prefix sums of tiles per row
    StepRow rows[kRowsPerLaunch];
};
static_assert(sizeof(StepParams) <= 32764, "kernel parameter space");

// Launch one fused step over p.nrows rows, all of correction width rho_bits
// and gradient width grad_bits (16: BF16, 32: FP32) (p.total_tiles > 0).
cudaError_t launch_step(Opt opt, int rho_bits, int grad_bits, const StepParams &p, cudaStream_t stream);

// Element-wise codecs.
cudaError_t launch_split(const float *theta, uint16_t *tp, void *rho, int64_t n, int rho_bits,
                         cudaStream_t stream);
cudaError_t launch_merge(const uint16_t *tp, const void *rho, float *theta, int64_t n, int rho_bits,
                         cudaStream_t stream);
cudaError_t launch_quant(const float *x, void *q, uint16_t *scales, int64_t n, int kind,
                         cudaStream_t stream);
cudaError_t launch_dequant(const void *q, const uint16_t *scales, float *x, int64_t n, int kind,
                           cudaStream_t stream);

// On-device enumeration of the fast path's hardware-dependent arithmetic
// (fo_verify.cu): kVerifyCounts mismatch counts written to `counts` (device).
constexpr int kVerifyCounts = 6;
cudaError_t launch_verify(unsigned long long *counts, cudaStream_t stream);

// Number of SMs of the current device (cached per device).
int sm_count();
// Kernel launches issued by this library so far.
void count_launch();

}  // namespace fo
