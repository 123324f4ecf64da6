/*
 * mp_oracle.h — plain, single-threaded CPU oracle of the mixed-precision
 * AdamW + stochastic-rounding optimizer step.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product (the CUDA library and its
 * Python binding) may include, link, load or call this code; only the tests,
 * the smoke check and the benchmark's CPU-baseline leg do. It shares no code,
 * header, table or constant generator with the CUDA path: every function here
 * is written from the pages' description of the method, cited per function.
 *
 * Sources (web pages, by title and section):
 *   [LLMC]  llm.c code walk-through, ch. 04 "Multi-GPU and mixed precision":
 *           §2.2 AdamW kernel, §2.3 stochastic rounding, §4 train step.
 *   [CMU13] CMU 11-667 lecture 13 notes, "Scaling up LLMs: optimization and
 *           parallel training": §1.7 bias correction and AdamW, §2.3 fp32
 *           master weights, §7.3 exercises 1 and 5.
 *
 * Precision: the pages fix fp32 for the update (fp32 master, fp32 m/v, the
 * bf16 grad converted to float before use), so the step is computed in fp32
 * with one rounding per written operation and an explicit fmaf() for each of
 * the two-FMA lerps; the gradient norm is a plain fp64 sum of squares.
 * Compiled with -ffp-contract=off and without fast-math.
 *
 * Parity unpinned: the exact 32-bit values of oracle_noise_u32. The pages
 * name SquirrelNoise5 but print no test vector, so the hash's constants and
 * shifts are pinned only by statistical tests (uniform, uncorrelated draws,
 * strict avalanche) that a different but equally good mixer would also
 * pass; a dropped mixing round fails the avalanche test. Every other
 * function here is pinned by values or properties the pages or mathematics
 * fix (tests/test_oracle_pins.py).
 */
#ifndef MP_ORACLE_H
#define MP_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct oracle_tensor {
    uint64_t offset; /* global element offset of the tensor */
    uint64_t size;   /* element count                        */
    int32_t decay;   /* 1: weight decay applies; 0: it does not */
    int32_t pad;
} oracle_tensor;

/* SquirrelNoise5 (Squirrel Eiserloh), 2D form, at (low32(k), high32(k)). */
uint32_t oracle_noise_u32(uint64_t k, uint32_t seed);
void oracle_noise_fill(uint32_t* out, uint64_t first, uint64_t n, uint32_t seed);

/* Stochastic rounding of one fp32 value with a given 16-bit random draw. */
uint16_t oracle_sr_with_rand(float x, uint32_t rand16);
/* Stochastic rounding keyed on (global index k, seed). */
uint16_t oracle_sr(float x, uint64_t k, uint32_t seed);
void oracle_stochastic_round(uint16_t* out, const float* in,
                             uint64_t global_offset, uint64_t n, uint32_t seed);
/* Stochastic rounding fp32 -> fp16 with a given 16-bit draw, and of a range
 * keyed on (global index, seed) with the same draws as the bf16 rounding. */
uint16_t oracle_sr_fp16_with_rand(float x, uint32_t rand16);
void oracle_stochastic_round_fp16(uint16_t* out, const float* in, uint64_t global_offset, uint64_t n,
                                  uint32_t seed);
/* acc[i] = SR((float)acc[i] + delta[i], global_offset + i, seed): a bf16
 * accumulator updated in fp32 and rounded back stochastically. */
void oracle_accumulate_sr(uint16_t* acc, const float* delta, uint64_t global_offset, uint64_t n,
                          uint32_t seed);

/* Gradient norm: plain fp64 sum of squares in index order, then sqrt. */
double oracle_sumsq(const uint16_t* grads, uint64_t n);
/* The same sum continued from a running total s, in index order: summing a
 * buffer in consecutive pieces gives exactly the one-pass sum. */
double oracle_sumsq_from(double s, const uint16_t* grads, uint64_t n);
float oracle_clip_scale(float norm, float clip);
/* ZeRO-1: norm and clip scale from per-rank sums of squares added in rank
 * order (fp64). */
void oracle_norm_from_parts(const double* parts, int32_t count, float clip,
                            double* sumsq, float* norm, float* scale);
/* Learning rate of the 1-based step t: kind 0 constant, 1 cosine, 2 linear,
 * 3 WSD, each after a linear warm-up; NaN for invalid arguments. */
float oracle_lr(int32_t kind, int64_t warmup, int64_t total, float lr_max, float lr_min,
                float decay_frac, int64_t t);
void oracle_grad_norm(const uint16_t* grads, uint64_t n, float clip,
                      double* sumsq, float* norm, float* scale);

/* Bias-correction denominators 1 - beta^t for the 1-based step t. */
void oracle_bias_corrections(float beta1, float beta2, int32_t t,
                             float* bc1, float* bc2);

/* One AdamW + SR step over [global_offset, global_offset + n) of the flat
 * buffer described by `table`. master == NULL selects the no-master variant.
 * Returns 0, or 5 (nothing written) if `scale` is not finite, or -1 if the
 * table leaves part of the range uncovered. */
int oracle_adamw_step(uint16_t* params, const uint16_t* grads, float* master,
                      float* m, float* v,
                      uint64_t global_offset, uint64_t n,
                      const oracle_tensor* table, int32_t n_tensors,
                      float lr, float beta1, float beta2, float eps,
                      float weight_decay, float scale,
                      int32_t t, uint32_t seed);

/* Grad-norm outlier check: window of the last 128 finite norms. */
#define ORACLE_OUTLIER_WINDOW 128
typedef struct oracle_outlier {
    double window[ORACLE_OUTLIER_WINDOW];
    uint64_t count; /* finite norms pushed so far */
} oracle_outlier;

/* z-score of `norm` against the window (NaN until it holds 128 norms); if z
 * exceeds a positive threshold, *scale becomes NaN and 8 is returned (skip),
 * else 0. A finite norm then enters the window, replacing the oldest. */
int oracle_outlier_check(oracle_outlier* st, float norm, float z_threshold,
                         float* scale, double* z);

#ifdef __cplusplus
}
#endif

#endif
