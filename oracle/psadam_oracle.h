/*
 * psadam_oracle.h — TEST INFRASTRUCTURE, not product code.
 *
 * Declarations of the plain, slow, single-threaded CPU oracle for the fused AdamW
 * update with compressed moment state (fp32, bf16 and block-wise 8-bit moments).
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg call it.
 * The CUDA library never includes this header and the oracle never includes the
 * library's; the two share no code.
 *
 * Sources the oracle follows (cited per function in psadam_oracle.c):
 *   [P814]  AiDotNet PR #814 "feat: add 8-bit Adam optimizer for memory efficiency":
 *           summary list, sequence diagram, options list, review of UpdateParameters.
 *   [P1745] AiDotNet PR #1745 "perf(training): make BF16-Adam fused-compatible
 *           (proper bf16 moment kernel, not a gate)": "What changed" / "The real fix".
 *   [PHILOX] J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw, "Parallel random
 *           numbers: as easy as 1, 2, 3", SC'11, section 3 (Philox).
 *   Textbook Adam (Kingma & Ba 2015, Algorithm 1) with decoupled weight decay
 *   (Loshchilov & Hutter 2019, AdamW).
 */
#ifndef PSADAM_ORACLE_H
#define PSADAM_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORC_BLOCK 2048 /* [P814] default BlockSize */

/* Hyper-parameters exactly as a caller hands them over (single precision). */
typedef struct {
    float lr, beta1, beta2, eps, weight_decay;
} orc_hparams;

/* Per-step single-precision constants, each computed in double and rounded once. */
typedef struct {
    float b1, omb1, b2, omb2, decay, step_size, inv_sqrt_bc2, eps;
} orc_scalars;

/* 8-bit moment options. */
typedef struct {
    int stochastic_rounding; /* 0 = round to nearest even, 1 = stochastic */
    uint64_t seed;           /* Philox key for stochastic rounding */
    float percentile;        /* scale basis percentile, (0, 100]; 100 = absmax */
    int static_scales;       /* 1: a block's nonzero scale is kept (frozen) instead of recomputed */
    int block_size;          /* elements per quantization block (>= 1; [P814] default 2048) */
} orc_q8opts;

/* Philox4x32-10 bijection of one 128-bit counter under a 64-bit key. */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);
void orc_philox4x32_10_many(int64_t n, const uint32_t* ctr, const uint32_t* key, uint32_t* out);

/* The uniform u in [0,1) used by stochastic rounding of element `elem` of tensor
 * `tensor_idx` for moment `moment` (0 = m, 1 = v) at step `step`. */
float orc_sr_uniform(uint64_t seed, int64_t step, int tensor_idx, int moment, int64_t elem);

/* bf16 storage: round to nearest, ties to even; exact widening. */
uint16_t orc_bf16_round(float x);
float orc_bf16_widen(uint16_t b);
void orc_bf16_round_many(int64_t n, const float* x, uint16_t* out);
void orc_bf16_widen_many(int64_t n, const uint16_t* b, float* out);

/* Step constants for 1-based step t. */
orc_scalars orc_make_scalars(const orc_hparams* hp, int64_t t);

/* Nearest-rank position k (1 = largest) of the percentile `pct` among n values. */
int64_t orc_percentile_rank(float pct, int64_t n);

/* k-th largest of |x[0..n)| (k is 1-based, 1 <= k <= n). */
float orc_kth_largest_abs(const float* x, int64_t n, int64_t k);

/* Quantize one block of n values (n <= the block size). is_signed: codes in [-127,127]
 * (written to codes_i8), else [0,255] (codes_u8). Returns the block's scale.
 * The stochastic variant draws element (elem0 + i)'s uniform from the step's stream.
 * With q->static_scales and a nonzero old_scale, that scale is kept (no new block
 * statistics); otherwise old_scale is ignored. */
float orc_quantize_block(const float* x, int64_t n, int is_signed, const orc_q8opts* q,
                         int64_t step, int tensor_idx, int64_t elem0, float old_scale,
                         int8_t* codes_i8, uint8_t* codes_u8);

/* Whole-tensor quantize / dequantize of a moment pair (block after block). */
void orc_quantize(int64_t n, const float* m, const float* v, const orc_q8opts* q,
                  int64_t step, int tensor_idx, int8_t* m_code, uint8_t* v_code,
                  float* m_scale, float* v_scale);
void orc_dequantize(int64_t n, int64_t block_size, const int8_t* m_code, const uint8_t* v_code,
                    const float* m_scale, const float* v_scale, float* m, float* v);

/* One AdamW step over one tensor of n elements, in place.
 * grad: float* when grad_bf16 == 0, else uint16_t* holding bf16 bits. */
void orc_step_fp32(int64_t n, float* p, const void* grad, int grad_bf16, float* m, float* v,
                   const orc_hparams* hp, int64_t t);
void orc_step_bf16m(int64_t n, float* p, const void* grad, int grad_bf16, uint16_t* m,
                    uint16_t* v, const orc_hparams* hp, int64_t t);
/* 8-bit moments over blocks [block_begin, block_end) of q->block_size elements; the rest of the
 * tensor is left untouched (steps are block-local, so a range is exact). */
void orc_step_q8(int64_t n, float* p, const void* grad, int grad_bf16, int8_t* m_code,
                 uint8_t* v_code, float* m_scale, float* v_scale, const orc_hparams* hp,
                 int64_t t, const orc_q8opts* q, int tensor_idx, int64_t block_begin,
                 int64_t block_end);

/* The same step for one block: cnt (<= q->block_size) valid elements that start at element
 * elem0 of their tensor; array pointers point at the block's first element and the
 * scale pointers at the block's own scale. */
void orc_step_q8_block(int64_t cnt, int64_t elem0, float* p, const void* grad, int grad_bf16,
                       int8_t* m_code, uint8_t* v_code, float* m_scale, float* v_scale,
                       const orc_hparams* hp, int64_t t, const orc_q8opts* q, int tensor_idx);

/* fp32 first moment, 8-bit second moment (the pages' CompressBothMoments = false):
 * whole-tensor (block range) and single-block forms, arguments as for the 8-bit step. */
void orc_step_q8v(int64_t n, float* p, const void* grad, int grad_bf16, float* m, uint8_t* v_code,
                  float* v_scale, const orc_hparams* hp, int64_t t, const orc_q8opts* q, int tensor_idx,
                  int64_t block_begin, int64_t block_end);
void orc_step_q8v_block(int64_t cnt, int64_t elem0, float* p, const void* grad, int grad_bf16, float* m,
                        uint8_t* v_code, float* v_scale, const orc_hparams* hp, int64_t t,
                        const orc_q8opts* q, int tensor_idx);

/* out[i] = grad[i] * unscale (one fp32 rounding; bf16 grads widened first). */
void orc_unscale_grads(int64_t n, const void* grad, int grad_bf16, float unscale, float* out);

/* Build-flag probe: returns a*b + c with two roundings. A build that let the
 * compiler contract this into one fused multiply-add would return the fused value. */
float orc_probe_mul_add(float a, float b, float c);

#ifdef __cplusplus
}
#endif

#endif /* PSADAM_ORACLE_H */
