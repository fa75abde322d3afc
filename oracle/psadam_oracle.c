/*
 * psadam_oracle.c — TEST INFRASTRUCTURE, not product code.
 *
 * A plain, slow, single-threaded CPU restatement of the fused AdamW update with
 * compressed moment state. It exists so that tests can check the CUDA library
 * element by element. Only tests/, the smoke check and the benchmark's CPU
 * baseline call it; the product library never links it and shares no code with it.
 *
 * Arithmetic: the pages' optimizer works in the parameter type T (float in every
 * workload), keeps fp32 per-block scale arrays next to the 8-bit codes, and forms
 * the bias corrections with Math.Pow on doubles ([P814] review of UpdateParameters).
 * So every per-element operation here is one IEEE single-precision operation, in the
 * order written, and only the per-step constants are formed in double and rounded
 * once. The file must be compiled with -ffp-contract=off (see orc_probe_mul_add).
 *
 * Source tags ([P814], [P1745], [PHILOX], textbook Adam/AdamW) are listed in
 * psadam_oracle.h.
 */
#include "psadam_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------------ */
/* Philox4x32-10 — [PHILOX] section 3: the Philox-4x32 round multiplies counter   */
/* words 0 and 2 by two fixed 32-bit constants, takes the high/low halves of the  */
/* 64-bit products, XORs the high halves with the other two counter words and the */
/* round key, and permutes; the key is bumped by the Weyl constants (golden ratio */
/* and sqrt(3)-1 in 32-bit fixed point) between rounds; ten rounds.               */
/* ------------------------------------------------------------------------------ */
#define PHILOX_M0 0xD2511F53u
#define PHILOX_M1 0xCD9E8D57u
#define PHILOX_W0 0x9E3779B9u
#define PHILOX_W1 0xBB67AE85u

void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    uint32_t x[4] = {ctr[0], ctr[1], ctr[2], ctr[3]};
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += PHILOX_W0;
            k1 += PHILOX_W1;
        }
        uint64_t prod0 = (uint64_t)PHILOX_M0 * (uint64_t)x[0];
        uint64_t prod1 = (uint64_t)PHILOX_M1 * (uint64_t)x[2];
        uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
        uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
        uint32_t y[4];
        y[0] = hi1 ^ x[1] ^ k0;
        y[1] = lo1;
        y[2] = hi0 ^ x[3] ^ k1;
        y[3] = lo0;
        memcpy(x, y, sizeof x);
    }
    memcpy(out, x, sizeof x);
}

void orc_philox4x32_10_many(int64_t n, const uint32_t* ctr, const uint32_t* key, uint32_t* out) {
    for (int64_t i = 0; i < n; ++i) orc_philox4x32_10(ctr + 4 * i, key + 2 * i, out + 4 * i);
}

/* Stochastic rounding stream ([P814] "Stochastic rounding option for reduced
 * quantization bias"; the pages' generator is a fixed-seed Random, replaced here by a
 * counter-based one so that a step is reproducible from (seed, step, index) alone).
 * Counter = (group index low, group index high, step, tensor_idx*2 + moment) with
 * group = elem / 4; key = seed; element elem takes output word elem % 4; the top 24
 * bits of that word, times 2^-24, give u in [0, 1). */
float orc_sr_uniform(uint64_t seed, int64_t step, int tensor_idx, int moment, int64_t elem) {
    uint64_t group = (uint64_t)elem / 4u;
    uint32_t ctr[4] = {(uint32_t)(group & 0xFFFFFFFFu), (uint32_t)(group >> 32), (uint32_t)step,
                       (uint32_t)tensor_idx * 2u + (uint32_t)moment};
    uint32_t key[2] = {(uint32_t)(seed & 0xFFFFFFFFu), (uint32_t)(seed >> 32)};
    uint32_t out[4];
    orc_philox4x32_10(ctr, key, out);
    uint32_t word = out[(uint64_t)elem % 4u];
    return (float)(word >> 8) * 0x1p-24f;
}

/* ------------------------------------------------------------------------------ */
/* bf16 moment storage — [P1745] keeps m and v in half-size 16-bit buffers: a bf16  */
/* the top 16 bits of an fp32. Storing rounds to the nearer of the two bf16 values */
/* around x, ties to the one with an even last bit; widening is exact.            */
/* ------------------------------------------------------------------------------ */
static uint32_t f32_bits(float x) {
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    return u;
}
static float f32_from_bits(uint32_t u) {
    float x;
    memcpy(&x, &u, sizeof x);
    return x;
}

uint16_t orc_bf16_round(float x) {
    uint32_t u = f32_bits(x);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    if (isnan(x)) return (uint16_t)((u >> 16) | 0x0040u); /* quiet NaN, sign kept */
    if (isinf(x)) return (uint16_t)(u >> 16);
    /* The bf16 just below |x| (truncation) and the next one up, as exact doubles. */
    uint16_t lo_mag = (uint16_t)((u >> 16) & 0x7FFFu);
    double lo = (double)f32_from_bits((uint32_t)lo_mag << 16);
    int exp_field = (int)((u >> 23) & 0xFFu);
    double spacing = ldexp(1.0, (exp_field == 0 ? 1 : exp_field) - 127 - 7);
    double hi = lo + spacing; /* 2^128 above the largest finite bf16: rounds to inf */
    double ax = fabs((double)x);
    double d_lo = ax - lo, d_hi = hi - ax; /* both exact in double */
    uint16_t mag;
    if (d_lo < d_hi)
        mag = lo_mag;
    else if (d_hi < d_lo)
        mag = (uint16_t)(lo_mag + 1u);
    else
        mag = (lo_mag & 1u) ? (uint16_t)(lo_mag + 1u) : lo_mag;
    return (uint16_t)(sign | mag);
}

float orc_bf16_widen(uint16_t b) { return f32_from_bits((uint32_t)b << 16); }

void orc_bf16_round_many(int64_t n, const float* x, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_round(x[i]);
}

void orc_bf16_widen_many(int64_t n, const uint16_t* b, float* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_widen(b[i]);
}

/* ------------------------------------------------------------------------------ */
/* Per-step constants — [P814] review of UpdateParameters: beta1, beta2, their     */
/* complements, epsilon and biasCorrection1/2 from Math.Pow on doubles and the     */
/* step count _t. With bc_i = 1 - beta_i^t (textbook Adam, Algorithm 1):           */
/*   step_size = lr / bc1, inv_sqrt_bc2 = 1 / sqrt(bc2), decay = 1 - lr * wd       */
/* (decoupled weight decay, AdamW). Each is formed in double and rounded once.    */
/* ------------------------------------------------------------------------------ */
orc_scalars orc_make_scalars(const orc_hparams* hp, int64_t t) {
    double lr = hp->lr, b1 = hp->beta1, b2 = hp->beta2, wd = hp->weight_decay;
    double bc1 = 1.0 - pow(b1, (double)t);
    double bc2 = 1.0 - pow(b2, (double)t);
    orc_scalars s;
    s.b1 = hp->beta1;
    s.omb1 = (float)(1.0 - b1);
    s.b2 = hp->beta2;
    s.omb2 = (float)(1.0 - b2);
    s.decay = (float)(1.0 - lr * wd);
    s.step_size = (float)(lr / bc1);
    s.inv_sqrt_bc2 = (float)(1.0 / sqrt(bc2));
    s.eps = hp->eps;
    return s;
}

/* One element of AdamW (textbook Adam with bias correction + decoupled decay):
 *   m' = b1*m + (1-b1)*g
 *   v' = b2*v + (1-b2)*g*g
 *   p' = p*(1 - lr*wd) - (lr/bc1) * m' / (sqrt(v')/sqrt(bc2) + eps)
 * which is p - lr*wd*p - lr * m_hat / (sqrt(v_hat) + eps) with m_hat = m'/bc1 and
 * v_hat = v'/bc2. The parameter update uses the unquantized m', v' ([P814] sequence
 * diagram: the updated m, v and parameters come back before Quantize(m), Quantize(v)). */
static void adam_element(float* p, float g, float* m, float* v, const orc_scalars* s) {
    float m_new = s->b1 * *m + s->omb1 * g;
    float v_new = s->b2 * *v + (s->omb2 * g) * g;
    float p_decayed = *p * s->decay;
    float denom = sqrtf(v_new) * s->inv_sqrt_bc2 + s->eps;
    float ratio = m_new / denom;
    *p = p_decayed - s->step_size * ratio;
    *m = m_new;
    *v = v_new;
}

static float load_grad(const void* grad, int grad_bf16, int64_t i) {
    if (grad_bf16) return orc_bf16_widen(((const uint16_t*)grad)[i]);
    return ((const float*)grad)[i];
}

void orc_step_fp32(int64_t n, float* p, const void* grad, int grad_bf16, float* m, float* v,
                   const orc_hparams* hp, int64_t t) {
    orc_scalars s = orc_make_scalars(hp, t);
    for (int64_t i = 0; i < n; ++i) adam_element(&p[i], load_grad(grad, grad_bf16, i), &m[i], &v[i], &s);
}

/* [P1745]: the bf16-moment kernel keeps m and v as bf16, widens, updates, and
 * stores them back rounded. */
void orc_step_bf16m(int64_t n, float* p, const void* grad, int grad_bf16, uint16_t* m,
                    uint16_t* v, const orc_hparams* hp, int64_t t) {
    orc_scalars s = orc_make_scalars(hp, t);
    for (int64_t i = 0; i < n; ++i) {
        float mf = orc_bf16_widen(m[i]);
        float vf = orc_bf16_widen(v[i]);
        adam_element(&p[i], load_grad(grad, grad_bf16, i), &mf, &vf, &s);
        m[i] = orc_bf16_round(mf);
        v[i] = orc_bf16_round(vf);
    }
}

/* ------------------------------------------------------------------------------ */
/* Block-wise 8-bit moments — [P814] summary: block-wise quantization, block 2048,  */
/* (options list: BlockSize, any positive size, default 2048),                     */
/* signed quantization for m and unsigned for v, dynamic scales, percentile-based  */
/* scaling (QuantizationPercentile, default 99.9, range 0..100), optional          */
/* stochastic rounding; review notes: "[-127, 127] to [1, 255] mapping (0 is       */
/* unused)". Reading: a linear code with the per-block fp32 scale equal to one code */
/* step: s = X / 127 for m and X / 255 for v, X the block's percentile magnitude.  */
/* ------------------------------------------------------------------------------ */

/* Nearest-rank percentile: the smallest value whose rank from the bottom is at least
 * ceil(pct/100 * n); as a position from the top that is k = n - ceil(pct*n/100) + 1. */
int64_t orc_percentile_rank(float pct, int64_t n) {
    int64_t from_bottom = (int64_t)ceil((double)pct * (double)n / 100.0);
    int64_t k = n - from_bottom + 1;
    if (k < 1) k = 1;
    if (k > n) k = n;
    return k;
}

static int cmp_desc(const void* a, const void* b) {
    float x = *(const float*)a, y = *(const float*)b;
    return (x < y) - (x > y);
}

float orc_kth_largest_abs(const float* x, int64_t n, int64_t k) {
    float* tmp = (float*)malloc((size_t)n * sizeof(float));
    for (int64_t i = 0; i < n; ++i) tmp[i] = fabsf(x[i]);
    qsort(tmp, (size_t)n, sizeof(float), cmp_desc);
    float r = tmp[k - 1];
    free(tmp);
    return r;
}

float orc_quantize_block(const float* x, int64_t n, int is_signed, const orc_q8opts* q,
                         int64_t step, int tensor_idx, int64_t elem0, float old_scale,
                         int8_t* codes_i8, uint8_t* codes_u8) {
    float qmax = is_signed ? 127.0f : 255.0f;
    float qmin = is_signed ? -127.0f : 0.0f;
    float scale;
    if (q->static_scales && old_scale != 0.0f) {
        /* [P814] options list: UseDynamicQuantization = false. Reading: the scale set by
         * the block's first quantization stays; values beyond it saturate. */
        scale = old_scale;
    } else {
        float absmax = 0.0f;
        for (int64_t i = 0; i < n; ++i)
            if (fabsf(x[i]) > absmax) absmax = fabsf(x[i]);
        int64_t k = orc_percentile_rank(q->percentile, n);
        float basis = orc_kth_largest_abs(x, n, k);
        if (basis == 0.0f) basis = absmax; /* a block whose percentile is 0 falls back to its max */
        scale = basis / qmax;
    }
    for (int64_t i = 0; i < n; ++i) {
        float r = 0.0f;
        if (scale != 0.0f) {
            float ratio = x[i] / scale;
            if (q->stochastic_rounding) {
                float u = orc_sr_uniform(q->seed, step, tensor_idx, is_signed ? 0 : 1, elem0 + i);
                r = floorf(ratio + u);
            } else {
                r = nearbyintf(ratio); /* default rounding mode: ties to even */
            }
            if (r > qmax) r = qmax;
            if (r < qmin) r = qmin;
        }
        if (is_signed)
            codes_i8[i] = (int8_t)(int)r;
        else
            codes_u8[i] = (uint8_t)(int)r;
    }
    return scale;
}

static int64_t block_count(int64_t n, int64_t bs) { return (n + bs - 1) / bs; }

void orc_quantize(int64_t n, const float* m, const float* v, const orc_q8opts* q,
                  int64_t step, int tensor_idx, int8_t* m_code, uint8_t* v_code,
                  float* m_scale, float* v_scale) {
    const int64_t bs = q->block_size;
    for (int64_t b = 0; b < block_count(n, bs); ++b) {
        int64_t lo = b * bs;
        int64_t cnt = n - lo < bs ? n - lo : bs;
        m_scale[b] = orc_quantize_block(m + lo, cnt, 1, q, step, tensor_idx, lo, m_scale[b], m_code + lo, NULL);
        v_scale[b] = orc_quantize_block(v + lo, cnt, 0, q, step, tensor_idx, lo, v_scale[b], NULL, v_code + lo);
    }
}

/* Dequantize: value = code * scale, one single-precision multiply. */
void orc_dequantize(int64_t n, int64_t block_size, const int8_t* m_code, const uint8_t* v_code,
                    const float* m_scale, const float* v_scale, float* m, float* v) {
    for (int64_t i = 0; i < n; ++i) {
        int64_t b = i / block_size;
        m[i] = (float)m_code[i] * m_scale[b];
        v[i] = (float)v_code[i] * v_scale[b];
    }
}

/* [P814] sequence diagram, per step: Dequantize(m), Dequantize(v), Adam update with
 * bias correction, Quantize(m), Quantize(v). Blocks never interact, so the four phases
 * run block by block. One block: `cnt` valid elements starting at element `elem0` of
 * its tensor; the array pointers point at the block's first element, the scale
 * pointers at the block's scale. */
void orc_step_q8_block(int64_t cnt, int64_t elem0, float* p, const void* grad, int grad_bf16,
                       int8_t* m_code, uint8_t* v_code, float* m_scale, float* v_scale,
                       const orc_hparams* hp, int64_t t, const orc_q8opts* q, int tensor_idx) {
    orc_scalars s = orc_make_scalars(hp, t);
    float* mf = (float*)malloc((size_t)cnt * sizeof(float));
    float* vf = (float*)malloc((size_t)cnt * sizeof(float));
    for (int64_t i = 0; i < cnt; ++i) mf[i] = (float)m_code[i] * *m_scale;
    for (int64_t i = 0; i < cnt; ++i) vf[i] = (float)v_code[i] * *v_scale;
    for (int64_t i = 0; i < cnt; ++i) adam_element(&p[i], load_grad(grad, grad_bf16, i), &mf[i], &vf[i], &s);
    *m_scale = orc_quantize_block(mf, cnt, 1, q, t, tensor_idx, elem0, *m_scale, m_code, NULL);
    *v_scale = orc_quantize_block(vf, cnt, 0, q, t, tensor_idx, elem0, *v_scale, NULL, v_code);
    free(mf);
    free(vf);
}

void orc_step_q8(int64_t n, float* p, const void* grad, int grad_bf16, int8_t* m_code,
                 uint8_t* v_code, float* m_scale, float* v_scale, const orc_hparams* hp,
                 int64_t t, const orc_q8opts* q, int tensor_idx, int64_t block_begin,
                 int64_t block_end) {
    size_t gsize = grad_bf16 ? sizeof(uint16_t) : sizeof(float);
    const int64_t bs = q->block_size;
    for (int64_t b = block_begin; b < block_end; ++b) {
        int64_t lo = b * bs;
        int64_t cnt = n - lo < bs ? n - lo : bs;
        orc_step_q8_block(cnt, lo, p + lo, (const char*)grad + (size_t)lo * gsize, grad_bf16,
                          m_code + lo, v_code + lo, m_scale + b, v_scale + b, hp, t, q, tensor_idx);
    }
}

/* [P814] summary: with CompressBothMoments = false the first moment stays in full
 * precision: m stays fp32, only v is block-quantized. Same step order
 * (dequantize v, update, quantize v), same v encoding and stream as the 8-bit step. */
void orc_step_q8v_block(int64_t cnt, int64_t elem0, float* p, const void* grad, int grad_bf16, float* m,
                        uint8_t* v_code, float* v_scale, const orc_hparams* hp, int64_t t,
                        const orc_q8opts* q, int tensor_idx) {
    orc_scalars s = orc_make_scalars(hp, t);
    float* vf = (float*)malloc((size_t)cnt * sizeof(float));
    for (int64_t i = 0; i < cnt; ++i) vf[i] = (float)v_code[i] * *v_scale;
    for (int64_t i = 0; i < cnt; ++i) adam_element(&p[i], load_grad(grad, grad_bf16, i), &m[i], &vf[i], &s);
    *v_scale = orc_quantize_block(vf, cnt, 0, q, t, tensor_idx, elem0, *v_scale, NULL, v_code);
    free(vf);
}

void orc_step_q8v(int64_t n, float* p, const void* grad, int grad_bf16, float* m, uint8_t* v_code,
                  float* v_scale, const orc_hparams* hp, int64_t t, const orc_q8opts* q, int tensor_idx,
                  int64_t block_begin, int64_t block_end) {
    size_t gsize = grad_bf16 ? sizeof(uint16_t) : sizeof(float);
    const int64_t bs = q->block_size;
    for (int64_t b = block_begin; b < block_end; ++b) {
        int64_t lo = b * bs;
        int64_t cnt = n - lo < bs ? n - lo : bs;
        orc_step_q8v_block(cnt, lo, p + lo, (const char*)grad + (size_t)lo * gsize, grad_bf16, m + lo,
                           v_code + lo, v_scale + b, hp, t, q, tensor_idx);
    }
}

/* Grad side of a mixed-precision step (the pages are silent; the plain reading of loss
 * scaling): each grad is multiplied by the inverse loss scale, one fp32 rounding, before
 * the update sees it. bf16 grads are widened first (exactly). */
void orc_unscale_grads(int64_t n, const void* grad, int grad_bf16, float unscale, float* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = load_grad(grad, grad_bf16, i) * unscale;
}

float orc_probe_mul_add(float a, float b, float c) { return a * b + c; }
