/*
 * psadam.h — C ABI of libpsadam.so: the fused AdamW parameter update with compressed
 * moment state, for sm_103a (GB300).
 *
 * One call performs one optimizer step over a multi-tensor list of fp32 parameters,
 * in place, with the moments stored in one of three forms:
 *   adam_step_fp32   fp32 m and v                                (28 bytes moved / param)
 *   adam_step_bf16m  bf16 m and v, round to nearest even         (20 bytes / param)
 *   adam_step_q8     8-bit block-wise codes + fp32 block scales  (16 bytes / param + scales)
 *   adam_step_q8v    fp32 m, 8-bit v codes + scales              (22 bytes / param + scales)
 * (byte counts for fp32 grads; bf16 grads move 2 bytes less.)
 *
 * Sources of the method:
 *   - AiDotNet PR #814 "feat: add 8-bit Adam optimizer for memory efficiency":
 *     block-wise quantization with block size 2048 (options list: BlockSize, any
 *     positive size), signed codes for m and unsigned codes for v, scales recomputed every step (its dynamic quantization),
 *     QuantizationPercentile (default 99.9, range 0..100) so that outliers do not set the scale,
 *     optional stochastic rounding; its sequence diagram fixes the step order:
 *     dequantize m and v, Adam update with bias correction, quantize m, quantize v.
 *   - AiDotNet PR #1745 "perf(training): make BF16-Adam fused-compatible (proper bf16
 *     moment kernel, not a gate)": the fused Adam/AdamW kernel over half-size bf16 m/v
 *     buffers, configured by (lr, beta1, beta2, eps, weight decay).
 *   - Adam (Kingma & Ba, Algorithm 1) with decoupled weight decay (Loshchilov & Hutter).
 *
 * What one element computes (fp32, each operation one rounding, no fused multiply-add):
 *   m' = beta1*m + (1-beta1)*g
 *   v' = beta2*v + ((1-beta2)*g)*g
 *   p' = p*(1 - lr*wd) - (lr/bc1) * (m' / (sqrt(v')*(1/sqrt(bc2)) + eps))
 * with bc1 = 1 - beta1^step and bc2 = 1 - beta2^step; the per-step constants
 * (1-beta1), (1-beta2), 1 - lr*wd, lr/bc1 and 1/sqrt(bc2) are formed in double on the
 * host and rounded once to fp32. By default every operation is IEEE-exact (the square root
 * and the quotient come from a fused correctly rounded pair inside a checked domain, with
 * the same bits as IEEE sqrt and division; see psadam_selftest_update_math).
 * psadam_list.approx_update opts into the hardware's approximate fp32 square root and
 * quotient in p' (relative errors within 2^-23 and 2 ulp): p' then lands within a few ulp
 * of the update term of the exact value (close normwise, not elementwise-relative where p'
 * passes near zero), while m', v' and every stored moment, code and scale stay exact; the
 * 8-bit step is 2-3 % faster. bf16 moments are widened exactly before and rounded to
 * nearest even after. 8-bit moments are decoded as code*scale, the update uses the
 * unquantized m', v', and each block of B elements (default 2048) is then re-encoded:
 *   X_m = k-th largest |m'| of the block, X_v = k-th largest v' (k = 1 for absmax)
 *   s_m = X_m / 127, s_v = X_v / 255  (if X = 0 the block's maximum is used instead)
 *   code = clamp(round(x / s), -127..127 for m, 0..255 for v); s = 0 gives code 0
 *   round = nearest even, or floor(x/s + u) with u in [0,1) from Philox4x32-10
 * where k = n - ceil(percentile * n / 100) + 1 among the block's n valid elements
 * (nearest-rank percentile, evaluated in double on the host).
 *
 * Conventions common to every entry point:
 *   - All arrays named "device" are device pointers; the host arrays that list them
 *     (and numel) are read during the call only. The caller owns every buffer.
 *   - Every device base pointer must be 16-byte aligned (PSADAM_ERR_MISALIGNED).
 *   - numel[i] >= 0; a tensor with numel 0 is skipped and its pointers may be NULL.
 *     n_tensors == 0 is a no-op.
 *   - Each tensor is split into consecutive blocks of B = block_size elements (2048 by
 *     default); the last block may be partial. Scale arrays hold ceil(numel/B) fp32
 *     entries per tensor.
 *   - step is the 1-based index of the step being taken (the caller increments it).
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default stream) and
 *     the call returns without synchronizing. Buffers must not alias one another.
 *   - Arguments are validated before anything is launched: on any error nothing has
 *     been written. PSADAM_ERR_CUDA means a launch failed; psadam_last_cuda_error()
 *     returns the cudaError_t value.
 *   - The library allocates no device memory: tensor metadata travels as kernel
 *     parameters; lists longer than one launch can carry are split into several launches.
 *     (psadam_step_from_host keeps a per-thread pool of CUDA events, created on first use.)
 */
#ifndef PSADAM_H
#define PSADAM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PSADAM_OK = 0,
    PSADAM_ERR_INVALID_ARG = 1, /* NULL pointer, negative size, step < 1, bad hyper-parameter */
    PSADAM_ERR_MISALIGNED = 2,  /* a device base pointer is not 16-byte aligned */
    PSADAM_ERR_UNSUPPORTED = 3, /* block size above 16384, or a block count above INT32_MAX */
    PSADAM_ERR_CUDA = 4         /* a kernel launch failed (see psadam_last_cuda_error) */
} psadam_status;

typedef enum { PSADAM_GRAD_F32 = 0, PSADAM_GRAD_BF16 = 1 } psadam_grad_dtype;

/* Hyper-parameters (PR #1745's fused config: lr, beta1, beta2, eps, weight decay).
 * Requirements: 0 <= beta1 < 1, 0 <= beta2 < 1, eps >= 0; all finite. */
typedef struct {
    float lr;
    float beta1;
    float beta2;
    float eps;
    float weight_decay; /* decoupled: p *= 1 - lr*weight_decay each step */
} psadam_hparams;

/* 8-bit options (PR #814's BlockSize, UseStochasticRounding, QuantizationPercentile).
 * Speed (identical results on every path for identical inputs):
 *   - block_size 2048 with a rank k <= 32 (percentile >= 98.5 on full blocks; 100 and the
 *     default 99.9 included) runs the pipelined 2048-block kernels, fastest at k <= 4;
 *   - power-of-two block sizes 16..1024 at rank 1 (absmax, or any percentile whose rank is
 *     1 at that size) and without grad-side options run as sub-blocks of the same kernels;
 *   - anything else runs a general kernel (tiles of whole blocks, shared-memory staging,
 *     radix select for ranks above 1). Blocks above 2048 with absmax scales whose staging
 *     would pass 32 KB are read twice instead of staged. */
typedef struct {
    int32_t block_size;          /* elements per block, 1..16384 (INVALID_ARG below 1,
                                    UNSUPPORTED above); PR #814's default is 2048 */
    int32_t stochastic_rounding; /* 0: round to nearest even; 1: Philox stochastic rounding */
    uint64_t seed;               /* Philox key (stochastic rounding only) */
    float percentile;            /* (0, 100]; 100 = absmax. PR #814's options list
                                    defaults to 99.9 (3rd largest of a full block) */
    int32_t static_scales;       /* 0: scales recomputed every step (PR #814's default
                                    UseDynamicQuantization = true). 1: a block keeps its scale
                                    once it is nonzero (set by its first quantization); values
                                    beyond it saturate. Steps only; quantize-only ignores it. */
} psadam_q8_opts;

/* The parameter/gradient side of a multi-tensor list, with the grad-side work that sits on
 * either side of the update in a mixed-precision training step. A zero-initialised tail
 * (grad_unscale 0, zero_grads 0, skip_if_set NULL, approx_update 0) changes nothing. */
typedef struct {
    int32_t n_tensors;
    int32_t grad_dtype;          /* psadam_grad_dtype: fp32 or bf16 grads (widened exactly) */
    const int64_t* numel;        /* host [n_tensors] element counts */
    float* const* param;         /* host [n_tensors] device fp32 params, updated in place */
    const void* const* grad;     /* host [n_tensors] device grads (float* or bf16 bits); read, and
                                    written only when zero_grads != 0 */
    float grad_unscale;          /* each grad is multiplied by this (one fp32 rounding) before use,
                                    e.g. 1/loss_scale; 0 reads as 1. Must be finite. */
    int32_t zero_grads;          /* nonzero: every grad is overwritten with 0 after it is read
                                    (adds 4 bytes/param of writes, 2 for bf16 grads) */
    const int32_t* skip_if_set;  /* device int32 or NULL: when it holds a nonzero value at launch
                                    the step changes nothing (e.g. psadam_check_grads found an
                                    inf/NaN). 4-byte aligned. */
    int32_t approx_update;       /* nonzero: approximate square root and quotient in the
                                    parameter update (see above); 0 = IEEE-exact */
} psadam_list;

/* One AdamW step with fp32 moments (PR #1745, "The real fix": the fused Adam/AdamW kernel
 * configured by (lr, beta1, beta2, eps, weight decay), fp32 moments being its default before
 * the bf16 option). m, v: host [n_tensors] of device float[numel], updated in place. Fresh
 * state is all zeros. */
int adam_step_fp32(const psadam_list* list, float* const* m, float* const* v, int64_t step,
                   const psadam_hparams* hp, void* stream);

/* One AdamW step with bf16 moments (PR #1745's half-size buffers). m, v: host
 * [n_tensors] of device uint16_t[numel] holding bf16 bit patterns, updated in place. */
int adam_step_bf16m(const psadam_list* list, uint16_t* const* m, uint16_t* const* v, int64_t step,
                    const psadam_hparams* hp, void* stream);

/* One AdamW step with 8-bit block-wise moments (PR #814): dequantize, update and
 * requantize in one pass. m_code: device int8_t[numel] in [-127,127]; v_code: device
 * uint8_t[numel]; m_scale, v_scale: device float[ceil(numel/block_size)]; all updated
 * in place. Fresh state is all zeros (codes 0, scales 0). Stochastic rounding of element e
 * of list tensor i draws word e%4 of Philox4x32-10(counter = (e/4 low, e/4 high,
 * step low 32 bits, 2*i + moment), key = seed), moment 0 for m and 1 for v; u is the
 * word's top 24 bits times 2^-24. */
int adam_step_q8(const psadam_list* list, int8_t* const* m_code, uint8_t* const* v_code,
                 float* const* m_scale, float* const* v_scale, int64_t step,
                 const psadam_hparams* hp, const psadam_q8_opts* q8, void* stream);

/* One AdamW step keeping the first moment in fp32 and only the second moment 8-bit (PR
 * #814's option CompressBothMoments = false, which leaves the first moment in full precision).
 * m: device float[numel]; v_code: device uint8_t[numel]; v_scale: device
 * float[ceil(numel/block_size)]; all updated in place. v is encoded exactly as adam_step_q8
 * encodes it (same percentile rule, rounding and stochastic-rounding stream, moment 1). */
int adam_step_q8v(const psadam_list* list, float* const* m, uint8_t* const* v_code, float* const* v_scale,
                  int64_t step, const psadam_hparams* hp, const psadam_q8_opts* q8, void* stream);

/* One step with host-resident grads and params (the end-to-end form of a step): copies each
 * grad from host_grad[i] (host memory, page-locked for asynchronous copies; fp32 or bf16 per
 * list->grad_dtype) into list->grad[i], steps, and copies the updated list->param[i] back to
 * host_param[i] (host fp32). mode: 0 fp32, 1 bf16m, 2 8-bit, 3 fp32 m + 8-bit v, with m, v,
 * m_scale, v_scale the arrays the matching adam_step_* call takes (NULL where that call has
 * none; q8 options only for modes 2 and 3). With stream_in and stream_out (two streams other
 * than `stream`) the list is cut into about n_chunks chunks (whole tensors; a larger tensor
 * at multiples of 4 quantization blocks and 16 elements, never past its first 4*INT_MAX
 * elements: the rest of a larger tensor is one slice) whose uploads (stream_in), steps
 * (stream) and downloads (stream_out) overlap; NULL streams run it all on `stream`. Either
 * way the results are bit for bit those of one adam_step_* call over the whole list (a
 * slice keeps its tensor's element offsets and list position for stochastic rounding), and
 * `stream` is ordered after every copy when the call returns. Within a chunk, consecutive
 * tensors whose host and device buffers both lie back to back (flat buffers) are moved by
 * one copy per direction. */
int psadam_step_from_host(int32_t mode, const psadam_list* list, const void* const* host_grad,
                          float* const* host_param, void* const* m, void* const* v,
                          float* const* m_scale, float* const* v_scale, int64_t step,
                          const psadam_hparams* hp, const psadam_q8_opts* q8, int32_t n_chunks,
                          void* stream, void* stream_in, void* stream_out);

/* Quantize-only (PR #814's Quantize(m), Quantize(v)): encodes fp32 m, v into codes and
 * scales exactly as adam_step_q8 encodes m', v' (same rounding, percentile and, for
 * stochastic rounding, the same Philox stream for `step`). For state initialisation
 * and checks. Inputs: device float m[numel], v[numel] with v >= 0. */
int psadam_q8_quantize(int32_t n_tensors, const int64_t* numel, const float* const* m,
                       const float* const* v, int8_t* const* m_code, uint8_t* const* v_code,
                       float* const* m_scale, float* const* v_scale, const psadam_q8_opts* q8,
                       int64_t step, void* stream);

/* Dequantize-only (PR #814's Dequantize): m = code*scale, v = code*scale (one fp32
 * multiply each, element e taking scale e / block_size) into device float m[numel],
 * v[numel]. block_size as in psadam_q8_opts. */
int psadam_q8_dequantize(int32_t n_tensors, const int64_t* numel, const int8_t* const* m_code,
                         const uint8_t* const* v_code, const float* const* m_scale,
                         const float* const* v_scale, float* const* m, float* const* v,
                         int32_t block_size, void* stream);

/* Non-finite grad check (the "found inf" test of a mixed-precision step): writes 0 to the
 * device int32 *found_nonfinite, then 1 if any grad of the list, multiplied by
 * list->grad_unscale, is +-inf or NaN. Only the grad side of `list` is used (param may be
 * NULL). Pass the same flag as skip_if_set of the following step to skip it. */
int psadam_check_grads(const psadam_list* list, int32_t* found_nonfinite, void* stream);

/* Bytes of optimizer state for a tensor of numel params (PR #814's GetMemoryUsage), B =
 * block_size (ignored by modes 0 and 1): mode 0 = fp32 (8*numel), 1 = bf16 (4*numel),
 * 2 = 8-bit (2*numel + 8*ceil(numel/B)), 3 = fp32 m + 8-bit v (5*numel + 4*ceil(numel/B)).
 * Returns 0 for an unknown mode, numel < 0, or B < 1 in modes 2 and 3. */
size_t psadam_state_bytes(int32_t mode, int64_t numel, int32_t block_size);

/* 1 if a kernel of the library gave up a bounded wait on its own asynchronous copies since
 * the last call (its results are then not to be trusted), 0 if not, -1 if the device could
 * not be queried. The call first waits for all work on the current device (every stream,
 * cudaDeviceSynchronize), then takes the word and clears it in one atomic exchange on the
 * legacy default stream, so a fault is never lost between the read and the clear. A CTA
 * gives up as a whole (its threads agree at a barrier) and stores nothing of the block it was
 * waiting for; blocks it finished before keep their results. */
int32_t psadam_device_fault(void);

/* Self-test of the failure path above: one thread waits on a barrier that nothing completes,
 * gives up after `cycles` SM cycles and sets the fault word (so the next
 * psadam_device_fault() returns 1). It never faults or hangs the device. cycles must lie in
 * [0, 2^31], the step kernels' own limit (PSADAM_ERR_INVALID_ARG otherwise). */
int psadam_selftest_bounded_wait(int64_t cycles, void* stream);

/* Self-test of the update's own square root and quotient. Where every moment of a thread's
 * elements lies in [2^-60, 2^64] (with eps in [2^-60, 2^20]), the IEEE-exact step takes them
 * from the hardware's reciprocal approximations plus one fused multiply-add correction each
 * instead of IEEE sqrt and division; they must give the same bits. The call counts, on the
 * device, the results that differ from IEEE sqrt / division: mismatches[0] over every float in
 * [2^-102, 2^128) (root), [1] over pairs of significands a, b in [1, 2) (quotient; full = 1:
 * all 2^46 pairs, about a minute; full = 0: 2^36 of them), [2] exponent-scaling checks of the
 * approximations that extend [1] to every exponent of the domain, [3] the step's arithmetic
 * on 2^25 random elements per setting of three (fused switch against the IEEE per-element
 * update; p, m and v). Every count is 0 on a correct build. mismatches: host, 4 entries.
 * Synchronous on `stream`. PSADAM_ERR_INVALID_ARG for a null array or full not 0/1. */
int psadam_selftest_update_math(int32_t full, uint64_t* mismatches, void* stream);

/* Static, human-readable name of a psadam_status value. */
const char* psadam_status_string(int32_t status);

/* cudaError_t of the most recent PSADAM_ERR_CUDA on the calling thread (0 if none). */
int32_t psadam_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* PSADAM_H */
