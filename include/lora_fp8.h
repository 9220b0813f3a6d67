/*
 * lora_fp8.h -- the LoRA linear layer with an fp8 (e4m3) frozen-W product.
 *
 * ch05 "Acceleration principles: Triton kernels and fused LoRA", §5.9 (fp8
 * mixed-precision training on fp8 tensor cores), applied to the frozen
 * weight of the LoRA layer of §5.3 (lora_linear.h); the low-rank extension
 * and dA / dB stay in bf16.  The pages fix no format or scaling recipe; the
 * one used here:
 *   - e4m3 (OCP: bias 7, largest finite value 448), round to nearest even,
 *     saturating;
 *   - power-of-two scales, so dividing by one is exact: a block with
 *     absolute maximum a > 0 gets 2^e, e the smallest integer with
 *     a <= 448 * 2^e (a = 0 gets 1);
 *   - W: one scale for the whole tensor, quantised once (it is frozen) in
 *     both orientations; X (forward) and dY (backward): one scale per row,
 *     quantised on every call.
 * With Q(.) the dequantised value (code times scale), s = alpha / r:
 *   Y  = Q(X) Q(W)^T + s (X A^T) B^T
 *   dX = Q(dY) Q(W)  + s (dY B) A,   dA = s (dY B)^T X,   dB = s dY^T (X A^T)
 * The fp32 accumulator of each tensor-core tile takes the e4m3 products
 * (kind::f8f6f4) and the bf16 extension (kind::f16), whose low-rank
 * activation is divided by the same product of power-of-two scales; the
 * epilogue multiplies by the row's scale times W's scale and rounds once to
 * bf16.
 *
 * bf16 X, A, B, dY, Y, dX, dA, dB as in lora_linear.h; d_in and d_out
 * multiples of 16; 1 <= r <= 256.  Errors, streams, the status word and the
 * timing hook are those of lora_linear.h.  Nothing is allocated.
 */
#ifndef LORA_FP8_H
#define LORA_FP8_H

#include "lora_linear.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Bytes of device workspace lora_fp8_quantize_w needs (a few words). */
size_t lora_fp8_quantize_w_workspace_bytes(void);

/*
 * Quantise the frozen W [d_out, d_in] (bf16) once: Wq [d_out, d_in] and its
 * transpose WqT [d_in, d_out] (e4m3 bytes), w_scale (one float, device).
 */
lora_status_t lora_fp8_quantize_w(const void *W, int64_t d_out, int64_t d_in, void *Wq,
                                  void *WqT, float *w_scale, void *workspace,
                                  size_t workspace_bytes, void *stream);

/*
 * The per-row quantiser the forward applies to X (and the backward to dY),
 * exposed on its own: x [rows, cols] bf16 (cols a multiple of 16) -> q
 * [rows, cols] e4m3 bytes and scale [rows] floats (powers of two).
 */
lora_status_t lora_fp8_quantize_rows(const void *x, int64_t rows, int64_t cols, void *q,
                                     float *scale, void *stream);

/* Bytes of device workspace needed by lora_fp8_fwd and lora_fp8_bwd. */
size_t lora_fp8_workspace_bytes(int64_t M, int64_t d_in, int64_t d_out, int r);

/*
 * Forward.  `saved` (lora_linear_saved_bytes(M, r, LORA_BF16) bytes) keeps
 * the low-rank activation for lora_fp8_bwd.  Three launches: quantise X, the
 * skinny s X A^T pass, the fp8 GEMM (and a pad of B when r % 8 != 0).
 */
lora_status_t lora_fp8_fwd(const void *X, const void *Wq, const float *w_scale, const void *A,
                           const void *B, float alpha, int r, int64_t M, int64_t d_in,
                           int64_t d_out, void *Y, void *saved, void *workspace,
                           size_t workspace_bytes, void *stream);

/*
 * Backward from dY and the forward's `saved` buffer (required).  dX may be
 * NULL to skip it.  Gradients are overwritten.
 */
lora_status_t lora_fp8_bwd(const void *dY, const void *X, const void *WqT, const float *w_scale,
                           const void *A, const void *B, const void *saved, float alpha, int r,
                           int64_t M, int64_t d_in, int64_t d_out, void *dX, void *dA, void *dB,
                           void *workspace, size_t workspace_bytes, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* LORA_FP8_H */
