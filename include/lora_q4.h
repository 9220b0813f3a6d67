/*
 * lora_q4.h -- the LoRA linear layer over a 4-bit frozen W (QLoRA-style).
 *
 * The frozen base weight of the LoRA layer of ch05 "Acceleration
 * principles: Triton kernels and fused LoRA", §5.3 (lora_linear.h), held in
 * 4 bits as in the Unsloth inference notes ("4-bit quantisation with
 * in-register dequantisation": weights read from HBM in a compact INT4
 * format and turned back into bf16 on chip, with their scales, right before
 * the tensor cores use them).  The pages fix no layout; the one used here:
 *   - symmetric INT4, q in [-8, 7], stored as the code q + 8;
 *   - one bf16 scale per group of 64 consecutive weights of a row of W
 *     (along d_in): scale = bf16(absmax / 7), 1 for an all-zero group, both
 *     the division and q = clamp(rint(w / scale), -8, 7) in IEEE fp32,
 *     rounding to nearest even;
 *   - the dequantised weight Wd = bf16((code - 8) * scale), the exact
 *     product rounded once.
 * Storage: codes [d_out][d_in / 2] bytes, element 2j of a row in the low
 * nibble of byte j and 2j + 1 in its high nibble; scales [d_in / 64][d_out]
 * bf16 (the scales of one group of columns are contiguous).  One copy serves
 * both the forward (W read along d_in) and the backward (W read along
 * d_out).
 *
 * With s = alpha / r the layer computes, in bf16 with fp32 accumulation:
 *   Y  = X Wd^T + s (X A^T) B^T
 *   dX = dY Wd + s (dY B) A,   dA = s (dY B)^T X,   dB = s dY^T (X A^T)
 * The main GEMMs stage the codes and scales of a K block in shared memory,
 * where four warps per CTA expand them to the bf16 tile the tensor cores
 * read; Wd never exists in HBM.
 *
 * Shapes: d_in a multiple of 64, d_out a multiple of 8, 1 <= r <= 256.
 * X, A, B, dY, Y, dX, dA, dB are as in lora_linear.h (bf16, row-major); the
 * saved buffer and the workspace are those of lora_linear_fwd /
 * lora_linear_bwd with LORA_BF16 (lora_linear_saved_bytes,
 * lora_linear_workspace_bytes).  Errors, streams, the status word and the
 * timing hook are those of lora_linear.h.  Nothing is allocated.
 */
#ifndef LORA_Q4_H
#define LORA_Q4_H

#include "lora_linear.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Quantise the frozen W [d_out, d_in] (bf16, device) once: codes
 * [d_out, d_in / 2] bytes and scales [d_in / 64, d_out] bf16 (device).  One
 * launch.
 */
lora_status_t lora_q4_quantize_w(const void *W, int64_t d_out, int64_t d_in, void *codes,
                                 void *scales, void *stream);

/* Wd [d_out, d_in] (bf16, device) from codes and scales.  One launch. */
lora_status_t lora_q4_dequantize_w(const void *codes, const void *scales, int64_t d_out,
                                   int64_t d_in, void *Wd, void *stream);

/*
 * Forward.  `saved` (lora_linear_saved_bytes(M, r, LORA_BF16) bytes) keeps
 * the low-rank activation for lora_q4_bwd.  Two launches (three when
 * r % 8 != 0): the skinny s X A^T pass and the dequantising GEMM.
 */
lora_status_t lora_q4_fwd(const void *X, const void *codes, const void *scales, const void *A,
                          const void *B, float alpha, int r, int64_t M, int64_t d_in,
                          int64_t d_out, void *Y, void *saved, void *workspace,
                          size_t workspace_bytes, void *stream);

/*
 * Backward from dY and the forward's `saved` buffer (NULL: recomputed into
 * the workspace, as in lora_linear_bwd).  dX may be NULL to skip it.
 * Gradients are overwritten.
 */
lora_status_t lora_q4_bwd(const void *dY, const void *X, const void *codes, const void *scales,
                          const void *A, const void *B, const void *saved, float alpha, int r,
                          int64_t M, int64_t d_in, int64_t d_out, void *dX, void *dA, void *dB,
                          void *workspace, size_t workspace_bytes, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* LORA_Q4_H */
