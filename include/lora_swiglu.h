/*
 * lora_swiglu.h -- the SwiGLU gate/up pair of LoRA layers, fused.
 *
 * ch05 "Acceleration principles: Triton kernels and fused LoRA", §5.6 (fused
 * SwiGLU): SwiGLU(x) = (W_g x * sigma(W_g x)) * W_u x, whose SiLU and
 * elementwise product are fused into the matmul epilogue; here each of the
 * gate and up projections is a LoRA layer of §5.3 (lora_linear.h) with the
 * same rank r and scale s = alpha / r.  Row-major, one token per row:
 *
 *   gate = X Wg^T + s (X Ag^T) Bg^T     up = X Wu^T + s (X Au^T) Bu^T
 *   H    = silu(gate) * up,             silu(z) = z / (1 + e^-z)
 *
 * Backward for the upstream gradient dH (Wg, Wu frozen):
 *   d_gate = dH * up * silu'(gate),  d_up = dH * silu(gate)
 *   dX  = d_gate Wg + s (d_gate Bg) Ag + d_up Wu + s (d_up Bu) Au
 *   dAg = s (d_gate Bg)^T X,  dBg = s d_gate^T (X Ag^T)   (same for up)
 *
 * Shapes: X [M, d_in]; Wg, Wu [d_ff, d_in]; Ag, Au [r, d_in];
 * Bg, Bu [d_ff, r]; H, dH [M, d_ff]; dX [M, d_in].  All bf16, row-major,
 * contiguous, 16-byte aligned device pointers.  bf16 only (LORA_FP32 returns
 * LORA_ERR_UNSUPPORTED); d_in and d_ff multiples of 8; 1 <= r <= 256.
 * Accumulation in fp32; gate and up are rounded to bf16 when saved, H once.
 *
 * Errors, streams, the status word and the timing hook are those of
 * lora_linear.h.  Nothing is allocated; no host synchronisation.
 */
#ifndef LORA_SWIGLU_H
#define LORA_SWIGLU_H

#include "lora_linear.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Bytes of the `saved` buffer the forward fills and the backward reads:
 * gate and up [M, d_ff] bf16, s X Ag^T and s X Au^T [M, 2 r_pad] and their
 * transposes (r_pad = r rounded up to 16).  0 for M = 0 or bad arguments. */
size_t lora_swiglu_saved_bytes(int64_t M, int64_t d_ff, int r);

/* Bytes of device workspace needed by lora_swiglu_fwd and lora_swiglu_bwd on
 * the current device (sized for a GB300 when none is usable). */
size_t lora_swiglu_workspace_bytes(int64_t M, int64_t d_in, int64_t d_ff, int r);

/*
 * Forward: H = silu(gate) * up, with gate and up written to `saved` for the
 * backward.  `saved` may be NULL (inference): then nothing is kept and the
 * forward skips writing gate and up (a third less output traffic).  Two
 * launches: one skinny pass for [s X Ag^T | s X Au^T], then one tensor-core
 * GEMM whose CTA pairs compute 128 columns of the gate
 * projection (even CTA) and of the up projection (odd CTA) for the same
 * 256 rows, and apply silu(gate) * up in the epilogue.
 *   workspace   device scratch of lora_swiglu_workspace_bytes bytes.
 */
lora_status_t lora_swiglu_fwd(const void *X, const void *Wg, const void *Ag, const void *Bg,
                              const void *Wu, const void *Au, const void *Bu, float alpha,
                              int r, int64_t M, int64_t d_in, int64_t d_ff, lora_dtype_t dtype,
                              void *H, void *saved, void *workspace, size_t workspace_bytes,
                              void *stream);

/*
 * Backward: dX (may be NULL to skip it), dAg, dBg, dAu, dBu, from dH and the
 * forward's `saved` buffer (required).  Gradients are overwritten.
 */
lora_status_t lora_swiglu_bwd(const void *dH, const void *X, const void *Wg, const void *Ag,
                              const void *Bg, const void *Wu, const void *Au, const void *Bu,
                              const void *saved, float alpha, int r, int64_t M, int64_t d_in,
                              int64_t d_ff, lora_dtype_t dtype, void *dX, void *dAg, void *dBg,
                              void *dAu, void *dBu, void *workspace, size_t workspace_bytes,
                              void *stream);

#ifdef __cplusplus
}
#endif

#endif /* LORA_SWIGLU_H */
