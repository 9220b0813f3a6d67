/*
 * lora_linear.h -- C ABI of the fused LoRA linear layer for one GB300 (sm_103a).
 *
 * The layer (ch05 "Acceleration principles: Triton kernels and fused LoRA",
 * §5.3, LoRA equation; ch01 "Project background", §1.2, dW = (alpha/r) B A),
 * written for row-major token batches:
 *
 *     s  = alpha / r
 *     Y  = X W^T + s (X A^T) B^T                     (forward)
 *     dX = dY W + s (dY B) A                         (backward, W frozen)
 *     dA = s (dY B)^T X
 *     dB = s dY^T (X A^T)
 *
 * ch05 §5.3 lists the backward's gradients as dL/dX, dL/dW ("if trained"),
 * dL/dA and dL/dB; W is frozen here, so dW is not computed.
 *
 * Tensors (all row-major and contiguous, all of the same dtype):
 *     X  [M, d_in]      W [d_out, d_in]     A [r, d_in]     B [d_out, r]
 *     Y  [M, d_out]     dY [M, d_out]       dX [M, d_in]
 *     dA [r, d_in]      dB [d_out, r]
 * M is the number of tokens (batch x sequence).
 *
 * Conventions shared by every entry point:
 *  - Ownership: the caller allocates and owns every buffer (device memory
 *    unless stated).  The library never allocates, frees or synchronises
 *    (lora_device_status excepted, which synchronises by design).
 *  - Execution: all work is enqueued on `stream` (a cudaStream_t passed as a
 *    void*; NULL = the legacy default stream) and completes asynchronously.
 *  - Outputs are overwritten, never accumulated into.
 *  - Validation: every argument is checked on the host before anything is
 *    launched.  A failed check returns a status and launches nothing.
 *  - Errors: launch failures return LORA_ERR_CUDA.  Device-side waits are
 *    bounded; a wait that runs out sets a device status word read by
 *    lora_device_status() (the kernel then returns early and its outputs
 *    are undefined).
 *  - Determinism: fixed-order reductions only (no floating-point atomics);
 *    the same inputs give bit-identical outputs run to run.
 *  - Thread safety: calls from several host threads are safe; the timing
 *    hook below is per host thread.
 *
 * dtype LORA_BF16: bf16 tensors, fp32 accumulation on the tcgen05 tensor
 *   cores, one round-to-nearest-even to bf16 per output.  The low-rank
 *   intermediates s*X A^T and s*dY B are rounded once to bf16 (they are
 *   tensor-core operands).  Requirements: d_in % 8 == 0, d_out % 8 == 0
 *   (16-byte row pitch for the TMA copies), 1 <= r <= 256, all pointers
 *   16-byte aligned.
 * dtype LORA_FP32: fp32 tensors, the same decomposition on CUDA cores
 *   (FFMA, fp32 accumulation): a debug mode for exact-as-fp32 comparisons.
 *   Requirements: 1 <= r <= 256, pointers 16-byte aligned.
 */
#ifndef LORA_LINEAR_H
#define LORA_LINEAR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LORA_OK = 0,
    LORA_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misalignment    */
    LORA_ERR_UNSUPPORTED = 2,  /* valid but unsupported shape or device   */
    LORA_ERR_WORKSPACE = 3,    /* workspace missing or too small          */
    LORA_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed       */
    LORA_ERR_TIMEOUT = 5       /* a bounded device-side wait ran out      */
} lora_status_t;

typedef enum {
    LORA_BF16 = 0,
    LORA_FP32 = 1
} lora_dtype_t;

/* Bytes of the `saved` buffer that lora_linear_fwd fills and
 * lora_linear_bwd reads: the low-rank activation s*X A^T, kept in the
 * layouts the backward's tensor-core passes read.  0 when M == 0. */
size_t lora_linear_saved_bytes(int64_t M, int r, lora_dtype_t dtype);

/* Bytes of device workspace needed by lora_linear_fwd and lora_linear_bwd
 * for this shape (the larger of the two, including room to recompute the
 * saved activation when bwd gets saved == NULL).  May be 0. */
size_t lora_linear_workspace_bytes(int64_t M, int64_t d_in, int64_t d_out,
                                   int r, lora_dtype_t dtype);

/*
 * Forward: Y = X W^T + s (X A^T) B^T with s = alpha / r.
 * (ch05 §5.3: the fused forward writes Y once and keeps the low-rank
 * intermediate out of the output pass.)
 *
 *   X, W, A, B  in, device, layouts above.
 *   alpha, r    LoRA scale numerator and rank; s = alpha / r.
 *   M           tokens (>= 0; M == 0 is an empty batch and launches nothing).
 *   Y           out, device, [M, d_out].
 *   saved       out, device, lora_linear_saved_bytes(M, r, dtype) bytes;
 *               pass it unchanged to lora_linear_bwd.
 *   workspace   device scratch of workspace_bytes bytes (>= the size from
 *               lora_linear_workspace_bytes; may be NULL if that is 0).
 *
 * Kernels: one skinny tensor-core pass writes s*X A^T (rounded to the
 * dtype), then one K-extended GEMM computes [X | s X A^T] . [W | B]^T in a
 * single fp32 accumulator and writes Y.
 */
lora_status_t lora_linear_fwd(const void *X, const void *W, const void *A,
                              const void *B, float alpha, int r, int64_t M,
                              int64_t d_in, int64_t d_out, lora_dtype_t dtype,
                              void *Y, void *saved, void *workspace,
                              size_t workspace_bytes, void *stream);

/*
 * Backward for the loss gradient dY = dL/dY:
 *   dX = dY W + s (dY B) A,  dA = s (dY B)^T X,  dB = s dY^T (X A^T).
 *
 *   dY, X, W, A, B  in, device.
 *   saved       in, device: the buffer lora_linear_fwd filled for the same
 *               X, A, alpha and r; or NULL, in which case s*X A^T is
 *               recomputed into the workspace first.
 *   dX          out, [M, d_in], or NULL to skip the dX GEMM.
 *   dA          out, [r, d_in].   dB  out, [d_out, r].
 *               With M == 0, dA and dB are set to zero.
 *   workspace   device scratch (lora_linear_workspace_bytes).
 *
 * Kernels: s*dY B is computed once (skinny tensor-core pass) and reused by
 * the K-extended dX GEMM over [dY | s dY B] . [W ; A] and by the dA pass;
 * dA and dB are skinny split-K passes whose partial sums are combined in
 * shared memory across a thread-block cluster in a fixed order.  The dA
 * pass starts on the SMs the dX GEMM frees in its last wave; work queued
 * after the call on the same stream still starts only once both are done.
 */
lora_status_t lora_linear_bwd(const void *dY, const void *X, const void *W,
                              const void *A, const void *B, const void *saved,
                              float alpha, int r, int64_t M, int64_t d_in,
                              int64_t d_out, lora_dtype_t dtype, void *dX,
                              void *dA, void *dB, void *workspace,
                              size_t workspace_bytes, void *stream);

/*
 * Backward without a caller-supplied workspace.  (The pages have no
 * counterpart: this is a convenience of this library.)
 *
 * For callers that cannot allocate device memory when they call the
 * backward -- for example a plugin running inside a host application that
 * owns all device memory and gives it no allocator, or a latency-critical
 * loop that must not call cudaMalloc (which may synchronise the device)
 * after start-up.  Arguments and results are those of lora_linear_bwd; the
 * scratch the kernels need comes from one array of
 * LORA_NOALLOC_SCRATCH_BYTES bytes that the library holds in device memory
 * on every GPU that loads it, until the process exits.
 *
 *  - Limit: shapes whose backward needs more than LORA_NOALLOC_SCRATCH_BYTES
 *    of scratch (lora_linear_workspace_bytes minus the recompute room when
 *    saved != NULL) are rejected with LORA_ERR_UNSUPPORTED and nothing runs.
 *    With saved != NULL, bf16 needs about 2*r_pad*(d_out + 2*M) bytes
 *    (r_pad = r rounded up to 16); every workload of the benchmark fits.
 *  - No allocation: it calls no cudaMalloc/cudaFree or allocating routine.
 *  - Set-up: the first call on each device looks up the array's device
 *    address (with that device current) and caches it; make that first call
 *    before any stream capture.  The cached address (like the device status
 *    word's, cached by every entry point) belongs to the device's primary
 *    context and does not survive cudaDeviceReset: a process that resets a
 *    device must not call into this library on it afterwards.
 *  - Errors: the argument checks of lora_linear_bwd, then the size limit
 *    below, then the device check that every entry point makes (a device
 *    this library was not built for gives LORA_ERR_UNSUPPORTED, as from
 *    lora_linear_bwd), all before the array is looked up.
 *  - Sharing: every call uses the same array.  Calls whose work overlaps on
 *    the GPU (other streams, other host threads) race on it and give wrong
 *    results; order them (one stream, or events).  The array keeps the last
 *    call's contents; nothing in it needs to start at zero.
 */
#define LORA_NOALLOC_SCRATCH_BYTES (16u << 20) /* 16 MiB */
lora_status_t lora_linear_bwd_noalloc(const void *dY, const void *X,
                                      const void *W, const void *A,
                                      const void *B, const void *saved,
                                      float alpha, int r, int64_t M,
                                      int64_t d_in, int64_t d_out,
                                      lora_dtype_t dtype, void *dX, void *dA,
                                      void *dB, void *stream);

/* Human-readable name of a status code (static string). */
const char *lora_status_string(lora_status_t status);

/* Detail message of the last failed call on this host thread ("" if none). */
const char *lora_last_error(void);

/* Reads the device status word that bounded waits set when they run out.
 * Synchronises the current device.  Returns LORA_OK, LORA_ERR_TIMEOUT or
 * LORA_ERR_CUDA.  If clear != 0 the word is reset to zero. */
lora_status_t lora_device_status(int clear);

/* Number of kernels this library has launched in this process. */
uint64_t lora_launch_count(void);

/* Kernel kinds reported by the timing hook. */
typedef enum {
    LORA_K_PREP = 0,      /* transpose / pad of B (tiny)                     */
    LORA_K_DOWN_FWD = 1,  /* s X A^T             (skinny, HBM-bound)         */
    LORA_K_MAIN_FWD = 2,  /* [X|sXA^T][W|B]^T    (K-extended GEMM)           */
    LORA_K_DOWN_BWD = 3,  /* s dY B              (skinny, HBM-bound)         */
    LORA_K_MAIN_BWD = 4,  /* [dY|sdYB][W;A]      (K-extended GEMM)           */
    LORA_K_GRAD_A = 5,    /* dA = (s dY B)^T X   (skinny split-K)            */
    LORA_K_GRAD_B = 6,    /* dB = dY^T (s X A^T) (skinny split-K)            */
    LORA_K_DOWN_BWD_GRAD_B = 7, /* s dY B and dB in one launch (both read dY) */
    LORA_K_SWIGLU_GRAD = 8,     /* SwiGLU pair: elementwise d_gate, d_up      */
    LORA_K_QUANT = 9,           /* fp8 variant: e4m3 quantisation of X or dY  */
    LORA_K_GRAD_A_B = 10        /* dA and dB in one launch, after the dX GEMM */
} lora_kernel_kind_t;

/*
 * Timing hook (per host thread).  While set, kernel launch j of the library
 * (j < n_pairs, counted from this call) records events[2j] on its stream
 * before the launch and events[2j+1] after it (cudaEvent_t handles passed
 * as void*), and stores its lora_kernel_kind_t in kinds[j] (kinds may be
 * NULL).  Pass events = NULL to clear.  lora_timing_used() returns how many
 * pairs have been recorded since the hook was set.
 */
lora_status_t lora_set_timing_events(void *const *events, int *kinds,
                                     int n_pairs);
int lora_timing_used(void);

/*
 * Test hook for the bounded device-side waits (the pages have no
 * counterpart; it exists so that the timeout path can be exercised without
 * faulting or hanging a GPU).  The next n bf16 backward dA passes (the last
 * launch of lora_linear_bwd, which carries dB as well when the GEMMs run
 * 256 x 512 tiles) launched by this process (any thread) leave the first
 * pipeline stage of their first dA CTA unfilled.  That CTA's MMA
 * wait then runs out after the wait limit (about 2 s), the kernel leaves
 * through its abort path (no fault, no hang), the caller's next
 * lora_device_status() returns LORA_ERR_TIMEOUT, and dA of that call is
 * undefined (dX and dB are complete).  n = 0 cancels.  Returns
 * LORA_ERR_INVALID_ARG for n < 0.
 */
lora_status_t lora_debug_withhold_arrive(int n);

/*
 * Test hook for the main GEMM's abort path (the pages have no counterpart).
 * The next n bf16 backward dX GEMMs (not the 4-bit layer's) launched by this
 * process leave one pipeline stage of the first CTA pair half filled: the
 * odd CTA never loads its first stage.  The MMA wait for it runs out after
 * the wait limit (about 2 s); both CTAs leave through their abort paths,
 * the even CTA first settling every phase of the pair's stage ring, so that
 * no copy is in flight when either CTA exits (no fault, no hang).  The
 * caller's next lora_device_status() returns LORA_ERR_TIMEOUT; dX of that
 * call is undefined.  n = 0 cancels; LORA_ERR_INVALID_ARG for n < 0.
 */
lora_status_t lora_debug_withhold_gemm_stage(int n);

/*
 * Test hook of the main GEMMs' tile width (the pages have no counterpart).
 * The GEMMs of the bf16, fp8 and SwiGLU layers run 256 x 512 or 256 x 256
 * pair tiles (either with the split of a short last wave where it applies),
 * chosen per GEMM and shape by a cost model of the waves.  width = 256 or
 * 512 forces that width for every later call in this process (512 only
 * where it is built: not for the 4-bit layer's GEMMs); 0 restores the cost
 * model.  Results differ between widths only by the rounding order of the
 * split tiles.  Workspace sizes do not depend on it.  Returns
 * LORA_ERR_INVALID_ARG for any other width.
 */
lora_status_t lora_debug_gemm_width(int width);

#ifdef __cplusplus
}
#endif

#endif /* LORA_LINEAR_H */
