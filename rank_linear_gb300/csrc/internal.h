// internal.h -- host-side interfaces shared by the library's translation
// units.  Not part of the public ABI (that is include/lora_linear.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace lora {

// ---- K-extended tensor-core GEMM (bf16 in, fp32 accumulate, bf16 out) ----
//   out[m, n] = sum_{k < K1} A(m, k) B(n, k)  +  sum_{k < k_ext} A2(m, k) B2(n, k)
// Computed in 256 x bn pair tiles (bn from main_gemm_pick_bn).
// A / A2 are K-major [M, K] tensor maps (box 64 x 128).  B / B2 are K-major
// [N, K] maps (box 64 x bn/2) or, with b_mn, MN-major [K, N] maps
// (box 64 x 64).
struct MainGemmArgs {
  CUtensorMap tmA, tmB, tmA2, tmB2;
  int M = 0, N = 0;
  int kb_main = 0;  // number of 64-wide K blocks of the first segment
  int k_ext = 0;    // K of the extension: a multiple of 16 in [0, 256]
  void *out = nullptr;
  int64_t ldo = 0;  // row pitch of out, elements
  bool b_mn = false;
  int bn = 256;     // pair-tile width
  // Split of the last, partial wave (see main_gemm_split): its split_rem
  // tiles are computed as split_k K-ranges each, on different pairs, whose
  // fp32 partials meet in `partials`; `counters` (2 * split_rem words) must
  // be zero when the kernel starts.
  int split_k = 1, split_rem = 0;
  float *partials = nullptr;
  unsigned *counters = nullptr;
  unsigned *dev_status = nullptr;
  // Gated (SwiGLU) pair: the pair's even CTA multiplies by B = tmB and
  // B2 = tmB2 (gate projection), the odd CTA by tmB3 and tmB4 (up
  // projection), whose extension columns are read ext_shift columns earlier
  // (K coordinate k - ext_shift) so that they meet the second half of the
  // extension A = [sH_g | sH_u].  A pair tile is 256 rows x 128 columns of
  // both projections; out = silu(gate) * up, aux0 = gate, aux1 = up (bf16,
  // row pitch ldo; aux0/aux1 may be null).  N counts output columns.
  bool gated = false;
  CUtensorMap tmB3, tmB4;
  int ext_shift = 0;
  void *aux0 = nullptr, *aux1 = nullptr;
  // Second B segment of the main K range (not gated): K blocks >= kb_switch
  // read B from tmB3 at K coordinate (kb - kb_switch) * 64.  -1: none.
  int kb_switch = -1;
  // fp8 main segment: A and B are e4m3 K-major maps (box 128 bytes x rows),
  // kb_main counts 128-wide K blocks, the extension stays bf16; the epilogue
  // multiplies row m of the result by row_scale[m] (times w_scale[0] if given).
  bool fp8 = false;
  const float *row_scale = nullptr, *w_scale = nullptr;
  // 4-bit W main segment (bn 256): tmB holds the packed codes [d_out][d_in/2]
  // bytes (box 32 bytes x 128 rows; with b_mn box 64 bytes x 64 rows) and
  // tmB3 the bf16 group scales [d_in/64][d_out] (box 128 x 1; with b_mn
  // 64 x 2).  Each CTA dequantises its half of the B tile to bf16 in shared
  // memory before the MMAs read it.
  bool q4 = false;
  // 256 x 512 pair tiles (two N = 256 MMAs per K step sharing A; all but the
  // 4-bit W; gated: 256 outputs of both projections); from main_gemm_plan
  bool wide = false;
  // The output as a TMA map (bf16 [M][N] with row pitch ldo, box 64 x 32,
  // 128-byte swizzle): the wide tiles' drain writes through it, and the
  // gated pair's through tmAux0 / tmAux1 (the same over aux0 / aux1) too.
  // Needed when wide (tmAux0 / tmAux1: when gated and aux0 / aux1 given).
  CUtensorMap tmOut, tmAux0, tmAux1;
  // Test hook of the abort path (not with 4-bit W): the odd CTA of the first
  // pair never loads its first stage.
  int withhold = 0;
};
constexpr int kMainBM = 128, kMainBK = 64;
int main_gemm_pick_bn(int M, int N, int num_sms);
// Number of CTA pairs the main GEMM runs on (resident clusters of two).
int main_gemm_pairs(bool b_mn, int num_sms);
struct MainSplit {
  int k = 1, rem = 0;
  size_t partial_bytes = 0, counter_bytes = 0;
  bool wide = false;  // 256 x 512 tiles
};
// Tail split for an M x N output on `pairs` CTA pairs in 256 x tile_n pair
// tiles: the last wave's rem tiles are split two ways (K ranges) when
// 2 * rem <= pairs.  For the gated pair pass N = 2 x roundup(output columns,
// 128): a pair tile of 256 (512) columns holds 128 (256) outputs of both
// projections.
MainSplit main_gemm_split(int M, int N, int pairs, int tile_n = 256);
// The plain layer's choice between 256 x 512 and 256 x 256 tiles, each with
// its tail split where that applies, by a cost model of the waves that
// weighs a split's fix-up against the tile's K blocks (kb_total, both
// segments).  allow_wide false: 256-wide tiles only, as main_gemm_split.
MainSplit main_gemm_plan(int M, int N, int pairs, bool allow_wide, int kb_total);
// Test hook: 0 = choose by the cost model, 256 or 512 = that width only
// (512 where allowed).
void main_gemm_force_width(int w);
cudaError_t launch_main_gemm(const MainGemmArgs &a, int num_sms, cudaStream_t s);

// ---- skinny tensor-core pass with cluster split-K -------------------------
//   acc[row, j] = sum_k A(row, k) B(j, k),  row < rows, j < RP (RP = r_pad)
//   out0[row * ld0 + j] = bf16(scale * acc)  for j < n0   (row-major, optional)
//   out1[j * ld1 + row] = bf16(scale * acc)  for j < n1   (transposed, optional)
// A is K-major [rows, K] (box 64 x 128) or, with a_mn, MN-major [K, rows]
// (box 64 x 64).  B is K-major [RP, K] (box 64 x RP) or, with b_mn,
// MN-major [K, >= 1 columns] (box 64 x 64; columns past the tensor read as
// zero and the MMA runs on whole 64-wide column blocks).  The K range is
// split over the CTAs of a cluster whose partial sums meet in distributed
// shared memory and are added in cluster-rank order.
struct SkinnyArgs {
  // optional: zero `zero_words` 32-bit words at `zero_ptr` (the next main
  // GEMM's split counters) once the preceding kernel has finished
  unsigned *zero_ptr = nullptr;
  int zero_words = 0;
  CUtensorMap tmA, tmB;
  bool a_mn = false, b_mn = false;
  int rows = 0, RP = 16, K = 0;
  float scale = 1.f;
  void *out0 = nullptr;
  int64_t ld0 = 0;
  int n0 = 0;
  void *out1 = nullptr;
  int64_t ld1 = 0;
  int n1 = 0;
  unsigned *dev_status = nullptr;
  // Test hook of the bounded waits: the first CTA's producer leaves its
  // first stage unfilled, so that CTA's MMA wait runs out (problem 0 only).
  int withhold_first_stage = 0;
  // Optional per-row divisor of out0 (powers of two, so exact): out0 row m
  // is divided by row_div[m]; out1 is not.
  const float *row_div = nullptr;
  // The preceding kernel is a main GEMM (it signals its dependents only once
  // every kernel before it has finished) and writes nothing this launch
  // reads: skip the wait at the start, so the launch streams on the SMs the
  // GEMM frees; the last cluster waits before it leaves, so the launch still
  // ends after the GEMM.  Not allowed with zero_ptr.
  int after_gemm = 0;
  // This pass feeds a main GEMM launched right after it, which needs its
  // result only at the end of each tile: when one CTA per 128 rows makes at
  // most kSkinnyFeedMaxCtas CTAs and K spans at most kSkinnyFeedMaxKb
  // blocks, run that way (no K split, no cluster), so that the GEMM's CTA
  // pairs start on the other SMs at once instead of waiting for this pass to
  // leave them.
  int feeds_gemm = 0;
  // With feeds_gemm: the GEMM gives every CTA pair two tiles or more, so the
  // pairs that start when this pass leaves end last; its CTAs (one per SM,
  // beside the GEMM's) then take a ring of twice the depth and leave sooner.
  int deep_ring = 0;
  // Largest K split (cluster size) the launch may take; 0: no limit.  Must
  // depend on the shape only, so that results do not depend on whether a
  // GEMM runs beside the pass.
  int max_split = 0;
};
constexpr int kSkinnyFeedMaxCtas = 64;
// One CTA streams its 128 rows at about 40 GB/s, so a 128-block (K = 8192)
// pass holds its SMs for ~50 us.  Longer, the pairs it delays start a full
// pass behind the others, which costs more than the overlap saves (at
// K = 14336 a 64-CTA pass held 64 SMs for ~90 us): such a pass runs split
// over all SMs before the GEMM instead.
constexpr int kSkinnyFeedMaxKb = 128;
// Runs one or two independent problems in one launch.
cudaError_t launch_skinny(const SkinnyArgs *probs, int nprob, int num_sms, cudaStream_t s);
int skinny_split(int rows, int K, int num_sms);

// ---- fp32 CUDA-core GEMM (debug dtype) ------------------------------------
//   c[m * c0 + n * c1] = alpha * (sum_{k<K1} a1(m,k) b1(k,n) + sum_{k<K2} a2(m,k) b2(k,n))
// with x(i, k) = p[i * s0 + k * s1] for an A operand and
//      x(k, n) = p[k * s0 + n * s1] for a B operand.
struct F32Operand {
  const float *p = nullptr;
  int64_t s0 = 0, s1 = 0;
};
struct F32GemmArgs {
  int M = 0, N = 0, K1 = 0, K2 = 0;
  F32Operand a1, b1, a2, b2;
  float alpha = 1.f;
  float *c = nullptr;
  int64_t c0 = 0, c1 = 0;
};
cudaError_t launch_f32_gemm(const F32GemmArgs &a, cudaStream_t s);

// ---- small bf16 copies of the adapter B ----------------------------------
// Bt[j * d_out + o] = (j < r) ? B[o * r + j] : 0     for j < r_pad
cudaError_t launch_transpose_pad_bf16(const void *B, int d_out, int r, int r_pad, void *Bt,
                                      cudaStream_t s);
// Bp[o * r_pad + j] = (j < r) ? B[o * r + j] : 0     for j < r_pad
cudaError_t launch_pad_cols_bf16(const void *B, int d_out, int r, int r_pad, void *Bp,
                                 cudaStream_t s);
// SwiGLU backward, elementwise: D = [dH * up * silu'(gate) | dH * silu(gate)]
// ([M][2 half] bf16, columns [d_ff, half) of each half zero).
cudaError_t launch_swiglu_grad_bf16(const void *dH, const void *gate, const void *up, int64_t M,
                                    int d_ff, int half, void *D, int num_sms, cudaStream_t s);
// dst [2 r_pad][d_in] = [Ag (r rows) ; 0 ; Au (r rows) ; 0].
cudaError_t launch_stack_rows_bf16(const void *Ag, const void *Au, int r, int r_pad, int64_t d_in,
                                   void *dst, cudaStream_t s);
// e4m3 with power-of-two scales: one scale per row of x [rows][cols]
// (cols % 8 == 0, cols <= 65536) -> q [rows][cols] bytes and scale [rows]
// floats, the row's scale times mul[0] when mul is given.
cudaError_t launch_quant_rows_e4m3(const void *x, int64_t rows, int64_t cols, void *q,
                                   float *scale, const float *mul, cudaStream_t s);
// Symmetric 4-bit W [d_out][d_in] (d_in % 64 == 0): packed codes
// [d_out][d_in / 2] bytes and bf16 group scales [d_in / 64][d_out]; and back.
cudaError_t launch_quant_q4(const void *w, int d_out, int d_in, void *codes, void *scales,
                            cudaStream_t s);
cudaError_t launch_dequant_q4(const void *codes, const void *scales, int d_out, int d_in, void *w,
                              int num_sms, cudaStream_t s);
// One scale for all of w [rows][cols]: q [rows][cols], qT [cols][rows],
// scale[0]; amax_bits is one word of device scratch.
cudaError_t launch_quant_tensor_e4m3(const void *w, int rows, int cols, unsigned *amax_bits,
                                     void *q, void *qT, float *scale, int num_sms,
                                     cudaStream_t s);
// out [cols][r_pad] = in^T / scale[0] for in [r][cols] (no scale: 1), zero-padded.
cudaError_t launch_transpose_scale_bf16(const void *in, int r, int64_t cols, int r_pad,
                                        const float *scale, void *out, cudaStream_t s);

}  // namespace lora
