// simt.cu -- CUDA-core kernels: the fp32 debug GEMM that runs the same
// decomposition as the bf16 tensor-core path, and the small copies of the
// adapter B that the tensor-core path reads.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "internal.h"
#include "ptx.cuh"

namespace lora {
namespace {

constexpr int TM = 64, TN = 64, TK = 16;  // block tile; 16 x 16 threads, 4 x 4 outputs each

// c = alpha * (A1 B1 + A2 B2) with strided operands, fp32 FFMA, one
// accumulator per output, K visited in increasing order (segment 1 first).
__global__ void __launch_bounds__(256) k_f32_gemm(F32GemmArgs a) {
  __shared__ float As[TK][TM + 1];
  __shared__ float Bs[TK][TN + 1];
  griddep_wait();
  griddep_launch_dependents();
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int m0 = blockIdx.y * TM, n0 = blockIdx.x * TN;
  float acc[4][4] = {};
  for (int seg = 0; seg < 2; ++seg) {
    const int K = seg == 0 ? a.K1 : a.K2;
    const F32Operand A = seg == 0 ? a.a1 : a.a2;
    const F32Operand B = seg == 0 ? a.b1 : a.b2;
    for (int k0 = 0; k0 < K; k0 += TK) {
      for (int i = threadIdx.x; i < TK * TM; i += 256) {
        const int kk = i / TM, mm = i % TM;
        const int m = m0 + mm, k = k0 + kk;
        As[kk][mm] = (m < a.M && k < K) ? A.p[m * A.s0 + k * A.s1] : 0.f;
      }
      for (int i = threadIdx.x; i < TK * TN; i += 256) {
        const int kk = i / TN, nn = i % TN;
        const int n = n0 + nn, k = k0 + kk;
        Bs[kk][nn] = (n < a.N && k < K) ? B.p[k * B.s0 + n * B.s1] : 0.f;
      }
      __syncthreads();
#pragma unroll
      for (int kk = 0; kk < TK; ++kk) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(As[kk][ty + 16 * i], Bs[kk][tx + 16 * j], acc[i][j]);
      }
      __syncthreads();
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int m = m0 + ty + 16 * i, n = n0 + tx + 16 * j;
      if (m < a.M && n < a.N) a.c[m * a.c0 + n * a.c1] = a.alpha * acc[i][j];
    }
}

// Bt[j][o] = B[o][j] (zero for j >= r), through a 32 x 32 shared tile.
__global__ void k_transpose_pad(const __nv_bfloat16 *__restrict__ B, int d_out, int r, int r_pad,
                                __nv_bfloat16 *__restrict__ Bt) {
  __shared__ __nv_bfloat16 tile[32][33];
  griddep_wait();
  griddep_launch_dependents();
  const int o0 = blockIdx.x * 32, j0 = blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int o = o0 + i, j = j0 + threadIdx.x;
    tile[i][threadIdx.x] = (o < d_out && j < r) ? B[static_cast<int64_t>(o) * r + j]
                                                : __float2bfloat16_rn(0.f);
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int j = j0 + i, o = o0 + threadIdx.x;
    if (j < r_pad && o < d_out) Bt[static_cast<int64_t>(j) * d_out + o] = tile[threadIdx.x][i];
  }
}

// Bp[o][j] = B[o][j] (zero for r <= j < r_pad).
__global__ void k_pad_cols(const __nv_bfloat16 *__restrict__ B, int d_out, int r, int r_pad,
                           __nv_bfloat16 *__restrict__ Bp) {
  griddep_wait();
  griddep_launch_dependents();
  const int64_t total = static_cast<int64_t>(d_out) * r_pad;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t o = i / r_pad;
    const int j = static_cast<int>(i % r_pad);
    Bp[i] = j < r ? B[o * r + j] : __float2bfloat16_rn(0.f);
  }
}

// SwiGLU backward, elementwise (ch05 "Acceleration principles: Triton kernels
// and fused LoRA", §5.6; the derivative of silu(g) * u), 8 columns per
// thread, fp32 arithmetic, one rounding to bf16:
//   D[m][j]        = dH * u * silu'(g),  silu'(g) = sig(g) (1 + g (1 - sig(g)))
//   D[m][half + j] = dH * silu(g),       silu(g) = g sig(g)
// for j < d_ff, with D's row pitch 2 * half; columns [d_ff, half) of both
// halves are written as zero.  d_ff and half are multiples of 8.
__global__ void k_swiglu_grad(const __nv_bfloat16 *__restrict__ dH,
                              const __nv_bfloat16 *__restrict__ gate,
                              const __nv_bfloat16 *__restrict__ up, int64_t M, int d_ff,
                              int half, __nv_bfloat16 *__restrict__ D) {
  griddep_wait();
  griddep_launch_dependents();
  const int per_row = half / 8;
  const int64_t total = M * per_row;
  for (int64_t v = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; v < total;
       v += int64_t(gridDim.x) * blockDim.x) {
    const int64_t m = v / per_row;
    const int j = static_cast<int>(v % per_row) * 8;
    uint4 dg = make_uint4(0u, 0u, 0u, 0u), du = dg;
    if (j < d_ff) {
      const int64_t src = m * d_ff + j;
      const uint4 h4 = *reinterpret_cast<const uint4 *>(dH + src);
      const uint4 g4 = *reinterpret_cast<const uint4 *>(gate + src);
      const uint4 u4 = *reinterpret_cast<const uint4 *>(up + src);
      const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&h4);
      const __nv_bfloat162 *g2 = reinterpret_cast<const __nv_bfloat162 *>(&g4);
      const __nv_bfloat162 *u2 = reinterpret_cast<const __nv_bfloat162 *>(&u4);
      __nv_bfloat162 *o_g = reinterpret_cast<__nv_bfloat162 *>(&dg);
      __nv_bfloat162 *o_u = reinterpret_cast<__nv_bfloat162 *>(&du);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 h = __bfloat1622float2(h2[i]);
        const float2 g = __bfloat1622float2(g2[i]);
        const float2 u = __bfloat1622float2(u2[i]);
        const float s0 = 1.f / (1.f + expf(-g.x)), s1 = 1.f / (1.f + expf(-g.y));
        o_g[i] = __floats2bfloat162_rn(h.x * u.x * s0 * (1.f + g.x * (1.f - s0)),
                                       h.y * u.y * s1 * (1.f + g.y * (1.f - s1)));
        o_u[i] = __floats2bfloat162_rn(h.x * g.x * s0, h.y * g.y * s1);
      }
    }
    __nv_bfloat16 *row = D + m * 2 * int64_t(half);
    *reinterpret_cast<uint4 *>(row + j) = dg;
    *reinterpret_cast<uint4 *>(row + half + j) = du;
  }
}

// dst [2 r_pad][d_in]: rows [0, r) = Ag, rows [r_pad, r_pad + r) = Au, the
// other rows zero (the extension operand [Ag ; Au] of the gated dX GEMM).
__global__ void k_stack_rows(const __nv_bfloat16 *__restrict__ Ag,
                             const __nv_bfloat16 *__restrict__ Au, int r, int r_pad,
                             int64_t d_in, __nv_bfloat16 *__restrict__ dst) {
  griddep_wait();
  griddep_launch_dependents();
  const int64_t total = 2 * int64_t(r_pad) * d_in;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int row = static_cast<int>(i / d_in);
    const int64_t k = i % d_in;
    __nv_bfloat16 v = __float2bfloat16_rn(0.f);
    if (row < r) v = Ag[row * d_in + k];
    else if (row >= r_pad && row < r_pad + r) v = Au[(row - r_pad) * d_in + k];
    dst[i] = v;
  }
}

// ---- e4m3 quantisation with power-of-two scales (fp8 frozen-W product) ----
// The scale of a block with absolute maximum a > 0 is 2^e, e the smallest
// integer with a <= 448 * 2^e (448 = 0.875 * 2^9, the largest e4m3 value);
// a = 0 gives 2^0.  Dividing by it is exact, so the one rounding is the
// conversion to e4m3 (nearest, ties to even, saturating).
__device__ __forceinline__ int pow2_exponent(float a) {
  if (!(a > 0.f)) return 0;
  int k;
  const float m = frexpf(a, &k);  // a = m 2^k, m in [0.5, 1)
  return m <= 0.875f ? k - 9 : k - 8;
}

__device__ __forceinline__ uint8_t to_e4m3(float v) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
}
// Two at once: f.x in the low byte, f.y in the high byte (one conversion
// instruction, the same rounding as to_e4m3).
__device__ __forceinline__ uint32_t to_e4m3x2(float2 f) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3));
}

// One block per row of x [rows][cols] (cols a multiple of 8), each thread
// holding up to 64 of the row's elements in registers (one pass over the
// row): scale[row] = 2^e * (mul ? mul[0] : 1) and the codes
// q[row][.] = round(x / 2^e).  blockDim.x * 64 >= cols.
__global__ void __launch_bounds__(1024) k_quant_rows(const __nv_bfloat16 *__restrict__ x,
                                                     int64_t cols, uint8_t *__restrict__ q,
                                                     float *__restrict__ scale,
                                                     const float *__restrict__ mul) {
  __shared__ float wmax[32];
  griddep_wait();
  griddep_launch_dependents();
  const int64_t row = blockIdx.x;
  const __nv_bfloat16 *xr = x + row * cols;
  uint4 v[8];
  float a = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int64_t c = (threadIdx.x + int64_t(j) * blockDim.x) * 8;
    v[j] = c < cols ? *reinterpret_cast<const uint4 *>(xr + c) : make_uint4(0u, 0u, 0u, 0u);
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&v[j]);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(h[i]);
      a = fmaxf(a, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = a;
  __syncthreads();
  const int nw = (blockDim.x + 31) >> 5;
  a = 0.f;
  for (int i = 0; i < nw; ++i) a = fmaxf(a, wmax[i]);
  const int e = pow2_exponent(a);
  const float inv = ldexpf(1.f, -e);
  if (threadIdx.x == 0) scale[row] = ldexpf(1.f, e) * (mul != nullptr ? mul[0] : 1.f);
  uint8_t *qr = q + row * cols;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int64_t c = (threadIdx.x + int64_t(j) * blockDim.x) * 8;
    if (c >= cols) break;
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&v[j]);
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(h[i]);
      const uint32_t pair = to_e4m3(f.x * inv) | (uint32_t(to_e4m3(f.y * inv)) << 8);
      if (i < 2) lo |= pair << (16 * i);
      else hi |= pair << (16 * (i - 2));
    }
    *reinterpret_cast<uint2 *>(qr + c) = make_uint2(lo, hi);
  }
}

// The same quantisation for rows of at most 4096 columns: one warp per row
// holds the whole row in registers (16 bytes x 16 per lane), so the row's
// maximum is a warp shuffle and four rows share a block with no block-wide
// barrier.  Rows this short left the block-per-row kernel latency-bound
// (two warps per block, a barrier between the maximum and the stores).
constexpr int kQuantWarpMaxCols = 4096;
__global__ void __launch_bounds__(128) k_quant_rows_warp(const __nv_bfloat16 *__restrict__ x,
                                                         int64_t rows, int64_t cols,
                                                         uint8_t *__restrict__ q,
                                                         float *__restrict__ scale,
                                                         const float *__restrict__ mul) {
  griddep_wait();
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t row = int64_t(blockIdx.x) * 4 + (threadIdx.x >> 5);
  if (row >= rows) return;
  const __nv_bfloat16 *xr = x + row * cols;
  constexpr int V = kQuantWarpMaxCols / (32 * 8);
  uint4 v[V];
#pragma unroll
  for (int j = 0; j < V; ++j) {
    const int64_t c = (lane + int64_t(j) * 32) * 8;
    v[j] = c < cols ? *reinterpret_cast<const uint4 *>(xr + c) : make_uint4(0u, 0u, 0u, 0u);
  }
  // |x| maximum in bf16 pairs (exact), four independent chains
  __nv_bfloat162 m[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) m[i] = __float2bfloat162_rn(0.f);
#pragma unroll
  for (int j = 0; j < V; ++j) {
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&v[j]);
#pragma unroll
    for (int i = 0; i < 4; ++i) m[i] = __hmax2(m[i], __habs2(h[i]));
  }
  const __nv_bfloat162 m2 = __hmax2(__hmax2(m[0], m[1]), __hmax2(m[2], m[3]));
  float a = fmaxf(__low2float(m2), __high2float(m2));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  const int e = pow2_exponent(a);
  const float inv = ldexpf(1.f, -e);
  if (lane == 0) scale[row] = ldexpf(1.f, e) * (mul != nullptr ? mul[0] : 1.f);
  uint8_t *qr = q + row * cols;
#pragma unroll
  for (int j = 0; j < V; ++j) {
    const int64_t c = (lane + int64_t(j) * 32) * 8;
    if (c >= cols) break;
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&v[j]);
    uint32_t p[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 f = __bfloat1622float2(h[i]);
      f.x *= inv;
      f.y *= inv;
      p[i] = to_e4m3x2(f);
    }
    *reinterpret_cast<uint2 *>(qr + c) = make_uint2(p[0] | (p[1] << 16), p[2] | (p[3] << 16));
  }
}

// amax_bits |= the bit pattern of max |w| (non-negative floats order like
// their bit patterns, so an unsigned atomicMax finds the largest).
__global__ void k_absmax_all(const __nv_bfloat16 *__restrict__ w, int64_t n,
                             unsigned *__restrict__ amax_bits) {
  griddep_wait();
  griddep_launch_dependents();
  float a = 0.f;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n;
       i += int64_t(gridDim.x) * blockDim.x)
    a = fmaxf(a, fabsf(__bfloat162float(w[i])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  if ((threadIdx.x & 31) == 0) atomicMax(amax_bits, __float_as_uint(a));
}

// W [rows][cols] -> e4m3 codes q [rows][cols] and their transpose qT
// [cols][rows], with one scale for the tensor (written to scale[0]); 32 x 32
// tiles through shared memory.
__global__ void k_quant_tensor(const __nv_bfloat16 *__restrict__ w, int rows, int cols,
                               const unsigned *__restrict__ amax_bits, uint8_t *__restrict__ q,
                               uint8_t *__restrict__ qT, float *__restrict__ scale) {
  __shared__ uint8_t tile[32][33];
  griddep_wait();
  griddep_launch_dependents();
  const int e = pow2_exponent(__uint_as_float(*amax_bits));
  const float inv = ldexpf(1.f, -e);
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0 && threadIdx.y == 0)
    scale[0] = ldexpf(1.f, e);
  const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int r = r0 + i, c = c0 + threadIdx.x;
    uint8_t v = 0;
    if (r < rows && c < cols) {
      v = to_e4m3(__bfloat162float(w[int64_t(r) * cols + c]) * inv);
      q[int64_t(r) * cols + c] = v;
    }
    tile[i][threadIdx.x] = v;
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int c = c0 + i, r = r0 + threadIdx.x;
    if (c < cols && r < rows) qT[int64_t(c) * rows + r] = tile[threadIdx.x][i];
  }
}

// out [cols][r_pad] = (j < r ? in[j][col] : 0) / scale[0]   (in: [r][cols];
// no scale: 1)
__global__ void k_transpose_scale(const __nv_bfloat16 *__restrict__ in, int r, int64_t cols,
                                  int r_pad, const float *__restrict__ scale,
                                  __nv_bfloat16 *__restrict__ out) {
  griddep_wait();
  griddep_launch_dependents();
  const float inv = scale != nullptr ? 1.f / scale[0] : 1.f;
  const int64_t total = cols * r_pad;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t k = i / r_pad;
    const int j = static_cast<int>(i % r_pad);
    out[i] = __float2bfloat16_rn(j < r ? __bfloat162float(in[j * cols + k]) * inv : 0.f);
  }
}

// ---- symmetric 4-bit W with bf16 scales per group of 64 along d_in ----
// Thread (row o, group g) of W [d_out][d_in]: scale = bf16(absmax / 7) (1
// when the group is all zero), code = clamp(rint(w / scale), -8, 7) + 8,
// both divisions IEEE fp32; codes[o][g * 32 + j] holds elements 2j (low
// nibble) and 2j + 1 of the group, scales[g][o] its scale.
__global__ void __launch_bounds__(128) k_quant_q4(const __nv_bfloat16 *__restrict__ w, int d_out,
                                                  int d_in, uint8_t *__restrict__ codes,
                                                  __nv_bfloat16 *__restrict__ scales) {
  griddep_wait();
  griddep_launch_dependents();
  const int o = blockIdx.x * blockDim.x + threadIdx.x, g = blockIdx.y;
  if (o >= d_out) return;
  const uint4 *src = reinterpret_cast<const uint4 *>(w + int64_t(o) * d_in + g * 64);
  float v[64];
  float a = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint4 u = src[j];
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(h[i]);
      v[8 * j + 2 * i] = f.x;
      v[8 * j + 2 * i + 1] = f.y;
      a = fmaxf(a, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
  __nv_bfloat16 sb = __float2bfloat16_rn(__fdiv_rn(a, 7.f));
  if (__bfloat162float(sb) == 0.f) sb = __float2bfloat16_rn(1.f);
  const float sc = __bfloat162float(sb);
  uint32_t word[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint32_t x = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float q = fminf(fmaxf(rintf(__fdiv_rn(v[8 * j + i], sc)), -8.f), 7.f);
      x |= static_cast<uint32_t>(static_cast<int>(q) + 8) << (4 * i);
    }
    word[j] = x;
  }
  uint4 *dst = reinterpret_cast<uint4 *>(codes + int64_t(o) * (d_in / 2) + g * 32);
  dst[0] = make_uint4(word[0], word[1], word[2], word[3]);
  dst[1] = make_uint4(word[4], word[5], word[6], word[7]);
  scales[int64_t(g) * d_out + o] = sb;
}

// W[o][k] = bf16((code - 8) * scale): the product is exact in fp32, so the
// one rounding is to bf16, nearest even.  One thread per 8 elements.
__global__ void k_dequant_q4(const uint8_t *__restrict__ codes,
                             const __nv_bfloat16 *__restrict__ scales, int d_out, int d_in,
                             __nv_bfloat16 *__restrict__ w) {
  griddep_wait();
  griddep_launch_dependents();
  const int64_t total = int64_t(d_out) * (d_in / 8);
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int o = static_cast<int>(i / (d_in / 8));
    const int k0 = static_cast<int>(i % (d_in / 8)) * 8;
    const uint32_t x = *reinterpret_cast<const uint32_t *>(codes + int64_t(o) * (d_in / 2) + k0 / 2);
    const float sc = __bfloat162float(scales[int64_t(k0 / 64) * d_out + o]);
    uint32_t out[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const float lo = static_cast<float>(static_cast<int>((x >> (8 * p)) & 0xF) - 8) * sc;
      const float hi = static_cast<float>(static_cast<int>((x >> (8 * p + 4)) & 0xF) - 8) * sc;
      const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
      out[p] = *reinterpret_cast<const uint32_t *>(&b);
    }
    *reinterpret_cast<uint4 *>(w + int64_t(o) * d_in + k0) = make_uint4(out[0], out[1], out[2], out[3]);
  }
}

// Launch with programmatic stream serialisation allowed (every kernel of the
// library waits on griddep_wait before touching global memory).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, cudaStream_t s,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace

cudaError_t launch_swiglu_grad_bf16(const void *dH, const void *gate, const void *up, int64_t M,
                                    int d_ff, int half, void *D, int num_sms, cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  const int64_t vecs = M * (half / 8);
  const int64_t want = (vecs + 255) / 256;
  const int blocks = static_cast<int>(want < 8LL * num_sms ? want : 8LL * num_sms);
  return launch_pdl(k_swiglu_grad, dim3(blocks), dim3(256), s,
                    static_cast<const __nv_bfloat16 *>(dH),
                    static_cast<const __nv_bfloat16 *>(gate),
                    static_cast<const __nv_bfloat16 *>(up), M, d_ff, half,
                    static_cast<__nv_bfloat16 *>(D));
}

cudaError_t launch_quant_rows_e4m3(const void *x, int64_t rows, int64_t cols, void *q,
                                   float *scale, const float *mul, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (cols > 1024 * 64) return cudaErrorInvalidValue;
  if (cols <= kQuantWarpMaxCols)
    return launch_pdl(k_quant_rows_warp, dim3(static_cast<unsigned>((rows + 3) / 4)), dim3(128), s,
                      static_cast<const __nv_bfloat16 *>(x), rows, cols, static_cast<uint8_t *>(q),
                      scale, mul);
  const int threads = static_cast<int>(((cols + 63) / 64 + 31) / 32 * 32);
  return launch_pdl(k_quant_rows, dim3(static_cast<unsigned>(rows)), dim3(threads), s,
                    static_cast<const __nv_bfloat16 *>(x), cols, static_cast<uint8_t *>(q), scale,
                    mul);
}

cudaError_t launch_quant_tensor_e4m3(const void *w, int rows, int cols, unsigned *amax_bits,
                                     void *q, void *qT, float *scale, int num_sms,
                                     cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(amax_bits, 0, sizeof(unsigned), s);
  if (e != cudaSuccess) return e;
  const int64_t n = int64_t(rows) * cols;
  const int64_t want = (n + 255) / 256;
  const int blocks = static_cast<int>(want < 4LL * num_sms ? want : 4LL * num_sms);
  e = launch_pdl(k_absmax_all, dim3(blocks > 0 ? blocks : 1), dim3(256), s,
                 static_cast<const __nv_bfloat16 *>(w), n, amax_bits);
  if (e != cudaSuccess) return e;
  dim3 grid((cols + 31) / 32, (rows + 31) / 32), block(32, 8);
  return launch_pdl(k_quant_tensor, grid, block, s, static_cast<const __nv_bfloat16 *>(w), rows,
                    cols, static_cast<const unsigned *>(amax_bits), static_cast<uint8_t *>(q),
                    static_cast<uint8_t *>(qT), scale);
}

cudaError_t launch_quant_q4(const void *w, int d_out, int d_in, void *codes, void *scales,
                            cudaStream_t s) {
  if (d_in % 64 != 0) return cudaErrorInvalidValue;
  dim3 grid((d_out + 127) / 128, d_in / 64);
  return launch_pdl(k_quant_q4, grid, dim3(128), s, static_cast<const __nv_bfloat16 *>(w), d_out,
                    d_in, static_cast<uint8_t *>(codes), static_cast<__nv_bfloat16 *>(scales));
}

cudaError_t launch_dequant_q4(const void *codes, const void *scales, int d_out, int d_in, void *w,
                              int num_sms, cudaStream_t s) {
  if (d_in % 64 != 0) return cudaErrorInvalidValue;
  const int64_t want = (int64_t(d_out) * (d_in / 8) + 255) / 256;
  const int blocks = static_cast<int>(want < 8LL * num_sms ? want : 8LL * num_sms);
  return launch_pdl(k_dequant_q4, dim3(blocks > 0 ? blocks : 1), dim3(256), s,
                    static_cast<const uint8_t *>(codes),
                    static_cast<const __nv_bfloat16 *>(scales), d_out, d_in,
                    static_cast<__nv_bfloat16 *>(w));
}

cudaError_t launch_transpose_scale_bf16(const void *in, int r, int64_t cols, int r_pad,
                                        const float *scale, void *out, cudaStream_t s) {
  const int64_t total = cols * r_pad;
  const int blocks = static_cast<int>(total / 256 + 1 < 4096 ? total / 256 + 1 : 4096);
  return launch_pdl(k_transpose_scale, dim3(blocks), dim3(256), s,
                    static_cast<const __nv_bfloat16 *>(in), r, cols, r_pad, scale,
                    static_cast<__nv_bfloat16 *>(out));
}

cudaError_t launch_stack_rows_bf16(const void *Ag, const void *Au, int r, int r_pad, int64_t d_in,
                                   void *dst, cudaStream_t s) {
  const int64_t total = 2 * int64_t(r_pad) * d_in;
  const int blocks = static_cast<int>(total / 256 + 1 < 4096 ? total / 256 + 1 : 4096);
  return launch_pdl(k_stack_rows, dim3(blocks), dim3(256), s,
                    static_cast<const __nv_bfloat16 *>(Ag),
                    static_cast<const __nv_bfloat16 *>(Au), r, r_pad, d_in,
                    static_cast<__nv_bfloat16 *>(dst));
}

cudaError_t launch_f32_gemm(const F32GemmArgs &a, cudaStream_t s) {
  if (a.M <= 0 || a.N <= 0) return cudaSuccess;
  dim3 grid((a.N + TN - 1) / TN, (a.M + TM - 1) / TM);
  return launch_pdl(k_f32_gemm, grid, dim3(256), s, a);
}

cudaError_t launch_transpose_pad_bf16(const void *B, int d_out, int r, int r_pad, void *Bt,
                                      cudaStream_t s) {
  dim3 grid((d_out + 31) / 32, (r_pad + 31) / 32), block(32, 8);
  return launch_pdl(k_transpose_pad, grid, block, s, static_cast<const __nv_bfloat16 *>(B), d_out,
                    r, r_pad, static_cast<__nv_bfloat16 *>(Bt));
}

cudaError_t launch_pad_cols_bf16(const void *B, int d_out, int r, int r_pad, void *Bp,
                                 cudaStream_t s) {
  const int64_t total = static_cast<int64_t>(d_out) * r_pad;
  const int blocks = static_cast<int>(total / 256 + 1 < 4096 ? total / 256 + 1 : 4096);
  return launch_pdl(k_pad_cols, dim3(blocks), dim3(256), s, static_cast<const __nv_bfloat16 *>(B),
                    d_out, r, r_pad, static_cast<__nv_bfloat16 *>(Bp));
}

}  // namespace lora
