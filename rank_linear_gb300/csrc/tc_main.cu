// tc_main.cu -- the K-extended tcgen05 GEMM of the forward and backward.
//
// Forward  (ch05 "Acceleration principles: Triton kernels and fused LoRA",
// §5.3, fused forward: one pass accumulates W x and the low-rank term and
// writes Y once):
//     Y  = [X | sH] . [W | B]^T            K = d_in + r_pad
// Backward (ch05 §5.3, dL/dX of the fused backward):
//     dX = [dY | sG] . [W ; A]             K = d_out + r_pad
// where sH = s X A^T and sG = s dY B come from the skinny passes.  Both
// segments accumulate into one fp32 TMEM accumulator; the concatenation is
// never materialised -- the producer switches tensor maps at the segment
// boundary.
//
// Structure: persistent CTAs (one per SM), 128 x 256 output tiles, 64-wide
// K blocks in a 4-stage TMA -> shared memory ring.  Warp 0 issues TMA loads,
// one thread of warp 1 issues tcgen05.mma into a double-buffered TMEM
// accumulator (2 x 256 columns), warps 2-5 drain the accumulator
// (tcgen05.ld -> bf16 -> 16-byte global stores) while the next tile's
// main loop runs.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace lora {
namespace {

constexpr int BM = kMainBM, BN = kMainBN, BK = kMainBK, STAGES = kMainStages;
constexpr uint32_t A_BYTES = BM * BK * 2;  // 16 KB
constexpr uint32_t B_BYTES = BN * BK * 2;  // 32 KB
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t TMEM_COLS = 2 * BN;  // two accumulators
constexpr int NUM_THREADS = 192;        // producer warp, MMA warp, 4 epilogue warps
constexpr int GROUP_M = 8;              // tile rasterisation: m-tiles per group

struct __align__(8) MainTail {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

constexpr size_t SMEM_BYTES = 1024 + size_t(STAGES) * STAGE_BYTES + sizeof(MainTail);

// Tile order: groups of GROUP_M m-tiles; within a group m varies fastest, so
// the CTAs of one wave share a few A panels and a few B panels in L2.
__device__ __forceinline__ void tile_coords(int tile, int m_tiles, int n_tiles, int &mb, int &nb) {
  const int per_group = GROUP_M * n_tiles;
  const int g = tile / per_group;
  const int first_m = g * GROUP_M;
  const int gm = min(GROUP_M, m_tiles - first_m);
  const int local = tile - g * per_group;
  mb = first_m + local % gm;
  nb = local / gm;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

template <bool B_MN>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    k_main_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB2,
                int M, int N, int kb_main, int k_ext, __nv_bfloat16 *__restrict__ out, int64_t ldo,
                unsigned *dev_status) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 128-B swizzle atoms need 1 KB alignment
  MainTail *tail = reinterpret_cast<MainTail *>(smem_raw + (base - raw) + STAGES * STAGE_BYTES);
  const uint32_t sA = base;
  const uint32_t sB = base + STAGES * A_BYTES;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int m_tiles = (M + BM - 1) / BM, n_tiles = (N + BN - 1) / BN;
  const int num_tiles = m_tiles * n_tiles;
  const int kb_total = kb_main + (k_ext + BK - 1) / BK;
  volatile int *abort_flag = &tail->abort_flag;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&tail->full[s]), 1);
      mbar_init(smem_u32(&tail->empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&tail->tfull[a]), 1);
      mbar_init(smem_u32(&tail->tempty[a]), 4);
    }
    mbar_init(smem_u32(&tail->drain), 1);
    tail->abort_flag = 0;
    fence_barrier_init();
    tma_prefetch(&tmA);
    tma_prefetch(&tmB);
    tma_prefetch(&tmA2);
    tma_prefetch(&tmB2);
  }
  // Everything above touches only this CTA's shared memory; inputs, outputs
  // and TMEM are used only after the preceding kernel has finished.
  griddep_wait();
  griddep_launch_dependents();
  if (warp == 1) {
    tmem_alloc(smem_u32(&tail->tmem_base), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tail->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t issued[STAGES];
      for (int s = 0; s < STAGES; ++s) issued[s] = 0;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        int mb, nb;
        tile_coords(tile, m_tiles, n_tiles, mb, nb);
        const int m0 = mb * BM, n0 = nb * BN;
        for (int kb = 0; kb < kb_total; ++kb) {
          if (!mbar_wait(smem_u32(&tail->empty[stage]), phase ^ 1u, abort_flag, dev_status)) {
            ok = false;
            break;
          }
          const uint32_t full = smem_u32(&tail->full[stage]);
          mbar_expect_tx(full, STAGE_BYTES);
          const bool ext = kb >= kb_main;
          const CUtensorMap *ta = ext ? &tmA2 : &tmA;
          const CUtensorMap *tb = ext ? &tmB2 : &tmB;
          const int k0 = (ext ? kb - kb_main : kb) * BK;
          tma_load_2d(sA + stage * A_BYTES, ta, full, k0, m0);
          if (B_MN) {
#pragma unroll
            for (int j = 0; j < BN / 64; ++j)
              tma_load_2d(sB + stage * B_BYTES + j * 8192u, tb, full, n0 + 64 * j, k0);
          } else {
            tma_load_2d(sB + stage * B_BYTES, tb, full, k0, n0);
          }
          issued[stage] += 1;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {  // let this CTA's copies in flight land before it exits
        for (int s = 0; s < STAGES; ++s)
          if (issued[s]) mbar_wait_drain(smem_u32(&tail->full[s]), (issued[s] - 1u) & 1u);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(BM, BN, false, B_MN);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int t = 0;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x, ++t) {
        const int acc = t & 1;
        const uint32_t use = static_cast<uint32_t>(t >> 1);
        if (!mbar_wait(smem_u32(&tail->tempty[acc]), (use & 1u) ^ 1u, abort_flag, dev_status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + acc * BN;
        for (int kb = 0; kb < kb_total; ++kb) {
          if (!mbar_wait(smem_u32(&tail->full[stage]), phase, abort_flag, dev_status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int nk = kb < kb_main ? BK / 16 : min(BK / 16, (k_ext - (kb - kb_main) * BK) / 16);
          const uint32_t a0 = sA + stage * A_BYTES, b0 = sB + stage * B_BYTES;
          for (int kk = 0; kk < nk; ++kk) {
            const uint64_t ad = sdesc_sw128(a0 + kk * 32, 16, 1024);
            const uint64_t bd = B_MN ? sdesc_sw128(b0 + kk * 2048, 8192, 1024)
                                     : sdesc_sw128(b0 + kk * 32, 16, 1024);
            tc_mma_bf16(d, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          tc_commit(smem_u32(&tail->empty[stage]));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(smem_u32(&tail->tfull[acc]));
      }
      if (!ok) {  // wait for this thread's MMAs in flight before TMEM is freed
        tc_commit(smem_u32(&tail->drain));
        mbar_wait_drain(smem_u32(&tail->drain), 0);
      }
    }
  } else {
    // ------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    int t = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++t) {
      const int acc = t & 1;
      const uint32_t use = static_cast<uint32_t>(t >> 1);
      int mb, nb;
      tile_coords(tile, m_tiles, n_tiles, mb, nb);
      const bool got = mbar_wait(smem_u32(&tail->tfull[acc]), use & 1u, abort_flag, dev_status);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after();
      const int row = mb * BM + q * 32 + lane;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      __nv_bfloat16 *orow = out + static_cast<int64_t>(row) * ldo;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        float v[32];
        tmem_ld_32cols(taddr + c * 32, v);
        const int col0 = nb * BN + c * 32;
        if (row < M) {
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const int col = col0 + g * 8;
            if (col < N) {  // N is a multiple of 8: a group is all in or all out
              uint4 pk;
              pk.x = pack_bf16x2(v[g * 8 + 0], v[g * 8 + 1]);
              pk.y = pack_bf16x2(v[g * 8 + 2], v[g * 8 + 3]);
              pk.z = pack_bf16x2(v[g * 8 + 4], v[g * 8 + 5]);
              pk.w = pack_bf16x2(v[g * 8 + 6], v[g * 8 + 7]);
              *reinterpret_cast<uint4 *>(orow + col) = pk;
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&tail->tempty[acc]));
    }
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace

size_t main_gemm_smem_bytes() { return SMEM_BYTES; }

cudaError_t launch_main_gemm(const MainGemmArgs &a, int num_sms, cudaStream_t s) {
  const int m_tiles = (a.M + BM - 1) / BM, n_tiles = (a.N + BN - 1) / BN;
  const int tiles = m_tiles * n_tiles;
  if (tiles == 0) return cudaSuccess;
  const int grid = tiles < num_sms ? tiles : num_sms;
  auto kern = a.b_mn ? k_main_gemm<true> : k_main_gemm<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(SMEM_BYTES));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a.tmA, a.tmB, a.tmA2, a.tmB2, a.M, a.N, a.kb_main,
                            a.k_ext, static_cast<__nv_bfloat16 *>(a.out), a.ldo, a.dev_status);
}

}  // namespace lora
