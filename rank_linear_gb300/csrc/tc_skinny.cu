// tc_skinny.cu -- the skinny (N = r) tensor-core passes of the layer.
//
// Four products of ch05 "Acceleration principles: Triton kernels and fused
// LoRA", §5.3 have one side of width r and are bound by the HBM read of the
// wide operand:
//     forward   sH  = s X A^T           rows = tokens, K = d_in   (A K-major)
//     backward  sG  = s dY B            rows = tokens, K = d_out  (A K-major,
//                                                                   B MN-major)
//               dA^T = X^T sG           rows = d_in,   K = tokens (A MN-major)
//               dB   = dY^T sH          rows = d_out,  K = tokens (A MN-major)
// (the last two are the dL/dA and dL/dB of the fused backward's gradient
// list; s is folded into sH and sG, so dA = s G^T X and dB = s dY^T H).
//
// One CTA owns 128 output rows and one slice of K.  The S CTAs that share
// the rows form a thread-block cluster: each accumulates its slice with
// tcgen05.mma (M = 128, N = RP) into TMEM; CTA c then adds rows
// [c*128/S, (c+1)*128/S) of all S fp32 partials in rank order.  Narrow
// accumulators (RP <= 64) are pushed into the owning CTA's staging area over
// distributed shared memory before one cluster barrier; wide ones stay in
// each CTA's shared memory and are pulled after the barrier.  The order is fixed, so results are bitwise
// reproducible and no partials touch HBM.  One launch may carry two
// independent problems (e.g. s dY B and dY^T sH, which both stream dY):
// the first CTAs of the grid work on problem 0, the rest on problem 1.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace lora {
namespace {

constexpr int BM = 128, BK = 64;
constexpr int MAX_STAGES = 12;
constexpr int NUM_THREADS = 192;
constexpr uint32_t A_BYTES = BM * BK * 2;   // 16 KB
constexpr size_t kSmemBudget = 100 * 1024;  // two CTAs per SM when RP <= 128
// The feeding layout's CTAs cannot share an SM with the GEMM beside them: with
// deep_ring each takes a ring of twice the depth, twice the bytes in flight.
constexpr size_t kSmemBudgetAlone = 200 * 1024;

struct __align__(8) SkinnyTail {
  uint64_t full[MAX_STAGES];
  uint64_t empty[MAX_STAGES];
  uint64_t tfull;
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

// Per-problem scalars (the tensor maps travel as separate kernel arguments).
struct Prob {
  int rows = 0, K = 0;
  int num_kb = 0, kb_per = 0, ctas = 0;
  int a_mn = 0, b_mn = 0;
  int RP = 16;   // N of the MMA
  int RK = 16;   // accumulator columns kept (<= RP, multiple of 16)
  float scale = 1.f;
  __nv_bfloat16 *out0 = nullptr;
  int64_t ld0 = 0;
  int n0 = 0;
  __nv_bfloat16 *out1 = nullptr;
  int64_t ld1 = 0;
  int n1 = 0;
  const float *row_div = nullptr;  // out0 row m divided by row_div[m]
};

struct Params {
  Prob p[2];
  int nprob = 1;
  int S = 1;
  unsigned *zero_ptr = nullptr;  // words zeroed by CTA 0 for the next kernel
  int zero_words = 0;
  unsigned *dev_status = nullptr;
  int withhold = 0;  // test hook: CTA 0 never fills its first stage
  int after_gemm = 0;  // no wait at the start; the last cluster waits at the end
  int alone = 0;       // feeding layout with deep_ring: the deep ring
};

struct SkinnyLayout {
  int stages;
  bool push;      // partials pushed into a dedicated staging area (1 barrier)
  uint32_t b_bytes, pipe_bytes, red_bytes, region_bytes, red_off;
  size_t smem_bytes;
  uint32_t tmem_cols;
};

__host__ __device__ inline SkinnyLayout skinny_layout(int RP, int RK, bool alone) {
  SkinnyLayout L;
  L.b_bytes = static_cast<uint32_t>(RP) * BK * 2;
  const uint32_t stage_bytes = A_BYTES + L.b_bytes;
  L.red_bytes = BM * (RK + 4) * 4;  // fp32 partials, row pitch RK + 4 floats
  // Narrow accumulators get a staging area of their own, so peers can push
  // their partials into it while this CTA's pipeline is still running;
  // wide ones overlay the pipeline buffers and are pulled after a barrier.
  L.push = RK <= 64;
  const size_t cap = alone ? kSmemBudgetAlone : kSmemBudget;
  const size_t budget = L.push ? cap + 10 * 1024 - L.red_bytes : cap;
  int st = static_cast<int>(budget / stage_bytes);
  st = st < 2 ? 2 : (st > MAX_STAGES ? MAX_STAGES : st);
  L.stages = st;
  L.pipe_bytes = st * stage_bytes;
  if (L.push) {
    L.red_off = L.pipe_bytes;
    L.region_bytes = L.pipe_bytes + L.red_bytes;
  } else {
    L.red_off = 0;
    L.region_bytes = L.pipe_bytes > L.red_bytes ? L.pipe_bytes : L.red_bytes;
  }
  L.smem_bytes = 1024 + L.region_bytes + sizeof(SkinnyTail);
  uint32_t c = 32;
  while (c < static_cast<uint32_t>(RP)) c <<= 1;
  L.tmem_cols = c;
  return L;
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    k_skinny(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmB0,
             const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmB1,
             const __grid_constant__ Params P) {
  const int S = P.S;
  const int which = (P.nprob > 1 && static_cast<int>(blockIdx.x) >= P.p[0].ctas) ? 1 : 0;
  const Prob &pr = P.p[which];
  const CUtensorMap *tmA = which ? &tmA1 : &tmA0;
  const CUtensorMap *tmB = which ? &tmB1 : &tmB0;
  const int block = static_cast<int>(blockIdx.x) - (which ? P.p[0].ctas : 0);
  const int RP = pr.RP, RK = pr.RK;
  const bool a_mn = pr.a_mn != 0, b_mn = pr.b_mn != 0;
  unsigned *dev_status = P.dev_status;

  extern __shared__ uint8_t smem_raw[];
  const SkinnyLayout L = skinny_layout(RP, RK, P.alone != 0);
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *base_ptr = smem_raw + (base - raw);
  SkinnyTail *tail = reinterpret_cast<SkinnyTail *>(base_ptr + L.region_bytes);
  float *red = reinterpret_cast<float *>(base_ptr + L.red_off);
  const uint32_t sA = base;
  const uint32_t sB = base + L.stages * A_BYTES;
  const int STAGES = L.stages;
  const int pitch = RK + 4;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int rank = static_cast<int>(cluster_ctarank());
  const int m0 = (block / S) * BM;
  const int kb_begin = rank * pr.kb_per;
  const int kb_end = min(pr.num_kb, kb_begin + pr.kb_per);
  const bool has_k = kb_end > kb_begin;
  volatile int *abort_flag = &tail->abort_flag;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&tail->full[s]), 1);
      mbar_init(smem_u32(&tail->empty[s]), 1);
    }
    mbar_init(smem_u32(&tail->tfull), 1);
    mbar_init(smem_u32(&tail->drain), 1);
    tail->abort_flag = 0;
    fence_barrier_init();
    tma_prefetch(tmA);
    tma_prefetch(tmB);
  }
  // Only this CTA's shared memory is touched above; global data and TMEM
  // are used only after the preceding kernel has finished -- or, after a
  // main GEMM, once that GEMM has signalled: then every kernel before it
  // has finished, and the GEMM writes nothing read here.
  if (!P.after_gemm) griddep_wait();
  griddep_launch_dependents();
  if (blockIdx.x == 0 && P.zero_ptr != nullptr)
    for (int i = threadIdx.x; i < P.zero_words; i += NUM_THREADS) P.zero_ptr[i] = 0u;
  if (warp == 1) {
    tmem_alloc(smem_u32(&tail->tmem_base), L.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tail->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t issued[MAX_STAGES];
      for (int s = 0; s < MAX_STAGES; ++s) issued[s] = 0;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      const uint32_t tx = A_BYTES + L.b_bytes;
      for (int kb = kb_begin; kb < kb_end; ++kb) {
        if (!mbar_wait(smem_u32(&tail->empty[stage]), phase ^ 1u, abort_flag, dev_status)) {
          ok = false;
          break;
        }
        if (P.withhold && blockIdx.x == 0 && kb == kb_begin) {
          // test hook: this stage is never filled, so the MMA thread's wait
          // for it runs out and the CTA leaves through its abort path
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
          continue;
        }
        const uint32_t full = smem_u32(&tail->full[stage]);
        mbar_expect_tx(full, tx);
        const int k0 = kb * BK;
        const uint32_t a_dst = sA + stage * A_BYTES, b_dst = sB + stage * L.b_bytes;
        if (a_mn) {  // A^T stored [K][rows]: two 64-wide boxes of rows
          tma_load_2d(a_dst, tmA, full, m0, k0);
          tma_load_2d(a_dst + 8192u, tmA, full, m0 + 64, k0);
        } else {
          tma_load_2d(a_dst, tmA, full, k0, m0);
        }
        if (b_mn) {  // B stored [K][N]: RP/64 boxes of 64 columns
          for (int j = 0; j < RP / 64; ++j) tma_load_2d(b_dst + j * 8192u, tmB, full, 64 * j, k0);
        } else {
          tma_load_2d(b_dst, tmB, full, k0, 0);
        }
        issued[stage] += 1;
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      // Stay until the MMAs have consumed every stage (their final commit).
      // If that wait gives up, the CTA is aborting and copies this thread
      // issued may still be in flight: let them land before the CTA exits.
      if (ok) ok = mbar_wait(smem_u32(&tail->tfull), 0, abort_flag, dev_status);
      if (!ok) {
        for (int s = 0; s < STAGES; ++s)
          if (issued[s]) mbar_wait_drain(smem_u32(&tail->full[s]), (issued[s] - 1u) & 1u);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(BM, static_cast<uint32_t>(RP), a_mn, b_mn);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int kb = kb_begin; kb < kb_end; ++kb) {
        if (!mbar_wait(smem_u32(&tail->full[stage]), phase, abort_flag, dev_status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = sA + stage * A_BYTES, b0 = sB + stage * L.b_bytes;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          const uint64_t ad = a_mn ? sdesc_sw128(a0 + kk * 2048, 8192, 1024)
                                   : sdesc_sw128(a0 + kk * 32, 16, 1024);
          const uint64_t bd = b_mn ? sdesc_sw128(b0 + kk * 2048, 8192, 1024)
                                   : sdesc_sw128(b0 + kk * 32, 16, 1024);
          tc_mma_bf16(tmem_base, ad, bd, idesc, (kb > kb_begin || kk > 0) ? 1u : 0u);
        }
        tc_commit(smem_u32(&tail->empty[stage]));
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok) {
        tc_commit(smem_u32(&tail->tfull));
      } else {
        tc_commit(smem_u32(&tail->drain));
        mbar_wait_drain(smem_u32(&tail->drain), 0);
      }
    }
  } else {
    // ------------------------------------------------------ TMEM -> staging
    // push: row rl of this CTA's partial belongs to CTA rl / R (which reduces
    // rows [c*R, (c+1)*R)) and is stored there, in slice `rank`.
    // pull: the partial stays in this CTA's (overlaid) staging area.
    const int q = warp & 3;
    const bool got = mbar_wait(smem_u32(&tail->tfull), 0, abort_flag, dev_status);
    if (__all_sync(0xffffffffu, got)) {
      tc_fence_after();
      const int rl = q * 32 + lane;
      const int R = BM / S;
      uint32_t dst;
      if (L.push) {
        const int slot = rank * R + rl % R;
        dst = dsmem_map(smem_u32(red) + static_cast<uint32_t>(slot * pitch) * 4u,
                        static_cast<uint32_t>(rl / R));
      } else {
        fence_proxy_async_smem();  // smem last read by the tensor cores is rewritten
        dst = smem_u32(red) + static_cast<uint32_t>(rl * pitch) * 4u;
      }
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      for (int c = 0; c < RK / 16; ++c) {
        float v[16];
        tmem_ld_16cols(taddr + c * 16, v);
        if (!has_k) {
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = 0.f;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
          dsmem_st_f4(dst + (c * 16 + 4 * i) * 4u,
                      make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]));
      }
    }
  }

  // ------------------------------------------------------ cluster reduction
  __syncwarp();
  cluster_sync();  // every partial is staged
  const int R = BM / S;
  const int r_lo = rank * R;
  const int c4n = RK / 4;
  const uint32_t red_addr = smem_u32(red);
  const bool vec0 = (pr.ld0 % 4 == 0) && (pr.n0 % 4 == 0);
  for (int e = threadIdx.x; e < R * c4n; e += NUM_THREADS) {
    const int rr = e / c4n;  // row within this CTA's slice
    const int c4 = e % c4n;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int p = 0; p < S; ++p) {  // partials added in cluster-rank order
      float4 v;
      if (L.push) {
        v = *reinterpret_cast<const float4 *>(red + (p * R + rr) * pitch + c4 * 4);
      } else {
        const uint32_t off = static_cast<uint32_t>(((r_lo + rr) * pitch + c4 * 4) * 4);
        v = dsmem_ld_f4(dsmem_map(red_addr + off, static_cast<uint32_t>(p)));
      }
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    acc.x *= pr.scale;
    acc.y *= pr.scale;
    acc.z *= pr.scale;
    acc.w *= pr.scale;
    // the result replaces a row only this thread reads: row rr of slice 0
    // (push) or this CTA's own row r_lo + rr (pull)
    const int keep = L.push ? rr : r_lo + rr;
    *reinterpret_cast<float4 *>(red + keep * pitch + c4 * 4) = acc;
    const int row = m0 + r_lo + rr;
    if (pr.out0 != nullptr && row < pr.rows) {
      if (pr.row_div != nullptr) {  // a power of two: the reciprocal is exact
        const float inv = 1.f / pr.row_div[row];
        acc.x *= inv;
        acc.y *= inv;
        acc.z *= inv;
        acc.w *= inv;
      }
      const int c = c4 * 4;
      __nv_bfloat16 *o = pr.out0 + static_cast<int64_t>(row) * pr.ld0 + c;
      if (vec0 && c + 4 <= pr.n0) {
        __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
        __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
        uint2 pk;
        pk.x = *reinterpret_cast<uint32_t *>(&lo);
        pk.y = *reinterpret_cast<uint32_t *>(&hi);
        *reinterpret_cast<uint2 *>(o) = pk;
      } else {
        const float vv[4] = {acc.x, acc.y, acc.z, acc.w};
        for (int i = 0; i < 4; ++i)
          if (c + i < pr.n0) o[i] = __float2bfloat16_rn(vv[i]);
      }
    }
  }
  // pull: peers must finish reading this CTA's staging area before it is
  // reused or the CTA exits; push: only local data is read after the barrier
  if (!L.push) cluster_sync();
  __syncthreads();

  if (pr.out1 != nullptr) {  // transposed copy: consecutive threads, consecutive rows
    for (int e = threadIdx.x; e < R * pr.n1; e += NUM_THREADS) {
      const int j = e / R;
      const int rr = e % R;
      const int row = m0 + r_lo + rr;
      const int keep = L.push ? rr : r_lo + rr;
      if (row < pr.rows)
        pr.out1[static_cast<int64_t>(j) * pr.ld1 + row] = __float2bfloat16_rn(red[keep * pitch + j]);
    }
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, L.tmem_cols);
  }
  // The launch must not end before the GEMM it overlapped: the kernels after
  // it rely on each kernel having finished after its predecessor.
  if (P.after_gemm && static_cast<int>(blockIdx.x) >= static_cast<int>(gridDim.x) - S)
    griddep_wait();
}

Prob to_prob(const SkinnyArgs &a, int S) {
  Prob p;
  p.rows = a.rows;
  p.K = a.K;
  p.num_kb = (a.K + BK - 1) / BK;
  p.kb_per = (p.num_kb + S - 1) / S;
  p.ctas = ((a.rows + BM - 1) / BM) * S;
  p.a_mn = a.a_mn ? 1 : 0;
  p.b_mn = a.b_mn ? 1 : 0;
  p.RK = a.RP;
  p.RP = a.b_mn ? (a.RP + 63) / 64 * 64 : a.RP;  // MN-major B: whole 64-wide atoms
  p.scale = a.scale;
  p.out0 = static_cast<__nv_bfloat16 *>(a.out0);
  p.ld0 = a.ld0;
  p.n0 = a.n0;
  p.out1 = static_cast<__nv_bfloat16 *>(a.out1);
  p.ld1 = a.ld1;
  p.n1 = a.n1;
  p.row_div = a.row_div;
  return p;
}

}  // namespace

// Cluster size for a launch of `total_mt` 128-row tiles (summed over its
// problems) whose longest problem has `max_kb` K blocks: the S in
// {1, 2, 4, 8} minimising  waves(S) x (t_kb * ceil(max_kb / S) + t_cta),
// where waves counts two CTAs per SM, t_kb ~ 0.15 us is the time of one K
// block of a CTA with every slot streaming and t_cta ~ 4 us is a CTA's fixed
// cost (start-up latency and the cluster reduction).  Ties go to fewer CTAs;
// the grid is then kept to about 1.2 waves.
int skinny_split_launch(int total_mt, int max_kb, int num_sms) {
  const int slots = 2 * num_sms;
  const double t_kb = 0.15, t_cta = 4.0;
  auto cost_of = [&](int S) {
    const double waves = static_cast<double>((total_mt * S + slots - 1) / slots);
    return waves * (t_kb * ((max_kb + S - 1) / S) + t_cta);
  };
  int best = 1;
  double best_cost = 1e300;
  for (int S = 1; S <= 8; S *= 2) {
    if (S > 1 && max_kb < 2 * S) break;  // keep at least two K blocks per CTA
    const double cost = cost_of(S);
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = S;
    }
  }
  // Grids of more than about 1.2 waves ran slower than the model says
  // (gate/up's grouped s dY B + dB launch: 82 us at 2.3 waves, 68 us at
  // 1.16): fewer, longer CTAs then.
  while (best > 1 && 10 * total_mt * best > 12 * slots) best /= 2;
  // A one-wave grid that can run one CTA per SM instead of two, for at most
  // a quarter more modelled time, takes the smaller grid: the pass is
  // HBM-bound either way, and the smaller grid leaves room beside the GEMMs
  // around it (the 4096^2 step's s X A^T and dA passes: 204.9 -> 201.3 us
  // with 128 CTAs instead of 256).
  if (best > 1 && total_mt * best <= slots && 5 * total_mt * (best / 2) >= 4 * num_sms &&
      cost_of(best / 2) <= 1.25 * cost_of(best))
    best /= 2;
  return best;
}

int skinny_split(int rows, int K, int num_sms) {
  return skinny_split_launch((rows + BM - 1) / BM, (K + BK - 1) / BK, num_sms);
}

cudaError_t launch_skinny(const SkinnyArgs *probs, int nprob, int num_sms, cudaStream_t s) {
  Params P;
  P.nprob = 0;
  const SkinnyArgs *use[2] = {nullptr, nullptr};
  for (int i = 0; i < nprob; ++i)
    if (probs[i].rows > 0) use[P.nprob++] = &probs[i];
  if (P.nprob == 0) return cudaSuccess;
  // one cluster size for the whole launch
  int total_mt = 0, max_kb = 0;
  for (int i = 0; i < P.nprob; ++i) {
    total_mt += (use[i]->rows + BM - 1) / BM;
    const int kb = (use[i]->K + BK - 1) / BK;
    max_kb = kb > max_kb ? kb : max_kb;
  }
  bool feeds = true, deep = true;
  for (int i = 0; i < P.nprob; ++i) {
    feeds = feeds && use[i]->feeds_gemm != 0;
    deep = deep && use[i]->deep_ring != 0;
  }
  const bool feed_layout =
      feeds && total_mt <= kSkinnyFeedMaxCtas && max_kb <= kSkinnyFeedMaxKb;
  int S = feed_layout ? 1 : skinny_split_launch(total_mt, max_kb, num_sms);
  for (int i = 0; i < P.nprob; ++i)
    while (use[i]->max_split > 0 && S > use[i]->max_split) S /= 2;
  P.S = S;
  P.alone = feed_layout && deep ? 1 : 0;
  size_t smem = 0;
  unsigned grid = 0;
  for (int i = 0; i < P.nprob; ++i) {
    P.p[i] = to_prob(*use[i], S);
    const SkinnyLayout L = skinny_layout(P.p[i].RP, P.p[i].RK, P.alone != 0);
    smem = L.smem_bytes > smem ? L.smem_bytes : smem;
    grid += static_cast<unsigned>(P.p[i].ctas);
  }
  P.dev_status = use[0]->dev_status;
  P.withhold = use[0]->withhold_first_stage;
  P.after_gemm = use[0]->after_gemm;
  for (int i = 0; i < nprob; ++i) {
    if (probs[i].after_gemm != P.after_gemm) return cudaErrorInvalidValue;
    if (probs[i].zero_ptr != nullptr) {
      if (P.after_gemm) return cudaErrorInvalidValue;  // would race the GEMM's counters
      P.zero_ptr = probs[i].zero_ptr;
      P.zero_words = probs[i].zero_words;
    }
  }
  cudaError_t e = cudaFuncSetAttribute(k_skinny, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(S);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const CUtensorMap &a1 = P.nprob > 1 ? use[1]->tmA : use[0]->tmA;
  const CUtensorMap &b1 = P.nprob > 1 ? use[1]->tmB : use[0]->tmB;
  return cudaLaunchKernelEx(&cfg, k_skinny, use[0]->tmA, use[0]->tmB, a1, b1, P);
}

}  // namespace lora
