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
// Structure: persistent CTA pairs (a cluster of two CTAs, one CTA per SM).
// A pair owns a 256 x 256 block of the output and computes it with
// tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16): CTA q holds the 128
// rows of A and of the accumulator of m-block 2p+q, and 128 of the 256 rows
// (columns of the output) of the B tile, so each SM stages only half of B.
// 64-wide K blocks flow through a 6-stage TMA ring per CTA; both CTAs' loads
// complete on the even CTA's barrier.  Warp 0 of each CTA issues its TMA
// loads; one thread of warp 1 of the even CTA issues the pair MMAs into a
// double-buffered TMEM accumulator (2 x 256 columns in each CTA) and
// releases each stage to both CTAs with a multicast commit; warps 2-5 of
// each CTA drain their half of the accumulator (tcgen05.ld -> bf16 ->
// 16-byte global stores) while the next tile's main loop runs.
//
// Tail split: when the last wave would leave at least half the pairs idle
// (rem tiles on P >= 2 rem pairs), those rem tiles are computed as two
// K-ranges each, on two different pairs.  Each range's CTA writes its fp32
// partial to `partials` (column-major, so a warp's stores coalesce) and
// counts itself in; the CTA that arrives second adds the other partial to
// its own, still in TMEM, and writes the bf16 tile.  fp32 addition of two
// terms is commutative, so the result does not depend on who is second.
//
// Instantiations beside the plain one (template flags of k_main_gemm):
//   GATED  the SwiGLU gate/up pair: the odd CTA streams the up projection,
//          the epilogue writes silu(gate) * up (and gate, up for training);
//   DUAL_B the pair's dX GEMM: the B map switches from Wg to Wu mid-K;
//   FP8    an e4m3 main segment (kind::f8f6f4, 128-wide K blocks) with the
//          bf16 extension in the same accumulator and per-row scales applied
//          in the epilogue;
//   Q4     a 4-bit W: each stage carries packed codes and bf16 group scales,
//          and six groups of two extra warps (one per ring stage) expand
//          them into the bf16 B tile in shared memory;
//   WIDE   256 x 512 pair tiles (all but Q4; gated: 256 outputs of both
//          projections, half h the gate and up of 128): each K step issues two
//          N = 256 pair MMAs that share the stage's A tile, into the two
//          256-column halves of TMEM (one accumulator, no double buffer).
//          Per SM a K block then moves A 16 KB + B 32 KB for 1024 MMA cycles
//          (48 B/clock) instead of 32 KB for 512 (64 B/clock, above the
//          ~58 B/clock the TMA feed sustains).  Eight epilogue warps drain
//          half 0 first; a half is released to the MMAs as soon as it has
//          been read into registers (plain and fp8 tiles), and the next
//          tile's half-0 MMAs go ahead while half 1 is still being read,
//          so the next tile runs under this one's stores.  A split wide
//          tile's partial holds both halves (256 x 512 fp32 per pair), and
//          its fix-up brings the other range's in one half at a time
//          through the stage ring.
#include <cuda_bf16.h>

#include <atomic>

#include "internal.h"
#include "ptx.cuh"

namespace lora {
namespace {

constexpr int BM = kMainBM, BK = kMainBK;
constexpr int CLUSTER = 2;                   // the CTA pair
constexpr uint16_t PAIR_MASK = 0x3;
constexpr uint32_t A_BYTES = BM * BK * 2;    // 16 KB: this CTA's 128 rows of A
constexpr int NUM_THREADS = 192;             // producer warp, MMA warp, 4 epilogue warps
constexpr int WIDE_THREADS = 320;            // producer warp, MMA warp, 8 epilogue warps
// 4-bit W: warps expanding codes to bf16, one group of them per ring stage
// (a stage is 128 lines of 64 weights)
constexpr int DQ_GROUP_WARPS = 2;
constexpr int DQ_GROUP_THREADS = 32 * DQ_GROUP_WARPS;
static_assert(128 % DQ_GROUP_THREADS == 0, "dequantising split");
// 4-bit W stage: 128 B-tile rows of 64 codes (32 bytes) or 64 K-rows of 128
// codes, then 128 bf16 scales
constexpr uint32_t RAW_CODE_BYTES = 4096, RAW_BYTES = RAW_CODE_BYTES + 256;
// Rasterisation: groups of GROUP_M_MIN..GROUP_M_MAX m-block pairs.  A
// group's A panels (group x 256 rows x K) should stay in L2 while the B
// panels stream past, so B is read from DRAM once per group: on the gate/up
// shape 2 times instead of 8 with groups of 4 (the power-capped GEMMs ran
// 1.5-2.5 % faster).  With K = 14336 a group of 16 holds 117 MB of A, which
// L2 does not keep; groups sized for about 60 MiB of A (8 there) cut the
// dX GEMM's DRAM traffic from 1.27 to 1.11 GB and the gate/up, down_proj and
// Qwen-class steps by 1.0-1.4 %.  Groups of 4 and 6 were slower.
constexpr int GROUP_M_MIN = 8, GROUP_M_MAX = 16;
constexpr int64_t kGroupABytes = 60ll << 20;
constexpr int EPI_ARRIVALS = 4 * CLUSTER;    // epilogue warps of both CTAs
constexpr int WIDE_EPI_ARRIVALS = 8 * CLUSTER;  // wide tiles: per accumulator half
constexpr size_t kStageBudget = 192 * 1024;  // shared memory for the stage ring

// Tile geometry for a pair tile of 256 x BN (BN = 128 or 256), or 256 x 2 BN
// (WIDE: two MMAs of width BN per K step); Q4 adds the raw 4-bit codes and
// scales of a stage.
template <int BN, bool Q4 = false, bool WIDE = false>
struct Geo {
  static constexpr int HALVES = WIDE ? 2 : 1;           // MMAs per K step
  static constexpr uint32_t B_HALF = BN / 2 * BK * 2;   // this CTA's share of one MMA's B
  static constexpr uint32_t B_BYTES = HALVES * B_HALF;
  static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES + (Q4 ? RAW_BYTES : 0);
  // bytes a stage's pair-TMA loads bring to the even CTA's barrier
  static constexpr uint32_t PAIR_TX = CLUSTER * (A_BYTES + B_BYTES);
  static constexpr int STAGES_RAW = static_cast<int>(kStageBudget / STAGE_BYTES);
  // 4-bit W: six stages (its chain from load to MMA is longer), in the room
  // the shared-memory limit leaves
  static constexpr int STAGES = Q4 ? 6 : (STAGES_RAW > 8 ? 8 : STAGES_RAW);
  static constexpr uint32_t TMEM_COLS = 2 * BN;  // two accumulators, or one wide one
  static constexpr int EPI_WARPS = WIDE ? 8 : 4;
};

// One dequantising group per stage of the 4-bit ring, so that each group
// waits on every phase of its stage's rawfull barrier in order (a parity
// wait never runs a phase ahead).
constexpr int DQ_GROUPS = Geo<256, true>::STAGES;
constexpr int Q4_THREADS = NUM_THREADS + DQ_GROUPS * DQ_GROUP_THREADS;
static_assert(DQ_GROUPS <= 15 && Q4_THREADS <= 1024, "named barriers 1..15");

template <int STAGES>
struct __align__(16) MainTail {
  uint64_t full[STAGES];    // even CTA: both CTAs' loads of a stage landed
  uint64_t rawfull[STAGES]; // each CTA (4-bit W): A and the raw codes landed
  uint64_t empty[STAGES];   // each CTA: the pair MMAs finished reading a stage
  uint64_t tfull[2];        // each CTA: an accumulator is complete
  uint64_t tempty[2];       // even CTA: both CTAs drained an accumulator
  uint64_t drain;
  uint64_t peer_done;       // even CTA: the odd CTA's issue counts are in peer_issued
  uint64_t settled;         // odd CTA: the even CTA saw every copy of the pair land
  uint64_t ebar;            // each CTA: the four epilogue warps meet (tail split)
  uint64_t fix;             // each CTA: the other K range's partial landed (tail split)
  uint32_t tmem_base;
  int abort_flag;
  int split_last;
  uint32_t peer_issued[STAGES];  // even CTA: phases the odd CTA loaded, per stage
  // 4-bit W: target of the odd CTA's 16-byte "stage expanded" copies
  alignas(16) uint8_t sig[16];
};

// Epilogue staging: per epilogue warp, one 32 x 32 bf16 chunk, 64 bytes a
// row; 16-byte segment i of row r sits at slot i ^ ((r >> 1) & 3), so that
// both the row-wise writes and the segment-wise reads of eight lanes cover
// all 32 banks.
constexpr uint32_t EPI_PITCH = 64;
constexpr uint32_t EPI_WARP_BYTES = 32 * EPI_PITCH;
// All but the 4-bit kernel (which has no shared memory to spare): per
// epilogue warp, one 32 x 64 bf16 chunk, 128 bytes a row (16-byte segment i
// of row r at slot i ^ (r & 7)), so that each global store instruction
// writes four whole 128-byte row segments instead of eight half segments:
// the drain of a 256-column accumulator half, bound by the SM's stores,
// took 2.0 instead of 2.6 us.
constexpr uint32_t EPI_PITCH_W = 128;
constexpr uint32_t EPI_WARP_BYTES_W = 32 * EPI_PITCH_W;
template <bool Q4>
__host__ __device__ constexpr uint32_t epi_warp_bytes() {
  return Q4 ? EPI_WARP_BYTES : EPI_WARP_BYTES_W;
}

template <int BN, bool Q4 = false, bool WIDE = false>
constexpr size_t smem_bytes() {
  using G = Geo<BN, Q4, WIDE>;
  return 1024 + size_t(G::STAGES) * G::STAGE_BYTES + G::EPI_WARPS * epi_warp_bytes<Q4>() +
         sizeof(MainTail<G::STAGES>);
}
static_assert(smem_bytes<256, true>() <= 227 * 1024 && smem_bytes<256>() <= 227 * 1024 &&
                  smem_bytes<256, false, true>() <= 227 * 1024,
              "shared memory per CTA");
static_assert(Geo<256, false, true>::STAGES == 4, "wide ring: four 48 KB stages");

// Work item -> tile and K-block range.  Items below split_first are whole
// tiles; the rest are range `chunk` of split tile `rel` (tile split_first+rel).
__device__ __forceinline__ void item_range(int item, int split_first, int split_k, int split_rem,
                                           int kb_total, int &tile, int &kb_lo, int &kb_hi,
                                           int &chunk, int &rel) {
  if (item < split_first) {
    tile = item;
    kb_lo = 0;
    kb_hi = kb_total;
    chunk = 0;
    rel = 0;
  } else {
    const int u = item - split_first;
    rel = u % split_rem;
    chunk = u / split_rem;
    tile = split_first + rel;
    kb_lo = chunk * kb_total / split_k;
    kb_hi = (chunk + 1) * kb_total / split_k;
  }
}

// Pair-tile order: groups of group_m m-pairs; within a group the m-pair
// varies fastest, so the pairs of one wave share a few A and B panels in L2.
__device__ __forceinline__ void tile_coords(int tile, int m_pairs, int n_tiles, int group_m,
                                            int &mp, int &nb) {
  const int per_group = group_m * n_tiles;
  const int g = tile / per_group;
  const int first = g * group_m;
  const int gm = min(group_m, m_pairs - first);
  const int local = tile - g * per_group;
  mp = first + local % gm;
  nb = local / gm;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

// Eight 4-bit codes (one 32-bit word, element 2j in the low nibble of byte
// j, 2j+1 in its high nibble) -> eight bf16 weights (code - 8) * scale.
// 0x4300 | c is the bf16 value 128 + c, exact for c < 16, so subtracting 136
// leaves c - 8 exactly; the product with the bf16 scale is then rounded once
// to bf16, nearest even.
__device__ __forceinline__ uint4 dequant8(uint32_t w, __nv_bfloat162 scale2) {
  const uint32_t lo = w & 0x0F0F0F0Fu, hi = (w >> 4) & 0x0F0F0F0Fu;
  const uint32_t p01 = __byte_perm(lo, hi, 0x5140);  // bytes lo0 hi0 lo1 hi1
  const uint32_t p23 = __byte_perm(lo, hi, 0x7362);  // bytes lo2 hi2 lo3 hi3
  const uint32_t x[4] = {__byte_perm(p01, 0x43434343u, 0x4140), __byte_perm(p01, 0x43434343u, 0x4342),
                         __byte_perm(p23, 0x43434343u, 0x4140), __byte_perm(p23, 0x43434343u, 0x4342)};
  const __nv_bfloat162 off = __floats2bfloat162_rn(136.f, 136.f);
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 c = __hsub2(*reinterpret_cast<const __nv_bfloat162 *>(&x[i]), off);
    const __nv_bfloat162 v = __hmul2(c, scale2);
    o[i] = *reinterpret_cast<const uint32_t *>(&v);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Writes a warp's 32 x 32 bf16 chunk (lane = row, pk = its 32 columns) to
// out rows row0.. and columns col0.. through the warp's staging buffer, so
// that each global store instruction covers 8 rows x 64 contiguous bytes.
__device__ __forceinline__ void store_chunk(const uint32_t (&pk)[16], uint8_t *stage, int lane,
                                           __nv_bfloat16 *out, int64_t ldo, int row0, int col0,
                                           int M, int N) {
  uint4 *my = reinterpret_cast<uint4 *>(stage + lane * EPI_PITCH);
  const int lsw = (lane >> 1) & 3;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    my[i ^ lsw] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
  __syncwarp();
  const int seg = lane & 3;  // 16-byte segment (8 columns) of a row
  const int col = col0 + seg * 8;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int r = 8 * j + (lane >> 2);
    const uint4 v =
        *reinterpret_cast<const uint4 *>(stage + r * EPI_PITCH + ((seg ^ ((r >> 1) & 3)) * 16));
    const int row = row0 + r;
    if (row < M && col < N)  // N is a multiple of 8: a segment is all in or all out
      *reinterpret_cast<uint4 *>(out + static_cast<int64_t>(row) * ldo + col) = v;
  }
  __syncwarp();
}

// Lane r's 64 packed bf16 (32 words) as row r of a 32 x 64 staging chunk of
// 128-byte rows, 16-byte segment i at slot i ^ (r & 7): the layout of a TMA
// map's 128-byte swizzle.
__device__ __forceinline__ void stage_chunk128(const uint32_t (&pk)[32], uint8_t *stage,
                                              int lane) {
  uint4 *my = reinterpret_cast<uint4 *>(stage + lane * EPI_PITCH_W);
  const int lsw = lane & 7;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    my[i ^ lsw] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
}
// As store_chunk for a 32 x 64 chunk (32 packed words per lane), through
// 128-byte staging rows: eight lanes store one row's 128 bytes.
__device__ __forceinline__ void store_chunk128(const uint32_t (&pk)[32], uint8_t *stage, int lane,
                                              __nv_bfloat16 *out, int64_t ldo, int row0,
                                              int col0, int M, int N) {
  stage_chunk128(pk, stage, lane);
  __syncwarp();
  const int seg = lane & 7;  // 16-byte segment (8 columns) of a row
  const int col = col0 + seg * 8;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int r = 4 * j + (lane >> 3);
    const uint4 v =
        *reinterpret_cast<const uint4 *>(stage + r * EPI_PITCH_W + ((seg ^ (r & 7)) * 16));
    const int row = row0 + r;
    if (row < M && col < N)  // N is a multiple of 8: a segment is all in or all out
      *reinterpret_cast<uint4 *>(out + static_cast<int64_t>(row) * ldo + col) = v;
  }
  __syncwarp();
}

// silu(g) * u in fp32, silu(z) = z / (1 + e^-z), the one expression both
// gated drains use: with the hardware exponential and division (__expf,
// __fdividef: relative error of order 1e-6, far below the result's one bf16
// rounding).  With expf and an IEEE division the SiLU's instructions, not
// the stores, bounded the wide gated tile's drain.  For g < -87 the
// exponential overflows and the quotient is 0, the limit of silu.
__device__ __forceinline__ float silu_mul(float g, float u) {
  return __fdividef(g * u, 1.f + __expf(-g));
}

// Gated (SwiGLU) epilogue of one 32-column chunk (ch05 "Acceleration
// principles: Triton kernels and fused LoRA", §5.6: SiLU and the elementwise
// product fused into the matmul epilogue): from fp32 gate g and up u, writes
// bf16 silu(g) * u to out, and g and u themselves (kept for the backward) to
// aux0 and aux1 (skipped when null).
__device__ __forceinline__ void store_gated(const float (&g)[32], const float (&u)[32],
                                           uint8_t *stage, int lane, __nv_bfloat16 *out,
                                           __nv_bfloat16 *aux0, __nv_bfloat16 *aux1,
                                           int64_t ldo, int row0, int col0, int M, int N) {
  uint32_t pk[16];
  if (aux0 != nullptr) {
#pragma unroll
    for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(g[2 * i], g[2 * i + 1]);
    store_chunk(pk, stage, lane, aux0, ldo, row0, col0, M, N);
  }
  if (aux1 != nullptr) {
#pragma unroll
    for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(u[2 * i], u[2 * i + 1]);
    store_chunk(pk, stage, lane, aux1, ldo, row0, col0, M, N);
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(silu_mul(g[2 * i], u[2 * i]),
                                                   silu_mul(g[2 * i + 1], u[2 * i + 1]));
  store_chunk(pk, stage, lane, out, ldo, row0, col0, M, N);
}

// One 32 x 64 staged chunk out through a TMA store (lane 0 issues it into
// its bulk group): first the buffer's previous store must have read it; a
// box wholly outside [M, N) is not issued.
__device__ __forceinline__ void tma_chunk128(const uint32_t (&pk)[32], uint8_t *stage, int lane,
                                             const CUtensorMap *tm, int col0, int row0, int M,
                                             int N) {
  if (lane == 0) bulk_wait_group_read0();
  __syncwarp();
  stage_chunk128(pk, stage, lane);
  fence_proxy_async_smem();  // this lane's stores, visible to the TMA
  __syncwarp();
  if (lane == 0 && col0 < N && row0 < M) {
    tma_store_2d(tm, smem_u32(stage), col0, row0);
    bulk_commit_group();
  }
}

// The wide gated drain of one warp's 64 outputs: gate columns g_col.., up
// columns u_col.. of TMEM; gate, up (when their maps are given) and
// silu(gate) * up, each through the staging buffer and a TMA store, one
// output at a time (TMEM is read again for the last, which keeps the live
// registers to one chunk).
__device__ __forceinline__ void drain_gated64(uint32_t g_col, uint32_t u_col, uint8_t *stage,
                                              int lane, const CUtensorMap *tm_gate,
                                              const CUtensorMap *tm_up, const CUtensorMap *tm_out,
                                              int col0, int row0, int M, int N) {
  uint32_t pk[32];
  const CUtensorMap *dst[2] = {tm_gate, tm_up};
  const uint32_t src[2] = {g_col, u_col};
#pragma unroll  // static indices: dst and src stay in registers
  for (int o = 0; o < 2; ++o) {
    if (dst[o] == nullptr) continue;
#pragma unroll
    for (int part = 0; part < 2; ++part) {
      float v[32];
      tmem_ld_32cols(src[o] + part * 32, v);
#pragma unroll
      for (int i = 0; i < 16; ++i) pk[part * 16 + i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
    }
    tma_chunk128(pk, stage, lane, dst[o], col0, row0, M, N);
  }
#pragma unroll
  for (int part = 0; part < 2; ++part) {
    float g[32], u[32];
    tmem_ld_32cols(g_col + part * 32, g);
    tmem_ld_32cols(u_col + part * 32, u);
#pragma unroll
    for (int i = 0; i < 16; ++i)
      pk[part * 16 + i] =
          pack_bf16x2(silu_mul(g[2 * i], u[2 * i]), silu_mul(g[2 * i + 1], u[2 * i + 1]));
  }
  tma_chunk128(pk, stage, lane, tm_out, col0, row0, M, N);
}

template <bool B_MN, int BN, bool SPLIT, bool GATED, bool DUAL_B, bool FP8, bool Q4, bool WIDE>
__global__ void __launch_bounds__(Q4 ? Q4_THREADS : WIDE ? WIDE_THREADS : NUM_THREADS, 1)
    k_main_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB2,
                const __grid_constant__ CUtensorMap tmB3, const __grid_constant__ CUtensorMap tmB4,
                const __grid_constant__ CUtensorMap tmOut,
                const __grid_constant__ CUtensorMap tmAux0, const __grid_constant__ CUtensorMap tmAux1,
                int M, int N, int kb_main, int k_ext, int kb_switch, int ext_shift, int group_m,
                __nv_bfloat16 *__restrict__ out, __nv_bfloat16 *__restrict__ aux0,
                __nv_bfloat16 *__restrict__ aux1, int64_t ldo, int split_k, int split_rem,
                float *__restrict__ partials, unsigned *counters, unsigned *dev_status,
                const float *__restrict__ row_scale, const float *__restrict__ w_scale,
                int withhold) {
  static_assert(!(GATED && B_MN), "the gated pair reads K-major B");
  static_assert(!(FP8 && (B_MN || GATED || DUAL_B)), "the fp8 product reads K-major operands");
  static_assert(!(Q4 && (GATED || DUAL_B || FP8)), "4-bit W: plain layer only");
  static_assert(!(WIDE && Q4), "wide tiles: not the 4-bit GEMM");
  // output columns per pair tile; the gated pair's accumulator half h holds
  // gate (columns h*BN + [0, GH)) and up (h*BN + [GH, BN)) of GH outputs
  constexpr int GH = BN / 2;
  constexpr int TN = GATED ? GH * (WIDE ? 2 : 1) : WIDE ? 2 * BN : BN;
  using G = Geo<BN, Q4, WIDE>;
  constexpr int STAGES = G::STAGES;
  constexpr uint32_t B_BYTES = G::B_BYTES, STAGE_BYTES = G::STAGE_BYTES, PAIR_TX = G::PAIR_TX;
  constexpr uint32_t B_HALF = G::B_HALF;
  constexpr uint32_t TMEM_COLS = G::TMEM_COLS;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 128-B swizzle atoms need 1 KB alignment
  uint8_t *epi_stage = smem_raw + (base - raw) + STAGES * STAGE_BYTES;
  constexpr uint32_t EPI_WB = epi_warp_bytes<Q4>();  // staging bytes per epilogue warp
  auto *tail = reinterpret_cast<MainTail<STAGES> *>(epi_stage + G::EPI_WARPS * EPI_WB);
  const uint32_t sA = base;
  const uint32_t sB = base + STAGES * A_BYTES;
  const uint32_t sRaw = sB + STAGES * B_BYTES;  // 4-bit W: codes and scales per stage

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int q = static_cast<int>(cluster_ctarank());  // 0: even (MMA-issuing) CTA, 1: odd
  const bool leader = q == 0;
  const int pair_id = blockIdx.x / CLUSTER, num_pairs = gridDim.x / CLUSTER;
  const int m_tiles = (M + BM - 1) / BM, n_tiles = (N + TN - 1) / TN;
  const int m_pairs = (m_tiles + 1) / 2;
  const int num_tiles = m_pairs * n_tiles;
  const int kb_total = kb_main + (k_ext + BK - 1) / BK;
  // work items: whole tiles [0, split_first), then split_k ranges of each of
  // the last split_rem tiles
  if (!SPLIT) {  // the lean instantiation runs whole tiles only
    split_k = 1;
    split_rem = 0;
  }
  const int split_first = num_tiles - split_rem;
  const int num_items = split_first + split_k * split_rem;
  volatile int *abort_flag = &tail->abort_flag;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      // the even CTA's expect_tx arrival: its producer's, or (4-bit W, main
      // segment) its dequantising group's, which expects the odd CTA's
      // 16-byte signal copy
      mbar_init(smem_u32(&tail->full[s]), 1);
      mbar_init(smem_u32(&tail->rawfull[s]), 1);
      mbar_init(smem_u32(&tail->empty[s]), 1);  // the even CTA's multicast commit
    }
    for (int a = 0; a < 2; ++a) {
      // wide: tfull[0] marks the accumulator complete, tempty[h] its half h
      // drained
      mbar_init(smem_u32(&tail->tfull[a]), 1);
      mbar_init(smem_u32(&tail->tempty[a]), WIDE ? WIDE_EPI_ARRIVALS : EPI_ARRIVALS);
    }
    mbar_init(smem_u32(&tail->drain), 1);
    mbar_init(smem_u32(&tail->peer_done), 1);
    mbar_init(smem_u32(&tail->settled), 1);
    mbar_init(smem_u32(&tail->ebar), G::EPI_WARPS);
    mbar_init(smem_u32(&tail->fix), 1);
    tail->abort_flag = 0;
    fence_barrier_init();
    tma_prefetch(&tmA);
    tma_prefetch(&tmB);
    tma_prefetch(&tmA2);
    tma_prefetch(&tmB2);
    if (GATED || DUAL_B || Q4) tma_prefetch(&tmB3);
    if (GATED) tma_prefetch(&tmB4);
  }
  // Both CTAs' barriers exist before either signals the other's.
  cluster_sync();
  // Programmatic dependent launch.  The preceding kernel in the stream (the
  // skinny pass producing sH or sG) waited for its own predecessor before
  // letting this grid start, so everything this kernel reads except the
  // low-rank operand of the K extension is already final, and nothing this
  // kernel writes is read by it.  The producer waits right before its first
  // load of the extension, so the main K segment overlaps the tail of the
  // preceding kernel.  One epilogue thread per CTA waits for the same
  // condition at the start and then signals the next kernel: once every
  // CTA has signalled (or left), every kernel before this one has finished,
  // which lets the backward's dA pass (it reads what the pass before this
  // GEMM wrote) start on the SMs this grid frees before the grid has ended.
  // (Signalling from the producer instead would wait for the extension of
  // each pair's first tile, a whole tile late in a pair that started after
  // the preceding pass left its SMs.)
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(&tail->tmem_base), TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tail->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t issued[STAGES];
      uint32_t rissued[STAGES];  // 4-bit W: main-segment loads on rawfull[s]
      for (int s = 0; s < STAGES; ++s) issued[s] = rissued[s] = 0;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      bool dep_done = false;
      for (int item = pair_id; item < num_items && ok; item += num_pairs) {
        int tile, kb_lo, kb_hi, chunk, rel;
        item_range(item, split_first, split_k, split_rem, kb_total, tile, kb_lo, kb_hi, chunk, rel);
        int mp, nb;
        tile_coords(tile, m_pairs, n_tiles, group_m, mp, nb);
        const int m0 = (2 * mp + q) * BM;
        // this CTA's half of the B tile: columns q*BN/2.. of the tile (of
        // each of its two BN-wide halves, wide), or for the gated pair the
        // same TN rows of its own projection
        const int n0 = GATED ? nb * TN : nb * TN + q * (BN / 2);
        for (int kb = kb_lo; kb < kb_hi; ++kb) {
          if (!mbar_wait(smem_u32(&tail->empty[stage]), phase ^ 1u, abort_flag, dev_status)) {
            ok = false;
            break;
          }
          if (!Q4 && withhold && blockIdx.x == 1 && item == pair_id && kb == kb_lo) {
            // test hook: the odd CTA of the first pair never loads its first
            // stage, so the MMA thread's wait for it runs out and both CTAs
            // leave through their abort paths
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          const uint32_t full_local = smem_u32(&tail->full[stage]);
          const uint32_t full = dsmem_map(full_local, 0);  // the even CTA's barrier
          const bool ext = kb >= kb_main;
          if constexpr (Q4) {
            if (!ext) {
              // this CTA's 4-bit codes and scales land on its own rawfull
              // barrier (issued first: the dequantising group waits for
              // them); the group turns them into the bf16 B tile and
              // signals the even CTA's full barrier
              const uint32_t rf = smem_u32(&tail->rawfull[stage]);
              const int k0 = kb * BK;
              const uint32_t rw = sRaw + stage * RAW_BYTES;
              mbar_expect_tx(rf, RAW_BYTES);
              if (B_MN) {  // 64 K-rows x 128 codes (64 bytes); scales of 2 column groups
                tma_load_2d(rw, &tmB, rf, n0 / 2, k0);
                tma_load_2d(rw + RAW_CODE_BYTES, &tmB3, rf, k0, n0 / 64);
              } else {  // 128 rows x 64 codes (32 bytes); their scales
                tma_load_2d(rw, &tmB, rf, k0 / 2, n0);
                tma_load_2d(rw + RAW_CODE_BYTES, &tmB3, rf, n0, k0 / 64);
              }
              // A as in the bf16 layer, onto the even CTA's full barrier
              // (its bytes are expected by the even CTA's dequantising group)
              tma_load_2d_pair(sA + stage * A_BYTES, &tmA, full, k0, m0);
              issued[stage] += 1;
              rissued[stage] += 1;
              if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
              }
              continue;
            }
            // extension stage: the pair loads as in the bf16 layer
            if (leader) mbar_expect_tx(full_local, PAIR_TX);
          } else {
            if (leader) mbar_expect_tx(full_local, PAIR_TX);
          }
          if (ext && !dep_done) {  // sH / sG come from the preceding kernel
            griddep_wait();
            dep_done = true;
          }
          const CUtensorMap *ta = ext ? &tmA2 : &tmA;
          // K of A: the fp8 main segment's 128-byte rows hold 2 x BK elements
          const int k0 = ext ? (kb - kb_main) * BK : kb * (FP8 ? 2 * BK : BK);
          // B: the odd CTA of the gated pair reads the up projection (its
          // extension shifted so it meets the second half of [sH_g | sH_u]);
          // otherwise the main segment switches to tmB3 at kb_switch
          const CUtensorMap *tb = ext ? &tmB2 : &tmB;
          int kB = k0;
          if constexpr (GATED) {
            if (q) {
              tb = ext ? &tmB4 : &tmB3;
              if (ext) kB = k0 - ext_shift;
            }
          } else if constexpr (DUAL_B) {
            if (!ext && kb >= kb_switch) {
              tb = &tmB3;
              kB = (kb - kb_switch) * BK;
            }
          }
          tma_load_2d_pair(sA + stage * A_BYTES, ta, full, k0, m0);
#pragma unroll
          for (int h = 0; h < G::HALVES; ++h) {  // wide: half h is BN columns further
            const uint32_t b_dst = sB + stage * B_BYTES + h * B_HALF;
            if (B_MN) {  // BN/128 boxes of [64 K x 64 N]
#pragma unroll
              for (int j = 0; j < BN / 128; ++j)
                tma_load_2d_pair(b_dst + j * 8192u, tb, full, n0 + h * BN + 64 * j, kB);
            } else {  // BN/2 rows of [N x 64 K]
              tma_load_2d_pair(b_dst, tb, full, kB, n0 + h * (GATED ? GH : BN));
            }
          }
          issued[stage] += 1;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      bool clean = ok;
      if (ok) {
        // The pair MMAs have released every stage this CTA filled: no commit
        // is still on its way to this CTA's barriers, and no copy in flight.
        for (int s = 0; s < STAGES; ++s)
          if (issued[s] && !mbar_wait(smem_u32(&tail->empty[s]), (issued[s] - 1u) & 1u,
                                      abort_flag, dev_status)) {
            clean = false;
            break;
          }
      }
      if (!clean) {  // aborting: let the pair's copies in flight land before exiting
        if constexpr (Q4) {
          // this CTA's own codes; then, for the pair loads and the signal
          // copies that complete on the even CTA's full barriers (phases
          // that need a dequantising group's arrival as well), 100 us
          for (int s = 0; s < STAGES; ++s)
            if (rissued[s]) mbar_wait_drain(smem_u32(&tail->rawfull[s]), (rissued[s] - 1u) & 1u);
          const uint64_t t0 = globaltimer_ns();
          while (globaltimer_ns() - t0 < 100000ull) {
          }
        }
      }
      if constexpr (!Q4) {
        // Both CTAs' copies complete on the even CTA's full barriers, which
        // only the even CTA can poll.  The odd CTA hands over how many
        // phases of each stage it loaded and, when aborting, stays until the
        // even CTA has seen every copy of the pair land.  Per stage at most
        // the last phase can be outstanding (a producer re-arms a stage only
        // after the MMAs consumed its previous phase, which needs both CTAs'
        // copies), and the two counts differ by at most one: the even CTA
        // settles a phase it armed but the odd CTA never loaded by counting
        // the odd CTA's bytes itself, arms a phase only the odd CTA loaded
        // for the odd CTA's bytes, and waits for the phase to complete.
        constexpr uint32_t CTA_TX = PAIR_TX / CLUSTER;
        if (!leader) {
          const uint32_t pi = smem_u32(tail->peer_issued);
          for (int s = 0; s < STAGES; ++s) dsmem_st_u32(dsmem_map(pi + 4u * s, 0), issued[s]);
          mbar_arrive_cluster(dsmem_map(smem_u32(&tail->peer_done), 0));  // release: the counts
          if (!clean) mbar_wait_drain(smem_u32(&tail->settled), 0);
        } else {
          if (!clean) {
            const bool counts = mbar_wait_drain<true>(smem_u32(&tail->peer_done), 0);
            for (int s = 0; s < STAGES; ++s) {
              const uint32_t e = issued[s];
              const uint32_t o = counts ? reinterpret_cast<volatile uint32_t *>(tail->peer_issued)[s] : e;
              const uint32_t n = e > o ? e : o;
              if (n == 0) continue;
              const uint32_t fs = smem_u32(&tail->full[s]);
              if (e == o + 1)
                mbar_complete_tx(fs, CTA_TX);
              else if (o == e + 1)
                mbar_expect_tx(fs, CTA_TX);
              mbar_wait_drain(fs, (n - 1u) & 1u);
            }
          }
          mbar_arrive_cluster(dsmem_map(smem_u32(&tail->settled), 1));
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer (even CTA)
    if (leader && lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(CLUSTER * BM, BN, false, B_MN);
      constexpr uint32_t idesc8 = idesc_e4m3(CLUSTER * BM, BN);
      // per 16-wide K step: 32 B along a K-major row, or two 1 KB MN-major
      // swizzle atoms (descriptor units of 16 B)
      constexpr uint64_t A_STEP = 32 >> 4, B_STEP = B_MN ? (2048 >> 4) : (32 >> 4);
      const uint64_t a_desc0 = sdesc_sw128(sA, 16, 1024);
      const uint64_t b_desc0 = B_MN ? sdesc_sw128(sB, 8192, 1024) : sdesc_sw128(sB, 16, 1024);
      // One K block's MMAs into accumulator columns dcol, from the stage
      // whose descriptors are ad / bd (fp8: four K = 32 steps of 32 bytes
      // each, like bf16's K = 16; the bf16 extension may be shorter).
      auto issue = [&](uint32_t dcol, uint64_t ad, uint64_t bd, int kb, uint32_t accum) {
        if (kb < kb_main) {
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            if constexpr (FP8)
              tc_mma_f8_pair(dcol, ad + kk * A_STEP, bd + kk * B_STEP, idesc8, kk ? 1u : accum);
            else
              tc_mma_bf16_pair(dcol, ad + kk * A_STEP, bd + kk * B_STEP, idesc, kk ? 1u : accum);
          }
        } else {
          const int nk = min(BK / 16, (k_ext - (kb - kb_main) * BK) / 16);
          for (int kk = 0; kk < nk; ++kk)
            tc_mma_bf16_pair(dcol, ad + kk * A_STEP, bd + kk * B_STEP, idesc, kk ? 1u : accum);
        }
      };
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int t = 0;
      for (int item = pair_id; item < num_items && ok; item += num_pairs, ++t) {
        int tile, kb_lo, kb_hi, chunk, rel;
        item_range(item, split_first, split_k, split_rem, kb_total, tile, kb_lo, kb_hi, chunk, rel);
        // wide: one accumulator (both TMEM halves), its half h free once
        // tempty[h] completes; half 1 is awaited just before its first MMA
        const int acc = WIDE ? 0 : (t & 1);
        const uint32_t use = static_cast<uint32_t>(WIDE ? t : (t >> 1));
        if (!mbar_wait(smem_u32(&tail->tempty[acc]), (use & 1u) ^ 1u, abort_flag, dev_status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + acc * BN;
        bool half1_free = !WIDE;
        // Descriptors of the current stage, advanced by addition: the
        // start-address field is the low 14 bits (address / 16) and every
        // stage lies below 256 KB, so the sums never carry out of it.
        // Between two MMAs the issuing thread runs as few instructions as
        // possible: anything longer than the tensor pipe's short queue
        // shows up as idle tensor cycles.
        uint64_t ad = a_desc0 + stage * (A_BYTES >> 4);
        uint64_t bd = b_desc0 + stage * (B_BYTES >> 4);
        uint32_t accum = 0, accum1 = 0;  // per accumulator half: 0 until its first MMA
        // Wide: while the previous tile's half 1 is still being drained, the
        // half-0 MMAs of up to STAGES - 1 K blocks go ahead; their stages
        // stay held until the half-1 MMAs catch up.
        int deferred = 0;
        for (int kb = kb_lo; kb < kb_hi; ++kb) {
          // 4-bit W: the phase also publishes the dequantising warps' stores,
          // some made by the other CTA of the pair
          if (!mbar_wait<Q4>(smem_u32(&tail->full[stage]), phase, abort_flag, dev_status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue(d, ad, bd, kb, accum);
          accum = 1u;
          bool hold = false;
          if constexpr (WIDE) {  // the same A tile against the second half of B
            if (!half1_free) {
              if (deferred + 1 < STAGES && kb + 1 < kb_hi &&
                  !mbar_peek(smem_u32(&tail->tempty[1]), (use & 1u) ^ 1u)) {
                ++deferred;
                hold = true;
              } else {
                if (!mbar_wait(smem_u32(&tail->tempty[1]), (use & 1u) ^ 1u, abort_flag,
                               dev_status)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
                half1_free = true;
                for (int j = deferred; j > 0; --j) {  // oldest first: K order within half 1
                  const int sj = stage >= j ? stage - j : stage - j + STAGES;
                  issue(d + BN, a_desc0 + sj * (A_BYTES >> 4),
                        b_desc0 + sj * (B_BYTES >> 4) + (B_HALF >> 4), kb - j, accum1);
                  accum1 = 1u;
                  tc_commit_pair_mc(smem_u32(&tail->empty[sj]), PAIR_MASK);
                }
                deferred = 0;
              }
            }
            if (!hold) {
              issue(d + BN, ad, bd + (B_HALF >> 4), kb, accum1);
              accum1 = 1u;
            }
          }
          if (!hold) tc_commit_pair_mc(smem_u32(&tail->empty[stage]), PAIR_MASK);  // free in both CTAs
          ad += A_BYTES >> 4;
          bd += B_BYTES >> 4;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
            ad = a_desc0;
            bd = b_desc0;
          }
        }
        if (!ok) break;
        tc_commit_pair_mc(smem_u32(&tail->tfull[acc]), PAIR_MASK);  // both halves complete
      }
      if (!ok) {  // wait for this thread's MMAs in flight before TMEM is freed
        tc_commit_pair(smem_u32(&tail->drain));
        mbar_wait_drain(smem_u32(&tail->drain), 0);
      }
    }
  } else if (Q4 && warp >= 6) {
    // ------------------------------------------------------ 4-bit W dequantisation (both CTAs)
    // Group g of warps owns ring stage g, so that several stages are
    // expanded at once.  On each main-segment use of its stage, a group
    // turns the codes and bf16 group scales into this CTA's bf16 half of the B tile,
    // in the layout the TMA writes for bf16 W (128-byte swizzle; K-major
    // forward, two MN-major atoms backward) and meets on a named barrier;
    // then one of its threads signals the even CTA's full barrier: there an
    // arrival expecting 16 bytes, here a 16-byte bulk copy into the even
    // CTA that completes them (a copy issued after the group's proxy fences
    // and barrier, so the tensor cores, reading through the async proxy
    // once the phase completes, see the expanded tile).  The stage's
    // previous B tile is free: its rawfull phase was armed only after the
    // pair MMAs released the stage.
    const int grp = (warp - 6) / DQ_GROUP_WARPS;
    const int gt = threadIdx.x - (6 + grp * DQ_GROUP_WARPS) * 32;  // 0 .. DQ_GROUP_THREADS - 1
    const uint32_t bar_id = 1 + grp;  // named barrier of the group (0 is __syncthreads)
    const uint8_t *raw_base = smem_raw + (sRaw - raw);
    uint8_t *b_base = smem_raw + (sB - raw);
    static_assert(!Q4 || DQ_GROUPS == STAGES, "one dequantising group per stage");
    int stage = 0;
    uint32_t rpar = 0;  // parity of the next rawfull phase of this group's stage
    bool ok = true;
    for (int item = pair_id; item < num_items && ok; item += num_pairs) {
      int tile, kb_lo, kb_hi, chunk, rel;
      item_range(item, split_first, split_k, split_rem, kb_total, tile, kb_lo, kb_hi, chunk, rel);
      for (int kb = kb_lo; kb < kb_hi; ++kb) {
        if (kb < kb_main && stage == grp) {
          const bool got = mbar_wait(smem_u32(&tail->rawfull[stage]), rpar, abort_flag,
                                     dev_status);
          if (named_bar_red_or(bar_id, DQ_GROUP_THREADS, !got)) {  // the group agrees
            ok = false;
            break;
          }
          const uint8_t *rw = raw_base + stage * RAW_BYTES;
          uint8_t *bt = b_base + stage * B_BYTES;
          // 128 lines of 128 bytes (a K-major row n, or K-row k of MN-major
          // atom a, line a * 64 + k): each line's 64 codes (32 bytes) and
          // scale; chunk c of a line sits at slot c ^ (line & 7)
#pragma unroll
          for (int li = 0; li < 128 / DQ_GROUP_THREADS; ++li) {
            const int line = gt + li * DQ_GROUP_THREADS;
            const uint8_t *src =
                B_MN ? rw + (line & 63) * 64 + (line >> 6) * 32 : rw + line * 32;
            // the 16-byte half read first alternates every 4 lines forward
            // (every 2 backward), so a quarter-warp's loads spread over the
            // banks; the halves are then put back in order, so that the
            // stores below (chunk c at slot c ^ (line & 7)) stay
            // conflict-free
            const int hx = B_MN ? (line >> 1) & 1 : (line >> 2) & 1;
            const uint4 ha = *reinterpret_cast<const uint4 *>(src + hx * 16);
            const uint4 hb = *reinterpret_cast<const uint4 *>(src + (hx ^ 1) * 16);
            const uint4 h0 = hx ? hb : ha, h1 = hx ? ha : hb;
            const uint32_t sb =
                *reinterpret_cast<const uint16_t *>(rw + RAW_CODE_BYTES + line * 2);
            const uint32_t s2 = sb * 0x10001u;
            const __nv_bfloat162 scale2 = *reinterpret_cast<const __nv_bfloat162 *>(&s2);
            uint8_t *dst = bt + (line >> 3) * 1024 + (line & 7) * 128;
            const int sw = line & 7;
            const uint32_t w[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
              *reinterpret_cast<uint4 *>(dst + ((i ^ sw) << 4)) = dequant8(w[i], scale2);
          }
          fence_proxy_async_smem();  // this thread's stores, visible to the tensor cores
          named_bar_sync(bar_id, DQ_GROUP_THREADS);
          if (gt == 0) {
            const uint32_t fl = smem_u32(&tail->full[stage]);
            const uint32_t sg = smem_u32(tail->sig);
            if (leader)  // both CTAs' A tiles and the odd CTA's signal
              mbar_expect_tx(fl, CLUSTER * A_BYTES + 16);
            else
              bulk_copy_s2c(dsmem_map(sg, 0), sg, 16, dsmem_map(fl, 0));
          }
          rpar ^= 1u;
        }
        if (++stage == STAGES) stage = 0;
      }
    }
  } else {
    // ------------------------------------------------------ epilogue (both CTAs)
    const int qd = warp & 3;  // TMEM lane quadrant this warp may access
    const int et = threadIdx.x - 64;  // 0..127 across the four epilogue warps
    if (warp == 2 && lane == 0) {  // signal the next kernel (see above)
      griddep_wait();
      griddep_launch_dependents();
    }
    int *last_flag = &tail->split_last;
    bool dep_done = false;
    uint32_t eph = 0;  // phase of ebar (the same sequence in every epilogue thread)
    // Bounded barrier among the four epilogue warps; false if it gave up.
    auto epi_sync = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&tail->ebar));
      const bool okw = mbar_wait(smem_u32(&tail->ebar), eph, abort_flag, dev_status);
      eph ^= 1u;
      return __all_sync(0xffffffffu, okw);
    };
    int t = 0;
    for (int item = pair_id; item < num_items; item += num_pairs, ++t) {
      int tile, kb_lo, kb_hi, chunk, rel;
      item_range(item, split_first, split_k, split_rem, kb_total, tile, kb_lo, kb_hi, chunk, rel);
      const bool split = SPLIT && item >= split_first;
      const int acc = WIDE ? 0 : (t & 1);
      const uint32_t use = static_cast<uint32_t>(WIDE ? t : (t >> 1));
      int mp, nb;
      tile_coords(tile, m_pairs, n_tiles, group_m, mp, nb);
      const bool got = mbar_wait(smem_u32(&tail->tfull[acc]), use & 1u, abort_flag, dev_status);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after();
      const int rl = qd * 32 + lane;  // row within this CTA's 128
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(qd * 32) << 16) + acc * BN;
      uint8_t *stage = epi_stage + qd * EPI_WB;
      const int row0 = (2 * mp + q) * BM + qd * 32;
      float sc = 1.f;  // fp8 product: this thread's row scale times W's scale
      if constexpr (FP8) {
        const int row = row0 + lane;
        sc = (row < M ? __ldg(row_scale + row) : 0.f) * (w_scale != nullptr ? __ldg(w_scale) : 1.f);
      }
      // wide: this warp's columns of each accumulator half (cpart)
      const int cpart = (warp - 2) >> 2;
      if (WIDE && GATED && (!SPLIT || !split)) {
        // as below; each warp of a quadrant drains 64 of a half's GH
        // outputs: silu(gate) * up, gate, up
        static_assert(GH == 128, "two warps of 64 outputs per half");
        uint8_t *wstage = epi_stage + (warp - 2) * EPI_WB;
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          const int c = cpart * 64;
          drain_gated64(taddr + h * BN + c, taddr + h * BN + GH + c, wstage, lane,
                        aux0 != nullptr ? &tmAux0 : nullptr, aux1 != nullptr ? &tmAux1 : nullptr,
                        &tmOut, nb * TN + h * GH + c, row0, M, N);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(dsmem_map(smem_u32(&tail->tempty[h]), 0));
        }
        continue;
      }
      if (WIDE && !GATED && (!SPLIT || !split)) {
        // Eight warps: warp w drains its lane quadrant's rows, columns
        // [h*BN + p*BN/2, +BN/2) of half h (p = which of the two warps of
        // the quadrant), half 0 first.  The warp reads its part of a half
        // out of TMEM (packed to bf16 in registers) before it stores any of
        // it, and releases the half to the MMA issuer as soon as it has read
        // it: the next tile's MMAs on that half then run under the stores.
        // Each 32 x 64 chunk goes out as one TMA store of the warp's staging
        // buffer (its layout is the map's 128-byte swizzle; the copy writes
        // only rows < M and columns < N); before the buffer is refilled the
        // previous store has read it.
        uint8_t *wstage = epi_stage + (warp - 2) * EPI_WB;
        constexpr int CH = BN / 128;  // 64-column chunks of a half per warp
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          uint32_t pk[CH][32];
#pragma unroll
          for (int c = 0; c < CH; ++c) {
            const int col = h * BN + cpart * (BN / 2) + c * 64;
            float v[32], u[32];
            tmem_ld_32cols(taddr + col, v);
            tmem_ld_32cols(taddr + col + 32, u);
            if constexpr (FP8) {
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                v[i] *= sc;
                u[i] *= sc;
              }
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              pk[c][i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
              pk[c][16 + i] = pack_bf16x2(u[2 * i], u[2 * i + 1]);
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(dsmem_map(smem_u32(&tail->tempty[h]), 0));
#pragma unroll
          for (int c = 0; c < CH; ++c)
            tma_chunk128(pk[c], wstage, lane, &tmOut,
                         nb * TN + h * BN + cpart * (BN / 2) + c * 64, row0, M, N);
        }
        continue;
      }
      if (!WIDE && (!SPLIT || !split)) {
        if constexpr (GATED) {  // columns [0, TN) gate, [TN, 2 TN) up
#pragma unroll 1
          for (int c = 0; c < TN / 32; ++c) {
            float g[32], u[32];
            tmem_ld_32cols(taddr + c * 32, g);
            tmem_ld_32cols(taddr + TN + c * 32, u);
            store_gated(g, u, stage, lane, out, aux0, aux1, ldo, row0, nb * TN + c * 32, M, N);
          }
        } else if constexpr (Q4) {
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            float v[32];
            tmem_ld_32cols(taddr + c * 32, v);
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
            store_chunk(pk, stage, lane, out, ldo, row0, nb * BN + c * 32, M, N);
          }
        } else {
#pragma unroll 1
          for (int c = 0; c < BN / 64; ++c) {  // 64 columns at a time
            float v[32], u[32];
            tmem_ld_32cols(taddr + c * 64, v);
            tmem_ld_32cols(taddr + c * 64 + 32, u);
            if constexpr (FP8) {
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                v[i] *= sc;
                u[i] *= sc;
              }
            }
            uint32_t pk[32];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              pk[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
              pk[16 + i] = pack_bf16x2(u[2 * i], u[2 * i + 1]);
            }
            store_chunk128(pk, stage, lane, out, ldo, row0, nb * BN + c * 64, M, N);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(dsmem_map(smem_u32(&tail->tempty[acc]), 0));
        continue;
      }
      if constexpr (SPLIT) {

      // ---- tail-split item (the last item of this pair): write the partial
      // [col][row] fp32, count in; the second to arrive adds the other one.
      // The accumulator is released only at the end (no item follows).
      // Wide: the partial holds both accumulator halves (2 BN columns), and
      // each of the eight warps takes its columns of each half.
      if (WIDE) {  // the staging buffer's last TMA store has read it
        if (lane == 0) bulk_wait_group_read0();
        __syncwarp();
      }
      constexpr int AC = WIDE ? 2 * BN : BN;  // accumulator columns
      constexpr int HALVES = WIDE ? 2 : 1;
      constexpr int WCOLS = WIDE ? BN / 2 : BN;  // this warp's columns of a half
      float *slot_mine = partials + static_cast<size_t>((rel * 2 + chunk) * 2 + q) * BM * AC;
      float *slot_other = partials + static_cast<size_t>((rel * 2 + (chunk ^ 1)) * 2 + q) * BM * AC;
      const int cbase = WIDE ? cpart * (BN / 2) : 0;  // first column of this warp in a half
      uint8_t *sstage = epi_stage + (WIDE ? (warp - 2) : qd) * EPI_WB;
#pragma unroll 1
      for (int h = 0; h < HALVES; ++h) {
#pragma unroll 1
        for (int c = 0; c < WCOLS / 32; ++c) {
          const int col = h * BN + cbase + c * 32;
          float v[32];
          tmem_ld_32cols(taddr + col, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) slot_mine[(col + i) * BM + rl] = v[i];
        }
      }
      if (!dep_done) {  // the counters were zeroed by the preceding kernel
        griddep_wait();
        dep_done = true;
      }
      __threadfence();            // this thread's partial is visible GPU-wide
      bool sync_ok = epi_sync();  // ... and so are the other threads'
      if (sync_ok && et == 0) {
        const unsigned prev = atomicAdd(&counters[rel * 2 + q], 1u);
        *last_flag = (prev == 1u) ? 1 : 0;
      }
      sync_ok = sync_ok && epi_sync();
      const bool last = sync_ok && *reinterpret_cast<volatile int *>(last_flag) != 0;
      if (last) {
        // The other range's partial (BM x AC fp32, column-major) comes in
        // with bulk copies on one barrier, into the stage ring, one half
        // (BM x BN, 128 KB) at a time: a split item is its pair's last, so
        // the ring's loads have all been consumed by the MMAs that completed
        // this accumulator.  One round trip per half instead of a dependent
        // chain of global loads per column block.
        constexpr uint32_t HALF_BYTES = BM * BN * 4, PIECE = 16384;
        static_assert(HALF_BYTES <= STAGES * STAGE_BYTES, "a half partial must fit the stage ring");
        const uint32_t fix = smem_u32(&tail->fix);
        const float *part = reinterpret_cast<const float *>(smem_raw + (base - raw));
        bool round_ok = true;
#pragma unroll 1
        for (int h = 0; h < HALVES && round_ok; ++h) {
          if (h > 0) {
            // every thread's reads of the previous half precede the copies
            // that overwrite it (generic reads, async-proxy writes)
            fence_proxy_async_smem();
            if (!epi_sync()) {
              round_ok = false;
              break;
            }
          }
          if (et == 0) {
            if (h == 0) {
              __threadfence();             // acquire: the other range's partial is final
              fence_proxy_async_global();  // ... and ordered before the bulk reads
            }
            mbar_expect_tx(fix, HALF_BYTES);
            const uint8_t *src = reinterpret_cast<const uint8_t *>(slot_other) + h * HALF_BYTES;
            for (uint32_t o = 0; o < HALF_BYTES; o += PIECE) bulk_load(base + o, src + o, PIECE, fix);
          }
          const bool landed = mbar_wait(fix, static_cast<uint32_t>(h) & 1u, abort_flag, dev_status);
          if (!__all_sync(0xffffffffu, landed)) {
            if (et == 0) mbar_wait_drain(fix, static_cast<uint32_t>(h) & 1u);  // copies land first
            round_ok = false;
            break;
          }
          if constexpr (GATED) {  // half h: gate, then up, of GH outputs
            const int c0 = WIDE ? cpart * (GH / 64) : 0, c1 = WIDE ? c0 + GH / 64 : GH / 32;
#pragma unroll 1
            for (int c = c0; c < c1; ++c) {
              float g[32], u[32];
              tmem_ld_32cols(taddr + h * BN + c * 32, g);
              tmem_ld_32cols(taddr + h * BN + GH + c * 32, u);
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                g[i] += part[(c * 32 + i) * BM + rl];
                u[i] += part[(GH + c * 32 + i) * BM + rl];
              }
              store_gated(g, u, sstage, lane, out, aux0, aux1, ldo, row0,
                          nb * TN + h * GH + c * 32, M, N);
            }
          } else {
#pragma unroll 1
            for (int c = 0; c < WCOLS / 32; ++c) {
              const int lc = cbase + c * 32;  // column within the half
              float o[32];
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = part[(lc + i) * BM + rl];
              float v[32];
              tmem_ld_32cols(taddr + h * BN + lc, v);
              uint32_t pk[16];
#pragma unroll
              for (int i = 0; i < 16; ++i)
                pk[i] = pack_bf16x2((v[2 * i] + o[2 * i]) * sc, (v[2 * i + 1] + o[2 * i + 1]) * sc);
              store_chunk(pk, sstage, lane, out, ldo, row0, nb * TN + h * BN + lc, M, N);
            }
          }
        }
        if (!round_ok) break;
      }
      if (sync_ok) sync_ok = epi_sync();  // the flag word is free again
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_cluster(dsmem_map(smem_u32(&tail->tempty[acc]), 0));
        if (WIDE) mbar_arrive_cluster(dsmem_map(smem_u32(&tail->tempty[1]), 0));
      }
      if (!sync_ok) break;
      }  // SPLIT
    }
    // this warp's TMA stores of the outputs are complete before the CTA leaves
    if (WIDE && lane == 0) bulk_wait_group0();
  }

  // Both CTAs are done with TMEM and with each other's barriers before the
  // collective deallocation; neither leaves while the other may still
  // touch its shared memory.
  __syncthreads();
  if (Q4 && !leader && threadIdx.x == 0 && tail->abort_flag) {
    // Aborting: a signal copy this CTA sent may still be on its way into
    // the even CTA, which leaves right after the cluster barrier.  (Without
    // an abort, the pair MMAs consumed every signal before the end.)  A copy
    // lands within microseconds: wait 100 us.
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 100000ull) {
    }
  }
  tc_fence_before();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

template <bool B_MN, int BN, bool SPLIT, bool GATED = false, bool DUAL_B = false,
          bool FP8 = false, bool Q4 = false, bool WIDE = false>
constexpr auto kernel_of() {
  return &k_main_gemm<B_MN, BN, SPLIT, GATED, DUAL_B, FP8, Q4, WIDE>;
}

int g_max_clusters[64][8] = {};

// Largest number of two-CTA clusters of a kernel variant that can be
// resident at once (queried once per device; the variant's shared-memory
// attribute must already be set).
template <bool B_MN, int BN, bool Q4 = false, bool WIDE = false>
int max_clusters(int num_sms) {
  int dev = 0;
  cudaGetDevice(&dev);
  int &n = g_max_clusters[dev & 63][(B_MN ? 1 : 0) + (Q4 ? 2 : 0) + (WIDE ? 4 : 0)];
  if (n == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(num_sms / CLUSTER * CLUSTER), 1, 1);
    cfg.blockDim = dim3(Q4 ? Q4_THREADS : WIDE ? WIDE_THREADS : NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem_bytes<BN, Q4, WIDE>();
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CLUSTER;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int c = 0;
    if (cudaOccupancyMaxActiveClusters(
            &c, kernel_of<B_MN, BN, false, false, false, false, Q4, WIDE>(), &cfg) != cudaSuccess ||
        c < 1) {
      cudaGetLastError();  // clear; fall back to one cluster per SM pair
      c = num_sms / CLUSTER;
    }
    n = c;
  }
  return n;
}

// m-block pairs per raster group for a main K segment of kb_main blocks
// (each 128 bytes of an A row, bf16 or e4m3).
int main_gemm_group_m(int kb_main) {
  const int64_t panel = int64_t(2 * BM) * kb_main * 128;  // A bytes of one m-block pair
  const int64_t g = panel > 0 ? kGroupABytes / panel : GROUP_M_MAX;
  return static_cast<int>(g < GROUP_M_MIN ? GROUP_M_MIN : g > GROUP_M_MAX ? GROUP_M_MAX : g);
}

template <bool B_MN, int BN, bool SPLIT, bool GATED, bool DUAL_B, bool FP8 = false,
          bool Q4 = false, bool WIDE = false>
cudaError_t launch_variant(const MainGemmArgs &a, int num_sms, cudaStream_t s) {
  constexpr int TN = GATED ? (BN / 2) * (WIDE ? 2 : 1) : WIDE ? 2 * BN : BN;
  const int m_tiles = (a.M + BM - 1) / BM, n_tiles = (a.N + TN - 1) / TN;
  const int tiles = ((m_tiles + 1) / 2) * n_tiles;  // pair tiles
  if (tiles == 0) return cudaSuccess;
  auto kern = kernel_of<B_MN, BN, SPLIT, GATED, DUAL_B, FP8, Q4, WIDE>();
  constexpr size_t smem = smem_bytes<BN, Q4, WIDE>();
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int maxc = max_clusters<B_MN, BN, Q4, WIDE>(num_sms);
  const int clusters = tiles < maxc ? tiles : maxc;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(clusters * CLUSTER), 1, 1);
  cfg.blockDim = dim3(Q4 ? Q4_THREADS : WIDE ? WIDE_THREADS : NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CLUSTER;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  // without a second B segment the switch point lies past every K block
  const int kb_switch = a.kb_switch >= 0 ? a.kb_switch : (1 << 30);
  const CUtensorMap &tmB3 = (GATED || Q4 || a.kb_switch >= 0) ? a.tmB3 : a.tmB;
  const CUtensorMap &tmB4 = GATED ? a.tmB4 : a.tmB2;
  // (the output maps are read only by the wide drains)
  const CUtensorMap &tmOut = WIDE ? a.tmOut : a.tmA;
  const CUtensorMap &tmAux0 = (WIDE && GATED && a.aux0 != nullptr) ? a.tmAux0 : a.tmA;
  const CUtensorMap &tmAux1 = (WIDE && GATED && a.aux1 != nullptr) ? a.tmAux1 : a.tmA;
  return cudaLaunchKernelEx(&cfg, kern, a.tmA, a.tmB, a.tmA2, a.tmB2, tmB3, tmB4, tmOut, tmAux0,
                            tmAux1, a.M, a.N,
                            a.kb_main, a.k_ext, kb_switch, a.ext_shift, main_gemm_group_m(a.kb_main),
                            static_cast<__nv_bfloat16 *>(a.out),
                            static_cast<__nv_bfloat16 *>(a.aux0),
                            static_cast<__nv_bfloat16 *>(a.aux1), a.ldo, a.split_k, a.split_rem,
                            a.partials, a.counters, a.dev_status, a.row_scale, a.w_scale,
                            a.withhold);
}

}  // namespace

int main_gemm_pairs(bool b_mn, int num_sms) {
  // the shared-memory attribute must be set before the occupancy query
  auto kern = b_mn ? kernel_of<true, 256, false>() : kernel_of<false, 256, false>();
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       static_cast<int>(smem_bytes<256>()));
  return b_mn ? max_clusters<true, 256>(num_sms) : max_clusters<false, 256>(num_sms);
}

std::atomic<int> g_force_width{0};

MainSplit main_gemm_split(int M, int N, int pairs, int tile_n) {
  MainSplit sp;
  if (pairs < 2) return sp;
  const int m_pairs = ((M + BM - 1) / BM + 1) / 2;
  const int tiles = m_pairs * ((N + tile_n - 1) / tile_n);
  const int rem = tiles % pairs;
  if (tiles <= pairs || rem == 0) return sp;  // one partial wave only, or none
  if (2 * rem > pairs) return sp;  // splitting would not shorten the last wave
  const int k = 2;
  sp.k = k;
  sp.rem = rem;
  sp.partial_bytes = static_cast<size_t>(rem) * k * 2 * BM * tile_n * sizeof(float);
  sp.counter_bytes = static_cast<size_t>(rem) * 2 * sizeof(unsigned);
  return sp;
}

// Pair-tile width.  256 is the only width built: 128-wide pair tiles ran at
// well under half the tensor rate of 256-wide ones on GB300.
int main_gemm_pick_bn(int, int, int) { return 256; }

// Time of one 256 x 512 tile in units of one 256 x 256 tile.  The narrow
// tile is bound by the TMA feed (~684 cycles per 64-wide K block against
// 512 of MMA); the wide one by its MMAs (1024 cycles per K block) plus the
// drain of the half the next tile waited for when this was measured.  The
// next tile now starts on a half as soon as it has been read out, so the
// figure errs towards narrow tiles; every benchmark shape picks the wide
// ones all the same.
constexpr double kWideTileCost = 1.6;
// A split tile's fix-up (its partial out, the other in, the combine and the
// drain), in microseconds, against a K block's time in the tile: 8 us
// against ~0.34 us for a 256-wide tile, 17 us against ~0.55 us for a
// 512-wide one (its partial is twice as large).
constexpr double kFixupNarrowUs = 8.0, kKbNarrowUs = 0.34;
constexpr double kFixupWideUs = 17.0, kKbWideUs = 0.55;

MainSplit main_gemm_plan(int M, int N, int pairs, bool allow_wide, int kb_total) {
  MainSplit narrow = main_gemm_split(M, N, pairs, 256);
  const int force = g_force_width.load();
  if (!allow_wide || pairs < 1 || force == 256) return narrow;
  MainSplit wide = main_gemm_split(M, N, pairs, 512);
  wide.wide = true;
  if (force == 512) return wide;
  const int kb = kb_total > 0 ? kb_total : 1;
  const int m_pairs = ((M + BM - 1) / BM + 1) / 2;
  const int tn = m_pairs * ((N + 255) / 256), tw = m_pairs * ((N + 511) / 512);
  const int rem = tn % pairs, rem_w = tw % pairs;
  // in 256 x 256 tile times
  const double cost_n =
      tn / pairs +
      (rem == 0 ? 0.0 : narrow.k > 1 ? 0.5 + kFixupNarrowUs / (kb * kKbNarrowUs) : 1.0);
  const double cost_w =
      kWideTileCost * (tw / pairs + (rem_w == 0 ? 0.0
                                                : wide.k > 1 ? 0.5 + kFixupWideUs / (kb * kKbWideUs)
                                                             : 1.0));
  return cost_w < cost_n ? wide : narrow;
}

void main_gemm_force_width(int w) { g_force_width.store(w); }

cudaError_t launch_main_gemm(const MainGemmArgs &a, int num_sms, cudaStream_t s) {
  // Every pair tile ends in the K extension, where the producer waits for the
  // preceding kernel.
  if (a.k_ext <= 0) return cudaErrorInvalidValue;
  const bool split = a.split_k > 1 && a.split_rem > 0;
  if (a.wide) {  // 256 x 512 pair tiles: not the 4-bit layer
    if (a.q4) return cudaErrorInvalidValue;
    if (a.gated) {
      if (a.b_mn || a.kb_switch >= 0 || a.fp8) return cudaErrorInvalidValue;
      return split ? launch_variant<false, 256, true, true, false, false, false, true>(a, num_sms, s)
                   : launch_variant<false, 256, false, true, false, false, false, true>(a, num_sms, s);
    }
    if (a.kb_switch >= 0) {
      if (!a.b_mn || a.fp8) return cudaErrorInvalidValue;
      return split ? launch_variant<true, 256, true, false, true, false, false, true>(a, num_sms, s)
                   : launch_variant<true, 256, false, false, true, false, false, true>(a, num_sms, s);
    }
    if (a.fp8) {
      if (a.b_mn || !a.row_scale) return cudaErrorInvalidValue;
      return split ? launch_variant<false, 256, true, false, false, true, false, true>(a, num_sms, s)
                   : launch_variant<false, 256, false, false, false, true, false, true>(a, num_sms, s);
    }
    if (a.b_mn)
      return split ? launch_variant<true, 256, true, false, false, false, false, true>(a, num_sms, s)
                   : launch_variant<true, 256, false, false, false, false, false, true>(a, num_sms, s);
    return split ? launch_variant<false, 256, true, false, false, false, false, true>(a, num_sms, s)
                 : launch_variant<false, 256, false, false, false, false, false, true>(a, num_sms, s);
  }
  if (a.q4) {  // 4-bit W: codes in tmB, bf16 group scales in tmB3
    if (a.fp8 || a.gated || a.kb_switch >= 0) return cudaErrorInvalidValue;
    if (a.b_mn)
      return split ? launch_variant<true, 256, true, false, false, false, true>(a, num_sms, s)
                   : launch_variant<true, 256, false, false, false, false, true>(a, num_sms, s);
    return split ? launch_variant<false, 256, true, false, false, false, true>(a, num_sms, s)
                 : launch_variant<false, 256, false, false, false, false, true>(a, num_sms, s);
  }
  if (a.fp8) {  // e4m3 main segment, K-major operands only
    if (a.b_mn || a.gated || a.kb_switch >= 0 || !a.row_scale)
      return cudaErrorInvalidValue;
    return split ? launch_variant<false, 256, true, false, false, true>(a, num_sms, s)
                 : launch_variant<false, 256, false, false, false, true>(a, num_sms, s);
  }
  if (a.gated) {
    if (a.b_mn || a.kb_switch >= 0) return cudaErrorInvalidValue;
    return split ? launch_variant<false, 256, true, true, false>(a, num_sms, s)
                 : launch_variant<false, 256, false, true, false>(a, num_sms, s);
  }
  if (a.kb_switch >= 0) {  // the gated pair's dX GEMM: [Wg ; Wu], MN-major
    if (!a.b_mn) return cudaErrorInvalidValue;
    return split ? launch_variant<true, 256, true, false, true>(a, num_sms, s)
                 : launch_variant<true, 256, false, false, true>(a, num_sms, s);
  }
  if (a.b_mn)
    return split ? launch_variant<true, 256, true, false, false>(a, num_sms, s)
                 : launch_variant<true, 256, false, false, false>(a, num_sms, s);
  return split ? launch_variant<false, 256, true, false, false>(a, num_sms, s)
               : launch_variant<false, 256, false, false, false>(a, num_sms, s);
}

}  // namespace lora
