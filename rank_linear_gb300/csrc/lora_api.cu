// lora_api.cu -- the C ABI of include/lora_linear.h: argument checks,
// buffer planning, TMA tensor maps and the launch sequence of the forward
// and backward passes.  No allocation, no synchronisation (except
// lora_device_status, which reads the device status word).
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>

#include "internal.h"
#include "lora_linear.h"
#include "lora_fp8.h"
#include "lora_q4.h"
#include "lora_swiglu.h"
#include "ptx.cuh"

namespace lora {
namespace {

__device__ unsigned g_dev_status = 0;

thread_local std::string t_err;

struct TimingHook {
  void *const *events = nullptr;
  int *kinds = nullptr;
  int n = 0;
  int used = 0;
};
thread_local TimingHook t_hook;
std::atomic<uint64_t> g_launches{0};
// backward dA passes still to launch with a withheld stage (test hook)
std::atomic<int> g_withhold{0};
// backward dX GEMMs still to launch with a withheld stage (test hook)
std::atomic<int> g_withhold_gemm{0};

// Takes one pending use of a test hook's counter; 1 if there was one.
int take_one(std::atomic<int> &counter) {
  int pending = counter.load();
  while (pending > 0 && !counter.compare_exchange_weak(pending, pending - 1)) {
  }
  return pending > 0 ? 1 : 0;
}

lora_status_t fail(lora_status_t st, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_err = buf;
  return st;
}

// ---------------------------------------------------------------- device
struct DevInfo {
  bool init = false;
  int sms = 0, major = 0, minor = 0;
  unsigned *status = nullptr;
};
std::mutex g_mtx;
constexpr int kMaxDevices = 64;
DevInfo g_dev[kMaxDevices];

lora_status_t device_info(DevInfo &out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(LORA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(LORA_ERR_UNSUPPORTED, "device index %d", dev);
  // Make the device's primary context current on this host thread (a fresh
  // thread, e.g. an autograd worker, may have none yet); the driver's
  // tensor-map encoder needs it.
  e = cudaSetDevice(dev);
  if (e != cudaSuccess) return fail(LORA_ERR_CUDA, "cudaSetDevice: %s", cudaGetErrorString(e));
  std::lock_guard<std::mutex> lock(g_mtx);
  DevInfo &d = g_dev[dev];
  if (!d.init) {
    if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev)) !=
            cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev)) !=
            cudaSuccess)
      return fail(LORA_ERR_CUDA, "device attributes: %s", cudaGetErrorString(e));
    void *p = nullptr;
    if ((e = cudaGetSymbolAddress(&p, g_dev_status)) != cudaSuccess)
      return fail(LORA_ERR_CUDA, "status word address: %s", cudaGetErrorString(e));
    d.status = static_cast<unsigned *>(p);
    d.init = true;
  }
  if (!(d.major == 10 && d.minor == 3))
    return fail(LORA_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a",
                dev, d.major, d.minor);
  out = d;
  return LORA_OK;
}

// ---------------------------------------------------------------- TMA maps
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D bf16 map over a row-major [outer][inner] tensor with the given row
// pitch; boxes of box_inner x box_outer elements, 128-byte swizzle,
// out-of-bounds elements read as zero.
lora_status_t tmap(CUtensorMap *tm, const void *ptr, uint64_t inner, uint64_t outer,
                   uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_outer, const char *what) {
  auto fn = encode_fn();
  if (!fn) return fail(LORA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {pitch_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(LORA_ERR_CUDA, "tensor map for %s (%llu x %llu, pitch %llu) failed: CUresult %d",
                what, (unsigned long long)outer, (unsigned long long)inner,
                (unsigned long long)pitch_bytes, static_cast<int>(r));
  return LORA_OK;
}

// The output maps of a main GEMM whose 256 x 512 tiles drain through TMA
// stores: bf16 [M][N] with row pitch ldo, boxes of 64 columns x 32 rows in
// the 128-byte swizzle of the drain's staging rows; for the gated pair also
// over gate (aux0) and up (aux1) when they are kept.
lora_status_t out_map(MainGemmArgs &a) {
  if (!a.wide) return LORA_OK;
  const uint64_t n = static_cast<uint64_t>(a.N), m = static_cast<uint64_t>(a.M);
  const uint64_t pitch = static_cast<uint64_t>(a.ldo) * 2;
  lora_status_t e = tmap(&a.tmOut, a.out, n, m, pitch, 64, 32, "output");
  if (e == LORA_OK && a.gated && a.aux0 != nullptr)
    e = tmap(&a.tmAux0, a.aux0, n, m, pitch, 64, 32, "gate");
  if (e == LORA_OK && a.gated && a.aux1 != nullptr)
    e = tmap(&a.tmAux1, a.aux1, n, m, pitch, 64, 32, "up");
  return e;
}

// Map without swizzle over a row-major [outer][inner] tensor of `dt`
// elements (the 4-bit W's packed codes and group scales, staged raw).
lora_status_t tmap_plain(CUtensorMap *tm, CUtensorMapDataType dt, const void *ptr, uint64_t inner,
                         uint64_t outer, uint64_t pitch_bytes, uint32_t box_inner,
                         uint32_t box_outer, const char *what) {
  auto fn = encode_fn();
  if (!fn) return fail(LORA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {pitch_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(tm, dt, 2, const_cast<void *>(ptr), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(LORA_ERR_CUDA, "tensor map for %s (%llu x %llu, pitch %llu) failed: CUresult %d",
                what, (unsigned long long)outer, (unsigned long long)inner,
                (unsigned long long)pitch_bytes, static_cast<int>(r));
  return LORA_OK;
}

// A frozen W held as 4-bit codes: packed [d_out][d_in / 2] bytes (element
// 2j in the low nibble of byte j) and bf16 group scales [d_in / 64][d_out].
struct Q4W {
  const void *codes = nullptr, *scales = nullptr;
};

// ---------------------------------------------------------------- launches
template <class F>
lora_status_t run(lora_kernel_kind_t kind, cudaStream_t s, const char *what, F &&launch) {
  int j = -1;
  if (t_hook.events != nullptr && t_hook.used < t_hook.n) {
    j = t_hook.used++;
    const cudaError_t er = cudaEventRecord(static_cast<cudaEvent_t>(t_hook.events[2 * j]), s);
    if (er != cudaSuccess)
      return fail(LORA_ERR_CUDA, "timing event before %s: %s", what, cudaGetErrorString(er));
    if (t_hook.kinds) t_hook.kinds[j] = static_cast<int>(kind);
  }
  const cudaError_t e = launch();
  if (e != cudaSuccess) return fail(LORA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  if (j >= 0) {
    const cudaError_t er = cudaEventRecord(static_cast<cudaEvent_t>(t_hook.events[2 * j + 1]), s);
    if (er != cudaSuccess)
      return fail(LORA_ERR_CUDA, "timing event after %s: %s", what, cudaGetErrorString(er));
  }
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return LORA_OK;
}

#define LORA_TRY(expr)                     \
  do {                                     \
    const lora_status_t st_ = (expr);      \
    if (st_ != LORA_OK) return st_;        \
  } while (0)

// ---------------------------------------------------------------- planning
int64_t rup(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// Byte layout of the saved buffer and of the workspace for one shape.
// The main GEMMs' tail-split region is optional: fwd_ws_min / bwd_ws_min
// leave it out, fwd_ws / bwd_ws include it (when the shape splits at all).
struct Plan {
  int r_pad = 0;     // bf16: r rounded up to 16 (K step of the MMA)
  int64_t Mp = 0;    // bf16: M rounded up to 8 (16-byte pitch of the transposed copies)
  size_t saved = 0;  // saved-buffer bytes
  size_t sHt_off = 0;
  // workspace offsets
  size_t bpad_off = 0, bt_off = 0, sg_off = 0, sgt_off = 0, resaved_off = 0;
  size_t fsplit_off = 0, fcnt_off = 0, bsplit_off = 0, bcnt_off = 0;
  MainSplit fsplit, bsplit;
  size_t fwd_ws = 0, bwd_ws = 0, fwd_ws_min = 0, bwd_ws_min = 0;
};

// pairs: CTA pairs of the main GEMM on the target device (0: no tail split).
// allow_wide: the GEMMs may take 256 x 512 tiles (the plain bf16 layer; the
// 4-bit layer's dequantising GEMM has 256-wide tiles only).
Plan make_plan(int64_t M, int64_t d_in, int64_t d_out, int r, lora_dtype_t dt, int pairs = 0,
               bool allow_wide = false) {
  Plan P;
  if (dt == LORA_BF16) {
    P.r_pad = static_cast<int>(rup(r, 16));
    P.Mp = rup(M, 8);
    const size_t sH = size_t(M) * P.r_pad * 2;
    P.sHt_off = rup(sH, 256);
    P.saved = M > 0 ? P.sHt_off + size_t(P.r_pad) * P.Mp * 2 : 0;
    // forward: [B padded (r % 8 != 0)] [split partials] [split counters]
    size_t off = (r % 8) ? rup(size_t(d_out) * P.r_pad * 2, 256) : 0;
    P.fwd_ws_min = off;
    // K blocks of a tile (main segment and extension), for the cost model
    const int kb_fwd = static_cast<int>((d_in + 63) / 64 + (P.r_pad + 63) / 64);
    const int kb_bwd = static_cast<int>((d_out + 63) / 64 + (P.r_pad + 63) / 64);
    if (pairs > 0 && M > 0) P.fsplit = main_gemm_plan(int(M), int(d_out), pairs, allow_wide, kb_fwd);
    P.fsplit_off = off;
    off += rup(P.fsplit.partial_bytes, 256);
    P.fcnt_off = off;
    off += rup(P.fsplit.counter_bytes, 256);
    P.fwd_ws = P.fsplit.k > 1 ? off : P.fwd_ws_min;
    // backward: [B^T] [sG] [sG^T] [split partials] [split counters] [recomputed saved]
    off = 0;
    P.bt_off = off;
    off += rup(size_t(P.r_pad) * d_out * 2, 256);
    P.sg_off = off;
    off += rup(size_t(M) * P.r_pad * 2, 256);
    P.sgt_off = off;
    off += rup(size_t(P.r_pad) * P.Mp * 2, 256);
    const size_t base_end = off;
    if (pairs > 0 && M > 0) P.bsplit = main_gemm_plan(int(M), int(d_in), pairs, allow_wide, kb_bwd);
    P.bsplit_off = off;
    off += rup(P.bsplit.partial_bytes, 256);
    P.bcnt_off = off;
    off += rup(P.bsplit.counter_bytes, 256);
    P.resaved_off = off;
    off += rup(P.saved, 256);
    P.bwd_ws = M > 0 ? off : 0;
    P.bwd_ws_min = M > 0 ? base_end : 0;  // with a saved buffer and no tail split
  } else {
    P.r_pad = r;
    P.Mp = M;
    P.saved = size_t(M) * r * 4;
    P.fwd_ws = 0;
    P.sg_off = 0;
    P.resaved_off = rup(size_t(M) * r * 4, 256);
    P.bwd_ws = M > 0 ? P.resaved_off + rup(P.saved, 256) : 0;
    P.bwd_ws_min = M > 0 ? P.resaved_off : 0;
  }
  return P;
}

// ---------------------------------------------------------------- checks
lora_status_t check_shape(int r, int64_t M, int64_t d_in, int64_t d_out, lora_dtype_t dt,
                          float alpha) {
  if (dt != LORA_BF16 && dt != LORA_FP32)
    return fail(LORA_ERR_INVALID_ARG, "dtype %d is not LORA_BF16 or LORA_FP32", int(dt));
  if (r < 1 || r > 256) return fail(LORA_ERR_INVALID_ARG, "r = %d is outside [1, 256]", r);
  if (M < 0) return fail(LORA_ERR_INVALID_ARG, "M = %lld is negative", (long long)M);
  if (d_in < 1 || d_out < 1)
    return fail(LORA_ERR_INVALID_ARG, "d_in = %lld, d_out = %lld must be >= 1", (long long)d_in,
                (long long)d_out);
  if (!std::isfinite(alpha)) return fail(LORA_ERR_INVALID_ARG, "alpha is not finite");
  const int64_t kMaxDim = int64_t(1) << 28;
  if (M > kMaxDim || d_in > kMaxDim || d_out > kMaxDim)
    return fail(LORA_ERR_UNSUPPORTED, "a dimension exceeds 2^28");
  const int64_t t1 = ((M + 127) / 128) * ((d_out + 255) / 256);
  const int64_t t2 = ((M + 127) / 128) * ((d_in + 255) / 256);
  if (t1 > INT32_MAX / 2 || t2 > INT32_MAX / 2)
    return fail(LORA_ERR_UNSUPPORTED, "too many output tiles");
  if (dt == LORA_BF16 && (d_in % 8 != 0 || d_out % 8 != 0))
    return fail(LORA_ERR_UNSUPPORTED,
                "bf16 needs d_in and d_out to be multiples of 8 (got %lld, %lld)",
                (long long)d_in, (long long)d_out);
  return LORA_OK;
}

lora_status_t check_ptr(const void *p, const char *name, bool may_be_null = false) {
  if (p == nullptr) {
    if (may_be_null) return LORA_OK;
    return fail(LORA_ERR_INVALID_ARG, "%s is NULL", name);
  }
  if (reinterpret_cast<uintptr_t>(p) % 16 != 0)
    return fail(LORA_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
  return LORA_OK;
}

lora_status_t check_ws(const void *ws, size_t have, size_t need) {
  if (need == 0) return LORA_OK;
  if (ws == nullptr || have < need)
    return fail(LORA_ERR_WORKSPACE, "workspace of %zu bytes needed, got %zu%s", need, have,
                ws == nullptr ? " (NULL)" : "");
  if (reinterpret_cast<uintptr_t>(ws) % 16 != 0)
    return fail(LORA_ERR_INVALID_ARG, "workspace is not 16-byte aligned");
  return LORA_OK;
}

uint8_t *at(void *base, size_t off) { return static_cast<uint8_t *>(base) + off; }

// ---------------------------------------------------------------- bf16 path
// At least two 256 x 512 pair tiles of an M x N output for every CTA pair.
bool many_wide_tiles(int64_t M, int64_t N, int pairs) {
  const int64_t tiles = ((M + 255) / 256) * ((N + 511) / 512);
  return tiles >= 2 * static_cast<int64_t>(pairs);
}

// sH = s X A^T into saved (row-major [M][r_pad]) and its transpose.
// feeds_gemm: the forward GEMM follows and may start beside this pass;
// deep_ring: that GEMM gives every pair two tiles or more.
lora_status_t down_fwd_bf16(const DevInfo &di, const Plan &P, const void *X, const void *A,
                            float s, int r, int64_t M, int64_t d_in, void *saved,
                            cudaStream_t st, unsigned *zero_ptr = nullptr, int zero_words = 0,
                            bool feeds_gemm = false, bool deep_ring = false) {
  SkinnyArgs f1;
  f1.feeds_gemm = feeds_gemm ? 1 : 0;
  f1.deep_ring = deep_ring ? 1 : 0;
  f1.zero_ptr = zero_ptr;
  f1.zero_words = zero_words;
  LORA_TRY(tmap(&f1.tmA, X, d_in, M, d_in * 2, 64, 128, "X"));
  LORA_TRY(tmap(&f1.tmB, A, d_in, r, d_in * 2, 64, P.r_pad, "A"));
  f1.a_mn = false;
  f1.rows = static_cast<int>(M);
  f1.RP = P.r_pad;
  f1.K = static_cast<int>(d_in);
  f1.scale = s;
  f1.out0 = saved;
  f1.ld0 = P.r_pad;
  f1.n0 = P.r_pad;
  f1.out1 = at(saved, P.sHt_off);
  f1.ld1 = P.Mp;
  f1.n1 = P.r_pad;
  f1.dev_status = di.status;
  return run(LORA_K_DOWN_FWD, st, "s X A^T pass", [&] { return launch_skinny(&f1, 1, di.sms, st); });
}

lora_status_t fwd_bf16(const void *X, const void *W, const void *A, const void *B, float alpha,
                       int r, int64_t M, int64_t d_in, int64_t d_out, void *Y, void *saved,
                       void *ws, size_t ws_bytes, cudaStream_t st, const Q4W *q4 = nullptr) {
  DevInfo di;
  LORA_TRY(device_info(di));
  Plan P = make_plan(M, d_in, d_out, r, LORA_BF16, main_gemm_pairs(false, di.sms), q4 == nullptr);
  const bool wide = P.fsplit.wide;
  const bool split = P.fsplit.k > 1 && ws != nullptr && ws_bytes >= P.fwd_ws;
  if (!split) P = make_plan(M, d_in, d_out, r, LORA_BF16);  // layout without the split region
  unsigned *counters = split ? reinterpret_cast<unsigned *>(at(ws, P.fcnt_off)) : nullptr;
  const float s = alpha / static_cast<float>(r);
  const void *Bsrc = B;
  int64_t b_inner = r;
  if (r % 8 != 0) {  // B's row pitch is not a multiple of 16 bytes: pad it
    void *Bp = at(ws, 0);
    LORA_TRY(run(LORA_K_PREP, st, "pad B", [&] {
      return launch_pad_cols_bf16(B, static_cast<int>(d_out), r, P.r_pad, Bp, st);
    }));
    Bsrc = Bp;
    b_inner = P.r_pad;
  }
  // with 256 x 512 tiles (about 33 us each at K = 4096) the pass can run
  // beside the GEMM's start: the pairs that start late have a tile's slack
  LORA_TRY(down_fwd_bf16(di, P, X, A, s, r, M, d_in, saved, st, counters,
                         split ? 2 * P.fsplit.rem : 0, wide,
                         wide && many_wide_tiles(M, d_out, main_gemm_pairs(false, di.sms))));
  MainGemmArgs f2;
  if (split) {
    f2.split_k = P.fsplit.k;
    f2.split_rem = P.fsplit.rem;
    f2.partials = reinterpret_cast<float *>(at(ws, P.fsplit_off));
    f2.counters = counters;
  }
  f2.bn = main_gemm_pick_bn(static_cast<int>(M), static_cast<int>(d_out), di.sms);
  LORA_TRY(tmap(&f2.tmA, X, d_in, M, d_in * 2, 64, 128, "X"));
  if (q4 != nullptr) {  // 128 rows x 64 codes, and their 128 scales, per K block
    LORA_TRY(tmap_plain(&f2.tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, q4->codes, d_in / 2, d_out,
                        d_in / 2, 32, 128, "W codes"));
    LORA_TRY(tmap_plain(&f2.tmB3, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, q4->scales, d_out, d_in / 64,
                        d_out * 2, 128, 1, "W scales"));
    f2.q4 = true;
  } else {
    LORA_TRY(tmap(&f2.tmB, W, d_in, d_out, d_in * 2, 64, f2.bn / 2, "W"));
  }
  LORA_TRY(tmap(&f2.tmA2, saved, P.r_pad, M, P.r_pad * 2, 64, 128, "sH"));
  LORA_TRY(tmap(&f2.tmB2, Bsrc, b_inner, d_out, b_inner * 2, 64, f2.bn / 2, "B"));
  f2.M = static_cast<int>(M);
  f2.N = static_cast<int>(d_out);
  f2.kb_main = static_cast<int>((d_in + 63) / 64);
  f2.k_ext = P.r_pad;
  f2.out = Y;
  f2.ldo = d_out;
  f2.b_mn = false;
  f2.wide = wide;
  f2.dev_status = di.status;
  LORA_TRY(out_map(f2));
  return run(LORA_K_MAIN_FWD, st, "forward GEMM", [&] { return launch_main_gemm(f2, di.sms, st); });
}

lora_status_t bwd_bf16(const void *dY, const void *X, const void *W, const void *A, const void *B,
                       const void *saved, float alpha, int r, int64_t M, int64_t d_in,
                       int64_t d_out, void *dX, void *dA, void *dB, void *ws, size_t ws_bytes,
                       cudaStream_t st, const Q4W *q4 = nullptr) {
  DevInfo di;
  LORA_TRY(device_info(di));
  Plan P = make_plan(M, d_in, d_out, r, LORA_BF16, main_gemm_pairs(true, di.sms), q4 == nullptr);
  const bool wide = P.bsplit.wide;
  // the dX GEMM's plan leaves its last wave short (no tail split): the pass
  // after it runs on the SMs that wave leaves idle (shape only, like `wide`)
  const bool idle_tail = wide && P.bsplit.k <= 1;
  // tail split of the dX GEMM only if the workspace holds its region (it sits
  // before the recompute room, so a saved buffer lets a shorter one suffice)
  const bool split = dX != nullptr && P.bsplit.k > 1 && ws != nullptr &&
                     ws_bytes >= (saved != nullptr ? P.resaved_off : P.bwd_ws);
  if (!split) P = make_plan(M, d_in, d_out, r, LORA_BF16);  // layout without the split region
  unsigned *counters = split ? reinterpret_cast<unsigned *>(at(ws, P.bcnt_off)) : nullptr;
  const float s = alpha / static_cast<float>(r);
  if (saved == nullptr) {  // recompute s X A^T into the workspace
    // with the forward's launch shape, so that the bits are the forward's
    const bool fwd_wide =
        make_plan(M, d_in, d_out, r, LORA_BF16, main_gemm_pairs(false, di.sms), q4 == nullptr)
            .fsplit.wide;
    void *re = at(ws, P.resaved_off);
    LORA_TRY(down_fwd_bf16(di, P, X, A, s, r, M, d_in, re, st, nullptr, 0, fwd_wide));
    saved = re;
  }
  const void *sHt = static_cast<const uint8_t *>(saved) + P.sHt_off;
  void *sG = at(ws, P.sg_off);
  void *sGt = at(ws, P.sgt_off);

  // With 256 x 512 tiles: sG = s dY B (and its transpose) alone, on few SMs
  // beside the dX GEMM's start; dB = dY^T sH after the GEMM together with
  // dA, on the SMs the GEMM's short last wave leaves idle.  With 256 x 256
  // tiles (whose tail split already fills the last wave): sG and dB in one
  // launch (both read dY), then dA beside the GEMM's last wave.  The choice
  // depends on the shape only, not on dX: the launches are the same without
  // dX (no GEMM between them), so dA and dB are the same bits either way
  // (each launch's split of K is its own).
  SkinnyArgs g[2];
  SkinnyArgs &b1 = g[0];
  LORA_TRY(tmap(&b1.tmA, dY, d_out, M, d_out * 2, 64, 128, "dY"));
  if (r % 8 == 0) {  // B [d_out, r] read directly as an MN-major operand
    LORA_TRY(tmap(&b1.tmB, B, r, d_out, int64_t(r) * 2, 64, 64, "B (MN-major)"));
    b1.b_mn = true;
  } else {  // B's row pitch is not a multiple of 16 bytes: transpose it first
    void *Bt = at(ws, P.bt_off);
    LORA_TRY(run(LORA_K_PREP, st, "transpose B", [&] {
      return launch_transpose_pad_bf16(B, static_cast<int>(d_out), r, P.r_pad, Bt, st);
    }));
    LORA_TRY(tmap(&b1.tmB, Bt, d_out, P.r_pad, d_out * 2, 64, P.r_pad, "B^T"));
    b1.b_mn = false;
  }
  b1.a_mn = false;
  b1.rows = static_cast<int>(M);
  b1.RP = P.r_pad;
  b1.K = static_cast<int>(d_out);
  b1.scale = s;
  b1.out0 = sG;
  b1.ld0 = P.r_pad;
  b1.n0 = P.r_pad;
  b1.out1 = sGt;
  b1.ld1 = P.Mp;
  b1.n1 = P.r_pad;
  b1.dev_status = di.status;
  b1.zero_ptr = counters;  // the dX GEMM's split counters
  b1.zero_words = split ? 2 * P.bsplit.rem : 0;

  SkinnyArgs &b4 = g[1];  // dB = dY^T sH   (rows = d_out, K = tokens)
  LORA_TRY(tmap(&b4.tmA, dY, d_out, M, d_out * 2, 64, 64, "dY^T"));
  LORA_TRY(tmap(&b4.tmB, sHt, M, P.r_pad, P.Mp * 2, 64, P.r_pad, "sH^T"));
  b4.a_mn = true;
  b4.rows = static_cast<int>(d_out);
  b4.RP = P.r_pad;
  b4.K = static_cast<int>(M);
  b4.scale = 1.f;
  b4.out0 = dB;
  b4.ld0 = r;
  b4.n0 = r;
  b4.dev_status = di.status;
  if (wide) {
    b1.feeds_gemm = 1;
    b1.deep_ring = many_wide_tiles(M, d_in, main_gemm_pairs(true, di.sms)) ? 1 : 0;
    LORA_TRY(run(LORA_K_DOWN_BWD, st, "s dY B pass",
                 [&] { return launch_skinny(&b1, 1, di.sms, st); }));
  } else {
    LORA_TRY(run(LORA_K_DOWN_BWD_GRAD_B, st, "s dY B and dB pass",
                 [&] { return launch_skinny(g, 2, di.sms, st); }));
  }

  // dX = [dY | sG] . [W ; A]
  if (dX != nullptr) {
    MainGemmArgs b2;
    b2.bn = main_gemm_pick_bn(static_cast<int>(M), static_cast<int>(d_in), di.sms);
    LORA_TRY(tmap(&b2.tmA, dY, d_out, M, d_out * 2, 64, 128, "dY"));
    if (q4 != nullptr) {  // 64 K-rows x 128 codes, and the scales of 2 column groups
      LORA_TRY(tmap_plain(&b2.tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, q4->codes, d_in / 2, d_out,
                          d_in / 2, 64, 64, "W codes (MN-major)"));
      LORA_TRY(tmap_plain(&b2.tmB3, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, q4->scales, d_out,
                          d_in / 64, d_out * 2, 64, 2, "W scales (MN-major)"));
      b2.q4 = true;
    } else {
      LORA_TRY(tmap(&b2.tmB, W, d_in, d_out, d_in * 2, 64, 64, "W (MN-major)"));
    }
    LORA_TRY(tmap(&b2.tmA2, sG, P.r_pad, M, P.r_pad * 2, 64, 128, "sG"));
    LORA_TRY(tmap(&b2.tmB2, A, d_in, r, d_in * 2, 64, 64, "A (MN-major)"));
    b2.M = static_cast<int>(M);
    b2.N = static_cast<int>(d_in);
    b2.kb_main = static_cast<int>((d_out + 63) / 64);
    b2.k_ext = P.r_pad;
    b2.out = dX;
    b2.ldo = d_in;
    b2.b_mn = true;
    b2.wide = wide;
    b2.dev_status = di.status;
    if (split) {
      b2.split_k = P.bsplit.k;
      b2.split_rem = P.bsplit.rem;
      b2.partials = reinterpret_cast<float *>(at(ws, P.bsplit_off));
      b2.counters = counters;
    }
    if (q4 == nullptr) b2.withhold = take_one(g_withhold_gemm);  // test hook
    LORA_TRY(out_map(b2));
    LORA_TRY(run(LORA_K_MAIN_BWD, st, "dX GEMM", [&] { return launch_main_gemm(b2, di.sms, st); }));
  }

  // dA^T = X^T sG   (rows = d_in, K = tokens), written transposed into dA
  SkinnyArgs b3;
  LORA_TRY(tmap(&b3.tmA, X, d_in, M, d_in * 2, 64, 64, "X^T"));
  LORA_TRY(tmap(&b3.tmB, sGt, M, P.r_pad, P.Mp * 2, 64, P.r_pad, "sG^T"));
  b3.a_mn = true;
  b3.rows = static_cast<int>(d_in);
  b3.RP = P.r_pad;
  b3.K = static_cast<int>(M);
  b3.scale = 1.f;
  b3.out1 = dA;
  b3.ld1 = d_in;
  b3.n1 = r;
  b3.dev_status = di.status;
  b3.after_gemm = dX != nullptr;  // overlaps the dX GEMM's last wave
  b3.withhold_first_stage = take_one(g_withhold);  // test hook of the bounded waits
  if (!wide)
    return run(LORA_K_GRAD_A, st, "dA pass", [&] { return launch_skinny(&b3, 1, di.sms, st); });
  // dA and dB in one launch (dA first: the test hook's problem).  Beside a
  // short last wave, CTAs of twice the length (K split at most in two) get
  // more of the pass done on the SMs that free early: the 4096^2 backward
  // took 87.6 instead of 95.2 us with 128 CTAs instead of 256.
  b4.after_gemm = b3.after_gemm;
  if (idle_tail) b3.max_split = b4.max_split = 2;
  SkinnyArgs ab[2] = {b3, b4};
  return run(LORA_K_GRAD_A_B, st, "dA and dB pass",
             [&] { return launch_skinny(ab, 2, di.sms, st); });
}

// ---------------------------------------------------------------- fp32 path
F32Operand op(const void *p, int64_t s0, int64_t s1) {
  F32Operand o;
  o.p = static_cast<const float *>(p);
  o.s0 = s0;
  o.s1 = s1;
  return o;
}

lora_status_t gemm32(lora_kernel_kind_t kind, const char *what, const F32GemmArgs &a,
                     cudaStream_t st) {
  return run(kind, st, what, [&] { return launch_f32_gemm(a, st); });
}

lora_status_t down_fwd_f32(const void *X, const void *A, float s, int r, int64_t M, int64_t d_in,
                           void *sH, cudaStream_t st) {
  F32GemmArgs f1;  // sH[m][i] = s sum_k X[m][k] A[i][k]
  f1.M = static_cast<int>(M);
  f1.N = r;
  f1.K1 = static_cast<int>(d_in);
  f1.a1 = op(X, d_in, 1);
  f1.b1 = op(A, 1, d_in);
  f1.alpha = s;
  f1.c = static_cast<float *>(sH);
  f1.c0 = r;
  f1.c1 = 1;
  return gemm32(LORA_K_DOWN_FWD, "s X A^T pass (fp32)", f1, st);
}

lora_status_t fwd_f32(const void *X, const void *W, const void *A, const void *B, float alpha,
                      int r, int64_t M, int64_t d_in, int64_t d_out, void *Y, void *saved,
                      cudaStream_t st) {
  DevInfo di;
  LORA_TRY(device_info(di));
  const float s = alpha / static_cast<float>(r);
  LORA_TRY(down_fwd_f32(X, A, s, r, M, d_in, saved, st));
  F32GemmArgs f2;  // Y[m][o] = sum_k X[m][k] W[o][k] + sum_i sH[m][i] B[o][i]
  f2.M = static_cast<int>(M);
  f2.N = static_cast<int>(d_out);
  f2.K1 = static_cast<int>(d_in);
  f2.a1 = op(X, d_in, 1);
  f2.b1 = op(W, 1, d_in);
  f2.K2 = r;
  f2.a2 = op(saved, r, 1);
  f2.b2 = op(B, 1, r);
  f2.c = static_cast<float *>(Y);
  f2.c0 = d_out;
  f2.c1 = 1;
  return gemm32(LORA_K_MAIN_FWD, "forward GEMM (fp32)", f2, st);
}

lora_status_t bwd_f32(const void *dY, const void *X, const void *W, const void *A, const void *B,
                      const void *saved, float alpha, int r, int64_t M, int64_t d_in,
                      int64_t d_out, void *dX, void *dA, void *dB, void *ws, cudaStream_t st) {
  DevInfo di;
  LORA_TRY(device_info(di));
  const Plan P = make_plan(M, d_in, d_out, r, LORA_FP32);
  const float s = alpha / static_cast<float>(r);
  if (saved == nullptr) {
    void *re = at(ws, P.resaved_off);
    LORA_TRY(down_fwd_f32(X, A, s, r, M, d_in, re, st));
    saved = re;
  }
  void *sG = at(ws, P.sg_off);
  F32GemmArgs b1;  // sG[m][i] = s sum_o dY[m][o] B[o][i]
  b1.M = static_cast<int>(M);
  b1.N = r;
  b1.K1 = static_cast<int>(d_out);
  b1.a1 = op(dY, d_out, 1);
  b1.b1 = op(B, r, 1);
  b1.alpha = s;
  b1.c = static_cast<float *>(sG);
  b1.c0 = r;
  b1.c1 = 1;
  LORA_TRY(gemm32(LORA_K_DOWN_BWD, "s dY B pass (fp32)", b1, st));

  F32GemmArgs b4;  // dB[o][i] = sum_m dY[m][o] sH[m][i]
  b4.M = static_cast<int>(d_out);
  b4.N = r;
  b4.K1 = static_cast<int>(M);
  b4.a1 = op(dY, 1, d_out);
  b4.b1 = op(saved, r, 1);
  b4.c = static_cast<float *>(dB);
  b4.c0 = r;
  b4.c1 = 1;
  LORA_TRY(gemm32(LORA_K_GRAD_B, "dB pass (fp32)", b4, st));

  if (dX != nullptr) {
    F32GemmArgs b2;  // dX[m][k] = sum_o dY[m][o] W[o][k] + sum_i sG[m][i] A[i][k]
    b2.M = static_cast<int>(M);
    b2.N = static_cast<int>(d_in);
    b2.K1 = static_cast<int>(d_out);
    b2.a1 = op(dY, d_out, 1);
    b2.b1 = op(W, d_in, 1);
    b2.K2 = r;
    b2.a2 = op(sG, r, 1);
    b2.b2 = op(A, d_in, 1);
    b2.c = static_cast<float *>(dX);
    b2.c0 = d_in;
    b2.c1 = 1;
    LORA_TRY(gemm32(LORA_K_MAIN_BWD, "dX GEMM (fp32)", b2, st));
  }

  F32GemmArgs b3;  // dA[i][k] = sum_m sG[m][i] X[m][k]
  b3.M = r;
  b3.N = static_cast<int>(d_in);
  b3.K1 = static_cast<int>(M);
  b3.a1 = op(sG, 1, r);
  b3.b1 = op(X, d_in, 1);
  b3.c = static_cast<float *>(dA);
  b3.c0 = d_in;
  b3.c1 = 1;
  return gemm32(LORA_K_GRAD_A, "dA pass (fp32)", b3, st);
}

// ---------------------------------------------------------------- SwiGLU pair
// Byte layout of the gated pair's saved buffer and workspace (bf16).
struct SwPlan {
  int r_pad = 0;
  int64_t Mp = 0, half = 0;  // half: d_ff rounded up to 64 (a column block of D)
  size_t gate_off = 0, up_off = 0, sh_off = 0, sht_off[2] = {0, 0}, saved = 0;
  size_t bpad_off[2] = {0, 0}, shws_off = 0, fsplit_off = 0, fcnt_off = 0, fwd_ws = 0,
         fwd_ws_min = 0;
  size_t d_off = 0, sg_off = 0, sgt_off[2] = {0, 0}, agu_off = 0, bt_off[2] = {0, 0};
  size_t bsplit_off = 0, bcnt_off = 0, bwd_ws = 0, bwd_ws_min = 0;
  MainSplit fsplit, bsplit;
};

SwPlan make_sw_plan(int64_t M, int64_t d_in, int64_t d_ff, int r, int pairs_f, int pairs_b,
                    bool allow_wide = true) {
  SwPlan P;
  P.r_pad = static_cast<int>(rup(r, 16));
  P.Mp = rup(M, 8);
  P.half = rup(d_ff, 64);
  // K blocks of a tile, for the tile-width cost model: the gated GEMM's X and
  // [sH_g | sH_u], the dX GEMM's [d_gate | d_up] and [sG_g | sG_u]
  const int kb_f = static_cast<int>((d_in + 63) / 64 + (2 * P.r_pad + 63) / 64);
  const int kb_b = static_cast<int>(2 * P.half / 64 + (2 * P.r_pad + 63) / 64);
  const size_t act = rup(size_t(M) * d_ff * 2, 256);
  const size_t tr = rup(size_t(P.r_pad) * P.Mp * 2, 256);
  // saved: [gate] [up] [sH_g | sH_u] [sH_g^T] [sH_u^T]
  size_t off = 0;
  P.gate_off = off;
  off += act;
  P.up_off = off;
  off += act;
  P.sh_off = off;
  off += rup(size_t(M) * 2 * P.r_pad * 2, 256);
  for (int p = 0; p < 2; ++p) {
    P.sht_off[p] = off;
    off += tr;
  }
  P.saved = M > 0 ? off : 0;
  // forward workspace: [Bg, Bu padded (r % 8 != 0)] [sH_g | sH_u when nothing
  // is saved] [split partials] [counters]
  off = 0;
  for (int p = 0; p < 2; ++p) {
    P.bpad_off[p] = off;
    if (r % 8) off += rup(size_t(d_ff) * P.r_pad * 2, 256);
  }
  P.shws_off = off;
  off += rup(size_t(M) * 2 * P.r_pad * 2, 256);
  P.fwd_ws_min = M > 0 ? off : 0;
  if (pairs_f > 0 && M > 0)
    P.fsplit = main_gemm_plan(int(M), int(2 * rup(d_ff, 128)), pairs_f, allow_wide, kb_f);
  P.fsplit_off = off;
  off += rup(P.fsplit.partial_bytes, 256);
  P.fcnt_off = off;
  off += rup(P.fsplit.counter_bytes, 256);
  P.fwd_ws = M > 0 ? (P.fsplit.k > 1 ? off : P.fwd_ws_min) : 0;
  // backward workspace: [D = d_gate | d_up] [sG_g | sG_u] [sG_g^T] [sG_u^T]
  // [Ag ; Au] [Bg^T, Bu^T (r % 8 != 0)] [split partials] [counters]
  off = 0;
  P.d_off = off;
  off += rup(size_t(M) * 2 * P.half * 2, 256);
  P.sg_off = off;
  off += rup(size_t(M) * 2 * P.r_pad * 2, 256);
  for (int p = 0; p < 2; ++p) {
    P.sgt_off[p] = off;
    off += tr;
  }
  P.agu_off = off;
  off += rup(size_t(2) * P.r_pad * d_in * 2, 256);
  for (int p = 0; p < 2; ++p) {
    P.bt_off[p] = off;
    if (r % 8) off += rup(size_t(P.r_pad) * d_ff * 2, 256);
  }
  P.bwd_ws_min = M > 0 ? off : 0;
  if (pairs_b > 0 && M > 0) P.bsplit = main_gemm_plan(int(M), int(d_in), pairs_b, allow_wide, kb_b);
  P.bsplit_off = off;
  off += rup(P.bsplit.partial_bytes, 256);
  P.bcnt_off = off;
  off += rup(P.bsplit.counter_bytes, 256);
  P.bwd_ws = M > 0 ? (P.bsplit.k > 1 ? off : P.bwd_ws_min) : 0;
  return P;
}

lora_status_t sw_fwd_bf16(const void *X, const void *Wg, const void *Ag, const void *Bg,
                          const void *Wu, const void *Au, const void *Bu, float alpha, int r,
                          int64_t M, int64_t d_in, int64_t d_ff, void *H, void *saved, void *ws,
                          size_t ws_bytes, cudaStream_t st) {
  DevInfo di;
  LORA_TRY(device_info(di));
  SwPlan P = make_sw_plan(M, d_in, d_ff, r, main_gemm_pairs(false, di.sms), 0);
  const bool wide = P.fsplit.wide;  // the gated GEMM's tile width
  const bool split = P.fsplit.k > 1 && ws != nullptr && ws_bytes >= P.fwd_ws;
  if (!split) P = make_sw_plan(M, d_in, d_ff, r, 0, 0);
  unsigned *counters = split ? reinterpret_cast<unsigned *>(at(ws, P.fcnt_off)) : nullptr;
  const float s = alpha / static_cast<float>(r);
  const void *A2[2] = {Ag, Au};
  const void *Bsrc[2] = {Bg, Bu};
  int64_t b_inner = r;
  if (r % 8 != 0) {  // B's row pitch is not a multiple of 16 bytes: pad it
    for (int p = 0; p < 2; ++p) {
      void *Bp = at(ws, P.bpad_off[p]);
      const void *B = Bsrc[p];
      LORA_TRY(run(LORA_K_PREP, st, "pad B", [&] {
        return launch_pad_cols_bf16(B, static_cast<int>(d_ff), r, P.r_pad, Bp, st);
      }));
      Bsrc[p] = Bp;
    }
    b_inner = P.r_pad;
  }
  // without a saved buffer (inference) the low-rank activations live in the
  // workspace and neither their transposes nor gate and up are written
  uint8_t *sh = saved != nullptr ? static_cast<uint8_t *>(saved) + P.sh_off
                                 : static_cast<uint8_t *>(at(ws, P.shws_off));
  // [s X Ag^T | s X Au^T] (and transposes): one launch, both read X
  SkinnyArgs f[2];
  for (int p = 0; p < 2; ++p) {
    LORA_TRY(tmap(&f[p].tmA, X, d_in, M, d_in * 2, 64, 128, "X"));
    LORA_TRY(tmap(&f[p].tmB, A2[p], d_in, r, d_in * 2, 64, P.r_pad, p ? "Au" : "Ag"));
    f[p].a_mn = false;
    f[p].rows = static_cast<int>(M);
    f[p].RP = P.r_pad;
    f[p].K = static_cast<int>(d_in);
    f[p].scale = s;
    f[p].out0 = sh + size_t(p) * P.r_pad * 2;
    f[p].ld0 = 2 * P.r_pad;
    f[p].n0 = P.r_pad;
    f[p].out1 = saved != nullptr ? at(saved, P.sht_off[p]) : nullptr;
    f[p].ld1 = P.Mp;
    f[p].n1 = P.r_pad;
    f[p].dev_status = di.status;
  }
  f[0].zero_ptr = counters;  // the gated GEMM's split counters
  f[0].zero_words = split ? 2 * P.fsplit.rem : 0;
  LORA_TRY(run(LORA_K_DOWN_FWD, st, "s X A^T passes (gate, up)",
               [&] { return launch_skinny(f, 2, di.sms, st); }));

  MainGemmArgs g;
  g.gated = true;
  g.bn = 256;
  g.wide = wide;
  LORA_TRY(tmap(&g.tmA, X, d_in, M, d_in * 2, 64, 128, "X"));
  LORA_TRY(tmap(&g.tmB, Wg, d_in, d_ff, d_in * 2, 64, 128, "Wg"));
  LORA_TRY(tmap(&g.tmB3, Wu, d_in, d_ff, d_in * 2, 64, 128, "Wu"));
  LORA_TRY(tmap(&g.tmA2, sh, 2 * P.r_pad, M, 2 * P.r_pad * 2, 64, 128, "[sH_g | sH_u]"));
  LORA_TRY(tmap(&g.tmB2, Bsrc[0], b_inner, d_ff, b_inner * 2, 64, 128, "Bg"));
  LORA_TRY(tmap(&g.tmB4, Bsrc[1], b_inner, d_ff, b_inner * 2, 64, 128, "Bu"));
  g.M = static_cast<int>(M);
  g.N = static_cast<int>(d_ff);
  g.kb_main = static_cast<int>((d_in + 63) / 64);
  g.k_ext = 2 * P.r_pad;
  g.ext_shift = P.r_pad;
  g.out = H;
  g.aux0 = saved != nullptr ? at(saved, P.gate_off) : nullptr;
  g.aux1 = saved != nullptr ? at(saved, P.up_off) : nullptr;
  g.ldo = d_ff;
  g.b_mn = false;
  g.dev_status = di.status;
  if (split) {
    g.split_k = P.fsplit.k;
    g.split_rem = P.fsplit.rem;
    g.partials = reinterpret_cast<float *>(at(ws, P.fsplit_off));
    g.counters = counters;
  }
  LORA_TRY(out_map(g));
  return run(LORA_K_MAIN_FWD, st, "gated GEMM", [&] { return launch_main_gemm(g, di.sms, st); });
}

lora_status_t sw_bwd_bf16(const void *dH, const void *X, const void *Wg, const void *Ag,
                          const void *Bg, const void *Wu, const void *Au, const void *Bu,
                          const void *saved, float alpha, int r, int64_t M, int64_t d_in,
                          int64_t d_ff, void *dX, void *dAg, void *dBg, void *dAu, void *dBu,
                          void *ws, size_t ws_bytes, cudaStream_t st) {
  DevInfo di;
  LORA_TRY(device_info(di));
  SwPlan P = make_sw_plan(M, d_in, d_ff, r, 0, main_gemm_pairs(true, di.sms));
  const bool wide = P.bsplit.wide;  // the dX GEMM's tile width (with or without the split)
  const bool split = dX != nullptr && P.bsplit.k > 1 && ws != nullptr && ws_bytes >= P.bwd_ws;
  if (!split) P = make_sw_plan(M, d_in, d_ff, r, 0, 0);
  unsigned *counters = split ? reinterpret_cast<unsigned *>(at(ws, P.bcnt_off)) : nullptr;
  const float s = alpha / static_cast<float>(r);
  const uint8_t *sv = static_cast<const uint8_t *>(saved);
  uint8_t *D = static_cast<uint8_t *>(at(ws, P.d_off));
  uint8_t *sG = static_cast<uint8_t *>(at(ws, P.sg_off));
  const int64_t half = P.half;

  // D = [d_gate | d_up]
  LORA_TRY(run(LORA_K_SWIGLU_GRAD, st, "SwiGLU backward (elementwise)", [&] {
    return launch_swiglu_grad_bf16(dH, sv + P.gate_off, sv + P.up_off, M, static_cast<int>(d_ff),
                                   static_cast<int>(half), D, di.sms, st);
  }));

  // per projection: s D_p B_p (and its transpose) and dB_p = D_p^T sH_p,
  // one launch (both read D_p)
  const void *Bs[2] = {Bg, Bu};
  void *dBs[2] = {dBg, dBu};
  for (int p = 0; p < 2; ++p) {
    const uint8_t *Dp = D + size_t(p) * half * 2;
    SkinnyArgs g[2];
    SkinnyArgs &b1 = g[0];
    LORA_TRY(tmap(&b1.tmA, Dp, d_ff, M, 2 * half * 2, 64, 128, p ? "d_up" : "d_gate"));
    if (r % 8 == 0) {
      LORA_TRY(tmap(&b1.tmB, Bs[p], r, d_ff, int64_t(r) * 2, 64, 64, "B (MN-major)"));
      b1.b_mn = true;
    } else {
      void *Bt = at(ws, P.bt_off[p]);
      const void *B = Bs[p];
      LORA_TRY(run(LORA_K_PREP, st, "transpose B", [&] {
        return launch_transpose_pad_bf16(B, static_cast<int>(d_ff), r, P.r_pad, Bt, st);
      }));
      LORA_TRY(tmap(&b1.tmB, Bt, d_ff, P.r_pad, d_ff * 2, 64, P.r_pad, "B^T"));
      b1.b_mn = false;
    }
    b1.a_mn = false;
    b1.rows = static_cast<int>(M);
    b1.RP = P.r_pad;
    b1.K = static_cast<int>(d_ff);
    b1.scale = s;
    b1.out0 = sG + size_t(p) * P.r_pad * 2;
    b1.ld0 = 2 * P.r_pad;
    b1.n0 = P.r_pad;
    b1.out1 = at(ws, P.sgt_off[p]);
    b1.ld1 = P.Mp;
    b1.n1 = P.r_pad;
    b1.dev_status = di.status;
    if (p == 0) {
      b1.zero_ptr = counters;  // the dX GEMM's split counters
      b1.zero_words = split ? 2 * P.bsplit.rem : 0;
    }
    SkinnyArgs &b4 = g[1];
    LORA_TRY(tmap(&b4.tmA, Dp, d_ff, M, 2 * half * 2, 64, 64, "D^T"));
    LORA_TRY(tmap(&b4.tmB, sv + P.sht_off[p], M, P.r_pad, P.Mp * 2, 64, P.r_pad, "sH^T"));
    b4.a_mn = true;
    b4.rows = static_cast<int>(d_ff);
    b4.RP = P.r_pad;
    b4.K = static_cast<int>(M);
    b4.scale = 1.f;
    b4.out0 = dBs[p];
    b4.ld0 = r;
    b4.n0 = r;
    b4.dev_status = di.status;
    LORA_TRY(run(LORA_K_DOWN_BWD_GRAD_B, st, "s D B and dB pass",
                 [&] { return launch_skinny(g, 2, di.sms, st); }));
  }

  // dX = [d_gate | d_up | sG_g | sG_u] . [Wg ; Wu ; Ag ; Au]
  if (dX != nullptr) {
    void *Agu = at(ws, P.agu_off);
    LORA_TRY(run(LORA_K_PREP, st, "stack Ag, Au", [&] {
      return launch_stack_rows_bf16(Ag, Au, r, P.r_pad, d_in, Agu, st);
    }));
    MainGemmArgs b2;
    b2.bn = 256;
    b2.wide = wide;
    LORA_TRY(tmap(&b2.tmA, D, 2 * half, M, 2 * half * 2, 64, 128, "[d_gate | d_up]"));
    LORA_TRY(tmap(&b2.tmB, Wg, d_in, d_ff, d_in * 2, 64, 64, "Wg (MN-major)"));
    LORA_TRY(tmap(&b2.tmB3, Wu, d_in, d_ff, d_in * 2, 64, 64, "Wu (MN-major)"));
    LORA_TRY(tmap(&b2.tmA2, sG, 2 * P.r_pad, M, 2 * P.r_pad * 2, 64, 128, "[sG_g | sG_u]"));
    LORA_TRY(tmap(&b2.tmB2, Agu, d_in, 2 * P.r_pad, d_in * 2, 64, 64, "[Ag ; Au] (MN-major)"));
    b2.M = static_cast<int>(M);
    b2.N = static_cast<int>(d_in);
    b2.kb_main = static_cast<int>(2 * half / 64);
    b2.kb_switch = static_cast<int>(half / 64);
    b2.k_ext = 2 * P.r_pad;
    b2.out = dX;
    b2.ldo = d_in;
    b2.b_mn = true;
    b2.dev_status = di.status;
    if (split) {
      b2.split_k = P.bsplit.k;
      b2.split_rem = P.bsplit.rem;
      b2.partials = reinterpret_cast<float *>(at(ws, P.bsplit_off));
      b2.counters = counters;
    }
    LORA_TRY(out_map(b2));
    LORA_TRY(run(LORA_K_MAIN_BWD, st, "gated dX GEMM",
                 [&] { return launch_main_gemm(b2, di.sms, st); }));
  }

  // dA_p^T = X^T sG_p, written transposed into dA_p: one launch, both read X
  SkinnyArgs a[2];
  void *dAs[2] = {dAg, dAu};
  for (int p = 0; p < 2; ++p) {
    LORA_TRY(tmap(&a[p].tmA, X, d_in, M, d_in * 2, 64, 64, "X^T"));
    LORA_TRY(tmap(&a[p].tmB, at(ws, P.sgt_off[p]), M, P.r_pad, P.Mp * 2, 64, P.r_pad, "sG^T"));
    a[p].a_mn = true;
    a[p].rows = static_cast<int>(d_in);
    a[p].RP = P.r_pad;
    a[p].K = static_cast<int>(M);
    a[p].scale = 1.f;
    a[p].out1 = dAs[p];
    a[p].ld1 = d_in;
    a[p].n1 = r;
    a[p].dev_status = di.status;
    a[p].after_gemm = dX != nullptr;
  }
  return run(LORA_K_GRAD_A, st, "dA passes (gate, up)",
             [&] { return launch_skinny(a, 2, di.sms, st); });
}

// ---------------------------------------------------------------- fp8 frozen W
// 2-D map over a row-major [outer][inner] tensor of bytes (e4m3 codes), box
// 128 bytes x box_outer rows, 128-byte swizzle.
lora_status_t tmap_u8(CUtensorMap *tm, const void *ptr, uint64_t inner, uint64_t outer,
                      uint64_t pitch_bytes, uint32_t box_outer, const char *what) {
  auto fn = encode_fn();
  if (!fn) return fail(LORA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {pitch_bytes};
  cuuint32_t box[2] = {128, box_outer};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(ptr), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(LORA_ERR_CUDA, "tensor map for %s (%llu x %llu bytes) failed: CUresult %d", what,
                (unsigned long long)outer, (unsigned long long)inner, static_cast<int>(r));
  return LORA_OK;
}

// Workspace layout of the fp8 forward and backward.
struct FpPlan {
  int r_pad = 0;
  int64_t Mp = 0;
  size_t xq_off = 0, xs_off = 0, bs_off = 0, fsplit_off = 0, fcnt_off = 0, fwd_ws = 0,
         fwd_ws_min = 0;
  size_t dq_off = 0, ds_off = 0, sg_off = 0, sgt_off = 0, at_off = 0, bt_off = 0,
         bsplit_off = 0, bcnt_off = 0, bwd_ws = 0, bwd_ws_min = 0;
  MainSplit fsplit, bsplit;
};

FpPlan make_fp_plan(int64_t M, int64_t d_in, int64_t d_out, int r, int pairs_f, int pairs_b,
                    bool allow_wide = true) {
  FpPlan P;
  P.r_pad = static_cast<int>(rup(r, 16));
  // K blocks of a tile (128-wide e4m3 main segment, 64-wide extension), for
  // the tile-width cost model: an e4m3 block of 128 takes the MMA time of a
  // bf16 block of 64
  const int kb_f = static_cast<int>((d_in + 127) / 128 + (P.r_pad + 63) / 64);
  const int kb_b = static_cast<int>((d_out + 127) / 128 + (P.r_pad + 63) / 64);
  P.Mp = rup(M, 8);
  // forward: [X codes] [X scales] [B / w_scale, padded] [split partials] [counters]
  size_t off = 0;
  P.xq_off = off;
  off += rup(size_t(M) * d_in, 256);
  P.xs_off = off;
  off += rup(size_t(M) * 4, 256);
  P.bs_off = off;
  off += rup(size_t(d_out) * P.r_pad * 2, 256);
  P.fwd_ws_min = M > 0 ? off : 0;
  if (pairs_f > 0 && M > 0) P.fsplit = main_gemm_plan(int(M), int(d_out), pairs_f, allow_wide, kb_f);
  P.fsplit_off = off;
  off += rup(P.fsplit.partial_bytes, 256);
  P.fcnt_off = off;
  off += rup(P.fsplit.counter_bytes, 256);
  P.fwd_ws = M > 0 ? (P.fsplit.k > 1 ? off : P.fwd_ws_min) : 0;
  // backward: [dY codes] [dY scales] [sG / dy_scale] [sG^T] [(A / w_scale)^T]
  // [B^T (r % 8 != 0)] [split partials] [counters]
  off = 0;
  P.dq_off = off;
  off += rup(size_t(M) * d_out, 256);
  P.ds_off = off;
  off += rup(size_t(M) * 4, 256);
  P.sg_off = off;
  off += rup(size_t(M) * P.r_pad * 2, 256);
  P.sgt_off = off;
  off += rup(size_t(P.r_pad) * P.Mp * 2, 256);
  P.at_off = off;
  off += rup(size_t(d_in) * P.r_pad * 2, 256);
  P.bt_off = off;
  if (r % 8) off += rup(size_t(P.r_pad) * d_out * 2, 256);
  P.bwd_ws_min = M > 0 ? off : 0;
  if (pairs_b > 0 && M > 0) P.bsplit = main_gemm_plan(int(M), int(d_in), pairs_b, allow_wide, kb_b);
  P.bsplit_off = off;
  off += rup(P.bsplit.partial_bytes, 256);
  P.bcnt_off = off;
  off += rup(P.bsplit.counter_bytes, 256);
  P.bwd_ws = M > 0 ? (P.bsplit.k > 1 ? off : P.bwd_ws_min) : 0;
  return P;
}

lora_status_t fp8_fwd(const void *X, const void *Wq, const float *w_scale, const void *A,
                      const void *B, float alpha, int r, int64_t M, int64_t d_in, int64_t d_out,
                      void *Y, void *saved, void *ws, size_t ws_bytes, cudaStream_t st) {
  DevInfo di;
  LORA_TRY(device_info(di));
  FpPlan P = make_fp_plan(M, d_in, d_out, r, main_gemm_pairs(false, di.sms), 0);
  const bool wide = P.fsplit.wide;  // 256 x 512 tiles (with or without the split)
  const bool split = P.fsplit.k > 1 && ws != nullptr && ws_bytes >= P.fwd_ws;
  if (!split) P = make_fp_plan(M, d_in, d_out, r, 0, 0);
  unsigned *counters = split ? reinterpret_cast<unsigned *>(at(ws, P.fcnt_off)) : nullptr;
  const Plan L = make_plan(M, d_in, d_out, r, LORA_BF16);  // the saved buffer's layout
  const float s = alpha / static_cast<float>(r);
  void *xq = at(ws, P.xq_off);
  float *xs = reinterpret_cast<float *>(at(ws, P.xs_off));  // x_scale * w_scale per row
  LORA_TRY(run(LORA_K_QUANT, st, "quantise X",
               [&] { return launch_quant_rows_e4m3(X, M, d_in, xq, xs, w_scale, st); }));
  const void *Bsrc = B;
  int64_t b_inner = r;
  if (r % 8 != 0) {  // B's row pitch is not a multiple of 16 bytes: pad it
    void *bs = at(ws, P.bs_off);
    LORA_TRY(run(LORA_K_PREP, st, "pad B", [&] {
      return launch_pad_cols_bf16(B, static_cast<int>(d_out), r, P.r_pad, bs, st);
    }));
    Bsrc = bs;
    b_inner = P.r_pad;
  }
  // sH / (x_scale w_scale) (row-major, the GEMM's extension: every tile's
  // accumulator is multiplied by x_scale w_scale in the epilogue) and sH^T
  // (unscaled, for the backward)
  SkinnyArgs f1;
  LORA_TRY(tmap(&f1.tmA, X, d_in, M, d_in * 2, 64, 128, "X"));
  LORA_TRY(tmap(&f1.tmB, A, d_in, r, d_in * 2, 64, P.r_pad, "A"));
  f1.a_mn = false;
  f1.rows = static_cast<int>(M);
  f1.RP = P.r_pad;
  f1.K = static_cast<int>(d_in);
  f1.scale = s;
  f1.out0 = saved;
  f1.ld0 = P.r_pad;
  f1.n0 = P.r_pad;
  f1.row_div = xs;
  f1.out1 = at(saved, L.sHt_off);
  f1.ld1 = P.Mp;
  f1.n1 = P.r_pad;
  f1.dev_status = di.status;
  f1.zero_ptr = counters;
  f1.zero_words = split ? 2 * P.fsplit.rem : 0;
  LORA_TRY(run(LORA_K_DOWN_FWD, st, "s X A^T pass", [&] { return launch_skinny(&f1, 1, di.sms, st); }));
  MainGemmArgs g;
  g.fp8 = true;
  g.bn = 256;
  g.wide = wide;
  LORA_TRY(tmap_u8(&g.tmA, xq, d_in, M, d_in, 128, "X (e4m3)"));
  LORA_TRY(tmap_u8(&g.tmB, Wq, d_in, d_out, d_in, 128, "W (e4m3)"));
  LORA_TRY(tmap(&g.tmA2, saved, P.r_pad, M, P.r_pad * 2, 64, 128, "sH / row scale"));
  LORA_TRY(tmap(&g.tmB2, Bsrc, b_inner, d_out, b_inner * 2, 64, 128, "B"));
  g.M = static_cast<int>(M);
  g.N = static_cast<int>(d_out);
  g.kb_main = static_cast<int>((d_in + 127) / 128);
  g.k_ext = P.r_pad;
  g.out = Y;
  g.ldo = d_out;
  g.row_scale = xs;
  g.dev_status = di.status;
  if (split) {
    g.split_k = P.fsplit.k;
    g.split_rem = P.fsplit.rem;
    g.partials = reinterpret_cast<float *>(at(ws, P.fsplit_off));
    g.counters = counters;
  }
  LORA_TRY(out_map(g));
  return run(LORA_K_MAIN_FWD, st, "fp8 forward GEMM", [&] { return launch_main_gemm(g, di.sms, st); });
}

lora_status_t fp8_bwd(const void *dY, const void *X, const void *WqT, const float *w_scale,
                      const void *A, const void *B, const void *saved, float alpha, int r,
                      int64_t M, int64_t d_in, int64_t d_out, void *dX, void *dA, void *dB,
                      void *ws, size_t ws_bytes, cudaStream_t st) {
  DevInfo di;
  LORA_TRY(device_info(di));
  FpPlan P = make_fp_plan(M, d_in, d_out, r, 0, main_gemm_pairs(false, di.sms));
  const bool wide = P.bsplit.wide;
  const bool split = dX != nullptr && P.bsplit.k > 1 && ws != nullptr && ws_bytes >= P.bwd_ws;
  if (!split) P = make_fp_plan(M, d_in, d_out, r, 0, 0);
  unsigned *counters = split ? reinterpret_cast<unsigned *>(at(ws, P.bcnt_off)) : nullptr;
  const Plan L = make_plan(M, d_in, d_out, r, LORA_BF16);
  const float s = alpha / static_cast<float>(r);
  const void *sHt = static_cast<const uint8_t *>(saved) + L.sHt_off;
  void *dq = at(ws, P.dq_off);
  float *ds = reinterpret_cast<float *>(at(ws, P.ds_off));  // dy_scale * w_scale per row
  void *sG = at(ws, P.sg_off);
  void *sGt = at(ws, P.sgt_off);
  LORA_TRY(run(LORA_K_QUANT, st, "quantise dY",
               [&] { return launch_quant_rows_e4m3(dY, M, d_out, dq, ds, w_scale, st); }));

  // sG / (dy_scale w_scale) (row-major, the dX GEMM's extension) and sG^T, and
  // dB = dY^T sH: one launch, both read dY
  SkinnyArgs g[2];
  SkinnyArgs &b1 = g[0];
  LORA_TRY(tmap(&b1.tmA, dY, d_out, M, d_out * 2, 64, 128, "dY"));
  if (r % 8 == 0) {
    LORA_TRY(tmap(&b1.tmB, B, r, d_out, int64_t(r) * 2, 64, 64, "B (MN-major)"));
    b1.b_mn = true;
  } else {
    void *Bt = at(ws, P.bt_off);
    LORA_TRY(run(LORA_K_PREP, st, "transpose B", [&] {
      return launch_transpose_pad_bf16(B, static_cast<int>(d_out), r, P.r_pad, Bt, st);
    }));
    LORA_TRY(tmap(&b1.tmB, Bt, d_out, P.r_pad, d_out * 2, 64, P.r_pad, "B^T"));
    b1.b_mn = false;
  }
  b1.a_mn = false;
  b1.rows = static_cast<int>(M);
  b1.RP = P.r_pad;
  b1.K = static_cast<int>(d_out);
  b1.scale = s;
  b1.out0 = sG;
  b1.ld0 = P.r_pad;
  b1.n0 = P.r_pad;
  b1.row_div = ds;
  b1.out1 = sGt;
  b1.ld1 = P.Mp;
  b1.n1 = P.r_pad;
  b1.dev_status = di.status;
  b1.zero_ptr = counters;
  b1.zero_words = split ? 2 * P.bsplit.rem : 0;
  SkinnyArgs &b4 = g[1];
  LORA_TRY(tmap(&b4.tmA, dY, d_out, M, d_out * 2, 64, 64, "dY^T"));
  LORA_TRY(tmap(&b4.tmB, sHt, M, P.r_pad, P.Mp * 2, 64, P.r_pad, "sH^T"));
  b4.a_mn = true;
  b4.rows = static_cast<int>(d_out);
  b4.RP = P.r_pad;
  b4.K = static_cast<int>(M);
  b4.scale = 1.f;
  b4.out0 = dB;
  b4.ld0 = r;
  b4.n0 = r;
  b4.dev_status = di.status;
  LORA_TRY(run(LORA_K_DOWN_BWD_GRAD_B, st, "s dY B and dB pass",
               [&] { return launch_skinny(g, 2, di.sms, st); }));

  // dX = Q(dY) Q(W) + sG A: the accumulator takes Q codes and sG / (dy_scale
  // w_scale), and the epilogue multiplies by dy_scale w_scale
  if (dX != nullptr) {
    void *at_ = at(ws, P.at_off);
    LORA_TRY(run(LORA_K_PREP, st, "A^T", [&] {
      return launch_transpose_scale_bf16(A, r, d_in, P.r_pad, nullptr, at_, st);
    }));
    MainGemmArgs b2;
    b2.fp8 = true;
    b2.bn = 256;
    b2.wide = wide;
    LORA_TRY(tmap_u8(&b2.tmA, dq, d_out, M, d_out, 128, "dY (e4m3)"));
    LORA_TRY(tmap_u8(&b2.tmB, WqT, d_out, d_in, d_out, 128, "W^T (e4m3)"));
    LORA_TRY(tmap(&b2.tmA2, sG, P.r_pad, M, P.r_pad * 2, 64, 128, "sG / row scale"));
    LORA_TRY(tmap(&b2.tmB2, at_, P.r_pad, d_in, P.r_pad * 2, 64, 128, "A^T"));
    b2.M = static_cast<int>(M);
    b2.N = static_cast<int>(d_in);
    b2.kb_main = static_cast<int>((d_out + 127) / 128);
    b2.k_ext = P.r_pad;
    b2.out = dX;
    b2.ldo = d_in;
    b2.row_scale = ds;
    b2.dev_status = di.status;
    if (split) {
      b2.split_k = P.bsplit.k;
      b2.split_rem = P.bsplit.rem;
      b2.partials = reinterpret_cast<float *>(at(ws, P.bsplit_off));
      b2.counters = counters;
    }
    LORA_TRY(out_map(b2));
    LORA_TRY(run(LORA_K_MAIN_BWD, st, "fp8 dX GEMM",
                 [&] { return launch_main_gemm(b2, di.sms, st); }));
  }

  // dA^T = X^T sG   (the unscaled transpose)
  SkinnyArgs b3;
  LORA_TRY(tmap(&b3.tmA, X, d_in, M, d_in * 2, 64, 64, "X^T"));
  LORA_TRY(tmap(&b3.tmB, sGt, M, P.r_pad, P.Mp * 2, 64, P.r_pad, "sG^T"));
  b3.a_mn = true;
  b3.rows = static_cast<int>(d_in);
  b3.RP = P.r_pad;
  b3.K = static_cast<int>(M);
  b3.scale = 1.f;
  b3.out1 = dA;
  b3.ld1 = d_in;
  b3.n1 = r;
  b3.dev_status = di.status;
  b3.after_gemm = dX != nullptr;
  return run(LORA_K_GRAD_A, st, "dA pass", [&] { return launch_skinny(&b3, 1, di.sms, st); });
}

}  // namespace
}  // namespace lora

using namespace lora;

// ---------------------------------------------------------------- no-alloc scratch
// Built-in scratch of lora_linear_bwd_noalloc: one file-scope device array of
// LORA_NOALLOC_SCRATCH_BYTES, held by every GPU that loads this library until
// the process exits.  All calls share it.
static __device__ __align__(256) unsigned char g_noalloc_scratch[LORA_NOALLOC_SCRATCH_BYTES];

namespace {
std::mutex g_noalloc_mtx;
void *g_noalloc_ptr[lora::kMaxDevices] = {};

// Device address of the scratch array on the current device.  The array's
// name is only a host-side stand-in, so the address is looked up once per
// device (with that device current) and cached.  The cached address belongs
// to the device's primary context (the one the runtime makes current); like
// the status-word address of device_info, it does not survive
// cudaDeviceReset.
lora_status_t noalloc_scratch(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return lora::fail(LORA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= lora::kMaxDevices)
    return lora::fail(LORA_ERR_UNSUPPORTED, "device index %d", dev);
  std::lock_guard<std::mutex> lock(g_noalloc_mtx);
  if (g_noalloc_ptr[dev] == nullptr) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr)
      return lora::fail(LORA_ERR_CUDA, "address of the built-in scratch: %s",
                        cudaGetErrorString(e));
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return LORA_OK;
}
}  // namespace


extern "C" {

size_t lora_linear_saved_bytes(int64_t M, int r, lora_dtype_t dtype) {
  if (M < 0 || r < 1 || r > 256 || (dtype != LORA_BF16 && dtype != LORA_FP32)) return 0;
  return make_plan(M, 1, 1, r, dtype).saved;
}

size_t lora_linear_workspace_bytes(int64_t M, int64_t d_in, int64_t d_out, int r,
                                   lora_dtype_t dtype) {
  if (M < 0 || d_in < 1 || d_out < 1 || r < 1 || r > 256 ||
      (dtype != LORA_BF16 && dtype != LORA_FP32))
    return 0;
  // sized for the current device (its number of main-GEMM CTA pairs); with
  // no usable device, for a GB300's 76 pairs
  int pairs = 76;
  if (dtype == LORA_BF16) {
    int dev = 0, sms = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) == cudaSuccess &&
        major == 10 && minor == 3)
      pairs = main_gemm_pairs(false, sms);
    cudaGetLastError();
  }
  // room for the tail split of either tile width (the 4-bit layer, sized
  // here too, has 256-wide tiles only)
  size_t need = 0;
  for (int allow_wide = 0; allow_wide < 2; ++allow_wide) {
    const Plan P = make_plan(M, d_in, d_out, r, dtype, pairs, allow_wide != 0);
    need = P.fwd_ws > need ? P.fwd_ws : need;
    need = P.bwd_ws > need ? P.bwd_ws : need;
  }
  return need;
}

lora_status_t lora_linear_fwd(const void *X, const void *W, const void *A, const void *B,
                              float alpha, int r, int64_t M, int64_t d_in, int64_t d_out,
                              lora_dtype_t dtype, void *Y, void *saved, void *workspace,
                              size_t workspace_bytes, void *stream) {
  t_err.clear();
  LORA_TRY(check_shape(r, M, d_in, d_out, dtype, alpha));
  const bool empty = M == 0;
  LORA_TRY(check_ptr(X, "X", empty));
  LORA_TRY(check_ptr(W, "W"));
  LORA_TRY(check_ptr(A, "A"));
  LORA_TRY(check_ptr(B, "B"));
  LORA_TRY(check_ptr(Y, "Y", empty));
  LORA_TRY(check_ptr(saved, "saved", empty));
  const Plan P = make_plan(M, d_in, d_out, r, dtype);
  LORA_TRY(check_ws(workspace, workspace_bytes, P.fwd_ws_min));
  if (empty) return LORA_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == LORA_BF16)
    return fwd_bf16(X, W, A, B, alpha, r, M, d_in, d_out, Y, saved, workspace, workspace_bytes, st);
  return fwd_f32(X, W, A, B, alpha, r, M, d_in, d_out, Y, saved, st);
}

lora_status_t lora_linear_bwd(const void *dY, const void *X, const void *W, const void *A,
                              const void *B, const void *saved, float alpha, int r, int64_t M,
                              int64_t d_in, int64_t d_out, lora_dtype_t dtype, void *dX, void *dA,
                              void *dB, void *workspace, size_t workspace_bytes, void *stream) {
  t_err.clear();
  LORA_TRY(check_shape(r, M, d_in, d_out, dtype, alpha));
  const bool empty = M == 0;
  LORA_TRY(check_ptr(dY, "dY", empty));
  LORA_TRY(check_ptr(X, "X", empty));
  LORA_TRY(check_ptr(W, "W"));
  LORA_TRY(check_ptr(A, "A"));
  LORA_TRY(check_ptr(B, "B"));
  LORA_TRY(check_ptr(saved, "saved", true));
  LORA_TRY(check_ptr(dX, "dX", true));
  LORA_TRY(check_ptr(dA, "dA"));
  LORA_TRY(check_ptr(dB, "dB"));
  const Plan P = make_plan(M, d_in, d_out, r, dtype);
  size_t need = saved != nullptr ? P.bwd_ws_min : P.bwd_ws;  // recompute room if no saved
  if (empty) need = 0;
  LORA_TRY(check_ws(workspace, workspace_bytes, need));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (empty) {  // sums over zero tokens
    const size_t es = dtype == LORA_BF16 ? 2 : 4;
    cudaError_t e = cudaMemsetAsync(dA, 0, size_t(r) * d_in * es, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(dB, 0, size_t(d_out) * r * es, st);
    if (e != cudaSuccess) return fail(LORA_ERR_CUDA, "zero dA/dB: %s", cudaGetErrorString(e));
    return LORA_OK;
  }
  if (dtype == LORA_BF16)
    return bwd_bf16(dY, X, W, A, B, saved, alpha, r, M, d_in, d_out, dX, dA, dB, workspace,
                    workspace_bytes, st);
  return bwd_f32(dY, X, W, A, B, saved, alpha, r, M, d_in, d_out, dX, dA, dB, workspace, st);
}

lora_status_t lora_linear_bwd_noalloc(const void *dY, const void *X, const void *W,
                                      const void *A, const void *B, const void *saved,
                                      float alpha, int r, int64_t M, int64_t d_in,
                                      int64_t d_out, lora_dtype_t dtype, void *dX, void *dA,
                                      void *dB, void *stream) {
  t_err.clear();
  LORA_TRY(check_shape(r, M, d_in, d_out, dtype, alpha));
  const bool empty = M == 0;
  LORA_TRY(check_ptr(dY, "dY", empty));
  LORA_TRY(check_ptr(X, "X", empty));
  LORA_TRY(check_ptr(W, "W"));
  LORA_TRY(check_ptr(A, "A"));
  LORA_TRY(check_ptr(B, "B"));
  LORA_TRY(check_ptr(saved, "saved", true));
  LORA_TRY(check_ptr(dX, "dX", true));
  LORA_TRY(check_ptr(dA, "dA"));
  LORA_TRY(check_ptr(dB, "dB"));
  const Plan P = make_plan(M, d_in, d_out, r, dtype);
  size_t need = saved != nullptr ? P.bwd_ws_min : P.bwd_ws;
  if (empty) need = 0;
  if (need > LORA_NOALLOC_SCRATCH_BYTES)
    return fail(LORA_ERR_UNSUPPORTED,
                "this shape needs %zu bytes of scratch; the built-in scratch of "
                "lora_linear_bwd_noalloc holds %zu (use lora_linear_bwd with a workspace)",
                need, static_cast<size_t>(LORA_NOALLOC_SCRATCH_BYTES));
  // Nothing in the scratch has to start at zero: every byte the kernels read
  // is written earlier in the same call (the dX GEMM's tail-split counters
  // are zeroed by the pass that precedes it).
  void *ws = nullptr;
  if (!empty) {
    // the device check of the other entry points comes first, so that a
    // device this library was not built for gets the same status here
    DevInfo di;
    LORA_TRY(device_info(di));
    LORA_TRY(noalloc_scratch(&ws));
  }
  return lora_linear_bwd(dY, X, W, A, B, saved, alpha, r, M, d_in, d_out, dtype, dX, dA, dB, ws,
                         LORA_NOALLOC_SCRATCH_BYTES, stream);
}

const char *lora_status_string(lora_status_t status) {
  switch (status) {
    case LORA_OK: return "LORA_OK";
    case LORA_ERR_INVALID_ARG: return "LORA_ERR_INVALID_ARG";
    case LORA_ERR_UNSUPPORTED: return "LORA_ERR_UNSUPPORTED";
    case LORA_ERR_WORKSPACE: return "LORA_ERR_WORKSPACE";
    case LORA_ERR_CUDA: return "LORA_ERR_CUDA";
    case LORA_ERR_TIMEOUT: return "LORA_ERR_TIMEOUT";
  }
  return "LORA_ERR_UNKNOWN";
}

const char *lora_last_error(void) { return t_err.c_str(); }

lora_status_t lora_device_status(int clear) {
  t_err.clear();
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return fail(LORA_ERR_CUDA, "synchronize: %s", cudaGetErrorString(e));
  unsigned v = 0;
  e = cudaMemcpyFromSymbol(&v, g_dev_status, sizeof(v));
  if (e != cudaSuccess) return fail(LORA_ERR_CUDA, "read status: %s", cudaGetErrorString(e));
  if (clear) {
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_dev_status, &zero, sizeof(zero));
    if (e != cudaSuccess) return fail(LORA_ERR_CUDA, "clear status: %s", cudaGetErrorString(e));
  }
  if (v & kDevErrTimeout) return fail(LORA_ERR_TIMEOUT, "a device-side wait ran out (0x%x)", v);
  return LORA_OK;
}

uint64_t lora_launch_count(void) { return g_launches.load(); }

lora_status_t lora_set_timing_events(void *const *events, int *kinds, int n_pairs) {
  t_err.clear();
  if (events != nullptr && n_pairs < 0)
    return fail(LORA_ERR_INVALID_ARG, "n_pairs = %d is negative", n_pairs);
  if (events != nullptr)
    for (int i = 0; i < 2 * n_pairs; ++i)
      if (events[i] == nullptr)
        return fail(LORA_ERR_INVALID_ARG, "timing event %d is NULL (not created yet?)", i);
  t_hook.events = events;
  t_hook.kinds = kinds;
  t_hook.n = events ? n_pairs : 0;
  t_hook.used = 0;
  return LORA_OK;
}

int lora_timing_used(void) { return t_hook.used; }

static int current_pairs(bool b_mn);

// ---------------------------------------------------------------- fp8 frozen W
static lora_status_t check_fp8_shape(int r, int64_t M, int64_t d_in, int64_t d_out,
                                     float alpha) {
  LORA_TRY(check_shape(r, M, d_in, d_out, LORA_BF16, alpha));
  if (d_in % 16 != 0 || d_out % 16 != 0 || d_in > 65536 || d_out > 65536)
    return fail(LORA_ERR_UNSUPPORTED,
                "the fp8 variant needs d_in and d_out to be multiples of 16, at most 65536 "
                "(got %lld, %lld)", (long long)d_in, (long long)d_out);
  return LORA_OK;
}

size_t lora_fp8_quantize_w_workspace_bytes(void) { return 256; }

lora_status_t lora_fp8_quantize_w(const void *W, int64_t d_out, int64_t d_in, void *Wq,
                                  void *WqT, float *w_scale, void *workspace,
                                  size_t workspace_bytes, void *stream) {
  t_err.clear();
  if (d_out < 1 || d_in < 1 || d_out % 16 != 0 || d_in % 16 != 0)
    return fail(LORA_ERR_UNSUPPORTED, "d_out, d_in must be positive multiples of 16");
  if (d_out > INT32_MAX / 2 || d_in > INT32_MAX / 2)
    return fail(LORA_ERR_UNSUPPORTED, "a dimension exceeds 2^30");
  LORA_TRY(check_ptr(W, "W"));
  LORA_TRY(check_ptr(Wq, "Wq"));
  LORA_TRY(check_ptr(WqT, "WqT"));
  if (w_scale == nullptr) return fail(LORA_ERR_INVALID_ARG, "w_scale is NULL");
  LORA_TRY(check_ws(workspace, workspace_bytes, lora_fp8_quantize_w_workspace_bytes()));
  DevInfo di;
  LORA_TRY(device_info(di));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return run(LORA_K_QUANT, st, "quantise W", [&] {
    return launch_quant_tensor_e4m3(W, static_cast<int>(d_out), static_cast<int>(d_in),
                                    static_cast<unsigned *>(workspace), Wq, WqT, w_scale, di.sms,
                                    st);
  });
}

lora_status_t lora_fp8_quantize_rows(const void *x, int64_t rows, int64_t cols, void *q,
                                     float *scale, void *stream) {
  t_err.clear();
  if (rows < 0 || cols < 1 || cols % 16 != 0 || rows > INT32_MAX || cols > 65536)
    return fail(LORA_ERR_UNSUPPORTED,
                "rows >= 0 and cols a positive multiple of 16, at most 65536, needed");
  if (rows == 0) return LORA_OK;
  LORA_TRY(check_ptr(x, "x"));
  LORA_TRY(check_ptr(q, "q"));
  if (scale == nullptr) return fail(LORA_ERR_INVALID_ARG, "scale is NULL");
  DevInfo di;
  LORA_TRY(device_info(di));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return run(LORA_K_QUANT, st, "quantise rows",
             [&] { return launch_quant_rows_e4m3(x, rows, cols, q, scale, nullptr, st); });
}

size_t lora_fp8_workspace_bytes(int64_t M, int64_t d_in, int64_t d_out, int r) {
  if (M < 0 || d_in < 1 || d_out < 1 || r < 1 || r > 256) return 0;
  // room for the tail split of either tile width
  size_t need = 0;
  for (int allow_wide = 0; allow_wide < 2; ++allow_wide) {
    const FpPlan P = make_fp_plan(M, d_in, d_out, r, current_pairs(false), current_pairs(false),
                                  allow_wide != 0);
    need = P.fwd_ws > need ? P.fwd_ws : need;
    need = P.bwd_ws > need ? P.bwd_ws : need;
  }
  return need;
}

lora_status_t lora_fp8_fwd(const void *X, const void *Wq, const float *w_scale, const void *A,
                           const void *B, float alpha, int r, int64_t M, int64_t d_in,
                           int64_t d_out, void *Y, void *saved, void *workspace,
                           size_t workspace_bytes, void *stream) {
  t_err.clear();
  LORA_TRY(check_fp8_shape(r, M, d_in, d_out, alpha));
  const bool empty = M == 0;
  LORA_TRY(check_ptr(X, "X", empty));
  LORA_TRY(check_ptr(Wq, "Wq"));
  if (w_scale == nullptr) return fail(LORA_ERR_INVALID_ARG, "w_scale is NULL");
  LORA_TRY(check_ptr(A, "A"));
  LORA_TRY(check_ptr(B, "B"));
  LORA_TRY(check_ptr(Y, "Y", empty));
  LORA_TRY(check_ptr(saved, "saved", empty));
  const FpPlan P = make_fp_plan(M, d_in, d_out, r, 0, 0);
  LORA_TRY(check_ws(workspace, workspace_bytes, P.fwd_ws_min));
  if (empty) return LORA_OK;
  return fp8_fwd(X, Wq, w_scale, A, B, alpha, r, M, d_in, d_out, Y, saved, workspace,
                 workspace_bytes, static_cast<cudaStream_t>(stream));
}

lora_status_t lora_fp8_bwd(const void *dY, const void *X, const void *WqT, const float *w_scale,
                           const void *A, const void *B, const void *saved, float alpha, int r,
                           int64_t M, int64_t d_in, int64_t d_out, void *dX, void *dA, void *dB,
                           void *workspace, size_t workspace_bytes, void *stream) {
  t_err.clear();
  LORA_TRY(check_fp8_shape(r, M, d_in, d_out, alpha));
  const bool empty = M == 0;
  LORA_TRY(check_ptr(dY, "dY", empty));
  LORA_TRY(check_ptr(X, "X", empty));
  LORA_TRY(check_ptr(WqT, "WqT"));
  if (w_scale == nullptr) return fail(LORA_ERR_INVALID_ARG, "w_scale is NULL");
  LORA_TRY(check_ptr(A, "A"));
  LORA_TRY(check_ptr(B, "B"));
  LORA_TRY(check_ptr(saved, "saved", empty));
  LORA_TRY(check_ptr(dX, "dX", true));
  LORA_TRY(check_ptr(dA, "dA"));
  LORA_TRY(check_ptr(dB, "dB"));
  const FpPlan P = make_fp_plan(M, d_in, d_out, r, 0, 0);
  LORA_TRY(check_ws(workspace, workspace_bytes, empty ? 0 : P.bwd_ws_min));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (empty) {  // sums over zero tokens
    cudaError_t e = cudaMemsetAsync(dA, 0, size_t(r) * d_in * 2, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(dB, 0, size_t(d_out) * r * 2, st);
    if (e != cudaSuccess) return fail(LORA_ERR_CUDA, "zero dA/dB: %s", cudaGetErrorString(e));
    return LORA_OK;
  }
  return fp8_bwd(dY, X, WqT, w_scale, A, B, saved, alpha, r, M, d_in, d_out, dX, dA, dB,
                 workspace, workspace_bytes, st);
}

// ---------------------------------------------------------------- SwiGLU pair
static lora_status_t check_sw_shape(int r, int64_t M, int64_t d_in, int64_t d_ff,
                                    lora_dtype_t dt, float alpha) {
  if (dt == LORA_FP32) return fail(LORA_ERR_UNSUPPORTED, "the SwiGLU pair is built for bf16 only");
  LORA_TRY(check_shape(r, M, d_in, d_ff, dt, alpha));
  // the gated GEMM's tiles are 128 output columns wide
  const int64_t t = ((M + 127) / 128) * ((d_ff + 127) / 128);
  if (t > INT32_MAX / 2) return fail(LORA_ERR_UNSUPPORTED, "too many output tiles");
  return LORA_OK;
}

static int current_pairs(bool b_mn) {
  int pairs = 76;  // a GB300's, when no usable device is current
  int dev = 0, sms = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) == cudaSuccess &&
      major == 10 && minor == 3)
    pairs = main_gemm_pairs(b_mn, sms);
  cudaGetLastError();
  return pairs;
}

size_t lora_swiglu_saved_bytes(int64_t M, int64_t d_ff, int r) {
  if (M < 0 || d_ff < 1 || r < 1 || r > 256) return 0;
  return make_sw_plan(M, 1, d_ff, r, 0, 0).saved;
}

size_t lora_swiglu_workspace_bytes(int64_t M, int64_t d_in, int64_t d_ff, int r) {
  if (M < 0 || d_in < 1 || d_ff < 1 || r < 1 || r > 256) return 0;
  // room for the dX GEMM's tail split at either tile width
  size_t need = 0;
  for (int allow_wide = 0; allow_wide < 2; ++allow_wide) {
    const SwPlan P = make_sw_plan(M, d_in, d_ff, r, current_pairs(false), current_pairs(true),
                                  allow_wide != 0);
    need = P.fwd_ws > need ? P.fwd_ws : need;
    need = P.bwd_ws > need ? P.bwd_ws : need;
  }
  return need;
}

lora_status_t lora_swiglu_fwd(const void *X, const void *Wg, const void *Ag, const void *Bg,
                              const void *Wu, const void *Au, const void *Bu, float alpha,
                              int r, int64_t M, int64_t d_in, int64_t d_ff, lora_dtype_t dtype,
                              void *H, void *saved, void *workspace, size_t workspace_bytes,
                              void *stream) {
  t_err.clear();
  LORA_TRY(check_sw_shape(r, M, d_in, d_ff, dtype, alpha));
  const bool empty = M == 0;
  LORA_TRY(check_ptr(X, "X", empty));
  LORA_TRY(check_ptr(Wg, "Wg"));
  LORA_TRY(check_ptr(Ag, "Ag"));
  LORA_TRY(check_ptr(Bg, "Bg"));
  LORA_TRY(check_ptr(Wu, "Wu"));
  LORA_TRY(check_ptr(Au, "Au"));
  LORA_TRY(check_ptr(Bu, "Bu"));
  LORA_TRY(check_ptr(H, "H", empty));
  LORA_TRY(check_ptr(saved, "saved", true));
  const SwPlan P = make_sw_plan(M, d_in, d_ff, r, 0, 0);
  LORA_TRY(check_ws(workspace, workspace_bytes, P.fwd_ws_min));
  if (empty) return LORA_OK;
  return sw_fwd_bf16(X, Wg, Ag, Bg, Wu, Au, Bu, alpha, r, M, d_in, d_ff, H, saved, workspace,
                     workspace_bytes, static_cast<cudaStream_t>(stream));
}

lora_status_t lora_swiglu_bwd(const void *dH, const void *X, const void *Wg, const void *Ag,
                              const void *Bg, const void *Wu, const void *Au, const void *Bu,
                              const void *saved, float alpha, int r, int64_t M, int64_t d_in,
                              int64_t d_ff, lora_dtype_t dtype, void *dX, void *dAg, void *dBg,
                              void *dAu, void *dBu, void *workspace, size_t workspace_bytes,
                              void *stream) {
  t_err.clear();
  LORA_TRY(check_sw_shape(r, M, d_in, d_ff, dtype, alpha));
  const bool empty = M == 0;
  LORA_TRY(check_ptr(dH, "dH", empty));
  LORA_TRY(check_ptr(X, "X", empty));
  LORA_TRY(check_ptr(Wg, "Wg"));
  LORA_TRY(check_ptr(Ag, "Ag"));
  LORA_TRY(check_ptr(Bg, "Bg"));
  LORA_TRY(check_ptr(Wu, "Wu"));
  LORA_TRY(check_ptr(Au, "Au"));
  LORA_TRY(check_ptr(Bu, "Bu"));
  LORA_TRY(check_ptr(saved, "saved", empty));
  LORA_TRY(check_ptr(dX, "dX", true));
  LORA_TRY(check_ptr(dAg, "dAg"));
  LORA_TRY(check_ptr(dBg, "dBg"));
  LORA_TRY(check_ptr(dAu, "dAu"));
  LORA_TRY(check_ptr(dBu, "dBu"));
  const SwPlan P = make_sw_plan(M, d_in, d_ff, r, 0, 0);
  LORA_TRY(check_ws(workspace, workspace_bytes, empty ? 0 : P.bwd_ws_min));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (empty) {  // sums over zero tokens
    cudaError_t e = cudaSuccess;
    for (void *p : {dAg, dAu})
      if (e == cudaSuccess) e = cudaMemsetAsync(p, 0, size_t(r) * d_in * 2, st);
    for (void *p : {dBg, dBu})
      if (e == cudaSuccess) e = cudaMemsetAsync(p, 0, size_t(d_ff) * r * 2, st);
    if (e != cudaSuccess) return fail(LORA_ERR_CUDA, "zero dA/dB: %s", cudaGetErrorString(e));
    return LORA_OK;
  }
  return sw_bwd_bf16(dH, X, Wg, Ag, Bg, Wu, Au, Bu, saved, alpha, r, M, d_in, d_ff, dX, dAg, dBg,
                     dAu, dBu, workspace, workspace_bytes, st);
}

// ---------------------------------------------------------------- 4-bit frozen W
static lora_status_t check_q4_dims(int64_t d_in, int64_t d_out) {
  if (d_in < 64 || d_out < 8 || d_in % 64 != 0 || d_out % 8 != 0)
    return fail(LORA_ERR_UNSUPPORTED,
                "the 4-bit variant needs d_in a positive multiple of 64 and d_out of 8 "
                "(got %lld, %lld)", (long long)d_in, (long long)d_out);
  if (d_in > INT32_MAX / 2 || d_out > INT32_MAX / 2)
    return fail(LORA_ERR_UNSUPPORTED, "a dimension exceeds 2^30");
  return LORA_OK;
}

lora_status_t lora_q4_quantize_w(const void *W, int64_t d_out, int64_t d_in, void *codes,
                                 void *scales, void *stream) {
  t_err.clear();
  LORA_TRY(check_q4_dims(d_in, d_out));
  LORA_TRY(check_ptr(W, "W"));
  LORA_TRY(check_ptr(codes, "codes"));
  LORA_TRY(check_ptr(scales, "scales"));
  DevInfo di;
  LORA_TRY(device_info(di));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return run(LORA_K_QUANT, st, "quantise W to 4 bits", [&] {
    return launch_quant_q4(W, static_cast<int>(d_out), static_cast<int>(d_in), codes, scales, st);
  });
}

lora_status_t lora_q4_dequantize_w(const void *codes, const void *scales, int64_t d_out,
                                   int64_t d_in, void *Wd, void *stream) {
  t_err.clear();
  LORA_TRY(check_q4_dims(d_in, d_out));
  LORA_TRY(check_ptr(codes, "codes"));
  LORA_TRY(check_ptr(scales, "scales"));
  LORA_TRY(check_ptr(Wd, "Wd"));
  DevInfo di;
  LORA_TRY(device_info(di));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return run(LORA_K_QUANT, st, "dequantise 4-bit W", [&] {
    return launch_dequant_q4(codes, scales, static_cast<int>(d_out), static_cast<int>(d_in), Wd,
                             di.sms, st);
  });
}

lora_status_t lora_q4_fwd(const void *X, const void *codes, const void *scales, const void *A,
                          const void *B, float alpha, int r, int64_t M, int64_t d_in,
                          int64_t d_out, void *Y, void *saved, void *workspace,
                          size_t workspace_bytes, void *stream) {
  t_err.clear();
  LORA_TRY(check_shape(r, M, d_in, d_out, LORA_BF16, alpha));
  LORA_TRY(check_q4_dims(d_in, d_out));
  const bool empty = M == 0;
  LORA_TRY(check_ptr(X, "X", empty));
  LORA_TRY(check_ptr(codes, "codes"));
  LORA_TRY(check_ptr(scales, "scales"));
  LORA_TRY(check_ptr(A, "A"));
  LORA_TRY(check_ptr(B, "B"));
  LORA_TRY(check_ptr(Y, "Y", empty));
  LORA_TRY(check_ptr(saved, "saved", empty));
  const Plan P = make_plan(M, d_in, d_out, r, LORA_BF16);
  LORA_TRY(check_ws(workspace, workspace_bytes, P.fwd_ws_min));
  if (empty) return LORA_OK;
  Q4W q4;
  q4.codes = codes;
  q4.scales = scales;
  return fwd_bf16(X, nullptr, A, B, alpha, r, M, d_in, d_out, Y, saved, workspace,
                  workspace_bytes, static_cast<cudaStream_t>(stream), &q4);
}

lora_status_t lora_q4_bwd(const void *dY, const void *X, const void *codes, const void *scales,
                          const void *A, const void *B, const void *saved, float alpha, int r,
                          int64_t M, int64_t d_in, int64_t d_out, void *dX, void *dA, void *dB,
                          void *workspace, size_t workspace_bytes, void *stream) {
  t_err.clear();
  LORA_TRY(check_shape(r, M, d_in, d_out, LORA_BF16, alpha));
  LORA_TRY(check_q4_dims(d_in, d_out));
  const bool empty = M == 0;
  LORA_TRY(check_ptr(dY, "dY", empty));
  LORA_TRY(check_ptr(X, "X", empty));
  LORA_TRY(check_ptr(codes, "codes"));
  LORA_TRY(check_ptr(scales, "scales"));
  LORA_TRY(check_ptr(A, "A"));
  LORA_TRY(check_ptr(B, "B"));
  LORA_TRY(check_ptr(saved, "saved", true));
  LORA_TRY(check_ptr(dX, "dX", true));
  LORA_TRY(check_ptr(dA, "dA"));
  LORA_TRY(check_ptr(dB, "dB"));
  const Plan P = make_plan(M, d_in, d_out, r, LORA_BF16);
  size_t need = saved != nullptr ? P.bwd_ws_min : P.bwd_ws;
  if (empty) need = 0;
  LORA_TRY(check_ws(workspace, workspace_bytes, need));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (empty) {  // sums over zero tokens
    cudaError_t e = cudaMemsetAsync(dA, 0, size_t(r) * d_in * 2, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(dB, 0, size_t(d_out) * r * 2, st);
    if (e != cudaSuccess) return fail(LORA_ERR_CUDA, "zero dA/dB: %s", cudaGetErrorString(e));
    return LORA_OK;
  }
  Q4W q4;
  q4.codes = codes;
  q4.scales = scales;
  return bwd_bf16(dY, X, nullptr, A, B, saved, alpha, r, M, d_in, d_out, dX, dA, dB, workspace,
                  workspace_bytes, st, &q4);
}

lora_status_t lora_debug_gemm_width(int width) {
  t_err.clear();
  if (width != 0 && width != 256 && width != 512)
    return fail(LORA_ERR_INVALID_ARG, "width %d is not 0, 256 or 512", width);
  main_gemm_force_width(width);
  return LORA_OK;
}

lora_status_t lora_debug_withhold_gemm_stage(int n) {
  t_err.clear();
  if (n < 0) return fail(LORA_ERR_INVALID_ARG, "n = %d is negative", n);
  g_withhold_gemm.store(n);
  return LORA_OK;
}

lora_status_t lora_debug_withhold_arrive(int n) {
  t_err.clear();
  if (n < 0) return fail(LORA_ERR_INVALID_ARG, "n = %d is negative", n);
  g_withhold.store(n);
  return LORA_OK;
}

}  // extern "C"
