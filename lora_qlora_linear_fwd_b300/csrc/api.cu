// C ABI of the library (declared in include/lora_b300.h): argument checks,
// TMA descriptor encoding, workspace carving and kernel launches.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "kernels.h"
#include "lora_b300.h"

using namespace lora;

namespace lora {
static std::atomic<uint64_t> g_launches{0};
void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
}  // namespace lora

namespace {

// ------------------------------------------------------------- device info
struct DeviceInfo {
  int sms = 0;
  bool ok = false;
};

lora_status_t device_info(DeviceInfo *out) {
  static thread_local int cached_dev = -1;
  static thread_local DeviceInfo cached;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LORA_ERR_CUDA;
  if (dev != cached_dev) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return LORA_ERR_CUDA;
    cached.sms = sms;
    cached.ok = (major == 10 && minor == 3);
    cached_dev = dev;
  }
  if (!cached.ok) return LORA_ERR_ARCH;
  *out = cached;
  return LORA_OK;
}

// ------------------------------------------------------------ tensor maps
using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                              const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                              const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  });
  return fn;
}

CUtensorMapSwizzle swizzle_for(int inner_bytes) {
  switch (inner_bytes) {
    case 128: return CU_TENSOR_MAP_SWIZZLE_128B;
    case 64: return CU_TENSOR_MAP_SWIZZLE_64B;
    case 32: return CU_TENSOR_MAP_SWIZZLE_32B;
    default: return CU_TENSOR_MAP_SWIZZLE_NONE;
  }
}

// 2-D map over a row-major matrix [outer, inner] with row pitch `pitch_bytes`.
bool make_map(CUtensorMap *m, CUtensorMapDataType dt, int esize, const void *ptr, uint64_t inner,
              uint64_t outer, uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_outer,
              bool swizzle) {
  EncodeFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {pitch_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapSwizzle sw =
      swizzle ? swizzle_for((int)(box_inner * esize)) : CU_TENSOR_MAP_SWIZZLE_NONE;
  return fn(m, dt, 2, const_cast<void *>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr CUtensorMapDataType kBF16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
constexpr CUtensorMapDataType kU8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;

// ---------------------------------------------------------------- checks
bool aligned16(const void *p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// Rank padded to a tensor-core N: 16/32/64 (and 128 for two merged rank-64
// projections).  The pair MMA needs N a multiple of 32.
int rank_pad(int r) { return r <= 16 ? 16 : (r <= 32 ? 32 : (r <= 64 ? 64 : 128)); }
int rank_pad_pair(int r) { return r <= 32 ? 32 : (r <= 64 ? 64 : 128); }
// GEMM variant: the two-SM kernel unless LORA_GEMM_VARIANT=1 selects the
// one-SM kernel (kept for comparison and testing).
bool use_pair_kernel() {
  static const bool pair = [] {
    const char *v = std::getenv("LORA_GEMM_VARIANT");
    return !(v && v[0] == '1');
  }();
  return pair;
}
bool rank_ok(int r) { return r == 8 || r == 16 || r == 32 || r == 64; }
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
constexpr int kBN = 256;

lora_status_t check_weight(const lora_weight_t &W, int n, int k) {
  if (W.type == LORA_WEIGHT_BF16) {
    if (!aligned16(W.w)) return LORA_ERR_INVALID_ARG;
  } else if (W.type == LORA_WEIGHT_NF4) {
    if (!aligned16(W.w) || !W.absmax || (reinterpret_cast<uintptr_t>(W.absmax) & 1u))
      return LORA_ERR_INVALID_ARG;
    if (W.blocksize != 64) return LORA_ERR_UNSUPPORTED;
  } else {
    return LORA_ERR_INVALID_ARG;
  }
  (void)n;
  (void)k;
  return LORA_OK;
}

lora_status_t check_shape(int M, int k, int n, int r) {
  if (M < 1 || k < 1 || n < 1 || M > (1 << 30) || k > (1 << 20) || n > (1 << 20))
    return LORA_ERR_INVALID_ARG;
  if (k % 64 || n % 64) return LORA_ERR_UNSUPPORTED;
  if (!rank_ok(r)) return LORA_ERR_UNSUPPORTED;
  return LORA_OK;
}

// ------------------------------------------------------------- schedule
// Static schedule for `slots` persistent workers over m_blocks x n_tiles
// tiles.  Cost model in tile times: each tile costs 1, forming the rank
// accumulator costs rank_cost more.  The grid schedule's makespan is
// ceil(Mb/gm)*ceil(Nt/gn) tiles; the contiguous one's is ceil(T/W) plus at
// most two rank formations, but it keeps the whole problem in flight, so it
// is used only when the streamed operands fit comfortably in L2.
Schedule pick_schedule(int m_blocks, int n_tiles, int slots, double rank_cost,
                       double operand_bytes) {
  Schedule best{1, 1, m_blocks, n_tiles, 0, 1};
  double best_cost = 1e300;
  for (int gm = 1; gm <= std::min(m_blocks, slots); ++gm) {
    const int gn = std::min(n_tiles, slots / gm);
    if (gn < 1) break;
    const int per_m = (m_blocks + gm - 1) / gm;
    const int per_n = (n_tiles + gn - 1) / gn;
    const double cost = (double)per_m * per_n + per_m * rank_cost;
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = Schedule{gm, gn, m_blocks, n_tiles, 0, gm * gn};
    }
  }
  const long long total = (long long)m_blocks * n_tiles;
  const int workers = (int)std::min<long long>(slots, total);
  const double per = (double)((total + workers - 1) / workers);
  const double cont_cost = per + std::min(2.0, 1.0 + per / n_tiles) * rank_cost;
  constexpr double kL2Comfortable = 96.0 * (1 << 20);
  // LORA_SCHEDULE=grid|contiguous overrides the choice (for measurements).
  static const int forced = [] {
    const char *v = std::getenv("LORA_SCHEDULE");
    if (!v) return -1;
    return v[0] == 'g' ? 0 : (v[0] == 'c' ? 1 : -1);
  }();
  const bool contiguous = forced >= 0 ? forced == 1
                                      : (operand_bytes <= kL2Comfortable &&
                                         cont_cost < best_cost - 0.5);
  if (contiguous) best = Schedule{1, 1, m_blocks, n_tiles, 1, workers};
  return best;
}

// --------------------------------------------------------- workspace plan
struct BwdPlan {
  int rp, Mp;
  int v_grid, v_max_segs;
  int g_grid, g_max_segs;
  size_t off_bt, off_ut_hi, off_ut_lo, off_vt_hi, off_vt_lo, off_part_v, off_part_a,
      off_part_b, off_counters, counters_bytes, total;
};

// Persistent skinny launch over `items` work items: the grid, and the most
// CTAs whose contiguous item ranges can touch one row tile of `chunks` items.
int stream_grid(long long items) {
  return (int)std::max<long long>(1, std::min<long long>(kSkinnyCtas, items));
}
int max_segs_for(int chunks, long long items, int grid) {
  const long long per = std::max<long long>(1, items / grid);
  return (int)((chunks + per - 1) / per + 1);
}

BwdPlan plan_bwd(int M, int k, int n, int r, size_t start) {
  BwdPlan b{};
  b.rp = rank_pad(r);
  b.Mp = (M + 63) & ~63;
  const int mt = (M + 127) / 128, kt = (k + 127) / 128, nt = (n + 127) / 128;
  const int v_chunks = k / 64, g_chunks = (M + 63) / 64;
  const long long v_items = (long long)mt * v_chunks;
  const long long g_items = (long long)(kt + nt) * g_chunks;
  b.v_grid = stream_grid(v_items);
  b.g_grid = stream_grid(g_items);
  b.v_max_segs = max_segs_for(v_chunks, v_items, b.v_grid);
  b.g_max_segs = max_segs_for(g_chunks, g_items, b.g_grid);
  size_t o = align256(start);
  const int ut_rows = std::max(b.rp, rank_pad_pair(r));  // rows the dX kernel may write
  b.off_bt = o;       o = align256(o + (size_t)r * n * 2);
  b.off_ut_hi = o;    o = align256(o + (size_t)ut_rows * b.Mp * 2);
  b.off_ut_lo = o;    o = align256(o + (size_t)ut_rows * b.Mp * 2);
  b.off_vt_hi = o;    o = align256(o + (size_t)b.rp * b.Mp * 2);
  b.off_vt_lo = o;    o = align256(o + (size_t)b.rp * b.Mp * 2);
  b.off_part_v = o;   o = align256(o + (size_t)mt * b.v_max_segs * 128 * b.rp * 4);
  b.off_part_a = o;   o = align256(o + (size_t)kt * b.g_max_segs * 128 * b.rp * 4);
  b.off_part_b = o;   o = align256(o + (size_t)nt * b.g_max_segs * 128 * b.rp * 4);
  b.off_counters = o;
  b.counters_bytes = (size_t)(mt + kt + nt) * 4;
  o = align256(o + b.counters_bytes);
  b.total = o;
  return b;
}

constexpr size_t kStatusBytes = 256;

lora_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? LORA_OK : LORA_ERR_CUDA; }

// ------------------------------------------------------ fused GEMM set-up
struct GroupArgs {
  lora_weight_t W;
  const void *r1;  // FWD: A [r,k]; DX: Bᵀ [r,n]
  const void *r2;  // FWD: B [n,r]; DX: A [r,k]
  void *out;
  int ncols;       // output columns
};

struct GemmOpts {
  int mode = kModeFwd;
  const void *act = nullptr;  // FWD: x [M, k]; DX: dY [M, n]
  int M = 0, Kred = 0;        // rows; reduction length (k in FWD, n in DX)
  const GroupArgs *ga = nullptr;
  int ng = 1;                 // projections along N (FWD)
  // DX: a second projection along the reduction: its W holds rows
  // [ksplit*64, Kred) of the combined reduction
  const lora_weight_t *W2 = nullptr;
  int ksplit = 0;
  int r_layout = 0;           // rank of the rank-r operands (r, or 2r merged)
  float scale = 0.0f;         // alpha / r of one projection
  bool merged_rank = false;
  bool rope = false;
  const int32_t *positions = nullptr;
  const float *cos_sin = nullptr;
  int max_pos = 0;
  void *ut_hi = nullptr, *ut_lo = nullptr;
  int accumulate = 0;
  bool need_pair = false;     // merged shapes exist only in the pair kernel
  uint32_t *status = nullptr;
};

bool make_w_map(CUtensorMap *m, const lora_weight_t &W, bool dx, bool nf4, int n, int k,
                uint32_t wrows) {
  if (!dx) {
    if (nf4) return make_map(m, kU8, 1, W.w, k / 2, n, (uint64_t)k / 2, 32, wrows, false);
    return make_map(m, kBF16, 2, W.w, k, n, (uint64_t)k * 2, 64, wrows, true);
  }
  if (nf4) return make_map(m, kU8, 1, W.w, k / 2, n, (uint64_t)k / 2, wrows / 2, 64, false);
  return make_map(m, kBF16, 2, W.w, k, n, (uint64_t)k * 2, 64, 64, true);
}

lora_status_t run_gemm(const GemmOpts &o, cudaStream_t st) {
  DeviceInfo di;
  lora_status_t s = device_info(&di);
  if (s != LORA_OK) return s;
  const bool pair = o.need_pair || use_pair_kernel();
  const int r = o.r_layout;
  const int rp = pair ? rank_pad_pair(r) : rank_pad(r);
  if (!pair && rp > 64) return LORA_ERR_UNSUPPORTED;
  const bool nf4 = o.ga[0].W.type == LORA_WEIGHT_NF4;
  const bool dx = o.mode == kModeDx;
  const uint32_t wrows = pair ? kBN / 2 : kBN;   // W / B rows staged per CTA
  const uint32_t r1rows = pair ? rp / 2 : rp;    // rank-operand rows per CTA
  const uint32_t r2cols = rp > 64 ? 64 : rp;     // FWD B tile: column block width
  GemmParams p;
  std::memset(&p, 0, sizeof(p));
  // activation: [M, Kred] K-major, box 64 x 128
  if (!make_map(&p.tm_act, kBF16, 2, o.act, o.Kred, o.M, (uint64_t)o.Kred * 2, 64, 128, true))
    return LORA_ERR_CUDA;
  int tiles = 0;
  for (int g = 0; g < o.ng; ++g) {
    GemmGroup &G = p.grp[g];
    const GroupArgs &a = o.ga[g];
    const int ncols = a.ncols;
    if (!dx) {
      const int n = ncols, k = o.Kred;
      if (!make_w_map(&G.tm_w, a.W, false, nf4, n, k, wrows) ||
          !make_map(&G.tm_r1, kBF16, 2, a.r1, k, r, (uint64_t)k * 2, 64, r1rows, true) ||
          !make_map(&G.tm_r2, kBF16, 2, a.r2, r, n, (uint64_t)r * 2, r2cols, wrows, true))
        return LORA_ERR_CUDA;
      G.ld_absmax = k / 64;
    } else {
      const int n = o.W2 ? o.ksplit * 64 : o.Kred, k = ncols;
      if (!make_w_map(&G.tm_w, a.W, true, nf4, n, k, wrows) ||
          !make_map(&G.tm_r1, kBF16, 2, a.r1, o.Kred, r, (uint64_t)o.Kred * 2, 64, r1rows,
                    true) ||
          !make_map(&G.tm_r2, kBF16, 2, a.r2, k, r, (uint64_t)k * 2, 64, rp, true))
        return LORA_ERR_CUDA;
      G.ld_absmax = k / 64;
    }
    G.out = static_cast<__nv_bfloat16 *>(a.out);
    G.absmax = static_cast<const __nv_bfloat16 *>(a.W.absmax);
    G.ncols = ncols;
    G.n_tiles = (ncols + kBN - 1) / kBN;
    G.tile_begin = tiles;
    tiles += G.n_tiles;
  }
  p.num_groups = o.ng;
  if (dx && o.W2) {  // second projection along the reduction
    GemmGroup &G1 = p.grp[1];
    const int k = o.ga[0].ncols, n2 = o.Kred - o.ksplit * 64;
    if (!make_w_map(&G1.tm_w, *o.W2, true, nf4, n2, k, wrows)) return LORA_ERR_CUDA;
    G1.absmax = static_cast<const __nv_bfloat16 *>(o.W2->absmax);
    G1.ld_absmax = k / 64;
    G1.ncols = k;
    p.kgroups = 2;
    p.ksplit = o.ksplit;
  } else {
    p.kgroups = 1;
  }
  p.merged_rank = o.merged_rank ? 1 : 0;
  p.M = o.M;
  p.K = o.Kred;
  p.scale = o.scale;
  int slots = di.sms;
  if (pair) {
    slots = gemm_pair_capacity(o.mode, rp, o.rope, nf4);
    if (slots < 1) return LORA_ERR_CUDA;
  }
  const int m_blocks = pair ? (o.M + 255) / 256 : (o.M + 127) / 128;
  double operand_bytes = (double)o.M * o.Kred * 2;   // activation
  for (int g = 0; g < o.ng; ++g)                        // weights
    operand_bytes += (double)o.ga[g].ncols * o.Kred * (nf4 ? 0.5 + 1.0 / 32 : 2.0);
  p.sched = pick_schedule(m_blocks, tiles, slots, (double)rp / kBN + 0.02, operand_bytes);
  p.ut_hi = static_cast<__nv_bfloat16 *>(o.ut_hi);
  p.ut_lo = static_cast<__nv_bfloat16 *>(o.ut_lo);
  p.accumulate = o.accumulate;
  p.positions = o.positions;
  p.cos_sin = o.cos_sin;
  p.max_pos = o.max_pos;
  p.status = o.status;
  const int grid = p.sched.workers;
  if (pair) return cuda_status(launch_gemm_pair(p, o.mode, rp, o.rope, nf4, grid, st));
  return cuda_status(launch_gemm(p, o.mode, rp, o.rope, nf4, grid, st));
}

// ------------------------------------------------------ backward phases
// The backward of one projection -- or of two projections sharing x, taken
// as one projection of rank 2r with A = [A1; A2] and B = diag(B1, B2) --
// split into phases that the caller orders on two streams:
//   v      v = x·Aᵀ recomputed -> vᵀ hi/lo   (needs x, A only)
//   dx     dX (+)= dY·W + s·(dY·B)·A, exports uᵀ = (dY·B)ᵀ hi/lo
//   grads  dA = s·uᵀ·x, dB = s·dYᵀ·v        (needs v and dx done)
struct BwdCall {
  const void *x, *A, *Bt, *dy;   // A [rl, k]; Bᵀ [rl, n] (prepared); dY [M, n]
  lora_weight_t W;               // W [n1, k] (the whole n unless merged)
  lora_weight_t W2;              // merged: W of projection 2, [n - n1, k]
  bool merged;
  void *dx;
  int accumulate;
  float *dA, *dB, *dA2, *dB2;    // per projection
  int M, k, n, n1;               // n: total reduction of dX; n1: rows of projection 1
  int r;                         // rank of one projection
  int rl;                        // layout rank (r, or 2r merged)
  float scale;
  uint32_t *status;
  BwdPlan b;
  uint8_t *ws;
  template <typename T>
  T *at(size_t off) const { return reinterpret_cast<T *>(ws + off); }
};

lora_status_t bwd_v(const BwdCall &c, cudaStream_t st) {
  const BwdPlan &b = c.b;
  SkinnyParams sp;
  std::memset(&sp, 0, sizeof(sp));
  SkinnyProblem &P = sp.pr[0];
  if (!make_map(&P.tm_p, kBF16, 2, c.x, c.k, c.M, (uint64_t)c.k * 2, 64, 128, true) ||
      !make_map(&P.tm_q_hi, kBF16, 2, c.A, c.k, c.rl, (uint64_t)c.k * 2, 64, b.rp, true))
    return LORA_ERR_CUDA;
  P.tm_q_lo = P.tm_q_hi;
  P.part = c.at<float>(b.off_part_v);
  P.counter = c.at<uint32_t>(b.off_counters);
  P.out_kind = kOutVt;
  P.out_hi = c.at<__nv_bfloat16>(b.off_vt_hi);
  P.out_lo = c.at<__nv_bfloat16>(b.off_vt_lo);
  P.out_ld = b.Mp;
  P.r = c.rl;
  P.nproj = 1;
  P.scale = 1.0f;
  P.rows = c.M;
  P.row_tiles = (c.M + 127) / 128;
  P.chunks = c.k / 64;
  P.max_segs = b.v_max_segs;
  sp.num_problems = 1;
  sp.total_items = (long long)P.row_tiles * P.chunks;
  sp.status = c.status;
  return cuda_status(launch_skinny(sp, false, b.rp, b.v_grid, st));
}

lora_status_t bwd_dx(const BwdCall &c, cudaStream_t st) {
  GroupArgs ga{c.W, c.Bt, c.A, c.dx, c.k};
  GemmOpts o;
  o.mode = kModeDx;
  o.act = c.dy;
  o.M = c.M;
  o.Kred = c.n;
  o.ga = &ga;
  o.ng = 1;
  if (c.merged) {
    o.W2 = &c.W2;
    o.ksplit = c.n1 / 64;
    o.merged_rank = true;
    o.need_pair = true;
  }
  o.r_layout = c.rl;
  o.scale = c.scale;
  o.ut_hi = c.at<__nv_bfloat16>(c.b.off_ut_hi);
  o.ut_lo = c.at<__nv_bfloat16>(c.b.off_ut_lo);
  o.accumulate = c.accumulate;
  o.status = c.status;
  return run_gemm(o, st);
}

lora_status_t bwd_grads(const BwdCall &c, cudaStream_t st) {
  const BwdPlan &b = c.b;
  const int M = c.M, k = c.k, n = c.n;
  SkinnyParams sp;
  std::memset(&sp, 0, sizeof(sp));
  SkinnyProblem &PA = sp.pr[0];
  SkinnyProblem &PB = sp.pr[1];
  if (!make_map(&PA.tm_p, kBF16, 2, c.x, k, M, (uint64_t)k * 2, 64, 64, true) ||
      !make_map(&PA.tm_q_hi, kBF16, 2, c.at<void>(b.off_ut_hi), M, b.rp, (uint64_t)b.Mp * 2, 64,
                b.rp, true) ||
      !make_map(&PA.tm_q_lo, kBF16, 2, c.at<void>(b.off_ut_lo), M, b.rp, (uint64_t)b.Mp * 2, 64,
                b.rp, true) ||
      !make_map(&PB.tm_p, kBF16, 2, c.dy, n, M, (uint64_t)n * 2, 64, 64, true) ||
      !make_map(&PB.tm_q_hi, kBF16, 2, c.at<void>(b.off_vt_hi), M, b.rp, (uint64_t)b.Mp * 2, 64,
                b.rp, true) ||
      !make_map(&PB.tm_q_lo, kBF16, 2, c.at<void>(b.off_vt_lo), M, b.rp, (uint64_t)b.Mp * 2, 64,
                b.rp, true))
    return LORA_ERR_CUDA;
  const int mt = (M + 127) / 128;
  uint32_t *counters = c.at<uint32_t>(b.off_counters);
  const int nproj = c.merged ? 2 : 1;
  PA.part = c.at<float>(b.off_part_a);
  PA.counter = counters + mt;
  PA.out_kind = kOutRowT;
  PA.out_f32 = c.dA;
  PA.out_f32b = c.dA2;
  PA.r = c.r;
  PA.nproj = nproj;
  PA.scale = c.scale;
  PA.rows = k;
  PA.row_tiles = (k + 127) / 128;
  PA.chunks = (M + 63) / 64;
  PA.max_segs = b.g_max_segs;
  PB.part = c.at<float>(b.off_part_b);
  PB.counter = counters + mt + PA.row_tiles;
  PB.out_kind = kOutRow;
  PB.out_f32 = c.dB;
  PB.out_f32b = c.dB2;
  PB.r = c.r;
  PB.nproj = nproj;
  PB.split_row = c.n1;
  PB.scale = c.scale;
  PB.rows = n;
  PB.row_tiles = (n + 127) / 128;
  PB.chunks = (M + 63) / 64;
  PB.max_segs = b.g_max_segs;
  sp.num_problems = 2;
  sp.total_items = (long long)(PA.row_tiles + PB.row_tiles) * PA.chunks;
  sp.status = c.status;
  return cuda_status(launch_skinny(sp, true, b.rp, b.g_grid, st));
}

// A helper stream (and events to order it against the caller's stream),
// created once per calling thread and device; the recomputation of
// v = x·Aᵀ runs on it while the dX GEMM runs on the caller's stream.
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t ev[2] = {nullptr, nullptr};
};

lora_status_t side_stream(SideStream **out) {
  constexpr int kMaxDev = 64;
  static thread_local SideStream per_dev[kMaxDev];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return LORA_ERR_CUDA;
  SideStream &ss = per_dev[dev];
  if (!ss.s) {
    if (cudaStreamCreateWithFlags(&ss.s, cudaStreamNonBlocking) != cudaSuccess)
      return LORA_ERR_CUDA;
    for (auto &e : ss.ev)
      if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess)
        return LORA_ERR_CUDA;
  }
  *out = &ss;
  return LORA_OK;
}

// `to` waits for everything issued on `from` so far (event `e`).
lora_status_t order_after(cudaStream_t to, cudaStream_t from, cudaEvent_t e) {
  if (cudaEventRecord(e, from) != cudaSuccess) return LORA_ERR_CUDA;
  return cuda_status(cudaStreamWaitEvent(to, e, 0));
}

// Run the phases: the x stream for v beside the dX GEMM, then dA/dB.
// Counters and Bᵀ must already be prepared on `st`.
lora_status_t run_bwd_phases(const BwdCall &c, cudaStream_t st) {
  SideStream *side = nullptr;
  lora_status_t s;
  if ((s = side_stream(&side))) return s;
  if ((s = order_after(side->s, st, side->ev[0]))) return s;   // fork
  if ((s = bwd_v(c, side->s))) return s;
  if ((s = bwd_dx(c, st))) return s;
  if ((s = order_after(st, side->s, side->ev[1]))) return s;   // join
  return bwd_grads(c, st);
}

size_t bwd_bytes(int M, int k, int n, int r) { return plan_bwd(M, k, n, r, 0).total; }

// q/k as one projection of rank 2r: A_qk = [Aq; Ak] [2r, hidden],
// B_qk = diag(Bq, Bk) [nq+nk, 2r] (forward) or its transpose (backward).
// Forward workspace: status | A_qk | B_qk.
struct QkFwdPlan {
  size_t off_a, off_b, total;
};
QkFwdPlan plan_qk_fwd(int k, int n, int r) {
  QkFwdPlan q{};
  size_t o = kStatusBytes;
  q.off_a = o;  o = align256(o + (size_t)2 * r * k * 2);
  q.off_b = o;  o = align256(o + (size_t)n * 2 * r * 2);
  q.total = o;
  return q;
}
// Backward workspace: status | rotated dY_qk [M, nq+nk] | A_qk | the
// rank-2r backward area (whose Bᵀ slot holds diag(Bq, Bk)ᵀ).
struct QkBwdPlan {
  size_t off_dy, off_a, off_area, total;
};
QkBwdPlan plan_qk_bwd(int M, int k, int n, int r) {
  QkBwdPlan q{};
  size_t o = kStatusBytes;
  q.off_dy = o;   o = align256(o + (size_t)M * n * 2);
  q.off_a = o;    o = align256(o + (size_t)2 * r * k * 2);
  q.off_area = o; o += bwd_bytes(M, k, n, 2 * r);
  q.total = o;
  return q;
}

lora_status_t build_a_qk(const void *Aq, const void *Ak, void *A_qk, int r, int k,
                         cudaStream_t st) {
  const size_t bytes = (size_t)r * k * 2;
  lora_status_t s;
  if ((s = cuda_status(cudaMemcpyAsync(A_qk, Aq, bytes, cudaMemcpyDeviceToDevice, st)))) return s;
  return cuda_status(cudaMemcpyAsync(static_cast<uint8_t *>(A_qk) + bytes, Ak, bytes,
                                     cudaMemcpyDeviceToDevice, st));
}

}  // namespace

// =================================================================== C ABI
extern "C" {

uint64_t lora_kernel_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char *lora_status_string(lora_status_t s) {
  switch (s) {
    case LORA_OK: return "LORA_OK";
    case LORA_ERR_INVALID_ARG: return "LORA_ERR_INVALID_ARG";
    case LORA_ERR_UNSUPPORTED: return "LORA_ERR_UNSUPPORTED";
    case LORA_ERR_WORKSPACE: return "LORA_ERR_WORKSPACE";
    case LORA_ERR_ARCH: return "LORA_ERR_ARCH";
    case LORA_ERR_CUDA: return "LORA_ERR_CUDA";
    case LORA_ERR_TIMEOUT: return "LORA_ERR_TIMEOUT";
  }
  return "LORA_ERR_UNKNOWN";
}

size_t lora_workspace_size(int op, int M, int k, int n, int r) {
  if (M < 1 || k < 1 || n < 1 || !rank_ok(r) || M > (1 << 30)) return 0;
  switch (op) {
    case LORA_OP_FWD:
      return kStatusBytes;
    case LORA_OP_BWD:
      return kStatusBytes + bwd_bytes(M, k, n, r);
    case LORA_OP_QK_ROPE_FWD:
      return plan_qk_fwd(k, n, r).total;
    case LORA_OP_QK_ROPE_BWD:
      return plan_qk_bwd(M, k, n, r).total;
  }
  return 0;
}

size_t lora_rope_cache_bytes(int max_pos, int head_dim) {
  if (max_pos < 1 || head_dim < 2) return 0;
  return align256((size_t)max_pos * head_dim * 4);
}

lora_status_t lora_linear_fwd(const void *x, lora_weight_t W, const void *A, const void *B,
                              void *y, int M, int k, int n, int r, float alpha, void *ws,
                              size_t ws_bytes, lora_stream_t stream) {
  lora_status_t s;
  if ((s = check_shape(M, k, n, r))) return s;
  if ((s = check_weight(W, n, k))) return s;
  if (!aligned16(x) || !aligned16(A) || !aligned16(B) || !aligned16(y) || !aligned16(ws))
    return LORA_ERR_INVALID_ARG;
  if (!std::isfinite(alpha)) return LORA_ERR_INVALID_ARG;
  if (ws_bytes < lora_workspace_size(LORA_OP_FWD, M, k, n, r)) return LORA_ERR_WORKSPACE;
  GroupArgs ga{W, A, B, y, n};
  GemmOpts o;
  o.mode = kModeFwd;
  o.act = x;
  o.M = M;
  o.Kred = k;
  o.ga = &ga;
  o.ng = 1;
  o.r_layout = r;
  o.scale = alpha / (float)r;
  o.status = static_cast<uint32_t *>(ws);
  return run_gemm(o, reinterpret_cast<cudaStream_t>(stream));
}

lora_status_t lora_linear_bwd(const void *x, lora_weight_t W, const void *A, const void *B,
                              const void *dy, void *dx, int accumulate_dx, float *dA, float *dB,
                              int M, int k, int n, int r, float alpha, void *ws, size_t ws_bytes,
                              lora_stream_t stream) {
  lora_status_t s;
  if ((s = check_shape(M, k, n, r))) return s;
  if ((s = check_weight(W, n, k))) return s;
  if (!aligned16(x) || !aligned16(A) || !aligned16(B) || !aligned16(dy) || !aligned16(dx) ||
      !aligned16(dA) || !aligned16(dB) || !aligned16(ws))
    return LORA_ERR_INVALID_ARG;
  if (!std::isfinite(alpha)) return LORA_ERR_INVALID_ARG;
  if (ws_bytes < lora_workspace_size(LORA_OP_BWD, M, k, n, r)) return LORA_ERR_WORKSPACE;
  DeviceInfo di;
  if ((s = device_info(&di))) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t *w8 = static_cast<uint8_t *>(ws);
  BwdCall c{};
  c.x = x;
  c.A = A;
  c.dy = dy;
  c.W = W;
  c.merged = false;
  c.dx = dx;
  c.accumulate = accumulate_dx;
  c.dA = dA;
  c.dB = dB;
  c.M = M;
  c.k = k;
  c.n = n;
  c.n1 = n;
  c.r = r;
  c.rl = r;
  c.scale = alpha / (float)r;
  c.status = static_cast<uint32_t *>(ws);
  c.b = plan_bwd(M, k, n, r, kStatusBytes);
  c.ws = w8;
  c.Bt = c.at<void>(c.b.off_bt);
  if ((s = cuda_status(cudaMemsetAsync(c.at<uint32_t>(c.b.off_counters), 0, c.b.counters_bytes,
                                       st))))
    return s;
  if ((s = cuda_status(launch_transpose_rank(static_cast<const __nv_bfloat16 *>(B),
                                             c.at<__nv_bfloat16>(c.b.off_bt), n, r, st))))
    return s;
  return run_bwd_phases(c, st);
}

static lora_status_t check_qk(const void *x, lora_weight_t Wq, const void *Aq, const void *Bq,
                              lora_weight_t Wk, const void *Ak, const void *Bk, int M, int hidden,
                              int nqh, int nkh, int head_dim, int r, float alpha,
                              const int32_t *positions, const float *cache, int max_pos,
                              double theta, void *ws) {
  lora_status_t s;
  if (head_dim != 128) return LORA_ERR_UNSUPPORTED;
  if (nqh < 1 || nkh < 1 || nqh > 4096 || nkh > 4096 || max_pos < 1) return LORA_ERR_INVALID_ARG;
  if ((s = check_shape(M, hidden, nqh * head_dim, r))) return s;
  if ((s = check_weight(Wq, nqh * head_dim, hidden))) return s;
  if ((s = check_weight(Wk, nkh * head_dim, hidden))) return s;
  if (Wq.type != Wk.type) return LORA_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(Aq) || !aligned16(Bq) || !aligned16(Ak) || !aligned16(Bk) ||
      !aligned16(ws) || !positions || (reinterpret_cast<uintptr_t>(positions) & 3u))
    return LORA_ERR_INVALID_ARG;
  if (cache && !aligned16(cache)) return LORA_ERR_INVALID_ARG;
  if (!cache && !(theta > 0.0 && std::isfinite(theta))) return LORA_ERR_INVALID_ARG;
  if (!std::isfinite(alpha)) return LORA_ERR_INVALID_ARG;
  return LORA_OK;
}

lora_status_t lora_qk_rope_fwd(const void *x, lora_weight_t Wq, const void *Aq, const void *Bq,
                               lora_weight_t Wk, const void *Ak, const void *Bk, void *q,
                               void *k_out, int M, int hidden, int n_q_heads, int n_kv_heads,
                               int head_dim, int r, float alpha, double rope_theta,
                               const int32_t *positions, const float *cos_sin_cache, int max_pos,
                               void *ws, size_t ws_bytes, lora_stream_t stream) {
  lora_status_t s;
  if ((s = check_qk(x, Wq, Aq, Bq, Wk, Ak, Bk, M, hidden, n_q_heads, n_kv_heads, head_dim, r,
                    alpha, positions, cos_sin_cache, max_pos, rope_theta, ws)))
    return s;
  if (!aligned16(q) || !aligned16(k_out)) return LORA_ERR_INVALID_ARG;
  const int nq = n_q_heads * head_dim, nk = n_kv_heads * head_dim;
  size_t need = lora_workspace_size(LORA_OP_QK_ROPE_FWD, M, hidden, nq + nk, r);
  const size_t cache_off = align256(need);
  if (!cos_sin_cache) need = cache_off + lora_rope_cache_bytes(max_pos, head_dim);
  if (ws_bytes < need) return LORA_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  DeviceInfo di;
  if ((s = device_info(&di))) return s;
  const float *cache = cos_sin_cache;
  if (!cache) {
    float *c = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + cache_off);
    if ((s = cuda_status(launch_rope_cache(c, max_pos, head_dim, rope_theta, st)))) return s;
    cache = c;
  }
  // one projection of rank 2r over both weights: the rank accumulator
  // x·A_qkᵀ is formed once per row block and serves the q and k tiles
  const QkFwdPlan qp = plan_qk_fwd(hidden, nq + nk, r);
  uint8_t *w8 = static_cast<uint8_t *>(ws);
  auto *B_qk = reinterpret_cast<__nv_bfloat16 *>(w8 + qp.off_b);
  if ((s = build_a_qk(Aq, Ak, w8 + qp.off_a, r, hidden, st))) return s;
  if ((s = cuda_status(launch_blockdiag_rank(static_cast<const __nv_bfloat16 *>(Bq),
                                             static_cast<const __nv_bfloat16 *>(Bk), B_qk, nq,
                                             nk, r, false, st))))
    return s;
  GroupArgs ga[2] = {{Wq, w8 + qp.off_a, B_qk, q, nq},
                     {Wk, w8 + qp.off_a, B_qk + (size_t)nq * 2 * r, k_out, nk}};
  GemmOpts o;
  o.mode = kModeFwd;
  o.act = x;
  o.M = M;
  o.Kred = hidden;
  o.ga = ga;
  o.ng = 2;
  o.r_layout = 2 * r;
  o.scale = alpha / (float)r;
  o.merged_rank = true;
  o.need_pair = true;
  o.rope = true;
  o.positions = positions;
  o.cos_sin = cache;
  o.max_pos = max_pos;
  o.status = static_cast<uint32_t *>(ws);
  return run_gemm(o, st);
}

lora_status_t lora_qk_rope_bwd(const void *x, lora_weight_t Wq, const void *Aq, const void *Bq,
                               lora_weight_t Wk, const void *Ak, const void *Bk, const void *dq,
                               const void *dk, void *dx, int accumulate_dx, float *dAq,
                               float *dBq, float *dAk, float *dBk, int M, int hidden,
                               int n_q_heads, int n_kv_heads, int head_dim, int r, float alpha,
                               double rope_theta, const int32_t *positions,
                               const float *cos_sin_cache, int max_pos, void *ws,
                               size_t ws_bytes, lora_stream_t stream) {
  lora_status_t s;
  if ((s = check_qk(x, Wq, Aq, Bq, Wk, Ak, Bk, M, hidden, n_q_heads, n_kv_heads, head_dim, r,
                    alpha, positions, cos_sin_cache, max_pos, rope_theta, ws)))
    return s;
  if (!aligned16(dq) || !aligned16(dk) || !aligned16(dx) || !aligned16(dAq) || !aligned16(dBq) ||
      !aligned16(dAk) || !aligned16(dBk))
    return LORA_ERR_INVALID_ARG;
  const int nq = n_q_heads * head_dim, nk = n_kv_heads * head_dim;
  size_t need = lora_workspace_size(LORA_OP_QK_ROPE_BWD, M, hidden, nq + nk, r);
  const size_t cache_off = align256(need);
  if (!cos_sin_cache) need = cache_off + lora_rope_cache_bytes(max_pos, head_dim);
  if (ws_bytes < need) return LORA_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  DeviceInfo di;
  if ((s = device_info(&di))) return s;
  uint8_t *w8 = static_cast<uint8_t *>(ws);
  uint32_t *status = static_cast<uint32_t *>(ws);
  const float *cache = cos_sin_cache;
  if (!cache) {
    float *c = reinterpret_cast<float *>(w8 + cache_off);
    if ((s = cuda_status(launch_rope_cache(c, max_pos, head_dim, rope_theta, st)))) return s;
    cache = c;
  }
  // rotate dq, dk back (RoPE is orthogonal) into one [M, nq+nk] gradient
  const int n = nq + nk;
  const QkBwdPlan qp = plan_qk_bwd(M, hidden, n, r);
  auto *dy_qk = reinterpret_cast<__nv_bfloat16 *>(w8 + qp.off_dy);
  if ((s = cuda_status(launch_rope_bwd(static_cast<const __nv_bfloat16 *>(dq), dy_qk, M, nq, n,
                                       positions, cache, max_pos, status, st))))
    return s;
  if ((s = cuda_status(launch_rope_bwd(static_cast<const __nv_bfloat16 *>(dk), dy_qk + nq, M, nk,
                                       n, positions, cache, max_pos, status, st))))
    return s;
  // then the backward of one projection of rank 2r, W = [Wq; Wk] along the
  // reduction of dX, with dA/dB split back per projection
  BwdCall c{};
  c.x = x;
  c.A = w8 + qp.off_a;
  c.dy = dy_qk;
  c.W = Wq;
  c.W2 = Wk;
  c.merged = true;
  c.dx = dx;
  c.accumulate = accumulate_dx;
  c.dA = dAq;
  c.dB = dBq;
  c.dA2 = dAk;
  c.dB2 = dBk;
  c.M = M;
  c.k = hidden;
  c.n = n;
  c.n1 = nq;
  c.r = r;
  c.rl = 2 * r;
  c.scale = alpha / (float)r;
  c.status = status;
  c.b = plan_bwd(M, hidden, n, 2 * r, 0);
  c.ws = w8 + qp.off_area;
  c.Bt = c.at<void>(c.b.off_bt);
  if ((s = build_a_qk(Aq, Ak, w8 + qp.off_a, r, hidden, st))) return s;
  if ((s = cuda_status(launch_blockdiag_rank(static_cast<const __nv_bfloat16 *>(Bq),
                                             static_cast<const __nv_bfloat16 *>(Bk),
                                             c.at<__nv_bfloat16>(c.b.off_bt), nq, nk, r, true,
                                             st))))
    return s;
  if ((s = cuda_status(cudaMemsetAsync(c.at<uint32_t>(c.b.off_counters), 0, c.b.counters_bytes,
                                       st))))
    return s;
  return run_bwd_phases(c, st);
}

lora_status_t nf4_dequant(const uint8_t *codes, const void *absmax, void *w_out, int n, int k,
                          int blocksize, lora_stream_t stream) {
  if (blocksize != 64) return LORA_ERR_UNSUPPORTED;
  if (n < 1 || k < 1 || k % 64) return LORA_ERR_INVALID_ARG;
  if (!aligned16(codes) || !absmax || (reinterpret_cast<uintptr_t>(absmax) & 1u) ||
      !aligned16(w_out))
    return LORA_ERR_INVALID_ARG;
  DeviceInfo di;
  lora_status_t s;
  if ((s = device_info(&di))) return s;
  return cuda_status(launch_nf4_dequant(codes, static_cast<const __nv_bfloat16 *>(absmax),
                                        static_cast<__nv_bfloat16 *>(w_out), n, k,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

lora_status_t nf4_quantize(const void *w, uint8_t *codes, void *absmax, int n, int k,
                           int blocksize, lora_stream_t stream) {
  if (blocksize != 64) return LORA_ERR_UNSUPPORTED;
  if (n < 1 || k < 1 || k % 64) return LORA_ERR_INVALID_ARG;
  if (!aligned16(w) || !aligned16(codes) || !absmax ||
      (reinterpret_cast<uintptr_t>(absmax) & 1u))
    return LORA_ERR_INVALID_ARG;
  DeviceInfo di;
  lora_status_t s;
  if ((s = device_info(&di))) return s;
  return cuda_status(launch_nf4_quantize(static_cast<const __nv_bfloat16 *>(w), codes,
                                         static_cast<__nv_bfloat16 *>(absmax), n, k,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

lora_status_t lora_rope_cache_build(float *cos_sin, int max_pos, int head_dim, double theta,
                                    lora_stream_t stream) {
  if (!aligned16(cos_sin) || max_pos < 1 || head_dim < 2 || head_dim % 2 ||
      !(theta > 0.0 && std::isfinite(theta)))
    return LORA_ERR_INVALID_ARG;
  DeviceInfo di;
  lora_status_t s;
  if ((s = device_info(&di))) return s;
  return cuda_status(
      launch_rope_cache(cos_sin, max_pos, head_dim, theta, reinterpret_cast<cudaStream_t>(stream)));
}

lora_status_t lora_read_device_status(const void *ws, uint32_t *status_out, lora_stream_t stream) {
  if (!ws || !status_out) return LORA_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return LORA_ERR_CUDA;
  uint32_t v = 0;
  if (cudaMemcpy(&v, ws, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return LORA_ERR_CUDA;
  *status_out = v;
  return (v & kDevTimeout) ? LORA_ERR_TIMEOUT : LORA_OK;
}

lora_status_t lora_clear_device_status(void *ws, lora_stream_t stream) {
  if (!ws) return LORA_ERR_INVALID_ARG;
  return cuda_status(cudaMemsetAsync(ws, 0, sizeof(uint32_t), reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
