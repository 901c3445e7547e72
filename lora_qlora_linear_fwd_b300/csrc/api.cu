// C ABI of the library (declared in include/lora_b300.h): argument checks,
// TMA descriptor encoding, workspace carving and kernel launches.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <random>
#include <vector>

#include "kernels.h"
#include "lora_b300.h"

using namespace lora;

namespace lora {
static std::atomic<uint64_t> g_launches{0};

namespace {
// Per-launch timing session (lora_profile_begin / lora_profile_end): event
// pairs created up front, consumed one pair per launch in launch order.
struct ProfileSession {
  std::mutex mu;
  std::atomic<bool> open{false};
  std::vector<cudaEvent_t> before, after;
  std::vector<const char *> names;
  int used = 0;
  bool pending = false;  // launch_begin recorded before[used]
};
ProfileSession &profile() {
  static ProfileSession s;
  return s;
}
}  // namespace

void launch_begin(cudaStream_t st) {
  ProfileSession &s = profile();
  if (!s.open.load(std::memory_order_acquire)) return;
  std::lock_guard<std::mutex> g(s.mu);
  if (s.used < (int)s.before.size()) s.pending = cudaEventRecord(s.before[s.used], st) == cudaSuccess;
}

void note_launch(const char *name, cudaStream_t st) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  ProfileSession &s = profile();
  if (!s.open.load(std::memory_order_acquire)) return;
  std::lock_guard<std::mutex> g(s.mu);
  if (!s.pending || s.used >= (int)s.after.size()) return;
  s.pending = false;
  if (cudaEventRecord(s.after[s.used], st) != cudaSuccess) return;
  s.names[s.used] = name;
  ++s.used;
}
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

constexpr CUtensorMapDataType kU8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
// Tensor-map type of the call's 16-bit tensors.
CUtensorMapDataType t16(bool f16) {
  return f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
}

// ---------------------------------------------------------------- checks
bool aligned16(const void *p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// Rank padded to a tensor-core N of the rank pass: 16/32/64 (and 128 for
// two merged rank-64 projections).
int rank_pad(int rl) { return rl <= 16 ? 16 : (rl <= 32 ? 32 : (rl <= 64 ? 64 : 128)); }
bool rank_ok(int r) { return r == 8 || r == 16 || r == 32 || r == 64; }
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
constexpr int kBN = 256;
// Time of an NF4 GEMM tile of two m-blocks, in tiles of one m-block.
constexpr double kMb2TileCost = 1.5;
constexpr size_t kStatusBytes = 256;

lora_status_t check_weight(const lora_weight_t &W) {
  if (W.dtype != LORA_DTYPE_BF16 && W.dtype != LORA_DTYPE_FP16) return LORA_ERR_INVALID_ARG;
  if (W.type == LORA_WEIGHT_DENSE) {
    if (!aligned16(W.w) || W.absmax_scale || W.absmax_offset) return LORA_ERR_INVALID_ARG;
  } else if (W.type == LORA_WEIGHT_NF4) {
    if (!aligned16(W.w) || !aligned16(W.absmax)) return LORA_ERR_INVALID_ARG;
    if ((W.absmax_scale == nullptr) != (W.absmax_offset == nullptr)) return LORA_ERR_INVALID_ARG;
    if (W.absmax_scale && (!aligned16(W.absmax_scale) || !aligned16(W.absmax_offset)))
      return LORA_ERR_INVALID_ARG;
    if (W.blocksize != 64) return LORA_ERR_UNSUPPORTED;
  } else {
    return LORA_ERR_INVALID_ARG;
  }
  return LORA_OK;
}

bool is_f16(const lora_weight_t &W) { return W.dtype == LORA_DTYPE_FP16; }
bool is_dq(const lora_weight_t &W) { return W.type == LORA_WEIGHT_NF4 && W.absmax_scale; }
Nf4Scales scales_of(const lora_weight_t &W) {
  return Nf4Scales{W.absmax, W.absmax_scale, W.absmax_offset};
}

lora_status_t check_shape(int M, int k, int n, int r) {
  if (M < 1 || k < 1 || n < 1 || M > (1 << 30) || k > (1 << 20) || n > (1 << 20))
    return LORA_ERR_INVALID_ARG;
  if (k % 64 || n % 64) return LORA_ERR_UNSUPPORTED;
  if (!rank_ok(r)) return LORA_ERR_UNSUPPORTED;
  return LORA_OK;
}

lora_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? LORA_OK : LORA_ERR_CUDA; }

// ------------------------------------------------------------- schedule
// Persistent GEMM schedule over tiles of `mb` m-blocks: as many CTA pairs
// as fit (one per two SMs), grouped raster of 8 m-blocks (8/mb tile rows).
Schedule make_schedule(int m_tiles, int n_tiles, int slots, int mb) {
  const long long total = (long long)m_tiles * n_tiles;
  Schedule s;
  s.m_blocks = m_tiles;
  s.n_tiles = n_tiles;
  s.group_m = std::max(1, std::min(m_tiles, 8 / mb));
  s.workers = (int)std::max<long long>(1, std::min<long long>(slots, total));
  s.contiguous = 0;
  return s;
}

// Whether a bf16 forward forms s·x·Aᵀ inside its GEMM (one launch) rather
// than in a rank pass before it.  Inside the GEMM, x·Aᵀ is formed once per
// m-block by the pair that meets it, so each pair must take its tiles as one
// contiguous m-major run; on B300 that spreads the pairs over all of x and W
// at once and loses the grouped raster's L2 reuse.  Measured on the
// Llama-3-8B q/k + RoPE and MLP forwards (8 to 12 tiles per pair) the
// one-launch form was 29-31% slower, so it is taken only when every tile has
// a pair of its own (one wave), where the rank pass's launch and its extra
// stream of x are what remains.
bool fused_fwd_pays(int M, int n_tiles, int rl, bool rope) {
  const long long tiles = (long long)((M + 255) / 256) * n_tiles;
  const int fv = rank_pad(rl) <= 64 ? 64 : 128;
  const int pairs = gemm_pair_capacity(kModeFwd, rope, false, 1, fv);
  return pairs > 0 && tiles <= pairs;
}

// NF4 weights staged in 16-bit.  The fused NF4 GEMMs decode the 4-bit codes
// while staging each W tile, reading 0.53 bytes per weight; at large M the
// kernels are tensor-bound and the decode costs MMA throughput (measured on
// B300: Qwen1.5-32B gate_proj at M = 8192, fused forward 1.62 ms against
// 1.38 ms for nf4_dequant followed by the bf16 GEMM; backward 2.31 against
// 1.68 ms).  So when M >= kNf4StageMinM and the caller's workspace has room
// past what the call needs, an NF4 weight is dequantised once into it and
// the call runs on the 16-bit copy; otherwise the fused decode runs.
constexpr int kNf4StageMinM = 2048;
size_t nf4_stage_bytes(int rows, int k) { return align256((size_t)rows * k * 2); }
// Room for the bf16 block scales of a double-quantised NF4 weight.
size_t dq_expand_bytes(int rows, int k) { return align256((size_t)rows * (k / 64) * 2); }

// Prepares NF4 descriptors W1 (n1 rows) and W2 (n2 rows; null: none) for the
// kernels: when staging applies (see above; stage area at `stage_off`)
// they are replaced by 16-bit copies dequantised there; otherwise
// double-quantised block scales are expanded to bf16 at `dq_off` (room:
// dq_expand_bytes per weight), the form the fused decode reads.
lora_status_t prepare_nf4(lora_weight_t *W1, int n1, lora_weight_t *W2, int n2, int k, int M,
                          void *ws, size_t ws_bytes, size_t dq_off, size_t stage_off,
                          cudaStream_t st) {
  if (W1->type != LORA_WEIGHT_NF4) return LORA_OK;
  lora_weight_t *W[2] = {W1, W2};
  const int rows[2] = {n1, n2};
  const int nw = W2 ? 2 : 1;
  uint8_t *w8 = static_cast<uint8_t *>(ws);
  stage_off = align256(stage_off);
  const size_t b1 = nf4_stage_bytes(n1, k), b2 = W2 ? nf4_stage_bytes(n2, k) : 0;
  if (M >= kNf4StageMinM && ws_bytes >= stage_off + b1 + b2) {
    for (int i = 0; i < nw; ++i) {
      auto *dst = reinterpret_cast<uint16_t *>(w8 + stage_off + (i ? b1 : 0));
      const cudaError_t e = launch_nf4_dequant(static_cast<const uint8_t *>(W[i]->w),
                                               scales_of(*W[i]), dst, rows[i], k, is_f16(*W[i]),
                                               st);
      if (e != cudaSuccess) return LORA_ERR_CUDA;
      lora_weight_t d{};
      d.type = LORA_WEIGHT_DENSE;
      d.w = dst;
      d.dtype = W[i]->dtype;
      *W[i] = d;
    }
    return LORA_OK;
  }
  size_t o = dq_off;
  for (int i = 0; i < nw; ++i) {
    if (!is_dq(*W[i])) continue;
    auto *dst = reinterpret_cast<uint16_t *>(w8 + o);
    const cudaError_t e =
        launch_nf4_dq_expand(scales_of(*W[i]), dst, (size_t)rows[i] * (k / 64), st);
    if (e != cudaSuccess) return LORA_ERR_CUDA;
    o += dq_expand_bytes(rows[i], k);
    W[i]->absmax = dst;
    W[i]->absmax_scale = nullptr;
    W[i]->absmax_offset = nullptr;
  }
  return LORA_OK;
}

// ------------------------------------------------------ fused GEMM set-up
struct GroupArgs {
  lora_weight_t W;
  const void *b;   // FWD: B [n_g, r] (K-major); DX: A [rl, k] (read MN-major)
  void *out;
  int ncols;       // output columns
  int sv_col;      // first column of this group's rank block in s·v / s·u
  int b_cols = 0;  // FWD: columns of B (0: the launch's rank_k)
  int b_shift = 0; // FWD: rank K-block e reads B from column 64·e + b_shift
};

struct GemmOpts {
  int mode = kModeFwd;
  bool f16 = false;           // 16-bit tensors are fp16 (else bf16)
  const void *act = nullptr;  // FWD: x [M, k]; DX: dY [M, n]
  int M = 0, Kred = 0;        // rows; main reduction length (k in FWD, n in DX)
  const GroupArgs *ga = nullptr;
  int ng = 1;                 // projections along N (FWD)
  // DX: a second projection along the reduction: its W holds rows
  // [ksplit*64, Kred) of the combined reduction
  const lora_weight_t *W2 = nullptr;
  int ksplit = 0;
  const void *sv = nullptr;   // s·v or s·u [M, rl] bf16
  int rl = 0;                 // columns of sv (r, or 2r merged)
  int rank_k = 0;             // rank columns each group reduces over (r FWD, rl DX)
  bool rope = false;
  const int32_t *positions = nullptr;
  const float *cos_sin = nullptr;
  int max_pos = 0;
  int accumulate = 0;
  uint32_t *status = nullptr;
  // SwiGLU pair (FWD, ng == 2: gate, up): h [M, n] out; the groups' `out`
  // receive g and u when both are non-null
  bool swiglu = false;
  void *h = nullptr;
  // DX read-modify-write scale (out = old + acc_scale·acc); overrides of the
  // activation's column count and of W's rows as the MN-major operand (both
  // default to Kred) for operands narrower than one 64-wide K-block, whose
  // missing columns / rows the copies fill with zeros
  float acc_scale = 1.0f;
  int act_cols = 0;
  int w_rows = 0;
  int w_cols = 0;  // FWD: columns of a 16-bit W narrower than Kred (read as zeros past it)
  // FWD, bf16 W: form s·v = s·x·[a1; a2]ᵀ inside the GEMM (no rank pass, no
  // s·v in memory; sv unused).  a2 null: one projection.
  bool fused_v = false;
  const void *a1 = nullptr, *a2 = nullptr;
  float fv_scale = 0.0f;
  // DX read-modify-write masked by LoRA dropout (bf16 kernel)
  bool dropout = false;
  uint32_t drop_thresh = 0;
  float drop_scale = 1.0f;
  uint64_t drop_seed = 0, drop_offset = 0;
};

bool make_w_map(CUtensorMap *m, const lora_weight_t &W, bool dx, bool nf4, int n, int k) {
  const CUtensorMapDataType dt = t16(is_f16(W));
  if (!dx) {
    if (nf4) return make_map(m, kU8, 1, W.w, k / 2, n, (uint64_t)k / 2, 32, 128, false);
    return make_map(m, dt, 2, W.w, k, n, (uint64_t)k * 2, 64, 128, true);
  }
  if (nf4) return make_map(m, kU8, 1, W.w, k / 2, n, (uint64_t)k / 2, 64, 64, false);
  return make_map(m, dt, 2, W.w, k, n, (uint64_t)k * 2, 64, 64, true);
}

lora_status_t run_gemm(const GemmOpts &o, cudaStream_t st) {
  DeviceInfo di;
  lora_status_t s = device_info(&di);
  if (s != LORA_OK) return s;
  const bool nf4 = o.ga[0].W.type == LORA_WEIGHT_NF4;
  const CUtensorMapDataType dt = t16(o.f16);
  // double-quantised scales reach the GEMMs expanded (prepare_nf4)
  if (is_dq(o.ga[0].W) || (o.ng > 1 && is_dq(o.ga[1].W)) || (o.W2 && is_dq(*o.W2)))
    return LORA_ERR_INVALID_ARG;
  const bool dx = o.mode == kModeDx;
  const int n_extra = (o.rank_k + 63) / 64;
  GemmParams p;
  std::memset(&p, 0, sizeof(p));
  // activation [M, Kred] and rank block [M, rl]: K-major, box 64 x 128
  const int act_cols = o.act_cols > 0 ? o.act_cols : o.Kred;
  // the down-projection in the GEMM (bf16 forward): v up to fv columns
  const int fv = (o.fused_v && !nf4 && !dx) ? (rank_pad(o.rl) <= 64 ? 64 : 128) : 0;
  if (!make_map(&p.tm_act, dt, 2, o.act, act_cols, o.M, (uint64_t)act_cols * 2, 64, 128, true) ||
      (o.rank_k > 0 && !fv &&
       !make_map(&p.tm_sv, dt, 2, o.sv, o.rl, o.M, (uint64_t)o.rl * 2, 64, 128, true)))
    return LORA_ERR_CUDA;
  if (fv) {
    // CTA c stages rows [c·nv/2, +nv/2) of [a1; a2] (padded with zero rows)
    const int nv = rank_pad(o.rl), h = nv / 2;
    const bool two = o.a2 != nullptr;
    const int rows = two ? o.rl / 2 : o.rl;
    if (!make_map(&p.tm_a[0], dt, 2, o.a1, o.Kred, rows, (uint64_t)o.Kred * 2, 64, h, true) ||
        (two &&
         !make_map(&p.tm_a[1], dt, 2, o.a2, o.Kred, rows, (uint64_t)o.Kred * 2, 64, h, true)))
      return LORA_ERR_CUDA;
    p.fv_nv = nv;
    p.fv_two = two ? 1 : 0;
    p.fv_scale = o.fv_scale;
  }
  int tiles = 0;
  const bool save_gu = o.swiglu && o.ga[0].out && o.ga[1].out;
  for (int g = 0; g < o.ng; ++g) {
    GemmGroup &G = p.grp[g];
    const GroupArgs &a = o.ga[g];
    const int ncols = a.ncols;
    if (!dx) {
      const int n = ncols, k = o.Kred;
      const int bc = a.b_cols > 0 ? a.b_cols : o.rank_k;
      if (!make_w_map(&G.tm_w, a.W, false, nf4, n, o.w_cols > 0 ? o.w_cols : k) ||
          (o.rank_k > 0 &&
           !make_map(&G.tm_b, dt, 2, a.b, bc, n, (uint64_t)bc * 2, 64, 128, true)))
        return LORA_ERR_CUDA;
      G.ld_absmax = k / 64;
      G.b_shift = a.b_shift;
    } else {
      const int n = o.W2 ? o.ksplit * 64 : (o.w_rows > 0 ? o.w_rows : o.Kred), k = ncols;
      if (!make_w_map(&G.tm_w, a.W, true, nf4, n, k) ||
          (o.rank_k > 0 &&
           !make_map(&G.tm_b, dt, 2, a.b, k, o.rl, (uint64_t)k * 2, 64, 64, true)))
        return LORA_ERR_CUDA;
      G.ld_absmax = k / 64;
    }
    if ((!o.swiglu || save_gu) &&
        !make_map(&G.tm_out, dt, 2, a.out, ncols, o.M, (uint64_t)ncols * 2, 32, 32, true))
      return LORA_ERR_CUDA;
    G.out = static_cast<uint16_t *>(a.out);
    G.absmax = static_cast<const __nv_bfloat16 *>(a.W.absmax);
    G.ncols = ncols;
    G.sv_col = a.sv_col;
    G.n_extra = n_extra;
    if (fv) {
      // rank K-blocks run over the 64-column atoms of the staged s·v from the
      // one holding sv_col; B is read shifted so its columns meet this
      // group's rank columns inside the atom
      G.b_shift = a.b_shift - a.sv_col % 64;
      G.n_extra = (a.sv_col % 64 + o.rank_k + 63) / 64;
    }
    if (o.swiglu) {  // both groups cover the same tiles of 128 output columns
      G.n_tiles = (ncols + 127) / 128;
      G.tile_begin = 0;
      tiles = G.n_tiles;
    } else {
      G.n_tiles = (ncols + kBN - 1) / kBN;
      G.tile_begin = tiles;
      tiles += G.n_tiles;
    }
  }
  p.num_groups = o.ng;
  if (o.swiglu) {
    p.swiglu = 1;
    p.save_gu = save_gu ? 1 : 0;
    if (!make_map(&p.tm_h, dt, 2, o.h, o.ga[0].ncols, o.M, (uint64_t)o.ga[0].ncols * 2, 32,
                  32, true))
      return LORA_ERR_CUDA;
  }
  if (dx && o.W2) {  // second projection along the reduction
    GemmGroup &G1 = p.grp[1];
    const int k = o.ga[0].ncols, n2 = o.Kred - o.ksplit * 64;
    if (!make_w_map(&G1.tm_w, *o.W2, true, nf4, n2, k)) return LORA_ERR_CUDA;
    G1.absmax = static_cast<const __nv_bfloat16 *>(o.W2->absmax);
    G1.ld_absmax = k / 64;
    G1.ncols = k;
    p.kgroups = 2;
    p.ksplit = o.ksplit;
  } else {
    p.kgroups = 1;
  }
  p.M = o.M;
  p.K = o.Kred;
  // Tiles of one or two m-blocks.  NF4: a two-m-block tile decodes each W
  // K-block once for 512 rows instead of 256; it is taken unless its coarser
  // waves of tiles cost more than that saves (an mb = 2 tile is timed at
  // kMb2TileCost mb = 1 tiles).
  const int m_blocks = (o.M + 255) / 256;
  int mb = 1;
  int slots = gemm_pair_capacity(o.mode, o.rope, nf4, 1, fv);
  if (slots < 1) return LORA_ERR_CUDA;
  if (nf4) {
    const int slots2 = gemm_pair_capacity(o.mode, o.rope, nf4, 2, 0);
    if (slots2 < 1) return LORA_ERR_CUDA;
    const long long w1 = ((long long)m_blocks * tiles + slots - 1) / slots;
    const long long w2 = ((long long)((m_blocks + 1) / 2) * tiles + slots2 - 1) / slots2;
    if ((double)w2 * kMb2TileCost < (double)w1) mb = 2, slots = slots2;
  }
  p.sched = make_schedule((m_blocks + mb - 1) / mb, tiles, slots, mb);
  p.sched.contiguous = fv ? 1 : 0;  // one run of tiles per m-block and pair
  p.accumulate = o.accumulate;
  p.acc_scale = o.acc_scale;
  if (o.dropout) {
    p.dropout = 1;
    p.drop_thresh = o.drop_thresh;
    p.drop_ld = o.ga[0].ncols;
    p.drop_scale = o.drop_scale;
    p.drop_seed = o.drop_seed;
    p.drop_offset = o.drop_offset;
  }
  p.positions = o.positions;
  p.cos_sin = o.cos_sin;
  p.max_pos = o.max_pos;
  p.status = o.status;
  return cuda_status(launch_gemm_pair(p, o.mode, o.rope, nf4, mb, fv, p.sched.workers, o.f16, st));
}

// ------------------------------------------------------------ rank passes
// One KMAJOR problem of the rank pass: g = P·Qᵀ over `K` (P [rows, K],
// Q [rl, K] bf16, or Q = [Q1; Q2] with q_rows1 rows each).
lora_status_t kmajor_problem(SkinnyProblem &P, const void *p_ptr, int rows, int K,
                             const void *q1, const void *q2, int q_rows1, int rl, int rp,
                             CUtensorMapDataType dt, bool tight_q = false) {
  if (!make_map(&P.tm_p, dt, 2, p_ptr, K, rows, (uint64_t)K * 2, 64, 128, true))
    return LORA_ERR_CUDA;
  if (q2) {
    if (!make_map(&P.tm_q, dt, 2, q1, K, q_rows1, (uint64_t)K * 2, 64, q_rows1, true) ||
        !make_map(&P.tm_q2, dt, 2, q2, K, q_rows1, (uint64_t)K * 2, 64, q_rows1, true))
      return LORA_ERR_CUDA;
    P.q_rows1 = q_rows1;
  } else {
    // tight_q (cluster schedule only): the box covers the rl real rows and
    // the kernel keeps the rest of the tile zero; rows past rl would be
    // zero-filled copies that still cross the L2-to-SM fabric
    const int box = tight_q ? rl : rp;
    if (!make_map(&P.tm_q, dt, 2, q1, K, rl, (uint64_t)K * 2, 64, box, true))
      return LORA_ERR_CUDA;
    P.q_rows1 = 0;
    P.q_rows = box;
  }
  if (q2) P.q_rows = rp;
  P.rows = rows;
  P.row_tiles = (rows + 127) / 128;
  P.chunks = K / 64;
  return LORA_OK;
}

// One MNMAJOR problem: g = Pᵀ·(Qhi + Qlo)ᵀ over M tokens (P [M, rows],
// Q hi/lo [rp, ld]).
lora_status_t mnmajor_problem(SkinnyProblem &P, const void *p_ptr, int M, int rows,
                              const void *q_hi, const void *q_lo, int ld, int rp,
                              CUtensorMapDataType dt) {
  if (!make_map(&P.tm_p, dt, 2, p_ptr, rows, M, (uint64_t)rows * 2, 64, 64, true) ||
      !make_map(&P.tm_q, dt, 2, q_hi, M, rp, (uint64_t)ld * 2, 64, rp, true) ||
      !make_map(&P.tm_q2, dt, 2, q_lo, M, rp, (uint64_t)ld * 2, 64, rp, true))
    return LORA_ERR_CUDA;
  P.rows = rows;
  P.row_tiles = (rows + 127) / 128;
  P.chunks = (M + 63) / 64;
  return LORA_OK;
}

// CTAs per cluster of the cluster schedule: the largest split the pass
// supports for which the grid still fits on the SMs at one CTA each and
// every CTA keeps >= 8 chunks.
int pick_split(int tiles, int min_chunks, int sms, bool mn, int rp, bool dec, bool two) {
  for (int s = 8; s > 1; --s)
    if (skinny_split_ok(mn, rp, dec, two, s) && tiles * s <= sms && min_chunks >= 8 * s) return s;
  return 1;
}

// A rank pass.  The cluster schedule (one tile per cluster) is taken unless
// the stream-K schedule (equal unit ranges on one CTA per SM) cuts the
// chunks of the busiest CTA to 3/4 or less: that happens when the tiles are
// too few to fill the SMs, or of unequal lengths.  Measured on B300, the
// stream-K form has a few microseconds of extra cost (parked partials, a
// second segment per CTA), so near-balanced cluster launches stay as they
// are.  `scratch` (skinny_scratch_bytes(rp)) holds the stream-K flags and
// parked partials.
// Epoch of a stream-K launch: a random 40-bit tag drawn once per process in
// the high bits and a launch counter in the low 24, so a flag word left in a
// reused workspace by another process, by older launches or by unrelated
// data (small integers, floats) does not equal this launch's epoch.
unsigned long long next_epoch() {
  static const unsigned long long tag = [] {
    std::random_device rd;
    const unsigned long long t = ((unsigned long long)rd() << 32) ^ rd() ^
        (unsigned long long)std::chrono::steady_clock::now().time_since_epoch().count();
    return (t & 0xFFFFFFFFFFull) | 1ull;  // never zero
  }();
  static std::atomic<unsigned long long> counter{0};
  const unsigned long long c = (counter.fetch_add(1, std::memory_order_relaxed) + 1) & 0xFFFFFFull;
  return (tag << 24) | c;
}

lora_status_t run_skinny(SkinnyParams &sp, bool mn, int rp, bool f16, uint32_t *status,
                         void *scratch, cudaStream_t st, bool cluster_only = false,
                         bool dec = false, bool two = false) {
  DeviceInfo di;
  lora_status_t s;
  if ((s = device_info(&di))) return s;
  int tiles = 0, min_chunks = 1 << 30;
  long long units = 0;
  for (int q = 0; q < sp.num_problems; ++q) {
    sp.pr[q].tile_begin = tiles;
    sp.pr[q].unit_begin = units;
    tiles += sp.pr[q].row_tiles;
    min_chunks = std::min(min_chunks, sp.pr[q].chunks);
    units += (long long)sp.pr[q].row_tiles * sp.pr[q].chunks;
  }
  if (units < 1) return LORA_ERR_INVALID_ARG;
  sp.status = status;
  // `two`: two CTAs share an SM, so twice the SMs' count of CTAs fit one wave
  sp.split = pick_split(tiles, min_chunks, two ? 2 * di.sms : di.sms, mn, rp, dec, two);
  long long w_cluster = 0;  // chunks of the busiest CTA
  for (int q = 0; q < sp.num_problems; ++q)
    w_cluster = std::max<long long>(w_cluster, (sp.pr[q].chunks + sp.split - 1) / sp.split);
  // stream-K: one CTA per SM, each with at least 8 chunks (a finisher adds
  // one parked partial per extra CTA on its tile)
  const int ctas = (int)std::max<long long>(
      1, std::min<long long>(std::min(di.sms, kSkinnyMaxCtas), units / 8));
  const long long w_sk = (units + ctas - 1) / ctas;
  if (cluster_only || 4 * w_sk > 3 * w_cluster)
    return cuda_status(launch_skinny_cluster(sp, mn, rp, f16, st, dec, two));
  sp.units = units;
  sp.ctas = ctas;
  uint8_t *s8 = static_cast<uint8_t *>(scratch);
  sp.flags = reinterpret_cast<unsigned long long *>(s8);
  sp.partials = reinterpret_cast<float *>(s8 + align256((size_t)kSkinnyMaxCtas * 8));
  sp.epoch = next_epoch();
  return cuda_status(launch_skinny_sk(sp, mn, rp, f16, st));
}

// ------------------------------------------------------------------ forward
// Workspace: status | s·v [M, rl] bf16 | rank-pass scratch.
size_t fwd_sv_bytes(int M, int rl) { return align256((size_t)M * rl * 2); }
size_t fwd_bytes(int M, int rl) {
  return kStatusBytes + fwd_sv_bytes(M, rl) + skinny_scratch_bytes(rank_pad(rl));
}

// s·v = s·x·[A1; A2]ᵀ into the workspace (A2 null: one projection).
lora_status_t fwd_rank(const void *x, const void *A1, const void *A2, int M, int k, int r,
                       float scale, void *sv, uint32_t *status, bool f16, cudaStream_t st) {
  const int nproj = A2 ? 2 : 1, rl = nproj * r, rp = rank_pad(rl);
  SkinnyParams sp;
  std::memset(&sp, 0, sizeof(sp));
  SkinnyProblem &P = sp.pr[0];
  lora_status_t s;
  if ((s = kmajor_problem(P, x, M, k, A1, A2, r, rl, rp, t16(f16)))) return s;
  P.out_kind = kOutRowBf16;
  P.out_bf16 = static_cast<uint16_t *>(sv);
  P.ld_row = rl;
  P.r = r;
  P.nproj = nproj;
  P.scale = scale;
  sp.num_problems = 1;
  return run_skinny(sp, false, rp, f16, status, static_cast<uint8_t *>(sv) + fwd_sv_bytes(M, rl),
                    st);
}

// Small-M forward: with at most kSmallM tokens a GEMM tile of 256 rows is
// mostly empty and the n/256 tiles leave most SMs idle, so the forward runs
// as a rank pass over the rows of W instead, in two launches:
//   1. one rank-pass launch with two problems over the same x (the narrow
//      operand, tokens padded to 64, 96 or 128): yᵀ = W·xᵀ over the rows of W,
//      and (s·v)ᵀ = s·A·xᵀ over the rows of A; the reduction over k split
//      across the CTAs of a cluster, both written transposed (y [M, n],
//      s·v [M, r]);
//   2. y += (s·v)·Bᵀ: the GEMM with s·v as its activation (K = r) and B as
//      its weight, adding to y in its epilogue.
// Every SM streams a share of W in the first launch; the second touches only
// y, s·v and B.
constexpr int kSmallM = 128;

// Whether a forward of M tokens takes the small-M form: at M <= kSmallM,
// for a dense and an NF4 W alike.  Measured on B300 at M = 16-64 with the
// NF4 decoding pass (a 64-code row per thread, 96 token columns): Qwen1.5-32B
// down_proj 86 us against 350 us for the fused NF4 GEMM, q_proj 35 against
// 76, k_proj 29 against 86, and gate_proj (107 GEMM tiles, so its pass runs
// in two waves of CTAs) 102-106 against 125.
bool small_m_pays(int M, int, bool) { return M <= kSmallM; }

lora_status_t small_m_fwd(const void *x, const lora_weight_t &W, const void *A, const void *B,
                          void *y, int M, int k, int n, int r, float scale, void *sv,
                          uint32_t *status, bool f16, cudaStream_t st) {
  lora_status_t s;
  const CUtensorMapDataType dt = t16(f16);
  // the token axis padded to 64 (or 128): narrower tiles would leave no room
  // to split the reduction across a cluster (16-column blocks per CTA).  An
  // NF4 W pads to 96 up to 96 tokens: its decoding pass then splits a tile
  // over 3 or 6 CTAs, and a 5120-row W fills 123 SMs rather than 82.
  const bool nf4 = W.type == LORA_WEIGHT_NF4;
  const int rp = nf4 && M <= 96 ? 96 : M <= 64 ? 64 : 128;
  SkinnyParams sp;
  std::memset(&sp, 0, sizeof(sp));
  SkinnyProblem &PW = sp.pr[0];
  SkinnyProblem &PA = sp.pr[1];
  if ((s = kmajor_problem(PW, W.w, n, k, x, nullptr, 0, M, rp, dt, true)) ||
      (s = kmajor_problem(PA, A, r, k, x, nullptr, 0, M, rp, dt, true)))
    return s;
  if (nf4) {  // P from the 4-bit codes, decoded in the kernel
    if (!make_map(&PW.tm_p, kU8, 1, W.w, k / 2, n, (uint64_t)k / 2, 32, 128, false))
      return LORA_ERR_CUDA;
    PW.nf4 = 1;
    PW.absmax = static_cast<const __nv_bfloat16 *>(W.absmax);
    PW.ld_absmax = k / 64;
  }
  PW.out_kind = PA.out_kind = kOutT16;
  PW.out_bf16 = static_cast<uint16_t *>(y);
  PW.ld_t = n;
  PW.scale = 1.0f;
  PA.out_bf16 = static_cast<uint16_t *>(sv);
  PA.ld_t = r;
  PA.scale = scale;
  PW.r = PA.r = M;  // valid columns of the transposed outputs
  PW.nproj = PA.nproj = 1;
  sp.num_problems = 2;
  // a dense W at up to 64 tokens: half-depth rings, two CTAs per SM (measured
  // 16-18% faster on the Qwen1.5-32B gate / down projections at M <= 64)
  const bool two = !nf4 && rp == 64;
  if ((s = run_skinny(sp, false, rp, f16, status, nullptr, st, true, nf4, two))) return s;
  lora_weight_t wb{};
  wb.type = LORA_WEIGHT_DENSE;
  wb.w = B;
  wb.dtype = W.dtype;
  GroupArgs ga{wb, nullptr, y, n, 0};
  GemmOpts o;
  o.mode = kModeFwd;
  o.f16 = f16;
  o.act = sv;
  o.act_cols = r;
  o.M = M;
  o.Kred = 64;
  o.w_cols = r;
  o.ga = &ga;
  o.ng = 1;
  o.rank_k = 0;
  o.accumulate = 1;
  o.acc_scale = 1.0f;
  o.status = status;
  return run_gemm(o, st);
}

// ----------------------------------------------------------------- backward
// The backward of one projection -- or of two projections sharing x, taken
// as one projection of rank rl = 2r with A = [A1; A2] and B = diag(B1, B2)
// -- in three launches after the set-up:
//   rank   v = x·Aᵀ -> vᵀ hi/lo;  u = dY·B -> uᵀ hi/lo and s·u   (one launch)
//   dx     dX (+)= [dY | s·u]·[W ; A]
//   grads  dA = s·uᵀ·x, dB = s·dYᵀ·v                           (one launch)
struct BwdPlan {
  int rp, Mp;
  size_t off_bt, off_su, off_ut_hi, off_ut_lo, off_vt_hi, off_vt_lo, off_scratch, total;
};

BwdPlan plan_bwd(int M, int n, int rl, size_t start) {
  BwdPlan b{};
  b.rp = rank_pad(rl);
  b.Mp = (M + 63) & ~63;
  size_t o = align256(start);
  b.off_bt = o;     o = align256(o + (size_t)rl * n * 2);
  b.off_su = o;     o = align256(o + (size_t)M * rl * 2);
  b.off_ut_hi = o;  o = align256(o + (size_t)b.rp * b.Mp * 2);
  b.off_ut_lo = o;  o = align256(o + (size_t)b.rp * b.Mp * 2);
  b.off_vt_hi = o;  o = align256(o + (size_t)b.rp * b.Mp * 2);
  b.off_vt_lo = o;  o = align256(o + (size_t)b.rp * b.Mp * 2);
  b.off_scratch = o; o = align256(o + skinny_scratch_bytes(b.rp));
  b.total = o;
  return b;
}

size_t bwd_bytes(int M, int n, int rl) { return plan_bwd(M, n, rl, 0).total; }

struct BwdCall {
  const void *x, *A, *dy;        // A [rl, k]; dY [M, n]
  lora_weight_t W;               // W [n1, k] (the whole n unless merged)
  lora_weight_t W2;              // merged: W of projection 2, [n - n1, k]
  bool merged;
  bool f16;                      // 16-bit tensors are fp16 (else bf16)
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

lora_status_t bwd_rank(const BwdCall &c, cudaStream_t st) {
  const BwdPlan &b = c.b;
  SkinnyParams sp;
  std::memset(&sp, 0, sizeof(sp));
  SkinnyProblem &PV = sp.pr[0];
  SkinnyProblem &PU = sp.pr[1];
  lora_status_t s;
  const CUtensorMapDataType dt = t16(c.f16);
  if ((s = kmajor_problem(PV, c.x, c.M, c.k, c.A, nullptr, 0, c.rl, b.rp, dt)) ||
      (s = kmajor_problem(PU, c.dy, c.M, c.n, c.at<void>(b.off_bt), nullptr, 0, c.rl, b.rp, dt)))
    return s;
  const int nproj = c.merged ? 2 : 1;
  PV.out_kind = kOutVt;
  PV.out_hi = c.at<uint16_t>(b.off_vt_hi);
  PV.out_lo = c.at<uint16_t>(b.off_vt_lo);
  PV.ld_t = b.Mp;
  PV.r = c.r;
  PV.nproj = nproj;
  PV.scale = 1.0f;
  PU.out_kind = kOutVt | kOutRowBf16;
  PU.out_hi = c.at<uint16_t>(b.off_ut_hi);
  PU.out_lo = c.at<uint16_t>(b.off_ut_lo);
  PU.ld_t = b.Mp;
  PU.out_bf16 = c.at<uint16_t>(b.off_su);
  PU.ld_row = c.rl;
  PU.r = c.r;
  PU.nproj = nproj;
  PU.scale = c.scale;
  sp.num_problems = 2;
  return run_skinny(sp, false, b.rp, c.f16, c.status, c.at<void>(b.off_scratch), st);
}

lora_status_t bwd_dx(const BwdCall &c, cudaStream_t st) {
  GroupArgs ga{c.W, c.A, c.dx, c.k, 0};
  GemmOpts o;
  o.mode = kModeDx;
  o.f16 = c.f16;
  o.act = c.dy;
  o.M = c.M;
  o.Kred = c.n;
  o.ga = &ga;
  o.ng = 1;
  if (c.merged) {
    o.W2 = &c.W2;
    o.ksplit = c.n1 / 64;
  }
  o.sv = c.at<void>(c.b.off_su);
  o.rl = c.rl;
  o.rank_k = c.rl;
  o.accumulate = c.accumulate;
  o.status = c.status;
  return run_gemm(o, st);
}

lora_status_t bwd_grads(const BwdCall &c, cudaStream_t st) {
  const BwdPlan &b = c.b;
  SkinnyParams sp;
  std::memset(&sp, 0, sizeof(sp));
  SkinnyProblem &PA = sp.pr[0];
  SkinnyProblem &PB = sp.pr[1];
  lora_status_t s;
  const CUtensorMapDataType dt = t16(c.f16);
  if ((s = mnmajor_problem(PA, c.x, c.M, c.k, c.at<void>(b.off_ut_hi), c.at<void>(b.off_ut_lo),
                           b.Mp, b.rp, dt)) ||
      (s = mnmajor_problem(PB, c.dy, c.M, c.n, c.at<void>(b.off_vt_hi), c.at<void>(b.off_vt_lo),
                           b.Mp, b.rp, dt)))
    return s;
  const int nproj = c.merged ? 2 : 1;
  PA.out_kind = kOutRowT;
  PA.out_f32 = c.dA;
  PA.out_f32b = c.dA2;
  PA.r = c.r;
  PA.nproj = nproj;
  PA.scale = c.scale;
  PB.out_kind = kOutRow;
  PB.out_f32 = c.dB;
  PB.out_f32b = c.dB2;
  PB.r = c.r;
  PB.nproj = nproj;
  PB.split_row = c.n1;
  PB.scale = c.scale;
  sp.num_problems = 2;
  return run_skinny(sp, true, b.rp, c.f16, c.status, c.at<void>(b.off_scratch), st);
}

// dA/dB run before dX: the dA/dB pass re-reads x and dY right after the
// u/v pass has read them, so on the smaller projections (x and dY within
// the L2) it reads them from the L2; dX does not depend on either.
lora_status_t run_bwd_phases(const BwdCall &c, cudaStream_t st) {
  lora_status_t s;
  if ((s = bwd_rank(c, st))) return s;
  if ((s = bwd_grads(c, st))) return s;
  return bwd_dx(c, st);
}

// The q/k backward runs q and k as one projection of rank 2r:
// A_qk = [Aq; Ak] [2r, hidden], B_qk = diag(Bq, Bk) [nq+nk, 2r] (exact:
// x·A_qkᵀ·B_qkᵀ = [x·Aqᵀ·Bqᵀ, x·Akᵀ·Bkᵀ]).
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
  q.off_area = o; o += bwd_bytes(M, n, 2 * r);
  q.total = o;
  return q;
}

}  // namespace

namespace lora {
lora_status_t check_bwd_args(const void *x, lora_weight_t W, const void *A, const void *B,
                             const void *dy, const void *dx, const float *dA, const float *dB,
                             int M, int k, int n, int r, float alpha) {
  lora_status_t s;
  if ((s = check_shape(M, k, n, r))) return s;
  if ((s = check_weight(W))) return s;
  if (!aligned16(x) || !aligned16(A) || !aligned16(B) || !aligned16(dy) || !aligned16(dx) ||
      !aligned16(dA) || !aligned16(dB))
    return LORA_ERR_INVALID_ARG;
  if (!std::isfinite(alpha)) return LORA_ERR_INVALID_ARG;
  return LORA_OK;
}

lora_status_t check_current_device() {
  DeviceInfo di;
  return device_info(&di);
}
}  // namespace lora

// =================================================================== C ABI
extern "C" {

uint64_t lora_kernel_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

lora_status_t lora_profile_begin(int capacity) {
  if (capacity < 1 || capacity > (1 << 16)) return LORA_ERR_INVALID_ARG;
  ProfileSession &s = profile();
  std::lock_guard<std::mutex> g(s.mu);
  if (s.open.load(std::memory_order_acquire)) return LORA_ERR_INVALID_ARG;
  s.before.assign(capacity, nullptr);
  s.after.assign(capacity, nullptr);
  s.names.assign(capacity, nullptr);
  s.used = 0;
  s.pending = false;
  for (int i = 0; i < capacity; ++i) {
    if (cudaEventCreate(&s.before[i]) != cudaSuccess || cudaEventCreate(&s.after[i]) != cudaSuccess) {
      for (cudaEvent_t e : s.before)
        if (e) cudaEventDestroy(e);
      for (cudaEvent_t e : s.after)
        if (e) cudaEventDestroy(e);
      s.before.clear();
      s.after.clear();
      return LORA_ERR_CUDA;
    }
  }
  s.open.store(true, std::memory_order_release);
  return LORA_OK;
}

lora_status_t lora_profile_end(const char **names, float *ms, int capacity, int *count) {
  ProfileSession &s = profile();
  std::lock_guard<std::mutex> g(s.mu);
  if (!s.open.load(std::memory_order_acquire)) return LORA_ERR_INVALID_ARG;
  s.open.store(false, std::memory_order_release);
  lora_status_t st = LORA_OK;
  int n = 0;
  for (int i = 0; i < s.used; ++i) {
    float t = 0.0f;
    if (cudaEventSynchronize(s.after[i]) != cudaSuccess ||
        cudaEventElapsedTime(&t, s.before[i], s.after[i]) != cudaSuccess) {
      st = LORA_ERR_CUDA;
      break;
    }
    if (n < capacity && names && ms) {
      names[n] = s.names[i];
      ms[n] = t;
    }
    ++n;
  }
  if (count) *count = std::min(n, capacity);
  for (cudaEvent_t e : s.before) cudaEventDestroy(e);
  for (cudaEvent_t e : s.after) cudaEventDestroy(e);
  s.before.clear();
  s.after.clear();
  s.names.clear();
  s.used = 0;
  return st;
}

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

}  // extern "C"

namespace {
// Workspace of an operation without the room for double-quantised scales.
size_t ws_base(int op, int M, int k, int n, int r) {
  switch (op) {
    case LORA_OP_FWD:
      return fwd_bytes(M, r);
    case LORA_OP_QK_ROPE_FWD:
      return fwd_bytes(M, 2 * r);
    case LORA_OP_BWD:
      return kStatusBytes + bwd_bytes(M, n, r);
    case LORA_OP_QK_ROPE_BWD:
      return plan_qk_bwd(M, k, n, r).total;
    case LORA_OP_SWIGLU_FWD:
      return fwd_bytes(M, 2 * r);
    case LORA_OP_SWIGLU_BWD:
      return plan_qk_bwd(M, k, 2 * n, r).total;
    case LORA_OP_FWD_DROPOUT:
      return fwd_bytes(M, r) + align256((size_t)M * k * 2);
    case LORA_OP_BWD_DROPOUT:
      return kStatusBytes + bwd_bytes(M, n, r) + align256((size_t)M * k * 2);
    case LORA_OP_MERGE:
      return kStatusBytes;
    case LORA_OP_MERGE_NF4:
      return kStatusBytes + align256((size_t)n * k * 2);
  }
  return 0;
}

// Room for the bf16 expansion of double-quantised block scales, past
// ws_base: one weight [n, k] (two for the q/k pair, whose n is the sum, and
// for gate / up); merges decode the scales directly.
size_t ws_dq(int op, int k, int n) {
  switch (op) {
    case LORA_OP_FWD:
    case LORA_OP_BWD:
    case LORA_OP_FWD_DROPOUT:
    case LORA_OP_BWD_DROPOUT:
      return dq_expand_bytes(n, k);
    case LORA_OP_QK_ROPE_FWD:
    case LORA_OP_QK_ROPE_BWD:
      return dq_expand_bytes(n, k) + 512;
    case LORA_OP_SWIGLU_FWD:
    case LORA_OP_SWIGLU_BWD:
      return 2 * dq_expand_bytes(n, k);
  }
  return 0;
}

int op_flags(const lora_weight_t &W1, const lora_weight_t *W2 = nullptr) {
  return (is_dq(W1) || (W2 && is_dq(*W2))) ? LORA_OP_FLAG_DQ : 0;
}
}  // namespace

extern "C" {

size_t lora_workspace_size(int op, int M, int k, int n, int r) {
  if (M < 1 || k < 1 || n < 1 || !rank_ok(r) || M > (1 << 30)) return 0;
  const bool dq = (op & LORA_OP_FLAG_DQ) != 0;
  op &= ~LORA_OP_FLAG_DQ;
  const size_t base = ws_base(op, M, k, n, r);
  if (base == 0) return 0;
  return base + (dq ? ws_dq(op, k, n) : 0);
}

size_t lora_nf4_stage_bytes(int n, int k) {
  if (n < 1 || k < 1) return 0;
  return nf4_stage_bytes(n, k);
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
  if ((s = check_weight(W))) return s;
  if (!aligned16(x) || !aligned16(A) || !aligned16(B) || !aligned16(y) || !aligned16(ws))
    return LORA_ERR_INVALID_ARG;
  if (!std::isfinite(alpha)) return LORA_ERR_INVALID_ARG;
  const size_t need = lora_workspace_size(LORA_OP_FWD | op_flags(W), M, k, n, r);
  if (ws_bytes < need) return LORA_ERR_WORKSPACE;
  DeviceInfo di;
  if ((s = device_info(&di))) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint32_t *status = static_cast<uint32_t *>(ws);
  void *sv = static_cast<uint8_t *>(ws) + kStatusBytes;
  const float scale = alpha / (float)r;
  const bool f16 = is_f16(W);
  if ((s = prepare_nf4(&W, n, nullptr, 0, k, M, ws, ws_bytes, ws_base(LORA_OP_FWD, M, k, n, r),
                       need, st)))
    return s;
  if (small_m_pays(M, n, W.type == LORA_WEIGHT_NF4))
    return small_m_fwd(x, W, A, B, y, M, k, n, r, scale, sv, status, f16, st);
  // 16-bit W, one wave of tiles: one launch, s·x·Aᵀ formed in the GEMM;
  // otherwise a rank pass first
  const bool fused = W.type == LORA_WEIGHT_DENSE && fused_fwd_pays(M, (n + 255) / 256, r, false);
  if (!fused && (s = fwd_rank(x, A, nullptr, M, k, r, scale, sv, status, f16, st))) return s;
  GroupArgs ga{W, B, y, n, 0};
  GemmOpts o;
  o.mode = kModeFwd;
  o.f16 = f16;
  o.act = x;
  o.M = M;
  o.Kred = k;
  o.ga = &ga;
  o.ng = 1;
  o.sv = sv;
  o.rl = r;
  o.rank_k = r;
  o.status = status;
  o.fused_v = fused;
  o.a1 = A;
  o.fv_scale = scale;
  return run_gemm(o, st);
}

lora_status_t lora_linear_bwd(const void *x, lora_weight_t W, const void *A, const void *B,
                              const void *dy, void *dx, int accumulate_dx, float *dA, float *dB,
                              int M, int k, int n, int r, float alpha, void *ws, size_t ws_bytes,
                              lora_stream_t stream) {
  lora_status_t s;
  if ((s = lora::check_bwd_args(x, W, A, B, dy, dx, dA, dB, M, k, n, r, alpha))) return s;
  if (!aligned16(ws)) return LORA_ERR_INVALID_ARG;
  const size_t need = lora_workspace_size(LORA_OP_BWD | op_flags(W), M, k, n, r);
  if (ws_bytes < need) return LORA_ERR_WORKSPACE;
  DeviceInfo di;
  if ((s = device_info(&di))) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t *w8 = static_cast<uint8_t *>(ws);
  const bool f16 = is_f16(W);
  if ((s = prepare_nf4(&W, n, nullptr, 0, k, M, ws, ws_bytes, ws_base(LORA_OP_BWD, M, k, n, r),
                       need, st)))
    return s;
  BwdCall c{};
  c.x = x;
  c.A = A;
  c.dy = dy;
  c.W = W;
  c.merged = false;
  c.f16 = f16;
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
  c.b = plan_bwd(M, n, r, kStatusBytes);
  c.ws = w8;
  // set-up: Bᵀ
  BwdPrep pp{};
  pp.M = M;
  pp.n1 = n;
  pp.k = k;
  pp.r = r;
  pp.nproj = 1;
  pp.B1 = static_cast<const uint16_t *>(B);
  pp.Bt = c.at<uint16_t>(c.b.off_bt);
  if ((s = cuda_status(launch_bwd_prep(pp, f16, st)))) return s;
  return run_bwd_phases(c, st);
}

// ------------------------------------------------------------- dropout
// Drop threshold on 16-bit uniforms and 1/q for a dropout rate p (the keep
// probability is q = 1 − thresh/65536); false if p is outside [0, 1).
static bool dropout_params(float p, uint32_t *thresh, float *inv_q) {
  if (!(p >= 0.0f && p < 1.0f)) return false;
  const double t = std::nearbyint((double)p * 65536.0);
  if (t >= 65536.0) return false;
  *thresh = (uint32_t)t;
  *inv_q = (float)(1.0 / (1.0 - t / 65536.0));
  return true;
}

lora_status_t lora_linear_fwd_dropout(const void *x, lora_weight_t W, const void *A,
                                      const void *B, void *y, int M, int k, int n, int r,
                                      float alpha, float dropout_p, uint64_t seed,
                                      uint64_t offset, void *ws, size_t ws_bytes,
                                      lora_stream_t stream) {
  lora_status_t s;
  if ((s = check_shape(M, k, n, r))) return s;
  if ((s = check_weight(W))) return s;
  if (!aligned16(x) || !aligned16(A) || !aligned16(B) || !aligned16(y) || !aligned16(ws))
    return LORA_ERR_INVALID_ARG;
  uint32_t thresh = 0;
  float inv_q = 1.0f;
  if (!std::isfinite(alpha) || !dropout_params(dropout_p, &thresh, &inv_q))
    return LORA_ERR_INVALID_ARG;
  const size_t need = lora_workspace_size(LORA_OP_FWD_DROPOUT | op_flags(W), M, k, n, r);
  if (ws_bytes < need) return LORA_ERR_WORKSPACE;
  DeviceInfo di;
  if ((s = device_info(&di))) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t *w8 = static_cast<uint8_t *>(ws);
  uint32_t *status = static_cast<uint32_t *>(ws);
  void *sv = w8 + kStatusBytes;
  auto *xd = reinterpret_cast<uint16_t *>(w8 + fwd_bytes(M, r));
  const float scale = alpha / (float)r;
  const bool f16 = is_f16(W);
  if ((s = prepare_nf4(&W, n, nullptr, 0, k, M, ws, ws_bytes,
                       ws_base(LORA_OP_FWD_DROPOUT, M, k, n, r), need, st)))
    return s;
  // x̃ = x ⊙ keep / q feeds the down-projection only; the base GEMM reads x
  if ((s = cuda_status(launch_dropout_x(static_cast<const uint16_t *>(x), xd, M, k, seed, offset,
                                        thresh, inv_q, f16, st))))
    return s;
  if ((s = fwd_rank(xd, A, nullptr, M, k, r, scale, sv, status, f16, st))) return s;
  GroupArgs ga{W, B, y, n, 0};
  GemmOpts o;
  o.mode = kModeFwd;
  o.f16 = f16;
  o.act = x;
  o.M = M;
  o.Kred = k;
  o.ga = &ga;
  o.ng = 1;
  o.sv = sv;
  o.rl = r;
  o.rank_k = r;
  o.status = status;
  return run_gemm(o, st);
}

lora_status_t lora_linear_bwd_dropout(const void *x, lora_weight_t W, const void *A,
                                      const void *B, const void *dy, void *dx, int accumulate_dx,
                                      float *dA, float *dB, int M, int k, int n, int r,
                                      float alpha, float dropout_p, uint64_t seed,
                                      uint64_t offset, void *ws, size_t ws_bytes,
                                      lora_stream_t stream) {
  lora_status_t s;
  if ((s = lora::check_bwd_args(x, W, A, B, dy, dx, dA, dB, M, k, n, r, alpha))) return s;
  if (!aligned16(ws)) return LORA_ERR_INVALID_ARG;
  uint32_t thresh = 0;
  float inv_q = 1.0f;
  if (!dropout_params(dropout_p, &thresh, &inv_q)) return LORA_ERR_INVALID_ARG;
  const size_t need = lora_workspace_size(LORA_OP_BWD_DROPOUT | op_flags(W), M, k, n, r);
  if (ws_bytes < need) return LORA_ERR_WORKSPACE;
  DeviceInfo di;
  if ((s = device_info(&di))) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t *w8 = static_cast<uint8_t *>(ws);
  auto *xd = reinterpret_cast<uint16_t *>(w8 + kStatusBytes + bwd_bytes(M, n, r));
  const bool f16 = is_f16(W);
  const int dtype = W.dtype;
  if ((s = prepare_nf4(&W, n, nullptr, 0, k, M, ws, ws_bytes,
                       ws_base(LORA_OP_BWD_DROPOUT, M, k, n, r), need, st)))
    return s;
  BwdCall c{};
  c.x = xd;  // the rank passes reduce over the dropped-out x (v and dA)
  c.A = A;
  c.dy = dy;
  c.W = W;
  c.merged = false;
  c.f16 = f16;
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
  c.b = plan_bwd(M, n, r, kStatusBytes);
  c.ws = w8;
  BwdPrep pp{};
  pp.M = M;
  pp.n1 = n;
  pp.k = k;
  pp.r = r;
  pp.nproj = 1;
  pp.B1 = static_cast<const uint16_t *>(B);
  pp.Bt = c.at<uint16_t>(c.b.off_bt);
  if ((s = cuda_status(launch_bwd_prep(pp, f16, st)))) return s;
  // the same mask as the forward, regenerated from (seed, offset)
  if ((s = cuda_status(launch_dropout_x(static_cast<const uint16_t *>(x), xd, M, k, seed, offset,
                                        thresh, inv_q, f16, st))))
    return s;
  if ((s = bwd_rank(c, st))) return s;
  if ((s = bwd_grads(c, st))) return s;  // before dX, as in run_bwd_phases
  // dX = dY·W (no adapter K-blocks) ...
  {
    GroupArgs ga{W, nullptr, dx, k, 0};
    GemmOpts o;
    o.mode = kModeDx;
    o.f16 = f16;
    o.act = dy;
    o.M = M;
    o.Kred = n;
    o.ga = &ga;
    o.ng = 1;
    o.rank_k = 0;
    o.accumulate = accumulate_dx;
    o.status = c.status;
    if ((s = run_gemm(o, st))) return s;
  }
  // ... + (s·u·A) ⊙ keep / q: the adapter term as its own K = r GEMM whose
  // read-modify-write epilogue applies the mask
  {
    lora_weight_t wa{};
    wa.type = LORA_WEIGHT_DENSE;
    wa.w = A;
    wa.dtype = dtype;
    GroupArgs ga{wa, nullptr, dx, k, 0};
    GemmOpts o;
    o.mode = kModeDx;
    o.f16 = f16;
    o.act = c.at<void>(c.b.off_su);
    o.act_cols = r;
    o.M = M;
    o.Kred = 64;
    o.w_rows = r;
    o.ga = &ga;
    o.ng = 1;
    o.rank_k = 0;
    o.accumulate = 1;
    o.status = c.status;
    o.dropout = true;
    o.drop_thresh = thresh;
    o.drop_scale = inv_q;
    o.drop_seed = seed;
    o.drop_offset = offset;
    return run_gemm(o, st);
  }
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
  if ((s = check_weight(Wq))) return s;
  if ((s = check_weight(Wk))) return s;
  if (Wq.type != Wk.type || Wq.dtype != Wk.dtype) return LORA_ERR_UNSUPPORTED;
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
  size_t need = lora_workspace_size(LORA_OP_QK_ROPE_FWD | op_flags(Wq, &Wk), M, hidden, nq + nk, r);
  const size_t cache_off = align256(need);
  if (!cos_sin_cache) need = cache_off + lora_rope_cache_bytes(max_pos, head_dim);
  if (ws_bytes < need) return LORA_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  DeviceInfo di;
  if ((s = device_info(&di))) return s;
  uint8_t *w8 = static_cast<uint8_t *>(ws);
  uint32_t *status = static_cast<uint32_t *>(ws);
  const bool f16 = is_f16(Wq);
  if ((s = prepare_nf4(&Wq, nq, &Wk, nk, hidden, M, ws, ws_bytes,
                       ws_base(LORA_OP_QK_ROPE_FWD, M, hidden, nq + nk, r), need, st)))
    return s;
  const float *cache = cos_sin_cache;
  if (!cache) {
    float *cb = reinterpret_cast<float *>(w8 + cache_off);
    if ((s = cuda_status(launch_rope_cache(cb, max_pos, head_dim, rope_theta, st)))) return s;
    cache = cb;
  }
  // s·v = s·x·[Aq; Ak]ᵀ [M, 2r]: formed in the GEMM for bf16 W, else by a
  // rank pass over both projections at once
  void *sv = w8 + kStatusBytes;
  const float scale = alpha / (float)r;
  const bool fused = Wq.type == LORA_WEIGHT_DENSE &&
                     fused_fwd_pays(M, (nq + 255) / 256 + (nk + 255) / 256, 2 * r, true);
  if (!fused && (s = fwd_rank(x, Aq, Ak, M, hidden, r, scale, sv, status, f16, st))) return s;
  // one GEMM launch over both weights; group g reduces over its r columns of s·v
  GroupArgs ga[2] = {{Wq, Bq, q, nq, 0}, {Wk, Bk, k_out, nk, r}};
  GemmOpts o;
  o.mode = kModeFwd;
  o.f16 = f16;
  o.act = x;
  o.M = M;
  o.Kred = hidden;
  o.ga = ga;
  o.ng = 2;
  o.sv = sv;
  o.rl = 2 * r;
  o.rank_k = r;
  o.rope = true;
  o.positions = positions;
  o.cos_sin = cache;
  o.max_pos = max_pos;
  o.status = status;
  o.fused_v = fused;
  o.a1 = Aq;
  o.a2 = Ak;
  o.fv_scale = scale;
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
  size_t need = lora_workspace_size(LORA_OP_QK_ROPE_BWD | op_flags(Wq, &Wk), M, hidden, nq + nk, r);
  const size_t cache_off = align256(need);
  if (!cos_sin_cache) need = cache_off + lora_rope_cache_bytes(max_pos, head_dim);
  if (ws_bytes < need) return LORA_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  DeviceInfo di;
  if ((s = device_info(&di))) return s;
  uint8_t *w8 = static_cast<uint8_t *>(ws);
  uint32_t *status = static_cast<uint32_t *>(ws);
  const bool f16 = is_f16(Wq);
  if ((s = prepare_nf4(&Wq, nq, &Wk, nk, hidden, M, ws, ws_bytes,
                       ws_base(LORA_OP_QK_ROPE_BWD, M, hidden, nq + nk, r), need, st)))
    return s;
  const float *cache = cos_sin_cache;
  if (!cache) {
    float *cb = reinterpret_cast<float *>(w8 + cache_off);
    if ((s = cuda_status(launch_rope_cache(cb, max_pos, head_dim, rope_theta, st)))) return s;
    cache = cb;
  }
  // the backward of one projection of rank 2r, W = [Wq; Wk] along the
  // reduction of dX, with dA/dB split back per projection
  const int n = nq + nk;
  const QkBwdPlan qp = plan_qk_bwd(M, hidden, n, r);
  BwdCall c{};
  c.x = x;
  c.A = w8 + qp.off_a;
  c.dy = w8 + qp.off_dy;
  c.W = Wq;
  c.W2 = Wk;
  c.merged = true;
  c.f16 = f16;
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
  c.b = plan_bwd(M, n, 2 * r, 0);
  c.ws = w8 + qp.off_area;
  // set-up: dq, dk rotated back (RoPE is orthogonal) into one [M, nq+nk]
  // gradient, A_qk, B_qkᵀ
  BwdPrep pp{};
  pp.dy1 = static_cast<const uint16_t *>(dq);
  pp.dy2 = static_cast<const uint16_t *>(dk);
  pp.dy_out = reinterpret_cast<uint16_t *>(w8 + qp.off_dy);
  pp.pos = positions;
  pp.cos_sin = cache;
  pp.max_pos = max_pos;
  pp.status = status;
  pp.M = M;
  pp.n1 = nq;
  pp.n2 = nk;
  pp.k = hidden;
  pp.r = r;
  pp.nproj = 2;
  pp.A1 = static_cast<const uint16_t *>(Aq);
  pp.A2 = static_cast<const uint16_t *>(Ak);
  pp.A_out = reinterpret_cast<uint16_t *>(w8 + qp.off_a);
  pp.B1 = static_cast<const uint16_t *>(Bq);
  pp.B2 = static_cast<const uint16_t *>(Bk);
  pp.Bt = c.at<uint16_t>(c.b.off_bt);
  if ((s = cuda_status(launch_bwd_prep(pp, f16, st)))) return s;
  return run_bwd_phases(c, st);
}

static lora_status_t check_pair(const void *x, lora_weight_t Wg, const void *Ag, const void *Bg,
                                lora_weight_t Wu, const void *Au, const void *Bu, int M, int k,
                                int n, int r, float alpha, const void *ws) {
  lora_status_t s;
  if ((s = check_shape(M, k, n, r))) return s;
  if ((s = check_weight(Wg))) return s;
  if ((s = check_weight(Wu))) return s;
  if (Wg.type != Wu.type || Wg.dtype != Wu.dtype) return LORA_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(Ag) || !aligned16(Bg) || !aligned16(Au) || !aligned16(Bu) ||
      !aligned16(ws))
    return LORA_ERR_INVALID_ARG;
  if (!std::isfinite(alpha)) return LORA_ERR_INVALID_ARG;
  return LORA_OK;
}

lora_status_t lora_swiglu_fwd(const void *x, lora_weight_t Wg, const void *Ag, const void *Bg,
                              lora_weight_t Wu, const void *Au, const void *Bu, void *h, void *g,
                              void *u, int M, int k, int n, int r, float alpha, void *ws,
                              size_t ws_bytes, lora_stream_t stream) {
  lora_status_t s;
  if ((s = check_pair(x, Wg, Ag, Bg, Wu, Au, Bu, M, k, n, r, alpha, ws))) return s;
  if (!aligned16(h) || (g == nullptr) != (u == nullptr) || (g && (!aligned16(g) || !aligned16(u))))
    return LORA_ERR_INVALID_ARG;
  const size_t need = lora_workspace_size(LORA_OP_SWIGLU_FWD | op_flags(Wg, &Wu), M, k, n, r);
  if (ws_bytes < need) return LORA_ERR_WORKSPACE;
  DeviceInfo di;
  if ((s = device_info(&di))) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint32_t *status = static_cast<uint32_t *>(ws);
  const bool f16 = is_f16(Wg);
  if ((s = prepare_nf4(&Wg, n, &Wu, n, k, M, ws, ws_bytes,
                       ws_base(LORA_OP_SWIGLU_FWD, M, k, n, r), need, st)))
    return s;
  void *sv = static_cast<uint8_t *>(ws) + kStatusBytes;
  const float scale = alpha / (float)r;
  // s·v = s·x·[Ag; Au]ᵀ [M, 2r]: formed in the GEMM for bf16 W, else by a
  // rank pass over both projections
  const bool fused = Wg.type == LORA_WEIGHT_DENSE && fused_fwd_pays(M, (n + 127) / 128, 2 * r, false);
  if (!fused && (s = fwd_rank(x, Ag, Au, M, k, r, scale, sv, status, f16, st))) return s;
  // one fused GEMM: CTA 0 of a pair stages gate rows, CTA 1 the up rows of
  // the same output columns; a rank K-block of [s·vg | s·vu] meets Bg in the
  // gate half and Bu (read r columns to the left, so it lines up with s·vu)
  // in the up half
  GroupArgs ga[2] = {{Wg, Bg, g, n, 0, r, 0}, {Wu, Bu, u, n, 0, r, -r}};
  GemmOpts o;
  o.mode = kModeFwd;
  o.f16 = f16;
  o.act = x;
  o.M = M;
  o.Kred = k;
  o.ga = ga;
  o.ng = 2;
  o.sv = sv;
  o.rl = 2 * r;
  o.rank_k = 2 * r;
  o.status = status;
  o.swiglu = true;
  o.h = h;
  o.fused_v = fused;
  o.a1 = Ag;
  o.a2 = Au;
  o.fv_scale = scale;
  return run_gemm(o, st);
}

lora_status_t lora_swiglu_bwd(const void *x, lora_weight_t Wg, const void *Ag, const void *Bg,
                              lora_weight_t Wu, const void *Au, const void *Bu, const void *g,
                              const void *u, const void *dh, void *dx, int accumulate_dx,
                              float *dAg, float *dBg, float *dAu, float *dBu, int M, int k, int n,
                              int r, float alpha, void *ws, size_t ws_bytes,
                              lora_stream_t stream) {
  lora_status_t s;
  if ((s = check_pair(x, Wg, Ag, Bg, Wu, Au, Bu, M, k, n, r, alpha, ws))) return s;
  if (!aligned16(g) || !aligned16(u) || !aligned16(dh) || !aligned16(dx) || !aligned16(dAg) ||
      !aligned16(dBg) || !aligned16(dAu) || !aligned16(dBu))
    return LORA_ERR_INVALID_ARG;
  const size_t need = lora_workspace_size(LORA_OP_SWIGLU_BWD | op_flags(Wg, &Wu), M, k, n, r);
  if (ws_bytes < need) return LORA_ERR_WORKSPACE;
  DeviceInfo di;
  if ((s = device_info(&di))) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t *w8 = static_cast<uint8_t *>(ws);
  const bool f16 = is_f16(Wg);
  if ((s = prepare_nf4(&Wg, n, &Wu, n, k, M, ws, ws_bytes,
                       ws_base(LORA_OP_SWIGLU_BWD, M, k, n, r), need, st)))
    return s;
  // gate and up as one projection of rank 2r over n_total = 2n outputs:
  // dY = [dg | du], A = [Ag; Au], B = diag(Bg, Bu), W = [Wg; Wu] along dX's
  // reduction (the q/k layout)
  const QkBwdPlan qp = plan_qk_bwd(M, k, 2 * n, r);
  BwdCall c{};
  c.x = x;
  c.A = w8 + qp.off_a;
  c.dy = w8 + qp.off_dy;
  c.W = Wg;
  c.W2 = Wu;
  c.merged = true;
  c.f16 = f16;
  c.dx = dx;
  c.accumulate = accumulate_dx;
  c.dA = dAg;
  c.dB = dBg;
  c.dA2 = dAu;
  c.dB2 = dBu;
  c.M = M;
  c.k = k;
  c.n = 2 * n;
  c.n1 = n;
  c.r = r;
  c.rl = 2 * r;
  c.scale = alpha / (float)r;
  c.status = static_cast<uint32_t *>(ws);
  c.b = plan_bwd(M, 2 * n, 2 * r, 0);
  c.ws = w8 + qp.off_area;
  BwdPrep pp{};
  pp.sw_dh = static_cast<const uint16_t *>(dh);
  pp.sw_g = static_cast<const uint16_t *>(g);
  pp.sw_u = static_cast<const uint16_t *>(u);
  pp.dy_out = reinterpret_cast<uint16_t *>(w8 + qp.off_dy);
  pp.status = c.status;
  pp.M = M;
  pp.n1 = n;
  pp.n2 = n;
  pp.k = k;
  pp.r = r;
  pp.nproj = 2;
  pp.A1 = static_cast<const uint16_t *>(Ag);
  pp.A2 = static_cast<const uint16_t *>(Au);
  pp.A_out = reinterpret_cast<uint16_t *>(w8 + qp.off_a);
  pp.B1 = static_cast<const uint16_t *>(Bg);
  pp.B2 = static_cast<const uint16_t *>(Bu);
  pp.Bt = c.at<uint16_t>(c.b.off_bt);
  if ((s = cuda_status(launch_bwd_prep(pp, f16, st)))) return s;
  return run_bwd_phases(c, st);
}

// W [n, k] 16-bit (in place) += sign·s·B·A on the tensor cores: the dX GEMM
// with B [n, r] as its activation (one 64-wide K-block, columns past r read
// as zero), A [r, k] as its MN-major weight (rows past r zero) and the
// read-modify-write epilogue scaled by sign·s.
static lora_status_t merge_dense(void *W, int dtype, const void *A, const void *B, int n, int k,
                                 int r, float scale, uint32_t *status, cudaStream_t st) {
  lora_weight_t wa{};
  wa.type = LORA_WEIGHT_DENSE;
  wa.w = A;
  wa.dtype = dtype;
  GroupArgs ga{wa, nullptr, W, k, 0};
  GemmOpts o;
  o.mode = kModeDx;
  o.f16 = dtype == LORA_DTYPE_FP16;
  o.act = B;
  o.act_cols = r;
  o.M = n;
  o.Kred = 64;
  o.w_rows = r;
  o.ga = &ga;
  o.ng = 1;
  o.rank_k = 0;
  o.accumulate = 1;
  o.acc_scale = scale;
  o.status = status;
  return run_gemm(o, st);
}

static lora_status_t check_merge(const void *A, const void *B, int n, int k, int r, float alpha,
                                 int sign, const void *ws) {
  if (n < 1 || k < 1 || n > (1 << 20) || k > (1 << 20)) return LORA_ERR_INVALID_ARG;
  if (k % 64 || n % 64) return LORA_ERR_UNSUPPORTED;
  if (!rank_ok(r)) return LORA_ERR_UNSUPPORTED;
  if (!aligned16(A) || !aligned16(B) || !aligned16(ws)) return LORA_ERR_INVALID_ARG;
  if (!std::isfinite(alpha) || (sign != 1 && sign != -1)) return LORA_ERR_INVALID_ARG;
  return LORA_OK;
}

lora_status_t lora_merge(lora_weight_t W, const void *A, const void *B, int n, int k, int r,
                         float alpha, int sign, void *ws, size_t ws_bytes, lora_stream_t stream) {
  lora_status_t s;
  if ((s = check_merge(A, B, n, k, r, alpha, sign, ws))) return s;
  if ((s = check_weight(W))) return s;
  const bool nf4 = W.type == LORA_WEIGHT_NF4;
  if (ws_bytes < lora_workspace_size(nf4 ? LORA_OP_MERGE_NF4 : LORA_OP_MERGE, 1, k, n, r))
    return LORA_ERR_WORKSPACE;
  DeviceInfo di;
  if ((s = device_info(&di))) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const float scale = (float)sign * alpha / (float)r;
  uint32_t *status = static_cast<uint32_t *>(ws);
  if (!nf4)
    return merge_dense(const_cast<void *>(W.w), W.dtype, A, B, n, k, r, scale, status, st);
  // dequantise into the workspace, merge there, quantise back in place
  // (the weight's own scale form: bf16 absmax or double-quantised)
  auto *wd = reinterpret_cast<uint16_t *>(static_cast<uint8_t *>(ws) + kStatusBytes);
  auto *codes = static_cast<uint8_t *>(const_cast<void *>(W.w));
  if ((s = cuda_status(launch_nf4_dequant(codes, scales_of(W), wd, n, k, is_f16(W), st))))
    return s;
  if ((s = merge_dense(wd, W.dtype, A, B, n, k, r, scale, status, st))) return s;
  return cuda_status(launch_nf4_quantize(wd, codes, const_cast<void *>(W.absmax),
                                         const_cast<float *>(W.absmax_scale),
                                         const_cast<float *>(W.absmax_offset), n, k, is_f16(W),
                                         st));
}

static lora_status_t check_nf4_call(const lora_weight_t &W, int n, int k) {
  lora_status_t s;
  if (W.type != LORA_WEIGHT_NF4) return LORA_ERR_INVALID_ARG;
  if ((s = check_weight(W))) return s;
  if (n < 1 || k < 1 || n > (1 << 20) || k > (1 << 20)) return LORA_ERR_INVALID_ARG;
  if (k % 64) return LORA_ERR_UNSUPPORTED;
  // double quantisation: the quantiser parks 16 bytes of statistics in each
  // group's scale codes, so the last group needs 16 blocks (n·k/64 % 16 == 0)
  if (W.absmax_scale && ((size_t)n * (k / 64)) % 16) return LORA_ERR_UNSUPPORTED;
  return LORA_OK;
}

lora_status_t nf4_dequant(lora_weight_t W, void *w_out, int n, int k, lora_stream_t stream) {
  lora_status_t s;
  if ((s = check_nf4_call(W, n, k))) return s;
  if (!aligned16(w_out)) return LORA_ERR_INVALID_ARG;
  DeviceInfo di;
  if ((s = device_info(&di))) return s;
  return cuda_status(launch_nf4_dequant(static_cast<const uint8_t *>(W.w), scales_of(W),
                                        static_cast<uint16_t *>(w_out), n, k, is_f16(W),
                                        reinterpret_cast<cudaStream_t>(stream)));
}

lora_status_t nf4_quantize(const void *w, lora_weight_t W_out, int n, int k,
                           lora_stream_t stream) {
  lora_status_t s;
  if ((s = check_nf4_call(W_out, n, k))) return s;
  if (!aligned16(w)) return LORA_ERR_INVALID_ARG;
  DeviceInfo di;
  if ((s = device_info(&di))) return s;
  return cuda_status(launch_nf4_quantize(
      static_cast<const uint16_t *>(w), static_cast<uint8_t *>(const_cast<void *>(W_out.w)),
      const_cast<void *>(W_out.absmax), const_cast<float *>(W_out.absmax_scale),
      const_cast<float *>(W_out.absmax_offset), n, k, is_f16(W_out),
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
