// Internal interface between the C-ABI host code (api.cu) and the kernels.
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "lora_b300.h"

namespace lora {

// ------------------------------------------------ per-device host state
// Devices the per-device caches below track (ordinals 0..63); calls on a
// higher ordinal skip the caches and query every time.
constexpr int kMaxDevices = 64;

// Raises the dynamic shared-memory limit of `kern` to `bytes` on the current
// device, once per device: the attribute belongs to the (kernel, device)
// pair, so a process that drives several GPUs sets it on each.  `done` is the
// calling launcher's per-kernel record (one bit per device); concurrent
// first calls may both set the attribute, which is harmless.
inline cudaError_t smem_attr_once(std::atomic<uint64_t> &done, const void *kern, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < kMaxDevices) ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Streaming multiprocessors of the current device (cached per device);
// 0 if the query fails.
inline int current_device_sms() {
  static std::atomic<int> cached[kMaxDevices];  // 0: not queried yet
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  const bool slot = dev >= 0 && dev < kMaxDevices;
  if (slot) {
    const int v = cached[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
  }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (slot) cached[dev].store(sms, std::memory_order_relaxed);
  return sms;
}

// The fused GEMM computes, per output tile, one reduction over the
// concatenated K axis [ main | rank ]:
//   FWD  y  = [x | s·v] · [W | B]ᵀ    (s·v = s·x·Aᵀ, from the rank pass)
//   DX   dX = [dY | s·u] · [W ; A]     (s·u = s·dY·B)
// The rank part is one to two extra 64-wide K-blocks that fill the same
// pipeline slots as the main K-blocks: the activation slot from tm_sv, the
// weight slot from the group's tm_b.
//   FWD: W [n,k] (K-major), tm_b = B [n, r] K-major, out = y [M, n].
//   DX:  W [n,k] read as an MN-major operand, tm_b = A [rl, k] MN-major,
//        out = dX [M, k].
// NF4 weights: tm_w maps the codes [n, k/2] bytes and absmax points at the
// bf16 block scales [n, k/64].
struct GemmGroup {
  CUtensorMap tm_w;
  CUtensorMap tm_b;
  CUtensorMap tm_out;  // out [M, ncols] 16-bit: box 32 x 32, 64-byte swizzle
  uint16_t *out;       // raw 16-bit words (bf16 or fp16, the kernel's type)
  const __nv_bfloat16 *absmax;
  int ncols;       // output columns of this group (n in FWD, k in DX)
  int n_tiles;     // ceil(ncols / 256)
  int tile_begin;  // first global n-tile index of this group
  int ld_absmax;   // k / 64 (NF4)
  int sv_col;      // first column of this group's rank block in s·v / s·u
  int n_extra;     // extra 64-wide K-blocks (ceil(rank / 64))
  int b_shift;     // FWD: x coordinate of rank K-block e in tm_b is 64·e + b_shift
};

struct GemmParams {
  CUtensorMap tm_act;  // x [M,k] (FWD) or dY [M,n] (DX): K-major, box 64 x 128
  CUtensorMap tm_sv;   // s·v or s·u [M, rl] bf16: K-major, box 64 x 128
  GemmGroup grp[kMaxGroups];
  int num_groups;
  int M;
  int K;          // main reduction length: k (FWD) or n (DX)
  // DX mode: W rows (the reduction) come from grp[0].tm_w for 64-chunks
  // [0, ksplit) and from grp[1].tm_w after, when kgroups == 2; the rank
  // blocks then use grp[0]'s tm_b and n_extra.
  int kgroups;
  int ksplit;
  Schedule sched;
  int accumulate;        // out += acc_scale·result instead of overwrite (DX; FWD without RoPE)
  float acc_scale;
  // DX read-modify-write of the bf16 kernel under LoRA dropout: the added
  // result is masked by the dropout keep bits of the output element
  // (philox.cuh; element index row·drop_ld + column) and scaled by drop_scale
  int dropout;
  uint32_t drop_thresh;
  int drop_ld;
  float drop_scale;
  uint64_t drop_seed, drop_offset;
  // SwiGLU pair (FWD): n-tile t covers output columns [128t, 128t + 128);
  // CTA c of a pair stages the rows of grp[c] (0: gate, 1: up), so a
  // tile's accumulator holds g in columns [0, 128) and u in [128, 256).
  // The epilogue stores h = silu(g)·u through tm_h and, when save_gu, g
  // and u through grp[0].tm_out and grp[1].tm_out.
  int swiglu;
  int save_gu;
  CUtensorMap tm_h;
  // Down-projection in the GEMM (FWD, contiguous schedule): on the first
  // tile of each m-block's run of tiles the pair also forms v = x·Aᵀ
  // (N = fv_nv, the padded rank; CTA c stages rows [c·fv_nv/2, +fv_nv/2) of
  // [A1; A2] from tm_a[c] when fv_two, else from tm_a[0] at that row), and
  // stages s·v (scaled by fv_scale) in shared memory as the rank K-blocks'
  // activation for every tile of the run.
  CUtensorMap tm_a[2];
  int fv_nv;
  int fv_two;
  float fv_scale;
  // RoPE epilogue (FWD mode)
  const int32_t *positions;
  const float *cos_sin;
  int max_pos;
  uint32_t *status;
};

enum GemmMode { kModeFwd = 0, kModeDx = 1 };

// Launch bookkeeping around every kernel launch of the library:
// launch_begin() just before it, note_launch() just after (with the kernel's
// name and stream).  note_launch counts launches (lora_kernel_launch_count);
// while a timing session is open (lora_profile_begin) the pair records a
// timing event on the stream on each side of the launch.
void launch_begin(cudaStream_t st);
void note_launch(const char *name, cudaStream_t st);

// Launch with programmatic stream serialization (the kernel calls
// grid_dep_wait() before touching global memory), and optionally cluster
// dimensions (cluster_x > 0; kernels with compile-time cluster dimensions
// pass 0).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(const char *name, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, unsigned cluster_x, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  unsigned na = 0;
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  if (cluster_x > 0) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = cluster_x;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  launch_begin(st);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args...);
  note_launch(name, st);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// Two-SM (CTA pair) fused GEMM: (256·mb) x 256 tiles over `pairs` persistent
// pairs; p.sched counts tiles of mb m-blocks.  mb = 2 exists for NF4
// weights; fv = 64 / 128 (the 16-bit-W forward with the down-projection
// formed in the GEMM, v up to fv columns wide) needs p.sched.contiguous.
// F16: the 16-bit operands and outputs are fp16 (else bf16).
template <bool F16>
cudaError_t launch_gemm_pair_t(const GemmParams &p, int mode, bool rope, bool nf4, int mb, int fv,
                               int pairs, cudaStream_t st);
template <bool F16>
int gemm_pair_capacity_t(int mode, bool rope, bool nf4, int mb, int fv);

inline cudaError_t launch_gemm_pair(const GemmParams &p, int mode, bool rope, bool nf4, int mb,
                                    int fv, int pairs, bool f16, cudaStream_t st) {
  return f16 ? launch_gemm_pair_t<true>(p, mode, rope, nf4, mb, fv, pairs, st)
             : launch_gemm_pair_t<false>(p, mode, rope, nf4, mb, fv, pairs, st);
}
// max co-resident pairs (the same for both element types: one pair per two
// SMs, bounded by shared memory)
inline int gemm_pair_capacity(int mode, bool rope, bool nf4, int mb, int fv) {
  return gemm_pair_capacity_t<false>(mode, rope, nf4, mb, fv);
}

// Skinny rank-r products on the tensor cores:
//   KMAJOR  (v, u):  g[t][j] = Σ_c P[t,c]·Q[j,c]            P = x or dY, Q = A or Bᵀ
//   MNMAJOR (dA,dB): g[o][j] = Σ_t P[t,o]·(Qhi+Qlo)[j,t]    P = x or dY, Q = uᵀ or vᵀ
// Two schedules over the units (problem, 128-row output tile, 64-wide
// reduction chunk):
//   cluster (skinny.cu):    a cluster of `split` CTAs owns one tile and adds
//                           its partials over distributed shared memory;
//   stream-K (skinny_sk.cu): `ctas` equal contiguous unit ranges, one per CTA;
//                           a tile shared by several CTAs is finished by the
//                           one holding its first chunks, which adds the
//                           others' fp32 partials (parked in `partials`,
//                           announced in `flags`) in CTA order.
// Both sum in a fixed order (deterministic).  Output kinds (a bit set):
//   kOutVt:      gᵀ as bf16 hi + lo parts [RP, ld_t] (unscaled; the Q operand
//                of the MNMAJOR pass)
//   kOutRowBf16: scale·g as bf16 [rows, ld_row] (the rank K-block of the
//                fused GEMM)
//   kOutRowT:    out[j][o] = scale·g[o][j] fp32 (dA [r, k]); with nproj == 2
//                columns [r, 2r) go to out_f32b
//   kOutRow:     out[o][j] = scale·g[o][j] fp32 (dB [n, r]); with nproj == 2
//                rows >= split_row go to out_f32b from columns [r, 2r)
//   kOutT16:     out_bf16[j][o] = scale·g[o][j], 16-bit, columns j < r only
//                (the small-M forward's y [M, n] and s·v [M, r], ld_t = n or r)
enum SkinnyOut { kOutVt = 1, kOutRowBf16 = 2, kOutRowT = 4, kOutRow = 8, kOutT16 = 16 };

constexpr int kSkinnyMaxCtas = 160;  // scratch slots (the grid is at most one CTA per SM)

struct SkinnyProblem {
  CUtensorMap tm_p;
  CUtensorMap tm_q;      // Q (MNMAJOR: its hi part)
  CUtensorMap tm_q2;     // MNMAJOR: lo part; KMAJOR with q_rows1 > 0: Q rows [q_rows1, 2·q_rows1)
  int q_rows1;           // KMAJOR: rows taken from tm_q when Q comes from two tensors, else 0
  int q_rows;            // KMAJOR: rows of the RP-row Q tile the copies fill; the rest is zero
  // NF4 P (the decoding variant): tm_p maps the codes [rows, K/2] bytes
  // (box 32 x 128), absmax the bf16 block scales [rows, ld_absmax]
  int nf4;
  const __nv_bfloat16 *absmax;
  int ld_absmax;
  float *out_f32;
  float *out_f32b;
  uint16_t *out_hi;  // 16-bit words (bf16 or fp16, the kernel's type)
  uint16_t *out_lo;
  uint16_t *out_bf16;
  int ld_t;              // leading dimension of the kOutVt output
  int ld_row;            // leading dimension of the kOutRowBf16 output
  int out_kind;
  int r;                 // rank of one projection
  int nproj;             // 1, or 2 for two projections merged as rank 2r
  int split_row;         // kOutRow with nproj == 2: first output row of projection 1
  float scale;
  int rows;              // output rows
  int row_tiles;         // ceil(rows / 128)
  int chunks;            // 64-wide reduction chunks
  int tile_begin;        // cluster: first cluster of this problem
  long long unit_begin;  // stream-K: units of the problems before this one
};

// The output fields of a problem, copied into registers before the output
// stores.  Read through a runtime problem index, the kernel-parameter fields
// are memory loads, and an fp32 output store may alias the float `scale`
// field: read in place, each fp32 store is followed by a reload that waits
// on it (on B300 the finishing CTAs of the dA/dB pass spent 11-14 us in
// their stores that way, 6-8 us with the fields in registers).
struct SkinnyDest {
  float *out_f32, *out_f32b;
  uint16_t *out_hi, *out_lo, *out_bf16;
  int ld_t, ld_row, out_kind, r, nproj, split_row, rows;
  float scale;
};
#ifdef __CUDACC__
__device__ __forceinline__ SkinnyDest skinny_dest(const SkinnyProblem &P) {
  return {P.out_f32, P.out_f32b, P.out_hi, P.out_lo, P.out_bf16, P.ld_t,  P.ld_row,
          P.out_kind, P.r,      P.nproj,  P.split_row, P.rows, P.scale};
}
#endif

struct SkinnyParams {
  SkinnyProblem pr[2];
  int num_problems;
  int split;                   // cluster: CTAs per cluster (1, 2, 4 or 8)
  int ctas;                    // stream-K: grid size (<= kSkinnyMaxCtas, <= units)
  long long units;             // Σ row_tiles · chunks
  float *partials;             // [kSkinnyMaxCtas][RP][128] fp32: CTA c's parked partial
  unsigned long long *flags;   // [kSkinnyMaxCtas]: CTA c's partial of this launch is parked
  unsigned long long epoch;    // unique per launch (flags of other launches never match)
  uint32_t *status;
};

// f16: the 16-bit operands (P, Q) and outputs (hi/lo, kOutRowBf16) are fp16.
// dec: the NF4-decoding variant (KMAJOR, rp 64, 96 or 128; problems with `nf4`
// set stream codes through tm_p and absmax instead of P).
// two: the variant with half-depth rings that runs two CTAs per SM (KMAJOR,
// rp 64, no decode).
cudaError_t launch_skinny_cluster(const SkinnyParams &p, bool mn_major, int rp, bool f16,
                                  cudaStream_t st, bool dec = false, bool two = false);
// Largest `split` the cluster kernel supports for (mn_major, rp, dec, two)
// (its epilogue buffers must fit in its pipeline ring).
int skinny_max_split(bool mn_major, int rp, bool dec = false, bool two = false);
// Whether `split` CTAs per cluster is a valid cluster schedule for the pass.
bool skinny_split_ok(bool mn_major, int rp, bool dec, bool two, int split);
// Scratch of one stream-K launch: flags, then partials (256-byte aligned).
size_t skinny_scratch_bytes(int rp);
cudaError_t launch_skinny_sk(const SkinnyParams &p, bool mn_major, int rp, bool f16,
                             cudaStream_t st);

// Elementwise / small helpers.
// Backward set-up (one launch): inverse RoPE of dy1|dy2 into dy_out (when
// dy1 is set) or the SwiGLU backward [dg | du] into dy_out (when sw_dh is
// set), A_out = [A1; A2] (nproj == 2), Bt = diag(B1, B2)ᵀ.
struct BwdPrep {
  const uint16_t *dy1, *dy2;   // [M, n1], [M, n2]; dy1 null: no rotation
  // SwiGLU (sw_dh set, n1 == n2 == n): dy_out = [dg | du] from the incoming
  // dh and the saved gate / up outputs g, u [M, n]
  const uint16_t *sw_dh, *sw_g, *sw_u;
  uint16_t *dy_out;            // [M, n1 + n2]
  const int32_t *pos;
  const float *cos_sin;
  int max_pos;
  uint32_t *status;
  int M, n1, n2, k, r, nproj;       // n2 = 0 for one projection
  const uint16_t *A1, *A2;     // [r, k] each
  uint16_t *A_out;                  // [2r, k]
  const uint16_t *B1, *B2;     // [n1, r], [n2, r]
  uint16_t *Bt;                     // [nproj·r, n1 + n2]
};
cudaError_t launch_bwd_prep(const BwdPrep &p, bool f16, cudaStream_t st);
cudaError_t launch_rope_cache(float *cos_sin, int max_pos, int head_dim, double theta,
                              cudaStream_t st);
// LoRA dropout on x [M, k]: out = x ⊙ keep / q (keep per philox.cuh).
cudaError_t launch_dropout_x(const uint16_t *x, uint16_t *out, int M, int k, uint64_t seed,
                             uint64_t offset, uint32_t thresh, float inv_q, bool f16,
                             cudaStream_t st);
// Block scales of an NF4 weight [n, k] (nb = n·k/64 blocks of 64): bf16
// absmax [nb] (dq_scale null), or double-quantised (nf4_levels.cuh): E4M3
// codes [nb] in `absmax`, fp32 scale per 256 blocks, one fp32 offset.
struct Nf4Scales {
  const void *absmax;
  const float *dq_scale;
  const float *dq_offset;
};
// W [n, k] in the 16-bit type (f16: fp16, else bf16) from codes and scales.
cudaError_t launch_nf4_dequant(const uint8_t *codes, const Nf4Scales &sc, uint16_t *w, int n,
                               int k, bool f16, cudaStream_t st);
// Double-quantised scales decoded to bf16 absmax [nb] (nb % 8 == 0).
cudaError_t launch_nf4_dq_expand(const Nf4Scales &sc, uint16_t *absmax_out, size_t nb,
                                 cudaStream_t st);
// Quantise W [n, k] (16-bit type per f16): codes and bf16 absmax, or with
// dq_scale set, E4M3 scale codes in `absmax`, dq_scale [ceil(nb/256)] and
// *dq_offset (three launches).
cudaError_t launch_nf4_quantize(const uint16_t *w, uint8_t *codes, void *absmax, float *dq_scale,
                                float *dq_offset, int n, int k, bool f16, cudaStream_t st);

// Argument checks of lora_linear_bwd other than the workspace (shape limits,
// weight descriptor, pointer alignment, finite alpha), shared with
// lora_linear_bwd_noalloc so that both reject the same calls before
// touching the device.
lora_status_t check_bwd_args(const void *x, lora_weight_t W, const void *A, const void *B,
                             const void *dy, const void *dx, const float *dA, const float *dB,
                             int M, int k, int n, int r, float alpha);

// LORA_OK if the current device is an sm_103 part (else LORA_ERR_ARCH, or
// LORA_ERR_CUDA if the query fails).
lora_status_t check_current_device();

}  // namespace lora
