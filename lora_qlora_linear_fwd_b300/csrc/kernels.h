// Internal interface between the C-ABI host code (api.cu) and the kernels.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace lora {

// One projection inside a fused GEMM launch.
//   FWD mode: W [n,k] bf16 (K-major operand), r1 = A [r,k] (down-projection
//             operand), r2 = B [n,r] (up-projection operand), out = y [M,n].
//   DX  mode: W [n,k] bf16 read as an MN-major operand (dY·W), r1 = Bᵀ [r,n]
//             (u = dY·B), r2 = A [r,k] read MN-major (s·u·A), out = dX [M,k].
// NF4 weights: tm_w maps the codes [n, k/2] bytes and absmax points at the
// bf16 block scales [n, k/64].
struct alignas(64) GemmGroup {
  CUtensorMap tm_w;
  CUtensorMap tm_r1;
  CUtensorMap tm_r2;
  __nv_bfloat16 *out;
  const __nv_bfloat16 *absmax;
  int ncols;       // output columns of this group (n in FWD, k in DX)
  int n_tiles;     // ceil(ncols / 256)
  int tile_begin;  // first global n-tile index of this group
  int ld_absmax;   // k / 64 (NF4)
};

struct alignas(64) GemmParams {
  CUtensorMap tm_act;  // x [M,k] (FWD) or dY [M,n] (DX): K-major, box 64 x 128
  GemmGroup grp[kMaxGroups];
  int num_groups;
  int M;
  int K;          // reduction length: k (FWD) or n (DX)
  float scale;    // s = alpha / r
  // Two projections sharing x as ONE projection of rank 2r (A = [A1; A2],
  // B = diag(B1, B2)): the rank accumulator is formed once per m-block
  // rather than again at the group switch.
  int merged_rank;
  // DX mode: W rows (the reduction) come from grp[0].tm_w for 64-chunks
  // [0, ksplit) and from grp[1].tm_w after, when kgroups == 2.
  int kgroups;
  int ksplit;
  Schedule sched;
  // DX mode
  __nv_bfloat16 *ut_hi;  // uᵀ [RP, M] high bf16 part (unscaled), written once per m-block
  __nv_bfloat16 *ut_lo;  // uᵀ low part: u - hi
  int accumulate;        // dX += result instead of overwrite
  // RoPE epilogue (FWD mode)
  const int32_t *positions;
  const float *cos_sin;
  int max_pos;
  uint32_t *status;
};

enum GemmMode { kModeFwd = 0, kModeDx = 1 };

// Count of kernel launches issued by the library (see lora_kernel_launch_count).
void note_launch();

cudaError_t launch_gemm(const GemmParams &p, int mode, int rp, bool rope, bool nf4, int grid,
                        cudaStream_t st);
// Two-SM (CTA pair) variant: 256 x 256 tiles, m-blocks of 256 rows, rp 32 or 64.
cudaError_t launch_gemm_pair(const GemmParams &p, int mode, int rp, bool rope, bool nf4,
                             int pairs, cudaStream_t st);
int gemm_pair_capacity(int mode, int rp, bool rope, bool nf4);  // max co-resident pairs

// Skinny rank-r GEMMs on the tensor cores, reduced over K-slices in-kernel:
//   KMAJOR  (v):     v[t][j]   = Σ_c P[t,c]·Q[j,c]             P = x [T,k], Q = A
//   MNMAJOR (dA,dB): g[o][j]   = Σ_t P[t,o]·(Qhi+Qlo)[j,t]     P = x or dY
// Every CTA writes the fp32 partial of its slice; the last CTA to finish a
// row tile (atomic counter) adds the slices in slice order (deterministic)
// and writes the final output:
//   kOutVt:   vᵀ as bf16 hi/lo [RP, ld] (the operand of the dB pass)
//   kOutRowT: out[j][o] = scale·g[o][j], j < r   (dA [r, k]); merged q/k:
//             columns [r, 2r) go to out_f32b
//   kOutRow:  out[o][j] = scale·g[o][j], j < r   (dB [n, r]); merged q/k:
//             rows >= split_row go to out_f32b from columns [r, 2r)
enum SkinnyOut { kOutVt = 0, kOutRowT = 1, kOutRow = 2 };

struct alignas(64) SkinnyProblem {
  CUtensorMap tm_p;
  CUtensorMap tm_q_hi;
  CUtensorMap tm_q_lo;
  float *part;           // [row_tiles, max_segs, 128, RP] fp32 partials
  uint32_t *counter;     // [row_tiles] arrival counters (zero on entry, reset on exit)
  float *out_f32;        // kOutRowT / kOutRow: projection 0
  float *out_f32b;       // kOutRowT / kOutRow: projection 1 (merged q/k), else null
  __nv_bfloat16 *out_hi; // kOutVt
  __nv_bfloat16 *out_lo;
  int out_kind;
  int out_ld;            // leading dimension of the vᵀ output (Mp)
  int r;                 // rank of one projection (columns written per projection)
  int nproj;             // 1, or 2 for two projections merged as rank 2r
  int split_row;         // kOutRow with nproj == 2: first output row of projection 1
  float scale;
  int rows;              // output rows (T for KMAJOR, Mo for MNMAJOR)
  int row_tiles;         // ceil(rows / 128)
  int chunks;            // 64-wide reduction chunks per row tile
  int max_segs;          // most CTAs that can share one row tile
};

struct alignas(64) SkinnyParams {
  SkinnyProblem pr[2];
  int num_problems;
  long long total_items;  // Σ row_tiles · chunks over the problems
  uint32_t *status;
};

// Persistent CTAs of the skinny kernel (one per SM of a B300); the workspace
// plan depends on it, so it is a constant rather than a device query.
constexpr int kSkinnyCtas = 148;

cudaError_t launch_skinny(const SkinnyParams &p, bool mn_major, int rp, int grid, cudaStream_t st);

// Elementwise / small helpers.
cudaError_t launch_transpose_rank(const __nv_bfloat16 *B, __nv_bfloat16 *Bt, int n, int r,
                                  cudaStream_t st);
cudaError_t launch_rope_bwd(const __nv_bfloat16 *dy, __nv_bfloat16 *out, int M, int ncols,
                            int out_ld, const int32_t *pos, const float *cos_sin, int max_pos,
                            uint32_t *status, cudaStream_t st);
cudaError_t launch_blockdiag_rank(const __nv_bfloat16 *B1, const __nv_bfloat16 *B2,
                                  __nv_bfloat16 *out, int n1, int n2, int r, bool transpose,
                                  cudaStream_t st);
cudaError_t launch_rope_cache(float *cos_sin, int max_pos, int head_dim, double theta,
                              cudaStream_t st);
cudaError_t launch_nf4_dequant(const uint8_t *codes, const __nv_bfloat16 *absmax,
                               __nv_bfloat16 *w, int n, int k, cudaStream_t st);
cudaError_t launch_nf4_quantize(const __nv_bfloat16 *w, uint8_t *codes, __nv_bfloat16 *absmax,
                                int n, int k, cudaStream_t st);

}  // namespace lora
