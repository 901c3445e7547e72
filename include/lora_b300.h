/*
 * lora_b300.h — C ABI of the fused LoRA / QLoRA projection library for
 * NVIDIA B300 (sm_103a).
 *
 * Sources of the operations (web pages about Unsloth, cited by title and
 * section):
 *   [P1] "UnSloth加速微调体验：在LoRA基础上再提速3倍的秘密":
 *        算子融合 (y = Wx + BAx computed in one pass, no intermediate in HBM),
 *        反向传播优化 (backward that recomputes Ax instead of caching it),
 *        RoPE缓存集成 (RoPE from a contiguous cos/sin cache applied inside the
 *        Q/K projection kernel).
 *   [P3] "Unsloth教程：本地微调大模型速度提升数倍，显存节省60%":
 *        显存优化策略 (QLoRA: frozen 4-bit NormalFloat4 base weight, only the
 *        adapter is trained).
 *   [QLoRA] Dettmers et al. 2023, §3 (the NF4 levels, and Double
 *        Quantization of the block scales; the pages only name the format).
 *
 * Conventions shared by every entry point
 *   - Row-major, contiguous tensors: x [M,k], W [n,k] (out x in), A [r,k],
 *     B [n,r], y and dY [M,n], dX [M,k], dA [r,k], dB [n,r].  The pages write
 *     column vectors (y = Wx + BAx); this is the same map in row form.
 *   - LoRA scale s = alpha / r multiplies the adapter branch.
 *   - x, W (dense form), A, B, y, dY, dX and every other 16-bit tensor of a
 *     call are of the call's 16-bit type, W.dtype: bfloat16 (the default) or
 *     float16 (the pages' API takes dtype = torch.float16 or torch.bfloat16,
 *     "UnSloth加速微调体验" usage example; "Unsloth自动化优化" §3.1 picks fp16
 *     where bf16 is unsupported).  dA, dB are float32; accumulation is
 *     float32 on the tensor cores; rounding to the 16-bit type is
 *     round-to-nearest-even.  fp16 has bf16's precision plus 3 bits but a
 *     range of ±65504: values past it become ±inf, as in any fp16 GEMM.
 *   - Every pointer is a DEVICE pointer owned by the caller, 16-byte
 *     aligned.  The library allocates no device memory (except the fixed
 *     scratch of lora_linear_bwd_noalloc) and keeps no state between calls
 *     other than per-device properties; TMA descriptors are encoded from
 *     the arguments on every call.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  Argument errors are returned before anything is
 *     launched.  LORA_ERR_CUDA reports a launch error seen immediately.
 *   - Device-side failures (an internal pipeline wait that exceeded its
 *     time limit, a position outside the RoPE cache) are recorded in a
 *     32-bit status word at the start of the caller's workspace; read it
 *     with lora_read_device_status() after the stream has finished.  The
 *     word is sticky: it is only cleared by lora_clear_device_status().
 *   - Shape limits: k % 64 == 0, n % 64 == 0, 1 <= M <= 2^30, r in
 *     {8, 16, 32, 64}, head_dim == 128; NF4 needs blocksize == 64.
 *   - Calls on the same workspace must not overlap on the GPU (use one
 *     stream, or one workspace per stream).  Every launch of a call goes to
 *     `stream`, in order.
 */
#ifndef LORA_B300_H
#define LORA_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without pulling in the CUDA headers. */
typedef struct CUstream_st *lora_stream_t;

typedef enum {
  LORA_OK = 0,
  LORA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad shape or value */
  LORA_ERR_UNSUPPORTED = 2, /* valid request outside the supported limits  */
  LORA_ERR_WORKSPACE = 3,   /* ws_bytes below lora_workspace_size()        */
  LORA_ERR_ARCH = 4,        /* current device is not sm_103                */
  LORA_ERR_CUDA = 5,        /* a CUDA runtime/driver call failed           */
  LORA_ERR_TIMEOUT = 6      /* device status: a pipeline wait timed out    */
} lora_status_t;

/* Bits of the device status word (see lora_read_device_status). */
#define LORA_DEVSTAT_TIMEOUT 0x1u     /* an mbarrier wait exceeded its limit */
#define LORA_DEVSTAT_BAD_POSITION 0x2u /* a RoPE position was outside [0,max_pos) */

/* Base weight descriptor (zero-initialise it, then set the fields).
 *   dtype: LORA_DTYPE_BF16 (0) or LORA_DTYPE_FP16 (1), the call's 16-bit type.
 *   type == LORA_WEIGHT_DENSE: w -> [n,k] of that type; absmax, absmax_scale,
 *     absmax_offset NULL; blocksize ignored.
 *   type == LORA_WEIGHT_NF4 : w -> uint8 codes [n, k/2] (byte j of a row holds
 *     element 2j in the high nibble, 2j+1 in the low nibble); blocksize must
 *     be 64; an element decodes to level[code] * absmax[block], rounded to
 *     the 16-bit type, with the 16 NF4 levels of [QLoRA].  The block scales
 *     (blocks numbered row-major, b = row·k/64 + j/64):
 *       absmax_scale == NULL: absmax -> bf16 [n·k/64].
 *       double quantisation ([QLoRA] §3; absmax_scale and absmax_offset
 *       both set): absmax -> uint8 E4M3 codes [n·k/64] (OCP FP8, 4 exponent
 *       bits, bias 7, 3 mantissa bits), absmax_scale -> float32
 *       [ceil(n·k/64 / 256)] (one per 256 consecutive blocks), absmax_offset
 *       -> one float32; block b's scale is
 *         bf16( e4m3(code[b]) · absmax_scale[b/256] + *absmax_offset )
 *       with the product and the sum each rounded to float32.  0.52 instead
 *       of 0.53 bytes per weight.
 *   Every pointer is 16-byte aligned. */
enum { LORA_WEIGHT_DENSE = 0, LORA_WEIGHT_NF4 = 1 };
#define LORA_WEIGHT_BF16 LORA_WEIGHT_DENSE /* earlier name of the dense type */
enum { LORA_DTYPE_BF16 = 0, LORA_DTYPE_FP16 = 1 };
typedef struct {
  int type;
  const void *w;
  const void *absmax;
  int blocksize;
  int dtype;
  const float *absmax_scale;
  const float *absmax_offset;
} lora_weight_t;

/* Operation ids for lora_workspace_size(). */
enum {
  LORA_OP_FWD = 0,
  LORA_OP_BWD = 1,
  LORA_OP_QK_ROPE_FWD = 2,
  LORA_OP_QK_ROPE_BWD = 3,
  LORA_OP_SWIGLU_FWD = 4,
  LORA_OP_SWIGLU_BWD = 5,
  LORA_OP_MERGE = 6,     /* pass M = 1 */
  LORA_OP_MERGE_NF4 = 7, /* pass M = 1 */
  LORA_OP_FWD_DROPOUT = 8,
  LORA_OP_BWD_DROPOUT = 9
};
/* OR'ed into the op of lora_workspace_size(): the call's NF4 weight (either
 * weight of a pair) has double-quantised block scales.  Adds room for their
 * bf16 expansion (n·k/32 bytes per weight), which the in-GEMM decode reads. */
#define LORA_OP_FLAG_DQ 0x100

/* Bytes of workspace an operation needs (always >= 256: the status word
 * lives at offset 0).  Besides the intermediates each call documents, every
 * operation holds a rank-pass scratch of 160 flags and 160 fp32 partials of
 * [r padded to 16/32/64/128, 128] (up to 10 MB), used when a rank pass runs
 * on its stream-K schedule.  A flag is matched against its launch's epoch (a
 * random per-process tag plus a launch counter) and cleared by the CTA that
 * consumes it, so stale or uninitialised workspace contents are not taken
 * for a new call's and a workspace needs no clearing between calls.  After
 * a call that reported LORA_ERR_TIMEOUT, zero the workspace before reusing
 * it (a partial parked after the timeout may have left its flag set for a
 * replay of the same launch).  For the q/k operations pass k = hidden and
 * n = (n_q_heads + n_kv_heads) * head_dim.  Returns 0 for an unknown op or
 * out-of-range sizes.  Pure host function. */
size_t lora_workspace_size(int op, int M, int k, int n, int r);

/* Room for NF4 weights staged in bf16 (n·k·2 bytes, 256-aligned).  An NF4
 * call (any of the forward and backward calls below) with M >= 2048 whose
 * workspace holds, past what lora_workspace_size() (plus the RoPE cache when
 * the call builds it) asks for, lora_nf4_stage_bytes() for each of its
 * weights (both weights of a q/k or gate/up pair, in that order), first
 * dequantises them there (nf4_dequant's rule) and then runs the bf16
 * kernels.  At that size the GEMMs are tensor-bound and the in-kernel
 * decode costs MMA throughput: on a B300, Qwen1.5-32B gate_proj at
 * M = 8192 ran forward 1.62 -> 1.38 ms and backward 2.31 -> 1.68 ms this way.
 * With a workspace of exactly lora_workspace_size(), or M < 2048, the NF4
 * codes are decoded inside the GEMMs while each W tile is staged.  Returns 0
 * for non-positive sizes. */
size_t lora_nf4_stage_bytes(int n, int k);

/* Fused forward, [P1] 算子融合:  y = x·Wᵀ + s·(x·Aᵀ)·Bᵀ.
 * Two launches.  The rank pass streams x once and writes the rank block
 * s·v = s·x·Aᵀ [M,r] (bf16, in the workspace: 2·M·r bytes, 1/(k/r) of x).
 * The fused GEMM then reduces each output tile over the concatenated axis
 * y = [x | s·v]·[W | B]ᵀ: base product and adapter land in the same fp32
 * tensor-memory accumulator before the single bf16 store of y, so neither
 * x·Wᵀ nor the adapter output goes to HBM.  An NF4 W is decoded tile by tile
 * in shared memory ([P3] 显存优化策略).
 * One launch when every 256 x 256 output tile has a CTA pair of its own and
 * W is 16-bit: s·x·Aᵀ is then formed inside the GEMM from the x tiles it
 * already holds and never leaves shared memory.
 * At M <= 128 the forward runs over the rows of W instead: one rank-pass
 * launch computes yᵀ = W·xᵀ and (s·v)ᵀ (NF4 codes decoded in that pass),
 * and a GEMM adds (s·v)·Bᵀ to y in its epilogue.
 *   x [M,k] bf16, W per lora_weight_t, A [r,k] bf16, B [n,r] bf16,
 *   y [M,n] bf16 (overwritten).  ws: >= lora_workspace_size(LORA_OP_FWD,...). */
lora_status_t lora_linear_fwd(const void *x, lora_weight_t W, const void *A,
                              const void *B, void *y, int M, int k, int n,
                              int r, float alpha, void *ws, size_t ws_bytes,
                              lora_stream_t stream);

/* Fused backward, [P1] 反向传播优化 (gradients derived from the forward; the
 * page's printed formulas have a garbled operand order and no scale):
 *   u  = dY·B, v = x·Aᵀ            (one rank pass; v recomputed, never cached)
 *   dX = [dY | s·u]·[W ; A]        (= dY·W + s·u·A; accumulate_dx != 0: dX += that)
 *   dA = s·uᵀ·x,   dB = s·dYᵀ·v    (one pass; overwritten, float32)
 * W is frozen: no weight gradient.  x [M,k], dy [M,n], dx [M,k] bf16;
 * dA [r,k], dB [n,r] float32.  ws: >= lora_workspace_size(LORA_OP_BWD,...). */
lora_status_t lora_linear_bwd(const void *x, lora_weight_t W, const void *A,
                              const void *B, const void *dy, void *dx,
                              int accumulate_dx, float *dA, float *dB, int M,
                              int k, int n, int r, float alpha, void *ws,
                              size_t ws_bytes, lora_stream_t stream);

/* q/k projections with RoPE, [P1] RoPE缓存集成: q = R(pos)·(x·Wqᵀ + s·(x·Aqᵀ)·Bqᵀ)
 * and the same for k: one rank pass for both (s·x·[Aq; Ak]ᵀ, [M,2r] in the
 * workspace), then ONE fused GEMM launch over both weights.
 * The rotation is applied in the epilogue to each 128-wide head, pairing
 * columns (i, i+64): y'[i] = y[i]·cos − y[i+64]·sin, y'[i+64] = y[i+64]·cos +
 * y[i]·sin, angle = pos[m]·theta^(−2i/128).
 *   x [M,hidden]; q [M, n_q_heads*128]; k_out [M, n_kv_heads*128] (bf16).
 *   positions int32 [M], each in [0, max_pos).
 *   cos_sin_cache float32 [max_pos, head_dim]: row p holds cos of the 64
 *     angles then their sin (see lora_rope_cache_build).  If NULL the call
 *     first builds it from rope_theta inside the workspace, which then needs
 *     lora_rope_cache_bytes(max_pos, head_dim) more bytes. */
lora_status_t lora_qk_rope_fwd(const void *x, lora_weight_t Wq, const void *Aq,
                               const void *Bq, lora_weight_t Wk, const void *Ak,
                               const void *Bk, void *q, void *k_out, int M,
                               int hidden, int n_q_heads, int n_kv_heads,
                               int head_dim, int r, float alpha,
                               double rope_theta, const int32_t *positions,
                               const float *cos_sin_cache, int max_pos,
                               void *ws, size_t ws_bytes, lora_stream_t stream);

/* Backward of lora_qk_rope_fwd: the incoming dq, dk are rotated back by the
 * transposed rotation R(pos)ᵀ into one [M, nq+nk] gradient; q and k then
 * run as ONE projection of rank 2r (A = [Aq; Ak], B = diag(Bq, Bk), exact)
 * through the passes of lora_linear_bwd, with dX reduced over [Wq; Wk] in
 * one GEMM (accumulate_dx != 0: dX += the sum).  dAq, dBq, dAk, dBk float32, overwritten.  Cache rules as in
 * lora_qk_rope_fwd. */
lora_status_t lora_qk_rope_bwd(const void *x, lora_weight_t Wq, const void *Aq,
                               const void *Bq, lora_weight_t Wk, const void *Ak,
                               const void *Bk, const void *dq, const void *dk,
                               void *dx, int accumulate_dx, float *dAq,
                               float *dBq, float *dAk, float *dBk, int M,
                               int hidden, int n_q_heads, int n_kv_heads,
                               int head_dim, int r, float alpha,
                               double rope_theta, const int32_t *positions,
                               const float *cos_sin_cache, int max_pos,
                               void *ws, size_t ws_bytes, lora_stream_t stream);

/* LoRA dropout on the adapter's input ([P2] "微调太慢？试试Unsloth" §3.3 table,
 * row E: lora_dropout 0.05; [P4] §2.2: lora_dropout=0.1): the base product
 * sees x, the adapter x̃ = x ⊙ keep / q.
 *   y = x·Wᵀ + s·(x̃·Aᵀ)·Bᵀ.
 * The mask is drawn from Philox4x64-10 (Salmon et al. 2011) and never
 * stored: element e = i·k + j of x takes 16-bit number e mod 16 of the block
 * with counter (e/16, offset, 0, 0) and key (seed, 0), and is kept iff that
 * number is >= round(dropout_p·65536); q = 1 − round(dropout_p·65536)/65536.
 * Pass the same (seed, offset) to the backward; change offset every step.
 * dropout_p in [0, 1).  Three launches: x̃ into the workspace (bf16), the rank
 * pass over x̃, the fused GEMM.
 *   ws: >= lora_workspace_size(LORA_OP_FWD_DROPOUT, M, k, n, r). */
lora_status_t lora_linear_fwd_dropout(const void *x, lora_weight_t W, const void *A,
                                      const void *B, void *y, int M, int k, int n,
                                      int r, float alpha, float dropout_p,
                                      uint64_t seed, uint64_t offset, void *ws,
                                      size_t ws_bytes, lora_stream_t stream);

/* Backward of lora_linear_fwd_dropout, the mask regenerated from (seed,
 * offset):  u = dY·B,  dX = dY·W + s·(u·A) ⊙ keep / q,  dA = s·uᵀ·x̃,
 * dB = s·dYᵀ·(x̃·Aᵀ) (x̃·Aᵀ recomputed).  dX's adapter term is its own K = r
 * tensor-core pass whose read-modify-write epilogue applies the mask.
 *   ws: >= lora_workspace_size(LORA_OP_BWD_DROPOUT, M, k, n, r). */
lora_status_t lora_linear_bwd_dropout(const void *x, lora_weight_t W, const void *A,
                                      const void *B, const void *dy, void *dx,
                                      int accumulate_dx, float *dA, float *dB, int M,
                                      int k, int n, int r, float alpha, float dropout_p,
                                      uint64_t seed, uint64_t offset, void *ws,
                                      size_t ws_bytes, lora_stream_t stream);

/* Gate and up projections of an MLP joined by SwiGLU, [P4] "Unsloth框架：
 * 高效LLM微调与LoRA优化实践" §3.1 计算图重写引擎 (adjacent linear layers merged
 * with their activation) and [P5] "Unsloth自动化优化" §1 模型结构自识别
 * (SwiGLU); SwiGLU itself as in Shazeer 2020, "GLU Variants Improve
 * Transformer" §2, since the pages only name it:
 *   g = x·Wgᵀ + s·(x·Agᵀ)·Bgᵀ,  u = x·Wuᵀ + s·(x·Auᵀ)·Buᵀ,
 *   h = silu(g)·u = g·u / (1 + e^(−g)).
 * One rank pass for both adapters (s·x·[Ag; Au]ᵀ, [M,2r] in the workspace),
 * then ONE fused GEMM launch over both weights: each CTA pair computes 128
 * columns of g and the same 128 of u into one accumulator and writes h
 * from its epilogue, so neither g nor u needs a second pass.
 *   x [M,k]; Wg, Wu [n,k] (both bf16 or both NF4); Ag, Au [r,k]; Bg, Bu [n,r];
 *   h [M,n] bf16 (the input of down_proj).  g, u [M,n] bf16 receive the
 *   pre-activation outputs, which lora_swiglu_bwd needs; pass both NULL to
 *   skip them (inference).
 *   ws: >= lora_workspace_size(LORA_OP_SWIGLU_FWD, M, k, n, r). */
lora_status_t lora_swiglu_fwd(const void *x, lora_weight_t Wg, const void *Ag,
                              const void *Bg, lora_weight_t Wu, const void *Au,
                              const void *Bu, void *h, void *g, void *u, int M,
                              int k, int n, int r, float alpha, void *ws,
                              size_t ws_bytes, lora_stream_t stream);

/* Backward of lora_swiglu_fwd for an incoming dh [M,n], from the saved g, u:
 *   dg = dh·u·σ(g)·(1 + g·(1 − σ(g))),  du = dh·g·σ(g)   (σ = sigmoid, one
 *   elementwise pass, rounded to bf16), then gate and up run as ONE
 *   projection of rank 2r (A = [Ag; Au], B = diag(Bg, Bu), dY = [dg | du])
 *   through the passes of lora_linear_bwd, with dX reduced over [Wg; Wu] in
 *   one GEMM (accumulate_dx != 0: dX += the sum).  dAg, dBg, dAu, dBu float32,
 *   overwritten.  ws: >= lora_workspace_size(LORA_OP_SWIGLU_BWD, M, k, n, r). */
lora_status_t lora_swiglu_bwd(const void *x, lora_weight_t Wg, const void *Ag,
                              const void *Bg, lora_weight_t Wu, const void *Au,
                              const void *Bu, const void *g, const void *u,
                              const void *dh, void *dx, int accumulate_dx,
                              float *dAg, float *dBg, float *dAu, float *dBu,
                              int M, int k, int n, int r, float alpha, void *ws,
                              size_t ws_bytes, lora_stream_t stream);

/* lora_linear_bwd without a workspace argument, for callers that cannot
 * allocate device memory where they run the backward (a plugin inside another
 * framework's runtime that is handed only its tensors; a latency-critical
 * loop that must not enter the driver's allocator).  The pages have no
 * counterpart: this is a packaging of lora_linear_bwd, same arguments and
 * results, minus ws/ws_bytes.
 *   Scratch: one fixed 32 MiB array in the library's device memory, held on
 *     every GPU that loads the library until the process exits.  Shapes
 *     needing more (lora_workspace_size(LORA_OP_BWD, ...) > 32 MiB) return
 *     LORA_ERR_WORKSPACE before any launch.
 *   The first call on a device looks up the array's address for that device
 *     (make it before any stream capture).  Calls share the array: calls
 *     that overlap on the GPU race and must be serialised.  Device-side
 *     timeouts are recorded in the array and not reported here. */
lora_status_t lora_linear_bwd_noalloc(const void *x, lora_weight_t W, const void *A,
                                      const void *B, const void *dy, void *dx,
                                      int accumulate_dx, float *dA, float *dB, int M, int k,
                                      int n, int r, float alpha, lora_stream_t stream);

/* Merge the adapter into its base weight for inference, or take it back out:
 * W <- W + sign·s·B·A (sign = +1 merge, -1 unmerge), s = alpha/r.  [P2]
 * "微调太慢？试试Unsloth" §5.1 (for_inference folds the LoRA weights into the
 * main weight so no adapter runs at generation time) and [P5] §3.2 (the
 * "A@B + original_weight" kernel).  In place, through W's pointers (the
 * descriptor's const qualifiers notwithstanding).  A [r,k], B [n,r] of
 * W.dtype.  n % 64 == 0, k % 64 == 0.
 *   Dense W [n,k]: B·A runs on the tensor cores (K = r) and each W element
 *   is read and written once (rounded once to W.dtype).
 *     ws: >= lora_workspace_size(LORA_OP_MERGE, 1, k, n, r) (status word).
 *   NF4 W: dequantised into the workspace (nf4_dequant's rule), merged
 *   there, and quantised back into the codes and block scales in place
 *   (nf4_quantize's rule, with double quantisation when W has it).  The
 *   merged weight is not representable in the old codes, so it is
 *   re-quantised; merging then unmerging returns a weight within NF4's
 *   quantisation error of the original, not the original codes.
 *     ws: >= lora_workspace_size(LORA_OP_MERGE_NF4, 1, k, n, r) (2·n·k
 *     bytes plus the status word). */
lora_status_t lora_merge(lora_weight_t W, const void *A, const void *B, int n,
                         int k, int r, float alpha, int sign, void *ws,
                         size_t ws_bytes, lora_stream_t stream);

/* Standalone NF4 dequantisation ([P3] 显存优化策略, [QLoRA] §3) of an NF4
 * descriptor (either scale form):
 *   w_out[i,j] = dtype( level[code(i,j)] * scale[block(i,j)] ), product in
 *   fp32, w_out [n,k] of W.dtype.  k % 64 == 0. */
lora_status_t nf4_dequant(lora_weight_t W, void *w_out, int n, int k,
                          lora_stream_t stream);

/* NF4 quantisation of a 16-bit w [n,k] of W_out.dtype into W_out's codes
 * and block scales (written through its pointers; type NF4, blocksize 64):
 *   absmax_scale NULL: absmax = bf16(max|w|) per 64-block (round to nearest
 *     even); code = index of the nearest level to w/absmax decided in IEEE
 *     fp32 (w/absmax clamped to [-1, 1]; ties to the lower index; absmax 0
 *     gives code 7, the exact zero).  One launch.
 *   double quantisation (absmax_scale, absmax_offset set; [QLoRA] §3):
 *     c[b] = max|w| of block b (exact in fp32); *absmax_offset = fp32 of the
 *     mean of all c[b]; per group G of 256 blocks, absmax_scale[G] =
 *     fp32( max_G |fp32(c[b] - offset)| / 448 ); code[b] = E4M3 of
 *     fp32((c[b] - offset) / scale) (round to nearest even; 0 when the
 *     group's scale is 0); then the NF4 codes as above against the scale
 *     code[b] decodes to (lora_weight_t).  Three launches.
 * k % 64 == 0; with double quantisation also n·k/64 % 16 == 0 (true
 * whenever n % 16 == 0). */
lora_status_t nf4_quantize(const void *w, lora_weight_t W_out, int n, int k,
                           lora_stream_t stream);

/* Bytes of a cos/sin cache for max_pos positions. */
size_t lora_rope_cache_bytes(int max_pos, int head_dim);

/* Build the contiguous RoPE cache ([P1] RoPE缓存集成): cos_sin [max_pos,
 * head_dim] float32, row p = cos(p·f_i) for i < head_dim/2, then sin(p·f_i),
 * f_i = theta^(−2i/head_dim).  Angles and trigonometry in fp64, stored
 * rounded to fp32. */
lora_status_t lora_rope_cache_build(float *cos_sin, int max_pos, int head_dim,
                                    double theta, lora_stream_t stream);

/* Synchronise `stream`, then copy the device status word at the start of
 * `ws` to *status_out (0 = no device-side failure).  Returns
 * LORA_ERR_TIMEOUT if the timeout bit is set, else LORA_OK (or
 * LORA_ERR_CUDA). */
lora_status_t lora_read_device_status(const void *ws, uint32_t *status_out,
                                      lora_stream_t stream);

/* Zero the device status word (asynchronous on `stream`). */
lora_status_t lora_clear_device_status(void *ws, lora_stream_t stream);

/* Number of kernels this library has launched in the calling process
 * (monotonic; a diagnostic for counting launches per step). */
uint64_t lora_kernel_launch_count(void);

/* Per-launch timing, a diagnostic (no counterpart in the pages): while a
 * session is open, each of the library's next `capacity` kernel launches (any
 * entry point, any stream) is bracketed by two timing events recorded on its
 * stream, one just before and one just after the launch, so the time between
 * them is that kernel's run time (it also keeps the kernel from starting
 * early under the previous one, which the library otherwise allows).
 * lora_profile_begin creates the 2*capacity events (host-side CUDA objects,
 * no device memory) and returns LORA_ERR_INVALID_ARG if a session is already
 * open or capacity is outside [1, 65536].  lora_profile_end waits for the
 * recorded events, writes the kernel name (a static string) and time in ms
 * of the first min(launches, capacity) launches, in launch order, to
 * names/ms, sets *count, destroys the events and closes the session.  One
 * session per process, driven from one host thread; do not capture the
 * library's launches into a CUDA graph while it is open. */
lora_status_t lora_profile_begin(int capacity);
lora_status_t lora_profile_end(const char **names, float *ms, int capacity, int *count);

/* Human-readable name of a status code. */
const char *lora_status_string(lora_status_t s);

#ifdef __cplusplus
}
#endif

#endif /* LORA_B300_H */
