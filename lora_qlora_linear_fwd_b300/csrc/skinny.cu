// Rank-r passes ("UnSloth加速微调体验" §算子融合, §反向传播优化):
//   forward   s·v = s·x·Aᵀ                      (KMAJOR: reduce over k)
//   backward  v = x·Aᵀ (recomputed), u = dY·B     (KMAJOR: reduce over k or n)
//             dA = s·uᵀ·x, dB = s·dYᵀ·v          (MNMAJOR: reduce over tokens)
//
// These stream x or dY once and are HBM-bound, so the kernel keeps HBM busy
// and avoids any traffic beyond the stream.  A cluster of `split` CTAs owns
// one 128-row output tile; each CTA streams its slice of the 64-wide
// reduction chunks through a deep TMA ring into one TMEM accumulator
// [128 x RP].  The non-leader CTAs then park their fp32 partials in their
// own (now idle) shared memory and the leader adds them over the cluster's
// distributed shared memory in cluster-rank order, so the result is
// deterministic and never round-trips through global memory.  In MNMAJOR
// mode the right-hand operand comes as bf16 hi + lo parts of an fp32 value
// (about 2^-17 relative) and both are multiplied, keeping near-fp32
// accuracy for dA and dB.
#include "kernels.h"

namespace lora {

template <bool MN, int RP>
struct SkinnySmem {
  static constexpr int P_BYTES = 128 * 128;  // [128 x 64] bf16 either way
  static constexpr int Q_BYTES = RP * 128;
  static constexpr int STAGE_BYTES = P_BYTES + (MN ? 2 : 1) * Q_BYTES;
  static constexpr int STAGES_FIT = (kSmemLimit - 4096) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 10 ? 10 : STAGES_FIT;
  // fp32 partial of a non-leader CTA: 128 rows, padded by 16 bytes so that
  // the rows of one 16-byte access pattern fall in different banks
  static constexpr int RED_STRIDE = RP * 4 + 16;
  static constexpr int RED_BYTES = 128 * RED_STRIDE;
  static constexpr int OFF_MISC = STAGES * STAGE_BYTES;
  static constexpr int TOTAL = OFF_MISC + 512 + 1024;
  static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");
  static_assert(STAGES >= 4, "pipeline depth");
  static_assert(RED_BYTES <= OFF_MISC, "partial fits in the ring");
  static_assert(TOTAL <= kSmemLimit, "shared memory budget");
};

// Columns [j0, j0+16) of output row `orow` (raw sums v) in every output
// form the problem asks for.
LORA_DEV void skinny_store16(const SkinnyProblem &P, int orow, int j0, const float (&v)[16]) {
  if (orow >= P.rows) return;
  const int cols = P.nproj * P.r;  // valid rank columns
  if (P.out_kind & kOutVt) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const __nv_bfloat16 hi = __float2bfloat16_rn(v[j]);
      P.out_hi[(size_t)(j0 + j) * P.ld_t + orow] = hi;
      P.out_lo[(size_t)(j0 + j) * P.ld_t + orow] = __float2bfloat16_rn(v[j] - __bfloat162float(hi));
    }
  }
  if (P.out_kind & kOutRowBf16) {
    __nv_bfloat16 *dst = P.out_bf16 + (size_t)orow * P.ld_row + j0;
    if (j0 + 16 <= cols) {
      uint4 w0, w1;
      w0.x = pack_bf16x2(v[0] * P.scale, v[1] * P.scale);
      w0.y = pack_bf16x2(v[2] * P.scale, v[3] * P.scale);
      w0.z = pack_bf16x2(v[4] * P.scale, v[5] * P.scale);
      w0.w = pack_bf16x2(v[6] * P.scale, v[7] * P.scale);
      w1.x = pack_bf16x2(v[8] * P.scale, v[9] * P.scale);
      w1.y = pack_bf16x2(v[10] * P.scale, v[11] * P.scale);
      w1.z = pack_bf16x2(v[12] * P.scale, v[13] * P.scale);
      w1.w = pack_bf16x2(v[14] * P.scale, v[15] * P.scale);
      reinterpret_cast<uint4 *>(dst)[0] = w0;
      reinterpret_cast<uint4 *>(dst)[1] = w1;
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (j0 + j < cols) dst[j] = __float2bfloat16_rn(v[j] * P.scale);
    }
  }
  if (P.out_kind & kOutRowT) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int jg = j0 + j;
      if (jg < cols) {
        const int pr = jg / P.r, jj = jg % P.r;
        float *out = pr ? P.out_f32b : P.out_f32;
        out[(size_t)jj * P.rows + orow] = v[j] * P.scale;
      }
    }
  }
  if (P.out_kind & kOutRow) {
    // dB: only the diagonal block of a merged pair is a real gradient
    const int pr = (P.nproj > 1 && orow >= P.split_row) ? 1 : 0;
    const int lo = pr * P.r;
    if (j0 + 16 <= lo || j0 >= lo + P.r) return;
    float *out = (pr ? P.out_f32b : P.out_f32) + (size_t)(orow - pr * P.split_row) * P.r;
    if (j0 >= lo && j0 + 16 <= lo + P.r) {
      float4 *dst = reinterpret_cast<float4 *>(out + (j0 - lo));
#pragma unroll
      for (int j = 0; j < 4; ++j)
        dst[j] = make_float4(v[4 * j] * P.scale, v[4 * j + 1] * P.scale, v[4 * j + 2] * P.scale,
                             v[4 * j + 3] * P.scale);
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (j0 + j >= lo && j0 + j < lo + P.r) out[j0 + j - lo] = v[j] * P.scale;
    }
  }
}

template <bool MN, int RP>
__global__ void __launch_bounds__(192, 1) lora_skinny_kernel(const __grid_constant__ SkinnyParams p) {
  using L = SkinnySmem<MN, RP>;
  constexpr int STAGES = L::STAGES;
  constexpr uint32_t kTmemCols = RP >= 32 ? RP : 32;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_addr(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (base - raw_base);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  const int S = p.split;
  const int cid = blockIdx.x / S;
  const int srank = blockIdx.x % S;  // this CTA's rank in the cluster
  const int pi = (p.num_problems > 1 && cid >= p.pr[1].tile_begin) ? 1 : 0;
  const SkinnyProblem &P = p.pr[pi];
  const int rt = cid - P.tile_begin;
  const int c_begin = (int)((long long)P.chunks * srank / S);
  const int c_end = (int)((long long)P.chunks * (srank + 1) / S);

  const uint32_t bar_full = base + L::OFF_MISC;
  const uint32_t bar_empty = bar_full + 8 * STAGES;
  const uint32_t bar_acc_full = bar_empty + 8 * STAGES;
  const uint32_t bar_drain = bar_acc_full + 8;
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::OFF_MISC + 8 * (2 * STAGES + 2));
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_acc_full, 1);
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_holder), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&P.tm_p);
      int stage = 0;
      uint32_t phase = 0;
      int fills[STAGES];
      for (int s = 0; s < STAGES; ++s) fills[s] = 0;
      for (int c = c_begin; c < c_end; ++c) {
        if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1u, abort_flag, p.status)) break;
        const uint32_t sp = base + stage * L::STAGE_BYTES;
        const uint32_t sq = sp + L::P_BYTES;
        const uint32_t fb = bar_full + 8 * stage;
        mbar_arrive_expect_tx(fb, L::STAGE_BYTES);
        if constexpr (MN) {
          // P [tokens, rows]: two boxes of [64 rows-of-output x 64 tokens]
          tma_load_2d(sp, &P.tm_p, fb, rt * 128, c * 64);
          tma_load_2d(sp + 8192, &P.tm_p, fb, rt * 128 + 64, c * 64);
          tma_load_2d(sq, &P.tm_q, fb, c * 64, 0);
          tma_load_2d(sq + L::Q_BYTES, &P.tm_q2, fb, c * 64, 0);
        } else {
          tma_load_2d(sp, &P.tm_p, fb, c * 64, rt * 128);
          if (P.q_rows1 > 0) {  // Q = [Q1; Q2] from two tensors
            tma_load_2d(sq, &P.tm_q, fb, c * 64, 0);
            tma_load_2d(sq + P.q_rows1 * 128, &P.tm_q2, fb, c * 64, 0);
          } else {
            tma_load_2d(sq, &P.tm_q, fb, c * 64, 0);
          }
        }
        ++fills[stage];
        if (++stage == STAGES) stage = 0, phase ^= 1u;
      }
      // drain: every issued copy has been consumed before the CTA may exit
      const uint64_t lim = *abort_flag ? 20000000ull : 1000000000ull;
      for (int s = 0; s < STAGES; ++s)
        if (fills[s] > 0) mbar_wait_quiet(bar_empty + 8 * s, (uint32_t)((fills[s] - 1) & 1), lim);
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc_bf16(128, RP, MN, false);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int c = c_begin; c < c_end; ++c) {
        if (!mbar_wait(bar_full + 8 * stage, phase, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sp = base + stage * L::STAGE_BYTES;
        const uint32_t sq = sp + L::P_BYTES;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint32_t accum = (c != c_begin || ks != 0) ? 1u : 0u;
          uint64_t da;
          if constexpr (MN)
            da = make_sdesc(sp + ks * 2048, 8192, 1024, kSw128);
          else
            da = make_sdesc(sp + ks * 32, 16, 1024, kSw128);
          tc_mma(tmem, da, make_sdesc(sq + ks * 32, 16, 1024, kSw128), idesc, accum);
          if constexpr (MN)
            tc_mma(tmem, da, make_sdesc(sq + L::Q_BYTES + ks * 32, 16, 1024, kSw128), idesc, 1u);
        }
        tc_commit(bar_empty + 8 * stage);
        if (++stage == STAGES) stage = 0, phase ^= 1u;
      }
      if (ok) tc_commit(bar_acc_full);
      if (*abort_flag) {
        tc_commit(bar_drain);
        mbar_wait_quiet(bar_drain, 0, 100000000ull);
      }
    }
  }

  // ---------------------------------------------- epilogue (warps 2-5)
  const bool epi = warp >= 2;
  const int row = (warp & 3) * 32 + lane;
  const uint32_t t_lane = (uint32_t)((warp & 3) * 32) << 16;
  const uint32_t my_red = base + row * L::RED_STRIDE;
  bool acc_ok = false;
  if (epi) {
    acc_ok = __all_sync(0xffffffffu, mbar_wait(bar_acc_full, 0, abort_flag, p.status));
    if (acc_ok) tc_fence_after();
    if (acc_ok && srank != 0) {
      // park the partial: the ring is idle (every MMA reading it completed)
#pragma unroll 1
      for (int c = 0; c < RP / 16; ++c) {
        uint32_t r[16];
        tmem_ld16(tmem + t_lane + c * 16, r);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 4; ++j)
          st_shared_v4(my_red + c * 64 + j * 16, r[4 * j], r[4 * j + 1], r[4 * j + 2],
                       r[4 * j + 3]);
      }
    }
  }
  __syncwarp();
  if (S > 1) cluster_sync_all();  // partials visible to the leader
  if (epi && srank == 0 && acc_ok) {
    const int orow = rt * 128 + row;
#pragma unroll 1
    for (int c = 0; c < RP / 16; ++c) {
      uint32_t r[16];
      tmem_ld16(tmem + t_lane + c * 16, r);
      tmem_ld_wait();
      float v[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
      for (int s = 1; s < S; ++s) {
        const uint32_t src = map_shared_rank(my_red + c * 64, (uint32_t)s);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float4 t = ld_shared_cluster_v4(src + j * 16);
          v[4 * j] += t.x;
          v[4 * j + 1] += t.y;
          v[4 * j + 2] += t.z;
          v[4 * j + 3] += t.w;
        }
      }
      skinny_store16(P, orow, c * 16, v);
    }
  }
  tc_fence_before();
  __syncwarp();
  if (S > 1)
    cluster_sync_all();  // the leader has read every partial before any CTA exits
  else
    __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <bool MN, int RP>
static cudaError_t launch_skinny_t(const SkinnyParams &p, cudaStream_t st) {
  using L = SkinnySmem<MN, RP>;
  auto kern = lora_skinny_kernel<MN, RP>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::TOTAL);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  int tiles = 0;
  for (int q = 0; q < p.num_problems; ++q) tiles += p.pr[q].row_tiles;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(tiles * p.split), 1, 1);
  cfg.blockDim = dim3(192, 1, 1);
  cfg.dynamicSmemBytes = L::TOTAL;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)p.split;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p);
  note_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_skinny(const SkinnyParams &p, bool mn_major, int rp, cudaStream_t st) {
  if (p.split != 1 && p.split != 2 && p.split != 4 && p.split != 8) return cudaErrorInvalidValue;
  switch (rp) {
    case 16: return mn_major ? launch_skinny_t<true, 16>(p, st) : launch_skinny_t<false, 16>(p, st);
    case 32: return mn_major ? launch_skinny_t<true, 32>(p, st) : launch_skinny_t<false, 32>(p, st);
    case 64: return mn_major ? launch_skinny_t<true, 64>(p, st) : launch_skinny_t<false, 64>(p, st);
    case 128: return mn_major ? launch_skinny_t<true, 128>(p, st) : launch_skinny_t<false, 128>(p, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace lora
