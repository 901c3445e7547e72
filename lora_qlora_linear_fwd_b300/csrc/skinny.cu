// Rank-r passes of the backward ("UnSloth加速微调体验" §反向传播优化):
//   v  = x·Aᵀ          (recomputed, KMAJOR mode: reduce over k)
//   dA = s·uᵀ·x        (MNMAJOR mode: reduce over tokens)
//   dB = s·dYᵀ·v       (MNMAJOR mode: reduce over tokens)
// Each CTA owns a 128-row output tile [128 x RP] and one slice of the
// reduction; it streams its operand tiles through a TMA ring into a tcgen05
// accumulator.  CTAs of one row tile meet through an arrival counter: each
// writes its fp32 partial, and the last to arrive adds all slices in slice
// order (deterministic) and writes the final output.  In MNMAJOR mode the
// bf16 right-hand operand comes as two parts (hi + lo = the fp32 value to
// about 2^-17 relative) and both are multiplied, so the result keeps
// near-fp32 accuracy while the large operand (x or dY) streams once.
#include "kernels.h"

namespace lora {

template <bool MN, int RP>
struct SkinnySmem {
  static constexpr int P_BYTES = 128 * 128;  // [128 x 64] bf16 either way
  static constexpr int Q_BYTES = RP * 128;
  static constexpr int STAGE_BYTES = P_BYTES + (MN ? 2 : 1) * Q_BYTES;
  // small enough that two CTAs share an SM
  static constexpr int STAGES_FIT = (110 * 1024 - 2048) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 6 ? 6 : STAGES_FIT;
  static constexpr int OFF_MISC = STAGES * STAGE_BYTES;
  static constexpr int TOTAL = OFF_MISC + 256 + 1024;
  static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");
  static_assert(STAGES >= 3, "pipeline depth");
};

LORA_DEV void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Final values of columns [j0, j0+16) of output row `orow`.
LORA_DEV void skinny_store16(const SkinnyProblem &P, int orow, int j0, const float (&v)[16]) {
  if (orow >= P.rows) return;
  if (P.out_kind == kOutVt) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const __nv_bfloat16 hi = __float2bfloat16_rn(v[j]);
      P.out_hi[(size_t)(j0 + j) * P.out_ld + orow] = hi;
      P.out_lo[(size_t)(j0 + j) * P.out_ld + orow] =
          __float2bfloat16_rn(v[j] - __bfloat162float(hi));
    }
  } else if (P.out_kind == kOutRowT) {
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (j0 + j < P.r) P.out_f32[(size_t)(j0 + j) * P.rows + orow] = v[j] * P.scale;
  } else {
    float4 *dst = reinterpret_cast<float4 *>(P.out_f32 + (size_t)orow * P.r + j0);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (j0 + 4 * j < P.r)
        dst[j] = make_float4(v[4 * j] * P.scale, v[4 * j + 1] * P.scale, v[4 * j + 2] * P.scale,
                             v[4 * j + 3] * P.scale);
  }
}

template <bool MN, int RP>
__global__ void __launch_bounds__(192, 2) lora_skinny_kernel(const __grid_constant__ SkinnyParams p) {
  using L = SkinnySmem<MN, RP>;
  constexpr int STAGES = L::STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_addr(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (base - raw_base);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  const uint32_t bar_full = base + L::OFF_MISC;
  const uint32_t bar_empty = bar_full + 8 * STAGES;
  const uint32_t bar_acc = bar_empty + 8 * STAGES;
  const uint32_t bar_drain = bar_acc + 8;
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::OFF_MISC + 8 * (2 * STAGES + 2));
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
  volatile int *last_flag = reinterpret_cast<volatile int *>(tmem_holder + 2);
  volatile int *epi_fail = reinterpret_cast<volatile int *>(tmem_holder + 3);

  const int pi = (p.num_problems > 1 && (int)blockIdx.x >= p.pr[1].cta_begin) ? 1 : 0;
  const SkinnyProblem &P = p.pr[pi];
  const int local = blockIdx.x - P.cta_begin;
  const int rt = local % P.row_tiles;
  const int slice = local / P.row_tiles;
  const int total_chunks = (P.red + 63) / 64;
  const int c_begin = slice * P.chunks_per_slice;
  const int c_end = min(total_chunks, c_begin + P.chunks_per_slice);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_acc, 1);
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    *last_flag = 0;
    *epi_fail = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_holder), 64);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&P.tm_p);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t fill_parity[STAGES];
      bool filled[STAGES];
      for (int s = 0; s < STAGES; ++s) filled[s] = false, fill_parity[s] = 0;
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
          tma_load_2d(sq, &P.tm_q_hi, fb, c * 64, 0);
          tma_load_2d(sq + L::Q_BYTES, &P.tm_q_lo, fb, c * 64, 0);
        } else {
          tma_load_2d(sp, &P.tm_p, fb, c * 64, rt * 128);
          tma_load_2d(sq, &P.tm_q_hi, fb, c * 64, 0);
        }
        filled[stage] = true;
        fill_parity[stage] = phase;
        if (++stage == STAGES) stage = 0, phase ^= 1u;
      }
      if (*abort_flag)
        for (int s = 0; s < STAGES; ++s)
          if (filled[s]) mbar_wait_quiet(bar_full + 8 * s, fill_parity[s], 100000000ull);
    }
  } else if (warp == 1) {
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
      if (ok) tc_commit(bar_acc);
      if (*abort_flag) {
        tc_commit(bar_drain);
        mbar_wait_quiet(bar_drain, 0, 100000000ull);
      }
    }
  } else {
    // ------------------------------------------------ epilogue + reduction
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int orow = rt * 128 + row;
    const bool ok = __all_sync(0xffffffffu, mbar_wait(bar_acc, 0, abort_flag, p.status));
    if (!ok && lane == 0) *epi_fail = 1;
    epi_bar();                 // every epilogue warp takes the same branch below
    if (!*epi_fail) {
      tc_fence_after();
      float v[RP];
#pragma unroll
      for (int c = 0; c < RP / 16; ++c) {
        uint32_t r[16];
        tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + c * 16, r);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) v[c * 16 + j] = __uint_as_float(r[j]);
      }
      if (P.slices == 1) {
#pragma unroll
        for (int c = 0; c < RP / 16; ++c) {
          float t[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) t[j] = v[c * 16 + j];
          skinny_store16(P, orow, c * 16, t);
        }
      } else {
        if (orow < P.rows) {
          float4 *dst = reinterpret_cast<float4 *>(P.part + ((size_t)slice * P.rows + orow) * RP);
#pragma unroll
          for (int j = 0; j < RP / 4; ++j)
            dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        }
        __threadfence();
        epi_bar();
        if (threadIdx.x == 64)
          *last_flag = (atomicAdd(P.counter + rt, 1u) == (uint32_t)(P.slices - 1)) ? 1 : 0;
        epi_bar();
        if (*last_flag) {
          __threadfence();
          // add the slices in slice order, 16 columns at a time
#pragma unroll
          for (int c = 0; c < RP / 16; ++c) {
            float sum[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) sum[j] = 0.0f;
            if (orow < P.rows) {
              for (int s = 0; s < P.slices; ++s) {
                if (s == slice) {
#pragma unroll
                  for (int j = 0; j < 16; ++j) sum[j] += v[c * 16 + j];
                } else {
                  const float4 *src = reinterpret_cast<const float4 *>(
                      P.part + ((size_t)s * P.rows + orow) * RP + c * 16);
#pragma unroll
                  for (int j = 0; j < 4; ++j) {
                    const float4 t = __ldcg(src + j);
                    sum[4 * j] += t.x;
                    sum[4 * j + 1] += t.y;
                    sum[4 * j + 2] += t.z;
                    sum[4 * j + 3] += t.w;
                  }
                }
              }
            }
            skinny_store16(P, orow, c * 16, sum);
          }
          if (threadIdx.x == 64) P.counter[rt] = 0u;   // ready for the next call
        }
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 64);
  }
}

template <bool MN, int RP>
static cudaError_t launch_skinny_t(const SkinnyParams &p, int grid, cudaStream_t st) {
  using L = SkinnySmem<MN, RP>;
  auto kern = lora_skinny_kernel<MN, RP>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::TOTAL);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  kern<<<grid, 192, L::TOTAL, st>>>(p);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_skinny(const SkinnyParams &p, bool mn_major, int rp, int grid, cudaStream_t st) {
  switch (rp) {
    case 16: return mn_major ? launch_skinny_t<true, 16>(p, grid, st) : launch_skinny_t<false, 16>(p, grid, st);
    case 32: return mn_major ? launch_skinny_t<true, 32>(p, grid, st) : launch_skinny_t<false, 32>(p, grid, st);
    case 64: return mn_major ? launch_skinny_t<true, 64>(p, grid, st) : launch_skinny_t<false, 64>(p, grid, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace lora
