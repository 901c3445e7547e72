// Rank-r passes of the backward ("UnSloth加速微调体验" §反向传播优化):
//   v  = x·Aᵀ          (recomputed, KMAJOR mode: reduce over k)
//   dA = s·uᵀ·x        (MNMAJOR mode: reduce over tokens)
//   dB = s·dYᵀ·v       (MNMAJOR mode: reduce over tokens)
//
// These are HBM-bound streams of x or dY, so the kernel is built to keep
// HBM busy: one persistent CTA per SM, each owning a contiguous, equal-sized
// range of work items (item = one 64-wide reduction chunk of one 128-row
// output tile), streamed back to back through a deep TMA ring.  A run of
// items of one row tile (a segment) accumulates in one of two TMEM buffers
// while the epilogue drains the other.  A row tile split over several CTAs
// meets through an arrival counter: each segment writes an fp32 partial and
// the last to arrive adds the partials in segment order (deterministic) and
// writes the final output.  In MNMAJOR mode the bf16 right-hand operand comes
// as hi + lo parts (the fp32 value to about 2^-17 relative) and both are
// multiplied, so the result keeps near-fp32 accuracy.
#include "kernels.h"

namespace lora {

template <bool MN, int RP>
struct SkinnySmem {
  static constexpr int P_BYTES = 128 * 128;  // [128 x 64] bf16 either way
  static constexpr int Q_BYTES = RP * 128;
  static constexpr int STAGE_BYTES = P_BYTES + (MN ? 2 : 1) * Q_BYTES;
  static constexpr int STAGES_FIT = (kSmemLimit - 4096) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 10 ? 10 : STAGES_FIT;
  static constexpr int OFF_MISC = STAGES * STAGE_BYTES;
  static constexpr int TOTAL = OFF_MISC + 512 + 1024;
  static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");
  static_assert(STAGES >= 4, "pipeline depth");
};

LORA_DEV void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Which CTA owns global work item i (ranges [floor(W*c/G), floor(W*(c+1)/G))).
LORA_DEV int item_owner(long long i, long long W, int G) {
  return (int)(((i + 1) * G - 1) / W);
}

// Problem, row tile and chunk of global work item i.
struct ItemPos {
  int pi, rt, c;
};

LORA_DEV ItemPos item_pos(const SkinnyParams &p, long long i) {
  ItemPos q;
  const long long items0 = (long long)p.pr[0].row_tiles * p.pr[0].chunks;
  q.pi = (p.num_problems > 1 && i >= items0) ? 1 : 0;
  const long long li = q.pi ? i - items0 : i;
  const int chunks = p.pr[q.pi].chunks;
  q.rt = (int)(li / chunks);
  q.c = (int)(li % chunks);
  return q;
}

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
    for (int j = 0; j < 16; ++j) {
      const int jg = j0 + j;
      if (jg < P.nproj * P.r) {
        const int pr = jg / P.r, jj = jg % P.r;
        float *out = pr ? P.out_f32b : P.out_f32;
        out[(size_t)jj * P.rows + orow] = v[j] * P.scale;
      }
    }
  } else {
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
  constexpr uint32_t kTmemCols = 2 * RP >= 32 ? 2 * RP : 32;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_addr(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (base - raw_base);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  const uint32_t bar_full = base + L::OFF_MISC;
  const uint32_t bar_empty = bar_full + 8 * STAGES;
  const uint32_t bar_acc_full = bar_empty + 8 * STAGES;  // [2]
  const uint32_t bar_acc_empty = bar_acc_full + 16;      // [2]
  const uint32_t bar_drain = bar_acc_empty + 16;
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::OFF_MISC + 8 * (2 * STAGES + 5));
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
  volatile int *last_flag = reinterpret_cast<volatile int *>(tmem_holder + 2);
  volatile int *epi_fail = reinterpret_cast<volatile int *>(tmem_holder + 3);

  const long long W = p.total_items;
  const int G = gridDim.x;
  const long long i_begin = W * blockIdx.x / G;
  const long long i_end = W * (blockIdx.x + 1) / G;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_acc_full, 1);
    mbar_init(bar_acc_full + 8, 1);
    mbar_init(bar_acc_empty, 128);
    mbar_init(bar_acc_empty + 8, 128);
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    *last_flag = 0;
    *epi_fail = 0;
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
      for (int q = 0; q < p.num_problems; ++q) tma_prefetch_desc(&p.pr[q].tm_p);
      int stage = 0;
      uint32_t phase = 0;
      int fills[STAGES];
      for (int s = 0; s < STAGES; ++s) fills[s] = 0;
      for (long long i = i_begin; i < i_end; ++i) {
        if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1u, abort_flag, p.status)) break;
        const ItemPos ip = item_pos(p, i);
        const SkinnyProblem &P = p.pr[ip.pi];
        const uint32_t sp = base + stage * L::STAGE_BYTES;
        const uint32_t sq = sp + L::P_BYTES;
        const uint32_t fb = bar_full + 8 * stage;
        mbar_arrive_expect_tx(fb, L::STAGE_BYTES);
        if constexpr (MN) {
          // P [tokens, rows]: two boxes of [64 rows-of-output x 64 tokens]
          tma_load_2d(sp, &P.tm_p, fb, ip.rt * 128, ip.c * 64);
          tma_load_2d(sp + 8192, &P.tm_p, fb, ip.rt * 128 + 64, ip.c * 64);
          tma_load_2d(sq, &P.tm_q_hi, fb, ip.c * 64, 0);
          tma_load_2d(sq + L::Q_BYTES, &P.tm_q_lo, fb, ip.c * 64, 0);
        } else {
          tma_load_2d(sp, &P.tm_p, fb, ip.c * 64, ip.rt * 128);
          tma_load_2d(sq, &P.tm_q_hi, fb, ip.c * 64, 0);
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
      int seg = 0;
      int used[2] = {0, 0};
      bool ok = true;
      long long i = i_begin;
      while (ok && i < i_end) {
        // one segment: the consecutive items of one row tile
        const ItemPos ip0 = item_pos(p, i);
        const int b = seg & 1;
        if (used[b] > 0 &&
            !mbar_wait(bar_acc_empty + 8 * b, (used[b] - 1) & 1, abort_flag, p.status))
          break;
        ++used[b];
        tc_fence_after();
        const uint32_t acc = tmem + b * RP;
        bool first = true;
        for (; i < i_end; ++i) {
          const ItemPos ip = item_pos(p, i);
          if (ip.pi != ip0.pi || ip.rt != ip0.rt) break;
          if (!mbar_wait(bar_full + 8 * stage, phase, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sp = base + stage * L::STAGE_BYTES;
          const uint32_t sq = sp + L::P_BYTES;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint32_t accum = (!first || ks != 0) ? 1u : 0u;
            uint64_t da;
            if constexpr (MN)
              da = make_sdesc(sp + ks * 2048, 8192, 1024, kSw128);
            else
              da = make_sdesc(sp + ks * 32, 16, 1024, kSw128);
            tc_mma(acc, da, make_sdesc(sq + ks * 32, 16, 1024, kSw128), idesc, accum);
            if constexpr (MN)
              tc_mma(acc, da, make_sdesc(sq + L::Q_BYTES + ks * 32, 16, 1024, kSw128), idesc, 1u);
          }
          tc_commit(bar_empty + 8 * stage);
          first = false;
          if (++stage == STAGES) stage = 0, phase ^= 1u;
        }
        if (!ok) break;
        tc_commit(bar_acc_full + 8 * b);
        ++seg;
      }
      if (*abort_flag) {
        tc_commit(bar_drain);
        mbar_wait_quiet(bar_drain, 0, 100000000ull);
      }
    }
  } else {
    // ------------------------------------------------ epilogue + reduction
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const uint32_t t_lane = (uint32_t)(q * 32) << 16;
    int seg = 0;
    long long i = i_begin;
    while (i < i_end) {
      const ItemPos ip0 = item_pos(p, i);
      const SkinnyProblem &P = p.pr[ip0.pi];
      // extent of this segment and of its row tile's work items
      const long long items0 = ip0.pi ? (long long)p.pr[0].row_tiles * p.pr[0].chunks : 0;
      const long long tile_first = items0 + (long long)ip0.rt * P.chunks;
      const long long tile_end = tile_first + P.chunks;
      const long long seg_end = tile_end < i_end ? tile_end : i_end;
      const int owner0 = item_owner(tile_first, W, G);
      const int nseg = item_owner(tile_end - 1, W, G) - owner0 + 1;
      const int slot = (int)blockIdx.x - owner0;
      const int b = seg & 1;
      const int orow = ip0.rt * 128 + row;

      const bool ok = __all_sync(
          0xffffffffu, mbar_wait(bar_acc_full + 8 * b, (seg >> 1) & 1, abort_flag, p.status));
      if (!ok && lane == 0) *epi_fail = 1;
      epi_bar();  // every epilogue warp takes the same branch below
      const bool failed = *epi_fail != 0;
      epi_bar();  // read before any warp can reach the next segment's wait
      if (failed) break;
      tc_fence_after();
      float *part_tile = P.part + (size_t)ip0.rt * P.max_segs * 128 * RP;
      float *my_part = part_tile + ((size_t)slot * 128 + row) * RP;
      // drain the accumulator 16 columns at a time: final values if this CTA
      // is the row tile's only contributor, else its fp32 partial
#pragma unroll
      for (int c = 0; c < RP / 16; ++c) {
        uint32_t r[16];
        tmem_ld16(tmem + t_lane + b * RP + c * 16, r);
        tmem_ld_wait();
        float t[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) t[j] = __uint_as_float(r[j]);
        if (nseg == 1) {
          skinny_store16(P, orow, c * 16, t);
        } else if (orow < P.rows) {
          float4 *dst = reinterpret_cast<float4 *>(my_part + c * 16);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            dst[j] = make_float4(t[4 * j], t[4 * j + 1], t[4 * j + 2], t[4 * j + 3]);
        }
      }
      tc_fence_before();
      mbar_arrive(bar_acc_empty + 8 * b);  // TMEM buffer b is free again

      if (nseg > 1) {
        __threadfence();
        epi_bar();
        if (threadIdx.x == 64)
          *last_flag = (atomicAdd(P.counter + ip0.rt, 1u) == (uint32_t)(nseg - 1)) ? 1 : 0;
        epi_bar();
        if (*last_flag) {
          __threadfence();
          // add the segments in segment order, 16 columns at a time
#pragma unroll 1
          for (int c = 0; c < RP / 16; ++c) {
            float sum[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) sum[j] = 0.0f;
            if (orow < P.rows) {
              for (int s = 0; s < nseg; ++s) {
                const float4 *src = reinterpret_cast<const float4 *>(
                    part_tile + ((size_t)s * 128 + row) * RP + c * 16);
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
            skinny_store16(P, orow, c * 16, sum);
          }
          if (threadIdx.x == 64) P.counter[ip0.rt] = 0u;  // ready for the next call
        }
        epi_bar();  // last_flag is reused by the next segment
      }
      i = seg_end;
      ++seg;
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
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
    case 128: return mn_major ? launch_skinny_t<true, 128>(p, grid, st) : launch_skinny_t<false, 128>(p, grid, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace lora
