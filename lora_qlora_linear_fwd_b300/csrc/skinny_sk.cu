// Rank-r passes, stream-K form: the same products as skinny.cu
// ("UnSloth加速微调体验" §算子融合, §反向传播优化), for the shapes whose row
// tiles do not spread evenly over the SMs as clusters (few or uneven tiles).
//
// These stream x or dY once and are HBM-bound, so every SM must stream for
// the whole launch.  The work is a list of units (problem, 128-row output
// tile, 64-wide reduction chunk), and a persistent grid of one CTA per SM
// takes equal contiguous ranges of it (a "stream-K" split): a CTA's range
// is cut into segments at tile boundaries, each reduced into one of two
// TMEM accumulators [128 x RP], so a segment's epilogue overlaps the next
// segment's stream.
//   * A segment that starts inside its tile (it is the first segment of its
//     CTA) parks its fp32 partial in the CTA's slot of the scratch area and
//     raises the CTA's flag (tagged with the launch's epoch).
//   * The segment that starts at the tile's first chunk -- the last segment
//     of its CTA, hence the last to finish -- waits for the flags of the
//     CTAs that took the rest of the tile, adds their partials in CTA order
//     (the sum is deterministic), and stores the outputs.
// In MNMAJOR mode the right-hand operand comes as bf16 hi + lo parts of an
// fp32 value (about 2^-17 relative) and both are multiplied, keeping
// near-fp32 accuracy for dA and dB.
#include "kernels.h"
#include "skinny_out.cuh"

namespace lora {
namespace sk {

template <bool MN, int RP>
struct SkSmem {
  static constexpr int P_BYTES = 128 * 128;  // [128 x 64] bf16 either way
  static constexpr int Q_BYTES = RP * 128;
  static constexpr int STAGE_BYTES = P_BYTES + (MN ? 2 : 1) * Q_BYTES;
  static constexpr int STAGES_FIT = (kSmemLimit - 4096) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 10 ? 10 : STAGES_FIT;
  static constexpr int OFF_MISC = STAGES * STAGE_BYTES;
  static constexpr int TOTAL = OFF_MISC + 512 + 1024;
  static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");
  static_assert(STAGES >= 4, "pipeline depth");
  static_assert(TOTAL <= kSmemLimit, "shared memory budget");
};

LORA_DEV unsigned long long ld_acquire_u64(const unsigned long long *p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
LORA_DEV void st_release_u64(unsigned long long *p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

#ifdef LORA_TEST_HOOKS
// Test-only build (liblora_b300_testhooks.so): the host can shorten the flag
// wait's limit and name one CTA that parks its partial without raising its
// flag (lora_test_stream_k_hooks), so that a test makes the finisher's wait
// run out and checks the reported status.  The product library has neither.
static __device__ unsigned long long g_flag_wait_limit_ns = kWaitLimitNs;
static __device__ int g_skip_flag_cta = -1;
LORA_DEV uint64_t flag_wait_limit_ns() { return g_flag_wait_limit_ns; }
LORA_DEV bool flag_skipped(int cta) { return cta == g_skip_flag_cta; }
#else
LORA_DEV uint64_t flag_wait_limit_ns() { return kWaitLimitNs; }
LORA_DEV bool flag_skipped(int) { return false; }
#endif

// Bounded wait for another CTA's flag to carry `epoch`.
LORA_DEV bool wait_flag(const unsigned long long *f, unsigned long long epoch,
                        volatile int *abort_flag, uint32_t *status) {
  const uint64_t t0 = global_timer_ns();
  const uint64_t limit = flag_wait_limit_ns();
  while (ld_acquire_u64(f) != epoch) {
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > limit) {
      *abort_flag = 1;
      atomicOr(status, kDevTimeout);
      return false;
    }
    __nanosleep(64);
  }
  return true;
}

// Walk over the segments of one CTA's unit range [u, end).
struct SegIter {
  long long u, end;
  int pi, rt, cb, ce;  // problem, row tile, chunk range [cb, ce)
  LORA_DEV bool next(const SkinnyParams &p) {
    if (u >= end) return false;
    pi = (p.num_problems > 1 && u >= p.pr[1].unit_begin) ? 1 : 0;
    const SkinnyProblem &P = p.pr[pi];
    const long long local = u - P.unit_begin;
    rt = (int)(local / P.chunks);
    cb = (int)(local - (long long)rt * P.chunks);
    const long long rest = end - u;
    ce = rest < (long long)(P.chunks - cb) ? cb + (int)rest : P.chunks;
    u += ce - cb;
    return true;
  }
};

LORA_DEV long long range_begin(const SkinnyParams &p, int cta) {
  return p.units * cta / p.ctas;
}

// Outputs of accumulator columns [j0, j0 + 16) of tile row `row` (final
// values, unscaled).  Transposed kinds: lanes hold consecutive rows, so
// each column is one contiguous run per warp; row-major kinds: each thread
// stores its row's 16 columns in 16-byte pieces.
template <bool F16>
LORA_DEV void skinny_store16(const SkinnyDest &P, int rt, int row, int j0, const float (&v)[16]) {
  const int grow = rt * 128 + row;
  if (grow >= P.rows) return;
  const int cols = P.nproj * P.r;  // valid rank columns
  if (P.out_kind & kOutVt) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const uint16_t hi = to16<F16>(v[j]);
      const uint16_t lo = to16<F16>(v[j] - from16<F16>(hi));
      P.out_hi[(size_t)(j0 + j) * P.ld_t + grow] = hi;
      P.out_lo[(size_t)(j0 + j) * P.ld_t + grow] = lo;
    }
  }
  if (P.out_kind & kOutRowT) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int jg = j0 + j;
      if (jg < cols) {
        const int pr = jg / P.r, jj = jg - pr * P.r;
        (pr ? P.out_f32b : P.out_f32)[(size_t)jj * P.rows + grow] = v[j] * P.scale;
      }
    }
  }
  if (P.out_kind & kOutRowBf16) {
    uint16_t *dst = P.out_bf16 + (size_t)grow * P.ld_row + j0;
    if (j0 + 16 <= cols) {
      uint32_t w[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) w[q] = pack2<F16>(v[2 * q] * P.scale, v[2 * q + 1] * P.scale);
      reinterpret_cast<uint4 *>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
      reinterpret_cast<uint4 *>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (j0 + j < cols) dst[j] = to16<F16>(v[j] * P.scale);
    }
  }
  if (P.out_kind & kOutRow) {
    // dB: only the diagonal block of a merged pair is a real gradient
    const int pr = (P.nproj > 1 && grow >= P.split_row) ? 1 : 0;
    const int lo = pr * P.r;
    float *dst = (pr ? P.out_f32b : P.out_f32) + (size_t)(grow - pr * P.split_row) * P.r;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int jg = j0 + 4 * q;
      if (jg >= lo && jg + 4 <= lo + P.r) {
        *reinterpret_cast<float4 *>(dst + (jg - lo)) =
            make_float4(v[4 * q] * P.scale, v[4 * q + 1] * P.scale, v[4 * q + 2] * P.scale,
                        v[4 * q + 3] * P.scale);
      } else {
        for (int e = 0; e < 4; ++e)
          if (jg + e >= lo && jg + e < lo + P.r) dst[jg + e - lo] = v[4 * q + e] * P.scale;
      }
    }
  }
}

template <bool MN, int RP, bool F16>
__global__ void __launch_bounds__(192, 1) lora_skinny_sk_kernel(const __grid_constant__ SkinnyParams p) {
  using L = SkSmem<MN, RP>;
  constexpr int STAGES = L::STAGES;
  constexpr uint32_t kTmemCols = 2 * RP >= 32 ? 2 * RP : 32;  // two accumulators
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_addr(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (base - raw_base);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int cta = blockIdx.x;
  const long long u_begin = range_begin(p, cta), u_end = range_begin(p, cta + 1);

  const uint32_t bar_full = base + L::OFF_MISC;
  const uint32_t bar_empty = bar_full + 8 * STAGES;
  const uint32_t bar_acc_full = bar_empty + 8 * STAGES;  // [2]
  const uint32_t bar_acc_empty = bar_acc_full + 16;      // [2] four epilogue warps
  const uint32_t bar_drain = bar_acc_empty + 16;
  // used at most once per launch: a CTA parks at most one partial (its
  // first segment) and finishes at most one tile that others share (its
  // last segment)
  const uint32_t bar_parked = bar_drain + 8;   // four epilogue warps stored the partial
  const uint32_t bar_ready = bar_parked + 8;   // the other CTAs' partials are visible
  const uint32_t bar_staged = bar_ready + 8;   // four epilogue warps staged the last tile
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::OFF_MISC + 8 * (2 * STAGES + 8));
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_acc_full + 8 * b, 1);
      mbar_init(bar_acc_empty + 8 * b, 4);
    }
    mbar_init(bar_drain, 1);
    mbar_init(bar_parked, 4);
    mbar_init(bar_ready, 1);
    mbar_init(bar_staged, 4);
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
  grid_dep_launch();
  grid_dep_wait();  // the previous kernel's outputs are complete

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      for (int q = 0; q < p.num_problems; ++q) tma_prefetch_desc(&p.pr[q].tm_p);
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;  // chunks issued: stage s took every STAGES-th from the s-th
      bool ok = true;
      SegIter sg{u_begin, u_end};
      while (ok && sg.next(p)) {
        const SkinnyProblem &P = p.pr[sg.pi];
        const int rt = sg.rt;
        for (int c = sg.cb; c < sg.ce; ++c) {
          if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
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
          ++issued;
          if (++stage == STAGES) stage = 0, phase ^= 1u;
        }
      }
      // drain: every issued copy has been consumed before the CTA may exit
      // (bounded: after an abort some never are)
      const uint64_t lim = *abort_flag ? 20000000ull : 1000000000ull;
      for (int s = 0; s < STAGES; ++s) {
        const int fills = issued > s ? (issued - s + STAGES - 1) / STAGES : 0;
        if (fills > 0) mbar_wait_quiet(bar_empty + 8 * s, (uint32_t)((fills - 1) & 1), lim);
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc(128, RP, MN, false, F16);
      int stage = 0;
      uint32_t phase = 0;
      int k = 0;  // segments issued: accumulator k & 1
      bool ok = true;
      SegIter sg{u_begin, u_end};
      while (ok && sg.next(p)) {
        const int b = k & 1;
        // the epilogue has drained this accumulator's previous segment
        if (k >= 2 && !mbar_wait(bar_acc_empty + 8 * b, (uint32_t)((k >> 1) - 1) & 1u, abort_flag,
                                 p.status))
          break;
        tc_fence_after();
        const uint32_t t_acc = tmem + (uint32_t)(b * RP);
        for (int c = sg.cb; c < sg.ce; ++c) {
          if (!mbar_wait(bar_full + 8 * stage, phase, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sp = base + stage * L::STAGE_BYTES;
          const uint32_t sq = sp + L::P_BYTES;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint32_t accum = (c != sg.cb || ks != 0) ? 1u : 0u;
            uint64_t da;
            if constexpr (MN)
              da = make_sdesc(sp + ks * 2048, 8192, 1024, kSw128);
            else
              da = make_sdesc(sp + ks * 32, 16, 1024, kSw128);
            tc_mma(t_acc, da, make_sdesc(sq + ks * 32, 16, 1024, kSw128), idesc, accum);
            if constexpr (MN)
              tc_mma(t_acc, da, make_sdesc(sq + L::Q_BYTES + ks * 32, 16, 1024, kSw128), idesc, 1u);
          }
          tc_commit(bar_empty + 8 * stage);
          if (++stage == STAGES) stage = 0, phase ^= 1u;
        }
        if (!ok) break;
        tc_commit(bar_acc_full + 8 * b);
        ++k;
      }
      if (*abort_flag) {
        tc_commit(bar_drain);
        mbar_wait_quiet(bar_drain, 0, 100000000ull);
      }
    }
  } else {
    // ------------------------------------------------------- epilogue (2-5)
    const int row = (warp & 3) * 32 + lane;
    const uint32_t t_lane = (uint32_t)((warp & 3) * 32) << 16;
    const bool leader = threadIdx.x == 64;
    float *my_part = p.partials + (size_t)cta * RP * 128 + row;  // slot [RP][128]
    int k = 0;
    SegIter sg{u_begin, u_end};
    while (sg.next(p)) {
      const int b = k & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(bar_acc_full + 8 * b, (uint32_t)(k >> 1) & 1u,
                                             abort_flag, p.status)))
        break;
      tc_fence_after();
      const SkinnyProblem &P = p.pr[sg.pi];
      const uint32_t t_acc = tmem + t_lane + (uint32_t)(b * RP);
      if (sg.cb > 0) {
        // the rest of a tile that another CTA finishes: park the partial
#pragma unroll 1
        for (int c = 0; c < RP / 16; ++c) {
          uint32_t r[16];
          tmem_ld16(t_acc + c * 16, r);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) __stcg(my_part + (c * 16 + j) * 128, __uint_as_float(r[j]));
        }
        __threadfence();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_parked);
        if (leader && mbar_wait(bar_parked, 0, abort_flag, p.status) && !flag_skipped(cta))
          st_release_u64(p.flags + cta, p.epoch);
      } else {
        // the tile's first chunks: add the partials of the CTAs that took
        // the rest of it (if any), then store
        const long long tile_end = P.unit_begin + (long long)(sg.rt + 1) * P.chunks;
        int n_part = 0;
        if (sg.ce < P.chunks)
          while (cta + n_part + 1 < p.ctas && range_begin(p, cta + n_part + 1) < tile_end) ++n_part;
        // The parked partials are bulk-copied into the TMA ring, idle by now
        // (this is the CTA's last segment and its MMAs have completed), when
        // they fit; element (j, row) of partial q then sits at word
        // (q·RP + j)·128 + row of the ring.
        constexpr uint32_t kPartBytes = RP * 128 * 4;
        const bool staged = n_part > 0 && (uint32_t)n_part * kPartBytes <= (uint32_t)L::OFF_MISC;
        bool ok = true;
        if (n_part > 0) {
          if (leader) {
            for (int q = 1; q <= n_part && ok; ++q)
              ok = wait_flag(p.flags + cta + q, p.epoch, abort_flag, p.status);
            // consumed (or given up on) by this launch: clear them, since a
            // replay of the same launch, e.g. from a CUDA graph, carries the
            // same epoch.  A partial parked after a timeout can still leave a
            // flag behind; the status word then reports the timeout.
            for (int q = 1; q <= n_part; ++q) p.flags[cta + q] = 0ull;
            if (ok) {
              if (staged) {
                // the partials were written with ordinary stores and made
                // visible by the acquire; order them before the copy
                // engine's reads
                asm volatile("fence.proxy.async.global;" ::: "memory");
                mbar_arrive_expect_tx(bar_ready, (uint32_t)n_part * kPartBytes);
                for (int q = 1; q <= n_part; ++q)
                  bulk_load(base + (uint32_t)(q - 1) * kPartBytes,
                            p.partials + (size_t)(cta + q) * RP * 128, kPartBytes, bar_ready);
              } else {
                mbar_arrive(bar_ready);
              }
            }
          }
          ok = __all_sync(0xffffffffu, mbar_wait(bar_ready, 0, abort_flag, p.status));
        }
        // The CTA's last segment leaves its ring idle: the tile is staged
        // there, behind the partials, and copied out with wide stores (each
        // thread's own row-by-row stores are many and narrow).
        constexpr SkinnyEpi E(RP, 1);
        const uint32_t soff = staged ? (uint32_t)n_part * kPartBytes : 0u;
        const bool stage_out =
            sg.u >= sg.end && soff + (uint32_t)E.bytes <= (uint32_t)L::OFF_MISC;
        const SkinnyDest out = skinny_dest(P);
        float *stage_t = reinterpret_cast<float *>(smem + soff + E.off_stage_t);
        float *stage_r = reinterpret_cast<float *>(smem + soff + E.off_stage_r);
        const bool want_t = (out.out_kind & (kOutVt | kOutRowT | kOutT16)) != 0;
        const bool want_r = (out.out_kind & (kOutRowBf16 | kOutRow)) != 0;
        if (ok) {
          const float *ring = reinterpret_cast<const float *>(smem) + row;
#pragma unroll 1
          for (int c = 0; c < RP / 16; ++c) {
            uint32_t r[16];
            tmem_ld16(t_acc + c * 16, r);
            tmem_ld_wait();
            float v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
            for (int q = 1; q <= n_part; ++q) {
              if (staged) {
                const float *src = ring + (size_t)(q - 1) * RP * 128;
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] += src[(c * 16 + j) * 128];
              } else {
                const float *src = p.partials + (size_t)(cta + q) * RP * 128 + row;
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] += __ldcg(src + (c * 16 + j) * 128);
              }
            }
            if (stage_out) {
              if (want_t) {
#pragma unroll
                for (int j = 0; j < 16; ++j) stage_t[(c * 16 + j) * 132 + row] = v[j];
              }
              if (want_r) {
                float4 *dst = reinterpret_cast<float4 *>(stage_r + row * (RP + 4) + c * 16);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                  dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
              }
            } else {
              skinny_store16<F16>(out, sg.rt, row, c * 16, v);
            }
          }
        }
        if (stage_out) {
          // every epilogue warp arrives, also one that gave up above (it has
          // raised the abort flag, so the others' bounded wait ends)
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_staged);
          if (__all_sync(0xffffffffu, mbar_wait(bar_staged, 0, abort_flag, p.status)) && ok)
            skinny_copy_out<F16>(out, sg.rt, 0, RP, stage_t, stage_r, threadIdx.x - 64);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_acc_empty + 8 * b);
      ++k;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <bool MN, int RP, bool F16>
static cudaError_t launch_skinny_t(const SkinnyParams &p, cudaStream_t st) {
  using L = SkSmem<MN, RP>;
  auto kern = lora_skinny_sk_kernel<MN, RP, F16>;
  static std::atomic<uint64_t> attr_done{0};
  const cudaError_t e = smem_attr_once(attr_done, reinterpret_cast<const void *>(kern), L::TOTAL);
  if (e != cudaSuccess) return e;
  const char *name =
      MN ? (F16 ? "lora_skinny_sk_kernel<mn_major,f16>" : "lora_skinny_sk_kernel<mn_major>")
         : (F16 ? "lora_skinny_sk_kernel<k_major,f16>" : "lora_skinny_sk_kernel<k_major>");
  return launch_pdl(name, kern,
                    dim3((unsigned)p.ctas), dim3(192), L::TOTAL, st, 0u, p);
}

}  // namespace sk

size_t skinny_scratch_bytes(int rp) {
  return (((size_t)kSkinnyMaxCtas * 8 + 255) & ~(size_t)255) + (size_t)kSkinnyMaxCtas * rp * 128 * 4;
}

template <bool F16>
static cudaError_t launch_skinny_sk_t(const SkinnyParams &p, bool mn_major, int rp,
                                      cudaStream_t st) {
  using namespace sk;
  switch (rp) {
    case 16: return mn_major ? launch_skinny_t<true, 16, F16>(p, st) : launch_skinny_t<false, 16, F16>(p, st);
    case 32: return mn_major ? launch_skinny_t<true, 32, F16>(p, st) : launch_skinny_t<false, 32, F16>(p, st);
    case 64: return mn_major ? launch_skinny_t<true, 64, F16>(p, st) : launch_skinny_t<false, 64, F16>(p, st);
    case 128:
      return mn_major ? launch_skinny_t<true, 128, F16>(p, st) : launch_skinny_t<false, 128, F16>(p, st);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_skinny_sk(const SkinnyParams &p, bool mn_major, int rp, bool f16,
                             cudaStream_t st) {
  if (p.ctas < 1 || p.ctas > kSkinnyMaxCtas || p.units < p.ctas) return cudaErrorInvalidValue;
  return f16 ? launch_skinny_sk_t<true>(p, mn_major, rp, st)
             : launch_skinny_sk_t<false>(p, mn_major, rp, st);
}

}  // namespace lora

#ifdef LORA_TEST_HOOKS
// Test-only entry point of liblora_b300_testhooks.so (declared in
// include/lora_b300_test_hooks.h): sets the stream-K flag wait's limit and
// the CTA that skips raising its flag (-1: none).  Synchronous.
extern "C" lora_status_t lora_test_stream_k_hooks(unsigned long long wait_limit_ns,
                                                  int skip_flag_cta) {
  if (cudaMemcpyToSymbol(lora::sk::g_flag_wait_limit_ns, &wait_limit_ns, sizeof(wait_limit_ns)) !=
          cudaSuccess ||
      cudaMemcpyToSymbol(lora::sk::g_skip_flag_cta, &skip_flag_cta, sizeof(skip_flag_cta)) !=
          cudaSuccess)
    return LORA_ERR_CUDA;
  return LORA_OK;
}
#endif
