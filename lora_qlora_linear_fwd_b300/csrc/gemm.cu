// Fused LoRA GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// FWD mode  ("UnSloth加速微调体验" §算子融合, §RoPE缓存集成):
//     y  = x·Wᵀ + s·(x·Aᵀ)·Bᵀ            [optionally RoPE-rotated per head]
// DX mode   (same page, §反向传播优化):
//     dX = dY·W + s·(dY·B)·A,  and u = dY·B is exported (as uᵀ, bf16 hi+lo)
//
// Both modes share one persistent, warp-specialised kernel:
//   warp 0       TMA producer.  Per 64-wide K stage: the activation tile
//                (x or dY) [128 x 64], the W tile (bf16 via TMA, or NF4 code
//                bytes for the decode warps), and the rank-r operand of the
//                down-projection (A in FWD, Bᵀ in DX) while it is needed.
//                Once per output tile: the rank-r operand of the
//                up-projection (B in FWD, A in DX).
//   warp 1       allocates TMEM and issues tcgen05.mma from one thread:
//                acc[128 x BN] += act·W and rank[128 x RP] += act·R1 in the
//                same K loop; after the loop acc += (s·rank)·R2 (K = RP).
//   warps 2-5    epilogue: rank -> s·rank in bf16 (shared memory) once per
//                m-block; acc -> (RoPE) -> bf16 -> global.
//   warps 6-9    (NF4 only) decode 4-bit codes through the 16-entry NF4
//                codebook held in shared memory, scale by the block absmax and
//                write the bf16 W tile in the swizzled layout the tensor core
//                reads ("Unsloth教程" §显存优化策略: NF4 base weight).
// TMEM: acc at columns [0, BN), rank at [BN, BN+RP); 512 columns allocated.
#include "kernels.h"

namespace lora {

// The 16 NormalFloat4 levels (QLoRA, Dettmers et al. 2023, appendix table),
// ascending; index 7 is the exact zero.
__constant__ float kNf4Levels[16] = {
    -1.0f, -0.6961928009986877f, -0.5250730514526367f, -0.39491748809814453f,
    -0.28444138169288635f, -0.18477343022823334f, -0.09105003625154495f, 0.0f,
    0.07958029955625534f, 0.16093020141124725f, 0.24611230194568634f, 0.33791524171829224f,
    0.44070982933044434f, 0.5626170039176941f, 0.7229568362236023f, 1.0f};

template <int BN, int RP, bool NF4>
struct GemmSmem {
  static constexpr int X_BYTES = kBM * 128;
  static constexpr int W_BYTES = BN * 128;
  static constexpr int R1_BYTES = RP * 128;
  static constexpr int C_BYTES = NF4 ? BN * 32 : 0;
  static constexpr int OFF_W = X_BYTES;
  static constexpr int OFF_R1 = OFF_W + W_BYTES;
  static constexpr int OFF_C = OFF_R1 + R1_BYTES;
  static constexpr int STAGE_BYTES = OFF_C + C_BYTES;
  static constexpr int R2_BYTES = BN * RP * 2;
  static constexpr int SR_BYTES = kBM * RP * 2;
  static constexpr int MISC_BYTES = 1024;
  static constexpr int FIXED = R2_BYTES + SR_BYTES + MISC_BYTES + 1024;  // + alignment slack
  static constexpr int STAGES_FIT = (kSmemLimit - FIXED) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 6 ? 6 : STAGES_FIT;
  static constexpr int OFF_R2 = STAGES * STAGE_BYTES;
  static constexpr int OFF_SR = OFF_R2 + R2_BYTES;
  static constexpr int OFF_MISC = OFF_SR + SR_BYTES;
  static constexpr int TOTAL = OFF_MISC + MISC_BYTES + 1024;
  static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");
  static_assert(STAGES >= 2, "pipeline depth");
  static_assert(TOTAL <= kSmemLimit, "shared memory budget");
};

constexpr uint32_t swz_mode_for_row_bytes(int rb) {
  return rb == 128 ? kSw128 : (rb == 64 ? kSw64 : kSw32);
}

LORA_DEV bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                        uint32_t *status) {
  const bool ok = mbar_wait(bar, parity, abort_flag, status);
  return __all_sync(0xffffffffu, ok);
}

LORA_DEV int group_of(const GemmParams &p, int nt) {
  return (p.num_groups > 1 && nt >= p.grp[1].tile_begin) ? 1 : 0;
}

LORA_DEV uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// Decode one 64-element row piece: 32 code bytes at `src` (shared), block
// scale `a`, into a 128-byte row of a 128-byte-swizzled tile at `dst`.
LORA_DEV void nf4_decode_piece(uint32_t src, uint32_t dst, float a, const float *levels) {
  const uint4 c01 = ld_shared_v4(src);
  const uint4 c23 = ld_shared_v4(src + 16);
  const uint32_t words[8] = {c01.x, c01.y, c01.z, c01.w, c23.x, c23.y, c23.z, c23.w};
  const uint32_t phase = (dst >> 7) & 7u;
#pragma unroll
  for (int ch = 0; ch < 8; ++ch) {
    const uint32_t w = words[ch];
    uint32_t o[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint32_t byte = (w >> (8 * b)) & 0xFFu;
      o[b] = pack_bf16x2(levels[byte >> 4] * a, levels[byte & 0xFu] * a);
    }
    st_shared_v4(dst + ((((uint32_t)ch) ^ phase) << 4), o[0], o[1], o[2], o[3]);
  }
}

template <int MODE, int BN, int RP, bool NF4, bool ROPE>
__global__ void __launch_bounds__(NF4 ? 320 : 192, 1)
    lora_gemm_kernel(const __grid_constant__ GemmParams p) {
  using L = GemmSmem<BN, RP, NF4>;
  constexpr int STAGES = L::STAGES;
  constexpr int RB = RP * 2;  // bytes per row of the rank-r operands
  constexpr uint32_t SWR = swz_mode_for_row_bytes(RB);
  constexpr bool DX = MODE == kModeDx;
  constexpr int NUM_DEC_WARPS = NF4 ? 4 : 0;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_addr(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (base - raw_base);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  // barriers
  const uint32_t bar_full = base + L::OFF_MISC;         // [STAGES] TMA landed
  const uint32_t bar_empty = bar_full + 8 * STAGES;     // [STAGES] MMA done reading
  const uint32_t bar_dec = bar_empty + 8 * STAGES;      // [STAGES] NF4 tile decoded
  const uint32_t bar_r2_full = bar_dec + 8 * STAGES;
  const uint32_t bar_r2_empty = bar_r2_full + 8;
  const uint32_t bar_rank_full = bar_r2_empty + 8;
  const uint32_t bar_sr_ready = bar_rank_full + 8;
  const uint32_t bar_acc_full = bar_sr_ready + 8;
  const uint32_t bar_acc_empty = bar_acc_full + 8;
  const uint32_t bar_drain = bar_acc_empty + 8;
  const int misc_words = (8 * (3 * STAGES + 7)) / 4;
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::OFF_MISC) + misc_words;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
  float *levels = reinterpret_cast<float *>(tmem_holder + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
      mbar_init(bar_dec + 8 * s, NUM_DEC_WARPS > 0 ? NUM_DEC_WARPS : 1);
    }
    mbar_init(bar_r2_full, 1);
    mbar_init(bar_r2_empty, 1);
    mbar_init(bar_rank_full, 1);
    mbar_init(bar_sr_ready, 128);
    mbar_init(bar_acc_full, 1);
    mbar_init(bar_acc_empty, 128);
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (NF4 && threadIdx.x < 16) levels[threadIdx.x] = kNf4Levels[threadIdx.x];
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tm_act);
    for (int g = 0; g < p.num_groups; ++g) {
      tma_prefetch_desc(&p.grp[g].tm_w);
      tma_prefetch_desc(&p.grp[g].tm_r1);
      tma_prefetch_desc(&p.grp[g].tm_r2);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_holder), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const int nk = p.K / kBK;

  if (warp == 0) {
    // ================================================================ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int tile_count = 0, prev_g = -1;
      uint32_t fill_parity[STAGES];
      bool filled[STAGES];
      for (int s = 0; s < STAGES; ++s) filled[s] = false, fill_parity[s] = 0;
      bool ok = true;
      TileIter it;
      for (it.init(p.sched, blockIdx.x); ok && it.valid(); it.next(), ++tile_count) {
        const int m = it.m(), nt = it.nt();
        const int g = group_of(p, nt);
        const bool need_rank = it.first_of_m() || g != prev_g;
        prev_g = g;
        const GemmGroup &G = p.grp[g];
        const int n0 = (nt - G.tile_begin) * BN;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          const uint32_t sx = base + stage * L::STAGE_BYTES;
          const uint32_t fb = bar_full + 8 * stage;
          const uint32_t wbytes = NF4 ? L::C_BYTES : L::W_BYTES;
          mbar_arrive_expect_tx(fb, L::X_BYTES + wbytes + (need_rank ? L::R1_BYTES : 0));
          tma_load_2d(sx, &p.tm_act, fb, kb * kBK, m * kBM);
          if constexpr (NF4) {
            if constexpr (DX)  // codes [64 rows of W, BN/2 bytes]
              tma_load_2d(sx + L::OFF_C, &G.tm_w, fb, n0 / 2, kb * kBK);
            else               // codes [BN rows of W, 32 bytes]
              tma_load_2d(sx + L::OFF_C, &G.tm_w, fb, kb * (kBK / 2), n0);
          } else {
            if constexpr (DX) {  // W as MN-major operand: BN/64 boxes [64 rows x 64]
#pragma unroll
              for (int j = 0; j < BN / 64; ++j)
                tma_load_2d(sx + L::OFF_W + j * 8192, &G.tm_w, fb, n0 + 64 * j, kb * kBK);
            } else {
              tma_load_2d(sx + L::OFF_W, &G.tm_w, fb, kb * kBK, n0);
            }
          }
          if (need_rank) tma_load_2d(sx + L::OFF_R1, &G.tm_r1, fb, kb * kBK, 0);
          filled[stage] = true;
          fill_parity[stage] = phase;
          if (++stage == STAGES) stage = 0, phase ^= 1u;
        }
        if (!ok) break;
        // up-projection operand of this output tile (used after the K loop)
        if (!mbar_wait(bar_r2_empty, (tile_count & 1) ^ 1, abort_flag, p.status)) break;
        mbar_arrive_expect_tx(bar_r2_full, L::R2_BYTES);
        if constexpr (DX) {  // A [r, k] read MN-major: BN/64 boxes [RP rows x 64]
#pragma unroll
          for (int j = 0; j < BN / 64; ++j)
            tma_load_2d(base + L::OFF_R2 + j * RP * 128, &G.tm_r2, bar_r2_full, n0 + 64 * j, 0);
        } else {  // B [n, r]: one box [BN rows x RP]
          tma_load_2d(base + L::OFF_R2, &G.tm_r2, bar_r2_full, 0, n0);
        }
      }
      if (*abort_flag) {
        for (int s = 0; s < STAGES; ++s)
          if (filled[s]) mbar_wait_quiet(bar_full + 8 * s, fill_parity[s], 100000000ull);
      }
    }
  } else if (warp == 1) {
    // ===================================================================== MMA
    if (lane == 0) {
      constexpr uint32_t idesc_main = make_idesc_bf16(kBM, BN, false, DX);
      constexpr uint32_t idesc_rank = make_idesc_bf16(kBM, RP, false, false);
      int stage = 0;
      uint32_t phase = 0;
      int tile_count = 0, rank_count = 0, prev_g = -1;
      bool ok = true;
      TileIter it;
      for (it.init(p.sched, blockIdx.x); ok && it.valid(); it.next(), ++tile_count) {
        const int g = group_of(p, it.nt());
        const bool need_rank = it.first_of_m() || g != prev_g;
        prev_g = g;
        if (!mbar_wait(bar_acc_empty, (tile_count & 1) ^ 1, abort_flag, p.status)) break;
        tc_fence_after();
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(bar_full + 8 * stage, phase, abort_flag, p.status)) {
            ok = false;
            break;
          }
          if (NF4 && !mbar_wait(bar_dec + 8 * stage, phase, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sx = base + stage * L::STAGE_BYTES;
          const uint32_t sw = sx + L::OFF_W;
          const uint32_t sr = sx + L::OFF_R1;
#pragma unroll
          for (int ks = 0; ks < kBK / 16; ++ks) {
            const uint64_t da = make_sdesc(sx + ks * 32, 16, 1024, kSw128);
            uint64_t dw;
            if constexpr (DX)  // MN-major: 16 K-rows per step; 64-wide MN blocks 8 KB apart
              dw = make_sdesc(sw + ks * 2048, 8192, 1024, kSw128);
            else
              dw = make_sdesc(sw + ks * 32, 16, 1024, kSw128);
            const uint32_t accum = (kb | ks) != 0;
            tc_mma(tmem, da, dw, idesc_main, accum);
            if (need_rank) {
              const uint64_t dr = make_sdesc(sr + ks * 32, 16, 1024, kSw128);
              tc_mma(tmem + BN, da, dr, idesc_rank, accum);
            }
          }
          tc_commit(bar_empty + 8 * stage);
          if (++stage == STAGES) stage = 0, phase ^= 1u;
        }
        if (!ok) break;
        if (need_rank) {
          tc_commit(bar_rank_full);
          if (!mbar_wait(bar_sr_ready, rank_count & 1, abort_flag, p.status)) break;
          ++rank_count;
          tc_fence_after();
        }
        if (!mbar_wait(bar_r2_full, tile_count & 1, abort_flag, p.status)) break;
        tc_fence_after();
#pragma unroll
        for (int kr = 0; kr < RP / 16; ++kr) {
          const uint64_t dsr = make_sdesc(base + L::OFF_SR + kr * 32, 16, 8 * RB, SWR);
          uint64_t db;
          if constexpr (DX)  // A tile MN-major: boxes of RP rows, 16 K-rows per step
            db = make_sdesc(base + L::OFF_R2 + kr * 2048, RP * 128, 1024, kSw128);
          else
            db = make_sdesc(base + L::OFF_R2 + kr * 32, 16, 8 * RB, SWR);
          tc_mma(tmem, dsr, db, idesc_main, 1u);
        }
        tc_commit(bar_r2_empty);
        tc_commit(bar_acc_full);
      }
      if (*abort_flag) {
        tc_commit(bar_drain);
        mbar_wait_quiet(bar_drain, 0, 100000000ull);
      }
    }
  } else if (warp < 6) {
    // ================================================================ epilogue
    const int q = warp & 3;  // TMEM lane quadrant accessible to this warp
    const int row = q * 32 + lane;
    const uint32_t t_lane = (uint32_t)(q * 32) << 16;
    const int Mp = (p.M + 63) & ~63;
    int tile_count = 0, rank_count = 0, prev_g = -1;
    TileIter it;
    for (it.init(p.sched, blockIdx.x); it.valid(); it.next(), ++tile_count) {
      const int m = it.m(), nt = it.nt();
      const int g = group_of(p, nt);
      const bool need_rank = it.first_of_m() || g != prev_g;
      prev_g = g;
      const GemmGroup &G = p.grp[g];
      const int n0 = (nt - G.tile_begin) * BN;
      const int grow = m * kBM + row;
      const bool row_ok = grow < p.M;
      if (need_rank) {
        if (!warp_wait(bar_rank_full, rank_count & 1, abort_flag, p.status)) break;
        ++rank_count;
        tc_fence_after();
        const bool write_ut = DX && nt == 0 && row_ok;
#pragma unroll
        for (int c = 0; c < RP / 16; ++c) {
          uint32_t r[16];
          tmem_ld16(tmem + t_lane + BN + c * 16, r);
          tmem_ld_wait();
          uint32_t pk[8];
#pragma unroll
          for (int j = 0; j < 8; ++j)
            pk[j] = pack_bf16x2(__uint_as_float(r[2 * j]) * p.scale,
                                __uint_as_float(r[2 * j + 1]) * p.scale);
          const uint32_t srow = base + L::OFF_SR;
          st_shared_v4(srow + swz_offset(row, 2 * c, RB), pk[0], pk[1], pk[2], pk[3]);
          st_shared_v4(srow + swz_offset(row, 2 * c + 1, RB), pk[4], pk[5], pk[6], pk[7]);
          if (write_ut) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float u = __uint_as_float(r[j]);
              const __nv_bfloat16 hi = __float2bfloat16_rn(u);
              const __nv_bfloat16 lo = __float2bfloat16_rn(u - __bfloat162float(hi));
              const size_t idx = (size_t)(c * 16 + j) * Mp + grow;
              p.ut_hi[idx] = hi;
              p.ut_lo[idx] = lo;
            }
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar_sr_ready);
      }
      if (!warp_wait(bar_acc_full, tile_count & 1, abort_flag, p.status)) break;
      tc_fence_after();
      const int ncols = min(BN, G.ncols - n0);
      __nv_bfloat16 *orow = G.out + (size_t)(row_ok ? grow : 0) * G.ncols + n0;
      if constexpr (!ROPE) {
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(tmem + t_lane + c * 32, r);
          tmem_ld_wait();
          if (row_ok && c * 32 < ncols) {
            uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
            float f[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(r[j]);
            if (DX && p.accumulate) {
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const uint4 old = dst[j];
                const uint32_t ow[4] = {old.x, old.y, old.z, old.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162 *>(&ow[e]);
                  f[8 * j + 2 * e] += __low2float(h);
                  f[8 * j + 2 * e + 1] += __high2float(h);
                }
              }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint4 w;
              w.x = pack_bf16x2(f[8 * j + 0], f[8 * j + 1]);
              w.y = pack_bf16x2(f[8 * j + 2], f[8 * j + 3]);
              w.z = pack_bf16x2(f[8 * j + 4], f[8 * j + 5]);
              w.w = pack_bf16x2(f[8 * j + 6], f[8 * j + 7]);
              dst[j] = w;
            }
          }
        }
      } else {
        // rotate-half RoPE per 128-wide head: columns (i, i+64) share a row,
        // so one thread holds both members of every pair.
        int pos = 0;
        if (row_ok) {
          pos = __ldg(p.positions + grow);
          if (pos < 0 || pos >= p.max_pos) {
            atomicOr(p.status, kDevBadPosition);
            pos = 0;
          }
        }
        const float *cs = p.cos_sin + (size_t)pos * 128;
#pragma unroll 1
        for (int h = 0; h < BN / 128; ++h) {
#pragma unroll 1
          for (int half = 0; half < 2; ++half) {
            const int c0 = h * 128 + half * 32;
            uint32_t ra[32], rb[32];
            tmem_ld32(tmem + t_lane + c0, ra);
            tmem_ld32(tmem + t_lane + c0 + 64, rb);
            tmem_ld_wait();
            if (row_ok && c0 < ncols) {
              const float4 *cp = reinterpret_cast<const float4 *>(cs + half * 32);
              const float4 *sp = reinterpret_cast<const float4 *>(cs + 64 + half * 32);
              uint4 *da = reinterpret_cast<uint4 *>(orow + c0);
              uint4 *db = reinterpret_cast<uint4 *>(orow + c0 + 64);
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const float4 c_lo = __ldg(cp + 2 * j), c_hi = __ldg(cp + 2 * j + 1);
                const float4 s_lo = __ldg(sp + 2 * j), s_hi = __ldg(sp + 2 * j + 1);
                const float co[8] = {c_lo.x, c_lo.y, c_lo.z, c_lo.w,
                                     c_hi.x, c_hi.y, c_hi.z, c_hi.w};
                const float si[8] = {s_lo.x, s_lo.y, s_lo.z, s_lo.w,
                                     s_hi.x, s_hi.y, s_hi.z, s_hi.w};
                float oa[8], ob[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                  const float a = __uint_as_float(ra[8 * j + e]);
                  const float b = __uint_as_float(rb[8 * j + e]);
                  oa[e] = a * co[e] - b * si[e];
                  ob[e] = b * co[e] + a * si[e];
                }
                uint4 wa, wb;
                wa.x = pack_bf16x2(oa[0], oa[1]);
                wa.y = pack_bf16x2(oa[2], oa[3]);
                wa.z = pack_bf16x2(oa[4], oa[5]);
                wa.w = pack_bf16x2(oa[6], oa[7]);
                wb.x = pack_bf16x2(ob[0], ob[1]);
                wb.y = pack_bf16x2(ob[2], ob[3]);
                wb.z = pack_bf16x2(ob[4], ob[5]);
                wb.w = pack_bf16x2(ob[6], ob[7]);
                da[j] = wa;
                db[j] = wb;
              }
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(bar_acc_empty);
    }
  } else if constexpr (NF4) {
    // ============================================================= NF4 decode
    // Piece index pc in [0, BN): FWD: row pc of the W tile [BN x 64];
    // DX: row (pc % 64) of box (pc / 64) of the MN-major tile [64 x BN].
    const int dt = threadIdx.x - 192;  // 0..127
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    TileIter it;
    for (it.init(p.sched, blockIdx.x); ok && it.valid(); it.next()) {
      const int nt = it.nt();
      const GemmGroup &G = p.grp[group_of(p, nt)];
      const int n0 = (nt - G.tile_begin) * BN;
      for (int kb = 0; kb < nk; ++kb) {
        // absmax of every piece this thread decodes in this stage
        float amax[BN / 128];
#pragma unroll
        for (int i = 0; i < BN / 128; ++i) {
          const int pc = dt + 128 * i;
          int wrow, kblk;
          if constexpr (DX) {
            wrow = kb * kBK + (pc & 63);
            kblk = (n0 >> 6) + (pc >> 6);
          } else {
            wrow = n0 + pc;
            kblk = kb;
          }
          const bool in = DX ? (kblk < G.ld_absmax) : (wrow < G.ncols);
          amax[i] = in ? __bfloat162float(G.absmax[(size_t)wrow * G.ld_absmax + kblk]) : 0.0f;
        }
        if (!warp_wait(bar_full + 8 * stage, phase, abort_flag, p.status)) {
          ok = false;
          break;
        }
        const uint32_t sx = base + stage * L::STAGE_BYTES;
#pragma unroll
        for (int i = 0; i < BN / 128; ++i) {
          const int pc = dt + 128 * i;
          uint32_t src, dst;
          if constexpr (DX) {
            src = sx + L::OFF_C + (pc & 63) * (BN / 2) + (pc >> 6) * 32;
            dst = sx + L::OFF_W + (pc >> 6) * 8192 + (pc & 63) * 128;
          } else {
            src = sx + L::OFF_C + pc * 32;
            dst = sx + L::OFF_W + pc * 128;
          }
          nf4_decode_piece(src, dst, amax[i], levels);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_dec + 8 * stage);
        if (++stage == STAGES) stage = 0, phase ^= 1u;
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int MODE, int BN, int RP, bool NF4, bool ROPE>
static cudaError_t launch_one(const GemmParams &p, int grid, cudaStream_t st) {
  using L = GemmSmem<BN, RP, NF4>;
  auto kern = lora_gemm_kernel<MODE, BN, RP, NF4, ROPE>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::TOTAL);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  kern<<<grid, NF4 ? 320 : 192, L::TOTAL, st>>>(p);
  note_launch();
  return cudaGetLastError();
}

template <int MODE, int RP>
static cudaError_t launch_rp(const GemmParams &p, bool rope, bool nf4, int grid, cudaStream_t st) {
  if (nf4) {
    if (rope) return launch_one<MODE, 256, RP, true, MODE == kModeFwd>(p, grid, st);
    return launch_one<MODE, 256, RP, true, false>(p, grid, st);
  }
  if (rope) return launch_one<MODE, 256, RP, false, MODE == kModeFwd>(p, grid, st);
  return launch_one<MODE, 256, RP, false, false>(p, grid, st);
}

cudaError_t launch_gemm(const GemmParams &p, int mode, int rp, bool rope, bool nf4, int grid,
                        cudaStream_t st) {
  if (mode == kModeFwd) {
    switch (rp) {
      case 16: return launch_rp<kModeFwd, 16>(p, rope, nf4, grid, st);
      case 32: return launch_rp<kModeFwd, 32>(p, rope, nf4, grid, st);
      case 64: return launch_rp<kModeFwd, 64>(p, rope, nf4, grid, st);
    }
  } else {
    switch (rp) {
      case 16: return launch_rp<kModeDx, 16>(p, false, nf4, grid, st);
      case 32: return launch_rp<kModeDx, 32>(p, false, nf4, grid, st);
      case 64: return launch_rp<kModeDx, 64>(p, false, nf4, grid, st);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace lora
