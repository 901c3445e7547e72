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
#include "gemm_common.cuh"

namespace lora {

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
        epi_rank_to_smem<RP>(tmem + t_lane + BN, base + L::OFF_SR, row, p.scale,
                             DX && nt == 0 && row_ok, p.ut_hi, p.ut_lo, Mp, grow);
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar_sr_ready);
      }
      if (!warp_wait(bar_acc_full, tile_count & 1, abort_flag, p.status)) break;
      tc_fence_after();
      const int ncols = min(BN, G.ncols - n0);
      __nv_bfloat16 *orow = G.out + (size_t)(row_ok ? grow : 0) * G.ncols + n0;
      const float *cs = ROPE ? rope_row(p, grow, row_ok) : nullptr;
      epi_store_tile<BN, ROPE>(tmem + t_lane, orow, row_ok, ncols, DX && p.accumulate, cs);
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
