// Fused LoRA GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// FWD mode  ("UnSloth加速微调体验" §算子融合, §RoPE缓存集成):
//     y  = x·Wᵀ + s·(x·Aᵀ)·Bᵀ = [x | s·v]·[W | B]ᵀ     [optionally RoPE per head]
// DX mode   (same page, §反向传播优化):
//     dX = dY·W + s·(dY·B)·A = [dY | s·u]·[W ; A]
// s·v = s·x·Aᵀ and s·u = s·dY·B come from the rank pass (skinny.cu), so the
// rank-r term is one or two extra 64-wide K-blocks at the end of each
// tile's reduction, streamed through the same pipeline slots as the main
// K-blocks.  Output tiles are therefore independent of each other.
//
// A cluster of two CTAs computes one (256·MB) x 256 output tile with
// tcgen05.mma.cta_group::2: for each of the tile's MB m-blocks (256 rows),
// CTA c (c = 0, 1) holds rows [128c, 128c+128) of the m-block's activation
// rows, and rows [128c, 128c+128) of the W tile (the N half); the tensor
// cores of both SMs work on the pair tile, and each SM stages half of the W
// bytes a one-SM 128 x 256 tile would need.  MB = 1: the two 256-column
// TMEM accumulators alternate between tiles, so a tile's epilogue overlaps
// the next tile's main loop.  MB = 2: each W K-block (decoded once, for NF4)
// feeds both m-blocks, one accumulator each; the MMA of a new tile waits for
// the drain of the accumulator it writes, m-block 0 being drained first.
//
// Roles (both CTAs unless noted; NF4 rings as in PairSmem):
//   warp 0     TMA producer: own halves of x/dY and (bf16) of W per main
//              K-block; own halves of s·v / s·u and (bf16) of B / A per
//              rank K-block.  Completion is counted on the even CTA's
//              barriers.
//   warp 1     TMEM owner (pair allocation, 2 x 256 columns); in the even
//              CTA also the single MMA issuer, whose commits are multicast
//              to both CTAs.
//   warps 2-5  epilogue of the CTA's own 128 rows: TMEM -> (RoPE) -> bf16
//              -> shared-memory staging -> TMA bulk store of whole lines
//              (dX with accumulate: plain loads/stores adding to the values
//              already there).
//   warps 6-13 NF4 only: decode the CTA's own half of the W tile through the
//              16-entry NF4 codebook, scaled by the block absmax ("Unsloth教程"
//              §显存优化策略: NF4 base weight).  Two groups of four warps take
//              alternate K-blocks, one thread per 64-element row piece, so
//              each group has two stage times per K-block it decodes.
//   warp 14    NF4 only: TMA producer of the CTA's own code bytes, into a
//              ring of its own that runs ahead of the x ring.
#pragma once
#include <string>

#include "gemm_common.cuh"

namespace lora {

// Threads per CTA: producer, MMA, 4 epilogue warps (+ 8 NF4 decode warps
// and the NF4 code producer).
constexpr int pair_threads(bool nf4) { return nf4 ? 480 : 192; }
constexpr int kNf4DecodeWarps = 8;

// Shared-memory layout.  bf16 W: each pipeline stage holds the x tile and
// the W tile.  NF4 W: three rings.  The x ring (released by the MMA) holds
// the activation tiles; the code ring holds the 4-bit codes of the CTA's W
// half and is released by the decoders as soon as they have read a slot, so
// that the codes run well ahead of the MMA (decoding sits between their
// landing and the MMA); the decoded W tiles have a ring of their own.  A
// rank K-block's B or A tile is copied straight into the W ring.  The two
// NF4 decode groups take alternate K-blocks.  A parity wait is only
// unambiguous for a waiter at most one phase ahead of the barrier, so each
// waiter must see every phase of its barrier: the code and W rings have an
// even number of slots, so that each slot belongs to one group.
template <bool NF4, bool STAGED_ROPE = false, int MB = 1, int FV = 0>
struct PairSmem {
  static constexpr int X_BYTES = 128 * 128;  // own 128 rows x 64 K of one m-block
  static constexpr int W_BYTES = 128 * 128;  // own 128 N-rows x 64 K
  static constexpr int C_BYTES = NF4 ? 128 * 32 : 0;  // own half of a K-block's codes
  static constexpr int OFF_W = MB * X_BYTES;  // bf16: W inside the stage
  static constexpr int STAGE_BYTES = MB * X_BYTES + (NF4 ? 0 : W_BYTES);
  static constexpr int C_STAGES = NF4 ? 4 : 0;
  static constexpr int W_STAGES = NF4 ? (MB == 2 ? 4 : 6) : 0;
  static constexpr int CRING_BYTES = C_STAGES * C_BYTES;
  static constexpr int WRING_BYTES = W_STAGES * W_BYTES;
  static constexpr int EPI_BYTES = 4 * 2 * 2048;  // per epilogue warp: two 2 KB staging buffers
  static constexpr int AMAX_PRE = NF4 ? 4 : 0;    // absmax prefetch distance (a group's K-blocks)
  static constexpr int AMAX_BYTES = AMAX_PRE * 256 * 4;  // per decode thread
  // RoPE with staged cos / sin: per epilogue warp 32 rows of one half
  static constexpr int CS_BYTES = STAGED_ROPE ? 4 * 32 * kRopeRowPitch : 0;
  // Down-projection in the GEMM (FV = padded width of v, 64 or 128): the s·v
  // operand of this CTA's 128 rows [FV/64 atoms of 128 rows x 128 B, 128-byte
  // swizzle], whose bytes also serve, while a segment's first tile forms v,
  // as a ring of four A tiles [FV/2 rows x 64 K each]
  static constexpr int SV_BYTES = FV * 256;
  static constexpr int A_SLOT_BYTES = FV * 64;
  static constexpr int MISC_BYTES = 1024;
  static constexpr int FIXED = WRING_BYTES + CRING_BYTES + EPI_BYTES + AMAX_BYTES + CS_BYTES +
                               SV_BYTES + MISC_BYTES + 1024;
  static constexpr int STAGES_FIT = (kSmemLimit - FIXED) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static constexpr int OFF_WRING = STAGES * STAGE_BYTES;
  static constexpr int OFF_CRING = OFF_WRING + WRING_BYTES;
  static constexpr int OFF_EPI = OFF_CRING + CRING_BYTES;
  static constexpr int OFF_AMAX = OFF_EPI + EPI_BYTES;
  static constexpr int OFF_CS = OFF_AMAX + AMAX_BYTES;
  static constexpr int OFF_SV = OFF_CS + CS_BYTES;
  static constexpr int OFF_MISC = OFF_SV + SV_BYTES;
  static constexpr int TOTAL = OFF_MISC + MISC_BYTES + 1024;
  static constexpr int NUM_BARS = 2 * STAGES + 2 * C_STAGES + 2 * W_STAGES + 5 +
                                  (STAGED_ROPE ? 4 : 0) + (FV ? 11 : 0);
  static_assert(OFF_SV % 1024 == 0, "s·v region alignment");
  static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");
  static_assert(STAGES >= 3 && (!NF4 || (W_STAGES >= 4 && C_STAGES >= 4)), "pipeline depth");
  static_assert(!NF4 || (W_STAGES % 2 == 0 && C_STAGES % 2 == 0), "one decode group per slot");
  static_assert(8 * NUM_BARS + 16 <= MISC_BYTES, "barriers fit");
  static_assert(TOTAL <= kSmemLimit, "shared memory budget");
};

// Walk of one NF4 decode thread over its absmax elements, K-block by
// K-block, across the tiles of its CTA pair (FWD: row nh + pc, column kb;
// DX: row kb·64 + pc/2 of the K-group's W, column nh/64 + pc%2).
template <bool DX>
struct Nf4Cursor {
  TileIter it;
  int kb, len;                        // K-block in the tile; K-blocks per tile
  const __nv_bfloat16 *e;             // absmax element of K-block kb
  const __nv_bfloat16 *p1;            // element at the first K-block of the second K-group
  long long step;                     // elements per K-block
  int split;                          // first K-block of the second K-group
  bool in;                            // the piece lies inside W
  __device__ void tile(const GemmParams &p, int pc, int crank, int nk) {
    const int nt = it.nt();
    const WHalf wh = w_half(p, nt, (uint32_t)crank);
    const GemmGroup &G = *wh.g;
    const int nh = wh.nh;
    len = nk + (DX ? p.grp[0].n_extra : G.n_extra);
    if constexpr (DX) {
      const int ld = p.grp[0].ld_absmax;
      const int kblk = (nh >> 6) + (pc & 1);
      in = kblk < ld;
      step = 64ll * ld;
      e = p.grp[0].absmax + (long long)(pc >> 1) * ld + kblk;
      p1 = p.kgroups > 1 ? p.grp[1].absmax + (long long)(pc >> 1) * ld + kblk : e;
      split = p.kgroups > 1 ? p.ksplit : nk;
    } else {
      const int wrow = nh + pc;
      in = wrow < G.ncols;
      step = 1;
      e = p1 = G.absmax + (long long)(in ? wrow : 0) * G.ld_absmax;
      split = nk;
    }
  }
  __device__ void init(const GemmParams &p, int worker, int pc, int crank, int nk) {
    it.init(p.sched, worker);
    kb = 0;
    if (it.valid()) tile(p, pc, crank, nk);
  }
  __device__ bool valid() const { return it.valid(); }
  __device__ const __nv_bfloat16 *elem() const { return e; }
  __device__ void advance(const GemmParams &p, int pc, int crank, int nk) {
    if (!it.valid()) return;
    if (++kb == len) {
      kb = 0;
      it.next();
      if (it.valid()) tile(p, pc, crank, nk);
    } else if (kb == split) {
      e = p1;
    } else {
      e += step;
    }
  }
};

template <int MODE, bool NF4, bool ROPE, int MB, int FV, bool F16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(pair_threads(NF4), 1)
    lora_gemm_pair_kernel(const __grid_constant__ GemmParams p) {
  // RoPE cos / sin staged in shared memory (bf16 W; the NF4 rings leave no room)
  constexpr bool STAGED = ROPE && !NF4;
  using L = PairSmem<NF4, STAGED, MB, FV>;
  static_assert(MB == 1 || MB == 2, "m-blocks per tile");
  static_assert(FV == 0 || (MODE == kModeFwd && !NF4 && MB == 1 && (FV == 64 || FV == 128)),
                "down-projection in the GEMM: bf16 forward, one m-block per tile");
  constexpr int STAGES = L::STAGES;
  constexpr int BN = 256;
  constexpr bool DX = MODE == kModeDx;
  constexpr int NUM_DEC_WARPS = kNf4DecodeWarps;
  constexpr uint16_t kBoth = 0x3;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_addr(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (base - raw_base);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint32_t crank = cluster_ctarank();
  const bool leader = crank == 0;
  const int pair = blockIdx.x >> 1;

  constexpr int WST = L::W_STAGES;
  constexpr int CST = L::C_STAGES;
  const uint32_t bar_full = base + L::OFF_MISC;       // [S] leader: TMA of both CTAs
  const uint32_t bar_empty = bar_full + 8 * STAGES;   // [S] both: pair MMA done
  const uint32_t bar_cfull = bar_empty + 8 * STAGES;  // [CST] both: own NF4 codes (or B) landed
  const uint32_t bar_cempty = bar_cfull + 8 * CST;    // [CST] both: the decode group read the slot
  const uint32_t bar_wfull = bar_cempty + 8 * CST;    // [WST] leader: W slot of both CTAs ready
  const uint32_t bar_wempty = bar_wfull + 8 * WST;    // [WST] both: pair MMA done with W slot
  const uint32_t bar_acc_full = bar_wempty + 8 * WST; // [2] both: accumulator b ready
  const uint32_t bar_acc_empty = bar_acc_full + 16;   // [2] leader: 8 warps drained b
  const uint32_t bar_drain = bar_acc_empty + 16;      // leader
  const uint32_t bar_cs = bar_drain + 8;              // [4] STAGED: cos / sin of epilogue warp q
  // FV: A-tile ring in the s·v region, v complete, s·v staged, s·v free
  const uint32_t bar_afull = bar_cs + (STAGED ? 32 : 0);  // [4] leader: A tiles of both CTAs
  const uint32_t bar_aempty = bar_afull + 32;              // [4] both: v MMAs done with the slot
  const uint32_t bar_vfull = bar_aempty + 32;              // both: v of the segment complete
  const uint32_t bar_svready = bar_vfull + 8;              // leader: 8 warps staged s·v
  const uint32_t bar_svfree = bar_svready + 8;             // both: the segment's MMAs read s·v
  const int misc_words = (8 * L::NUM_BARS) / 4;
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::OFF_MISC) + misc_words;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int c = 0; c < CST; ++c) {
      mbar_init(bar_cfull + 8 * c, 1);
      mbar_init(bar_cempty + 8 * c, NUM_DEC_WARPS / 2);  // the four warps of one group
    }
    for (int w = 0; w < WST; ++w) {
      mbar_init(bar_wfull + 8 * w, NUM_DEC_WARPS);  // one decode group in each of 2 CTAs
      mbar_init(bar_wempty + 8 * w, 1);
    }
    mbar_init(bar_acc_full, 1);
    mbar_init(bar_acc_full + 8, 1);
    mbar_init(bar_acc_empty, 8);
    mbar_init(bar_acc_empty + 8, 8);
    mbar_init(bar_drain, 1);
    if constexpr (STAGED)
      for (int q = 0; q < 4; ++q) mbar_init(bar_cs + 8 * q, 1);
    if constexpr (FV > 0) {
      for (int a = 0; a < 4; ++a) {
        mbar_init(bar_afull + 8 * a, 1);
        mbar_init(bar_aempty + 8 * a, 1);
      }
      mbar_init(bar_vfull, 1);
      mbar_init(bar_svready, 8);
      mbar_init(bar_svfree, 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {  // one warp in each CTA of the pair allocates together
    tmem_alloc_pair(smem_addr(tmem_holder), 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // barriers of both CTAs initialised before any remote use
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  grid_dep_launch();
  grid_dep_wait();  // the previous kernel's outputs (s·v, dY) are complete
  const int nk = p.K / kBK;  // main K-blocks
  // the even CTA's copies of the barriers the pair shares
  const uint32_t lead_full = map_shared_rank(bar_full, 0);
  const uint32_t lead_wfull = map_shared_rank(bar_wfull, 0);
  const uint32_t lead_acc_empty = map_shared_rank(bar_acc_empty, 0);
  const uint32_t lead_afull = FV > 0 ? map_shared_rank(bar_afull, 0) : 0u;
  const uint32_t lead_svready = FV > 0 ? map_shared_rank(bar_svready, 0) : 0u;
  const uint32_t sv_base = base + L::OFF_SV;

  if (warp == 0) {
    // ================================================================ producer
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_act);
      tma_prefetch_desc(&p.tm_sv);
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;  // K-blocks issued: stage s took every STAGES-th from the s-th
      int aslot = 0;   // FV: A-tile ring
      uint32_t aphase = 0;
      int a_issued = 0;
      int segs = 0;    // FV: segments started
      const int fv_h = p.fv_nv / 2;  // A rows per CTA
      bool ok = true;
      TileIter it;
      for (it.init(p.sched, pair); ok && it.valid(); it.next()) {
        const bool vtile = FV > 0 && it.seg_start();
        if (vtile) {
          // the previous segment's rank MMAs are done with the s·v region
          if (segs > 0 &&
              !mbar_wait(bar_svfree, (uint32_t)(segs - 1) & 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          ++segs;
        }
        const int m = it.m(), nt = it.nt();
        const WHalf wh = w_half(p, nt, crank);
        const GemmGroup &G = *wh.g;             // this CTA's weight group
        const int nh = wh.nh;                   // first N index of this CTA's half
        const int row0 = m * (256 * MB) + (int)crank * 128;  // m-block mb: + 256·mb
        const int ne = DX ? p.grp[0].n_extra : G.n_extra;
        for (int kb = 0; kb < nk + ne; ++kb) {
          if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          const uint32_t sx = base + stage * L::STAGE_BYTES;
          const uint32_t fb = lead_full + 8 * stage;
          if (kb < nk) {
            if (leader)
              mbar_arrive_expect_tx(bar_full + 8 * stage,
                                    2 * (MB * L::X_BYTES + (NF4 ? 0 : L::W_BYTES)));
#pragma unroll
            for (int mb = 0; mb < MB; ++mb)
              tma_load_2d_pair(sx + mb * L::X_BYTES, &p.tm_act, fb, kb * kBK, row0 + mb * 256);
            // DX: the reduction may run over two projections' W (K-groups)
            const int gk = (DX && p.kgroups > 1 && kb >= p.ksplit) ? 1 : 0;
            const CUtensorMap *tw = DX ? &p.grp[gk].tm_w : &G.tm_w;
            const int wk = kb - (gk ? p.ksplit : 0);
            if constexpr (!NF4) {
              if constexpr (DX) {  // W as MN-major operand: 2 boxes [64 rows x 64]
                tma_load_2d_pair(sx + L::OFF_W, tw, fb, nh, wk * kBK);
                tma_load_2d_pair(sx + L::OFF_W + 8192, tw, fb, nh + 64, wk * kBK);
              } else {
                tma_load_2d_pair(sx + L::OFF_W, tw, fb, kb * kBK, nh);
              }
            }
            if (vtile) {
              // this CTA's rows of the A tile of K-block kb into the ring
              if (!mbar_wait(bar_aempty + 8 * aslot, aphase ^ 1u, abort_flag, p.status)) {
                ok = false;
                break;
              }
              if (leader) mbar_arrive_expect_tx(bar_afull + 8 * aslot, 2 * fv_h * 128);
              tma_load_2d_pair(sv_base + aslot * L::A_SLOT_BYTES,
                               p.fv_two ? &p.tm_a[crank] : &p.tm_a[0], lead_afull + 8 * aslot,
                               kb * kBK, p.fv_two ? 0 : (int)crank * fv_h);
              ++a_issued;
              if (++aslot == 4) aslot = 0, aphase ^= 1u;
            }
          } else if (FV > 0) {
            // rank K-block e: B only (s·v is staged in shared memory)
            const int e = kb - nk;
            if (leader) mbar_arrive_expect_tx(bar_full + 8 * stage, 2 * L::W_BYTES);
            tma_load_2d_pair(sx + L::OFF_W, &G.tm_b, fb, e * kBK + G.b_shift, nh);
          } else {
            // rank K-block e: s·v (or s·u) columns and the matching B (or A)
            const int e = kb - nk;
            const GemmGroup &R = DX ? p.grp[0] : G;
            if constexpr (NF4) {
              // B / A goes straight into the W ring (copied by the decode
              // group that owns the slot, see the code producer)
              if (leader) mbar_arrive_expect_tx(bar_full + 8 * stage, 2 * MB * L::X_BYTES);
#pragma unroll
              for (int mb = 0; mb < MB; ++mb)
                tma_load_2d_pair(sx + mb * L::X_BYTES, &p.tm_sv, fb, R.sv_col + e * kBK,
                                 row0 + mb * 256);
            } else {
              if (leader)
                mbar_arrive_expect_tx(bar_full + 8 * stage, 2 * (MB * L::X_BYTES + L::W_BYTES));
#pragma unroll
              for (int mb = 0; mb < MB; ++mb)
                tma_load_2d_pair(sx + mb * L::X_BYTES, &p.tm_sv, fb, R.sv_col + e * kBK,
                                 row0 + mb * 256);
              if constexpr (DX) {  // A [rl, k] MN-major: 2 boxes [64 k-columns x 64 rank rows]
                tma_load_2d_pair(sx + L::OFF_W, &R.tm_b, fb, nh, e * kBK);
                tma_load_2d_pair(sx + L::OFF_W + 8192, &R.tm_b, fb, nh + 64, e * kBK);
              } else {             // B [n, r] K-major: own 128 rows x 64
                tma_load_2d_pair(sx + L::OFF_W, &R.tm_b, fb, e * kBK + R.b_shift, nh);
              }
            }
          }
          ++issued;
          if (++stage == STAGES) stage = 0, phase ^= 1u;
        }
      }
      // Let every completion the leader multicasts to this CTA land before
      // the CTA may exit (bounded: after an abort some never come).
      const uint64_t lim = *abort_flag ? 20000000ull : 1000000000ull;
      for (int s = 0; s < STAGES; ++s) {
        const int fills = issued > s ? (issued - s + STAGES - 1) / STAGES : 0;
        if (fills > 0) mbar_wait_quiet(bar_empty + 8 * s, (uint32_t)((fills - 1) & 1), lim);
      }
      if constexpr (FV > 0) {
        for (int a = 0; a < 4; ++a) {
          const int uses = a_issued > a ? (a_issued - a + 3) / 4 : 0;
          if (uses > 0) mbar_wait_quiet(bar_aempty + 8 * a, (uint32_t)((uses - 1) & 1), lim);
        }
        if (segs > 0) mbar_wait_quiet(bar_svfree, (uint32_t)((segs - 1) & 1), lim);
      }
    }
  } else if (warp == 1) {
    // ===================================================== MMA (even CTA)
    if (leader && lane == 0) {
      constexpr uint32_t idesc = make_idesc(256, BN, false, DX, F16);
      const uint32_t idesc_v = make_idesc(256, FV > 0 ? p.fv_nv : 16, false, false, F16);
      int stage = 0;
      uint32_t phase = 0;
      int wslot = 0;
      uint32_t wphase = 0;
      int aslot = 0;  // FV: A-tile ring
      uint32_t aphase = 0;
      int segs = 0;
      int tile_count = 0;
      int used[2] = {0, 0};  // tiles issued into each accumulator buffer
      bool ok = true;
      TileIter it;
      for (it.init(p.sched, pair); ok && it.valid(); it.next(), ++tile_count) {
        const GemmGroup &G = p.grp[group_of(p, it.nt())];
        const int ne = DX ? p.grp[0].n_extra : G.n_extra;
        const int buf = tile_count & 1;  // MB = 1: the accumulator of this tile
        const bool vtile = FV > 0 && it.seg_start();
        if constexpr (MB == 1) {
          if (used[buf] > 0 && !mbar_wait_cluster(bar_acc_empty + 8 * buf, (used[buf] - 1) & 1,
                                                  abort_flag, p.status))
            break;
          ++used[buf];
          // v goes to the other buffer's first columns: its previous tile
          // must be drained
          if (vtile && used[buf ^ 1] > 0 &&
              !mbar_wait_cluster(bar_acc_empty + 8 * (buf ^ 1), (used[buf ^ 1] - 1) & 1,
                                 abort_flag, p.status))
            break;
        }
        if (vtile) ++segs;
        tc_fence_after();
        for (int kb = 0; ok && kb < nk + ne; ++kb) {
          if (!mbar_wait(bar_full + 8 * stage, phase, abort_flag, p.status)) {
            ok = false;
            break;
          }
          if (NF4 && !mbar_wait_cluster(bar_wfull + 8 * wslot, wphase, abort_flag, p.status)) {
            ok = false;
            break;
          }
          if (vtile && kb < nk &&
              !mbar_wait(bar_afull + 8 * aslot, aphase, abort_flag, p.status)) {
            ok = false;
            break;
          }
          if (FV > 0 && vtile && kb == nk &&
              !mbar_wait_cluster(bar_svready, (uint32_t)(segs - 1) & 1u, abort_flag, p.status)) {
            ok = false;  // the first rank K-block needs the segment's s·v staged
            break;
          }
          tc_fence_after();
          const uint32_t sx = base + stage * L::STAGE_BYTES;
          const uint32_t sw = NF4 ? base + L::OFF_WRING + wslot * L::W_BYTES : sx + L::OFF_W;
          // FV rank K-block: the activation is atom (sv_col/64 + e) of s·v
          const uint32_t sa = (FV > 0 && kb >= nk)
                                  ? sv_base + (uint32_t)(G.sv_col / 64 + (kb - nk)) * 16384u
                                  : sx;
#pragma unroll
          for (int mb = 0; mb < MB; ++mb) {
            if (MB == 2 && kb == 0 && tile_count > 0) {
              // accumulator mb is free once the previous tile's m-block mb is drained
              if (!mbar_wait_cluster(bar_acc_empty + 8 * mb, (tile_count - 1) & 1, abort_flag,
                                     p.status)) {
                ok = false;
                break;
              }
              tc_fence_after();
            }
            const uint32_t t_acc = tmem + (MB == 1 ? buf : mb) * BN;
#pragma unroll
            for (int ks = 0; ks < kBK / 16; ++ks) {
              const uint64_t da = make_sdesc(sa + mb * L::X_BYTES + ks * 32, 16, 1024, kSw128);
              uint64_t dw;
              if constexpr (DX)  // MN-major: 16 K-rows per step; two 64-wide blocks 8 KB apart
                dw = make_sdesc(sw + ks * 2048, 8192, 1024, kSw128);
              else
                dw = make_sdesc(sw + ks * 32, 16, 1024, kSw128);
              tc_mma_pair(t_acc, da, dw, idesc, (kb | ks) != 0 ? 1u : 0u);
            }
            // MB = 2: m-block mb's accumulator is complete after its last
            // K-block, before the other m-block's MMAs of that K-block
            if (MB == 2 && kb == nk + ne - 1) tc_commit_pair(bar_acc_full + 8 * mb, kBoth);
          }
          if (!ok) break;
          if (vtile && kb < nk) {
            // v += x·Aᵀ on the same x tile (v in the other buffer's columns)
            const uint32_t t_v = tmem + (buf ^ 1) * BN;
            const uint32_t sa_ring = sv_base + aslot * L::A_SLOT_BYTES;
#pragma unroll
            for (int ks = 0; ks < kBK / 16; ++ks)
              tc_mma_pair(t_v, make_sdesc(sx + ks * 32, 16, 1024, kSw128),
                          make_sdesc(sa_ring + ks * 32, 16, 1024, kSw128), idesc_v,
                          (kb | ks) != 0 ? 1u : 0u);
            tc_commit_pair(bar_aempty + 8 * aslot, kBoth);
            if (++aslot == 4) aslot = 0, aphase ^= 1u;
            if (kb == nk - 1) tc_commit_pair(bar_vfull, kBoth);  // v complete
          }
          tc_commit_pair(bar_empty + 8 * stage, kBoth);
          if (++stage == STAGES) stage = 0, phase ^= 1u;
          if constexpr (NF4) {
            tc_commit_pair(bar_wempty + 8 * wslot, kBoth);
            if (++wslot == WST) wslot = 0, wphase ^= 1u;
          }
        }
        if (!ok) break;
        // the run's last tile: its rank MMAs were the last reads of s·v
        if (FV > 0 && it.seg_last()) tc_commit_pair(bar_svfree, kBoth);
        if constexpr (MB == 1) tc_commit_pair(bar_acc_full + 8 * buf, kBoth);
      }
      if (*abort_flag) {
        tc_commit_pair(bar_drain, 0x1);
        mbar_wait_quiet(bar_drain, 0, 100000000ull);
      }
    }
  } else if (warp < 6) {
    // ================================================================ epilogue
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const uint32_t t_lane = (uint32_t)(q * 32) << 16;
    const uint32_t epi_buf = base + L::OFF_EPI + (uint32_t)q * 4096u;
    const uint32_t cs_bar = bar_cs + 8 * q;
    const uint32_t srow = base + L::OFF_CS + (uint32_t)row * kRopeRowPitch;
    uint32_t cs_phase = 0;
    uint32_t nstore = 0;  // SwiGLU: stores issued by this warp
    int segs = 0;         // FV: segments whose s·v this warp staged
    bool cs_pending = false;  // a staged half has not been waited for
    int tile_count = 0;
    TileIter it;
    bool ok = true;
    for (it.init(p.sched, pair); ok && it.valid(); it.next(), ++tile_count) {
      const int m = it.m(), nt = it.nt();
      const GemmGroup &G = p.grp[group_of(p, nt)];
      if (FV > 0 && it.seg_start()) {
        // v of the segment (in the other buffer): s·v into the operand region
        if (!warp_wait(bar_vfull, (uint32_t)segs & 1u, abort_flag, p.status)) break;
        ++segs;
        tc_fence_after();
        stage_sv<FV, F16>(tmem + t_lane + ((tile_count & 1) ^ 1) * BN, base + L::OFF_SV, row, p.fv_nv,
                     p.fv_scale);
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(lead_svready);
      }
      // output columns of the tile (SwiGLU: 128 of h, g and u)
      const int n0 = p.swiglu ? nt * 128 : (nt - G.tile_begin) * BN;
      const int ncols = min(p.swiglu ? 128 : BN, G.ncols - n0);
#pragma unroll 1
      for (int mb = 0; mb < MB; ++mb) {
        const int acc = MB == 1 ? (tile_count & 1) : mb;
        const uint32_t par = MB == 1 ? (uint32_t)(tile_count >> 1) & 1u : (uint32_t)tile_count & 1u;
        const int wrow0 = (m * MB + mb) * 256 + (int)crank * 128 + q * 32;  // warp's first row
        const int grow = wrow0 + lane;
        const bool row_ok = grow < p.M;
        const float *cs = ROPE ? rope_row(p, grow, row_ok) : nullptr;
        if constexpr (STAGED) {  // fetched while the accumulator is still being produced
          rope_stage(cs, 0, srow, cs_bar, lane);
          cs_pending = true;
        }
        if (!warp_wait(bar_acc_full + 8 * acc, par, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if ((DX || !ROPE) && p.accumulate) {  // read-modify-write of the output: plain loads and stores
          uint16_t *orow = G.out + (size_t)(row_ok ? grow : 0) * G.ncols + n0;
          if (!NF4 && p.dropout)   // the masked adapter term of dX under LoRA dropout
            epi_accumulate_tile<BN, F16, !NF4>(tmem + t_lane + acc * BN, orow, row_ok, ncols,
                                               p.acc_scale, &p, grow, n0);
          else
            epi_accumulate_tile<BN, F16>(tmem + t_lane + acc * BN, orow, row_ok, ncols,
                                         p.acc_scale);
        } else if (!DX && !ROPE && p.swiglu) {
          epi_store_swiglu<F16>(tmem + t_lane + acc * BN, epi_buf, p, n0, wrow0, ncols, lane, nstore);
        } else {
          if (!epi_store_tile_tma<BN, ROPE, STAGED, F16>(tmem + t_lane + acc * BN, epi_buf, &G.tm_out,
                                                    n0, wrow0, ncols, cs, srow, cs_bar, cs_phase,
                                                    lane, abort_flag, p.status)) {
            ok = false;
            break;
          }
          cs_pending = false;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(lead_acc_empty + 8 * acc);
      }
    }
    if (STAGED && cs_pending)  // no copy may land after the CTA exits
      mbar_wait_quiet(cs_bar, cs_phase, 100000000ull);
    if (lane == 0) bulk_wait_all();  // every output store has completed
    __syncwarp();
  } else if constexpr (NF4) {
    if (warp < 6 + kNf4DecodeWarps) {
    // ============================================================= NF4 decode
    // Group gr = 0 / 1 (warps 6-9 / 10-13) decodes the K-blocks whose running
    // index across the CTA's tiles is even / odd; thread pc of a group
    // decodes row piece pc:
    // FWD: piece pc = row pc of this CTA's W half [128 rows x 64].
    // DX:  the half is [64 n-rows x 128 k-columns] = two boxes of [64 x 64];
    //      piece pc = row pc / 2 of box pc % 2 (a warp's pieces are then
    //      one contiguous kilobyte of the code slot).
    // The codes of running K-block g sit in code slot g % CST; the group
    // releases the slot once it has decoded them.
    // A rank K-block's B / A tile is copied into the W slot by one lane of
    // the group (counted on the code slot's barrier); the group waits for
    // it and passes the slot on.
    // Decoded tiles go to the W ring (slot g % WST for running K-block g),
    // whose slots the MMA releases through bar_wempty.
    // The absmax of a piece is fetched AMAX_PRE of the group's K-blocks
    // ahead (cp.async into a per-thread shared ring) by a look-ahead cursor:
    // loaded at decode time it would stall every K-block by a memory latency.
    const int dt = threadIdx.x - 192;  // 0..255
    const int gr = dt >> 7, pc = dt & 127;
    constexpr int PRE = L::AMAX_PRE;
    const uint32_t ring = base + L::OFF_AMAX + (uint32_t)dt * 4u;  // slot j at ring + 1024 j
    float lvl[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) lvl[i] = kNf4Levels[i];
    Nf4Cursor<DX> cur, ahead;
    cur.init(p, pair, pc, (int)crank, nk);
    if (gr) cur.advance(p, pc, (int)crank, nk);  // group 1 starts at the second K-block
    ahead = cur;
    auto prefetch = [&](uint32_t slot) {
      if (ahead.valid() && ahead.kb < nk && ahead.in)
        cp_async_4(ring + slot * 1024u,
                   reinterpret_cast<const void *>(reinterpret_cast<uintptr_t>(ahead.elem()) &
                                                  ~uintptr_t(3)));
      cp_async_commit();
      ahead.advance(p, pc, (int)crank, nk);
      ahead.advance(p, pc, (int)crank, nk);
    };
    for (int j = 0; j < PRE; ++j) prefetch((uint32_t)j);
    // 32-byte code pieces of consecutive threads are contiguous: threads
    // whose pieces start in the same half of the 32 banks read their two
    // 16-byte halves in opposite orders, so each load touches every bank
    const uint32_t flip = (uint32_t)(pc >> 2) & 1u;
    const uint32_t c_off = DX ? (uint32_t)((pc >> 1) * 64 + (pc & 1) * 32) : (uint32_t)(pc * 32);
    const uint32_t w_off = DX ? (uint32_t)((pc & 1) * 8192 + (pc >> 1) * 128) : (uint32_t)(pc * 128);
    int gk = gr;     // running K-block index of this group (gr, gr + 2, ...)
    int wslot = gr;  // and every other slot of the W ring
    uint32_t wphase = 0;
    int ng = 0;      // K-blocks this group took a W slot for
    uint32_t slot = 0;
    while (cur.valid()) {
      const int kb = cur.kb;
      const int cst = gk % CST;
      const uint32_t cphase = (uint32_t)(gk / CST) & 1u;
      const uint32_t cbar = bar_cfull + 8 * cst;
      cp_async_wait<PRE - 1>();  // this K-block's absmax has landed
      float amax = 0.0f;
      if (kb < nk && cur.in) {
        const uint32_t w = ld_shared_u32(ring + slot * 1024u);
        const bool high = (reinterpret_cast<uintptr_t>(cur.elem()) & 2u) != 0;
        amax = __uint_as_float((high ? (w >> 16) : (w & 0xFFFFu)) << 16);
      }
      prefetch(slot);  // the slot just read refills for the group's K-block PRE ahead
      if (++slot == (uint32_t)PRE) slot = 0;
      // the W slot is free once the MMA of its previous use has completed
      if (!warp_wait(bar_wempty + 8 * wslot, wphase ^ 1u, abort_flag, p.status)) break;
      ++ng;
      const uint32_t sw = base + L::OFF_WRING + wslot * L::W_BYTES;
      if (kb >= nk && (warp & 3) == 2 && lane == 0) {
        // rank K-block e: this CTA's half of B [n, r] (K-major) or of A [rl, k]
        // (MN-major) into the W slot, counted on the code slot's barrier
        // (armed by the code producer)
        const int e = kb - nk;
        const WHalf wh = w_half(p, cur.it.nt(), crank);
        const GemmGroup &R = DX ? p.grp[0] : *wh.g;
        const int nh = wh.nh;
        if constexpr (DX) {
          tma_load_2d(sw, &R.tm_b, cbar, nh, e * kBK);
          tma_load_2d(sw + 8192, &R.tm_b, cbar, nh + 64, e * kBK);
        } else {
          tma_load_2d(sw, &R.tm_b, cbar, e * kBK + R.b_shift, nh);
        }
      }
      // this K-block's codes (or rank tile) landed
      if (!warp_wait(cbar, cphase, abort_flag, p.status)) break;
      if (kb < nk) {
        uint32_t words[8];
        nf4_load_codes(base + L::OFF_CRING + cst * L::C_BYTES + c_off, flip, words);
        nf4_decode_words(words, sw + w_off, nf4_table<F16>(lvl, amax));
        fence_proxy_async_smem();
        // the slot is released once its codes have been consumed: a release
        // right after the loads let the next copy overwrite bytes that some
        // lanes had not read yet
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_cempty + 8 * cst);
      } else {
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_cempty + 8 * cst);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(lead_wfull + 8 * wslot);
      // next K-block of this group: two code and W slots on
      gk += 2;
      wslot += 2;
      if (wslot >= WST) wslot -= WST, wphase ^= 1u;
      cur.advance(p, pc, (int)crank, nk);
      cur.advance(p, pc, (int)crank, nk);
    }
    cp_async_wait<0>();  // no copy may land after the CTA exits
    // and no release of the group's W slots (multicast by the MMA) may
    // still be in flight (bounded: after an abort some never come); the
    // group's j-th W slot took every (WST/2)-th of its K-blocks from the j-th
    if (lane == 0) {
      const uint64_t lim = *abort_flag ? 20000000ull : 1000000000ull;
      for (int j = 0; j < WST / 2; ++j) {
        const int uses = ng > j ? (ng - j + WST / 2 - 1) / (WST / 2) : 0;
        if (uses > 0)
          mbar_wait_quiet(bar_wempty + 8 * (gr + 2 * j), (uint32_t)((uses - 1) & 1), lim);
      }
    }
    } else if (lane == 0) {
      // ===================================================== NF4 code producer
      // Fills the code ring in running K-block order, paced by the decode
      // groups' releases only: the codes run up to CST K-blocks ahead of
      // decoding.  A rank K-block's slot carries no codes; its barrier is
      // armed for the B / A tile that the decode group copies into its W slot.
      int cst = 0;
      uint32_t cph = 0;
      int issued = 0;
      bool ok = true;
      TileIter it;
      for (it.init(p.sched, pair); ok && it.valid(); it.next()) {
        const int nt = it.nt();
        const WHalf wh = w_half(p, nt, crank);
        const GemmGroup &G = *wh.g;
        const int nh = wh.nh;
        const int ne = DX ? p.grp[0].n_extra : G.n_extra;
        for (int kb = 0; kb < nk + ne; ++kb) {
          if (!mbar_wait(bar_cempty + 8 * cst, cph ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          const uint32_t cb = bar_cfull + 8 * cst;
          if (kb < nk) {
            // DX: the reduction may run over two projections' W (K-groups)
            const int gk = (DX && p.kgroups > 1 && kb >= p.ksplit) ? 1 : 0;
            const CUtensorMap *tw = DX ? &p.grp[gk].tm_w : &G.tm_w;
            const int wk = kb - (gk ? p.ksplit : 0);
            const uint32_t sc = base + L::OFF_CRING + cst * L::C_BYTES;
            mbar_arrive_expect_tx(cb, L::C_BYTES);
            if constexpr (DX)  // codes [64 rows of W, 64 bytes = 128 k-columns]
              tma_load_2d(sc, tw, cb, nh / 2, wk * kBK);
            else               // codes [128 rows of W, 32 bytes]
              tma_load_2d(sc, tw, cb, kb * (kBK / 2), nh);
          } else {
            mbar_arrive_expect_tx(cb, L::W_BYTES);
          }
          ++issued;
          if (++cst == CST) cst = 0, cph ^= 1u;
        }
      }
      // no copy may land after the CTA exits: the last phase of every slot
      // completes (bounded: after an abort some never do)
      const uint64_t lim = *abort_flag ? 20000000ull : 1000000000ull;
      for (int c = 0; c < CST; ++c) {
        const int uses = issued > c ? (issued - c + CST - 1) / CST : 0;
        if (uses > 0) mbar_wait_quiet(bar_cfull + 8 * c, (uint32_t)((uses - 1) & 1), lim);
      }
    }
  }

  __syncthreads();
  cluster_sync_all();  // no remote arrival may target a CTA that has exited
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

// Name of a variant in the launch log:
// lora_gemm_pair_kernel<fwd|dx, bf16|f16|nf4[,rope][,mb2][,xa][,f16 for nf4]>.
inline std::string pair_kernel_name(bool fwd, bool nf4, bool rope, bool mb2, bool xa, bool f16) {
  std::string n = std::string("lora_gemm_pair_kernel<") + (fwd ? "fwd," : "dx,") +
                  (nf4 ? "nf4" : (f16 ? "f16" : "bf16"));
  if (rope) n += ",rope";
  if (mb2) n += ",mb2";
  if (xa) n += ",xa";
  if (nf4 && f16) n += ",f16";
  return n + ">";
}

template <int MODE, bool NF4, bool ROPE, int MB, int FV, bool F16>
static cudaError_t launch_pair_one(const GemmParams &p, int pairs, cudaStream_t st) {
  using L = PairSmem<NF4, ROPE && !NF4, MB, FV>;
  auto kern = lora_gemm_pair_kernel<MODE, NF4, ROPE, MB, FV, F16>;
  static std::atomic<uint64_t> attr_done{0};
  const cudaError_t e = smem_attr_once(attr_done, reinterpret_cast<const void *>(kern), L::TOTAL);
  if (e != cudaSuccess) return e;
  static const std::string name_s =
      pair_kernel_name(MODE == kModeFwd, NF4, ROPE, MB == 2, FV != 0, F16);
  const char *name = name_s.c_str();
  return launch_pdl(name, kern, dim3(2 * pairs), dim3(pair_threads(NF4)), L::TOTAL, st, 0u, p);
}

// Co-resident CTA pairs of one kernel on the current device (cached per
// device; 0 if the query fails).
template <int MODE, bool NF4, bool ROPE, int MB, int FV, bool F16>
static int pair_capacity() {
  using L = PairSmem<NF4, ROPE && !NF4, MB, FV>;
  auto kern = lora_gemm_pair_kernel<MODE, NF4, ROPE, MB, FV, F16>;
  static std::atomic<uint64_t> attr_done{0};
  static std::atomic<int> cached[kMaxDevices];  // pairs + 1; 0: not queried yet
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  const bool slot = dev >= 0 && dev < kMaxDevices;
  if (slot) {
    const int v = cached[dev].load(std::memory_order_relaxed);
    if (v > 0) return v - 1;
  }
  if (smem_attr_once(attr_done, reinterpret_cast<const void *>(kern), L::TOTAL) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(pair_threads(NF4), 1, 1);
  cfg.dynamicSmemBytes = L::TOTAL;
  int n = 0;  // cluster shape comes from the kernel's compile-time cluster dims
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) return 0;
  if (slot) cached[dev].store(n + 1, std::memory_order_relaxed);
  return n;
}

template <int MODE, bool NF4, bool ROPE, int MB, int FV, bool F16>
static cudaError_t run_or_query(const GemmParams &p, int pairs, int *cap, cudaStream_t st) {
  if (cap) return *cap = pair_capacity<MODE, NF4, ROPE, MB, FV, F16>(), cudaSuccess;
  return launch_pair_one<MODE, NF4, ROPE, MB, FV, F16>(p, pairs, st);
}

// Launch (cap == nullptr) or capacity query (*cap) of the variant
// (MODE, NF4, rope, mb, fv).  RoPE applies to the forward only; two
// m-blocks per tile are compiled for NF4 weights, the down-projection in the
// GEMM (fv = 64 or 128, the padded width of v it stages) for the bf16
// forward.
template <int MODE, bool NF4, bool F16>
static cudaError_t pair_dispatch(const GemmParams &p, bool rope, int mb, int fv, int pairs,
                                 int *cap, cudaStream_t st) {
  constexpr bool FWD = MODE == kModeFwd;
  if constexpr (NF4) {
    if (fv != 0) return cudaErrorInvalidValue;
    if (mb == 2)
      return (FWD && rope) ? run_or_query<MODE, NF4, FWD, 2, 0, F16>(p, pairs, cap, st)
                           : run_or_query<MODE, NF4, false, 2, 0, F16>(p, pairs, cap, st);
  } else if constexpr (FWD) {
    if (fv == 64)
      return rope ? run_or_query<MODE, NF4, true, 1, 64, F16>(p, pairs, cap, st)
                  : run_or_query<MODE, NF4, false, 1, 64, F16>(p, pairs, cap, st);
    if (fv == 128)
      return rope ? run_or_query<MODE, NF4, true, 1, 128, F16>(p, pairs, cap, st)
                  : run_or_query<MODE, NF4, false, 1, 128, F16>(p, pairs, cap, st);
  }
  if (mb != 1 || fv != 0) return cudaErrorInvalidValue;
  return (FWD && rope) ? run_or_query<MODE, NF4, FWD, 1, 0, F16>(p, pairs, cap, st)
                       : run_or_query<MODE, NF4, false, 1, 0, F16>(p, pairs, cap, st);
}

}  // namespace lora
