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
//
// DEC variant (KMAJOR, the small-M forward over the rows of an NF4 W): eight
// more warps decode P from 4-bit codes.  A problem with `nf4` set streams its
// codes [128 rows x 32 bytes] per chunk instead of P, through a deep ring of
// (Q, codes) stages (the codes are a quarter of P's bytes, so many chunks are
// in flight); each decode thread takes half a row (32 codes), looks them up
// in a 16-entry table scaled by the block's absmax (fetched a few chunks
// ahead by cp.async) and writes the 16-bit values, 128-byte swizzled, into a
// short ring of P tiles that the MMA reads.  A problem without codes loads P
// into that ring by TMA.
#include "gemm_common.cuh"
#include "kernels.h"
#include "skinny_out.cuh"

namespace lora {

// PER_SM = 2: a ring half as deep, so that two CTAs share an SM (the
// small-M forward's pass over W, where more CTAs in flight pay).
template <bool MN, int RP, bool DEC = false, int PER_SM = 1>
struct SkinnySmem {
  static constexpr int SMEM_BUDGET = PER_SM == 2 ? 115712 : kSmemLimit;
  static constexpr int P_BYTES = 128 * 128;  // [128 x 64] bf16 either way
  static constexpr int Q_BYTES = RP * 128;
  static constexpr int C_BYTES = DEC ? 128 * 32 : 0;  // NF4 codes of a P tile
  static constexpr int AMAX_PRE = 8;                  // absmax prefetch distance (chunks)
  static constexpr int DEC_THREADS = DEC ? 256 : 0;   // two per P row
  static constexpr int AMAX_BYTES = DEC ? AMAX_PRE * DEC_THREADS * 4 : 0;
  static constexpr int PST = DEC ? 4 : 0;             // DEC: ring of P tiles
  // a TMA stage: P (not DEC) and Q (MN: its hi and lo parts), codes (DEC)
  static constexpr int STAGE_BYTES = (DEC ? 0 : P_BYTES) + (MN ? 2 : 1) * Q_BYTES + C_BYTES;
  static constexpr int STAGES_FIT =
      (SMEM_BUDGET - 4096 - AMAX_BYTES - PST * P_BYTES) / STAGE_BYTES;
  static constexpr int STAGES_MAX = DEC ? 16 : 10;
  static constexpr int STAGES = STAGES_FIT > STAGES_MAX ? STAGES_MAX : STAGES_FIT;
  static constexpr int OFF_PRING = STAGES * STAGE_BYTES;
  static constexpr int OFF_AMAX = OFF_PRING + PST * P_BYTES;
  static constexpr int OFF_MISC = OFF_AMAX + AMAX_BYTES;
  static constexpr int TOTAL = OFF_MISC + 512 + 1024;
  static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");
  static_assert(STAGES >= 4, "pipeline depth");
  static_assert(TOTAL <= SMEM_BUDGET, "shared memory budget");
};

template <bool MN, int RP, bool F16, bool DEC, int PER_SM = 1>
__global__ void __launch_bounds__(DEC ? 448 : 192, PER_SM)
    lora_skinny_kernel(const __grid_constant__ SkinnyParams p) {
  using L = SkinnySmem<MN, RP, DEC, PER_SM>;
  static_assert(!DEC || !MN, "NF4 decode: KMAJOR only");
  static_assert(SkinnyEpi(RP, 1).bytes <= L::OFF_AMAX, "epilogue buffers fit in the ring");
  constexpr int STAGES = L::STAGES;
  constexpr uint32_t kTmemCols = RP <= 32 ? 32 : RP <= 64 ? 64 : RP <= 128 ? 128 : 256;
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
  const int n_chunks = (int)((long long)P.chunks * (srank + 1) / S) - c_begin;
  // Row tiles start at staggered chunks of their slice (and wrap around), so
  // the CTAs in flight read different Q chunks instead of all hitting the
  // same L2 lines at once; the order is fixed, so results stay deterministic.
  const int c_rot = n_chunks > 0 ? (int)(((long long)rt * n_chunks) / P.row_tiles) % n_chunks : 0;

  const uint32_t bar_full = base + L::OFF_MISC;
  const uint32_t bar_empty = bar_full + 8 * STAGES;
  const uint32_t bar_acc_full = bar_empty + 8 * STAGES;
  const uint32_t bar_drain = bar_acc_full + 8;
  constexpr int PST = L::PST;
  const uint32_t bar_pfull = bar_drain + 8;      // [PST] DEC: P tile ready (four warps of a decode group)
  const uint32_t bar_pempty = bar_pfull + 8 * PST;  // [PST] DEC: the MMA read the P tile
  uint32_t *tmem_holder =
      reinterpret_cast<uint32_t *>(smem + L::OFF_MISC + 8 * (2 * STAGES + 2 + 2 * PST));
  // Q of TMA stage s; P of TMA stage s or (DEC) of P-ring slot ps
  auto slot_q = [&](int st) {
    return base + (uint32_t)st * L::STAGE_BYTES + (DEC ? 0u : (uint32_t)L::P_BYTES);
  };
  auto slot_p = [&](int st, int ps) {
    return DEC ? base + L::OFF_PRING + (uint32_t)ps * L::P_BYTES
               : base + (uint32_t)st * L::STAGE_BYTES;
  };
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_acc_full, 1);
    mbar_init(bar_drain, 1);
    for (int s = 0; s < PST; ++s) {
      mbar_init(bar_pfull + 8 * s, 4);  // the four warps of one decode group
      mbar_init(bar_pempty + 8 * s, 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_holder), kTmemCols);
    tmem_relinquish();
  }
  if (!MN && P.q_rows < RP) {
    // rows [q_rows, RP) of every Q slot stay zero (the copies fill the rest)
    const uint32_t row_bytes = (uint32_t)(RP - P.q_rows) * 128u;
    for (uint32_t o = threadIdx.x * 16u; o < (uint32_t)STAGES * row_bytes; o += blockDim.x * 16u) {
      const uint32_t st = o / row_bytes;
      st_shared_v4(slot_q((int)st) + (uint32_t)P.q_rows * 128u + (o - st * row_bytes), 0u, 0u, 0u,
                   0u);
    }
    fence_proxy_async_smem();
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
      tma_prefetch_desc(&P.tm_p);
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;  // chunks issued: stage s took every STAGES-th from the s-th
      int pslot = 0, pissued = 0;  // DEC, P by TMA: the P ring
      uint32_t pphase = 0;
      for (int i = 0; i < n_chunks; ++i) {
        const int c = c_begin + (i + c_rot) % n_chunks;
        if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1u, abort_flag, p.status)) break;
        const uint32_t sp = slot_p(stage, 0);
        const uint32_t sq = slot_q(stage);
        const uint32_t fb = bar_full + 8 * stage;
        if constexpr (DEC) {
          if (P.nf4) {  // Q and the codes of the P tile (decoded by the decode warps)
            mbar_arrive_expect_tx(fb, L::C_BYTES + P.q_rows * 128);
            tma_load_2d(sq + L::Q_BYTES, &P.tm_p, fb, c * 32, rt * 128);
            tma_load_2d(sq, &P.tm_q, fb, c * 64, 0);
          } else {      // Q, and P straight into the P ring
            if (!mbar_wait(bar_pempty + 8 * pslot, pphase ^ 1u, abort_flag, p.status)) break;
            mbar_arrive_expect_tx(fb, L::P_BYTES + P.q_rows * 128);
            tma_load_2d(slot_p(stage, pslot), &P.tm_p, fb, c * 64, rt * 128);
            tma_load_2d(sq, &P.tm_q, fb, c * 64, 0);
            ++pissued;
            if (++pslot == PST) pslot = 0, pphase ^= 1u;
          }
          ++issued;
          if (++stage == STAGES) stage = 0, phase ^= 1u;
          continue;
        }
        mbar_arrive_expect_tx(fb, MN ? L::STAGE_BYTES : L::P_BYTES + P.q_rows * 128);
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
      // drain: every issued copy has been consumed before the CTA may exit
      // (bounded: after an abort some never are)
      const uint64_t lim = *abort_flag ? 20000000ull : 1000000000ull;
      for (int s = 0; s < STAGES; ++s) {
        const int fills = issued > s ? (issued - s + STAGES - 1) / STAGES : 0;
        if (fills > 0) mbar_wait_quiet(bar_empty + 8 * s, (uint32_t)((fills - 1) & 1), lim);
      }
      if constexpr (DEC) {  // the P ring exists only in the decoding variant
        for (int s = 0; s < PST; ++s) {
          const int fills = pissued > s ? (pissued - s + PST - 1) / PST : 0;
          if (fills > 0) mbar_wait_quiet(bar_pempty + 8 * s, (uint32_t)((fills - 1) & 1), lim);
        }
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc(128, RP, MN, false, F16);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int pslot = 0;  // DEC: P ring
      uint32_t pphase = 0;
      for (int i = 0; i < n_chunks; ++i) {
        if (!mbar_wait(bar_full + 8 * stage, phase, abort_flag, p.status) ||
            (DEC && !mbar_wait(bar_pfull + 8 * pslot, pphase, abort_flag, p.status))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sp = slot_p(stage, pslot);
        const uint32_t sq = slot_q(stage);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint32_t accum = (i != 0 || ks != 0) ? 1u : 0u;
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
        if constexpr (DEC) {
          tc_commit(bar_pempty + 8 * pslot);
          if (++pslot == PST) pslot = 0, pphase ^= 1u;
        }
      }
      if (ok) tc_commit(bar_acc_full);
      if (*abort_flag) {
        tc_commit(bar_drain);
        mbar_wait_quiet(bar_drain, 0, 100000000ull);
      }
    }
  } else if (DEC && warp >= 6) {
    // ------------------------------------------------------- NF4 decode
    // Two groups of four warps take alternate chunks (group gr: chunks gr,
    // gr + 2, ...); thread pr of a group decodes row pr of the chunk's P
    // tile (64 codes, one scaled table).  A problem without codes passes its
    // stages straight on.
    const int t = threadIdx.x - 192;  // 0..255
    const int gr = t >> 7, prow = t & 127;
    const bool dec = P.nf4 != 0;
    const int wrow = rt * 128 + prow;
    const bool row_in = wrow < P.rows;
    constexpr int PRE = L::AMAX_PRE;
    constexpr uint32_t kSlot = L::DEC_THREADS * 4;
    const uint32_t ring = base + L::OFF_AMAX + (uint32_t)t * 4u;  // slot j at ring + kSlot j
    float lvl[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) lvl[i] = kNf4Levels[i];
    const __nv_bfloat16 *arow = P.absmax + (size_t)(row_in ? wrow : 0) * P.ld_absmax + c_begin;
    // The absmax of chunk i is arow[(i + c_rot) % n_chunks]; the offsets of
    // the group's chunk being decoded (cur) and of its chunk PRE of its own
    // chunks ahead (ahead) advance by two with wrap-around.
    auto step2 = [&](int &o) {
      o += 2;
      while (o >= n_chunks && n_chunks > 0) o -= n_chunks;
    };
    int cur = n_chunks > 0 ? (c_rot + gr) % n_chunks : 0, ahead = cur;
    int ia = gr;  // chunk of the next prefetch
    auto prefetch = [&](uint32_t slot) {
      if (dec && row_in && ia < n_chunks)
        cp_async_4(ring + slot * kSlot, reinterpret_cast<const void *>(
                                            reinterpret_cast<uintptr_t>(arow + ahead) & ~uintptr_t(3)));
      cp_async_commit();
      step2(ahead);
      ia += 2;
    };
    for (int j = 0; j < PRE; ++j) prefetch((uint32_t)j);
    // 32-byte code rows of consecutive threads are contiguous: threads whose
    // rows start in the same half of the 32 banks read their two 16-byte
    // halves in opposite orders, so each load touches every bank
    const uint32_t flip = (uint32_t)(prow >> 2) & 1u;
    int stage = gr;
    uint32_t phase = 0;
    uint32_t slot = 0;
    int pslot = gr;
    uint32_t pphase = 0;
    for (int i = gr; i < n_chunks; i += 2) {
      if (!warp_wait(bar_full + 8 * stage, phase, abort_flag, p.status)) break;
      // the P slot is free once the MMA of its previous use has completed
      // (for P loaded by TMA the producer waited for that)
      if (dec && !warp_wait(bar_pempty + 8 * pslot, pphase ^ 1u, abort_flag, p.status)) break;
      if (dec) {
        cp_async_wait<PRE - 1>();  // this chunk's absmax has landed
        float amax = 0.0f;
        if (row_in) {
          const uint32_t w = ld_shared_u32(ring + slot * kSlot);
          const bool high = (reinterpret_cast<uintptr_t>(arow + cur) & 2u) != 0;
          amax = __uint_as_float((high ? (w >> 16) : (w & 0xFFFFu)) << 16);
        }
        step2(cur);
        prefetch(slot);  // the slot just read refills for PRE of the group's chunks ahead
        if (++slot == (uint32_t)PRE) slot = 0;
        uint32_t words[8];
        nf4_load_codes(slot_q(stage) + L::Q_BYTES + (uint32_t)prow * 32u, flip, words);
        nf4_decode_words(words, slot_p(stage, pslot) + (uint32_t)prow * 128u,
                         nf4_table<F16>(lvl, amax));
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_pfull + 8 * pslot);
      stage += 2;
      if (stage >= STAGES) stage -= STAGES, phase ^= 1u;
      pslot += 2;
      if (pslot >= PST) pslot -= PST, pphase ^= 1u;
    }
    cp_async_wait<0>();  // no copy may land after the CTA exits
  }

  // ---------------------------------------------- epilogue (warps 2-5)
  // 1. every CTA's accumulator is complete (its ring is idle)
  // 2. each CTA pushes its partial of the other CTAs' column blocks into
  //    their recv slots (distributed shared memory stores)
  // 3. each CTA adds the S partials of its own block in cluster-rank order
  //    (deterministic), stages the result and copies it out
  const bool epi = warp >= 2 && warp < 6;
  const int row = (warp & 3) * 32 + lane;
  const uint32_t t_lane = (uint32_t)((warp & 3) * 32) << 16;
  const SkinnyEpi E(RP, S);
  const int CW = E.cw;
  float *recv = reinterpret_cast<float *>(smem);
  float *stage_t = reinterpret_cast<float *>(smem + E.off_stage_t);
  float *stage_r = reinterpret_cast<float *>(smem + E.off_stage_r);
  bool acc_ok = false;
  if (epi) {
    acc_ok = __all_sync(0xffffffffu, mbar_wait(bar_acc_full, 0, abort_flag, p.status));
    if (acc_ok) tc_fence_after();
  }
  __syncwarp();
  if (S > 1) cluster_sync_all();  // every ring of the cluster is idle
  if (epi && acc_ok && S > 1) {
    const uint32_t my_slot = smem_addr(recv + ((size_t)srank * 128 + row) * E.recv_stride);
    for (int b = 0; b < S; ++b) {
      if (b == srank) continue;
      const uint32_t dst = map_shared_rank(my_slot, (uint32_t)b);
#pragma unroll 1
      for (int c = 0; c < CW / 16; ++c) {
        uint32_t r[16];
        tmem_ld16(tmem + t_lane + b * CW + c * 16, r);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 4; ++j)
          st_shared_cluster_v4(dst + c * 64 + j * 16, r[4 * j], r[4 * j + 1], r[4 * j + 2],
                               r[4 * j + 3]);
      }
    }
  }
  __syncwarp();
  if (S > 1) cluster_sync_all();  // pushed partials have landed
  const bool want_t = (P.out_kind & (kOutVt | kOutRowT | kOutT16)) != 0;
  const bool want_r = (P.out_kind & (kOutRowBf16 | kOutRow)) != 0;
  if (epi && acc_ok) {
#pragma unroll 1
    for (int c = 0; c < CW / 16; ++c) {
      uint32_t r[16];
      tmem_ld16(tmem + t_lane + srank * CW + c * 16, r);
      tmem_ld_wait();
      float v[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = 0.0f;
      for (int s = 0; s < S; ++s) {
        if (s == srank) {
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] += __uint_as_float(r[j]);
        } else {
          const float4 *src = reinterpret_cast<const float4 *>(
              recv + ((size_t)s * 128 + row) * E.recv_stride + c * 16);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float4 t = src[j];
            v[4 * j] += t.x;
            v[4 * j + 1] += t.y;
            v[4 * j + 2] += t.z;
            v[4 * j + 3] += t.w;
          }
        }
      }
      if (want_t) {
#pragma unroll
        for (int j = 0; j < 16; ++j) stage_t[(c * 16 + j) * 132 + row] = v[j];
      }
      if (want_r) {
        float4 *dst = reinterpret_cast<float4 *>(stage_r + row * (CW + 4) + c * 16);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
      }
    }
  }
  if (epi) {
    epi_bar();
    if (acc_ok)
      skinny_copy_out<F16>(skinny_dest(P), rt, srank * CW, CW, stage_t, stage_r, threadIdx.x - 64);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <bool MN, int RP, bool F16, bool DEC, int PER_SM = 1>
static cudaError_t launch_skinny_t(const SkinnyParams &p, cudaStream_t st) {
  using L = SkinnySmem<MN, RP, DEC, PER_SM>;
  auto kern = lora_skinny_kernel<MN, RP, F16, DEC, PER_SM>;
  static std::atomic<uint64_t> attr_done{0};
  const cudaError_t e = smem_attr_once(attr_done, reinterpret_cast<const void *>(kern), L::TOTAL);
  if (e != cudaSuccess) return e;
  int tiles = 0;
  for (int q = 0; q < p.num_problems; ++q) tiles += p.pr[q].row_tiles;
  const char *name =
      DEC ? (F16 ? "lora_skinny_kernel<k_major,nf4,f16>" : "lora_skinny_kernel<k_major,nf4>")
      : PER_SM == 2 ? (F16 ? "lora_skinny_kernel<k_major,2cta,f16>" : "lora_skinny_kernel<k_major,2cta>")
      : MN ? (F16 ? "lora_skinny_kernel<mn_major,f16>" : "lora_skinny_kernel<mn_major>")
           : (F16 ? "lora_skinny_kernel<k_major,f16>" : "lora_skinny_kernel<k_major>");
  return launch_pdl(name, kern, dim3((unsigned)(tiles * p.split)), dim3(DEC ? 448 : 192),
                    L::TOTAL, st, (unsigned)p.split, p);
}

template <bool MN, int RP, bool DEC = false, int PER_SM = 1>
static int max_split_t() {
  using L = SkinnySmem<MN, RP, DEC, PER_SM>;
  int s = 1;
  while (s < 8 && RP / (2 * s) >= 16 && SkinnyEpi(RP, 2 * s).bytes <= L::OFF_AMAX) s *= 2;
  return s;
}

// The NF4 decoding pass with 96 token columns splits a tile over 1, 2, 3 or
// 6 CTAs (16-column blocks); 41 row tiles (a 5120-row W and A) then fill 123
// SMs instead of 82.
static_assert(SkinnyEpi(96, 6).bytes <= SkinnySmem<false, 96, true>::OFF_AMAX,
              "epilogue buffers of the 96-column decoding pass fit in its ring");

bool skinny_split_ok(bool mn_major, int rp, bool dec, bool two, int split) {
  if (split < 1 || split > 8 || rp % (16 * split) != 0) return false;
  if (dec && !mn_major && !two && rp == 96) return split == 1 || split == 2 || split == 3 || split == 6;
  if ((split & (split - 1)) != 0) return false;
  return split <= skinny_max_split(mn_major, rp, dec, two);
}

int skinny_max_split(bool mn_major, int rp, bool dec, bool two) {
  if (two) return (!mn_major && !dec && rp == 64) ? max_split_t<false, 64, false, 2>() : 1;
  if (dec) {
    if (mn_major) return 1;
    if (rp == 96) return 6;
    return rp == 64 ? max_split_t<false, 64, true>() : rp == 128 ? max_split_t<false, 128, true>() : 1;
  }
  switch (rp) {
    case 16: return mn_major ? max_split_t<true, 16>() : max_split_t<false, 16>();
    case 32: return mn_major ? max_split_t<true, 32>() : max_split_t<false, 32>();
    case 64: return mn_major ? max_split_t<true, 64>() : max_split_t<false, 64>();
    case 128: return mn_major ? max_split_t<true, 128>() : max_split_t<false, 128>();
  }
  return 1;
}

template <bool F16>
static cudaError_t launch_skinny_cluster_t(const SkinnyParams &p, bool mn_major, int rp, bool dec,
                                           bool two, cudaStream_t st) {
  if (two) {
    if (mn_major || dec || rp != 64) return cudaErrorInvalidValue;
    return launch_skinny_t<false, 64, F16, false, 2>(p, st);
  }
  if (dec) {
    if (mn_major) return cudaErrorInvalidValue;
    if (rp == 64) return launch_skinny_t<false, 64, F16, true>(p, st);
    if (rp == 96) return launch_skinny_t<false, 96, F16, true>(p, st);
    if (rp == 128) return launch_skinny_t<false, 128, F16, true>(p, st);
    return cudaErrorInvalidValue;
  }
  switch (rp) {
    case 16: return mn_major ? launch_skinny_t<true, 16, F16, false>(p, st) : launch_skinny_t<false, 16, F16, false>(p, st);
    case 32: return mn_major ? launch_skinny_t<true, 32, F16, false>(p, st) : launch_skinny_t<false, 32, F16, false>(p, st);
    case 64: return mn_major ? launch_skinny_t<true, 64, F16, false>(p, st) : launch_skinny_t<false, 64, F16, false>(p, st);
    case 128: return mn_major ? launch_skinny_t<true, 128, F16, false>(p, st) : launch_skinny_t<false, 128, F16, false>(p, st);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_skinny_cluster(const SkinnyParams &p, bool mn_major, int rp, bool f16,
                                  cudaStream_t st, bool dec, bool two) {
  if (!skinny_split_ok(mn_major, rp, dec, two, p.split)) return cudaErrorInvalidValue;
  return f16 ? launch_skinny_cluster_t<true>(p, mn_major, rp, dec, two, st)
             : launch_skinny_cluster_t<false>(p, mn_major, rp, dec, two, st);
}

}  // namespace lora
