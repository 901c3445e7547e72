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
  static constexpr int OFF_MISC = STAGES * STAGE_BYTES;
  static constexpr int TOTAL = OFF_MISC + 512 + 1024;
  static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");
  static_assert(STAGES >= 4, "pipeline depth");
  static_assert(TOTAL <= kSmemLimit, "shared memory budget");
};

// Epilogue buffers, laid over the (then idle) TMA ring.  A CTA of a cluster
// of S finalises the column block [CW·rank, CW·rank + CW), CW = RP / S:
//   recv    [S][128][CW + 4] fp32: slot s holds CTA s's partial of this block
//   stage_t [CW][128 + 4] fp32:   final values, transposed (kOutVt, kOutRowT)
//   stage_r [128][CW + 4] fp32:   final values, row-major (kOutRowBf16, kOutRow)
// Rows are padded by 16 bytes so the 16-byte accesses of a warp hit distinct
// banks.
struct SkinnyEpi {
  int cw, recv_stride, off_stage_t, off_stage_r, bytes;
  __host__ __device__ constexpr SkinnyEpi(int rp, int split)
      : cw(rp / split),
        recv_stride(rp / split + 4),
        off_stage_t(split > 1 ? split * 128 * (rp / split + 4) * 4 : 0),
        off_stage_r((split > 1 ? split * 128 * (rp / split + 4) * 4 : 0) +
                    (rp / split) * (128 + 4) * 4),
        bytes((split > 1 ? split * 128 * (rp / split + 4) * 4 : 0) +
              (rp / split) * (128 + 4) * 4 + 128 * (rp / split + 4) * 4) {}
};


LORA_DEV void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Copy-out of one CTA's column block [col0, col0 + cw) of row tile rt from
// the staging buffers, by the 128 epilogue threads (e = 0..127).  Every
// warp-wide store covers contiguous runs of 256 to 512 bytes.
template <bool F16>
LORA_DEV void skinny_copy_out(const SkinnyProblem &P, int rt, int col0, int cw,
                              const float *stage_t, const float *stage_r, int e) {
  const int cols = P.nproj * P.r;  // valid rank columns
  const int row0 = rt * 128;
  const int w = e >> 5, l = e & 31;
  // transposed outputs: warp w takes block columns j = w, w + 4, ...; lane l
  // takes rows [4l, 4l + 4) of the tile
  if (P.out_kind & (kOutVt | kOutRowT)) {
    const int orow = row0 + 4 * l;
    const bool full = orow + 4 <= P.rows;
    for (int j = w; j < cw; j += 4) {
      const float4 t = *reinterpret_cast<const float4 *>(stage_t + j * 132 + 4 * l);
      const float f[4] = {t.x, t.y, t.z, t.w};
      const int jg = col0 + j;
      if (P.out_kind & kOutVt) {
        uint16_t hi[4], lo[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          hi[q] = to16<F16>(f[q]);
          lo[q] = to16<F16>(f[q] - from16<F16>(hi[q]));
        }
        uint16_t *dh = P.out_hi + (size_t)jg * P.ld_t + orow;
        uint16_t *dl = P.out_lo + (size_t)jg * P.ld_t + orow;
        if (full) {
          *reinterpret_cast<uint2 *>(dh) = *reinterpret_cast<const uint2 *>(hi);
          *reinterpret_cast<uint2 *>(dl) = *reinterpret_cast<const uint2 *>(lo);
        } else {
          for (int q = 0; q < 4; ++q)
            if (orow + q < P.rows) dh[q] = hi[q], dl[q] = lo[q];
        }
      }
      if ((P.out_kind & kOutRowT) && jg < cols) {
        const int pr = jg / P.r, jj = jg - pr * P.r;
        float *dst = (pr ? P.out_f32b : P.out_f32) + (size_t)jj * P.rows + orow;
        if (full) {
          *reinterpret_cast<float4 *>(dst) =
              make_float4(f[0] * P.scale, f[1] * P.scale, f[2] * P.scale, f[3] * P.scale);
        } else {
          for (int q = 0; q < 4; ++q)
            if (orow + q < P.rows) dst[q] = f[q] * P.scale;
        }
      }
    }
  }
  // row-major outputs: a row is cw columns; lanes cover 8 (bf16) or 4 (fp32)
  // consecutive columns, several rows per warp-wide store
  if (P.out_kind & kOutRowBf16) {
    const int lpr = cw / 8;  // lanes per row (cw >= 16)
    const int rpw = 32 / lpr;
    const int c = (l % lpr) * 8;
    for (int rr = w * rpw + l / lpr; rr < 128; rr += 4 * rpw) {
      const int orow = row0 + rr;
      if (orow >= P.rows) break;
      const float *src = stage_r + rr * (cw + 4) + c;
      const float4 a = *reinterpret_cast<const float4 *>(src);
      const float4 b = *reinterpret_cast<const float4 *>(src + 4);
      uint16_t *dst = P.out_bf16 + (size_t)orow * P.ld_row + col0 + c;
      if (col0 + c + 8 <= cols) {
        uint4 o;
        o.x = pack2<F16>(a.x * P.scale, a.y * P.scale);
        o.y = pack2<F16>(a.z * P.scale, a.w * P.scale);
        o.z = pack2<F16>(b.x * P.scale, b.y * P.scale);
        o.w = pack2<F16>(b.z * P.scale, b.w * P.scale);
        *reinterpret_cast<uint4 *>(dst) = o;
      } else {
        const float f[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        for (int q = 0; q < 8; ++q)
          if (col0 + c + q < cols) dst[q] = to16<F16>(f[q] * P.scale);
      }
    }
  }
  if (P.out_kind & kOutRow) {
    // dB: only the diagonal block of a merged pair is a real gradient
    const int lpr = cw / 4;
    const int rpw = lpr >= 32 ? 1 : 32 / lpr;
    for (int cb = 0; cb < cw; cb += 128) {   // column groups of 32 lanes x 4
      const int c = cb + (l % (lpr >= 32 ? 32 : lpr)) * 4;
      if (c >= cw) continue;
      for (int rr = w * rpw + (lpr >= 32 ? 0 : l / lpr); rr < 128; rr += 4 * rpw) {
        const int orow = row0 + rr;
        if (orow >= P.rows) break;
        const int pr = (P.nproj > 1 && orow >= P.split_row) ? 1 : 0;
        const int jg = col0 + c, lo = pr * P.r;
        if (jg < lo || jg >= lo + P.r) continue;
        const float4 t = *reinterpret_cast<const float4 *>(stage_r + rr * (cw + 4) + c);
        float *dst = (pr ? P.out_f32b : P.out_f32) + (size_t)(orow - pr * P.split_row) * P.r +
                     (jg - lo);
        if (jg + 4 <= lo + P.r) {
          *reinterpret_cast<float4 *>(dst) =
              make_float4(t.x * P.scale, t.y * P.scale, t.z * P.scale, t.w * P.scale);
        } else {
          const float f[4] = {t.x, t.y, t.z, t.w};
          for (int q = 0; q < 4 && jg + q < lo + P.r; ++q) dst[q] = f[q] * P.scale;
        }
      }
    }
  }
}

template <bool MN, int RP, bool F16>
__global__ void __launch_bounds__(192, 1) lora_skinny_kernel(const __grid_constant__ SkinnyParams p) {
  using L = SkinnySmem<MN, RP>;
  static_assert(SkinnyEpi(RP, 1).bytes <= L::OFF_MISC, "epilogue buffers fit in the ring");
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
  const int n_chunks = (int)((long long)P.chunks * (srank + 1) / S) - c_begin;
  // Row tiles start at staggered chunks of their slice (and wrap around), so
  // the CTAs in flight read different Q chunks instead of all hitting the
  // same L2 lines at once; the order is fixed, so results stay deterministic.
  const int c_rot = n_chunks > 0 ? (int)(((long long)rt * n_chunks) / P.row_tiles) % n_chunks : 0;

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
  grid_dep_launch();
  grid_dep_wait();  // the previous kernel's outputs are complete

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&P.tm_p);
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;  // chunks issued: stage s took every STAGES-th from the s-th
      for (int i = 0; i < n_chunks; ++i) {
        const int c = c_begin + (i + c_rot) % n_chunks;
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
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc(128, RP, MN, false, F16);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int i = 0; i < n_chunks; ++i) {
        if (!mbar_wait(bar_full + 8 * stage, phase, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sp = base + stage * L::STAGE_BYTES;
        const uint32_t sq = sp + L::P_BYTES;
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
      }
      if (ok) tc_commit(bar_acc_full);
      if (*abort_flag) {
        tc_commit(bar_drain);
        mbar_wait_quiet(bar_drain, 0, 100000000ull);
      }
    }
  }

  // ---------------------------------------------- epilogue (warps 2-5)
  // 1. every CTA's accumulator is complete (its ring is idle)
  // 2. each CTA pushes its partial of the other CTAs' column blocks into
  //    their recv slots (distributed shared memory stores)
  // 3. each CTA adds the S partials of its own block in cluster-rank order
  //    (deterministic), stages the result and copies it out
  const bool epi = warp >= 2;
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
  const bool want_t = (P.out_kind & (kOutVt | kOutRowT)) != 0;
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
    if (acc_ok) skinny_copy_out<F16>(P, rt, srank * CW, CW, stage_t, stage_r, threadIdx.x - 64);
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
  using L = SkinnySmem<MN, RP>;
  auto kern = lora_skinny_kernel<MN, RP, F16>;
  static std::atomic<uint64_t> attr_done{0};
  const cudaError_t e = smem_attr_once(attr_done, reinterpret_cast<const void *>(kern), L::TOTAL);
  if (e != cudaSuccess) return e;
  int tiles = 0;
  for (int q = 0; q < p.num_problems; ++q) tiles += p.pr[q].row_tiles;
  const char *name = MN ? (F16 ? "lora_skinny_kernel<mn_major,f16>" : "lora_skinny_kernel<mn_major>")
                        : (F16 ? "lora_skinny_kernel<k_major,f16>" : "lora_skinny_kernel<k_major>");
  return launch_pdl(name, kern,
                    dim3((unsigned)(tiles * p.split)), dim3(192), L::TOTAL, st,
                    (unsigned)p.split, p);
}

template <bool MN, int RP>
static int max_split_t() {
  using L = SkinnySmem<MN, RP>;
  int s = 1;
  while (s < 8 && RP / (2 * s) >= 16 && SkinnyEpi(RP, 2 * s).bytes <= L::OFF_MISC) s *= 2;
  return s;
}

int skinny_max_split(bool mn_major, int rp) {
  switch (rp) {
    case 16: return mn_major ? max_split_t<true, 16>() : max_split_t<false, 16>();
    case 32: return mn_major ? max_split_t<true, 32>() : max_split_t<false, 32>();
    case 64: return mn_major ? max_split_t<true, 64>() : max_split_t<false, 64>();
    case 128: return mn_major ? max_split_t<true, 128>() : max_split_t<false, 128>();
  }
  return 1;
}

template <bool F16>
static cudaError_t launch_skinny_cluster_t(const SkinnyParams &p, bool mn_major, int rp,
                                           cudaStream_t st) {
  switch (rp) {
    case 16: return mn_major ? launch_skinny_t<true, 16, F16>(p, st) : launch_skinny_t<false, 16, F16>(p, st);
    case 32: return mn_major ? launch_skinny_t<true, 32, F16>(p, st) : launch_skinny_t<false, 32, F16>(p, st);
    case 64: return mn_major ? launch_skinny_t<true, 64, F16>(p, st) : launch_skinny_t<false, 64, F16>(p, st);
    case 128: return mn_major ? launch_skinny_t<true, 128, F16>(p, st) : launch_skinny_t<false, 128, F16>(p, st);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_skinny_cluster(const SkinnyParams &p, bool mn_major, int rp, bool f16,
                                  cudaStream_t st) {
  if (p.split != 1 && p.split != 2 && p.split != 4 && p.split != 8) return cudaErrorInvalidValue;
  if (p.split > skinny_max_split(mn_major, rp)) return cudaErrorInvalidValue;
  return f16 ? launch_skinny_cluster_t<true>(p, mn_major, rp, st)
             : launch_skinny_cluster_t<false>(p, mn_major, rp, st);
}

}  // namespace lora
