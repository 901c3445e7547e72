// Device helpers of the fused GEMM kernel: the NF4 level table and row
// decode, and the output epilogue (TMEM -> optional rotate-half RoPE ->
// bf16 -> global).
#pragma once

#include "kernels.h"
#include "nf4_levels.cuh"
#include "philox.cuh"

namespace lora {


LORA_DEV bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                        uint32_t *status) {
  const bool ok = mbar_wait(bar, parity, abort_flag, status);
  return __all_sync(0xffffffffu, ok);
}

// Group of n-tile nt (its output columns, rank blocks and epilogue); the
// SwiGLU pair's tiles belong to group 0 for these purposes.
LORA_DEV int group_of(const GemmParams &p, int nt) {
  return (!p.swiglu && p.num_groups > 1 && nt >= p.grp[1].tile_begin) ? 1 : 0;
}

// This CTA's half of the W tile of n-tile nt: its weight group and first N
// row.  Normally rows [256·(nt − tile_begin) + 128·crank, +128) of the
// tile's group; for the SwiGLU pair rows [128·nt, +128) of group crank
// (gate or up).
struct WHalf {
  const GemmGroup *g;
  int nh;
};
LORA_DEV WHalf w_half(const GemmParams &p, int nt, uint32_t crank) {
  if (p.swiglu) return {&p.grp[crank], nt * 128};
  const GemmGroup &G = p.grp[group_of(p, nt)];
  return {&G, (nt - G.tile_begin) * 256 + (int)crank * 128};
}

LORA_DEV uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// NF4 decode without shared-memory lookups.  Per K-block each decode
// thread forms the 16 values level_i·a of its row (fp32 product rounded once
// to bf16) and keeps them as two byte planes in registers: lo[q] holds the
// low bytes of values 4q..4q+3, hi[q] their high bytes.  A 4-bit code then
// selects its two bytes with byte permutes (prmt picks any of 8 bytes, so
// values 0-7 and 8-15 are picked separately and merged by the code's top
// bit).
struct Nf4Table {
  uint32_t lo[4], hi[4];
};

template <bool F16>
LORA_DEV Nf4Table nf4_table(const float (&lv)[16], float a) {
  uint32_t pk[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) pk[j] = pack2<F16>(lv[2 * j] * a, lv[2 * j + 1] * a);
  Nf4Table t;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    t.lo[q] = __byte_perm(pk[2 * q], pk[2 * q + 1], 0x6420);
    t.hi[q] = __byte_perm(pk[2 * q], pk[2 * q + 1], 0x7531);
  }
  return t;
}

// Four codes, the nibbles of the 16-bit value c = [e1 | e0 << 4 | e3 << 8 |
// e2 << 12] (two code bytes: element 2j in a byte's high nibble), to the
// bf16 pairs (e0, e1) and (e2, e3).
LORA_DEV void nf4_lookup4(const Nf4Table &t, uint32_t c, uint32_t &p01, uint32_t &p23) {
  const uint32_t s7 = c & 0x7777u;                        // index within a half table
  const uint32_t sel = 0x3210u | ((c >> 1) & 0x4444u);    // which half, per byte
  const uint32_t lo = __byte_perm(__byte_perm(t.lo[0], t.lo[1], s7),
                                  __byte_perm(t.lo[2], t.lo[3], s7), sel);
  const uint32_t hi = __byte_perm(__byte_perm(t.hi[0], t.hi[1], s7),
                                  __byte_perm(t.hi[2], t.hi[3], s7), sel);
  // lo/hi bytes are in code order e1, e0, e3, e2
  p01 = __byte_perm(lo, hi, 0x5140 ^ 0x1111);  // bytes lo.1, hi.1, lo.0, hi.0 -> (e0, e1)
  p23 = __byte_perm(lo, hi, 0x7362 ^ 0x1111);  // bytes lo.3, hi.3, lo.2, hi.2 -> (e2, e3)
}

// The 32 code bytes of one 64-element row piece at `src` (shared), read as
// two 16-byte halves in the order `flip` gives (flip = 1: second half
// first), returned in order.
LORA_DEV void nf4_load_codes(uint32_t src, uint32_t flip, uint32_t (&w)[8]) {
  const uint4 a = ld_shared_v4(src + (flip << 4));
  const uint4 b = ld_shared_v4(src + ((flip ^ 1u) << 4));
  const uint4 lo = flip ? b : a, hi = flip ? a : b;
  w[0] = lo.x, w[1] = lo.y, w[2] = lo.z, w[3] = lo.w;
  w[4] = hi.x, w[5] = hi.y, w[6] = hi.z, w[7] = hi.w;
}

// Decode one 64-element row piece (its 32 code bytes in `words`) into a
// 128-byte row of a 128-byte-swizzled tile at `dst`.
LORA_DEV void nf4_decode_words(const uint32_t (&words)[8], uint32_t dst, const Nf4Table &t) {
  const uint32_t phase = (dst >> 7) & 7u;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    uint32_t o[4];
    nf4_lookup4(t, words[q] & 0xFFFFu, o[0], o[1]);
    nf4_lookup4(t, words[q] >> 16, o[2], o[3]);
    st_shared_v4(dst + ((((uint32_t)q) ^ phase) << 4), o[0], o[1], o[2], o[3]);
  }
}

// Read-modify-write epilogue for one thread: BN accumulator columns at
// `t_acc` of one output row are scaled by `scale` and added to the bf16
// values already at `orow` (ncols valid columns), rounding once to bf16.
// Used where the result accumulates into its destination (dX += ..., and
// W ± s·B·A when merging an adapter into its weight).
// DROPOUT: the result is multiplied by the dropout keep bit of its output
// element (row `grow`, column col0 + column in tile) times p.drop_scale.
template <int BN, bool F16, bool DROPOUT = false>
LORA_DEV void epi_accumulate_tile(uint32_t t_acc, uint16_t *orow, bool row_ok, int ncols,
                                  float scale, const GemmParams *p = nullptr, int grow = 0,
                                  int col0 = 0) {
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    uint32_t r[32];
    tmem_ld32(t_acc + c * 32, r);
    tmem_ld_wait();
    if (row_ok && c * 32 < ncols) {
      uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
      float f[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(r[j]) * scale;
      if constexpr (DROPOUT) {
        // 32 columns = two 16-element Philox blocks (row·ld and the column are
        // multiples of 16)
        const uint64_t e0 = (uint64_t)grow * (uint64_t)p->drop_ld + (uint64_t)(col0 + c * 32);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t keep =
              dropout_keep16(e0 / 16 + h, p->drop_seed, p->drop_offset, p->drop_thresh);
#pragma unroll
          for (int j = 0; j < 16; ++j)
            f[16 * h + j] = (keep >> j) & 1u ? f[16 * h + j] * p->drop_scale : 0.0f;
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 old = dst[j];
        const uint32_t ow[4] = {old.x, old.y, old.z, old.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 h = unpack2<F16>(ow[e]);
          f[8 * j + 2 * e] += h.x;
          f[8 * j + 2 * e + 1] += h.y;
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint4 w;
        w.x = pack2<F16>(f[8 * j + 0], f[8 * j + 1]);
        w.y = pack2<F16>(f[8 * j + 2], f[8 * j + 3]);
        w.z = pack2<F16>(f[8 * j + 4], f[8 * j + 5]);
        w.w = pack2<F16>(f[8 * j + 6], f[8 * j + 7]);
        dst[j] = w;
      }
    }
  }
}

// cos / sin of one half (32 rotation pairs) of a cache row, in registers.
struct RopeHalf {
  float4 c[8], s[8];
  // from a staged row [32 cos | 32 sin]
  LORA_DEV void load_shared(uint32_t srow) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint4 a = ld_shared_v4(srow + 16 * i), b = ld_shared_v4(srow + 128 + 16 * i);
      c[i] = make_float4(__uint_as_float(a.x), __uint_as_float(a.y), __uint_as_float(a.z),
                         __uint_as_float(a.w));
      s[i] = make_float4(__uint_as_float(b.x), __uint_as_float(b.y), __uint_as_float(b.z),
                         __uint_as_float(b.w));
    }
  }
};

// Row pitch of a staged cos / sin half: 256 bytes of data plus 16 of padding,
// so that 32 lanes reading 16 bytes each of their own rows fall on distinct
// bank quads (four wavefronts, the minimum for 512 bytes).
constexpr int kRopeRowPitch = 272;

// Stages half `half` of this lane's cache row `cs` (32 cos, then 32 sin
// values) into its shared-memory row `srow` with two bulk copies, which the
// copy engine rather than the load/store pipe carries (the 32 lanes of a
// warp read 32 different rows: as plain loads each instruction would touch
// 32 cache lines).  Lane 0 arms the warp's barrier for all 32 rows.
LORA_DEV void rope_stage(const float *cs, int half, uint32_t srow, uint32_t bar, int lane) {
  if (lane == 0) mbar_arrive_expect_tx(bar, 32 * 256);
  fence_proxy_async_smem();  // this lane's reads of its row precede the overwrite
  bulk_load(srow, cs + half * 32, 128, bar);
  bulk_load(srow + 128, cs + 64 + half * 32, 128, bar);
}

// Output epilogue through shared memory and TMA for one warp (32 rows of
// the CTA's 128): per 32-column chunk, TMEM -> (RoPE) -> bf16 into one of
// two 2 KB staging buffers [32 rows x 64 bytes, 64-byte swizzle, the layout
// the output tensor map names], then lane 0 stores the chunk with one bulk
// tensor copy (whole lines, clipped at the tensor's extent).  `buf` is the
// warp's staging area; `cs` the cos/sin row of this lane's output row.  The
// epilogue of a tile overlaps the next tile's K loop, so two buffers do.
// RoPE takes the row's cos / sin one half (32 rotation pairs) at a time,
// both heads of the tile per half.  STAGED: the halves come from the lane's
// shared-memory row `srow`, filled by rope_stage() on barrier `cs_bar` (the
// caller stages half 0 before the accumulator is ready; half 1 is staged
// here as soon as half 0 sits in registers).  Otherwise each 32-column
// chunk reads its cos / sin from the cache directly.  Returns false when a
// wait gave up.
template <int BN, bool ROPE, bool STAGED, bool F16>
LORA_DEV bool epi_store_tile_tma(uint32_t t_acc, uint32_t buf, const CUtensorMap *tm_out,
                                 int col0, int row0, int ncols, const float *cs, uint32_t srow,
                                 uint32_t cs_bar, uint32_t &cs_phase, int lane,
                                 volatile int *abort_flag, uint32_t *status) {
  // byte offset of 16-byte chunk q of this lane's row in a staging buffer
  auto at = [&](int q) -> uint32_t {
    return (uint32_t)(lane * 64 + ((q ^ ((lane >> 1) & 3)) << 4));
  };
  if constexpr (!ROPE) {
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      uint32_t r[32];
      tmem_ld32(t_acc + c * 32, r);
      tmem_ld_wait();
      if (c * 32 >= ncols) continue;
      const uint32_t b = buf + (uint32_t)(c & 1) * 2048u;
      if (lane == 0) bulk_wait_read<1>();  // buffer (c & 1) no longer read by an older copy
      __syncwarp();
#pragma unroll
      for (int q = 0; q < 4; ++q)
        st_shared_v4(b + at(q), pack2<F16>(__uint_as_float(r[8 * q + 0]), __uint_as_float(r[8 * q + 1])),
                     pack2<F16>(__uint_as_float(r[8 * q + 2]), __uint_as_float(r[8 * q + 3])),
                     pack2<F16>(__uint_as_float(r[8 * q + 4]), __uint_as_float(r[8 * q + 5])),
                     pack2<F16>(__uint_as_float(r[8 * q + 6]), __uint_as_float(r[8 * q + 7])));
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(tm_out, b, col0 + c * 32, row0);
        bulk_commit();
      }
    }
  } else if constexpr (!STAGED) {
    // cos / sin straight from the cache (the register budget of the NF4
    // kernel holds one 32-column chunk of them at a time)
#pragma unroll 1
    for (int h = 0; h < BN / 128; ++h) {
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        const int c0 = h * 128 + half * 32;
        uint32_t ra[32], rb[32];
        tmem_ld32(t_acc + c0, ra);
        tmem_ld32(t_acc + c0 + 64, rb);
        tmem_ld_wait();
        if (c0 >= ncols) continue;
        const uint32_t ba = buf;
        const uint32_t bb = buf + 2048u;
        if (lane == 0) bulk_wait_read<0>();  // both buffers are free again
        __syncwarp();
        const float4 *cp = reinterpret_cast<const float4 *>(cs + half * 32);
        const float4 *sp = reinterpret_cast<const float4 *>(cs + 64 + half * 32);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 c_lo = __ldg(cp + 2 * q), c_hi = __ldg(cp + 2 * q + 1);
          const float4 s_lo = __ldg(sp + 2 * q), s_hi = __ldg(sp + 2 * q + 1);
          const float co[8] = {c_lo.x, c_lo.y, c_lo.z, c_lo.w, c_hi.x, c_hi.y, c_hi.z, c_hi.w};
          const float si[8] = {s_lo.x, s_lo.y, s_lo.z, s_lo.w, s_hi.x, s_hi.y, s_hi.z, s_hi.w};
          float oa[8], ob[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float a = __uint_as_float(ra[8 * q + e]);
            const float bv = __uint_as_float(rb[8 * q + e]);
            oa[e] = a * co[e] - bv * si[e];
            ob[e] = bv * co[e] + a * si[e];
          }
          st_shared_v4(ba + at(q), pack2<F16>(oa[0], oa[1]), pack2<F16>(oa[2], oa[3]),
                       pack2<F16>(oa[4], oa[5]), pack2<F16>(oa[6], oa[7]));
          st_shared_v4(bb + at(q), pack2<F16>(ob[0], ob[1]), pack2<F16>(ob[2], ob[3]),
                       pack2<F16>(ob[4], ob[5]), pack2<F16>(ob[6], ob[7]));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(tm_out, ba, col0 + c0, row0);
          tma_store_2d(tm_out, bb, col0 + c0 + 64, row0);
          bulk_commit();
        }
      }
    }
  } else {
    RopeHalf v;
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {
      if (!warp_wait(cs_bar, cs_phase, abort_flag, status)) return false;
      cs_phase ^= 1u;
      v.load_shared(srow);
      if (half == 0) rope_stage(cs, 1, srow, cs_bar, lane);  // the row is in registers now
#pragma unroll 1
      for (int h = 0; h < BN / 128; ++h) {
        const int c0 = h * 128 + half * 32;
        uint32_t ra[32], rb[32];
        tmem_ld32(t_acc + c0, ra);
        tmem_ld32(t_acc + c0 + 64, rb);
        tmem_ld_wait();
        if (c0 >= ncols) continue;
        const uint32_t ba = buf;
        const uint32_t bb = buf + 2048u;
        if (lane == 0) bulk_wait_read<0>();  // both buffers are free again
        __syncwarp();
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float co[8] = {v.c[2 * q].x,     v.c[2 * q].y,     v.c[2 * q].z,     v.c[2 * q].w,
                               v.c[2 * q + 1].x, v.c[2 * q + 1].y, v.c[2 * q + 1].z, v.c[2 * q + 1].w};
          const float si[8] = {v.s[2 * q].x,     v.s[2 * q].y,     v.s[2 * q].z,     v.s[2 * q].w,
                               v.s[2 * q + 1].x, v.s[2 * q + 1].y, v.s[2 * q + 1].z, v.s[2 * q + 1].w};
          float oa[8], ob[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float a = __uint_as_float(ra[8 * q + e]);
            const float bv = __uint_as_float(rb[8 * q + e]);
            oa[e] = a * co[e] - bv * si[e];
            ob[e] = bv * co[e] + a * si[e];
          }
          st_shared_v4(ba + at(q), pack2<F16>(oa[0], oa[1]), pack2<F16>(oa[2], oa[3]),
                       pack2<F16>(oa[4], oa[5]), pack2<F16>(oa[6], oa[7]));
          st_shared_v4(bb + at(q), pack2<F16>(ob[0], ob[1]), pack2<F16>(ob[2], ob[3]),
                       pack2<F16>(ob[4], ob[5]), pack2<F16>(ob[6], ob[7]));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(tm_out, ba, col0 + c0, row0);
          tma_store_2d(tm_out, bb, col0 + c0 + 64, row0);
          bulk_commit();
        }
      }
    }
  }
  return true;
}

// SwiGLU epilogue for one warp (32 rows of the CTA's 128), [P4] §3.1 (the
// activation joined to the linear layers before it): the tile's accumulator
// holds the gate output g in columns [0, 128) and the up output u in
// [128, 256).  Per 32-column chunk it stores g and u (when saved for the
// backward) and h = silu(g)·u = g·u / (1 + e^{-g}), each rounded once from
// fp32 to bf16, through the warp's two 2 KB staging buffers in turn and TMA
// bulk stores at output column col0 + 32·chunk, row row0.  `nstore` counts
// the warp's stores (it picks the buffer).
template <bool F16>
LORA_DEV void epi_store_swiglu(uint32_t t_acc, uint32_t buf, const GemmParams &p, int col0,
                               int row0, int ncols, int lane, uint32_t &nstore) {
  auto at = [&](int q) -> uint32_t {
    return (uint32_t)(lane * 64 + ((q ^ ((lane >> 1) & 3)) << 4));
  };
  auto store = [&](const uint32_t (&v)[32], const CUtensorMap *map, int col) {
    const uint32_t b = buf + (nstore & 1u) * 2048u;
    ++nstore;
    if (lane == 0) bulk_wait_read<1>();  // this buffer's previous store has read it
    __syncwarp();
#pragma unroll
    for (int q = 0; q < 4; ++q)
      st_shared_v4(b + at(q), pack2<F16>(__uint_as_float(v[8 * q + 0]), __uint_as_float(v[8 * q + 1])),
                   pack2<F16>(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
                   pack2<F16>(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
                   pack2<F16>(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])));
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(map, b, col, row0);
      bulk_commit();
    }
  };
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    uint32_t rg[32], ru[32];
    tmem_ld32(t_acc + c * 32, rg);
    tmem_ld32(t_acc + 128 + c * 32, ru);
    tmem_ld_wait();
    if (c * 32 >= ncols) continue;
    if (p.save_gu) {
      store(rg, &p.grp[0].tm_out, col0 + c * 32);
      store(ru, &p.grp[1].tm_out, col0 + c * 32);
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float g = __uint_as_float(rg[j]);
      rg[j] = __float_as_uint(g * __uint_as_float(ru[j]) / (1.0f + expf(-g)));
    }
    store(rg, &p.tm_h, col0 + c * 32);
  }
}

// Down-projection in the GEMM: this thread's row of v (TMEM columns
// [0, nv) at t_v, fp32) scaled by `scale`, rounded to bf16 and written into
// the s·v operand region `sv` [FV/64 atoms][128 rows x 128 B] in the
// 128-byte-swizzled K-major layout the MMA reads.  Columns from nv on are
// written as zeros (the rank K-blocks read whole 64-column atoms).
template <int FV, bool F16>
LORA_DEV void stage_sv(uint32_t t_v, uint32_t sv, int row, int nv, float scale) {
#pragma unroll 1
  for (int c = 0; c < FV / 32; ++c) {
    uint32_t r[32];
    if (c * 32 < nv) {  // nv is uniform across the warp
      tmem_ld32(t_v + c * 32, r);
      tmem_ld_wait();
    }
#pragma unroll
    for (int j = 0; j < 32; ++j)
      r[j] = __float_as_uint(c * 32 + j < nv ? __uint_as_float(r[j]) * scale : 0.0f);
    const uint32_t rowp = sv + (uint32_t)(c >> 1) * 16384u + (uint32_t)row * 128u;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t chunk = (uint32_t)((c & 1) * 4 + q);
      st_shared_v4(rowp + ((chunk ^ ((uint32_t)row & 7u)) << 4),
                   pack2<F16>(__uint_as_float(r[8 * q + 0]), __uint_as_float(r[8 * q + 1])),
                   pack2<F16>(__uint_as_float(r[8 * q + 2]), __uint_as_float(r[8 * q + 3])),
                   pack2<F16>(__uint_as_float(r[8 * q + 4]), __uint_as_float(r[8 * q + 5])),
                   pack2<F16>(__uint_as_float(r[8 * q + 6]), __uint_as_float(r[8 * q + 7])));
    }
  }
}

// Position of output row `grow` for the RoPE epilogue; an out-of-range
// position is reported in the status word and replaced by 0 (no read
// outside the cache).
LORA_DEV const float *rope_row(const GemmParams &p, int grow, bool row_ok) {
  int pos = 0;
  if (row_ok) {
    pos = __ldg(p.positions + grow);
    if (pos < 0 || pos >= p.max_pos) {
      atomicOr(p.status, kDevBadPosition);
      pos = 0;
    }
  }
  return p.cos_sin + (size_t)pos * 128;
}

}  // namespace lora
