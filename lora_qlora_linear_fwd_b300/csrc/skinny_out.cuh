// Output stage of the rank passes (skinny.cu, skinny_sk.cu): the final
// [128 x cw] fp32 block of a row tile, staged in shared memory, is written out
// in the layouts of the SkinnyOut kinds with warp-wide stores of 256-512
// contiguous bytes.
#pragma once

#include "kernels.h"

namespace lora {

// Epilogue buffers, laid over the (then idle) TMA ring.  In the cluster
// schedule a CTA of a cluster of S finalises the column block
// [CW·rank, CW·rank + CW), CW = RP / S; the stream-K schedule stages a whole
// tile (S = 1, no recv slots):
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
LORA_DEV void skinny_copy_out(const SkinnyDest &P, int rt, int col0, int cw,
                              const float *stage_t, const float *stage_r, int e) {
  const int cols = P.nproj * P.r;  // valid rank columns
  const int row0 = rt * 128;
  const int w = e >> 5, l = e & 31;
  // transposed outputs: warp w takes block columns j = w, w + 4, ...; lane l
  // takes rows [4l, 4l + 4) of the tile
  if (P.out_kind & (kOutVt | kOutRowT | kOutT16)) {
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
      if ((P.out_kind & kOutT16) && jg < cols) {
        uint16_t *dst = P.out_bf16 + (size_t)jg * P.ld_t + orow;
        const uint32_t w0 = pack2<F16>(f[0] * P.scale, f[1] * P.scale);
        const uint32_t w1 = pack2<F16>(f[2] * P.scale, f[3] * P.scale);
        if (full) {
          *reinterpret_cast<uint2 *>(dst) = make_uint2(w0, w1);
        } else {
          for (int q = 0; q < 4; ++q)
            if (orow + q < P.rows) dst[q] = to16<F16>(f[q] * P.scale);
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

}  // namespace lora
