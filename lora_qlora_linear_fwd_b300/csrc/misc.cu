// Small kernels around the fused GEMMs: the backward set-up (inverse RoPE
// rotation of incoming gradients, merged A and Bᵀ), the cos/sin
// cache builder, and the standalone NF4 dequantise / quantise.
#include "kernels.h"
#include "nf4_levels.cuh"
#include "philox.cuh"

#include <cuda_fp8.h>

namespace lora {

// Blocks for `items` work items of `per_block` each, capped at
// `per_sm` resident blocks on every SM of the current device (grid-stride
// loops take the rest).
static int grid_for(size_t items, int per_block, int per_sm) {
  const size_t g = (items + per_block - 1) / per_block;
  const int sms = current_device_sms();
  const size_t cap = (size_t)(sms > 0 ? sms : 1) * (size_t)per_sm;
  return (int)(g < cap ? (g > 0 ? g : 1) : cap);
}

// ------------------------------------------------------- backward set-up
// Everything the backward needs before its GEMM and rank-r passes, in one
// launch (three independent jobs over one flat index space):
//   rope     dY[:, :n1] = R(pos)ᵀ·dy1, dY[:, n1:] = R(pos)ᵀ·dy2 (inverse
//            rotate-half per 128-wide head; one item = one row, head and
//            group of 8 pair indices)
//   A        A_out = [A1; A2] (two projections merged as rank 2r)
//   Bᵀ       Bt [nproj·r, n] = diag(B1, B2)ᵀ (just B1ᵀ for one projection)
template <bool F16>
LORA_DEV void rope_bwd_item(const BwdPrep &p, size_t i) {
  const int hq = p.n1 / 128, hk = p.n2 / 128, heads = hq + hk;
  const int g = (int)(i % 8);
  const size_t mh = i / 8;
  const int h = (int)(mh % heads);
  const int m = (int)(mh / heads);
  int pos = p.pos[m];
  if (pos < 0 || pos >= p.max_pos) {
    atomicOr(p.status, kDevBadPosition);
    pos = 0;
  }
  const float *c = p.cos_sin + (size_t)pos * 128 + g * 8;
  const float *s = c + 64;
  const uint16_t *src = h < hq ? p.dy1 + (size_t)m * p.n1 + h * 128
                               : p.dy2 + (size_t)m * p.n2 + (h - hq) * 128;
  uint16_t *dst = p.dy_out + (size_t)m * (p.n1 + p.n2) + h * 128;
  const uint4 ua = *reinterpret_cast<const uint4 *>(src + g * 8);
  const uint4 ub = *reinterpret_cast<const uint4 *>(src + g * 8 + 64);
  const uint32_t wa[4] = {ua.x, ua.y, ua.z, ua.w}, wb[4] = {ub.x, ub.y, ub.z, ub.w};
  const float4 c0 = *reinterpret_cast<const float4 *>(c);
  const float4 c1 = *reinterpret_cast<const float4 *>(c + 4);
  const float4 s0 = *reinterpret_cast<const float4 *>(s);
  const float4 s1 = *reinterpret_cast<const float4 *>(s + 4);
  const float cc[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  const float ss[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
  uint32_t oa[4], ob[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 a = unpack2<F16>(wa[e]), b = unpack2<F16>(wb[e]);
    const float x0 = cc[2 * e], x1 = cc[2 * e + 1], y0 = ss[2 * e], y1 = ss[2 * e + 1];
    oa[e] = pack2<F16>(a.x * x0 + b.x * y0, a.y * x1 + b.y * y1);
    ob[e] = pack2<F16>(b.x * x0 - a.x * y0, b.y * x1 - a.y * y1);
  }
  *reinterpret_cast<uint4 *>(dst + g * 8) = make_uint4(oa[0], oa[1], oa[2], oa[3]);
  *reinterpret_cast<uint4 *>(dst + g * 8 + 64) = make_uint4(ob[0], ob[1], ob[2], ob[3]);
}

// SwiGLU backward of 8 consecutive columns of one row ("Unsloth框架" §3.1;
// SwiGLU as in "GLU Variants Improve Transformer" §2): with σ = sigmoid(g),
//   dg = dh·u·σ·(1 + g·(1 − σ)),   du = dh·g·σ,
// in fp32 from the 16-bit dh, g, u, each rounded once to the 16-bit type
// into dY = [dg | du].
template <bool F16>
LORA_DEV void swiglu_bwd_item(const BwdPrep &p, size_t i) {
  const int n = p.n1;
  const size_t m = i / (n / 8);
  const int c = (int)(i % (n / 8)) * 8;
  const size_t off = m * n + c;
  const uint4 vh = *reinterpret_cast<const uint4 *>(p.sw_dh + off);
  const uint4 vg = *reinterpret_cast<const uint4 *>(p.sw_g + off);
  const uint4 vu = *reinterpret_cast<const uint4 *>(p.sw_u + off);
  const uint32_t h2[4] = {vh.x, vh.y, vh.z, vh.w};
  const uint32_t g2[4] = {vg.x, vg.y, vg.z, vg.w};
  const uint32_t u2[4] = {vu.x, vu.y, vu.z, vu.w};
  uint32_t og[4], ou[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float dg[2], du[2];
    const float2 fh = unpack2<F16>(h2[e]), fg = unpack2<F16>(g2[e]), fu = unpack2<F16>(u2[e]);
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const float dh = t ? fh.y : fh.x;
      const float g = t ? fg.y : fg.x;
      const float u = t ? fu.y : fu.x;
      const float sg = 1.0f / (1.0f + expf(-g));
      dg[t] = dh * u * sg * (1.0f + g * (1.0f - sg));
      du[t] = dh * g * sg;
    }
    og[e] = pack2<F16>(dg[0], dg[1]);
    ou[e] = pack2<F16>(du[0], du[1]);
  }
  uint16_t *dst = p.dy_out + m * (size_t)(2 * n) + c;
  *reinterpret_cast<uint4 *>(dst) = make_uint4(og[0], og[1], og[2], og[3]);
  *reinterpret_cast<uint4 *>(dst + n) = make_uint4(ou[0], ou[1], ou[2], ou[3]);
}

// Work items of the gradient job: rotation (8 per row and head) or SwiGLU
// (one per 8 columns of a row).
__host__ __device__ static inline size_t dy_items(const BwdPrep &p) {
  const int n = p.n1 + p.n2;
  if (p.dy1) return (size_t)p.M * (n / 128) * 8;
  if (p.sw_dh) return (size_t)p.M * (p.n1 / 8);
  return 0;
}

template <bool F16>
__global__ void bwd_prep_kernel(const BwdPrep p) {
  grid_dep_launch();
  grid_dep_wait();
  const int n = p.n1 + p.n2, rl = p.nproj * p.r;
  const size_t n_rope = dy_items(p);
  const size_t n_a = p.nproj > 1 ? (size_t)rl * p.k / 8 : 0;   // 16-byte pieces
  const size_t n_b = (size_t)rl * n;
  const size_t total = n_rope + n_a + n_b;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x) {
    if (i < n_rope) {
      if (p.dy1)
        rope_bwd_item<F16>(p, i);
      else
        swiglu_bwd_item<F16>(p, i);
    } else if (i < n_rope + n_a) {
      const size_t q = i - n_rope, half = (size_t)p.r * p.k / 8;
      const uint4 *src = reinterpret_cast<const uint4 *>(q < half ? p.A1 : p.A2);
      reinterpret_cast<uint4 *>(p.A_out)[q] = src[q < half ? q : q - half];
    } else {
      const size_t q = i - n_rope - n_a;
      const int j = (int)(q / n), o = (int)(q % n);   // Bt row j (rank), column o
      uint16_t v = 0;  // +0 in either 16-bit type
      if (o < p.n1 && j < p.r) v = p.B1[(size_t)o * p.r + j];
      else if (o >= p.n1 && j >= p.r) v = p.B2[(size_t)(o - p.n1) * p.r + (j - p.r)];
      p.Bt[q] = v;
    }
  }
}

cudaError_t launch_bwd_prep(const BwdPrep &p, bool f16, cudaStream_t st) {
  const int n = p.n1 + p.n2, rl = p.nproj * p.r;
  const size_t total = dy_items(p) + (p.nproj > 1 ? (size_t)rl * p.k / 8 : 0) + (size_t)rl * n;
  const dim3 grid(grid_for(total, 256, 16));
  return f16 ? launch_pdl("bwd_prep_kernel<f16>", bwd_prep_kernel<true>, grid, dim3(256), 0, st,
                          0u, p)
             : launch_pdl("bwd_prep_kernel", bwd_prep_kernel<false>, grid, dim3(256), 0, st, 0u, p);
}

// --------------------------------------------------------------- RoPE cache
// cos_sin [max_pos, D]: row p = cos(p·f_i) (i < D/2), then sin(p·f_i),
// f_i = theta^(-2i/D); fp64 angle and trigonometry, stored as fp32.
__global__ void rope_cache_kernel(float *__restrict__ cs, int max_pos, int D, double theta) {
  const int h = D / 2;
  const size_t total = (size_t)max_pos * h;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x) {
    const int p = (int)(i / h), f = (int)(i % h);
    const double inv_freq = pow(theta, -2.0 * (double)f / (double)D);
    double s, c;
    sincos((double)p * inv_freq, &s, &c);
    cs[(size_t)p * D + f] = (float)c;
    cs[(size_t)p * D + h + f] = (float)s;
  }
}

cudaError_t launch_rope_cache(float *cos_sin, int max_pos, int head_dim, double theta,
                              cudaStream_t st) {
  const size_t total = (size_t)max_pos * (head_dim / 2);
  const int grid = grid_for(total, 256, 16);
  launch_begin(st);
  rope_cache_kernel<<<grid, 256, 0, st>>>(cos_sin, max_pos, head_dim, theta);
  note_launch("rope_cache_kernel", st);
  return cudaGetLastError();
}

// --------------------------------------------------------------- dropout
// x̃ = x ⊙ keep / q into `out` (16-bit, rounded once from the fp32 product),
// one 16-element Philox block per thread and trip (k % 16 == 0, so a block
// never straddles a row).  HBM-bound: reads and writes 2·M·k bytes.
template <bool F16>
__global__ void __launch_bounds__(256) dropout_x_kernel(const uint16_t *__restrict__ x,
                                                        uint16_t *__restrict__ out,
                                                        size_t n_blocks, uint64_t seed,
                                                        uint64_t offset, uint32_t thresh,
                                                        float inv_q) {
  grid_dep_launch();
  grid_dep_wait();
  for (size_t b = blockIdx.x * (size_t)blockDim.x + threadIdx.x; b < n_blocks;
       b += (size_t)gridDim.x * blockDim.x) {
    const uint32_t keep = dropout_keep16(b, seed, offset, thresh);
    const uint4 *src = reinterpret_cast<const uint4 *>(x) + 2 * b;
    uint4 *dst = reinterpret_cast<uint4 *>(out) + 2 * b;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint4 v = __ldcs(src + h);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 t = unpack2<F16>(w[e]);
        const int i0 = 8 * h + 2 * e;
        const float f0 = (keep >> i0) & 1u ? t.x * inv_q : 0.0f;
        const float f1 = (keep >> (i0 + 1)) & 1u ? t.y * inv_q : 0.0f;
        o[e] = pack2<F16>(f0, f1);
      }
      dst[h] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

cudaError_t launch_dropout_x(const uint16_t *x, uint16_t *out, int M, int k, uint64_t seed,
                             uint64_t offset, uint32_t thresh, float inv_q, bool f16,
                             cudaStream_t st) {
  const size_t blocks = (size_t)M * k / 16;
  const dim3 grid(grid_for(blocks, 256, 8));
  return f16 ? launch_pdl("dropout_x_kernel<f16>", dropout_x_kernel<true>, grid, dim3(256), 0, st,
                          0u, x, out, blocks, seed, offset, thresh, inv_q)
             : launch_pdl("dropout_x_kernel", dropout_x_kernel<false>, grid, dim3(256), 0, st, 0u,
                          x, out, blocks, seed, offset, thresh, inv_q);
}

// ------------------------------------------------------------ NF4 dequant

// One thread per 32-bit code word (8 elements, 16 output bytes), so a
// warp's code loads are 128 contiguous bytes and its stores 512; the eight
// threads of a 64-element block read the same block scale.  Each element is
// the fp32 product level·absmax rounded once to the 16-bit type, the level
// read from a 16-entry shared table (conflict-free: 16 banks, equal codes
// broadcast).  Four words per thread per trip keep more loads in flight.
// HBM-bound: reads n·k/2 + n·k/32 bytes (n·k/64 + 1/64 of that with double
// quantisation), writes 2·n·k bytes.
template <bool F16>
__device__ __forceinline__ uint4 dq_word(uint32_t c, float a, const float *lv) {
  uint32_t o[4];
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const uint32_t byte = (c >> (8 * b)) & 0xFFu;
    o[b] = pack2<F16>(lv[byte >> 4] * a, lv[byte & 0xFu] * a);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Block scale of 64-element block b.
template <bool DQ>
__device__ __forceinline__ float block_scale(const Nf4Scales &sc, size_t b, float offset) {
  if constexpr (DQ)
    return dq_absmax(__ldg(static_cast<const uint8_t *>(sc.absmax) + b),
                     __ldg(sc.dq_scale + b / kDqGroup), offset);
  else
    return __bfloat162float(static_cast<const __nv_bfloat16 *>(sc.absmax)[b]);
}

template <bool F16, bool DQ>
__global__ void __launch_bounds__(256) nf4_dequant_kernel(const uint8_t *__restrict__ codes,
                                                          const Nf4Scales sc,
                                                          uint16_t *__restrict__ w,
                                                          size_t n_words) {
  __shared__ float lv[16];
  if (threadIdx.x < 16) lv[threadIdx.x] = kNf4Levels[threadIdx.x];
  __syncthreads();
  const float offset = DQ ? __ldg(sc.dq_offset) : 0.0f;
  const uint32_t *c32 = reinterpret_cast<const uint32_t *>(codes);
  uint4 *w4 = reinterpret_cast<uint4 *>(w);
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n_words; i += 4 * stride) {
    uint32_t c[4];
    float a[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      c[u] = __ldcs(c32 + i + u * stride);
      a[u] = block_scale<DQ>(sc, (i + u * stride) >> 3, offset);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) __stcs(w4 + i + u * stride, dq_word<F16>(c[u], a[u], lv));
  }
  for (; i < n_words; i += stride)
    __stcs(w4 + i, dq_word<F16>(__ldcs(c32 + i), block_scale<DQ>(sc, i >> 3, offset), lv));
}

cudaError_t launch_nf4_dequant(const uint8_t *codes, const Nf4Scales &sc, uint16_t *w, int n,
                               int k, bool f16, cudaStream_t st) {
  const size_t words = (size_t)n * k / 8;
  const int grid = grid_for(words, 256, 8);
  const bool dq = sc.dq_scale != nullptr;
  launch_begin(st);
  if (f16) {
    if (dq)
      nf4_dequant_kernel<true, true><<<grid, 256, 0, st>>>(codes, sc, w, words);
    else
      nf4_dequant_kernel<true, false><<<grid, 256, 0, st>>>(codes, sc, w, words);
  } else {
    if (dq)
      nf4_dequant_kernel<false, true><<<grid, 256, 0, st>>>(codes, sc, w, words);
    else
      nf4_dequant_kernel<false, false><<<grid, 256, 0, st>>>(codes, sc, w, words);
  }
  note_launch(f16 ? (dq ? "nf4_dequant_kernel<f16,dq>" : "nf4_dequant_kernel<f16>")
                  : (dq ? "nf4_dequant_kernel<dq>" : "nf4_dequant_kernel"),
              st);
  return cudaGetLastError();
}

// Double-quantised block scales expanded to bf16 [nb] (the form the fused
// GEMMs read): one thread per 8 blocks (8 code bytes in, 16 bytes out; the 8
// share a group, 256 % 8 == 0).  nb % 8 == 0.
__global__ void __launch_bounds__(256) nf4_dq_expand_kernel(const Nf4Scales sc,
                                                            uint16_t *__restrict__ out,
                                                            size_t n8) {
  grid_dep_launch();
  grid_dep_wait();
  const float offset = __ldg(sc.dq_offset);
  const uint2 *q8 = static_cast<const uint2 *>(sc.absmax);
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n8;
       i += (size_t)gridDim.x * blockDim.x) {
    const uint2 q = __ldg(q8 + i);
    const float s = __ldg(sc.dq_scale + (8 * i) / kDqGroup);
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t word = e < 2 ? q.x : q.y;
      const int sh = 16 * (e & 1);
      o[e] = pack_bf16x2(dq_absmax((word >> sh) & 0xFFu, s, offset),
                         dq_absmax((word >> (sh + 8)) & 0xFFu, s, offset));
    }
    reinterpret_cast<uint4 *>(out)[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

cudaError_t launch_nf4_dq_expand(const Nf4Scales &sc, uint16_t *absmax_out, size_t nb,
                                 cudaStream_t st) {
  const size_t n8 = nb / 8;
  return launch_pdl("nf4_dq_expand_kernel", nf4_dq_expand_kernel, dim3(grid_for(n8, 256, 8)),
                    dim3(256), 0, st, 0u, sc, absmax_out, n8);
}

// ----------------------------------------------------------- NF4 quantise
// Codes of one 64-element block against block scale `a`: the first index
// minimising |w/a - level| in IEEE fp32 (w/a clamped to [-1, 1]); a == 0
// gives code 7 (the exact zero).  Packed two per byte, high nibble first,
// into 32 bytes at `dst`.
LORA_DEV void nf4_code_block(const float (&v)[64], float a, const float *lv, uint8_t *dst) {
  uint32_t out[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) out[q] = 0;
#pragma unroll
  for (int e = 0; e < 64; ++e) {
    uint32_t best = 7;
    if (a != 0.0f) {
      float ratio = __fdiv_rn(v[e], a);
      ratio = fminf(fmaxf(ratio, -1.0f), 1.0f);
      float bestd = fabsf(__fsub_rn(ratio, lv[0]));
      best = 0;
#pragma unroll
      for (int t = 1; t < 16; ++t) {
        const float d = fabsf(__fsub_rn(ratio, lv[t]));
        if (d < bestd) bestd = d, best = t;
      }
    }
    // byte j = (code[2j] << 4) | code[2j+1]; bytes little-endian in words
    const int byte = e >> 1;
    const uint32_t nib = (e & 1) ? best : (best << 4);
    out[byte >> 2] |= nib << (8 * (byte & 3));
  }
  uint4 *d4 = reinterpret_cast<uint4 *>(dst);
  d4[0] = make_uint4(out[0], out[1], out[2], out[3]);
  d4[1] = make_uint4(out[4], out[5], out[6], out[7]);
}

// The 64 elements of block b as fp32, and their max |w| (exact).
template <bool F16>
LORA_DEV float load_block64(const uint16_t *w, size_t b, float (&v)[64]) {
  const uint4 *src = reinterpret_cast<const uint4 *>(w + b * 64);
  float am = 0.0f;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const uint4 u = src[q];
    const uint32_t ws[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 h = unpack2<F16>(ws[e]);
      v[8 * q + 2 * e] = h.x;
      v[8 * q + 2 * e + 1] = h.y;
      am = fmaxf(am, fmaxf(fabsf(h.x), fabsf(h.y)));
    }
  }
  return am;
}

// Single-level scales: one thread per 64-element block, absmax =
// bf16(max|w|) (round to nearest even; exact for bf16 inputs).
template <bool F16>
__global__ void nf4_quantize_kernel(const uint16_t *__restrict__ w, uint8_t *__restrict__ codes,
                                    __nv_bfloat16 *__restrict__ absmax, size_t n_blocks) {
  __shared__ float lv[16];
  if (threadIdx.x < 16) lv[threadIdx.x] = kNf4Levels[threadIdx.x];
  __syncthreads();
  for (size_t b = blockIdx.x * (size_t)blockDim.x + threadIdx.x; b < n_blocks;
       b += (size_t)gridDim.x * blockDim.x) {
    float v[64];
    const __nv_bfloat16 amb = __float2bfloat16_rn(load_block64<F16>(w, b, v));
    absmax[b] = amb;
    nf4_code_block(v, __bfloat162float(amb), lv, codes + b * 32);
  }
}

// Double quantisation, pass 1: one CTA per group of 256 blocks, a thread per
// block.  Writes the group's Σ max|w| (fp64, fixed reduction order), min and
// max into the first 16 bytes of the group's 256 code bytes (overwritten by
// pass 3; the last group holds at least 64 blocks because n % 64 == 0).
struct DqStats {
  double sum;
  float mn, mx;
};

template <bool F16>
__global__ void __launch_bounds__(256) nf4_dq_stats_kernel(const uint16_t *__restrict__ w,
                                                           uint8_t *__restrict__ qcodes,
                                                           size_t nb) {
  __shared__ double ssum[256];
  __shared__ float smn[256], smx[256];
  const size_t b = (size_t)blockIdx.x * kDqGroup + threadIdx.x;
  float c1 = 0.0f;
  const bool in = b < nb;
  if (in) {
    float v[64];
    c1 = load_block64<F16>(w, b, v);
  }
  ssum[threadIdx.x] = in ? (double)c1 : 0.0;
  smn[threadIdx.x] = in ? c1 : INFINITY;
  smx[threadIdx.x] = in ? c1 : -INFINITY;
  __syncthreads();
  for (int h = 128; h > 0; h >>= 1) {
    if ((int)threadIdx.x < h) {
      ssum[threadIdx.x] += ssum[threadIdx.x + h];
      smn[threadIdx.x] = fminf(smn[threadIdx.x], smn[threadIdx.x + h]);
      smx[threadIdx.x] = fmaxf(smx[threadIdx.x], smx[threadIdx.x + h]);
    }
    __syncthreads();
  }
  if (threadIdx.x == 0)
    *reinterpret_cast<DqStats *>(qcodes + (size_t)blockIdx.x * kDqGroup) =
        DqStats{ssum[0], smn[0], smx[0]};
}

// Pass 2, one CTA of 1024 threads: offset = fp32(Σ / nb) (each thread sums
// its groups in order, then a fixed tree), and per group
// scale = fp32(max(|mx - offset|, |mn - offset|) / 448), the fp32 differences
// rounded to nearest (max |c1 - offset| over the group, because rounding is
// monotonic).
__global__ void __launch_bounds__(1024) nf4_dq_scale_kernel(const uint8_t *__restrict__ qcodes,
                                                            float *__restrict__ scale,
                                                            float *__restrict__ offset,
                                                            size_t nb, int ng) {
  __shared__ double ssum[1024];
  __shared__ float s_off;
  double acc = 0.0;
  for (int g = threadIdx.x; g < ng; g += 1024)
    acc += reinterpret_cast<const DqStats *>(qcodes + (size_t)g * kDqGroup)->sum;
  ssum[threadIdx.x] = acc;
  __syncthreads();
  for (int h = 512; h > 0; h >>= 1) {
    if ((int)threadIdx.x < h) ssum[threadIdx.x] += ssum[threadIdx.x + h];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    s_off = (float)(ssum[0] / (double)nb);
    *offset = s_off;
  }
  __syncthreads();
  const float off = s_off;
  for (int g = threadIdx.x; g < ng; g += 1024) {
    const DqStats st = *reinterpret_cast<const DqStats *>(qcodes + (size_t)g * kDqGroup);
    const float m = fmaxf(fabsf(__fsub_rn(st.mx, off)), fabsf(__fsub_rn(st.mn, off)));
    scale[g] = __fdiv_rn(m, kE4m3Max);
  }
}

// Pass 3: one CTA per group, a thread per block: the first-level constant
// again (max|w|), its E4M3 code of fp32((c1 - offset) / scale) (round to
// nearest even, saturating; code 0 when the group's scale is 0), and the
// NF4 codes against the block scale that code decodes to.
template <bool F16>
__global__ void __launch_bounds__(256) nf4_dq_quantize_kernel(const uint16_t *__restrict__ w,
                                                              uint8_t *__restrict__ codes,
                                                              uint8_t *__restrict__ qcodes,
                                                              const float *__restrict__ scale,
                                                              const float *__restrict__ offset,
                                                              size_t nb) {
  __shared__ float lv[16];
  if (threadIdx.x < 16) lv[threadIdx.x] = kNf4Levels[threadIdx.x];
  __syncthreads();
  const size_t b = (size_t)blockIdx.x * kDqGroup + threadIdx.x;
  const float s = scale[blockIdx.x], off = *offset;
  if (b >= nb) return;
  float v[64];
  const float c1 = load_block64<F16>(w, b, v);
  uint32_t q = 0;
  if (s > 0.0f)
    q = (uint32_t)__nv_cvt_float_to_fp8(__fdiv_rn(__fsub_rn(c1, off), s), __NV_SATFINITE,
                                        __NV_E4M3);
  qcodes[b] = (uint8_t)q;
  nf4_code_block(v, dq_absmax(q, s, off), lv, codes + b * 32);
}

cudaError_t launch_nf4_quantize(const uint16_t *w, uint8_t *codes, void *absmax, float *dq_scale,
                                float *dq_offset, int n, int k, bool f16, cudaStream_t st) {
  const size_t blocks = (size_t)n * k / 64;
  if (!dq_scale) {
    const int grid = grid_for(blocks, 128, 8);
    launch_begin(st);
    if (f16)
      nf4_quantize_kernel<true><<<grid, 128, 0, st>>>(w, codes, static_cast<__nv_bfloat16 *>(absmax),
                                                      blocks);
    else
      nf4_quantize_kernel<false><<<grid, 128, 0, st>>>(w, codes,
                                                       static_cast<__nv_bfloat16 *>(absmax), blocks);
    note_launch(f16 ? "nf4_quantize_kernel<f16>" : "nf4_quantize_kernel", st);
    return cudaGetLastError();
  }
  const int ng = (int)((blocks + kDqGroup - 1) / kDqGroup);
  uint8_t *q = static_cast<uint8_t *>(absmax);
  launch_begin(st);
  if (f16)
    nf4_dq_stats_kernel<true><<<ng, 256, 0, st>>>(w, q, blocks);
  else
    nf4_dq_stats_kernel<false><<<ng, 256, 0, st>>>(w, q, blocks);
  note_launch("nf4_dq_stats_kernel", st);
  launch_begin(st);
  nf4_dq_scale_kernel<<<1, 1024, 0, st>>>(q, dq_scale, dq_offset, blocks, ng);
  note_launch("nf4_dq_scale_kernel", st);
  launch_begin(st);
  if (f16)
    nf4_dq_quantize_kernel<true><<<ng, 256, 0, st>>>(w, codes, q, dq_scale, dq_offset, blocks);
  else
    nf4_dq_quantize_kernel<false><<<ng, 256, 0, st>>>(w, codes, q, dq_scale, dq_offset, blocks);
  note_launch("nf4_dq_quantize_kernel", st);
  return cudaGetLastError();
}

}  // namespace lora
