// Small kernels around the fused GEMMs: the backward set-up (inverse RoPE
// rotation of incoming gradients, merged A and Bᵀ), the cos/sin
// cache builder, and the standalone NF4 dequantise / quantise.
#include "kernels.h"
#include "nf4_levels.cuh"

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
  const __nv_bfloat16 *src = h < hq ? p.dy1 + (size_t)m * p.n1 + h * 128
                                    : p.dy2 + (size_t)m * p.n2 + (h - hq) * 128;
  __nv_bfloat16 *dst = p.dy_out + (size_t)m * (p.n1 + p.n2) + h * 128;
  const uint4 ua = *reinterpret_cast<const uint4 *>(src + g * 8);
  const uint4 ub = *reinterpret_cast<const uint4 *>(src + g * 8 + 64);
  const __nv_bfloat162 *a2 = reinterpret_cast<const __nv_bfloat162 *>(&ua);
  const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&ub);
  const float4 c0 = *reinterpret_cast<const float4 *>(c);
  const float4 c1 = *reinterpret_cast<const float4 *>(c + 4);
  const float4 s0 = *reinterpret_cast<const float4 *>(s);
  const float4 s1 = *reinterpret_cast<const float4 *>(s + 4);
  const float cc[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  const float ss[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
  uint32_t oa[4], ob[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float a0 = __low2float(a2[e]), a1 = __high2float(a2[e]);
    const float b0 = __low2float(b2[e]), b1 = __high2float(b2[e]);
    const float x0 = cc[2 * e], x1 = cc[2 * e + 1], y0 = ss[2 * e], y1 = ss[2 * e + 1];
    oa[e] = pack_bf16x2(a0 * x0 + b0 * y0, a1 * x1 + b1 * y1);
    ob[e] = pack_bf16x2(b0 * x0 - a0 * y0, b1 * x1 - a1 * y1);
  }
  *reinterpret_cast<uint4 *>(dst + g * 8) = make_uint4(oa[0], oa[1], oa[2], oa[3]);
  *reinterpret_cast<uint4 *>(dst + g * 8 + 64) = make_uint4(ob[0], ob[1], ob[2], ob[3]);
}

// SwiGLU backward of 8 consecutive columns of one row ("Unsloth框架" §3.1;
// SwiGLU as in "GLU Variants Improve Transformer" §2): with σ = sigmoid(g),
//   dg = dh·u·σ·(1 + g·(1 − σ)),   du = dh·g·σ,
// in fp32 from the bf16 dh, g, u, each rounded once to bf16 into dY = [dg | du].
LORA_DEV void swiglu_bwd_item(const BwdPrep &p, size_t i) {
  const int n = p.n1;
  const size_t m = i / (n / 8);
  const int c = (int)(i % (n / 8)) * 8;
  const size_t off = m * n + c;
  const uint4 vh = *reinterpret_cast<const uint4 *>(p.sw_dh + off);
  const uint4 vg = *reinterpret_cast<const uint4 *>(p.sw_g + off);
  const uint4 vu = *reinterpret_cast<const uint4 *>(p.sw_u + off);
  const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&vh);
  const __nv_bfloat162 *g2 = reinterpret_cast<const __nv_bfloat162 *>(&vg);
  const __nv_bfloat162 *u2 = reinterpret_cast<const __nv_bfloat162 *>(&vu);
  uint32_t og[4], ou[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float dg[2], du[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const float dh = t ? __high2float(h2[e]) : __low2float(h2[e]);
      const float g = t ? __high2float(g2[e]) : __low2float(g2[e]);
      const float u = t ? __high2float(u2[e]) : __low2float(u2[e]);
      const float sg = 1.0f / (1.0f + expf(-g));
      dg[t] = dh * u * sg * (1.0f + g * (1.0f - sg));
      du[t] = dh * g * sg;
    }
    og[e] = pack_bf16x2(dg[0], dg[1]);
    ou[e] = pack_bf16x2(du[0], du[1]);
  }
  __nv_bfloat16 *dst = p.dy_out + m * (size_t)(2 * n) + c;
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
        rope_bwd_item(p, i);
      else
        swiglu_bwd_item(p, i);
    } else if (i < n_rope + n_a) {
      const size_t q = i - n_rope, half = (size_t)p.r * p.k / 8;
      const uint4 *src = reinterpret_cast<const uint4 *>(q < half ? p.A1 : p.A2);
      reinterpret_cast<uint4 *>(p.A_out)[q] = src[q < half ? q : q - half];
    } else {
      const size_t q = i - n_rope - n_a;
      const int j = (int)(q / n), o = (int)(q % n);   // Bt row j (rank), column o
      __nv_bfloat16 v = __float2bfloat16_rn(0.0f);
      if (o < p.n1 && j < p.r) v = p.B1[(size_t)o * p.r + j];
      else if (o >= p.n1 && j >= p.r) v = p.B2[(size_t)(o - p.n1) * p.r + (j - p.r)];
      p.Bt[q] = v;
    }
  }
}

cudaError_t launch_bwd_prep(const BwdPrep &p, cudaStream_t st) {
  const int n = p.n1 + p.n2, rl = p.nproj * p.r;
  const size_t total = dy_items(p) + (p.nproj > 1 ? (size_t)rl * p.k / 8 : 0) + (size_t)rl * n;
  return launch_pdl("bwd_prep_kernel", bwd_prep_kernel, dim3(grid_for(total, 256, 16)), dim3(256), 0, st, 0u,
                    p);
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

// ------------------------------------------------------------ NF4 dequant

// One thread per 32-bit code word (8 elements, 16 output bytes), so a
// warp's code loads are 128 contiguous bytes and its stores 512; the eight
// threads of a 64-element block read the same absmax.  Each element is the
// fp32 product level·absmax rounded once to bf16, the level read from a
// 16-entry shared table (conflict-free: 16 banks, equal codes broadcast).
// Four words per thread per trip keep more loads in flight.  HBM-bound:
// reads n·k/2 + n·k/32 bytes, writes 2·n·k bytes.
__device__ __forceinline__ uint4 dq_word(uint32_t c, float a, const float *lv) {
  uint32_t o[4];
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const uint32_t byte = (c >> (8 * b)) & 0xFFu;
    o[b] = pack_bf16x2(lv[byte >> 4] * a, lv[byte & 0xFu] * a);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

__global__ void __launch_bounds__(256) nf4_dequant_kernel(const uint8_t *__restrict__ codes,
                                                          const __nv_bfloat16 *__restrict__ absmax,
                                                          __nv_bfloat16 *__restrict__ w,
                                                          size_t n_words) {
  __shared__ float lv[16];
  if (threadIdx.x < 16) lv[threadIdx.x] = kNf4Levels[threadIdx.x];
  __syncthreads();
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
      a[u] = __bfloat162float(absmax[(i + u * stride) >> 3]);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) __stcs(w4 + i + u * stride, dq_word(c[u], a[u], lv));
  }
  for (; i < n_words; i += stride)
    __stcs(w4 + i, dq_word(__ldcs(c32 + i), __bfloat162float(absmax[i >> 3]), lv));
}

cudaError_t launch_nf4_dequant(const uint8_t *codes, const __nv_bfloat16 *absmax,
                               __nv_bfloat16 *w, int n, int k, cudaStream_t st) {
  const size_t words = (size_t)n * k / 8;
  const int grid = grid_for(words, 256, 8);
  launch_begin(st);
  nf4_dequant_kernel<<<grid, 256, 0, st>>>(codes, absmax, w, words);
  note_launch("nf4_dequant_kernel", st);
  return cudaGetLastError();
}

// ----------------------------------------------------------- NF4 quantise
// One thread per 64-element block: absmax = max|w| (exact in bf16 because
// the inputs are bf16), code = first index minimising |w/absmax - level|
// in IEEE fp32; all-zero blocks get code 7.
__global__ void nf4_quantize_kernel(const __nv_bfloat16 *__restrict__ w, uint8_t *__restrict__ codes,
                                    __nv_bfloat16 *__restrict__ absmax, size_t n_blocks) {
  __shared__ float lv[16];
  if (threadIdx.x < 16) lv[threadIdx.x] = kNf4Levels[threadIdx.x];
  __syncthreads();
  for (size_t b = blockIdx.x * (size_t)blockDim.x + threadIdx.x; b < n_blocks;
       b += (size_t)gridDim.x * blockDim.x) {
    const uint4 *src = reinterpret_cast<const uint4 *>(w + b * 64);
    float v[64];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const uint4 u = src[q];
      const uint32_t ws[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162 *>(&ws[e]);
        v[8 * q + 2 * e] = __low2float(h);
        v[8 * q + 2 * e + 1] = __high2float(h);
      }
    }
    float am = 0.0f;
#pragma unroll
    for (int e = 0; e < 64; ++e) am = fmaxf(am, fabsf(v[e]));
    const __nv_bfloat16 amb = __float2bfloat16_rn(am);
    absmax[b] = amb;
    const float a = __bfloat162float(amb);
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
    uint4 *dst = reinterpret_cast<uint4 *>(codes + b * 32);
    dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
    dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
  }
}

cudaError_t launch_nf4_quantize(const __nv_bfloat16 *w, uint8_t *codes, __nv_bfloat16 *absmax,
                                int n, int k, cudaStream_t st) {
  const size_t blocks = (size_t)n * k / 64;
  const int grid = grid_for(blocks, 128, 8);
  launch_begin(st);
  nf4_quantize_kernel<<<grid, 128, 0, st>>>(w, codes, absmax, blocks);
  note_launch("nf4_quantize_kernel", st);
  return cudaGetLastError();
}

}  // namespace lora
