// Small kernels around the fused GEMMs: slice reductions of the rank-r
// passes, the inverse RoPE rotation of incoming gradients, the cos/sin cache
// builder, the Bᵀ copy, and the standalone NF4 dequantise / quantise.
#include "kernels.h"

namespace lora {

static int grid_for(size_t items, int per_block, int cap) {
  const size_t g = (items + per_block - 1) / per_block;
  return (int)(g < (size_t)cap ? (g > 0 ? g : 1) : (size_t)cap);
}

// ---------------------------------------------------------------- Bᵀ copy
// Bt [r, n] <- B [n, r]
__global__ void transpose_rank_kernel(const __nv_bfloat16 *__restrict__ B,
                                      __nv_bfloat16 *__restrict__ Bt, int n, int r) {
  const size_t total = (size_t)n * r;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x) {
    const int j = (int)(i / n), c = (int)(i % n);  // output index: row j, column c
    Bt[i] = B[(size_t)c * r + j];
  }
}

cudaError_t launch_transpose_rank(const __nv_bfloat16 *B, __nv_bfloat16 *Bt, int n, int r,
                                  cudaStream_t st) {
  const size_t total = (size_t)n * r;
  const int grid = grid_for(total, 256, 4096);
  transpose_rank_kernel<<<grid, 256, 0, st>>>(B, Bt, n, r);
  note_launch();
  return cudaGetLastError();
}

// ------------------------------------------------------------- RoPE backward
// out = R(pos)ᵀ · dy per 128-wide head (inverse rotate-half), bf16 in/out.
// dy rows have ncols elements; out rows start out_ld elements apart (so two
// projections can be written side by side).  One thread per (row, head,
// group of 8 pair indices).
__global__ void rope_bwd_kernel(const __nv_bfloat16 *__restrict__ dy,
                                __nv_bfloat16 *__restrict__ out, int M, int ncols, int out_ld,
                                const int32_t *__restrict__ pos, const float *__restrict__ cs,
                                int max_pos, uint32_t *status) {
  const int heads = ncols / 128;
  const size_t total = (size_t)M * heads * 8;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x) {
    const int g = (int)(i % 8);
    const size_t mh = i / 8;
    const int h = (int)(mh % heads);
    const int m = (int)(mh / heads);
    int p = pos[m];
    if (p < 0 || p >= max_pos) {
      atomicOr(status, kDevBadPosition);
      p = 0;
    }
    const float *c = cs + (size_t)p * 128 + g * 8;
    const float *s = c + 64;
    const size_t o = (size_t)m * ncols + h * 128 + g * 8;
    const size_t oo = (size_t)m * out_ld + h * 128 + g * 8;
    const uint4 ua = *reinterpret_cast<const uint4 *>(dy + o);
    const uint4 ub = *reinterpret_cast<const uint4 *>(dy + o + 64);
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
    *reinterpret_cast<uint4 *>(out + oo) = make_uint4(oa[0], oa[1], oa[2], oa[3]);
    *reinterpret_cast<uint4 *>(out + oo + 64) = make_uint4(ob[0], ob[1], ob[2], ob[3]);
  }
}

cudaError_t launch_rope_bwd(const __nv_bfloat16 *dy, __nv_bfloat16 *out, int M, int ncols,
                            int out_ld, const int32_t *pos, const float *cos_sin, int max_pos,
                            uint32_t *status, cudaStream_t st) {
  const size_t total = (size_t)M * (ncols / 128) * 8;
  const int grid = grid_for(total, 256, 148 * 16);
  rope_bwd_kernel<<<grid, 256, 0, st>>>(dy, out, M, ncols, out_ld, pos, cos_sin, max_pos, status);
  note_launch();
  return cudaGetLastError();
}

// ------------------------------------------ block-diagonal pair of B factors
// Two projections sharing x taken as one projection of rank 2r:
// B = diag(B1, B2) with B1 [n1, r], B2 [n2, r].  transpose == 0 writes
// B [n1+n2, 2r]; transpose == 1 writes Bᵀ [2r, n1+n2].
__global__ void blockdiag_rank_kernel(const __nv_bfloat16 *__restrict__ B1,
                                      const __nv_bfloat16 *__restrict__ B2,
                                      __nv_bfloat16 *__restrict__ out, int n1, int n2, int r,
                                      int transpose) {
  const int n = n1 + n2, r2 = 2 * r;
  const size_t total = (size_t)n * r2;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x) {
    int o, j;
    if (transpose) {
      j = (int)(i / n);
      o = (int)(i % n);
    } else {
      o = (int)(i / r2);
      j = (int)(i % r2);
    }
    __nv_bfloat16 v = __float2bfloat16_rn(0.0f);
    if (o < n1 && j < r) v = B1[(size_t)o * r + j];
    else if (o >= n1 && j >= r) v = B2[(size_t)(o - n1) * r + (j - r)];
    out[i] = v;
  }
}

cudaError_t launch_blockdiag_rank(const __nv_bfloat16 *B1, const __nv_bfloat16 *B2,
                                  __nv_bfloat16 *out, int n1, int n2, int r, bool transpose,
                                  cudaStream_t st) {
  const size_t total = (size_t)(n1 + n2) * 2 * r;
  blockdiag_rank_kernel<<<grid_for(total, 256, 4096), 256, 0, st>>>(B1, B2, out, n1, n2, r,
                                                                    transpose ? 1 : 0);
  note_launch();
  return cudaGetLastError();
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
  const int grid = grid_for(total, 256, 148 * 16);
  rope_cache_kernel<<<grid, 256, 0, st>>>(cos_sin, max_pos, head_dim, theta);
  note_launch();
  return cudaGetLastError();
}

// ------------------------------------------------------------ NF4 dequant
// The 16 NormalFloat4 levels (QLoRA, Dettmers et al. 2023, appendix table).
__constant__ float kNf4LevelsMisc[16] = {
    -1.0f, -0.6961928009986877f, -0.5250730514526367f, -0.39491748809814453f,
    -0.28444138169288635f, -0.18477343022823334f, -0.09105003625154495f, 0.0f,
    0.07958029955625534f, 0.16093020141124725f, 0.24611230194568634f, 0.33791524171829224f,
    0.44070982933044434f, 0.5626170039176941f, 0.7229568362236023f, 1.0f};

// One thread per 16 code bytes (32 elements; half of a 64-element block).
// HBM-bound: reads n·k/2 + n·k/32 bytes, writes 2·n·k bytes.
__global__ void __launch_bounds__(256) nf4_dequant_kernel(const uint8_t *__restrict__ codes,
                                                          const __nv_bfloat16 *__restrict__ absmax,
                                                          __nv_bfloat16 *__restrict__ w,
                                                          size_t n_chunks) {
  __shared__ float lv[16];
  if (threadIdx.x < 16) lv[threadIdx.x] = kNf4LevelsMisc[threadIdx.x];
  __syncthreads();
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n_chunks;
       i += (size_t)gridDim.x * blockDim.x) {
    const uint4 c = __ldg(reinterpret_cast<const uint4 *>(codes) + i);
    const float a = __bfloat162float(absmax[i >> 1]);
    const uint32_t words[4] = {c.x, c.y, c.z, c.w};
    uint4 *dst = reinterpret_cast<uint4 *>(w) + 4 * i;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t o[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const uint32_t byte = (words[q] >> (8 * b)) & 0xFFu;
        o[b] = pack_bf16x2(lv[byte >> 4] * a, lv[byte & 0xFu] * a);
      }
      dst[q] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

cudaError_t launch_nf4_dequant(const uint8_t *codes, const __nv_bfloat16 *absmax,
                               __nv_bfloat16 *w, int n, int k, cudaStream_t st) {
  const size_t chunks = (size_t)n * k / 32;
  const int grid = grid_for(chunks, 256, 148 * 8);
  nf4_dequant_kernel<<<grid, 256, 0, st>>>(codes, absmax, w, chunks);
  note_launch();
  return cudaGetLastError();
}

// ----------------------------------------------------------- NF4 quantise
// One thread per 64-element block: absmax = max|w| (exact in bf16 because
// the inputs are bf16), code = first index minimising |w/absmax - level|
// in IEEE fp32; all-zero blocks get code 7.
__global__ void nf4_quantize_kernel(const __nv_bfloat16 *__restrict__ w, uint8_t *__restrict__ codes,
                                    __nv_bfloat16 *__restrict__ absmax, size_t n_blocks) {
  __shared__ float lv[16];
  if (threadIdx.x < 16) lv[threadIdx.x] = kNf4LevelsMisc[threadIdx.x];
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
  const int grid = grid_for(blocks, 128, 148 * 8);
  nf4_quantize_kernel<<<grid, 128, 0, st>>>(w, codes, absmax, blocks);
  note_launch();
  return cudaGetLastError();
}

}  // namespace lora
