// The 16 NormalFloat4 levels (QLoRA, Dettmers et al. 2023, appendix table),
// ascending; index 7 is the exact zero.  The one copy of the table that the
// fused GEMM's decode and the standalone dequantise / quantise kernels read.
#pragma once

#include <cuda_bf16.h>

#include "ptx.cuh"

namespace lora {

static __constant__ float kNf4Levels[16] = {
    -1.0f, -0.6961928009986877f, -0.5250730514526367f, -0.39491748809814453f,
    -0.28444138169288635f, -0.18477343022823334f, -0.09105003625154495f, 0.0f,
    0.07958029955625534f, 0.16093020141124725f, 0.24611230194568634f, 0.33791524171829224f,
    0.44070982933044434f, 0.5626170039176941f, 0.7229568362236023f, 1.0f};

}  // namespace lora

namespace lora {

// Double quantisation of the block scales (QLoRA, Dettmers et al. 2023, §3
// "Double Quantization"): the first-level constants of 256 consecutive
// blocks (row-major block order) share one fp32 second-level scale, and one
// fp32 offset (the mean of all first-level constants) is subtracted before
// they are quantised to 8-bit floats (E4M3: 1 sign, 4 exponent bits with
// bias 7, 3 mantissa bits; 0x7F / 0xFF are NaN).
constexpr int kDqGroup = 256;
constexpr float kE4m3Max = 448.0f;

// Value of an E4M3 code, from the format's definition (exact in fp32).
LORA_DEV float e4m3_value(uint32_t c) {
  const uint32_t e = (c >> 3) & 15u, m = c & 7u;
  float v;
  if ((c & 0x7Fu) == 0x7Fu)
    v = __uint_as_float(0x7FC00000u);
  else if (e == 0)
    v = (float)m * 0x1p-9f;  // subnormal: m · 2^-9
  else
    v = __uint_as_float(((e + 120u) << 23) | (m << 20));  // (1 + m/8) · 2^(e-7)
  return (c & 0x80u) ? -v : v;
}

// Block scale as the NF4 decode uses it: fp32 product code·scale, then fp32
// sum with the offset, each rounded to nearest, then rounded to bf16 (the
// type a single-level block scale is stored in).  Returned as an fp32 value.
LORA_DEV float dq_absmax(uint32_t code, float scale, float offset) {
  const float a = __fadd_rn(__fmul_rn(e4m3_value(code), scale), offset);
  return __bfloat162float(__float2bfloat16_rn(a));
}

}  // namespace lora
