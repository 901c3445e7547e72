// The 16 NormalFloat4 levels (QLoRA, Dettmers et al. 2023, appendix table),
// ascending; index 7 is the exact zero.  The one copy of the table that the
// fused GEMM's decode and the standalone dequantise / quantise kernels read.
#pragma once

namespace lora {

static __constant__ float kNf4Levels[16] = {
    -1.0f, -0.6961928009986877f, -0.5250730514526367f, -0.39491748809814453f,
    -0.28444138169288635f, -0.18477343022823334f, -0.09105003625154495f, 0.0f,
    0.07958029955625534f, 0.16093020141124725f, 0.24611230194568634f, 0.33791524171829224f,
    0.44070982933044434f, 0.5626170039176941f, 0.7229568362236023f, 1.0f};

}  // namespace lora
