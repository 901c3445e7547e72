// bf16 instantiation of the fused GEMM variants (fp16: gemm_f16.cu).
#define LORA_GEMM_F16 false
#include "gemm_inst.cuh"
