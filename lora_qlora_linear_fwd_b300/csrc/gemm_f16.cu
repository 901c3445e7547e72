// fp16 instantiation of the fused GEMM variants (bf16: gemm.cu).
#define LORA_GEMM_F16 true
#include "gemm_inst.cuh"
