// Entry points of the fused GEMM variants for the 16-bit element type
// LORA_GEMM_F16 (false: bf16, true: fp16); gemm.cu and gemm_f16.cu each
// compile one of them.  The kernel and its dispatch live in gemm_pair.cuh.
#pragma once
#include "gemm_pair.cuh"

namespace lora {

// the other element type is compiled in the other translation unit
extern template cudaError_t launch_gemm_pair_t<!LORA_GEMM_F16>(const GemmParams &, int, bool, bool,
                                                               int, int, int, cudaStream_t);
extern template int gemm_pair_capacity_t<!LORA_GEMM_F16>(int, bool, bool, int, int);

template <bool F16>
cudaError_t launch_gemm_pair_t(const GemmParams &p, int mode, bool rope, bool nf4, int mb, int fv,
                               int pairs, cudaStream_t st) {
  if (mode == kModeFwd)
    return nf4 ? pair_dispatch<kModeFwd, true, F16>(p, rope, mb, fv, pairs, nullptr, st)
               : pair_dispatch<kModeFwd, false, F16>(p, rope, mb, fv, pairs, nullptr, st);
  return nf4 ? pair_dispatch<kModeDx, true, F16>(p, false, mb, fv, pairs, nullptr, st)
             : pair_dispatch<kModeDx, false, F16>(p, false, mb, fv, pairs, nullptr, st);
}

template <bool F16>
int gemm_pair_capacity_t(int mode, bool rope, bool nf4, int mb, int fv) {
  int cap = 0;
  GemmParams dummy;
  if (mode == kModeFwd)
    nf4 ? pair_dispatch<kModeFwd, true, F16>(dummy, rope, mb, fv, 0, &cap, nullptr)
        : pair_dispatch<kModeFwd, false, F16>(dummy, rope, mb, fv, 0, &cap, nullptr);
  else
    nf4 ? pair_dispatch<kModeDx, true, F16>(dummy, false, mb, fv, 0, &cap, nullptr)
        : pair_dispatch<kModeDx, false, F16>(dummy, false, mb, fv, 0, &cap, nullptr);
  return cap;
}

// this translation unit's element type
template cudaError_t launch_gemm_pair_t<LORA_GEMM_F16>(const GemmParams &, int, bool, bool, int,
                                                       int, int, cudaStream_t);
template int gemm_pair_capacity_t<LORA_GEMM_F16>(int, bool, bool, int, int);

}  // namespace lora
