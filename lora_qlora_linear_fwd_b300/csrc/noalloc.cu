// lora_linear_bwd_noalloc: the fused backward of lora_linear_bwd for callers
// that cannot allocate device memory at the point of the call.
//
// Some callers cannot call cudaMalloc (or any allocating routine) when they
// run the backward: a plugin executed inside another framework's runtime
// that is handed only its tensors, or a latency-critical training loop that
// must never enter the driver's allocator (which can synchronise the device
// and stall every stream).  This entry point takes the same inputs and
// outputs as lora_linear_bwd but no workspace: its scratch (the transposed B,
// the 16-bit hi/lo parts of uᵀ and vᵀ, the rank-pass flags and parked
// partials, and the device status word) lives in one fixed array in the
// library's own device memory, declared below.
//
// Properties a caller must know:
//   * The array holds kNoAllocScratchBytes (32 MiB) on every GPU that loads
//     this library, from module load until the process exits.
//   * Shapes whose scratch need (lora_workspace_size(LORA_OP_BWD, ...), with
//     LORA_OP_FLAG_DQ for double-quantised NF4 scales)
//     exceeds that size are rejected with LORA_ERR_WORKSPACE before anything
//     is launched.
//   * The first call on each device looks up the array's device address
//     (cudaGetSymbolAddress, with that device current) and caches it; make
//     that first call before any stream capture.
//   * Every call uses the same array, which keeps the previous call's
//     contents: each call zeroes the status word; the rank-pass flags
//     carry a per-launch epoch (stale ones never match), and everything
//     else is fully written before it is read.
//     Two calls that overlap on the GPU (e.g. on two streams of one device)
//     race on the array and give wrong results; serialise them.
//   * Device-side failures (a pipeline wait past its time limit) are
//     recorded in the array's status word, which this entry point does not
//     report; use lora_linear_bwd with a workspace to observe them.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "kernels.h"
#include "lora_b300.h"

namespace {

constexpr size_t kNoAllocScratchBytes = 32ull << 20;

// Scratch of lora_linear_bwd_noalloc (one copy per device).  In host code
// this name is only a handle for cudaGetSymbolAddress, never an address.
static __device__ __align__(256) unsigned char g_bwd_scratch[kNoAllocScratchBytes];

// Device address of g_bwd_scratch on the current device, looked up once per
// device.  Returns nullptr (and sets *err) if the lookup fails.
void *scratch_address(cudaError_t *err) {
  static std::mutex mu;
  static void *addr[lora::kMaxDevices] = {};
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= lora::kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void *p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_bwd_scratch);
    if (*err != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace

extern "C" lora_status_t lora_linear_bwd_noalloc(const void *x, lora_weight_t W, const void *A,
                                                 const void *B, const void *dy, void *dx,
                                                 int accumulate_dx, float *dA, float *dB, int M,
                                                 int k, int n, int r, float alpha,
                                                 lora_stream_t stream) {
  // every check lora_linear_bwd makes comes first, so a call it would
  // reject enqueues nothing (not even the status-word reset below)
  lora_status_t s = lora::check_bwd_args(x, W, A, B, dy, dx, dA, dB, M, k, n, r, alpha);
  if (s != LORA_OK) return s;
  const int dq = (W.type == LORA_WEIGHT_NF4 && W.absmax_scale) ? LORA_OP_FLAG_DQ : 0;
  const size_t need = lora_workspace_size(LORA_OP_BWD | dq, M, k, n, r);
  if (need == 0) return LORA_ERR_INVALID_ARG;
  if (need > kNoAllocScratchBytes) return LORA_ERR_WORKSPACE;
  if ((s = lora::check_current_device()) != LORA_OK) return s;
  cudaError_t err = cudaSuccess;
  void *scratch = scratch_address(&err);
  if (!scratch) return LORA_ERR_CUDA;
  // the status word starts each call at zero
  if (cudaMemsetAsync(scratch, 0, 256, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return LORA_ERR_CUDA;
  return lora_linear_bwd(x, W, A, B, dy, dx, accumulate_dx, dA, dB, M, k, n, r, alpha, scratch,
                         kNoAllocScratchBytes, stream);
}
