// tcgen05 tensor-core path of the A-MiX x W-MX matmul (placeholder until the
// kernel lands) and the per-device error word used by bounded waits.
#include <cuda_runtime.h>

#include "mix_internal.h"

namespace mixk {

__device__ unsigned g_mix_device_error;

cudaError_t read_device_error(unsigned* word, bool clear) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbol(word, g_mix_device_error, sizeof(unsigned));
  if (e != cudaSuccess) return e;
  if (clear) {
    const unsigned z = 0;
    e = cudaMemcpyToSymbol(g_mix_device_error, &z, sizeof(unsigned));
  }
  return e;
}

cudaError_t launch_gemm_tc(const mix_gemm_desc_t& d, cudaStream_t st, mix_status_t* why) {
  (void)d; (void)st;
  *why = MIX_ERR_UNSUPPORTED;
  return cudaSuccess;
}

}  // namespace mixk
