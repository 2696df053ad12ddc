// Host-side launchers shared between the library's translation units.  The
// C ABI (include/mix.h) validates arguments and then calls these.
#pragma once
#include <cuda_runtime.h>
#include <cstdint>

#include "../../include/mix.h"

namespace mixk {

int num_sms();

cudaError_t launch_mix_quantize(const void* x, bool bf16, int64_t rows, int64_t k, int64_t ld,
                                int type, int ebias, bool asym, uint8_t* codes, void* shared,
                                cudaStream_t st);
cudaError_t launch_mx_quantize_rows(const void* x, bool bf16, int64_t rows, int64_t k, int64_t ld,
                                    bool fp4, bool floor_rule, uint8_t* codes, uint8_t* scales,
                                    cudaStream_t st);
cudaError_t launch_mx_quantize_cols(const void* x, bool bf16, int64_t kdim, int64_t n, int64_t ld,
                                    bool fp4, bool floor_rule, uint8_t* codes, uint8_t* scales,
                                    cudaStream_t st);
cudaError_t launch_mix_dequantize(const uint8_t* codes, const void* shared, int64_t rows, int64_t k,
                                  int type, int ebias, float* out, cudaStream_t st);
cudaError_t launch_mx_dequantize(const uint8_t* codes, const uint8_t* scales, int64_t rows, int64_t k,
                                 bool fp4, float* out, cudaStream_t st);

// GEMM paths.  Descriptor already validated.
size_t gemv_workspace_bytes(const mix_gemm_desc_t& d);
cudaError_t launch_gemv_shiftadd(const mix_gemm_desc_t& d, void* ws, cudaStream_t st);
cudaError_t launch_gemm_tc(const mix_gemm_desc_t& d, cudaStream_t st, mix_status_t* why);

// K-smoothing.
size_t ksmooth_ws_bytes(int64_t tokens, int heads, int head_dim);
cudaError_t launch_ksmooth(const void* k, bool bf16, int64_t tokens, int heads, int head_dim,
                           int64_t ld, float* mean, int mode, float* k_out, void* ws,
                           cudaStream_t st);

// K-smoothing with the library's built-in scratch (no caller workspace).
size_t ksmooth_noalloc_scratch_bytes();
cudaError_t launch_ksmooth_noalloc(const void* k, bool bf16, int64_t tokens, int heads, int head_dim,
                                   int64_t ld, float* mean, int mode, float* k_out, cudaStream_t st);

// Device error word (bounded waits).
cudaError_t read_device_error(unsigned* word, bool clear);

}  // namespace mixk
