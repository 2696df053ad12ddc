// C ABI of libmix.so (include/mix.h): host-side validation, then one or more
// launches on the caller's stream.  Nothing here allocates device memory.
#include <cuda_runtime.h>

#include <cstdint>

#include "mix_internal.h"

using namespace mixk;

namespace {

constexpr int kVersion = 10301;  // 1.3.1

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

mix_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? MIX_OK : MIX_ERR_CUDA; }

bool valid_dtype(mix_dtype_t d) { return d == MIX_DT_F32 || d == MIX_DT_BF16; }
int esize(mix_dtype_t d) { return d == MIX_DT_F32 ? 4 : 2; }

// A packed plane addressed by element offsets: codes at offset/2 bytes,
// shared (or scales) at offset/32 entries.  Strides must keep every row on a
// 16-byte codes boundary.
bool plane_strides_ok(int64_t ld, int64_t bs, int64_t k) {
  return ld >= k && ld % 32 == 0 && bs % 32 == 0 && bs >= 0;
}

// The element-wise kernels number their work items (blocks, 16-byte vectors,
// 8-element groups) with 32 bits: rows * per_row must stay below 2^32 - 1.
bool items_fit(int64_t rows, int64_t per_row) {
  return per_row <= 0 || rows <= (int64_t)(UINT32_MAX - 1u) / per_row;
}

}  // namespace

extern "C" {

size_t mix_codes_bytes(int64_t rows, int64_t k) {
  if (rows < 0 || k < 0 || k % 32 != 0) return 0;
  return (size_t)rows * (size_t)(k / 2);
}

size_t mix_shared_bytes(mix_type_t type, int64_t rows, int64_t k) {
  if (rows < 0 || k < 0 || k % 32 != 0 || (type != MIX_T1_4P25 && type != MIX_T2_4P5)) return 0;
  return (size_t)rows * (size_t)(k / 32) * (type == MIX_T1_4P25 ? 1u : 2u);
}

size_t mx_scales_bytes(int64_t rows, int64_t k) {
  if (rows < 0 || k < 0 || k % 32 != 0) return 0;
  return (size_t)rows * (size_t)(k / 32);
}

const char* mix_status_str(mix_status_t s) {
  switch (s) {
    case MIX_OK: return "ok";
    case MIX_ERR_INVALID_ARG: return "invalid argument";
    case MIX_ERR_SHAPE: return "unsupported shape (K and quantised N must be multiples of 32)";
    case MIX_ERR_ALIGN: return "misaligned pointer or stride";
    case MIX_ERR_UNSUPPORTED: return "unsupported combination";
    case MIX_ERR_CUDA: return "CUDA error";
    case MIX_ERR_WORKSPACE: return "workspace missing or too small";
    case MIX_ERR_DEVICE: return "a kernel wait ran out (device error word set)";
  }
  return "unknown status";
}

int mix_version(void) { return kVersion; }

mix_status_t mix_selftest_wait_timeout(void* workspace, size_t workspace_bytes, mix_stream_t stream) {
  if (workspace == nullptr || workspace_bytes < MIX_SELFTEST_WORKSPACE_BYTES) return MIX_ERR_WORKSPACE;
  if (!aligned(workspace, 16)) return MIX_ERR_ALIGN;
  if (selftest_ws_bytes() > MIX_SELFTEST_WORKSPACE_BYTES) return MIX_ERR_UNSUPPORTED;
  return from_cuda(launch_selftest_wait_timeout(workspace, 1LL << 20, reinterpret_cast<cudaStream_t>(stream)));
}

mix_status_t mix_device_error(unsigned* word, int clear) {
  if (word == nullptr) return MIX_ERR_INVALID_ARG;
  return from_cuda(read_device_error(word, clear != 0));
}

mix_status_t mix_quantize(const void* x, mix_dtype_t dtype, int64_t rows, int64_t k, int64_t ld,
                          mix_type_t type, int ebias, unsigned flags, uint8_t* codes, void* shared,
                          mix_stream_t stream) {
  if (!valid_dtype(dtype) || (type != MIX_T1_4P25 && type != MIX_T2_4P5)) return MIX_ERR_INVALID_ARG;
  if (rows < 0 || k < 0 || ld < k || ebias < -100 || ebias > 100 || (flags & ~1u)) return MIX_ERR_INVALID_ARG;
  if (k % 32 != 0) return MIX_ERR_SHAPE;
  if (rows == 0 || k == 0) return MIX_OK;
  if (x == nullptr || codes == nullptr || shared == nullptr) return MIX_ERR_INVALID_ARG;
  if (!aligned(x, 16) || (ld * esize(dtype)) % 16 != 0 || !aligned(codes, 16) ||
      !aligned(shared, type == MIX_T1_4P25 ? 1 : 2))
    return MIX_ERR_ALIGN;
  if (!items_fit(rows, k / 32)) return MIX_ERR_UNSUPPORTED;
  return from_cuda(launch_mix_quantize(x, dtype == MIX_DT_BF16, rows, k, ld, (int)type, ebias,
                                       (flags & MIX_ASYM_ZERO) != 0, codes, shared,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

mix_status_t mix_auto_ebias(const void* x, mix_dtype_t dtype, int64_t rows, int64_t k, int64_t ld, int* ebias,
                            mix_stream_t stream) {
  if (!valid_dtype(dtype) || rows < 0 || k < 0 || ld < k || ebias == nullptr) return MIX_ERR_INVALID_ARG;
  if (k % 32 != 0) return MIX_ERR_SHAPE;
  if (!aligned(ebias, 4)) return MIX_ERR_ALIGN;
  if (rows > 0 && k > 0) {
    if (x == nullptr) return MIX_ERR_INVALID_ARG;
    if (!aligned(x, 16) || (ld * esize(dtype)) % 16 != 0) return MIX_ERR_ALIGN;
    if (!items_fit(rows, k * esize(dtype) / 16)) return MIX_ERR_UNSUPPORTED;
  }
  return from_cuda(launch_auto_ebias(x, dtype == MIX_DT_BF16, rows, k, ld, ebias,
                                     reinterpret_cast<cudaStream_t>(stream)));
}

mix_status_t mix_quantize_auto(const void* x, mix_dtype_t dtype, int64_t rows, int64_t k, int64_t ld,
                               mix_type_t type, unsigned flags, uint8_t* codes, void* shared, int* ebias,
                               mix_stream_t stream) {
  if (!valid_dtype(dtype) || (type != MIX_T1_4P25 && type != MIX_T2_4P5)) return MIX_ERR_INVALID_ARG;
  if (rows < 0 || k < 0 || ld < k || (flags & ~1u) || ebias == nullptr) return MIX_ERR_INVALID_ARG;
  if (k % 32 != 0) return MIX_ERR_SHAPE;
  if (!aligned(ebias, 4)) return MIX_ERR_ALIGN;
  const bool empty = rows == 0 || k == 0;
  if (!empty) {
    if (x == nullptr || codes == nullptr || shared == nullptr) return MIX_ERR_INVALID_ARG;
    if (!aligned(x, 16) || (ld * esize(dtype)) % 16 != 0 || !aligned(codes, 16) ||
        !aligned(shared, type == MIX_T1_4P25 ? 1 : 2))
      return MIX_ERR_ALIGN;
    if (!items_fit(rows, k / 32) || !items_fit(rows, k * esize(dtype) / 16)) return MIX_ERR_UNSUPPORTED;
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = launch_auto_ebias(x, dtype == MIX_DT_BF16, rows, k, ld, ebias, st);
  if (e != cudaSuccess || empty) return from_cuda(e);
  return from_cuda(launch_mix_quantize(x, dtype == MIX_DT_BF16, rows, k, ld, (int)type, 0,
                                       (flags & MIX_ASYM_ZERO) != 0, codes, shared, st, ebias));
}

mix_status_t mx_quantize(const void* x, mix_dtype_t dtype, int64_t rows, int64_t cols, int64_t ld,
                         int axis, mx_type_t type, unsigned flags, uint8_t* codes, uint8_t* scales,
                         mix_stream_t stream) {
  if (!valid_dtype(dtype) || (type != MX_INT4 && type != MX_FP4_E2M1) || (axis != 0 && axis != 1))
    return MIX_ERR_INVALID_ARG;
  if (rows < 0 || cols < 0 || ld < cols || (flags & ~14u) || (flags & 6u) == 6u) return MIX_ERR_INVALID_ARG;
  const int64_t K = axis ? cols : rows, N = axis ? rows : cols;
  if (K % 32 != 0) return MIX_ERR_SHAPE;
  if (N == 0 || K == 0) return MIX_OK;
  if (x == nullptr || codes == nullptr || scales == nullptr) return MIX_ERR_INVALID_ARG;
  if (!aligned(x, 16) || (ld * esize(dtype)) % 16 != 0 || !aligned(codes, 16)) return MIX_ERR_ALIGN;
  if (axis == 1 && !items_fit(N, K / 32)) return MIX_ERR_UNSUPPORTED;
  const bool fp4 = type == MX_FP4_E2M1, g16 = (flags & MX_BLOCK16) != 0;
  const int fl = mx_rule_of(flags);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (axis == 1)
    return from_cuda(launch_mx_quantize_rows(x, dtype == MIX_DT_BF16, N, K, ld, fp4, fl, g16, codes, scales, st));
  return from_cuda(launch_mx_quantize_cols(x, dtype == MIX_DT_BF16, K, N, ld, fp4, fl, g16, codes, scales, st));
}

mix_status_t nvfp4_quantize(const void* x, mix_dtype_t dtype, int64_t rows, int64_t k, int64_t ld,
                            uint8_t* codes, uint8_t* scales, float* tensor_scale, mix_stream_t stream) {
  if (!valid_dtype(dtype) || rows < 0 || k < 0 || ld < k || tensor_scale == nullptr) return MIX_ERR_INVALID_ARG;
  if (k % 16 != 0) return MIX_ERR_SHAPE;
  if (!aligned(tensor_scale, 4)) return MIX_ERR_ALIGN;
  if (rows > 0 && k > 0) {
    if (x == nullptr || codes == nullptr || scales == nullptr) return MIX_ERR_INVALID_ARG;
    if (!aligned(x, 16) || (ld * esize(dtype)) % 16 != 0 || !aligned(codes, 8)) return MIX_ERR_ALIGN;
    if (!items_fit(rows, k / 16) || !items_fit(rows, k * esize(dtype) / 16)) return MIX_ERR_UNSUPPORTED;
  }
  return from_cuda(launch_nvfp4_quantize(x, dtype == MIX_DT_BF16, rows, k, ld, codes, scales, tensor_scale,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

mix_status_t mix_underflow_count(const void* x, mix_dtype_t dtype, int64_t rows, int64_t k, int64_t ld,
                                 const uint8_t* codes, mix_underflow_fmt_t fmt, unsigned long long* count,
                                 mix_stream_t stream) {
  if (!valid_dtype(dtype) || rows < 0 || k < 0 || ld < k || count == nullptr) return MIX_ERR_INVALID_ARG;
  if (fmt != MIX_UF_MIX && fmt != MIX_UF_MXINT4 && fmt != MIX_UF_E2M1) return MIX_ERR_INVALID_ARG;
  if (k % 16 != 0) return MIX_ERR_SHAPE;
  if (!aligned(count, 8)) return MIX_ERR_ALIGN;
  if (rows > 0 && k > 0) {
    if (x == nullptr || codes == nullptr) return MIX_ERR_INVALID_ARG;
    if (!aligned(x, 16) || (ld * esize(dtype)) % 16 != 0 || !aligned(codes, 4)) return MIX_ERR_ALIGN;
    if (!items_fit(rows, k / 8)) return MIX_ERR_UNSUPPORTED;
  }
  return from_cuda(launch_underflow_count(x, dtype == MIX_DT_BF16, rows, k, ld, codes, (int)fmt, count,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

mix_status_t mix_clamp_count(const void* x, mix_dtype_t dtype, int64_t rows, int64_t k, int64_t ld, int ebias,
                             unsigned long long* counts, mix_stream_t stream) {
  if (!valid_dtype(dtype) || rows < 0 || k < 0 || ld < k || counts == nullptr || ebias < -100 || ebias > 100)
    return MIX_ERR_INVALID_ARG;
  if (k % 32 != 0) return MIX_ERR_SHAPE;
  if (!aligned(counts, 8)) return MIX_ERR_ALIGN;
  if (rows > 0 && k > 0) {
    if (x == nullptr) return MIX_ERR_INVALID_ARG;
    if (!aligned(x, 16) || (ld * esize(dtype)) % 16 != 0) return MIX_ERR_ALIGN;
    if (!items_fit(rows, k / 32)) return MIX_ERR_UNSUPPORTED;
  }
  return from_cuda(launch_clamp_count(x, dtype == MIX_DT_BF16, rows, k, ld, ebias, counts,
                                      reinterpret_cast<cudaStream_t>(stream)));
}

static mix_status_t validate_attn(const mix_decode_attn_desc_t* d) {
  if (d == nullptr) return MIX_ERR_INVALID_ARG;
  if (d->tokens < 1 || d->q_heads < 1 || d->kv_heads < 1 || d->q_heads % d->kv_heads != 0 ||
      d->q_heads / d->kv_heads > 8 || !valid_dtype(d->dtype))
    return MIX_ERR_INVALID_ARG;
  if (d->head_dim != 128 || d->v_ld % 32 != 0 || d->v_ld < d->tokens) return MIX_ERR_SHAPE;
  if (d->q_ebias < -100 || d->q_ebias > 100 || d->p_ebias < -100 || d->p_ebias > 100) return MIX_ERR_INVALID_ARG;
  if (d->q == nullptr || d->k_codes == nullptr || d->k_scales == nullptr || d->v_codes == nullptr ||
      d->v_scales == nullptr || d->out == nullptr || (d->k_new != nullptr && d->k_mean == nullptr) ||
      ((d->p_codes == nullptr) != (d->p_shared == nullptr)))
    return MIX_ERR_INVALID_ARG;
  if (!aligned(d->k_codes, 16) || !aligned(d->k_scales, 4) || !aligned(d->v_codes, 16) ||
      (d->p_codes != nullptr && (!aligned(d->p_codes, 16) || !aligned(d->p_shared, 2))) ||
      (d->p_values != nullptr && !aligned(d->p_values, 4)))
    return MIX_ERR_ALIGN;
  if (d->tokens >= (int64_t)1 << 40) return MIX_ERR_SHAPE;
  return MIX_OK;
}

size_t mix_decode_attention_workspace_bytes(const mix_decode_attn_desc_t* d) {
  if (validate_attn(d) != MIX_OK) return 0;
  return decode_attention_ws_bytes(*d);
}

mix_status_t mix_decode_attention(const mix_decode_attn_desc_t* d, void* workspace, size_t workspace_bytes,
                                  mix_stream_t stream) {
  const mix_status_t s = validate_attn(d);
  if (s != MIX_OK) return s;
  if (workspace == nullptr || workspace_bytes < decode_attention_ws_bytes(*d)) return MIX_ERR_WORKSPACE;
  return from_cuda(launch_decode_attention(*d, workspace, reinterpret_cast<cudaStream_t>(stream)));
}

mix_status_t mix_dequantize(const uint8_t* codes, const void* shared, int64_t rows, int64_t k,
                            mix_type_t type, int ebias, float* out, mix_stream_t stream) {
  if ((type != MIX_T1_4P25 && type != MIX_T2_4P5) || rows < 0 || k < 0 || ebias < -100 || ebias > 100)
    return MIX_ERR_INVALID_ARG;
  if (k % 32 != 0) return MIX_ERR_SHAPE;
  if (rows == 0 || k == 0) return MIX_OK;
  if (codes == nullptr || shared == nullptr || out == nullptr) return MIX_ERR_INVALID_ARG;
  if (!aligned(codes, 16) || !aligned(out, 16) || !aligned(shared, type == MIX_T1_4P25 ? 1 : 2))
    return MIX_ERR_ALIGN;
  return from_cuda(launch_mix_dequantize(codes, shared, rows, k, (int)type, ebias, out,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

mix_status_t mx_dequantize(const uint8_t* codes, const uint8_t* scales, int64_t rows, int64_t k,
                           mx_type_t type, float* out, mix_stream_t stream) {
  if ((type != MX_INT4 && type != MX_FP4_E2M1) || rows < 0 || k < 0) return MIX_ERR_INVALID_ARG;
  if (k % 32 != 0) return MIX_ERR_SHAPE;
  if (rows == 0 || k == 0) return MIX_OK;
  if (codes == nullptr || scales == nullptr || out == nullptr) return MIX_ERR_INVALID_ARG;
  if (!aligned(codes, 16) || !aligned(out, 16)) return MIX_ERR_ALIGN;
  return from_cuda(launch_mx_dequantize(codes, scales, rows, k, type == MX_FP4_E2M1, out,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

static mix_status_t validate_gemm(const mix_gemm_desc_t* d) {
  if (d == nullptr) return MIX_ERR_INVALID_ARG;
  if (d->M < 0 || d->N < 0 || d->K < 0 || d->batch < 1 || d->b_group < 1) return MIX_ERR_INVALID_ARG;
  if (d->a_type != MIX_T1_4P25 && d->a_type != MIX_T2_4P5) return MIX_ERR_INVALID_ARG;
  if (d->b_type != MX_INT4 && d->b_type != MX_FP4_E2M1) return MIX_ERR_INVALID_ARG;
  if (d->b_block != 0 && d->b_block != 16 && d->b_block != 32) return MIX_ERR_INVALID_ARG;
  if (d->a_ebias < -100 || d->a_ebias > 100 || d->epi_ebias < -100 || d->epi_ebias > 100)
    return MIX_ERR_INVALID_ARG;
  if (d->epi < MIX_EPI_NONE || d->epi > MIX_EPI_MXFP4) return MIX_ERR_INVALID_ARG;
  if ((d->epi_flags & ~7u) || (d->epi_flags & 6u) == 6u) return MIX_ERR_INVALID_ARG;
  if (d->algo < MIX_GEMM_AUTO || d->algo > MIX_GEMM_TCGEN05_FUSED) return MIX_ERR_INVALID_ARG;
  if (d->b_prepared != nullptr && !aligned(d->b_prepared, 16)) return MIX_ERR_ALIGN;
  if (d->a_causal != 0 && d->a_causal != 1) return MIX_ERR_INVALID_ARG;
  if (d->a_causal && (d->a_causal_shift <= -(int64_t)INT32_MAX || d->a_causal_shift >= (int64_t)INT32_MAX))
    return MIX_ERR_INVALID_ARG;
  if (d->K % 32 != 0) return MIX_ERR_SHAPE;
  if (d->epi != MIX_EPI_NONE && d->N % 32 != 0) return MIX_ERR_SHAPE;
  if (d->epi == MIX_EPI_NONE && d->c == nullptr) return MIX_ERR_INVALID_ARG;
  if (d->M == 0 || d->N == 0) return MIX_OK;
  if (d->K > 0) {
    if (d->a_codes == nullptr || d->a_shared == nullptr || d->b_codes == nullptr || d->b_scales == nullptr)
      return MIX_ERR_INVALID_ARG;
    if (!plane_strides_ok(d->a_ld, d->a_batch_stride, d->K) || !plane_strides_ok(d->b_ld, d->b_batch_stride, d->K))
      return MIX_ERR_ALIGN;
    if (!aligned(d->a_codes, 16) || !aligned(d->b_codes, 16) ||
        !aligned(d->a_shared, d->a_type == MIX_T1_4P25 ? 1 : 2))
      return MIX_ERR_ALIGN;
  }
  if (d->c != nullptr) {
    if (d->ldc < d->N || d->c_batch_stride < 0 || !aligned(d->c, 16) || d->ldc % 4 != 0 || d->c_batch_stride % 4 != 0)
      return MIX_ERR_ALIGN;
  }
  if (d->epi != MIX_EPI_NONE) {
    if (d->out_codes == nullptr || d->out_shared == nullptr) return MIX_ERR_INVALID_ARG;
    if (!plane_strides_ok(d->out_ld, d->out_batch_stride, d->N) || !aligned(d->out_codes, 16) ||
        !aligned(d->out_shared, d->epi == MIX_EPI_MIX_T2 ? 2 : 1))
      return MIX_ERR_ALIGN;
  }
  return MIX_OK;
}

static bool use_shiftadd(const mix_gemm_desc_t* d) {
  if (d->algo == MIX_GEMM_SHIFTADD) return true;
  if (d->algo != MIX_GEMM_AUTO) return false;
  return d->M <= 16;
}

size_t mix_mx_gemm_workspace_bytes(const mix_gemm_desc_t* d) {
  if (validate_gemm(d) != MIX_OK || d->M == 0 || d->N == 0) return 0;
  if (use_shiftadd(d)) return gemv_workspace_bytes(*d);
  return gemm_tc_workspace_bytes(*d);
}

size_t mix_mx_gemm_prepare_b_bytes(const mix_gemm_desc_t* d) {
  if (validate_gemm(d) != MIX_OK || d->M == 0 || d->N == 0 || d->K == 0 || use_shiftadd(d)) return 0;
  return gemm_tc_prepare_b_bytes(*d);
}

mix_status_t mix_mx_gemm_prepare_b(const mix_gemm_desc_t* d, void* prepared, size_t prepared_bytes,
                                   mix_stream_t stream) {
  mix_status_t s = validate_gemm(d);
  if (s != MIX_OK) return s;
  const size_t need = mix_mx_gemm_prepare_b_bytes(d);
  if (need == 0) return MIX_ERR_UNSUPPORTED;
  if (prepared == nullptr || prepared_bytes < need) return MIX_ERR_WORKSPACE;
  if (!aligned(prepared, 16)) return MIX_ERR_ALIGN;
  return from_cuda(launch_gemm_tc_prepare_b(*d, prepared, reinterpret_cast<cudaStream_t>(stream)));
}

mix_status_t mix_mx_gemm(const mix_gemm_desc_t* d, void* workspace, size_t workspace_bytes,
                         mix_stream_t stream) {
  mix_status_t s = validate_gemm(d);
  if (s != MIX_OK || d->M == 0 || d->N == 0) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (use_shiftadd(d)) {
    if (d->M > 16) return MIX_ERR_UNSUPPORTED;
    if (d->epi != MIX_EPI_NONE) {
      // the shift-add path quantises dense fp32 rows into dense planes
      if (d->out_ld != d->N || d->out_batch_stride != d->M * d->N) return MIX_ERR_UNSUPPORTED;
      if (d->c != nullptr && (d->ldc % 4 != 0)) return MIX_ERR_UNSUPPORTED;
    }
    const size_t need = gemv_workspace_bytes(*d);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return MIX_ERR_WORKSPACE;
    if (d->K == 0) return MIX_ERR_UNSUPPORTED;
    return from_cuda(launch_gemv_shiftadd(*d, workspace, st));
  }
  mix_status_t why = MIX_OK;
  if (workspace != nullptr && !aligned(workspace, 16)) return MIX_ERR_ALIGN;
  cudaError_t e = launch_gemm_tc(*d, workspace, workspace_bytes, st, &why);
  if (why != MIX_OK) return why;
  return from_cuda(e);
}

size_t ksmooth_workspace_bytes(int64_t tokens, int heads, int head_dim) {
  if (tokens <= 0 || heads <= 0 || head_dim <= 0) return 0;
  return ksmooth_ws_bytes(tokens, heads, head_dim);
}

mix_status_t ksmooth_kv(const void* k, mix_dtype_t dtype, int64_t tokens, int heads, int head_dim,
                        int64_t ld, float* mean, int mode, float* k_out, void* workspace,
                        size_t workspace_bytes, mix_stream_t stream) {
  if (!valid_dtype(dtype) || tokens < 0 || heads <= 0 || head_dim <= 0) return MIX_ERR_INVALID_ARG;
  if (mode != KSMOOTH_COMPUTE && mode != KSMOOTH_APPLY_FROZEN) return MIX_ERR_INVALID_ARG;
  const int64_t C = (int64_t)heads * head_dim;
  if (ld < C) return MIX_ERR_INVALID_ARG;
  if (C % 8 != 0) return MIX_ERR_SHAPE;
  if (mean == nullptr) return MIX_ERR_INVALID_ARG;
  if (mode == KSMOOTH_COMPUTE && tokens == 0) return MIX_ERR_INVALID_ARG;  // mean of nothing
  if (tokens > 0 && (k == nullptr)) return MIX_ERR_INVALID_ARG;
  if (!aligned(k, 16) || (ld * esize(dtype)) % 16 != 0 || !aligned(mean, 16) || (k_out && !aligned(k_out, 16)))
    return MIX_ERR_ALIGN;
  if (mode == KSMOOTH_COMPUTE) {
    const size_t need = ksmooth_ws_bytes(tokens, heads, head_dim);
    if (workspace == nullptr || workspace_bytes < need) return MIX_ERR_WORKSPACE;
    if (!aligned(workspace, 16)) return MIX_ERR_ALIGN;
  }
  return from_cuda(launch_ksmooth(k, dtype == MIX_DT_BF16, tokens, heads, head_dim, ld, mean, mode, k_out,
                                  workspace, reinterpret_cast<cudaStream_t>(stream)));
}

mix_status_t ksmooth_kv_noalloc(const void* k, mix_dtype_t dtype, int64_t tokens, int heads, int head_dim,
                                int64_t ld, float* mean, int mode, float* k_out, mix_stream_t stream) {
  if (!valid_dtype(dtype) || tokens < 0 || heads <= 0 || head_dim <= 0) return MIX_ERR_INVALID_ARG;
  if (mode != KSMOOTH_COMPUTE && mode != KSMOOTH_APPLY_FROZEN) return MIX_ERR_INVALID_ARG;
  const int64_t C = (int64_t)heads * head_dim;
  if (ld < C) return MIX_ERR_INVALID_ARG;
  if (C % 8 != 0) return MIX_ERR_SHAPE;
  if (mean == nullptr) return MIX_ERR_INVALID_ARG;
  if (mode == KSMOOTH_COMPUTE && tokens == 0) return MIX_ERR_INVALID_ARG;
  if (tokens > 0 && k == nullptr) return MIX_ERR_INVALID_ARG;
  // the built-in scratch holds at most KSMOOTH_NOALLOC_SCRATCH_BYTES of partial sums
  if (mode == KSMOOTH_COMPUTE && ksmooth_ws_bytes(tokens, heads, head_dim) > ksmooth_noalloc_scratch_bytes())
    return MIX_ERR_WORKSPACE;
  if (!aligned(k, 16) || (ld * esize(dtype)) % 16 != 0 || !aligned(mean, 16) || (k_out && !aligned(k_out, 16)))
    return MIX_ERR_ALIGN;
  return from_cuda(launch_ksmooth_noalloc(k, dtype == MIX_DT_BF16, tokens, heads, head_dim, ld, mean, mode,
                                          k_out, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
