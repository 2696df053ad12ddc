// Host-side launchers shared between the library's translation units.  The
// C ABI (include/mix.h) validates arguments and then calls these.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "../../include/mix.h"

namespace mixk {

int num_sms();

// MX shared-exponent rules: the paper's ceil (the default), the OCP floor, and
// the tight rule (the smallest exponent at which no element saturates).
enum { MX_RULE_CEIL = 0, MX_RULE_FLOOR = 1, MX_RULE_TIGHT = 2 };
__host__ __device__ inline int mx_rule_of(unsigned flags) {
  return (flags & MX_SCALE_FLOOR) ? MX_RULE_FLOOR : (flags & MX_SCALE_TIGHT) ? MX_RULE_TIGHT : MX_RULE_CEIL;
}

// ebias_dev, when given, overrides ebias with the int it points at (read on
// the device: the automatic two-pass mode).
cudaError_t launch_mix_quantize(const void* x, bool bf16, int64_t rows, int64_t k, int64_t ld,
                                int type, int ebias, bool asym, uint8_t* codes, void* shared,
                                cudaStream_t st, const int* ebias_dev = nullptr);
// NVFP4 comparison quantiser (tensor scale written to *tensor_scale) and the
// dead-zone count (fmt 0 MiX, 1 MXINT4, 2 E2M1).
cudaError_t launch_nvfp4_quantize(const void* x, bool bf16, int64_t rows, int64_t k, int64_t ld, uint8_t* codes,
                                  uint8_t* scales, float* tensor_scale, cudaStream_t st);
cudaError_t launch_underflow_count(const void* x, bool bf16, int64_t rows, int64_t k, int64_t ld, const uint8_t* codes,
                                   int fmt, unsigned long long* count, cudaStream_t st);
// Clamped-block count of the MiX quantiser at ebias (counts[0] high, [1] low).
cudaError_t launch_clamp_count(const void* x, bool bf16, int64_t rows, int64_t k, int64_t ld, int ebias,
                               unsigned long long* counts, cudaStream_t st);
// Automatic ebias into one device int (clear, max-reduction, finish).
cudaError_t launch_auto_ebias(const void* x, bool bf16, int64_t rows, int64_t k, int64_t ld, int* ebias,
                              cudaStream_t st);
cudaError_t launch_mx_quantize_rows(const void* x, bool bf16, int64_t rows, int64_t k, int64_t ld,
                                    bool fp4, int rule, bool g16, uint8_t* codes, uint8_t* scales,
                                    cudaStream_t st);
cudaError_t launch_mx_quantize_cols(const void* x, bool bf16, int64_t kdim, int64_t n, int64_t ld,
                                    bool fp4, int rule, bool g16, uint8_t* codes, uint8_t* scales,
                                    cudaStream_t st);
cudaError_t launch_mix_dequantize(const uint8_t* codes, const void* shared, int64_t rows, int64_t k,
                                  int type, int ebias, float* out, cudaStream_t st);
cudaError_t launch_mx_dequantize(const uint8_t* codes, const uint8_t* scales, int64_t rows, int64_t k,
                                 bool fp4, float* out, cudaStream_t st);

// GEMM paths.  Descriptor already validated.
size_t gemv_workspace_bytes(const mix_gemm_desc_t& d);
cudaError_t launch_gemv_shiftadd(const mix_gemm_desc_t& d, void* ws, cudaStream_t st);
cudaError_t launch_gemm_tc(const mix_gemm_desc_t& d, void* ws, size_t ws_bytes, cudaStream_t st,
                           mix_status_t* why);
size_t gemm_tc_workspace_bytes(const mix_gemm_desc_t& d);
// Prepared B (the tensor-core path's B staging, written once for fixed weights).
size_t gemm_tc_prepare_b_bytes(const mix_gemm_desc_t& d);
cudaError_t launch_gemm_tc_prepare_b(const mix_gemm_desc_t& d, void* prepared, cudaStream_t st);

// Staged tensor-core matmul: the operands are expanded once per call into the
// caller's workspace -- e4m3 planes [batch][rows][k_pad] (k_pad = K rounded up
// to 128, zero padded) and UE8M0 block-scale words grouped per (row tile,
// 128-deep k-step): 128-row tiles for A (512 bytes), kStagedBN-row tiles for
// B stored as 256-row groups (1024 bytes, two 128-row halves, the rows past
// kStagedBN padding).  Inside a 128-row group, 32-bit word
// 4 l + i holds the four k-block scales (byte j = k-block 4 kt + j) of row
// 32 i + l, so one tcgen05.cp of 32 rows x 128 bits puts row 32 i + l at TMEM
// lane l (of every lane quadrant), column i.  MXFP4 weights that the
// unpacking TMA can read in place are not expanded: only their scales are
// regrouped.
//
// Tile schedule of the persistent staged kernel (grid `grid`, one CTA per SM).
// Without a split, CTA c takes tiles c, c + grid, ...  With one (`split`),
// the first `nd` waves of whole tiles go that way and the last
// R = tiles - nd * grid tiles, which would leave most SMs idle in a final
// wave, are cut along K: their R * kt k-steps (sk_len) are divided evenly
// over all CTAs, CTA c taking k-steps [c * sk_len / grid, (c + 1) * sk_len /
// grid) of them, tile by tile.  A CTA whose share starts inside a tile writes
// that part's fp32 sums to its slot of `off_sk` and raises per-warp flags;
// the CTA holding the tile's first k-step adds the later parts in k order
// and runs the epilogue.
struct StagedPlan {
  bool b_native;
  int64_t k_pad, kt, mt, nt, bb;
  // offsets from the 1024-aligned workspace base; off_sfe: per-32-block scale
  // bytes of g16 weights ([bb][N][k_pad / 32]), in B-only plans; off_sk: the
  // split parts' partial sums ([grid][128 x 224] fp32) and their flags
  // ([grid][12] words), present when split
  size_t off_a, off_sfa, off_sk, off_b, off_sfb, off_sfe, bytes;
  int grid, split, nd;
  int64_t sk_tile0, sk_len;
};
// Weights with one scale per 16 elements (MXINT4g16 / MXFP4g16).
inline bool b_g16(const mix_gemm_desc_t& d) { return d.b_block == 16; }
constexpr int kStagedAlign = 1024;
constexpr int kStagedBN = 224;  // output columns per tile of the staged matmul
constexpr int kSkSlotBytes = 128 * kStagedBN * 4;  // one split part's fp32 sums
constexpr int kSkFlags = 12;                        // flags per part: one per epilogue warp
StagedPlan staged_plan(const mix_gemm_desc_t& d);
StagedPlan staged_plan_b_only(const mix_gemm_desc_t& d);  // B expansion alone (fused-decode path)
bool staged_fp4_native_ok(const mix_gemm_desc_t& d);
int64_t expand_a_threads(const mix_gemm_desc_t& d, const StagedPlan& sp);
int64_t expand_b_threads(const StagedPlan& sp);
cudaError_t launch_expand_a(const mix_gemm_desc_t& d, const StagedPlan& sp, unsigned char* base, cudaStream_t st);
cudaError_t launch_expand_b(const mix_gemm_desc_t& d, const StagedPlan& sp, unsigned char* base, cudaStream_t st);

// Fused decode attention.
size_t decode_attention_ws_bytes(const mix_decode_attn_desc_t& d);
cudaError_t launch_decode_attention(const mix_decode_attn_desc_t& d, void* ws, cudaStream_t st);

// K-smoothing.
size_t ksmooth_ws_bytes(int64_t tokens, int heads, int head_dim);
cudaError_t launch_ksmooth(const void* k, bool bf16, int64_t tokens, int heads, int head_dim,
                           int64_t ld, float* mean, int mode, float* k_out, void* ws,
                           cudaStream_t st);

// K-smoothing with the library's built-in scratch (no caller workspace).
size_t ksmooth_noalloc_scratch_bytes();
cudaError_t launch_ksmooth_noalloc(const void* k, bool bf16, int64_t tokens, int heads, int head_dim,
                                   int64_t ld, float* mean, int mode, float* k_out, cudaStream_t st);

// Device error word (bounded waits), and the launch that makes one run out.
cudaError_t read_device_error(unsigned* word, bool clear);
cudaError_t device_error_word(unsigned** word);  // device address of the error word
size_t selftest_ws_bytes();
cudaError_t launch_selftest_wait_timeout(void* ws, long long limit_cycles, cudaStream_t st);

}  // namespace mixk
