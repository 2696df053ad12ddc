/*
 * mix.h -- C ABI of libmix.so: the MiX (Micro-Inverted-Scaling) hot path on
 * one NVIDIA B300 (sm_103a).
 *
 * Source of every operation: "MiX: Micro-Inverted-Scaling for End-to-End
 * Low-Bit Vision-Language Model Acceleration" (Liao and Seo, MICRO 2026), as
 * digested on the pchao.org page "MiX：面向端到端低比特视觉语言模型加速的微反缩放"
 * (sections named below are that page's).
 *
 * Bit layouts (the page gives field widths only; orders are this library's):
 *  - MiX element nibble: bit 3 sign, bits 2..0 delta-e; 0x7 is zero; 0xF is
 *    the recycled "-0", a positive value (1.mshared) * 2^(Emax - 7).
 *  - MiX-4.25b shared byte: bits 3..0 Emax - ebias, bits 6..4 mshared, bit 7 0.
 *  - MiX-4.5b shared uint16: bits 3..0 Emax - ebias, then the mshared of
 *    sub-blocks 0..3 in bits 6..4, 9..7, 12..10, 15..13.
 *  - MX element nibble: OCP E2M1 (MXFP4) or two's complement q (MXINT4);
 *    scale byte X + 127 (E8M0).
 *
 * Conventions for every call:
 *  - Pointers named x, codes, shared, scales, c, out_*, mean, k_out and
 *    workspace are DEVICE pointers owned by the caller; the library allocates
 *    no device memory and keeps no pointer after a call returns.
 *  - Calls are asynchronous on `stream` (NULL = the legacy default stream).
 *  - Arguments are validated on the host before any launch; a rejected call
 *    launches nothing and returns a MIX_ERR_* status.  A launch failure
 *    returns MIX_ERR_CUDA.
 *  - Non-finite inputs never fault: NaN is coded as zero and +-Inf saturates.
 *  - The element-wise kernels number their work items with 32 bits.  A call
 *    that would need 2^32 - 1 or more returns MIX_ERR_UNSUPPORTED before any
 *    launch.  The items are 32-element blocks for mix_quantize and for
 *    mx_quantize along rows; 16-element blocks for nvfp4_quantize; 8-element
 *    groups for mix_underflow_count; and 16-byte vectors of x for the amax
 *    pass of mix_auto_ebias, mix_quantize_auto and nvfp4_quantize.  The
 *    tightest of these is the amax pass, at 64 GiB of input (2^35 bf16 or
 *    2^34 fp32 elements).
 *  - Sizes are in elements unless a name ends in _bytes.  The packed planes
 *    of a matrix with R rows and K columns are: codes R x K/2 bytes (element
 *    2j in the low nibble of byte j, 16-byte aligned rows), shared R x K/32
 *    entries (uint8 for MiX-4.25b, uint16 for MiX-4.5b), scales R x K/32
 *    E8M0 bytes.  K must be a multiple of 32.
 */
#ifndef MIX_H_
#define MIX_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MIX_API __attribute__((visibility("default")))
#else
#define MIX_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* mix_stream_t; /* same handle as cudaStream_t */

typedef enum {
  MIX_OK = 0,
  MIX_ERR_INVALID_ARG = 1, /* null pointer, unknown enum value, negative size  */
  MIX_ERR_SHAPE = 2,       /* K % 32 != 0, N % 32 != 0 for a quantising epilogue */
  MIX_ERR_ALIGN = 3,       /* a plane or stride breaks its alignment rule       */
  MIX_ERR_UNSUPPORTED = 4, /* a valid request this build does not implement     */
  MIX_ERR_CUDA = 5,        /* a CUDA runtime error at launch                     */
  MIX_ERR_WORKSPACE = 6,   /* workspace missing or smaller than required         */
  MIX_ERR_DEVICE = 7       /* a kernel's bounded wait ran out (see below)        */
} mix_status_t;

typedef enum { MIX_T1_4P25 = 1, MIX_T2_4P5 = 2 } mix_type_t;
typedef enum { MX_INT4 = 0, MX_FP4_E2M1 = 1 } mx_type_t;
typedef enum { MIX_DT_F32 = 0, MIX_DT_BF16 = 1 } mix_dtype_t;

/* Quantiser flags. */
enum {
  MIX_ASYM_ZERO = 1,  /* MiX: recycle the -0 code for one more positive binade
                         (Method section, accelerator bullet).  Default on.   */
  MX_SCALE_FLOOR = 2, /* MXFP4: OCP floor shared exponent instead of the ceil
                         rule the paper uses for every MXFP4 (Key results).   */
  MX_SCALE_TIGHT = 4, /* MX: the smallest shared exponent at which no element
                         of the block saturates -- ceil(log2(amax / 6)) for
                         MXFP4 (the alternative to the ceil rule named beside
                         it in Key results), ceil(log2(amax / 1.75)) for
                         MXINT4.  Not combinable with MX_SCALE_FLOOR.         */
  MX_BLOCK16 = 8      /* mx_quantize: one scale per 16 elements (MXINT4g16 /
                         MXFP4g16, the g16 weights of "MiX-INT4g16"); the
                         scale plane is N x K/16.                             */
};

/* ---------------------------------------------------------------------- */
/* Plane sizes (host only, no device work).                                */
/* ---------------------------------------------------------------------- */

/* rows * k / 2.  Returns 0 for negative sizes or k % 32 != 0. */
MIX_API size_t mix_codes_bytes(int64_t rows, int64_t k);
/* rows * k/32 * (1 for MiX-4.25b, 2 for MiX-4.5b).  4.25 and 4.5 bits per
 * element together with the codes (Method section, MiX-4.25b and MiX-4.5b
 * bullets: (8 + 128)/32 and (4 + 4*3 + 32*4)/32 bits). */
MIX_API size_t mix_shared_bytes(mix_type_t type, int64_t rows, int64_t k);
/* rows * k / 32 E8M0 scale bytes of an MX plane. */
MIX_API size_t mx_scales_bytes(int64_t rows, int64_t k);

/* ---------------------------------------------------------------------- */
/* MiX activation quantiser -- Algorithm 1 (Method section).               */
/* ---------------------------------------------------------------------- */
/* Per 32-element block along k: Emax from the block's largest magnitude,
 * mshared from that element's mantissa (rounded to 3 bits, nearest-even), then
 * per element the delta-e of least error among {de-1, de, de+1}; de = 7 codes
 * zero; with MIX_ASYM_ZERO the -0 code is a positive level below de = 6.
 * MiX-4.5b (Type 2) keeps one Emax per block and one mshared per 8-element
 * sub-block.  Emax is stored as Emax - ebias in 4 bits (clamped).
 *   x      rows x k input, row stride ld >= k elements, fp32 or bf16,
 *          16-byte aligned with ld * sizeof(elem) a multiple of 16.
 *   ebias  -100 .. 100; -8 suits activations, -15 softmax probabilities.
 *   codes  rows x k/2 bytes (dense, 16-byte aligned).
 *   shared rows x k/32 uint8 (Type 1) or uint16 (Type 2), dense.
 * Output is bit-identical to the plain CPU definition. */
MIX_API mix_status_t mix_quantize(const void* x, mix_dtype_t dtype, int64_t rows, int64_t k, int64_t ld,
                          mix_type_t type, int ebias, unsigned flags, uint8_t* codes,
                          void* shared, mix_stream_t stream);

/* Data-dependent ebias (a two-pass mode; the Method section fixes only the
 * 4-bit width of Emax).  Pass 1 finds the largest block exponent f over the
 * tensor -- floor(log2) of a block maximum after Algorithm 1 rounds its
 * mantissa to three bits, carry included -- and sets ebias = f - 15, so that
 * block takes the top code and no block clamps from above; clamped to
 * [-100, 100].  +-Inf and NaN elements are left out (they saturate / code zero
 * under any ebias); a tensor with no nonzero finite element gets -8.
 *   x, dtype, rows, k, ld   as for mix_quantize (same alignment rules).
 *   ebias   one int in DEVICE memory (4-byte aligned), written on `stream`;
 *           the host reads it only after synchronising.
 * Three launches: a clear, a max-reduction over x, a one-warp finish. */
MIX_API mix_status_t mix_auto_ebias(const void* x, mix_dtype_t dtype, int64_t rows, int64_t k, int64_t ld,
                                    int* ebias, mix_stream_t stream);
/* mix_auto_ebias followed by mix_quantize with that ebias, all on `stream`
 * with no host round trip (the quantiser reads *ebias on the device).  The
 * ebias stays in *ebias for dequantisation and the matmul's a_ebias. */
MIX_API mix_status_t mix_quantize_auto(const void* x, mix_dtype_t dtype, int64_t rows, int64_t k, int64_t ld,
                                       mix_type_t type, unsigned flags, uint8_t* codes, void* shared,
                                       int* ebias, mix_stream_t stream);

/* ---------------------------------------------------------------------- */
/* W-MX quantiser (MXINT4 / MXFP4, block 32, E8M0 scale).                  */
/* ---------------------------------------------------------------------- */
/* Blocks run along the reduction dimension K; outputs are N x K planes.
 * With MX_BLOCK16 the blocks hold 16 elements (K still a multiple of 32) and
 * the scales plane is N x K/16; the rules below apply per 16-block.
 *   axis = 1: x is N x K (rows = N, cols = K), row stride ld >= K.
 *   axis = 0: x is K x N (rows = K, cols = N), row stride ld >= N -- a
 *             weight stored for x @ W; it is read down its columns and the
 *             planes are written transposed (N x K).
 * MXFP4 shared exponent: ceil(log2 amax) - 2 (the paper's ceil rule, Key
 * results section), the OCP floor with MX_SCALE_FLOOR, or the tight rule with
 * MX_SCALE_TIGHT (both flags together: MIX_ERR_INVALID_ARG); elements E2M1,
 * nearest-even, saturating at 6.  MXINT4: X = floor(log2 amax), elements
 * q * 2^(X-2), q in [-7, 7] two's complement, nearest-even.
 *   codes  N x K/2 bytes; scales N x K/32 bytes (X + 127). */
MIX_API mix_status_t mx_quantize(const void* x, mix_dtype_t dtype, int64_t rows, int64_t cols, int64_t ld,
                         int axis, mx_type_t type, unsigned flags, uint8_t* codes,
                         uint8_t* scales, mix_stream_t stream);

/* ---------------------------------------------------------------------- */
/* Comparison formats and the dead-zone count.                             */
/* ---------------------------------------------------------------------- */
/* NVFP4, the 16-element comparison format the pages set MiX against (blocks
 * of 16 E2M1 elements, an E4M3 block scale, one FP32 tensor scale).  Every
 * step is one IEEE fp32 operation, in this order: amax_t = the largest finite
 * |x| of the tensor; s_t = amax_t / 2688 (1 if amax_t is 0, the smallest
 * positive float if the quotient underflows); per 16-block t = (amax_b / s_t)
 * / 6 (NaN left out of amax_b, +-Inf included) and its E4M3 code sb (nearest,
 * ties even, saturating at 448); d = e4m3(sb) * s_t; each element the E2M1
 * code of x / d (nearest, ties even, saturating at 6; NaN codes +0; -0 is
 * written as +0); a block with sb = 0 stores zero codes.
 *   x       rows x k, k % 16 == 0, row stride ld (alignment as mix_quantize).
 *   codes   rows x k/2 bytes (8-byte aligned); scales rows x k/16 E4M3 bytes.
 *   tensor_scale  one float in DEVICE memory, written on `stream`.
 * Four launches: a clear, the amax reduction, a one-warp finish, the quantiser. */
MIX_API mix_status_t nvfp4_quantize(const void* x, mix_dtype_t dtype, int64_t rows, int64_t k, int64_t ld,
                                    uint8_t* codes, uint8_t* scales, float* tensor_scale, mix_stream_t stream);

/* Clamped-block count of the MiX quantiser (Method section, MiX-4.25b
 * bullet: Emax has 4 bits, so with Emax = field + ebias a block exponent
 * outside [ebias, ebias + 15] is clamped).  For every 32-element block of x
 * (rows x k, row stride ld elements, bf16 or fp32): f = the exponent that
 * steps 1-2 of Algorithm 1 give the block maximum, its 3-bit mantissa
 * rounding and carry included.  counts[0] = blocks with f > ebias + 15 (the
 * elements saturate; +-Inf blocks count here); counts[1] = blocks with a
 * nonzero maximum and f < ebias (small elements flush to zero).  NaN counts
 * as zero.  counts: two uint64 in device memory, 8-byte aligned, overwritten
 * (stream-ordered).  x 16-byte aligned, ld * element size a multiple of 16,
 * k % 32 == 0, ebias in [-100, 100]. */
MIX_API mix_status_t mix_clamp_count(const void* x, mix_dtype_t dtype, int64_t rows, int64_t k, int64_t ld,
                                     int ebias, unsigned long long* counts, mix_stream_t stream);

/* Dead-zone count (the key-underflow comparison of the Key results section,
 * made synthetic): how many finite nonzero elements of x have a zero code in
 * `codes` -- 0x7 for MiX (the recycled -0 code 0xF is not zero), 0 for MXINT4,
 * +-0 (nibble & 7 == 0) for E2M1 formats (MXFP4, NVFP4).
 *   x       rows x k (k % 16 == 0), row stride ld; codes rows x k/2 (dense, 4-byte aligned).
 *   count   one unsigned long long in DEVICE memory, written on `stream`. */
typedef enum { MIX_UF_MIX = 0, MIX_UF_MXINT4 = 1, MIX_UF_E2M1 = 2 } mix_underflow_fmt_t;
MIX_API mix_status_t mix_underflow_count(const void* x, mix_dtype_t dtype, int64_t rows, int64_t k, int64_t ld,
                                         const uint8_t* codes, mix_underflow_fmt_t fmt, unsigned long long* count,
                                         mix_stream_t stream);

/* Test aids: decode packed planes to fp32 (rows x k, dense).  MiX: the rule
 * (-1)^s (1.mshared)_2 2^(Emax - de) of the Method section, de = 7 zero, code
 * 0xF the recycled positive level.  MX: w * 2^X. */
MIX_API mix_status_t mix_dequantize(const uint8_t* codes, const void* shared, int64_t rows, int64_t k,
                            mix_type_t type, int ebias, float* out, mix_stream_t stream);
MIX_API mix_status_t mx_dequantize(const uint8_t* codes, const uint8_t* scales, int64_t rows, int64_t k,
                           mx_type_t type, float* out, mix_stream_t stream);

/* ---------------------------------------------------------------------- */
/* A-MiX x W-MX block matmul with optional fused output quantiser.         */
/* ---------------------------------------------------------------------- */
/* C[b][m][n] = sum over 32-blocks of Eq. (6) (Method section, dual-format
 * matmul bullet): per block (1.mshared) * 2^(Emax + X) * sum_i s_i w_i
 * 2^(-de_i), per 8-sub-block mshared for MiX-4.5b.  A (activations, MiX) is
 * batch x M x K; B (weights or K/V, MX) is (batch / b_group) x N x K with
 * blocks along K -- exactly what mx_quantize writes.  fp32 accumulation.
 *
 * Epilogue (Method section, accelerator bullet: accumulator -> fused MiX/MX
 * quantiser -> DRAM): each 32-column block of each output row is quantised
 * as mix_quantize / mx_quantize(axis 1) would quantise the fp32 row, into
 * out_codes / out_shared (MiX shared, or MX scales).  C may be written too.
 *
 * Strides are in ELEMENTS of the logical matrix and must be multiples of 32:
 * the codes of row m, batch b of A start at byte (b*a_batch_stride +
 * m*a_ld)/2 of a_codes, its shared entries at index (b*a_batch_stride +
 * m*a_ld)/32 of a_shared; likewise for B and the epilogue planes.  C is fp32
 * with its own element strides ldc and c_batch_stride.
 *
 * algo: MIX_GEMM_AUTO picks the integer shift-add path for M <= 16 and the
 * tcgen05 tensor-core path otherwise; the others force a path.  The
 * shift-add path evaluates Eq. (6) literally (integer shift-add trees, one
 * multiply by the shared mantissa, one exponent add) and splits K across
 * CTAs when there are few outputs, summing the partials in a fixed order in
 * the caller's workspace (see mix_mx_gemm_workspace_bytes).
 *
 * The tensor-core path has two variants.  Every product is exact and the
 * fp32 sums run in K order in both, so their results are identical, except
 * where the staged variant cuts a tile along K (below):
 *  - staged (MIX_GEMM_TCGEN05_STAGED; chosen by AUTO / TCGEN05 when N > 256):
 *    A, and B unless it is MXFP4 that the unpacking TMA reads in place, are
 *    first expanded into exact e4m3 planes and UE8M0 scale words in the
 *    caller's workspace, then a TMA-fed tcgen05 kernel multiplies them.  The
 *    workspace holds batch*M*Kp + bB*N*Kp bytes (Kp = K rounded up to 128,
 *    bB = ceil(batch / b_group); the B plane only when B is expanded) plus
 *    the scale words and alignment; mix_mx_gemm_workspace_bytes gives the
 *    exact size and a smaller workspace returns MIX_ERR_WORKSPACE.  When
 *    the output tiles (128 x 224) leave a last wave that would keep most SMs
 *    idle, those tiles' K loops are shared out over all SMs: each part's fp32
 *    sums go through the workspace (one 128 x 224 fp32 slot and 12 flag
 *    words per SM) and the SM holding a tile's first k-steps adds the later
 *    parts in K order before the epilogue.  Such tiles can differ from the
 *    fused variant in the last bits of C; the result is deterministic for a
 *    given device.  Such a launch is cooperative (all its CTAs, one per SM,
 *    resident together); a part that never arrives ends its wait with bit 9
 *    of the device error word.
 *  - fused decode (MIX_GEMM_TCGEN05_FUSED; chosen when N <= 256): decoder
 *    warps expand each A tile inside the matmul; B enters by TMA, MXFP4 in
 *    place (no workspace) or else expanded once into e4m3 in the workspace
 *    (bB*N*Kp bytes plus its scale words and alignment).
 */
typedef enum { MIX_EPI_NONE = 0, MIX_EPI_MIX_T1 = 1, MIX_EPI_MIX_T2 = 2,
               MIX_EPI_MXINT4 = 3, MIX_EPI_MXFP4 = 4 } mix_epilogue_t;
typedef enum { MIX_GEMM_AUTO = 0, MIX_GEMM_TCGEN05 = 1, MIX_GEMM_SHIFTADD = 2,
               MIX_GEMM_TCGEN05_STAGED = 3, MIX_GEMM_TCGEN05_FUSED = 4 } mix_gemm_algo_t;

typedef struct {
  int64_t M, N, K;
  int64_t batch;   /* >= 1 */
  int64_t b_group; /* >= 1; batch b reads B batch b / b_group (GQA) */
  const uint8_t* a_codes;
  const void* a_shared;
  mix_type_t a_type;
  int a_ebias;
  int64_t a_ld, a_batch_stride;
  const uint8_t* b_codes;
  const uint8_t* b_scales;
  mx_type_t b_type;
  int b_block;     /* elements per B scale: 32 (0 means 32) or 16 (g16) */
  int64_t b_ld, b_batch_stride;
  float* c; /* optional fp32 output (NULL: epilogue planes only) */
  int64_t ldc, c_batch_stride;
  mix_epilogue_t epi;
  int epi_ebias;       /* MiX epilogues */
  unsigned epi_flags;  /* MIX_ASYM_ZERO / MX_SCALE_FLOOR / MX_SCALE_TIGHT */
  uint8_t* out_codes;  /* batch x M x N/2 codes of the quantised output */
  void* out_shared;    /* MiX shared entries or MX scale bytes */
  int64_t out_ld, out_batch_stride;
  mix_gemm_algo_t algo;
  /* Optional: B in the tensor-core path's prepared form, written by
   * mix_mx_gemm_prepare_b for a descriptor with the same M, N, K, batch,
   * b_group, B fields and algo (NULL: B is prepared inside every call). */
  const void* b_prepared;
  /* Optional causal bound of A (a_causal = 0: none).  a_causal = 1 asserts
   * that in every batch A[m][k] is zero for every k > m + a_causal_shift:
   * the masked part of a causal attention P (a_causal_shift = keys -
   * queries, 0 for a square self-attention P; |a_causal_shift| < 2^31).
   * The fused-decode variant then neither loads nor multiplies the 128-deep
   * k-steps that lie wholly past the bound of a 128-row tile, and starts the
   * tiles with the longest K loops first; the other variants ignore it.
   * When the assertion holds the result is the same bits as without it (the
   * skipped steps would only add exact zeros); when it does not, the entries
   * of those steps are taken as zero. */
  int a_causal;
  int64_t a_causal_shift;
} mix_gemm_desc_t;

/* Bytes of device workspace mix_mx_gemm needs for this descriptor (0 if
 * none).  The workspace is scratch owned by the caller; its contents on entry
 * do not matter.  With b_prepared set it covers A's staging only. */
MIX_API size_t mix_mx_gemm_workspace_bytes(const mix_gemm_desc_t* desc);
MIX_API mix_status_t mix_mx_gemm(const mix_gemm_desc_t* desc, void* workspace, size_t workspace_bytes,
                         mix_stream_t stream);

/* Prepared weights.  The tensor-core path feeds the MMA from B in a fixed
 * form: the UE8M0 scale bytes regrouped into the words the MMA's scale
 * columns take (one 32-bit word per row and 128-deep k-step, in tiles of
 * rows), plus, unless B is MXFP4 that the unpacking TMA reads in place, the
 * exact e4m3 expansion of every element (Kp = K rounded up to 128 bytes per
 * row).  This is a layout transform of B alone: no arithmetic of the method
 * moves out of the matmul, and the products are the same bits.  Weights are
 * fixed, so a caller can prepare them once, when they are quantised, and
 * pass the result in desc->b_prepared on every call; without it each call
 * prepares B again in its workspace.
 *   mix_mx_gemm_prepare_b_bytes: bytes of the prepared form (0: this
 *     descriptor takes no prepared B -- the shift-add path, or MXFP4 on the
 *     fused-decode variant, which reads B as it is).
 *   mix_mx_gemm_prepare_b: writes it into `prepared` (device memory owned by
 *     the caller, any alignment of 16 bytes or more; valid while B's planes
 *     are unchanged).  desc->b_prepared is ignored here. */
MIX_API size_t mix_mx_gemm_prepare_b_bytes(const mix_gemm_desc_t* desc);
MIX_API mix_status_t mix_mx_gemm_prepare_b(const mix_gemm_desc_t* desc, void* prepared, size_t prepared_bytes,
                                           mix_stream_t stream);

/* ---------------------------------------------------------------------- */
/* K-smoothing (SageAttention style; Method section, accelerator bullet,   */
/* and Caveats section on the static prefill mean).                        */
/* ---------------------------------------------------------------------- */
/* k: tokens x heads x head_dim keys (bf16 or fp32), token stride ld >= heads *
 * head_dim elements.  KSMOOTH_COMPUTE: mean[h][d] = mean over the tokens,
 * summed as fp32 pairs (about 48 bits, Knuth's two-sum) in a fixed order,
 * divided by the token count in fp64 and rounded once to fp32 (the prefill
 * mean).  KSMOOTH_APPLY_FROZEN: mean is an input (frozen at prefill; decode
 * does not re-read the cache).  Both modes write k_out = fp32(k) - mean (one
 * fp32 subtraction), tokens x heads x head_dim dense, when k_out != NULL.
 * COMPUTE splits the tokens across CTAs and keeps per-chunk partial sums
 * (fp32 pairs, about 48 bits) in the caller's workspace
 * (ksmooth_workspace_bytes); APPLY needs none.  When every CTA's run of
 * tokens fits in shared memory (a few MB of keys in all, e.g. one layer's
 * prefill), COMPUTE is one cooperative launch whose CTAs meet at a barrier
 * counter in the workspace; longer inputs take three kernels.  The two
 * orders of summation can differ in the last bit of the mean. */
enum { KSMOOTH_COMPUTE = 0, KSMOOTH_APPLY_FROZEN = 1 };
MIX_API size_t ksmooth_workspace_bytes(int64_t tokens, int heads, int head_dim);
MIX_API mix_status_t ksmooth_kv(const void* k, mix_dtype_t dtype, int64_t tokens, int heads, int head_dim,
                        int64_t ld, float* mean, int mode, float* k_out, void* workspace,
                        size_t workspace_bytes, mix_stream_t stream);

/* No-allocation variant of ksmooth_kv.  The paper has no counterpart for
 * this entry point; it exists for callers that cannot give the library device
 * memory: hosts whose device memory all belongs to their own allocator (a
 * framework's pool that hands out no raw buffers), and serving or decode loops
 * that must not call cudaMalloc, which can synchronise the whole device and
 * stall every stream.  Arguments and results are
 * those of ksmooth_kv; the caller still passes k, mean and k_out.  COMPUTE
 * keeps its partial sums in a fixed array built into the library
 * (KSMOOTH_NOALLOC_SCRATCH_BYTES, held on every GPU that loads the library
 * until the process exits) and allocates nothing.
 *  - Size limit: a COMPUTE call whose ksmooth_workspace_bytes(tokens, heads,
 *    head_dim) exceeds KSMOOTH_NOALLOC_SCRATCH_BYTES is rejected with
 *    MIX_ERR_WORKSPACE before any launch.
 *  - The first call on a device looks up the array's device address (with
 *    that device current); make that first call before any stream capture.
 *    The address is kept for the life of that device's CUDA context: a call
 *    made under a new context (after cudaDeviceReset, say) looks it up again.
 *  - All calls share the array.  Calls ordered on one stream are safe; calls
 *    whose kernels overlap on the GPU (other streams, other threads) race.
 *    Nothing has to be cleared between calls: each call writes every partial
 *    sum it later reads. */
#define KSMOOTH_NOALLOC_SCRATCH_BYTES ((size_t)2 << 20)
MIX_API mix_status_t ksmooth_kv_noalloc(const void* k, mix_dtype_t dtype, int64_t tokens, int heads,
                                        int head_dim, int64_t ld, float* mean, int mode, float* k_out,
                                        mix_stream_t stream);

/* ---------------------------------------------------------------------- */
/* Fused decode attention over an MX KV cache.                             */
/* ---------------------------------------------------------------------- */
/* One decode step for one sequence (one query token per head, GQA), in the
 * dataflow of the Method section's accelerator bullet: the new key is
 * smoothed with the frozen prefill mean and appended to the MXINT4 K' cache,
 * S = q K'^T by Eq. (6) with q quantised to MiX-4.5b, P = softmax(sm_scale S)
 * over the cache, P requantised to MiX-4.5b (32-token blocks, ebias p_ebias),
 * O = P V by Eq. (6) against the MXINT4 V cache (blocks along tokens).  One
 * cooperative launch (KV heads x token chunks, filling the SMs once) keeps
 * each chunk's keys, values and scores in shared memory and meets at two
 * bounded grid barriers (a counter in the workspace; bit 11 of the device
 * error word on timeout): after the chunk statistics, and after the partial
 * outputs, which are then summed in chunk order.  A cache too long for that
 * (chunks over 200 KB of shared memory, tens of thousands of tokens) runs as
 * two kernels, the last CTA of each KV head summing the partials.
 * Products are exact integers per block; block terms, S and the softmax are
 * fp32 (expf); O matches the oracle's fp64 composition within 1e-3 of each
 * head's largest |O|. */
typedef struct {
  int64_t tokens;        /* cache length including the new token (>= 1)        */
  int q_heads, kv_heads; /* q_heads % kv_heads == 0, q_heads / kv_heads <= 8    */
  int head_dim;          /* 128                                                 */
  mix_dtype_t dtype;     /* of q and k_new                                      */
  const void* q;         /* [q_heads][head_dim]                                  */
  const void* k_new;     /* [kv_heads][head_dim], or NULL: no append             */
  const float* k_mean;   /* [kv_heads][head_dim] frozen prefill mean (with k_new) */
  uint8_t* k_codes;      /* K' cache [tokens][kv_heads][head_dim/2], MXINT4 along
                            head_dim; row tokens-1 is written when k_new is set */
  uint8_t* k_scales;     /* [tokens][kv_heads][head_dim/32], 4-byte aligned rows  */
  const uint8_t* v_codes;  /* V cache [kv_heads][head_dim][v_ld/2], MXINT4 along tokens */
  const uint8_t* v_scales; /* [kv_heads][head_dim][v_ld/32]                         */
  int64_t v_ld;          /* token capacity of the V planes: a multiple of 32 >= tokens */
  float sm_scale;        /* softmax temperature (1/sqrt(head_dim) typically)     */
  int q_ebias, p_ebias;  /* MiX ebias of q (-8) and of P (-15)                   */
  float* out;            /* O [q_heads][head_dim] fp32                           */
  uint8_t* p_codes;      /* optional P planes [q_heads][v_ld/2] (NULL: not kept); only
                            the 32-token blocks that hold a token are written    */
  void* p_shared;        /* [q_heads][v_ld/32] uint16 MiX-4.5b shared fields     */
  float* p_values;       /* optional [q_heads][v_ld] fp32 (NULL: not kept): the
                            probabilities the kernel quantised into p_codes, for
                            checking the quantiser on the kernel's own P; only the
                            32-token blocks that hold a token are written, with 0
                            past the last token                                   */
} mix_decode_attn_desc_t;

/* Device workspace bytes (the per-chunk statistics and partial outputs, the
 * barrier counter; S as well on the two-kernel path). */
MIX_API size_t mix_decode_attention_workspace_bytes(const mix_decode_attn_desc_t* desc);
MIX_API mix_status_t mix_decode_attention(const mix_decode_attn_desc_t* desc, void* workspace, size_t workspace_bytes,
                                          mix_stream_t stream);

/* ---------------------------------------------------------------------- */
/* Status and device error word.                                           */
/* ---------------------------------------------------------------------- */
MIX_API const char* mix_status_str(mix_status_t status);
/* Kernels never spin without bound: a wait that runs out records a bit in a
 * per-device error word and the kernel returns early (its outputs are then
 * undefined).  This reads the word for the current device (synchronising the
 * device) and clears it when `clear` is nonzero.  MIX_OK if the read worked.
 * Bits 0..9: a wait of the matmul kernels (which one, by role); bit 10:
 * the grid barrier of the one-pass K-smoothing kernel; bit 11: a grid
 * barrier of the one-kernel decode attention. */
MIX_API mix_status_t mix_device_error(unsigned* word, int clear);
/* Test aid for the bounded waits.  Launches the staged tensor-core matmul
 * kernel once, on a single 128 x 224 tile, with its producer switched off
 * and every wait limited to 2^20 SM clocks (about half a millisecond): the
 * MMA thread's wait for the first stage runs out with no copy or MMA in
 * flight, the kernel records it in the device error word (bit 1, or bit 5
 * if a scale warp's wait runs out first), its other roles see the CTA's
 * abort flag, and the CTA frees its TMEM and exits.  The device stays
 * usable; read and clear the word with mix_device_error afterwards.
 * workspace: device memory, 16-byte aligned, at least
 * MIX_SELFTEST_WORKSPACE_BYTES (its contents are never read). */
#define MIX_SELFTEST_WORKSPACE_BYTES ((size_t)64 << 10)
MIX_API mix_status_t mix_selftest_wait_timeout(void* workspace, size_t workspace_bytes, mix_stream_t stream);
/* Library version, major * 10000 + minor * 100 + patch. */
MIX_API int mix_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MIX_H_ */
