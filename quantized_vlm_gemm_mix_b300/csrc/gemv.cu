// Integer shift-add path of the A-MiX x W-MX matmul for decode shapes
// (M <= 16): Eq. (6) of the pchao.org digest of "MiX: Micro-Inverted-Scaling
// ..." (Method section, dual-format matmul bullet) evaluated literally on CUDA
// cores.  Per 32-block: each W-MX element's integer mantissa is shifted by
// the MiX element's delta-e (the MXFP4 element's own exponent added first),
// the terms of each 8-element sub-tree are summed as integers, each sub-tree
// sum is multiplied by its shared mantissa (8 + m3, the 4.5b PE) or all by one
// (4.25b), and one exponent add 2^(Emax + X - 10 - c_B) scales the block.
// Block sums are exact (|sum| < 2^20); blocks are accumulated in fp32.
//
// Layout of work: a CTA owns one batch, one K-chunk and a range of output
// columns n.  The chunk of A (all M rows) is decoded once into shared memory
// as per-element factors s * 2^(7 - de) (0 for the zero code, +1 for the
// recycled -0 code).  T lanes share one n and split its blocks; T = 32 for
// long K (one warp per n), down to 1 for K = 128 (one lane per n).  When the
// output is too small to fill the GPU the K range is split across CTAs and
// the fp32 partials go to the caller's workspace, then are summed in a fixed
// order.
#include <cuda_runtime.h>

#include "decode.cuh"
#include "mix_internal.h"

namespace mixk {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxM = 16;

struct GemvArgs {
  const uint8_t* a_codes;
  const void* a_shared;
  const uint8_t* b_codes;
  const uint8_t* b_scales;
  float* out;  // C (splits == 1) or the partial buffer
  int64_t M, N, K, b_group;
  int64_t a_ld, a_bs, b_ld, b_bs;
  int64_t out_ld, out_bs, out_split_stride;
  int64_t kc;  // elements per K-chunk (multiple of 32)
  int a_type, a_ebias, b_fp4, tpn;
};

__device__ __forceinline__ int a_factor(uint32_t c) {
  const int d = (int)(c & 7u);
  if (c == 7u) return 0;   // zero code
  if (c == 15u) return 1;  // recycled -0: + 2^0 (one binade below de = 6)
  const int v = 128 >> d;  // 2^(7 - de)
  return (c & 8u) ? -v : v;
}

// W-MX element code -> int8 value through two 8-entry byte tables and a
// byte select by the sign bit (dec8): E2M1 in half units (0, 1, 2, 3, 4, 6,
// 8, 12 and their negatives), INT4 as its two's complement value.
__device__ __forceinline__ DecTab fp4_int8_tab() { return DecTab{0x03020100u, 0x0C080604u, 0xFDFEFF00u, 0xF4F8FAFCu}; }
__device__ __forceinline__ DecTab int4_int8_tab() { return DecTab{0x03020100u, 0x07060504u, 0xFBFAF9F8u, 0xFFFEFDFCu}; }

// G16: weights with one scale per 16 elements; each 32-block's two halves
// (sub-trees 0-1 and 2-3) take their own exponent add.
template <bool G16>
__global__ void __launch_bounds__(kThreads) gemv_shiftadd_kernel(GemvArgs p) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int64_t bt = blockIdx.z;
  const int64_t split = blockIdx.y;
  const int64_t k0 = split * p.kc;
  const int64_t kc = min(p.kc, p.K - k0);
  const int nbc = (int)(kc / 32);
  const int64_t nbc_max = p.kc / 32;
  int16_t* fa = reinterpret_cast<int16_t*>(smem);                                 // [M][nbc][32]
  int2* ash = reinterpret_cast<int2*>(smem + (size_t)p.M * nbc_max * 32 * sizeof(int16_t));  // [M][nbc]

  // Decode this CTA's chunk of A once.
  const int64_t words = p.M * (kc / 8);
  for (int64_t w = threadIdx.x; w < words; w += blockDim.x) {
    const int64_t m = w / (kc / 8), j = w - m * (kc / 8);
    const int64_t e0 = bt * p.a_bs + m * p.a_ld + k0 + j * 8;
    const uint32_t cw = *reinterpret_cast<const uint32_t*>(p.a_codes + e0 / 2);
    int16_t* dst = fa + (m * nbc_max + j / 4) * 32 + (j & 3) * 8;
#pragma unroll
    for (int i = 0; i < 8; ++i) dst[i] = (int16_t)a_factor((cw >> (4 * i)) & 0xFu);
  }
  const int64_t blocks = p.M * nbc;
  for (int64_t w = threadIdx.x; w < blocks; w += blockDim.x) {
    const int64_t m = w / nbc, b = w - m * nbc;
    const int64_t idx = (bt * p.a_bs + m * p.a_ld + k0) / 32 + b;
    int emax, mk;
    if (p.a_type == 1) {
      const uint32_t s = static_cast<const uint8_t*>(p.a_shared)[idx];
      const uint32_t m3 = (s >> 4) & 7u;
      emax = (int)(s & 0xFu) + p.a_ebias;
      mk = (int)(m3 | (m3 << 8) | (m3 << 16) | (m3 << 24));
    } else {
      const uint32_t s = static_cast<const uint16_t*>(p.a_shared)[idx];
      emax = (int)(s & 0xFu) + p.a_ebias;
      mk = (int)(((s >> 4) & 7u) | (((s >> 7) & 7u) << 8) | (((s >> 10) & 7u) << 16) | (((s >> 13) & 7u) << 24));
    }
    ash[m * nbc_max + b] = make_int2(emax, mk);
  }
  __syncthreads();

  const int tpn = p.tpn;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sub = lane % tpn;
  const int64_t n = (int64_t)blockIdx.x * (kThreads / tpn) + warp * (32 / tpn) + lane / tpn;
  const int cB = p.b_fp4 ? 1 : 2;
  float acc[kMaxM];
#pragma unroll
  for (int m = 0; m < kMaxM; ++m) acc[m] = 0.0f;
  if (n < p.N) {
    const int64_t gb = bt / p.b_group;
    const uint8_t* brow = p.b_codes + (gb * p.b_bs + n * p.b_ld + k0) / 2;
    const uint8_t* bsc = p.b_scales + (gb * p.b_bs + n * p.b_ld + k0) / (G16 ? 16 : 32);
    for (int b = sub; b < nbc; b += tpn) {
      const uint4 cw = *reinterpret_cast<const uint4*>(brow + b * 16);
      const int X = (int)bsc[G16 ? 2 * b : b] - 127;
      const int X1 = G16 ? (int)bsc[2 * b + 1] - 127 : 0;
      // the block's 32 weights as int8, four per word (element order)
      const DecTab tb = p.b_fp4 ? fp4_int8_tab() : int4_int8_tab();
      const uint2 bw[4] = {dec8(cw.x, tb), dec8(cw.y, tb), dec8(cw.z, tb), dec8(cw.w, tb)};
#pragma unroll
      for (int m = 0; m < kMaxM; ++m) {
        if (m < p.M) {
          const int16_t* f = fa + (m * nbc_max + b) * 32;
          const int2 sh = ash[m * nbc_max + b];
          int blockv = 0, half0 = 0;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int4 f0 = *reinterpret_cast<const int4*>(f + 8 * q);
            const int fw[4] = {f0.x, f0.y, f0.z, f0.w};
            // one 8-way shift-add sub-tree: four 2-way 16 x 8-bit dot products
            int S = __dp2a_lo(fw[0], (int)bw[q].x, 0);
            S = __dp2a_hi(fw[1], (int)bw[q].x, S);
            S = __dp2a_lo(fw[2], (int)bw[q].y, S);
            S = __dp2a_hi(fw[3], (int)bw[q].y, S);
            blockv += S * (8 + ((sh.y >> (8 * q)) & 0xFF));  // x (1.mshared_k) in eighths
            if (G16 && q == 1) {
              half0 = blockv;
              blockv = 0;
            }
          }
          if (G16) {
            acc[m] += ldexpf((float)half0, sh.x + X - 10 - cB);
            acc[m] += ldexpf((float)blockv, sh.x + X1 - 10 - cB);
          } else {
            acc[m] += ldexpf((float)blockv, sh.x + X - 10 - cB);  // one exponent add
          }
        }
      }
    }
  }
  // Reduce the tpn lanes that share n (fixed butterfly order).
  for (int off = 1; off < tpn; off <<= 1) {
#pragma unroll
    for (int m = 0; m < kMaxM; ++m) acc[m] += __shfl_xor_sync(0xFFFFFFFFu, acc[m], off);
  }
  if (n < p.N && sub == 0) {
    float* o = p.out + split * p.out_split_stride + bt * p.out_bs + n;
#pragma unroll
    for (int m = 0; m < kMaxM; ++m)
      if (m < p.M) o[m * p.out_ld] = acc[m];
  }
}

__global__ void gemv_reduce_kernel(const float* __restrict__ part, int64_t splits, int64_t split_stride,
                                   int64_t batch, int64_t M, int64_t N, float* __restrict__ c,
                                   int64_t ldc, int64_t cbs) {
  const int64_t total = batch * M * N;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    float acc = 0.0f;
    for (int64_t s = 0; s < splits; ++s) acc += part[s * split_stride + i];
    const int64_t bt = i / (M * N), r = i - bt * M * N, m = r / N, n = r - m * N;
    c[bt * cbs + m * ldc + n] = acc;
  }
}

struct Plan {
  int tpn;
  int64_t kc, splits;
  size_t part_bytes, c_bytes;
};

Plan make_plan(const mix_gemm_desc_t& d) {
  Plan pl{};
  const int64_t nb = d.K / 32;
  // Chunk length: bounded by shared memory (16 rows x 2048 x 2 B = 64 KB).
  int64_t kc = d.K < 2048 ? d.K : 2048;
  int64_t splits = (d.K + kc - 1) / kc;
  // Split K further while the grid would leave most SMs idle (one warp per n).
  const int64_t ctas = ((d.N + 7) / 8) * d.batch;
  while (ctas * splits < 2 * (int64_t)num_sms() && kc > 256 && (kc / 2) % 32 == 0) {
    kc /= 2;
    splits = (d.K + kc - 1) / kc;
  }
  // Lanes per output column: enough to cover the chunk's blocks, at most 32.
  int tpn = 32;
  while (tpn > 1 && tpn / 2 >= kc / 32) tpn >>= 1;
  (void)nb;
  pl.tpn = tpn;
  pl.kc = kc;
  pl.splits = splits;
  pl.part_bytes = splits > 1 ? (size_t)splits * d.batch * d.M * d.N * sizeof(float) : 0;
  pl.c_bytes = (d.c == nullptr && d.epi != MIX_EPI_NONE) ? (size_t)d.batch * d.M * d.N * sizeof(float) : 0;
  return pl;
}

}  // namespace

size_t gemv_workspace_bytes(const mix_gemm_desc_t& d) {
  const Plan pl = make_plan(d);
  return pl.part_bytes + pl.c_bytes;
}

cudaError_t launch_gemv_shiftadd(const mix_gemm_desc_t& d, void* ws, cudaStream_t st) {
  const Plan pl = make_plan(d);
  float* cbuf = d.c;
  int64_t ldc = d.ldc, cbs = d.c_batch_stride;
  char* wsb = static_cast<char*>(ws);
  if (cbuf == nullptr) {  // epilogue only: C lives in the workspace, dense
    cbuf = reinterpret_cast<float*>(wsb + pl.part_bytes);
    ldc = d.N;
    cbs = d.M * d.N;
  }
  GemvArgs p{};
  p.a_codes = d.a_codes; p.a_shared = d.a_shared; p.b_codes = d.b_codes; p.b_scales = d.b_scales;
  p.M = d.M; p.N = d.N; p.K = d.K; p.b_group = d.b_group;
  p.a_ld = d.a_ld; p.a_bs = d.a_batch_stride; p.b_ld = d.b_ld; p.b_bs = d.b_batch_stride;
  p.kc = pl.kc; p.a_type = (int)d.a_type; p.a_ebias = d.a_ebias; p.b_fp4 = d.b_type == MX_FP4_E2M1;
  p.tpn = pl.tpn;
  if (pl.splits > 1) {
    p.out = reinterpret_cast<float*>(wsb);
    p.out_ld = d.N; p.out_bs = d.M * d.N; p.out_split_stride = d.batch * d.M * d.N;
  } else {
    p.out = cbuf; p.out_ld = ldc; p.out_bs = cbs; p.out_split_stride = 0;
  }
  const size_t smem = (size_t)d.M * (pl.kc / 32) * (32 * sizeof(int16_t) + sizeof(int2));
  const bool g16 = b_g16(d);
  if (smem > 48 * 1024) {
    cudaError_t e = g16 ? cudaFuncSetAttribute(gemv_shiftadd_kernel<true>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)
                        : cudaFuncSetAttribute(gemv_shiftadd_kernel<false>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  const dim3 grid((unsigned)((d.N + (kThreads / pl.tpn) - 1) / (kThreads / pl.tpn)), (unsigned)pl.splits,
                  (unsigned)d.batch);
  if (g16) gemv_shiftadd_kernel<true><<<grid, kThreads, smem, st>>>(p);
  else gemv_shiftadd_kernel<false><<<grid, kThreads, smem, st>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (pl.splits > 1) {
    const int64_t total = d.batch * d.M * d.N;
    int64_t g = (total + 255) / 256;
    if (g > (int64_t)num_sms() * 8) g = (int64_t)num_sms() * 8;
    gemv_reduce_kernel<<<(unsigned)(g > 0 ? g : 1), 256, 0, st>>>(p.out, pl.splits, p.out_split_stride,
                                                                 d.batch, d.M, d.N, cbuf, ldc, cbs);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (d.epi != MIX_EPI_NONE) {  // quantise the fp32 rows, as mix/mx_quantize would
    for (int64_t bt = 0; bt < d.batch; ++bt) {
      const float* cb = cbuf + bt * cbs;
      uint8_t* oc = d.out_codes + bt * d.out_batch_stride / 2;
      if (d.epi == MIX_EPI_MIX_T1 || d.epi == MIX_EPI_MIX_T2) {
        const int t = d.epi == MIX_EPI_MIX_T1 ? 1 : 2;
        void* os = static_cast<char*>(d.out_shared) + (bt * d.out_batch_stride / 32) * (t == 1 ? 1 : 2);
        e = launch_mix_quantize(cb, false, d.M, d.N, ldc, t, d.epi_ebias, (d.epi_flags & MIX_ASYM_ZERO) != 0,
                                oc, os, st);
      } else {
        uint8_t* os = static_cast<uint8_t*>(d.out_shared) + bt * d.out_batch_stride / 32;
        e = launch_mx_quantize_rows(cb, false, d.M, d.N, ldc, d.epi == MIX_EPI_MXFP4,
                                    mx_rule_of(d.epi_flags), false, oc, os, st);
      }
      if (e != cudaSuccess) return e;
    }
  }
  return cudaSuccess;
}

}  // namespace mixk
