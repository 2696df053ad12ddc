// Staging pass of the tensor-core matmul: each operand is expanded ONCE per
// call into exact e4m3 bytes plus UE8M0 block-scale words in the caller's
// workspace, so that the matmul's main loop is TMA -> tcgen05.st of the
// scale words -> MMA with no per-tile decode.  Without it every CTA of a row panel re-decodes the same
// A tile (N / 256 times for a wide layer).
//
// The arithmetic is the decode of "MiX: Micro-Inverted-Scaling for End-to-End
// Low-Bit Vision-Language Model Acceleration" (pchao.org digest, section
// "Method", dual-format matmul bullet): MiX element -> +-(1.m3) 2^(1 - de)
// with block scale 2^(Emax - 1); MX element -> (q / 4) or its E2M1 value with
// block scale 2^X.  Every value is exact in e4m3 and every scale exact in
// UE8M0, so the expanded operands multiply to the same products as Eq. (6).
#include <cuda_runtime.h>

#include <cstdint>

#include "decode.cuh"
#include "mix_common.cuh"
#include "mix_internal.h"

namespace mixk {

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ uint32_t quad_or(uint32_t v) {
  v |= __shfl_xor_sync(0xFFFFFFFFu, v, 1);
  v |= __shfl_xor_sync(0xFFFFFFFFu, v, 2);
  return v;
}

// One thread per 32-element block of a (padded) row of A.  Rows run to the
// last full 128-row tile so every scale word of the tile is written; only
// rows < M get e4m3 bytes (the matmul's TMA zero-fills rows >= M).  Warps
// iterate in lockstep (the trip count is rounded to the warp) so the quad
// shuffles that assemble a scale word always see all 32 lanes.
template <int TYPE>
__global__ void __launch_bounds__(kThreads) expand_a_kernel(const uint8_t* __restrict__ codes,
                                                            const void* __restrict__ shared, int64_t M,
                                                            int64_t K, int64_t a_ld, int64_t a_bs, int ebias,
                                                            int64_t batch, int64_t k_pad, int64_t mt, int64_t kt_n,
                                                            FastDiv f_kbp, FastDiv f_rows,
                                                            uint8_t* __restrict__ a_e4m3, uint32_t* __restrict__ sfa,
                                                            uint32_t* __restrict__ clear, int nclear) {
  const int64_t kbv = K / 32;
  // the matmul's split-part flags start at zero (the matmul runs after this
  // pass on the same stream)
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < nclear; i += gridDim.x * blockDim.x) clear[i] = 0u;
  const uint32_t total = (uint32_t)(batch * (int64_t)f_rows.d * f_kbp.d);
  const uint32_t total_w = (total + 31u) & ~31u;
  const uint32_t stride = gridDim.x * blockDim.x;
  const unsigned char* tabs;
  __shared__ uint4 tab_s[8];
  if (threadIdx.x < 8) {
    const DecTab t = mix_tab(threadIdx.x);
    tab_s[threadIdx.x] = make_uint4(t.plo, t.phi, t.nlo, t.nhi);
  }
  __syncthreads();
  tabs = reinterpret_cast<const unsigned char*>(tab_s);
  auto tab = [&](uint32_t m3) {
    const uint4 t = *reinterpret_cast<const uint4*>(tabs + 16 * m3);
    return DecTab{t.x, t.y, t.z, t.w};
  };
  for (uint32_t t = blockIdx.x * blockDim.x + threadIdx.x; t < total_w; t += stride) {
    const bool valid = t < total;
    const uint32_t rr = fdiv(t, f_kbp), kb = t - rr * f_kbp.d;
    const uint32_t b = fdiv(rr, f_rows), r = rr - b * f_rows.d;
    uint32_t sbyte = 127u;
    if (valid && r < M) {
      uint4 out0 = make_uint4(0, 0, 0, 0), out1 = make_uint4(0, 0, 0, 0);
      if (kb < kbv) {
        const int64_t e = (int64_t)b * a_bs + (int64_t)r * a_ld + 32 * (int64_t)kb;
        const uint4 cv = __ldg(reinterpret_cast<const uint4*>(codes + e / 2));
        const uint32_t sh = TYPE == 1 ? (uint32_t)__ldg(static_cast<const uint8_t*>(shared) + e / 32)
                                      : (uint32_t)__ldg(static_cast<const uint16_t*>(shared) + e / 32);
        uint2 d0, d1, d2, d3;
        if (TYPE == 1) {
          const DecTab tt = tab((sh >> 4) & 7u);
          d0 = dec8(cv.x, tt); d1 = dec8(cv.y, tt); d2 = dec8(cv.z, tt); d3 = dec8(cv.w, tt);
        } else {
          d0 = dec8(cv.x, tab((sh >> 4) & 7u));
          d1 = dec8(cv.y, tab((sh >> 7) & 7u));
          d2 = dec8(cv.z, tab((sh >> 10) & 7u));
          d3 = dec8(cv.w, tab((sh >> 13) & 7u));
        }
        out0 = make_uint4(d0.x, d0.y, d1.x, d1.y);
        out1 = make_uint4(d2.x, d2.y, d3.x, d3.y);
        const int emax = (int)(sh & 0xFu) + ebias;
        sbyte = (uint32_t)clampi(emax + 126, 1, 254);  // 2^(Emax - 1)
      }
      uint4* dst = reinterpret_cast<uint4*>(a_e4m3 + ((int64_t)b * M + r) * k_pad + 32 * (int64_t)kb);
      dst[0] = out0;
      dst[1] = out1;
    }
    // scale word of (row r, k-step kb / 4): byte kb % 4, assembled across the quad
    const uint32_t word = quad_or(sbyte << (8 * (kb & 3u)));
    if (valid && (kb & 3u) == 0) {
      const int64_t tile = r >> 7, rin = r & 127;
      const int64_t idx = (((int64_t)b * mt + tile) * kt_n + (kb >> 2)) * 128 + (rin & 31) * 4 + (rin >> 5);
      sfa[idx] = word;
    }
  }
}

// B: MX plane -> e4m3 of q / 4 (MXINT4) or the E2M1 value, and the MX scale
// bytes regrouped into tiles of `tile_rows` (<= 256) rows, each stored as a
// 256-row group (two 128-row halves; the words of rows tile_rows .. 255 are
// padding and hold scale 1).  Threads walk the padded 256-row index space.
//
// G16 (MXINT4g16 / MXFP4g16, one scale per 16 elements): the matmul takes one
// UE8M0 scale per 32-deep block, so each block gets S = max(X0, X1) - C and
// each half's elements are stored multiplied by 2^(X_h - S) (C = 7 for
// MXINT4, 6 for MXFP4: the larger half's largest element still fits e4m3).
// A half whose exponent is within 14 binades of the other's stays exact; a
// farther one is rounded to the nearest e4m3 subnormal.  The per-block S
// bytes also go to `eff_scales` ([bb][N][k_pad / 32]) when it is given, for
// the fused-decode matmul, which reads block scale bytes directly.
constexpr int kG16ShiftMin = -24, kG16Shifts = 32;  // shifts -24 .. 7; -24 already zeroes every code

template <bool FP4, bool G16>
__global__ void __launch_bounds__(kThreads) expand_b_kernel(const uint8_t* __restrict__ codes,
                                                            const uint8_t* __restrict__ scales, int64_t N,
                                                            int64_t K, int64_t b_ld, int64_t b_bs, int64_t bb,
                                                            int64_t k_pad, int tile_rows, int64_t kt_n,
                                                            FastDiv f_kbp, FastDiv f_rows,
                                                            uint8_t* __restrict__ b_e4m3, uint32_t* __restrict__ sfb,
                                                            uint8_t* __restrict__ eff_scales) {
  const int64_t kbv = K / 32;
  const uint32_t total = (uint32_t)(bb * (int64_t)f_rows.d * f_kbp.d);
  const uint32_t total_w = (total + 31u) & ~31u;
  const uint32_t stride = gridDim.x * blockDim.x;
  const int64_t nt = f_rows.d / 256;
  const DecTab tt = FP4 ? fp4_tab() : int4_tab();
  __shared__ __align__(16) uint8_t g16_tab[G16 ? kG16Shifts * 16 : 16];
  if (G16) {
    for (int i = threadIdx.x; i < kG16Shifts * 16; i += blockDim.x)
      g16_tab[i] = (uint8_t)mx_scaled_entry(i & 15, FP4, kG16ShiftMin + (i >> 4));
    __syncthreads();
  }
  for (uint32_t t = blockIdx.x * blockDim.x + threadIdx.x; t < total_w; t += stride) {
    const bool valid = t < total;
    const uint32_t rr = fdiv(t, f_kbp), kb = t - rr * f_kbp.d;
    const uint32_t b = fdiv(rr, f_rows), vr = rr - b * f_rows.d;   // padded row
    const uint32_t tile = vr >> 8, rin = vr & 255u;
    const int64_t r = (int64_t)tile * tile_rows + rin;              // matrix row
    uint32_t sbyte = 127u;
    if (valid && (int)rin < tile_rows && r < N) {
      uint4 out0 = make_uint4(0, 0, 0, 0), out1 = make_uint4(0, 0, 0, 0);
      if (kb < kbv) {
        const int64_t e = (int64_t)b * b_bs + r * b_ld + 32 * (int64_t)kb;
        const uint4 cv = __ldg(reinterpret_cast<const uint4*>(codes + e / 2));
        if (G16) {
          const int x0 = (int)__ldg(scales + e / 16), x1 = (int)__ldg(scales + e / 16 + 1);  // biased
          const int s = max(max(x0, x1) - (FP4 ? 6 : 7), 0);
          sbyte = (uint32_t)s;
          const uint4 t0 = *reinterpret_cast<const uint4*>(g16_tab + 16 * (max(x0 - s, kG16ShiftMin) - kG16ShiftMin));
          const uint4 t1 = *reinterpret_cast<const uint4*>(g16_tab + 16 * (max(x1 - s, kG16ShiftMin) - kG16ShiftMin));
          const DecTab h0{t0.x, t0.y, t0.z, t0.w}, h1{t1.x, t1.y, t1.z, t1.w};
          const uint2 d0 = dec8(cv.x, h0), d1 = dec8(cv.y, h0), d2 = dec8(cv.z, h1), d3 = dec8(cv.w, h1);
          out0 = make_uint4(d0.x, d0.y, d1.x, d1.y);
          out1 = make_uint4(d2.x, d2.y, d3.x, d3.y);
        } else {
          sbyte = (uint32_t)__ldg(scales + e / 32);
          const uint2 d0 = dec8(cv.x, tt), d1 = dec8(cv.y, tt), d2 = dec8(cv.z, tt), d3 = dec8(cv.w, tt);
          out0 = make_uint4(d0.x, d0.y, d1.x, d1.y);
          out1 = make_uint4(d2.x, d2.y, d3.x, d3.y);
        }
      }
      uint4* dst = reinterpret_cast<uint4*>(b_e4m3 + ((int64_t)b * N + r) * k_pad + 32 * (int64_t)kb);
      dst[0] = out0;
      dst[1] = out1;
      if (G16 && eff_scales != nullptr) eff_scales[((int64_t)b * N + r) * (k_pad / 32) + kb] = (uint8_t)sbyte;
    }
    const uint32_t word = quad_or(sbyte << (8 * (kb & 3u)));
    if (valid && (kb & 3u) == 0) {
      const uint32_t h = rin >> 7, rq = rin & 127u;
      const int64_t idx = ((((int64_t)b * nt + tile) * kt_n + (kb >> 2)) * 2 + h) * 128 + (rq & 31) * 4 + (rq >> 5);
      sfb[idx] = word;
    }
  }
}

// Scales only (MXFP4 weights read in place): one thread per 32-bit scale
// word, i.e. per (row, 128-deep k-step) of the padded 256-row groups; the
// k-step runs fastest so the four scale bytes are read contiguously.
__global__ void __launch_bounds__(kThreads) b_scales_kernel(const uint8_t* __restrict__ scales, int64_t N,
                                                            int64_t K, int64_t b_ld, int64_t b_bs, int64_t bb,
                                                            int tile_rows, int64_t kt_n, FastDiv f_kt,
                                                            FastDiv f_rows, uint32_t* __restrict__ sfb) {
  const int64_t kbv = K / 32;
  const uint32_t total = (uint32_t)(bb * (int64_t)f_rows.d * f_kt.d);
  const int64_t nt = f_rows.d / 256;
  for (uint32_t t = blockIdx.x * blockDim.x + threadIdx.x; t < total; t += gridDim.x * blockDim.x) {
    const uint32_t rr = fdiv(t, f_kt), kt = t - rr * f_kt.d;
    const uint32_t b = fdiv(rr, f_rows), vr = rr - b * f_rows.d;
    const uint32_t tile = vr >> 8, rin = vr & 255u;
    const int64_t r = (int64_t)tile * tile_rows + rin;
    uint32_t word = 0x7F7F7F7Fu;
    if ((int)rin < tile_rows && r < N) {
      const uint8_t* src = scales + ((int64_t)b * b_bs + r * b_ld) / 32;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int64_t kb = 4 * (int64_t)kt + j;
        if (kb < kbv) word = (word & ~(0xFFu << (8 * j))) | ((uint32_t)__ldg(src + kb) << (8 * j));
      }
    }
    const uint32_t h = rin >> 7, rq = rin & 127u;
    sfb[((((int64_t)b * nt + tile) * kt_n + kt) * 2 + h) * 128 + (rq & 31) * 4 + (rq >> 5)] = word;
  }
}

int grid_for(int64_t threads) {
  const int64_t cap = (int64_t)num_sms() * 8;
  int64_t g = (threads + kThreads - 1) / kThreads;
  if (g > cap) g = cap;
  return (int)(g < 1 ? 1 : g);
}

size_t align_up(size_t v) { return (v + kStagedAlign - 1) / kStagedAlign * kStagedAlign; }

}  // namespace

bool staged_fp4_native_ok(const mix_gemm_desc_t& d) {
  if (d.b_type != MX_FP4_E2M1 || d.K % 128 != 0 || b_g16(d)) return false;
  if ((reinterpret_cast<uintptr_t>(d.b_codes) & 31) != 0 || (d.b_ld / 2) % 32 != 0) return false;
  const int64_t bb = (d.batch + d.b_group - 1) / d.b_group;
  if (bb > 1 && (d.b_batch_stride / 2) % 32 != 0) return false;
  return true;
}

StagedPlan staged_plan(const mix_gemm_desc_t& d) {
  StagedPlan sp{};
  sp.b_native = staged_fp4_native_ok(d);
  sp.k_pad = (d.K + 127) / 128 * 128;
  sp.kt = sp.k_pad / 128;
  sp.mt = (d.M + 127) / 128;
  sp.nt = (d.N + kStagedBN - 1) / kStagedBN;
  sp.bb = (d.batch + d.b_group - 1) / d.b_group;
  // the schedule: split the last partial wave along K when that shortens it
  // by more than the cost of passing the parts (about four k-steps).  Only
  // long K loops gain: measured on this part, the split took the 18944-deep
  // down projection from 0.270 to 0.252 ms but made 3584- and 5120-deep
  // calls 2-6 % slower (a partial last wave of whole tiles runs faster per
  // k-step than a full one).
  const int64_t tiles = d.batch * sp.mt * sp.nt, P = num_sms();
  sp.grid = (int)(tiles < P ? tiles : P);
  sp.split = 0;
  sp.nd = 0;
  sp.sk_tile0 = 0;
  sp.sk_len = 0;
  if (tiles > 0 && sp.kt >= 64) {
    const int64_t nd = tiles / P, R = tiles - nd * P;
    if (R > 0 && R * sp.kt >= 2 * P && R * sp.kt + 4 * P <= sp.kt * P) {
      sp.grid = (int)P;
      sp.split = 1;
      sp.nd = (int)nd;
      sp.sk_tile0 = nd * P;
      sp.sk_len = R * sp.kt;
    }
  }
  size_t off = 0;
  sp.off_a = off;
  off = align_up(off + (size_t)d.batch * d.M * sp.k_pad);
  sp.off_sfa = off;
  off = align_up(off + (size_t)d.batch * sp.mt * sp.kt * 512);
  sp.off_sk = off;
  if (sp.split) off = align_up(off + (size_t)sp.grid * (kSkSlotBytes + kSkFlags * 4));
  sp.off_b = off;
  if (!sp.b_native) off = align_up(off + (size_t)sp.bb * d.N * sp.k_pad);
  sp.off_sfb = off;
  off = align_up(off + (size_t)sp.bb * sp.nt * sp.kt * 1024);
  sp.off_sfe = off;
  sp.bytes = off;
  return sp;
}

StagedPlan staged_plan_b_only(const mix_gemm_desc_t& d) {
  StagedPlan sp = staged_plan(d);
  sp.b_native = false;
  sp.split = 0;
  size_t off = 0;
  sp.off_a = sp.off_sfa = sp.off_sk = 0;
  sp.off_b = off;
  off = align_up(off + (size_t)sp.bb * d.N * sp.k_pad);
  sp.off_sfb = off;
  off = align_up(off + (size_t)sp.bb * sp.nt * sp.kt * 1024);
  sp.off_sfe = off;
  if (b_g16(d)) off = align_up(off + (size_t)sp.bb * d.N * (sp.k_pad / 32));  // per-block S bytes
  sp.bytes = off;
  return sp;
}

// Thread counts of the two passes; the staged path is taken only when both
// index spaces fit 32 bits.
int64_t expand_a_threads(const mix_gemm_desc_t& d, const StagedPlan& sp) { return d.batch * sp.mt * 128 * (sp.k_pad / 32); }
int64_t expand_b_threads(const StagedPlan& sp) { return sp.bb * sp.nt * 256 * (sp.k_pad / 32); }

cudaError_t launch_expand_a(const mix_gemm_desc_t& d, const StagedPlan& sp, unsigned char* base, cudaStream_t st) {
  const int64_t threads = expand_a_threads(d, sp);
  const FastDiv fk = make_fastdiv((uint32_t)(sp.k_pad / 32)), fr = make_fastdiv((uint32_t)(sp.mt * 128));
  uint8_t* a = base + sp.off_a;
  uint32_t* sfa = reinterpret_cast<uint32_t*>(base + sp.off_sfa);
  uint32_t* flags = sp.split ? reinterpret_cast<uint32_t*>(base + sp.off_sk + (size_t)sp.grid * kSkSlotBytes) : nullptr;
  const int nflags = sp.split ? sp.grid * kSkFlags : 0;
  if (d.a_type == MIX_T1_4P25)
    expand_a_kernel<1><<<grid_for(threads), kThreads, 0, st>>>(d.a_codes, d.a_shared, d.M, d.K, d.a_ld,
                                                               d.a_batch_stride, d.a_ebias, d.batch, sp.k_pad,
                                                               sp.mt, sp.kt, fk, fr, a, sfa, flags, nflags);
  else
    expand_a_kernel<2><<<grid_for(threads), kThreads, 0, st>>>(d.a_codes, d.a_shared, d.M, d.K, d.a_ld,
                                                               d.a_batch_stride, d.a_ebias, d.batch, sp.k_pad,
                                                               sp.mt, sp.kt, fk, fr, a, sfa, flags, nflags);
  return cudaGetLastError();
}

cudaError_t launch_expand_b(const mix_gemm_desc_t& d, const StagedPlan& sp, unsigned char* base, cudaStream_t st) {
  const int64_t threads = expand_b_threads(sp);
  const FastDiv fk = make_fastdiv((uint32_t)(sp.k_pad / 32)), fr = make_fastdiv((uint32_t)(sp.nt * 256));
  const int tr = kStagedBN;
  uint8_t* b = base + sp.off_b;
  uint32_t* sfb = reinterpret_cast<uint32_t*>(base + sp.off_sfb);
  const int g = grid_for(threads);
  const int64_t bs = sp.bb > 1 ? d.b_batch_stride : 0;
  if (sp.b_native) {
    const int64_t words = sp.bb * sp.nt * 256 * sp.kt;
    b_scales_kernel<<<grid_for(words), kThreads, 0, st>>>(d.b_scales, d.N, d.K, d.b_ld, bs, sp.bb, tr, sp.kt,
                                                          make_fastdiv((uint32_t)sp.kt), fr, sfb);
    return cudaGetLastError();
  }
  // the per-block scale bytes exist only in a B-only plan with g16 weights
  uint8_t* sfe = (b_g16(d) && sp.bytes > sp.off_sfe) ? base + sp.off_sfe : nullptr;
#define EXPAND_B(FP4, G16)                                                                                   \
  expand_b_kernel<FP4, G16><<<g, kThreads, 0, st>>>(d.b_codes, d.b_scales, d.N, d.K, d.b_ld, bs, sp.bb, sp.k_pad, \
                                                    tr, sp.kt, fk, fr, b, sfb, sfe)
  if (d.b_type == MX_FP4_E2M1) {
    if (b_g16(d)) EXPAND_B(true, true);
    else EXPAND_B(true, false);
  } else {
    if (b_g16(d)) EXPAND_B(false, true);
    else EXPAND_B(false, false);
  }
#undef EXPAND_B
  return cudaGetLastError();
}

}  // namespace mixk
