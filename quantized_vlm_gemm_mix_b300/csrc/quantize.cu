// MiX and MX quantiser kernels (sm_103a).
//
// MiX (Algorithm 1, Method section of the pchao.org digest of "MiX:
// Micro-Inverted-Scaling ..."): one thread owns one 32-element block (four
// 16-byte loads of bf16, eight of fp32), computes the block's Emax and
// mshared once, codes the 32 elements with integer compares on their fp32
// bit patterns and stores 16 code bytes; a warp's stores are 512 contiguous
// bytes.  MX along rows: four lanes per block, eight elements each, the block
// maximum by two butterfly shuffles.
//
// The kernels are HBM-bound: a bf16 element costs 2 bytes in and 0.53125
// (T1) / 0.5625 (T2) bytes out.  Each thread keeps two blocks in flight and
// the grid is a multiple of the SM count.
#include <cuda_runtime.h>

#include <atomic>

#include "mix_common.cuh"
#include "mix_internal.h"

namespace mixk {

// SM count of the current device, looked up once per device.  Host threads
// may call this concurrently: each entry is an atomic, and a race only makes
// two threads store the same value.
int num_sms() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

namespace {

constexpr int kThreads = 256;
constexpr int kQuadsPerCta = kThreads / 4;
constexpr int kUnroll = 2;

// Eight consecutive elements as fp32 bit patterns.
template <bool BF16>
__device__ __forceinline__ void load8(const void* base, int64_t elem, uint32_t* u) {
  if (BF16) {
    uint4 v = __ldcs(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + elem));
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      u[2 * i] = w[i] << 16;
      u[2 * i + 1] = w[i] & 0xFFFF0000u;
    }
  } else {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const float*>(base) + elem);
    uint4 a = __ldcs(p), b = __ldcs(p + 1);
    u[0] = a.x; u[1] = a.y; u[2] = a.z; u[3] = a.w;
    u[4] = b.x; u[5] = b.y; u[6] = b.z; u[7] = b.w;
  }
}

__device__ __forceinline__ uint32_t pair_max(uint32_t v) {
  return max(v, __shfl_xor_sync(0xFFFFFFFFu, v, 1));
}

__device__ __forceinline__ uint32_t quad_max(uint32_t v) {
  v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, 1));
  return max(v, __shfl_xor_sync(0xFFFFFFFFu, v, 2));
}

// One thread per 32-element block: the block's parameters are computed once
// and no lane exchange is needed.  |x| is formed once per element and feeds
// both the block maximum and the element decision; a block holding a NaN
// (rare) takes a slow path that codes the NaNs as zero first.
template <bool BF16>
__device__ __forceinline__ void load32(const void* base, int64_t elem, uint32_t* u) {
  if (BF16) {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + elem);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 v = p[j];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        u[8 * j + 2 * i] = w[i] << 16;
        u[8 * j + 2 * i + 1] = w[i] & 0xFFFF0000u;
      }
    }
  } else {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const float*>(base) + elem);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint4 v = p[j];
      u[4 * j] = v.x; u[4 * j + 1] = v.y; u[4 * j + 2] = v.z; u[4 * j + 3] = v.w;
    }
  }
}

// DEV_EB: ebias is read from device memory (the automatic two-pass mode), in
// its own instantiation so the fixed-ebias kernel keeps ebias in the
// parameter bank rather than in a register.
template <bool BF16, int TYPE, bool DEV_EB>
__global__ void __launch_bounds__(kThreads, 4) mix_quantize_kernel(
    const void* __restrict__ x, int64_t rows, int64_t nb, int64_t ld, int ebias, int asym,
    uint8_t* __restrict__ codes, void* __restrict__ shared, FastDiv fnb, const int* __restrict__ ebias_dev) {
  if (DEV_EB) ebias = *ebias_dev;
  const int64_t total = rows * nb;
  for (int64_t g = (int64_t)blockIdx.x * kThreads + threadIdx.x; g < total; g += (int64_t)gridDim.x * kThreads) {
    const uint32_t row = fdiv((uint32_t)g, fnb);
    const int64_t b = g - (int64_t)row * nb;
    uint4 cw;
    uint32_t sh;
    if (BF16) {  // packed step: two elements per integer operation
      const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(x) + (int64_t)row * ld + b * 32);
      uint32_t w[16];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 v = p[j];
        w[4 * j] = v.x; w[4 * j + 1] = v.y; w[4 * j + 2] = v.z; w[4 * j + 3] = v.w;
      }
      mix_block32_bf16<TYPE>(w, ebias, asym != 0, cw, sh);
    } else {
      uint32_t u[32];
      load32<BF16>(x, (int64_t)row * ld + b * 32, u);
      mix_block32<TYPE>(u, ebias, asym != 0, cw, sh);
    }
    __stcs(reinterpret_cast<uint4*>(codes + g * 16), cw);
    if (TYPE == 1) static_cast<uint8_t*>(shared)[g] = (uint8_t)sh;
    else static_cast<uint16_t*>(shared)[g] = (uint16_t)sh;
  }
}

// NVFP4 (a comparison format: 16-element blocks of E2M1, an E4M3 block scale
// and one fp32 tensor scale).  One thread per 16-element block; every
// decision is an IEEE fp32 operation in the order the definition fixes:
// t = (amax_b / s_t) / 6, its E4M3 code (nearest even, saturating), d =
// e4m3(sb) * s_t, then E2M1 of x / d.  s_t comes from the tensor's largest
// finite |x| (the automatic-ebias reduction), finished in place.
__device__ __forceinline__ uint32_t e4m3_rn_satfinite(float t) {
  uint32_t r;
  asm("{\n\t.reg .b16 h;\n\tcvt.rn.satfinite.e4m3x2.f32 h, %1, %2;\n\tcvt.u32.u16 %0, h;\n\t}"
      : "=r"(r)
      : "f"(0.0f), "f"(t));
  return r & 0xFFu;
}

__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {  // b <= 0x7E
  const uint32_t e = (b >> 3) & 15u, m = b & 7u;
  return e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : (float)m * 0x1p-9f;
}

__global__ void nvfp4_scale_finish_kernel(float* __restrict__ ts) {
  if (threadIdx.x != 0) return;
  const uint32_t key = *reinterpret_cast<const unsigned*>(ts);
  float s = 1.0f;
  if (key != 0u) {
    s = __fdiv_rn(__uint_as_float(key), 2688.0f);
    if (s == 0.0f) s = 0x1p-149f;
  }
  *ts = s;
}

template <bool BF16>
__global__ void __launch_bounds__(kThreads) nvfp4_quantize_kernel(const void* __restrict__ x, int64_t rows,
                                                                  int64_t nb, int64_t ld, FastDiv fnb,
                                                                  const float* __restrict__ ts,
                                                                  uint8_t* __restrict__ codes,
                                                                  uint8_t* __restrict__ scales) {
  const float st = *ts;
  const int64_t total = rows * nb;
  for (int64_t g = (int64_t)blockIdx.x * kThreads + threadIdx.x; g < total; g += (int64_t)gridDim.x * kThreads) {
    const uint32_t row = fdiv((uint32_t)g, fnb);
    const int64_t e = (int64_t)row * ld + (g - (int64_t)row * nb) * 16;
    uint32_t u[16];
    load8<BF16>(x, e, u);
    load8<BF16>(x, e + 8, u + 8);
    uint32_t kb = max_abs_bits<16>(u);
    if (kb > 0x7F800000u) {
      zero_nans<16>(u);
      kb = max_abs_bits<16>(u);
    }
    const float t = __fdiv_rn(__fdiv_rn(__uint_as_float(kb), st), 6.0f);
    const uint32_t sb = e4m3_rn_satfinite(t);
    uint2 w = make_uint2(0u, 0u);
    if (sb != 0u) {
      const float d = __fmul_rn(e4m3_to_f32(sb), st);
      uint32_t c[2] = {0u, 0u};
#pragma unroll
      for (int i = 0; i < 8; ++i)
        c[i >> 2] |= e2m1x2(__fdiv_rn(__uint_as_float(u[2 * i]), d), __fdiv_rn(__uint_as_float(u[2 * i + 1]), d))
                     << (8 * (i & 3));
#pragma unroll
      for (int j = 0; j < 2; ++j) {  // -0 (nibble 0x8) -> +0
        const uint32_t tt = c[j] ^ 0x88888888u;
        const uint32_t nz = (tt | (tt >> 1) | (tt >> 2) | (tt >> 3)) & 0x11111111u;
        c[j] &= ~((~nz & 0x11111111u) << 3);
      }
      w = make_uint2(c[0], c[1]);
    }
    __stcs(reinterpret_cast<uint2*>(codes + g * 8), w);
    scales[g] = (uint8_t)sb;
  }
}

// Dead-zone count: finite nonzero inputs whose code is a zero code (MiX 0x7,
// MXINT4 0, E2M1 +-0).  One thread per eight elements (one code word), one
// atomic per warp.
template <bool BF16>
__global__ void __launch_bounds__(kThreads) underflow_count_kernel(const void* __restrict__ x, int64_t rows,
                                                                   int64_t wpr, int64_t ld, FastDiv fw, int fmt,
                                                                   const uint8_t* __restrict__ codes,
                                                                   unsigned long long* __restrict__ count) {
  const int64_t total = rows * wpr;
  unsigned n = 0;
  for (int64_t g = (int64_t)blockIdx.x * kThreads + threadIdx.x; g < total; g += (int64_t)gridDim.x * kThreads) {
    const uint32_t row = fdiv((uint32_t)g, fw);
    const int64_t j = g - (int64_t)row * wpr;
    uint32_t u[8];
    load8<BF16>(x, (int64_t)row * ld + j * 8, u);
    const uint32_t cw = __ldcs(reinterpret_cast<const uint32_t*>(codes) + g);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t a = u[i] & 0x7FFFFFFFu, c = (cw >> (4 * i)) & 0xFu;
      const bool zero = fmt == 0 ? c == 7u : (fmt == 1 ? c == 0u : (c & 7u) == 0u);
      n += (a != 0u && a < 0x7F800000u && zero) ? 1u : 0u;
    }
  }
  n = __reduce_add_sync(0xFFFFFFFFu, n);
  if ((threadIdx.x & 31) == 0 && n != 0u) atomicAdd(count, (unsigned long long)n);
}

// Clamped blocks of the MiX quantiser at `ebias`: one thread per 32-element
// block, the block exponent f of Algorithm 1's first two steps (mantissa
// rounding and carry included); counts[0] += [f > ebias + 15] (+-Inf too),
// counts[1] += [nonzero maximum and f < ebias].  A subnormal maximum is below
// any allowed ebias (>= -100).  NaN counts as zero.  One atomic per warp.
template <bool BF16>
__global__ void __launch_bounds__(kThreads) clamp_count_kernel(const void* __restrict__ x, int64_t rows,
                                                               int64_t nb, int64_t ld, FastDiv fb, int ebias,
                                                               unsigned long long* __restrict__ counts) {
  const int64_t total = rows * nb;
  unsigned hi = 0, lo = 0;
  for (int64_t g = (int64_t)blockIdx.x * kThreads + threadIdx.x; g < total; g += (int64_t)gridDim.x * kThreads) {
    const uint32_t row = fdiv((uint32_t)g, fb);
    const int64_t b = g - (int64_t)row * nb;
    uint32_t u[32];
    load32<BF16>(x, (int64_t)row * ld + b * 32, u);
    uint32_t key = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const uint32_t a = u[i] & 0x7FFFFFFFu;
      key = max(key, a <= 0x7F800000u ? a : 0u);
    }
    if (key == 0u) continue;
    int f = 0, m3 = 0;
    if (!max_exp_mant(key, &f, &m3)) {  // subnormal maximum
      ++lo;
      continue;
    }
    hi += f > ebias + 15 ? 1u : 0u;
    lo += f < ebias ? 1u : 0u;
  }
  hi = __reduce_add_sync(0xFFFFFFFFu, hi);
  lo = __reduce_add_sync(0xFFFFFFFFu, lo);
  if ((threadIdx.x & 31) == 0) {
    if (hi != 0u) atomicAdd(counts, (unsigned long long)hi);
    if (lo != 0u) atomicAdd(counts + 1, (unsigned long long)lo);
  }
}

// Automatic ebias, pass 1: the largest finite |x| of the tensor, as the
// integer maximum of the magnitude bits (the order of non-negative floats).
// Rounding a block maximum to three mantissa bits never lowers a larger one
// below a smaller one, so the largest rounded block exponent is the rounded
// exponent of the global maximum and the pass needs no block structure.
// bf16 pairs are compared two at a time in 16-bit SIMD lanes.  One 16-byte
// vector per load, four in flight per thread, one atomic per warp.
constexpr int kAmaxUnroll = 4;

template <bool BF16>
__global__ void __launch_bounds__(kThreads) amax_bits_kernel(const void* __restrict__ x, int64_t rows,
                                                             int64_t vpr, int64_t ld_bytes, FastDiv fv,
                                                             unsigned* __restrict__ key) {
  const int64_t total = rows * vpr;
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  uint32_t m = 0u;   // fp32 magnitude bits, or two bf16 magnitudes
  for (int64_t g0 = (int64_t)blockIdx.x * kThreads + threadIdx.x; g0 < total; g0 += stride * kAmaxUnroll) {
    uint4 v[kAmaxUnroll];
#pragma unroll
    for (int r = 0; r < kAmaxUnroll; ++r) {
      const int64_t g = g0 + r * stride;
      v[r] = make_uint4(0u, 0u, 0u, 0u);
      if (g < total) {
        const uint32_t row = fdiv((uint32_t)g, fv);
        const int64_t c = g - (int64_t)row * vpr;
        v[r] = __ldg(reinterpret_cast<const uint4*>(static_cast<const char*>(x) + (int64_t)row * ld_bytes + c * 16));
      }
    }
#pragma unroll
    for (int r = 0; r < kAmaxUnroll; ++r) {
      const uint32_t w[4] = {v[r].x, v[r].y, v[r].z, v[r].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (BF16) {
          const uint32_t a = w[i] & 0x7FFF7FFFu;
          m = __vmaxu2(m, a & __vcmpltu2(a, 0x7F807F80u));   // +-Inf and NaN drop out
        } else {
          const uint32_t a = w[i] & 0x7FFFFFFFu;
          m = max(m, a < 0x7F800000u ? a : 0u);
        }
      }
    }
  }
  if (BF16) m = max(m >> 16, m & 0xFFFFu) << 16;
  m = __reduce_max_sync(0xFFFFFFFFu, m);
  if ((threadIdx.x & 31) == 0 && m != 0u) atomicMax(key, m);
}

// Pass 1 finish: key (fp32 magnitude bits of the largest finite |x|, 0 if
// none) -> ebias in place.  The exponent is Algorithm 1's: the significand
// rounded to three fraction bits, nearest-even, a round-up to 2 carrying
// into the exponent (fraction >= 15/16).
__global__ void auto_ebias_finish_kernel(int* __restrict__ ebias) {
  if (threadIdx.x != 0) return;
  const uint32_t key = *reinterpret_cast<const unsigned*>(ebias);
  int e = -8;
  if (key != 0u) {
    const Elem el = split_f32(key);
    const int f = el.f + ((el.sig & 0x7FFFFFu) >= 0x780000u ? 1 : 0);
    e = clampi(f - 15, -100, 100);
  }
  *ebias = e;
}

// G16: a pair of lanes per 16-element block (one scale per pair).
template <bool BF16, bool FP4, bool G16>
__global__ void __launch_bounds__(kThreads, 4) mx_quantize_rows_kernel(
    const void* __restrict__ x, int64_t rows, int64_t nb, int64_t ld, int rule,
    uint8_t* __restrict__ codes, uint8_t* __restrict__ scales, FastDiv fnb) {
  const int q = threadIdx.x & 3;
  const int64_t total = rows * nb;
  const int64_t stride = (int64_t)gridDim.x * kQuadsPerCta;
  for (int64_t base = (int64_t)blockIdx.x * kQuadsPerCta; base < total; base += stride * kUnroll) {
    uint32_t u[kUnroll][8];
    int64_t g[kUnroll];
    uint32_t row[kUnroll] = {0u};
#pragma unroll
    for (int r = 0; r < kUnroll; ++r) {
      g[r] = base + r * stride + (threadIdx.x >> 2);
      if (g[r] < total) {
        row[r] = fdiv((uint32_t)g[r], fnb);
        const int64_t b = g[r] - (int64_t)row[r] * nb;
        load8<BF16>(x, (int64_t)row[r] * ld + b * 32 + q * 8, u[r]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) u[r][i] = 0;
      }
    }
#pragma unroll
    for (int r = 0; r < kUnroll; ++r) {
      uint32_t kb = G16 ? pair_max(max_abs_bits<8>(u[r])) : quad_max(max_abs_bits<8>(u[r]));
      if (__any_sync(0xFFFFFFFFu, kb > 0x7F800000u)) {  // a NaN in some block of the warp
        zero_nans<8>(u[r]);
        kb = G16 ? pair_max(max_abs_bits<8>(u[r])) : quad_max(max_abs_bits<8>(u[r]));
      }
      uint32_t word = 0u, sc = 0u;
      if (kb != 0u) {
        const int X = mx_shared_exp(kb, FP4, rule);
        word = mx_codes8(u[r], X, FP4);
        sc = (uint32_t)(X + 127);
      }
      if (g[r] < total) {
        __stcs(reinterpret_cast<uint32_t*>(codes + g[r] * 16 + q * 4), word);
        if (G16) {
          if ((q & 1) == 0) scales[2 * g[r] + (q >> 1)] = (uint8_t)sc;
        } else if (q == 0) {
          scales[g[r]] = (uint8_t)sc;
        }
      }
    }
  }
}

// axis 0: x is K x N row-major; block kb of column n is x[32kb .. 32kb+31][n].
// A warp owns one k-block and 64 columns (two per lane): every load is a
// contiguous 128-byte (bf16) or 256-byte (fp32) row segment.  The eight warps
// of a CTA own eight consecutive k-blocks, so each column's 128 code bytes are
// written by one CTA.
// bf16 input, 32-element blocks: the same work with the two columns of a
// lane kept packed (one 32-bit word per row) until each column is coded, so
// a thread holds 32 words rather than 64 and four CTAs fit on an SM.  NaNs
// are cleared in the packed words (a 16-bit lane compare per word).
template <bool FP4>
__global__ void __launch_bounds__(kThreads, 4) mx_quantize_cols_bf16_kernel(
    const uint16_t* __restrict__ x, int64_t kdim, int64_t n, int64_t ld, int rule,
    uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
  // The CTA's 64 columns x 8 k-blocks of output are staged in shared memory
  // ([column][k-block], one pad slot per column), then written out whole: a
  // column's codes for the 8 k-blocks are 128 contiguous bytes, its scales 8.
  __shared__ uint4 cs[64][9];
  __shared__ uint8_t ss[64][8];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t nbk = kdim / 32;
  const int64_t kb = (int64_t)blockIdx.y * 8 + warp;
  const int64_t n0 = (int64_t)blockIdx.x * 64 + 2 * lane;
  if (kb < nbk && n0 < n) {
    const bool two = n0 + 1 < n;
    uint32_t v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const uint16_t* p = x + (kb * 32 + i) * ld + n0;
      v[i] = two ? __ldcs(reinterpret_cast<const unsigned int*>(p)) : (uint32_t)__ldcs(p);
    }
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) m = vmax_u16x2(m, v[i] & 0x7FFF7FFFu);
    if (((m & 0xFFFFu) > 0x7F80u) || ((m >> 16) > 0x7F80u)) {  // a NaN in one of the two blocks
      m = 0;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        v[i] &= ~__vcmpgtu2(v[i] & 0x7FFF7FFFu, 0x7F807F80u);
        m = vmax_u16x2(m, v[i] & 0x7FFF7FFFu);
      }
    }
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const uint32_t kbits = c ? (m & 0xFFFF0000u) : (m << 16);
      uint4 w = make_uint4(0u, 0u, 0u, 0u);
      uint32_t sc = 0u;
      if (kbits != 0u) {
        const int X = mx_shared_exp(kbits, FP4, rule);
        uint32_t wd[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t t[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) t[i] = c ? (v[8 * j + i] & 0xFFFF0000u) : (v[8 * j + i] << 16);
          wd[j] = mx_codes8(t, X, FP4);
        }
        w = make_uint4(wd[0], wd[1], wd[2], wd[3]);
        sc = (uint32_t)(X + 127);
      }
      cs[2 * lane + c][warp] = w;
      ss[2 * lane + c][warp] = (uint8_t)sc;
    }
  }
  __syncthreads();
  const int64_t c0 = (int64_t)blockIdx.x * 64, k0 = (int64_t)blockIdx.y * 8;
  for (int i = threadIdx.x; i < 64 * 8; i += blockDim.x) {
    const int cl = i >> 3, kl = i & 7;
    const int64_t col = c0 + cl, kbo = k0 + kl;
    if (col < n && kbo < nbk) {
      *reinterpret_cast<uint4*>(codes + col * (kdim / 2) + kbo * 16) = cs[cl][kl];
      scales[col * nbk + kbo] = ss[cl][kl];
    }
  }
}

template <bool BF16, bool FP4, bool G16>
__global__ void __launch_bounds__(kThreads) mx_quantize_cols_kernel(
    const void* __restrict__ x, int64_t kdim, int64_t n, int64_t ld, int rule,
    uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
  // outputs staged per CTA as in mx_quantize_cols_bf16_kernel: a column's 8
  // k-blocks of codes (128 bytes) and of scales (8, or 16 for g16) contiguous
  constexpr int SPB = G16 ? 2 : 1;  // scale bytes per 32-row block
  __shared__ uint4 cs[64][9];
  __shared__ uint8_t ss[64][8 * SPB];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t nbk = kdim / 32;
  const int64_t kb = (int64_t)blockIdx.y * 8 + warp;
  const int64_t n0 = (int64_t)blockIdx.x * 64 + 2 * lane;
  if (kb < nbk && n0 < n) {
    const bool two = n0 + 1 < n;
    uint32_t u0[32], u1[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int64_t off = (kb * 32 + i) * ld + n0;
      if (BF16) {
        const uint16_t* p = static_cast<const uint16_t*>(x) + off;
        if (two) {
          const uint32_t v = __ldcs(reinterpret_cast<const unsigned int*>(p));
          u0[i] = v << 16;
          u1[i] = v & 0xFFFF0000u;
        } else {
          u0[i] = (uint32_t)__ldcs(p) << 16;
          u1[i] = 0;
        }
      } else {
        const float* p = static_cast<const float*>(x) + off;
        if (two) {
          const float2 v = __ldcs(reinterpret_cast<const float2*>(p));
          u0[i] = __float_as_uint(v.x);
          u1[i] = __float_as_uint(v.y);
        } else {
          u0[i] = __float_as_uint(__ldcs(p));
          u1[i] = 0;
        }
      }
    }
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      uint32_t* u = c ? u1 : u0;
      const int cl = 2 * lane + c;
      if (G16) {
        uint2 w0, w1;
        uint32_t s0, s1;
        mx_block16<FP4>(u, rule, w0, s0);
        mx_block16<FP4>(u + 16, rule, w1, s1);
        cs[cl][warp] = make_uint4(w0.x, w0.y, w1.x, w1.y);
        ss[cl][2 * warp] = (uint8_t)s0;
        ss[cl][2 * warp + 1] = (uint8_t)s1;
      } else {
        uint4 w;
        uint32_t sc;
        mx_block32<FP4>(u, rule, w, sc);
        cs[cl][warp] = w;
        ss[cl][warp] = (uint8_t)sc;
      }
    }
  }
  __syncthreads();
  const int64_t c0 = (int64_t)blockIdx.x * 64, k0 = (int64_t)blockIdx.y * 8;
  for (int i = threadIdx.x; i < 64 * 8; i += blockDim.x) {
    const int cl = i >> 3, kl = i & 7;
    const int64_t col = c0 + cl, kbo = k0 + kl;
    if (col < n && kbo < nbk) {
      *reinterpret_cast<uint4*>(codes + col * (kdim / 2) + kbo * 16) = cs[cl][kl];
#pragma unroll
      for (int j = 0; j < SPB; ++j) scales[(col * nbk + kbo) * SPB + j] = ss[cl][SPB * kl + j];
    }
  }
}

// Test aid: the dequantisation rule (-1)^s (1.mshared)_2 2^(Emax - de).
__global__ void mix_dequant_kernel(const uint8_t* __restrict__ codes, const void* __restrict__ shared,
                                   int64_t rows, int64_t k, int type, int ebias, float* __restrict__ out) {
  const int64_t words = rows * (k / 8);
  for (int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; w < words;
       w += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = w / (k / 8), j = w - row * (k / 8);
    const int64_t blk = row * (k / 32) + j / 4;
    uint32_t ec, m3;
    if (type == 1) {
      const uint32_t s = static_cast<const uint8_t*>(shared)[blk];
      ec = s & 0xF; m3 = (s >> 4) & 7;
    } else {
      const uint32_t s = static_cast<const uint16_t*>(shared)[blk];
      ec = s & 0xF; m3 = (s >> (4 + 3 * (j & 3))) & 7;
    }
    const int emax = (int)ec + ebias;
    const uint32_t cw = reinterpret_cast<const uint32_t*>(codes + row * (k / 2))[j];
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t c = (cw >> (4 * i)) & 0xF;
      const int d = c & 7;
      const float mag = ldexpf((float)(8 + m3), emax - 3 - d);
      v[i] = (d == 7) ? ((c >> 3) ? mag : 0.0f) : ((c >> 3) ? -mag : mag);
    }
    float4* o = reinterpret_cast<float4*>(out + row * k + j * 8);
    o[0] = make_float4(v[0], v[1], v[2], v[3]);
    o[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
}

__global__ void mx_dequant_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales,
                                  int64_t rows, int64_t k, int fp4, float* __restrict__ out) {
  const int64_t words = rows * (k / 8);
  for (int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; w < words;
       w += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = w / (k / 8), j = w - row * (k / 8);
    const int X = (int)scales[row * (k / 32) + j / 4] - 127;
    const uint32_t cw = reinterpret_cast<const uint32_t*>(codes + row * (k / 2))[j];
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t c = (cw >> (4 * i)) & 0xF;
      if (fp4) {
        const uint32_t e = (c >> 1) & 3, m = c & 1;
        const int half_units = e ? (int)((2 + m) << (e - 1)) : (int)m;  // value * 2
        const float mag = ldexpf((float)half_units, X - 1);
        v[i] = (c & 8) ? -mag : mag;
      } else {
        const int qv = (c & 8) ? (int)c - 16 : (int)c;
        v[i] = ldexpf((float)qv, X - 2);
      }
    }
    float4* o = reinterpret_cast<float4*>(out + row * k + j * 8);
    o[0] = make_float4(v[0], v[1], v[2], v[3]);
    o[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
}

int grid_for(int64_t quads) {
  const int64_t want = (quads + kQuadsPerCta * kUnroll - 1) / (kQuadsPerCta * kUnroll);
  const int64_t cap = (int64_t)num_sms() * 8;  // 8 resident CTAs of 256 threads per SM
  int64_t g = want < cap ? want : cap;
  return (int)(g > 0 ? g : 1);
}

}  // namespace

cudaError_t launch_mix_quantize(const void* x, bool bf16, int64_t rows, int64_t k, int64_t ld,
                                int type, int ebias, bool asym, uint8_t* codes, void* shared,
                                cudaStream_t st, const int* ebias_dev) {
  const int64_t nb = k / 32;
  if (rows * nb >= (int64_t)UINT32_MAX) return cudaErrorInvalidValue;  // 32-bit block index
  int64_t gb = (rows * nb + kThreads - 1) / kThreads;
  if (gb > (int64_t)num_sms() * 4) gb = (int64_t)num_sms() * 4;  // one wave of 4 resident CTAs per SM
  const int grid = (int)(gb > 0 ? gb : 1);
  const FastDiv f = make_fastdiv((uint32_t)nb);
  const bool dev = ebias_dev != nullptr;
#define MIXQ_LAUNCH(BF, T)                                                                                   \
  (dev ? mix_quantize_kernel<BF, T, true><<<grid, kThreads, 0, st>>>(x, rows, nb, ld, ebias, asym, codes,   \
                                                                      shared, f, ebias_dev)                  \
       : mix_quantize_kernel<BF, T, false><<<grid, kThreads, 0, st>>>(x, rows, nb, ld, ebias, asym, codes,  \
                                                                       shared, f, ebias_dev))
  if (bf16) {
    if (type == 1) MIXQ_LAUNCH(true, 1);
    else MIXQ_LAUNCH(true, 2);
  } else {
    if (type == 1) MIXQ_LAUNCH(false, 1);
    else MIXQ_LAUNCH(false, 2);
  }
#undef MIXQ_LAUNCH
  return cudaGetLastError();
}

// The largest finite |x| bit pattern into *key (cleared first).
cudaError_t launch_auto_ebias_key(const void* x, bool bf16, int64_t rows, int64_t k, int64_t ld, unsigned* key,
                                  cudaStream_t st) {
  const int es = bf16 ? 2 : 4;
  const int64_t vpr = k * es / 16;   // 16-byte vectors per row (k % 16 == 0)
  if (rows * vpr >= (int64_t)UINT32_MAX) return cudaErrorInvalidValue;  // 32-bit vector index
  cudaError_t e = cudaMemsetAsync(key, 0, sizeof(unsigned), st);
  if (e != cudaSuccess) return e;
  if (rows > 0 && vpr > 0) {
    int64_t gb = (rows * vpr + (int64_t)kThreads * kAmaxUnroll - 1) / ((int64_t)kThreads * kAmaxUnroll);
    if (gb > (int64_t)num_sms() * 8) gb = (int64_t)num_sms() * 8;
    const FastDiv f = make_fastdiv((uint32_t)vpr);
    if (bf16) amax_bits_kernel<true><<<(int)gb, kThreads, 0, st>>>(x, rows, vpr, ld * es, f, key);
    else amax_bits_kernel<false><<<(int)gb, kThreads, 0, st>>>(x, rows, vpr, ld * es, f, key);
    e = cudaGetLastError();
  }
  return e;
}

cudaError_t launch_auto_ebias(const void* x, bool bf16, int64_t rows, int64_t k, int64_t ld, int* ebias,
                              cudaStream_t st) {
  cudaError_t e = launch_auto_ebias_key(x, bf16, rows, k, ld, reinterpret_cast<unsigned*>(ebias), st);
  if (e != cudaSuccess) return e;
  auto_ebias_finish_kernel<<<1, 32, 0, st>>>(ebias);
  return cudaGetLastError();
}

cudaError_t launch_nvfp4_quantize(const void* x, bool bf16, int64_t rows, int64_t k, int64_t ld, uint8_t* codes,
                                  uint8_t* scales, float* tensor_scale, cudaStream_t st) {
  cudaError_t e = launch_auto_ebias_key(x, bf16, rows, k, ld, reinterpret_cast<unsigned*>(tensor_scale), st);
  if (e != cudaSuccess) return e;
  nvfp4_scale_finish_kernel<<<1, 32, 0, st>>>(tensor_scale);
  e = cudaGetLastError();
  if (e != cudaSuccess || rows == 0 || k == 0) return e;
  const int64_t nb = k / 16;
  if (rows * nb >= (int64_t)UINT32_MAX) return cudaErrorInvalidValue;
  int64_t gb = (rows * nb + kThreads - 1) / kThreads;
  if (gb > (int64_t)num_sms() * 8) gb = (int64_t)num_sms() * 8;
  const FastDiv f = make_fastdiv((uint32_t)nb);
  if (bf16) nvfp4_quantize_kernel<true><<<(int)gb, kThreads, 0, st>>>(x, rows, nb, ld, f, tensor_scale, codes, scales);
  else nvfp4_quantize_kernel<false><<<(int)gb, kThreads, 0, st>>>(x, rows, nb, ld, f, tensor_scale, codes, scales);
  return cudaGetLastError();
}

cudaError_t launch_clamp_count(const void* x, bool bf16, int64_t rows, int64_t k, int64_t ld, int ebias,
                               unsigned long long* counts, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(counts, 0, 2 * sizeof(unsigned long long), st);
  if (e != cudaSuccess || rows == 0 || k == 0) return e;
  const int64_t nb = k / 32;
  if (rows * nb >= (int64_t)UINT32_MAX) return cudaErrorInvalidValue;
  int64_t gb = (rows * nb + kThreads - 1) / kThreads;
  if (gb > (int64_t)num_sms() * 8) gb = (int64_t)num_sms() * 8;
  const FastDiv f = make_fastdiv((uint32_t)nb);
  if (bf16) clamp_count_kernel<true><<<(int)gb, kThreads, 0, st>>>(x, rows, nb, ld, f, ebias, counts);
  else clamp_count_kernel<false><<<(int)gb, kThreads, 0, st>>>(x, rows, nb, ld, f, ebias, counts);
  return cudaGetLastError();
}

cudaError_t launch_underflow_count(const void* x, bool bf16, int64_t rows, int64_t k, int64_t ld, const uint8_t* codes,
                                   int fmt, unsigned long long* count, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(count, 0, sizeof(unsigned long long), st);
  if (e != cudaSuccess || rows == 0 || k == 0) return e;
  const int64_t wpr = k / 8;
  if (rows * wpr >= (int64_t)UINT32_MAX) return cudaErrorInvalidValue;
  int64_t gb = (rows * wpr + kThreads - 1) / kThreads;
  if (gb > (int64_t)num_sms() * 8) gb = (int64_t)num_sms() * 8;
  const FastDiv f = make_fastdiv((uint32_t)wpr);
  if (bf16) underflow_count_kernel<true><<<(int)gb, kThreads, 0, st>>>(x, rows, wpr, ld, f, fmt, codes, count);
  else underflow_count_kernel<false><<<(int)gb, kThreads, 0, st>>>(x, rows, wpr, ld, f, fmt, codes, count);
  return cudaGetLastError();
}


cudaError_t launch_mx_quantize_rows(const void* x, bool bf16, int64_t rows, int64_t k, int64_t ld,
                                    bool fp4, int rule, bool g16, uint8_t* codes, uint8_t* scales,
                                    cudaStream_t st) {
  const int64_t nb = k / 32;
  if (rows * nb >= (int64_t)UINT32_MAX) return cudaErrorInvalidValue;  // 32-bit block index
  const int grid = grid_for(rows * nb);
  const FastDiv f = make_fastdiv((uint32_t)nb);
#define MXR(BF, F4, G)                                                                                 \
  mx_quantize_rows_kernel<BF, F4, G><<<grid, kThreads, 0, st>>>(x, rows, nb, ld, rule, codes, scales, f)
  if (bf16) {
    if (fp4) { if (g16) MXR(true, true, true); else MXR(true, true, false); }
    else { if (g16) MXR(true, false, true); else MXR(true, false, false); }
  } else {
    if (fp4) { if (g16) MXR(false, true, true); else MXR(false, true, false); }
    else { if (g16) MXR(false, false, true); else MXR(false, false, false); }
  }
#undef MXR
  return cudaGetLastError();
}

cudaError_t launch_mx_quantize_cols(const void* x, bool bf16, int64_t kdim, int64_t n, int64_t ld,
                                    bool fp4, int rule, bool g16, uint8_t* codes, uint8_t* scales,
                                    cudaStream_t st) {
  const dim3 grid((unsigned)((n + 63) / 64), (unsigned)((kdim / 32 + 7) / 8));
#define MXC(BF, F4, G) \
  mx_quantize_cols_kernel<BF, F4, G><<<grid, kThreads, 0, st>>>(x, kdim, n, ld, rule, codes, scales)
  if (bf16 && !g16) {
    const uint16_t* xb = static_cast<const uint16_t*>(x);
    if (fp4) mx_quantize_cols_bf16_kernel<true><<<grid, kThreads, 0, st>>>(xb, kdim, n, ld, rule, codes, scales);
    else mx_quantize_cols_bf16_kernel<false><<<grid, kThreads, 0, st>>>(xb, kdim, n, ld, rule, codes, scales);
  } else if (bf16) {
    if (fp4) MXC(true, true, true);
    else MXC(true, false, true);
  } else {
    if (fp4) { if (g16) MXC(false, true, true); else MXC(false, true, false); }
    else { if (g16) MXC(false, false, true); else MXC(false, false, false); }
  }
#undef MXC
  return cudaGetLastError();
}

cudaError_t launch_mix_dequantize(const uint8_t* codes, const void* shared, int64_t rows, int64_t k,
                                  int type, int ebias, float* out, cudaStream_t st) {
  const int64_t words = rows * (k / 8);
  int64_t g = (words + 255) / 256;
  if (g > (int64_t)num_sms() * 16) g = (int64_t)num_sms() * 16;
  mix_dequant_kernel<<<(int)(g > 0 ? g : 1), 256, 0, st>>>(codes, shared, rows, k, type, ebias, out);
  return cudaGetLastError();
}

cudaError_t launch_mx_dequantize(const uint8_t* codes, const uint8_t* scales, int64_t rows, int64_t k,
                                 bool fp4, float* out, cudaStream_t st) {
  const int64_t words = rows * (k / 8);
  int64_t g = (words + 255) / 256;
  if (g > (int64_t)num_sms() * 16) g = (int64_t)num_sms() * 16;
  mx_dequant_kernel<<<(int)(g > 0 ? g : 1), 256, 0, st>>>(codes, scales, rows, k, fp4 ? 1 : 0, out);
  return cudaGetLastError();
}

}  // namespace mixk
