// Device-side numerics of the MiX and MX formats, shared by the quantiser
// kernels and the GEMM epilogue.  Every decision is integer arithmetic on the
// fp32 bit pattern (bf16 inputs are widened exactly first), so a block gives
// the same codes wherever it is quantised.
//
// Source: "MiX: Micro-Inverted-Scaling for End-to-End Low-Bit Vision-Language
// Model Acceleration", pchao.org digest, section "Method" (MiX-4.25b /
// MiX-4.5b layouts, Algorithm 1 with the +-1 exponent refinement, asymmetric
// zero), section "Key results" (MXFP4 ceil shared exponent).
#pragma once
#include <cstdint>

namespace mixk {

// An fp32 value split for integer decisions.
//   cls 0: zero or NaN (both quantise to zero), 1: finite nonzero, 2: +-Inf.
//   sig: 24-bit significand with its leading one at bit 23 (normalised, also
//        for subnormals); f = floor(log2 |x|); s = sign bit.
struct Elem {
  uint32_t sig;
  int f;
  int s;
  int cls;
};

__device__ __forceinline__ Elem split_f32(uint32_t u) {
  Elem e;
  e.s = (int)(u >> 31);
  uint32_t ex = (u >> 23) & 0xFFu, m = u & 0x7FFFFFu;
  if (ex == 0xFFu) {
    e.cls = m ? 0 : 2;
    e.sig = 0x800000u;
    e.f = 128;
  } else if (ex == 0u) {
    if (m == 0u) {
      e.cls = 0; e.sig = 0; e.f = 0;
    } else {
      int p = 31 - __clz(m);  // 0 .. 22
      e.cls = 1;
      e.sig = m << (23 - p);
      e.f = p - 149;
    }
  } else {
    e.cls = 1;
    e.sig = m | 0x800000u;
    e.f = (int)ex - 127;
  }
  return e;
}

// Magnitude key of an fp32 bit pattern for block maxima: NaN maps to 0, so a
// NaN is never a maximum; +-Inf is the largest key.
__device__ __forceinline__ uint32_t mag_key(uint32_t u) {
  uint32_t a = u & 0x7FFFFFFFu;
  return a > 0x7F800000u ? 0u : a;
}

__device__ __forceinline__ uint32_t bf16_to_f32_bits(uint32_t h) { return h << 16; }

// Algorithm 1, first two steps, on the maximum magnitude (key != 0): its
// exponent and its mantissa rounded to 3 bits nearest-even; a carry out of the
// 3 bits gives mantissa 0 and exponent + 1.  Inf: mantissa 0, huge exponent.
__device__ __forceinline__ void max_exp_mant(uint32_t key, int* f, int* m3) {
  if (key >= 0x7F800000u) { *f = 1 << 20; *m3 = 0; return; }
  Elem e = split_f32(key);
  uint32_t q = (e.sig >> 20) & 7u, r = e.sig & 0xFFFFFu;
  if (r > 0x80000u || (r == 0x80000u && (q & 1u))) ++q;
  int ff = e.f;
  if (q == 8u) { q = 0; ++ff; }
  *f = ff;
  *m3 = (int)q;
}

__device__ __forceinline__ int clampi(int v, int lo, int hi) { return v < lo ? lo : (v > hi ? hi : v); }

// Algorithm 1, element step: the code of least |x - xhat| among the refinement
// candidates, ties to the larger magnitude.  M = 8 + mshared (the shared
// significand in eighths).  The nearest level M/8 * 2^j has j in {f-1, f,
// f+1}; the two midpoints 1.5 * M/8 * 2^(f-1) and 1.5 * M/8 * 2^f become the
// integer compares sig >= 12M * 2^16 and sig >= 24M * 2^16 (the hardware's
// 4-bit residual against 0.5).  Below the smallest level the choice is zero
// versus that level, an exact compare against half of it.
__device__ __forceinline__ uint32_t mix_code(const Elem& x, int emax, int M, bool asym) {
  if (x.cls == 0) return 7u;
  if (x.cls == 2) return (uint32_t)x.s << 3;
  const uint32_t t_lo = (uint32_t)(12 * M) << 16, t_hi = (uint32_t)(24 * M) << 16;
  int j = x.f + (x.sig >= t_hi ? 1 : 0) - (x.sig < t_lo ? 1 : 0);
  int d = emax - j;
  if (d < 0) d = 0;  // above the top level: saturate at de = 0
  const int dmax = (asym && x.s == 0) ? 7 : 6;
  if (d <= dmax) return d == 7 ? 0xFu : (((uint32_t)x.s << 3) | (uint32_t)d);
  const int sh = emax - dmax - x.f + 19;  // x >= half the smallest level?
  const bool up = sh < 21 && x.sig >= ((uint32_t)M << sh);
  if (!up) return 7u;
  return dmax == 7 ? 0xFu : (((uint32_t)x.s << 3) | 6u);
}

// Eight elements -> eight nibbles (element i in bits 4i..4i+3).
__device__ __forceinline__ uint32_t mix_codes8(const uint32_t* u, int emax, int M, bool asym) {
  uint32_t w = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) w |= mix_code(split_f32(u[i]), emax, M, asym) << (4 * i);
  return w;
}

__device__ __forceinline__ uint32_t max_key8(const uint32_t* u) {
  uint32_t k = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) k = max(k, mag_key(u[i]));
  return k;
}

// ---------------------------------------------------------------------------
// MX (MXINT4 / MXFP4)
// ---------------------------------------------------------------------------

// Shared exponent X from the block maximum key (key != 0).  MXFP4: the OCP
// rule floor(log2 amax) - 2 with the floor replaced by a ceil (the paper's
// MXFP4), or the OCP floor on request.  MXINT4: floor(log2 amax).
__device__ __forceinline__ int mx_shared_exp(uint32_t key, bool fp4, bool floor_rule) {
  if (key >= 0x7F800000u) return 127;
  Elem e = split_f32(key);
  int X;
  if (fp4) {
    int ce = (e.sig == 0x800000u) ? e.f : e.f + 1;
    X = floor_rule ? e.f - 2 : ce - 2;
  } else {
    X = e.f;
  }
  return clampi(X, -127, 127);
}

__device__ __forceinline__ uint32_t rne_shift(uint32_t sig, int sh) {
  // round-half-even of sig / 2^sh for 1 <= sh <= 31
  uint32_t q = sig >> sh, r = sig & ((1u << sh) - 1u), half = 1u << (sh - 1);
  if (r > half || (r == half && (q & 1u))) ++q;
  return q;
}

// E2M1 code of x / 2^X: nearest, ties to the even code, saturating at 6, -0
// written as +0.
__device__ __forceinline__ uint32_t mx_fp4_code(const Elem& x, int X) {
  if (x.cls == 0) return 0u;
  if (x.cls == 2) return ((uint32_t)x.s << 3) | 7u;
  int ey = x.f - X;
  uint32_t code;
  if (ey >= 3) {
    code = 7u;
  } else if (ey >= 0) {
    uint32_t q = rne_shift(x.sig, 22);  // 2 .. 4 in units of 2^(ey-1)
    if (q == 4u) { q = 2u; ++ey; }
    code = (ey >= 3) ? 7u : ((uint32_t)((ey + 1) << 1) | (q - 2u));
  } else {
    const int sh = 22 - ey;  // >= 23: units of 0.5
    code = (sh >= 25) ? 0u : rne_shift(x.sig, sh);  // 0, 1 (0.5) or 2 (1.0)
  }
  return code ? (((uint32_t)x.s << 3) | code) : 0u;
}

// INT4 code of x / 2^(X-2): nearest-even, clamped to [-7, 7], two's complement.
__device__ __forceinline__ uint32_t mx_int4_code(const Elem& x, int X) {
  if (x.cls == 0) return 0u;
  int q;
  if (x.cls == 2) {
    q = 7;
  } else {
    const int d = x.f - X;
    if (d >= 1) {
      q = 7;
    } else {
      const int sh = 21 - d;
      q = (sh >= 25) ? 0 : (int)rne_shift(x.sig, sh);
      if (q > 7) q = 7;
    }
  }
  return (uint32_t)(x.s ? -q : q) & 0xFu;
}

__device__ __forceinline__ uint32_t mx_codes8(const uint32_t* u, int X, bool fp4) {
  uint32_t w = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    Elem e = split_f32(u[i]);
    w |= (fp4 ? mx_fp4_code(e, X) : mx_int4_code(e, X)) << (4 * i);
  }
  return w;
}

}  // namespace mixk
