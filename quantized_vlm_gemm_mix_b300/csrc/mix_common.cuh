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

#include "mix_internal.h"

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

__device__ __forceinline__ uint32_t bf16_to_f32_bits(uint32_t h) { return h << 16; }

// Algorithm 1, first two steps, on the maximum magnitude (key != 0): its
// exponent and its mantissa rounded to 3 bits nearest-even; a carry out of the
// 3 bits gives mantissa 0 and exponent + 1.  Inf: mantissa 0, huge exponent.
// Returns false for a zero or subnormal maximum: with Emax >= ebias >= -100
// every element of such a (sub-)block quantises to the zero code, which is the
// canonical all-zero block.
// The rounding adds 2^19 - 1 plus the kept lowest mantissa bit below bit 20
// (ties to even), so a carry out of the mantissa raises the exponent field
// by itself (checked against the compare form for every normal key).
__device__ __forceinline__ bool max_exp_mant(uint32_t key, int* f, int* m3) {
  if (key < 0x00800000u) { *f = 0; *m3 = 0; return false; }
  if (key >= 0x7F800000u) { *f = 1 << 20; *m3 = 0; return true; }
  const uint32_t t = key + 0x7FFFFu + ((key >> 20) & 1u);
  *f = (int)(t >> 23) - 127;
  *m3 = (int)((t >> 20) & 7u);
  return true;
}

__device__ __forceinline__ int clampi(int v, int lo, int hi) { return v < lo ? lo : (v > hi ? hi : v); }

// Algorithm 1, element step, for one (sub-)block with shared exponent emax and
// shared significand M = 8 + mshared.  The levels M/8 * 2^(emax - de) form a
// geometric sequence, so do the midpoints between neighbouring levels:
// t_de = 3M * 2^(emax - 5 - de), whose fp32 bit patterns differ by exactly
// 2^23 per step.  The level nearest to |x| (ties to the larger) is therefore
// de = ceil((bits(t_0) - bits(|x|)) / 2^23) clamped at 0, an integer
// subtract and shift; below the smallest level the choice is zero versus that
// level, one compare against half of it.  This is the page's single-cycle
// "4-bit residual against 0.5" test, evaluated on bit patterns.
struct MixBlk {
  uint32_t t0;   // bits of the midpoint between the two largest levels
  uint32_t zp;   // bits of half the smallest positive level (de 7 with the recycled -0, else 6)
  uint32_t zn;   // bits of half the smallest negative level (de 6)
  int dmaxp;     // largest positive de: 7 with the recycled -0, else 6
};

__device__ __forceinline__ MixBlk mix_blk(int emax, int M, bool asym) {
  MixBlk b;
  const uint32_t m3M = 3u * (uint32_t)M;  // 24 .. 45
  const int p = m3M >= 32u ? 5 : 4;
  b.t0 = ((uint32_t)(emax - 5 + p + 127) << 23) | ((m3M - (1u << p)) << (23 - p));
  b.zn = ((uint32_t)(emax - 7 + 127) << 23) | ((uint32_t)(M - 8) << 20);  // (M/8) 2^(emax-6) / 2
  b.zp = asym ? b.zn - (1u << 23) : b.zn;
  b.dmaxp = asym ? 7 : 6;
  return b;
}

// Element step for a block known to hold no NaN (|x| bit pattern a given).
__device__ __forceinline__ uint32_t mix_code_nonan(uint32_t u, uint32_t a, const MixBlk& b) {
  int d = ((int)(b.t0 - a) + 0x7FFFFF) >> 23;
  const bool neg = (int)u < 0;
  const int dd = min(max(d, 0), neg ? 6 : b.dmaxp);
  const uint32_t code = (uint32_t)dd | ((u >> 28) & 8u) | ((uint32_t)(dd + 1) & 8u);
  return a < (neg ? b.zn : b.zp) ? 7u : code;
}

// Algorithm 1 on one 32-element block held as fp32 bit patterns (TYPE 1:
// MiX-4.25b, one shared mantissa; TYPE 2: MiX-4.5b, one per 8-element
// sub-block).  NaNs are coded as zero: the rare block holding one has them
// replaced by +0 first, so the element step never sees a NaN.  Writes the
// 16 code bytes and the shared field (zero for an all-zero block).
template <int TYPE>
__device__ __forceinline__ void mix_block32(uint32_t* u, int ebias, bool asym, uint4& cw, uint32_t& sh) {
  uint32_t ks[4];
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    uint32_t k = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) k = max(k, u[8 * s + i] & 0x7FFFFFFFu);
    ks[s] = k;
  }
  uint32_t kb = max(max(ks[0], ks[1]), max(ks[2], ks[3]));
  if (kb > 0x7F800000u) {  // a NaN in the block: code it as zero
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if ((u[i] & 0x7FFFFFFFu) > 0x7F800000u) u[i] = 0u;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      uint32_t k = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) k = max(k, u[8 * s + i] & 0x7FFFFFFFu);
      ks[s] = k;
    }
    kb = max(max(ks[0], ks[1]), max(ks[2], ks[3]));
  }
  cw = make_uint4(0x77777777u, 0x77777777u, 0x77777777u, 0x77777777u);
  sh = 0;
  int f, m3;
  if (max_exp_mant(kb, &f, &m3)) {
    const int emax = clampi(f, ebias, ebias + 15);
    uint32_t w[4];
    uint32_t m3bits = 0;
    bool all_zero = true;
    const MixBlk b1 = mix_blk(emax, 8 + m3, asym);
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      int ms = m3;
      MixBlk bb = b1;
      if (TYPE == 2) {
        int fs;
        if (!max_exp_mant(ks[s], &fs, &ms)) ms = 0;
        bb = mix_blk(emax, 8 + ms, asym);
      }
      uint32_t word = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t v = u[8 * s + i];
        word |= mix_code_nonan(v, v & 0x7FFFFFFFu, bb) << (4 * i);
      }
      w[s] = word;
      const bool z = word == 0x77777777u;
      all_zero &= z;
      if (z) ms = 0;
      m3bits |= (uint32_t)ms << (4 + 3 * s);
    }
    cw = make_uint4(w[0], w[1], w[2], w[3]);
    if (!all_zero) {
      const uint32_t ec = (uint32_t)(emax - ebias);
      sh = TYPE == 1 ? (ec | ((uint32_t)m3 << 4)) : (ec | m3bits);
    }
  }
}

// ---------------------------------------------------------------------------
// Packed element step: two elements per 32-bit word (element 2j in the low
// half of word j), one integer operation for both.  The inputs are the top
// 16 bits of the fp32 patterns (bf16 inputs as they are).  Exact because
// every threshold of the element step (t0, zn, zp above) has zero low 16
// bits, so comparing the top halves gives the same decisions:
//   d   = ceil((t0 - |x|) / 2^23) = floor((T - a + 127) / 128), T = t0 >> 16,
//         a = the top-half magnitude; computed per 16-bit lane as
//         X = 0x807F + T - a (the 0x8000 guard keeps every lane positive, so
//         no borrow crosses lanes), clamped with max/min.u16x2 to
//         [0x8000, 0x8000 + 128 cap + 127] (cap 6 for negative elements,
//         dmaxp for positive ones), then shifted right by 7: the low three
//         bits of each lane are d (clamping before the shift needs no mask),
//   code = d | sign << 3 | ((d + 1) & 8), and the zero code 7 where a < z,
//         the lane compare read from bit 15 of a + (0x8000 - z).
// Per-lane sign and compare masks come from one byte permute each (prmt
// replicates the sign bit of a byte), and the caps and zero thresholds of
// the two signs are chosen by those masks.  Checked against the scalar step
// exhaustively (every top-half pattern in each lane, every Emax of seven
// ebias values, every mshared, both zero modes) in an emulation before use.
__device__ __forceinline__ uint32_t vmax_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t vmin_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("min.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// Byte permute in its generic mode: a selector nibble with bit 3 set
// replicates the sign bit of the selected byte.
__device__ __forceinline__ uint32_t prmt_sel(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

struct MixBlk2 {
  uint32_t c1;   // (0x807F + T) in both lanes
  uint32_t kp2;  // 0x8000 - ZP in both lanes (positive elements)
  uint32_t kn2;  // 0x8000 - ZN in both lanes (ZN = ZP + 128 with the recycled -0, else ZP)
  uint32_t capn; // what the positive lanes' clamp adds: 128 with the recycled -0 (cap 7), else 0 (cap 6)
};

// The packed-step constants of a (sub-)block are the top halves of mix_blk's
// t0, zn, zp: in units of the top half, T = 128 Emax + 16192 + 24 m (m < 3,
// where 3 M < 32) or 16224 + 12 m, ZN = 128 Emax + 15360 + 16 m, ZP = ZN - 128
// with the recycled -0 (checked against mix_blk for every Emax in [-100, 115]
// and every m).  They split into a per-block part (Emax) and a per-sub-block
// part (mshared), linear in both -- T's mshared offset is 24 m - max(12 m -
// 32, 0) -- exact modulo 2^32 because every lane's final value lies in
// [0, 2^16) (checked against the formulas above for every Emax, m and zero
// mode).
struct MixBlkBase {
  uint32_t b1;    // (0x807F + 16192 + 128 Emax) in both lanes
  uint32_t b2;    // (0x8000 - 15360 - 128 Emax) in both lanes
  uint32_t ak;    // 128 in both lanes with the recycled -0, else 0
  uint32_t capn;
};
__device__ __forceinline__ MixBlkBase mix_blk_base(int emax, bool asym) {
  MixBlkBase b;
  const int e7 = emax * 128;
  b.b1 = (uint32_t)(0x807F + 16192 + e7) * 0x00010001u;
  b.b2 = (uint32_t)(0x8000 - 15360 - e7) * 0x00010001u;
  b.ak = asym ? 0x00800080u : 0u;
  b.capn = asym ? 0x00800080u : 0u;
  return b;
}
__device__ __forceinline__ MixBlk2 mix_blk2_lin(const MixBlkBase& b, int ms) {
  MixBlk2 q;
  const uint32_t m12 = (uint32_t)max(12 * ms - 32, 0);
  q.c1 = b.b1 + (uint32_t)ms * (24u * 0x00010001u) - m12 * 0x00010001u;
  q.kn2 = b.b2 - (uint32_t)ms * (16u * 0x00010001u);
  q.kp2 = q.kn2 + b.ak;
  q.capn = b.capn;
  return q;
}

// Codes of the two elements of word w (magnitudes a = w & 0x7FFF7FFF), at
// bits 0..3 (low element) and 16..19 (high element); every other bit zero.
__device__ __forceinline__ uint32_t mix_code_pair(uint32_t w, uint32_t a, const MixBlk2& q) {
  const uint32_t s = prmt_sel(w, w, 0xBB99u);              // 0xFFFF in negative lanes
  uint32_t x = vmax_u16x2(q.c1 - a, 0x80008000u);
  x = vmin_u16x2(x, 0x837F837Fu | (~s & q.capn));
  const uint32_t d = x >> 7;                                // d in bits 0..2 of each lane
  const uint32_t code = (d & 0x00070007u) | (((d + 0x00010001u) | s) & 0x00080008u);
  const uint32_t y = a + ((s & q.kn2) | (~s & q.kp2));
  const uint32_t m = prmt_sel(y, 0u, 0x4B49u);              // 0x00FF where |x| >= z
  return (code & m) | (0x00070007u & ~m);
}

// Eight codes of words w[0..3] (magnitudes a[0..3]) as one 32-bit word
// (element 2j in the low nibble of byte j): two pairs meet in a half-word by
// a multiply-add and a shift, two half-words in a word by a byte permute.
__device__ __forceinline__ uint32_t mix_codes8_packed(const uint32_t* w, const uint32_t* a, const MixBlk2& q) {
  uint32_t p0 = mix_code_pair(w[0], a[0], q) + mix_code_pair(w[1], a[1], q) * 256u;
  uint32_t p1 = mix_code_pair(w[2], a[2], q) + mix_code_pair(w[3], a[3], q) * 256u;
  p0 |= p0 >> 12;
  p1 |= p1 >> 12;
  return prmt_sel(p0, p1, 0x5410u);
}

// The packed part of Algorithm 1 for one NaN-free block: w holds the top 16
// bits of the 32 elements (element 2j in the low half of word j), ks the exact
// fp32 magnitude bits of each 8-element sub-block's maximum and kb the
// block's (they set Emax and mshared, whose rounding needs every mantissa
// bit).
template <int TYPE>
__device__ __forceinline__ void mix_block32_packed(const uint32_t* w, const uint32_t* a, const uint32_t* ks,
                                                   uint32_t kb, int ebias, bool asym, uint4& cw, uint32_t& sh) {
  cw = make_uint4(0x77777777u, 0x77777777u, 0x77777777u, 0x77777777u);
  sh = 0;
  int f, m3;
  if (!max_exp_mant(kb, &f, &m3)) return;
  const int emax = clampi(f, ebias, ebias + 15);
  uint32_t wd[4];
  uint32_t m3bits = 0;
  bool all_zero = true;
  const MixBlkBase base = mix_blk_base(emax, asym);
  const MixBlk2 q1 = mix_blk2_lin(base, m3);
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    int ms = m3;
    MixBlk2 q = q1;
    if (TYPE == 2) {
      int fs;
      if (!max_exp_mant(ks[s], &fs, &ms)) ms = 0;
      q = mix_blk2_lin(base, ms);
    }
    const uint32_t word = mix_codes8_packed(w + 4 * s, a + 4 * s, q);
    wd[s] = word;
    const bool z = word == 0x77777777u;
    all_zero &= z;
    if (z) ms = 0;
    m3bits |= (uint32_t)ms << (4 + 3 * s);
  }
  cw = make_uint4(wd[0], wd[1], wd[2], wd[3]);
  if (!all_zero) {
    const uint32_t ec = (uint32_t)(emax - ebias);
    sh = TYPE == 1 ? (ec | ((uint32_t)m3 << 4)) : (ec | m3bits);
  }
}

// Algorithm 1 on one block of 32 bf16 elements held as 16 packed words;
// same results as mix_block32 on the widened elements (a block holding a NaN
// goes through mix_block32, which codes NaN as zero).
template <int TYPE>
__device__ __forceinline__ void mix_block32_bf16(const uint32_t* w, int ebias, bool asym, uint4& cw, uint32_t& sh) {
  uint32_t a[16], ks[4];
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    uint32_t m = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      a[4 * s + j] = w[4 * s + j] & 0x7FFF7FFFu;
      m = vmax_u16x2(m, a[4 * s + j]);
    }
    ks[s] = max(m >> 16, m & 0xFFFFu) << 16;
  }
  const uint32_t kb = max(max(ks[0], ks[1]), max(ks[2], ks[3]));
  if (kb > 0x7F800000u) {  // a NaN in the block
    uint32_t u[32];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      u[2 * j] = w[j] << 16;
      u[2 * j + 1] = w[j] & 0xFFFF0000u;
    }
    mix_block32<TYPE>(u, ebias, asym, cw, sh);
    return;
  }
  mix_block32_packed<TYPE>(w, a, ks, kb, ebias, asym, cw, sh);
}

// Algorithm 1 on one block of 32 fp32 elements (bit patterns; u may be
// overwritten).  Emax and mshared come from the exact fp32 maxima; the element
// step runs packed on the top 16 bits of each element, which decides exactly
// as on all 32: every threshold is a multiple of 2^16 in bit-pattern space,
// and for such a t, |x| < t holds exactly when its top 16 bits are below t's.
// max(|a|, |b|, |c|) in one instruction, NaN if any input is NaN.  For
// values that are not NaN the result is the largest magnitude with its sign
// clear, and non-negative floats order as their bit patterns do, so its bits
// are the integer maximum of the magnitude bit patterns (checked on the GPU
// for every fp32 pattern as an input).
__device__ __forceinline__ float absmax3(float a, float b, float c) {
  float d;
  asm("max.NaN.abs.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

template <int TYPE>
__device__ __forceinline__ void mix_block32_f32(uint32_t* u, int ebias, bool asym, uint4& cw, uint32_t& sh) {
  // the sub-block maxima of |x|, eight elements in four 3-input steps; a NaN
  // makes the maximum a NaN pattern, above every finite and infinite one
  uint32_t ks[4];
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const uint32_t* v = u + 8 * s;
    float m = absmax3(__uint_as_float(v[0]), __uint_as_float(v[1]), __uint_as_float(v[2]));
    m = absmax3(m, __uint_as_float(v[3]), __uint_as_float(v[4]));
    m = absmax3(m, __uint_as_float(v[5]), __uint_as_float(v[6]));
    m = absmax3(m, __uint_as_float(v[7]), __uint_as_float(v[7]));
    ks[s] = __float_as_uint(m);
  }
  const uint32_t kb = max(max(ks[0], ks[1]), max(ks[2], ks[3]));
  if (kb > 0x7F800000u) {  // a NaN in the block: the scalar path codes it as zero
    mix_block32<TYPE>(u, ebias, asym, cw, sh);
    return;
  }
  uint32_t w[16], a[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    w[j] = __byte_perm(u[2 * j], u[2 * j + 1], 0x7632);
    a[j] = w[j] & 0x7FFF7FFFu;
  }
  mix_block32_packed<TYPE>(w, a, ks, kb, ebias, asym, cw, sh);
}

// Division by a runtime constant d (1 <= d < 2^31) of 32-bit numerators with
// a multiply-high and a shift (Granlund and Montgomery, "Division by invariant
// integers using multiplication", 1994): m = floor(2^32 (2^l - d) / d) + 1
// with l = ceil(log2 d), q = (mulhi(n, m) + n) >> l.
struct FastDiv {
  uint32_t d, m, l;
};
inline FastDiv make_fastdiv(uint32_t d) {
  FastDiv f;
  f.d = d;
  f.l = 0;
  while ((1ull << f.l) < d) ++f.l;
  f.m = (uint32_t)((((1ull << 32) * ((1ull << f.l) - d)) / d) + 1);
  return f;
}
__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv& f) {
  return (uint32_t)(((uint64_t)__umulhi(n, f.m) + n) >> f.l);
}

// ---------------------------------------------------------------------------
// MX (MXINT4 / MXFP4)
// ---------------------------------------------------------------------------

// Shared exponent X from the block maximum key (key != 0), amax = sig 2^f
// with sig in [1, 2).  MXFP4: the OCP rule floor(log2 amax) - 2 with the
// floor replaced by a ceil (the paper's MXFP4), the OCP floor, or the tight
// ceil(log2(amax / 6)) = f - 2 + [sig > 1.5].  MXINT4 (elements q 2^(X-2),
// |q| <= 7): floor(log2 amax), or the tight f + [sig > 1.75].
__device__ __forceinline__ int mx_shared_exp(uint32_t key, bool fp4, int rule) {
  if (key >= 0x7F800000u) return 127;
  Elem e = split_f32(key);
  int X;
  if (fp4) {
    if (rule == MX_RULE_TIGHT) X = e.f - 2 + (e.sig > 0xC00000u ? 1 : 0);
    else if (rule == MX_RULE_FLOOR) X = e.f - 2;
    else X = (e.sig == 0x800000u) ? e.f - 2 : e.f - 1;
  } else {
    X = e.f + ((rule == MX_RULE_TIGHT && e.sig > 0xE00000u) ? 1 : 0);
  }
  return clampi(X, -127, 127);
}

// 2^k as an fp32 factor, k in [-126, 127].
__device__ __forceinline__ float pow2f(int k) { return __int_as_float((uint32_t)(k + 127) << 23); }

// Two elements -> one byte of E2M1 codes (first element in the low nibble):
// x / 2^X rounded to nearest-even on the E2M1 grid with saturation at 6 is the
// hardware conversion cvt.rn.satfinite.e2m1x2.f32.
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// Eight elements of an MX block with shared exponent X -> eight nibbles.
// MXFP4: E2M1 codes of x / 2^X, -0 written as +0.  MXINT4: q = round-half-even
// of x / 2^(X-2) (an fp32 add of 1.5 * 2^23 rounds to an integer exactly),
// clamped to [-7, 7], two's complement.  The 2^-X factor is applied as two
// exact power-of-two multiplies so that it never overflows.  The elements
// hold no NaN (mx_block32 / the callers replace NaNs by +0 first).
__device__ __forceinline__ uint32_t mx_codes8(const uint32_t* u, int X, bool fp4) {
  const int k = fp4 ? -X : 2 - X;
  const int k1 = k / 2, k2 = k - k1;
  const float s1 = pow2f(k1), s2 = pow2f(k2);
  uint32_t w = 0;
  if (fp4) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      w |= e2m1x2(__uint_as_float(u[2 * i]) * s1 * s2, __uint_as_float(u[2 * i + 1]) * s1 * s2) << (8 * i);
    // -0 (nibble 0x8) -> +0
    const uint32_t t = w ^ 0x88888888u;
    const uint32_t nz = (t | (t >> 1) | (t >> 2) | (t >> 3)) & 0x11111111u;
    w &= ~((~nz & 0x11111111u) << 3);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float y = __uint_as_float(u[i]) * s1 * s2;
      int q = __float_as_int(y + 12582912.0f) - 0x4B400000;
      q = clampi(q, -7, 7);
      w |= ((uint32_t)q & 0xFu) << (4 * i);
    }
  }
  return w;
}

// Largest |x| bit pattern of n >= 3 elements, or a NaN pattern (above every
// other) when one of them is NaN: two elements per 3-input abs max.
template <int N>
__device__ __forceinline__ uint32_t max_abs_bits(const uint32_t* u) {
  float m = absmax3(__uint_as_float(u[0]), __uint_as_float(u[1]), __uint_as_float(u[2]));
#pragma unroll
  for (int i = 3; i < N; i += 2)
    m = absmax3(m, __uint_as_float(u[i]), __uint_as_float(u[i + 1 < N ? i + 1 : i]));
  return __float_as_uint(m);
}

// NaN -> +0 in place (NaN is coded as zero and is never a block maximum).
template <int N>
__device__ __forceinline__ void zero_nans(uint32_t* u) {
#pragma unroll
  for (int i = 0; i < N; ++i)
    if ((u[i] & 0x7FFFFFFFu) > 0x7F800000u) u[i] = 0u;
}

// One MX block of 32 elements (in place: NaNs become +0): the shared
// exponent X, the 16 code bytes and the E8M0 scale byte X + 127 (zero codes
// and scale for an all-zero block).
template <bool FP4>
__device__ __forceinline__ void mx_block32(uint32_t* u, int rule, uint4& w, uint32_t& sc) {
  uint32_t kb = max_abs_bits<32>(u);
  if (kb > 0x7F800000u) {
    zero_nans<32>(u);
    kb = max_abs_bits<32>(u);
  }
  w = make_uint4(0, 0, 0, 0);
  sc = 0;
  if (kb != 0u) {
    const int X = mx_shared_exp(kb, FP4, rule);
    w = make_uint4(mx_codes8(u, X, FP4), mx_codes8(u + 8, X, FP4), mx_codes8(u + 16, X, FP4),
                   mx_codes8(u + 24, X, FP4));
    sc = (uint32_t)(X + 127);
  }
}

// One 16-element MX block (the g16 weight formats), as mx_block32.
template <bool FP4>
__device__ __forceinline__ void mx_block16(uint32_t* u, int rule, uint2& w, uint32_t& sc) {
  uint32_t kb = max_abs_bits<16>(u);
  if (kb > 0x7F800000u) {
    zero_nans<16>(u);
    kb = max_abs_bits<16>(u);
  }
  w = make_uint2(0, 0);
  sc = 0;
  if (kb != 0u) {
    const int X = mx_shared_exp(kb, FP4, rule);
    w = make_uint2(mx_codes8(u, X, FP4), mx_codes8(u + 8, X, FP4));
    sc = (uint32_t)(X + 127);
  }
}

}  // namespace mixk
