// Exact conversion of 4-bit MiX and MX element codes to e4m3 operand bytes,
// eight nibbles at a time, for the tcgen05 matmul (in-kernel decode and the
// staging pass that expands an operand once per call).
//
// "MiX: Micro-Inverted-Scaling for End-to-End Low-Bit Vision-Language Model
// Acceleration", pchao.org digest, section "Method": a MiX element (sign s,
// exponent offset de) with its block's shared mantissa m3 is
// +-(1.m3) 2^(Emax - de); with the block scale 2^(Emax - 1) factored out it is
// +-(1.m3) 2^(1 - de), always a normal e4m3 (exponents 1 .. -5; code 0x7 is
// zero, the recycled -0 code 0xF is +(1.m3) 2^-6).  An MXINT4 element q with
// scale 2^X is (q / 4) 2^X, and E2M1 codes keep their value; both are exact in
// e4m3 with the MX scale byte as the UE8M0 block scale.
#pragma once
#include <cstdint>

#include "tc_ptx.cuh"

namespace mixk {
namespace {

// Nibble -> e4m3 byte through two 8-entry tables (by the low three bits) and
// a byte select by the sign bit: one prmt per table half and one to pick
// between the positive and the negative candidate of every byte.
struct DecTab {
  uint32_t plo, phi, nlo, nhi;
};
// MiX element (s, de) with shared mantissa m3: +-(1.m3) 2^(1-de); code 0x7
// is zero and 0xF the recycled -0, +(1.m3) 2^-6.
__device__ __forceinline__ DecTab mix_tab(uint32_t m3) {
  const uint32_t m3x = m3 * 0x01010101u;
  DecTab t;
  t.plo = 0x28303840u | m3x;
  t.phi = 0x00101820u | (m3x & 0x00FFFFFFu);
  t.nlo = t.plo | 0x80808080u;
  t.nhi = 0x089098A0u | m3x;
  return t;
}
// INT4 two's complement q -> q / 4; E2M1 -> its value.
__device__ __forceinline__ DecTab int4_tab() { return DecTab{0x34302800u, 0x3E3C3A38u, 0xBABCBEC0u, 0xA8B0B4B8u}; }
__device__ __forceinline__ DecTab fp4_tab() { return DecTab{0x3C383000u, 0x4C484440u, 0xBCB8B080u, 0xCCC8C4C0u}; }

// e4m3 byte of +-mant 2^e (0 <= mant <= 15): exact when it fits, otherwise
// rounded to the nearest (ties to even) subnormal, and clipped to 448 above.
__device__ __forceinline__ uint32_t e4m3_of(int mant, int e, bool neg) {
  uint32_t b = 0u;
  if (mant != 0) {
    const int p = 31 - __clz(mant);  // leading bit
    const int E = p + e;
    if (E > 8) {
      b = 0x7Eu;
    } else if (E >= -6) {
      b = ((uint32_t)(E + 7) << 3) | ((uint32_t)((mant << 3) >> p) & 7u);
    } else {  // subnormal: m 2^-9
      const int s = e + 9;
      if (s >= 0) {
        b = (uint32_t)(mant << s);
      } else {
        const int r = -s;
        if (r <= 5) {
          const uint32_t q = (uint32_t)mant >> r, rem = (uint32_t)mant & ((1u << r) - 1u), half = 1u << (r - 1);
          b = q + ((rem > half || (rem == half && (q & 1u))) ? 1u : 0u);  // 8 is the smallest normal
        }
      }
    }
  }
  return (neg ? 0x80u : 0u) | b;
}

// The MX element tables (int4_tab / fp4_tab) with every value multiplied by
// 2^sh, as 16 bytes in code order (codes 0..7 then 8..15): MXINT4 q / 4,
// E2M1 in half units.
__device__ __forceinline__ uint32_t mx_scaled_entry(int code, bool fp4, int sh) {
  if (fp4) {
    const int e = (code >> 1) & 3, m = code & 1;
    const int half_units = e ? ((2 + m) << (e - 1)) : m;  // 0, 1, 2, 3, 4, 6, 8, 12
    return e4m3_of(half_units, sh - 1, (code & 8) != 0);
  }
  const int q = (code & 8) ? code - 16 : code;
  return e4m3_of(q < 0 ? -q : q, sh - 2, q < 0);
}

// Eight nibbles (element i in bits 4i..4i+3) -> eight e4m3 bytes.
__device__ __forceinline__ uint2 dec8(uint32_t v, const DecTab& t) {
  const uint32_t s7 = v & 0x77777777u, s2 = (v >> 1) & 0x44444444u;
  const uint32_t s7h = s7 >> 16, s2h = s2 >> 16;
  uint2 r;
  r.x = ptx::prmt(ptx::prmt(t.plo, t.phi, s7), ptx::prmt(t.nlo, t.nhi, s7), s2 | 0x3210u);
  r.y = ptx::prmt(ptx::prmt(t.plo, t.phi, s7h), ptx::prmt(t.nlo, t.nhi, s7h), s2h | 0x3210u);
  return r;
}

}  // namespace
}  // namespace mixk
