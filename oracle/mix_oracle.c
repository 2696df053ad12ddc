/*
 * Plain, slow, scalar CPU oracle for the MiX hot path.  TEST INFRASTRUCTURE
 * ONLY: it is built and called by the tests, by the smoke check and by the
 * bench's CPU-baseline leg, never by the library.  It shares no code, header,
 * table or helper with the CUDA sources.
 *
 * Source: "MiX: Micro-Inverted-Scaling for End-to-End Low-Bit Vision-Language
 * Model Acceleration" (Liao and Seo, MICRO 2026), as digested on the pchao.org
 * page, section "Method" (方法概览): the MiX-4.25b and MiX-4.5b block formats,
 * Algorithm 1 with the +-1 exponent refinement, Eq. (6), the asymmetric zero,
 * K-smoothing; "Key results" (关键结果) for the MXFP4 ceil rule.
 *
 * Arithmetic: every value handled here is an exact binary quantity.  Inputs
 * (bf16 / fp32) are widened to double exactly; code values are (1.m3) * 2^j
 * with a 3-bit m3; GEMM block sums are int64; the cross-block sum is fp64.
 *
 * Readings of points the page leaves open: field orders as in the library
 * header; mshared rounded to nearest-even with a carry into Emax; equal
 * errors resolved toward the larger magnitude; an all-zero (sub-)block stores
 * zero shared fields; NaN counts as zero, +-Inf saturates; MXFP4 scale
 * ceil(log2 amax) - 2, MXINT4 scale floor(log2 amax) with q in [-7, 7].
 * Optional rules beyond the page: the OCP floor for MXFP4, and the "tight"
 * shared exponent (the smallest one at which no element saturates: the
 * ceil(log2(amax / 6)) alternative the page's ceil rule is contrasted with);
 * the automatic ebias puts the largest block's Emax at the top of the 4-bit
 * range.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F32 = 0, ORC_BF16 = 1 };
enum { ORC_T1 = 1, ORC_T2 = 2 };
enum { ORC_MXINT4 = 0, ORC_MXFP4 = 1 };
enum { ORC_ASYM_ZERO = 1, ORC_MX_FLOOR = 2, ORC_MX_TIGHT = 4 };

/* A test may plant one deliberate mistake here to prove the pins catch it. */
static int g_mutation = 0;
void orc_set_mutation(int m) { g_mutation = m; }

/* ----------------------------------------------------------------------- */
/* Input widening (exact).                                                  */
/* ----------------------------------------------------------------------- */
static double load_elem(const void* x, int dtype, int64_t idx) {
  if (dtype == ORC_F32) {
    float f;
    memcpy(&f, (const char*)x + 4 * idx, 4);
    return (double)f;
  }
  uint16_t h;
  memcpy(&h, (const char*)x + 2 * idx, 2);
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Magnitude used for the block maximum: NaN counts as 0 (never a maximum). */
static double mag(double v) { return isnan(v) ? 0.0 : fabs(v); }

/* floor(log2 |v|) for finite nonzero v, exactly (frexp handles subnormals). */
static int floor_log2(double v) {
  int e;
  frexp(fabs(v), &e);
  return e - 1;
}

/* Round-half-to-even of a non-negative double to an integer. */
static double rne(double t) {
  double f = floor(t);
  double r = t - f;
  if (r > 0.5) return f + 1.0;
  if (r < 0.5) return f;
  return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

/* ----------------------------------------------------------------------- */
/* MiX: Algorithm 1                                                         */
/* ----------------------------------------------------------------------- */

/* Steps 1-2 of Algorithm 1 for a set of magnitudes with maximum amax > 0:
 * the exponent f of amax and the 3-bit shared mantissa taken from amax's own
 * mantissa, rounded to nearest-even; a carry out of the 3 bits makes the
 * mantissa 0 and moves f up by one.  Inf gives m3 = 0 and a huge f. */
static void max_exp_mant(double amax, int* f_out, int* m3_out) {
  if (isinf(amax)) { *f_out = 100000; *m3_out = 0; return; }
  int f = floor_log2(amax);
  double sig = ldexp(amax, -f);            /* in [1, 2) */
  double t = (sig - 1.0) * 8.0;            /* exact */
  int m3 = (g_mutation == 1) ? (int)floor(t) : (int)rne(t);
  if (m3 == 8) { m3 = 0; f += 1; }
  *f_out = f;
  *m3_out = m3;
}

/* Value of element code (s, d) under shared exponent emax and mantissa m3.
 * d = 7 is the zero code when s = 0; (s = 1, d = 7) is the recycled "-0"
 * (asymmetric zero), a positive value one binade below d = 6. */
static double mix_value(int s, int d, int emax, int m3) {
  double M = 1.0 + m3 / 8.0;
  if (g_mutation == 2) M = m3 / 8.0;       /* planted: implicit leading 1 dropped */
  if (d == 7 && s && g_mutation == 13) return -ldexp(M, emax - 7);   /* planted: recycled -0 negative */
  if (d == 7) return s ? ldexp(M, emax - 7) : 0.0;
  double v = ldexp(M, emax - d);
  return s ? -v : v;
}

/* Step 3-4 of Algorithm 1 for one element: naive delta-e from the element's
 * own exponent, then the refinement search over {de-1, de, de+1} (clipped to
 * the code range) for the smallest reconstruction error.  Equal errors go to
 * the larger magnitude.  Returns the 4-bit code (sign << 3 | delta-e). */
static int mix_element(double x, int emax, int m3, int asym) {
  if (isnan(x) || x == 0.0) return 0x7;
  int s = x < 0.0;
  if (isinf(x)) return (s << 3) | 0;
  int naive = emax - floor_log2(x);
  if (g_mutation == 3) naive = emax - floor_log2(x) + 1;
  int best_code = 0x7;
  double best_err = fabs(x);               /* the zero code */
  double best_mag = 0.0;
  int lo = naive - 1, hi = naive + 1;
  if (g_mutation == 4) { lo = naive; hi = naive; }   /* planted: no refinement */
  for (int c = lo; c <= hi; ++c) {
    int d = c < 0 ? 0 : (c > 7 ? 7 : c);
    for (int ss = 0; ss <= 1; ++ss) {
      int sc = (d == 7) ? ss : s;          /* d = 7: zero (s=0) or asym (s=1) */
      if (d == 7 && sc == 1 && !asym) continue;
      if (d == 7 && sc == 0) continue;     /* zero already seeded */
      if (d < 7 && ss == 1) continue;      /* one sign per d < 7 */
      double v = mix_value(sc, d, emax, m3);
      double err = fabs(x - v);
      double m = fabs(v);
      if (err < best_err || (err == best_err && m > best_mag)) {
        best_err = err;
        best_mag = m;
        best_code = (sc << 3) | d;
      }
    }
  }
  return best_code;
}

/* Quantise one 32-element block.  type T1: one m3 for the block; T2: the
 * block splits into four 8-element sub-blocks, each with its own m3 taken
 * from its own maximum, all sharing the block's Emax. */
static void mix_block(const double* v, int type, int ebias, unsigned flags,
                      int* codes, int* emax_code, int* m3s) {
  int asym = (flags & ORC_ASYM_ZERO) != 0;
  double amax = 0.0;
  for (int i = 0; i < 32; ++i) { double a = mag(v[i]); if (a > amax) amax = a; }
  for (int k = 0; k < 4; ++k) m3s[k] = 0;
  *emax_code = 0;
  if (amax == 0.0) { for (int i = 0; i < 32; ++i) codes[i] = 0x7; return; }
  int f, m3;
  max_exp_mant(amax, &f, &m3);
  int emax = f < ebias ? ebias : (f > ebias + 15 ? ebias + 15 : f);
  if (type == ORC_T1) {
    for (int k = 0; k < 4; ++k) m3s[k] = m3;
  } else {
    for (int k = 0; k < 4; ++k) {
      double sm = 0.0;
      for (int i = 0; i < 8; ++i) { double a = mag(v[8 * k + i]); if (a > sm) sm = a; }
      int fk = 0, mk = 0;
      if (sm > 0.0) max_exp_mant(sm, &fk, &mk);
      m3s[k] = mk;                         /* a carry only zeroes mk; Emax stays */
      if (g_mutation == 12) m3s[k] = m3;   /* planted: sub-block mantissa from the block max */
    }
  }
  for (int i = 0; i < 32; ++i) codes[i] = mix_element(v[i], emax, m3s[i / 8], asym);
  /* Canonical form: an all-zero (sub-)block stores m3 = 0; an all-zero block
   * stores a zero Emax field as well. */
  int all_zero = 1;
  for (int k = 0; k < 4; ++k) {
    int z = 1;
    for (int i = 0; i < 8; ++i) if (codes[8 * k + i] != 0x7) z = 0;
    if (z && type == ORC_T2) m3s[k] = 0;
    all_zero &= z;
  }
  if (all_zero) { for (int k = 0; k < 4; ++k) m3s[k] = 0; return; }
  *emax_code = emax - ebias;
}

/* x: rows x k (leading dimension ld elements).  codes: rows x k/2 bytes,
 * element 2j in the low nibble of byte j.  shared: rows x k/32 entries,
 * uint8 for T1 ([3:0] Emax-ebias, [6:4] m3), uint16 for T2 ([3:0] Emax-ebias,
 * then m3 of sub-blocks 0..3 at [6:4], [9:7], [12:10], [15:13]). */
int orc_mix_quantize(const void* x, int dtype, int64_t rows, int64_t k, int64_t ld,
                     int type, int ebias, unsigned flags, uint8_t* codes, void* shared) {
  if (k % 32 != 0 || (type != ORC_T1 && type != ORC_T2)) return 1;
  int64_t nb = k / 32;
  double v[32];
  int c[32], ec, m3s[4];
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      for (int i = 0; i < 32; ++i) v[i] = load_elem(x, dtype, r * ld + b * 32 + i);
      mix_block(v, type, ebias, flags, c, &ec, m3s);
      uint8_t* out = codes + r * (k / 2) + b * 16;
      for (int j = 0; j < 16; ++j)
        out[j] = g_mutation == 18 ? (uint8_t)((c[2 * j] << 4) | c[2 * j + 1])   /* planted: nibble order */
                                  : (uint8_t)(c[2 * j] | (c[2 * j + 1] << 4));
      if (type == ORC_T1) {
        ((uint8_t*)shared)[r * nb + b] = (uint8_t)(ec | (m3s[0] << 4));
      } else {
        uint16_t w = (uint16_t)(ec | (m3s[0] << 4) | (m3s[1] << 7) | (m3s[2] << 10) | (m3s[3] << 13));
        if (g_mutation == 20)   /* planted: sub-blocks packed in reverse order (unpacked the same way) */
          w = (uint16_t)(ec | (m3s[3] << 4) | (m3s[2] << 7) | (m3s[1] << 10) | (m3s[0] << 13));
        ((uint16_t*)shared)[r * nb + b] = w;
      }
    }
  }
  return 0;
}

/* Field access for one block of MiX shared data. */
static void mix_shared_fields(const void* shared, int type, int64_t idx, int* ec, int* m3s) {
  if (type == ORC_T1) {
    uint8_t s = ((const uint8_t*)shared)[idx];
    *ec = s & 0xF;
    for (int k = 0; k < 4; ++k) m3s[k] = (s >> 4) & 7;
  } else {
    uint16_t s = ((const uint16_t*)shared)[idx];
    *ec = s & 0xF;
    for (int k = 0; k < 4; ++k) m3s[k] = (s >> (4 + 3 * (g_mutation == 20 ? 3 - k : k))) & 7;
  }
}

static int nibble(const uint8_t* codes, int64_t i) {
  uint8_t b = codes[i >> 1];
  return (i & 1) ? (b >> 4) : (b & 0xF);
}

/* Dequantisation rule: (-1)^s * (1.mshared)_2 * 2^(Emax - de), de = 7 zero. */
int orc_mix_dequantize(const uint8_t* codes, const void* shared, int64_t rows, int64_t k,
                       int type, int ebias, double* out) {
  if (k % 32 != 0) return 1;
  int64_t nb = k / 32;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t b = 0; b < nb; ++b) {
      int ec, m3s[4];
      mix_shared_fields(shared, type, r * nb + b, &ec, m3s);
      for (int i = 0; i < 32; ++i) {
        int c = nibble(codes + r * (k / 2), b * 32 + i);
        out[r * k + b * 32 + i] = mix_value(c >> 3, c & 7, ec + ebias, m3s[i / 8]);
      }
    }
  return 0;
}

/* Clamped blocks of the MiX quantiser at a given ebias (the page gives Emax
 * only its 4-bit width, so Emax = field + ebias and an exponent outside
 * [ebias, ebias + 15] is clamped).  Per 32-element block: f = the exponent
 * steps 1-2 of Algorithm 1 give the block maximum (mshared rounding and its
 * carry included).  counts[0]: blocks with f > ebias + 15 (+-Inf included);
 * counts[1]: blocks with a nonzero maximum and f < ebias.  NaN counts as 0. */
int orc_mix_clamp_count(const void* x, int dtype, int64_t rows, int64_t k, int64_t ld, int ebias,
                        int64_t* counts) {
  if (k % 32 != 0) return 1;
  counts[0] = counts[1] = 0;
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t b = 0; b < k / 32; ++b) {
      double amax = 0.0;
      for (int i = 0; i < 32; ++i) {
        double a = mag(load_elem(x, dtype, r * ld + b * 32 + i));
        if (a > amax) amax = a;
      }
      if (amax == 0.0) continue;
      int f, m3;
      max_exp_mant(amax, &f, &m3);
      if (g_mutation == 21) { f = floor_log2(amax); }   /* planted: carry ignored */
      if (f > ebias + 15) counts[0] += 1;
      else if (f < ebias) counts[1] += 1;
    }
  }
  return 0;
}

/* Automatic ebias (a two-pass mode; the page fixes only the 4-bit width of
 * Emax): the largest block exponent f over the tensor -- floor(log2) of the
 * block maximum after its mantissa is rounded to three bits, carry included,
 * i.e. the Emax that block would take unclamped -- less 15, so that block
 * sits at the top of the range; clamped to [-100, 100].  Infinite elements
 * saturate under any ebias and are left out of the scan, as NaN is; a tensor
 * without a nonzero finite element gets -8. */
int orc_mix_auto_ebias(const void* x, int dtype, int64_t rows, int64_t k, int64_t ld) {
  if (k % 32 != 0) return -1000;
  int have = 0, fmax = 0;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t b = 0; b < k / 32; ++b) {
      double amax = 0.0;
      for (int i = 0; i < 32; ++i) {
        double a = mag(load_elem(x, dtype, r * ld + b * 32 + i));
        if (!isinf(a) && a > amax) amax = a;
      }
      if (amax == 0.0) continue;
      int f, m3;
      max_exp_mant(amax, &f, &m3);   /* Algorithm 1's first two steps, carry included */
      if (g_mutation == 9) f = floor_log2(amax);   /* planted: carry dropped */
      if (!have || f > fmax) fmax = f;
      have = 1;
    }
  if (!have) return -8;
  int e = fmax - 15;
  if (e < -100) e = -100;
  if (e > 100) e = 100;
  return e;
}

/* ----------------------------------------------------------------------- */
/* MX: MXINT4 / MXFP4, block 32, E8M0 shared scale                          */
/* ----------------------------------------------------------------------- */
static const double E2M1_GRID[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

/* Shared exponent X of a block with maximum magnitude amax > 0.
 * MXFP4: OCP rule floor(log2 amax) - 2 with the floor replaced by a ceil
 * (every "MXFP4" of the paper uses ceil); the OCP floor on request.
 * MXINT4: floor(log2 amax); elements are q * 2^(X-2), q in [-7, 7]. */
static int mx_shared_exp(double amax, int type, unsigned flags) {
  int X;
  if (isinf(amax)) return 127;
  int fl = floor_log2(amax);
  if (flags & ORC_MX_TIGHT) {
    /* smallest X with amax <= cap * 2^X: cap 6 (the largest E2M1 value) for
     * MXFP4, 7 * 2^-2 for MXINT4 (elements q * 2^(X-2), |q| <= 7) */
    const double cap = (type == ORC_MXFP4) ? 6.0 : 1.75;
    X = fl - 4;
    while (amax > ldexp(cap, X) || (g_mutation == 8 && amax == ldexp(cap, X))) ++X;
  } else if (type == ORC_MXFP4) {
    int is_pow2 = ldexp(amax, -fl) == 1.0;
    int ce = is_pow2 ? fl : fl + 1;
    X = (flags & ORC_MX_FLOOR) ? fl - 2 : ce - 2;
    if (g_mutation == 5) X = fl - 2;       /* planted: floor used for ceil */
  } else {
    X = fl;
  }
  if (X < -127) X = -127;
  if (X > 127) X = 127;
  return X;
}

/* E2M1 code of y = x / 2^X: nearest grid point, ties to the even code
 * (mantissa bit 0), saturating at 6; -0 is written as +0. */
static int e2m1_code(double y) {
  if (isnan(y)) return 0;
  int s = y < 0.0;
  double a = fabs(y);
  int best = 7;
  if (a < 6.0) {
    best = 0;
    for (int i = 1; i < 8; ++i) {
      double e0 = fabs(a - E2M1_GRID[best]), e1 = fabs(a - E2M1_GRID[i]);
      if (e1 < e0 || (e1 == e0 && (i & 1) == 0)) best = i;
    }
  }
  if (best == 0) s = 0;
  return (s << 3) | best;
}

/* INT4 code of y = x / 2^(X-2): round half to even, clamp to [-7, 7]. */
static int int4_code(double y) {
  if (isnan(y)) return 0;
  double a = fabs(y);
  double q = isinf(a) ? 7.0 : rne(a);
  if (q > 7.0) q = 7.0;
  if (g_mutation == 14 && isfinite(a) && rne(a) >= 8.0) q = 8.0;   /* planted: clamp at 8 */
  int qi = (int)q;
  if (y < 0.0) qi = -qi;
  return qi & 0xF;
}

/* One MX block of n (32, or 16 for the g16 variants) elements. */
static void mx_block(const double* v, int n, int type, unsigned flags, int* codes, int* scale) {
  double amax = 0.0;
  for (int i = 0; i < n; ++i) { double a = mag(v[i]); if (a > amax) amax = a; }
  if (amax == 0.0) {
    *scale = 0;
    for (int i = 0; i < n; ++i) codes[i] = 0;
    return;
  }
  int X = mx_shared_exp(amax, type, flags);
  *scale = X + 127;
  for (int i = 0; i < n; ++i) {
    double x = isnan(v[i]) ? 0.0 : v[i];
    if (type == ORC_MXFP4) {
      codes[i] = isinf(x) ? ((x < 0) << 3 | 7) : e2m1_code(ldexp(x, -X));
    } else {
      codes[i] = int4_code(isinf(x) ? x : ldexp(x, 2 - X));
    }
  }
}

/* Quantise a matrix to MX with blocks of `block` (32; 16 for MXINT4g16 /
 * MXFP4g16) elements along the reduction dimension K.
 * axis = 1: x is N x K (row-major, ld >= K), blocks along its rows.
 * axis = 0: x is K x N (row-major, ld >= N), blocks down its columns; the
 *           output is written transposed, i.e. as N x K.
 * codes: N x K/2 bytes; scales: N x K/block E8M0 bytes (X + 127). */
int orc_mx_quantize_blk(const void* x, int dtype, int64_t rows, int64_t cols, int64_t ld,
                        int axis, int type, unsigned flags, int block, uint8_t* codes, uint8_t* scales) {
  int64_t N = axis ? rows : cols, K = axis ? cols : rows;
  if (block != 32 && block != 16) return 1;
  if (K % 32 != 0) return 1;
  if ((flags & ORC_MX_FLOOR) && (flags & ORC_MX_TIGHT)) return 1;   /* two exponent rules */
  int64_t nb = K / block;
  double v[32];
  int c[32], sc;
  for (int64_t n = 0; n < N; ++n)
    for (int64_t b = 0; b < nb; ++b) {
      for (int i = 0; i < block; ++i) {
        int64_t kk = b * block + i;
        v[i] = load_elem(x, dtype, axis ? n * ld + kk : kk * ld + n);
      }
      mx_block(v, block, type, flags, c, &sc);
      uint8_t* out = codes + n * (K / 2) + b * (block / 2);
      for (int j = 0; j < block / 2; ++j) out[j] = (uint8_t)(c[2 * j] | (c[2 * j + 1] << 4));
      scales[n * nb + b] = (uint8_t)sc;
    }
  return 0;
}

int orc_mx_quantize(const void* x, int dtype, int64_t rows, int64_t cols, int64_t ld,
                    int axis, int type, unsigned flags, uint8_t* codes, uint8_t* scales) {
  return orc_mx_quantize_blk(x, dtype, rows, cols, ld, axis, type, flags, 32, codes, scales);
}

static double mx_value(int code, int X, int type) {
  if (type == ORC_MXFP4) {
    double v = ldexp(E2M1_GRID[code & 7], X);
    return (code & 8) ? -v : v;
  }
  int q = (code & 8) ? code - 16 : code;
  if (g_mutation == 19) return ldexp((double)q, X - 1);   /* planted: INT4 step of 2^(X-1) */
  return ldexp((double)q, X - 2);
}

int orc_mx_dequantize_blk(const uint8_t* codes, const uint8_t* scales, int64_t n_rows, int64_t k,
                          int type, int block, double* out) {
  if (k % 32 != 0 || (block != 32 && block != 16)) return 1;
  int64_t nb = k / block;
  for (int64_t n = 0; n < n_rows; ++n)
    for (int64_t kk = 0; kk < k; ++kk) {
      int X = (int)scales[n * nb + kk / block] - 127;
      out[n * k + kk] = mx_value(nibble(codes + n * (k / 2), kk), X, type);
    }
  return 0;
}

int orc_mx_dequantize(const uint8_t* codes, const uint8_t* scales, int64_t n_rows, int64_t k,
                      int type, double* out) {
  return orc_mx_dequantize_blk(codes, scales, n_rows, k, type, 32, out);
}

/* ----------------------------------------------------------------------- */
/* NVFP4 (a comparison format of the pages: blocks of 16 E2M1 elements, an  */
/* E4M3 block scale and one FP32 tensor scale)                              */
/* ----------------------------------------------------------------------- */

/* Value of a non-negative E4M3 code (no NaN: codes up to 0x7E). */
static double e4m3_value(int code) {
  int e = (code >> 3) & 15, m = code & 7;
  return e ? ldexp(1.0 + m / 8.0, e - 7) : ldexp(m / 8.0, -6);
}

/* E4M3 code nearest to t >= 0 (ties to the even code), saturating at 448. */
static int e4m3_code_of(double t) {
  if (!(t < 448.0)) return 0x7E;
  int best = 0;
  for (int c = 1; c <= 0x7E; ++c) {
    if (g_mutation == 11 && e4m3_value(c) > t) break;   /* planted: truncation */
    double e0 = fabs(t - e4m3_value(best)), e1 = fabs(t - e4m3_value(c));
    if (e1 < e0 || (e1 == e0 && (c & 1) == 0)) best = c;
  }
  return best;
}

/* x: rows x k (ld elements), k % 16 == 0.  All arithmetic is fp32 with one
 * rounding per operation, in this order:
 *   amax_t = the largest finite |x| of the tensor (NaN and +-Inf left out);
 *   amax_b = the block's largest |x| (NaN left out; +-Inf gives sb = 448);
 *   s_t    = amax_t / 2688 (2688 = 6 * 448; 1 when amax_t is 0; the smallest
 *            positive float if the quotient underflows), stored as fp32;
 *   per 16-block: t = (amax_b / s_t) / 6, its E4M3 code sb (nearest, ties
 *            even, saturating at 448);
 *   d = e4m3(sb) * s_t, and each element's E2M1 code of x / d (nearest,
 *            ties even, saturating at 6; NaN codes +0, +-Inf saturates).
 * A block whose sb is 0 stores zero codes.  codes rows x k/2, scales rows x
 * k/16 E4M3 bytes, *tensor_scale = s_t. */
int orc_nvfp4_quantize(const void* x, int dtype, int64_t rows, int64_t k, int64_t ld,
                       uint8_t* codes, uint8_t* scales, float* tensor_scale) {
  if (k % 16 != 0) return 1;
  float amax_t = 0.0f;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t i = 0; i < k; ++i) {
      double a = mag(load_elem(x, dtype, r * ld + i));
      if (!isinf(a) && (float)a > amax_t) amax_t = (float)a;
    }
  float s_t = 1.0f;
  if (amax_t > 0.0f) {
    volatile float q = amax_t / 2688.0f;
    s_t = q > 0.0f ? q : 0x1p-149f;
  }
  *tensor_scale = s_t;
  int64_t nb = k / 16;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t b = 0; b < nb; ++b) {
      float amax_b = 0.0f, v[16];
      for (int i = 0; i < 16; ++i) {
        v[i] = (float)load_elem(x, dtype, r * ld + b * 16 + i);
        double a = mag(v[i]);
        if ((float)a > amax_b) amax_b = (float)a;     /* +-Inf included: its block saturates */
      }
      volatile float t1 = amax_b / s_t;
      volatile float t = t1 / 6.0f;
      int sb = e4m3_code_of((double)t);
      scales[r * nb + b] = (uint8_t)sb;
      volatile float d = (float)e4m3_value(sb) * s_t;
      uint8_t* out = codes + r * (k / 2) + b * 8;
      for (int j = 0; j < 8; ++j) {
        int c[2];
        for (int h = 0; h < 2; ++h) {
          float xv = v[2 * j + h];
          if (sb == 0 || isnan(xv)) { c[h] = 0; continue; }
          if (isinf(xv)) { c[h] = (xv < 0 ? 8 : 0) | 7; continue; }
          volatile float y = xv / d;
          c[h] = e2m1_code((double)y);
        }
        out[j] = (uint8_t)(c[0] | (c[1] << 4));
      }
    }
  return 0;
}

int orc_nvfp4_dequantize(const uint8_t* codes, const uint8_t* scales, float tensor_scale, int64_t rows,
                         int64_t k, double* out) {
  if (k % 16 != 0) return 1;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t i = 0; i < k; ++i) {
      int c = nibble(codes + r * (k / 2), i);
      double g = E2M1_GRID[c & 7] * e4m3_value(scales[r * (k / 16) + i / 16]) * (double)tensor_scale;
      out[r * k + i] = (c & 8) ? -g : g;
    }
  return 0;
}

/* ----------------------------------------------------------------------- */
/* Dead-zone count: nonzero inputs whose code is zero                       */
/* ----------------------------------------------------------------------- */

/* Counts elements of x (rows x k, ld) that are finite and nonzero but whose
 * 4-bit code in `codes` (rows x k/2) is a zero code: MiX 0x7 (fmt 0), MXINT4
 * 0 (fmt 1), E2M1 +-0 for MXFP4 and NVFP4 (fmt 2). */
int64_t orc_underflow_count(const void* x, int dtype, int64_t rows, int64_t k, int64_t ld,
                            const uint8_t* codes, int fmt) {
  int64_t n = 0;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t i = 0; i < k; ++i) {
      double v = load_elem(x, dtype, r * ld + i);
      if (isnan(v) || (v == 0.0 && g_mutation != 16) || isinf(v)) continue;   /* 16 planted: zeros counted */
      int c = nibble(codes + r * (k / 2), i);
      int zero = fmt == 0 ? c == 0x7 : fmt == 1 ? c == 0 : (c & 7) == 0;
      n += zero;
    }
  return n;
}

/* ----------------------------------------------------------------------- */
/* A-MiX x W-MX block matmul, Eq. (6)                                       */
/* ----------------------------------------------------------------------- */

/* The W-MX element as an integer mantissa and a pre-shift: MXINT4 gives its
 * two's complement q with no shift (value q * 2^(X-2)); MXFP4 gives the E2M1
 * significand in half units (0/1 subnormal, 2/3 normal) and its exponent,
 * which Eq. (6) adds to the MiX element's delta-e before the shift
 * (value mant * 2^shift * 2^(X-1)). */
static void mx_int_parts(int code, int type, int* mant, int* shift) {
  if (type == ORC_MXINT4) { *mant = (code & 8) ? code - 16 : code; *shift = 0; return; }
  int e = (code >> 1) & 3, m = code & 1;
  int v = e ? (2 + m) : m;
  *mant = (code & 8) ? -v : v;
  *shift = e ? e - 1 : 0;
}

/* C[b, m, n] = sum over 32-blocks of
 *    (1.mshared) * 2^(Emax + X) * sum_i sign_i * w_i * 2^(-de_i)      (Eq. 6)
 * evaluated as an exact int64 shift-add per block (per 8-sub-block for T2,
 * each multiplied by its own 8 + m3), one multiply by the shared mantissa,
 * one exponent add, and an fp64 sum across blocks in K order.  With g16
 * weights (b_block 16) the block splits into its two 16-element halves, each
 * scaled by its own X: two exponent adds per 32-block, in K order.
 * A: batch x M x K MiX; B: (batch / b_group) x N x K MX.  Planes dense. */
int orc_gemm_blk(const uint8_t* a_codes, const void* a_shared, int a_type, int a_ebias,
                 const uint8_t* b_codes, const uint8_t* b_scales, int b_type, int b_block,
                 int64_t batch, int64_t b_group, int64_t M, int64_t N, int64_t K, double* c) {
  if (K % 32 != 0 || b_group < 1 || (b_block != 32 && b_block != 16)) return 1;
  int64_t nb = K / 32, nbb = K / b_block;
  int cB = (b_type == ORC_MXFP4) ? 1 : 2;
  size_t ssz = (a_type == ORC_T1) ? 1 : 2;
  for (int64_t bt = 0; bt < batch; ++bt) {
    const uint8_t* ac = a_codes + bt * M * (K / 2);
    const char* as = (const char*)a_shared + bt * M * nb * ssz;
    const uint8_t* bc = b_codes + (bt / b_group) * N * (K / 2);
    const uint8_t* bs = b_scales + (bt / b_group) * N * nbb;
    for (int64_t m = 0; m < M; ++m)
      for (int64_t n = 0; n < N; ++n) {
        double acc = 0.0;
        for (int64_t b = 0; b < nb; ++b) {
          int ec, m3s[4];
          mix_shared_fields(as, a_type, m * nb + b, &ec, m3s);
          int emax = ec + a_ebias;
          int64_t block = 0;
          for (int sb = 0; sb < 4; ++sb) {
            int64_t S = 0;                  /* shift-add tree of one sub-block */
            for (int i = 8 * sb; i < 8 * sb + 8; ++i) {
              int ca = nibble(ac + m * (K / 2), b * 32 + i);
              int cb = nibble(bc + n * (K / 2), b * 32 + i);
              int s = ca >> 3, d = ca & 7;
              if (d == 7 && s == 0) continue;          /* zero code */
              if (d == 7 && g_mutation == 17) continue;   /* planted: recycled -0 dropped */
              if (d == 7) s = 0;                       /* recycled -0: positive */
              int wm, ws;
              mx_int_parts(cb, b_type, &wm, &ws);
              /* w' 2^(7 - de + ws) as a product: a shift of a negative w' is not defined in C */
              int64_t t = (int64_t)wm * ((int64_t)1 << (7 - d + ws));
              if (g_mutation == 6) t = (int64_t)wm * ((int64_t)1 << (7 - d));   /* planted: FP4 exponent dropped */
              S += s ? -t : t;
            }
            block += S * (8 + m3s[g_mutation == 15 ? 0 : sb]);   /* x (1.mshared) in eighths */
            if (b_block == 16 && (sb & 1)) {  /* end of a 16-element half */
              int X = (int)bs[n * nbb + 2 * b + (g_mutation == 10 ? 0 : (sb >> 1))] - 127;
              acc += ldexp((double)block, emax + X - 10 - cB);
              block = 0;
            }
          }
          /* A = s (8+m3) 2^(Emax-3-de), B = w 2^ws 2^(X-cB): the block is
           * block * 2^(Emax + X - 10 - cB). */
          if (b_block == 32) acc += ldexp((double)block, emax + (int)bs[n * nbb + b] - 127 - 10 - cB);
        }
        c[(bt * M + m) * N + n] = acc;
      }
  }
  return 0;
}

int orc_gemm(const uint8_t* a_codes, const void* a_shared, int a_type, int a_ebias,
             const uint8_t* b_codes, const uint8_t* b_scales, int b_type,
             int64_t batch, int64_t b_group, int64_t M, int64_t N, int64_t K, double* c) {
  return orc_gemm_blk(a_codes, a_shared, a_type, a_ebias, b_codes, b_scales, b_type, 32, batch, b_group,
                      M, N, K, c);
}

/* ----------------------------------------------------------------------- */
/* K-smoothing (SageAttention): gamma(K) = K - mean_t(K)                     */
/* ----------------------------------------------------------------------- */

/* k: tokens x heads x head_dim (token stride ld elements).  mean: heads x
 * head_dim, the fp64 mean over tokens, summed in token order. */
int orc_ksmooth_mean(const void* k, int dtype, int64_t tokens, int heads, int head_dim,
                     int64_t ld, double* mean) {
  if (tokens <= 0) return 1;
  for (int h = 0; h < heads; ++h)
    for (int d = 0; d < head_dim; ++d) {
      double s = 0.0;
      for (int64_t t = 0; t < tokens; ++t) s += load_elem(k, dtype, t * ld + (int64_t)h * head_dim + d);
      mean[h * head_dim + d] = s / (double)tokens;
    }
  return 0;
}

/* K' = K - mu with K widened to fp32 and one fp32 subtraction (the difference
 * of two fp32 values formed exactly in fp64, then rounded once to fp32). */
int orc_ksmooth_apply(const void* k, int dtype, int64_t tokens, int heads, int head_dim,
                      int64_t ld, const float* mu, float* out) {
  for (int64_t t = 0; t < tokens; ++t)
    for (int h = 0; h < heads; ++h)
      for (int d = 0; d < head_dim; ++d) {
        double kv = load_elem(k, dtype, t * ld + (int64_t)h * head_dim + d);
        double m = (double)mu[h * head_dim + d];
        if (g_mutation == 7) m = -m;
        out[(t * heads + h) * head_dim + d] = (float)(kv - m);
      }
  return 0;
}
