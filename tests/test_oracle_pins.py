"""Pins for the CPU oracle: each checks it against something other than itself.

Sources (the MiX paper as digested on the pchao.org page
'MiX：面向端到端低比特视觉语言模型加速的微反缩放'):
  * section 方法概览 (Method), MiX-4.25b / MiX-4.5b bullets: bit layouts,
    dequantisation (-1)^s (1.mshared)_2 2^(Emax - de), de = 7 as zero;
  * same section, Algorithm 1 bullet: Emax from the block maximum, mshared from
    the maximum's mantissa, refinement over {de-1, de, de+1} for minimum error;
  * same section, Eq. (6) bullet: the factorised block dot product;
  * same section, accelerator bullet: asymmetric zero (the -0 code recycled
    for positives), K-smoothing gamma(K) = K - mean(K), softmax shift invariance;
  * section 关键结果 (Key results): about 40% of block maxima unrepresentable
    under the OCP floor rule for MXFP4.

Pins used: brute force with exact rationals (fractions.Fraction) over every
code, closed-form special values, invariants (round trip, softmax shift
invariance, zero-mean after smoothing), the printed bit accounting and the
printed ~40% statistic.  ``test_planted_mistakes_are_caught`` plants each of
the oracle's deliberate mutations and checks that some pin fails.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from quantized_vlm_gemm_mix_b300 import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(1234)


# ----------------------------------------------------------------------------
# Independent helpers written from the definitions (not from the oracle).
# ----------------------------------------------------------------------------

def bf16_to_fraction(bits: int) -> Fraction:
    """Exact value of a finite bf16 bit pattern, from the IEEE field definition."""
    s = (bits >> 15) & 1
    e = (bits >> 7) & 0xFF
    m = bits & 0x7F
    if e == 0:
        v = Fraction(m, 128) * Fraction(2) ** -126
    else:
        v = (1 + Fraction(m, 128)) * Fraction(2) ** (e - 127)
    return -v if s else v


def f32_to_fraction(x: float) -> Fraction:
    return Fraction(float(np.float32(x)))


def mix_code_value(code: int, emax: int, m3: int) -> Fraction:
    """Dequantisation rule of the Method section, with the recycled -0 code."""
    s, d = code >> 3, code & 7
    M = 1 + Fraction(m3, 8)
    if d == 7:
        return M * Fraction(2) ** (emax - 7) if s else Fraction(0)
    v = M * Fraction(2) ** (emax - d)
    return -v if s else v


def brute_mix_code(x: Fraction, emax: int, m3: int, asym: bool) -> int:
    """argmin over all 16 codes of |x - value|; ties to the larger magnitude,
    and between two zero codes to 0x7."""
    best = None
    for code in range(16):
        if code == 0xF and not asym:
            continue
        v = mix_code_value(code, emax, m3)
        key = (abs(x - v), -abs(v), code != 0x7)
        if best is None or key < best[0]:
            best = (key, code)
    return best[1]


def nearest_mantissa(amax: Fraction):
    """Round amax to 4 significant bits (nearest, ties to even); returns (f, m3)."""
    f = math.floor(math.log2(amax))
    while Fraction(2) ** f > amax:
        f -= 1
    while Fraction(2) ** (f + 1) <= amax:
        f += 1
    cands = [(Fraction(8 + j, 8) * Fraction(2) ** f, j) for j in range(9)]
    best = min(cands, key=lambda c: (abs(amax - c[0]), c[1] % 2))
    j = best[1]
    return (f + 1, 0) if j == 8 else (f, j)


def unpack_nibbles(codes: np.ndarray) -> np.ndarray:
    lo = codes & 0xF
    hi = codes >> 4
    return np.stack([lo, hi], axis=-1).reshape(codes.shape[0], -1)


def t1_fields(sh):
    return int(sh) & 0xF, [(int(sh) >> 4) & 7] * 4


def t2_fields(sh):
    sh = int(sh)
    return sh & 0xF, [(sh >> (4 + 3 * k)) & 7 for k in range(4)]


def e2m1_magnitudes():
    """E2M1 magnitudes from the field definition: e = 0 subnormal m * 0.5,
    else (1 + m/2) * 2^(e-1)."""
    out = []
    for code in range(8):
        e, m = code >> 1, code & 1
        out.append(Fraction(m, 2) if e == 0 else (1 + Fraction(m, 2)) * Fraction(2) ** (e - 1))
    return out


def random_bf16_block_bits(n_blocks, spread=12, zeros=0.1):
    """Random bf16 bit patterns with a wide exponent spread and some zeros."""
    exps = RNG.integers(127 - spread, 127 + 4, size=(n_blocks, 32))
    mant = RNG.integers(0, 128, size=(n_blocks, 32))
    sign = RNG.integers(0, 2, size=(n_blocks, 32))
    bits = (sign << 15) | (exps << 7) | mant
    bits[RNG.random((n_blocks, 32)) < zeros] = 0
    return bits.astype(np.uint16)


# ----------------------------------------------------------------------------
# Pins (plain functions so the planted-mistake test can re-run them).
# ----------------------------------------------------------------------------

def pin_bit_accounting(orc):
    g = json.load(open(os.path.join(GOLD, "bit_accounting.json")))
    rows, k = 8, 256
    x = synth.to_bf16_bits(synth.laplace(0, 1, rows * k, 0.3).reshape(rows, k))
    c1, s1 = orc.mix_quantize(x, orc.T1)
    c2, s2 = orc.mix_quantize(x, orc.T2)
    assert (c1.nbytes + s1.nbytes) * 8 == rows * k * g["mix_4p25"]["bits_per_element"]
    assert (c2.nbytes + s2.nbytes) * 8 == rows * k * g["mix_4p5"]["bits_per_element"]
    assert (c2.nbytes + s2.nbytes) * 8 // (rows * k // 32) == g["mix_4p5"]["bits_per_block"]
    # T1 shared field: Emax (4 bits) + mshared (3 bits) padded to 8 bits -> bit 7 unused
    assert int(np.max(s1)) < 128
    # T2: 4 + 4 x 3 bits occupy the whole 16-bit field, nothing more
    assert s2.dtype == np.uint16


def pin_dequant_special_values(orc):
    """Closed-form values of single codes: implicit leading one, de = 7 zero,
    one binade per de step, sign, and the recycled -0."""
    ebias = -8
    for ec in (0, 5, 8, 15):
        emax = ec + ebias
        for m3 in range(8):
            codes = np.zeros((1, 16), dtype=np.uint8)
            nib = [0x0, 0x1, 0x2, 0x3, 0x4, 0x5, 0x6, 0x7, 0x8, 0x9, 0xA, 0xE, 0xF] + [0x7] * 19
            for j in range(16):
                codes[0, j] = nib[2 * j] | (nib[2 * j + 1] << 4)
            sh = np.array([[ec | (m3 << 4)]], dtype=np.uint8)
            v = orc.mix_dequantize(codes, sh, orc.T1, ebias)[0]
            M = 1.0 + m3 / 8.0
            assert v[0] == M * 2.0 ** emax                   # de = 0 is the block maximum
            for d in range(6):
                assert v[d] == 2.0 * v[d + 1]                # one binade per de
            assert v[7] == 0.0                               # de = 7 encodes zero
            assert v[8] == -v[0] and v[9] == -v[1] and v[10] == -v[2] and v[11] == -v[6]
            assert v[12] == M * 2.0 ** (emax - 7) and v[12] > 0   # recycled -0
    # a worked value: m3 = 4 is (1.100)_2 = 1.5; Emax = 3, de = 2 -> 1.5 * 2 = 3
    codes = np.full((1, 16), 0x77, dtype=np.uint8)
    codes[0, 0] = 0x72
    sh = np.array([[(3 + 8) | (4 << 4)]], dtype=np.uint8)
    assert orc.mix_dequantize(codes, sh, orc.T1, -8)[0, 0] == 3.0


def pin_refinement_brute_force(orc, n_blocks=300):
    """Every element code is the exact minimum-error code (all 16 tried),
    and Emax / mshared come from the block (sub-block) maximum rounded to
    nearest-even at 4 significant bits."""
    bits = random_bf16_block_bits(n_blocks)
    for mix_type in (1, 2):
        for asym in (True, False):
            flags = 1 if asym else 0
            ebias = -12
            codes, shared = orc.mix_quantize(bits, mix_type, ebias, flags)
            nib = unpack_nibbles(codes)
            for b in range(n_blocks):
                xs = [bf16_to_fraction(int(v)) for v in bits[b]]
                ec, m3s = (t1_fields if mix_type == 1 else t2_fields)(shared[b, 0])
                amax = max(abs(v) for v in xs)
                if amax == 0:
                    assert all(int(c) == 7 for c in nib[b]) and ec == 0
                    continue
                f, m3 = nearest_mantissa(amax)
                emax = min(max(f, ebias), ebias + 15)
                all_zero = all(int(c) == 7 for c in nib[b])
                if not all_zero:
                    assert ec + ebias == emax
                for k in range(4):
                    sub = xs[8 * k:8 * k + 8]
                    smax = max(abs(v) for v in sub)
                    want_m3 = m3 if mix_type == 1 else (nearest_mantissa(smax)[1] if smax else 0)
                    sub_zero = all(int(c) == 7 for c in nib[b, 8 * k:8 * k + 8])
                    if (mix_type == 2 and sub_zero) or all_zero:
                        want_m3 = 0
                        assert m3s[k] == 0
                    else:
                        assert m3s[k] == want_m3
                    for i in range(8):
                        x = sub[i]
                        use_m3 = m3 if mix_type == 1 else (nearest_mantissa(smax)[1] if smax else 0)
                        want = brute_mix_code(x, emax, use_m3, asym)
                        assert int(nib[b, 8 * k + i]) == want, (b, k, i, x, emax, use_m3)


def pin_exhaustive_sweep(orc):
    """Every bf16 magnitude in [2^(Emax-10), 2^(Emax+1)) of either sign, for
    each of the 8 shared mantissas, as the second element of a block whose
    first element M * 2^Emax fixes the block maximum."""
    emax = 0
    xs = []
    for e in range(127 + emax - 10, 127 + emax + 1):
        for m in range(128):
            xs.append((e << 7) | m)
    xs = np.array(xs, dtype=np.uint16)
    for m3 in range(8):
        M_bits = ((127 + emax) << 7) | (m3 << 4)           # (1.m3) * 2^emax exactly
        Mv = bf16_to_fraction(M_bits)
        for sgn in (0, 0x8000):
            blk = np.full((len(xs), 32), 0, dtype=np.uint16)
            blk[:, 0] = M_bits
            blk[:, 1] = xs | sgn
            for mix_type in (1, 2):
                codes, shared = orc.mix_quantize(blk, mix_type, -8, 1)
                nib = unpack_nibbles(codes)
                for r in range(len(xs)):
                    x = bf16_to_fraction(int(blk[r, 1]))
                    if abs(x) > Mv:
                        continue                               # x became the maximum
                    want = brute_mix_code(x, emax, m3, True)
                    assert int(nib[r, 1]) == want, (m3, hex(int(blk[r, 1])))
                    assert int(nib[r, 0]) == 0                 # the maximum: de = 0


def pin_t2_shared_layout(orc):
    """The Type 2 shared half-word read by hand against the format's bit
    positions (Method section, MiX-4.5b bullet, for the fields; their order is
    the format's reading): Emax - ebias in bits 3..0, then the mshared of
    sub-blocks 0..3 in bits 6..4, 9..7, 12..10, 15..13."""
    ebias, ec = -8, 9
    m3 = [5, 2, 7, 1]
    word = ec | (m3[0] << 4) | (m3[1] << 7) | (m3[2] << 10) | (m3[3] << 13)
    codes = np.full((1, 16), 0x77, dtype=np.uint8)
    for k in range(4):
        codes[0, 4 * k] = 0x70                       # element 8k: de = 0, element 8k + 1: zero
    sh = np.array([[word]], dtype=np.uint16)
    v = orc.mix_dequantize(codes, sh, orc.T2, ebias)[0]
    for k in range(4):
        assert v[8 * k] == (1.0 + m3[k] / 8.0) * 2.0 ** (ec + ebias)
    # and the quantiser writes that layout: each sub-block's maximum is its own
    # (1.m3) 2^Emax, so the word comes back bit for bit
    x = np.zeros((1, 32), dtype=np.float32)
    for k in range(4):
        x[0, 8 * k] = (1.0 + m3[k] / 8.0) * 2.0 ** (ec + ebias)   # all in the binade of 2^(ec + ebias)
    c, s = orc.mix_quantize(x, orc.T2, ebias, 1)
    assert int(s[0, 0]) == word
    for k in range(4):
        assert c[0, 4 * k] == 0x70                  # de = 0 at element 8k, zero at 8k + 1


def pin_asymmetric_zero(orc):
    """The recycled -0 code gives positive values one more binade (accelerator
    bullet of the Method section)."""
    emax, m3 = 2, 5
    M = 1 + m3 / 8
    base = np.zeros((1, 32), dtype=np.float32)
    base[0, 0] = M * 2.0 ** emax
    vmin_pos = M * 2.0 ** (emax - 7)
    for x, asym, want in [
        (vmin_pos, True, 0xF),              # exactly the recycled level
        (vmin_pos * 0.51, True, 0xF),       # above half-way to zero
        (vmin_pos * 0.49, True, 0x7),       # below half-way: zero
        (-vmin_pos * 0.99, True, 0x7),      # negative side has no such level: zero
        (-vmin_pos, True, 0xE),             # half-way to -2*vmin: the tie goes to the larger
        (vmin_pos * 0.99, False, 0x7),      # flag off: nearest of {0, 2*vmin} is 0
        (vmin_pos, False, 0x6),             # flag off: the tie goes to de = 6
        (vmin_pos * 2.0, True, 0x6),
    ]:
        b = base.copy()
        b[0, 5] = x
        codes, _ = orc.mix_quantize(b, orc.T1, -8, 1 if asym else 0)
        got = unpack_nibbles(codes)[0, 5]
        assert int(got) == want, (x, asym, int(got), want)


def pin_round_trip(orc, n=400):
    """quantise(decode(c)) == c for canonical code blocks with a de = 0 element."""
    for mix_type in (1, 2):
        ebias = -8
        nib = RNG.integers(0, 16, size=(n, 32))
        nib[:, 0] = RNG.integers(0, 2, size=n) << 3        # a de = 0 element
        ec = RNG.integers(0, 16, size=n)
        m3 = RNG.integers(0, 8, size=(n, 4))
        if mix_type == 1:
            m3[:, 1:] = m3[:, :1]
        for b in range(n):                                  # canonical: all-zero sub-blocks
            for k in range(4):
                if mix_type == 2 and all(nib[b, 8 * k:8 * k + 8] == 7):
                    m3[b, k] = 0
        codes = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
        if mix_type == 1:
            sh = (ec | (m3[:, 0] << 4)).astype(np.uint8)[:, None]
        else:
            sh = (ec | (m3[:, 0] << 4) | (m3[:, 1] << 7) | (m3[:, 2] << 10) | (m3[:, 3] << 13)).astype(np.uint16)[:, None]
        v = orc.mix_dequantize(codes, sh, mix_type, ebias).astype(np.float32)
        c2, s2 = orc.mix_quantize(v, mix_type, ebias, 1)
        assert np.array_equal(c2, codes)
        assert np.array_equal(s2, sh)


def pin_nonfinite_and_zero_blocks(orc):
    x = np.zeros((3, 32), dtype=np.float32)
    x[0, 3] = np.nan                                     # NaN alone: zero block
    x[1, 0] = np.inf
    x[1, 1] = 1.0
    x[1, 2] = -np.inf
    x[2, :] = 1e-30                                      # far below 2^ebias: all zero codes
    codes, sh = orc.mix_quantize(x, orc.T1, -8, 1)
    nib = unpack_nibbles(codes)
    assert all(nib[0] == 7) and sh[0, 0] == 0
    assert nib[1, 0] == 0 and nib[1, 2] == 8 and (sh[1, 0] & 0xF) == 15
    assert all(nib[2] == 7) and sh[2, 0] == 0            # canonical zero block


def pin_e2m1_and_int4_brute_force(orc):
    grid = e2m1_magnitudes()
    assert [float(g) for g in grid] == [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    # a block whose maximum fixes X, then sweep the other elements
    vals = np.linspace(-7.5, 7.5, 961).astype(np.float32)
    for mx_type in (0, 1):
        nblk = (len(vals) + 30) // 31
        x = np.zeros((nblk, 32), dtype=np.float32)
        x[:, 0] = 4.0 if mx_type == 1 else 7.0               # X = 0 (FP4, floor rule) / X = 2 (INT4)
        flat = np.concatenate([vals, np.zeros(nblk * 31 - len(vals), np.float32)])
        x[:, 1:] = flat.reshape(nblk, 31)
        # the OCP floor rule keeps X = 0 for every block here, so the rounding
        # and the saturation above 6 are both exercised
        codes, scales = orc.mx_quantize(x, 1, mx_type, orc.MX_FLOOR if mx_type == 1 else 0)
        nib = unpack_nibbles(codes)
        for b in range(nblk):
            X = int(scales[b, 0]) - 127
            for i in range(1, 32):
                xv = Fraction(float(x[b, i]))
                if mx_type == 1:
                    assert X == 0
                    y = xv / Fraction(2) ** X
                    if abs(y) >= 6:
                        want = 7
                    else:
                        want = min(range(8), key=lambda c: (abs(abs(y) - grid[c]), c % 2))
                    want |= (8 if (y < 0 and want != 0) else 0)
                else:
                    assert X == 2
                    y = xv / Fraction(2) ** (X - 2)
                    q = round(y)                          # Python rounds half to even
                    q = max(-7, min(7, q))
                    want = q & 0xF
                assert int(nib[b, i]) == want, (mx_type, float(xv), int(nib[b, i]), want)


def pin_mx_scale_rule(orc):
    """About 40% of block maxima are unrepresentable under the floor rule; none
    under ceil (Key results section); ceil puts amax / 2^X in (2, 4]."""
    g = json.load(open(os.path.join(GOLD, "mxfp4_floor_rule.json")))
    w = synth.to_bf16_bits(synth.gaussian_weights(7, 3, 1024, 512))
    xf = synth.bf16_bits_to_f32(w).astype(np.float64)
    for flags, lo, hi in ((2, 0.35, 0.46), (0, 0.0, 0.0)):
        codes, scales = orc.mx_quantize(w, 0, orc.MXFP4, flags)
        X = scales.astype(np.int64) - 127                   # [N, K/32]
        amax = np.abs(xf).reshape(32, 32, 512).max(axis=1).T  # [N, K/32]
        frac = float(np.mean(amax / np.exp2(X) > 6.0))
        assert lo <= frac <= hi, (flags, frac)
        if flags == 0:
            r = amax / np.exp2(X)
            assert np.all((r > 2) & (r <= 4))
    assert abs(g["floor_unrepresentable_fraction_about"] - math.log2(2 / 1.5)) < 0.02


def pin_mx_axis_consistency(orc):
    x = synth.to_bf16_bits(synth.normal(3, 9, 96 * 160, 0, 0.02).reshape(96, 160))
    for t in (0, 1):
        c0, s0 = orc.mx_quantize(x, 0, t)                   # blocks down the columns
        c1, s1 = orc.mx_quantize(np.ascontiguousarray(x.T), 1, t)
        assert np.array_equal(c0, c1) and np.array_equal(s0, s1)


def frac_mx_value(code, scale, mx_type):
    X = int(scale) - 127
    if mx_type == 1:
        v = e2m1_magnitudes()[code & 7] * Fraction(2) ** X
        return -v if code & 8 else v
    q = code - 16 if code & 8 else code
    return q * Fraction(2) ** (X - 2)


def pin_gemm_eq6_exact(orc):
    """Eq. (6) evaluated as int64 shift-add equals the exact sum of products of
    dequantised values (the plain definition), on tiny matrices, exactly."""
    M, N, K = 3, 4, 96
    a = synth.to_bf16_bits(synth.vlm_activations(5, 0, M, K, visual_rows=2))
    w = synth.to_bf16_bits(synth.gaussian_weights(5, 1, K, N))
    for at in (1, 2):
        ac, ash = orc.mix_quantize(a, at, -8, 1)
        an = unpack_nibbles(ac)
        for bt in (0, 1):
            bc, bs = orc.mx_quantize(w, 0, bt)
            bn = unpack_nibbles(bc)
            c = orc.gemm(ac, ash, at, -8, bc, bs, bt)
            for m in range(M):
                for n in range(N):
                    tot = Fraction(0)
                    for kk in range(K):
                        ec, m3s = (t1_fields if at == 1 else t2_fields)(ash[m, kk // 32])
                        av = mix_code_value(int(an[m, kk]), ec - 8, m3s[(kk % 32) // 8])
                        bv = frac_mx_value(int(bn[n, kk]), bs[n, kk // 32], bt)
                        tot += av * bv
                    assert Fraction(c[m, n]) == tot, (at, bt, m, n)


def pin_gemm_against_dequant_matmul(orc):
    M, N, K = 24, 40, 320
    a = synth.to_f32(synth.vlm_activations(6, 0, M, K, visual_rows=16))
    w = synth.to_bf16_bits(synth.gaussian_weights(6, 1, K, N))
    for at in (1, 2):
        ac, ash = orc.mix_quantize(a, at, -8, 1)
        ad = orc.mix_dequantize(ac, ash, at, -8)
        for bt in (0, 1):
            bc, bs = orc.mx_quantize(w, 0, bt)
            bd = orc.mx_dequantize(bc, bs, bt)
            c = orc.gemm(ac, ash, at, -8, bc, bs, bt)
            ref = ad @ bd.T
            scale = np.abs(ad) @ np.abs(bd).T + 1e-300
            assert np.max(np.abs(c - ref) / scale) < 1e-13


def pin_gemm_reduces_to_mx_dot(orc):
    """m3 = 0 and every de = 0: each A element is +-2^Emax, so the product is a
    plain MX dot product with a sign vector."""
    N, K = 6, 64
    sgn = RNG.integers(0, 2, size=(1, K))
    a = np.where(sgn == 1, -1.0, 1.0).astype(np.float32) * 2.0
    w = synth.to_bf16_bits(synth.gaussian_weights(8, 1, K, N))
    ac, ash = orc.mix_quantize(a, orc.T1, -8, 1)
    assert np.all((unpack_nibbles(ac) & 7) == 0) and int(ash[0, 0]) >> 4 == 0
    for bt in (0, 1):
        bc, bs = orc.mx_quantize(w, 0, bt)
        bd = orc.mx_dequantize(bc, bs, bt)
        c = orc.gemm(ac, ash, orc.T1, -8, bc, bs, bt)
        want = np.array([sum(float(a[0, k]) * bd[n, k] for k in range(K)) for n in range(N)])
        assert np.array_equal(c[0], want)


def pin_gemm_batch_gqa_indexing(orc):
    B, G, M, N, K = 6, 3, 5, 7, 64
    a = synth.to_f32(synth.laplace(9, 0, B * M * K, 0.3).reshape(B * M, K))
    w = synth.to_bf16_bits(synth.normal(9, 1, (B // G) * N * K, 0, 0.02).reshape((B // G) * N, K))
    ac, ash = orc.mix_quantize(a, orc.T2, -8, 1)
    bc, bs = orc.mx_quantize(w, 1, orc.MXINT4)
    c = orc.gemm(ac.reshape(B, M, -1), ash.reshape(B, M, -1), orc.T2, -8,
                 bc.reshape(B // G, N, -1), bs.reshape(B // G, N, -1), orc.MXINT4, b_group=G)
    for b in range(B):
        g = b // G
        c2 = orc.gemm(ac[b * M:(b + 1) * M], ash[b * M:(b + 1) * M], orc.T2, -8,
                      bc[g * N:(g + 1) * N], bs[g * N:(g + 1) * N], orc.MXINT4)
        assert np.array_equal(c[b], c2)


def pin_ksmooth(orc):
    """gamma(K) = K - mean(K): zero mean per channel afterwards, exact means of
    closed-form inputs, and softmax(qK^T) unchanged (shift invariance)."""
    T, H, D = 64, 2, 32
    # closed form: K[t, h, d] = c[h, d] + t * delta (exact in fp32) -> mean = c + delta (T-1)/2
    c = np.arange(H * D, dtype=np.float32).reshape(H, D) * 0.25 - 3.0
    delta = np.float32(0.125)
    k = (c[None] + delta * np.arange(T, dtype=np.float32)[:, None, None]).astype(np.float32)
    mu = orc.ksmooth_mean(k)
    assert np.array_equal(mu, c.astype(np.float64) + float(delta) * (T - 1) / 2)
    q, kk, _ = synth.attention_qkv(11, T, q_heads=2, kv_heads=2, head_dim=D)
    kb = synth.to_bf16_bits(kk)
    mu = orc.ksmooth_mean(kb)
    ks = orc.ksmooth_apply(kb, mu.astype(np.float32))
    assert np.max(np.abs(ks.astype(np.float64).mean(axis=0))) < 1e-5 * np.max(np.abs(mu))
    kf = synth.bf16_bits_to_f32(kb).astype(np.float64)
    for h in range(2):
        s0 = q[:, h] @ kf[:, h].T
        s1 = q[:, h] @ (kf[:, h] - mu[h]).T
        p0 = np.exp(s0 - s0.max(1, keepdims=True)); p0 /= p0.sum(1, keepdims=True)
        p1 = np.exp(s1 - s1.max(1, keepdims=True)); p1 /= p1.sum(1, keepdims=True)
        assert np.max(np.abs(p0 - p1)) < 1e-12
    # a frozen mean (from a prefix of the tokens) is still a per-channel shift
    mu_f = orc.ksmooth_mean(kb[: T // 2])
    ks_f = orc.ksmooth_apply(kb, mu_f.astype(np.float32)).astype(np.float64)
    want = kf - mu_f.astype(np.float32).astype(np.float64)[None]
    assert np.max(np.abs(ks_f - want)) <= np.max(np.abs(want)) * 2.0 ** -23


def brute_mx_code(y: Fraction, mx_type: int) -> int:
    """Element code of y = x / 2^X (MXFP4) or x / 2^(X-2) (MXINT4), by search."""
    if mx_type == 1:
        grid = e2m1_magnitudes()
        if abs(y) >= 6:
            c = 7
        else:
            c = min(range(8), key=lambda j: (abs(abs(y) - grid[j]), j % 2))
        return c | (8 if (y < 0 and c != 0) else 0)
    q = max(-7, min(7, round(y)))                       # half to even
    return q & 0xF


def exact_f_m(a: Fraction):
    """a = m * 2^f with m in [1, 2), exactly."""
    f = 0
    while Fraction(2) ** f > a:
        f -= 1
    while Fraction(2) ** (f + 1) <= a:
        f += 1
    return f, a / Fraction(2) ** f


def pin_mx_tight_rule(orc):
    """The tight MX exponent, the ceil(log2(amax / 6)) alternative to the ceil
    rule (Key results section): the smallest X at which no element of the
    block saturates.  With amax = m 2^f, m in [1, 2), it has the closed forms
    MXFP4 X = f - 2 + [m > 1.5] and MXINT4 X = f + [m > 1.75] (elements
    q 2^(X-2), |q| <= 7); it is never above the ceil rule and at most one
    below it."""
    rng = np.random.default_rng(21)
    maxima = [m * 2.0 ** f for f in (-30, -3, 0, 7)
              for m in (1.0, 1.25, 1.5, 1.5 + 2 ** -7, 1.75, 1.75 + 2 ** -7, 2 - 2 ** -7)]
    x = (rng.uniform(-0.99, 0.99, (len(maxima), 32)) * np.array(maxima)[:, None]).astype(np.float32)
    for b, a in enumerate(maxima):
        x[b, rng.integers(32)] = a if b % 2 else -a
    w = synth.bf16_bits_to_f32(synth.to_bf16_bits(synth.gaussian_weights(5, 3, 256, 64)))
    for xx, brute in ((x, True), (w, False)):
        for mx_type, cap in ((1, Fraction(6)), (0, Fraction(7, 4))):
            codes, scales = orc.mx_quantize(xx, 1, mx_type, orc.MX_TIGHT)
            _, ceil_scales = orc.mx_quantize(xx, 1, mx_type, 0)
            nib = unpack_nibbles(codes)
            X_all = scales.astype(np.int64) - 127
            for r in range(xx.shape[0]):
                for b in range(xx.shape[1] // 32):
                    blk = [Fraction(float(v)) for v in xx[r, 32 * b: 32 * b + 32]]
                    amax = max(abs(v) for v in blk)
                    X = int(X_all[r, b])
                    f, m = exact_f_m(amax)
                    want = f - 2 + (m > Fraction(3, 2)) if mx_type == 1 else f + (m > Fraction(7, 4))
                    assert X == want, (mx_type, float(amax), X, want)
                    assert amax <= cap * Fraction(2) ** X < 2 * amax   # fits; X - 1 would not
                    dx = int(ceil_scales[r, b]) - 127 - X
                    assert dx in ((0, 1) if mx_type == 1 else (0, -1)), (mx_type, float(amax), dx)
                    if brute:
                        step = Fraction(2) ** (X if mx_type == 1 else X - 2)
                        for i in range(32):
                            assert int(nib[r, 32 * b + i]) == brute_mx_code(blk[i] / step, mx_type)
    # about log2(1.5) of gaussian block maxima move down one binade under MXFP4
    _, s_t = orc.mx_quantize(w, 1, 1, orc.MX_TIGHT)
    _, s_c = orc.mx_quantize(w, 1, 1, 0)
    frac = float(np.mean(s_t != s_c))
    assert 0.45 < frac < 0.72, frac
    with pytest.raises(ValueError):
        orc.mx_quantize(w, 1, 1, orc.MX_TIGHT | orc.MX_FLOOR)


def pin_auto_ebias(orc):
    """Automatic ebias: the largest block exponent (the block maximum rounded
    to a 3-bit mantissa, carry included, as in Algorithm 1) lands on the top
    4-bit code, so no block clamps from above and the range below it is the
    widest the 4-bit Emax field allows (Format section)."""
    x = np.zeros((3, 96), np.float32)
    x[0, 5] = 3.0                       # f = 1
    x[1, 40] = -2.0 ** -7
    x[2, 70] = 15.0                     # 1.875 * 2^3: f = 3, no carry
    assert orc.mix_auto_ebias(x) == 3 - 15
    x[2, 70] = 15.5                     # rounds to 16: the carry makes f = 4
    assert orc.mix_auto_ebias(x) == 4 - 15
    x[2, 70] = np.inf                   # saturates under any ebias; left out
    x[2, 71] = np.nan
    assert orc.mix_auto_ebias(x) == 1 - 15
    assert orc.mix_auto_ebias(np.zeros((2, 64), np.float32)) == -8
    x = np.zeros((1, 32), np.float32)
    x[0, 3] = -np.inf
    assert orc.mix_auto_ebias(x) == -8
    big = np.full((1, 32), 2.0 ** 120, np.float32)
    assert orc.mix_auto_ebias(big) == 100                  # clamped
    # brute force on a wide-range tensor, f32 and bf16 alike
    xa = synth.vlm_activations(4, 1, 64, 256, visual_rows=48, outlier_frac=0.01)
    xb = synth.to_bf16_bits(xa)
    for xx, vals in ((xa.astype(np.float32), xa.astype(np.float32)), (xb, synth.bf16_bits_to_f32(xb))):
        fs = []
        for r in range(vals.shape[0]):
            for b in range(vals.shape[1] // 32):
                amax = max(abs(Fraction(float(v))) for v in vals[r, 32 * b: 32 * b + 32])
                if amax:
                    fs.append(nearest_mantissa(amax)[0])
        eb = orc.mix_auto_ebias(xx)
        assert eb == max(fs) - 15
        for t in (1, 2):
            _, sh = orc.mix_quantize(xx, t, eb)
            assert int(np.max(sh.astype(np.int64) & 0xF)) == 15


def pin_mx_g16(orc):
    """MXINT4g16 / MXFP4g16 (Method and Key results sections: the weight
    formats of MiX-INT4g16 and the g16 MX baselines): one E8M0 scale per 16
    elements.  Every 16-element block obeys the 32-block rules (ceil for
    MXFP4, floor for MXINT4; element codes by brute force), and equals the
    32-block quantiser applied to that block padded with zeros."""
    w = synth.to_bf16_bits(synth.gaussian_weights(9, 4, 96, 40))        # K = 96, N = 40
    wf = synth.bf16_bits_to_f32(w)
    for t in (0, 1):
        for flags in (0, 4):
            c16, s16 = orc.mx_quantize(w, 0, t, flags, block=16)
            assert c16.shape == (40, 48) and s16.shape == (40, 6)
            nib = unpack_nibbles(c16)
            for n in range(40):
                for b in range(6):
                    blk = [Fraction(float(v)) for v in wf[16 * b: 16 * b + 16, n]]
                    pad = np.zeros((32, 1), np.float32)
                    pad[:16, 0] = wf[16 * b: 16 * b + 16, n]
                    cp, sp = orc.mx_quantize(pad, 0, t, flags)
                    assert s16[n, b] == sp[0, 0]
                    assert np.array_equal(nib[n, 16 * b: 16 * b + 16], unpack_nibbles(cp)[0, :16])
                    amax = max(abs(v) for v in blk)
                    f, m = exact_f_m(amax)
                    if flags == 0:
                        want = (f - 2 + (m > 1)) if t == 1 else f
                    else:
                        want = (f - 2 + (m > Fraction(3, 2))) if t == 1 else f + (m > Fraction(7, 4))
                    X = int(s16[n, b]) - 127
                    assert X == want
                    step = Fraction(2) ** (X if t == 1 else X - 2)
                    for i in range(16):
                        assert int(nib[n, 16 * b + i]) == brute_mx_code(blk[i] / step, t)
            d = orc.mx_dequantize(c16, s16, t, block=16)
            for n in range(0, 40, 7):
                for kk in range(96):
                    assert Fraction(d[n, kk]) == frac_mx_value(int(nib[n, kk]), s16[n, kk // 16], t)


def pin_gemm_g16(orc):
    """Eq. (6) with g16 weights: each 32-block of the MiX operand meets two
    weight scales, one per 16-element half.  Exact against the sum of
    products of dequantised values; equal to the 32-block matmul when both
    halves carry the 32-block's scale."""
    M, N, K = 3, 5, 96
    a = synth.to_bf16_bits(synth.vlm_activations(7, 0, M, K, visual_rows=2))
    w = synth.to_bf16_bits(synth.gaussian_weights(7, 1, K, N) * np.repeat(np.exp2(np.arange(6) % 4 - 1.5), 16)[:, None])
    for at in (1, 2):
        ac, ash = orc.mix_quantize(a, at, -8, 1)
        an = unpack_nibbles(ac)
        for bt in (0, 1):
            bc, bs = orc.mx_quantize(w, 0, bt, 0, block=16)
            assert np.any(bs[:, 0::2] != bs[:, 1::2])          # the halves' scales differ
            bn = unpack_nibbles(bc)
            c = orc.gemm(ac, ash, at, -8, bc, bs, bt, b_block=16)
            for m in range(M):
                for n in range(N):
                    tot, mag_sum = Fraction(0), Fraction(0)
                    for kk in range(K):
                        ec, m3s = (t1_fields if at == 1 else t2_fields)(ash[m, kk // 32])
                        av = mix_code_value(int(an[m, kk]), ec - 8, m3s[(kk % 32) // 8])
                        p = av * frac_mx_value(int(bn[n, kk]), bs[n, kk // 16], bt)
                        tot += p
                        mag_sum += abs(p)
                    # half-block sums are exact; only the fp64 additions across them round
                    assert abs(Fraction(c[m, n]) - tot) <= mag_sum * Fraction(1, 2 ** 50), (at, bt, m, n)
            bc32, bs32 = orc.mx_quantize(w, 0, bt)
            c32 = orc.gemm(ac, ash, at, -8, bc32, bs32, bt)
            c16 = orc.gemm(ac, ash, at, -8, bc32, np.repeat(bs32, 2, axis=1), bt, b_block=16)
            assert np.max(np.abs(c16 - c32)) <= np.max(np.abs(c32)) * 2.0 ** -50


def e4m3_magnitudes():
    """Every finite non-negative E4M3 value by code (0 .. 0x7E), exactly."""
    out = []
    for c in range(0x7F):
        e, m = c >> 3, c & 7
        out.append(Fraction(m, 8) * Fraction(2) ** -6 if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7))
    return out


def brute_e4m3(t: Fraction) -> int:
    vals = e4m3_magnitudes()
    if t >= 448:
        return 0x7E
    return min(range(0x7F), key=lambda c: (abs(t - vals[c]), c % 2))


def pin_nvfp4(orc):
    """NVFP4 (named by the pages as the 16-element, E4M3-block-scale,
    FP32-tensor-scale comparison format): block scales are the nearest E4M3
    (ties even, saturating) of (amax_b / s_t) / 6 with s_t = amax_t / 2688;
    elements the nearest E2M1 of x / (e4m3(sb) s_t).  Checked by enumerating
    both grids on exact rationals, by scale equivariance and by the
    reconstruction bound."""
    vals = e4m3_magnitudes()
    # an anchor element 2688 makes s_t exactly 1, so t = amax_b / 6 exactly;
    # targets: every E4M3 value, every midpoint between neighbours, and
    # points just off the midpoints
    targets = []
    for c in range(0x7E):
        lo, hi = vals[c], vals[c + 1]
        mid = (lo + hi) / 2
        targets += [lo, mid, mid + (hi - lo) / 64, mid - (hi - lo) / 64]
    targets += [Fraction(448)]
    nb = len(targets) + 1
    x = np.zeros((1, 16 * nb), np.float32)
    x[0, 0] = 2688.0
    for i, t in enumerate(targets):
        x[0, 16 * (i + 1) + 5] = np.float32(float(6 * t))
        assert Fraction(float(x[0, 16 * (i + 1) + 5])) == 6 * t      # exactly representable
    codes, scales, ts = orc.nvfp4_quantize(x)
    assert ts == np.float32(1.0)
    for i, t in enumerate(targets):
        assert int(scales[0, i + 1]) == brute_e4m3(t), (float(t), int(scales[0, i + 1]), brute_e4m3(t))
    # element codes on random blocks (general s_t), both grids by enumeration
    rng = np.random.default_rng(41)
    xr = (rng.standard_normal((6, 64)) * np.exp2(rng.integers(-8, 8, (6, 1)))).astype(np.float32)
    xr[2, 5] = 0.0
    codes, scales, ts = orc.nvfp4_quantize(xr)
    amax_t = np.float32(np.max(np.abs(xr)))
    assert ts == np.float32(amax_t / np.float32(2688.0))
    grid = e2m1_magnitudes()
    nib = unpack_nibbles(codes)
    for r in range(6):
        for b in range(4):
            blk = xr[r, 16 * b: 16 * b + 16]
            t = np.float32(np.float32(np.max(np.abs(blk)) / ts) / np.float32(6.0))
            sb = brute_e4m3(Fraction(float(t)))
            assert int(scales[r, b]) == sb
            d = np.float32(np.float32(float(vals[sb])) * ts)
            for i in range(16):
                y = Fraction(float(np.float32(blk[i] / d)))
                c = 7 if abs(y) >= 6 else min(range(8), key=lambda j: (abs(abs(y) - grid[j]), j % 2))
                want = c | (8 if (y < 0 and c) else 0)
                assert int(nib[r, 16 * b + i]) == want
    # scale equivariance: x 2^j keeps codes and block scales, s_t scales exactly
    for j in (-20, 3, 40):
        c2, s2, t2 = orc.nvfp4_quantize((xr * np.float32(2.0 ** j)).astype(np.float32))
        assert np.array_equal(c2, codes) and np.array_equal(s2, scales) and t2 == np.float32(ts * 2.0 ** j)
    # reconstruction: within half an E2M1 step (at most 1 unit of d) plus saturation
    deq = orc.nvfp4_dequantize(codes, scales, ts)
    for r in range(6):
        for b in range(4):
            d = float(vals[int(scales[r, b])]) * float(ts)
            err = np.abs(deq[r, 16 * b: 16 * b + 16] - xr[r, 16 * b: 16 * b + 16].astype(np.float64))
            assert np.all(err <= d * 1.0 + 1e-30)
    # +-Inf saturates its block, NaN codes zero, an all-zero tensor gives s_t = 1
    xs = np.zeros((1, 32), np.float32)
    xs[0, 3], xs[0, 4], xs[0, 20] = np.inf, np.nan, 1.0
    c3, s3, t3 = orc.nvfp4_quantize(xs)
    n3 = unpack_nibbles(c3)
    assert t3 == np.float32(1.0 / 2688.0) and int(s3[0, 0]) == 0x7E and n3[0, 3] == 7 and n3[0, 4] == 0
    assert orc.nvfp4_quantize(np.zeros((2, 32), np.float32))[2] == np.float32(1.0)


def pin_underflow_count(orc):
    """The dead-zone count (Key results section's key-underflow comparison,
    made synthetic): finite nonzero inputs whose code is a zero code, equal to
    the count of nonzero inputs that dequantise to exactly zero, per format;
    and a hand-counted MXFP4 block."""
    x = np.zeros((1, 32), np.float32)
    x[0, :6] = [4.0, 0.2, 0.24, 0.26, -0.25, 0.0]          # X = 0: 0.2, 0.24 and -0.25 fall to zero
    c, s = orc.mx_quantize(x, 1, 1)
    assert orc.underflow_count(x, c, orc.UF_E2M1) == 3
    a = synth.attention_qkv(3, 256, n_outlier=4)[1].reshape(-1, 128)           # K [tokens * heads, 128]
    a = synth.to_bf16_bits(a)
    af = synth.bf16_bits_to_f32(a).astype(np.float64)
    nz = (af != 0)
    for fmt, codes, deq in (
            (orc.UF_MIX,) + (lambda cs: (cs[0], orc.mix_dequantize(cs[0], cs[1], 2, -8)))(orc.mix_quantize(a, 2)),
            (orc.UF_MXINT4,) + (lambda cs: (cs[0], orc.mx_dequantize(cs[0], cs[1], 0)))(orc.mx_quantize(a, 1, 0)),
            (orc.UF_E2M1,) + (lambda cs: (cs[0], orc.mx_dequantize(cs[0], cs[1], 1)))(orc.mx_quantize(a, 1, 1)),
            (orc.UF_E2M1,) + (lambda cs: (cs[0], orc.nvfp4_dequantize(*cs)))(orc.nvfp4_quantize(a))):
        n = orc.underflow_count(a, codes, fmt)
        assert n == int(np.sum(nz & (deq == 0))), fmt
        assert n > 0


def pin_decode_attention(orc):
    """One decode step composed in the pages' order (frozen-mean K-smoothing
    on append, Q-K^T, softmax, MiX requantisation of P, P-V): S and O equal
    the fp64 products of the dequantised planes with head h reading KV head
    h // G; P is a softmax (rows sum to 1, shift-invariant); the appended K'
    row dequantises to fp32(k_new) - mean within half an MXINT4 step."""
    HQ, HK, D, T = 6, 2, 128, 80
    G = HQ // HK
    q, k, v = synth.attention_qkv(9, T, q_heads=HQ, kv_heads=HK, head_dim=D)
    mean = orc.ksmooth_mean(synth.to_bf16_bits(k[:48]))
    kp = orc.ksmooth_apply(synth.to_bf16_bits(k[:T - 1]), mean.astype(np.float32))
    kc = np.zeros((T, HK, D // 2), np.uint8)
    ks = np.zeros((T, HK, D // 32), np.uint8)
    c, s = orc.mx_quantize(kp.reshape(-1, D).astype(np.float32), 1, 0)
    kc[:T - 1], ks[:T - 1] = c.reshape(T - 1, HK, -1), s.reshape(T - 1, HK, -1)
    Tv = 96
    vv = np.zeros((Tv, HK, D))
    vv[:T] = v
    vc, vs = orc.mx_quantize(synth.to_bf16_bits(vv.reshape(Tv, HK * D)), 0, 0)   # [HK*D, Tv/2]
    vc, vs = vc.reshape(HK, D, -1), vs.reshape(HK, D, -1)
    qb = synth.to_bf16_bits(q[T - 1])
    kn = synth.to_bf16_bits(k[T - 1])
    O, Pm, (pc, ps), S = orc.decode_attention(qb, kc, ks, vc, vs, T, 0.088, k_new=kn, k_mean=mean)
    # the appended row
    kd = orc.mx_dequantize(kc[T - 1], ks[T - 1], 0)
    want = synth.bf16_bits_to_f32(kn).astype(np.float64) - mean.astype(np.float32).astype(np.float64)
    step = np.exp2(ks[T - 1].astype(np.float64) - 127 - 2).repeat(32, axis=1)
    sat = np.abs(want) > 7 * step                     # above the largest level 7 * 2^(X-2)
    err = np.abs(kd - want)
    assert np.all(err[~sat] <= step[~sat] / 2 + 1e-12) and np.all(err[sat] < step[sat])
    # S and O against dequantised planes
    qc, qs = orc.mix_quantize(qb, 2, -8)
    qd = orc.mix_dequantize(qc, qs, 2, -8)
    pd = orc.mix_dequantize(pc, ps, 2, -15)
    for h in range(HQ):
        g = h // G
        kdq = orc.mx_dequantize(np.ascontiguousarray(kc[:T, g]), np.ascontiguousarray(ks[:T, g]), 0)
        assert np.max(np.abs(S[h] - kdq @ qd[h])) <= 1e-12 * np.max(np.abs(S[h]))
        vdq = orc.mx_dequantize(vc[g], vs[g], 0)                    # [D, Tv]
        assert np.max(np.abs(O[h] - vdq @ pd[h])) <= 1e-12 * np.max(np.abs(O[h]))
    # softmax properties
    assert np.all(np.abs(Pm.astype(np.float64).sum(axis=1) - 1.0) < 1e-5)
    assert np.all(pd[:, T:] == 0)
    z = S * 0.088
    e = np.exp(z + 7.0 - (z + 7.0).max(axis=1, keepdims=True))
    assert np.allclose(e / e.sum(axis=1, keepdims=True), Pm, rtol=1e-6, atol=1e-12)


def pin_clamp_count(orc):
    """The clamped-block count against blocks built by hand and against an
    independent restatement in Python: the block exponent is the floor of
    log2 of the maximum, plus one when rounding its mantissa to three bits
    (half to even, Python's round) carries out."""
    import math
    ebias = -8
    # hand-built blocks: (block values, expected (high, low))
    cases = [
        ([1.875 * 2.0 ** 7], (0, 0)),          # f = 7 = ebias + 15: top code, not clamped
        ([1.9375 * 2.0 ** 7], (1, 0)),         # rounds to 2^8: carried past the top
        ([2.0 ** 8], (1, 0)),
        ([2.0 ** -8], (0, 0)),                 # f = ebias: bottom code
        ([1.9375 * 2.0 ** -9], (0, 0)),        # rounds up to 2^-8: carried into range
        ([1.875 * 2.0 ** -9], (0, 1)),
        ([2.0 ** -140], (0, 1)),               # fp32 subnormal
        ([np.inf], (1, 0)),
        ([-np.inf, 1.0], (1, 0)),
        ([np.nan], (0, 0)),                    # NaN counts as zero
        ([0.0], (0, 0)),
        ([-3.0 * 2.0 ** 9, 1.0], (1, 0)),
    ]
    for vals, want in cases:
        x = np.zeros((1, 32), np.float32)
        x[0, :len(vals)] = vals
        assert orc.mix_clamp_count(x, ebias) == want, (vals, want)
    # random blocks over a wide exponent range, fp32 and bf16, several ebias
    rng = np.random.default_rng(21)
    x = (rng.standard_normal((64, 256)) * np.exp2(rng.integers(-30, 30, (64, 256)))).astype(np.float32)
    x[3, :32] = 0.0
    for eb in (-15, -8, 0):
        for arr in (x, synth.to_bf16_bits(x.astype(np.float64))):
            vals = synth.bf16_bits_to_f32(arr) if arr.dtype == np.uint16 else arr
            hi = lo = 0
            for blk in vals.reshape(-1, 32).astype(np.float64):
                amax = float(np.max(np.abs(blk)))
                if amax == 0.0:
                    continue
                m, e = math.frexp(amax)           # amax = m 2^e, m in [0.5, 1)
                f = e - 1
                if round((2.0 * m - 1.0) * 8.0) == 8:
                    f += 1
                hi += f > eb + 15
                lo += f < eb
            assert orc.mix_clamp_count(arr, eb) == (hi, lo), eb


ALL_PINS = [pin_bit_accounting, pin_dequant_special_values, pin_refinement_brute_force,
            pin_exhaustive_sweep, pin_asymmetric_zero, pin_round_trip,
            pin_nonfinite_and_zero_blocks, pin_e2m1_and_int4_brute_force, pin_mx_scale_rule,
            pin_mx_axis_consistency, pin_gemm_eq6_exact, pin_gemm_against_dequant_matmul,
            pin_gemm_reduces_to_mx_dot, pin_gemm_batch_gqa_indexing, pin_ksmooth,
            pin_mx_tight_rule, pin_auto_ebias, pin_mx_g16, pin_gemm_g16, pin_nvfp4, pin_underflow_count,
            pin_decode_attention, pin_t2_shared_layout, pin_clamp_count]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    orc.set_mutation(0)
    pin(orc)


# Mutations planted in the oracle (see orc_set_mutation): 1 mshared truncated
# instead of rounded, 2 implicit leading one dropped, 3 naive de off by one,
# 4 refinement search removed, 5 MXFP4 floor instead of ceil, 6 FP4 exponent
# dropped from the Eq. (6) shift, 7 smoothing adds the mean, 8 the tight MX
# exponent steps past a block maximum on the boundary, 9 the automatic ebias
# drops the rounding carry, 10 the g16 matmul reads the first half's scale
# for both halves, 11 the E4M3 rounding of the NVFP4 block scale truncates,
# 12 a Type 2 sub-block takes its mantissa from the whole block's maximum,
# 13 the recycled -0 decodes as a negative value, 14 MXINT4 saturates at 8
# (which wraps to the code of -8), 15 the Type 2 matmul scales every
# sub-block by sub-block 0's mantissa, 16 the underflow count also counts
# elements that were zero before quantisation, 17 the matmul drops the
# recycled -0 as if it coded zero, 18 element nibbles are packed high nibble
# first, 19 the MXINT4 element step is 2^(X-1) instead of 2^(X-2), 20 the
# Type 2 sub-block mantissas are packed and unpacked in reverse order, 21 the
# clamped-block count ignores the mantissa rounding's carry.
FAST_PINS = [pin_dequant_special_values, pin_round_trip, pin_asymmetric_zero,
             pin_e2m1_and_int4_brute_force, pin_mx_scale_rule, pin_gemm_eq6_exact,
             pin_gemm_against_dequant_matmul, pin_ksmooth, pin_nonfinite_and_zero_blocks,
             pin_mx_tight_rule, pin_auto_ebias, pin_gemm_g16, pin_nvfp4, pin_underflow_count,
             pin_t2_shared_layout, pin_clamp_count,
             lambda o: pin_refinement_brute_force(o, n_blocks=40)]


@pytest.mark.parametrize("mutation", list(range(1, 22)))
def test_planted_mistakes_are_caught(orc, mutation):
    failed = []
    try:
        orc.set_mutation(mutation)
        for pin in FAST_PINS:
            try:
                pin(orc)
            except AssertionError:
                failed.append(getattr(pin, "__name__", "pin"))
    finally:
        orc.set_mutation(0)
    assert failed, f"mutation {mutation} slipped through every pin"


def test_synthetic_activation_ratio():
    """Visual vs text mean |x| follows the Fig. 1 statistics (about 34x)."""
    g = json.load(open(os.path.join(GOLD, "activation_stats.json")))
    x = synth.vlm_activations(0, 0, 512, 512, visual_rows=384, outlier_frac=0.0)
    r = np.abs(x[:384]).mean() / np.abs(x[384:]).mean()
    assert abs(r - g["ratio_about"]) < 3.0
