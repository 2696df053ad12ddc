"""GPU parity of the quantiser kernels against the CPU oracle: bit-exact codes
and packed bytes (MiX-4.25b / MiX-4.5b, MXINT4 / MXFP4 along rows and down
columns), on the paper-shaped workloads and on edge cases."""
import numpy as np
import pytest

from quantized_vlm_gemm_mix_b300 import synth
from helpers import to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mix():
    import torch
    assert torch.cuda.is_available()
    from quantized_vlm_gemm_mix_b300 import mix as m
    return m


def gpu_mix(mix, x_np, mix_type, ebias=-8, flags=1):
    codes, shared = mix.quantize_mix(to_dev(x_np), mix_type, ebias, flags)
    return to_host(codes), to_host(shared)


def check_mix(mix, orc, x_np, mix_type, ebias=-8, flags=1):
    c_ref, s_ref = orc.mix_quantize(x_np, mix_type, ebias, flags)
    c, s = gpu_mix(mix, x_np, mix_type, ebias, flags)
    assert np.array_equal(c, c_ref), f"codes differ at {np.argwhere(c != c_ref)[:5]}"
    assert np.array_equal(s.astype(s_ref.dtype), s_ref), f"shared differs at {np.argwhere(s != s_ref)[:5]}"


# ---------------------------------------------------------------------------
# MiX


def test_mix_tiny_fp32_config(mix, orc):
    """fp32 A [128 x 512]: visual rows with 4 outlier channels x30, text rows."""
    a = synth.to_f32(synth.vlm_activations(0, 0, 128, 512, visual_rows=96, n_outlier=4))
    for t in (1, 2):
        check_mix(mix, orc, a, t)


@pytest.mark.parametrize("t", [1, 2])
def test_mix_quantizer_sweep_bf16_full(mix, orc, t):
    """bf16 activations 4096 x 3584 (3072 visual rows, 1% outlier channels x30)."""
    a = synth.to_bf16_bits(synth.vlm_activations(0, 1, 4096, 3584, visual_rows=3072))
    check_mix(mix, orc, a, t)


@pytest.mark.parametrize("rows,k", [(1, 32), (3, 96), (7, 160), (33, 224), (5, 4128)])
@pytest.mark.parametrize("t", [1, 2])
@pytest.mark.parametrize("asym", [0, 1])
def test_mix_ragged_shapes(mix, orc, rows, k, t, asym):
    a = synth.to_bf16_bits(synth.vlm_activations(3, rows, rows, k, visual_rows=rows // 2 + 1))
    check_mix(mix, orc, a, t, flags=asym)
    f = synth.to_f32(synth.laplace(4, rows, rows * k, 0.5).reshape(rows, k))
    check_mix(mix, orc, f, t, ebias=-12, flags=asym)


def test_mix_edge_values(mix, orc):
    """Zeros, NaN, +-Inf, subnormals, saturation above 2^(ebias+15), values far
    below 2^ebias, and every bf16 magnitude of a 12-binade window."""
    rng = np.random.default_rng(5)
    blocks = []
    z = np.zeros(32, np.float32)
    blocks.append(z.copy())
    b = z.copy(); b[3] = np.nan; blocks.append(b)
    b = z.copy(); b[0] = np.inf; b[1] = -np.inf; b[2] = 1.0; b[5] = np.nan; blocks.append(b)
    b = (rng.standard_normal(32) * 1e-41).astype(np.float32); blocks.append(b)       # subnormal fp32
    b = (rng.standard_normal(32) * 1e6).astype(np.float32); blocks.append(b)         # saturates
    b = (rng.standard_normal(32) * 1e-9).astype(np.float32); blocks.append(b)        # under 2^ebias
    b = z.copy(); b[:8] = 1e-30; b[8:] = rng.standard_normal(24); blocks.append(b)   # one dead sub-block
    b = z.copy(); b[0] = 1.9375; b[1:] = rng.standard_normal(31) * 0.1; blocks.append(b)  # carry
    x = np.stack(blocks).astype(np.float32)
    for t in (1, 2):
        for flags in (0, 1):
            check_mix(mix, orc, x, t, flags=flags)
            check_mix(mix, orc, x, t, ebias=-100, flags=flags)
            check_mix(mix, orc, x, t, ebias=100, flags=flags)
    bits = np.arange(0x3A00, 0x4000 + 0x600, dtype=np.uint32)
    bits = np.concatenate([bits, bits | 0x8000]).astype(np.uint16)
    bits = bits[: (len(bits) // 31) * 31].reshape(-1, 31)
    for m3 in range(8):
        head = np.full((bits.shape[0], 1), (127 << 7) | (m3 << 4), dtype=np.uint16)
        xb = np.concatenate([head, bits], axis=1)
        for t in (1, 2):
            check_mix(mix, orc, xb, t)


def test_mix_every_bf16_pattern(mix, orc):
    """All 65536 bf16 bit patterns (NaNs, +-Inf, +-0, subnormals, every
    magnitude) through the bf16 quantiser, bit-exact against the oracle: once
    shuffled together (most blocks then hold a NaN: the scalar path), once
    without NaNs (every block on the packed two-elements-per-word path); both
    types, both zero modes, ebias at both ends of its range and in between."""
    rng = np.random.default_rng(11)
    every = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    no_nan = every[(every & 0x7FFF) <= 0x7F80]
    mixed = rng.permutation(every).reshape(256, 256)
    clean = rng.permutation(no_nan)
    clean = clean[: (clean.size // 256) * 256].reshape(-1, 256)
    # blocks of one binade band each, so many blocks neither saturate nor flush
    banded = np.sort(clean.reshape(-1) & 0x7FFF).astype(np.uint16)
    banded = (banded[: (banded.size // 256) * 256] | (rng.integers(0, 2, banded.size // 256 * 256) << 15)
              ).astype(np.uint16).reshape(-1, 256)
    for x in (mixed, clean, banded):
        for t in (1, 2):
            for flags in (0, 1):
                for ebias in (-100, -8, 30, 100):
                    check_mix(mix, orc, x, t, ebias=ebias, flags=flags)


def test_mix_strided_input(mix, orc):
    import torch
    a = synth.to_bf16_bits(synth.vlm_activations(8, 0, 64, 512, visual_rows=48))
    big = np.zeros((64, 640), np.uint16)
    big[:, :512] = a
    x = to_dev(big)
    codes = torch.empty((64, 256), dtype=torch.uint8, device="cuda")
    shared = torch.empty((64, 16), dtype=torch.int16, device="cuda")
    mix.mix_quantize(x, 64, 512, 640, mix.MIX_T2_4P5, -8, 1, codes, shared)
    c_ref, s_ref = orc.mix_quantize(a, 2)
    assert np.array_equal(to_host(codes), c_ref) and np.array_equal(to_host(shared), s_ref)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("rows,k", [(777, 96), (1, 32032), (4099, 160)])
def test_mix_contiguous_and_strided_paths(mix, orc, dtype, rows, k):
    """A contiguous x goes through the TMA-fed kernel (several chunks, an odd
    block count whose last bf16 block lies past the last whole 128-byte row);
    the same values in a strided buffer through the direct-load kernel.  Both
    equal the oracle bit for bit."""
    import torch
    a = synth.vlm_activations(12, rows, rows, k, visual_rows=rows // 2 + 1)
    a = synth.to_bf16_bits(a) if dtype == "bf16" else synth.to_f32(a)
    for t in (1, 2):
        check_mix(mix, orc, a, t)
        big = np.zeros((rows, k + 64), a.dtype)
        big[:, :k] = a
        x = to_dev(big)
        codes = torch.empty((rows, k // 2), dtype=torch.uint8, device="cuda")
        shared = torch.empty((rows, k // 32), dtype=torch.int16 if t == 2 else torch.uint8, device="cuda")
        mix.mix_quantize(x, rows, k, k + 64, t, -8, 1, codes, shared)
        c_ref, s_ref = orc.mix_quantize(a, t)
        assert np.array_equal(to_host(codes), c_ref)
        assert np.array_equal(to_host(shared).astype(s_ref.dtype), s_ref)
    assert mix.mix_device_error() == 0


def test_mix_dequantize_matches_oracle(mix, orc):
    import torch
    a = synth.to_bf16_bits(synth.vlm_activations(9, 0, 64, 256, visual_rows=40))
    for t in (1, 2):
        c, s = orc.mix_quantize(a, t)
        out = torch.empty((64, 256), dtype=torch.float32, device="cuda")
        mix.mix_dequantize(to_dev(c), to_dev(s), 64, 256, t, -8, out)
        assert np.array_equal(to_host(out).astype(np.float64), orc.mix_dequantize(c, s, t))


# ---------------------------------------------------------------------------
# MX


def check_mx(mix, orc, x_np, axis, t, flags=0):
    c_ref, s_ref = orc.mx_quantize(x_np, axis, t, flags)
    c, s = mix.quantize_mx(to_dev(x_np), axis, t, flags)
    c, s = to_host(c), to_host(s)
    assert np.array_equal(c, c_ref), f"codes differ at {np.argwhere(c != c_ref)[:5]}"
    assert np.array_equal(s, s_ref), f"scales differ at {np.argwhere(s != s_ref)[:5]}"


@pytest.mark.parametrize("axis", [0, 1])
@pytest.mark.parametrize("t", [0, 1])
def test_mx_tiny_weights(mix, orc, axis, t):
    w = synth.to_f32(synth.gaussian_weights(0, 2, 512, 256))
    x = w if axis == 0 else np.ascontiguousarray(w.T)
    check_mx(mix, orc, x, axis, t)
    check_mx(mix, orc, x, axis, t, flags=2)
    check_mx(mix, orc, x, axis, t, flags=4)


@pytest.mark.parametrize("t", [0, 1])
def test_mx_sweep_weights_full_sampled(mix, orc, t):
    """bf16 W 3584 x 18944 quantised down its columns on the GPU; every code of
    a sampled set of 512 columns checked against the oracle."""
    w = synth.to_bf16_bits(synth.gaussian_weights(0, 3, 3584, 18944))
    c, s = mix.quantize_mx(to_dev(w), 0, t)
    c, s = to_host(c), to_host(s)
    cols = np.sort(np.random.default_rng(0).choice(18944, 512, replace=False))
    c_ref, s_ref = orc.mx_quantize(np.ascontiguousarray(w[:, cols]), 0, t)
    assert np.array_equal(c[cols], c_ref) and np.array_equal(s[cols], s_ref)


@pytest.mark.parametrize("shape", [(32, 1), (64, 63), (96, 130), (4128, 5)])
@pytest.mark.parametrize("t", [0, 1])
def test_mx_cols_ragged(mix, orc, shape, t):
    kdim, n = shape
    ldn = (n + 7) // 8 * 8
    w = synth.to_bf16_bits(synth.normal(1, n, kdim * ldn, 0, 0.02).reshape(kdim, ldn))
    import torch
    x = to_dev(w)
    codes = torch.empty((n, kdim // 2), dtype=torch.uint8, device="cuda")
    scales = torch.empty((n, kdim // 32), dtype=torch.uint8, device="cuda")
    mix.mx_quantize(x, kdim, n, ldn, 0, t, 0, codes, scales)
    c_ref, s_ref = orc.mx_quantize(np.ascontiguousarray(w[:, :n]), 0, t)
    assert np.array_equal(to_host(codes), c_ref) and np.array_equal(to_host(scales), s_ref)


@pytest.mark.parametrize("shape", [(32, 8), (96, 200), (4128, 72), (288, 1024)])
def test_mx_cols_bf16_aligned_edges(mix, orc, shape):
    """bf16 weights quantised down their columns (n and the row stride
    multiples of 8), partial column groups and k-block groups, and edge
    values planted in some blocks: NaN
    (coded as zero, never the maximum), +-Inf, an all-zero block, bf16
    subnormals and values near the bf16 maximum; both formats and all three
    scale rules, bit for bit against the oracle."""
    kdim, n = shape
    rng = np.random.default_rng(kdim + n)
    w = rng.standard_normal((kdim, n)).astype(np.float32) * 0.02
    w[3, 1] = np.nan
    w[5, n - 1] = np.inf
    w[40 % kdim, n // 2] = -np.inf
    w[:32, min(3, n - 1)] = 0.0
    w[:32, n - 2] = (rng.standard_normal(32) * 1e-40).astype(np.float32)
    if n > 8:
        w[kdim - 32:, 8] = (rng.uniform(-1.1, 1.1, 32) * 3e38).astype(np.float32)
        w[kdim - 1, 9] = np.nan
    wb = synth.to_bf16_bits(w)
    for t in (0, 1):
        for flags in (0, 2, 4):
            check_mx(mix, orc, wb, 0, t, flags)


def test_mx_edge_values(mix, orc):
    rng = np.random.default_rng(6)
    rows = [np.zeros(32, np.float32)]
    b = np.zeros(32, np.float32); b[2] = np.nan; b[3] = 1.0; rows.append(b)
    b = rng.standard_normal(32).astype(np.float32); b[4] = np.inf; b[9] = -np.inf; rows.append(b)
    rows.append((rng.standard_normal(32) * 1e-40).astype(np.float32))
    with np.errstate(over="ignore"):                  # some of these round past the fp32 range: +-Inf
        rows.append((rng.standard_normal(32) * 3e38).astype(np.float32))
    rows.append(np.linspace(-7.5, 7.5, 32).astype(np.float32))
    b = np.full(32, 0.25, np.float32); b[0] = 4.0; rows.append(b)
    rows.append(np.linspace(-6.5, 0.25, 32).astype(np.float32))
    x = np.stack(rows)                      # 8 rows: the transposed copy has ld = 8
    for t in (0, 1):
        for flags in (0, 2, 4):
            check_mx(mix, orc, x, 1, t, flags)
            check_mx(mix, orc, np.ascontiguousarray(x.T), 0, t, flags)


def test_mx_dequantize_matches_oracle(mix, orc):
    import torch
    w = synth.to_bf16_bits(synth.gaussian_weights(2, 2, 128, 96))
    for t in (0, 1):
        c, s = orc.mx_quantize(w, 0, t)
        out = torch.empty((96, 128), dtype=torch.float32, device="cuda")
        mix.mx_dequantize(to_dev(c), to_dev(s), 96, 128, t, out)
        assert np.array_equal(to_host(out).astype(np.float64), orc.mx_dequantize(c, s, t))


@pytest.mark.parametrize("bf16", [False, True])
def test_mx_tight_rule_boundaries(mix, orc, bf16):
    """Tight shared exponent on blocks whose maximum sits on, just above and
    just below the rule's switch points (significand 1.5 for MXFP4, 1.75 for
    MXINT4), on powers of two and on subnormal and near-overflow maxima."""
    rng = np.random.default_rng(31)
    sig = [1.0, 1.0 + 2 ** -7, 1.25, 1.5 - 2 ** -7, 1.5, 1.5 + 2 ** -7, 1.75 - 2 ** -7, 1.75,
           1.75 + 2 ** -7, 2 - 2 ** -7]
    maxima = [s * 2.0 ** e for e in (-133, -126, -40, -1, 0, 3, 60, 127) for s in sig]
    x = (rng.uniform(-1, 1, (len(maxima), 64)) * np.array(maxima)[:, None]).astype(np.float32)
    for r, a in enumerate(maxima):
        x[r, rng.integers(32)] = a if r % 2 else -a
        x[r, 32 + rng.integers(32)] = a
    x = synth.to_bf16_bits(x) if bf16 else x
    for t in (0, 1):
        check_mx(mix, orc, x, 1, t, 4)
        check_mx(mix, orc, np.ascontiguousarray(x.T), 0, t, 4)


def gpu_auto_ebias(mix, x_np, ld=None):
    import torch
    rows, k = x_np.shape
    xd = to_dev(x_np)
    if ld is not None:   # the same tensor read through a wider row stride
        wide = torch.zeros((rows, ld), dtype=xd.dtype, device="cuda")
        wide[:, :k] = xd
        xd = wide
    e = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    mix.mix_auto_ebias(xd, rows, k, xd.stride(0) if rows else k, e)
    return int(to_host(e)[0])


def auto_ebias_cases():
    a = synth.vlm_activations(3, 1, 96, 512, visual_rows=64, n_outlier=4)
    z = np.zeros((4, 64), np.float32)
    special = np.zeros((3, 96), np.float32)
    special[0, 5], special[1, 40], special[2, 70] = 3.0, -2.0 ** -7, 15.5   # 15.5 rounds up: carry
    inf_nan = special.copy()
    inf_nan[2, 70], inf_nan[2, 71], inf_nan[0, 1] = np.inf, np.nan, -np.inf
    tiny = (np.random.default_rng(4).standard_normal((5, 32)) * 1e-42).astype(np.float32)
    huge = np.full((2, 32), 3e38, np.float32)
    return {"activations_f32": synth.to_f32(a), "activations_bf16": synth.to_bf16_bits(a),
            "zeros": z, "carry": special, "inf_nan": inf_nan, "inf_nan_bf16": synth.to_bf16_bits(inf_nan),
            "subnormal": tiny, "huge": huge, "empty": np.zeros((0, 64), np.float32)}


@pytest.mark.parametrize("case", list(auto_ebias_cases()))
def test_auto_ebias_matches_oracle(mix, orc, case):
    x = auto_ebias_cases()[case]
    want = orc.mix_auto_ebias(x) if x.shape[0] else -8
    assert gpu_auto_ebias(mix, x) == want
    if x.shape[0]:
        assert gpu_auto_ebias(mix, x, ld=x.shape[1] + 32) == want


@pytest.mark.parametrize("t", [1, 2])
def test_quantize_auto_matches_oracle(mix, orc, t):
    """Two passes on one stream, no host round trip: the codes are the oracle's
    quantiser run with the oracle's automatic ebias; every block stays
    unclamped from above and the largest lands on code 15."""
    a = synth.vlm_activations(8, 2, 600, 1024, visual_rows=500, n_outlier=8) * 300.0
    for x in (synth.to_bf16_bits(a), synth.to_f32(a)):
        eb = orc.mix_auto_ebias(x)
        c_ref, s_ref = orc.mix_quantize(x, t, eb, 1)
        c, s, e = mix.quantize_mix_auto(to_dev(x), t)
        assert int(to_host(e)[0]) == eb
        assert np.array_equal(to_host(c), c_ref)
        assert np.array_equal(to_host(s).astype(s_ref.dtype), s_ref)
        assert int(np.max(s_ref.astype(np.int64) & 0xF)) == 15
