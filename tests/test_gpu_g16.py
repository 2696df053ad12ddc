"""GPU parity of the g16 weight formats (MXINT4g16 / MXFP4g16: one E8M0
scale per 16 elements; the weights of "MiX-INT4g16") against the CPU
oracle: bit-exact quantiser planes, and the A-MiX x W-MX g16 matmul on the
staged and fused-decode tensor-core variants and on the shift-add path,
within the row-relative tolerance."""
import numpy as np
import pytest

from quantized_vlm_gemm_mix_b300 import synth
from helpers import GEMM_REL_TOL, row_rel_err, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mix():
    import torch
    assert torch.cuda.is_available()
    from quantized_vlm_gemm_mix_b300 import mix as m
    return m


def check_mx16(mix, orc, x, axis, t, flags=0):
    c_ref, s_ref = orc.mx_quantize(x, axis, t, flags, block=16)
    c, s = mix.quantize_mx(to_dev(x), axis, t, flags | mix.MX_BLOCK16)
    c, s = to_host(c), to_host(s)
    assert s.shape == s_ref.shape
    assert np.array_equal(c, c_ref), f"codes differ at {np.argwhere(c != c_ref)[:5]}"
    assert np.array_equal(s, s_ref), f"scales differ at {np.argwhere(s != s_ref)[:5]}"


def g16_weights(seed, tid, k, n):
    """N(0, 0.02) with a per-16-row gain of 2^(0 .. 3), so the two halves of a
    32-block usually carry different scales."""
    w = synth.gaussian_weights(seed, tid, k, n)
    return w * np.exp2(np.arange(k) // 16 % 4)[:, None]


@pytest.mark.parametrize("axis", [0, 1])
@pytest.mark.parametrize("t", [0, 1])
@pytest.mark.parametrize("flags", [0, 4])
def test_mx_g16_quantiser(mix, orc, axis, t, flags):
    w = synth.to_bf16_bits(g16_weights(1, 2, 512, 160))
    x = w if axis == 0 else np.ascontiguousarray(w.T)
    check_mx16(mix, orc, x, axis, t, flags)
    check_mx16(mix, orc, synth.bf16_bits_to_f32(x).astype(np.float32), axis, t, flags)


@pytest.mark.parametrize("t", [0, 1])
def test_mx_g16_edges_and_ragged(mix, orc, t):
    rng = np.random.default_rng(8)
    x = rng.standard_normal((8, 96)).astype(np.float32)   # 8 rows: the transposed copy keeps 16-byte rows
    x[0] = 0.0
    x[1, 3], x[1, 20] = np.nan, np.inf
    x[2, 17:32] = 0.0                       # one zero half
    x[3] *= 1e-40
    x[4, :16] *= 2.0 ** 40                  # halves 40 binades apart
    x[5, 16] = -np.inf
    for axis in (0, 1):
        xx = x if axis == 1 else np.ascontiguousarray(x.T)
        for flags in (0, 2, 4):
            check_mx16(mix, orc, xx, axis, t, flags)


def run(mix, ac, ash, at, bc, bs, bt, M, N, K, algo, batch=1, b_group=1):
    import torch
    c = torch.empty((batch, M, N), dtype=torch.float32, device="cuda")
    d = mix.gemm_desc(M, N, K, to_dev(ac), to_dev(ash), at, -8, to_dev(bc), to_dev(bs), bt, c=c, algo=algo,
                      b_block=16, batch=batch, b_group=b_group)
    mix.gemm(d)
    torch.cuda.synchronize()
    assert mix.mix_device_error() == 0
    return to_host(c)


# the shift-add path takes at most 16 rows, so it gets only the shapes within that
G16_SHAPES = [(1, 64, 96), (16, 256, 512), (130, 288, 416), (300, 544, 1024)]
G16_CASES = [(algo, shape) for algo in ("staged", "fused", "shiftadd") for shape in G16_SHAPES
             if algo != "shiftadd" or shape[0] <= 16]


@pytest.mark.parametrize("at,bt", [(2, 0), (2, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("algo,shape", G16_CASES)
def test_g16_gemm_matches_eq6(mix, orc, algo, shape, at, bt):
    M, N, K = shape
    a = synth.to_bf16_bits(synth.vlm_activations(M + K, 0, M, K, visual_rows=(3 * M) // 4))
    w = synth.to_bf16_bits(g16_weights(N, 1, K, N))
    ac, ash = orc.mix_quantize(a, at)
    bc, bs = orc.mx_quantize(w, 0, bt, 0, block=16)
    ref = orc.gemm(ac, ash, at, -8, bc, bs, bt, b_block=16)
    algo_id = {"staged": mix.MIX_GEMM_TCGEN05_STAGED, "fused": mix.MIX_GEMM_TCGEN05_FUSED,
               "shiftadd": mix.MIX_GEMM_SHIFTADD}[algo]
    c = run(mix, ac, ash, at, bc, bs, bt, M, N, K, algo_id)[0]
    err = row_rel_err(c, ref)
    assert err <= GEMM_REL_TOL, err
    assert err < 1e-5, err   # every product is exact; only fp32 accumulation rounds


@pytest.mark.parametrize("algo", ["staged", "fused"])
def test_g16_gemm_batched_gqa(mix, orc, algo):
    B, G, M, N, K = 6, 3, 96, 288, 256
    a = synth.to_bf16_bits(synth.vlm_activations(3, 0, B * M, K, visual_rows=B * M // 2))
    w = synth.to_bf16_bits(g16_weights(4, 1, K, (B // G) * N))
    ac, ash = orc.mix_quantize(a, 2)
    bc, bs = orc.mx_quantize(w, 0, 0, 0, block=16)
    ac, ash = ac.reshape(B, M, -1), ash.reshape(B, M, -1)
    bc, bs = bc.reshape(B // G, N, -1), bs.reshape(B // G, N, -1)
    ref = orc.gemm(ac, ash, 2, -8, bc, bs, 0, b_group=G, b_block=16)
    algo_id = mix.MIX_GEMM_TCGEN05_STAGED if algo == "staged" else mix.MIX_GEMM_TCGEN05_FUSED
    c = run(mix, ac, ash, 2, bc, bs, 0, M, N, K, algo_id, batch=B, b_group=G)
    for b in range(B):
        assert row_rel_err(c[b], ref[b]) < 1e-5


@pytest.mark.parametrize("algo", ["staged", "fused", "shiftadd"])
def test_g16_halves_far_apart(mix, orc, algo):
    """Halves ~10 binades apart stay exact on the tensor cores; 20 apart, the
    smaller half is rounded to e4m3 relative to the larger (the integer
    shift-add path stays exact), an error bounded by that half's share."""
    M, N, K = 8, 64, 64
    a = synth.to_bf16_bits(synth.vlm_activations(5, 0, M, K, visual_rows=4))
    ac, ash = orc.mix_quantize(a, 2)
    algo_id = {"staged": mix.MIX_GEMM_TCGEN05_STAGED, "fused": mix.MIX_GEMM_TCGEN05_FUSED,
               "shiftadd": mix.MIX_GEMM_SHIFTADD}[algo]
    for bt in (0, 1):
        for gap in (10, 20):
            w = synth.gaussian_weights(6, 1, K, N) * np.where(np.arange(K) % 32 < 16, 1.0, 2.0 ** -gap)[:, None]
            bc, bs = orc.mx_quantize(synth.to_bf16_bits(w), 0, bt, 0, block=16)
            ref = orc.gemm(ac, ash, 2, -8, bc, bs, bt, b_block=16)
            c = run(mix, ac, ash, 2, bc, bs, bt, M, N, K, algo_id)[0]
            if gap == 10 or algo == "shiftadd":
                assert row_rel_err(c, ref) < 1e-5
            else:
                # the rounded half's terms are below 2^-14 of the row's scale
                assert row_rel_err(c, ref) < 2.0 ** -12
