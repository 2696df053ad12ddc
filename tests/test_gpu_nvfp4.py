"""GPU parity of the NVFP4 comparison quantiser (16-element E2M1 blocks, E4M3
block scale, fp32 tensor scale) and of the dead-zone count against the CPU
oracle: bit-exact codes, block scales and tensor scale, exact counts."""
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


def check_nvfp4(mix, orc, x):
    c_ref, s_ref, t_ref = orc.nvfp4_quantize(x)
    c, s, t = mix.quantize_nvfp4(to_dev(x))
    c, s, t = to_host(c), to_host(s), to_host(t)
    assert t[0] == t_ref, (t[0], t_ref)
    assert np.array_equal(s, s_ref), f"scales differ at {np.argwhere(s != s_ref)[:5]}"
    assert np.array_equal(c, c_ref), f"codes differ at {np.argwhere(c != c_ref)[:5]}"


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_nvfp4_activations_and_weights(mix, orc, dtype):
    conv = synth.to_bf16_bits if dtype == "bf16" else synth.to_f32
    check_nvfp4(mix, orc, conv(synth.vlm_activations(0, 1, 512, 3584, visual_rows=384)))
    check_nvfp4(mix, orc, conv(synth.gaussian_weights(0, 3, 256, 1024)))
    q, k, v = synth.attention_qkv(2, 256)
    check_nvfp4(mix, orc, conv(k.reshape(-1, 128)))


@pytest.mark.parametrize("k", [16, 48, 4112])
def test_nvfp4_ragged_and_edges(mix, orc, k):
    rng = np.random.default_rng(k)
    x = rng.standard_normal((6, k)).astype(np.float32)
    x[0] = 0.0
    x[1, 3], x[1, 4] = np.nan, np.inf
    x[2, :16] *= 1e-38                       # subnormal block
    x[3, 5] = -np.inf
    x[4] *= 1e30
    check_nvfp4(mix, orc, x)
    check_nvfp4(mix, orc, np.zeros((3, k), np.float32))
    check_nvfp4(mix, orc, (rng.standard_normal((4, k)) * 1e-42).astype(np.float32))


def test_nvfp4_strided(mix, orc):
    import torch
    x = synth.to_bf16_bits(synth.vlm_activations(4, 1, 64, 256, visual_rows=48))
    wide = torch.zeros((64, 320), dtype=torch.bfloat16, device="cuda")
    wide[:, :256] = to_dev(x)
    codes = torch.empty((64, 128), dtype=torch.uint8, device="cuda")
    scales = torch.empty((64, 16), dtype=torch.uint8, device="cuda")
    ts = torch.empty((1,), dtype=torch.float32, device="cuda")
    mix.nvfp4_quantize(wide, 64, 256, 320, codes, scales, ts)
    c_ref, s_ref, t_ref = orc.nvfp4_quantize(x)
    assert to_host(ts)[0] == t_ref
    assert np.array_equal(to_host(codes), c_ref) and np.array_equal(to_host(scales), s_ref)


def test_dead_zone_counts(mix, orc):
    """Keys of the attention workload (K and the frozen-mean-smoothed K'):
    every format's zero-code count on the GPU equals the oracle's, on the
    GPU's own codes (themselves bit-exact with the oracle's)."""
    q, k, v = synth.attention_qkv(5, 1024)
    kk = k.reshape(-1, 128)
    kp = (k - k[:512].mean(axis=0, keepdims=True)).reshape(-1, 128)
    for raw in (kk, kp):
        x = synth.to_bf16_bits(raw)
        xd = to_dev(x)
        planes = {
            "mix": (mix.quantize_mix(xd, mix.MIX_T2_4P5)[0], mix.MIX_UF_MIX, orc.mix_quantize(x, 2)[0]),
            "mxint4": (mix.quantize_mx(xd, 1, mix.MX_INT4)[0], mix.MIX_UF_MXINT4, orc.mx_quantize(x, 1, 0)[0]),
            "mxfp4": (mix.quantize_mx(xd, 1, mix.MX_FP4_E2M1)[0], mix.MIX_UF_E2M1, orc.mx_quantize(x, 1, 1)[0]),
            "nvfp4": (mix.quantize_nvfp4(xd)[0], mix.MIX_UF_E2M1, orc.nvfp4_quantize(x)[0]),
        }
        for name, (codes, fmt, ref_codes) in planes.items():
            assert np.array_equal(to_host(codes), ref_codes), name
            n = int(to_host(mix.underflow_count(xd, codes, fmt))[0])
            assert n == orc.underflow_count(x, ref_codes, fmt), name
    # MiX's recycled -0 code is a value, not a zero
    x = np.zeros((1, 32), np.float32)
    x[0, 0], x[0, 1] = 1.0, 1.0 / 128 * 1.05
    c, _ = mix.quantize_mix(to_dev(x), mix.MIX_T2_4P5)
    n = int(to_host(mix.underflow_count(to_dev(x), c, mix.MIX_UF_MIX))[0])
    assert n == orc.underflow_count(x, orc.mix_quantize(x, 2)[0], orc.UF_MIX)
