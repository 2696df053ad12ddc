"""The benchmark's algorithmic accounting, checked on the CPU: the bytes it
charges each call are the library's own plane sizes (each input read once,
each output written once) and its flops are 2 M N K of the named shapes."""
import re

import pytest

import bench


@pytest.fixture(scope="module")
def mix():
    from quantized_vlm_gemm_mix_b300 import mix as m
    return m


@pytest.mark.parametrize("rows,k", [(1, 32), (96, 3584), (4096, 18944), (114688, 4096)])
def test_plane_bytes_are_the_library_plane_sizes(mix, rows, k):
    codes = mix.mix_codes_bytes(rows, k)
    assert bench.plane_bytes(rows, k, 1) == codes + mix.mix_shared_bytes(mix.MIX_T1_4P25, rows, k)
    assert bench.plane_bytes(rows, k, 2) == codes + mix.mix_shared_bytes(mix.MIX_T2_4P5, rows, k)
    assert bench.plane_bytes(rows, k, 0) == codes + mix.mx_scales_bytes(rows, k)
    # quantisers: the bf16 input once plus the planes they write
    assert bench.mix_bytes(rows, k, 1) == 2 * rows * k + bench.plane_bytes(rows, k, 1)
    assert bench.mix_bytes(rows, k, 2) == 2 * rows * k + bench.plane_bytes(rows, k, 2)
    assert bench.mx_bytes(rows, k) == 2 * rows * k + bench.plane_bytes(rows, k, 0)
    assert bench.mx_bytes(rows, k, 4) == 4 * rows * k + bench.plane_bytes(rows, k, 0)


@pytest.mark.parametrize("small", [False, 2])
def test_step_table_flops_and_shapes(small):
    rows = bench.step_table(small)
    names = [r[0] for r in rows]
    assert len(names) == len(set(names)) == 20
    for name, nbytes, flops, launches, cpu in rows:
        assert nbytes > 0 and launches >= 1
        m = re.fullmatch(r"gemm_\w+?_(\d+)x(\d+)x(\d+)", name)
        if m:                                        # gemm_<name>_MxKxN
            M, K, N = map(int, m.groups())
            assert flops == 2.0 * M * N * K
            assert cpu == ("gemm", M * N * (K // 32))
        m = re.fullmatch(r"bmm_(qk|pv)_(\d+)x(\d+)x(\d+)x(\d+)", name)
        if m and m.group(1) == "qk":                 # bmm_qk_heads x M x N x K
            H, M, N, K = map(int, m.groups()[1:])
            assert flops == 2.0 * H * M * N * K
        if m and m.group(1) == "pv":                 # causal P (M = K tokens): products below the mask,
            H, M, N, K = map(int, m.groups()[1:])    # P's blocks holding an unmasked entry
            assert M == K and flops == 2.0 * H * N * M * (M + 1) / 2
            blocks = H * sum(r // 32 + 1 for r in range(M))
            assert nbytes == blocks * 18 + bench.plane_bytes(N * H // 7, K, 0) + H * M * N * 4
        if name.startswith(("mix_quantize", "mx_quantize", "ksmooth")):
            assert flops == 0.0
        m = re.fullmatch(r"decode_attention_(\d+)x(\d+)x(\d+)x(\d+)", name)
        if m:                                        # kv heads x group x cache tokens x head_dim
            HK, G, TC, D = map(int, m.groups())
            assert flops == 2.0 * 2.0 * HK * G * TC * D          # q K'^T and P V
            assert launches == 1


def test_decode_attention_bytes():
    """The fused decode step reads the MXINT4 K' cache (64 code and 4 scale
    bytes per token and KV head) and the V planes along tokens once, plus q,
    the new key and the mean, and writes the appended row and the output."""
    TC, HQ, HK, D = 8192, 28, 4, 128
    want = TC * HK * 68 + HK * D * (TC // 2 + TC // 32) + HQ * D * 2 + HK * D * 6 + HK * 68 + HQ * D * 4
    assert bench.decode_attention_bytes(TC, HQ, HK, D) == want


def test_ksmooth_reads_keys_once():
    g = bench.dims()
    T, HK, D = g["T"], g["HK"], g["D"]
    row = dict((r[0], r) for r in bench.step_table())[f"ksmooth_compute_{T}x{HK}x{D}"]
    # bf16 K read once, fp32 K' written once, fp32 mean written once
    assert row[1] == T * HK * D * (2 + 4) + HK * D * 4


def test_roofline_time_is_the_larger_bound():
    assert bench.roof_seconds(bench.HBM * 1e9, 0.0) == pytest.approx(1.0)
    assert bench.roof_seconds(0.0, bench.MX8_TFLOPS * 1e12) == pytest.approx(1.0)
    assert bench.roof_seconds(bench.HBM * 1e9, 2 * bench.MX8_TFLOPS * 1e12) == pytest.approx(2.0)
