"""The C ABI without a GPU: the library loads, exports every symbol the header
declares, and answers its host-only queries (sizes, validation, strings)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mix.h")


def declared_symbols():
    src = open(HEADER).read()
    return re.findall(r"MIX_API\s+[\w\s\*]+?\b(\w+)\s*\(", src)


@pytest.fixture(scope="module")
def mix():
    from quantized_vlm_gemm_mix_b300 import _build
    _build.build()
    from quantized_vlm_gemm_mix_b300 import mix as m
    return m


def test_header_lists_the_entry_points():
    syms = declared_symbols()
    for want in ("mix_quantize", "mx_quantize", "mix_mx_gemm", "ksmooth_kv", "mix_status_str"):
        assert want in syms


def test_library_exports_every_declared_symbol(mix):
    lib = ctypes.CDLL(mix.LIB_PATH)
    for s in declared_symbols():
        assert hasattr(lib, s), s
    assert set(declared_symbols()) == set(mix.EXPORTS)


def test_plane_sizes_match_bit_accounting(mix):
    rows, k = 96, 3584
    assert mix.mix_codes_bytes(rows, k) == rows * k // 2
    t1 = mix.mix_codes_bytes(rows, k) + mix.mix_shared_bytes(mix.MIX_T1_4P25, rows, k)
    t2 = mix.mix_codes_bytes(rows, k) + mix.mix_shared_bytes(mix.MIX_T2_4P5, rows, k)
    assert t1 * 8 == rows * k * 4.25 and t2 * 8 == rows * k * 4.5
    assert mix.mx_scales_bytes(rows, k) == rows * k // 32
    assert mix.mix_codes_bytes(rows, 33) == 0 and mix.mix_shared_bytes(7, rows, k) == 0


def test_validation_rejects_before_launch(mix):
    L = mix.lib
    # k not a multiple of 32, bad enum, bad ebias, negative rows: no device work happens
    assert L.mix_quantize(None, 1, 4, 40, 40, 2, -8, 1, None, None, None) == mix.MIX_ERR_SHAPE
    assert L.mix_quantize(None, 1, 4, 64, 64, 3, -8, 1, None, None, None) == mix.MIX_ERR_INVALID_ARG
    assert L.mix_quantize(None, 1, 4, 64, 64, 2, -200, 1, None, None, None) == mix.MIX_ERR_INVALID_ARG
    assert L.mix_quantize(None, 1, -1, 64, 64, 2, -8, 1, None, None, None) == mix.MIX_ERR_INVALID_ARG
    assert L.mix_quantize(None, 1, 0, 64, 64, 2, -8, 1, None, None, None) == mix.MIX_OK  # empty: no-op
    assert L.mx_quantize(None, 1, 48, 64, 64, 0, 1, 0, None, None, None) == mix.MIX_ERR_SHAPE
    assert L.mx_quantize(None, 1, 64, 64, 64, 2, 1, 0, None, None, None) == mix.MIX_ERR_INVALID_ARG
    d = mix.GemmDesc()
    d.M, d.N, d.K, d.batch, d.b_group = 8, 64, 48, 1, 1
    d.a_type, d.b_type = 2, 1
    assert L.mix_mx_gemm(ctypes.byref(d), None, 0, None) == mix.MIX_ERR_SHAPE
    d.K, d.batch = 64, 0
    assert L.mix_mx_gemm(ctypes.byref(d), None, 0, None) == mix.MIX_ERR_INVALID_ARG
    d.batch, d.epi, d.N = 1, mix.MIX_EPI_MIX_T2, 48
    assert L.mix_mx_gemm(ctypes.byref(d), None, 0, None) == mix.MIX_ERR_SHAPE
    assert L.ksmooth_kv(None, 1, 16, 4, 12, 48, None, 0, None, None, 0, None) in (mix.MIX_ERR_SHAPE,
                                                                                 mix.MIX_ERR_INVALID_ARG)


def test_status_strings(mix):
    for s in range(8):
        assert isinstance(mix.status_str(s), str) and mix.status_str(s)
    assert mix.mix_version() >= 10000
