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
    # floor and tight rules together; an unknown flag bit
    assert L.mx_quantize(None, 1, 64, 64, 64, 1, 1, 6, None, None, None) == mix.MIX_ERR_INVALID_ARG
    assert L.mx_quantize(None, 1, 64, 64, 64, 1, 1, 8, None, None, None) == mix.MIX_ERR_INVALID_ARG
    # automatic ebias: the result pointer is required, k % 32, alignment of the result int
    assert L.mix_auto_ebias(None, 1, 4, 64, 64, None, None) == mix.MIX_ERR_INVALID_ARG
    assert L.mix_auto_ebias(None, 1, 4, 40, 40, 16, None) == mix.MIX_ERR_SHAPE
    assert L.mix_auto_ebias(None, 1, 4, 64, 64, 18, None) == mix.MIX_ERR_ALIGN
    assert L.mix_quantize_auto(None, 1, 4, 64, 64, 2, 2, None, None, 16, None) == mix.MIX_ERR_INVALID_ARG
    assert L.mix_quantize_auto(None, 1, 4, 64, 64, 3, 1, None, None, 16, None) == mix.MIX_ERR_INVALID_ARG
    d = mix.GemmDesc()
    d.M, d.N, d.K, d.batch, d.b_group = 8, 64, 48, 1, 1
    d.a_type, d.b_type = 2, 1
    assert L.mix_mx_gemm(ctypes.byref(d), None, 0, None) == mix.MIX_ERR_SHAPE
    d.K, d.batch = 64, 0
    assert L.mix_mx_gemm(ctypes.byref(d), None, 0, None) == mix.MIX_ERR_INVALID_ARG
    d.batch, d.epi, d.N = 1, mix.MIX_EPI_MIX_T2, 48
    assert L.mix_mx_gemm(ctypes.byref(d), None, 0, None) == mix.MIX_ERR_SHAPE
    d.N, d.epi, d.epi_flags = 64, mix.MIX_EPI_MXFP4, mix.MX_SCALE_FLOOR | mix.MX_SCALE_TIGHT
    assert L.mix_mx_gemm(ctypes.byref(d), None, 0, None) == mix.MIX_ERR_INVALID_ARG
    d.epi, d.epi_flags = mix.MIX_EPI_MIX_T2, 1
    d.b_block = 8                                   # only 32 (or 0) and 16 exist
    assert L.mix_mx_gemm(ctypes.byref(d), None, 0, None) == mix.MIX_ERR_INVALID_ARG
    d.b_block = 0
    d.a_causal = 2                                  # the causal bound is off (0) or on (1)
    assert L.mix_mx_gemm(ctypes.byref(d), None, 0, None) == mix.MIX_ERR_INVALID_ARG
    d.a_causal, d.a_causal_shift = 1, 1 << 31       # |shift| < 2^31
    assert L.mix_mx_gemm(ctypes.byref(d), None, 0, None) == mix.MIX_ERR_INVALID_ARG
    d.a_causal_shift = -(1 << 31)
    assert L.mix_mx_gemm(ctypes.byref(d), None, 0, None) == mix.MIX_ERR_INVALID_ARG
    d.a_causal, d.a_causal_shift = 0, 0
    assert L.mx_quantize(None, 1, 64, 64, 64, 1, 1, 16, None, None, None) == mix.MIX_ERR_INVALID_ARG
    assert L.ksmooth_kv(None, 1, 16, 4, 12, 48, None, 0, None, None, 0, None) in (mix.MIX_ERR_SHAPE,
                                                                                 mix.MIX_ERR_INVALID_ARG)


def test_status_strings(mix):
    for s in range(8):
        assert isinstance(mix.status_str(s), str) and mix.status_str(s)
    assert mix.mix_version() >= 10000


def _staged_desc(mix, M, N, K, b_type, batch=1, b_group=1, algo=None):
    # fake, suitably aligned device addresses: nothing is launched
    d = mix.GemmDesc()
    d.M, d.N, d.K, d.batch, d.b_group = M, N, K, batch, b_group
    d.a_type, d.a_ebias, d.b_type = mix.MIX_T2_4P5, -8, b_type
    d.a_codes, d.a_shared, d.b_codes, d.b_scales, d.c = 0x100000, 0x200000, 0x300000, 0x400000, 0x500000
    d.a_ld, d.a_batch_stride, d.b_ld, d.b_batch_stride = K, M * K, K, N * K
    d.ldc, d.c_batch_stride = N, M * N
    d.algo = mix.MIX_GEMM_TCGEN05 if algo is None else algo
    return d


def test_staged_gemm_workspace_size_and_check(mix):
    """The staged tensor-core path needs batch*M*Kp bytes of e4m3 A, 512 bytes
    of A scale words per (128-row tile, 128-deep k-step), the same for an
    expanded B (bB*N*Kp bytes, 1024 bytes per 224-row tile and k-step), each
    part rounded up to 1 KiB, plus 1 KiB of alignment slack; a call without
    that workspace is refused before anything is launched."""
    L = mix.lib
    kib = lambda v: (v + 1023) // 1024 * 1024
    M, N, K = 300, 520, 416                      # MXINT4 weights: B expanded
    kp, kt, mt, nt = 512, 4, 3, 3
    want = kib(M * kp) + kib(mt * kt * 512) + kib(N * kp) + kib(nt * kt * 1024) + 1024
    d = _staged_desc(mix, M, N, K, mix.MX_INT4)
    assert L.mix_mx_gemm_workspace_bytes(ctypes.byref(d)) == want
    assert L.mix_mx_gemm(ctypes.byref(d), None, 0, None) == mix.MIX_ERR_WORKSPACE
    assert L.mix_mx_gemm(ctypes.byref(d), ctypes.c_void_p(0x600000), want - 1, None) == mix.MIX_ERR_WORKSPACE
    # prepared once, B's part (expanded plane and scale words) moves out of the workspace
    assert L.mix_mx_gemm_prepare_b_bytes(ctypes.byref(d)) == kib(N * kp) + kib(nt * kt * 1024) + 1024
    assert L.mix_mx_gemm_prepare_b(ctypes.byref(d), None, 0, None) == mix.MIX_ERR_WORKSPACE
    d.b_prepared = 0x700000
    assert L.mix_mx_gemm_workspace_bytes(ctypes.byref(d)) == kib(M * kp) + kib(mt * kt * 512) + 1024
    d.b_prepared = 0x700008                      # not 16-byte aligned
    assert L.mix_mx_gemm_workspace_bytes(ctypes.byref(d)) == 0
    d.b_prepared = None
    # MXFP4 with K % 128 == 0 is read in place: only its scale words are staged
    M, N, K, B, G = 160, 4096, 512, 6, 3
    d = _staged_desc(mix, M, N, K, mix.MX_FP4_E2M1, batch=B, b_group=G)
    want = kib(B * M * K) + kib(B * 2 * 4 * 512) + kib((B // G) * 19 * 4 * 1024) + 1024   # 19 = ceil(4096 / 224)
    assert L.mix_mx_gemm_workspace_bytes(ctypes.byref(d)) == want
    # one 256-column tile: the fused-decode variant; it stages only B, and
    # MXFP4 read in place needs no workspace at all
    d = _staged_desc(mix, 300, 256, 416, mix.MX_INT4)
    assert L.mix_mx_gemm_workspace_bytes(ctypes.byref(d)) == kib(256 * 512) + kib(2 * 4 * 1024) + 1024
    d = _staged_desc(mix, 300, 520, 416, mix.MX_INT4, algo=mix.MIX_GEMM_TCGEN05_FUSED)
    assert L.mix_mx_gemm_workspace_bytes(ctypes.byref(d)) == kib(520 * 512) + kib(3 * 4 * 1024) + 1024
    d = _staged_desc(mix, 300, 256, 512, mix.MX_FP4_E2M1)
    assert L.mix_mx_gemm_workspace_bytes(ctypes.byref(d)) == 0
    d = _staged_desc(mix, 300, 256, 416, mix.MX_INT4, algo=mix.MIX_GEMM_TCGEN05_STAGED)
    assert L.mix_mx_gemm_workspace_bytes(ctypes.byref(d)) > 0
    d.algo = 5
    assert L.mix_mx_gemm(ctypes.byref(d), None, 0, None) == mix.MIX_ERR_INVALID_ARG


def test_selftest_validation(mix):
    """The bounded-wait self-test refuses a missing, short or misaligned
    workspace before launching anything."""
    L = mix.lib
    assert L.mix_selftest_wait_timeout(None, 0, None) == mix.MIX_ERR_WORKSPACE
    assert L.mix_selftest_wait_timeout(ctypes.c_void_p(0x600000), 1024, None) == mix.MIX_ERR_WORKSPACE
    assert L.mix_selftest_wait_timeout(ctypes.c_void_p(0x600004), mix.MIX_SELFTEST_WORKSPACE_BYTES,
                                       None) == mix.MIX_ERR_ALIGN


def test_decode_attention_validation(mix):
    """Host-side checks of the fused decode attention (no launch)."""
    import ctypes
    L = mix.lib
    d = mix.DecodeAttnDesc()
    d.tokens, d.q_heads, d.kv_heads, d.head_dim, d.dtype = 100, 28, 4, 128, mix.MIX_DT_BF16
    d.q = d.k_codes = d.k_scales = d.v_codes = d.v_scales = d.out = 4096   # placeholders, never dereferenced
    d.v_ld, d.sm_scale, d.q_ebias, d.p_ebias = 128, 0.088, -8, -15
    need = L.mix_decode_attention_workspace_bytes(ctypes.byref(d))
    # one cooperative kernel over 4 KV heads x NC chunks of at least 32 tokens
    # (the SMs shared out per KV head: 100 tokens -> 4 chunks of 32 here):
    # statistics [4][NC][7] float2 + partial O [4][NC][7][128] + the barrier
    # counter, each 256-aligned, + 256
    nc = 4
    al = lambda v: (v + 255) // 256 * 256
    assert need == al(4 * nc * 7 * 8) + al(4 * nc * 7 * 128 * 4) + 256 + 256
    assert L.mix_decode_attention(ctypes.byref(d), None, 0, None) == mix.MIX_ERR_WORKSPACE
    for field, value, want in (("q_heads", 64, mix.MIX_ERR_INVALID_ARG),     # 16 query heads per KV head
                               ("q_heads", 30, mix.MIX_ERR_INVALID_ARG),     # not a multiple of kv_heads
                               ("head_dim", 64, mix.MIX_ERR_SHAPE),
                               ("v_ld", 96, mix.MIX_ERR_SHAPE),              # below the token count
                               ("v_ld", 120, mix.MIX_ERR_SHAPE),             # not a multiple of 32
                               ("tokens", 0, mix.MIX_ERR_INVALID_ARG),
                               ("k_new", 4096, mix.MIX_ERR_INVALID_ARG)):    # a new key without the mean
        saved = getattr(d, field)
        setattr(d, field, value)
        assert L.mix_decode_attention(ctypes.byref(d), None, 0, None) == want, field
        assert L.mix_decode_attention_workspace_bytes(ctypes.byref(d)) == 0
        setattr(d, field, saved)



# ---------------------------------------------------------------------------
# The ctypes binding mirrors the header: every enum and define it repeats, and
# the byte layout of both descriptor structs, read from a C program compiled
# against include/mix.h.

_MIRRORED = ["MIX_OK", "MIX_ERR_INVALID_ARG", "MIX_ERR_SHAPE", "MIX_ERR_ALIGN", "MIX_ERR_UNSUPPORTED",
             "MIX_ERR_CUDA", "MIX_ERR_WORKSPACE", "MIX_ERR_DEVICE", "MIX_T1_4P25", "MIX_T2_4P5", "MX_INT4",
             "MX_FP4_E2M1", "MIX_DT_F32", "MIX_DT_BF16", "MIX_ASYM_ZERO", "MX_SCALE_FLOOR", "MX_SCALE_TIGHT",
             "MX_BLOCK16", "MIX_UF_MIX", "MIX_UF_MXINT4", "MIX_UF_E2M1", "MIX_EPI_NONE", "MIX_EPI_MIX_T1",
             "MIX_EPI_MIX_T2", "MIX_EPI_MXINT4", "MIX_EPI_MXFP4", "MIX_GEMM_AUTO", "MIX_GEMM_TCGEN05",
             "MIX_GEMM_SHIFTADD", "MIX_GEMM_TCGEN05_STAGED", "MIX_GEMM_TCGEN05_FUSED", "KSMOOTH_COMPUTE",
             "KSMOOTH_APPLY_FROZEN", "KSMOOTH_NOALLOC_SCRATCH_BYTES"]


def _header_layout(mix):
    import subprocess
    out = os.path.join(ROOT, "_build", "abi_layout")
    os.makedirs(out, exist_ok=True)
    lines = ['#include <stddef.h>', '#include <stdio.h>', '#include "mix.h"', "int main(void) {"]
    for name in _MIRRORED:
        lines.append(f'  printf("{name} %lld\\n", (long long)({name}));')
    for struct, cls in (("mix_gemm_desc_t", mix.GemmDesc), ("mix_decode_attn_desc_t", mix.DecodeAttnDesc)):
        lines.append(f'  printf("sizeof.{struct} %zu\\n", sizeof({struct}));')
        for field, _ in cls._fields_:
            lines.append(f'  printf("{struct}.{field} %zu\\n", offsetof({struct}, {field}));')
    lines += ["  return 0;", "}"]
    src = os.path.join(out, f"layout.{os.getpid()}.c")
    exe = os.path.join(out, f"layout.{os.getpid()}")
    with open(src, "w") as f:
        f.write("\n".join(lines) + "\n")
    try:
        subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), src, "-o", exe],
                       check=True, capture_output=True)
        out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout
    finally:
        for p in (src, exe):
            if os.path.exists(p):
                os.remove(p)
    return dict((k, int(v)) for k, v in (line.split() for line in out.splitlines()))


def test_binding_mirrors_header_constants_and_struct_layouts(mix):
    got = _header_layout(mix)
    for name in _MIRRORED:
        assert getattr(mix, name) == got[name], name
    for struct, cls in (("mix_gemm_desc_t", mix.GemmDesc), ("mix_decode_attn_desc_t", mix.DecodeAttnDesc)):
        assert ctypes.sizeof(cls) == got[f"sizeof.{struct}"], struct
        for field, _ in cls._fields_:
            assert getattr(cls, field).offset == got[f"{struct}.{field}"], f"{struct}.{field}"


def test_work_item_limits_are_rejected_before_launch(mix):
    """Calls past a kernel's 32-bit work-item count return MIX_ERR_UNSUPPORTED
    from validation.  The device addresses are fake but aligned; nothing is
    launched, on a GPU machine or not."""
    L = mix.lib
    X, C, S, R = 0x100000, 0x200000, 0x300000, 0x400000
    BF, F32 = mix.MIX_DT_BF16, mix.MIX_DT_F32
    UN = mix.MIX_ERR_UNSUPPORTED
    # 32-element blocks: rows * k/32 reaches 2^32 - 1 at k = 64 from rows = 2^31
    assert L.mix_quantize(X, BF, 2 ** 31, 64, 64, 2, -8, 1, C, S, None) == UN
    assert L.mx_quantize(X, BF, 2 ** 31, 64, 64, 1, 1, 0, C, S, None) == UN
    # 16-byte vectors of x: bf16 k = 64 is 8 per row, fp32 16 per row
    assert L.mix_auto_ebias(X, BF, 2 ** 29, 64, 64, R, None) == UN
    assert L.mix_auto_ebias(X, F32, 2 ** 28, 64, 64, R, None) == UN
    assert L.mix_quantize_auto(X, BF, 2 ** 29, 64, 64, 2, 1, C, S, R, None) == UN
    assert L.nvfp4_quantize(X, BF, 2 ** 29, 64, 64, C, S, R, None) == UN
    # 8-element groups
    assert L.mix_underflow_count(X, BF, 2 ** 29, 64, 64, C, mix.MIX_UF_MIX, R, None) == UN
    # just below each limit the size check passes; a GPU-less machine then fails at the launch
    if not mix_has_gpu():
        assert L.mix_underflow_count(X, BF, 2 ** 29 - 1, 64, 64, C, mix.MIX_UF_MIX, R, None) == mix.MIX_ERR_CUDA
        assert L.mix_quantize(X, BF, 2 ** 31 - 1, 64, 64, 2, -8, 1, C, S, None) == mix.MIX_ERR_CUDA


def mix_has_gpu():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return True      # when in doubt, skip the calls that would launch


def test_helpers_reject_tensors_without_unit_row_stride(mix):
    import torch
    x = torch.zeros((64, 8), dtype=torch.float32).t()          # [8, 64] with stride (1, 8)
    for call in (lambda: mix.quantize_mix(x), lambda: mix.quantize_mx(x, 1, mix.MX_INT4),
                 lambda: mix.quantize_nvfp4(x), lambda: mix.quantize_mix_auto(x)):
        with pytest.raises(ValueError):
            call()
    with pytest.raises(ValueError):
        mix.quantize_mix(torch.zeros(64))                       # not 2-D
