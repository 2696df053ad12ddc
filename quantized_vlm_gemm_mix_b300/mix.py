"""Thin ctypes binding of libmix.so (include/mix.h).

Argument marshalling only: every step of the hot path runs in the library's
CUDA kernels.  Tensors are torch CUDA tensors (PyTorch supplies device memory
and streams); the calls are asynchronous on the current torch stream unless a
stream is given.  There is no CPU fallback: importing this module without the
built library, or calling it on a machine without a GPU, raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmix.so")

# enums and flags (mirror include/mix.h)
MIX_OK, MIX_ERR_INVALID_ARG, MIX_ERR_SHAPE, MIX_ERR_ALIGN = 0, 1, 2, 3
MIX_ERR_UNSUPPORTED, MIX_ERR_CUDA, MIX_ERR_WORKSPACE, MIX_ERR_DEVICE = 4, 5, 6, 7
MIX_T1_4P25, MIX_T2_4P5 = 1, 2
MX_INT4, MX_FP4_E2M1 = 0, 1
MIX_DT_F32, MIX_DT_BF16 = 0, 1
MIX_ASYM_ZERO, MX_SCALE_FLOOR, MX_SCALE_TIGHT, MX_BLOCK16 = 1, 2, 4, 8
MIX_UF_MIX, MIX_UF_MXINT4, MIX_UF_E2M1 = 0, 1, 2
MIX_EPI_NONE, MIX_EPI_MIX_T1, MIX_EPI_MIX_T2, MIX_EPI_MXINT4, MIX_EPI_MXFP4 = 0, 1, 2, 3, 4
MIX_GEMM_AUTO, MIX_GEMM_TCGEN05, MIX_GEMM_SHIFTADD, MIX_GEMM_TCGEN05_STAGED, MIX_GEMM_TCGEN05_FUSED = 0, 1, 2, 3, 4
KSMOOTH_COMPUTE, KSMOOTH_APPLY_FROZEN = 0, 1

EXPORTS = ["mix_codes_bytes", "mix_shared_bytes", "mx_scales_bytes", "mix_quantize", "mix_auto_ebias",
           "mix_quantize_auto", "mx_quantize", "nvfp4_quantize", "mix_underflow_count", "mix_clamp_count",
           "mix_decode_attention_workspace_bytes", "mix_decode_attention",
           "mix_dequantize", "mx_dequantize", "mix_mx_gemm_workspace_bytes", "mix_mx_gemm",
           "mix_mx_gemm_prepare_b_bytes", "mix_mx_gemm_prepare_b",
           "ksmooth_workspace_bytes", "ksmooth_kv", "ksmooth_kv_noalloc", "mix_status_str", "mix_device_error",
           "mix_selftest_wait_timeout", "mix_version"]
KSMOOTH_NOALLOC_SCRATCH_BYTES = 2 << 20
MIX_SELFTEST_WORKSPACE_BYTES = 64 << 10


class MixError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {status_str(status)} (status {status})")
        self.status = status


class GemmDesc(ctypes.Structure):
    """mix_gemm_desc_t."""
    _fields_ = [
        ("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
        ("batch", ctypes.c_int64), ("b_group", ctypes.c_int64),
        ("a_codes", ctypes.c_void_p), ("a_shared", ctypes.c_void_p),
        ("a_type", ctypes.c_int), ("a_ebias", ctypes.c_int),
        ("a_ld", ctypes.c_int64), ("a_batch_stride", ctypes.c_int64),
        ("b_codes", ctypes.c_void_p), ("b_scales", ctypes.c_void_p), ("b_type", ctypes.c_int),
        ("b_block", ctypes.c_int),
        ("b_ld", ctypes.c_int64), ("b_batch_stride", ctypes.c_int64),
        ("c", ctypes.c_void_p), ("ldc", ctypes.c_int64), ("c_batch_stride", ctypes.c_int64),
        ("epi", ctypes.c_int), ("epi_ebias", ctypes.c_int), ("epi_flags", ctypes.c_uint),
        ("out_codes", ctypes.c_void_p), ("out_shared", ctypes.c_void_p),
        ("out_ld", ctypes.c_int64), ("out_batch_stride", ctypes.c_int64),
        ("algo", ctypes.c_int), ("b_prepared", ctypes.c_void_p),
        ("a_causal", ctypes.c_int), ("a_causal_shift", ctypes.c_int64),
    ]


class DecodeAttnDesc(ctypes.Structure):
    """mix_decode_attn_desc_t."""
    _fields_ = [
        ("tokens", ctypes.c_int64), ("q_heads", ctypes.c_int), ("kv_heads", ctypes.c_int),
        ("head_dim", ctypes.c_int), ("dtype", ctypes.c_int),
        ("q", ctypes.c_void_p), ("k_new", ctypes.c_void_p), ("k_mean", ctypes.c_void_p),
        ("k_codes", ctypes.c_void_p), ("k_scales", ctypes.c_void_p),
        ("v_codes", ctypes.c_void_p), ("v_scales", ctypes.c_void_p), ("v_ld", ctypes.c_int64),
        ("sm_scale", ctypes.c_float), ("q_ebias", ctypes.c_int), ("p_ebias", ctypes.c_int),
        ("out", ctypes.c_void_p), ("p_codes", ctypes.c_void_p), ("p_shared", ctypes.c_void_p),
        ("p_values", ctypes.c_void_p),
    ]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libmix.so is not built ({LIB_PATH}); run __graft_entry__.build()")
    L = ctypes.CDLL(LIB_PATH)
    P, I64, I, U, S = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint, ctypes.c_size_t
    sig = {
        "mix_codes_bytes": (S, [I64, I64]),
        "mix_shared_bytes": (S, [I, I64, I64]),
        "mx_scales_bytes": (S, [I64, I64]),
        "mix_quantize": (I, [P, I, I64, I64, I64, I, I, U, P, P, P]),
        "mix_auto_ebias": (I, [P, I, I64, I64, I64, P, P]),
        "nvfp4_quantize": (I, [P, I, I64, I64, I64, P, P, P, P]),
        "mix_decode_attention_workspace_bytes": (S, [P]),
        "mix_decode_attention": (I, [P, P, S, P]),
        "mix_underflow_count": (I, [P, I, I64, I64, I64, P, I, P, P]),
        "mix_clamp_count": (I, [P, I, I64, I64, I64, I, P, P]),
        "mix_quantize_auto": (I, [P, I, I64, I64, I64, I, U, P, P, P, P]),
        "mx_quantize": (I, [P, I, I64, I64, I64, I, I, U, P, P, P]),
        "mix_dequantize": (I, [P, P, I64, I64, I, I, P, P]),
        "mx_dequantize": (I, [P, P, I64, I64, I, P, P]),
        "mix_mx_gemm_workspace_bytes": (S, [ctypes.POINTER(GemmDesc)]),
        "mix_mx_gemm": (I, [ctypes.POINTER(GemmDesc), P, S, P]),
        "mix_mx_gemm_prepare_b_bytes": (S, [ctypes.POINTER(GemmDesc)]),
        "mix_mx_gemm_prepare_b": (I, [ctypes.POINTER(GemmDesc), P, S, P]),
        "ksmooth_workspace_bytes": (S, [I64, I, I]),
        "ksmooth_kv": (I, [P, I, I64, I, I, I64, P, I, P, P, S, P]),
        "ksmooth_kv_noalloc": (I, [P, I, I64, I, I, I64, P, I, P, P]),
        "mix_status_str": (ctypes.c_char_p, [I]),
        "mix_device_error": (I, [ctypes.POINTER(ctypes.c_uint), I]),
        "mix_selftest_wait_timeout": (I, [P, S, P]),
        "mix_version": (I, []),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    return L


lib = _load()


def status_str(status: int) -> str:
    return lib.mix_status_str(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != MIX_OK:
        raise MixError(status, where)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t) -> int:
    if t is None:
        return 0
    if not t.is_cuda:
        raise ValueError("libmix takes CUDA tensors (device pointers)")
    return t.data_ptr()


def _rows_of(x, name: str = "x"):
    """(rows, cols) of a 2-D tensor whose elements run contiguously along a row."""
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError(f"{name} must be 2-D with unit stride along its rows (got shape {tuple(x.shape)}, "
                         f"strides {tuple(x.stride())})")
    return x.shape


def _dtype(t) -> int:
    if t.dtype == torch.float32:
        return MIX_DT_F32
    if t.dtype == torch.bfloat16:
        return MIX_DT_BF16
    raise TypeError(f"unsupported input dtype {t.dtype}")


# ----------------------------------------------------------------------------
# 1:1 wrappers (same names as the C ABI)
# ----------------------------------------------------------------------------

def mix_codes_bytes(rows: int, k: int) -> int:
    return lib.mix_codes_bytes(rows, k)


def mix_shared_bytes(mix_type: int, rows: int, k: int) -> int:
    return lib.mix_shared_bytes(mix_type, rows, k)


def mx_scales_bytes(rows: int, k: int) -> int:
    return lib.mx_scales_bytes(rows, k)


def mix_quantize(x, rows, k, ld, mix_type, ebias, flags, codes, shared, stream=None) -> None:
    _check(lib.mix_quantize(_ptr(x), _dtype(x), rows, k, ld, mix_type, ebias, flags, _ptr(codes),
                            _ptr(shared), _stream(stream)), "mix_quantize")


def mix_auto_ebias(x, rows, k, ld, ebias, stream=None) -> None:
    _check(lib.mix_auto_ebias(_ptr(x), _dtype(x), rows, k, ld, _ptr(ebias), _stream(stream)), "mix_auto_ebias")


def mix_quantize_auto(x, rows, k, ld, mix_type, flags, codes, shared, ebias, stream=None) -> None:
    _check(lib.mix_quantize_auto(_ptr(x), _dtype(x), rows, k, ld, mix_type, flags, _ptr(codes), _ptr(shared),
                                 _ptr(ebias), _stream(stream)), "mix_quantize_auto")


def nvfp4_quantize(x, rows, k, ld, codes, scales, tensor_scale, stream=None) -> None:
    _check(lib.nvfp4_quantize(_ptr(x), _dtype(x), rows, k, ld, _ptr(codes), _ptr(scales), _ptr(tensor_scale),
                              _stream(stream)), "nvfp4_quantize")


def mix_underflow_count(x, rows, k, ld, codes, fmt, count, stream=None) -> None:
    _check(lib.mix_underflow_count(_ptr(x), _dtype(x), rows, k, ld, _ptr(codes), fmt, _ptr(count), _stream(stream)),
           "mix_underflow_count")


def mix_clamp_count(x, rows, k, ld, ebias, counts, stream=None) -> None:
    _check(lib.mix_clamp_count(_ptr(x), _dtype(x), rows, k, ld, ebias, _ptr(counts), _stream(stream)),
           "mix_clamp_count")


def decode_attention_desc(q, k_codes, k_scales, v_codes, v_scales, tokens, sm_scale, out, k_new=None, k_mean=None,
                          q_ebias=-8, p_ebias=-15, p_codes=None, p_shared=None, p_values=None) -> DecodeAttnDesc:
    """q [HQ, 128]; K' cache codes [T, HK, 64], scales [T, HK, 4]; V planes [HK, 128, Tv/2], [HK, 128, Tv/32]."""
    d = DecodeAttnDesc()
    d._keep = [t for t in (q, k_codes, k_scales, v_codes, v_scales, out, k_new, k_mean, p_codes, p_shared,
                           p_values) if t is not None]
    d.tokens, d.q_heads, d.kv_heads, d.head_dim = tokens, q.shape[0], k_codes.shape[1], q.shape[1]
    d.dtype = _dtype(q)
    d.q, d.k_new, d.k_mean = _ptr(q), _ptr(k_new), _ptr(k_mean)
    d.k_codes, d.k_scales, d.v_codes, d.v_scales = _ptr(k_codes), _ptr(k_scales), _ptr(v_codes), _ptr(v_scales)
    d.v_ld = v_codes.shape[-1] * 2
    d.sm_scale, d.q_ebias, d.p_ebias = sm_scale, q_ebias, p_ebias
    d.out, d.p_codes, d.p_shared, d.p_values = _ptr(out), _ptr(p_codes), _ptr(p_shared), _ptr(p_values)
    return d


def decode_attention(desc: DecodeAttnDesc, workspace=None, stream=None):
    """mix_decode_attention; allocates the workspace with torch when none is given."""
    need = lib.mix_decode_attention_workspace_bytes(ctypes.byref(desc))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
    _check(lib.mix_decode_attention(ctypes.byref(desc), _ptr(workspace), workspace.numel(), _stream(stream)),
           "mix_decode_attention")
    return workspace


def mx_quantize(x, rows, cols, ld, axis, mx_type, flags, codes, scales, stream=None) -> None:
    _check(lib.mx_quantize(_ptr(x), _dtype(x), rows, cols, ld, axis, mx_type, flags, _ptr(codes),
                           _ptr(scales), _stream(stream)), "mx_quantize")


def mix_dequantize(codes, shared, rows, k, mix_type, ebias, out, stream=None) -> None:
    _check(lib.mix_dequantize(_ptr(codes), _ptr(shared), rows, k, mix_type, ebias, _ptr(out),
                              _stream(stream)), "mix_dequantize")


def mx_dequantize(codes, scales, rows, k, mx_type, out, stream=None) -> None:
    _check(lib.mx_dequantize(_ptr(codes), _ptr(scales), rows, k, mx_type, _ptr(out), _stream(stream)),
           "mx_dequantize")


def mix_mx_gemm_workspace_bytes(desc: GemmDesc) -> int:
    return lib.mix_mx_gemm_workspace_bytes(ctypes.byref(desc))


def mix_mx_gemm(desc: GemmDesc, workspace=None, stream=None) -> None:
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib.mix_mx_gemm(ctypes.byref(desc), _ptr(workspace), ws_bytes, _stream(stream)), "mix_mx_gemm")


def mix_mx_gemm_prepare_b_bytes(desc: GemmDesc) -> int:
    return lib.mix_mx_gemm_prepare_b_bytes(ctypes.byref(desc))


def mix_mx_gemm_prepare_b(desc: GemmDesc, prepared, stream=None) -> None:
    nbytes = prepared.numel() * prepared.element_size()
    _check(lib.mix_mx_gemm_prepare_b(ctypes.byref(desc), _ptr(prepared), nbytes, _stream(stream)),
           "mix_mx_gemm_prepare_b")


def prepare_b(desc: GemmDesc, stream=None):
    """Prepare desc's B once (a device buffer allocated by torch) and set
    desc.b_prepared to it; returns the buffer, or None when this descriptor
    takes B as it is."""
    need = mix_mx_gemm_prepare_b_bytes(desc)
    if not need:
        return None
    buf = torch.empty(need, dtype=torch.uint8, device=torch.device("cuda"))
    mix_mx_gemm_prepare_b(desc, buf, stream)
    desc.b_prepared = _ptr(buf)
    desc._keep.append(buf)
    return buf


def ksmooth_workspace_bytes(tokens: int, heads: int, head_dim: int) -> int:
    return lib.ksmooth_workspace_bytes(tokens, heads, head_dim)


def ksmooth_kv(k, tokens, heads, head_dim, ld, mean, mode, k_out, workspace=None, stream=None) -> None:
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib.ksmooth_kv(_ptr(k), _dtype(k), tokens, heads, head_dim, ld, _ptr(mean), mode, _ptr(k_out),
                          _ptr(workspace), ws_bytes, _stream(stream)), "ksmooth_kv")


def ksmooth_kv_noalloc(k, tokens, heads, head_dim, ld, mean, mode, k_out, stream=None) -> None:
    """ksmooth_kv without a workspace: for callers that cannot allocate device
    memory (an allocator that owns all of it, loops that must not call
    cudaMalloc).  COMPUTE is limited to
    KSMOOTH_NOALLOC_SCRATCH_BYTES of partial sums; see include/mix.h."""
    _check(lib.ksmooth_kv_noalloc(_ptr(k), _dtype(k), tokens, heads, head_dim, ld, _ptr(mean), mode,
                                  _ptr(k_out), _stream(stream)), "ksmooth_kv_noalloc")


def mix_device_error(clear: bool = True) -> int:
    w = ctypes.c_uint(0)
    _check(lib.mix_device_error(ctypes.byref(w), 1 if clear else 0), "mix_device_error")
    return w.value


def mix_version() -> int:
    return lib.mix_version()


# ----------------------------------------------------------------------------
# Allocating helpers (torch owns the memory)
# ----------------------------------------------------------------------------

def quantize_mix(x: torch.Tensor, mix_type: int = MIX_T2_4P5, ebias: int = -8, flags: int = MIX_ASYM_ZERO,
                 stream=None):
    """x [rows, k] (row stride x.stride(0)) -> (codes uint8 [rows, k/2], shared [rows, k/32])."""
    rows, k = _rows_of(x)
    codes = torch.empty((rows, k // 2), dtype=torch.uint8, device=x.device)
    shared = torch.empty((rows, k // 32), dtype=torch.uint8 if mix_type == MIX_T1_4P25 else torch.int16,
                         device=x.device)
    mix_quantize(x, rows, k, x.stride(0), mix_type, ebias, flags, codes, shared, stream)
    return codes, shared


def quantize_mix_auto(x: torch.Tensor, mix_type: int = MIX_T2_4P5, flags: int = MIX_ASYM_ZERO, stream=None):
    """Two-pass MiX quantiser -> (codes, shared, ebias int32 [1] on the device)."""
    rows, k = _rows_of(x)
    codes = torch.empty((rows, k // 2), dtype=torch.uint8, device=x.device)
    shared = torch.empty((rows, k // 32), dtype=torch.uint8 if mix_type == MIX_T1_4P25 else torch.int16,
                         device=x.device)
    ebias = torch.empty((1,), dtype=torch.int32, device=x.device)
    mix_quantize_auto(x, rows, k, x.stride(0), mix_type, flags, codes, shared, ebias, stream)
    return codes, shared, ebias


def quantize_nvfp4(x: torch.Tensor, stream=None):
    """x [rows, k] -> (codes uint8 [rows, k/2], E4M3 scales uint8 [rows, k/16], tensor scale float32 [1])."""
    rows, k = _rows_of(x)
    codes = torch.empty((rows, k // 2), dtype=torch.uint8, device=x.device)
    scales = torch.empty((rows, k // 16), dtype=torch.uint8, device=x.device)
    ts = torch.empty((1,), dtype=torch.float32, device=x.device)
    nvfp4_quantize(x, rows, k, x.stride(0), codes, scales, ts, stream)
    return codes, scales, ts


def underflow_count(x: torch.Tensor, codes: torch.Tensor, fmt: int, stream=None) -> torch.Tensor:
    """Device count (int64 [1]) of finite nonzero x whose code is a zero code."""
    rows, k = _rows_of(x)
    n = torch.empty((1,), dtype=torch.int64, device=x.device)
    mix_underflow_count(x, rows, k, x.stride(0), codes, fmt, n, stream)
    return n


def clamp_count(x: torch.Tensor, ebias: int = -8, stream=None) -> torch.Tensor:
    """Device counts (int64 [2]) of the MiX blocks of x clamped down (block
    exponent above ebias + 15) and clamped up (nonzero, below ebias)."""
    rows, k = _rows_of(x)
    n = torch.empty((2,), dtype=torch.int64, device=x.device)
    mix_clamp_count(x, rows, k, x.stride(0), ebias, n, stream)
    return n


def quantize_mx(x: torch.Tensor, axis: int, mx_type: int, flags: int = 0, stream=None):
    """axis=1: x [N, K]; axis=0: x [K, N] -> (codes [N, K/2], scales [N, K/32], or K/16 with MX_BLOCK16)."""
    rows, cols = _rows_of(x)
    N, K = (rows, cols) if axis == 1 else (cols, rows)
    codes = torch.empty((N, K // 2), dtype=torch.uint8, device=x.device)
    scales = torch.empty((N, K // (16 if flags & MX_BLOCK16 else 32)), dtype=torch.uint8, device=x.device)
    mx_quantize(x, rows, cols, x.stride(0), axis, mx_type, flags, codes, scales, stream)
    return codes, scales


def gemm_desc(M, N, K, a_codes, a_shared, a_type, a_ebias, b_codes, b_scales, b_type, c=None,
              epi=MIX_EPI_NONE, epi_ebias=-8, epi_flags=MIX_ASYM_ZERO, out_codes=None, out_shared=None,
              batch=1, b_group=1, a_ld=None, a_batch_stride=None, b_ld=None, b_batch_stride=None,
              ldc=None, c_batch_stride=None, out_ld=None, out_batch_stride=None, algo=MIX_GEMM_AUTO, b_block=32,
              a_causal=0, a_causal_shift=0) -> GemmDesc:
    d = GemmDesc()
    # the descriptor holds raw device pointers: keep the tensors alive with it
    d._keep = [t for t in (a_codes, a_shared, b_codes, b_scales, c, out_codes, out_shared) if t is not None]
    d.M, d.N, d.K, d.batch, d.b_group = M, N, K, batch, b_group
    d.a_codes, d.a_shared, d.a_type, d.a_ebias = _ptr(a_codes), _ptr(a_shared), a_type, a_ebias
    d.a_ld = K if a_ld is None else a_ld
    d.a_batch_stride = M * d.a_ld if a_batch_stride is None else a_batch_stride
    d.b_codes, d.b_scales, d.b_type, d.b_block = _ptr(b_codes), _ptr(b_scales), b_type, b_block
    d.b_ld = K if b_ld is None else b_ld
    d.b_batch_stride = N * d.b_ld if b_batch_stride is None else b_batch_stride
    d.c = _ptr(c)
    d.ldc = N if ldc is None else ldc
    d.c_batch_stride = M * d.ldc if c_batch_stride is None else c_batch_stride
    d.epi, d.epi_ebias, d.epi_flags = epi, epi_ebias, epi_flags
    d.out_codes, d.out_shared = _ptr(out_codes), _ptr(out_shared)
    d.out_ld = N if out_ld is None else out_ld
    d.out_batch_stride = M * d.out_ld if out_batch_stride is None else out_batch_stride
    d.algo = algo
    d.a_causal, d.a_causal_shift = a_causal, a_causal_shift
    return d


def gemm(desc: GemmDesc, device=None, stream=None) -> None:
    """mix_mx_gemm with a workspace allocated by torch when one is needed."""
    need = mix_mx_gemm_workspace_bytes(desc)
    ws = None
    if need:
        ws = torch.empty(need, dtype=torch.uint8, device=device or torch.device("cuda"))
    mix_mx_gemm(desc, ws, stream)
    return ws
