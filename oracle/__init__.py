"""CPU oracle for the MiX hot path -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library never calls it, and it
shares no code with the CUDA sources.  The arithmetic lives in
``mix_oracle.c`` (plain scalar C, exact binary arithmetic, fp64 sums); this
module only compiles it with gcc and marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mix_oracle.c")
_LIB = os.path.join(_HERE, "liborcmix.so")

F32, BF16 = 0, 1
T1, T2 = 1, 2
MXINT4, MXFP4 = 0, 1
ASYM_ZERO, MX_FLOOR, MX_TIGHT = 1, 2, 4

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library with gcc (no OpenMP: one host thread)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                               "-fno-fast-math", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        P, I64, I, U = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint
        L.orc_mix_quantize.argtypes = [P, I, I64, I64, I64, I, I, U, P, P]
        L.orc_mix_dequantize.argtypes = [P, P, I64, I64, I, I, P]
        L.orc_mx_quantize.argtypes = [P, I, I64, I64, I64, I, I, U, P, P]
        L.orc_mx_dequantize.argtypes = [P, P, I64, I64, I, P]
        L.orc_gemm.argtypes = [P, P, I, I, P, P, I, I64, I64, I64, I64, I64, P]
        L.orc_ksmooth_mean.argtypes = [P, I, I64, I, I, I64, P]
        L.orc_ksmooth_apply.argtypes = [P, I, I64, I, I, I64, P, P]
        L.orc_set_mutation.argtypes = [I]
        L.orc_mix_auto_ebias.argtypes = [P, I, I64, I64, I64]
        L.orc_mx_quantize_blk.argtypes = [P, I, I64, I64, I64, I, I, U, I, P, P]
        L.orc_mx_dequantize_blk.argtypes = [P, P, I64, I64, I, I, P]
        L.orc_gemm_blk.argtypes = [P, P, I, I, P, P, I, I, I64, I64, I64, I64, I64, P]
        L.orc_nvfp4_quantize.argtypes = [P, I, I64, I64, I64, P, P, P]
        L.orc_nvfp4_dequantize.argtypes = [P, P, ctypes.c_float, I64, I64, P]
        L.orc_underflow_count.argtypes = [P, I, I64, I64, I64, P, I]
        L.orc_mix_clamp_count.argtypes = [P, I, I64, I64, I64, I, P]
        L.orc_underflow_count.restype = I64
        for f in ("orc_mix_quantize", "orc_mix_dequantize", "orc_mx_quantize",
                  "orc_mx_dequantize", "orc_gemm", "orc_ksmooth_mean", "orc_ksmooth_apply",
                  "orc_mix_auto_ebias", "orc_mx_quantize_blk", "orc_mx_dequantize_blk", "orc_gemm_blk",
                  "orc_nvfp4_quantize", "orc_nvfp4_dequantize", "orc_mix_clamp_count"):
            getattr(L, f).restype = ctypes.c_int
        L.orc_set_mutation.restype = None
        _lib = L
    return _lib


def set_mutation(m: int) -> None:
    """Plant mistake number ``m`` in the oracle (0 = none).  Tests only."""
    lib().orc_set_mutation(int(m))


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _dtype_of(x: np.ndarray) -> int:
    if x.dtype == np.float32:
        return F32
    if x.dtype == np.uint16:
        return BF16
    raise TypeError("oracle input must be float32 or bfloat16 bit patterns (uint16)")


def _check(rc: int) -> None:
    if rc != 0:
        raise ValueError("oracle rejected the arguments")


def mix_quantize(x: np.ndarray, mix_type: int, ebias: int = -8, flags: int = ASYM_ZERO):
    """x: [rows, k] float32 or bf16 bits -> (codes uint8 [rows, k/2], shared)."""
    x = np.ascontiguousarray(x)
    rows, k = x.shape
    codes = np.zeros((rows, k // 2), dtype=np.uint8)
    shared = np.zeros((rows, k // 32), dtype=np.uint8 if mix_type == T1 else np.uint16)
    _check(lib().orc_mix_quantize(_ptr(x), _dtype_of(x), rows, k, k, mix_type, ebias,
                                  flags, _ptr(codes), _ptr(shared)))
    return codes, shared


def mix_auto_ebias(x: np.ndarray) -> int:
    """The automatic ebias of x [rows, k] (float32 or bf16 bits)."""
    x = np.ascontiguousarray(x)
    rows, k = x.shape
    e = lib().orc_mix_auto_ebias(_ptr(x), _dtype_of(x), rows, k, k)
    if e == -1000:
        raise ValueError("k must be a multiple of 32")
    return e


def mix_clamp_count(x: np.ndarray, ebias: int = -8):
    """(blocks clamped down, blocks clamped up) of the MiX quantiser of x
    [rows, k] at this ebias: the block exponent of Algorithm 1's steps 1-2
    above ebias + 15, or (nonzero blocks) below ebias."""
    x = np.ascontiguousarray(x)
    rows, k = x.shape
    out = np.zeros(2, dtype=np.int64)
    _check(lib().orc_mix_clamp_count(_ptr(x), _dtype_of(x), rows, k, k, int(ebias), _ptr(out)))
    return int(out[0]), int(out[1])


def mix_dequantize(codes: np.ndarray, shared: np.ndarray, mix_type: int, ebias: int = -8):
    codes = np.ascontiguousarray(codes)
    shared = np.ascontiguousarray(shared)
    rows, kh = codes.shape
    out = np.zeros((rows, kh * 2), dtype=np.float64)
    _check(lib().orc_mix_dequantize(_ptr(codes), _ptr(shared), rows, kh * 2, mix_type, ebias,
                                    _ptr(out)))
    return out


def mx_quantize(x: np.ndarray, axis: int, mx_type: int, flags: int = 0, block: int = 32):
    """axis=1: x is [N, K]; axis=0: x is [K, N].  -> (codes [N, K/2], scales [N, K/block])."""
    x = np.ascontiguousarray(x)
    rows, cols = x.shape
    N, K = (rows, cols) if axis == 1 else (cols, rows)
    codes = np.zeros((N, K // 2), dtype=np.uint8)
    scales = np.zeros((N, K // block), dtype=np.uint8)
    _check(lib().orc_mx_quantize_blk(_ptr(x), _dtype_of(x), rows, cols, cols, axis, mx_type,
                                     flags, block, _ptr(codes), _ptr(scales)))
    return codes, scales


def mx_dequantize(codes: np.ndarray, scales: np.ndarray, mx_type: int, block: int = 32):
    codes = np.ascontiguousarray(codes)
    scales = np.ascontiguousarray(scales)
    n, kh = codes.shape
    out = np.zeros((n, kh * 2), dtype=np.float64)
    _check(lib().orc_mx_dequantize_blk(_ptr(codes), _ptr(scales), n, kh * 2, mx_type, block, _ptr(out)))
    return out


def nvfp4_quantize(x: np.ndarray):
    """x [rows, k] float32 or bf16 bits -> (codes [rows, k/2], E4M3 scales [rows, k/16], fp32 tensor scale)."""
    x = np.ascontiguousarray(x)
    rows, k = x.shape
    codes = np.zeros((rows, k // 2), dtype=np.uint8)
    scales = np.zeros((rows, k // 16), dtype=np.uint8)
    ts = np.zeros(1, dtype=np.float32)
    _check(lib().orc_nvfp4_quantize(_ptr(x), _dtype_of(x), rows, k, k, _ptr(codes), _ptr(scales), _ptr(ts)))
    return codes, scales, ts[0]


def nvfp4_dequantize(codes: np.ndarray, scales: np.ndarray, tensor_scale):
    codes = np.ascontiguousarray(codes)
    scales = np.ascontiguousarray(scales)
    rows, kh = codes.shape
    out = np.zeros((rows, kh * 2), dtype=np.float64)
    _check(lib().orc_nvfp4_dequantize(_ptr(codes), _ptr(scales), float(tensor_scale), rows, kh * 2, _ptr(out)))
    return out


UF_MIX, UF_MXINT4, UF_E2M1 = 0, 1, 2


def underflow_count(x: np.ndarray, codes: np.ndarray, fmt: int) -> int:
    """Finite nonzero elements of x [rows, k] whose code in codes [rows, k/2] is a zero code."""
    x = np.ascontiguousarray(x)
    codes = np.ascontiguousarray(codes)
    rows, k = x.shape
    return int(lib().orc_underflow_count(_ptr(x), _dtype_of(x), rows, k, k, _ptr(codes), fmt))


def gemm(a_codes, a_shared, a_type, a_ebias, b_codes, b_scales, b_type, b_group: int = 1, b_block: int = 32):
    """Eq. (6) reference.  a_*: [batch, M, ...] or [M, ...]; b_*: [batch_b, N, ...] or [N, ...].

    Returns C fp64 [batch, M, N] (or [M, N] for 2-D inputs).
    """
    squeeze = a_codes.ndim == 2
    ac = np.ascontiguousarray(a_codes if a_codes.ndim == 3 else a_codes[None])
    ash = np.ascontiguousarray(a_shared if a_shared.ndim == 3 else a_shared[None])
    bc = np.ascontiguousarray(b_codes if b_codes.ndim == 3 else b_codes[None])
    bs = np.ascontiguousarray(b_scales if b_scales.ndim == 3 else b_scales[None])
    batch, M, kh = ac.shape
    N = bc.shape[1]
    c = np.zeros((batch, M, N), dtype=np.float64)
    _check(lib().orc_gemm_blk(_ptr(ac), _ptr(ash), a_type, a_ebias, _ptr(bc), _ptr(bs), b_type, b_block,
                              batch, b_group, M, N, kh * 2, _ptr(c)))
    return c[0] if squeeze else c


def ksmooth_mean(k: np.ndarray):
    """k: [tokens, heads, head_dim] float32 or bf16 bits -> fp64 mean [heads, head_dim]."""
    k = np.ascontiguousarray(k)
    t, h, d = k.shape
    mean = np.zeros((h, d), dtype=np.float64)
    _check(lib().orc_ksmooth_mean(_ptr(k), _dtype_of(k), t, h, d, h * d, _ptr(mean)))
    return mean


def ksmooth_apply(k: np.ndarray, mu: np.ndarray):
    """K' = fp32(K) - mu (mu float32 [heads, head_dim]) -> float32 [tokens, heads, head_dim]."""
    k = np.ascontiguousarray(k)
    mu = np.ascontiguousarray(mu, dtype=np.float32)
    t, h, d = k.shape
    out = np.zeros((t, h, d), dtype=np.float32)
    _check(lib().orc_ksmooth_apply(_ptr(k), _dtype_of(k), t, h, d, h * d, _ptr(mu), _ptr(out)))
    return out


def decode_attention(q, k_cache_codes, k_cache_scales, v_codes, v_scales, tokens, sm_scale,
                     k_new=None, k_mean=None, q_ebias=-8, p_ebias=-15):
    """One decode step of MiX attention over an MX KV cache, in the order the
    pages give (Method section, accelerator bullet: K-smoothing with the
    frozen prefill mean, Q-K^T on the dual-format matmul, the softmax of the
    SFU, the MiX requantisation of P, P-V on the dual-format matmul).

    q: [HQ, D] float32 or bf16 bits.  K' cache: codes [T, HK, D/2], scales
    [T, HK, D/32] (MXINT4 along D).  k_new: [HK, D] (float32 or bf16 bits) or
    None; when given, K' = fp32(k_new) - k_mean is quantised to MXINT4 and
    written to cache row tokens - 1 (the arrays are updated in place).
    V: codes [HK, D, Tv/2], scales [HK, D, Tv/32] (MXINT4 along tokens, Tv a
    multiple of 32 >= tokens).  Returns (O fp64 [HQ, D], P fp32 [HQ, tokens],
    the MiX-4.5b planes of P over Tv tokens, S fp64 [HQ, tokens]).
    """
    HQ, D = q.shape
    HK = k_cache_codes.shape[1]
    G = HQ // HK
    Tv = v_codes.shape[2] * 2
    if k_new is not None:
        kp = ksmooth_apply(np.ascontiguousarray(k_new).reshape(1, HK, D), k_mean.astype(np.float32))
        c, s = mx_quantize(kp.reshape(HK, D).astype(np.float32), 1, MXINT4)
        k_cache_codes[tokens - 1] = c
        k_cache_scales[tokens - 1] = s
    qc, qs = mix_quantize(q, T2, q_ebias)
    S = np.zeros((HQ, tokens))
    for g in range(HK):
        kc = np.ascontiguousarray(k_cache_codes[:tokens, g])
        ks = np.ascontiguousarray(k_cache_scales[:tokens, g])
        S[g * G:(g + 1) * G] = gemm(qc[g * G:(g + 1) * G], qs[g * G:(g + 1) * G], T2, q_ebias, kc, ks, MXINT4)
    z = S * sm_scale
    e = np.exp(z - z.max(axis=1, keepdims=True))
    P = (e / e.sum(axis=1, keepdims=True)).astype(np.float32)
    Pp = np.zeros((HQ, Tv), np.float32)
    Pp[:, :tokens] = P
    pc, ps = mix_quantize(Pp, T2, p_ebias)
    O = np.zeros((HQ, D))
    for g in range(HK):
        O[g * G:(g + 1) * G] = gemm(pc[g * G:(g + 1) * G], ps[g * G:(g + 1) * G], T2, p_ebias,
                                    np.ascontiguousarray(v_codes[g]), np.ascontiguousarray(v_scales[g]), MXINT4)
    return O, P, (pc, ps), S
