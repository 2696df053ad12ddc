"""Seeded synthetic tensors shaped like the VLM layers the MiX paper evaluates.

This module only draws random numbers; it holds none of the quantisation or
matmul arithmetic, so that the CPU oracle and the CUDA path can both be fed
the very same bytes.

Generator: splitmix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014) used counter-style.  Element ``i`` of the
tensor with id ``tid`` under ``seed`` takes the 64-bit word
``mix64(key + (i + 1) * GAMMA)`` with ``key = mix64(seed * GAMMA ^ tid * C1)``.
Uniforms in (0, 1) are ``((u >> 11) + 0.5) * 2**-53``.  Laplace samples use the
inverse CDF; normal samples use Box-Muller on the words of counters ``2i`` and
``2i + 1``.  Values are produced in float64 and rounded once, to float32 (RNE)
or to bfloat16 (RNE from the float32 value).

Workload shapes and value distributions follow the MiX paper's setup
(Qwen2-VL-7B decoder linears, a ViT MLP and GQA attention) and its activation
statistics ("Fig. 1": visual tokens about 34x larger than text tokens; "Fig. 2":
Q/K channel outliers on all tokens, V outliers on early tokens).
"""
from __future__ import annotations

import math

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_C1 = np.uint64(0xD1B54A32D192ED03)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _key(seed: int, tid: int) -> np.uint64:
    with np.errstate(over="ignore"):
        k = np.array([np.uint64(seed) * GAMMA ^ np.uint64(tid) * _C1], dtype=np.uint64)
        return _mix64(k)[0]


def words(seed: int, tid: int, start: int, count: int) -> np.ndarray:
    """Raw 64-bit words for counters ``start .. start+count-1``."""
    key = _key(seed, tid)
    ctr = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(key + ctr * GAMMA)


def uniform(seed: int, tid: int, start: int, count: int) -> np.ndarray:
    w = words(seed, tid, start, count)
    return ((w >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)


def laplace(seed: int, tid: int, n: int, b: float) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    for s in range(0, n, _CHUNK):
        c = min(_CHUNK, n - s)
        u = uniform(seed, tid, s, c) - 0.5
        out[s:s + c] = -b * np.sign(u) * np.log1p(-2.0 * np.abs(u))
    return out


def normal(seed: int, tid: int, n: int, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    for s in range(0, n, _CHUNK):
        c = min(_CHUNK, n - s)
        u = uniform(seed, tid, 2 * s, 2 * c)
        u1, u2 = u[0::2], u[1::2]
        out[s:s + c] = mean + std * np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)
    return out


def permutation(seed: int, tid: int, n: int) -> np.ndarray:
    """Seeded permutation of range(n): argsort of n random words (stable)."""
    return np.argsort(words(seed, tid, 0, n), kind="stable")


def to_f32(x: np.ndarray) -> np.ndarray:
    return x.astype(np.float32)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float64 -> float32 (RNE) -> bfloat16 (RNE); returns the uint16 bit patterns."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(f)
    if nan.any():
        r[nan] = np.uint16(0x7FC0)
    return r


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


# --------------------------------------------------------------------------- #
# Workload recipes.  Every recipe returns float64 values; callers round them.  #
# --------------------------------------------------------------------------- #

def outlier_channels(seed: int, tid: int, k: int, frac: float) -> np.ndarray:
    n = int(math.ceil(frac * k - 1e-9))
    return np.sort(permutation(seed, tid, k)[:n])


def vlm_activations(seed: int, tid: int, rows: int, k: int, visual_rows: int,
                    b_visual: float = 0.30, b_text: float = 0.009,
                    outlier_frac: float = 0.01, outlier_scale: float = 30.0,
                    n_outlier: int | None = None) -> np.ndarray:
    """Visual rows first (Laplace(0, b_visual), outlier channels scaled), then text rows.

    ``n_outlier`` fixes the outlier channel count directly (else ``ceil(frac*k)``).
    """
    x = np.empty((rows, k), dtype=np.float64)
    nv = min(visual_rows, rows)
    if nv:
        x[:nv] = laplace(seed, tid, nv * k, b_visual).reshape(nv, k)
        if n_outlier is None:
            ch = outlier_channels(seed, tid + 1000, k, outlier_frac)
        else:
            ch = np.sort(permutation(seed, tid + 1000, k)[:n_outlier])
        x[:nv, ch] *= outlier_scale
    if rows > nv:
        x[nv:] = laplace(seed, tid + 1, (rows - nv) * k, b_text).reshape(rows - nv, k)
    return x


def gaussian_weights(seed: int, tid: int, k: int, n: int, std: float = 0.02) -> np.ndarray:
    """Weight matrix W[k x n] (row-major, as used in x @ W)."""
    return normal(seed, tid, k * n, 0.0, std).reshape(k, n)


def attention_qkv(seed: int, tokens: int, q_heads: int = 28, kv_heads: int = 4,
                  head_dim: int = 128, n_outlier: int = 4, qk_scale: float = 20.0,
                  v_spike_tokens: int = 16, v_scale: float = 15.0):
    """Q[t,hq,d], K[t,hk,d], V[t,hk,d] in float64.

    Q and K: N(b_c, 1) per (head, channel) with b_c ~ N(0, 1); the same seeded
    set of ``n_outlier`` channels is scaled by ``qk_scale`` on every token.
    V: N(0, 1) with the first ``v_spike_tokens`` tokens scaled by ``v_scale``.
    Token t of every tensor depends only on (seed, t), so a longer draw extends a
    shorter one (a decode cache grows by appending tokens).
    """
    ch = np.sort(permutation(seed, 50, head_dim)[:n_outlier])
    bq = normal(seed, 51, q_heads * head_dim).reshape(q_heads, head_dim)
    bk = normal(seed, 52, kv_heads * head_dim).reshape(kv_heads, head_dim)
    q = normal(seed, 53, tokens * q_heads * head_dim).reshape(tokens, q_heads, head_dim) + bq
    k = normal(seed, 54, tokens * kv_heads * head_dim).reshape(tokens, kv_heads, head_dim) + bk
    v = normal(seed, 55, tokens * kv_heads * head_dim).reshape(tokens, kv_heads, head_dim)
    q[:, :, ch] *= qk_scale
    k[:, :, ch] *= qk_scale
    v[:min(v_spike_tokens, tokens)] *= v_scale
    return q, k, v
