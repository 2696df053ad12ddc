"""GPU parity of the fused MiX decode attention (frozen-mean K append, Q-K^T,
softmax, MiX requantisation of P, P-V; one cooperative launch, or two for a
cache too long for it) against the oracle's
composition of the pinned steps.  The appended K' row is bit-exact; O is
within 1e-3 of each head's largest |O|; the kernel's own fp32 P (a debug
output) is within fp32 rounding of the oracle's softmax, and the P planes are
bit-exact against the oracle quantiser applied to that P."""
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


def make_cache(orc, seed, T, HQ, HK, prefill, dtype="bf16"):
    """K' cache rows 0..T-2 (smoothed with the frozen prefill mean), the new
    token's raw key, and the V cache along tokens (capacity rounded to 32)."""
    q, k, v = synth.attention_qkv(seed, T, q_heads=HQ, kv_heads=HK)
    conv = synth.to_bf16_bits if dtype == "bf16" else synth.to_f32
    mean = orc.ksmooth_mean(synth.to_bf16_bits(k[:prefill])).astype(np.float32)
    kc = np.zeros((T, HK, 64), np.uint8)
    ks = np.zeros((T, HK, 4), np.uint8)
    if T > 1:
        kp = orc.ksmooth_apply(synth.to_bf16_bits(k[:T - 1]), mean)
        c, s = orc.mx_quantize(kp.reshape(-1, 128).astype(np.float32), 1, 0)
        kc[:T - 1], ks[:T - 1] = c.reshape(T - 1, HK, 64), s.reshape(T - 1, HK, 4)
    Tv = (T + 31) // 32 * 32
    vv = np.zeros((Tv, HK, 128))
    vv[:T] = v
    vc, vs = orc.mx_quantize(synth.to_bf16_bits(vv.reshape(Tv, HK * 128)), 0, 0)
    return conv(q[T - 1]), conv(k[T - 1]), mean, kc, ks, vc.reshape(HK, 128, -1), vs.reshape(HK, 128, -1)


def run_both(mix, orc, q, kn, mean, kc, ks, vc, vs, T, sm, append=True):
    import torch
    HQ = q.shape[0]
    Tv = vc.shape[2] * 2
    kc_g, ks_g = to_dev(kc.copy()), to_dev(ks.copy())
    out = torch.empty((HQ, 128), dtype=torch.float32, device="cuda")
    pc = torch.zeros((HQ, Tv // 2), dtype=torch.uint8, device="cuda")
    psh = torch.zeros((HQ, Tv // 32), dtype=torch.int16, device="cuda")
    pval = torch.full((HQ, Tv), -1.0, dtype=torch.float32, device="cuda")
    d = mix.decode_attention_desc(to_dev(q), kc_g, ks_g, to_dev(vc), to_dev(vs), T, sm, out,
                                  k_new=to_dev(kn) if append else None,
                                  k_mean=to_dev(mean) if append else None, p_codes=pc, p_shared=psh,
                                  p_values=pval)
    mix.decode_attention(d)
    torch.cuda.synchronize()
    assert mix.mix_device_error() == 0
    kc_o, ks_o = kc.copy(), ks.copy()
    O, P, (rpc, rps), S = orc.decode_attention(q, kc_o, ks_o, vc, vs, T, sm, k_new=kn if append else None,
                                               k_mean=mean if append else None)
    got = (to_host(out), to_host(kc_g), to_host(ks_g), to_host(pc), to_host(psh), to_host(pval))
    return got, (O, kc_o, ks_o, rpc, rps, P, S)


def check_p(T, sm, got, ref, orc):
    """The kernel's P: within fp32 rounding of the oracle's softmax, and its
    MiX-4.5b planes bit-exact against the oracle quantiser on that same P."""
    _, _, _, pc, psh, pval = got
    P, S = ref[5], ref[6]
    nb = (T + 31) // 32
    pv = pval[:, :32 * nb]
    assert np.all(pv[:, T:] == 0.0)
    # S leaves the kernel as an fp32 sum of four exact block terms (a few
    # roundings of 2^-24 of the row's largest |S|), which moves z = sm S and
    # so P by that much relative; expf, the fp32 divide and the chunk sums
    # add a few ulp.
    tol = 2.0 * sm * 2.0 ** -21 * np.max(np.abs(S), axis=1, keepdims=True) + 4e-6
    err = np.abs(pv[:, :T].astype(np.float64) - P) / np.max(P, axis=1, keepdims=True)
    assert np.all(err <= tol), float(np.max(err - tol))
    rc, rs = orc.mix_quantize(np.ascontiguousarray(pv), 2, -15, 1)
    assert np.array_equal(pc[:, :16 * nb], rc)
    assert np.array_equal(psh[:, :nb].view(np.uint16), rs)


@pytest.mark.parametrize("T,HQ,HK", [(8192, 28, 4), (80, 28, 4), (1, 28, 4), (257, 28, 4), (300, 4, 4),
                                     (1000, 16, 2), (40000, 8, 4)])
def test_decode_attention_matches_oracle(mix, orc, T, HQ, HK):
    """Up to a few tens of thousands of tokens the step is one kernel whose
    chunks of keys, values and scores stay in shared memory; the 40000-token
    cache (chunks of 1088 tokens) is too long for it and takes two kernels."""
    q, kn, mean, kc, ks, vc, vs = make_cache(orc, T + HQ, T, HQ, HK, prefill=max(1, T // 2))
    got, ref = run_both(mix, orc, q, kn, mean, kc, ks, vc, vs, T, 1 / np.sqrt(128.0))
    o, kcg, ksg = got[:3]
    O, kco, kso = ref[:3]
    assert np.array_equal(kcg, kco) and np.array_equal(ksg, kso)      # the append, bit for bit
    assert row_rel_err(o, O) <= GEMM_REL_TOL, row_rel_err(o, O)
    check_p(T, 1 / np.sqrt(128.0), got, ref, orc)


def test_decode_attention_no_append_f32(mix, orc):
    T, HQ, HK = 600, 28, 4
    q, kn, mean, kc, ks, vc, vs = make_cache(orc, 3, T, HQ, HK, prefill=300, dtype="f32")
    # the cache already holds the last row: fill it as an earlier step would have
    kp = orc.ksmooth_apply(kn.reshape(1, HK, 128), mean)
    c, s = orc.mx_quantize(kp.reshape(HK, 128).astype(np.float32), 1, 0)
    kc[T - 1], ks[T - 1] = c, s
    got, ref = run_both(mix, orc, q, kn, mean, kc, ks, vc, vs, T, 0.05, append=False)
    assert np.array_equal(got[1], kc)
    assert row_rel_err(got[0], ref[0]) <= GEMM_REL_TOL
    check_p(T, 0.05, got, ref, orc)


def test_decode_attention_repeat_is_identical(mix, orc):
    """The barrier counter reset and the chunk-order reductions make repeated
    calls give identical bits."""
    import torch
    T, HQ, HK = 2048, 28, 4
    q, kn, mean, kc, ks, vc, vs = make_cache(orc, 11, T, HQ, HK, prefill=1024)
    out = torch.empty((HQ, 128), dtype=torch.float32, device="cuda")
    d = mix.decode_attention_desc(to_dev(q), to_dev(kc), to_dev(ks), to_dev(vc), to_dev(vs), T, 0.088, out,
                                  k_new=to_dev(kn), k_mean=to_dev(mean))
    ws = mix.decode_attention(d)
    first = to_host(out).copy()
    for _ in range(3):
        mix.decode_attention(d, ws)
    torch.cuda.synchronize()
    assert np.array_equal(to_host(out), first)
