"""GPU parity of the fused MiX decode attention (frozen-mean K append, Q-K^T,
softmax, MiX requantisation of P, P-V; two launches) against the oracle's
composition of the pinned steps.  The appended K' row is bit-exact; O is
within 1e-3 of each head's largest |O|; the P planes agree except where the
fp32 softmax (expf) and the oracle's fp64 one straddle a rounding boundary."""
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
    d = mix.decode_attention_desc(to_dev(q), kc_g, ks_g, to_dev(vc), to_dev(vs), T, sm, out,
                                  k_new=to_dev(kn) if append else None,
                                  k_mean=to_dev(mean) if append else None, p_codes=pc, p_shared=psh)
    mix.decode_attention(d)
    torch.cuda.synchronize()
    kc_o, ks_o = kc.copy(), ks.copy()
    O, P, (rpc, rps), S = orc.decode_attention(q, kc_o, ks_o, vc, vs, T, sm, k_new=kn if append else None,
                                               k_mean=mean if append else None)
    return (to_host(out), to_host(kc_g), to_host(ks_g), to_host(pc), to_host(psh)), (O, kc_o, ks_o, rpc, rps)


@pytest.mark.parametrize("T,HQ,HK", [(8192, 28, 4), (80, 28, 4), (1, 28, 4), (257, 28, 4), (300, 4, 4),
                                     (1000, 16, 2)])
def test_decode_attention_matches_oracle(mix, orc, T, HQ, HK):
    q, kn, mean, kc, ks, vc, vs = make_cache(orc, T + HQ, T, HQ, HK, prefill=max(1, T // 2))
    (o, kcg, ksg, pc, psh), (O, kco, kso, rpc, rps) = run_both(mix, orc, q, kn, mean, kc, ks, vc, vs, T,
                                                               1 / np.sqrt(128.0))
    assert np.array_equal(kcg, kco) and np.array_equal(ksg, kso)      # the append, bit for bit
    assert row_rel_err(o, O) <= GEMM_REL_TOL, row_rel_err(o, O)
    nb = (T + 31) // 32
    diff = np.mean(pc[:, :nb * 16] != rpc[:, :nb * 16])
    assert diff <= 1e-3, diff
    assert np.mean(psh[:, :nb].view(np.uint16) != rps[:, :nb]) <= 1e-2


def test_decode_attention_no_append_f32(mix, orc):
    T, HQ, HK = 600, 28, 4
    q, kn, mean, kc, ks, vc, vs = make_cache(orc, 3, T, HQ, HK, prefill=300, dtype="f32")
    # the cache already holds the last row: fill it as an earlier step would have
    kp = orc.ksmooth_apply(kn.reshape(1, HK, 128), mean)
    c, s = orc.mx_quantize(kp.reshape(HK, 128).astype(np.float32), 1, 0)
    kc[T - 1], ks[T - 1] = c, s
    (o, kcg, ksg, _, _), (O, _, _, _, _) = run_both(mix, orc, q, kn, mean, kc, ks, vc, vs, T, 0.05, append=False)
    assert np.array_equal(kcg, kc)
    assert row_rel_err(o, O) <= GEMM_REL_TOL


def test_decode_attention_repeat_is_identical(mix, orc):
    """The ticket reset and the chunk-order reduction make repeated calls give
    identical bits."""
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
