"""GPU parity of the prefill attention matmuls in exactly the call forms the
benchmark times: 28 query heads over 4 KV heads (GQA groups of 7), head_dim
128, 4096 tokens.

  * S = Q K'^T: A is the MiX-4.5b Q read in place from its [token][head][128]
    layout (row stride 28*128, batch stride 128), B the MXINT4 K' read in
    place from [token][kv head][128] (row stride 4*128, batch stride 128).
  * O = P V: A is a causal softmax P [head][token][token] in MiX-4.5b with
    ebias -15, B the MXINT4 V planes quantised down the token axis.
  * The MiX quantiser of P at its full size, 114688 x 4096.

Every oracle input comes from the seeded generators (or from torch, for the
softmax that builds P) and is quantised by the oracle on the host; the GPU's
planes are compared with the oracle's bit for bit, and the matmul outputs on
sampled rows of sampled heads (all four KV groups) within 1e-3 of each row's
largest reference magnitude."""
import math

import numpy as np
import pytest

from quantized_vlm_gemm_mix_b300 import synth
from helpers import GEMM_REL_TOL, row_rel_err, to_dev, to_host

pytestmark = pytest.mark.gpu

T, HQ, HK, D = 4096, 28, 4, 128
G = HQ // HK
HEADS = (0, 6, 7, 13, 15, 20, 27)   # both ends of every KV group


@pytest.fixture(scope="module")
def mix():
    import torch
    assert torch.cuda.is_available()
    from quantized_vlm_gemm_mix_b300 import mix as m
    return m


def sample_rows(rng, n):
    """n token rows, always including the first and last few (the mostly-zero
    and the full causal rows)."""
    mid = rng.choice(np.arange(4, T - 4), n - 8, replace=False)
    return np.sort(np.concatenate([np.arange(4), mid, np.arange(T - 4, T)]))


def test_qk_prefill_bench_form(mix, orc):
    import torch
    q, k, _ = synth.attention_qkv(11, T, HQ, HK, D)
    qb = np.ascontiguousarray(synth.to_bf16_bits(q).reshape(T, HQ * D))
    kb = synth.to_bf16_bits(k)                                      # [T, HK, D]
    mu = orc.ksmooth_mean(kb).astype(np.float32)
    kp = orc.ksmooth_apply(kb, mu).reshape(T * HK, D)               # rows (token, kv head)
    qc, qs = orc.mix_quantize(qb.reshape(T * HQ, D), 2)             # rows (token, head)
    kc, ks = orc.mx_quantize(kp, 1, 0)
    # the GPU quantisers on the same inputs, in the bench's call forms
    qc_g, qs_g = mix.quantize_mix(to_dev(qb).view(T * HQ, D), mix.MIX_T2_4P5)
    kc_g, ks_g = mix.quantize_mx(to_dev(kp), 1, mix.MX_INT4)
    assert np.array_equal(to_host(qc_g), qc) and np.array_equal(to_host(qs_g), qs)
    assert np.array_equal(to_host(kc_g), kc) and np.array_equal(to_host(ks_g), ks)
    S = torch.empty((HQ, T, T), dtype=torch.float32, device="cuda")
    d = mix.gemm_desc(T, T, D, qc_g, qs_g, mix.MIX_T2_4P5, -8, kc_g, ks_g, mix.MX_INT4, c=S, batch=HQ,
                      b_group=G, a_ld=HQ * D, a_batch_stride=D, b_ld=HK * D, b_batch_stride=D,
                      algo=mix.MIX_GEMM_TCGEN05)
    mix.gemm(d)
    torch.cuda.synchronize()
    assert mix.mix_device_error() == 0
    rng = np.random.default_rng(12)
    kc3, ks3 = kc.reshape(T, HK, D // 2), ks.reshape(T, HK, D // 32)
    qc3, qs3 = qc.reshape(T, HQ, D // 2), qs.reshape(T, HQ, D // 32)
    for h in HEADS:
        rows = sample_rows(rng, 64)
        g = h // G
        ref = orc.gemm(np.ascontiguousarray(qc3[rows, h]), np.ascontiguousarray(qs3[rows, h]), 2, -8,
                       np.ascontiguousarray(kc3[:, g]), np.ascontiguousarray(ks3[:, g]), 0)
        got = to_host(S[h, torch.from_numpy(rows).cuda()])
        err = row_rel_err(got, ref)
        assert err <= GEMM_REL_TOL, (h, err)


def causal_softmax_bf16(seed):
    """A causal softmax P [HQ, T, T] (bf16) of seeded scores, made by torch on
    the device (the softmax is outside the library)."""
    import torch
    g = torch.Generator(device="cuda").manual_seed(seed)
    P = torch.empty((HQ, T, T), dtype=torch.bfloat16, device="cuda")
    causal = torch.ones((T, T), dtype=torch.bool, device="cuda").tril()
    for h in range(HQ):
        s = torch.randn((T, T), device="cuda", generator=g) * 3.0
        P[h] = torch.softmax((s / math.sqrt(D)).masked_fill(~causal, float("-inf")), dim=-1).to(torch.bfloat16)
    return P


def test_pv_prefill_bench_form_and_full_size_p_quantiser(mix, orc):
    import torch
    P = causal_softmax_bf16(13)
    pc_g = torch.empty((HQ * T, T // 2), dtype=torch.uint8, device="cuda")
    ps_g = torch.empty((HQ * T, T // 32), dtype=torch.int16, device="cuda")
    mix.mix_quantize(P, HQ * T, T, T, mix.MIX_T2_4P5, -15, 1, pc_g, ps_g)
    _, _, v = synth.attention_qkv(14, T, HQ, HK, D)
    vb = np.ascontiguousarray(synth.to_bf16_bits(v).reshape(T, HK * D))
    vc, vs = orc.mx_quantize(vb, 0, 0)                              # [HK*D, T/2], [HK*D, T/32]
    vqc_g = torch.empty((HK, D, T // 2), dtype=torch.uint8, device="cuda")
    vqs_g = torch.empty((HK, D, T // 32), dtype=torch.uint8, device="cuda")
    mix.mx_quantize(to_dev(vb), T, HK * D, HK * D, 0, mix.MX_INT4, 0, vqc_g, vqs_g)
    assert np.array_equal(to_host(vqc_g).reshape(HK * D, -1), vc)
    assert np.array_equal(to_host(vqs_g).reshape(HK * D, -1), vs)
    # the benchmark's form states P's causal bound (a_causal); the same call
    # without it reads every k-step and must give the same bits
    outs = []
    for causal in (1, 0):
        O = torch.empty((HQ, T, D), dtype=torch.float32, device="cuda")
        d = mix.gemm_desc(T, D, T, pc_g, ps_g, mix.MIX_T2_4P5, -15, vqc_g, vqs_g, mix.MX_INT4, c=O, batch=HQ,
                          b_group=G, algo=mix.MIX_GEMM_TCGEN05, a_causal=causal)
        mix.gemm(d)
        torch.cuda.synchronize()
        assert mix.mix_device_error() == 0
        outs.append(O)
    assert torch.equal(outs[0], outs[1])
    O = outs[0]
    vc3, vs3 = vc.reshape(HK, D, -1), vs.reshape(HK, D, -1)
    rng = np.random.default_rng(15)
    for h in HEADS:
        rows = sample_rows(rng, 64)
        ridx = torch.from_numpy(h * T + rows).cuda()
        p_rows = to_host(P.view(HQ * T, T)[ridx])                      # bf16 bits
        pc, ps = orc.mix_quantize(p_rows, 2, -15)
        # the full-size P quantiser, bit for bit on these rows
        assert np.array_equal(to_host(pc_g[ridx]), pc), h
        assert np.array_equal(to_host(ps_g[ridx]), ps), h
        ref = orc.gemm(pc, ps, 2, -15, vc3[h // G], vs3[h // G], 0)
        got = to_host(O[h, torch.from_numpy(rows).cuda()])
        err = row_rel_err(got, ref)
        assert err <= GEMM_REL_TOL, (h, err)


@pytest.mark.parametrize("algo", ["staged", "fused"])
@pytest.mark.parametrize("N", [128, 288])
def test_strided_a_and_b_gqa(mix, orc, algo, N):
    """Both operands read in place through interleaved strides, at a size the
    oracle checks in full: A rows of batch b at m * (B*K) + b * K, B rows of
    KV group g at n * (BB*K) + g * K (the [token][head][dim] layouts of Q and
    K'), batch 6 in groups of 3."""
    import torch
    B, GR, M, K = 6, 3, 160, 128
    BB = B // GR
    a = synth.to_bf16_bits(synth.vlm_activations(40, 0, B * M, K, visual_rows=B * M // 2))
    w = synth.to_bf16_bits(synth.normal(41, 1, BB * N * K, 0, 0.5).reshape(BB * N, K))
    ac, ash = orc.mix_quantize(a, 2)
    bc, bs = orc.mx_quantize(w, 1, 0)
    acb = ac.reshape(B, M, K // 2).transpose(1, 0, 2).copy()        # [M, B, K/2]
    ashb = ash.reshape(B, M, K // 32).transpose(1, 0, 2).copy()
    bcb = bc.reshape(BB, N, K // 2).transpose(1, 0, 2).copy()       # [N, BB, K/2]
    bsb = bs.reshape(BB, N, K // 32).transpose(1, 0, 2).copy()
    c = torch.empty((B, M, N), dtype=torch.float32, device="cuda")
    algo_id = mix.MIX_GEMM_TCGEN05_STAGED if algo == "staged" else mix.MIX_GEMM_TCGEN05_FUSED
    d = mix.gemm_desc(M, N, K, to_dev(acb), to_dev(ashb), 2, -8, to_dev(bcb), to_dev(bsb), 0, c=c, batch=B,
                      b_group=GR, a_ld=B * K, a_batch_stride=K, b_ld=BB * K, b_batch_stride=K, algo=algo_id)
    mix.gemm(d)
    torch.cuda.synchronize()
    assert mix.mix_device_error() == 0
    ref = orc.gemm(ac.reshape(B, M, -1), ash.reshape(B, M, -1), 2, -8, bc.reshape(BB, N, -1),
                   bs.reshape(BB, N, -1), 0, b_group=GR)
    assert row_rel_err(to_host(c), ref) <= GEMM_REL_TOL


def test_clamp_count_matches_oracle(mix, orc):
    """The clamped-block count on wide-range inputs (fp32 and bf16, strided
    rows, several ebias) and on the step's activations, which must show
    none at ebias -8."""
    import torch
    rng = np.random.default_rng(16)
    x = (rng.standard_normal((300, 320)) * np.exp2(rng.integers(-40, 40, (300, 320)))).astype(np.float32)
    x[5, :32] = 0.0
    x[6, 3] = np.inf
    x[7, 40] = np.nan
    x[8, 70] = 2.0 ** -140
    for arr in (x, synth.to_bf16_bits(x.astype(np.float64))):
        for eb in (-30, -8, 0, 20):
            got = to_host(mix.clamp_count(to_dev(arr), eb))
            assert tuple(int(v) for v in got) == orc.mix_clamp_count(arr, eb), eb
        wide = np.zeros((arr.shape[0], 384), dtype=arr.dtype)
        wide[:, :320] = arr
        dev = to_dev(wide)[:, :320]
        got = torch.empty((2,), dtype=torch.int64, device="cuda")
        mix.mix_clamp_count(dev, arr.shape[0], 320, 384, -8, got)
        assert tuple(int(v) for v in to_host(got)) == orc.mix_clamp_count(arr, -8)
    act = synth.to_bf16_bits(synth.vlm_activations(0, 1, 4096, 3584, visual_rows=3072))
    assert tuple(int(v) for v in to_host(mix.clamp_count(to_dev(act), -8))) == orc.mix_clamp_count(act, -8) == (0, 0)
