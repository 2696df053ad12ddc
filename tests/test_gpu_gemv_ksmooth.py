"""GPU parity of the integer shift-add matmul path (decode shapes) and of
K-smoothing against the CPU oracle."""
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


def make_operands(orc, seed, batch, bgroups, M, N, K, at, bt):
    a = synth.to_bf16_bits(synth.vlm_activations(seed, 0, batch * M, K, visual_rows=(batch * M * 3) // 4))
    w = synth.to_bf16_bits(synth.normal(seed, 1, bgroups * N * K, 0, 0.02).reshape(bgroups * N, K))
    ac, ash = orc.mix_quantize(a, at)
    bc, bs = orc.mx_quantize(w, 1, bt)
    return ac, ash, bc, bs


@pytest.mark.parametrize("M,N,K", [(1, 64, 32), (7, 96, 128), (16, 40, 416), (5, 128, 8192), (3, 2048, 1024)])
@pytest.mark.parametrize("at,bt", [(1, 0), (2, 1), (2, 0), (1, 1)])
def test_shiftadd_gemm_matches_eq6(mix, orc, M, N, K, at, bt):
    import torch
    ac, ash, bc, bs = make_operands(orc, M + N, 1, 1, M, N, K, at, bt)
    ref = orc.gemm(ac, ash, at, -8, bc, bs, bt)
    c = torch.empty((M, N), dtype=torch.float32, device="cuda")
    d = mix.gemm_desc(M, N, K, to_dev(ac), to_dev(ash), at, -8, to_dev(bc), to_dev(bs), bt, c=c,
                      algo=mix.MIX_GEMM_SHIFTADD)
    ws = mix.gemm(d)
    torch.cuda.synchronize()
    assert row_rel_err(to_host(c), ref) <= GEMM_REL_TOL
    # blocks are exact integers; only the fp32 cross-block sum rounds
    assert row_rel_err(to_host(c), ref) < 1e-5


def test_shiftadd_batched_gqa(mix, orc):
    import torch
    B, G, M, N, K = 8, 4, 7, 200, 256
    ac, ash, bc, bs = make_operands(orc, 77, B, B // G, M, N, K, 2, 0)
    ref = orc.gemm(ac.reshape(B, M, -1), ash.reshape(B, M, -1), 2, -8,
                   bc.reshape(B // G, N, -1), bs.reshape(B // G, N, -1), 0, b_group=G)
    c = torch.empty((B, M, N), dtype=torch.float32, device="cuda")
    d = mix.gemm_desc(M, N, K, to_dev(ac), to_dev(ash), 2, -8, to_dev(bc), to_dev(bs), 0, c=c,
                      batch=B, b_group=G, algo=mix.MIX_GEMM_SHIFTADD)
    mix.gemm(d)
    torch.cuda.synchronize()
    assert row_rel_err(to_host(c), ref) < 1e-5


@pytest.mark.parametrize("epi,mx_flags", [(1, 0), (2, 0), (3, 0), (4, 0), (3, 4), (4, 4)])
def test_shiftadd_epilogue_codes_are_quantised_c(mix, orc, epi, mx_flags):
    """The fused output quantiser's planes equal the oracle quantiser applied
    to the GPU's own fp32 C, bit for bit."""
    import torch
    M, N, K = 9, 256, 512
    ac, ash, bc, bs = make_operands(orc, 5, 1, 1, M, N, K, 2, 1)
    c = torch.empty((M, N), dtype=torch.float32, device="cuda")
    oc = torch.empty((M, N // 2), dtype=torch.uint8, device="cuda")
    osh = torch.empty((M, N // 32), dtype=torch.int16 if epi == 2 else torch.uint8, device="cuda")
    d = mix.gemm_desc(M, N, K, to_dev(ac), to_dev(ash), 2, -8, to_dev(bc), to_dev(bs), 1, c=c, epi=epi,
                      epi_ebias=-6, epi_flags=1 if epi <= 2 else mx_flags, out_codes=oc, out_shared=osh,
                      algo=mix.MIX_GEMM_SHIFTADD)
    mix.gemm(d)
    torch.cuda.synchronize()
    ch = to_host(c)
    if epi <= 2:
        rc, rs = orc.mix_quantize(ch, epi, -6, 1)
    else:
        rc, rs = orc.mx_quantize(ch, 1, 0 if epi == 3 else 1, mx_flags)
    assert np.array_equal(to_host(oc), rc) and np.array_equal(to_host(osh).astype(rs.dtype), rs)


def test_decode_attention_shapes(mix, orc):
    """Batch-1 decode over an 8192-token cache, GQA 28/4, head_dim 128:
    S = q K'^T (K' MX along head_dim) and O = P V (V MX along tokens)."""
    import torch
    T, HQ, HK, D = 8192, 28, 4, 128
    q, k, v = synth.attention_qkv(0, T, HQ, HK, D)
    kb = synth.to_bf16_bits(k)
    mu = orc.ksmooth_mean(kb[:4096])
    ks = orc.ksmooth_apply(kb, mu.astype(np.float32))            # [T, HK, D]
    qd = synth.to_bf16_bits(q[-1])                               # [HQ, D] the newest query
    qc, qs = orc.mix_quantize(qd, 2)
    kc_list, ks_list, vc_list, vs_list = [], [], [], []
    vb = synth.to_bf16_bits(v)
    for h in range(HK):
        c_, s_ = orc.mx_quantize(np.ascontiguousarray(ks[:, h]), 1, 0)   # [T, D] blocks along D
        kc_list.append(c_); ks_list.append(s_)
        c_, s_ = orc.mx_quantize(np.ascontiguousarray(vb[:, h]), 0, 0)   # V[T, D] -> [D, T]
        vc_list.append(c_); vs_list.append(s_)
    kc, kss = np.stack(kc_list), np.stack(ks_list)
    s_gpu = torch.empty((HK, 7, T), dtype=torch.float32, device="cuda")
    d = mix.gemm_desc(7, T, D, to_dev(qc), to_dev(qs), 2, -8, to_dev(kc), to_dev(kss), 0, c=s_gpu,
                      batch=HK, b_group=1, algo=mix.MIX_GEMM_AUTO)
    mix.gemm(d)
    torch.cuda.synchronize()
    s_ref = orc.gemm(qc.reshape(HK, 7, -1), qs.reshape(HK, 7, -1), 2, -8, kc, kss, 0)
    assert row_rel_err(to_host(s_gpu), s_ref) < 1e-5
    # P from a softmax of the oracle scores (scaled by 1/sqrt(D)), quantised with ebias -15
    sr = s_ref.reshape(HQ, T) / np.sqrt(D)
    p = np.exp(sr - sr.max(1, keepdims=True)); p /= p.sum(1, keepdims=True)
    pc, ps = orc.mix_quantize(p.astype(np.float32), 2, -15)
    vc, vs = np.stack(vc_list), np.stack(vs_list)
    o_gpu = torch.empty((HK, 7, D), dtype=torch.float32, device="cuda")
    d = mix.gemm_desc(7, D, T, to_dev(pc), to_dev(ps), 2, -15, to_dev(vc), to_dev(vs), 0, c=o_gpu,
                      batch=HK, algo=mix.MIX_GEMM_AUTO)
    mix.gemm(d)
    torch.cuda.synchronize()
    o_ref = orc.gemm(pc.reshape(HK, 7, -1), ps.reshape(HK, 7, -1), 2, -15, vc, vs, 0)
    assert row_rel_err(to_host(o_gpu), o_ref) < 1e-5


# ---------------------------------------------------------------------------
# K-smoothing


@pytest.mark.parametrize("tokens,bf16", [(1, True), (1, False), (33, True), (33, False), (4096, True),
                                         (4096, False), (16384, False), (32768, True)])
def test_ksmooth_compute_and_apply(mix, orc, tokens, bf16):
    """Up to 4096 tokens the keys fit the one-pass kernel (each CTA keeps its
    run of tokens in shared memory); the two largest cases are too long for it
    and take the partial / finalize / apply kernels."""
    import torch
    HK, D = 4, 128
    _, k, _ = synth.attention_qkv(1, tokens, 2, HK, D)
    kk = synth.to_bf16_bits(k) if bf16 else synth.to_f32(k)
    mu_ref = orc.ksmooth_mean(kk)
    kd = to_dev(kk.reshape(tokens, HK * D))
    mean = torch.empty((HK, D), dtype=torch.float32, device="cuda")
    kout = torch.empty((tokens, HK, D), dtype=torch.float32, device="cuda")
    ws = torch.empty(mix.ksmooth_workspace_bytes(tokens, HK, D), dtype=torch.uint8, device="cuda")
    mix.ksmooth_kv(kd, tokens, HK, D, HK * D, mean, mix.KSMOOTH_COMPUTE, kout, ws)
    torch.cuda.synchronize()
    mu = to_host(mean).astype(np.float64)
    assert np.max(np.abs(mu - mu_ref) / np.maximum(np.abs(mu_ref), 1e-30)) <= 1e-6
    want = orc.ksmooth_apply(kk, to_host(mean))
    assert np.array_equal(to_host(kout), want)


def test_ksmooth_frozen_mean_decode(mix, orc):
    import torch
    HK, D = 4, 128
    _, k, _ = synth.attention_qkv(2, 4100, 2, HK, D)
    kb = synth.to_bf16_bits(k)
    mu = orc.ksmooth_mean(kb[:4096]).astype(np.float32)
    new = np.ascontiguousarray(kb[4096:])
    kout = torch.empty((4, HK, D), dtype=torch.float32, device="cuda")
    mean = to_dev(mu)
    mix.ksmooth_kv(to_dev(new.reshape(4, HK * D)), 4, HK, D, HK * D, mean, mix.KSMOOTH_APPLY_FROZEN, kout)
    torch.cuda.synchronize()
    assert np.array_equal(to_host(kout), orc.ksmooth_apply(new, mu))
    assert np.array_equal(to_host(mean), mu)   # the frozen mean is an input only
