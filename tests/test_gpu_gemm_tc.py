"""GPU parity of the tcgen05 A-MiX x W-MX matmul and its fused output
quantiser against the CPU oracle (Eq. (6): int64 shift-add per block, fp64
across blocks).  Floating-point results: max error relative to each output
row's largest reference magnitude <= 1e-3.  Quantised outputs: bit-exact
against the oracle quantiser applied to the GPU's own fp32 C."""
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


def operands(orc, seed, M, N, K, at, bt, a_dtype="bf16", batch=1, bb=1):
    a = synth.vlm_activations(seed, 0, batch * M, K, visual_rows=(batch * M * 3) // 4)
    a = synth.to_bf16_bits(a) if a_dtype == "bf16" else synth.to_f32(a)
    w = synth.to_bf16_bits(synth.normal(seed, 1, bb * N * K, 0, 0.02).reshape(bb * N, K))
    ac, ash = orc.mix_quantize(a, at)
    bc, bs = orc.mx_quantize(w, 1, bt)
    return ac, ash, bc, bs


ALGOS = ["staged", "fused"]


def algo_id(mix, algo):
    return {"auto": mix.MIX_GEMM_TCGEN05, "staged": mix.MIX_GEMM_TCGEN05_STAGED,
            "fused": mix.MIX_GEMM_TCGEN05_FUSED}[algo]


def run_tc(mix, ac, ash, at, bc, bs, bt, M, N, K, epi=0, epi_ebias=-8, epi_flags=1, batch=1, b_group=1,
           want_c=True, algo="auto", **kw):
    import torch
    c = torch.empty((batch, M, N), dtype=torch.float32, device="cuda") if want_c else None
    oc = osh = None
    if epi:
        oc = torch.empty((batch, M, N // 2), dtype=torch.uint8, device="cuda")
        osh = torch.empty((batch, M, N // 32), dtype=torch.int16 if epi == 2 else torch.uint8, device="cuda")
    d = mix.gemm_desc(M, N, K, to_dev(ac), to_dev(ash), at, -8, to_dev(bc), to_dev(bs), bt, c=c, epi=epi,
                      epi_ebias=epi_ebias, epi_flags=epi_flags, out_codes=oc, out_shared=osh, batch=batch,
                      b_group=b_group, algo=algo_id(mix, algo), **kw)
    mix.gemm(d)
    torch.cuda.synchronize()
    assert mix.mix_device_error() == 0
    return (to_host(c) if want_c else None), (to_host(oc) if epi else None), (to_host(osh) if epi else None)


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("at,bt", [(2, 1), (1, 0), (2, 0), (1, 1)])
@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (300, 520, 416), (1, 32, 32), (17, 288, 3584)])
def test_tc_matches_eq6(mix, orc, M, N, K, at, bt, algo):
    ac, ash, bc, bs = operands(orc, M * 7 + N + K, M, N, K, at, bt)
    ref = orc.gemm(ac, ash, at, -8, bc, bs, bt)
    c, _, _ = run_tc(mix, ac, ash, at, bc, bs, bt, M, N, K, algo=algo)
    err = row_rel_err(c[0], ref)
    assert err <= GEMM_REL_TOL, err


@pytest.mark.parametrize("at,bt", [(2, 1), (1, 0)])
@pytest.mark.parametrize("M,N,K,batch,b_group", [(300, 544, 416, 1, 1), (130, 768, 1024, 1, 1),
                                                 (160, 288, 128, 6, 3), (257, 1024, 96, 1, 1)])
def test_staged_equals_fused_bitwise(mix, orc, M, N, K, batch, b_group, at, bt):
    """The staged variant (operands expanded once into the workspace, scales
    moved by tcgen05.cp) and the fused-decode variant feed the MMA the same
    exact operand values in the same K order, so their fp32 outputs agree bit
    for bit; the fused MiX epilogue planes then agree too."""
    ac, ash, bc, bs = operands(orc, 31 + M + N + K, M, N, K, at, bt, batch=batch, bb=batch // b_group)
    c1, o1, s1 = run_tc(mix, ac, ash, at, bc, bs, bt, M, N, K, epi=2, batch=batch, b_group=b_group, algo="staged")
    c2, o2, s2 = run_tc(mix, ac, ash, at, bc, bs, bt, M, N, K, epi=2, batch=batch, b_group=b_group, algo="fused")
    assert np.array_equal(c1.view(np.uint32), c2.view(np.uint32))
    assert np.array_equal(o1, o2) and np.array_equal(s1, s2)
    ref = orc.gemm(ac.reshape(batch, M, -1), ash.reshape(batch, M, -1), at, -8,
                   bc.reshape(batch // b_group, N, -1), bs.reshape(batch // b_group, N, -1), bt, b_group=b_group)
    assert row_rel_err(c1, ref) <= GEMM_REL_TOL


def test_tc_agrees_with_shiftadd_path(mix, orc):
    import torch
    M, N, K = 16, 512, 1024
    ac, ash, bc, bs = operands(orc, 3, M, N, K, 2, 1)
    c_tc, _, _ = run_tc(mix, ac, ash, 2, bc, bs, 1, M, N, K)
    c2 = torch.empty((M, N), dtype=torch.float32, device="cuda")
    d = mix.gemm_desc(M, N, K, to_dev(ac), to_dev(ash), 2, -8, to_dev(bc), to_dev(bs), 1, c=c2,
                      algo=mix.MIX_GEMM_SHIFTADD)
    mix.gemm(d)
    torch.cuda.synchronize()
    assert row_rel_err(c_tc[0], to_host(c2).astype(np.float64)) <= GEMM_REL_TOL


def test_tiny_end_to_end_config(mix, orc):
    """fp32 A [128 x 512] -> MiX-4.5b; W [512 x 256] N(0, 0.02) -> MXFP4 along K;
    C = A W in fp32 plus the fused MiX-4.5b output quantiser; seed 0."""
    import torch
    a = synth.to_f32(synth.vlm_activations(0, 0, 128, 512, visual_rows=96, n_outlier=4))
    w = synth.to_f32(synth.gaussian_weights(0, 2, 512, 256))
    ac_g, ash_g = mix.quantize_mix(to_dev(a), mix.MIX_T2_4P5)
    bc_g, bs_g = mix.quantize_mx(to_dev(w), 0, mix.MX_FP4_E2M1)
    ac, ash = orc.mix_quantize(a, 2)
    bc, bs = orc.mx_quantize(w, 0, 1)
    assert np.array_equal(to_host(ac_g), ac) and np.array_equal(to_host(ash_g), ash)
    assert np.array_equal(to_host(bc_g), bc) and np.array_equal(to_host(bs_g), bs)
    c, oc, osh = run_tc(mix, ac, ash, 2, bc, bs, 1, 128, 256, 512, epi=2)
    ref = orc.gemm(ac, ash, 2, -8, bc, bs, 1)
    assert row_rel_err(c[0], ref) <= GEMM_REL_TOL
    rc, rs = orc.mix_quantize(c[0], 2, -8, 1)
    assert np.array_equal(oc[0], rc) and np.array_equal(osh[0], rs)
    # against the oracle's own C the codes may differ only at rounding ties
    rc2, _ = orc.mix_quantize(ref.astype(np.float32), 2, -8, 1)
    assert np.mean(oc[0] != rc2) < 1e-3


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("epi,mx_flags", [(1, 0), (2, 0), (3, 0), (4, 0), (3, 4), (4, 4), (4, 2)])
def test_tc_epilogue_formats(mix, orc, epi, mx_flags, algo):
    """The fused output quantiser (MiX, MX with the ceil, tight or floor
    exponent rule) equals the oracle quantiser applied to the GPU's own C."""
    M, N, K = 200, 512, 640
    ac, ash, bc, bs = operands(orc, 11 + epi, M, N, K, 1, 0)
    c, oc, osh = run_tc(mix, ac, ash, 1, bc, bs, 0, M, N, K, epi=epi, epi_ebias=-6,
                        epi_flags=1 if epi <= 2 else mx_flags, algo=algo)
    if epi <= 2:
        rc, rs = orc.mix_quantize(c[0], epi, -6, 1)
    else:
        rc, rs = orc.mx_quantize(c[0], 1, 0 if epi == 3 else 1, mx_flags)
    assert np.array_equal(oc[0], rc) and np.array_equal(osh[0].astype(rs.dtype), rs)


def test_tc_epilogue_only_no_c(mix, orc):
    M, N, K = 130, 256, 256
    ac, ash, bc, bs = operands(orc, 19, M, N, K, 2, 1)
    c, _, _ = run_tc(mix, ac, ash, 2, bc, bs, 1, M, N, K)
    _, oc, osh = run_tc(mix, ac, ash, 2, bc, bs, 1, M, N, K, epi=2, want_c=False)
    rc, rs = orc.mix_quantize(c[0], 2, -8, 1)
    assert np.array_equal(oc[0], rc) and np.array_equal(osh[0], rs)


@pytest.mark.parametrize("algo", ALGOS)
def test_tc_batched_gqa_and_strides(mix, orc, algo):
    """Batch 6 in groups of 3 sharing B; A read through an interleaved row
    stride (the (token, head) layout of a QKV projection)."""
    B, G, M, N, K = 6, 3, 160, 288, 128
    ac, ash, bc, bs = operands(orc, 23, M, N, K, 2, 0, batch=B, bb=B // G)
    # interleave: row m of batch b at element offset m * (B*K) + b * K
    acb = ac.reshape(B, M, K // 2).transpose(1, 0, 2).copy()      # [M, B, K/2]
    ashb = ash.reshape(B, M, K // 32).transpose(1, 0, 2).copy()
    c, _, _ = run_tc(mix, acb, ashb, 2, bc, bs, 0, M, N, K, batch=B, b_group=G, a_ld=B * K, a_batch_stride=K,
                     algo=algo)
    ref = orc.gemm(ac.reshape(B, M, -1), ash.reshape(B, M, -1), 2, -8, bc.reshape(B // G, N, -1),
                   bs.reshape(B // G, N, -1), 0, b_group=G)
    assert row_rel_err(c, ref) <= GEMM_REL_TOL


def sampled_check(orc, c, ac, ash, at, bc, bs, bt, rows, cols, ebias=-8):
    ref = orc.gemm(ac[rows], ash[rows], at, ebias, bc[cols], bs[cols], bt)
    return row_rel_err(c[np.ix_(rows, cols)], ref)


@pytest.mark.parametrize("name,K,N", [("qkv", 3584, 4608), ("o", 3584, 3584), ("gate_up", 3584, 37888),
                                      ("down", 18944, 3584)])
def test_qwen2vl_prefill_linears_sampled(mix, orc, name, K, N):
    """M = 4096 tokens, A-MiX-4.5b x W-MXFP4, fused MiX-4.5b epilogue, at full
    size; the oracle checks 96 sampled rows x 256 sampled columns of C, and the
    epilogue planes of the sampled rows bit for bit."""
    import torch
    M = 4096
    x = synth.to_bf16_bits(synth.vlm_activations(1, 10 + K, M, K, visual_rows=3072))
    w = synth.to_bf16_bits(synth.gaussian_weights(1, 20 + N, K, N))
    ac_g, ash_g = mix.quantize_mix(to_dev(x), mix.MIX_T2_4P5)
    bc_g, bs_g = mix.quantize_mx(to_dev(w), 0, mix.MX_FP4_E2M1)
    del w
    c = torch.empty((M, N), dtype=torch.float32, device="cuda")
    oc = torch.empty((M, N // 2), dtype=torch.uint8, device="cuda")
    osh = torch.empty((M, N // 32), dtype=torch.int16, device="cuda")
    d = mix.gemm_desc(M, N, K, ac_g, ash_g, 2, -8, bc_g, bs_g, 1, c=c, epi=2, out_codes=oc, out_shared=osh,
                      algo=mix.MIX_GEMM_TCGEN05)
    mix.gemm(d)
    torch.cuda.synchronize()
    rng = np.random.default_rng(K + N)
    rows = np.sort(rng.choice(M, 96, replace=False))
    cols = np.sort(rng.choice(N, 256, replace=False))
    ac, ash = to_host(ac_g), to_host(ash_g)
    bc, bs = to_host(bc_g), to_host(bs_g)
    ch = to_host(c)
    assert sampled_check(orc, ch, ac, ash, 2, bc, bs, 1, rows, cols) <= GEMM_REL_TOL
    rc, rs = orc.mix_quantize(np.ascontiguousarray(ch[rows]), 2, -8, 1)
    assert np.array_equal(to_host(oc)[rows], rc) and np.array_equal(to_host(osh)[rows], rs)


def test_vit_mlp_chain_sampled(mix, orc):
    """M = 16384 patch tokens, A-MiX-4.25b x W-MXINT4: fc1 1280 -> 5120 with the
    fused MiX-4.25b epilogue feeding fc2 5120 -> 1280 directly."""
    import torch
    M, D, H = 16384, 1280, 5120
    x = synth.to_bf16_bits(synth.vlm_activations(2, 0, M, D, visual_rows=M, outlier_frac=0.02,
                                                 outlier_scale=20.0))
    w1 = synth.to_bf16_bits(synth.gaussian_weights(2, 1, D, H))
    w2 = synth.to_bf16_bits(synth.gaussian_weights(2, 2, H, D))
    ac_g, ash_g = mix.quantize_mix(to_dev(x), mix.MIX_T1_4P25)
    b1c, b1s = mix.quantize_mx(to_dev(w1), 0, mix.MX_INT4)
    b2c, b2s = mix.quantize_mx(to_dev(w2), 0, mix.MX_INT4)
    c1 = torch.empty((M, H), dtype=torch.float32, device="cuda")
    hc = torch.empty((M, H // 2), dtype=torch.uint8, device="cuda")
    hs = torch.empty((M, H // 32), dtype=torch.uint8, device="cuda")
    mix.gemm(mix.gemm_desc(M, H, D, ac_g, ash_g, 1, -8, b1c, b1s, 0, c=c1, epi=1, out_codes=hc, out_shared=hs,
                           algo=mix.MIX_GEMM_TCGEN05))
    c2 = torch.empty((M, D), dtype=torch.float32, device="cuda")
    mix.gemm(mix.gemm_desc(M, D, H, hc, hs, 1, -8, b2c, b2s, 0, c=c2, algo=mix.MIX_GEMM_TCGEN05))
    torch.cuda.synchronize()
    rng = np.random.default_rng(4)
    rows = np.sort(rng.choice(M, 64, replace=False))
    ac, ash = to_host(ac_g), to_host(ash_g)
    c1h = to_host(c1)
    assert sampled_check(orc, c1h, ac, ash, 1, to_host(b1c), to_host(b1s), 0, rows,
                         np.sort(rng.choice(H, 256, replace=False))) <= GEMM_REL_TOL
    rc, rs = orc.mix_quantize(np.ascontiguousarray(c1h[rows]), 1, -8, 1)
    assert np.array_equal(to_host(hc)[rows], rc) and np.array_equal(to_host(hs)[rows], rs)
    assert sampled_check(orc, to_host(c2), to_host(hc), to_host(hs), 1, to_host(b2c), to_host(b2s), 0, rows,
                         np.sort(rng.choice(D, 256, replace=False))) <= GEMM_REL_TOL


def split_schedule(M, N, K, sms):
    """The staged kernel's schedule rule, restated: 128 x 224 tiles; when the
    last wave is partial and cutting it along K shortens it by more than
    about four k-steps, its R tiles' k-steps are shared out over all SMs."""
    mt, nt, kt = -(-M // 128), -(-N // 224), -(-K // 128)
    tiles = mt * nt
    nd, R = divmod(tiles, sms)
    split = kt >= 64 and R > 0 and R * kt >= 2 * sms and R * kt + 4 * sms <= kt * sms
    return split, mt, nd * sms


@pytest.mark.parametrize("M,N,K,at,bt", [(1000, 2208, 8192, 2, 1), (1536, 3136, 8192, 1, 0),
                                         (4096, 3584, 8192, 2, 1)])
def test_staged_split_last_wave(mix, orc, M, N, K, at, bt):
    """Tiles of a partial last wave cut along K across every SM: the CTA that
    holds a tile's first k-steps adds the later parts' fp32 sums in k order
    before its epilogue.  Shapes: fewer tiles than SMs with ragged edges (two
    parts a tile), 20 tiles past a full wave (seven or eight parts a tile),
    and 68 past three waves (two or three parts; the 18944-deep down
    projection of the full-size test is cut the same way).  Whole rows of C (every column,
    cut tiles and whole ones) match the oracle on rows sampled mostly from
    the cut tiles; the fused MiX epilogue is bit-exact given C; two calls
    agree bit for bit."""
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    split, mt, first = split_schedule(M, N, K, sms)
    if sms == 148:
        assert split  # the shapes are chosen to be cut on this part
    ac, ash, bc, bs = operands(orc, 77 + M + N, M, N, K, at, bt)
    outs = [run_tc(mix, ac, ash, at, bc, bs, bt, M, N, K, epi=2, algo="staged") for _ in range(2)]
    assert np.array_equal(outs[0][0].view(np.uint32), outs[1][0].view(np.uint32))
    assert np.array_equal(outs[0][1], outs[1][1]) and np.array_equal(outs[0][2], outs[1][2])
    c, oc, osh = outs[0]
    c = c[0]
    rng = np.random.default_rng(M + N + K)
    cut_rows = sorted({min(M - 1, 128 * (t % mt) + int(r)) for t in range(first, mt * (-(-N // 224)))
                       for r in rng.choice(128, 2, replace=False)}) if split else []
    rows = np.array(sorted(set(cut_rows[:48]) | set(rng.choice(M, 16, replace=False).tolist())))
    ref = orc.gemm(ac[rows], ash[rows], at, -8, bc, bs, bt)
    assert row_rel_err(c[rows], ref) <= GEMM_REL_TOL
    rc, rs = orc.mix_quantize(np.ascontiguousarray(c[rows]), 2, -8, 1)
    assert np.array_equal(oc[0][rows], rc) and np.array_equal(osh[0][rows], rs)


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("N", [128, 256])
def test_tc_zero_blocks_causal(mix, orc, algo, N):
    """An A operand with all-zero 32-blocks and all-zero 128-deep tiles (a
    causal attention P: row m is zero past column m), a tile whose first
    k-step is zero but not its later ones, and an all-zero row tile: the
    stages whose A tile is all zero are skipped on the fused path, and the
    result still equals the oracle's."""
    M, K = 384, 1024
    rng = np.random.default_rng(5)
    a = rng.random((M, K)).astype(np.float32)
    a[np.arange(K)[None, :] > np.arange(M)[:, None] * 2] = 0.0      # causal-like: zero tiles to the right
    a[128:256, :128] = 0.0                                          # first k-step zero, later ones not
    a[256:384] = 0.0                                                # an all-zero row tile
    a[260, 700] = 0.5                                               # ... but one nonzero block in it
    w = synth.to_bf16_bits(synth.normal(9, 1, N * K, 0, 0.5).reshape(N, K))
    ac, ash = orc.mix_quantize(a, 2, -15)
    bc, bs = orc.mx_quantize(w, 1, 0)
    import torch
    c = torch.empty((1, M, N), dtype=torch.float32, device="cuda")
    d = mix.gemm_desc(M, N, K, to_dev(ac), to_dev(ash), 2, -15, to_dev(bc), to_dev(bs), 0, c=c,
                      algo=algo_id(mix, algo))
    mix.gemm(d)
    torch.cuda.synchronize()
    assert mix.mix_device_error() == 0
    ref = orc.gemm(ac, ash, 2, -15, bc, bs, 0)
    got = to_host(c)[0]
    assert row_rel_err(got, ref) <= GEMM_REL_TOL
    assert np.all(got[256:260] == 0) and np.all(got[261:] == 0)


@pytest.mark.parametrize("shift,M,K,batch,N", [(0, 384, 1024, 2, 128), (200, 300, 640, 1, 128),
                                               (-300, 520, 896, 2, 128), (0, 1000, 1024, 1, 256),
                                               (64, 300, 640, 3, 544)])
def test_tc_causal_bound(mix, orc, shift, M, K, batch, N):
    """A stated causal bound (a_causal): A is zero past column m + shift in
    every batch, and the fused-decode kernel skips the k-steps past each row
    tile's bound and takes the row tiles last first.  The result is the same
    bits as the same call without the bound, and the oracle's within the
    matmul tolerance.  A negative shift leaves whole row tiles zero (their
    loop keeps step 0), a positive one (more keys than queries) moves the
    bound right, M is ragged in three cases, the 256-column tile runs too,
    and N = 544 gives three column tiles, which the reordering walks with
    the row tiles and the batches."""
    import torch
    rng = np.random.default_rng(17 + M)
    a = rng.random((batch, M, K)).astype(np.float32)
    a[:, np.arange(K)[None, :] > np.arange(M)[:, None] + shift] = 0.0
    ac, ash = orc.mix_quantize(a.reshape(batch * M, K), 2, -15)
    w = synth.to_bf16_bits(synth.normal(18, 1, N * K, 0, 0.5).reshape(N, K))
    bc, bs = orc.mx_quantize(w, 1, 0)
    outs = []
    for causal in (0, 1):
        c = torch.empty((batch, M, N), dtype=torch.float32, device="cuda")
        d = mix.gemm_desc(M, N, K, to_dev(ac), to_dev(ash), 2, -15, to_dev(bc), to_dev(bs), 0, c=c, batch=batch,
                          b_group=batch, algo=mix.MIX_GEMM_TCGEN05_FUSED, a_causal=causal, a_causal_shift=shift)
        mix.gemm(d)
        torch.cuda.synchronize()
        assert mix.mix_device_error() == 0
        outs.append(to_host(c))
    assert np.array_equal(outs[0], outs[1])
    for b in range(batch):
        ref = orc.gemm(ac[b * M:(b + 1) * M], ash[b * M:(b + 1) * M], 2, -15, bc, bs, 0)
        assert row_rel_err(outs[1][b], ref) <= GEMM_REL_TOL, b
    if shift < 0:
        assert np.all(outs[1][:, :-shift] == 0)


PREP_CASES = [(algo, bt, blk) for algo in ALGOS for bt, blk in ((1, 32), (0, 32), (0, 16), (1, 16))
              if not (algo == "fused" and bt == 1 and blk == 32)]   # MXFP4 on the fused path: read as it is


@pytest.mark.parametrize("algo,bt,b_block", PREP_CASES)
def test_prepared_b_equals_per_call(mix, orc, algo, bt, b_block):
    """B prepared once (mix_mx_gemm_prepare_b) gives the same bits as B
    prepared inside the call, with and without the fused epilogue, and a
    second call on the same prepared B gives them again."""
    import torch
    M, K = 200, 640
    N = 544 if algo == "staged" else 224
    a = synth.to_bf16_bits(synth.vlm_activations(50, 0, M, K, visual_rows=150))
    w = synth.to_bf16_bits(synth.normal(51, 1, K * N, 0, 0.02).reshape(K, N))
    ac, ash = orc.mix_quantize(a, 2)
    bc, bs = orc.mx_quantize(w, 0, bt, 0, block=b_block)
    outs = []
    for prep in (False, True, True):
        c = torch.empty((M, N), dtype=torch.float32, device="cuda")
        oc = torch.empty((M, N // 2), dtype=torch.uint8, device="cuda")
        osh = torch.empty((M, N // 32), dtype=torch.int16, device="cuda")
        d = mix.gemm_desc(M, N, K, to_dev(ac), to_dev(ash), 2, -8, to_dev(bc), to_dev(bs), bt, c=c, epi=2,
                          out_codes=oc, out_shared=osh, algo=algo_id(mix, algo), b_block=b_block)
        ws_plain = mix.mix_mx_gemm_workspace_bytes(d)
        if prep:
            assert mix.prepare_b(d) is not None
            assert mix.mix_mx_gemm_workspace_bytes(d) < ws_plain
        mix.gemm(d)
        torch.cuda.synchronize()
        assert mix.mix_device_error() == 0
        outs.append((to_host(c), to_host(oc), to_host(osh)))
    for o in outs[1:]:
        assert np.array_equal(o[0].view(np.uint32), outs[0][0].view(np.uint32))
        assert np.array_equal(o[1], outs[0][1]) and np.array_equal(o[2], outs[0][2])
    ref = orc.gemm(ac, ash, 2, -8, bc, bs, bt, b_block=b_block)
    assert row_rel_err(outs[0][0], ref) <= GEMM_REL_TOL


def test_prepare_b_not_taken(mix, orc):
    """MXFP4 weights on the fused-decode variant are read as they are: no
    prepared form (0 bytes) and prepare_b says so."""
    import ctypes
    import torch
    M, N, K = 128, 128, 256
    ac, ash, bc, bs = operands(orc, 52, M, N, K, 2, 1)
    c = torch.empty((M, N), dtype=torch.float32, device="cuda")
    d = mix.gemm_desc(M, N, K, to_dev(ac), to_dev(ash), 2, -8, to_dev(bc), to_dev(bs), 1, c=c,
                      algo=mix.MIX_GEMM_TCGEN05_FUSED)
    assert mix.mix_mx_gemm_prepare_b_bytes(d) == 0
    st = mix.lib.mix_mx_gemm_prepare_b(ctypes.byref(d), ctypes.c_void_p(c.data_ptr()), 1 << 20, None)
    assert st == mix.MIX_ERR_UNSUPPORTED
