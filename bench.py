"""Benchmark of the MiX hot path on one B300 (or N replicas).

One step runs every stage of the path once, at the paper-shaped sizes:
  * quantiser sweep: 4096 x 3584 bf16 activations -> MiX-4.25b and MiX-4.5b;
    3584 x 18944 bf16 weights -> MXINT4 and MXFP4 (down the columns, as stored);
  * Qwen2-VL-7B-shaped prefill linears (M = 4096): activations -> MiX-4.5b,
    QKV / O / gate+up / down as A-MiX-4.5b x W-MXFP4 with the fused MiX-4.5b
    output quantiser (the down projection's 18944-wide input is quantised too);
  * ViT MLP (M = 16384): activations -> MiX-4.25b, fc1 (fused MiX-4.25b
    output) feeding fc2 directly, A-MiX-4.25b x W-MXINT4;
  * GQA attention (28 / 4 heads, d 128), prefill 4096: K-smoothing (mean +
    subtraction), Q -> MiX-4.5b, K' -> MXINT4, S = Q K'^T (fp32), P (a fixed
    softmax output) -> MiX-4.5b, V -> MXINT4 along tokens, O = P V;
  * decode over an 8192-token MX cache: one fused call -- the new key
    smoothed with the frozen prefill mean and appended to the K' cache,
    q K'^T, the softmax, P -> MiX-4.5b, P V (one cooperative launch).
Weights (and their MMA-ready form) and caches are made once at set-up;
everything above is timed.

value = 100 * (sum over the step's launches of max(bytes / HBM peak, flops /
tensor peak)) / measured step time, i.e. the step's throughput as a percentage
of the B300 roofline; absolute GB/s and TOPS of every call are in "parts".
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import re
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MiX quantize GB/s + MiX×MX GEMM eff. TOPS, % of B300 roofline"
UNIT = "% of B300 roofline"
WORKLOAD = "qwen2vl7b_vit_attention_hot_path"


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d["bf16_tflops_sustained"], "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


PEAKS = load_peaks()
# kind::mxf8f6f4 (FP8-rate) dense peak: the measured bf16 peak x the nominal
# 2x fp8/bf16 ratio.  A call timed on its own (a fraction of a millisecond,
# at full clock) is graded against the burst figure; the sustained one was
# measured seconds into a loop at the power cap's lower clock, and applies
# only to a run whose own clock record shows that cap pulling the clock down.
MX8_TFLOPS_BURST = PEAKS["bf16_tflops"] * 2.0
MX8_TFLOPS_SUSTAINED = PEAKS["bf16_tflops_sustained"] * 2.0
MX8_TFLOPS = MX8_TFLOPS_BURST
HBM = PEAKS["hbm_gbs"]


def step_mma_peak(clk):
    """The MMA peak that matches the step's timed run: burst unless the SM
    clock sampled during it had a median below 90 % of its maximum (the
    power cap at work), then sustained."""
    sm, mx = clk.get("sm_mhz"), clk.get("sm_max_mhz")
    if sm and mx and sm < 0.9 * mx:
        return MX8_TFLOPS_SUSTAINED, f"sustained (median SM clock {sm:.0f} of {mx:.0f} MHz)"
    return MX8_TFLOPS_BURST, (f"burst (median SM clock {sm:.0f} of {mx:.0f} MHz)" if sm and mx
                              else "burst (no clock record)")


EXT_INPUTS = {}   # step tensors the extension measurements reuse
CLAMP = {}        # what the clamped-block report reads (filled by build_workload)


def with_prepared(d, src):
    """d with the prepared B of the descriptor src (same B and shapes)."""
    d.b_prepared = src.b_prepared
    return d


def clamp_report(torch, mix, ws):
    """Clamped MiX blocks of every MiX quantisation in the step, at its ebias:
    [blocks clamped down (exponent above ebias + 15), blocks clamped up
    (nonzero, below ebias), blocks].  The matmul epilogues are counted on
    their fp32 C, made once here by the same matmul with an fp32 output
    (outside the timed region)."""
    out = {}
    for name, x, eb in CLAMP["inputs"]:
        n = mix.clamp_count(x, eb)
        out[name] = [int(v) for v in n.tolist()] + [x.shape[0] * (x.shape[1] // 32)]
    big = max(m * n for _, _, m, n, _ in CLAMP["epi"])
    cbuf = torch.empty(big, dtype=torch.float32, device=ws.device)
    for name, make, m, n, eb in CLAMP["epi"]:
        c = cbuf[:m * n].view(m, n)
        d = make(c)
        mix.mix_mx_gemm(d, ws)
        cnt = mix.clamp_count(c, eb)
        out[name + ":epilogue"] = [int(v) for v in cnt.tolist()] + [m * (n // 32)]
    del cbuf
    torch.cuda.synchronize()
    return out


class Call:
    """One library call of the step with its algorithmic bytes and flops."""

    def __init__(self, name, fn, nbytes, flops=0.0, launches=1, kind="hbm"):
        self.name, self.fn, self.bytes, self.flops, self.launches, self.kind = name, fn, nbytes, flops, launches, kind

    def roof_s(self, mma_tflops=None):
        t_mem = self.bytes / (HBM * 1e9)
        t_mma = self.flops / ((mma_tflops or MX8_TFLOPS) * 1e12) if self.flops else 0.0
        return max(t_mem, t_mma)


def mix_bytes(rows, k, t, in_bytes=2):
    return rows * k * in_bytes + rows * k // 2 + rows * (k // 32) * (1 if t == 1 else 2)


def mx_bytes(n, k, in_bytes=2):
    return n * k * in_bytes + n * k // 2 + n * (k // 32)


def plane_bytes(rows, k, t):
    """Packed MiX planes (t = 1 / 2) or MX planes (t = 0)."""
    return rows * k // 2 + rows * (k // 32) * (2 if t == 2 else 1)


# ---------------------------------------------------------------------------
# The step: every call with its algorithmic bytes and flops (shapes only)
# ---------------------------------------------------------------------------

def dims(small=False):
    """Sizes of the step; small = a divisor of the token counts (True means 8)."""
    s = (8 if small is True else int(small)) if small else 1
    return dict(M=4096 // s, DM=3584, DF=18944, QKV=4608, MV=16384 // s, T=4096 // s, TC=8192 // s,
                HQ=28, HK=4, D=128)


def tc_launches(n, b_in_place=False, prepared=False):
    """Launches of one tensor-core matmul call: outputs wider than one 256-column
    tile take the staged variant (expand A, expand B or its scales unless B was
    prepared once, matmul); narrower ones the fused-decode variant (expand B
    unless it is MXFP4 read in place or prepared, matmul)."""
    if n > 256:
        return 2 if prepared else 3
    return 1 if (b_in_place or prepared) else 2


def step_table(small=False):
    """[(name, bytes, flops, launches, cpu work)] in launch order.  The cpu work
    (kind, count) lets the CPU baseline extrapolate the oracle's sampled cost:
    elements for quantisers and smoothing, outputs x 32-blocks for matmuls."""
    g = dims(small)
    M, DM, DF, QKV, MV, T, TC, HQ, HK, D = (g[k] for k in ("M", "DM", "DF", "QKV", "MV", "T", "TC", "HQ", "HK", "D"))
    rows = []

    def add(name, nbytes, flops=0.0, launches=1, cpu=None):
        rows.append((name, float(nbytes), float(flops), launches, cpu))

    add(f"mix_quantize_t1_{M}x{DM}", mix_bytes(M, DM, 1), cpu=("mix1", M * DM))
    add(f"mix_quantize_t2_{M}x{DM}", mix_bytes(M, DM, 2), cpu=("mix2", M * DM))
    add(f"mx_quantize_int4_{DM}x{DF}", mx_bytes(DF, DM), cpu=("mx", DF * DM))
    add(f"mx_quantize_fp4_{DM}x{DF}", mx_bytes(DF, DM), cpu=("mx", DF * DM))
    add(f"mix_quantize_t2_{M}x{DF}", mix_bytes(M, DF, 2), cpu=("mix2", M * DF))
    for name, k, n in (("qkv", DM, QKV), ("o", DM, DM), ("gate_up", DM, 2 * DF), ("down", DF, DM)):
        add(f"gemm_{name}_{M}x{k}x{n}", plane_bytes(M, k, 2) + plane_bytes(n, k, 0) + plane_bytes(M, n, 2),
            2.0 * M * n * k, launches=tc_launches(n, prepared=True), cpu=("gemm", M * n * (k // 32)))
    add(f"mix_quantize_t1_{MV}x1280", mix_bytes(MV, 1280, 1), cpu=("mix1", MV * 1280))
    add(f"gemm_vit_fc1_{MV}x1280x5120", plane_bytes(MV, 1280, 1) + plane_bytes(5120, 1280, 0) +
        plane_bytes(MV, 5120, 1), 2.0 * MV * 5120 * 1280, launches=tc_launches(5120, prepared=True),
        cpu=("gemm", MV * 5120 * 40))
    add(f"gemm_vit_fc2_{MV}x5120x1280", plane_bytes(MV, 5120, 1) + plane_bytes(1280, 5120, 0) +
        plane_bytes(MV, 1280, 1), 2.0 * MV * 1280 * 5120, launches=tc_launches(1280, prepared=True),
        cpu=("gemm", MV * 1280 * 160))
    # one cooperative kernel (after a counter reset): the 4 MB of prefill keys
    # fit the one-pass path
    add(f"ksmooth_compute_{T}x{HK}x{D}", T * HK * D * (2 + 4) + HK * D * 4, launches=1,
        cpu=("ks", 2 * T * HK * D))   # K read once, K' (fp32) and the mean written once
    add(f"mix_quantize_t2_q_{T * HQ}x{D}", mix_bytes(T * HQ, D, 2), cpu=("mix2", T * HQ * D))
    add(f"mx_quantize_int4_kprime_{T * HK}x{D}", mx_bytes(T * HK, D, 4), cpu=("mx", T * HK * D))
    add(f"bmm_qk_{HQ}x{T}x{T}x{D}", plane_bytes(T * HQ, D, 2) + plane_bytes(T * HK, D, 0) + HQ * T * T * 4,
        2.0 * HQ * T * T * D, launches=tc_launches(T), cpu=("gemm", HQ * T * T * (D // 32)))
    add(f"mix_quantize_t2_p_{HQ * T}x{T}", mix_bytes(HQ * T, T, 2), cpu=("mix2", HQ * T * T))
    add(f"mx_quantize_int4_v_{T}x{HK * D}", mx_bytes(HK * D, T), cpu=("mx", HK * D * T))
    # P is causal and the call says so: the work is P's 32-blocks that hold an
    # unmasked entry (row r: blocks 0 .. r // 32; 16 code bytes and a 2-byte
    # shared field each) and the products below the mask
    pv_blocks = HQ * 32 * (T // 32) * (T // 32 + 1) // 2
    add(f"bmm_pv_{HQ}x{T}x{D}x{T}", pv_blocks * 18 + plane_bytes(HK * D, T, 0) + HQ * T * D * 4,
        2.0 * HQ * D * T * (T + 1) / 2, launches=tc_launches(D), cpu=("gemm", HQ * T * D * (T // 32)))
    # decode over the TC-token MX cache: one fused call (frozen-mean K append,
    # Q.K'^T, softmax, MiX requantisation of P, P.V; one cooperative kernel
    # after a counter reset)
    add(f"decode_attention_{HK}x7x{TC}x{D}", decode_attention_bytes(TC, HQ, HK, D), 2.0 * 2.0 * HQ * TC * D,
        launches=1, cpu=("gemm", HQ * TC * (D // 32) + HQ * D * (TC // 32)))
    return rows


def decode_attention_bytes(TC, HQ, HK, D):
    """The fused decode step's algorithmic bytes: the MXINT4 K' and V caches
    read once, q, the new key and the frozen mean read, the appended K' row
    and the output written."""
    kcache = TC * HK * (D // 2 + D // 32)
    vcache = HK * D * (TC // 2 + TC // 32)
    return kcache + vcache + HQ * D * 2 + HK * D * (2 + 4) + HK * (D // 2 + D // 32) + HQ * D * 4


MATMUL_SOURCES = ("gemm_tc.cu", "expand.cu", "decode.cuh", "mix_common.cuh", "tc_ptx.cuh")


def matmul_source_sha():
    """sha256 over the matmul's kernel sources with comments and blank space
    removed: a recorded DRAM-traffic figure counts only for the code it was
    measured on, and an edit of a comment does not change that code."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in MATMUL_SOURCES:
        with open(os.path.join(ROOT, "quantized_vlm_gemm_mix_b300", "csrc", f), encoding="utf-8") as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)   # block comments
        src = re.sub(r"//[^\n]*", " ", src)                  # line comments
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()


def _require(ok, what: str) -> None:
    """A check that holds under python -O too (unlike assert)."""
    if not ok:
        raise RuntimeError(what)


def roof_seconds(nbytes, flops, mma_tflops=None):
    return max(nbytes / (HBM * 1e9), flops / ((mma_tflops or MX8_TFLOPS) * 1e12) if flops else 0.0)


# ---------------------------------------------------------------------------
# Replicas (N > 1): every rank runs the whole step on its own GPU; the only
# exchanges are the barriers around the timed region and the max of the
# ranks' times.  No collective touches the data path.
# ---------------------------------------------------------------------------

def max_over_ranks(torch, dist, v, device):
    """The largest of the ranks' values v (every rank gets it); v itself with
    no process group."""
    if dist is None:
        return v
    t = torch.tensor([v], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(roof_s, world, ms_step):
    """Whole-job throughput as a percentage of ONE B300's roofline: the work
    of all `world` replicas (each one step's roofline time roof_s) over the
    slowest rank's time per step."""
    return 100.0 * roof_s * world / (ms_step * 1e-3)


# ---------------------------------------------------------------------------
# Workload
# ---------------------------------------------------------------------------

def build_workload(torch, mix, synth, dev, seed=0, small=False):
    """Inputs on the device, weights and caches quantised once, and one closure
    per call of the step.  Returns (calls, h2d pairs, d2h tensors, host arrays,
    tensors to keep alive)."""
    bf16 = torch.bfloat16
    T2, T1 = mix.MIX_T2_4P5, mix.MIX_T1_4P25
    FP4, INT4 = mix.MX_FP4_E2M1, mix.MX_INT4
    g = dims(small)
    M, DM, DF, QKV, MV, T, TC, HQ, HK, D = (g[k] for k in ("M", "DM", "DF", "QKV", "MV", "T", "TC", "HQ", "HK", "D"))
    fns, h2d, d2h, host, keep = {}, [], [], {}, []
    # MiX quantiser inputs (tensor, ebias) and the matmuls with a fused MiX
    # epilogue (a descriptor maker taking an fp32 C, its M x N, ebias), for
    # the clamped-block report
    CLAMP["inputs"], CLAMP["epi"] = [], []

    def dev_bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(bf16)

    def new(shape, dtype):
        t = torch.empty(shape, dtype=dtype, device=dev)
        keep.append(t)
        return t

    # one workspace serves every tensor-core matmul of the step (they run in
    # sequence on one stream); sized by the largest request
    tc_descs = []

    def tc_call(d):
        tc_descs.append(d)
        return lambda: mix.mix_mx_gemm(d, ws_tc[0])

    # weights are fixed: their MMA-ready form (scale words regrouped, MXINT4
    # expanded to e4m3) is made once here, when they are quantised
    def weight_call(d):
        buf = mix.prepare_b(d)
        if buf is not None:
            keep.append(buf)
        return tc_call(d)

    ws_tc = [None]

    # ----- per-step activations
    x_np = synth.to_bf16_bits(synth.vlm_activations(seed, 1, M, DM, visual_rows=(3 * M) // 4))
    xd_np = synth.to_bf16_bits(synth.vlm_activations(seed, 2, M, DF, visual_rows=(3 * M) // 4))
    xv_np = synth.to_bf16_bits(synth.vlm_activations(seed, 3, MV, 1280, visual_rows=MV, outlier_frac=0.02,
                                                     outlier_scale=20.0))
    host.update(x=x_np, xd=xd_np, xv=xv_np)
    x, xd, xv = dev_bf16(x_np), dev_bf16(xd_np), dev_bf16(xv_np)
    h2d += [(x, x_np), (xd, xd_np), (xv, xv_np)]

    # ----- resident weights, quantised at set-up (down the columns, as stored)
    def weight(tid, k, n):
        return dev_bf16(synth.to_bf16_bits(synth.gaussian_weights(seed, tid, k, n)))

    w_gu = weight(30, DM, 2 * DF)        # gate+up 3584 x 37888; its first 18944 columns are the sweep weight
    keep.append(w_gu)
    EXT_INPUTS.update(w_gu=w_gu, xd=xd, x=x, g=g)
    wq = {"gate_up": mix.quantize_mx(w_gu, 0, FP4)}
    for name, tid, k, n in (("qkv", 31, DM, QKV), ("o", 32, DM, DM), ("down", 33, DF, DM)):
        w = weight(tid, k, n)
        wq[name] = mix.quantize_mx(w, 0, FP4)
        del w
    w1, w2 = weight(34, 1280, 5120), weight(35, 5120, 1280)
    wv1, wv2 = mix.quantize_mx(w1, 0, INT4), mix.quantize_mx(w2, 0, INT4)
    del w1, w2
    keep += [wq, wv1, wv2]

    # ----- 1. quantiser sweep
    a1c, a1s = new((M, DM // 2), torch.uint8), new((M, DM // 32), torch.uint8)
    a2c, a2s = new((M, DM // 2), torch.uint8), new((M, DM // 32), torch.int16)
    wic, wis = new((DF, DM // 2), torch.uint8), new((DF, DM // 32), torch.uint8)
    wfc, wfs = new((DF, DM // 2), torch.uint8), new((DF, DM // 32), torch.uint8)
    fns[f"mix_quantize_t1_{M}x{DM}"] = lambda: mix.mix_quantize(x, M, DM, DM, T1, -8, 1, a1c, a1s)
    fns[f"mix_quantize_t2_{M}x{DM}"] = lambda: mix.mix_quantize(x, M, DM, DM, T2, -8, 1, a2c, a2s)
    fns[f"mx_quantize_int4_{DM}x{DF}"] = lambda: mix.mx_quantize(w_gu, DM, DF, 2 * DF, 0, INT4, 0, wic, wis)
    fns[f"mx_quantize_fp4_{DM}x{DF}"] = lambda: mix.mx_quantize(w_gu, DM, DF, 2 * DF, 0, FP4, 0, wfc, wfs)

    # ----- 2. prefill linears: A = the MiX-4.5b activations; epilogue-only outputs
    adc, ads = new((M, DF // 2), torch.uint8), new((M, DF // 32), torch.int16)
    fns[f"mix_quantize_t2_{M}x{DF}"] = lambda: mix.mix_quantize(xd, M, DF, DF, T2, -8, 1, adc, ads)
    outs = {}
    for name, k, n, (ac_, as_) in (("qkv", DM, QKV, (a2c, a2s)), ("o", DM, DM, (a2c, a2s)),
                                   ("gate_up", DM, 2 * DF, (a2c, a2s)), ("down", DF, DM, (adc, ads))):
        oc, os_ = new((M, n // 2), torch.uint8), new((M, n // 32), torch.int16)
        outs[name] = oc
        bc, bs = wq[name]
        d = mix.gemm_desc(M, n, k, ac_, as_, T2, -8, bc, bs, FP4, c=None, epi=mix.MIX_EPI_MIX_T2, out_codes=oc,
                          out_shared=os_, algo=mix.MIX_GEMM_TCGEN05)
        fns[f"gemm_{name}_{M}x{k}x{n}"] = weight_call(d)
        CLAMP["epi"].append((f"gemm_{name}_{M}x{k}x{n}", (lambda c, k=k, n=n, ac_=ac_, as_=as_, bc=bc, bs=bs, d=d:
                             with_prepared(mix.gemm_desc(M, n, k, ac_, as_, T2, -8, bc, bs, FP4, c=c,
                                                         algo=mix.MIX_GEMM_TCGEN05), d)), M, n, -8))
    d2h.append(outs["down"])

    # ----- 3. ViT MLP: fc1's fused MiX-4.25b output is fc2's input
    vc, vs = new((MV, 640), torch.uint8), new((MV, 40), torch.uint8)
    hc, hs = new((MV, 2560), torch.uint8), new((MV, 160), torch.uint8)
    yc, ys = new((MV, 640), torch.uint8), new((MV, 40), torch.uint8)
    fns[f"mix_quantize_t1_{MV}x1280"] = lambda: mix.mix_quantize(xv, MV, 1280, 1280, T1, -8, 1, vc, vs)
    d1 = mix.gemm_desc(MV, 5120, 1280, vc, vs, T1, -8, wv1[0], wv1[1], INT4, epi=mix.MIX_EPI_MIX_T1, out_codes=hc,
                       out_shared=hs, algo=mix.MIX_GEMM_TCGEN05)
    d2 = mix.gemm_desc(MV, 1280, 5120, hc, hs, T1, -8, wv2[0], wv2[1], INT4, epi=mix.MIX_EPI_MIX_T1, out_codes=yc,
                       out_shared=ys, algo=mix.MIX_GEMM_TCGEN05)
    fns[f"gemm_vit_fc1_{MV}x1280x5120"] = weight_call(d1)
    fns[f"gemm_vit_fc2_{MV}x5120x1280"] = weight_call(d2)
    CLAMP["epi"].append((f"gemm_vit_fc1_{MV}x1280x5120", lambda c: with_prepared(mix.gemm_desc(
        MV, 5120, 1280, vc, vs, T1, -8, wv1[0], wv1[1], INT4, c=c, algo=mix.MIX_GEMM_TCGEN05), d1), MV, 5120, -8))
    CLAMP["epi"].append((f"gemm_vit_fc2_{MV}x5120x1280", lambda c: with_prepared(mix.gemm_desc(
        MV, 1280, 5120, hc, hs, T1, -8, wv2[0], wv2[1], INT4, c=c, algo=mix.MIX_GEMM_TCGEN05), d2), MV, 1280, -8))
    CLAMP["inputs"] += [(f"mix_quantize_t1_{M}x{DM}", x, -8), (f"mix_quantize_t2_{M}x{DF}", xd, -8),
                        (f"mix_quantize_t1_{MV}x1280", xv, -8)]
    d2h.append(yc)

    # ----- 4. attention prefill (28 query / 4 KV heads, d 128)
    q_np, k_np, v_np = synth.attention_qkv(seed, TC, HQ, HK, D)
    qb = np.ascontiguousarray(synth.to_bf16_bits(q_np[:T]).reshape(T, HQ * D))
    kb = synth.to_bf16_bits(k_np).reshape(TC, HK * D)
    vb = synth.to_bf16_bits(v_np).reshape(TC, HK * D)
    q_last = synth.to_bf16_bits(q_np[TC - 1]).reshape(HQ, D)
    del q_np, k_np, v_np
    host.update(q=qb, k=kb, v=vb)
    q_d, k_d, v_d = dev_bf16(qb), dev_bf16(kb), dev_bf16(vb)
    h2d += [(q_d, qb), (k_d, kb), (v_d, vb)]
    k_pre = k_d[:T]
    mean = new((HK, D), torch.float32)
    kprime = new((T, HK, D), torch.float32)
    ws_k = new(mix.ksmooth_workspace_bytes(T, HK, D), torch.uint8)
    fns[f"ksmooth_compute_{T}x{HK}x{D}"] = lambda: mix.ksmooth_kv(k_pre, T, HK, D, HK * D, mean,
                                                                  mix.KSMOOTH_COMPUTE, kprime, ws_k)
    qc, qs = new((T * HQ, 64), torch.uint8), new((T * HQ, 4), torch.int16)         # rows (token, head)
    fns[f"mix_quantize_t2_q_{T * HQ}x{D}"] = lambda: mix.mix_quantize(q_d, T * HQ, D, D, T2, -8, 1, qc, qs)
    kc, ks = new((T * HK, 64), torch.uint8), new((T * HK, 4), torch.uint8)         # rows (token, head)
    fns[f"mx_quantize_int4_kprime_{T * HK}x{D}"] = lambda: mix.mx_quantize(kprime, T * HK, D, D, 1, INT4, 0, kc, ks)
    S = new((HQ, T, T), torch.float32)
    dqk = mix.gemm_desc(T, T, D, qc, qs, T2, -8, kc, ks, INT4, c=S, batch=HQ, b_group=HQ // HK, a_ld=HQ * D,
                        a_batch_stride=D, b_ld=HK * D, b_batch_stride=D, algo=mix.MIX_GEMM_TCGEN05)
    fns[f"bmm_qk_{HQ}x{T}x{T}x{D}"] = tc_call(dqk)
    ws_tc[0] = new(max(16, max(mix.mix_mx_gemm_workspace_bytes(d) for d in tc_descs)), torch.uint8)
    CLAMP["ws"] = ws_tc[0]
    # P: a fixed causal softmax of S, made once here (softmax is not on the path)
    for f in (f"ksmooth_compute_{T}x{HK}x{D}", f"mix_quantize_t2_q_{T * HQ}x{D}",
              f"mx_quantize_int4_kprime_{T * HK}x{D}", f"bmm_qk_{HQ}x{T}x{T}x{D}"):
        fns[f]()
    P = new((HQ, T, T), bf16)
    causal = torch.ones((T, T), dtype=torch.bool, device=dev).tril()
    for h in range(HQ):
        P[h] = torch.softmax((S[h] / math.sqrt(D)).masked_fill(~causal, float("-inf")), dim=-1).to(bf16)
    del causal
    CLAMP["inputs"] += [(f"mix_quantize_t2_q_{T * HQ}x{D}", q_d.view(T * HQ, D), -8),
                        (f"mix_quantize_t2_p_{HQ * T}x{T}", P.view(HQ * T, T), -15)]
    pc, ps = new((HQ * T, T // 2), torch.uint8), new((HQ * T, T // 32), torch.int16)
    fns[f"mix_quantize_t2_p_{HQ * T}x{T}"] = lambda: mix.mix_quantize(P, HQ * T, T, T, T2, -15, 1, pc, ps)
    # V [T, HK*D] quantised down its columns in one call: column h*D + d is
    # row (h, d) of the [HK][D][T/2] planes the PV matmul reads
    vqc, vqs = new((HK, D, T // 2), torch.uint8), new((HK, D, T // 32), torch.uint8)
    v_pre = v_d[:T]
    fns[f"mx_quantize_int4_v_{T}x{HK * D}"] = lambda: mix.mx_quantize(v_pre, T, HK * D, HK * D, 0, INT4, 0, vqc, vqs)
    O = new((HQ, T, D), torch.float32)
    # P is causal: the call states it, and the matmul skips the masked k-steps
    dpv = mix.gemm_desc(T, D, T, pc, ps, T2, -15, vqc, vqs, INT4, c=O, batch=HQ, b_group=HQ // HK,
                        algo=mix.MIX_GEMM_TCGEN05, a_causal=1)
    _require(mix.mix_mx_gemm_workspace_bytes(dpv) <= ws_tc[0].numel(), "P.V workspace exceeds the shared staging buffer")
    fns[f"bmm_pv_{HQ}x{T}x{D}x{T}"] = tc_call(dpv)
    d2h.append(O)

    # ----- 5. decode over a TC-token cache smoothed with the frozen prefill mean
    mean_f = new((HK, D), torch.float32)
    mean_f.copy_(mean)
    kp_all = new((TC, HK, D), torch.float32)
    mix.ksmooth_kv(k_d, TC, HK, D, HK * D, mean_f, mix.KSMOOTH_APPLY_FROZEN, kp_all)
    kcc, kcs = new((TC * HK, 64), torch.uint8), new((TC * HK, 4), torch.uint8)
    mix.mx_quantize(kp_all, TC * HK, D, D, 1, INT4, 0, kcc, kcs)
    vcc, vcs = new((HK, D, TC // 2), torch.uint8), new((HK, D, TC // 32), torch.uint8)
    for h in range(HK):
        mix.mx_quantize(v_d[:, h * D:(h + 1) * D], TC, D, HK * D, 0, INT4, 0, vcc[h], vcs[h])
    q_new = dev_bf16(q_last)
    keep.append(q_new)
    k_new = k_d[TC - 1:TC]
    dec_out = new((HQ, D), torch.float32)
    pdc, pds = new((HQ, TC // 2), torch.uint8), new((HQ, TC // 32), torch.int16)
    p_val = new((HQ, TC), torch.float32)
    dda = mix.decode_attention_desc(q_new, kcc.view(TC, HK, 64), kcs.view(TC, HK, 4), vcc, vcs, TC,
                                    1.0 / math.sqrt(D), dec_out, k_new=k_new[0], k_mean=mean_f)
    ws_dec = new(mix.lib.mix_decode_attention_workspace_bytes(ctypes.byref(dda)), torch.uint8)
    fns[f"decode_attention_{HK}x7x{TC}x{D}"] = lambda: mix.decode_attention(dda, ws_dec)
    d2h.append(dec_out)
    # once at set-up: the same step with its P kept, for the clamp report and
    # for the unfused shift-add matmuls timed beside the step
    ddp = mix.decode_attention_desc(q_new, kcc.view(TC, HK, 64), kcs.view(TC, HK, 4), vcc, vcs, TC,
                                    1.0 / math.sqrt(D), dec_out, k_new=k_new[0], k_mean=mean_f, p_codes=pdc,
                                    p_shared=pds, p_values=p_val)
    mix.decode_attention(ddp, ws_dec)
    qdc, qds = mix.quantize_mix(q_new, T2)
    keep += [qdc, qds]
    CLAMP["inputs"] += [(f"decode_q_{HQ}x{D}", q_new, -8), (f"decode_p_{HQ}x{TC}", p_val, -15)]
    s_dec = new((HK, 7, TC), torch.float32)
    dd1 = mix.gemm_desc(7, TC, D, qdc, qds, T2, -8, kcc, kcs, INT4, c=s_dec, batch=HK, b_ld=HK * D,
                        b_batch_stride=D, algo=mix.MIX_GEMM_SHIFTADD)
    o_dec = new((HK, 7, D), torch.float32)
    dd2 = mix.gemm_desc(7, D, TC, pdc, pds, T2, -15, vcc, vcs, INT4, c=o_dec, batch=HK, algo=mix.MIX_GEMM_SHIFTADD)
    EXT_INPUTS.update(gemv=dict(dd1=dd1, ws1=new(max(16, mix.mix_mx_gemm_workspace_bytes(dd1)), torch.uint8),
                                dd2=dd2, ws2=new(max(16, mix.mix_mx_gemm_workspace_bytes(dd2)), torch.uint8),
                                TC=TC, HQ=HQ, HK=HK, D=D,
                                dec=lambda: mix.decode_attention(dda, ws_dec)))

    calls = []
    for name, nbytes, flops, launches, _ in step_table(small):
        calls.append(Call(name, fns.pop(name), nbytes, flops, launches))
    _require(not fns, f"closures without a table entry: {list(fns)}")
    keep += [P, S, O, kprime, kp_all]
    return calls, h2d, d2h, host, keep


# ---------------------------------------------------------------------------
# Clocks
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0):
        self.index, self.rows, self.proc = index, [], None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([c.strip() for c in line.split(",")])

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm = [float(r[1]) for r in self.rows if len(r) >= 9 and r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if len(r) >= 9 and r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            if len(r) >= 9:
                for n, v in zip(names, r[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU baseline: the oracle, as it stands, on a bounded sample of the step
# ---------------------------------------------------------------------------

def oracle_unit_costs(budget_s=10.0, part=0):
    """Seconds per unit of work of the oracle (one host thread), measured on
    seeded samples of the step's tensors sized to take about budget_s: per
    element for the quantisers and smoothing, per output x 32-block for the
    matmul.  `part` picks the seed, so parallel workers time distinct samples."""
    import oracle as orc
    from quantized_vlm_gemm_mix_b300 import synth
    r = max(16, int(64 * math.sqrt(budget_s / 0.11)) // 16 * 16)
    x = synth.to_bf16_bits(synth.vlm_activations(part, 1, r, 3584, visual_rows=(3 * r) // 4))
    w = synth.to_bf16_bits(synth.gaussian_weights(part, 30, 3584, r))
    _, k_np, _ = synth.attention_qkv(part, 4 * r, 2, 4, 128)
    kb = synth.to_bf16_bits(k_np)
    cost = {}

    def timed(fn):
        t0 = time.perf_counter()
        out = fn()
        return time.perf_counter() - t0, out

    t, _ = timed(lambda: orc.mix_quantize(x, orc.T1))
    cost["mix1"] = t / x.size
    t, (ac, ash) = timed(lambda: orc.mix_quantize(x, orc.T2))
    cost["mix2"] = t / x.size
    t, (bc, bs) = timed(lambda: orc.mx_quantize(w, 0, orc.MXFP4))
    cost["mx"] = t / w.size
    t, _ = timed(lambda: orc.ksmooth_mean(kb))
    cost["ks"] = t / kb.size
    rr = max(1, r // 4)
    t, _ = timed(lambda: orc.gemm(ac[:rr], ash[:rr], orc.T2, -8, bc, bs, orc.MXFP4))
    cost["gemm"] = t / (rr * bc.shape[0] * (3584 // 32))
    sample = (f"oracle on {r} x 3584 activations (MiX T1, T2), 3584 x {r} weights (MXFP4), "
              f"{4 * r} x 4 x 128 keys (mean), {rr} x {r} outputs of K 3584 (Eq. (6) matmul); "
              f"per-unit costs extrapolated to every call of one full step")
    return cost, sample


def _oracle_worker(task):
    """One process of the parallel leg: the unmodified one-thread oracle on
    its own seeded sample."""
    part, budget_s = task
    sys.path.insert(0, ROOT)
    return oracle_unit_costs(budget_s, part)


def oracle_unit_costs_parallel(budget_s, procs):
    """The oracle as it stands, run in `procs` spawned processes at once (one
    per host core, each on its own seeded sample of the same shapes); the
    host's aggregate rate, as seconds per unit of work for the whole host."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    with ctx.Pool(procs) as pool:
        res = pool.map(_oracle_worker, [(i + 1, budget_s) for i in range(procs)])
    cost = {k: 1.0 / sum(1.0 / c[k] for c, _ in res) for k in res[0][0]}
    sample = (f"{procs} processes at once, each: " + res[0][1]).replace("; per-unit costs", "; aggregate per-unit costs")
    return cost, sample


def host_cpu():
    """The host's CPU model and logical core count, for the CPU-baseline record."""
    model = None
    try:
        with open("/proc/cpuinfo", encoding="utf-8") as f:
            for line in f:
                if line.startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    return {"cpu_model": model, "host_logical_cpus": os.cpu_count()}


def cpu_step_seconds(cost, small=False):
    return sum(cost[c[0]] * c[1] for *_, c in step_table(small))


def run_reference(args, rank, world):
    """--impl reference: the CPU oracle as it stands, on the host cores, each
    step a bounded sample of the workload extrapolated to the full step."""
    if rank != 0:
        return
    roof = sum(roof_seconds(b, f) for _, b, f, _, _ in step_table())
    est = []
    sample = ""
    budget = min(10.0, 150.0 / max(1, args.warmup + args.steps))   # whole run within a few minutes
    procs = max(1, os.cpu_count() or 1)
    for i in range(args.warmup + args.steps):
        cost, sample = oracle_unit_costs_parallel(budget, procs)
        if i >= args.warmup:
            est.append(cpu_step_seconds(cost))
    sec = float(np.mean(est))
    val = 100.0 * roof / sec
    out = {"impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": args.gpus,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64 / int64 (scalar C oracle)",
           "data": "synthetic (seeded)", "config": {"workload": WORKLOAD, "sample": sample},
           "cpu_baseline": {"value": val, "unit": UNIT, "cores": procs, "kind": "oracle", "sample": sample,
                            **host_cpu()},
           "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------

def measure_fp8_peak(local):
    """Dense FP8 e4m3 x e4m3 -> fp32 tensor rate on this GPU, measured the way
    the bf16 peak in MEASURED_PEAKS.json was: an 8192^3 cuBLASLt matmul, best
    of 10 (burst) and back to back for 4 s (sustained), with the SM clock
    sampled.  kind::mxf8f6f4 runs on the same FP8 tensor rate."""
    import torch
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    n = 8192
    g = torch.Generator(device=dev).manual_seed(0)
    a = torch.randn((n, n), device=dev, generator=g).to(torch.float8_e4m3fn)
    b = torch.randn((n, n), device=dev, generator=g).to(torch.float8_e4m3fn).t()
    one = torch.ones((), device=dev)

    def mm():
        return torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.float32)

    for _ in range(5):
        mm()
    torch.cuda.synchronize()
    flops = 2.0 * n ** 3
    best = float("inf")
    for _ in range(10):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        mm()
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    clocks = ClockSampler(local)
    clocks.start()
    reps, t_start = 0, time.time()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    while time.time() - t_start < 4.0:
        for _ in range(20):
            mm()
        reps += 20
        torch.cuda.synchronize()
    e1.record()
    torch.cuda.synchronize()
    ck = clocks.stop()
    line = {"what": "dense FP8 e4m3 tensor rate, cuBLASLt 8192^3, fp32 out",
            "fp8_tflops_burst": round(flops / (best * 1e-3) / 1e12, 1),
            "fp8_tflops_sustained": round(flops * reps / (e0.elapsed_time(e1) * 1e-3) / 1e12, 1),
            "bf16_tflops_measured": PEAKS["bf16_tflops"], "bf16_tflops_sustained_measured": PEAKS["bf16_tflops_sustained"],
            "clocks": ck}
    print(json.dumps(line))


def measure_extensions(torch, mix, stream, iters=10):
    """Kernels beyond the step (the tight MX exponent, the automatic ebias),
    timed like the step's calls: CUDA events on the launching stream around
    each launch, a spin kernel ahead of it, inputs larger than L2.  Each
    entry gives its algorithmic bytes and the fraction of measured HBM copy
    bandwidth reached."""
    g, w_gu, xd, x = EXT_INPUTS["g"], EXT_INPUTS["w_gu"], EXT_INPUTS["xd"], EXT_INPUTS["x"]
    M, DM, DF = g["M"], g["DM"], g["DF"]
    dev = xd.device
    FP4, INT4, T2 = mix.MX_FP4_E2M1, mix.MX_INT4, mix.MIX_T2_4P5
    # MiX-INT4g16: MiX-4.5b activations x MXINT4g16 weights, at the gate/up shape
    a2c, a2s = mix.quantize_mix(x, T2)
    g16c, g16s = mix.quantize_mx(w_gu, 0, INT4, mix.MX_BLOCK16)
    g32c, g32s = mix.quantize_mx(w_gu, 0, INT4)
    oc = torch.empty((M, DF), dtype=torch.uint8, device=dev)
    osh = torch.empty((M, 2 * DF // 32), dtype=torch.int16, device=dev)
    d16 = mix.gemm_desc(M, 2 * DF, DM, a2c, a2s, T2, -8, g16c, g16s, INT4, epi=mix.MIX_EPI_MIX_T2, out_codes=oc,
                        out_shared=osh, algo=mix.MIX_GEMM_TCGEN05, b_block=16)
    d32 = mix.gemm_desc(M, 2 * DF, DM, a2c, a2s, T2, -8, g32c, g32s, INT4, epi=mix.MIX_EPI_MIX_T2, out_codes=oc,
                        out_shared=osh, algo=mix.MIX_GEMM_TCGEN05)
    mix.prepare_b(d16)   # weights: prepared once, as in the step
    mix.prepare_b(d32)
    gws = torch.empty(max(mix.mix_mx_gemm_workspace_bytes(d16), mix.mix_mx_gemm_workspace_bytes(d32)),
                      dtype=torch.uint8, device=dev)
    g16_bytes = plane_bytes(M, DM, 2) + 2 * DF * DM // 2 + 2 * DF * DM // 16 + plane_bytes(M, 2 * DF, 2)
    g32_bytes = plane_bytes(M, DM, 2) + plane_bytes(2 * DF, DM, 0) + plane_bytes(M, 2 * DF, 2)
    gflops = 2.0 * M * 2 * DF * DM
    nvc = torch.empty((M, DM // 2), dtype=torch.uint8, device=dev)
    nvs = torch.empty((M, DM // 16), dtype=torch.uint8, device=dev)
    nvt = torch.empty((1,), dtype=torch.float32, device=dev)
    ufn = torch.empty((1,), dtype=torch.int64, device=dev)
    wc = torch.empty((DF, DM // 2), dtype=torch.uint8, device=dev)
    ws = torch.empty((DF, DM // 32), dtype=torch.uint8, device=dev)
    ac = torch.empty((M, DF // 2), dtype=torch.uint8, device=dev)
    ash = torch.empty((M, DF // 32), dtype=torch.int16, device=dev)
    eb = torch.empty((1,), dtype=torch.int32, device=dev)
    table = [
        (f"gemm_gate_up_mix_int4g16_{M}x{DM}x{2 * DF}", "MiX-4.5b x MXINT4g16 (staged; the g16 scales folded "
         "into the e4m3 expansion, prepared once)", g16_bytes, 2, lambda: mix.mix_mx_gemm(d16, gws), gflops),
        (f"gemm_gate_up_mix_int4_{M}x{DM}x{2 * DF}", "MiX-4.5b x MXINT4 (32-blocks), same call for comparison",
         g32_bytes, 2, lambda: mix.mix_mx_gemm(d32, gws), gflops),
        (f"mx_quantize_int4_g16_{DM}x{DF}", "MXINT4g16 weight quantiser (down the columns)",
         DF * DM * 2 + DF * DM // 2 + DF * DM // 16, 1,
         lambda: mix.mx_quantize(w_gu, DM, DF, 2 * DF, 0, INT4, mix.MX_BLOCK16, g16c, g16s)),
        (f"nvfp4_quantize_{M}x{DM}", "NVFP4 comparison quantiser (tensor amax pass, then 16-blocks; x read twice)",
         2 * M * DM * 2 + M * DM // 2 + M * DM // 16 + 4, 4,
         lambda: mix.nvfp4_quantize(x, M, DM, DM, nvc, nvs, nvt)),
        (f"mix_underflow_count_{M}x{DM}", "dead-zone count over the MiX-4.5b plane of x",
         M * DM * 2 + M * DM // 2 + 8, 2, lambda: mix.mix_underflow_count(x, M, DM, DM, a2c, mix.MIX_UF_MIX, ufn)),
        (f"mx_quantize_fp4_tight_{DM}x{DF}", "tight MX shared exponent", mx_bytes(DF, DM), 1,
         lambda: mix.mx_quantize(w_gu, DM, DF, 2 * DF, 0, FP4, mix.MX_SCALE_TIGHT, wc, ws)),
        (f"mx_quantize_fp4_ceil_{DM}x{DF}", "the ceil rule, same call (for comparison)", mx_bytes(DF, DM), 1,
         lambda: mix.mx_quantize(w_gu, DM, DF, 2 * DF, 0, FP4, 0, wc, ws)),
        (f"mix_auto_ebias_{M}x{DF}", "automatic ebias, pass 1 (clear, max-reduction, finish)", M * DF * 2 + 4, 3,
         lambda: mix.mix_auto_ebias(xd, M, DF, DF, eb)),
        (f"mix_quantize_auto_t2_{M}x{DF}", "automatic ebias + MiX-4.5b quantiser (x read twice)",
         mix_bytes(M, DF, 2) + M * DF * 2, 4,
         lambda: mix.mix_quantize_auto(xd, M, DF, DF, T2, 1, ac, ash, eb)),
    ]
    out = {}
    for row in table:
        name, what, nbytes, launches, fn = row[:5]
        flops = row[5] if len(row) > 5 else 0.0
        for _ in range(3):
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
        for a, b in ev:
            torch.cuda._sleep(400000)
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        ms = float(np.median([a.elapsed_time(b) for a, b in ev]))
        gbs = nbytes / (ms * 1e-3) / 1e9
        out[name] = {"what": what, "ms": round(ms, 5), "bytes": int(nbytes), "GB/s": round(gbs, 1),
                     "frac_hbm": round(gbs / HBM, 3), "launches": launches}
        if flops:
            tf = flops / (ms * 1e-3) / 1e12
            out[name].update({"TFLOP/s": round(tf, 1), "frac_mma": round(tf / MX8_TFLOPS, 3)})
    _require(mix.mix_device_error() == 0, "a kernel reported a timed-out wait")
    out.update(measure_unfused_decode(torch, mix, stream, iters))
    out["dead_zone"] = dead_zone_table(torch, mix, dev)
    return out


def decode_l2_states(torch, stream, iters, name, nbytes, fn):
    """The fused decode attention with its caches cold in L2 (a 256 MB buffer
    written before every launch) and warm (launched back to back, so the 4.5
    MB of caches stay in L2 from the previous call), each against HBM."""
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    res = {}
    for state in ("cold_l2", "warm_l2"):
        for _ in range(3):
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
        for a, b in ev:
            if state == "cold_l2":
                flush.zero_()
            torch.cuda._sleep(400000)
            if state == "warm_l2":
                fn()                                  # the caches the timed call reads, just read
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        ms = float(np.median([a.elapsed_time(b) for a, b in ev]))
        gbs = nbytes / (ms * 1e-3) / 1e9
        res[f"{name}_{state}"] = {"what": "the fused decode attention, one call, caches " +
                                  ("evicted from L2 first" if state == "cold_l2" else "resident in L2"),
                                  "ms": round(ms, 5), "bytes": int(nbytes), "GB/s": round(gbs, 1),
                                  "frac_hbm": round(gbs / HBM, 3), "launches": 1}
    del flush
    return res


def measure_unfused_decode(torch, mix, stream, iters):
    """The decode step's two matmuls on the integer shift-add path alone (the
    fused call of the step does the same arithmetic): S = q K'^T over the
    cache, and P V with the P planes the fused call produced at set-up."""
    e = EXT_INPUTS["gemv"]
    TC, HQ, HK, D = e["TC"], e["HQ"], e["HK"], e["D"]
    rows = [(f"gemv_qk_decode_{HK}x{HQ // HK}x{TC}x{D}", "S = q K'^T, shift-add (Eq. (6) literally), 1 launch",
             plane_bytes(HQ, D, 2) + plane_bytes(TC * HK, D, 0) + HQ * TC * 4, 2.0 * HQ * TC * D, 1,
             lambda: mix.mix_mx_gemm(e["dd1"], e["ws1"])),
            (f"gemv_pv_decode_{HK}x{HQ // HK}x{D}x{TC}", "O = P V, shift-add, split over K (2 launches)",
             plane_bytes(HQ, TC, 2) + plane_bytes(HK * D, TC, 0) + HQ * D * 4, 2.0 * HQ * D * TC, 2,
             lambda: mix.mix_mx_gemm(e["dd2"], e["ws2"]))]
    out = {}
    out.update(decode_l2_states(torch, stream, iters, f"decode_attention_{HK}x{HQ // HK}x{TC}x{D}",
                                decode_attention_bytes(TC, HQ, HK, D), e["dec"]))
    for name, what, nbytes, flops, launches, fn in rows:
        for _ in range(3):
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
        for a, b in ev:
            torch.cuda._sleep(400000)
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        ms = float(np.median([a.elapsed_time(b) for a, b in ev]))
        gbs = nbytes / (ms * 1e-3) / 1e9
        out[name] = {"what": what, "ms": round(ms, 5), "bytes": int(nbytes), "GB/s": round(gbs, 1),
                     "frac_hbm": round(gbs / HBM, 3), "TFLOP/s": round(flops / (ms * 1e-3) / 1e12, 2),
                     "launches": launches}
    return out


def dead_zone_table(torch, mix, dev, tokens=4096):
    """Fraction of nonzero key elements that each 4-bit format codes as zero,
    on the attention workload's synthetic keys (4 KV heads x 128, channel
    outliers), raw and smoothed with the frozen prefill mean: a synthetic
    analogue of the pages' key-underflow comparison."""
    from quantized_vlm_gemm_mix_b300 import synth
    q, k, v = synth.attention_qkv(0, tokens)
    res = {}
    for name, arr in (("K", k), ("K_smoothed", k - k[: tokens // 2].mean(axis=0, keepdims=True))):
        xb = synth.to_bf16_bits(arr.reshape(-1, 128))
        xd = torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)
        nz = int(np.count_nonzero(synth.bf16_bits_to_f32(xb)))
        planes = {"MiX-4.5b": (mix.quantize_mix(xd, mix.MIX_T2_4P5)[0], mix.MIX_UF_MIX),
                  "MXINT4": (mix.quantize_mx(xd, 1, mix.MX_INT4)[0], mix.MIX_UF_MXINT4),
                  "MXFP4": (mix.quantize_mx(xd, 1, mix.MX_FP4_E2M1)[0], mix.MIX_UF_E2M1),
                  "NVFP4": (mix.quantize_nvfp4(xd)[0], mix.MIX_UF_E2M1)}
        res[name] = {f: round(int(mix.underflow_count(xd, c, fmt).item()) / nz, 4) for f, (c, fmt) in planes.items()}
    return res


def single_call(args):
    """--call NAME: only that call of the step, its operands alone on the
    device (a few hundred MB), run warm-up + steps times with CUDA events
    around each launch; for profiler captures of one kernel and for quick
    timing.  Prints one JSON line with the median time."""
    import torch
    from quantized_vlm_gemm_mix_b300 import _build
    _build.build()
    from quantized_vlm_gemm_mix_b300 import mix, synth
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    g = dims()
    M, DM, DF, QKV, MV = g["M"], g["DM"], g["DF"], g["QKV"], g["MV"]
    T1, T2, FP4, INT4 = mix.MIX_T1_4P25, mix.MIX_T2_4P5, mix.MX_FP4_E2M1, mix.MX_INT4

    def bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    table = {r[0]: r for r in step_table()}
    name = args.call
    _require(name in table, f"--call takes one of: {', '.join(table)}")
    _, nbytes, flops, _, _ = table[name]
    gemms = {f"gemm_qkv_{M}x{DM}x{QKV}": (M, DM, QKV, 31, T2, FP4, 1), f"gemm_o_{M}x{DM}x{DM}": (M, DM, DM, 32, T2, FP4, 1),
             f"gemm_gate_up_{M}x{DM}x{2 * DF}": (M, DM, 2 * DF, 30, T2, FP4, 1),
             f"gemm_down_{M}x{DF}x{DM}": (M, DF, DM, 33, T2, FP4, 2),
             f"gemm_vit_fc1_{MV}x1280x5120": (MV, 1280, 5120, 34, T1, INT4, 3),
             f"gemm_vit_fc2_{MV}x5120x1280": (MV, 5120, 1280, 35, T1, INT4, 4)}
    if name in gemms:
        m, k, n, wid, at, bt, aid = gemms[name]
        x = bf16(synth.to_bf16_bits(synth.vlm_activations(0, aid, m, k, visual_rows=(3 * m) // 4 if m == M else m)))
        ac, ash = mix.quantize_mix(x, at)
        del x
        w = bf16(synth.to_bf16_bits(synth.gaussian_weights(0, wid, k, n)))
        bc, bs = mix.quantize_mx(w, 0, bt)
        del w
        oc = torch.empty((m, n // 2), dtype=torch.uint8, device=dev)
        os_ = torch.empty((m, n // 32), dtype=torch.uint8 if at == T1 else torch.int16, device=dev)
        d = mix.gemm_desc(m, n, k, ac, ash, at, -8, bc, bs, bt, epi=at, out_codes=oc, out_shared=os_,
                          algo=mix.MIX_GEMM_TCGEN05)
        mix.prepare_b(d)
        ws = torch.empty(max(16, mix.mix_mx_gemm_workspace_bytes(d)), dtype=torch.uint8, device=dev)
        fn = lambda: mix.mix_mx_gemm(d, ws)
    elif name.startswith("bmm_pv_"):
        # a causal softmax P (made by torch: the softmax is outside the
        # library) in MiX-4.5b at ebias -15, V in MXINT4 along tokens
        T, HQ, HK, D = g["T"], g["HQ"], g["HK"], g["D"]
        gen = torch.Generator(device=dev).manual_seed(0)
        P = torch.empty((HQ, T, T), dtype=torch.bfloat16, device=dev)
        causal = torch.ones((T, T), dtype=torch.bool, device=dev).tril()
        for h in range(HQ):
            sc = torch.randn((T, T), device=dev, generator=gen) * 3.0
            P[h] = torch.softmax((sc / math.sqrt(D)).masked_fill(~causal, float("-inf")), dim=-1).to(torch.bfloat16)
        del causal, sc
        pc = torch.empty((HQ * T, T // 2), dtype=torch.uint8, device=dev)
        ps = torch.empty((HQ * T, T // 32), dtype=torch.int16, device=dev)
        mix.mix_quantize(P, HQ * T, T, T, T2, -15, 1, pc, ps)
        del P
        _, _, v = synth.attention_qkv(0, T, HQ, HK, D)
        vb = bf16(synth.to_bf16_bits(v).reshape(T, HK * D))
        vqc = torch.empty((HK, D, T // 2), dtype=torch.uint8, device=dev)
        vqs = torch.empty((HK, D, T // 32), dtype=torch.uint8, device=dev)
        mix.mx_quantize(vb, T, HK * D, HK * D, 0, INT4, 0, vqc, vqs)
        O = torch.empty((HQ, T, D), dtype=torch.float32, device=dev)
        d = mix.gemm_desc(T, D, T, pc, ps, T2, -15, vqc, vqs, INT4, c=O, batch=HQ, b_group=HQ // HK,
                          algo=mix.MIX_GEMM_TCGEN05, a_causal=1)
        ws = torch.empty(max(16, mix.mix_mx_gemm_workspace_bytes(d)), dtype=torch.uint8, device=dev)
        fn = lambda: mix.mix_mx_gemm(d, ws)
    elif name.startswith("bmm_qk_"):
        # Q (MiX-4.5b, rows (token, head)) x K' (MXINT4 along head_dim), GQA,
        # both read in place with head strides; fp32 scores out
        T, HQ, HK, D = g["T"], g["HQ"], g["HK"], g["D"]
        q, k, _ = synth.attention_qkv(0, T, HQ, HK, D)
        qd = bf16(synth.to_bf16_bits(q).reshape(T, HQ * D))
        kd = bf16(synth.to_bf16_bits(k).reshape(T, HK * D))
        del q, k
        qc = torch.empty((T * HQ, D // 2), dtype=torch.uint8, device=dev)
        qs = torch.empty((T * HQ, D // 32), dtype=torch.int16, device=dev)
        mix.mix_quantize(qd, T * HQ, D, D, T2, -8, 1, qc, qs)
        kc = torch.empty((T * HK, D // 2), dtype=torch.uint8, device=dev)
        ks = torch.empty((T * HK, D // 32), dtype=torch.uint8, device=dev)
        mix.mx_quantize(kd.float(), T * HK, D, D, 1, INT4, 0, kc, ks)
        S = torch.empty((HQ, T, T), dtype=torch.float32, device=dev)
        d = mix.gemm_desc(T, T, D, qc, qs, T2, -8, kc, ks, INT4, c=S, batch=HQ, b_group=HQ // HK, a_ld=HQ * D,
                          a_batch_stride=D, b_ld=HK * D, b_batch_stride=D, algo=mix.MIX_GEMM_TCGEN05)
        ws = torch.empty(max(16, mix.mix_mx_gemm_workspace_bytes(d)), dtype=torch.uint8, device=dev)
        fn = lambda: mix.mix_mx_gemm(d, ws)
    elif name.startswith("ksmooth_compute_"):
        # the prefill keys of one layer: mean over the tokens and K' = K - mean
        T, HK, D = g["T"], g["HK"], g["D"]
        _, k, _ = synth.attention_qkv(0, T, g["HQ"], HK, D)
        kd = bf16(synth.to_bf16_bits(k).reshape(T, HK * D))
        del k
        mean = torch.empty((HK, D), dtype=torch.float32, device=dev)
        kout = torch.empty((T, HK, D), dtype=torch.float32, device=dev)
        ws = torch.empty(mix.ksmooth_workspace_bytes(T, HK, D), dtype=torch.uint8, device=dev)
        fn = lambda: mix.ksmooth_kv(kd, T, HK, D, HK * D, mean, mix.KSMOOTH_COMPUTE, kout, ws)
    elif name.startswith("decode_attention_"):
        # one decode step over the TC-token MX cache (K' smoothed with the mean
        # of its first half, the new key appended each call)
        TC, HQ, HK, D = g["TC"], g["HQ"], g["HK"], g["D"]
        q, k, v = synth.attention_qkv(0, TC, HQ, HK, D)
        kd = bf16(synth.to_bf16_bits(k).reshape(TC, HK * D))
        vd = bf16(synth.to_bf16_bits(v).reshape(TC, HK * D))
        qn = bf16(synth.to_bf16_bits(q[TC - 1]).reshape(HQ, D))
        del q, k, v
        mean = torch.empty((HK, D), dtype=torch.float32, device=dev)
        kp = torch.empty((TC, HK, D), dtype=torch.float32, device=dev)
        wsk = torch.empty(mix.ksmooth_workspace_bytes(TC // 2, HK, D), dtype=torch.uint8, device=dev)
        mix.ksmooth_kv(kd, TC // 2, HK, D, HK * D, mean, mix.KSMOOTH_COMPUTE, kp[:TC // 2], wsk)
        mix.ksmooth_kv(kd, TC, HK, D, HK * D, mean, mix.KSMOOTH_APPLY_FROZEN, kp)
        kc = torch.empty((TC * HK, 64), dtype=torch.uint8, device=dev)
        ks = torch.empty((TC * HK, 4), dtype=torch.uint8, device=dev)
        mix.mx_quantize(kp, TC * HK, D, D, 1, INT4, 0, kc, ks)
        vc = torch.empty((HK, D, TC // 2), dtype=torch.uint8, device=dev)
        vs = torch.empty((HK, D, TC // 32), dtype=torch.uint8, device=dev)
        for h in range(HK):
            mix.mx_quantize(vd[:, h * D:(h + 1) * D], TC, D, HK * D, 0, INT4, 0, vc[h], vs[h])
        out = torch.empty((HQ, D), dtype=torch.float32, device=dev)
        dd = mix.decode_attention_desc(qn, kc.view(TC, HK, 64), ks.view(TC, HK, 4), vc, vs, TC, 1.0 / math.sqrt(D),
                                       out, k_new=kd[TC - 1].view(HK, D), k_mean=mean)
        ws = torch.empty(mix.lib.mix_decode_attention_workspace_bytes(ctypes.byref(dd)), dtype=torch.uint8,
                         device=dev)
        fn = lambda: mix.decode_attention(dd, ws)
    elif re.fullmatch(r"mix_quantize_t[12]_\d+x\d+", name):
        # the activation quantisers (the sweep's, the MLP's and the ViT's)
        t = T1 if name.startswith("mix_quantize_t1") else T2
        rows, k = map(int, name.rsplit("_", 1)[1].split("x"))
        x = bf16(synth.to_bf16_bits(synth.vlm_activations(0, 1, rows, k, visual_rows=(3 * rows) // 4)))
        c = torch.empty((rows, k // 2), dtype=torch.uint8, device=dev)
        sh = torch.empty((rows, k // 32), dtype=torch.uint8 if t == T1 else torch.int16, device=dev)
        fn = lambda: mix.mix_quantize(x, rows, k, k, t, -8, 1, c, sh)
    else:
        raise SystemExit(f"--call supports the prefill matmuls, the attention Q.K'^T and P.V, K-smoothing, the "
                         f"decode attention and the MiX activation quantisers, not {name}")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)   # larger than L2
    times = []
    for i in range(args.warmup + args.steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(200000)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        if i >= args.warmup:
            times.append(a.elapsed_time(b))
    _require(mix.mix_device_error() == 0, "a kernel reported a timed-out wait")
    ms = float(np.median(times))
    out = {"call": name, "ms": round(ms, 5), "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1),
           "frac_hbm": round(nbytes / (ms * 1e-3) / 1e9 / HBM, 3), "steps": args.steps, "warmup": args.warmup,
           "l2": "256 MB buffer written before every launch"}
    if flops:
        out.update({"TFLOP/s": round(flops / (ms * 1e-3) / 1e12, 1),
                    "frac_mma": round(flops / (ms * 1e-3) / 1e12 / MX8_TFLOPS, 3)})
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--small", action="store_true", help="1/8-size workload (for profiler captures)")
    ap.add_argument("--div", type=int, default=0,
                    help="divide the token counts by this instead (2 or 4: profiler captures of steady-state tiles)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-baseline leg")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer leg")
    ap.add_argument("--no-ext", action="store_true", help="skip the kernels measured beside the step")
    ap.add_argument("--call", default=None, help="run one call of the step alone (see single_call)")
    ap.add_argument("--mma-peak", action="store_true",
                    help="measure the dense FP8 (e4m3) tensor rate instead: cuBLASLt 8192^3, burst and sustained")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if args.mma_peak:
        return measure_fp8_peak(local)
    if args.call:
        return single_call(args)

    import torch
    from quantized_vlm_gemm_mix_b300 import _build
    _build.build()
    from quantized_vlm_gemm_mix_b300 import mix, synth
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    if args.div > 1:
        args.small = args.div
    calls, h2d, d2h, host, keep = build_workload(torch, mix, synth, dev, small=args.small)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()

    def step(events=None):
        for i, c in enumerate(calls):
            if events is not None:
                events[i][0].record(stream)
            c.fn()
            if events is not None:
                events[i][1].record(stream)

    def barrier():
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(max(3, args.warmup)):
        step()
    barrier()
    _require(mix.mix_device_error() == 0, "a kernel reported a timed-out wait")
    clamped = clamp_report(torch, mix, CLAMP["ws"])

    # One step captured as a CUDA graph: the ~30 launches replay without host
    # gaps (every library call is asynchronous and allocation-free).
    run, timing_mode = step, "eager"
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        run, timing_mode = graph.replay, "cuda graph"
        for _ in range(2):
            run()
        barrier()
    except Exception as exc:  # keep measuring eagerly, and say so
        timing_mode = f"eager (graph capture failed: {type(exc).__name__})"
        barrier()

    # headline: K back-to-back steps, no per-call events
    clocks = ClockSampler(local)
    clocks.start()
    barrier()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        run()
    t1.record(stream)
    barrier()
    clk = clocks.stop()
    ms_step = max_over_ranks(torch, dist, t0.elapsed_time(t1), dev) / args.steps
    _require(mix.mix_device_error() == 0, "a kernel reported a timed-out wait")

    # Per-call durations: a second timed pass, CUDA events on the launching
    # stream around each call.  A short spin kernel before every call keeps
    # the GPU busy while the host enqueues it, so the events bracket device
    # time only, not host launch gaps.
    per_call = np.zeros(len(calls))
    percall_mode = "events per call, spin kernel ahead of each launch"
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in calls]
    for _ in range(args.steps):
        # the first kernel after a synchronise runs slow; an untimed launch of
        # the (small, cache-cold-insensitive) last call takes that cost, and
        # no timed call's inputs are touched by it
        torch.cuda._sleep(100000)
        calls[-1].fn()
        for i, c in enumerate(calls):
            torch.cuda._sleep(400000)
            ev[i][0].record(stream)
            c.fn()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        per_call += np.array([a.elapsed_time(b) for a, b in ev])
    per_call /= args.steps

    step_peak, step_peak_source = step_mma_peak(clk)
    roof_s = sum(c.roof_s(step_peak) for c in calls)
    value = job_value(roof_s, world, ms_step)
    ext = None if args.no_ext else measure_extensions(torch, mix, stream)

    e2e = None
    if not args.no_e2e:
        # Host buffers in, host buffers out, every step.  Two steps are in
        # flight: step i+1's inputs upload on a copy stream into a second
        # device staging set while step i computes, and step i's outputs go
        # back on a third stream, as a serving loop would overlap them.  The
        # main stream moves each step's inputs from staging into place (and
        # its outputs out to staging) with device copies.
        pin_in = [(d, torch.from_numpy(h.view(np.int16) if h.dtype == np.uint16 else h).pin_memory())
                  for d, h in h2d]
        pin_out = [(d, torch.empty(d.shape, dtype=d.dtype).pin_memory()) for d in d2h]
        bi = sum(p.numel() * p.element_size() for _, p in pin_in)
        bo = sum(p.numel() * p.element_size() for _, p in pin_out)
        up_s, down_s = torch.cuda.Stream(), torch.cuda.Stream()
        stage_in = [[torch.empty(p.shape, dtype=p.dtype, device=dev) for _, p in pin_in] for _ in range(2)]
        stage_out = [[torch.empty_like(d) for d in d2h] for _ in range(2)]
        ev = lambda: torch.cuda.Event()
        in_ready, in_free = [ev(), ev()], [ev(), ev()]
        out_ready, out_free = [ev(), ev()], [ev(), ev()]
        used = set()

        def e2e_step(i):
            b = i % 2
            with torch.cuda.stream(up_s):
                if ("in", b) in used:
                    up_s.wait_event(in_free[b])
                for (_, p), sb in zip(pin_in, stage_in[b]):
                    sb.copy_(p, non_blocking=True)
                in_ready[b].record(up_s)
            stream.wait_event(in_ready[b])
            for (d, p), sb in zip(pin_in, stage_in[b]):
                d.view(p.dtype).copy_(sb)
            in_free[b].record(stream)
            run()
            if ("out", b) in used:
                stream.wait_event(out_free[b])
            for d, so in zip(d2h, stage_out[b]):
                so.copy_(d)
            out_ready[b].record(stream)
            with torch.cuda.stream(down_s):
                down_s.wait_event(out_ready[b])
                for (_, p), so in zip(pin_out, stage_out[b]):
                    p.copy_(so, non_blocking=True)
                out_free[b].record(down_s)
            used.update({("in", b), ("out", b)})

        def e2e_run(n, start_ev=None):
            if start_ev is not None:
                up_s.wait_event(start_ev)
            for i in range(n):
                e2e_step(i)
            stream.wait_event(out_free[(n - 1) % 2])   # the last result is on the host

        e2e_run(2)
        torch.cuda.synchronize()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        e2e_run(args.steps, e0)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        ms_e2e = max_over_ranks(torch, dist, e0.elapsed_time(e1), dev) / args.steps
        e2e = {"value": round(job_value(roof_s, world, ms_e2e), 3), "unit": UNIT,
               "ms_per_step": round(ms_e2e, 4), "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
               "overlap": "2 steps in flight: upload, compute and download on separate streams"}

    parts = {}
    for c, ms in zip(calls, per_call):
        e = {"ms": round(float(ms), 5), "GB/s": round(c.bytes / (ms * 1e-3) / 1e9, 1),
             "frac_hbm": round(c.bytes / (ms * 1e-3) / 1e9 / HBM, 3), "roofline_ms": round(c.roof_s() * 1e3, 5)}
        if c.flops:
            e["TFLOP/s"] = round(c.flops / (ms * 1e-3) / 1e12, 1)
            e["frac_mma"] = round(c.flops / (ms * 1e-3) / 1e12 / MX8_TFLOPS, 3)
        parts[c.name] = e
    dom = max(range(len(calls)), key=lambda i: calls[i].roof_s())
    dc = calls[dom]
    ach = dc.flops / (per_call[dom] * 1e-3) / 1e12
    traffic = None
    tp = os.path.join(ROOT, "profiles", "dominant_kernel_traffic.json")
    if os.path.exists(tp) and not args.small:
        tj = json.load(open(tp))
        if tj.get("call") == dc.name and tj.get("source_sha256") == matmul_source_sha():
            traffic = tj.get("dram_bytes_per_launch")
    fp8 = None
    fp = os.path.join(ROOT, "profiles", "fp8_peak.json")
    if os.path.exists(fp):
        fj = json.load(open(fp))
        fp8 = {"fp8_tflops_burst_direct": fj["fp8_tflops_burst"],
               "frac_of_direct": round(ach / fj["fp8_tflops_burst"], 4), "how": fj["command"]}
    roofline = {"bound": "tensor", "kernel": dc.name, "achieved": round(ach, 1), "peak": round(MX8_TFLOPS, 1),
                "unit": "TFLOP/s", "frac": round(ach / MX8_TFLOPS, 4), "traffic": traffic, "fp8_measured": fp8,
                "algorithmic_bytes": dc.bytes, "algorithmic_flops": dc.flops,
                "peak_source": f"2 x measured bf16 burst ({PEAKS['source']}; the call is timed on its own, "
                               f"at full clock); sustained would be {MX8_TFLOPS_SUSTAINED:.0f} TFLOP/s"}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cost1, sample1 = oracle_unit_costs(10.0)
        sec1 = cpu_step_seconds(cost1, args.small)
        procs = max(1, os.cpu_count() or 1)
        costp, samplep = oracle_unit_costs_parallel(10.0, procs)
        secp = cpu_step_seconds(costp, args.small)
        cpu = {"value": 100.0 * roof_s / secp, "unit": UNIT, "cores": procs, "kind": "oracle", "sample": samplep,
               "seconds_per_step": round(secp, 2), **host_cpu(),
               "single_thread": {"value": 100.0 * roof_s / sec1, "cores": 1, "sample": sample1,
                                 "seconds_per_step": round(sec1, 2)}}
    out = {"metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
           "warmup": max(3, args.warmup), "ms_per_step": round(ms_step, 4), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None,
           "dtype": "e4m3 x e4m3 -> fp32 (tcgen05 kind::mxf8f6f4); int32 shift-add; u8 codes",
           "data": "synthetic (seeded; Qwen2-VL-7B / ViT / GQA-attention shapes, paper activation statistics)",
           "config": {"workload": WORKLOAD + (f"_div{8 if args.small is True else args.small}" if args.small else ""),
                      "l2": "inputs larger than L2 (several GB per step; each tensor is evicted before reuse)",
                      "parallelism": f"replicas x{world}", "roofline_ms_per_step": round(roof_s * 1e3, 4),
                      "hbm_peak_gbs": HBM, "mma_peak_tflops_per_call": round(MX8_TFLOPS, 1),
                      "mma_peak_tflops_step": round(step_peak, 1), "mma_peak_step_source": step_peak_source,
                      "timing": timing_mode,
                      "per_call_timing": percall_mode},
           "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clamped_blocks": clamped,
           "gpu_launches": int(sum(c.launches for c in calls) * args.steps), "clocks": clk, "parts": parts,
           "extensions": ext}
    if rank == 0:
        print(json.dumps(out), flush=True)
    del keep
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
