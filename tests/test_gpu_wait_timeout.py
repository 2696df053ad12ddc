"""The bounded waits of the tensor-core matmul, made to run out on purpose
and safely: the staged kernel is launched on one tile with its producer
switched off (no TMA, bulk copy or tcgen05 operation is ever issued), so the
MMA thread's wait for the first stage times out with nothing in flight.  The
kernel must record the timeout in the device error word, drain, free its TMEM
and return; the device must then run an ordinary matmul correctly."""
import ctypes

import numpy as np
import pytest

from quantized_vlm_gemm_mix_b300 import synth
from helpers import GEMM_REL_TOL, row_rel_err, to_dev, to_host

pytestmark = pytest.mark.gpu


def test_wait_runs_out_and_device_recovers(orc):
    import torch
    from quantized_vlm_gemm_mix_b300 import mix
    mix.mix_device_error()                                   # start from a clear word
    ws = torch.empty(mix.MIX_SELFTEST_WORKSPACE_BYTES, dtype=torch.uint8, device="cuda")
    st = mix.lib.mix_selftest_wait_timeout(ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                                           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == mix.MIX_OK, mix.status_str(st)
    torch.cuda.synchronize()
    word = mix.mix_device_error(clear=True)
    assert word & (2 | 32), word                             # the MMA thread's (or a scale warp's) wait
    assert mix.mix_device_error() == 0                       # cleared
    # too small a workspace is refused before any launch
    st = mix.lib.mix_selftest_wait_timeout(ctypes.c_void_p(ws.data_ptr()), 1024, None)
    assert st == mix.MIX_ERR_WORKSPACE
    # an ordinary staged matmul afterwards
    M, N, K = 256, 448, 512
    a = synth.to_bf16_bits(synth.vlm_activations(60, 0, M, K, visual_rows=192))
    w = synth.to_bf16_bits(synth.normal(61, 1, N * K, 0, 0.02).reshape(N, K))
    ac, ash = orc.mix_quantize(a, 2)
    bc, bs = orc.mx_quantize(w, 1, 1)
    c = torch.empty((M, N), dtype=torch.float32, device="cuda")
    d = mix.gemm_desc(M, N, K, to_dev(ac), to_dev(ash), 2, -8, to_dev(bc), to_dev(bs), 1, c=c,
                      algo=mix.MIX_GEMM_TCGEN05_STAGED)
    mix.gemm(d)
    torch.cuda.synchronize()
    assert mix.mix_device_error() == 0
    assert row_rel_err(to_host(c), orc.gemm(ac, ash, 2, -8, bc, bs, 1)) <= GEMM_REL_TOL
