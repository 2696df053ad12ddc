"""The no-allocation K-smoothing entry point (ksmooth_kv_noalloc).

Some callers cannot give the library device memory: hosts whose allocator owns
all device memory, and loops that must never call cudaMalloc because it can
synchronise the whole device.  This entry point keeps its partial sums in a
fixed array inside the library.  These tests call it through the C ABI twice
in a row and check each result against the workspace-taking ksmooth_kv on the
same input.  Both run the same kernels with the same token chunking and the
same fixed-order sums, so the results must agree bit for bit: a tolerance
would hide a stale partial sum that perturbs only the last bits.  The file
runs last so that a failure here leaves every other test already run."""
import ctypes

import numpy as np
import pytest

from quantized_vlm_gemm_mix_b300 import synth
from helpers import to_dev, to_host

pytestmark = pytest.mark.gpu


def _with_workspace(mix, kd, tokens, heads, dim):
    import torch
    mean = torch.empty((heads, dim), dtype=torch.float32, device="cuda")
    kout = torch.empty((tokens, heads, dim), dtype=torch.float32, device="cuda")
    ws = torch.empty(mix.ksmooth_workspace_bytes(tokens, heads, dim), dtype=torch.uint8, device="cuda")
    mix.ksmooth_kv(kd, tokens, heads, dim, heads * dim, mean, mix.KSMOOTH_COMPUTE, kout, ws)
    return mean, kout


def _no_alloc(mix, kd, tokens, heads, dim):
    import torch
    mean = torch.empty((heads, dim), dtype=torch.float32, device="cuda")
    kout = torch.empty((tokens, heads, dim), dtype=torch.float32, device="cuda")
    st = mix.lib.ksmooth_kv_noalloc(ctypes.c_void_p(kd.data_ptr()), mix.MIX_DT_BF16, tokens, heads, dim,
                                    heads * dim, ctypes.c_void_p(mean.data_ptr()), mix.KSMOOTH_COMPUTE,
                                    ctypes.c_void_p(kout.data_ptr()),
                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == mix.MIX_OK, mix.status_str(st)
    return mean, kout


def test_no_alloc_matches_workspace_entry_point_on_two_calls():
    import torch
    from quantized_vlm_gemm_mix_b300 import mix
    # two different calls in a row: the second has fewer tokens and other keys,
    # so anything left over in the shared array from the first would show
    for seed, tokens in ((3, 4096), (4, 1000)):
        _, k, _ = synth.attention_qkv(seed, tokens, 2, 4, 128)
        kd = to_dev(synth.to_bf16_bits(k).reshape(tokens, 512))
        m_ref, k_ref = _with_workspace(mix, kd, tokens, 4, 128)
        m, ko = _no_alloc(mix, kd, tokens, 4, 128)
        torch.cuda.synchronize()
        assert np.array_equal(to_host(m).view(np.uint32), to_host(m_ref).view(np.uint32))
        assert np.array_equal(to_host(ko).view(np.uint32), to_host(k_ref).view(np.uint32))


def test_no_alloc_rejects_requests_beyond_its_scratch():
    import torch
    from quantized_vlm_gemm_mix_b300 import mix
    heads, dim = 264, 1024                      # 270336 channels need more than 2 MiB of partial sums
    assert mix.ksmooth_workspace_bytes(64, heads, dim) > mix.KSMOOTH_NOALLOC_SCRATCH_BYTES
    dummy = torch.zeros(64, dtype=torch.float32, device="cuda")
    st = mix.lib.ksmooth_kv_noalloc(ctypes.c_void_p(dummy.data_ptr()), mix.MIX_DT_BF16, 64, heads, dim,
                                    heads * dim, ctypes.c_void_p(dummy.data_ptr()), mix.KSMOOTH_COMPUTE, None,
                                    None)
    assert st == mix.MIX_ERR_WORKSPACE
