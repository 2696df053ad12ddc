"""The N > 1 launch of bench.py (replicas only: each rank runs the whole step
on its own GPU).  Its host logic runs here as two gloo ranks on the CPU, each
a separate process started the way torchrun starts them (RANK, WORLD_SIZE,
MASTER_ADDR/PORT in the environment)."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_RANK_SCRIPT = r"""
import json, os, sys
sys.path.insert(0, {root!r})
import torch
import torch.distributed as dist
import bench
dist.init_process_group("gloo")
rank, world = dist.get_rank(), dist.get_world_size()
ms = [2.5, 3.25][rank]                       # this rank's time per step
dev = torch.device("cpu")
worst = bench.max_over_ranks(torch, dist, ms, dev)
dist.barrier()
print(json.dumps({{"rank": rank, "world": world, "max_ms": worst,
                   "value": bench.job_value(0.0015, world, worst)}}), flush=True)
dist.destroy_process_group()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _launch(args, world, env_extra=None, timeout=120):
    port = _free_port()
    procs = []
    for r in range(world):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE=str(world),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), **(env_extra or {}))
        procs.append(subprocess.Popen(args, cwd=ROOT, env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    try:
        for p in procs:
            out, err = p.communicate(timeout=timeout)
            outs.append((p.returncode, out, err))
    finally:
        for p in procs:
            if p.poll() is None:
                p.kill()
    return outs


def test_max_over_ranks_and_job_value_two_gloo_ranks():
    outs = _launch([sys.executable, "-c", _RANK_SCRIPT.format(root=ROOT)], world=2)
    lines = []
    for rc, out, err in outs:
        assert rc == 0, err[-2000:]
        lines.append(json.loads(out.strip().splitlines()[-1]))
    for r, d in enumerate(lines):
        assert d["rank"] == r and d["world"] == 2
        assert d["max_ms"] == 3.25                     # the slowest rank's time, on every rank
        # two replicas' work over the slowest time: 2 x 1.5 ms of roofline in 3.25 ms
        assert d["value"] == pytest.approx(100.0 * 2 * 0.0015 / 3.25e-3)


def test_job_value_single_rank():
    import bench
    assert bench.max_over_ranks(None, None, 1.75, None) == 1.75
    assert bench.job_value(0.0015, 1, 2.0) == pytest.approx(75.0)
    # weak scaling: twice the ranks at the same time per step is twice the value
    assert bench.job_value(0.0015, 2, 2.0) == pytest.approx(2 * bench.job_value(0.0015, 1, 2.0))


def test_reference_arm_other_ranks_exit_without_work():
    """Under torchrun only rank 0 runs the oracle arm and prints its line."""
    outs = _launch([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
                    "--warmup", "0"], world=2, timeout=300)
    rc1, out1, err1 = outs[1]
    assert rc1 == 0, err1[-2000:]
    assert out1.strip() == ""
    rc0, out0, err0 = outs[0]
    assert rc0 == 0, err0[-2000:]
    line = json.loads(out0.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
