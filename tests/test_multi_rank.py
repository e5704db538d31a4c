"""The benchmark's multi-rank plumbing, with two gloo ranks on the CPU.

Each GPU runs its own replica of the workload; the only cross-rank operations are a
barrier and a max over ranks of the timed region.  The reference arm runs on rank 0 only.
"""

import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import os, sys, json
sys.path.insert(0, %(root)r)
import torch.distributed as dist
import bench
rank = int(os.environ["RANK"]); world = int(os.environ["WORLD_SIZE"])
dist.init_process_group("gloo")
bench.barrier(world)
elapsed = [10.0, 25.0][rank]
mx = bench.max_over_ranks(world, elapsed, device="cpu")
value = bench.job_throughput(world, 1_000_000_000, 4, mx)
print(json.dumps({"rank": rank, "max": mx, "value": value}), flush=True)
dist.destroy_process_group()
"""


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _launch(code, world=2, extra_env=None):
    port = _free_port()
    procs = []
    for r in range(world):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE=str(world),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), **(extra_env or {}))
        procs.append(subprocess.Popen([sys.executable, "-c", code], env=env, cwd=ROOT,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err[-2000:]
        outs.append(out)
    return outs


def test_max_over_ranks_and_weak_scaling_value():
    import json
    outs = _launch(WORKER % {"root": ROOT})
    res = [json.loads(o.strip().splitlines()[-1]) for o in outs]
    assert all(r["max"] == 25.0 for r in res)
    # 2 ranks x 1 GB x 4 steps in 25 ms (the slowest rank) = 320 GB/s
    assert all(abs(r["value"] - 320.0) < 1e-9 for r in res)


def test_reference_arm_runs_on_rank_zero_only():
    code = (f"import sys; sys.path.insert(0, {ROOT!r}); import bench; "
            "sys.argv=['bench.py','--impl','reference','--steps','1','--warmup','3','--ref-units','16']; "
            "sys.exit(bench.main())")
    outs = _launch(code)
    assert outs[1].strip() == ""                      # rank 1 exits 0 without work or output
    import json
    line = json.loads(outs[0].strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
