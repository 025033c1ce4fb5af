"""Host logic of the bench's N > 1 path (replicas), on CPU with gloo.

The layer does not shard: `bench.py --gpus N` runs N independent replicas.
What is rank-dependent is the timing reduction (the job's time is its slowest
replica's), the whole-job value, and that the reference arm runs on rank 0
only.  These run here as two gloo ranks; no GPU is needed.
"""
import json
import os
import socket
import subprocess
import sys
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


RANK_SCRIPT = textwrap.dedent("""
    import json, os, sys
    sys.path.insert(0, {root!r})
    import torch
    import torch.distributed as dist
    import bench
    rank, world, _ = bench.dist_env()
    dist.init_process_group("gloo")
    times = [0.25, 0.75]
    t = bench.max_over_ranks(times[rank], world, torch.device("cpu"))
    v = bench.job_value(world, 1e9, t)
    print(json.dumps({{"rank": rank, "t_max": t, "value": v}}), flush=True)
    dist.barrier()
    dist.destroy_process_group()
""")


@pytest.mark.timeout(300)
def test_two_gloo_ranks_take_the_slowest_replica():
    port = _free_port()
    script = RANK_SCRIPT.format(root=ROOT)
    procs = []
    for r in range(2):
        env = dict(os.environ, RANK=str(r), WORLD_SIZE="2", LOCAL_RANK=str(r), MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", script], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=240)
        assert p.returncode == 0, err
        outs.append(json.loads(out.strip().splitlines()[-1]))
    for o in outs:
        assert o["t_max"] == 0.75                        # every rank sees the slowest replica
        assert abs(o["value"] - 2 * 1e9 / 0.75 / 1e12) < 1e-12   # whole job: both replicas' bytes


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        steps, warmup = 1, 0

    called = []
    monkeypatch.setattr(bench, "time_oracle", lambda *a, **k: called.append(1))
    assert bench.run_reference(Args(), None) == 0
    assert called == [] and capsys.readouterr().out == ""


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.5, 1, None) == 1.5
    assert bench.job_value(1, 2e12, 1.0) == 2.0
