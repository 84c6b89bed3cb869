"""Multi-process paths of bench.py, on CPU.

The benchmark runs one independent replica per GPU (no collective on the data
path); the only cross-rank steps are the barrier and the max over ranks of the
timed interval.  Those run here with the gloo backend at world size 2.
"""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

from tests.conftest import ROOT


def _worker(rank, world, port, values, results):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        dist.barrier()
        m = bench.reduce_max_over_ranks(values[rank], world, torch.device("cpu"))
        results[rank] = (m, bench.job_throughput(100, world, m))
    finally:
        dist.destroy_process_group()


def _free_port():
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_max_over_ranks_and_job_throughput_gloo():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        values = [12.5, 40.0]
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, values, results)) for r in range(2)]
        for pr in procs:
            pr.start()
        for pr in procs:
            pr.join(timeout=120)
            assert pr.exitcode == 0
        for r in range(2):
            m, tput = results[r]
            assert m == 40.0
            assert abs(tput - 2 * 100 / 0.040) < 1e-6


def _run_reference(rank, world):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    return subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", str(world),
                           "--steps", "1", "--warmup", "0"], cwd=ROOT, env=env,
                          capture_output=True, text=True, timeout=600)


def test_reference_arm_other_ranks_exit_without_work():
    r = _run_reference(1, 2)
    assert r.returncode == 0 and r.stdout.strip() == ""


@pytest.mark.timeout(600)
def test_reference_arm_prints_one_line():
    r = _run_reference(0, 1)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "tokens/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
