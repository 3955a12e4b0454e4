"""The N > 1 path of bench.py on CPU: two ranks over gloo (no GPU).

The hot path does not shard (each GPU runs an independent replica), so the only
multi-rank logic is the launch and timing plumbing: rank set-up from the
torchrun environment, the barriers around the timed region, the max over ranks
of the elapsed time, and the reference arm, which rank 0 alone runs and prints.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    w, r, _ = bench.dist_setup()
    bench.barrier(w)
    elapsed = bench.max_over_ranks(10.0 + r, w)  # each rank's "elapsed time"
    bench.barrier(w)
    q.put((r, w, elapsed))
    torch.distributed.destroy_process_group()


@pytest.mark.skipif(torch.cuda.is_available(), reason="the gloo path is the one without GPUs")
def test_two_gloo_ranks_time_with_the_slowest():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 2, 11.0), (1, 2, 11.0)]


@pytest.mark.skipif(torch.cuda.is_available(), reason="the gloo path is the one without GPUs")
@pytest.mark.parametrize("mode", [[], ["--scheduler"], ["--reuse-cached"]])
def test_reference_arm_under_torchrun_prints_once(mode):
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--workload", "tiny", "--steps", "2", "--warmup", "1",
           "--ref-seconds", "0.5"] + mode
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
    if mode == ["--scheduler"]:
        assert "window scheduler" in d["cpu_baseline"]["sample"] and "scheduler" in d["config"]
    if mode == ["--reuse-cached"]:
        assert "kept cached part" in d["cpu_baseline"]["sample"]
