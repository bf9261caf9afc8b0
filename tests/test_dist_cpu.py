"""The multi-process path on CPU: gloo ranks, world size 2.

The verify step does not shard (sequences are independent), so several GPUs run
replicas: each rank times its own step, the job's device time is the maximum over
ranks and the units are summed.  These tests run that aggregation and the reference
arm's rank handling as real gloo process groups on the host.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist()
    d.barrier()
    t = d.max(1.0 + rank)          # per-rank device time: the job takes the slowest
    u = d.sum(10.0 * (rank + 1))   # per-rank units: the job processed all of them
    d.barrier()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"max": t, "sum": u, "world": d.world}, f)
    d.close()


def test_replica_aggregation_gloo(tmp_path):
    world, port = 2, _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    for r in range(world):
        res = json.load(open(tmp_path / f"rank{r}.json"))
        assert res == {"max": 2.0, "sum": 30.0, "world": 2}


@pytest.mark.timeout(300)
def test_reference_arm_under_torchrun_two_ranks(tmp_path):
    """Rank 0 alone runs the oracle and prints one JSON line; rank 1 exits 0."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "1",
           "--steps", "1", "--warmup", "0", "--gpus", "2"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=280)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    res = json.loads(lines[0])
    assert res["impl"] == "reference" and res["n_gpus"] == 2 and res["value"] > 0
    assert res["cpu_baseline"]["kind"] == "oracle"
    assert res["e2e"]["h2d_bytes_per_step"] == 0
