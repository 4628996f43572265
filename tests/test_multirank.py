"""The multi-process (N > 1) host logic of bench.py on CPU: two ranks over
gloo agree on the slowest rank's time and pass the barrier, and the reference
arm launched as two ranks runs and prints on rank 0 only.  (Multi-GPU runs
are independent replicas: there is no data-path collective to test.)"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
torch = pytest.importorskip("torch")


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, local = bench.dist_info()
    bench.barrier(w)
    # each rank's "step time"; every rank must see the slowest one
    got = bench.max_over_ranks(1.5 + rank, w)
    bench.barrier(w)
    dist.destroy_process_group()
    with open(os.path.join(out, f"rank{rank}.json"), "w") as f:
        json.dump({"rank": r, "world": w, "local": local, "max": got}, f)


def test_two_gloo_ranks_agree_on_the_slowest_time(tmp_path):
    port = free_port()
    torch.multiprocessing.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2,
                                join=True)
    for rank in range(2):
        rec = json.load(open(tmp_path / f"rank{rank}.json"))
        assert rec == {"rank": rank, "world": 2, "local": rank, "max": 2.5}


def test_reference_arm_runs_on_rank_zero_only():
    env0 = dict(os.environ, RANK="0", WORLD_SIZE="2", LOCAL_RANK="0")
    env1 = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
           "--steps", "1", "--warmup", "3"]
    p1 = subprocess.run(cmd, env=env1, capture_output=True, text=True, cwd=ROOT,
                        timeout=300)
    assert p1.returncode == 0 and p1.stdout.strip() == ""
    p0 = subprocess.run(cmd, env=env0, capture_output=True, text=True, cwd=ROOT,
                        timeout=300)
    assert p0.returncode == 0, p0.stderr[-2000:]
    lines = [l for l in p0.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle"
    assert rec["e2e"]["h2d_bytes_per_step"] == 0
