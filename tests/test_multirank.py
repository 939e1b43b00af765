"""The N > 1 host path on the CPU, world size 2 over gloo (127.0.0.1).

bench.py runs one replica per rank: every rank draws its own seeded prompts,
times its stack, and rank 0 prints one JSON line with the slowest rank's time
(max over ranks) and the job's total tokens.  These tests run that host logic
with real processes and a real process group, without a GPU:
  * `bench.py --impl reference` launched by torch.distributed.run (2 ranks):
    rank 0 alone times the oracle and prints, the other rank exits 0;
  * bench's max-over-ranks reduction, barrier and per-rank seeds inside a
    2-rank gloo group.
"""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
torch = pytest.importorskip("torch")


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_reference_arm_under_torchrun_two_ranks():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "1"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]


def _rank_body(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_info()[:2] == (rank, world)
        # the slowest rank's time is the job's time
        t = bench.max_over_ranks(10.0 + rank, world)
        bench.barrier(world)
        # every rank draws its own prompts (replicas of independent prompts)
        layer = bench.make_layers(rank, n_layers=1)[0]
        digest = float(np.asarray(layer.qkv[:64], np.float64).sum())
        got = [None] * world
        dist.all_gather_object(got, digest)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"max": t, "digests": got}, f)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_barrier_and_replica_seeds(tmp_path):
    import torch.multiprocessing as mp
    port = _free_port()
    mp.spawn(_rank_body, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    assert res[0]["max"] == res[1]["max"] == 11.0
    d0, d1 = res[0]["digests"]
    assert res[0]["digests"] == res[1]["digests"] and d0 != d1
