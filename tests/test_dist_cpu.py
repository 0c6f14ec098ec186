"""The multi-process path of bench.py on CPU (gloo, world size 2): the max-over-ranks reduction
of the timings, and the reference arm under torchrun, which runs on rank 0 alone and prints one
JSON line while the other rank exits 0 without work."""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench

    dist, r, w, _ = bench.dist_setup()
    try:
        assert dist is not None and (r, w) == (rank, world)
        out[rank] = (dist.get_backend(), bench.dist_max(dist, float(10 + 3 * rank), "cpu"))
    finally:
        dist.destroy_process_group()


def test_dist_max_over_two_gloo_ranks():
    import torch.multiprocessing as mp

    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(2, port, out), nprocs=2, start_method="spawn", join=True)
        res = dict(out)
    assert res[0] == ("gloo", 13.0) and res[1] == ("gloo", 13.0)


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
           "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"), "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    p = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
