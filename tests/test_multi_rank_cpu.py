"""The benchmark's multi-process harness on CPU (gloo, two ranks): process
group set-up, the barrier and the max-over-ranks timing reduction, and the
reference arm under torchrun (rank 0 alone prints the one JSON line, the
other rank exits 0).  The GPU path runs replicas only -- every rank attends
its own copy of the workload -- so these host pieces are what N > 1 adds."""
from __future__ import annotations

import json
import multiprocessing as mp
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, port: int, q) -> None:
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": "2",
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "CUDA_VISIBLE_DEVICES": ""})
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    world, r, local = bench.dist_setup()
    bench.barrier(world)
    got = bench.max_over_ranks(float(10 * (rank + 1)), world)
    q.put((r, world, dist.get_backend(), got))
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_max():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert sorted(r for r, *_ in results) == [0, 1]
    for _, world, backend, got in results:
        assert world == 2 and backend == "gloo" and got == 20.0


def test_reference_arm_under_torchrun_prints_once():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "3", "--workload", "tiny"]
    res = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, res.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["cpu_baseline"]["kind"] == "oracle" and line["value"] > 0
