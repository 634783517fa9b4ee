"""The benchmark's multi-rank path on the CPU (gloo, world size 2): the
max-over-ranks timing reduction and the barrier, and the launch of the
reference arm under torchrun, where rank 0 alone runs and prints one line and
the other rank exits 0 without work.  The path runs N independent replicas (the
attention work does not shard, see the design notes), so these are its only
collectives."""
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


def _rank(rank: int, ws: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    got_ws, got_rank, _ = bench.dist_init()
    assert (got_ws, got_rank) == (ws, rank) and dist.get_backend() == "gloo"
    bench.barrier(ws)
    # each rank's step time; the job's time is the slowest rank's
    m = bench.reduce_max(1.5 + rank, ws)
    bench.barrier(ws)
    dist.destroy_process_group()
    q.put((rank, m))


def test_reduce_max_and_barrier_over_two_gloo_ranks():
    ws, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(ws))
    assert got == {0: 2.5, 1: 2.5}


def test_reduce_max_is_the_identity_on_one_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(3.25, 1) == 3.25
    bench.barrier(1)  # no process group: a no-op


@pytest.mark.timeout(600)
def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["steps"] == 1
    assert rec["value"] > 0 and rec["cpu_baseline"]["kind"] == "oracle"
    assert rec["e2e"]["h2d_bytes_per_step"] == 0
