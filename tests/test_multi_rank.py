"""The multi-rank path of bench.py on CPU with the gloo backend, world size 2: one process per
rank, each with its own seeded batch (weak scaling, no data-path collective), the timing
reduced by max and the work by sum over ranks, and the reference arm printed by rank 0 only.
No GPU: the GPU arm needs one, but its rank logic is the code exercised here."""
import json
import multiprocessing as mp
import os
import socket
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist, r, w, _ = bench.dist_setup(world)
    assert dist is not None and (r, w) == (rank, world)
    dist.barrier()
    mx = bench.max_over_ranks(dist, float(rank + 1), "cpu")
    sm = bench.sum_over_ranks(dist, float(10 * (rank + 1)), "cpu")
    out.put((rank, mx, sm))
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_time_by_max_and_work_by_sum():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == [(0, 2.0, 30.0), (1, 2.0, 30.0)]


def test_each_rank_builds_its_own_batch():
    """Weak scaling: the same shapes, different seeded values per rank."""
    sys.path.insert(0, ROOT)
    import bench
    d0, c0 = bench.make_workload("swa64", seed=0)
    d1, c1 = bench.make_workload("swa64", seed=1)
    assert d0 == d1 and [c.q.shape for c in c0] == [c.q.shape for c in c1]
    assert not torch.equal(c0[0].q, c1[0].q)


def test_reference_arm_prints_one_line_from_rank_zero():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3",
           "--workload", "swa64", "--ref-step-seconds", "0.4"]
    res = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300,
                         env={**os.environ, "OMP_NUM_THREADS": "2"})
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [json.loads(l) for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
