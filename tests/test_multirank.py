"""The N>1 benchmark path on CPU: two gloo ranks, independent replicas.

Each rank draws its own id batches (no two ranks decode the same batch), and
the step time is the maximum over ranks.  No data-path collective exists."""

import os
import socket

import numpy as np
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, lr = bench.dist_env()
        t = bench.max_over_ranks(1.0 + rank, w)
        ids = bench.make_batches("tiny", 2048, 2, bench.batch_seed_offset(r))
        bench.barrier(w)
        q.put((r, w, lr, t, ids))
    finally:
        dist.destroy_process_group()


def test_two_rank_replicas_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in res] == [0, 1] and all(r[1] == world for r in res)
    assert all(r[3] == 2.0 for r in res)  # max over ranks
    a, b = res[0][4], res[1][4]
    assert a.shape == b.shape and not np.array_equal(a, b)


def test_reference_arm_under_torchrun_prints_one_line():
    """Two ranks launched as the multi-GPU bench is: rank 0 alone times the
    oracle and prints the line; the other rank exits 0 without work."""
    import json
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--config", "dense_gnn", "--rows", "20000", "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=root, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
