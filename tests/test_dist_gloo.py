"""The bench's multi-rank plumbing on CPU: two gloo ranks on 127.0.0.1.

Each rank runs its own population (seeds offset by rank * pop, so no two ranks
regenerate the same noise) and only the timing is reduced (max over ranks);
there is no data-path collective."""

import os
import socket

import pytest
import torch
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
    from virtual_noise_perturbed_gb300 import workloads

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_env()
        wl = workloads.make(1)
        seeds = wl.seeds + r * wl.pop
        bench.barrier(w)
        mx = bench.max_over_ranks(float(10 + 5 * r), w, None)
        q.put((r, w, local, mx, seeds.tolist()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_timing_and_shard_population():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    assert [x[0] for x in res] == [0, 1] and all(x[1] == 2 for x in res)
    assert all(x[3] == 15.0 for x in res)                 # max over ranks
    s0, s1 = set(res[0][4]), set(res[1][4])
    assert not (s0 & s1)                                   # disjoint populations


def test_single_rank_defaults():
    import bench
    for v in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        os.environ.pop(v, None)
    assert bench.dist_env() == (1, 0, 0)
    assert bench.max_over_ranks(3.5, 1) == 3.5


def test_reference_arm_under_torchrun_prints_once():
    """The reference arm launched as the multi-GPU bench is: rank 0 alone times the
    oracle and prints the one JSON line; the other rank exits 0 without work."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(root, "bench.py"), "--impl", "reference", "--workload", "tiny",
           "--gpus", "2", "--steps", "1", "--warmup", "3"]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=root)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
