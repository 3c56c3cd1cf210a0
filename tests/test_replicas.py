"""Multi-replica path of bench.py on the CPU (gloo, world size 2).

An iteration has no exchange step, so the multi-GPU form is independent
replicas: each rank plans and runs its own batch, a barrier brackets the
timed region, and the job's rate is all ranks' rows over the slowest
rank's time.  These tests run that host logic with two gloo ranks: the
rendezvous and helpers, one planner per replica through the C ABI, and the
reference arm under torchrun (rank 0 alone runs it; the other rank exits 0).
"""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _replica(rank, world, port, queue):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    import chunked_prefill_hybrid_tau_gb300 as hb
    w, r, _ = bench.dist_setup(None)
    assert (w, r) == (world, rank)
    # each replica owns its queue: rank-dependent decodes and one prompt
    rng = np.random.default_rng(100 + rank)
    dec_ctx = [int(c) for c in rng.integers(1, 300, 3 + rank)]
    dec_pages = [list(range(i * 20, i * 20 + (c + 15) // 16)) for i, c in enumerate(dec_ctx)]
    pool = list(range(200, 400))
    hp = hb.hb_plan_batch(dec_ctx, dec_pages, [500], [0], [[]], pool, 64, 64)
    bench.barrier(world)
    t_mine = 0.01 * (rank + 1)  # stand-in for this rank's timed region
    t_max = bench.max_over_ranks(t_mine, world)
    queue.put((rank, hp.n_rows, len(dec_ctx), t_max))
    bench.barrier(world)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_replica_helpers_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_replica, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=5) for _ in range(2))
    # both ranks see the slowest rank's time; each planned its own full budget
    assert [g[3] for g in got] == [0.02, 0.02]
    assert [g[1] for g in got] == [64, 64]
    assert [g[2] for g in got] == [3, 4]
    # the job's rate as bench.py reports it: all ranks' rows over the max time
    steps = 10
    value = sum(g[1] for g in got) * steps / got[0][3]
    assert value == pytest.approx(2 * 64 * steps / 0.02)


@pytest.mark.slow
def test_reference_arm_under_torchrun_two_ranks():
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout  # rank 0 alone prints
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
