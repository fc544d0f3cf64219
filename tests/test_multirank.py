"""Multi-rank host logic of bench.py on CPU: world_size-2 gloo process groups.

The hot path shards by independent problems (each rank runs its own batch of
sequences, weak scaling); the only cross-rank steps are the barrier around the
timed region and the max over ranks of the elapsed time.  Both are exercised
here with the gloo backend, rendezvous on 127.0.0.1.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, loc = bench.dist_env()
        assert (w, r, loc) == (world, rank, rank)
        bench.barrier(world)
        # each rank times a different elapsed; every rank must see the slowest
        mx = bench.max_over_ranks(10.0 + 7.5 * rank, world)
        bench.barrier(world)
        q.put((rank, mx))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    codes = [p.exitcode for p in procs]
    for p in procs:
        if p.is_alive():
            p.kill()
    assert codes == [0, 0], codes
    got = dict(q.get(timeout=5) for _ in range(world))
    assert got == {0: 17.5, 1: 17.5}


def test_single_rank_identity():
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25
    bench.barrier(1)  # no process group needed


def test_reference_arm_nonzero_rank_does_no_work(capsys):
    """Under torchrun only rank 0 runs the oracle and prints the line."""
    import argparse

    import bench
    from block_sparse_gqa_causal_gb300.workloads import BY_NAME
    args = argparse.Namespace(steps=1, warmup=0)
    assert bench.run_reference(args, BY_NAME["train_n128k"], 2, 1) is None
    assert capsys.readouterr().out == ""


def test_weak_scaling_value_counts_all_ranks():
    """The whole-job value is world x per-rank work over the slowest rank's time."""
    import bench
    from block_sparse_gqa_causal_gb300.workloads import BY_NAME
    w = BY_NAME["train_n128k"]
    f1 = sum(bench.useful_flops(w).values())
    assert f1 > 0
    # doubling the batch doubles the useful FLOPs: per-rank work is additive
    f2 = sum(bench.useful_flops(w.scaled(B=2 * w.B)).values())
    assert f2 == pytest.approx(2 * f1, rel=1e-12)
