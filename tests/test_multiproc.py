"""The bench's multi-process host logic on CPU: two gloo ranks (world size 2)
run the process-group set-up, the max-over-ranks timing and the barrier that
`bench.py --gpus N` uses under torchrun, and the reference arm prints its one
line from rank 0 only while the other rank exits 0 without output."""
import argparse
import contextlib
import io
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

WORLD = 2

# bench.dist_setup picks gloo only without a GPU (NCCL otherwise, one GPU per
# rank): this is the CPU test of the multi-rank host path
pytestmark = pytest.mark.skipif(torch.cuda.is_available(), reason="gloo path runs on CPU-only hosts")


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _env(rank: int, port: int):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(WORLD), RANK=str(rank),
                      LOCAL_RANK=str(rank))


def _timing_worker(rank: int, port: int, q):
    _env(rank, port)
    import torch
    import torch.distributed as dist
    import bench
    try:
        r, world, local = bench.dist_setup(WORLD)
        # each rank reports its own step time; the job's time is the slowest rank's
        ms = bench.max_over_ranks(1.5 * (rank + 1), world, torch.device("cpu"))
        bench.barrier(world)
        q.put((rank, r, world, local, ms))
    finally:
        if dist.is_initialized():
            dist.destroy_process_group()


def _reference_worker(rank: int, port: int, q):
    _env(rank, port)
    import torch.distributed as dist
    import bench
    import kvq_synth as synth
    args = argparse.Namespace(gpus=WORLD, seed=1, oracle_units=1, warmup=1, steps=1)
    out = io.StringIO()
    try:
        with contextlib.redirect_stdout(out):
            rc = bench.run_reference(args, synth.WORKLOADS["tiny"])
        q.put((rank, rc, out.getvalue()))
    finally:
        if dist.is_initialized():
            dist.destroy_process_group()


def _run(target):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=target, args=(r, port, q)) for r in range(WORLD)]
    for p in procs:
        p.start()
    results = [q.get(timeout=240) for _ in range(WORLD)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return sorted(results)


def test_two_ranks_max_over_ranks_and_barrier():
    res = _run(_timing_worker)
    for rank, (got_rank, r, world, local, ms) in enumerate(res):
        assert (got_rank, r, world, local) == (rank, rank, WORLD, rank)
        assert ms == pytest.approx(3.0)  # both ranks see the slower rank's time


def test_reference_arm_prints_on_rank_zero_only():
    import json
    res = _run(_reference_worker)
    (r0, rc0, out0), (r1, rc1, out1) = res
    assert (r0, rc0, r1, rc1) == (0, 0, 1, 0)
    assert out1 == ""
    line = json.loads(out0.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == WORLD and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
