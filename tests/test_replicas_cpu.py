"""The N > 1 path of bench.py on CPU (gloo, world size 2): the path shards
into independent replicas, so the only cross-rank steps are the barrier and
the max over ranks of the timings; each rank draws its own inputs; the
whole-job value counts every rank's tokens over the slowest rank's time;
only rank 0 prints (the reference arm: the other ranks do no work)."""

from __future__ import annotations

import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    import bench
    from workloads import LM_F1
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(10.0 + 5.0 * rank, world, "cpu")
        dist.barrier()
        seeds = [bench.replica_seed(LM_F1, rank, i) for i in range(4)]
        all_seeds = [None] * world
        dist.all_gather_object(all_seeds, seeds)
        buf = io.StringIO()
        with redirect_stdout(buf):  # the reference arm prints on rank 0 only
            class A:
                warmup, steps, gpus = 0, 0, world
            if rank != 0:
                bench.run_reference(A, LM_F1, rank)
        out[rank] = (ms, all_seeds, buf.getvalue())
    finally:
        dist.destroy_process_group()


def test_replicas_gloo_world2():
    world, port = 2, _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
    assert set(out.keys()) == {0, 1}
    for r in range(world):
        ms, all_seeds, printed = out[r]
        assert ms == 15.0                        # every rank sees the slowest rank's time
        assert len(set(all_seeds[0]) & set(all_seeds[1])) == 0  # independent batches
        assert printed == ""


def test_job_throughput_counts_every_rank():
    import bench
    from workloads import LM_F1
    one = bench.job_tokens_per_s(LM_F1, 1, 0.1)
    assert bench.job_tokens_per_s(LM_F1, 4, 0.1) == pytest.approx(4 * one)
    assert bench.max_over_ranks(3.0, 1, "cpu") == 3.0


def test_roofline_byte_counts():
    """The numerators of the reported roofline fractions, by hand for the
    headline workload (8 x 2048 x 12 heads, d = 64, bf16): q, k, v in and o
    out at 128 bytes a row, beta and lambda at 4 bytes a step, the final
    state once (96 heads x 64 x 64 fp32); the sequential kernel's share is
    q, k, o and the state."""
    import bench
    from workloads import LM_F1, LONG_F1
    rows = 8 * 2048 * 12
    state = 96 * 64 * 64 * 4
    assert bench.algorithmic_bytes(LM_F1) == rows * 4 * 128 + rows * 8 + state == 103809024
    assert bench.kernel_bytes(LM_F1, ["tc_wyu_kernel", "tc_fwd_chain_kernel"]) == [
        rows * 2 * 128 + rows * 8, rows * 3 * 128 + state]
    rows_l = 2 * 16384 * 16
    assert bench.kernel_bytes(LONG_F1, ["tc_wyu_kernel", "tc_fwd_kernel"])[1] == \
        rows_l * 3 * 256 + 32 * 128 * 128 * 4
