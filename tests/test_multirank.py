"""The benchmark's multi-replica host logic on CPU ranks (gloo, world size 2): the step time
is the slowest rank's, the value counts every replica's bytes, and the reference arm runs on
rank 0 alone.  The hot path itself shards into independent replicas with no collective."""
import os
import socket
import sys
from pathlib import Path

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = Path(__file__).resolve().parent.parent


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    sys.path.insert(0, str(ROOT))
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        local_us = [150.0, 172.5][rank]
        m = bench.max_over_ranks(local_us, torch.device("cpu"))
        results[rank] = (m, bench.job_value_gbs(1_000_000, world, m))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_step():
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        mp.start_processes(_rank_main, args=(2, port, results), nprocs=2, join=True, start_method="spawn")
        got = dict(results)
    assert got[0][0] == got[1][0] == 172.5
    assert got[0][1] == pytest.approx(2 * 1_000_000 / 172.5 / 1e3)


def test_single_process_needs_no_process_group():
    sys.path.insert(0, str(ROOT))
    import bench
    assert bench.max_over_ranks(3.5, torch.device("cpu")) == 3.5
    assert bench.job_value_gbs(587_829_248, 1, 168.8) == pytest.approx(3482.4, rel=1e-3)


def test_reference_arm_runs_on_rank_0_only():
    sys.path.insert(0, str(ROOT))
    import bench
    args = bench.argparse.Namespace(gpus=2, steps=1, warmup=3, impl="reference", no_cpu_baseline=True, only=None)
    assert bench.run_reference(args, 2, 1) == 0  # returns at once, no oracle work, no output


def test_profile_traffic_is_keyed_to_code_not_comments():
    """The DRAM traffic a committed ncu summary reports is used only while the kernel sources
    hash the same, comments and blank lines aside: a comment edit keeps it, a code edit drops it."""
    import bench
    src = "int f(int x) {  // doubles\n\n    /* note */ return 2 * x;\n}\n"
    same = "// a header line\nint f(int x) {  // twice x\n    return 2 * x;   \n}\n"
    other = "int f(int x) {\n    return 3 * x;\n}\n"
    assert bench._code_only(src) == bench._code_only(same)
    assert bench._code_only(src) != bench._code_only(other)
    # every committed summary's traffic line still matches its kernels' sources
    for kind, workload in (("prefill", "chunked_prefill"), ("decode", "batched_decode"), ("splitkv", "splitkv_4x8192")):
        assert bench.profiled_traffic(kind, workload) is not None, (kind, workload)
