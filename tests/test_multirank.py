"""Host-side logic of bench.py's multi-rank (replicas) path on two gloo ranks, CPU only.

The path has no data exchange: under torchrun every rank runs an independent
replica of the workload, the step time is the maximum over ranks and the
whole-job rate counts every rank's query tokens.  These tests run that
reduction on two processes with the gloo backend (rendezvous on 127.0.0.1),
and check that a non-zero rank of the reference arm exits without work.
"""

import json
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # every rank measured a different time; all of them must see the largest
        ms = bench.max_over_ranks(10.0 + 3.0 * rank, world, device="cpu")
        rate = bench.whole_job_rate(256, world, 20, ms)
        # the reference arm: ranks other than 0 return at once (rank 0 is not run here)
        ran_reference = None
        if rank != 0:
            args = type("A", (), dict(workload=1, steps=1, warmup=0))()
            bench.run_reference(args)
            ran_reference = "returned"
        dist.barrier()
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"ms": ms, "rate": rate, "env": list(bench.dist_env()), "reference": ran_reference}, f)
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_gloo_ranks_take_max_time_and_sum_tokens(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    expect_ms = 13.0  # max(10, 13)
    for r, d in enumerate(res):
        assert d["ms"] == pytest.approx(expect_ms)
        # 2 ranks x 256 query tokens x 20 steps in 13 ms
        assert d["rate"] == pytest.approx(2 * 256 * 20 / 13e-3)
        assert d["env"] == [r, r, world]
    assert res[1]["reference"] == "returned"


def test_single_rank_reduction_is_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(7.5, 1) == 7.5
    assert bench.whole_job_rate(100, 1, 4, 2.0) == pytest.approx(100 * 4 / 2e-3)
