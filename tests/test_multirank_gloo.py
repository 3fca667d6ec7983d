"""The bench's multi-rank path on CPU: two gloo ranks, replicas only.

Each rank runs its own replica (its own seeded batch); the job's rate is the
units all ranks processed over the slowest rank's time, taken with a MAX
all-reduce. No collective is part of the attention path itself.
"""

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    from paged_kv_cache_hkv_gb300 import synth

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 10.0 + 5.0 * rank  # rank 1 is the slowest
        slowest = bench.max_over_ranks(local_ms, dist)
        step = synth.mixed_step(seed=bench.replica_seed(3, rank), num_decodes=16,
                                materialize=False)
        rate = bench.whole_job_rate(step.num_tokens, world, slowest)
        lens = ",".join(str(int(x)) for x in step.seq_lens)
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(f"{slowest}\n{rate}\n{lens}\n")
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_rank(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    r0 = open(tmp_path / "rank0.txt").read().split("\n")
    r1 = open(tmp_path / "rank1.txt").read().split("\n")
    assert float(r0[0]) == float(r1[0]) == 15.0  # max over ranks
    assert float(r0[1]) == float(r1[1])
    tokens = 512 + 8 * 64 + 16
    assert abs(float(r0[1]) - tokens * 2 / 15e-3) < 1e-6
    assert r0[2] != r1[2]  # each replica has its own batch


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_rate(100, 1, 2.0) == 50000.0
