"""Multi-process (replicas) path of bench.py on the CPU: two gloo ranks exercise the rank-side
logic that a multi-GPU run uses -- the barrier, the max-over-ranks timing reduction, the sum
reduction, per-rank synthetic inputs and the whole-job rate. The decoder path has no exchange
step (each rank serves its own sequences), so there is no data-path collective to test."""

import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, out_dir: str) -> None:
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    import synth
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        mx = bench.reduce_max(10.0 * (rank + 1), world)  # per-rank elapsed ms
        sm = bench.reduce_sum(float(rank + 1), world)
        seed = bench.rank_token_seed(1, rank)
        toks = synth.make_tokens(synth.QWEN3_0_6B.vocab, 5, seed)
        np.save(os.path.join(out_dir, f"r{rank}.npy"), np.array([mx, sm, seed] + toks.tolist(), dtype=np.float64))
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_replica_logic(tmp_path):
    mp = pytest.importorskip("torch.multiprocessing")
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    r = [np.load(tmp_path / f"r{i}.npy") for i in range(world)]
    for x in r:
        assert x[0] == 20.0  # max over ranks
        assert x[1] == 3.0   # sum over ranks
    assert r[0][2] != r[1][2]  # each replica draws its own prompts
    assert not np.array_equal(r[0][3:], r[1][3:])


def test_whole_job_rate():
    sys.path.insert(0, ROOT)
    import bench
    # 2 ranks x 65 tokens per step x 10 steps in at most 500 ms -> 2600 tok/s for the job
    assert bench.whole_job_rate(65, 10, 2, 500.0) == pytest.approx(2600.0)
    assert bench.whole_job_rate(65, 10, 1, 500.0) == pytest.approx(1300.0)
