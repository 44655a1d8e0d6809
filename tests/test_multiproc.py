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


class _Ev:
    """Stand-in for a CUDA event: elapsed_time in ms between two recorded times."""

    def __init__(self, t_ms):
        self.t = t_ms

    def elapsed_time(self, other):
        return other.t - self.t


def test_step_stats_median_and_nearest_rank_p95():
    import bench
    # 20 intervals: 18 of 0.5 ms, one of 0.4 ms, one of 2.0 ms
    times = [0.0]
    for d in [0.5] * 9 + [0.4] + [0.5] * 9 + [2.0]:
        times.append(times[-1] + d)
    st = bench.step_stats([_Ev(t) for t in times])
    assert st["n"] == 20
    assert st["median_us"] == pytest.approx(500.0)
    assert st["p95_us"] == pytest.approx(500.0)  # nearest rank 19 of 20: the outlier is the 20th
    times.append(times[-1] + 3.0)  # a 21st interval: rank ceil(0.95 * 21) = 20 -> 2.0 ms
    assert bench.step_stats([_Ev(t) for t in times])["p95_us"] == pytest.approx(2000.0)


def test_ncu_traffic_needs_the_captured_source():
    import bench
    # every entry names a tracked source; an unknown kernel or a stale hash gives no traffic
    for (cfg, kernel), (nbytes, src, sha) in bench.NCU_TRAFFIC.items():
        assert nbytes > 0 and len(sha) == 64
    assert bench.ncu_traffic(1, "no such kernel") is None
    key = next(iter(bench.NCU_TRAFFIC))
    saved = bench.NCU_TRAFFIC[key]
    try:
        bench.NCU_TRAFFIC[key] = (saved[0], saved[1], "0" * 64)
        assert bench.ncu_traffic(*key) is None
    finally:
        bench.NCU_TRAFFIC[key] = saved


def test_gpus_flag_spawns_replica_processes():
    """`bench.py --gpus 2` without a launcher re-runs itself as two processes under
    torch.distributed.run (127.0.0.1). Checked with the reference arm, which needs no GPU:
    rank 0 alone runs the oracle and prints the one line, the other rank exits 0."""
    import json
    import subprocess
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR",
                                                             "MASTER_PORT")}
    env["OMP_NUM_THREADS"] = "2"
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--impl", "reference",
                        "--config", "0", "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, timeout=900, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    out = json.loads(lines[0])
    assert out["impl"] == "reference" and out["n_gpus"] == 2 and out["value"] > 0


def test_replica_command():
    sys.path.insert(0, ROOT)
    import bench
    cmd = bench.replica_command(4, ["--steps", "5"])
    assert cmd[1:3] == ["-m", "torch.distributed.run"]
    assert "--nproc-per-node=4" in cmd and "--master-addr=127.0.0.1" in cmd
    assert cmd[-3:] == [os.path.join(ROOT, "bench.py"), "--steps", "5"]
