"""The multi-process benchmark path on the CPU: two gloo ranks on 127.0.0.1.

The linear does not shard across GPUs here: under torchrun every rank runs its
own replica of the step, with no data-path collective.  What N > 1 adds is
host logic, tested here without a GPU:
* the rank bookkeeping, the barrier and the max-over-ranks of the timed region
  (every rank must see the slowest rank's time);
* the whole-job value: N replicas, each doing a fixed amount of work, timed at
  the slowest rank;
* the reference arm runs on rank 0 only: other ranks exit at once, print
  nothing and do no work.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir, times):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist("gloo")
    d.barrier()
    slowest = d.max(times[rank])
    d.barrier()
    res = {"rank": d.rank, "world": d.world, "on": d.on, "max": slowest}
    d.close()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump(res, f)


def test_two_gloo_ranks_agree_on_the_slowest_time(tmp_path):
    world, times = 2, [1.5, 7.25]
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path), times), nprocs=world,
                       start_method="spawn", join=True)
    for r in range(world):
        res = json.load(open(tmp_path / f"rank{r}.json"))
        assert res == {"rank": r, "world": world, "on": True, "max": max(times)}


def test_single_process_needs_no_process_group(monkeypatch):
    for k in ("RANK", "LOCAL_RANK", "WORLD_SIZE"):
        monkeypatch.delenv(k, raising=False)
    import bench
    d = bench.Dist("gloo")
    assert not d.on and d.world == 1 and d.rank == 0
    assert d.max(3.0) == 3.0
    d.barrier()
    d.close()


def test_whole_job_value_counts_every_replica():
    import bench
    one = bench.replica_gbs(4.0e9, 10, 1, 20.0)
    assert one == pytest.approx(4.0e9 * 10 / 0.020 / 1e9)
    # weak scaling: twice the replicas at the same (slowest-rank) time is twice the whole-job throughput
    assert bench.replica_gbs(4.0e9, 10, 2, 20.0) == pytest.approx(2 * one)
    # a slower rank lowers the whole job's number
    assert bench.replica_gbs(4.0e9, 10, 2, 40.0) == pytest.approx(one)


def test_reference_arm_is_rank_zero_only():
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2", MASTER_ADDR="127.0.0.1", MASTER_PORT="29599")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
