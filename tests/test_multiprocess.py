"""Host logic of the N > 1 bench path on CPU: two gloo ranks.

The step shards by request with no data exchange (independent replicas), so
the only cross-rank operations are the barrier around the timed region and
the max over ranks of the step time; the job value is the sum over replicas.
"""
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, local = bench.dist_setup(None)
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(w)
    step_ms = [0.25, 0.40][rank]             # rank 1 is the slow replica
    ms_max = bench.max_over_ranks(step_ms, w)
    value = bench.replica_value(128, w, ms_max)
    bench.barrier(w)
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(f"{ms_max} {value}")
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_step(tmp_path):
    port = _free_port()
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    got = [open(tmp_path / f"rank{r}.txt").read().split() for r in range(2)]
    for ms_max, value in got:
        assert float(ms_max) == 0.40
        assert float(value) == pytest.approx(2 * 128 / 0.40e-3)


def test_replica_value_is_weak_scaling_sum():
    one = bench.replica_value(128, 1, 0.2)
    assert bench.replica_value(128, 4, 0.2) == pytest.approx(4 * one)
    assert bench.replica_value(128, 2, 0.4) == pytest.approx(one)


def test_reference_arm_non_zero_rank_exits_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "1"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
