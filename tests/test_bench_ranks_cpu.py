"""bench.py's multi-rank plumbing on CPU: two gloo ranks agree on the job's
time (the slowest rank's) and the whole-job throughput, and the reference
arm runs on rank 0 only."""

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        ms_max = bench.reduce_max_ms(times[rank], world, "cpu")
        q.put((rank, ms_max, bench.job_gbs(1000, 10, world, ms_max), bench.env_rank()))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    times = [2.5, 4.0]
    q = mp.get_context("spawn").SimpleQueue()   # a pipe: no files, no manager process
    mp.start_processes(_rank_main, args=(world, port, times, q), nprocs=world, join=True, start_method="spawn")
    res = {}
    while not q.empty():
        rank, ms_max, gbs, env = q.get()
        res[rank] = (ms_max, gbs, env)
    assert sorted(res) == [0, 1]
    for rank in range(world):
        ms_max, gbs, env = res[rank]
        assert ms_max == 4.0
        assert gbs == pytest.approx(1000 * 10 * world / 4.0e-3 / 1e9)
        assert env == (rank, rank, world)


def test_single_rank_is_local_time():
    assert bench.reduce_max_ms(3.25, 1, "cpu") == 3.25
    assert bench.job_gbs(2000, 4, 1, 2.0) == pytest.approx(2000 * 4 / 2.0e-3 / 1e9)


def test_reference_arm_runs_on_rank_0_only(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        steps, warmup, gpus = 1, 3, 2
    assert bench.run_reference(Args()) == 0   # returns before loading the oracle or timing anything


def test_reference_arm_prints_one_contract_line():
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, check=True, env=env, timeout=600)
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "GB/s"
    assert d["value"] > 0 and d["higher_is_better"] is True and d["steps"] == 1 and d["warmup"] == 3
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == bench.WORKLOAD
