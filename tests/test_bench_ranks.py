"""Host-side logic of bench.py's multi-rank path, on CPU: two gloo ranks
agree on the slowest rank's time and on the whole-job rate, and the
reference arm prints nothing on ranks other than 0."""
import json
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
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank, world_size=world)
    try:
        # rank r "took" 10 + 5 r ms per step over 4 steps
        total = bench.max_over_ranks(4 * (10.0 + 5.0 * rank), world)
        ms = total / 4
        rate = bench.whole_job_rate(1e9, ms, world, 1e9)
        with open(os.path.join(out_dir, "r%d.json" % rank), "w") as f:
            json.dump({"ms": ms, "rate": rate}, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(tmp_path / ("r%d.json" % r))) for r in range(world)]
    for r in res:
        assert r["ms"] == pytest.approx(15.0)          # the slower rank's 15 ms per step
        assert r["rate"] == pytest.approx(2 * 1.0 / 15e-3)  # 2 replicas x 1 GB per 15 ms


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_rate(2e12, 10.0, 1, 1e12) == pytest.approx(200.0)


def test_reference_arm_is_silent_on_other_ranks():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
