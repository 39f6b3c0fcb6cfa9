"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): the timed
region's max-over-ranks reduction and barrier, the whole-job throughput, and the
reference arm printing on rank 0 only."""
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, secs, out_path):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist()
    d.init("gloo")
    d.barrier()
    slowest = d.max(secs[rank])
    value = bench.whole_job_throughput(d.world, 8192, 10, slowest)
    d.barrier()
    with open("%s.%d" % (out_path, rank), "w") as f:
        f.write("%r %r\n" % (slowest, value))
    d.close()


def test_max_over_ranks_and_throughput(tmp_path):
    import torch.multiprocessing as mp
    world, port = 2, _free_port()
    secs = [0.25, 0.5]
    out = str(tmp_path / "r")
    mp.start_processes(_rank_main, args=(world, port, secs, out), nprocs=world, join=True, start_method="spawn")
    for r in range(world):
        slowest, value = map(float, open("%s.%d" % (out, r)).read().split())
        assert slowest == 0.5
        assert value == pytest.approx(world * 8192 * 10 / 0.5)


def test_whole_job_throughput_is_weak_scaling():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.whole_job_throughput(1, 100.0, 4, 2.0)
    two = bench.whole_job_throughput(2, 100.0, 4, 2.0)
    assert one == 200.0 and two == 2 * one


def test_reference_arm_prints_on_rank_zero_only():
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2", MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
