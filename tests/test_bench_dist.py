"""Host logic of bench.py on CPU: the multi-rank timed region (gloo, world size
2: max-over-ranks reduction and barrier), the whole-job throughput, the
reference arm printing on rank 0 only, the clock record's sample selection, and
the guard that keeps a profile's DRAM traffic only while its sources match."""
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


def test_clock_sampler_uses_samples_inside_the_timed_window():
    import datetime
    sys.path.insert(0, ROOT)
    import bench
    t0 = datetime.datetime(2026, 1, 2, 3, 4, 5)

    def row(dt_ms, sm, reasons=("Not Active",) * 4):
        stamp = (t0 + datetime.timedelta(milliseconds=dt_ms)).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        return ", ".join([stamp, "0", str(sm), "2070", "300.0", "0x0"] + list(reasons))

    text = "\n".join([row(0, 1200), row(20, 2070), row(40, 2055),
                      row(60, 1800, ("Not Active", "Not Active", "Not Active", "Active"))])
    window = ((t0 + datetime.timedelta(milliseconds=10)).timestamp(),
              (t0 + datetime.timedelta(milliseconds=45)).timestamp())
    c = bench.ClockSampler.summarise(text, window, 20)
    assert c["samples"] == 4 and c["samples_in_timed_region"] == 2
    assert c["sm_mhz"] == (2070 + 2055) / 2 and c["sm_max_mhz"] == 2070
    assert c["reasons"] == ["sw_power_cap"]
    # no sample inside the window: the median of all samples
    c = bench.ClockSampler.summarise(text, (0.0, 1.0), 20)
    assert c["samples_in_timed_region"] == 0 and c["sm_mhz"] == (1800 + 2055) / 2


def test_profile_traffic_only_while_the_source_matches(tmp_path, monkeypatch):
    """roofline.traffic comes from a committed ncu summary only while the SHA-256 of
    the kernel sources it names still matches: a changed source gives None."""
    import hashlib
    sys.path.insert(0, ROOT)
    import bench
    (tmp_path / "profiles").mkdir()
    (tmp_path / "k").mkdir()
    src_a, src_b = tmp_path / "k" / "a.cu", tmp_path / "k" / "b.cuh"
    src_a.write_bytes(b"kernel a\n")
    src_b.write_bytes(b"header b\n")
    sha = hashlib.sha256(src_a.read_bytes() + src_b.read_bytes()).hexdigest()
    (tmp_path / "profiles" / "demo.md").write_text(
        "# demo\n\ntraffic_bytes_per_launch: 12345\nsource_file: k/a.cu, k/b.cuh\nsource_sha256: %s\n" % sha)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.ncu_traffic("demo") == 12345
    assert bench.ncu_traffic("missing") is None
    src_b.write_bytes(b"header b, changed\n")
    assert bench.ncu_traffic("demo") is None
