"""Host-side logic of bench.py that needs no GPU: the whole-job aggregation across ranks
(world size 2 over gloo on CPU), the clock-sample parsing and the argument contract."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist

    bench.init_dist(world, "gloo")
    bench.barrier(world)
    elapsed, units = bench.aggregate(1.0 + rank, 10.0 * (rank + 1), world)
    q.put((rank, elapsed, units))
    dist.destroy_process_group()


def test_aggregate_two_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    # max of elapsed over ranks, sum of units: whole-job throughput = 30 / 2
    assert got == [(0, 2.0, 30.0), (1, 2.0, 30.0)]


def test_aggregate_single_rank_is_identity():
    assert bench.aggregate(1.5, 7.0, 1) == (1.5, 7.0)


def test_clock_sampler_parsing():
    cs = bench.ClockSampler("0")

    class P:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            pass

    cs.proc = P()
    cs.skip = 1
    cs.lines = ["1900, 2070, 500.1, Not Active, Not Active, Not Active, Not Active",
                "1600, 2070, 1380.0, Not Active, Not Active, Not Active, Active",
                "1620, 2070, 1390.0, Not Active, Not Active, Not Active, Active",
                "1640, 2070, 1385.0, Not Active, Not Active, Not Active, Not Active"]
    out = cs.stop()
    assert out["sm_mhz"] == 1620.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"] and out["samples"] == 3


def test_cli_contract():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])      # the contract wants at least 3 warm-up steps
    with pytest.raises(SystemExit):
        bench.main(["--workload", "nope"])


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    # Under torchrun only rank 0 runs the CPU reference and prints its line; others return 0.
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"]) == 0
    assert capsys.readouterr().out.strip() == ""


def test_host_cpu_names_a_model_and_falls_back_without_lscpu(monkeypatch):
    import platform
    import subprocess

    assert bench.host_cpu().endswith(f"({platform.machine()})")

    def no_lscpu(*args, **kwargs):
        raise FileNotFoundError("lscpu")

    monkeypatch.setattr(subprocess, "run", no_lscpu)
    got = bench.host_cpu()  # /proc/cpuinfo, else "unknown"
    assert got.endswith(f"({platform.machine()})") and len(got) > len(platform.machine()) + 3


def test_single_thread_oracle_is_null_when_its_child_fails(monkeypatch):
    import subprocess

    class Done:
        stdout, stderr, returncode = "Traceback: no json here", "", 1

    monkeypatch.setattr(subprocess, "run", lambda *a, **k: Done())
    assert bench.single_thread_oracle() is None

    def timeout(*a, **k):
        raise subprocess.TimeoutExpired("python", 1.0)

    monkeypatch.setattr(subprocess, "run", timeout)
    assert bench.single_thread_oracle() is None
