"""The bench's across-rank logic on the CPU with two gloo ranks: the job's time
is the slowest rank's, its units are every rank's together, and the
reference arm runs on rank 0 only."""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=2)
    import bench
    cpu = torch.device("cpu")
    ms = bench.slowest_rank_ms(10.0 + 5.0 * rank, cpu)
    units = bench.job_units(100 + rank, cpu)
    q.put((rank, ms, units))
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_all_units():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for _, ms, units in got:
        assert ms == 15.0 and units == 201


def test_one_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.slowest_rank_ms(7.5, torch.device("cpu")) == 7.5
    assert bench.job_units(42, torch.device("cpu")) == 42


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference"])
    assert bench.run_reference(bench.parse()) is None
    assert capsys.readouterr().out == ""


def test_oracle_single_thread_leg():
    # the CPU leg's one-core sample runs one request at one thread and leaves
    # the oracle's thread count as it found it
    sys.path.insert(0, ROOT)
    import bench
    import oracle
    from speculative_decoding_02_gb300 import workloads as wl
    w = wl.WORKLOADS["tiny"]
    _, hs = bench.host_sample(w, 2, "cpu")
    thr = oracle.num_threads()
    st = bench.single_thread_sample(w, hs)
    assert oracle.num_threads() == thr
    assert st["cores"] == 1 and st["unit"] == bench.UNIT and st["value"] >= 0
    assert "1 of 2 requests" in st["sample"]
