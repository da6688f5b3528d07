"""The N>1 host logic of bench.py on CPU: two gloo ranks in separate processes (no GPU).

bench.py runs one full replica per rank; the step shards by sequence with no exchange on the
data path. What crosses ranks is the timing: the job takes as long as its slowest rank, and
the reported rate is every rank's units over that time. The reference arm runs on rank 0
alone.
"""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, ms_of_rank, units, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out[rank] = bench.job_rate(ms_of_rank[rank], units, world, device="cpu")
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_rank_and_whole_job_units():
    torch = pytest.importorskip("torch")
    mp = torch.multiprocessing.get_context("spawn")
    world, units = 2, 32 * 8   # batch 32, 8 steps per rank
    ms_of_rank = [10.0, 12.5]
    with mp.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [mp.Process(target=_rank_main, args=(r, world, port, ms_of_rank, units, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
        res = dict(out)
    assert len(res) == world
    for r in range(world):
        ms, total, rate = res[r]
        assert ms == 12.5                      # max over ranks
        assert total == units * world          # whole-job units
        assert rate == pytest.approx(units * world / 0.0125)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_rate(4.0, 100, 1) == (4.0, 100, 100 / 0.004)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    import workloads as wl
    monkeypatch.setenv("RANK", "1")
    assert bench.run_reference(None, wl.W_GPT2XL_B256, wl.W_GPT2_BF16_PREFILL) == 0   # returns before any work
