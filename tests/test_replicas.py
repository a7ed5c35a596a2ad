"""The N > 1 path of bench.py (one independent replica per rank, no data-path
collective) on two CPU ranks over gloo: the timed region's length is the
slowest rank's, the rate counts every rank's units, and the reference arm
prints on rank 0 only."""
import argparse
import multiprocessing
import os
import socket
import sys


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, times, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE="2")
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=2)
    try:
        t = bench.max_over_ranks(times[rank], 2, device="cpu")
        out.put((rank, t, bench.whole_job_rate(100.0, 2, t)))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_count_all_units():
    ctx = multiprocessing.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    times = [1.25, 4.0]
    procs = [ctx.Process(target=_rank_main, args=(r, port, times, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    codes = [p.exitcode for p in procs]
    for p in procs:
        if p.is_alive():
            p.kill()
    assert codes == [0, 0], codes
    res = sorted(out.get(timeout=10) for _ in range(2))
    assert [r[1] for r in res] == [4.0, 4.0]       # both ranks report the slowest
    assert [r[2] for r in res] == [50.0, 50.0]     # 2 ranks x 100 units / 4.0


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_rate(12.0, 1, 3.0) == 4.0


def test_reference_arm_prints_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.run_reference(argparse.Namespace(steps=1, warmup=3))
    assert capsys.readouterr().out == ""
