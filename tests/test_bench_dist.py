"""Multi-rank plumbing of bench.py on CPU (gloo, world size 2): the barrier, the
maximum over ranks used for the timed region, the whole-job throughput, and
the reference arm's rank gating.  No GPU is used."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, w = bench.init_dist("gloo")
    bench.barrier()
    # each rank "measured" a different time; the job time is the slowest rank's
    m = bench.reduce_max(10.0 + 5.0 * r)
    thr = bench.aggregate_throughput(1000.0, w, m / 1e3)
    bench.barrier()
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(f"{r} {w} {m} {thr}\n")
    dist.destroy_process_group()


def test_reduce_max_and_throughput_two_ranks(tmp_path):
    import torch.multiprocessing as mp
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    rows = []
    for r in range(2):
        with open(tmp_path / f"rank{r}.txt") as f:
            rows.append(f.read().split())
    for r, row in enumerate(rows):
        rr, w, m, thr = int(row[0]), int(row[1]), float(row[2]), float(row[3])
        assert rr == r and w == 2
        assert m == pytest.approx(15.0)            # max over ranks, seen by every rank
        # 1000 units per rank, 2 ranks, over the slowest rank's 15 ms
        assert thr == pytest.approx(1000.0 * 2 / 0.015)


def test_single_process_helpers_without_process_group():
    import bench
    assert bench.reduce_max(3.25) == 3.25
    assert bench.aggregate_throughput(10.0, 1, 2.0) == 5.0
    bench.barrier()   # no process group: a no-op


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        gpus, steps, warmup, ref_budget = 2, 1, 3, 0.1

    assert bench.run_reference(A()) == 0
    assert capsys.readouterr().out == ""


def test_roofline_entry_per_launch_and_held_sm_rates():
    """The roofline object: FLOPs per launch over the average launch duration
    against the peak, plus the rate on the SMs the launches hold (device time x
    SM share)."""
    import bench
    agg = {"launches": 4, "ms": 0.4, "flops": 4.0e12 * 0.4e-3, "sm_ms": 0.1}
    r = bench.roofline_entry("no_such_kernel", agg, 2000.0, "test")
    assert r["kernel"] == "no_such_kernel" and r["bound"] == "tensor"
    assert abs(r["achieved"] - 4.0) < 1e-9               # 0.4 GFLOP per 0.1 ms launch
    assert abs(r["frac"] - 0.002) < 1e-12
    assert abs(r["avg_launch_us"] - 100.0) < 1e-9
    assert abs(r["avg_sm_share"] - 0.25) < 1e-12
    assert abs(r["achieved_on_held_sms"] - 16.0) < 1e-9  # same FLOPs over a quarter of the time
    assert r["traffic"] is None                           # no committed summary for it
