"""Process-layout logic of bench.py on CPU (no GPU is used): a job on more
than one GPU is refused with one line from rank 0 and exit status 0 on every
rank, the reference arm runs on rank 0 only, and the roofline object's
arithmetic."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _run_rank(rank, world, extra):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
               MASTER_ADDR="127.0.0.1", MASTER_PORT="29555", CUDA_VISIBLE_DEVICES="")
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *extra], env=env,
                          capture_output=True, text=True, timeout=300, cwd=ROOT)


def test_two_rank_job_is_refused_on_every_rank():
    """Two ranks launched as torchrun would (RANK / WORLD_SIZE set): rank 0
    prints one refusal line, rank 1 prints nothing, both exit 0."""
    procs = [_run_rank(r, 2, ["--gpus", "2", "--steps", "2", "--warmup", "3"]) for r in (0, 1)]
    for p in procs:
        assert p.returncode == 0, p.stderr
    lines = [ln for ln in procs[0].stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["n_gpus"] == 2 and line["value"] is None
    assert "single-GPU" in line["unavailable"]
    assert procs[1].stdout.strip() == ""


def test_gpus_flag_alone_is_refused(monkeypatch):
    import bench
    monkeypatch.delenv("WORLD_SIZE", raising=False)

    class A:
        gpus, steps, warmup = 4, 1, 3

    r = bench.single_gpu_refusal(A())
    assert r is not None and r["n_gpus"] == 4
    A.gpus = 1
    assert bench.single_gpu_refusal(A()) is None


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        gpus, steps, warmup, ref_budget, workload = 2, 1, 3, 0.1, "lm760m"

    assert bench.run_reference(A()) == 0
    assert capsys.readouterr().out == ""


def test_reference_arm_line_on_rank_zero(monkeypatch, capsys):
    """Rank 0 of the reference arm prints one line with the oracle's rate
    (a tiny budget: one run of the sampled chunks)."""
    import bench
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")

    class A:
        gpus, steps, warmup, ref_budget, workload = 1, 1, 0, 0.01, "nvs-strided"

    assert bench.run_reference(A()) == 0
    line = json.loads(capsys.readouterr().out.strip())
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["config"]["update_chunks"] == [1, 1, 1, 1, 0, 0, 0, 0]
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_layer_flops_per_workload():
    """FLOP counts written out per workload: 18 b d m per chunk and head
    (12 for an update, 6 for an apply) plus Muon's s (4 r c^2 + 2 c^3) per
    matrix and update."""
    import bench
    import workloads as W
    assert bench.layer_flops(W.LM_760M) == pytest.approx(1.348082860032e12)
    # strided: 2 heads x (4 updates x 12 + 8 applies x 6) b d m
    assert bench.layer_flops(W.NVS_STRIDED) == pytest.approx(2 * 96 * 8192 * 384 * 768)
    assert bench.layer_flops(W.LONG_1M) == pytest.approx(25.98e12, rel=1e-3)


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
