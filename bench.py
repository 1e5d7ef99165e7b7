#!/usr/bin/env python
"""Benchmark: TTT-KVB (LaCT) layer forward tokens/s on GB300 and the share of
the dense-BF16 tensor-core peak it reaches.

Workload: the 760M-scale language-model layer (d = 1536, 4 TTT heads):
B = 2, H = 4, d_h = m_h = 384, N = 32768 tokens, chunk 2048, apply-then-update
mask, momentum beta = 0.9, Muon with 5 Newton-Schulz steps, L2-Normalize,
bf16 q/k/v (L2-normed keys), fp32 fast weights; seeded synthetic inputs from
``workloads.py``.  One step is one full ``ttt_layer_forward`` call over the
sequence (every chunk: projections + gating, weight gradients, momentum,
Muon, normalisation, apply).

Under torchrun with N ranks every rank runs its own copy of the workload on
its own GPU (weak scaling, no collective on the data path); rank 0 prints one
JSON line.  ``--impl reference`` times the fp64 CPU oracle instead, on a
bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "TTT-layer fwd tokens/sec on 1 GB300; % of dense BF16 tensor-core peak"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---------------------------------------------------------------------------
# distributed plumbing (weak scaling: each rank runs its own workload copy)

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def init_dist(backend: str):
    import torch.distributed as dist
    rank, world, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return rank, world


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def reduce_max(x: float, device=None) -> float:
    """Maximum of x over ranks (x itself on one rank)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Whole-job throughput: the units every rank processed over the slowest rank's time."""
    return units_per_rank * world / max_seconds


# ---------------------------------------------------------------------------
# GPU clocks during the timed region

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index=None):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if self.gpu_index is not None:
            cmd += ["-i", str(self.gpu_index)]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [s for s, p in zip(sm, power) if p > 0.25 * max(power)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power)}


# ---------------------------------------------------------------------------
# algorithmic work of the workload

def layer_flops(wl) -> float:
    """18 b d m per chunk and head for update + apply (f_W(k) is not needed
    under the dot-product loss), plus Muon's s (4 r c^2 + 2 c^3) per matrix
    (r = max(d, m), c = min(d, m)) on every update."""
    nc = wl.N // wl.chunk
    n_upd = nc if wl.update_chunks is None else sum(1 for x in wl.update_chunks if x)
    d, m, b = wl.d_h, wl.m_h, wl.chunk
    r, c = max(d, m), min(d, m)
    per_head = n_upd * 12 * b * d * m + nc * 6 * b * d * m
    per_head += n_upd * wl.muon_steps * 3 * (4 * r * c * c + 2 * c ** 3)
    return float(per_head * wl.B * wl.H)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def cpu_cores() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n and n[0]:
            return int(n[0])
    except Exception:
        pass
    return os.cpu_count() or 1


# ---------------------------------------------------------------------------
# the oracle on a bounded sample (CPU baseline / reference arm)

def oracle_sample(wl, inputs, budget_s: float = 12.0, chunks_per_run: int = 2):
    """Runs the fp64 oracle, as it stands, on the first ``chunks_per_run``
    chunks of one (batch, head) sequence after another until about
    ``budget_s`` seconds have passed.  Every chunk does the same work, so the
    rate extrapolates to the whole workload.  Returns (layer tokens/s, sample
    description, seconds)."""
    from oracle import ttt_oracle as O
    q, k, v, eta, W1, W2, W3 = inputs
    n = min(chunks_per_run, wl.N // wl.chunk)
    sl = slice(0, n * wl.chunk)
    runs, elapsed = 0, 0.0
    pairs = [(b, h) for b in range(wl.B) for h in range(wl.H)]
    while elapsed < budget_s:
        b, h = pairs[runs % len(pairs)]
        x = [t[b:b + 1, h:h + 1, sl].double().numpy() for t in (q, k, v)]
        e = eta[b:b + 1, h:h + 1, sl].double().numpy()
        w = [t[h:h + 1].double().numpy() for t in (W1, W2, W3)]
        ts = time.perf_counter()
        O.ttt_layer_forward(*x, e, *w, wl.chunk, wl.mode, l2norm=wl.l2norm,
                            muon_steps=wl.muon_steps, momentum_beta=wl.momentum_beta)
        elapsed += time.perf_counter() - ts
        runs += 1
    head_tokens = runs * n * wl.chunk
    rate = head_tokens / elapsed / wl.H   # every layer token costs H head-tokens
    desc = (f"fp64 oracle on the first {n} chunks of {runs} (batch, head) sequences of the "
            f"workload ({head_tokens} head-tokens in {elapsed:.1f} s); layer tokens/s = "
            f"head-tokens/s / H")
    return rate, desc, elapsed


# ---------------------------------------------------------------------------

def run_reference(args):
    """Reference arm: the fp64 CPU oracle, as it stands, on the machine's cores."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import workloads
    wl = workloads.LM_760M
    inputs = workloads.layer_inputs(wl)
    per_step = []
    for _ in range(args.warmup):
        oracle_sample(wl, inputs, budget_s=1.0)
    for _ in range(args.steps):
        rate, desc, el = oracle_sample(wl, inputs, budget_s=args.ref_budget)
        per_step.append(rate)
    value = statistics.median(per_step)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": wl.B * wl.N / value * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "B": wl.B, "H": wl.H, "N": wl.N, "d_h": wl.d_h,
                   "m_h": wl.m_h, "chunk": wl.chunk, "mask": "apply-then-update",
                   "muon_steps": wl.muon_steps, "momentum_beta": wl.momentum_beta,
                   "l2norm": wl.l2norm, "parallelism": "replicas"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# kernel -> (ncu summary under profiles/, sources whose hash the summary records)
KERNEL_PROFILE = {
    "ns_half_kernel": ("profiles/ns_half_kernel_lm760m.md",
                       ("chunked_linear_attention_gb300/csrc/ns_half.cu",
                        "chunked_linear_attention_gb300/csrc/common.cuh")),
    "ns_panel_kernel": ("profiles/ns_panel_kernel_lm760m.md",
                        ("chunked_linear_attention_gb300/csrc/ns_panel.cu",
                         "chunked_linear_attention_gb300/csrc/common.cuh")),
    "umma_gemm_kernel": ("profiles/umma_gemm_kernel_lm760m.md",
                         ("chunked_linear_attention_gb300/csrc/gemm_umma.cu",
                          "chunked_linear_attention_gb300/csrc/umma_core.cuh",
                          "chunked_linear_attention_gb300/csrc/tc_epilogue.cuh",
                          "chunked_linear_attention_gb300/csrc/common.cuh")),
}


def source_hash(paths):
    import hashlib
    h = hashlib.sha256()
    for rel in paths:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel):
    """DRAM bytes per launch from the committed ncu summary of `kernel`, or None
    when there is none or the kernel's sources changed since it was taken."""
    entry = KERNEL_PROFILE.get(kernel)
    if not entry:
        return None, None
    path = os.path.join(ROOT, entry[0])
    if not os.path.exists(path):
        return None, None
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line and line.strip().startswith("- "):
                k_, v_ = line.strip()[2:].split(":", 1)
                vals[k_.strip()] = v_.strip().strip("`")
    if vals.get("source_hash") != source_hash(entry[1]):
        return None, entry[0]
    try:
        return float(vals["dram_bytes_per_launch"]), entry[0]
    except (KeyError, ValueError):
        return None, entry[0]


def roofline_entry(name, agg, peak, peak_src):
    """Roofline of the dominant kernel: algorithmic FLOPs per launch over its
    average launch duration (CUDA events on its own stream, profiled step)."""
    n = max(agg["launches"], 1)
    avg_ms = agg["ms"] / n
    fl = agg["flops"] / n
    achieved = fl / (avg_ms / 1e3) / 1e12 if avg_ms > 0 else None
    traffic, src = recorded_traffic(name)
    share = agg["sm_ms"] / agg["ms"] if agg.get("ms") else None
    return {"bound": "tensor", "kernel": name, "achieved": achieved, "peak": peak,
            "unit": "TFLOP/s", "frac": achieved / peak if achieved and peak else None,
            "peak_kind": f"bf16 sustained ({peak_src}): the kernel runs inside a long step",
            "traffic": traffic, "traffic_unit": "bytes per launch (ncu dram read + write)",
            "traffic_source": src, "launches_per_step": agg["launches"],
            "flops_per_launch": fl, "avg_launch_us": avg_ms * 1e3,
            "dominance": "most GPU time: device time x fraction of SMs the grid holds",
            "gpu_ms_per_step": agg.get("sm_ms"), "avg_sm_share": share,
            "achieved_on_held_sms": (agg["flops"] / (agg["sm_ms"] / 1e3) / 1e12
                                     if agg.get("sm_ms") else None),
            "achieved_on_held_sms_note": "FLOPs over device time x SM share: the rate on the "
                                         "SMs the launches hold, scaled to the whole GPU"}


def time_steps(torch, fn, steps, warmup, stream):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    return e0.elapsed_time(e1)


def run_ours(args):
    import torch
    import chunked_linear_attention_gb300 as cla
    import workloads
    from chunked_linear_attention_gb300 import _build

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist("nccl")
    _build.build()
    cla.library()

    wl = workloads.LM_760M
    if args.seq_len:
        wl = dataclasses.replace(wl, N=args.seq_len)
    B, H, N, d, m, b = wl.B, wl.H, wl.N, wl.d_h, wl.m_h, wl.chunk
    host = workloads.layer_inputs(wl, seed=wl.seed + rank)
    pinned = [t.pin_memory() for t in host]
    q, k, v, eta, W1, W2, W3 = [t.to(dev) for t in pinned]
    rule = cla.update_rule(l2norm=wl.l2norm, muon_steps=wl.muon_steps,
                           momentum_beta=wl.momentum_beta)
    out = torch.empty_like(q)
    Wf = (torch.empty((B, H, m, d), device=dev), torch.empty((B, H, d, m), device=dev),
          torch.empty((B, H, m, d), device=dev))
    ws = torch.empty(cla.layer_workspace_size(B, H, N, d, m, b, cla.TTT_BF16, wl.mode, rule),
                     device=dev, dtype=torch.uint8)
    stream = torch.cuda.current_stream(dev)

    def step():
        cla.ttt_layer_forward(q, k, v, eta, W1, W2, W3, b, wl.mode, rule, out=out, W_final=Wf,
                              workspace=ws)

    # device-resident timing, clocks sampled during the timed region
    clocks = ClockSampler(gpu_index=None if world > 1 else local)
    step()
    torch.cuda.synchronize()
    st = cla.device_status()
    if st != 0:
        raise RuntimeError(f"device status {st}: {cla.status_string(st)}")
    launches0 = cla.launch_count()
    clocks.start()
    ms = time_steps(torch, step, args.steps, args.warmup, stream)
    clk = clocks.stop()
    launches = (cla.launch_count() - launches0) // (args.steps + args.warmup) * args.steps
    max_ms = reduce_max(ms, dev)
    ms_step = max_ms / args.steps
    tokens = B * N
    value = aggregate_throughput(tokens * args.steps, world, max_ms / 1e3)

    # end to end through the public host-buffer call: page-locked inputs in,
    # outputs and final weights back in page-locked host memory; the library
    # overlaps each chunk's transfers with the kernels
    h_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    h_W = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in Wf]
    hq, hk, hv, heta, hW1, hW2, hW3 = pinned
    ws_host = torch.empty(cla.layer_host_workspace_size(B, H, N, d, m, b, cla.TTT_BF16, wl.mode,
                                                        rule), device=dev, dtype=torch.uint8)

    def e2e_step():
        cla.ttt_layer_forward_host(hq, hk, hv, heta, hW1, hW2, hW3, b, wl.mode, rule, out=h_out,
                                   W_final=h_W, workspace=ws_host)

    e2e_steps = max(1, min(args.steps, 10))
    ms_e2e = time_steps(torch, e2e_step, e2e_steps, 1, stream)
    max_e2e = reduce_max(ms_e2e, dev)
    e2e_value = aggregate_throughput(tokens * e2e_steps, world, max_e2e / 1e3)
    h2d = sum(t.numel() * t.element_size() for t in pinned)
    d2h = h_out.numel() * h_out.element_size() + sum(t.numel() * t.element_size() for t in h_W)

    # per-launch profile of one more step (CUDA events around every launch)
    cla.profile_start()
    step()
    prof = cla.profile_stop()
    tc_kernels = ("umma_gemm_kernel", "ns_cluster_kernel", "ns_panel_kernel", "ns_half_kernel")
    gemm = [p for p in prof if p["kernel"] in tc_kernels]
    g_fl = sum(p["flops"] for p in gemm)
    g_n = sum(p["launches"] for p in gemm)
    # The dominant kernel: most GPU time in the profiled step, counted as each
    # launch's device time x the fraction of the SMs its grid holds (launches
    # of the stream groups and the apply streams run side by side, several of
    # them on a part of the GPU).
    per_kernel = {}
    for p in gemm:
        k_ = per_kernel.setdefault(p["kernel"], {"launches": 0, "ms": 0.0, "flops": 0.0,
                                                 "sm_ms": 0.0})
        k_["launches"] += p["launches"]
        k_["ms"] += p["ms"]
        k_["flops"] += p["flops"]
        k_["sm_ms"] += p.get("sm_ms", p["ms"])
    dom_name, dom = max(per_kernel.items(), key=lambda kv: kv[1]["sm_ms"])
    peaks, peak_src = load_peaks()
    peak_sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    peak_burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    flops_step = layer_flops(wl)
    step_tflops = flops_step / (ms_step / 1e3) / 1e12
    # Launches of different (batch, head) sequences overlap on separate
    # streams, so per-launch durations do not add up to the step: the
    # tensor-core kernels' achieved rate is their algorithmic FLOPs (which
    # are all of the step's FLOPs) over the timed step.
    achieved = g_fl / (ms_step / 1e3) / 1e12

    # chunked linear attention (the linear-fast-weight reduction), HBM-bound
    lin = None
    if rank == 0 and not args.skip_linattn:
        lw = workloads.LINATTN_C2
        lq, lk, lv, leta, _ = [t.to(dev) if t is not None else None
                               for t in workloads.linattn_inputs(lw)]
        lo = torch.empty_like(lq)
        lS = torch.empty((lw.B, lw.H, lw.d_v, lw.d_k), device=dev)
        lws = torch.empty(cla.linattn_workspace_size(lw.B, lw.H, lw.N, lw.d_k, lw.d_v, lw.chunk,
                                                     cla.TTT_BF16, lw.mode),
                          device=dev, dtype=torch.uint8)
        lstep = lambda: cla.linattn_chunked_forward(lq, lk, lv, leta, lw.chunk, lw.mode, out=lo,
                                                    S_final=lS, workspace=lws)
        flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
        tot = 0.0
        reps = 20
        for i in range(reps + 3):
            flush.zero_()    # evict the inputs from L2 between repetitions
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            lstep()
            e1.record(stream)
            torch.cuda.synchronize()
            if i >= 3:
                tot += e0.elapsed_time(e1)
        lms = tot / reps
        io_bytes = (3 * lq.numel() * 2 + leta.numel() * 4 + lo.numel() * 2)
        hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        lin = {"workload": lw.name, "us_per_call": lms * 1e3,
               "tokens_per_s": lw.B * lw.N / (lms / 1e3),
               "gbs": io_bytes / (lms / 1e3) / 1e9, "hbm_frac": io_bytes / (lms / 1e3) / 1e9 / hbm,
               "io_bytes": io_bytes, "l2": "flushed (256 MB write) before each call"}

    cpu = None
    if rank == 0 and not args.skip_cpu_baseline:
        rate, desc, _ = oracle_sample(wl, host, budget_s=args.ref_budget)
        cpu = {"value": rate, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
               "sample": desc}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": wl.name, "B": B, "H": H, "N": N, "d_h": d, "m_h": m,
                       "chunk": b, "mask": "apply-then-update", "muon_steps": wl.muon_steps,
                       "momentum_beta": wl.momentum_beta, "l2norm": wl.l2norm,
                       "io": "bf16 q/k/v, fp32 eta and fast weights",
                       "l2": "inputs larger than L2 (q, k, v: %.0f MB per step)"
                             % (3 * q.numel() * 2 / 1e6),
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "pct_bf16_peak": {"step_tflops": step_tflops, "frac_of_burst": step_tflops / peak_burst,
                              "frac_of_sustained": step_tflops / peak_sus,
                              "flops_per_step": flops_step, "peaks": peak_src},
            "roofline": roofline_entry(dom_name, dom, peak_sus, peak_src),
            "tensor_kernels": {"launches_per_step": g_n, "flops_per_step": g_fl,
                               "achieved_tflops_over_step": achieved,
                               "note": "all tensor-core launches' algorithmic FLOPs over the "
                                       "step time (stream groups overlap)"},
            "breakdown_note": "summed launch durations of one profiled step; launches of "
                              "different sequences overlap, so sums exceed the step time",
            "breakdown": {p["name"]: {"launches": p["launches"], "ms": p["ms"],
                                      "gpu_ms": p.get("sm_ms"),
                                      "tflops": p["flops"] / (p["ms"] / 1e3) / 1e12
                                      if p["flops"] and p["ms"] else None,
                                      "gbs": p["bytes"] / (p["ms"] / 1e3) / 1e9
                                      if p["bytes"] and p["ms"] else None}
                          for p in prof},
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": max_e2e / e2e_steps},
            "cpu_baseline": cpu,
            "gpu_launches": launches,
            "clocks": clk,
            "linattn": lin,
        }
        print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--ref-budget", type=float, default=12.0,
                    help="seconds of oracle work per CPU-baseline sample")
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--skip-linattn", action="store_true")
    ap.add_argument("--seq-len", type=int, default=None,
                    help="override the workload's sequence length (small profiling cases)")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)   # timing rule: at least 3 warm-up steps
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
