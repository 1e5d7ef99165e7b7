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

The same line carries the view-synthesis strided workload (B1 H2 d384
m768, 8 chunks of 8192, update on chunks 0-3) and the million-token context
(B1 H4 d=m=512, N = 1,048,576, chunk 8192, Muon 5) under "workloads";
``--workload`` makes either of them the headline instead.

The library is single-GPU: the layer runs on one GPU without sharding
(the (batch, head) sequences shard only as independent replicas, and no
replica mode is provided).  A launch on
more than one GPU (``--gpus N`` with N > 1, or torchrun with WORLD_SIZE > 1)
prints one line saying so and exits 0 without touching a GPU.
``--impl reference`` times the fp64 CPU oracle instead, on a bounded sample of
the same workload (rank 0 only under torchrun).
"""
from __future__ import annotations

import argparse
import dataclasses
import json
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
# process layout: one process, one GPU

def dist_env():
    """(rank, world size, local rank) from the launcher's environment."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def single_gpu_refusal(args):
    """The line printed instead of a measurement when the job spans more than
    one GPU (None when it does not)."""
    _, world, _ = dist_env()
    n = max(world, args.gpus)
    if n <= 1:
        return None
    return {"metric": METRIC, "value": None, "unit": UNIT, "n_gpus": n, "steps": args.steps,
            "warmup": args.warmup, "higher_is_better": True,
            "unavailable": "single-GPU build: the layer runs on one GPU without sharding; its "
                           "(batch, head) sequences shard only as independent replicas and no "
                           "replica mode is provided"}


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
               "-lms", "25"]
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

def oracle_sample(wl, budget_s: float = 12.0, max_chunks: int = 2):
    """Runs the fp64 oracle, as it stands, on one (batch, head) sequence after
    another until about ``budget_s`` seconds have passed, each run covering
    the first ``max_chunks`` chunks of the workload (every chunk of a
    strided workload, whose chunks differ in work).  The inputs are drawn
    with the workload's recipe at the sampled length.  Every sampled run
    does the work of the same chunks, so the rate extrapolates to the whole
    workload.  Returns (layer tokens/s, sample description, seconds)."""
    import workloads
    from oracle import ttt_oracle as O
    nc = wl.N // wl.chunk
    n = nc if wl.update_chunks is not None else min(max_chunks, nc)
    q, k, v, eta, W1, W2, W3 = workloads.layer_inputs(wl, B=1, H=1, N=n * wl.chunk)
    x = [t.double().numpy() for t in (q, k, v)]
    e = eta.double().numpy()
    w = [t.double().numpy() for t in (W1, W2, W3)]
    flags = None if wl.update_chunks is None else list(wl.update_chunks)[:n]
    runs, elapsed = 0, 0.0
    while elapsed < budget_s:
        ts = time.perf_counter()
        O.ttt_layer_forward(*x, e, *w, wl.chunk, wl.mode, update_chunks=flags, l2norm=wl.l2norm,
                            muon_steps=wl.muon_steps, momentum_beta=wl.momentum_beta)
        elapsed += time.perf_counter() - ts
        runs += 1
    head_tokens = runs * n * wl.chunk
    rate = head_tokens / elapsed / wl.H   # every layer token costs H head-tokens
    desc = (f"fp64 oracle on the first {n} of {nc} chunks of one (batch, head) sequence, "
            f"{runs} runs ({head_tokens} head-tokens in {elapsed:.1f} s); "
            f"layer tokens/s = head-tokens/s / H")
    return rate, desc, elapsed


# workloads bench.py can time (--workload); the default is the first
WORKLOADS = ("lm760m", "nvs-strided", "long-1m")


def workload_by_key(key):
    import workloads
    return {"lm760m": workloads.LM_760M, "nvs-strided": workloads.NVS_STRIDED,
            "long-1m": workloads.LONG_1M}[key]


def workload_config(wl):
    mask = {0: "apply-then-update", 1: "block-causal", 2: "bidirectional", 3: "strided"}[wl.mode]
    cfg = {"workload": wl.name, "B": wl.B, "H": wl.H, "N": wl.N, "d_h": wl.d_h, "m_h": wl.m_h,
           "chunk": wl.chunk, "mask": mask, "muon_steps": wl.muon_steps,
           "momentum_beta": wl.momentum_beta, "l2norm": wl.l2norm}
    if wl.update_chunks is not None:
        cfg["update_chunks"] = list(wl.update_chunks)
    return cfg


# ---------------------------------------------------------------------------

def run_reference(args):
    """Reference arm: the fp64 CPU oracle, as it stands, on the machine's cores."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    wl = workload_by_key(args.workload)
    per_step = []
    for _ in range(args.warmup):
        oracle_sample(wl, budget_s=1.0)
    desc = ""
    for _ in range(args.steps):
        rate, desc, el = oracle_sample(wl, budget_s=args.ref_budget)
        per_step.append(rate)
    value = statistics.median(per_step)
    cfg = workload_config(wl)
    cfg["parallelism"] = "single process (host cores)"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": max(world, args.gpus), "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": wl.B * wl.N / value * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": cfg,
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
    """CUDA-event time (ms) of `steps` calls of fn after `warmup` untimed ones,
    with the device synchronised on both sides."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


# inputs above this many q elements are drawn on the device
HOST_DRAW_LIMIT = 1 << 28


def device_inputs(torch, wl, dev):
    """(device inputs, page-locked host copies or None) for a layer workload."""
    import workloads
    if wl.B * wl.H * wl.N * wl.d_h > HOST_DRAW_LIMIT:
        return list(workloads.layer_inputs_on_device(wl, dev)), None
    pinned = [t.pin_memory() for t in workloads.layer_inputs(wl)]
    return [t.to(dev) for t in pinned], pinned


class LayerCall:
    """One ttt_layer_forward call over a workload with preallocated outputs
    and workspace (device-resident inputs)."""

    def __init__(self, torch, cla, wl, dev, inputs):
        self.cla, self.wl = cla, wl
        self.q, self.k, self.v, self.eta, self.W1, self.W2, self.W3 = inputs
        B, H, N, d, m, b = wl.B, wl.H, wl.N, wl.d_h, wl.m_h, wl.chunk
        self.rule = cla.update_rule(l2norm=wl.l2norm, muon_steps=wl.muon_steps,
                                    momentum_beta=wl.momentum_beta)
        self.out = torch.empty_like(self.q)
        self.Wf = (torch.empty((B, H, m, d), device=dev), torch.empty((B, H, d, m), device=dev),
                   torch.empty((B, H, m, d), device=dev))
        self.ws = torch.empty(cla.layer_workspace_size(B, H, N, d, m, b, cla.TTT_BF16, wl.mode,
                                                       self.rule), device=dev, dtype=torch.uint8)

    def __call__(self):
        self.cla.ttt_layer_forward(self.q, self.k, self.v, self.eta, self.W1, self.W2, self.W3,
                                   self.wl.chunk, self.wl.mode, self.rule,
                                   update_chunks=self.wl.update_chunks, out=self.out,
                                   W_final=self.Wf, workspace=self.ws)


def check_status(cla):
    st = cla.device_status()
    if st != 0:
        raise RuntimeError(f"device status {st}: {cla.status_string(st)}")


def time_extra_workload(torch, cla, wl, dev, stream, peaks, steps, warmup):
    """ms per call, tokens/s and share of the bf16 peak of a further workload."""
    inputs, _ = device_inputs(torch, wl, dev)
    call = LayerCall(torch, cla, wl, dev, inputs)
    call()
    torch.cuda.synchronize()
    check_status(cla)
    ms = time_steps(torch, call, steps, warmup, stream) / steps
    check_status(cla)
    fl = layer_flops(wl)
    tfl = fl / (ms / 1e3) / 1e12
    res = {"config": workload_config(wl), "ms_per_call": ms, "steps": steps, "warmup": warmup,
           "tokens_per_s": wl.B * wl.N / (ms / 1e3), "flops_per_call": fl, "tflops": tfl,
           "frac_of_burst": tfl / float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])),
           "inputs": "drawn on the device" if wl.B * wl.H * wl.N * wl.d_h > HOST_DRAW_LIMIT
           else "drawn on the host, copied once"}
    del call, inputs
    torch.cuda.empty_cache()
    return res


def time_linattn(torch, cla, dev, stream, peaks):
    """The chunked linear-attention workload (HBM-bound), CUDA-event time per
    call.  Main figure: calls back to back over three independently drawn
    input sets whose I/O together (3 x 134.7 MB) is three times L2, so every
    call reads its inputs from HBM.  Beside it: the call alone after a 256 MB
    write flush, whose dirty lines are written back during the call."""
    import workloads
    lw = workloads.LINATTN_C2
    nsets = 3
    sets = []
    for j in range(nsets):
        lq, lk, lv, leta, _ = [t.to(dev) if t is not None else None
                               for t in workloads.linattn_inputs(lw, seed=lw.seed + j)]
        sets.append((lq, lk, lv, leta, torch.empty_like(lq),
                     torch.empty((lw.B, lw.H, lw.d_v, lw.d_k), device=dev)))
    lws = torch.empty(cla.linattn_workspace_size(lw.B, lw.H, lw.N, lw.d_k, lw.d_v, lw.chunk,
                                                 cla.TTT_BF16, lw.mode),
                      device=dev, dtype=torch.uint8)

    def call(j):
        q_, k_, v_, eta_, o_, S_ = sets[j % nsets]
        cla.linattn_chunked_forward(q_, k_, v_, eta_, lw.chunk, lw.mode, out=o_, S_final=S_,
                                    workspace=lws)

    for j in range(3 * nsets):
        call(j)
    torch.cuda.synchronize()
    check_status(cla)
    reps = 10 * nsets
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    # keep the GPU busy (~1.5 ms) while the host enqueues the calls, so the
    # timed calls run back to back on the device whatever the host's pace
    torch.cuda._sleep(3_000_000)
    h0 = time.perf_counter()
    e0.record(stream)
    for j in range(reps):
        call(j)
    e1.record(stream)
    host_us = (time.perf_counter() - h0) * 1e6 / reps
    torch.cuda.synchronize()
    lms = e0.elapsed_time(e1) / reps

    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    tot, nf = 0.0, 10
    for i in range(nf + 3):
        flush.zero_()
        f0 = torch.cuda.Event(enable_timing=True)
        f1 = torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        call(0)
        f1.record(stream)
        torch.cuda.synchronize()
        if i >= 3:
            tot += f0.elapsed_time(f1)
    check_status(cla)
    fms = tot / nf
    lq, leta, lo = sets[0][0], sets[0][3], sets[0][4]
    io_bytes = (3 * lq.numel() * 2 + leta.numel() * 4 + lo.numel() * 2)
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    return {"workload": lw.name, "us_per_call": lms * 1e3,
            "tokens_per_s": lw.B * lw.N / (lms / 1e3),
            "gbs": io_bytes / (lms / 1e3) / 1e9, "hbm_frac": io_bytes / (lms / 1e3) / 1e9 / hbm,
            "io_bytes": io_bytes, "host_enqueue_us_per_call": host_us,
            "l2": "inputs larger than L2: calls back to back over %d input sets (%.0f MB of I/O)"
                  % (nsets, nsets * io_bytes / 1e6),
            "after_write_flush": {"us_per_call": fms * 1e3,
                                  "gbs": io_bytes / (fms / 1e3) / 1e9,
                                  "note": "one call after a 256 MB write to L2; the flush's "
                                          "dirty lines are written back during the call"}}


def time_variants(torch, cla, dev, stream, steps=10, warmup=3):
    """The reduction path of the linear-attention paper (sec. 6.1, Table 2:
    TTT-layer tokens/s, recurrent and parallel forms) on the LM workload's
    shapes and inputs: LaCT; Variant 1 (only W2 updates); Variant 2 (no
    normalisation; recurrent and parallel); Variants 3-5 (a single linear
    fast weight d x d with Muon; momentum; per-token or constant eta; parallel
    form); Variant 6 (plain chunked linear attention)."""
    import workloads
    wl = workloads.LM_760M
    B, H, N, d, m, b = wl.B, wl.H, wl.N, wl.d_h, wl.m_h, wl.chunk
    q, k, v, eta, W1, W2, W3 = [t.to(dev) for t in workloads.layer_inputs(wl)]
    nc = N // b
    res = {}

    def timed(name, fn, form):
        fn()
        torch.cuda.synchronize()
        check_status(cla)
        ms = time_steps(torch, fn, steps, warmup, stream) / steps
        check_status(cla)
        res[name] = {"form": form, "ms_per_call": ms, "tokens_per_s": B * N / (ms / 1e3)}

    out = torch.empty_like(q)
    Wf = (torch.empty((B, H, m, d), device=dev), torch.empty((B, H, d, m), device=dev),
          torch.empty((B, H, m, d), device=dev))
    for name, kw, form in (
            ("lact", dict(), "recurrent"),
            ("v1", dict(last_layer_only=True), "recurrent"),
            ("v2_recurrent", dict(last_layer_only=True, l2norm=False,
                                  form=cla.FORM_RECURRENT), "recurrent"),
            ("v2_parallel", dict(last_layer_only=True, l2norm=False,
                                 form=cla.FORM_PARALLEL), "parallel")):
        rk = dict(l2norm=True, muon_steps=wl.muon_steps, momentum_beta=wl.momentum_beta)
        rk.update(kw)
        rule = cla.update_rule(**rk)
        ws = torch.empty(cla.layer_workspace_size(B, H, N, d, m, b, cla.TTT_BF16, wl.mode, rule),
                         device=dev, dtype=torch.uint8)
        timed(name, lambda: cla.ttt_layer_forward(q, k, v, eta, W1, W2, W3, b, wl.mode, rule,
                                                  out=out, W_final=Wf, workspace=ws), form)
        del ws
    # a single linear fast weight S [d, d] (Variants 3-6), S0 ~ N(0, 1/d)
    S0 = W2.unsqueeze(0).expand(B, H, d, m).contiguous()
    beta = torch.full((B, H, nc), wl.momentum_beta, device=dev)
    eta_c = torch.full_like(eta, 1.0 / b)
    S = torch.empty((B, H, d, m), device=dev)
    lo = torch.empty_like(q)
    for name, e_, al, steps_ in (("v3", eta, beta, wl.muon_steps),
                                 ("v4", eta_c, beta, wl.muon_steps),
                                 ("v5", eta_c, None, wl.muon_steps),
                                 ("v6", eta_c, None, 0)):
        rule = cla.linattn_rule(alpha=al, muon_steps=steps_)
        ws = torch.empty(cla.library().linattn_rule_workspace_size(
            B, H, N, d, d, b, cla.TTT_BF16, wl.mode, ctypes_ref(rule)), device=dev,
            dtype=torch.uint8)
        timed(name, lambda: cla.linattn_chunked_forward_rule(
            q, k, v, e_, b, wl.mode, S0=S0, alpha=al, muon_steps=steps_, out=lo, S_final=S,
            workspace=ws), "parallel")
        del ws
    res["note"] = ("LM workload shapes (B2 H4 d=m=384 N32768 chunk 2048, beta 0.9, Muon 5); "
                   "Variants 3-6 use q, k, v directly with a 384 x 384 state")
    return res


def ctypes_ref(x):
    import ctypes
    return ctypes.byref(x)


def run_ours(args):
    import torch
    import chunked_linear_attention_gb300 as cla
    from chunked_linear_attention_gb300 import _build

    refusal = single_gpu_refusal(args)
    if refusal is not None:
        if dist_env()[0] == 0:
            print(json.dumps(refusal), flush=True)
        return 0
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    _build.build()
    cla.library()

    wl = workload_by_key(args.workload)
    if args.seq_len:
        wl = dataclasses.replace(wl, N=args.seq_len,
                                 update_chunks=None if wl.update_chunks is None
                                 else wl.update_chunks[:args.seq_len // wl.chunk])
    B, H, N, d, m, b = wl.B, wl.H, wl.N, wl.d_h, wl.m_h, wl.chunk
    inputs, pinned = device_inputs(torch, wl, dev)
    step = LayerCall(torch, cla, wl, dev, inputs)
    stream = torch.cuda.current_stream(dev)
    peaks, peak_src = load_peaks()

    # device-resident timing, clocks sampled during the timed region
    clocks = ClockSampler(gpu_index=dev.index)
    step()
    torch.cuda.synchronize()
    check_status(cla)
    launches0 = cla.launch_count()
    clocks.start()
    ms = time_steps(torch, step, args.steps, args.warmup, stream)
    clk = clocks.stop()
    check_status(cla)
    launches = (cla.launch_count() - launches0) // (args.steps + args.warmup) * args.steps
    ms_step = ms / args.steps
    tokens = B * N
    value = tokens * args.steps / (ms / 1e3)

    # end to end through the public host-buffer call: page-locked inputs in,
    # outputs and final weights back in page-locked host memory; the library
    # overlaps each chunk's transfers with the kernels
    if pinned is None:
        pinned = [t.cpu().pin_memory() for t in inputs]
    h_out = torch.empty(step.out.shape, dtype=step.out.dtype, pin_memory=True)
    h_W = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in step.Wf]
    hq, hk, hv, heta, hW1, hW2, hW3 = pinned
    ws_host = torch.empty(cla.layer_host_workspace_size(B, H, N, d, m, b, cla.TTT_BF16, wl.mode,
                                                        step.rule), device=dev, dtype=torch.uint8)

    def e2e_step():
        cla.ttt_layer_forward_host(hq, hk, hv, heta, hW1, hW2, hW3, b, wl.mode, step.rule,
                                   update_chunks=wl.update_chunks, out=h_out, W_final=h_W,
                                   workspace=ws_host)
        # the step's result is read on the host: wait for the call to complete
        stream.synchronize()

    e2e_steps = max(1, min(args.steps, 20))
    ms_e2e = time_steps(torch, e2e_step, e2e_steps, 3, stream)
    check_status(cla)
    e2e_value = tokens * e2e_steps / (ms_e2e / 1e3)
    h2d = sum(t.numel() * t.element_size() for t in pinned)
    d2h = h_out.numel() * h_out.element_size() + sum(t.numel() * t.element_size() for t in h_W)
    del ws_host

    # per-launch profile of one more step (CUDA events around every launch)
    cla.profile_start()
    step()
    prof = cla.profile_stop()
    check_status(cla)
    tc_kernels = ("umma_gemm_kernel", "ns_cluster_kernel", "ns_half_kernel")
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
    peak_sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    peak_burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    flops_step = layer_flops(wl)
    step_tflops = flops_step / (ms_step / 1e3) / 1e12
    # Launches of different (batch, head) sequences overlap on separate
    # streams, so per-launch durations do not add up to the step: the
    # tensor-core kernels' achieved rate is their algorithmic FLOPs (which
    # are all of the step's FLOPs) over the timed step.
    achieved = g_fl / (ms_step / 1e3) / 1e12
    q_bytes = 3 * inputs[0].numel() * inputs[0].element_size()
    del step, inputs
    torch.cuda.empty_cache()

    lin = None
    if not args.skip_linattn:
        lin = time_linattn(torch, cla, dev, stream, peaks)

    extra = {}
    if not args.skip_workloads:
        for key in WORKLOADS:
            if key == args.workload:
                continue
            ew = workload_by_key(key)
            big = ew.B * ew.H * ew.N * ew.d_h > HOST_DRAW_LIMIT
            extra[key] = time_extra_workload(torch, cla, ew, dev, stream, peaks,
                                             steps=5 if big else 20, warmup=3)

    variants = None
    if not args.skip_variants:
        variants = time_variants(torch, cla, dev, stream)

    cpu = None
    if not args.skip_cpu_baseline:
        rate, desc, _ = oracle_sample(wl, budget_s=args.ref_budget)
        cpu = {"value": rate, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
               "sample": desc}

    cfg = workload_config(wl)
    cfg.update({"io": "bf16 q/k/v, fp32 eta and fast weights",
                "l2": "inputs larger than L2 (q, k, v: %.0f MB per step)" % (q_bytes / 1e6),
                "parallelism": "single GPU"})
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": cfg,
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
                "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e / e2e_steps,
                "steps": e2e_steps},
        "cpu_baseline": cpu,
        "gpu_launches": launches,
        "clocks": clk,
        "linattn": lin,
        "workloads": extra,
        "variants": variants,
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=WORKLOADS, default=WORKLOADS[0],
                    help="the workload of the headline figure")
    ap.add_argument("--ref-budget", type=float, default=12.0,
                    help="seconds of oracle work per CPU-baseline sample")
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--skip-linattn", action="store_true")
    ap.add_argument("--skip-workloads", action="store_true",
                    help="time only the headline workload")
    ap.add_argument("--skip-variants", action="store_true",
                    help="skip the reduction variants (Table 2 forms) on the LM workload")
    ap.add_argument("--seq-len", type=int, default=None,
                    help="override the workload's sequence length (small profiling cases)")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)   # timing rule: at least 3 warm-up steps
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
