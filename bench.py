#!/usr/bin/env python3
"""Benchmark of the GQA decode step on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--no-cpu-baseline]

One step = one gqa_decode call over the whole batch of the workload (default:
the Llama-2/3-70B-shaped long-context decode, B=8, Hq=64, Hkv=8, D=128,
seq_len=8192, bf16).  Inputs are synthetic, seeded, and resident in HBM when
the timed region starts; they exceed the 126 MB L2 (268 MB for the default
workload) and the kernel loads K/V with an L2 evict-first hint, so nothing is
flushed between steps.  Each step is bracketed by CUDA events recorded on the
launching stream; the timed region is bracketed by a barrier and
torch.cuda.synchronize() on both sides.

Printed (rank 0, one JSON line): the metric (us/step, lower is better), KV
GB/s and the HBM roofline fraction, an end-to-end figure through the public
API with host buffers (pinned H2D of the step's inputs + decode + D2H of the
output), SM clocks sampled during the timed region, and the fp64 CPU oracle
timed on a bounded sample of the same workload (``cpu_baseline``).

``--impl reference`` times only that oracle (the reference arm): each step is
a bounded sample of the workload, extrapolated to the metric's unit.

Multi-GPU (torchrun): every rank runs an independent replica of the workload
(the decode step has no exchange between GPUs); rank 0 reports the maximum
step time over ranks and the aggregate KV bandwidth.
"""
from __future__ import annotations

import argparse
import json
import os
import signal
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("GQA decode attention µs/step, KV-cache GB/s and % of B300 HBM "
          "peak (1 GPU)")
FALLBACK_HBM_GBS = 6400.0
SPEC_HBM_GBS = 8000.0
L2_BYTES = 126 * 1024 * 1024


KERNEL_SOURCES = ("gqa_decode_kernel.cuh", "ptx.cuh", "gqa_api.cu")
GRAPH_STEPS = 100  # steps per captured CUDA graph (--graph, --op append)


def _code_only(text: str) -> str:
    """C++ source without comments and with whitespace runs collapsed, so
    that an edit of comments or layout leaves the hash unchanged (string and
    character literals are kept as they are)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_sources_sha256() -> str:
    """Hash of the CUDA sources the profiled kernel was built from (their
    code only: comments and whitespace do not count)."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "grouped_query_attention_11_b300", "csrc")
    for name in KERNEL_SOURCES:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()


def profiled_traffic(workload: str):
    """DRAM bytes (read + write) per launch of the decode kernel on this
    workload, from the ncu summary committed under profiles/, or None when
    there is none or the kernel sources changed since it was captured."""
    path = os.path.join(ROOT, "profiles", f"gqa_decode_kernel__{workload}.md")
    try:
        with open(path) as f:
            text = f.read()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        line = line.strip().lstrip("-").strip()
        if ":" in line and line.startswith(("traffic_bytes_per_launch",
                                            "kernel_sources_sha256")):
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_sources_sha256") != kernel_sources_sha256():
        return None
    try:
        return int(vals["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 200):
        self.proc = None
        self.rows = []
        self.gpu_index = gpu_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}",
                 f"--query-gpu=timestamp,{self.FIELDS}",
                 "--format=csv,noheader,nounits", f"-lms={period_ms}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.send_signal(signal.SIGTERM)
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 10:
                self.rows.append(parts)

    def summary(self):
        if not self.rows:
            return None
        sm = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in self.rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        reasons = set()
        for r in self.rows:
            for name, val in zip(names, r[6:10]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(self.rows)}


# ------------------------------------------------------------ CPU baseline

def cpu_baseline(w, inp, budget_s: float = 10.0):
    """fp64 oracle on the host cores: whole sequences, one at a time, until
    ``budget_s`` has passed; extrapolated to one full step (us/step)."""
    import numpy as np
    import oracle
    import torch
    oracle.build()
    threads = oracle.max_threads()
    lens = inp["seq_lens"]
    done_tokens = 0
    total_tokens = int(lens.sum())
    t0 = time.perf_counter()
    n_seq = 0
    order = list(range(w.B))
    for b in order:
        sl = slice(b, b + 1)
        ks = inp["k_scale"][sl] if inp["k_scale"] is not None else None
        vs = inp["v_scale"][sl] if inp["v_scale"] is not None else None
        oracle.gqa_decode(inp["q"][sl], inp["k"][sl], inp["v"][sl], lens[sl],
                          inp["scale"], k_scale=ks, v_scale=vs,
                          nthreads=threads)
        done_tokens += int(lens[b])
        n_seq += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    el = time.perf_counter() - t0
    frac = done_tokens / total_tokens if total_tokens else 1.0
    us_per_step = el / frac * 1e6 if frac > 0 else el * 1e6
    return {"value": us_per_step, "unit": "us/step", "cores": threads,
            "kind": "oracle",
            "sample": (f"{n_seq} of {w.B} sequences ({done_tokens} of "
                       f"{total_tokens} tokens, all {w.Hq} query heads), fp64 "
                       f"C oracle, {el:.2f} s wall, extrapolated by tokens")}


# ------------------------------------------------------------------ runner

def bench_append(a, w, name, peak, peak_kind):
    """K back-to-back gqa_append_kv calls on the workload's shape (1 GPU):
    every call appends one token to every sequence, from a length that
    leaves room for all of them.  FP8 scales start at 1 (N(0,1) rows fit, so
    no earlier code is re-encoded: the common step)."""
    import torch
    import grouped_query_attention_11_b300 as gq
    dev = torch.device("cuda", torch.cuda.current_device())
    K, warmup = a.steps, max(3, a.warmup)
    start_len = max(0, w.Smax - K - warmup - 2)
    g = torch.Generator().manual_seed(w.seed)
    qdt = {"f16": torch.float16, "bf16": torch.bfloat16}[w.dtype]
    cdt = {"same": qdt, "e4m3": torch.float8_e4m3fn,
           "e5m2": torch.float8_e5m2}[w.kv]
    kn = torch.randn((w.B, w.Hkv, w.D), generator=g).to(qdt).to(dev)
    vn = torch.randn((w.B, w.Hkv, w.D), generator=g).to(qdt).to(dev)
    shape = (w.B, w.Hkv, w.Smax, w.D)
    kc = torch.zeros(shape, dtype=torch.uint8 if w.kv != "same" else qdt,
                     device=dev)
    vc = torch.zeros_like(kc)
    if w.kv != "same":
        kc, vc = kc.view(cdt), vc.view(cdt)
        ks = torch.ones((w.B, w.Hkv), dtype=torch.float32, device=dev)
        vs = torch.ones_like(ks)
    else:
        ks = vs = None
    lens = torch.full((w.B,), start_len, dtype=torch.int32, device=dev)
    # a side stream: the library's per-stream scratch is set up on it before
    # the steps are captured into graphs
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())

    # checked once through the public wrapper, then one C-ABI call per step
    gq.gqa_append_kv(kn, vn, kc, vc, lens, k_scale=ks, v_scale=vs,
                     stream=stream)
    torch.cuda.synchronize()
    lens.fill_(start_len)
    fn = gq.lib().gqa_append_kv
    code = {"f16": gq.GQA_F16, "bf16": gq.GQA_BF16}[w.dtype]
    ccode = {"same": code, "e4m3": gq.GQA_E4M3, "e5m2": gq.GQA_E5M2}[w.kv]
    args = (kn.data_ptr(), vn.data_ptr(), kc.data_ptr(), vc.data_ptr(),
            ks.data_ptr() if ks is not None else None,
            vs.data_ptr() if vs is not None else None, lens.data_ptr(), w.B,
            w.Hkv, w.Smax, w.D, code, ccode, stream.cuda_stream)

    def step():
        if fn(*args) != gq.GQA_OK:
            raise RuntimeError("gqa_append_kv failed")

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            step()
    torch.cuda.synchronize()
    # K steps as CUDA graphs of GRAPH_STEPS captured calls: each call is one
    # kernel of a few microseconds, so launching them one by one from the
    # host would time the driver's launch path, not the GPU
    graphs, left = [], K
    while left > 0:
        n = min(GRAPH_STEPS, left)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(n):
                step()
        graphs.append(g)
        left -= n
    lens.fill_(start_len + warmup)
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(torch.cuda.current_device())
    time.sleep(1.0 if sampler.proc else 0)
    torch.cuda.synchronize()
    ev0.record(stream)
    for g in graphs:
        g.replay()
    launches = K
    ev1.record(stream)
    torch.cuda.synchronize()
    sampler.stop()
    assert gq.gqa_device_errors(stream) == 0
    assert int(lens[0]) == start_len + K + warmup
    us = ev0.elapsed_time(ev1) * 1e3 / K
    eb = 1 if w.kv != "same" else 2
    # bytes per append: new rows read (16-bit) + cache rows written + lens
    algo = 2 * w.B * w.Hkv * w.D * (2 + eb) + 8 * w.B + (
        16 * w.B * w.Hkv if w.kv != "same" else 0)
    achieved = algo / (us * 1e-6) / 1e9
    line = {"metric": "GQA cache append us/step (1 GPU)", "value": us,
            "unit": "us/step", "n_gpus": 1, "steps": K, "warmup": warmup,
            "ms_per_step": us / 1e3, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype if w.kv == "same" else
            f"{w.kv} KV / {w.dtype} rows", "data": "synthetic",
            "config": {"workload": name, "op": "append",
                       "launch": f"CUDA graphs of {GRAPH_STEPS} steps",
                       "B": w.B,
                       "Hkv": w.Hkv, "D": w.D, "Smax": w.Smax,
                       "start_len": start_len},
            "algorithmic_bytes_per_step": algo,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak,
                         "unit": "GB/s", "frac": achieved / peak,
                         "peak_kind": peak_kind, "traffic": None,
                         "note": "a few KB per call: launch-latency bound"},
            "gpu_launches": launches, "clocks": sampler.summary()}
    print(json.dumps(line), flush=True)
    return 0


def job_us_per_step(us: float, ws: int, device) -> float:
    """Whole-job time per step of ws replicas that each ran the same steps:
    the slowest rank's time (max over ranks, one all-reduce on the timing
    only) divided by the ws steps the job completed in it."""
    if ws > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([us], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        us = float(t.item())
    return us / ws


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=None)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--op", default="decode", choices=["decode", "append"],
                    help="decode: the decode step (default); append: the "
                         "cache-append step before it")
    a = ap.parse_args(argv)

    from grouped_query_attention_11_b300.workloads import (HEADLINE,
                                                           WORKLOADS,
                                                           make_inputs)
    name = a.workload or HEADLINE
    w = WORKLOADS[name]
    ws, rank, local = dist_env()
    peak, peak_kind = load_peaks()
    cfg = {"workload": name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "G": w.G,
           "D": w.D, "seq_len": (w.Smax if w.lens[0] == "uniform" else
                                 f"uniform[{w.lens[1]},{w.lens[2]}]"),
           "Smax": w.Smax, "qo_dtype": w.dtype,
           "kv_dtype": w.kv if w.kv != "same" else w.dtype,
           "l2": "inputs larger than L2, K/V loaded evict-first; no flush",
           "parallelism": "replicas" if a.gpus > 1 else "single"}
    warmup = max(3, a.warmup)

    if a.impl == "reference":
        if rank != 0:
            return 0
        inp = make_inputs(w, pad="zero")
        # Warm-up: the oracle on one sequence per warm-up step, untimed (it
        # builds and loads the oracle library and touches the inputs).
        for _ in range(warmup):
            cpu_baseline(w, inp, budget_s=0.0)
        # Each step is a bounded sample (about 10 s of oracle work); at most
        # ~60 s in all, whatever --steps asks for.
        n_steps = max(1, min(a.steps, 6))
        budget = max(2.0, 60.0 / n_steps)
        vals = []
        last = None
        for _ in range(n_steps):
            last = cpu_baseline(w, inp, budget_s=budget)
            vals.append(last["value"])
        v = statistics.median(vals)
        line = {"metric": METRIC, "value": v, "unit": "us/step",
                "impl": "reference", "n_gpus": a.gpus, "steps": len(vals),
                "warmup": warmup, "ms_per_step": v / 1e3,
                "higher_is_better": False,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": cfg,
                "cpu_baseline": dict(last, value=v),
                "e2e": {"value": v, "unit": "us/step",
                        "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return 0

    import torch
    import grouped_query_attention_11_b300 as gq

    if a.op == "append":
        return bench_append(a, w, name, peak, peak_kind)

    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    gq.lib()

    inp = make_inputs(w, pad="zero", seed=w.seed + rank)
    # a paged workload also carries its contiguous copy (for checks): not an
    # input of the step
    inp.pop("k_contig", None)
    inp.pop("v_contig", None)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v)
         for k, v in inp.items()}
    out = torch.empty_like(d["q"])
    stream = torch.cuda.current_stream()

    step = gq.BoundDecode(d, out, stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    assert gq.gqa_device_errors(stream) == 0

    algo_bytes = w.algorithmic_bytes(inp["seq_lens"])
    K = a.steps
    # K steps back to back between one pair of events on the launching
    # stream; the host only enqueues (one C-ABI call per step), so the device
    # time per step is not inflated by Python overhead.
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)

    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    time.sleep(1.0 if sampler and sampler.proc else 0)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    launches = 0
    t_wall0 = time.perf_counter()
    ev0.record(stream)
    for i in range(K):
        step()
        launches += gq.gqa_last_launch_count()
    ev1.record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    if ws > 1:
        torch.distributed.barrier()
    if sampler:
        sampler.stop()
    assert gq.gqa_device_errors(stream) == 0

    us = ev0.elapsed_time(ev1) * 1e3 / K
    # replicas: every rank ran K steps; the job's time is the slowest rank's
    job_us = job_us_per_step(us, ws, dev)

    # ---- end to end through the public API, host buffers ----
    e2e = None
    ek = max(1, a.e2e_steps)
    host = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v)
            for k, v in inp.items()}
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in host.values()
              if isinstance(v, torch.Tensor))
    d2h = h_out.numel() * h_out.element_size()
    dd = {k: (torch.empty_like(v, device=dev) if isinstance(v, torch.Tensor)
              else v) for k, v in host.items()}

    def e2e_step():
        for k, v in host.items():
            if isinstance(v, torch.Tensor):
                dd[k].copy_(v, non_blocking=True)
        gq.decode_inputs(dd, out=out, stream=stream)
        h_out.copy_(out, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(
        enable_timing=True)
    es.record(stream)
    for _ in range(ek):
        e2e_step()
    ee.record(stream)
    torch.cuda.synchronize()
    e2e_us = es.elapsed_time(ee) * 1e3 / ek
    e2e = {"value": job_us_per_step(e2e_us, ws, dev), "unit": "us/step",
           "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "steps": ek}
    del dd

    if rank != 0:
        if ws > 1:
            torch.distributed.destroy_process_group()
        return 0

    achieved = algo_bytes / (us * 1e-6) / 1e9
    traffic = profiled_traffic(name)
    clocks = sampler.summary() if sampler else None
    cpu = None
    if not a.no_cpu_baseline and ws == 1:
        cpu = cpu_baseline(w, inp, budget_s=10.0)
    line = {
        "metric": METRIC, "value": job_us, "unit": "us/step",
        "n_gpus": ws, "steps": K, "warmup": warmup,
        "ms_per_step": job_us / 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype if
        w.kv == "same" else f"{w.kv} KV / {w.dtype} q,out", "data": "synthetic",
        "config": cfg,
        "kv_gbs": achieved * ws, "hbm_frac_of_" + peak_kind: achieved / peak,
        "hbm_frac_of_spec_8tbs": achieved / SPEC_HBM_GBS,
        "wall_s_timed_region": t_wall,
        "algorithmic_bytes_per_step": algo_bytes,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": peak_kind, "traffic": traffic},
        "e2e": e2e, "gpu_launches": launches, "clocks": clocks,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
