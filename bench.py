#!/usr/bin/env python3
"""Benchmark of the GQA decode step on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--no-cpu-baseline]
                    [--no-per-config] [--op decode|append]
                    [--kernel-path 0|1|2] [--num-ctas N] [--tune BITS]
                    [--profile-launches N [--batch B]]

The last four are diagnostics: A/B arms of single design choices (kernel
choice, block count, GQA_TUNE_* bits) and a profiling mode that only launches
N steps (optionally of a smaller batch of the same shape) for ncu.

One step = one gqa_decode call over the whole batch of the workload (default:
the Llama-2/3-70B-shaped long-context decode, B=8, Hq=64, Hkv=8, D=128,
seq_len=8192, bf16).  Inputs are synthetic, seeded, and resident in HBM when
the timed region starts.

Protocol of the headline line:

1. the nvidia-smi clock sampler starts and settles (1 s, the GPU idle);
2. W warm-up steps, then back-to-back steps until SETTLE_S seconds have passed
   since the warm-up began ("settle"): the first ~1 ms of work after an idle
   GPU runs up to 25 % slower, with the SM and memory clocks already at their
   maximum, so a short timed region that follows an idle gap measures that
   ramp rather than the kernel;
3. barrier + synchronize, then EXACTLY K steps back to back between two CUDA
   events on the launching stream (one pre-marshalled C-ABI call per step),
   barrier + synchronize.  The inputs (268 MB) exceed the 126 MB L2 and K/V are
   loaded evict-first, so nothing is flushed between steps.

After the timed region (not part of ``value``): the same K-step region
repeated (median, p10, p90) and the per-launch time of steps that each start
with a flushed L2 (a 256 MB buffer written before every step; median, p10,
p90 of 200).

``per_config`` (N=1): every other named workload measured in the same process
by the same steps, with inputs drawn on the device.  Workloads whose bytes
per step exceed twice the L2 are timed back to back; smaller ones (tiny, the
8B shape, MQA) with L2 flushed before every step, so that their figure is an
HBM figure.  Each entry carries us/step, KV GB/s, the roofline fraction, the
profiled DRAM traffic (when current) and the CPU oracle on a bounded sample.

The headline line also carries an end-to-end figure through the public API
with host buffers (pinned H2D of the step's inputs + decode + D2H of the
output), SM clocks sampled from the warm-up to the end of the timed region,
and the fp64 CPU oracle timed on a bounded sample of the same workload
(``cpu_baseline``).

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


KERNEL_SOURCES = ("gqa_decode_kernel.cuh", "gqa_decode_umma.cuh", "ptx.cuh",
                  "gqa_api.cu", "gqa_umma.cu")
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


TRAFFIC_SUMMARY = os.path.join("profiles",
                               "gqa_decode__dram_traffic_all_workloads.md")


def profiled_traffic(workload: str, algo_bytes: int = 0):
    """DRAM bytes (read + write) per launch of the decode kernel on this
    workload, from the ncu summary committed under profiles/ (scaled by this
    run's algorithmic bytes when they differ from the captured step's), or
    None when there is none or the kernel sources changed since it was
    captured."""
    path = os.path.join(ROOT, TRAFFIC_SUMMARY)
    try:
        with open(path) as f:
            text = f.read()
    except OSError:
        return None
    sha, found = None, None
    for line in text.splitlines():
        line = line.strip().lstrip("-").strip()
        if line.startswith("kernel_sources_sha256:"):
            sha = line.split(":", 1)[1].strip().strip("`")
        elif line.startswith(f"traffic_bytes_per_launch {workload}:"):
            parts = [x for x in line.split("`") if x.strip().isdigit()]
            if len(parts) >= 2:
                found = (int(parts[0]), int(parts[1]))
    if sha != kernel_sources_sha256() or found is None:
        return None
    traffic, algo = found
    if algo_bytes and algo and algo_bytes != algo:
        return int(round(traffic * algo_bytes / algo))
    return traffic


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

    def __init__(self, gpu_index: int, period_ms: int = 100):
        self.proc = None
        self.rows = []
        self.gpu_index = gpu_index
        self.t_mark = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}",
                 f"--query-gpu=timestamp,{self.FIELDS}",
                 "--format=csv,noheader,nounits", f"-lms={period_ms}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def mark(self):
        """Only samples taken from now on count in summary()."""
        import datetime
        self.t_mark = datetime.datetime.now()

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

    def _window(self):
        if self.t_mark is None:
            return self.rows
        import datetime
        kept = []
        for r in self.rows:
            try:
                t = datetime.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f")
            except ValueError:
                continue
            if t >= self.t_mark:
                kept.append(r)
        return kept or self.rows[-1:]

    def summary(self):
        rows = self._window()
        if not rows:
            return None
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        reasons = set()
        for r in rows:
            for name, val in zip(names, r[6:10]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# ------------------------------------------------------------ CPU baseline

def _host_sequence(inp: dict, b: int, pool_host: dict) -> dict:
    """Sequence b of a workload's inputs as host tensors (the inputs may be
    on the device; a paged cache's page pool is copied to the host once)."""
    out = {"scale": inp["scale"]}
    sl = slice(b, b + 1)
    for key in ("q", "seq_lens", "k_scale", "v_scale", "block_table"):
        v = inp.get(key)
        out[key] = v[sl].cpu() if v is not None else None
    if inp.get("block_table") is not None:
        for key in ("k", "v"):
            if key not in pool_host:
                pool_host[key] = inp[key].cpu()
            out[key] = pool_host[key]
    else:
        for key in ("k", "v"):
            out[key] = inp[key][sl].cpu()
    return out


def cpu_baseline(w, inp, budget_s: float = 10.0):
    """fp64 oracle on the host cores: whole sequences, one at a time, until
    ``budget_s`` of oracle time has passed; extrapolated to one full step
    (us/step).  Only the oracle calls are timed (not the copies of each
    sequence's inputs to the host)."""
    import oracle
    oracle.build()
    threads = oracle.max_threads()
    lens = inp["seq_lens"].cpu()
    total_tokens = int(lens.sum())
    done_tokens, n_seq, el = 0, 0, 0.0
    pool_host = {}
    for b in range(w.B):
        h = _host_sequence(inp, b, pool_host)
        t0 = time.perf_counter()
        if h["q"].dim() == 4:
            oracle.gqa_decode_chunk(h["q"], h["k"], h["v"], h["seq_lens"],
                                    h["scale"], nthreads=threads)
        elif h["block_table"] is not None:
            oracle.gqa_decode_paged(h["q"], h["k"], h["v"], h["block_table"],
                                    h["seq_lens"], h["scale"],
                                    nthreads=threads)
        else:
            oracle.gqa_decode(h["q"], h["k"], h["v"], h["seq_lens"],
                              h["scale"], k_scale=h["k_scale"],
                              v_scale=h["v_scale"], nthreads=threads)
        el += time.perf_counter() - t0
        done_tokens += int(lens[b])
        n_seq += 1
        if el >= budget_s:
            break
    frac = done_tokens / total_tokens if total_tokens else 1.0
    us_per_step = el / frac * 1e6 if frac > 0 else el * 1e6
    return {"value": us_per_step, "unit": "us/step", "cores": threads,
            "kind": "oracle",
            "sample": (f"{n_seq} of {w.B} sequences ({done_tokens} of "
                       f"{total_tokens} tokens, all {w.Hq} query heads"
                       f"{f', {w.T} tokens each' if w.T > 1 else ''}), fp64 "
                       f"C oracle, {el:.2f} s, extrapolated by tokens")}


# ------------------------------------------------------------------ timing

SETTLE_S = 0.25        # back-to-back steps after the warm-up, seconds
COLD_STEPS = 200       # flushed-L2 launches timed one by one
REPEATS = 30           # K-step regions repeated after the timed one


def _pct(xs, q):
    xs = sorted(xs)
    if not xs:
        return None
    k = (len(xs) - 1) * q
    lo = int(k)
    hi = min(lo + 1, len(xs) - 1)
    return xs[lo] + (xs[hi] - xs[lo]) * (k - lo)


def _dist(xs):
    return {"median_us": _pct(xs, 0.5), "p10_us": _pct(xs, 0.1),
            "p90_us": _pct(xs, 0.9), "n": len(xs)}


def time_region(step, K: int, stream) -> float:
    """us per step of K back-to-back steps between two events on the
    launching stream (synchronised on both sides)."""
    import torch
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(K):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / K


def settle(step, seconds: float) -> int:
    """Back-to-back steps until `seconds` of host time have passed (the
    launch queue keeps the GPU busy throughout); returns their number."""
    n, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        for _ in range(20):
            step()
        n += 20
    return n


def cold_launches(step, n: int, stream, flush) -> list:
    """Per-launch us of n steps, each after writing a buffer twice the size
    of L2 (so the step finds none of its inputs in L2 and no earlier decode
    launch to overlap with)."""
    import torch
    evs = []
    for i in range(n):
        flush.fill_(i & 0xFF)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step()
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) * 1e3 for a, b in evs]


def measure_config(name, w, dev, stream, flush, warmup, K, peak, peak_kind,
                   cpu_budget):
    """One per_config entry: the workload's inputs drawn on the device, warm-up
    and settle as for the headline, then either K-step back-to-back regions
    (bytes per step > 2 x L2) or flushed-L2 launches one by one."""
    import torch
    import grouped_query_attention_11_b300 as gq
    from grouped_query_attention_11_b300.workloads import make_inputs
    inp = make_inputs(w, pad="zero", device=dev)
    inp.pop("k_contig", None)
    inp.pop("v_contig", None)
    out = torch.empty_like(inp["q"])
    step = gq.BoundDecode(inp, out, stream)
    algo = w.algorithmic_bytes(inp["seq_lens"].cpu())
    for _ in range(warmup):
        step()
    settle(step, 0.1)
    torch.cuda.synchronize()
    assert gq.gqa_device_errors(stream) == 0
    b2b = [time_region(step, K, stream) for _ in range(5)]
    cold = cold_launches(step, 50, stream, flush)
    big = algo > 2 * L2_BYTES
    us = _pct(b2b, 0.5) if big else _pct(cold, 0.5)
    assert gq.gqa_device_errors(stream) == 0
    achieved = algo / (us * 1e-6) / 1e9
    entry = {
        "workload": name, "us_per_step": us,
        "l2": ("back to back: inputs larger than 2 x L2, median of 5 "
               f"regions of {K} steps") if big else
              "L2 flushed before every step: median of 50 launches",
        "kv_gbs": achieved, "frac": achieved / peak, "peak": peak,
        "peak_kind": peak_kind, "algorithmic_bytes_per_step": algo,
        "traffic": profiled_traffic(name, algo),
        "back_to_back": _dist(b2b), "cold_l2": _dist(cold),
        "launches_per_step": gq.gqa_last_launch_count(),
    }
    if cpu_budget > 0:
        entry["cpu_baseline"] = cpu_baseline(w, inp, budget_s=cpu_budget)
    del inp, out, step
    torch.cuda.empty_cache()
    return entry


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


def profile_launches(w, name, dev, n: int) -> int:
    """Profiling mode: the workload's inputs drawn on the device, then n
    decode launches back to back and nothing else, for a profiler to capture
    (``-s`` skips the first ones)."""
    import torch
    import grouped_query_attention_11_b300 as gq
    from grouped_query_attention_11_b300.workloads import make_inputs
    inp = make_inputs(w, pad="zero", device=dev)
    inp.pop("k_contig", None)
    inp.pop("v_contig", None)
    out = torch.empty_like(inp["q"])
    stream = torch.cuda.current_stream()
    step = gq.BoundDecode(inp, out, stream)
    torch.cuda.synchronize()
    for _ in range(n):
        step()
    torch.cuda.synchronize()
    err = gq.gqa_device_errors(stream)
    print(json.dumps({"profile_launches": n, "workload": name, "B": w.B,
                      "algorithmic_bytes_per_step":
                          w.algorithmic_bytes(inp["seq_lens"].cpu()),
                      "device_errors": err,
                      "launches_per_step": gq.gqa_last_launch_count()}),
          flush=True)
    return 0 if err == 0 else 1


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
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-workload measurements (headline only)")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--op", default="decode", choices=["decode", "append"],
                    help="decode: the decode step (default); append: the "
                         "cache-append step before it")
    ap.add_argument("--kernel-path", type=int, default=0, choices=[0, 1, 2],
                    help="0 automatic kernel choice (default); 1 the "
                         "warp-level mma kernel only; 2 the tensor-core "
                         "kernel wherever it applies (for A/B comparisons)")
    ap.add_argument("--num-ctas", type=int, default=0,
                    help="blocks per launch (0: the library's own choice, "
                         "the default; for A/B comparisons of the split)")
    ap.add_argument("--tune", type=int, default=0,
                    help="GQA_TUNE_* bits: design choices turned off for "
                         "A/B comparisons (1 no L2 warm-up, 2 no clusters, "
                         "4 no narrow rows); 0 (default) keeps all")
    ap.add_argument("--profile-launches", type=int, default=0,
                    help="profiling mode: build the workload's inputs, "
                         "launch exactly this many decode steps, check the "
                         "error flags and exit (no timing, no other "
                         "kernels after the inputs are drawn)")
    ap.add_argument("--batch", type=int, default=0,
                    help="profiling mode only: the workload with this many "
                         "sequences instead of its own B (a smaller capture "
                         "of the same shape; per-sequence figures scale)")
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
    gq.gqa_set_num_ctas(a.num_ctas)
    gq.gqa_set_kernel_path(a.kernel_path)
    gq.gqa_set_tuning(a.tune)
    if a.tune:
        cfg["tune"] = a.tune
    if a.num_ctas:
        cfg["num_ctas"] = a.num_ctas
    cfg["kernel_path"] = ("automatic", "warp-level mma",
                          "tensor core where it applies")[a.kernel_path]

    if a.profile_launches > 0:
        if a.batch > 0:
            import dataclasses
            w = dataclasses.replace(w, B=a.batch)
        return profile_launches(w, name, dev, a.profile_launches)

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
    algo_bytes = w.algorithmic_bytes(inp["seq_lens"])
    K = a.steps

    # clock sampler first, while the GPU is idle; then warm-up and settle, so
    # that the timed steps follow back-to-back work directly
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    time.sleep(1.0 if sampler and sampler.proc else 0)
    if sampler:
        sampler.mark()
    for _ in range(warmup):
        step()
    n_settle = settle(step, SETTLE_S)

    # ---- the timed region: exactly K steps ----
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    launches = 0
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    t_wall0 = time.perf_counter()
    ev0.record(stream)
    for _ in range(K):
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

    # ---- distributions (after the timed region; not part of value) ----
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    repeats = [time_region(step, K, stream) for _ in range(REPEATS)]
    cold = cold_launches(step, COLD_STEPS, stream, flush)
    assert gq.gqa_device_errors(stream) == 0

    # ---- end to end through the public API, host buffers ----
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
    traffic = profiled_traffic(name, algo_bytes)
    clocks = sampler.summary() if sampler else None
    if clocks is not None:
        clocks["window"] = "warm-up, settle and timed region"
    cpu = None
    if not a.no_cpu_baseline and ws == 1:
        cpu = cpu_baseline(w, inp, budget_s=10.0)

    per_config = None
    if ws == 1 and not a.no_per_config:
        del d, step
        torch.cuda.empty_cache()
        per_config = {}
        pc_sampler = ClockSampler(torch.cuda.current_device())
        time.sleep(1.0 if pc_sampler.proc else 0)
        pc_sampler.mark()
        for cname, cw in WORKLOADS.items():
            if cname == name:
                continue
            per_config[cname] = measure_config(
                cname, cw, dev, stream, flush, warmup, max(K, 20), peak,
                peak_kind, 0.0 if a.no_cpu_baseline else 2.0)
        pc_sampler.stop()
        per_config["clocks"] = pc_sampler.summary()

    line = {
        "metric": METRIC, "value": job_us, "unit": "us/step",
        "n_gpus": ws, "steps": K, "warmup": warmup,
        "ms_per_step": job_us / 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype if
        w.kv == "same" else f"{w.kv} KV / {w.dtype} q,out", "data": "synthetic",
        "config": cfg,
        "settle": {"steps": n_settle, "seconds": SETTLE_S,
                   "note": "untimed back-to-back steps after the warm-up"},
        "kv_gbs": achieved * ws, "hbm_frac_of_" + peak_kind: achieved / peak,
        "hbm_frac_of_spec_8tbs": achieved / SPEC_HBM_GBS,
        "wall_s_timed_region": t_wall,
        "algorithmic_bytes_per_step": algo_bytes,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": peak_kind, "traffic": traffic},
        "repeats": dict(_dist(repeats), steps_per_region=K),
        "cold_l2": _dist(cold),
        "e2e": e2e, "gpu_launches": launches, "clocks": clocks,
        "cpu_baseline": cpu,
        "per_config": per_config,
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
