"""Benchmark of the paged-KV GQA attention hot path on GB300.

One step = one pass of the hot path over one batch of synthetic input:
  pa_write_cache (the batch's new tokens) -> pa_decode_partitions -> pa_decode_merge
on the Llama-3-8B-shaped decode workload (64 sequences, 32 q / 8 kv heads,
head_dim 128, 16-token pages, seq_lens U[512, 4096], shuffled block tables).
The metric is decode KV-bytes GB/s (K and V of every visible token per step).
The other workloads (long-context split decode, tiny decode, ragged prefill,
chunked paged prefill, and the legs of the sliding window, the FP8 cache, the
single pass, the ungrouped split and the page copies) are measured in the same
run.  Each is then checked on its whole output against the fp64 CPU oracle,
which is timed on the host cores doing so (outside every GPU-timed region).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Output: one JSON line on stdout.  Its last key, "configs", summarises the five
named workloads (step throughput, kernel time, roofline fractions of the
measured and the nominal peak, median / min step time over 30 individually
timed steps, the oracle's throughput on all host cores and on one, and the
max / mean absolute error of the whole output against the oracle); "next", just
before it, does the same for the other legs.  The full per-workload records go
to stderr as one JSON line.

Under torchrun (N > 1) every rank runs its own replica of the workload (no
data-path collective); the step time is the max over ranks and `value` is the
bytes all ranks processed divided by it.  `--impl reference` times the fp64 CPU
oracle on a bounded sample of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode KV HBM GB/s & ragged prefill TFLOP/s, as fraction of GB300 roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Nominal peaks of one GB300, the denominators the decode and prefill targets are stated
# against: HBM3e at 8 TB/s, and dense BF16 tensor throughput of 2.25 PFLOP/s (NVIDIA's
# HGX B300 specification gives 36 PFLOPS FP16/BF16 per 8 GPUs with 2:4 sparsity, i.e.
# 4.5 sparse = 2.25 dense per GPU).
NOMINAL = {"hbm_gbs": 8000.0, "bf16_tflops": 2250.0}
# The targets: decode at >= 70 % of nominal HBM on the long-context workload, ragged
# prefill at >= 50 % of the nominal dense BF16 peak.
TARGETS = {"long_context_decode": 0.70, "ragged_prefill": 0.50}
# The five named workloads, by their index in the workload list.
CONFIGS = {"tiny_decode": 1, "llama8b_decode": 2, "long_context_decode": 3,
           "ragged_prefill": 4, "chunked_paged_prefill": 5}
STAT_REPS = 30          # individually timed steps behind the median / min figures
PARITY_MAX_ABS, PARITY_MEAN_ABS = 2e-2, 2e-3

# DRAM bytes (read + write) per launch from ncu captures, keyed by kernel, valid only
# for the source file hash they were measured on (otherwise reported as null).
TRAFFIC = {
    # ncu capture of one decode_tc_kernel<4> launch on the Llama-8B decode workload:
    # dram__bytes_read.sum 568.34 MB + dram__bytes_write.sum 5.08 MB
    "decode_partitions:llama8b_decode_b64_h32kv8_d128": {
        "src": "e53731200feeaa9e", "bytes_per_launch": 573424896},
    # ncu capture of one prefill_kernel<128,64,ragged> launch on the 16-request ragged
    # causal prefill: dram__bytes_read.sum 298.53 MB + dram__bytes_write.sum 108.54 MB
    "ragged_prefill:ragged_prefill_r16_h32kv8_d128": {
        "src": "fe29602adfbe4d3a", "bytes_per_launch": 407071488},
    # ncu capture of one prefill_kernel<256,64,paged> launch on the chunked paged prefill:
    # dram__bytes_read.sum 396.10 MB + dram__bytes_write.sum 23.06 MB
    "ragged_prefill:chunked_paged_prefill_r8_h16kv8_d256": {
        "src": "fe29602adfbe4d3a", "bytes_per_launch": 419157248},
    # ncu capture of one decode_tc8_kernel<4> launch on the Llama-8B decode workload over
    # an FP8 cache: dram__bytes_read.sum 284.49 MB + dram__bytes_write.sum 4.33 MB
    "decode_partitions:llama8b_decode_fp8_b64_h32kv8_d128": {
        "src": "c96d19f3ccc7f4f1", "bytes_per_launch": 288820224},
}


# ---------------------------------------------------------------------------------------
# host-side helpers (also exercised by the CPU tests)
# ---------------------------------------------------------------------------------------

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, \
            "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def source_hash(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "paged_kv_gqa_15_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_for(kernel, src_files, launches_bytes=None):
    rec = TRAFFIC.get(kernel)
    if not rec or rec.get("src") != source_hash(*src_files):
        return None
    return rec["bytes_per_launch"]


def roofline(bound, achieved, peak, unit, traffic, peak_kind):
    return {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
            "frac": round(achieved / peak, 4) if peak else None, "traffic": traffic,
            "peak_source": peak_kind}


def reduce_max(x: float, device=None) -> float:
    """Max of a float over all ranks (identity without torch.distributed)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(x: float, device=None) -> float:
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def aggregate_throughput(units_per_step_local: float, ms_per_step_local: float, device=None):
    """(whole-job units per second, max-over-ranks ms per step)."""
    ms = reduce_max(ms_per_step_local, device)
    units = reduce_sum(units_per_step_local, device)
    return units / (ms / 1e3), ms


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running.  Samples
    are time-stamped; `phase()` brackets a GPU-timed interval, and `summary_of_phases()`
    keeps only the samples taken inside such intervals (host-only work in between, such
    as the oracle legs, would otherwise add idle clocks)."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id=None, interval_ms=50):
        self.gpu_id = gpu_id
        self.interval_ms = interval_ms
        self.proc = None
        self.lines = []           # (monotonic time, csv line)
        self.phases = []          # (start, end) of GPU-timed intervals

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               f"--loop-ms={self.interval_ms}"]
        if self.gpu_id:
            cmd.insert(1, f"--id={self.gpu_id}")
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    class _Phase:
        def __init__(self, owner):
            self.owner = owner

        def __enter__(self):
            self.t0 = time.monotonic()
            return self

        def __exit__(self, *exc):
            self.owner.phases.append((self.t0, time.monotonic()))
            return False

    def phase(self):
        return ClockSampler._Phase(self)

    def _stop_proc(self):
        if self.proc is None:
            return False
        time.sleep(self.interval_ms / 1000.0 * 2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        return True

    def stop(self):
        if not self._stop_proc():
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        return self.summary([ln for _, ln in self.lines])

    def phase_lines(self):
        """The samples taken inside a GPU-timed phase (with one sampling interval of
        slack on either side)."""
        slack = self.interval_ms / 1000.0
        return [ln for t, ln in self.lines
                if any(a - slack <= t <= b + slack for a, b in self.phases)]

    def summary_of_phases(self):
        if not self._stop_proc():
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        return self.summary(self.phase_lines())

    @staticmethod
    def summary(lines):
        sm, smax, reasons, power = [], [], set(), []
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------------------
# GPU arms
# ---------------------------------------------------------------------------------------

# FP8 caches hold E4M3 codes of x / FP8_SCALE: N(0, 1) inputs then use the format's
# range (|x| / FP8_SCALE up to 448 for |x| <= 7) and read back as code value * FP8_SCALE.
FP8_SCALE = 1.0 / 64


def decode_setup(w, dev, split=True):
    import paged_kv_gqa_15_gb300 as pa
    t = w.tensors(dev)
    if w.kv_fp8:   # input preparation, outside any timed region
        for name in ("k_cache", "v_cache"):
            t[name] = (t[name].float() / FP8_SCALE).to(torch.float8_e4m3fn)
            torch.cuda.empty_cache()
    s = {"t": t,
         "bt": torch.from_numpy(w.block_tables).to(dev),
         "sl": torch.from_numpy(w.seq_lens).to(dev),
         "out": torch.empty_like(t["q"])}
    if w.new_token_write:
        s["slots"] = torch.from_numpy(w.slot_mapping).to(dev)
    s["ws"] = pa.alloc_workspace(pa.decode_split_workspace_size(
        w.batch, w.num_q_heads, w.head_dim, max(w.max_seq_len, 1)), dev)
    return s


def decode_step(w, s, stream, evs=None):
    """One hot-path step; records an event after each kernel when evs is a list."""
    import paged_kv_gqa_15_gb300 as pa
    t = s["t"]
    n = 0
    if evs is not None:
        evs.append(_ev(stream))
    scales = dict(k_scale=FP8_SCALE, v_scale=FP8_SCALE) if w.kv_fp8 else {}
    if w.new_token_write:
        pa.pa_write_cache(t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], s["slots"],
                          stream=stream, **scales)
        n += 1
        if evs is not None:
            evs.append(_ev(stream))
    if not w.split:   # the workload's decode is one pass over each sequence
        pa.pa_decode(s["out"], t["q"], t["k_cache"], t["v_cache"], s["bt"], s["sl"], w.scale,
                     stream=stream, sliding_window=w.window, **scales)
        if evs is not None:
            evs.append(_ev(stream))
        return n + 1
    L = max(w.max_seq_len, 1)
    pa.pa_decode_partitions(t["q"], t["k_cache"], t["v_cache"], s["bt"], s["sl"], w.scale, L,
                            s["ws"], stream=stream, sliding_window=w.window, **scales)
    if evs is not None:
        evs.append(_ev(stream))
    pa.pa_decode_merge(s["out"], s["sl"], L, s["ws"], stream=stream, sliding_window=w.window)
    if evs is not None:
        evs.append(_ev(stream))
    return n + 2


def _ev(stream):
    e = torch.cuda.Event(enable_timing=True)
    e.record(stream)
    return e


L2_FLUSH_BYTES = 512 << 20    # > 3x the 129 MB L2
_flush_buf = {}


def flush_l2(stream, device):
    """Overwrites a buffer much larger than L2 on `stream` (evicts the workload), then
    reads it back: the read evicts the buffer's own dirty lines, so their write-backs
    happen here and not inside the next timed step, which starts with L2 holding only
    clean lines of the flush buffer."""
    buf = _flush_buf.get(str(device))
    if buf is None:
        buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
        _flush_buf[str(device)] = buf
    with torch.cuda.stream(stream):
        buf.fill_(1)
        buf.sum(dtype=torch.int64)


def step_stats(ms_list):
    """Median, min, max and mean of individually timed steps (ms)."""
    return {"reps": len(ms_list), "median_ms": round(statistics.median(ms_list), 5),
            "min_ms": round(min(ms_list), 5), "max_ms": round(max(ms_list), 5),
            "mean_ms": round(sum(ms_list) / len(ms_list), 5)}


def time_steps(step, steps, warmup, stream, device, labels, flush=False, reps=STAT_REPS):
    """Warm up, then time exactly `steps` steps with CUDA events on `stream`.
    Without flush the step time comes from one pass with events only around the whole
    loop; with flush, L2 is flushed before every step, outside the timed intervals, and
    each step is timed on its own between two events.  Either way no event sits between
    a step's kernels, so the dependent launches overlap as in use.  A second pass times
    `reps` steps one by one (flushed the same way) for the median / min figures, and a
    third pass of `steps` steps with an event after every kernel gives the per-kernel
    times.  Returns {"ms": ms per step, "per": {label: avg ms}, "launches": launches of
    the timed pass, "stats": step_stats of the second pass}."""
    import torch.distributed as dist
    for _ in range(warmup):
        if flush:
            flush_l2(stream, device)
        step(None)
    torch.cuda.synchronize()
    if dist.is_available() and dist.is_initialized():
        dist.barrier()
    torch.cuda.synchronize()
    launches = 0
    if not flush:
        start = _ev(stream)
        for _ in range(steps):
            launches += step(None)
        end = _ev(stream)
        torch.cuda.synchronize()
        ms_whole = start.elapsed_time(end) / steps
    else:
        spans = []
        for _ in range(steps):
            flush_l2(stream, device)
            a = _ev(stream)
            launches += step(None)
            spans.append((a, _ev(stream)))
        torch.cuda.synchronize()
        ms_whole = sum(a.elapsed_time(b) for a, b in spans) / steps
    if dist.is_available() and dist.is_initialized():
        dist.barrier()
    spans = []
    for _ in range(reps):
        if flush:
            flush_l2(stream, device)
        a = _ev(stream)
        step(None)
        spans.append((a, _ev(stream)))
    torch.cuda.synchronize()
    stats = step_stats([a.elapsed_time(b) for a, b in spans])
    all_evs = []
    for _ in range(steps):
        if flush:
            flush_l2(stream, device)
        evs = []
        step(evs)
        all_evs.append(evs)
    torch.cuda.synchronize()
    if dist.is_available() and dist.is_initialized():
        dist.barrier()
    per = {l: 0.0 for l in labels}
    for evs in all_evs:
        for i, l in enumerate(labels):
            per[l] += evs[i].elapsed_time(evs[i + 1])
    per = {l: v / steps for l, v in per.items()}
    return {"ms": ms_whole, "per": per, "launches": launches, "stats": stats}


def decode_footprint(w):
    return 2 * w.num_blocks * w.num_kv_heads * w.block_size * w.head_dim * (1 if w.kv_fp8 else 2)


def prefill_footprint(w):
    qo = 2 * w.total_qo * w.num_q_heads * w.head_dim * 2
    if w.paged:
        return qo + 2 * w.num_blocks * w.num_kv_heads * w.block_size * w.head_dim * 2
    return qo + 2 * w.total_kv * w.num_kv_heads * w.head_dim * 2


def nominal_frac(achieved, bound):
    peak = NOMINAL["hbm_gbs"] if bound == "hbm" else NOMINAL["bf16_tflops"]
    return round(achieved / peak, 4)


def decode_kernel_sources(w):
    if not w.split:
        return ("pa_decode_kernel.cuh", "pa_device.cuh")
    if w.head_dim == 128 and w.num_q_heads // w.num_kv_heads in (4, 8):
        return (("pa_decode_tc_fp8.cu" if w.kv_fp8 else "pa_decode_tc.cu"), "pa_tcgen05.cuh",
                "pa_device.cuh")
    return ("pa_decode_kernel.cuh", "pa_device.cuh")


def bench_decode(w, steps, warmup, dev, stream, peaks, peak_kind, snapshot=False):
    """Times the decode step of workload w.  With snapshot, the step's inputs are copied
    to the host first (for the oracle leg) and the step's output after the timing."""
    s = decode_setup(w, dev)
    snap = decode_snapshot(w, s) if snapshot else None
    flush = decode_footprint(w) < L2_FLUSH_BYTES
    labels = (["write_cache"] if w.new_token_write else []) + (
        ["decode_partitions", "decode_merge"] if w.split else ["decode"])

    def step(evs):
        return decode_step(w, s, stream, evs)

    tm = time_steps(step, steps, warmup, stream, dev, labels, flush)
    kv = w.kv_bytes()
    value, ms_max = aggregate_throughput(kv, tm["ms"], dev)
    kern_ms = tm["per"]["decode_partitions" if w.split else "decode"]
    achieved = kv / (kern_ms / 1e3) / 1e9
    res = {
        "value": value / 1e9, "unit": "GB/s", "ms_per_step": ms_max,
        "kv_bytes_per_step": kv, "launches": tm["launches"], "step_stats": tm["stats"],
        "kernels_ms": {k: round(v, 5) for k, v in tm["per"].items()},
        "roofline": roofline("hbm", achieved, peaks["hbm_gbs"], "GB/s",
                             traffic_for("decode_partitions:" + w.name,
                                         decode_kernel_sources(w)), peak_kind),
        "roofline_nominal_frac": nominal_frac(achieved, "hbm"),
    }
    if snap is not None:
        snap["out"] = W_bits(s["out"])
    res["graph"] = bench_decode_graph(w, s, steps, warmup, dev, stream, flush)
    return res, s, snap


def W_bits(t):
    from paged_kv_gqa_15_gb300 import workloads as W
    return W.to_bits(t)


def decode_snapshot(w, s):
    """Host copies of a decode step's inputs, before any step ran: q and the new rows
    as bf16 bits, the pools as bf16 bits or E4M3 codes."""
    t = s["t"]
    snap = {"q": W_bits(t["q"]), "k_cache": host_pool(w, t["k_cache"]),
            "v_cache": host_pool(w, t["v_cache"])}
    if w.new_token_write:
        snap["k_new"], snap["v_new"] = W_bits(t["k_new"]), W_bits(t["v_new"])
    return snap


def bench_decode_graph(w, s, steps, warmup, dev, stream, flush):
    """The same step captured once in a CUDA graph and replayed (serving replays a
    captured decode); one graph launch replaces the step's kernel launches."""
    with torch.cuda.stream(stream):
        decode_step(w, s, stream, None)   # one-time set-up happens outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        n = decode_step(w, s, stream, None)
    torch.cuda.synchronize()

    def replay(evs):
        if evs is not None:
            evs.append(_ev(stream))
        with torch.cuda.stream(stream):
            graph.replay()
        if evs is not None:
            evs.append(_ev(stream))
        return n

    tm = time_steps(replay, steps, warmup, stream, dev, ["step"], flush)
    value, ms_max = aggregate_throughput(w.kv_bytes(), tm["ms"], dev)
    del graph
    return {"value": round(value / 1e9, 3), "unit": "GB/s", "ms_per_step": round(ms_max, 5),
            "kernels_per_replay": n, "median_ms": tm["stats"]["median_ms"]}


def bench_decode_e2e(w, s, steps, warmup, dev, stream):
    """Same step through the public calls with pinned host inputs copied in and the
    output copied out inside the timed region, pipelined as a serving loop does: the
    inputs and output are double-buffered on the device, a copy stream uploads step
    k + 1's inputs and reads back step k's output while the compute stream runs step k
    (events order the two), and the timed region ends after the last read-back."""
    import torch.distributed as dist
    t = s["t"]
    names = ["q", "bt", "sl"] + (["k_new", "v_new", "slots"] if w.new_token_write else [])

    def dev_of(state, name):
        return state["t"][name] if name in ("q", "k_new", "v_new") else state[name]

    # A step's inputs sit in one pinned staging buffer (256-byte-aligned fields), so each
    # step uploads them with one copy; the kernels read typed views of the device copy.
    offs, total = {}, 0
    for n in names:
        src = dev_of(s, n)
        offs[n] = (total, src.dtype, tuple(src.shape))
        total += (src.numel() * src.element_size() + 255) // 256 * 256
    stage_h = torch.empty(total, dtype=torch.uint8).pin_memory()
    stage_d = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(2)]

    def view(buf, n):
        o, dt, shape = offs[n]
        nbytes = int(np.prod(shape)) * torch.empty(0, dtype=dt).element_size()
        return buf[o:o + nbytes].view(dt).view(shape)

    for n in names:
        view(stage_h, n).copy_(dev_of(s, n).cpu())
    states = []
    for i in range(2):
        st = dict(s)
        st["t"] = dict(t)
        for n in names:
            if n in ("q", "k_new", "v_new"):
                st["t"][n] = view(stage_d[i], n)
            else:
                st[n] = view(stage_d[i], n)
        st["out"] = torch.empty_like(s["out"])
        states.append(st)
    out_h = [torch.empty(s["out"].shape, dtype=s["out"].dtype).pin_memory() for _ in range(2)]
    h2d = total                                # the staging copy, alignment padding included
    d2h = out_h[0].numel() * out_h[0].element_size()
    copy = torch.cuda.Stream(device=dev)
    uploaded = [torch.cuda.Event() for _ in range(2)]
    computed = [torch.cuda.Event() for _ in range(2)]
    for e in computed:
        e.record(stream)

    def upload(k):
        i = k % 2
        copy.wait_event(computed[i])          # step k - 2 no longer reads these buffers
        with torch.cuda.stream(copy):
            stage_d[i].copy_(stage_h, non_blocking=True)
            uploaded[i].record(copy)

    def run(k):
        i = k % 2
        stream.wait_event(uploaded[i])
        n = decode_step(w, states[i], stream, None)
        computed[i].record(stream)
        copy.wait_event(computed[i])
        with torch.cuda.stream(copy):
            out_h[i].copy_(states[i]["out"], non_blocking=True)
        return n

    def loop(k0, count):
        n = 0
        upload(k0)
        for k in range(k0, k0 + count):
            if k + 1 < k0 + count:
                upload(k + 1)                 # overlaps step k's kernels
            n += run(k)
        return n

    loop(0, max(warmup, 3))
    torch.cuda.synchronize()
    if dist.is_available() and dist.is_initialized():
        dist.barrier()
    torch.cuda.synchronize()
    start = _ev(stream)
    copy.wait_event(start)
    loop(0, steps)
    stream.wait_stream(copy)                  # the last read-back is inside the region
    end = _ev(stream)
    torch.cuda.synchronize()
    if dist.is_available() and dist.is_initialized():
        dist.barrier()
    ms = start.elapsed_time(end) / steps
    value, ms_max = aggregate_throughput(w.kv_bytes(), ms, dev)
    return {"value": round(value / 1e9, 3), "unit": "GB/s", "ms_per_step": round(ms_max, 5),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "pipelining": "double-buffered inputs and output; copies on a second stream "
                          "overlap the previous step's kernels"}


def prefill_setup(w, dev):
    import paged_kv_gqa_15_gb300 as pa
    t = w.tensors(dev)
    return {"t": t,
            "qo_d": torch.from_numpy(w.qo_indptr).to(dev),
            "kv_d": torch.from_numpy(w.kv_indptr).to(dev),
            "out": torch.empty_like(t["q"]),
            "ws": pa.alloc_workspace(pa.ragged_prefill_workspace_size(
                w.batch, w.total_qo, w.num_q_heads, w.head_dim), dev),
            "bt": torch.from_numpy(w.block_tables).to(dev) if w.paged else None,
            "slots": torch.from_numpy(w.chunk_slot_mapping).to(dev) if w.chunk_write else None}


def prefill_step(w, s, stream, evs=None):
    """One prefill step: the chunk's cache write (paged chunked prefill), then the ragged
    prefill; records an event after each kernel when evs is a list."""
    import paged_kv_gqa_15_gb300 as pa
    t = s["t"]
    n = 0
    if evs is not None:
        evs.append(_ev(stream))
    if w.chunk_write:
        pa.pa_write_cache(t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], s["slots"],
                          stream=stream)
        n += 1
        if evs is not None:
            evs.append(_ev(stream))
    k = t["k_cache"] if w.paged else t["k"]
    v = t["v_cache"] if w.paged else t["v"]
    pa.pa_ragged_prefill(s["out"], t["q"], k, v, w.qo_indptr, w.kv_indptr, s["qo_d"],
                         s["kv_d"], w.scale, causal=w.causal, block_tables=s["bt"],
                         workspace=s["ws"], stream=stream, sliding_window=w.window)
    if evs is not None:
        evs.append(_ev(stream))
    return n + 1


def bench_prefill(w, steps, warmup, dev, stream, peaks, peak_kind, snapshot=False):
    """Times the prefill step of workload w (with its chunk's cache write if it has one).
    With snapshot, the inputs go to the host first and the output after the timing."""
    s = prefill_setup(w, dev)
    snap = prefill_snapshot(w, s["t"]) if snapshot else None
    labels = (["write_cache"] if w.chunk_write else []) + ["ragged_prefill"]

    def step(evs):
        return prefill_step(w, s, stream, evs)

    tm = time_steps(step, steps, warmup, stream, dev, labels,
                    prefill_footprint(w) < L2_FLUSH_BYTES)
    flops = w.flops()
    value, ms_max = aggregate_throughput(flops, tm["ms"], dev)
    kern_ms = tm["per"]["ragged_prefill"]
    achieved = flops / (kern_ms / 1e3) / 1e12
    if snap is not None:
        snap["out"] = W_bits(s["out"])
    return {"value": value / 1e12, "unit": "TFLOP/s", "ms_per_step": ms_max,
            "flops_per_step": flops, "launches": tm["launches"], "step_stats": tm["stats"],
            "kernels_ms": {k: round(v, 5) for k, v in tm["per"].items()},
            "roofline": roofline("tensor", achieved, peaks["bf16_tflops"], "TFLOP/s",
                                 traffic_for("ragged_prefill:" + w.name,
                                             ("pa_prefill.cu", "pa_device.cuh")), peak_kind),
            "roofline_nominal_frac": nominal_frac(achieved, "tensor")}, snap


def prefill_snapshot(w, t):
    """Host copies of a prefill step's inputs (bf16 bits), before any step ran."""
    return {n: W_bits(v) for n, v in t.items()}


# Page-copy legs: a Llama-3-8B-shaped cache (32 layers x K and V pools of 1024
# 16-token pages, 8 kv heads x head_dim 128 bf16 = 32 KB per page, 2 GiB in all) and
# 256 pages per pool per call (a 4096-token context): 512 MiB of pages per call.
BLOCK_LEGS = ("copy_blocks_fork", "swap_blocks")
BLOCK_LAYERS, BLOCK_POOL_PAGES, BLOCK_PAIRS, BLOCK_PAGE = 32, 1024, 256, (8, 16, 128)


def blocks_config(name):
    cfg = {"workload": name, "layers": BLOCK_LAYERS, "pools": 2 * BLOCK_LAYERS,
           "pages_per_pool": BLOCK_POOL_PAGES, "pairs_per_call": BLOCK_PAIRS,
           "page_bytes": int(np.prod(BLOCK_PAGE)) * 2,
           "page": "8 kv heads x 16 tokens x head_dim 128 bf16", "l2": "inputs > L2 (no flush)"}
    if name == "swap_blocks":
        cfg["host_pool_pages"] = BLOCK_PAIRS
    return cfg


def bench_blocks(name, steps, warmup, dev, stream, peaks, peak_kind):
    """copy_blocks_fork: one pa_copy_blocks call duplicates 256 pages in all 64 pools
    (read + write 1 GiB of HBM).  swap_blocks: the same pages go out to pinned host pools
    and come back to other device pages, one pa_swap_blocks call per direction; the link
    is judged against a contiguous copy-engine copy of the same bytes timed here."""
    import paged_kv_gqa_15_gb300 as pa
    rng = np.random.default_rng(2024)
    perm = rng.permutation(BLOCK_POOL_PAGES)
    pools = [torch.empty((BLOCK_POOL_PAGES,) + BLOCK_PAGE, dtype=torch.bfloat16,
                         device=dev).normal_() for _ in range(2 * BLOCK_LAYERS)]
    page_bytes = int(np.prod(BLOCK_PAGE)) * 2
    moved = BLOCK_PAIRS * len(pools) * page_bytes          # bytes of pages per call
    stats = {}

    def timed(call, label):
        def step(evs):
            if evs is not None:
                evs.append(_ev(stream))
            call()
            if evs is not None:
                evs.append(_ev(stream))
            return 1
        tm = time_steps(step, steps, warmup, stream, dev, [label])
        stats[label] = tm["stats"]
        return tm["ms"], tm["launches"]

    if name == "copy_blocks_fork":
        pairs = np.stack([perm[:BLOCK_PAIRS], perm[BLOCK_PAIRS:2 * BLOCK_PAIRS]], 1)
        m = torch.from_numpy(pairs.astype(np.int64)).to(dev)
        keys, vals = pools[0::2], pools[1::2]
        call = lambda: pa.pa_copy_blocks(keys, vals, m, stream=stream)
        # A direct call costs the host about as long as the kernel runs (the binding
        # gathers 64 pool pointers), so timed call by call the device can idle between
        # kernels and the figure follows the host's speed.  The call is captured once in
        # a CUDA graph and replayed, so the timing is the device's; the host's cost per
        # direct call is reported beside it.
        with torch.cuda.stream(stream):
            call()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            call()
        torch.cuda.synchronize()

        def replay():
            with torch.cuda.stream(stream):
                graph.replay()
        ms, n = timed(replay, "copy_blocks")
        t0 = time.perf_counter()
        for _ in range(20):
            call()
        host_us = (time.perf_counter() - t0) / 20 * 1e6
        torch.cuda.synchronize()
        ms_direct, _ = timed(call, "copy_blocks_direct")
        del graph
        hbm = 2 * moved / (ms / 1e3) / 1e9                  # read + write
        st = stats["copy_blocks"]
        return {"value": round(hbm, 2), "unit": "GB/s", "ms_per_step": round(ms, 5),
                "bytes_per_step": 2 * moved, "launches": n, "step_stats": st,
                "median_GB/s": round(2 * moved / (st["median_ms"] / 1e3) / 1e9, 2),
                "max_GB/s": round(2 * moved / (st["min_ms"] / 1e3) / 1e9, 2),
                "kernels_ms": {"copy_blocks": round(ms, 5)},
                "timing": "CUDA graph replays of one captured pa_copy_blocks call",
                "direct_calls": {"GB/s": round(2 * moved / (ms_direct / 1e3) / 1e9, 2),
                                 "host_us_per_call": round(host_us, 1)},
                "roofline": roofline("hbm", hbm, peaks["hbm_gbs"], "GB/s", None, peak_kind),
                "roofline_nominal_frac": nominal_frac(hbm, "hbm"),
                "config": blocks_config(name)}

    host = [torch.empty((BLOCK_PAIRS,) + BLOCK_PAGE, dtype=torch.bfloat16).pin_memory()
            for _ in pools]
    out_pairs = np.stack([perm[:BLOCK_PAIRS], np.arange(BLOCK_PAIRS)], 1).astype(np.int64)
    in_pairs = np.stack([np.arange(BLOCK_PAIRS), perm[2 * BLOCK_PAIRS:3 * BLOCK_PAIRS]],
                        1).astype(np.int64)
    m_out = torch.from_numpy(out_pairs).to(dev)
    m_in = torch.from_numpy(in_pairs).to(dev)
    ms_out, n1 = timed(lambda: pa.pa_swap_blocks(pools, host, m_out, stream=stream), "swap_out")
    ms_in, n2 = timed(lambda: pa.pa_swap_blocks(host, pools, m_in, stream=stream), "swap_in")
    # the link's copy-engine rate for the same bytes, as one contiguous copy each way
    dbuf = torch.empty(moved, dtype=torch.uint8, device=dev)
    hbuf = torch.empty(moved, dtype=torch.uint8).pin_memory()

    def ce(dst, src):
        with torch.cuda.stream(stream):
            dst.copy_(src, non_blocking=True)
    ce_out, _ = timed(lambda: ce(hbuf, dbuf), "ce_out")
    ce_in, _ = timed(lambda: ce(dbuf, hbuf), "ce_in")
    del dbuf, hbuf, host
    gbs = lambda ms: moved / (ms / 1e3) / 1e9
    both, both_ce = 2 * moved / ((ms_out + ms_in) / 1e3) / 1e9, \
        2 * moved / ((ce_out + ce_in) / 1e3) / 1e9
    rl = roofline("link", both, round(both_ce, 2), "GB/s", None,
                  "measured here: one contiguous cudaMemcpyAsync of the same bytes each way "
                  "between pinned host memory and the device")
    return {"value": round(both, 2), "unit": "GB/s", "ms_per_step": round(ms_out + ms_in, 5),
            "bytes_per_step": 2 * moved, "launches": n1 + n2,
            "kernels_ms": {"swap_out": round(ms_out, 5), "swap_in": round(ms_in, 5)},
            "out": {"GB/s": round(gbs(ms_out), 2), "copy_engine_GB/s": round(gbs(ce_out), 2)},
            "in": {"GB/s": round(gbs(ms_in), 2), "copy_engine_GB/s": round(gbs(ce_in), 2)},
            "step_stats": {"swap_out": stats["swap_out"], "swap_in": stats["swap_in"]},
            "roofline": rl, "config": blocks_config(name)}


# ---------------------------------------------------------------------------------------
# oracle (CPU) arm
# ---------------------------------------------------------------------------------------

def oracle_decode_time(w, t_host, seqs, nthreads):
    """Runs the fp64 oracle on the given sequences; returns (seconds, KV bytes)."""
    import oracle
    q, kc, vc = t_host
    seqs = np.asarray(seqs)
    t0 = time.perf_counter()
    oracle.decode(q[seqs], kc, vc, w.block_tables[seqs], w.seq_lens[seqs], w.num_kv_heads,
                  w.block_size, w.scale, nthreads=nthreads, window=w.window, kv_fp8=w.kv_fp8,
                  k_scale=FP8_SCALE, v_scale=FP8_SCALE)
    dt = time.perf_counter() - t0
    lens = w.seq_lens[seqs].astype(np.int64)
    if w.window > 0:
        lens = np.minimum(lens, w.window)
    kv = int(lens.sum()) * w.num_kv_heads * w.head_dim * 2 * (1 if w.kv_fp8 else 2)
    return dt, kv


def oracle_decode_sample(w, t_host, target_s=12.0, nthreads=None):
    """Times the fp64 oracle on a bounded sample of the workload lasting about target_s
    seconds: the first n sequences if the whole batch takes longer than that, else
    whole passes over the batch, repeated.  Returns (GB/s, seconds, n, passes, threads)."""
    import oracle
    nthreads = nthreads or oracle.default_threads()
    one, _ = oracle_decode_time(w, t_host, [0], nthreads)
    n = int(max(1, min(w.batch, math.floor(target_s / max(one, 1e-4)))))
    dt, kv = oracle_decode_time(w, t_host, np.arange(n), nthreads)
    passes = 1
    while n == w.batch and dt < target_s and passes < 10000:
        d, b = oracle_decode_time(w, t_host, np.arange(n), nthreads)
        dt, kv, passes = dt + d, kv + b, passes + 1
    return kv / dt / 1e9, dt, n, passes, nthreads


def _parity(got_bits, ref):
    """Max / mean absolute error of a bf16 output (bits) against the fp64 oracle, over
    every element; ok when both are inside the bounds the tests use."""
    from paged_kv_gqa_15_gb300 import workloads as W
    got = W.bits_to_float(got_bits).astype(np.float64)
    finite = bool(np.isfinite(got).all())
    err = np.abs(got - ref)
    mx, mean = float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0
    return {"max_abs": round(mx, 6), "mean_abs": round(mean, 7), "elements": int(err.size),
            "ok": finite and mx <= PARITY_MAX_ABS and mean <= PARITY_MEAN_ABS}


def oracle_leg(w, snap, one_thread=False, target_1t_s=3.0):
    """The fp64 oracle run once over the whole workload on all host cores, on the host
    copies of the step's inputs: the step's cache write (if any), then the attention.
    That run is timed (the oracle's throughput in the workload's unit) and its result is
    compared with the GPU step's output on every element.  With one_thread, the oracle
    is also timed on one thread over a bounded sample (whole sequences, about
    target_1t_s seconds)."""
    import oracle
    from paged_kv_gqa_15_gb300 import workloads as W
    th = oracle.default_threads()
    scales = dict(k_scale=FP8_SCALE, v_scale=FP8_SCALE)
    if isinstance(w, W.DecodeWorkload):
        kc, vc = snap["k_cache"], snap["v_cache"]
        t0 = time.perf_counter()
        if w.new_token_write:
            oracle.write_cache(snap["k_new"], snap["v_new"], kc, vc, w.slot_mapping,
                               w.block_size, kv_fp8=w.kv_fp8, **scales)
        ref = oracle.decode(snap["q"], kc, vc, w.block_tables, w.seq_lens, w.num_kv_heads,
                            w.block_size, w.scale, nthreads=th, window=w.window,
                            kv_fp8=w.kv_fp8, **scales)
        dt = time.perf_counter() - t0
        cpu = {"value": round(w.kv_bytes() / dt / 1e9, 4), "unit": "GB/s", "cores": th,
               "kind": "oracle", "seconds": round(dt, 3),
               "sample": "the whole workload once (cache write + decode of every sequence "
                         "and head)"}
        if one_thread:
            n, dt1, kv1 = 0, 0.0, 0
            while n < w.batch and dt1 < target_1t_s:
                d, b = oracle_decode_time(w, (snap["q"], kc, vc), [n], 1)
                dt1, kv1, n = dt1 + d, kv1 + b, n + 1
            cpu["one_thread"] = {"value": round(kv1 / dt1 / 1e9, 4), "unit": "GB/s",
                                 "sample": f"{n} of {w.batch} sequences, {dt1:.1f} s"}
    else:
        q = snap["q"]
        t0 = time.perf_counter()
        if w.paged:
            k, v = snap["k_cache"], snap["v_cache"]
            if w.chunk_write:
                oracle.write_cache(snap["k_new"], snap["v_new"], k, v, w.chunk_slot_mapping,
                                   w.block_size)
        else:
            k, v = snap["k"], snap["v"]
        ref = oracle.prefill(q, k, v, w.qo_indptr, w.kv_indptr, w.num_kv_heads, w.scale,
                             causal=w.causal, block_tables=w.block_tables if w.paged else None,
                             block_size=w.block_size, nthreads=th, window=w.window)
        dt = time.perf_counter() - t0
        cpu = {"value": round(w.flops() / dt / 1e12, 5), "unit": "TFLOP/s", "cores": th,
               "kind": "oracle", "seconds": round(dt, 3),
               "sample": "the whole workload once (every query row and head" +
                         (", after the chunk's cache write)" if w.chunk_write else ")")}
    return cpu, _parity(snap["out"], ref)


def host_pool(w, pool):
    """Host copy of a pool for the oracle: bf16 bits, or E4M3 codes of an fp8
    workload (quantised here if the pool is still bf16)."""
    from paged_kv_gqa_15_gb300 import workloads as W
    if not w.kv_fp8:
        return W.to_bits(pool)
    if pool.dtype == torch.bfloat16:
        pool = (pool.float() / FP8_SCALE).to(torch.float8_e4m3fn)
    return pool.cpu().view(torch.uint8).numpy()


def host_decode_inputs(w, t):
    from paged_kv_gqa_15_gb300 import workloads as W
    return W.to_bits(t["q"]), host_pool(w, t["k_cache"]), host_pool(w, t["v_cache"])


def run_reference(args, w, rank):
    """The oracle as the reference arm: each step is a bounded sample (n of the
    workload's sequences, cycling through the batch) sized so that the whole
    --warmup + --steps run takes about 90 s of host time."""
    if rank != 0:
        return None
    import oracle
    from paged_kv_gqa_15_gb300 import workloads as W
    t = w.tensors("cpu")
    host = host_decode_inputs(w, t)
    th = oracle.default_threads()
    per_step = 90.0 / max(args.steps + args.warmup, 1)
    one, _ = oracle_decode_time(w, host, [0], th)
    n = int(max(1, min(w.batch, math.floor(per_step / max(one, 1e-4)))))
    cursor = 0

    def next_seqs():
        nonlocal cursor
        seqs = [(cursor + i) % w.batch for i in range(n)]
        cursor = (cursor + n) % w.batch
        return seqs

    for _ in range(args.warmup):
        oracle_decode_time(w, host, next_seqs(), th)
    tot_s, tot_b = 0.0, 0
    for _ in range(args.steps):
        dt, kv = oracle_decode_time(w, host, next_seqs(), th)
        tot_s += dt
        tot_b += kv
    value = tot_b / tot_s / 1e9
    sample = (f"fp64 oracle decode of {n} of the {w.batch} sequences per step (all "
              f"{w.num_q_heads} heads, cycling through the batch), {tot_s:.1f} s over "
              f"{args.steps} steps")
    return {"metric": METRIC, "impl": "reference", "value": round(value, 4), "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(tot_s / max(args.steps, 1) * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(w),
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": th,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def l2_note(footprint):
    if footprint < L2_FLUSH_BYTES:
        return ("inputs %.0f MB: L2 flushed (512 MB written, then read back) before every "
                "timed step, outside the timed intervals" % (footprint / 1e6))
    return "inputs larger than L2 (%.0f MB > 129 MB); no flush" % (footprint / 1e6)


def workload_config(w):
    from paged_kv_gqa_15_gb300 import workloads as W
    if isinstance(w, W.DecodeWorkload):
        return {"workload": w.name, "batch": w.batch, "num_q_heads": w.num_q_heads,
                "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
                "block_size": w.block_size,
                "seq_lens": f"U[{int(w.seq_lens.min())},{int(w.seq_lens.max())}] seed {w.seed}",
                "num_blocks": w.num_blocks, "kv_bytes_per_step": w.kv_bytes(),
                "sliding_window": w.window or None,
                "kv_cache_dtype": "fp8_e4m3" if w.kv_fp8 else "bf16",
                "kv_scales": FP8_SCALE if w.kv_fp8 else None, "l2": l2_note(decode_footprint(w))}
    return {"workload": w.name, "batch": w.batch, "num_q_heads": w.num_q_heads,
            "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "causal": w.causal,
            "paged": w.paged, "total_qo": w.total_qo, "total_kv": w.total_kv,
            "sliding_window": w.window or None, "flops_per_step": w.flops(),
            "l2": l2_note(prefill_footprint(w))}


# ---------------------------------------------------------------------------------------

def compact(name, r):
    """A short summary of one workload's record, for the tail of the printed line."""
    if "unavailable" in r:
        return {"unavailable": r["unavailable"]}
    e = {r["unit"]: round(r["value"], 2)}
    rl = r.get("roofline") or {}
    km = r.get("kernels_ms") or {}
    main_k = next((k for k in ("decode_partitions", "decode", "ragged_prefill", "copy_blocks")
                   if k in km), None)
    if main_k:
        e["kernel_ms"] = km[main_k]
    if rl.get("frac") is not None:
        e["frac"] = rl["frac"]
    if "roofline_nominal_frac" in r:
        e["frac_nominal"] = r["roofline_nominal_frac"]
    st = r.get("step_stats") or {}
    if "median_ms" in st:
        e["median_ms"], e["min_ms"] = st["median_ms"], st["min_ms"]
    if name in TARGETS:
        e["target_nominal"] = TARGETS[name]
        e["met"] = r.get("roofline_nominal_frac", 0) >= TARGETS[name]
    cpu = r.get("cpu")
    if cpu:
        e["oracle"] = cpu["value"]
        e["oracle_cores"] = cpu["cores"]
        if "one_thread" in cpu:
            e["oracle_1t"] = cpu["one_thread"]["value"]
    par = r.get("parity")
    if par:
        e["max_abs"], e["mean_abs"], e["parity_ok"] = par["max_abs"], par["mean_abs"], par["ok"]
    return e


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama8b_decode")
    ap.add_argument("--extra", default="tiny_decode,long_context_decode,ragged_prefill,"
                                       "chunked_paged_prefill,window_decode,window_prefill,"
                                       "llama8b_decode_fp8,long_context_decode_fp8,"
                                       "llama8b_decode_single,mha_decode,gqa7_decode,"
                                       "copy_blocks_fork,swap_blocks",
                    help="other workloads measured in the same run (N=1 only); 'none' for none")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the oracle legs (timing and whole-output parity)")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)

    from paged_kv_gqa_15_gb300 import workloads as W
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    w = W.WORKLOADS[args.workload]()

    if args.impl == "reference":
        res = run_reference(args, w, rank)
        if res is not None:
            print(json.dumps(res), flush=True)
        return 0

    import __graft_entry__
    import paged_kv_gqa_15_gb300 as pa
    if not os.path.exists(pa.LIB_PATH):
        __graft_entry__.build_library()
    pa.load()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    stream = torch.cuda.Stream(device=dev)
    peaks, peak_kind = load_peaks()
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        uuid = None
    oracle_on = rank == 0 and world == 1 and not args.no_cpu_baseline

    clocks = ClockSampler(uuid)
    clocks.start()
    is_decode = isinstance(w, W.DecodeWorkload)
    if is_decode:
        res, state, snap = bench_decode(w, args.steps, args.warmup, dev, stream, peaks,
                                        peak_kind, snapshot=oracle_on)
    else:
        (res, snap), state = bench_prefill(w, args.steps, args.warmup, dev, stream, peaks,
                                           peak_kind, snapshot=oracle_on), None
    clk_main = clocks.stop()
    e2e = bench_decode_e2e(w, state, args.steps, args.warmup, dev, stream) if is_decode else None
    status = pa.device_status(stream)
    if snap is not None:
        res["cpu"], res["parity"] = oracle_leg(w, snap, one_thread=args.workload in
                                               ("tiny_decode", "llama8b_decode",
                                                "long_context_decode"))
        del snap
    records = {args.workload: res}

    clocks_all = ClockSampler(uuid)
    clocks_all.start()
    if world == 1 and args.extra:
        for name in [x for x in args.extra.split(",") if x and x not in ("none", args.workload)]:
            if name in BLOCK_LEGS:
                with clocks_all.phase():
                    records[name] = bench_blocks(name, max(STAT_REPS, min(args.steps, 50)),
                                                 args.warmup, dev, stream, peaks, peak_kind)
                torch.cuda.empty_cache()
                continue
            wx = W.WORKLOADS[name]()
            snap = None
            try:
                with clocks_all.phase():
                    if isinstance(wx, W.DecodeWorkload):
                        steps = max(3, min(args.steps, 50)) if wx.kv_bytes() > 1e9 \
                            else args.steps
                        r, _, snap = bench_decode(wx, steps, args.warmup, dev, stream, peaks,
                                                  peak_kind, snapshot=oracle_on)
                    else:
                        r, snap = bench_prefill(wx, max(3, min(args.steps, 50)), args.warmup,
                                                dev, stream, peaks, peak_kind,
                                                snapshot=oracle_on)
                r["config"] = workload_config(wx)
                records[name] = r
            except pa.PaError as e:
                records[name] = {"unavailable": str(e)}
            torch.cuda.empty_cache()
            if snap is not None:     # host-only work, outside the clock phases
                records[name]["cpu"], records[name]["parity"] = oracle_leg(
                    wx, snap, one_thread=CONFIGS.get(name, 0) in (1, 2, 3))
                del snap
        status |= pa.device_status(stream)
    clk_all = clocks_all.summary_of_phases()
    clk = dict(clk_main)
    clk["extra_workloads"] = clk_all

    cpu = None
    if oracle_on and is_decode:
        # the contract's CPU baseline: the oracle on the headline workload, whole passes
        # repeated for about 12 s (the single pass above is too short to time alone)
        t = state["t"]
        host = host_decode_inputs(w, t)
        gbs, dt, n, passes, th = oracle_decode_sample(w, host)
        cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": th, "kind": "oracle",
               "sample": f"fp64 oracle decode of {n} of {w.batch} sequences x {passes} "
                         f"pass(es) (all {w.num_q_heads} heads, {dt:.1f} s)"}

    if rank == 0:
        configs = {f"c{CONFIGS[n]}_{n}": compact(n, r)
                   for n, r in sorted(records.items(), key=lambda kv: CONFIGS.get(kv[0], 0))
                   if n in CONFIGS}
        nxt = {n: compact(n, r) for n, r in records.items() if n not in CONFIGS}
        parity_ok = all(r.get("parity", {}).get("ok", True) for r in records.values())
        line = {
            "metric": METRIC, "value": round(res["value"], 3), "unit": res["unit"],
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(res["ms_per_step"], 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16 (fp32 accumulate)",
            "data": "synthetic", "config": workload_config(w),
            "roofline": res["roofline"], "roofline_nominal_frac": res["roofline_nominal_frac"],
            "kernels_ms": res["kernels_ms"], "step_stats": res["step_stats"],
            "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": res["launches"], "clocks": clk, "device_status": status,
            "graph": res.get("graph"),
            "parity_all_ok": parity_ok if oracle_on else None,
            "nominal_peaks": NOMINAL,
            "next": nxt,
            "configs": configs,
        }
        sys.stderr.write("bench records: " + json.dumps(records, default=float) + "\n")
        sys.stderr.flush()
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
