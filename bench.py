"""Benchmark of the paged-KV GQA attention hot path on GB300.

One step = one pass of the hot path over one batch of synthetic input:
  pa_write_cache (the batch's new tokens) -> pa_decode_partitions -> pa_decode_merge
on the Llama-3-8B-shaped decode workload (64 sequences, 32 q / 8 kv heads,
head_dim 128, 16-token pages, seq_lens U[512, 4096], shuffled block tables).
The metric is decode KV-bytes GB/s (K and V of every visible token per step).
The other workloads (long-context split decode, tiny decode, ragged prefill,
chunked paged prefill) are measured in the same run and reported under
"workloads", each with its own roofline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

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

# DRAM bytes (read + write) per launch from ncu captures, keyed by kernel, valid only
# for the source file hash they were measured on (otherwise reported as null).
TRAFFIC = {
    # ncu capture of one decode_tc_kernel<4> launch on the Llama-8B decode workload:
    # dram__bytes_read.sum 568.32 MB + dram__bytes_write.sum 5.49 MB
    "decode_partitions:llama8b_decode_b64_h32kv8_d128": {
        "src": "23c62bb4aa65e8f7", "bytes_per_launch": 573813760},
    # ncu capture of one prefill_kernel<128,64,ragged> launch on the 16-request ragged
    # causal prefill: dram__bytes_read.sum 294.99 MB + dram__bytes_write.sum 108.21 MB
    # (captured on source 024cc71c5a1bbe51; re-keyed after a comment-only edit)
    "ragged_prefill:ragged_prefill_r16_h32kv8_d128": {
        "src": "3ff2430e17fafd35", "bytes_per_launch": 403205632},
    # ncu capture of one decode_tc8_kernel<4> launch on the Llama-8B decode workload over
    # an FP8 cache: dram__bytes_read.sum 284.47 MB + dram__bytes_write.sum 4.72 MB
    "decode_partitions:llama8b_decode_fp8_b64_h32kv8_d128": {
        "src": "a9c251812034d7df", "bytes_per_launch": 289189888},
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
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id=None, interval_ms=50):
        self.gpu_id = gpu_id
        self.interval_ms = interval_ms
        self.proc = None
        self.lines = []

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
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(self.interval_ms / 1000.0 * 2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        return self.summary(self.lines)

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


def time_steps(step, steps, warmup, stream, device, labels, flush=False):
    """Warm up, then time exactly `steps` steps with CUDA events on `stream`.
    Without flush the step time comes from one pass with events only around the whole
    loop; with flush, L2 is flushed before every step, outside the timed intervals, and
    each step is timed on its own between two events.  Either way no event sits between
    a step's kernels, so the dependent launches overlap as in use.  A second pass of
    `steps` steps with an event after every kernel gives the per-kernel times.
    Returns (ms per step, {label: avg ms}, launches per timed pass)."""
    import torch.distributed as dist
    for _ in range(warmup):
        if flush:
            flush_l2(stream, device)
        step(None)
    torch.cuda.synchronize()
    if dist.is_available() and dist.is_initialized():
        dist.barrier()
    torch.cuda.synchronize()
    if not flush:
        start = _ev(stream)
        for _ in range(steps):
            step(None)
        end = _ev(stream)
        torch.cuda.synchronize()
        ms_whole = start.elapsed_time(end) / steps
    else:
        spans = []
        for _ in range(steps):
            flush_l2(stream, device)
            a = _ev(stream)
            step(None)
            spans.append((a, _ev(stream)))
        torch.cuda.synchronize()
        ms_whole = sum(a.elapsed_time(b) for a, b in spans) / steps
    all_evs = []
    launches = 0
    for _ in range(steps):
        if flush:
            flush_l2(stream, device)
        evs = []
        launches += step(evs)
        all_evs.append(evs)
    torch.cuda.synchronize()
    if dist.is_available() and dist.is_initialized():
        dist.barrier()
    per = {l: 0.0 for l in labels}
    for evs in all_evs:
        for i, l in enumerate(labels):
            per[l] += evs[i].elapsed_time(evs[i + 1])
    per = {l: v / steps for l, v in per.items()}
    return ms_whole, per, launches


def decode_footprint(w):
    return 2 * w.num_blocks * w.num_kv_heads * w.block_size * w.head_dim * (1 if w.kv_fp8 else 2)


def prefill_footprint(w):
    qo = 2 * w.total_qo * w.num_q_heads * w.head_dim * 2
    if w.paged:
        return qo + 2 * w.num_blocks * w.num_kv_heads * w.block_size * w.head_dim * 2
    return qo + 2 * w.total_kv * w.num_kv_heads * w.head_dim * 2


def bench_decode(w, steps, warmup, dev, stream, peaks, peak_kind):
    s = decode_setup(w, dev)
    flush = decode_footprint(w) < L2_FLUSH_BYTES
    labels = (["write_cache"] if w.new_token_write else []) + (
        ["decode_partitions", "decode_merge"] if w.split else ["decode"])

    def step(evs):
        return decode_step(w, s, stream, evs)

    ms, per, launches = time_steps(step, steps, warmup, stream, dev, labels, flush)
    kv = w.kv_bytes()
    value, ms_max = aggregate_throughput(kv, ms, dev)
    kern_ms = per["decode_partitions" if w.split else "decode"]
    src = (("pa_decode_tc_fp8.cu" if w.kv_fp8 else "pa_decode_tc.cu"), "pa_tcgen05.cuh",
           "pa_device.cuh") if w.split else ("pa_decode_kernel.cuh", "pa_device.cuh")
    res = {
        "value": value / 1e9, "unit": "GB/s", "ms_per_step": ms_max,
        "kv_bytes_per_step": kv, "launches": launches,
        "kernels_ms": {k: round(v, 5) for k, v in per.items()},
        "roofline": roofline("hbm", kv / (kern_ms / 1e3) / 1e9, peaks["hbm_gbs"], "GB/s",
                             traffic_for("decode_partitions:" + w.name, src), peak_kind),
        "roofline_nominal_frac": round(kv / (kern_ms / 1e3) / 1e9 / 8000.0, 4),
    }
    res["graph"] = bench_decode_graph(w, s, steps, warmup, dev, stream, flush)
    return res, s


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

    ms, _, _ = time_steps(replay, steps, warmup, stream, dev, ["step"], flush)
    value, ms_max = aggregate_throughput(w.kv_bytes(), ms, dev)
    del graph
    return {"value": round(value / 1e9, 3), "unit": "GB/s", "ms_per_step": round(ms_max, 5),
            "kernels_per_replay": n}


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


def bench_prefill(w, steps, warmup, dev, stream, peaks, peak_kind):
    import paged_kv_gqa_15_gb300 as pa
    t = w.tensors(dev)
    qo_d = torch.from_numpy(w.qo_indptr).to(dev)
    kv_d = torch.from_numpy(w.kv_indptr).to(dev)
    o = torch.empty_like(t["q"])
    ws = pa.alloc_workspace(pa.ragged_prefill_workspace_size(w.batch, w.total_qo, w.num_q_heads,
                                                             w.head_dim), dev)
    bt = torch.from_numpy(w.block_tables).to(dev) if w.paged else None
    slots = torch.from_numpy(w.chunk_slot_mapping).to(dev) if w.chunk_write else None
    labels = (["write_cache"] if w.chunk_write else []) + ["ragged_prefill"]

    def step(evs):
        n = 0
        if evs is not None:
            evs.append(_ev(stream))
        if w.chunk_write:
            pa.pa_write_cache(t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], slots,
                              stream=stream)
            n += 1
            if evs is not None:
                evs.append(_ev(stream))
        k = t["k_cache"] if w.paged else t["k"]
        v = t["v_cache"] if w.paged else t["v"]
        pa.pa_ragged_prefill(o, t["q"], k, v, w.qo_indptr, w.kv_indptr, qo_d, kv_d, w.scale,
                             causal=w.causal, block_tables=bt, workspace=ws, stream=stream,
                             sliding_window=w.window)
        if evs is not None:
            evs.append(_ev(stream))
        return n + 1

    ms, per, launches = time_steps(step, steps, warmup, stream, dev, labels,
                                   prefill_footprint(w) < L2_FLUSH_BYTES)
    flops = w.flops()
    value, ms_max = aggregate_throughput(flops, ms, dev)
    kern_ms = per["ragged_prefill"]
    achieved = flops / (kern_ms / 1e3) / 1e12
    return {"value": value / 1e12, "unit": "TFLOP/s", "ms_per_step": ms_max,
            "flops_per_step": flops, "launches": launches,
            "kernels_ms": {k: round(v, 5) for k, v in per.items()},
            "roofline": roofline("tensor", achieved, peaks["bf16_tflops"], "TFLOP/s",
                                 traffic_for("ragged_prefill:" + w.name,
                                             ("pa_prefill.cu", "pa_device.cuh")), peak_kind),
            "roofline_nominal_frac": round(achieved / 2250.0, 4)}


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

    def timed(call, label):
        def step(evs):
            if evs is not None:
                evs.append(_ev(stream))
            call()
            if evs is not None:
                evs.append(_ev(stream))
            return 1
        ms, _, n = time_steps(step, steps, warmup, stream, dev, [label])
        return ms, n

    if name == "copy_blocks_fork":
        pairs = np.stack([perm[:BLOCK_PAIRS], perm[BLOCK_PAIRS:2 * BLOCK_PAIRS]], 1)
        m = torch.from_numpy(pairs.astype(np.int64)).to(dev)
        ms, n = timed(lambda: pa.pa_copy_blocks(pools[0::2], pools[1::2], m, stream=stream),
                      "copy_blocks")
        hbm = 2 * moved / (ms / 1e3) / 1e9                  # read + write
        return {"value": round(hbm, 2), "unit": "GB/s", "ms_per_step": round(ms, 5),
                "bytes_per_step": 2 * moved, "launches": n,
                "kernels_ms": {"copy_blocks": round(ms, 5)},
                "roofline": roofline("hbm", hbm, peaks["hbm_gbs"], "GB/s", None, peak_kind),
                "roofline_nominal_frac": round(hbm / 8000.0, 4),
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

def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama8b_decode")
    ap.add_argument("--extra", default="long_context_decode,tiny_decode,ragged_prefill,"
                                       "chunked_paged_prefill,window_decode,window_prefill,"
                                       "llama8b_decode_fp8,long_context_decode_fp8,"
                                       "copy_blocks_fork,swap_blocks",
                    help="other workloads measured in the same run (N=1 only); 'none' for none")
    ap.add_argument("--no-cpu-baseline", action="store_true")
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

    clocks = ClockSampler(uuid)
    clocks.start()
    is_decode = isinstance(w, W.DecodeWorkload)
    if is_decode:
        res, state = bench_decode(w, args.steps, args.warmup, dev, stream, peaks, peak_kind)
    else:
        res, state = bench_prefill(w, args.steps, args.warmup, dev, stream, peaks,
                                   peak_kind), None
    clk_main = clocks.stop()
    e2e = bench_decode_e2e(w, state, args.steps, args.warmup, dev, stream) if is_decode else None
    status = pa.device_status(stream)
    clocks_all = ClockSampler(uuid)
    clocks_all.start()

    extra = {}
    if world == 1 and args.extra:
        for name in [x for x in args.extra.split(",") if x and x not in ("none", args.workload)]:
            if name in BLOCK_LEGS:
                extra[name] = bench_blocks(name, max(3, min(args.steps, 50)), args.warmup, dev,
                                           stream, peaks, peak_kind)
                torch.cuda.empty_cache()
                continue
            wx = W.WORKLOADS[name]()
            try:
                if isinstance(wx, W.DecodeWorkload):
                    steps = max(3, min(args.steps, 50)) if wx.kv_bytes() > 1e9 else args.steps
                    r, _ = bench_decode(wx, steps, args.warmup, dev, stream, peaks, peak_kind)
                else:
                    r = bench_prefill(wx, max(3, min(args.steps, 50)), args.warmup, dev, stream,
                                      peaks, peak_kind)
                r["config"] = workload_config(wx)
                extra[name] = r
            except pa.PaError as e:
                extra[name] = {"unavailable": str(e)}
            torch.cuda.empty_cache()
        status |= pa.device_status(stream)
    clk_all = clocks_all.stop()
    clk = dict(clk_main)
    clk["extra_workloads"] = clk_all

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and is_decode:
        t = state["t"]
        host = host_decode_inputs(w, t)
        gbs, dt, n, passes, th = oracle_decode_sample(w, host)
        cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": th, "kind": "oracle",
               "sample": f"fp64 oracle decode of {n} of {w.batch} sequences x {passes} "
                         f"pass(es) (all {w.num_q_heads} heads, {dt:.1f} s)"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(res["value"], 3), "unit": res["unit"],
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(res["ms_per_step"], 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16 (fp32 accumulate)",
            "data": "synthetic", "config": workload_config(w),
            "roofline": res["roofline"], "roofline_nominal_frac": res["roofline_nominal_frac"],
            "kernels_ms": res["kernels_ms"], "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": res["launches"], "clocks": clk, "device_status": status,
            "graph": res.get("graph"),
            "workloads": extra,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
