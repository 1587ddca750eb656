"""Host-side logic of bench.py on the CPU: multi-rank aggregation over gloo
(world size 2), clock-sample parsing, the oracle reference arm, the source-keyed
traffic records and the L2 note."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # rank r processed (r + 1) GB in (10 + 5 r) ms per step
    value, ms = bench.aggregate_throughput((rank + 1) * 1e9, 10.0 + 5.0 * rank)
    q.put((rank, value, ms, bench.reduce_max(float(rank))))
    dist.destroy_process_group()


def test_two_rank_aggregation_over_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, value, ms, mx in res:
        assert ms == pytest.approx(15.0)                  # max over ranks
        assert value == pytest.approx(3e9 / 0.015)        # all ranks' units / max time
        assert mx == 1.0


def test_single_process_aggregation_is_identity():
    value, ms = bench.aggregate_throughput(2e9, 4.0)
    assert ms == 4.0 and value == pytest.approx(5e11)


def test_clock_summary_parsing():
    lines = ["1965, 2070, 610.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
             "2070, 2070, 900.1, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
             "garbage line"]
    s = bench.ClockSampler.summary(lines)
    assert s["sm_mhz"] == pytest.approx((1965 + 2070) / 2)
    assert s["sm_max_mhz"] == 2070 and s["samples"] == 2
    assert s["reasons"] == ["sw_power_cap"]


def test_reference_arm_prints_one_json_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload",
                          "tiny_decode", "--steps", "2", "--warmup", "3"], cwd=ROOT,
                         capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_window_and_fp8_accounting():
    """Algorithmic work of the windowed and fp8 workloads: visible (query, key) pairs
    counted against a brute-force mask, and fp8 decode bytes half of bf16."""
    import numpy as np
    from paged_kv_gqa_15_gb300 import workloads as W
    for causal in (True, False):
        for window in (0, 1, 5, 40):
            w = W.make_prefill("acc", [3, 17, 40], [9, 17, 60], 4, 2, 64, seed=1, causal=causal,
                               window=window)
            n = 0
            for qo, kv in zip(w.qo_lens, w.kv_lens):
                for i in range(qo):
                    pos = i + kv - qo
                    for j in range(kv):
                        ok = (j <= pos or not causal) and (window <= 0 or j > pos - window)
                        n += ok
            assert w.visible_pairs() == n, (causal, window)
    a = W.make_decode("b", [100, 7000], 32, 8, 128, seed=2)
    f = W.make_decode("f", [100, 7000], 32, 8, 128, seed=2, kv_fp8=True)
    assert f.kv_bytes() * 2 == a.kv_bytes()
    wdw = W.make_decode("w", [100, 7000], 32, 8, 128, seed=2, window=4096)
    assert wdw.visible_tokens() == 100 + 4096


def test_traffic_records_follow_their_sources(tmp_path, monkeypatch):
    # a record applies only to the source it was measured on: any other hash reads null
    name = "decode_partitions:llama8b_decode_b64_h32kv8_d128"
    src = ("pa_decode_tc.cu", "pa_tcgen05.cuh", "pa_device.cuh")
    rec = bench.TRAFFIC[name]
    monkeypatch.setitem(bench.TRAFFIC, name, dict(rec, src=bench.source_hash(*src)))
    assert bench.traffic_for(name, src) == rec["bytes_per_launch"]
    monkeypatch.setitem(bench.TRAFFIC, name, dict(rec, src="0" * 16))
    assert bench.traffic_for(name, src) is None
    assert bench.traffic_for("no_such_kernel:no_such_workload", src) is None


def test_l2_note_names_flush_or_size():
    small = bench.l2_note(100e6)
    large = bench.l2_note(600e6)
    assert "flushed" in small and "read back" in small
    assert "no flush" in large and "600 MB" in large


def test_clock_phases_keep_only_gpu_timed_samples():
    c = bench.ClockSampler(interval_ms=50)
    busy = "2070, 2070, 900, 0x0, Not Active, Not Active, Not Active, Not Active"
    idle = "345, 2070, 120, 0x1, Not Active, Not Active, Not Active, Not Active"
    c.lines = [(0.0, idle), (1.0, busy), (1.5, busy), (3.0, idle), (5.02, busy)]
    c.phases = [(0.9, 1.6), (4.0, 5.0)]
    kept = c.phase_lines()
    assert kept == [busy, busy, busy]          # 5.02 is within one interval of slack
    assert bench.ClockSampler.summary(kept)["sm_mhz"] == 2070


def test_step_stats_and_compact_summary():
    st = bench.step_stats([0.3, 0.1, 0.2, 0.4])
    assert st["median_ms"] == 0.25 and st["min_ms"] == 0.1 and st["reps"] == 4
    rec = {"value": 1000.0, "unit": "TFLOP/s", "kernels_ms": {"ragged_prefill": 0.18},
           "roofline": {"frac": 0.55}, "roofline_nominal_frac": 0.49, "step_stats": st,
           "cpu": {"value": 0.01, "cores": 16}, "parity": {"max_abs": 0.004,
                                                           "mean_abs": 1e-4, "ok": True}}
    e = bench.compact("ragged_prefill", rec)
    assert e["TFLOP/s"] == 1000.0 and e["kernel_ms"] == 0.18 and e["frac"] == 0.55
    assert e["target_nominal"] == 0.50 and e["met"] is False      # 0.49 of nominal
    assert e["median_ms"] == 0.25 and e["oracle"] == 0.01 and e["parity_ok"] is True
    assert "target_nominal" not in bench.compact("chunked_paged_prefill", rec)


def test_parity_record_counts_every_element():
    import numpy as np
    from paged_kv_gqa_15_gb300 import workloads as W
    ref = np.linspace(-2, 2, 24).reshape(2, 3, 4)
    bits = W.float_to_bits(ref.astype(np.float32))          # bf16 of the reference
    p = bench._parity(bits, ref)
    assert p["ok"] and p["elements"] == 24 and p["max_abs"] <= 2 ** -8 * 2
    bad = bits.copy()
    bad[1, 2, 3] = W.float_to_bits(np.float32(5.0))
    assert not bench._parity(bad, ref)["ok"]
    nan = bits.copy()
    nan[0, 0, 0] = np.uint16(0x7FC0)
    assert not bench._parity(nan, ref)["ok"]
