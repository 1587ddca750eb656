"""Whole-output GPU parity of every benchmarked workload at its full size, in the launch
configuration the benchmark times: the benchmark's own set-up and step functions (one
stream, the step's cache write first where it has one, dependent launches), run twice as
the timed loop repeats them, then every element of the output compared with the fp64
oracle on the same inputs ("paged_attn.py", PagedAttention.forward_decode V1 / V2 and
_forward_prefix_pytorch; "spark_runtime/flashinfer.rs", ragged_prefill_bf16_hd256 and its
CPU reference)."""
import numpy as np
import pytest
import torch

import bench
import oracle
import paged_kv_gqa_15_gb300 as pa
from paged_kv_gqa_15_gb300 import workloads as W
from tests.gpu_util import assert_close_bf16

pytestmark = pytest.mark.gpu
DEV = "cuda"

DECODE = ["tiny_decode", "llama8b_decode", "long_context_decode", "window_decode",
          "llama8b_decode_fp8", "long_context_decode_fp8", "llama8b_decode_single",
          "mha_decode", "gqa7_decode"]
PREFILL = ["ragged_prefill", "chunked_paged_prefill", "window_prefill"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    yield
    assert pa.device_status() == 0


@pytest.mark.parametrize("name", DECODE)
def test_decode_workload_whole_output(name):
    w = W.WORKLOADS[name]()
    stream = torch.cuda.Stream()
    s = bench.decode_setup(w, DEV)
    t = s["t"]
    q = W.to_bits(t["q"])
    kc, vc = bench.host_pool(w, t["k_cache"]), bench.host_pool(w, t["v_cache"])
    for _ in range(2):
        bench.decode_step(w, s, stream)
    stream.synchronize()
    scales = dict(k_scale=bench.FP8_SCALE, v_scale=bench.FP8_SCALE)
    if w.new_token_write:
        oracle.write_cache(W.to_bits(t["k_new"]), W.to_bits(t["v_new"]), kc, vc,
                           w.slot_mapping, w.block_size, kv_fp8=w.kv_fp8, **scales)
        # the cache write is bit-exact on every page it touched
        touched = np.unique(w.slot_mapping[w.slot_mapping >= 0] // w.block_size)
        idx = torch.from_numpy(touched).to(DEV)
        np.testing.assert_array_equal(bench.host_pool(w, t["k_cache"][idx]), kc[touched])
        np.testing.assert_array_equal(bench.host_pool(w, t["v_cache"][idx]), vc[touched])
    ref = oracle.decode(q, kc, vc, w.block_tables, w.seq_lens, w.num_kv_heads, w.block_size,
                        w.scale, window=w.window, kv_fp8=w.kv_fp8, **scales)
    assert_close_bf16(s["out"], ref, what=name)
    assert pa.device_status(stream) == 0


@pytest.mark.parametrize("name", PREFILL)
def test_prefill_workload_whole_output(name):
    w = W.WORKLOADS[name]()
    stream = torch.cuda.Stream()
    s = bench.prefill_setup(w, DEV)
    host = {n: W.to_bits(v) for n, v in s["t"].items()}
    for _ in range(2):
        bench.prefill_step(w, s, stream)
    stream.synchronize()
    if w.paged:
        k, v = host["k_cache"], host["v_cache"]
        if w.chunk_write:
            oracle.write_cache(host["k_new"], host["v_new"], k, v, w.chunk_slot_mapping,
                               w.block_size)
    else:
        k, v = host["k"], host["v"]
    ref = oracle.prefill(host["q"], k, v, w.qo_indptr, w.kv_indptr, w.num_kv_heads, w.scale,
                         causal=w.causal, block_tables=w.block_tables if w.paged else None,
                         block_size=w.block_size, window=w.window)
    assert_close_bf16(s["out"], ref, what=name)
    # the work counters are left zero for the next call
    assert int(s["ws"][:8].view(torch.int32).abs().sum()) == 0
    assert pa.device_status(stream) == 0
