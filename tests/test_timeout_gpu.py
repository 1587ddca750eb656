"""The bounded pipeline wait on the GPU: a wait that nothing completes runs out after
its limit, records PA_ERR_TIMEOUT in the device status word instead of hanging, and
leaves the context usable (a decode right after it matches the oracle)."""
import time

import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_15_gb300 as pa
from paged_kv_gqa_15_gb300 import workloads as W
from tests.gpu_util import assert_close_bf16

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    yield
    assert pa.device_status() == 0


def test_a_wait_that_runs_out_reports_timeout_and_the_context_survives():
    assert pa.device_status() == 0
    t0 = time.monotonic()
    pa.selftest_wait_timeout()
    status = pa.device_status()          # synchronises, reads and clears
    elapsed = time.monotonic() - t0
    assert status == 1 << pa.PA_ERR_TIMEOUT
    assert 0.9 < elapsed < 30.0          # the 1 s per-wait limit, not a hang
    assert pa.device_status() == 0       # the read cleared it

    w = W.make_decode("after_timeout", [17, 600], 8, 2, 128, seed=91)
    t = w.tensors(DEV)
    out = torch.empty_like(t["q"])
    pa.pa_decode(out, t["q"], t["k_cache"], t["v_cache"], torch.from_numpy(w.block_tables).to(DEV),
                 torch.from_numpy(w.seq_lens).to(DEV), w.scale)
    torch.cuda.synchronize()
    ref = oracle.decode(W.to_bits(t["q"].cpu()), W.to_bits(t["k_cache"].cpu()),
                        W.to_bits(t["v_cache"].cpu()), w.block_tables, w.seq_lens, 2, 16, w.scale)
    assert_close_bf16(out, ref, what="decode after a timeout")
    assert pa.device_status() == 0
