"""pa_decode_split_static: the split decode for callers that cannot allocate
device memory (its partials live in a fixed array inside the library instead of
a caller workspace).  Collected last on purpose: it checks the static-scratch
entry point against the workspace entry point, through the C ABI, on two calls
in a row (the second with fewer sequences but more partitions each, so stale
partials left by the first call would show up), and the second call against
the fp64 oracle."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_15_gb300 as pa
from paged_kv_gqa_15_gb300 import workloads as W
from tests.gpu_util import MAX_ABS, MEAN_ABS, assert_close_bf16, bf16_out

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(w):
    t = w.tensors(DEV)
    return (t["q"], t["k_cache"], t["v_cache"], torch.from_numpy(w.block_tables).to(DEV),
            torch.from_numpy(w.seq_lens).to(DEV))


def _static_call(lib, out, q, kc, vc, bt, sl, w, max_seq_len):
    sb, sh, st = pa.pool_strides(kc)
    return lib.pa_decode_split_static(
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(q.data_ptr()),
        ctypes.c_void_p(kc.data_ptr()), ctypes.c_void_p(vc.data_ptr()),
        ctypes.c_void_p(bt.data_ptr()), ctypes.c_void_p(sl.data_ptr()), w.batch,
        w.num_q_heads, w.num_kv_heads, w.head_dim, 16, bt.shape[1], w.num_blocks, sb, sh, st,
        ctypes.c_float(w.scale), 0, 0, ctypes.c_float(1.0), ctypes.c_float(1.0), max_seq_len,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _check_pair(lib, w):
    """One call of each entry point on the same inputs; returns the static call's output
    and the inputs (q, k_cache, v_cache)."""
    q, kc, vc, bt, sl = _inputs(w)
    L = w.max_seq_len
    ref = torch.empty_like(q)
    ws = pa.alloc_workspace(pa.decode_split_workspace_size(w.batch, w.num_q_heads,
                                                           w.head_dim, L), DEV)
    pa.pa_decode_split(ref, q, kc, vc, bt, sl, w.scale, L, ws)
    out = torch.full_like(q, float("nan"))
    rc = _static_call(lib, out, q, kc, vc, bt, sl, w, L)
    assert rc == pa.PA_OK, lib.pa_last_error()
    torch.cuda.synchronize()
    got, want = bf16_out(out), bf16_out(ref)
    assert np.isfinite(got).all()
    err = np.abs(got - want)
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, (err.max(), err.mean())
    return got, (q, kc, vc)


def test_static_scratch_matches_workspace_entry_point_on_two_calls():
    import __graft_entry__
    __graft_entry__.build()
    lib = pa.load()
    rng = np.random.default_rng(2024)
    # The second call has fewer sequences but more partitions per sequence (up to 49,
    # past the 32 the one-warp merge handles) than the first, so partials the first call
    # left in the shared array lie inside the rows the second call merges.
    first = W.make_decode("no_alloc_1", rng.integers(1, 6000, size=24), 32, 8, 128, seed=71)
    second = W.make_decode("no_alloc_2", [24577, 16385, 3, 511], 32, 8, 128, seed=72)
    need = pa.decode_split_workspace_size(second.batch, 32, 128, second.max_seq_len)
    assert need <= 16 << 20
    _check_pair(lib, first)
    got, (q, kc, vc) = _check_pair(lib, second)
    # the second call also against the fp64 oracle, on the same (device-generated) inputs
    ref = oracle.decode(W.to_bits(q), W.to_bits(kc), W.to_bits(vc), second.block_tables,
                        second.seq_lens, second.num_kv_heads, second.block_size, second.scale)
    assert_close_bf16(got, ref, what="static split vs oracle")
    assert pa.device_status() == 0


def test_static_scratch_rejects_batches_beyond_its_size():
    lib = pa.load()
    w = W.make_decode("no_alloc_big", [16], 32, 8, 128, seed=73)
    q, kc, vc, bt, sl = _inputs(w)
    out = torch.empty_like(q)
    # 64 seqs x 32 heads x 256 partitions x 128 dims x 4 B = 64 MiB > the fixed scratch
    big = torch.zeros((64, 8192), dtype=torch.int32, device=DEV)
    sl64 = torch.full((64,), 16, dtype=torch.int32, device=DEV)
    q64 = torch.zeros((64, 32, 128), dtype=torch.bfloat16, device=DEV)
    sb, sh, st = pa.pool_strides(kc)
    rc = lib.pa_decode_split_static(
        ctypes.c_void_p(q64.data_ptr()), ctypes.c_void_p(q64.data_ptr()),
        ctypes.c_void_p(kc.data_ptr()), ctypes.c_void_p(vc.data_ptr()),
        ctypes.c_void_p(big.data_ptr()), ctypes.c_void_p(sl64.data_ptr()), 64, 32, 8, 128, 16,
        8192, w.num_blocks, sb, sh, st, ctypes.c_float(w.scale), 0, 0, ctypes.c_float(1.0),
        ctypes.c_float(1.0), 131072,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == pa.PA_ERR_WORKSPACE
    assert b"PA_STATIC_SCRATCH_BYTES" in lib.pa_last_error()
    del out
