"""The decode step (cache write, split partitions, merge) captured once in a CUDA graph
and replayed with new inputs: each replay's cache and output must match the fp64
oracle run on a host copy of the cache that the oracle's own scatter keeps up to date.
Between replays every sequence grows by one token (taking a fresh page whenever it
crosses a page boundary) and the changed block-table rows go up through
pa_block_table_sync, which must report exactly those rows."""
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


@pytest.mark.parametrize("nq,nkv", [(32, 8), (8, 8)])
def test_decode_step_replayed_from_a_cuda_graph(nq, nkv):
    hd, bs, steps = 128, 16, 4
    # the third length sits one token before a page boundary, the fourth on one
    lens0 = np.array([100, 700, 1503, 48], np.int32)
    need = int(sum((L + steps + bs - 1) // bs for L in lens0))
    w = W.make_decode("graph", lens0, nq, nkv, hd, seed=61, new_token_write=True, split=True,
                      num_blocks=need + 8, max_blocks=(int(lens0.max()) + steps) // bs + 2)
    t = w.tensors("cpu")
    kc_h, vc_h = W.to_bits(t["k_cache"]), W.to_bits(t["v_cache"])
    bt_h = w.block_tables.copy()
    used = set(int(x) for x in bt_h[bt_h >= 0].ravel())
    free = [b for b in range(w.num_blocks) if b not in used]
    sl_h = w.seq_lens.copy()
    slots_h = w.slot_mapping.copy()

    # static device buffers the graph is captured with
    q_d = t["q"].to(DEV)
    kn_d, vn_d = t["k_new"].to(DEV), t["v_new"].to(DEV)
    kc_d, vc_d = t["k_cache"].to(DEV), t["v_cache"].to(DEV)
    bt_d = torch.from_numpy(bt_h).to(DEV)
    snap = torch.from_numpy(bt_h.copy()).pin_memory()
    sl_d = torch.from_numpy(sl_h).to(DEV)
    slots_d = torch.from_numpy(slots_h).to(DEV)
    out_d = torch.empty_like(q_d)
    L_cap = int(lens0.max()) + steps          # the split grid is sized for this bound
    ws = pa.alloc_workspace(pa.decode_split_workspace_size(w.batch, nq, hd, L_cap), DEV)
    stream = torch.cuda.Stream()

    def step():
        pa.pa_write_cache(kn_d, vn_d, kc_d, vc_d, slots_d, stream=stream)
        pa.pa_decode_partitions(q_d, kc_d, vc_d, bt_d, sl_d, w.scale, L_cap, ws, stream=stream)
        pa.pa_decode_merge(out_d, sl_d, L_cap, ws, stream=stream)

    # warm up outside the capture (one-time set-up such as shared-memory opt-ins), on a
    # scratch copy of the pools so the replays start from the original cache
    kc_save, vc_save = kc_d.clone(), vc_d.clone()
    with torch.cuda.stream(stream):
        step()
    stream.synchronize()
    kc_d.copy_(kc_save)
    vc_d.copy_(vc_save)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    torch.cuda.synchronize()

    rng = np.random.default_rng(62)
    for it in range(steps):
        if it > 0:   # one more token per sequence; new q and new K/V rows
            changed = set()
            for b in range(w.batch):
                pos = int(sl_h[b])                 # position of the new token
                if pos % bs == 0:                  # first token of a new page
                    bt_h[b, pos // bs] = free.pop()
                    changed.add(b)
                sl_h[b] = pos + 1
                slots_h[b] = int(bt_h[b, pos // bs]) * bs + pos % bs
            assert pa.pa_block_table_sync(bt_h, snap, bt_d, stream=stream) == len(changed)
            for name, dst in (("q", q_d), ("k_new", kn_d), ("v_new", vn_d)):
                src = W.bf16_normal(tuple(dst.shape), int(rng.integers(1 << 30)), "cpu")
                t[name] = src
                dst.copy_(src)
            sl_d.copy_(torch.from_numpy(sl_h))
            slots_d.copy_(torch.from_numpy(slots_h))
            torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        oracle.write_cache(W.to_bits(t["k_new"]), W.to_bits(t["v_new"]), kc_h, vc_h, slots_h, bs)
        assert np.array_equal(W.to_bits(kc_d.cpu()), kc_h), f"replay {it}: K cache"
        assert np.array_equal(W.to_bits(vc_d.cpu()), vc_h), f"replay {it}: V cache"
        ref = oracle.decode(W.to_bits(t["q"]), kc_h, vc_h, bt_h, sl_h, nkv, bs, w.scale)
        assert_close_bf16(out_d.cpu(), ref, what=f"graph replay {it}")
