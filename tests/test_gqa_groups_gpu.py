"""GPU parity for GQA group sizes beyond 1, 2, 4 and 8 ("paged_attn.py", forward_decode's
num_queries_per_kv = num_heads // num_kv_heads, any integer; query head h reads kv head
h / g), through the C ABI, against the fp64 oracle on every output element.

The decode kernels serve some group sizes directly (on the tensor cores: bf16 3-16 at
head_dim 128 and 3-8 at head_dim 64, fp8 3-8 at head_dim 128; the CUDA-core kernel 1, 2,
4 and 8).  Any other size runs as several kernel groups per kv head, each of a divisor of
g.  The cases below reach every kind of dispatch:
  - a tensor-core group of its own (bf16 3, 5, 6, 7, 11, 12, 16 at head_dim 128, 3 and 6
    at head_dim 64; fp8 3, 5, 6, 7);
  - tensor-core groups of a divisor (bf16 32 = 2 x 16, 12 = 2 x 6 at head_dim 64;
    fp8 10 = 2 x 5, 12 = 2 x 6, 16 = 2 x 8);
  - CUDA-core groups of a divisor (bf16 17 = 17 x 1; fp8 11 = 11 x 1; head_dim 256 with
    3, 6 and 12).
The prefill kernel takes the group size at run time; it is checked at 3 and 6, contiguous
and paged."""
import numpy as np
import pytest

from paged_kv_gqa_15_gb300 import workloads as W
from tests.gpu_util import assert_close_bf16
from tests.test_decode_gpu import _run_decode
from tests.test_fp8_gpu import _fp8_pools, _run as _run_fp8
from tests.test_prefill_gpu import _contig_case, _paged_case

pytestmark = pytest.mark.gpu

LENS = [0, 1, 15, 16, 17, 100, 511, 512, 513, 1100, 2049]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    import paged_kv_gqa_15_gb300 as pa
    __graft_entry__.build()
    yield
    assert pa.device_status() == 0


@pytest.mark.parametrize("nq,nkv", [(6, 2), (10, 2), (12, 2), (14, 2), (24, 2), (32, 2),
                                    (22, 2), (28, 4), (64, 2), (34, 2)])
@pytest.mark.parametrize("split", [False, True])
def test_bf16_decode_group_sizes_hd128(nq, nkv, split):
    w = W.make_decode("gqa", LENS, nq, nkv, 128, seed=120 + nq)
    out, ref, _, _ = _run_decode(w, split)
    assert_close_bf16(out, ref, what=f"bf16 g{nq // nkv} split={split}")


@pytest.mark.parametrize("hd", [64, 256])
@pytest.mark.parametrize("nq,nkv", [(6, 2), (12, 2), (24, 2)])
@pytest.mark.parametrize("split", [False, True])
def test_bf16_decode_group_sizes_other_head_dims(hd, nq, nkv, split):
    w = W.make_decode("gqa_cc", LENS, nq, nkv, hd, seed=130 + nq + hd)
    out, ref, _, _ = _run_decode(w, split)
    assert_close_bf16(out, ref, what=f"hd{hd} g{nq // nkv} split={split}")


@pytest.mark.parametrize("nq,nkv", [(12, 2), (6, 2), (10, 2), (14, 2), (20, 2), (24, 2),
                                    (32, 2), (22, 2)])
@pytest.mark.parametrize("split", [False, True])
def test_fp8_decode_group_sizes_hd128(nq, nkv, split):
    w = W.make_decode("gqa8", LENS, nq, nkv, 128, seed=140 + nq)
    kc, vc = _fp8_pools(w, seed=141)
    out, ref, _, _ = _run_fp8(w, kc, vc, split)
    assert_close_bf16(out, ref, what=f"fp8 g{nq // nkv} split={split}")


@pytest.mark.parametrize("nq,nkv", [(12, 2), (32, 2), (6, 2)])
@pytest.mark.parametrize("split", [False, True])
def test_windowed_decode_group_sizes(nq, nkv, split):
    w = W.make_decode("gqaw", LENS + [4000], nq, nkv, 128, seed=150 + nq, window=700)
    out, ref, _, _ = _run_decode(w, split)
    assert_close_bf16(out, ref, what=f"window g{nq // nkv} split={split}")


@pytest.mark.parametrize("nq,nkv", [(6, 2), (12, 2)])
@pytest.mark.parametrize("hd", [64, 128, 256])
def test_prefill_group_sizes(nq, nkv, hd):
    o, ref, _ = _contig_case([5, 130, 300], [5, 200, 300], nq, nkv, hd, seed=160 + nq + hd)
    assert_close_bf16(o, ref, what=f"prefill g{nq // nkv} hd{hd}")
    o, ref, _ = _paged_case([64, 129], [300, 129], nq, nkv, hd, seed=170 + nq + hd)
    assert_close_bf16(o, ref, what=f"paged prefill g{nq // nkv} hd{hd}")


@pytest.mark.parametrize("nq,nkv", [(12, 2), (14, 2), (34, 2)])
def test_static_entry_and_graph_replay_take_any_group(nq, nkv):
    """The fixed-scratch split entry and a captured split step (the regrouping happens
    on the host, before the launch, so a replay repeats the same kernels)."""
    import oracle
    import torch
    import paged_kv_gqa_15_gb300 as pa
    w = W.make_decode("gqas", [1, 513, 1500, 33], nq, nkv, 128, seed=180 + nq)
    t = w.tensors("cuda")
    q, kc, vc = t["q"], t["k_cache"], t["v_cache"]
    bt = torch.from_numpy(w.block_tables).to("cuda")
    sl = torch.from_numpy(w.seq_lens).to("cuda")
    L = w.max_seq_len
    ref = oracle.decode(W.to_bits(q), W.to_bits(kc), W.to_bits(vc), w.block_tables,
                        w.seq_lens, nkv, 16, w.scale)
    out = torch.full_like(q, float("nan"))
    pa.pa_decode_split_static(out, q, kc, vc, bt, sl, w.scale, L)
    torch.cuda.synchronize()
    assert_close_bf16(out, ref, what=f"static g{nq // nkv}")
    ws = pa.alloc_workspace(pa.decode_split_workspace_size(w.batch, nq, 128, L), "cuda")
    out2 = torch.full_like(q, float("nan"))
    stream = torch.cuda.Stream()
    pa.pa_decode_split(out2, q, kc, vc, bt, sl, w.scale, L, ws, stream=stream)   # warm-up
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        pa.pa_decode_split(out2, q, kc, vc, bt, sl, w.scale, L, ws, stream=stream)
    for _ in range(2):
        out2.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert_close_bf16(out2, ref, what=f"graph g{nq // nkv}")
