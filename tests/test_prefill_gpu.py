"""GPU parity of the ragged / paged prefill (tcgen05 kernel) against the fp64
oracle, through the C ABI."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_15_gb300 as pa
from paged_kv_gqa_15_gb300 import workloads as W
from tests.gpu_util import assert_close_bf16, bf16_out

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    yield
    assert pa.device_status() == 0


def _to_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV).view(torch.bfloat16)


def run_contiguous(q, k, v, qo_ind, kv_ind, scale, causal):
    o = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device=DEV)
    pa.pa_ragged_prefill(o, _to_dev(q), _to_dev(k), _to_dev(v), qo_ind, kv_ind,
                         torch.from_numpy(qo_ind).to(DEV), torch.from_numpy(kv_ind).to(DEV),
                         scale, causal=causal)
    torch.cuda.synchronize()
    return o


def _contig_case(qo, kv, nq, nkv, hd, seed, causal=True):
    w = W.make_prefill("c", qo, kv, nq, nkv, hd, seed=seed, causal=causal)
    t = w.tensors("cpu")
    q, k, v = (W.to_bits(t[n]) for n in ("q", "k", "v"))
    o = run_contiguous(q, k, v, w.qo_indptr, w.kv_indptr, w.scale, causal)
    ref = oracle.prefill(q, k, v, w.qo_indptr, w.kv_indptr, nkv, w.scale, causal=causal)
    return o, ref, w


def test_t1_shape_hash_inputs():
    """2 requests of 6 and 10 tokens, 4 qo / 2 kv heads, hd 256, causal, counter-hash
    inputs in [-0.25, 0.25) (the worked test of the "spark_runtime/flashinfer.rs" page)."""
    hd, nq, nkv = 256, 4, 2
    lens = np.array([6, 10])
    ind = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(lens.sum())
    q = W.float_to_bits(W.hash_uniform(np.arange(T * nq * hd)).astype(np.float32))
    k = W.float_to_bits(W.hash_uniform(np.arange(T * nkv * hd) ^ 0x1111).astype(np.float32))
    v = W.float_to_bits(W.hash_uniform(np.arange(T * nkv * hd) ^ 0x2222).astype(np.float32))
    q, k, v = q.reshape(T, nq, hd), k.reshape(T, nkv, hd), v.reshape(T, nkv, hd)
    scale = 1.0 / math.sqrt(hd)
    o = run_contiguous(q, k, v, ind, ind, scale, True)
    ref = oracle.prefill(q, k, v, ind, ind, nkv, scale, causal=True)
    assert_close_bf16(o, ref, what="T1")
    got = bf16_out(o)
    cos = (got * ref).sum(-1) / (np.linalg.norm(got, axis=-1) * np.linalg.norm(ref, axis=-1))
    assert cos.min() > 0.99


@pytest.mark.parametrize("hd", [64, 128, 256])
@pytest.mark.parametrize("causal", [True, False])
def test_single_tile_square(hd, causal):
    o, ref, _ = _contig_case([128], [128], 2, 1, hd, seed=hd, causal=causal)
    assert_close_bf16(o, ref, what=f"hd{hd} causal={causal}")


@pytest.mark.parametrize("hd", [64, 128, 256])
def test_ragged_multi_tile(hd):
    # several query tiles, several key tiles, ragged tails, chunk-after-prefix (kv > qo)
    qo = [1, 130, 300, 17, 256]
    kv = [1, 130, 700, 400, 256]
    o, ref, _ = _contig_case(qo, kv, 8, 2, hd, seed=100 + hd)
    assert_close_bf16(o, ref, what=f"ragged hd{hd}")


@pytest.mark.parametrize("hd", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
def test_query_block_boundaries(hd, causal):
    # query lengths on both sides of the 128- and 256-row boundaries: a block whose
    # second tile is empty, partial or full, and keys shorter than the queries
    qo = [255, 256, 257, 383, 384, 385, 513, 129]
    kv = [255, 300, 257, 383, 900, 385, 513, 60]
    o, ref, _ = _contig_case(qo, kv, 4, 2, hd, seed=200 + hd + causal, causal=causal)
    assert_close_bf16(o, ref, what=f"block boundaries hd{hd} causal={causal}")


@pytest.mark.parametrize("hd", [64, 128])
def test_paged_query_block_boundaries(hd):
    o, ref, _ = _paged_case([257, 384, 100], [400, 384, 1000], 4, 1, hd, seed=210 + hd)
    assert_close_bf16(o, ref, what=f"paged block boundaries hd{hd}")


def test_output_only_16_byte_aligned():
    # an output buffer that is 16- but not 32-byte aligned takes the 16-byte store path
    w = W.make_prefill("al", [200, 70], [200, 300], 4, 2, 128, seed=220)
    t = w.tensors("cpu")
    q, k, v = (W.to_bits(t[n]) for n in ("q", "k", "v"))
    n = q.size
    backing = torch.full((n + 8,), float("nan"), dtype=torch.bfloat16, device=DEV)
    o = backing[8:].view(q.shape)
    assert o.data_ptr() % 32 == 16
    pa.pa_ragged_prefill(o, _to_dev(q), _to_dev(k), _to_dev(v), w.qo_indptr, w.kv_indptr,
                         torch.from_numpy(w.qo_indptr).to(DEV), torch.from_numpy(w.kv_indptr).to(DEV),
                         w.scale, causal=True)
    torch.cuda.synchronize()
    ref = oracle.prefill(q, k, v, w.qo_indptr, w.kv_indptr, 2, w.scale, causal=True)
    assert_close_bf16(o, ref, what="16-byte aligned output")


@pytest.mark.parametrize("nq,nkv", [(4, 4), (8, 4), (16, 4), (32, 4)])
def test_group_sizes(nq, nkv):
    o, ref, _ = _contig_case([200, 77], [200, 300], nq, nkv, 128, seed=nq)
    assert_close_bf16(o, ref, what=f"g{nq // nkv}")


def test_non_causal_ragged():
    o, ref, _ = _contig_case([50, 129, 3], [400, 129, 700], 8, 2, 128, seed=5, causal=False)
    assert_close_bf16(o, ref, what="non-causal")


def test_rows_without_keys_are_zero():
    # kv < qo: the first qo - kv rows see nothing and must come out as zeros
    o, ref, _ = _contig_case([300, 40], [100, 0], 4, 2, 128, seed=6)
    got = bf16_out(o)
    assert (got[:200] == 0).all() and (got[300:] == 0).all()
    assert_close_bf16(got, ref, what="kv < qo")


def test_empty_requests_in_batch():
    o, ref, _ = _contig_case([0, 5, 0, 140], [0, 5, 9, 140], 4, 2, 64, seed=7)
    assert_close_bf16(o, ref, what="empty requests")


def test_large_logits():
    w = W.make_prefill("big", [150], [150], 4, 2, 128, seed=8)
    t = w.tensors("cpu")
    q, k, v = (W.to_bits(t[n]) for n in ("q", "k", "v"))
    scale = 1.0   # scores of tens: exercises the running-max rescale of O
    o = run_contiguous(q, k, v, w.qo_indptr, w.kv_indptr, scale, True)
    ref = oracle.prefill(q, k, v, w.qo_indptr, w.kv_indptr, 2, scale, causal=True)
    assert_close_bf16(o, ref, what="large logits")


def test_growing_logits_force_rescale():
    """Keys whose scores grow along the sequence force the O rescale on later tiles."""
    qo, kv, hd = 64, 640, 128
    rng = np.random.default_rng(9)
    q = np.zeros((qo, 2, hd), np.float32)
    q[:, :, 0] = 1.0
    k = rng.standard_normal((kv, 1, hd)).astype(np.float32) * 0.1
    k[:, 0, 0] = np.linspace(0, 40, kv)          # score grows by ~8 per 128-key tile
    v = rng.standard_normal((kv, 1, hd)).astype(np.float32)
    qb, kb, vb = W.float_to_bits(q), W.float_to_bits(k), W.float_to_bits(v)
    ind_q = np.array([0, qo], np.int32)
    ind_k = np.array([0, kv], np.int32)
    o = run_contiguous(qb, kb, vb, ind_q, ind_k, 1.0, False)
    ref = oracle.prefill(qb, kb, vb, ind_q, ind_k, 1, 1.0, causal=False)
    assert_close_bf16(o, ref, what="growing logits")


# ---- paged mode -------------------------------------------------------------------------------


def _paged_case(qo, kv, nq, nkv, hd, seed, layout="HND", causal=True, chunk_write=False):
    w = W.make_prefill("p", qo, kv, nq, nkv, hd, seed=seed, causal=causal, paged=True,
                       chunk_write=chunk_write)
    t = w.tensors("cpu")
    q = W.to_bits(t["q"])
    kc, vc = W.to_bits(t["k_cache"]), W.to_bits(t["v_cache"])
    kc_d, vc_d = _to_dev(kc), _to_dev(vc)
    if layout == "NHD":
        kc_d = kc_d.permute(0, 2, 1, 3).contiguous()
        vc_d = vc_d.permute(0, 2, 1, 3).contiguous()
    if chunk_write:
        kn, vn = W.to_bits(t["k_new"]), W.to_bits(t["v_new"])
        pa.pa_write_cache(_to_dev(kn), _to_dev(vn), kc_d, vc_d,
                          torch.from_numpy(w.chunk_slot_mapping).to(DEV), layout=layout)
        oracle.write_cache(kn, vn, kc, vc, w.chunk_slot_mapping, 16)
    o = torch.full(t["q"].shape, float("nan"), dtype=torch.bfloat16, device=DEV)
    pa.pa_ragged_prefill(o, _to_dev(q), kc_d, vc_d, w.qo_indptr, w.kv_indptr,
                         torch.from_numpy(w.qo_indptr).to(DEV),
                         torch.from_numpy(w.kv_indptr).to(DEV), w.scale, causal=causal,
                         block_tables=torch.from_numpy(w.block_tables).to(DEV), layout=layout)
    torch.cuda.synchronize()
    ref = oracle.prefill(q, kc, vc, w.qo_indptr, w.kv_indptr, nkv, w.scale, causal=causal,
                         block_tables=w.block_tables, block_size=16)
    return o, ref, w


@pytest.mark.parametrize("hd", [64, 128, 256])
@pytest.mark.parametrize("layout", ["HND", "NHD"])
def test_paged_chunk_after_prefix(hd, layout):
    o, ref, _ = _paged_case([64, 130, 1], [300, 130, 517], 8, 4, hd, seed=20 + hd,
                            layout=layout, chunk_write=True)
    assert_close_bf16(o, ref, what=f"paged hd{hd} {layout}")


def test_paged_equals_contiguous():
    qo, kv = [100, 33], [260, 33]
    o_p, ref, w = _paged_case(qo, kv, 4, 2, 128, seed=30)
    assert_close_bf16(o_p, ref, what="paged")


def test_paged_bad_block_id_is_flagged():
    w = W.make_prefill("bad", [20], [40], 4, 2, 64, seed=31, paged=True)
    t = w.tensors("cpu")
    bt = w.block_tables.copy()
    bt[0, 1] = w.num_blocks + 3
    o = torch.empty_like(t["q"]).to(DEV)
    pa.pa_ragged_prefill(o, t["q"].to(DEV), t["k_cache"].to(DEV), t["v_cache"].to(DEV),
                         w.qo_indptr, w.kv_indptr, torch.from_numpy(w.qo_indptr).to(DEV),
                         torch.from_numpy(w.kv_indptr).to(DEV), w.scale,
                         block_tables=torch.from_numpy(bt).to(DEV))
    assert pa.device_status() & (1 << pa.PA_ERR_DEVICE_BOUNDS)
    assert torch.isfinite(o.float()).all()


def test_paged_stale_nan_rows_do_not_leak():
    """Rows of a request's last page past its kv length may hold anything (here NaN):
    they are masked out and must not reach the output."""
    w = W.make_prefill("stale", [20, 7], [37, 70], 4, 2, 128, seed=40, paged=True)
    t = w.tensors("cpu")
    q = W.to_bits(t["q"])
    kc, vc = W.to_bits(t["k_cache"]), W.to_bits(t["v_cache"])
    nan = np.uint16(0x7FC0)
    for r, kv in enumerate(w.kv_lens):
        if kv % 16:
            page = w.block_tables[r, kv // 16]
            kc[page, :, kv % 16:, :] = nan
            vc[page, :, kv % 16:, :] = nan
    o = torch.empty(t["q"].shape, dtype=torch.bfloat16, device=DEV)
    pa.pa_ragged_prefill(o, _to_dev(q), _to_dev(kc), _to_dev(vc), w.qo_indptr, w.kv_indptr,
                         torch.from_numpy(w.qo_indptr).to(DEV),
                         torch.from_numpy(w.kv_indptr).to(DEV), w.scale, causal=True,
                         block_tables=torch.from_numpy(w.block_tables).to(DEV))
    torch.cuda.synchronize()
    ref = oracle.prefill(q, kc, vc, w.qo_indptr, w.kv_indptr, 2, w.scale, causal=True,
                         block_tables=w.block_tables, block_size=16)
    assert_close_bf16(o, ref, what="stale NaN rows")


def test_rejects_non_positive_scale():
    w = W.make_prefill("s", [4], [4], 2, 1, 64, seed=41)
    t = w.tensors("cpu")
    o = torch.empty(t["q"].shape, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(pa.PaError):
        pa.pa_ragged_prefill(o, t["q"].to(DEV), t["k"].to(DEV), t["v"].to(DEV), w.qo_indptr,
                             w.kv_indptr, torch.from_numpy(w.qo_indptr).to(DEV),
                             torch.from_numpy(w.kv_indptr).to(DEV), 0.0)


# ---- work list: built on the host (<= 1024 query tiles) or by the schedule kernel ------

def test_work_list_longer_than_the_inline_limit():
    # 1100 one-tile requests: the work list is built on the device, not on the host
    rng = np.random.default_rng(40)
    lens = rng.integers(1, 129, size=1100)
    o, ref, _ = _contig_case(lens, lens, 4, 2, 64, seed=41)
    assert pa.device_status() == 0
    assert_close_bf16(o, ref, what="1100 query tiles")


def test_calls_leave_the_work_counters_zero():
    # one workspace through host-built and device-built work lists, alternately: each
    # launch must find its counters at zero and leave them so
    small = W.make_prefill("s", [130, 5, 300], [200, 5, 300], 8, 2, 128, seed=42)
    rng = np.random.default_rng(43)
    many_lens = rng.integers(1, 129, size=1100)
    many = W.make_prefill("m", many_lens, many_lens, 4, 2, 128, seed=44)
    size = max(pa.ragged_prefill_workspace_size(w.batch, w.total_qo, w.num_q_heads, 128)
               for w in (small, many))
    ws = pa.alloc_workspace(size, DEV)
    for w in (small, many, small, many):
        t = w.tensors("cpu")
        q, k, v = (W.to_bits(t[n]) for n in ("q", "k", "v"))
        o = torch.full((w.total_qo, w.num_q_heads, 128), float("nan"), dtype=torch.bfloat16,
                       device=DEV)
        pa.pa_ragged_prefill(o, _to_dev(q), _to_dev(k), _to_dev(v), w.qo_indptr, w.kv_indptr,
                             torch.from_numpy(w.qo_indptr).to(DEV),
                             torch.from_numpy(w.kv_indptr).to(DEV), w.scale, causal=True,
                             workspace=ws)
        torch.cuda.synchronize()
        assert int(ws[:8].view(torch.int32).abs().sum()) == 0
        ref = oracle.prefill(q, k, v, w.qo_indptr, w.kv_indptr, w.num_kv_heads, w.scale,
                             causal=True)
        assert_close_bf16(o, ref, what=f"batch {w.batch}")
    assert pa.device_status() == 0
