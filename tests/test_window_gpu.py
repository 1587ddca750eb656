"""GPU parity of the sliding window (a query at position pos sees keys j > pos - W;
"paged_attn.py", forward_prefix's sliding_window, and "libmir-cuda attention/mod.rs",
active_partitions(token_count, window)) in decode -- single pass, split on the tensor
cores and on the CUDA cores -- and in ragged prefill over contiguous and paged K/V,
against the fp64 oracle through the C ABI.

Pages that lie wholly before a window get invalid block-table entries (-1) and the
rows before the window in its first page hold NaN: the outputs must match the oracle
(which reads neither) and no bounds flag may fire, so neither is ever read into a
result."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_15_gb300 as pa
from paged_kv_gqa_15_gb300 import workloads as W
from tests.gpu_util import assert_close_bf16, bf16_out, stale_fill_last_pages

pytestmark = pytest.mark.gpu
DEV = "cuda"
LENS = [0, 1, 15, 16, 17, 100, 511, 512, 513, 1100, 2049, 4000]
NAN_BITS = W.float_to_bits(np.float32("nan"))


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    yield
    assert pa.device_status() == 0


def _to_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV).view(torch.bfloat16)


def _poison_before(kc, vc, bt, first_keys, bs=16):
    """Sequence / request b sees no key before first_keys[b]: its table entries for the
    pages wholly before that key become -1 and that page's earlier rows become NaN."""
    bt = bt.copy()
    for b, lo in enumerate(first_keys):
        lo = int(lo)
        if lo <= 0:
            continue
        bt[b, :lo // bs] = -1
        if lo % bs:
            page = bt[b, lo // bs]
            kc[page, :, :lo % bs, :] = NAN_BITS
            vc[page, :, :lo % bs, :] = NAN_BITS
    return bt


def _decode_case(hd, nq, nkv, window, seed):
    w = W.make_decode("win", LENS, nq, nkv, hd, seed=seed, window=window)
    t = w.tensors("cpu")
    q, kc, vc = W.to_bits(t["q"]), W.to_bits(t["k_cache"]), W.to_bits(t["v_cache"])
    stale_fill_last_pages(kc, vc, w.block_tables, w.seq_lens, 16)
    lens = w.seq_lens.astype(np.int64)
    bt = _poison_before(kc, vc, w.block_tables, np.maximum(lens - window, 0))
    ref = oracle.decode(q, kc, vc, bt, w.seq_lens, nkv, 16, w.scale, window=window)
    return w, q, kc, vc, bt, ref


# (head_dim, nq, nkv): tensor-core split at GQA 4 and 8, CUDA-core kernels otherwise
SHAPES = [(128, 32, 8), (128, 64, 8), (64, 8, 8), (256, 16, 8), (128, 8, 4)]


@pytest.mark.parametrize("hd,nq,nkv", SHAPES)
@pytest.mark.parametrize("window", [1, 100, 512, 700, 3000])
@pytest.mark.parametrize("split", [False, True])
def test_windowed_decode_matches_oracle(hd, nq, nkv, window, split):
    w, q, kc, vc, bt, ref = _decode_case(hd, nq, nkv, window, seed=51 + hd + nq)
    q_d, kc_d, vc_d = _to_dev(q), _to_dev(kc), _to_dev(vc)
    bt_d = torch.from_numpy(bt).to(DEV)
    sl = torch.from_numpy(w.seq_lens).to(DEV)
    out = torch.full_like(q_d, float("nan"))
    if split:
        L = w.max_seq_len
        ws = pa.alloc_workspace(pa.decode_split_workspace_size(w.batch, nq, hd, L), DEV)
        ws.fill_(0xFF)   # partitions before a window are never written and never read
        pa.pa_decode_split(out, q_d, kc_d, vc_d, bt_d, sl, w.scale, L, ws,
                           sliding_window=window)
    else:
        pa.pa_decode(out, q_d, kc_d, vc_d, bt_d, sl, w.scale, sliding_window=window)
    assert pa.device_status() == 0
    assert_close_bf16(out, ref, what=f"decode hd {hd} g {nq // nkv} W {window} split {split}")


@pytest.mark.parametrize("hd,nq,nkv", [(128, 32, 8), (64, 8, 4)])
def test_windowed_partials_match_oracle_partitions(hd, nq, nkv):
    window = 700          # the first active partition is cut by the window
    w, q, kc, vc, bt, _ = _decode_case(hd, nq, nkv, window, seed=60)
    L = w.max_seq_len
    P = (L + 511) // 512
    ws = pa.alloc_workspace(pa.decode_split_workspace_size(w.batch, nq, hd, L), DEV)
    pa.pa_decode_partitions(_to_dev(q), _to_dev(kc), _to_dev(vc), torch.from_numpy(bt).to(DEV),
                            torch.from_numpy(w.seq_lens).to(DEV), w.scale, L, ws,
                            sliding_window=window)
    po, pm, pl = pa.decode_split_workspace_views(ws, w.batch, nq, hd, L)
    m, l, o = oracle.decode_partitions(q, kc, vc, bt, w.seq_lens, nkv, 16, w.scale, P,
                                       window=window)
    vf = W.bits_to_float(vc)
    vmax = float(np.abs(vf[np.isfinite(vf)]).max())
    for b, Lb in enumerate(LENS):
        p0, p1 = max(0, Lb - window) // 512, (Lb + 511) // 512
        gm, gl, go = (x[b, :, p0:p1].cpu().numpy().astype(np.float64) for x in (pm, pl, po))
        np.testing.assert_allclose(gm, m[b, :, p0:p1], atol=1e-4, rtol=0)
        np.testing.assert_allclose(gl, l[b, :, p0:p1], rtol=1e-4, atol=0)
        # P enters the tensor-core P.V as bf16: up to 2^-9 max|V| per partial output
        np.testing.assert_allclose(go, o[b, :, p0:p1], atol=2.0 ** -9 * vmax + 1e-5, rtol=0)


def test_window_covering_every_sequence_equals_no_window():
    w, q, kc, vc, bt, ref = _decode_case(128, 32, 8, 5000, seed=61)
    outs = []
    for window in (0, 5000):
        out = torch.empty((w.batch, 32, 128), dtype=torch.bfloat16, device=DEV)
        ws = pa.alloc_workspace(pa.decode_split_workspace_size(w.batch, 32, 128, 4000), DEV)
        pa.pa_decode_split(out, _to_dev(q), _to_dev(kc), _to_dev(vc),
                           torch.from_numpy(bt).to(DEV), torch.from_numpy(w.seq_lens).to(DEV),
                           w.scale, 4000, ws, sliding_window=window)
        outs.append(out)
    assert torch.equal(outs[0], outs[1])
    assert_close_bf16(outs[1], ref, what="W >= L")


def test_static_entry_point_takes_the_window():
    w, q, kc, vc, bt, ref = _decode_case(128, 32, 8, 700, seed=62)
    args = (_to_dev(q), _to_dev(kc), _to_dev(vc), torch.from_numpy(bt).to(DEV),
            torch.from_numpy(w.seq_lens).to(DEV), w.scale, w.max_seq_len)
    a = torch.empty((w.batch, 32, 128), dtype=torch.bfloat16, device=DEV)
    b = torch.empty_like(a)
    ws = pa.alloc_workspace(pa.decode_split_workspace_size(w.batch, 32, 128, w.max_seq_len), DEV)
    pa.pa_decode_split(a, *args, ws, sliding_window=700)
    pa.pa_decode_split_static(b, *args, sliding_window=700)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert_close_bf16(b, ref, what="static")


# ---- prefill ------------------------------------------------------------------------

QO = [1, 130, 300, 5, 700, 64]
KV = [1, 200, 300, 40, 900, 64]


@pytest.mark.parametrize("hd,nq,nkv", [(64, 4, 2), (128, 8, 2), (256, 4, 4)])
@pytest.mark.parametrize("window", [1, 7, 64, 100, 300, 5000])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("paged", [False, True])
def test_windowed_prefill_matches_oracle(hd, nq, nkv, window, causal, paged):
    w = W.make_prefill("win", QO, KV, nq, nkv, hd, seed=70 + hd, causal=causal, paged=paged,
                       window=window)
    t = w.tensors("cpu")
    q = W.to_bits(t["q"])
    qo_d = torch.from_numpy(w.qo_indptr).to(DEV)
    kv_d = torch.from_numpy(w.kv_indptr).to(DEV)
    o = torch.full((w.total_qo, nq, hd), float("nan"), dtype=torch.bfloat16, device=DEV)
    if paged:
        kc, vc = W.to_bits(t["k_cache"]), W.to_bits(t["v_cache"])
        stale_fill_last_pages(kc, vc, w.block_tables, w.kv_lens, 16)
        # a request's first query row sees keys from kv - qo - W + 1 on, and later rows
        # see even later keys: nothing before that key is ever needed
        first = np.maximum(w.kv_lens.astype(np.int64) - w.qo_lens - window + 1, 0)
        bt = _poison_before(kc, vc, w.block_tables, first)
        pa.pa_ragged_prefill(o, _to_dev(q), _to_dev(kc), _to_dev(vc), w.qo_indptr, w.kv_indptr,
                             qo_d, kv_d, w.scale, causal=causal,
                             block_tables=torch.from_numpy(bt).to(DEV), sliding_window=window)
        ref = oracle.prefill(q, kc, vc, w.qo_indptr, w.kv_indptr, nkv, w.scale, causal=causal,
                             block_tables=bt, window=window)
    else:
        k, v = W.to_bits(t["k"]), W.to_bits(t["v"])
        pa.pa_ragged_prefill(o, _to_dev(q), _to_dev(k), _to_dev(v), w.qo_indptr, w.kv_indptr,
                             qo_d, kv_d, w.scale, causal=causal, sliding_window=window)
        ref = oracle.prefill(q, k, v, w.qo_indptr, w.kv_indptr, nkv, w.scale, causal=causal,
                             window=window)
    assert pa.device_status() == 0
    assert_close_bf16(o, ref, what=f"prefill hd {hd} W {window} causal {causal} paged {paged}")


def test_windowed_decode_equals_last_row_of_windowed_prefill():
    lens = [40, 513, 1000, 2100]
    window = 77
    w = W.make_decode("win", lens, 32, 8, 128, seed=71, window=window)
    t = w.tensors(DEV)
    bt = torch.from_numpy(w.block_tables).to(DEV)
    sl = torch.from_numpy(w.seq_lens).to(DEV)
    dec = torch.empty_like(t["q"])
    pa.pa_decode(dec, t["q"], t["k_cache"], t["v_cache"], bt, sl, w.scale,
                 sliding_window=window)
    qo_indptr = np.arange(len(lens) + 1, dtype=np.int32)
    kv_indptr = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    pre = torch.empty_like(t["q"])
    pa.pa_ragged_prefill(pre, t["q"], t["k_cache"], t["v_cache"], qo_indptr, kv_indptr,
                         torch.from_numpy(qo_indptr).to(DEV), torch.from_numpy(kv_indptr).to(DEV),
                         w.scale, causal=True, block_tables=bt, sliding_window=window)
    torch.cuda.synchronize()
    ref = oracle.decode(W.to_bits(t["q"].cpu()), W.to_bits(t["k_cache"].cpu()),
                        W.to_bits(t["v_cache"].cpu()), w.block_tables, w.seq_lens, 8, 16,
                        w.scale, window=window)
    assert_close_bf16(dec, ref, what="decode")
    assert_close_bf16(pre, ref, what="prefill")
    # two different kernels (P in fp32 vs bf16): agree to the output rounding
    assert np.abs(bf16_out(dec) - bf16_out(pre)).max() <= 2 * 2 ** -8 * max(1.0, np.abs(ref).max())
