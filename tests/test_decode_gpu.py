"""GPU parity of the cache write and the paged decode (single pass and split-KV)
against the fp64 oracle, through the C ABI."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_15_gb300 as pa
from paged_kv_gqa_15_gb300 import workloads as W
from tests.gpu_util import assert_close_bf16, bf16_out, stale_fill_last_pages

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    yield
    assert pa.device_status() == 0


def _to_dev(bits):
    return torch.from_numpy(bits.view(np.int16)).to(DEV).view(torch.bfloat16)


def _run_decode(w, split, layout="HND", stale=True, q_zero=False):
    t = w.tensors("cpu")
    q = W.to_bits(t["q"])
    if q_zero:
        q[:] = 0
    kc, vc = W.to_bits(t["k_cache"]), W.to_bits(t["v_cache"])
    if stale:
        stale_fill_last_pages(kc, vc, w.block_tables, w.seq_lens, w.block_size)
    strides = oracle.hnd_strides(w.num_kv_heads, w.block_size, w.head_dim)
    kc_d, vc_d = _to_dev(kc), _to_dev(vc)
    if layout == "NHD":
        kc_d = kc_d.permute(0, 2, 1, 3).contiguous()
        vc_d = vc_d.permute(0, 2, 1, 3).contiguous()
    q_d = _to_dev(q)
    bt = torch.from_numpy(w.block_tables).to(DEV)
    sl = torch.from_numpy(w.seq_lens).to(DEV)
    out = torch.full_like(q_d, float("nan"))
    ws = None
    if split:
        L = max(w.max_seq_len, 1)
        ws = pa.alloc_workspace(pa.decode_split_workspace_size(w.batch, w.num_q_heads,
                                                               w.head_dim, L), DEV)
        ws.fill_(0xFF)  # NaN pattern: partitions that are never written must never be read
        pa.pa_decode_split(out, q_d, kc_d, vc_d, bt, sl, w.scale, L, ws, layout=layout,
                           sliding_window=w.window)
    else:
        pa.pa_decode(out, q_d, kc_d, vc_d, bt, sl, w.scale, layout=layout,
                     sliding_window=w.window)
    torch.cuda.synchronize()
    ref = oracle.decode(q, kc, vc, w.block_tables, w.seq_lens, w.num_kv_heads, w.block_size,
                        w.scale, strides=strides, window=w.window)
    return out, ref, ws, (q, kc, vc)


# ---- cache write ---------------------------------------------------------------------


@pytest.mark.parametrize("hd", [64, 128, 256])
@pytest.mark.parametrize("layout", ["HND", "NHD"])
def test_write_cache_bit_exact(hd, layout):
    rng = np.random.default_rng(hd)
    nb, nkv, bs, T = 40, 4, 16, 300
    sentinel = np.uint16(0x7F7F)
    kc = np.full((nb, nkv, bs, hd), sentinel, np.uint16)
    vc = np.full_like(kc, sentinel)
    k = rng.integers(0, 0xFFFF, size=(T, nkv, hd)).astype(np.uint16)   # any bit pattern
    v = rng.integers(0, 0xFFFF, size=(T, nkv, hd)).astype(np.uint16)
    slots = rng.choice(nb * bs, size=T, replace=False).astype(np.int64)
    slots[::9] = -1
    kc_d, vc_d = _to_dev(kc), _to_dev(vc)
    if layout == "NHD":
        kc_d = kc_d.permute(0, 2, 1, 3).contiguous()
        vc_d = vc_d.permute(0, 2, 1, 3).contiguous()
    pa.pa_write_cache(_to_dev(k), _to_dev(v), kc_d, vc_d, torch.from_numpy(slots).to(DEV),
                      layout=layout)
    oracle.write_cache(k, v, kc, vc, slots, bs)
    got_k, got_v = W.to_bits(kc_d), W.to_bits(vc_d)
    if layout == "NHD":
        got_k, got_v = got_k.transpose(0, 2, 1, 3), got_v.transpose(0, 2, 1, 3)
    np.testing.assert_array_equal(got_k, kc)
    np.testing.assert_array_equal(got_v, vc)
    assert pa.device_status() == 0


def test_write_cache_out_of_range_slot_is_flagged_not_written():
    nb, nkv, bs, hd = 4, 2, 16, 64
    kc = torch.zeros((nb, nkv, bs, hd), dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    k = torch.ones((2, nkv, hd), dtype=torch.bfloat16, device=DEV)
    slots = torch.tensor([nb * bs, 5], dtype=torch.int64, device=DEV)
    pa.pa_write_cache(k, k, kc, vc, slots)
    st = pa.device_status()
    assert st & (1 << pa.PA_ERR_DEVICE_BOUNDS)
    assert kc.float().sum().item() == nkv * hd       # only slot 5 was written
    assert kc[0, :, 5].float().min().item() == 1.0


def test_write_cache_empty_is_a_no_op():
    kc = torch.zeros((2, 1, 16, 64), dtype=torch.bfloat16, device=DEV)
    k = torch.zeros((0, 1, 64), dtype=torch.bfloat16, device=DEV)
    pa.pa_write_cache(k, k, kc, kc.clone(), torch.zeros(0, dtype=torch.int64, device=DEV))
    assert pa.device_status() == 0


# ---- decode ------------------------------------------------------------------------------


def test_tiny_config_single_pass():
    out, ref, _, _ = _run_decode(W.tiny_decode(), split=False)
    assert_close_bf16(out, ref, what="tiny decode")


@pytest.mark.parametrize("window", [0, 5000])
@pytest.mark.parametrize("hd,nq,nkv", [(128, 32, 8), (64, 8, 8), (256, 16, 2)])
def test_single_pass_cluster_split_of_long_sequences(hd, nq, nkv, window):
    """Few (sequence, kv head) items with long sequences: the single pass spreads each
    over a 4-CTA cluster that merges its partial results in distributed shared memory.
    Lengths cover page counts not divisible by 4, fewer pages than ranks, and 0."""
    lens = [70001, 4099, 3, 0, 1025]
    w = W.make_decode("cluster", lens, nq, nkv, hd, seed=hd + window, window=window)
    out, ref, _, _ = _run_decode(w, split=False)
    assert_close_bf16(out, ref, what=f"cluster single pass hd{hd} window {window}")
    assert pa.device_status() == 0


@pytest.mark.parametrize("window", [0, 700])
@pytest.mark.parametrize("nq,nkv", [(32, 8), (64, 8)])
def test_tensor_core_single_pass(nq, nkv, window):
    """The single pass at head_dim 128 with GQA 4 or 8 runs on the tensor cores: each CTA
    owns whole (sequence, kv head) pairs (snake order over the sequences sorted by their
    partitions) and merges the partitions in registers.  Lengths include 0, 1, partition
    edges, ties and long sequences."""
    rng = np.random.default_rng(nq + window)
    lens = np.concatenate([[0, 1, 511, 512, 513, 4096, 4096, 9000, 0],
                           rng.integers(1, 3000, size=40)])
    w = W.make_decode("tc_single", lens, nq, nkv, 128, seed=nq * 3 + window, window=window)
    out, ref, _, _ = _run_decode(w, split=False)
    assert_close_bf16(out, ref, what=f"tensor-core single pass nq{nq} window {window}")
    assert pa.device_status() == 0


def test_tiny_config_split():
    out, ref, _, _ = _run_decode(W.tiny_decode(), split=True)
    assert_close_bf16(out, ref, what="tiny split decode")


LENS = [0, 1, 15, 16, 17, 100, 511, 512, 513, 1024, 1500, 2049]


@pytest.mark.parametrize("hd", [64, 128, 256])
@pytest.mark.parametrize("nq,nkv", [(4, 4), (8, 4), (16, 4), (32, 4)])
@pytest.mark.parametrize("split", [False, True])
def test_decode_shapes_and_ragged_lengths(hd, nq, nkv, split):
    w = W.make_decode("grid", LENS, nq, nkv, hd, seed=hd * 100 + nq)
    out, ref, _, _ = _run_decode(w, split)
    assert_close_bf16(out, ref, what=f"hd{hd} g{nq // nkv} split={split}")


@pytest.mark.parametrize("split", [False, True])
def test_decode_nhd_layout(split):
    w = W.make_decode("nhd", [33, 700, 5], 8, 2, 128, seed=31)
    out, ref, _, _ = _run_decode(w, split, layout="NHD")
    assert_close_bf16(out, ref, what="NHD")


def test_zero_query_returns_mean_of_values():
    w = W.make_decode("q0", [3, 40, 600], 8, 2, 128, seed=32)
    out, ref, _, (q, kc, vc) = _run_decode(w, split=True, q_zero=True)
    assert_close_bf16(out, ref, what="q=0")


def test_split_partials_match_oracle_partitions():
    w = W.make_decode("parts", [1, 512, 513, 1700, 3000], 8, 2, 128, seed=33)
    out, ref, ws, (q, kc, vc) = _run_decode(w, split=True)
    L = w.max_seq_len
    P = (L + 511) // 512
    po, pm, pl = pa.decode_split_workspace_views(ws, w.batch, w.num_q_heads, w.head_dim, L)
    m, l, o = oracle.decode_partitions(q, kc, vc, w.block_tables, w.seq_lens, 2, 16, w.scale, P)
    vmax = float(np.abs(W.bits_to_float(vc)).max())
    for b, Lb in enumerate(w.seq_lens):
        np_ = (int(Lb) + 511) // 512
        gm, gl, go = (x[b, :, :np_].cpu().numpy().astype(np.float64) for x in (pm, pl, po))
        np.testing.assert_allclose(gm, m[b, :, :np_], atol=1e-4, rtol=0)
        np.testing.assert_allclose(gl, l[b, :, :np_], rtol=1e-4, atol=0)
        # The partial output is a p-weighted mean of V rows; the tensor-core P.V takes
        # P rounded to bf16 (relative error <= 2^-9 per weight), which can move it by up
        # to 2^-9 * max|V| (fp32 P on the CUDA-core path stays far inside this bound).
        np.testing.assert_allclose(go, o[b, :, :np_], atol=2.0 ** -9 * vmax + 1e-5, rtol=0)
    assert_close_bf16(out, ref, what="split")


def test_split_equals_single_pass():
    w = W.make_decode("eq", [700, 4096, 2500, 1], 32, 8, 128, seed=34)
    single, ref, _, _ = _run_decode(w, split=False)
    split, _, _, _ = _run_decode(w, split=True)
    a, b = bf16_out(single), bf16_out(split)
    assert np.abs(a - b).max() <= 2 * 2 ** -8 * max(1.0, np.abs(ref).max())


def test_page_permutation_invariance_on_gpu():
    w = W.make_decode("perm", [300, 77], 8, 2, 128, seed=35)
    out1, ref, _, (q, kc, vc) = _run_decode(w, split=True, stale=False)
    rng = np.random.default_rng(1)
    perm = rng.permutation(w.num_blocks)
    bt2 = w.block_tables.copy()
    used = bt2 != W.PAD_ENTRY
    bt2[used] = perm[bt2[used]]
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[perm], vc2[perm] = kc, vc
    out2 = torch.empty_like(out1)
    ws = pa.alloc_workspace(pa.decode_split_workspace_size(2, 8, 128, 300), DEV)
    pa.pa_decode_split(out2, _to_dev(q), _to_dev(kc2), _to_dev(vc2),
                       torch.from_numpy(bt2).to(DEV), torch.from_numpy(w.seq_lens).to(DEV),
                       w.scale, 300, ws)
    np.testing.assert_array_equal(W.to_bits(out1), W.to_bits(out2))


@pytest.mark.parametrize("split", [False, True])
def test_bad_block_id_is_flagged_and_contributes_nothing(split):
    w = W.make_decode("bad", [40, 40], 4, 2, 64, seed=36)
    t = w.tensors("cpu")
    q, kc, vc = (W.to_bits(t[n]) for n in ("q", "k_cache", "v_cache"))
    bt = w.block_tables.copy()
    bt[1, 1] = w.num_blocks + 5        # tokens 16..31 of sequence 1 point nowhere
    out = torch.empty_like(_to_dev(q))
    args = (out, _to_dev(q), _to_dev(kc), _to_dev(vc), torch.from_numpy(bt).to(DEV),
            torch.from_numpy(w.seq_lens).to(DEV), w.scale)
    if split:
        ws = pa.alloc_workspace(pa.decode_split_workspace_size(2, 4, 64, 40), DEV)
        pa.pa_decode_split(*args, 40, ws)
    else:
        pa.pa_decode(*args)
    st = pa.device_status()
    assert st & (1 << pa.PA_ERR_DEVICE_BOUNDS)
    # sequence 0 is untouched by the bad entry
    ref = oracle.decode(q, kc, vc, w.block_tables, w.seq_lens, 2, 16, w.scale)
    assert_close_bf16(bf16_out(out)[0], ref[0], what="good sequence")
    # sequence 1 equals attention over its tokens without the missing page
    keep = np.r_[0:16, 32:40]
    bt_keep = np.full((1, 2), W.PAD_ENTRY, np.int32)
    # rebuild as an explicit token list through a scratch pool
    nb = 3
    kc1 = np.zeros((nb, 2, 16, 64), np.uint16)
    vc1 = np.zeros_like(kc1)
    for j, src in enumerate(keep):
        page, row = w.block_tables[1, src // 16], src % 16
        kc1[j // 16, :, j % 16] = kc[page, :, row]
        vc1[j // 16, :, j % 16] = vc[page, :, row]
    bt_keep[0] = [0, 1]
    ref1 = oracle.decode(q[1:2], kc1, vc1, bt_keep, np.array([len(keep)], np.int32), 2, 16,
                         w.scale)
    assert_close_bf16(bf16_out(out)[1], ref1[0], what="sequence with a bad page")


def test_seq_len_beyond_table_is_clamped_and_flagged():
    w = W.make_decode("clamp", [32], 4, 2, 64, seed=37)
    t = w.tensors("cpu")
    sl = torch.tensor([10_000], dtype=torch.int32, device=DEV)   # table holds 2 pages
    out = torch.empty_like(t["q"].to(DEV))
    pa.pa_decode(out, t["q"].to(DEV), t["k_cache"].to(DEV), t["v_cache"].to(DEV),
                 torch.from_numpy(w.block_tables).to(DEV), sl, w.scale)
    assert pa.device_status() & (1 << pa.PA_ERR_DEVICE_BOUNDS)
    q, kc, vc = (W.to_bits(t[n]) for n in ("q", "k_cache", "v_cache"))
    ref = oracle.decode(q, kc, vc, w.block_tables, w.seq_lens, 2, 16, w.scale)
    assert_close_bf16(out, ref, what="clamped")


# ---- full-size workloads -------------------------------------------------------------------


def test_llama8b_config_write_then_split_decode_full_parity():
    """64 sequences, 32 q / 8 kv heads, hd 128, seq_lens U[512, 4096]: the new token
    goes in through pa_write_cache, then the split decode; every output row is compared."""
    w = W.llama8b_decode()
    t = w.tensors(DEV)
    kc_h, vc_h = W.to_bits(t["k_cache"]), W.to_bits(t["v_cache"])
    slots = torch.from_numpy(w.slot_mapping).to(DEV)
    pa.pa_write_cache(t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], slots)
    oracle.write_cache(W.to_bits(t["k_new"]), W.to_bits(t["v_new"]), kc_h, vc_h, w.slot_mapping,
                       16)
    bt = torch.from_numpy(w.block_tables).to(DEV)
    sl = torch.from_numpy(w.seq_lens).to(DEV)
    out = torch.empty_like(t["q"])
    ws = pa.alloc_workspace(pa.decode_split_workspace_size(w.batch, 32, 128, w.max_seq_len), DEV)
    pa.pa_decode_split(out, t["q"], t["k_cache"], t["v_cache"], bt, sl, w.scale, w.max_seq_len,
                       ws)
    out1 = torch.empty_like(out)
    pa.pa_decode(out1, t["q"], t["k_cache"], t["v_cache"], bt, sl, w.scale)
    ref = oracle.decode(W.to_bits(t["q"]), kc_h, vc_h, w.block_tables, w.seq_lens, 8, 16,
                        w.scale)
    assert_close_bf16(out, ref, what="llama8b split")
    assert_close_bf16(out1, ref, what="llama8b single pass")
    # the cache write itself is bit-exact on the touched pages
    touched = np.unique(w.slot_mapping // 16)
    np.testing.assert_array_equal(W.to_bits(t["k_cache"][torch.from_numpy(touched).to(DEV)]),
                                  kc_h[touched])
