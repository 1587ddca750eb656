"""Pins of the oracle's sliding window (a query at position pos sees keys j with
pos - W < j; "paged_attn.py", forward_prefix's sliding_window, and "libmir-cuda
attention/mod.rs", active_partitions(token_count, window)) against brute force with a
window mask (tests/brute.py), closed forms and invariants that do not come from the
oracle."""
import numpy as np
import pytest

import oracle
from paged_kv_gqa_15_gb300 import workloads as W
from tests import brute

LENS = [1, 15, 16, 17, 100, 511, 512, 513, 1100, 2049]


def _decode_inputs(w):
    t = w.tensors("cpu")
    return W.to_bits(t["q"]), W.to_bits(t["k_cache"]), W.to_bits(t["v_cache"])


@pytest.mark.parametrize("window", [1, 16, 100, 512, 700, 5000])
def test_windowed_decode_matches_brute_force(oracle_lib, window):
    w = W.make_decode("win", LENS, 8, 2, 64, seed=31)
    q, kc, vc = _decode_inputs(w)
    got = oracle.decode(q, kc, vc, w.block_tables, w.seq_lens, 2, 16, w.scale, window=window)
    ref = brute.brute_decode(q, kc, vc, w.block_tables, w.seq_lens, 2, 16, w.scale,
                             oracle.hnd_strides(2, 16, 64), window=window)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_window_covering_the_sequence_changes_nothing(oracle_lib):
    w = W.make_decode("win", LENS, 4, 2, 64, seed=32)
    q, kc, vc = _decode_inputs(w)
    full = oracle.decode(q, kc, vc, w.block_tables, w.seq_lens, 2, 16, w.scale)
    for window in (int(max(LENS)), int(max(LENS)) + 1, 1 << 20):
        got = oracle.decode(q, kc, vc, w.block_tables, w.seq_lens, 2, 16, w.scale,
                            window=window)
        np.testing.assert_array_equal(got, full)
    # and W <= 0 is no window at all
    np.testing.assert_array_equal(
        oracle.decode(q, kc, vc, w.block_tables, w.seq_lens, 2, 16, w.scale, window=-3), full)


def test_window_of_one_returns_the_newest_value_row(oracle_lib):
    w = W.make_decode("win", LENS, 4, 2, 64, seed=33)
    q, kc, vc = _decode_inputs(w)
    got = oracle.decode(q, kc, vc, w.block_tables, w.seq_lens, 2, 16, w.scale, window=1)
    v = brute.widen(vc)
    for b, L in enumerate(LENS):
        page = w.block_tables[b, (L - 1) // 16]
        for h in range(4):
            np.testing.assert_array_equal(got[b, h], v[page, h // 2, (L - 1) % 16])


def test_page_aligned_window_equals_the_truncated_table(oracle_lib):
    # a window starting on a page boundary sees exactly the pages from that one on
    lens = np.array([160, 1040, 48], np.int32)
    window = 32
    w = W.make_decode("win", lens, 4, 1, 64, seed=34)
    q, kc, vc = _decode_inputs(w)
    got = oracle.decode(q, kc, vc, w.block_tables, lens, 1, 16, w.scale, window=window)
    bt2 = np.full_like(w.block_tables, W.PAD_ENTRY)
    for b, L in enumerate(lens):
        first = (L - window) // 16
        n = (L + 15) // 16 - first
        bt2[b, :n] = w.block_tables[b, first:first + n]
    ref = oracle.decode(q, kc, vc, bt2, np.full(3, window, np.int32), 1, 16, w.scale)
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("window", [1, 300, 512, 513, 1024, 1500])
def test_windowed_split_merge_equals_windowed_single_pass(oracle_lib, window):
    w = W.make_decode("win", LENS, 8, 2, 64, seed=35)
    q, kc, vc = _decode_inputs(w)
    single = oracle.decode(q, kc, vc, w.block_tables, w.seq_lens, 2, 16, w.scale,
                           window=window)
    m, l, o = oracle.decode_partitions(q, kc, vc, w.block_tables, w.seq_lens, 2, 16, w.scale,
                                       5, window=window)
    for b, L in enumerate(LENS):
        first = max(0, L - window) // 512
        assert np.isnan(m[b, :, :first]).all()           # wholly before the window
        assert np.isfinite(m[b, :, first:(L + 511) // 512]).all()
    merged = oracle.merge_partitions(m, l, o, w.seq_lens, window=window)
    np.testing.assert_allclose(merged, single, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("window", [1, 7, 64, 200])
def test_windowed_prefill_matches_brute_force(oracle_lib, causal, window):
    qo, kv = np.array([6, 130, 3, 70]), np.array([6, 200, 9, 70])
    w = W.make_prefill("win", qo, kv, 4, 2, 64, seed=36)
    t = w.tensors("cpu")
    q, k, v = (W.to_bits(t[n]) for n in ("q", "k", "v"))
    got = oracle.prefill(q, k, v, w.qo_indptr, w.kv_indptr, 2, w.scale, causal=causal,
                         window=window)
    ref = brute.brute_prefill_contiguous(q, k, v, w.qo_indptr, w.kv_indptr, 2, w.scale,
                                         causal, window=window)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_windowed_decode_equals_last_row_of_windowed_paged_prefill(oracle_lib):
    lens = [40, 513, 1000]
    window = 77
    w = W.make_decode("win", lens, 4, 2, 64, seed=37)
    q, kc, vc = _decode_inputs(w)
    dec = oracle.decode(q, kc, vc, w.block_tables, w.seq_lens, 2, 16, w.scale, window=window)
    qo_indptr = np.arange(len(lens) + 1, dtype=np.int32)         # one query row each
    kv_indptr = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    pre = oracle.prefill(q, kc, vc, qo_indptr, kv_indptr, 2, w.scale, causal=True,
                         block_tables=w.block_tables, window=window)
    np.testing.assert_array_equal(pre, dec)
