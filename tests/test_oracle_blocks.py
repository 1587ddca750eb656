"""Pins of the oracle's page copies (copy_blocks / swap_blocks, "paged_attn.py",
PagedAttention.copy_blocks and swap_blocks) against facts that do not come from the
oracle: per-page digests taken before the copy, round trips, and the attention
output of a sequence forked onto copied pages."""
import hashlib

import numpy as np

import oracle
from paged_kv_gqa_15_gb300 import workloads as W


def _digests(pool):
    return [hashlib.sha256(pool[b].tobytes()).hexdigest() for b in range(pool.shape[0])]


def _random_pools(n, num_blocks, page_shape, seed):
    rng = np.random.default_rng(seed)
    return [rng.integers(0, 256, size=(num_blocks,) + page_shape, dtype=np.uint8)
            for _ in range(n)]


def test_copy_blocks_moves_exactly_the_mapped_pages(oracle_lib):
    pools = _random_pools(3, 12, (3, 16), seed=1)
    before = [_digests(p) for p in pools]
    # a source may feed several destinations (a page shared by many forks)
    pairs = [(0, 5), (3, 7), (3, 9), (-1, 2), (4, -1), (12, 1), (2, 12), (11, 0)]
    bad = oracle.copy_blocks(pools, pairs)
    assert bad == 2 * len(pools)          # (12, 1) and (2, 12) in every pool
    moved = {5: 0, 7: 3, 9: 3, 0: 11}
    for p, d0 in zip(pools, before):
        after = _digests(p)
        for b in range(12):
            assert after[b] == d0[moved.get(b, b)], f"page {b}"


def test_identity_pairs_leave_the_pool_unchanged(oracle_lib):
    pools = _random_pools(2, 6, (64,), seed=2)
    ref = [p.copy() for p in pools]
    assert oracle.copy_blocks(pools, [(b, b) for b in range(6)]) == 0
    for p, r in zip(pools, ref):
        np.testing.assert_array_equal(p, r)


def test_swap_out_and_back_restores_the_pages(oracle_lib):
    dev = _random_pools(1, 20, (2, 16, 8), seed=3)[0]
    host = np.zeros((6,) + dev.shape[1:], np.uint8)
    src_pages = [17, 2, 9, 0]
    out_pairs = [(s, h) for h, s in enumerate(src_pages)]
    assert oracle.swap_blocks(dev, host, out_pairs) == 0
    for h, s in enumerate(src_pages):
        np.testing.assert_array_equal(host[h], dev[s])
    np.testing.assert_array_equal(host[4:], 0)   # pages no pair wrote stay as they were
    back = np.zeros_like(dev)
    new_pages = [3, 4, 18, 11]
    assert oracle.swap_blocks(host, back, [(h, n) for h, n in enumerate(new_pages)]) == 0
    for s, n in zip(src_pages, new_pages):
        np.testing.assert_array_equal(back[n], dev[s])
    untouched = [b for b in range(20) if b not in new_pages]
    np.testing.assert_array_equal(back[untouched], 0)


def test_swap_counts_pairs_outside_either_pool(oracle_lib):
    src = _random_pools(1, 4, (16,), seed=4)[0]
    dst = np.zeros((2, 16), np.uint8)
    assert oracle.swap_blocks(src, dst, [(0, 1), (4, 0), (1, 2), (3, 0)]) == 2
    np.testing.assert_array_equal(dst[1], src[0])
    np.testing.assert_array_equal(dst[0], src[3])


def test_forked_sequence_attends_exactly_like_the_original(oracle_lib):
    # copy-on-write fork: the child's block table names copies of the parent's pages,
    # so decode over the child's table must equal decode over the parent's, exactly
    w = W.make_decode("fork", [70, 33], 4, 2, 64, seed=5, num_blocks=24)
    t = w.tensors("cpu")
    q, kc, vc = (W.to_bits(t[n]) for n in ("q", "k_cache", "v_cache"))
    bt = w.block_tables
    used = sorted(set(int(x) for x in bt[bt != W.PAD_ENTRY].ravel()))
    free = [b for b in range(w.num_blocks) if b not in used]
    child = bt.copy()
    pairs = []
    for b in range(w.batch):
        for i in range((int(w.seq_lens[b]) + 15) // 16):
            new = free.pop()
            pairs.append((int(bt[b, i]), new))
            child[b, i] = new
    # the child's pages hold zeros until copied: without the copy the outputs differ
    kc_z, vc_z = kc.copy(), vc.copy()
    for _, d in pairs:
        kc_z[d] = 0
        vc_z[d] = 0
    before = oracle.decode(q, kc_z, vc_z, child, w.seq_lens, 2, 16, w.scale)
    parent = oracle.decode(q, kc_z, vc_z, bt, w.seq_lens, 2, 16, w.scale)
    assert not np.array_equal(before, parent)
    assert oracle.copy_blocks([kc_z, vc_z], pairs) == 0
    forked = oracle.decode(q, kc_z, vc_z, child, w.seq_lens, 2, 16, w.scale)
    np.testing.assert_array_equal(forked, parent)
