"""Planted mistakes: each mutation of a COPY of the oracle source must be caught.

A plausible slip anywhere in the oracle (a dropped term, a wrong index or
sign, a transposed operand) has to fail at least one pin, otherwise the pins
do not really tie the oracle down.  The copies are compiled into a temporary
directory on the CPU and exercised in a child process (a mutated index can
read or write out of bounds, which must not corrupt the test process); a
failed check or a crash of the child both count as caught.  The committed
oracle is never modified.
"""
import math
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
from paged_kv_gqa_15_gb300 import workloads as W
from tests import brute

SRC = os.path.join(os.path.dirname(oracle.__file__), "pa_oracle.c")

MUTATIONS = {
    "dropped_scale": ("        s *= scale;\n        scores[j] = s;", "        scores[j] = s;"),
    "gqa_modulo": ("int kh = h / g; /* contiguous GQA groups */", "int kh = h % c->nkv;"),
    "top_left_causal": ("int64_t lim = i + (kv - qo) + 1;", "int64_t lim = i + 1;"),
    "page_row_swapped": ("(j % c->bs) * c->s_token;\n}", "(j / c->bs) * c->s_token;\n}"),
    "merge_without_lp": ("double w = l[bh * max_parts + p] * exp(m[bh * max_parts + p] - M);",
                         "double w = exp(m[bh * max_parts + p] - M);"),
    "slot_div_mod_swapped": ("int64_t page = slot / bs, row = slot % bs;",
                             "int64_t page = slot % bs, row = slot / bs;"),
    "unnormalised_output": ("    for (int d = 0; d < hd; ++d) out[d] /= den;\n", ""),
    "partition_unnormalised": ("for (int e = 0; e < d->hd; ++e) op[e] /= lsum;", ""),
    "max_not_subtracted": ("double p = exp(scores[j] - mx);", "double p = exp(scores[j]);"),
    "wrong_exp_sign": ("double w = exp(sc[j - j0] - mx);", "double w = exp(mx - sc[j - j0]);"),
    "pair_columns_swapped": ("int64_t s = mapping[2 * i], d = mapping[2 * i + 1];",
                             "int64_t d = mapping[2 * i], s = mapping[2 * i + 1];"),
    "copy_from_destination_index": ("const uint8_t *from = src + s * block_bytes;",
                                    "const uint8_t *from = src + d * block_bytes;"),
    "half_page_copied": ("for (int64_t b = 0; b < block_bytes; ++b) to[b] = from[b];",
                         "for (int64_t b = 0; b < block_bytes / 2; ++b) to[b] = from[b];"),
    "page_bound_off_by_one": ("if (s >= src_blocks || d >= dst_blocks) {",
                              "if (s > src_blocks || d > dst_blocks) {"),
    "first_pool_only": ("for (int t = 0; t < num_pools; ++t)\n        bad +=",
                        "for (int t = 0; t < 1; ++t)\n        bad +="),
    "window_one_key_wider": ("    return pos - w + 1;\n}", "    return pos - w;\n}"),
    "decode_window_from_length": ("int64_t j0 = L > 0 ? window_first(L - 1, c->window) : 0;",
                                  "int64_t j0 = L > 0 ? window_first(L, c->window) : 0;"),
    "partition_not_clipped_to_window": ("        if (j0 < jw) j0 = jw;\n", ""),
    "merge_from_partition_zero": (
        "int64_t p0 = (L > 0 ? window_first(L - 1, window) : 0) / part;", "int64_t p0 = 0;"),
    "prefill_window_ignored": ("int64_t lo = window_first(i + (kv - qo), c->window);",
                               "int64_t lo = 0;"),
    "e4m3_bias_off_by_one": ("ldexp(1.0 + m / 8.0, e - 7)", "ldexp(1.0 + m / 8.0, e - 8)"),
    "e4m3_subnormal_exponent": ("ldexp(m / 8.0, -6)", "ldexp(m / 8.0, -7)"),
    "e4m3_ties_to_odd": ("(err == best_err && (c & 1) == 0)", "(err == best_err && (c & 1) == 1)"),
    "fp8_write_multiplies_by_scale": ("oracle_e4m3_encode(kx / k_scale)",
                                      "oracle_e4m3_encode(kx * k_scale)"),
    "fp8_read_ignores_scale": (
        "return oracle_e4m3_value(((const uint8_t *)p->base)[idx]) * p->scale;",
        "return oracle_e4m3_value(((const uint8_t *)p->base)[idx]);"),
}


def _check_decode():
    w = W.make_decode("mut", [17, 33, 64, 100], 4, 2, 64, seed=1000, num_blocks=64)
    t = w.tensors("cpu")
    q, kc, vc = (W.to_bits(t[n]) for n in ("q", "k_cache", "v_cache"))
    got = oracle.decode(q, kc, vc, w.block_tables, w.seq_lens, 2, 16, w.scale)
    ref = brute.brute_decode(q, kc, vc, w.block_tables, w.seq_lens, 2, 16, w.scale,
                             oracle.hnd_strides(2, 16, 64))
    np.testing.assert_allclose(got, ref, atol=1e-12, rtol=0)


def _check_prefill():
    qo, kv = np.array([6, 10, 3]), np.array([6, 14, 9])
    w = W.make_prefill("mut", qo, kv, 4, 2, 64, seed=7)
    t = w.tensors("cpu")
    q, k, v = (W.to_bits(t[n]) for n in ("q", "k", "v"))
    got = oracle.prefill(q, k, v, w.qo_indptr, w.kv_indptr, 2, w.scale, causal=True)
    ref = brute.brute_prefill_contiguous(q, k, v, w.qo_indptr, w.kv_indptr, 2, w.scale, True)
    np.testing.assert_allclose(got, ref, atol=1e-12, rtol=0)


def _check_split():
    w = W.make_decode("mut", [300, 1100, 2000], 4, 2, 64, seed=13)
    t = w.tensors("cpu")
    q, kc, vc = (W.to_bits(t[n]) for n in ("q", "k_cache", "v_cache"))
    strides = oracle.hnd_strides(2, 16, 64)
    ref = brute.brute_decode(q, kc, vc, w.block_tables, w.seq_lens, 2, 16, w.scale, strides)
    m, l, o = oracle.decode_partitions(q, kc, vc, w.block_tables, w.seq_lens, 2, 16, w.scale, 4)
    merged = oracle.merge_partitions(m, l, o, w.seq_lens)
    np.testing.assert_allclose(merged, ref, atol=1e-12, rtol=0)


def _check_write():
    rng = np.random.default_rng(3)
    kc = np.zeros((8, 2, 16, 64), np.uint16)
    vc = np.zeros_like(kc)
    k = rng.integers(1, 0x7F00, size=(20, 2, 64)).astype(np.uint16)
    v = rng.integers(1, 0x7F00, size=(20, 2, 64)).astype(np.uint16)
    slots = rng.choice(8 * 16, size=20, replace=False).astype(np.int64)
    oracle.write_cache(k, v, kc, vc, slots, 16)
    for t, s in enumerate(slots):
        np.testing.assert_array_equal(kc[s // 16, :, s % 16], k[t])
        np.testing.assert_array_equal(vc[s // 16, :, s % 16], v[t])


def _check_large_logits():
    # scores of several hundred: exp() overflows unless the row max is subtracted
    w = W.make_decode("mut", [40, 90], 2, 1, 64, seed=21)
    t = w.tensors("cpu")
    q, kc, vc = (W.to_bits(t[n]) for n in ("q", "k_cache", "v_cache"))
    got = oracle.decode(q, kc, vc, w.block_tables, w.seq_lens, 1, 16, 100.0)
    ref = brute.brute_decode(q, kc, vc, w.block_tables, w.seq_lens, 1, 16, 100.0,
                             oracle.hnd_strides(1, 16, 64))
    np.testing.assert_allclose(got, ref, atol=1e-12, rtol=0)


def _check_blocks():
    rng = np.random.default_rng(8)
    pools = [rng.integers(0, 256, size=(6, 48), dtype=np.uint8) for _ in range(3)]
    ref = [p.copy() for p in pools]
    # pairs past the end of the pool must be skipped: (5, 6) would write one page past it,
    # so the pools get a guard page that has to stay untouched
    guarded = [np.concatenate([p, np.full((1, 48), 0xAB, np.uint8)]) for p in pools]
    views = [g[:6] for g in guarded]
    bad = oracle.copy_blocks(views, [(1, 4), (2, 0), (5, 6), (6, 3)])
    assert bad == 2 * len(pools)
    for g, r in zip(guarded, ref):
        exp = r.copy()
        exp[4] = r[1]
        exp[0] = r[2]
        np.testing.assert_array_equal(g[:6], exp)
        np.testing.assert_array_equal(g[6], 0xAB)


def _check_window():
    lens = [1, 17, 300, 513, 1100]
    w = W.make_decode("mut", lens, 4, 2, 64, seed=40)
    t = w.tensors("cpu")
    q, kc, vc = (W.to_bits(t[n]) for n in ("q", "k_cache", "v_cache"))
    strides = oracle.hnd_strides(2, 16, 64)
    for window in (1, 100, 600):
        ref = brute.brute_decode(q, kc, vc, w.block_tables, w.seq_lens, 2, 16, w.scale,
                                 strides, window=window)
        got = oracle.decode(q, kc, vc, w.block_tables, w.seq_lens, 2, 16, w.scale,
                            window=window)
        np.testing.assert_allclose(got, ref, atol=1e-12, rtol=0)
        m, l, o = oracle.decode_partitions(q, kc, vc, w.block_tables, w.seq_lens, 2, 16,
                                           w.scale, 3, window=window)
        merged = oracle.merge_partitions(m, l, o, w.seq_lens, window=window)
        np.testing.assert_allclose(merged, ref, atol=1e-12, rtol=0)
    qo, kv = np.array([6, 40, 3]), np.array([6, 50, 9])
    wp = W.make_prefill("mut", qo, kv, 4, 2, 64, seed=41)
    tp = wp.tensors("cpu")
    qq, k, v = (W.to_bits(tp[n]) for n in ("q", "k", "v"))
    for causal in (True, False):
        got = oracle.prefill(qq, k, v, wp.qo_indptr, wp.kv_indptr, 2, wp.scale, causal=causal,
                             window=5)
        ref = brute.brute_prefill_contiguous(qq, k, v, wp.qo_indptr, wp.kv_indptr, 2, wp.scale,
                                             causal, window=5)
        np.testing.assert_allclose(got, ref, atol=1e-12, rtol=0)


def _check_fp8():
    import torch
    table = np.array([float(torch.tensor([c], dtype=torch.uint8).view(torch.float8_e4m3fn)
                            .float()[0]) for c in range(256)])
    for c in range(256):
        got = oracle.e4m3_value(c)
        assert (np.isnan(got) and np.isnan(table[c])) or got == table[c], hex(c)
    mids = np.array([1.0625, 1.1875, 2.0 ** -10, 3 * 2.0 ** -10], np.float32)
    np.testing.assert_array_equal(oracle.e4m3_encode(mids), [0x38, 0x3A, 0x00, 0x02])
    # write then decode through non-unit scales, against numpy / torch on the side
    rng = np.random.default_rng(9)
    nb, nkv, bs, hd, T = 6, 2, 16, 64, 40
    kc = np.zeros((nb, nkv, bs, hd), np.uint8)
    vc = np.zeros_like(kc)
    k = W.float_to_bits(rng.standard_normal((T, nkv, hd)).astype(np.float32))
    v = W.float_to_bits(rng.standard_normal((T, nkv, hd)).astype(np.float32))
    slots = np.arange(T, dtype=np.int64) + 8
    oracle.write_cache(k, v, kc, vc, slots, bs, kv_fp8=True, k_scale=0.05, v_scale=0.02)
    kq = W.bits_to_float(k).astype(np.float32) / np.float32(0.05)
    ref = torch.from_numpy(np.clip(kq, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8)
    for t, s in enumerate(slots):
        np.testing.assert_array_equal(kc[s // bs, :, s % bs], ref.numpy()[t])
    w = W.make_decode("mut", [48], 4, 2, 64, seed=42, num_blocks=nb)
    bt = np.array([[0, 1, 2, 3]], np.int32)
    q = W.to_bits(w.tensors("cpu")["q"])
    got = oracle.decode(q, kc, vc, bt, np.array([48], np.int32), 2, 16, 0.125, kv_fp8=True,
                        k_scale=0.05, v_scale=0.02)
    ref = brute.brute_decode_values(q, table[kc] * 0.05, table[vc] * 0.02, bt,
                                    np.array([48], np.int32), 2, 16, 0.125,
                                    oracle.hnd_strides(2, 16, 64))
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


CHECKS = [_check_decode, _check_prefill, _check_split, _check_write, _check_large_logits,
          _check_blocks, _check_window, _check_fp8]


def _run_checks_in_child(lib_path):
    """Returns (exit code, stdout) of a child running every check against lib_path."""
    code = ("import sys; sys.path.insert(0, %r); import oracle; "
            "from tests import test_oracle_mutations as m; "
            "failed = []\n"
            "with oracle.using_library(%r):\n"
            "    for chk in m.CHECKS:\n"
            "        try:\n"
            "            chk()\n"
            "        except AssertionError:\n"
            "            failed.append(chk.__name__)\n"
            "print('FAILED', failed); sys.exit(1 if failed else 0)")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    res = subprocess.run([sys.executable, "-c", code % (root, lib_path)], capture_output=True,
                         text=True, timeout=300, cwd=root)
    return res.returncode, res.stdout + res.stderr


def _compile(src_path, lib_path):
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                           str(src_path), "-o", str(lib_path), "-lm"])


def test_unmutated_copy_passes_every_check(tmp_path):
    lib = tmp_path / "clean.so"
    _compile(SRC, lib)
    rc, out = _run_checks_in_child(str(lib))
    assert rc == 0, out


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(tmp_path, name):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    mutated = tmp_path / "mut.c"
    mutated.write_text(src.replace(old, new))
    lib = tmp_path / "mut.so"
    _compile(mutated, lib)
    rc, out = _run_checks_in_child(str(lib))
    assert rc != 0, f"planted mistake {name} passed every pin:\n{out}"
