"""Pins of the oracle's fp8 KV cache (kv_cache_dtype "fp8" with k_scale / v_scale,
"paged_attn.py" write_to_paged_cache and forward_decode; the format is OCP FP8 E4M3):
hand-derived code values and rounding cases (tests/golden/e4m3_codes.txt), torch's
independent float8_e4m3fn conversion, round trips, and attention over a quantised
cache against brute force on the dequantised values."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_gqa_15_gb300 import workloads as W
from tests import brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_codes.txt")


def _golden():
    values, rounding = [], []
    section = values
    for line in open(GOLDEN):
        if line.startswith("# x "):
            section = rounding
        if not line.strip() or line.startswith("#") and section is values:
            continue
        parts = line.lstrip("#").split()
        if section is values:
            values.append((int(parts[0], 16), float(parts[1])))
        elif len(parts) >= 2 and parts[1].startswith("0x"):
            rounding.append((float(parts[0]), int(parts[1], 16)))
    return values, rounding


def _torch_value(code):
    return float(torch.tensor([code], dtype=torch.uint8).view(torch.float8_e4m3fn).float()[0])


def test_golden_code_values(oracle_lib):
    values, _ = _golden()
    assert len(values) == 16
    for code, v in values:
        got = oracle.e4m3_value(code)
        if math.isnan(v):
            assert math.isnan(got), hex(code)
        else:
            assert got == v and math.copysign(1, got) == math.copysign(1, v), hex(code)


def test_golden_rounding_cases(oracle_lib):
    _, rounding = _golden()
    assert len(rounding) == 9
    xs = np.array([x for x, _ in rounding], np.float32)
    np.testing.assert_array_equal(oracle.e4m3_encode(xs), [c for _, c in rounding])


def test_every_code_value_matches_torch(oracle_lib):
    for code in range(256):
        got, ref = oracle.e4m3_value(code), _torch_value(code)
        if math.isnan(ref):
            assert math.isnan(got), hex(code)
        else:
            assert got == ref, hex(code)


def test_rounding_matches_torch_below_saturation(oracle_lib):
    rng = np.random.default_rng(3)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * 3,
        rng.uniform(-463.9, 463.9, 5000).astype(np.float32),
        (rng.standard_normal(5000) * 2.0 ** -8).astype(np.float32),   # subnormal range
        # every midpoint between neighbouring codes, and just either side of it
        *[np.array([(a + b) / 2 * f for a, b in zip(v[:-1], v[1:]) for f in (1 - 1e-6, 1, 1 + 1e-6)],
                   np.float32) for v in [[oracle.e4m3_value(c) for c in range(0x7F)]]],
    ])
    x = x[np.abs(x) < 464]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(oracle.e4m3_encode(x), ref)


def test_finite_codes_round_trip(oracle_lib):
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = np.array([oracle.e4m3_value(c) for c in codes], np.float32)
    np.testing.assert_array_equal(oracle.e4m3_encode(vals), codes)


def test_encode_is_monotone(oracle_lib):
    x = np.linspace(-600, 600, 200001).astype(np.float32)
    vals = np.array([oracle.e4m3_value(c) for c in oracle.e4m3_encode(x)])
    assert np.all(np.diff(vals) >= 0)
    assert vals.max() == 448 and vals.min() == -448


def test_fp8_write_stores_codes_of_the_fp32_quotient(oracle_lib):
    rng = np.random.default_rng(4)
    nb, nkv, bs, hd, T = 10, 2, 16, 64, 30
    kc = np.full((nb, nkv, bs, hd), 0x55, np.uint8)
    vc = np.full_like(kc, 0x55)
    k = W.float_to_bits(rng.standard_normal((T, nkv, hd)).astype(np.float32) * 40)
    v = W.float_to_bits(rng.standard_normal((T, nkv, hd)).astype(np.float32) * 40)
    slots = rng.choice(nb * bs, size=T, replace=False).astype(np.int64)
    slots[::7] = -1
    ks, vs = np.float32(0.0371), np.float32(0.213)
    assert oracle.write_cache(k, v, kc, vc, slots, bs, kv_fp8=True, k_scale=ks, v_scale=vs) == 0
    kf = W.bits_to_float(k).astype(np.float32) / ks        # numpy's own fp32 division
    vf = W.bits_to_float(v).astype(np.float32) / vs
    ref_k = torch.from_numpy(np.clip(kf, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ref_v = torch.from_numpy(np.clip(vf, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    written = np.zeros((nb, bs), bool)
    for t, s in enumerate(slots):
        if s < 0:
            continue
        np.testing.assert_array_equal(kc[s // bs, :, s % bs], ref_k[t])
        np.testing.assert_array_equal(vc[s // bs, :, s % bs], ref_v[t])
        written[s // bs, s % bs] = True
    assert (kc.transpose(0, 2, 1, 3)[~written] == 0x55).all()
    assert (vc.transpose(0, 2, 1, 3)[~written] == 0x55).all()


def _fp8_decode_inputs(seed, lens, nq=8, nkv=2, hd=64):
    w = W.make_decode("fp8", lens, nq, nkv, hd, seed=seed)
    rng = np.random.default_rng(seed)
    q = W.to_bits(w.tensors("cpu")["q"])
    kc = rng.integers(0, 256, size=w.pool_shape, dtype=np.uint8)
    vc = rng.integers(0, 256, size=w.pool_shape, dtype=np.uint8)
    for c in (kc, vc):                                   # no NaN codes in the cache
        c[(c & 0x7F) == 0x7F] = 0x7E
    return w, q, kc, vc


def _dequant(codes, scale):
    table = np.array([_torch_value(c) for c in range(256)])
    return table[codes] * scale


def test_fp8_decode_matches_brute_force_on_dequantised_pools(oracle_lib):
    w, q, kc, vc = _fp8_decode_inputs(5, [1, 17, 300, 513, 1100])
    ks, vs = 0.05, 0.3
    got = oracle.decode(q, kc, vc, w.block_tables, w.seq_lens, 2, 16, w.scale, kv_fp8=True,
                        k_scale=ks, v_scale=vs)
    ref = brute.brute_decode_values(q, _dequant(kc, ks), _dequant(vc, vs), w.block_tables,
                                    w.seq_lens, 2, 16, w.scale, oracle.hnd_strides(2, 16, 64))
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_fp8_scales_act_as_exact_factors(oracle_lib):
    w, q, kc, vc = _fp8_decode_inputs(6, [40, 600])
    base = oracle.decode(q, kc, vc, w.block_tables, w.seq_lens, 2, 16, w.scale, kv_fp8=True,
                         k_scale=0.05, v_scale=0.25)
    # v_scale multiplies the output (a power of two: exactly)
    twice = oracle.decode(q, kc, vc, w.block_tables, w.seq_lens, 2, 16, w.scale, kv_fp8=True,
                          k_scale=0.05, v_scale=0.5)
    np.testing.assert_array_equal(twice, 2 * base)
    # k_scale multiplies every score, as sm_scale does
    folded = oracle.decode(q, kc, vc, w.block_tables, w.seq_lens, 2, 16, w.scale * 0.05,
                           kv_fp8=True, k_scale=1.0, v_scale=0.25)
    np.testing.assert_allclose(folded, base, rtol=1e-12, atol=1e-12)


def test_fp8_split_merge_equals_single_pass(oracle_lib):
    w, q, kc, vc = _fp8_decode_inputs(7, [1, 511, 512, 513, 2049])
    kw = dict(kv_fp8=True, k_scale=0.07, v_scale=0.4)
    single = oracle.decode(q, kc, vc, w.block_tables, w.seq_lens, 2, 16, w.scale, **kw)
    m, l, o = oracle.decode_partitions(q, kc, vc, w.block_tables, w.seq_lens, 2, 16, w.scale, 5,
                                       **kw)
    # values reach a few hundred (codes up to 448 times the scale): relative rounding bound
    np.testing.assert_allclose(oracle.merge_partitions(m, l, o, w.seq_lens), single,
                               rtol=1e-12, atol=1e-12)


def test_bf16_cache_of_the_dequantised_values_gives_the_same_decode(oracle_lib):
    # with unit scales and codes whose values are bf16-representable (all of them are),
    # an fp8 cache and a bf16 cache holding the decoded values attend identically
    w, q, kc, vc = _fp8_decode_inputs(8, [33, 700])
    kb = W.float_to_bits(_dequant(kc, 1.0).astype(np.float32))
    vb = W.float_to_bits(_dequant(vc, 1.0).astype(np.float32))
    a = oracle.decode(q, kc, vc, w.block_tables, w.seq_lens, 2, 16, w.scale, kv_fp8=True)
    b = oracle.decode(q, kb, vb, w.block_tables, w.seq_lens, 2, 16, w.scale)
    np.testing.assert_array_equal(a, b)
