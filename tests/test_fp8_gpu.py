"""GPU parity of the FP8 E4M3 KV cache (kv_cache_dtype "fp8" with k_scale / v_scale,
"paged_attn.py" write_to_paged_cache and forward_decode) through the C ABI: the cache
write is compared code for code with the oracle, and the decode (single pass and
split) with the fp64 oracle reading the same codes."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_15_gb300 as pa
from paged_kv_gqa_15_gb300 import workloads as W
from tests.gpu_util import assert_close_bf16

pytestmark = pytest.mark.gpu
DEV = "cuda"
KS, VS = 1.0 / 64, 1.0 / 48        # codes then hold about 64 / 48 x N(0, 1)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    yield
    assert pa.device_status() == 0


def _codes(values, scale):
    """E4M3 codes of values / scale (torch's conversion; inputs stay below 448)."""
    v = np.clip(np.asarray(values, np.float32), -6.0, 6.0)
    return (torch.from_numpy(v) / scale).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _fp8_pools(w, seed, stale_nan=True):
    rng = np.random.default_rng(seed)
    kc = _codes(rng.standard_normal(w.pool_shape), KS)
    vc = _codes(rng.standard_normal(w.pool_shape), VS)
    if stale_nan:   # rows past each sequence's end in its last page hold NaN codes
        for b, L in enumerate(w.seq_lens):
            L = int(L)
            if L % 16:
                page = w.block_tables[b, L // 16]
                kc[page, :, L % 16:, :] = 0x7F
                vc[page, :, L % 16:, :] = 0xFF
    return kc, vc


def _dev_u8(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


# ---- cache write -------------------------------------------------------------------------


@pytest.mark.parametrize("hd", [64, 128, 256])
@pytest.mark.parametrize("layout", ["HND", "NHD"])
def test_fp8_write_cache_matches_oracle_codes(hd, layout):
    rng = np.random.default_rng(hd)
    nb, nkv, bs, T = 40, 4, 16, 300
    kx = rng.standard_normal((T, nkv, hd)).astype(np.float32)
    vx = rng.standard_normal((T, nkv, hd)).astype(np.float32)
    # magnitudes past saturation, in the subnormal range, signed zeros and infinities
    kx[0, 0, :8] = [1e5, -1e5, 3e-4, -3e-4, 0.0, -0.0, np.inf, -np.inf]
    kx[1] *= 50.0
    vx[2] *= 1e-3
    k = W.float_to_bits(kx)
    v = W.float_to_bits(vx)
    slots = rng.choice(nb * bs, size=T, replace=False).astype(np.int64)
    slots[5::9] = -1                           # padding tokens (rows 0..2 keep their slots)
    kc = np.full((nb, nkv, bs, hd), 0x55, np.uint8)
    vc = np.full_like(kc, 0x55)
    kc_d, vc_d = _dev_u8(kc), _dev_u8(vc)
    if layout == "NHD":
        kc_d = kc_d.permute(0, 2, 1, 3).contiguous()
        vc_d = vc_d.permute(0, 2, 1, 3).contiguous()
    kb = torch.from_numpy(k.view(np.int16)).to(DEV).view(torch.bfloat16)
    vb = torch.from_numpy(v.view(np.int16)).to(DEV).view(torch.bfloat16)
    pa.pa_write_cache(kb, vb, kc_d, vc_d, torch.from_numpy(slots).to(DEV), layout=layout,
                      k_scale=0.0371, v_scale=0.213)
    got_k, got_v = kc_d.cpu().numpy(), vc_d.cpu().numpy()
    if layout == "NHD":
        got_k, got_v = got_k.transpose(0, 2, 1, 3), got_v.transpose(0, 2, 1, 3)
    oracle.write_cache(k, v, kc, vc, slots, bs, kv_fp8=True, k_scale=0.0371, v_scale=0.213)
    assert np.array_equal(got_k, kc), np.argwhere(got_k != kc)[:5]
    assert np.array_equal(got_v, vc)
    assert pa.device_status() == 0


def test_fp8_write_of_nan_gives_a_nan_code():
    kx = np.zeros((1, 1, 64), np.float32)
    kx[0, 0, 3] = np.nan
    kb = torch.from_numpy(W.float_to_bits(kx).view(np.int16)).to(DEV).view(torch.bfloat16)
    kc = torch.zeros((2, 1, 16, 64), dtype=torch.uint8, device=DEV)
    vc = torch.zeros_like(kc)
    pa.pa_write_cache(kb, kb, kc, vc, torch.tensor([5], dtype=torch.int64, device=DEV),
                      k_scale=1.0, v_scale=1.0)
    row = kc[0, 0, 5].cpu().numpy()
    assert row[3] & 0x7F == 0x7F          # a NaN code (either sign)
    assert (np.delete(row, 3) == 0).all()


# ---- decode ------------------------------------------------------------------------------

LENS = [0, 1, 15, 16, 17, 100, 511, 512, 513, 1100, 2049]
SHAPES = [(128, 32, 8), (128, 64, 8), (64, 8, 8), (256, 16, 8), (128, 8, 4)]


def _run(w, kc, vc, split, window=0):
    q = W.to_bits(w.tensors("cpu")["q"])
    q_d = torch.from_numpy(q.view(np.int16)).to(DEV).view(torch.bfloat16)
    kc_d = _dev_u8(kc).view(torch.float8_e4m3fn)
    vc_d = _dev_u8(vc).view(torch.float8_e4m3fn)
    bt = torch.from_numpy(w.block_tables).to(DEV)
    sl = torch.from_numpy(w.seq_lens).to(DEV)
    out = torch.full_like(q_d, float("nan"))
    ws = None
    if split:
        L = max(w.max_seq_len, 1)
        ws = pa.alloc_workspace(pa.decode_split_workspace_size(w.batch, w.num_q_heads,
                                                               w.head_dim, L), DEV)
        pa.pa_decode_split(out, q_d, kc_d, vc_d, bt, sl, w.scale, L, ws, sliding_window=window,
                           k_scale=KS, v_scale=VS)
    else:
        pa.pa_decode(out, q_d, kc_d, vc_d, bt, sl, w.scale, sliding_window=window, k_scale=KS,
                     v_scale=VS)
    torch.cuda.synchronize()
    ref = oracle.decode(q, kc, vc, w.block_tables, w.seq_lens, w.num_kv_heads, 16, w.scale,
                        window=window, kv_fp8=True, k_scale=KS, v_scale=VS)
    return out, ref, ws, q


@pytest.mark.parametrize("hd,nq,nkv", SHAPES)
@pytest.mark.parametrize("split", [False, True])
def test_fp8_decode_matches_oracle(hd, nq, nkv, split):
    w = W.make_decode("fp8", LENS, nq, nkv, hd, seed=80 + hd + nq)
    kc, vc = _fp8_pools(w, seed=81)
    out, ref, _, _ = _run(w, kc, vc, split)
    assert pa.device_status() == 0
    assert_close_bf16(out, ref, what=f"fp8 decode hd {hd} g {nq // nkv} split {split}")


@pytest.mark.parametrize("split", [False, True])
def test_fp8_decode_with_a_sliding_window(split):
    w = W.make_decode("fp8w", LENS, 32, 8, 128, seed=82)
    kc, vc = _fp8_pools(w, seed=83)
    out, ref, _, _ = _run(w, kc, vc, split, window=300)
    assert_close_bf16(out, ref, what="fp8 + window")


def test_fp8_partials_match_oracle_partitions():
    w = W.make_decode("fp8p", [1, 512, 513, 1700, 3000], 32, 8, 128, seed=84)
    kc, vc = _fp8_pools(w, seed=85)
    out, ref, ws, q = _run(w, kc, vc, split=True)
    L = w.max_seq_len
    P = (L + 511) // 512
    po, pm, pl = pa.decode_split_workspace_views(ws, w.batch, 32, 128, L)
    m, l, o = oracle.decode_partitions(q, kc, vc, w.block_tables, w.seq_lens, 8, 16, w.scale, P,
                                       kv_fp8=True, k_scale=KS, v_scale=VS)
    # The tensor-core fp8 path multiplies K by q carried as two E4M3 codes per element
    # (hi = e4m3(q s), lo = e4m3(q s - hi), s a power of two with max|q s| in [128, 256)),
    # which is q to within |dq| <= 2^-8 |q| + 2^-17 max|q|.  A score then moves by at most
    # db_j = sm_scale * sum_d |dq_d| |k_jd|; m by the largest db_j of the partition, l by a
    # factor within exp(+-2 db), and o (a weighted mean of V) by 2 db max|V|.  P reaches
    # the P.V as two E4M3 codes too (R17: hi = e4m3(256 p), lo = e4m3(256 p - hi)), so
    # |dp| <= 2^-8 p + 2^-18; with l >= 1 (the partition's largest weight is 1) and at
    # most 512 weights, o moves by at most (2^-8 + 2^-9) max|V| more.
    qf = W.bits_to_float(q).astype(np.float64)
    table = np.array([float(torch.tensor([c], dtype=torch.uint8).view(torch.float8_e4m3fn)
                            .float()) if c & 0x7F != 0x7F else 0.0 for c in range(256)])
    kf = table[kc] * KS                        # NaN codes sit only in unread stale rows
    vmax = float(np.abs(table[vc] * VS).max())
    for b, Lb in enumerate(w.seq_lens):
        n = (int(Lb) + 511) // 512
        gm, gl, go = (x[b, :, :n].cpu().numpy().astype(np.float64) for x in (pm, pl, po))
        for h in range(32):
            kh = h // 4
            dq = 2.0 ** -8 * np.abs(qf[b, h]) + 2.0 ** -17 * np.abs(qf[b, h]).max()
            for pidx in range(n):
                j0, j1 = pidx * 512, min(Lb, pidx * 512 + 512)
                rows = np.array([kf[w.block_tables[b, j // 16], kh, j % 16] for j in range(j0, j1)])
                db = w.scale * (np.abs(rows) @ dq).max()
                assert abs(gm[h, pidx] - m[b, h, pidx]) <= db + 1e-4, (b, h, pidx)
                assert abs(gl[h, pidx] / l[b, h, pidx] - 1) <= np.expm1(2 * db) + 1e-4, (b, h, pidx)
                np.testing.assert_allclose(go[h, pidx], o[b, h, pidx],
                                           atol=(2 * db + 2.0 ** -8 + 2.0 ** -9) * vmax + 1e-5,
                                           rtol=0)
    assert_close_bf16(out, ref, what="fp8 split")


def test_fp8_write_then_decode_step():
    # the Llama-3-8B decode step on a small batch: quantise the new token into the fp8
    # cache, then decode through it
    lens = np.array([700, 33, 1500, 16], np.int32)
    w = W.make_decode("fp8s", lens, 32, 8, 128, seed=86, new_token_write=True, split=True)
    kc, vc = _fp8_pools(w, seed=87, stale_nan=False)
    t = w.tensors("cpu")
    kn, vn = W.to_bits(t["k_new"]), W.to_bits(t["v_new"])
    kc_d = _dev_u8(kc).view(torch.float8_e4m3fn)
    vc_d = _dev_u8(vc).view(torch.float8_e4m3fn)
    pa.pa_write_cache(t["k_new"].to(DEV), t["v_new"].to(DEV), kc_d, vc_d,
                      torch.from_numpy(w.slot_mapping).to(DEV), k_scale=KS, v_scale=VS)
    oracle.write_cache(kn, vn, kc, vc, w.slot_mapping, 16, kv_fp8=True, k_scale=KS, v_scale=VS)
    assert np.array_equal(kc_d.view(torch.uint8).cpu().numpy(), kc)
    assert np.array_equal(vc_d.view(torch.uint8).cpu().numpy(), vc)
    out, ref, _, _ = _run(w, kc, vc, split=True)
    assert_close_bf16(out, ref, what="fp8 write + decode")
