"""Helpers shared by the GPU parity tests (comparison and host copies only)."""
import numpy as np

from paged_kv_gqa_15_gb300 import workloads as W

# bf16 outputs on N(0, 1) inputs: max-abs 2e-2 and mean-abs 2e-3 against the fp64 oracle
MAX_ABS = 2e-2
MEAN_ABS = 2e-3


def bf16_out(t):
    return W.bits_to_float(W.to_bits(t)).astype(np.float64)


def assert_close_bf16(got_tensor_or_array, ref, max_abs=MAX_ABS, mean_abs=MEAN_ABS, what=""):
    got = got_tensor_or_array
    if not isinstance(got, np.ndarray):
        got = bf16_out(got)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    assert err.max() <= max_abs, f"{what}: max abs err {err.max():.4g} > {max_abs}"
    assert err.mean() <= mean_abs, f"{what}: mean abs err {err.mean():.4g} > {mean_abs}"
    return float(err.max()), float(err.mean())


def stale_fill_last_pages(kc_bits, vc_bits, block_tables, seq_lens, block_size, value=1.0e4):
    """Write large finite values into the rows of each sequence's last page that lie
    past its length, so a kernel that reads them without masking fails loudly."""
    big = W.float_to_bits(np.float32(value))
    neg = W.float_to_bits(np.float32(-value))
    for b, L in enumerate(seq_lens):
        L = int(L)
        if L % block_size == 0 or L == 0:
            continue
        page = block_tables[b, L // block_size]
        for row in range(L % block_size, block_size):
            kc_bits[page, :, row, :] = big if row % 2 else neg
            vc_bits[page, :, row, :] = neg if row % 2 else big
