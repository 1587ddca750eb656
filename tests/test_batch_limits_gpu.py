"""GPU parity at the batch-size limits of the decode kernels ("paged_attn.py",
forward_decode over a batch of sequences), through the C ABI.

The tensor-core decodes (head_dim 128, GQA 4 or 8) and the CUDA-core persistent split
kernel keep a per-sequence table of 2048 entries in shared memory: 2048 sequences is the
largest batch they take, and 2049 goes to the next path (the CUDA-core kernel, or its
one-CTA-per-partition grid).  Each case runs mostly short sequences (0-40 tokens) with a
few long ones, so that items of one, several and many partitions meet the limit, and
compares every output element with the fp64 oracle."""
import numpy as np
import pytest

from paged_kv_gqa_15_gb300 import workloads as W
from tests.gpu_util import assert_close_bf16
from tests.test_decode_gpu import _run_decode
from tests.test_fp8_gpu import _fp8_pools, _run as _run_fp8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    import paged_kv_gqa_15_gb300 as pa
    __graft_entry__.build()
    yield
    assert pa.device_status() == 0


def _lens(batch, seed):
    rng = np.random.default_rng(seed)
    lens = rng.integers(0, 40, size=batch, endpoint=True)
    lens[0], lens[batch // 2], lens[-1] = 1500, 700, 513   # one, two and three partitions
    return lens


@pytest.mark.parametrize("batch", [2048, 2049])
@pytest.mark.parametrize("split", [False, True])
def test_bf16_tensor_core_shape_at_the_batch_limit(batch, split):
    w = W.make_decode("limit", _lens(batch, 90 + batch), 8, 2, 128, seed=91 + batch)
    out, ref, _, _ = _run_decode(w, split)
    assert_close_bf16(out, ref, what=f"bf16 B={batch} split={split}")


@pytest.mark.parametrize("batch", [2048, 2049])
def test_bf16_cuda_core_split_at_the_batch_limit(batch):
    w = W.make_decode("limit64", _lens(batch, 92 + batch), 8, 4, 64, seed=93 + batch)
    out, ref, _, _ = _run_decode(w, split=True)
    assert_close_bf16(out, ref, what=f"hd64 B={batch}")


@pytest.mark.parametrize("batch", [2048, 2049])
@pytest.mark.parametrize("split", [False, True])
def test_fp8_tensor_core_shape_at_the_batch_limit(batch, split):
    w = W.make_decode("limit8", _lens(batch, 94 + batch), 8, 2, 128, seed=95 + batch)
    kc, vc = _fp8_pools(w, seed=96)
    out, ref, _, _ = _run_fp8(w, kc, vc, split)
    assert_close_bf16(out, ref, what=f"fp8 B={batch} split={split}")


@pytest.mark.parametrize("split", [False, True])
def test_windowed_decode_at_the_batch_limit(split):
    w = W.make_decode("limitw", _lens(2048, 97), 8, 2, 128, seed=98, window=600)
    out, ref, _, _ = _run_decode(w, split)
    assert_close_bf16(out, ref, what=f"window B=2048 split={split}")
