"""fp64 CPU oracle for paged-KV GQA attention -- TEST INFRASTRUCTURE ONLY.

Only the test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its binding) never imports it, and it never imports the product path.

``build()`` compiles ``pa_oracle.c`` with gcc into ``libpa_oracle.so`` beside
it; the wrappers below take numpy arrays (bf16 data as ``uint16`` bit
patterns) and return float64 results.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_LIB = os.path.join(_HERE, "libpa_oracle.so")
_lib = None

PARTITION = 512  # tokens per split-KV partition ("paged_attn.py", _PARTITION_SIZE)


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc, -O2, pthreads)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def load_library(path: str):
    """Load an oracle library from `path` (used by the planted-mistake tests)."""
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I, L, D = ctypes.c_int, ctypes.c_int64, ctypes.c_double
    F = ctypes.c_float
    lib.oracle_write_cache.argtypes = [P, P, P, P, P, L, I, I, I, L, L, L, L, I, F, F]
    lib.oracle_write_cache.restype = L
    lib.oracle_decode.argtypes = [P, P, P, P, L, L, L, P, P, I, I, I, I, I, I, D, P, L, I, I, I,
                                  D, D]
    lib.oracle_decode.restype = I
    lib.oracle_decode_partitions.argtypes = [P, P, P, P, P, P, L, L, L, P, P, I, I, I, I,
                                             I, I, D, I, I, I, I, I, D, D]
    lib.oracle_decode_partitions.restype = I
    lib.oracle_merge_partitions.argtypes = [P, P, P, P, P, I, I, I, I, I, I]
    lib.oracle_merge_partitions.restype = I
    lib.oracle_prefill.argtypes = [P, P, P, P, P, P, P, I, I, L, L, L, I, I, I, I, D, I,
                                   P, L, I, I]
    lib.oracle_prefill.restype = I
    lib.oracle_swap_blocks.argtypes = [P, P, P, L, L, L, L]
    lib.oracle_swap_blocks.restype = L
    lib.oracle_copy_blocks.argtypes = [P, I, P, L, L, L]
    lib.oracle_copy_blocks.restype = L
    lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_value.restype = D
    lib.oracle_e4m3_encode_array.argtypes = [P, P, L]
    lib.oracle_e4m3_encode_array.restype = None
    return lib


class using_library:
    """Context manager: route the wrappers below through another oracle build."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        self.saved = _lib
        _lib = load_library(self.path)
        return _lib

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved
        return False


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = load_library(_LIB)
    return _lib


def default_threads() -> int:
    return os.cpu_count() or 1


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def hnd_strides(num_kv_heads: int, block_size: int, head_dim: int):
    """Element strides (block, head, token) of a [blocks][nkv][bs][hd] pool."""
    return (num_kv_heads * block_size * head_dim, block_size * head_dim, head_dim)


def e4m3_value(code: int) -> float:
    """Value of one FP8 E4M3 code."""
    return _load().oracle_e4m3_value(int(code) & 0xFF)


def e4m3_encode(x):
    """E4M3 codes (uint8) of float32 values: nearest, ties to even, saturating."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint8)
    _load().oracle_e4m3_encode_array(_ptr(x), _ptr(out), x.size)
    return out


def write_cache(k, v, k_cache, v_cache, slot_mapping, block_size, strides=None, kv_fp8=False,
                k_scale=1.0, v_scale=1.0):
    """In-place scatter of k/v [T][nkv][hd] (uint16 bf16 bits) into the caches (uint16, or
    uint8 E4M3 codes of x / scale with kv_fp8); returns #bad slots."""
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    sm = _c(slot_mapping, np.int64)
    cache_t = np.uint8 if kv_fp8 else np.uint16
    assert k_cache.dtype == cache_t and k_cache.flags.c_contiguous
    assert v_cache.dtype == cache_t and v_cache.flags.c_contiguous
    T, nkv, hd = k.shape
    if strides is None:
        strides = hnd_strides(nkv, block_size, hd)
    nblocks = k_cache.size // strides[0]
    return _load().oracle_write_cache(_ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), _ptr(sm),
                                      T, nkv, hd, block_size, nblocks, *strides,
                                      1 if kv_fp8 else 0, float(k_scale), float(v_scale))


def _pool(a, kv_fp8):
    return _c(a, np.uint8 if kv_fp8 else np.uint16)


def decode(q, k_cache, v_cache, block_tables, seq_lens, num_kv_heads, block_size, scale,
           strides=None, items=None, nthreads=None, out=None, window=0, kv_fp8=False,
           k_scale=1.0, v_scale=1.0):
    """softmax(scale q K^T) V per (sequence, query head), fp64 [B][nq][hd]; window > 0
    keeps the last `window` keys of each sequence; kv_fp8 reads E4M3 pools (uint8)
    as code value * k_scale / v_scale."""
    q = _c(q, np.uint16)
    B, nq, hd = q.shape
    bt = _c(block_tables, np.int32)
    sl = _c(seq_lens, np.int32)
    if strides is None:
        strides = hnd_strides(num_kv_heads, block_size, hd)
    if out is None:
        out = np.zeros((B, nq, hd), np.float64)
    it = None if items is None else _c(items, np.int32)
    rc = _load().oracle_decode(_ptr(out), _ptr(q), _ptr(_pool(k_cache, kv_fp8)),
                               _ptr(_pool(v_cache, kv_fp8)), *strides, _ptr(bt), _ptr(sl),
                               B, nq, num_kv_heads, hd, block_size, bt.shape[1], scale,
                               _ptr(it), 0 if it is None else it.size,
                               nthreads or default_threads(), int(window), 1 if kv_fp8 else 0,
                               float(k_scale), float(v_scale))
    assert rc == 0
    return out


def decode_partitions(q, k_cache, v_cache, block_tables, seq_lens, num_kv_heads, block_size,
                      scale, max_parts, strides=None, part=PARTITION, nthreads=None, window=0,
                      kv_fp8=False, k_scale=1.0, v_scale=1.0):
    """Per-partition (m, l, o) of the split-KV pass; untouched entries are NaN."""
    q = _c(q, np.uint16)
    B, nq, hd = q.shape
    bt = _c(block_tables, np.int32)
    sl = _c(seq_lens, np.int32)
    if strides is None:
        strides = hnd_strides(num_kv_heads, block_size, hd)
    m = np.full((B, nq, max_parts), np.nan)
    l = np.full((B, nq, max_parts), np.nan)
    o = np.full((B, nq, max_parts, hd), np.nan)
    rc = _load().oracle_decode_partitions(_ptr(m), _ptr(l), _ptr(o), _ptr(q),
                                          _ptr(_pool(k_cache, kv_fp8)),
                                          _ptr(_pool(v_cache, kv_fp8)), *strides, _ptr(bt),
                                          _ptr(sl), B, nq, num_kv_heads, hd, block_size,
                                          bt.shape[1], scale, part, max_parts,
                                          nthreads or default_threads(), int(window),
                                          1 if kv_fp8 else 0, float(k_scale), float(v_scale))
    assert rc == 0
    return m, l, o


def merge_partitions(m, l, o, seq_lens, part=PARTITION, window=0):
    """Log-sum-exp merge of partition results, fp64 [B][nq][hd]."""
    m = _c(m, np.float64)
    l = _c(l, np.float64)
    o = _c(o, np.float64)
    B, nq, P, hd = o.shape
    out = np.zeros((B, nq, hd), np.float64)
    rc = _load().oracle_merge_partitions(_ptr(out), _ptr(m), _ptr(l), _ptr(o),
                                         _ptr(_c(seq_lens, np.int32)), B, nq, hd, part, P,
                                         int(window))
    assert rc == 0
    return out


def prefill(q, k, v, qo_indptr, kv_indptr, num_kv_heads, scale, causal=True,
            block_tables=None, block_size=16, strides=None, rows=None, nthreads=None,
            out=None, window=0):
    """Ragged prefill, fp64 [total_qo][nq][hd]; contiguous (block_tables None) or paged."""
    q = _c(q, np.uint16)
    total_qo, nq, hd = q.shape
    qi = _c(qo_indptr, np.int32)
    ki = _c(kv_indptr, np.int32)
    batch = qi.size - 1
    bt = None if block_tables is None else _c(block_tables, np.int32)
    if bt is not None and strides is None:
        strides = hnd_strides(num_kv_heads, block_size, hd)
    if strides is None:
        strides = (0, 0, 0)
    if out is None:
        out = np.zeros((total_qo, nq, hd), np.float64)
    rw = None if rows is None else _c(rows, np.int64)
    rc = _load().oracle_prefill(_ptr(out), _ptr(q), _ptr(_c(k, np.uint16)),
                                _ptr(_c(v, np.uint16)), _ptr(qi), _ptr(ki), _ptr(bt),
                                0 if bt is None else bt.shape[1], block_size, *strides,
                                batch, nq, num_kv_heads, hd, scale, 1 if causal else 0,
                                _ptr(rw), 0 if rw is None else rw.size,
                                nthreads or default_threads(), int(window))
    assert rc == 0
    return out


def _pages(pool):
    """(num_blocks, block_bytes) of a C-contiguous numpy pool [num_blocks, ...]."""
    assert pool.flags.c_contiguous
    return pool.shape[0], pool.nbytes // max(1, pool.shape[0])


def swap_blocks(src, dst, block_mapping):
    """In-place page copies src -> dst (numpy pools) for the int64 [n, 2] pairs;
    returns the number of out-of-range pairs."""
    bm = _c(block_mapping, np.int64).reshape(-1, 2)
    snb, sbb = _pages(src)
    dnb, dbb = _pages(dst)
    assert sbb == dbb
    return _load().oracle_swap_blocks(_ptr(src), _ptr(dst), _ptr(bm), bm.shape[0], snb, dnb, sbb)


def copy_blocks(pools, block_mapping):
    """In-place page copies inside each numpy pool of the list; returns the number of
    out-of-range pairs summed over the pools."""
    bm = _c(block_mapping, np.int64).reshape(-1, 2)
    nb, bb = _pages(pools[0])
    for p in pools:
        assert _pages(p) == (nb, bb)
    arr = (ctypes.c_void_p * len(pools))(*[p.ctypes.data for p in pools])
    return _load().oracle_copy_blocks(arr, len(pools), _ptr(bm), bm.shape[0], nb, bb)
