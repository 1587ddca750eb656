"""Paged-KV GQA attention for GB300 (sm_103a).

A thin ctypes binding over the C ABI in include/pa.h (libpa.so, built in-tree
by ``paged_kv_gqa_15_gb300.build``).  Functions take torch CUDA tensors and
only marshal pointers, shapes and strides: every step of the computation runs
in the library's CUDA kernels.  There is no CPU fallback -- if libpa.so is
missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpa.so")
PARTITION_TOKENS = 512
_lib = None

PA_OK, PA_ERR_INVALID, PA_ERR_UNSUPPORTED, PA_ERR_CUDA, PA_ERR_WORKSPACE, PA_ERR_TIMEOUT, \
    PA_ERR_DEVICE_BOUNDS = range(7)
PA_KV_BF16, PA_KV_FP8_E4M3 = 0, 1   # pa_kv_dtype
STATUS_NAMES = {1: "INVALID", 2: "UNSUPPORTED", 3: "CUDA", 4: "WORKSPACE", 5: "TIMEOUT",
                6: "DEVICE_BOUNDS"}


class PaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"pa error {code} ({STATUS_NAMES.get(code, '?')}): {msg}")
        self.code = code


def load():
    """Load libpa.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"CUDA library {LIB_PATH} is missing: build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, L, F, Z = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                     ctypes.c_size_t)
    lib.pa_write_cache.argtypes = [P, P, P, P, P, L, I, I, I, L, L, L, L, I, F, F, P]
    lib.pa_decode.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, L, L, L, L, F, I, I, F, F, P]
    lib.pa_decode_split_workspace_size.argtypes = [I, I, I, I]
    lib.pa_decode_split_workspace_size.restype = Z
    lib.pa_decode_split_workspace_offsets.argtypes = [I, I, I, I, P, P, P]
    lib.pa_decode_split_workspace_offsets.restype = None
    lib.pa_decode_split.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, L, L, L, L, F, I, I, F,
                                    F, I, P, Z, P]
    lib.pa_decode_partitions.argtypes = [P, P, P, P, P, I, I, I, I, I, I, L, L, L, L, F, I, I, F,
                                         F, I, P, Z, P]
    lib.pa_decode_merge.argtypes = [P, P, I, I, I, I, I, P, Z, P]
    lib.pa_decode_split_static.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, L, L, L, L, F, I,
                                           I, F, F, I, P]
    lib.pa_decode_split_static.restype = I
    lib.pa_ragged_prefill_workspace_size.argtypes = [I, I, I, I]
    lib.pa_ragged_prefill_workspace_size.restype = Z
    lib.pa_ragged_prefill.argtypes = [P, P, P, P, P, P, P, P, P, I, I, L, L, L, L, I, I, I, I, I,
                                      I, F, I, I, P, Z, P]
    lib.pa_get_device_status.argtypes = [P, P]
    lib.pa_selftest_wait_timeout.argtypes = [P]
    lib.pa_block_table_sync.argtypes = [P, P, P, I, I, P, P]
    lib.pa_block_table_sync.restype = I
    lib.pa_copy_blocks.argtypes = [P, I, P, L, L, L, P]
    lib.pa_copy_blocks.restype = I
    lib.pa_swap_blocks.argtypes = [P, P, I, P, L, L, L, L, P]
    lib.pa_swap_blocks.restype = I
    lib.pa_last_error.restype = ctypes.c_char_p
    for name in ("pa_write_cache", "pa_decode", "pa_decode_split", "pa_decode_partitions",
                 "pa_decode_merge", "pa_ragged_prefill",
                 "pa_get_device_status"):
        getattr(lib, name).restype = I
    _lib = lib
    return lib


def _check(rc: int):
    if rc != PA_OK:
        raise PaError(rc, load().pa_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def pool_strides(cache: torch.Tensor, layout: str = "HND"):
    """(block, head, token) element strides of a 4-D pool tensor.

    HND: [num_blocks][num_kv_heads][block_size][head_dim];
    NHD: [num_blocks][block_size][num_kv_heads][head_dim]."""
    s = cache.stride()
    assert cache.dim() == 4 and s[3] == 1, "pool must be 4-D with a contiguous head_dim"
    return (s[0], s[1], s[2]) if layout == "HND" else (s[0], s[2], s[1])


def kv_dtype_of(cache: torch.Tensor) -> int:
    """pa_kv_dtype of a pool tensor: bf16, or FP8 E4M3 codes (float8_e4m3fn or uint8)."""
    if cache.dtype == torch.bfloat16:
        return PA_KV_BF16
    if cache.dtype in (torch.uint8, getattr(torch, "float8_e4m3fn", torch.uint8)):
        return PA_KV_FP8_E4M3
    raise TypeError(f"unsupported KV cache dtype {cache.dtype}")


def _pool_geometry(cache, layout):
    nb = cache.shape[0]
    if layout == "HND":
        nkv, bs, hd = cache.shape[1], cache.shape[2], cache.shape[3]
    else:
        bs, nkv, hd = cache.shape[1], cache.shape[2], cache.shape[3]
    return nb, nkv, bs, hd


def _host_ptr(a):
    """Address of a C-contiguous host array (numpy or CPU torch tensor)."""
    if isinstance(a, torch.Tensor):
        assert a.device.type == "cpu" and a.is_contiguous()
        return ctypes.c_void_p(a.data_ptr())
    assert a.flags["C_CONTIGUOUS"]
    return ctypes.c_void_p(a.ctypes.data)


def pa_block_table_sync(host_table, snapshot, device_table, stream=None) -> int:
    """Uploads the rows of host_table (int32 [rows, cols], host) that differ from
    snapshot (a pinned int32 host tensor holding what was last uploaded) into
    device_table, refreshing the snapshot; returns the number of rows copied."""
    rows, cols = host_table.shape
    assert tuple(snapshot.shape) == (rows, cols) and tuple(device_table.shape) == (rows, cols)
    n = ctypes.c_int(0)
    _check(load().pa_block_table_sync(_host_ptr(host_table), _host_ptr(snapshot),
                                      _ptr(device_table), rows, cols, ctypes.byref(n),
                                      _stream(stream) if torch.cuda.is_available() else None))
    return n.value


def _page_geometry(pools):
    """(num_blocks, block_bytes) shared by a list of pools, each [num_blocks, ...] with
    densely packed pages (page b = bytes [b * block_bytes, (b + 1) * block_bytes))."""
    nb, bb = None, None
    for t in pools:
        page_elems = t[0].numel() if t.shape[0] > 0 else 0
        assert t.stride(0) == page_elems and t[0].is_contiguous(), \
            "pool pages must be densely packed"
        b = page_elems * t.element_size()
        assert (nb, bb) in ((None, None), (t.shape[0], b)), "pools differ in geometry"
        nb, bb = t.shape[0], b
    return nb, bb


def _pointer_array(tensors):
    arr = (ctypes.c_void_p * max(1, len(tensors)))()
    for i, t in enumerate(tensors):
        arr[i] = t.data_ptr()
    return arr


def pa_copy_blocks(key_caches, value_caches, block_mapping, stream=None):
    """copy_blocks: for every (src, dst) row of block_mapping (int64 [n, 2], on the
    device), page src of every layer's key and value pool is copied to page dst."""
    pools = [t for kv in zip(key_caches, value_caches) for t in kv]
    if not pools or block_mapping.numel() == 0:
        return
    assert block_mapping.dtype == torch.int64 and block_mapping.is_contiguous()
    nb, bb = _page_geometry(pools)
    _check(load().pa_copy_blocks(_pointer_array(pools), len(pools), _ptr(block_mapping),
                                 block_mapping.shape[0], nb, bb, _stream(stream)))


def pa_swap_blocks(src, dst, block_mapping, stream=None):
    """swap_blocks: page src of each source pool to page dst of the matching
    destination pool, for every row of block_mapping (int64 [n, 2]).  src / dst are a
    pool or a list of pools, each on the device or in pinned host memory; the mapping
    may be on either side too."""
    src = list(src) if isinstance(src, (list, tuple)) else [src]
    dst = list(dst) if isinstance(dst, (list, tuple)) else [dst]
    assert len(src) == len(dst)
    if not src or block_mapping.numel() == 0:
        return
    assert block_mapping.dtype == torch.int64 and block_mapping.is_contiguous()
    snb, sbb = _page_geometry(src)
    dnb, dbb = _page_geometry(dst)
    assert sbb == dbb, "source and destination pages differ in size"
    _check(load().pa_swap_blocks(_pointer_array(src), _pointer_array(dst), len(src),
                                 _ptr(block_mapping), block_mapping.shape[0], snb, dnb, sbb,
                                 _stream(stream)))


def pa_write_cache(k, v, k_cache, v_cache, slot_mapping, layout="HND", stream=None,
                   k_scale=1.0, v_scale=1.0):
    """reshape_and_cache: scatter k/v [T, nkv, hd] into the pools at slot_mapping [T];
    an FP8 pool (float8_e4m3fn or uint8) stores the E4M3 codes of x / k_scale (v_scale)."""
    nb, nkv, bs, hd = _pool_geometry(k_cache, layout)
    sb, sh, st = pool_strides(k_cache, layout)
    _check(load().pa_write_cache(_ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache),
                                 _ptr(slot_mapping), k.shape[0], nkv, hd, bs, nb, sb, sh, st,
                                 kv_dtype_of(k_cache), float(k_scale), float(v_scale),
                                 _stream(stream)))


def pa_decode(out, q, k_cache, v_cache, block_tables, seq_lens, sm_scale, layout="HND",
              stream=None, sliding_window=0, k_scale=1.0, v_scale=1.0):
    """Single-pass paged GQA decode into out [B, nq, hd]; sliding_window > 0 keeps the
    last sliding_window keys of each sequence."""
    nb, nkv, bs, hd = _pool_geometry(k_cache, layout)
    sb, sh, st = pool_strides(k_cache, layout)
    B, nq, _ = q.shape
    _check(load().pa_decode(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                            _ptr(seq_lens), B, nq, nkv, hd, bs, block_tables.shape[1], nb, sb,
                            sh, st, float(sm_scale), int(sliding_window), kv_dtype_of(k_cache),
                            float(k_scale), float(v_scale), _stream(stream)))


def decode_split_workspace_size(num_seqs, num_q_heads, head_dim, max_seq_len) -> int:
    return int(load().pa_decode_split_workspace_size(num_seqs, num_q_heads, head_dim,
                                                     max_seq_len))


def decode_split_workspace_views(workspace, num_seqs, num_q_heads, head_dim, max_seq_len):
    """(partial_out, partial_max, partial_sum) float32 views of a split workspace."""
    oo, om, ol = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    load().pa_decode_split_workspace_offsets(num_seqs, num_q_heads, head_dim, max_seq_len,
                                             ctypes.byref(oo), ctypes.byref(om),
                                             ctypes.byref(ol))
    P = (max_seq_len + PARTITION_TOKENS - 1) // PARTITION_TOKENS
    n = num_seqs * num_q_heads * P
    ws = workspace.view(torch.uint8)
    po = ws[oo.value:oo.value + n * head_dim * 4].view(torch.float32).view(num_seqs, num_q_heads,
                                                                           P, head_dim)
    pm = ws[om.value:om.value + n * 4].view(torch.float32).view(num_seqs, num_q_heads, P)
    pl = ws[ol.value:ol.value + n * 4].view(torch.float32).view(num_seqs, num_q_heads, P)
    return po, pm, pl


def alloc_workspace(nbytes: int, device) -> torch.Tensor:
    """A zeroed, 256-byte-aligned uint8 device buffer of at least nbytes (the prefill's
    work counters must start at zero)."""
    buf = torch.zeros(max(int(nbytes), 1) + 256, dtype=torch.uint8, device=device)
    off = (-buf.data_ptr()) % 256
    return buf[off:off + max(int(nbytes), 1)]


def pa_decode_split(out, q, k_cache, v_cache, block_tables, seq_lens, sm_scale, max_seq_len,
                    workspace, layout="HND", stream=None, sliding_window=0, k_scale=1.0,
                    v_scale=1.0):
    """Split-KV paged GQA decode (512-token partitions + LSE merge) into out [B, nq, hd]."""
    nb, nkv, bs, hd = _pool_geometry(k_cache, layout)
    sb, sh, st = pool_strides(k_cache, layout)
    B, nq, _ = q.shape
    _check(load().pa_decode_split(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                  _ptr(block_tables), _ptr(seq_lens), B, nq, nkv, hd, bs,
                                  block_tables.shape[1], nb, sb, sh, st, float(sm_scale),
                                  int(sliding_window), kv_dtype_of(k_cache), float(k_scale),
                                  float(v_scale), int(max_seq_len), _ptr(workspace),
                                  workspace.numel(), _stream(stream)))


STATIC_SCRATCH_BYTES = 16 * 1024 * 1024  # PA_STATIC_SCRATCH_BYTES in include/pa.h


def pa_decode_split_static(out, q, k_cache, v_cache, block_tables, seq_lens, sm_scale,
                           max_seq_len, layout="HND", stream=None, sliding_window=0,
                           k_scale=1.0, v_scale=1.0):
    """pa_decode_split with the library's fixed device scratch instead of a workspace,
    for callers that cannot allocate device memory.  Batches needing more than
    STATIC_SCRATCH_BYTES of partials are rejected; concurrent calls on one device race."""
    nb, nkv, bs, hd = _pool_geometry(k_cache, layout)
    sb, sh, st = pool_strides(k_cache, layout)
    B, nq, _ = q.shape
    _check(load().pa_decode_split_static(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                         _ptr(block_tables), _ptr(seq_lens), B, nq, nkv, hd, bs,
                                         block_tables.shape[1], nb, sb, sh, st, float(sm_scale),
                                         int(sliding_window), kv_dtype_of(k_cache),
                                         float(k_scale), float(v_scale), int(max_seq_len),
                                         _stream(stream)))


def pa_decode_partitions(q, k_cache, v_cache, block_tables, seq_lens, sm_scale, max_seq_len,
                         workspace, layout="HND", stream=None, sliding_window=0, k_scale=1.0,
                         v_scale=1.0):
    """Split-KV pass 1: per-partition (m, l, o) into the workspace."""
    nb, nkv, bs, hd = _pool_geometry(k_cache, layout)
    sb, sh, st = pool_strides(k_cache, layout)
    B, nq, _ = q.shape
    _check(load().pa_decode_partitions(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                       _ptr(seq_lens), B, nq, nkv, hd, bs, block_tables.shape[1],
                                       nb, sb, sh, st, float(sm_scale), int(sliding_window),
                                       kv_dtype_of(k_cache), float(k_scale), float(v_scale),
                                       int(max_seq_len), _ptr(workspace), workspace.numel(),
                                       _stream(stream)))


def pa_decode_merge(out, seq_lens, max_seq_len, workspace, stream=None, sliding_window=0):
    """Split-KV pass 2: log-sum-exp merge of the workspace partitions into out (the
    same sliding_window as pass 1)."""
    B, nq, hd = out.shape
    _check(load().pa_decode_merge(_ptr(out), _ptr(seq_lens), B, nq, hd, int(max_seq_len),
                                  int(sliding_window), _ptr(workspace), workspace.numel(),
                                  _stream(stream)))


def ragged_prefill_workspace_size(batch, total_qo_rows, num_q_heads, head_dim) -> int:
    return int(load().pa_ragged_prefill_workspace_size(batch, total_qo_rows, num_q_heads,
                                                       head_dim))


def pa_ragged_prefill(o, q, k, v, qo_indptr_h, kv_indptr_h, qo_indptr_d, kv_indptr_d, sm_scale,
                      causal=True, block_tables=None, num_kv_heads=None, layout="HND",
                      workspace=None, stream=None, sliding_window=0):
    """Ragged prefill.  Contiguous mode: k, v [total_kv, nkv, hd].  Paged mode
    (block_tables given): k, v are pools and kv_indptr only carries lengths.
    qo_indptr_h / kv_indptr_h are int32 host tensors (or numpy arrays)."""
    import numpy as np
    qh = np.ascontiguousarray(np.asarray(qo_indptr_h, np.int32))
    kh = np.ascontiguousarray(np.asarray(kv_indptr_h, np.int32))
    batch = qh.size - 1
    total_qo, nq, hd = q.shape
    if block_tables is None:
        nkv = k.shape[1]
        nb, bs, sb, sh, st, mb = 1, 16, 8, 8, 8, 1
        total_kv = k.shape[0]
    else:
        nb, nkv, bs, _ = _pool_geometry(k, layout)
        sb, sh, st = pool_strides(k, layout)
        mb = block_tables.shape[1]
        total_kv = int(kh[-1])
    if workspace is None:
        workspace = alloc_workspace(ragged_prefill_workspace_size(batch, total_qo, nq, hd),
                                    q.device)
    _check(load().pa_ragged_prefill(
        _ptr(o), _ptr(q), _ptr(k), _ptr(v), qh.ctypes.data_as(ctypes.c_void_p),
        kh.ctypes.data_as(ctypes.c_void_p), _ptr(qo_indptr_d), _ptr(kv_indptr_d),
        _ptr(block_tables), mb, bs, nb, sb, sh, st, batch, total_qo, total_kv, nq, nkv, hd,
        float(sm_scale), 1 if causal else 0, int(sliding_window), _ptr(workspace),
        workspace.numel(), _stream(stream)))


def selftest_wait_timeout(stream=None):
    """Runs one bounded wait that nothing completes (about 1 s); the device status
    then holds the PA_ERR_TIMEOUT bit."""
    _check(load().pa_selftest_wait_timeout(_stream(stream)))


def device_status(stream=None) -> int:
    """Synchronise the stream, then read and clear the device status bits."""
    st = ctypes.c_int(0)
    _check(load().pa_get_device_status(ctypes.byref(st), _stream(stream)))
    return st.value
