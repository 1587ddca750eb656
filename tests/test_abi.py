"""CPU-side checks of the C ABI: the library loads, exports every declared
symbol, and rejects bad arguments on the host before touching the GPU."""
import ctypes
import os
import re

import pytest

import paged_kv_gqa_15_gb300 as pa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pa.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build_library()
    return pa.load()


def test_header_declares_the_four_operations():
    names = declared_functions()
    for op in ("pa_write_cache", "pa_decode", "pa_decode_split", "pa_ragged_prefill"):
        assert op in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/pa.h but not exported"


FAKE = ctypes.c_void_p(0x10000)          # never dereferenced: validation fails first
FAKE_ODD = ctypes.c_void_p(0x10008)


def _decode(lib, **kw):
    a = dict(out=FAKE, q=FAKE, kc=FAKE, vc=FAKE, bt=FAKE, sl=FAKE, B=2, nq=8, nkv=2, hd=128,
             bs=16, mb=4, nb=100, sb=2 * 16 * 128, sh=16 * 128, st=128, scale=0.1)
    a.update(kw)
    return lib.pa_decode(a["out"], a["q"], a["kc"], a["vc"], a["bt"], a["sl"], a["B"], a["nq"],
                         a["nkv"], a["hd"], a["bs"], a["mb"], a["nb"], a["sb"], a["sh"], a["st"],
                         a["scale"], 0, 0, 1.0, 1.0, None)


@pytest.mark.parametrize("kw,code", [
    (dict(hd=96), pa.PA_ERR_UNSUPPORTED),
    (dict(nq=6, nkv=4), pa.PA_ERR_INVALID),
    (dict(bs=32), pa.PA_ERR_UNSUPPORTED),
    (dict(nb=0), pa.PA_ERR_INVALID),
    (dict(mb=0), pa.PA_ERR_INVALID),
    (dict(q=None), pa.PA_ERR_INVALID),
    (dict(out=FAKE_ODD), pa.PA_ERR_INVALID),
    (dict(st=100), pa.PA_ERR_INVALID),               # token stride not a multiple of 8
    (dict(st=64), pa.PA_ERR_INVALID),                # token stride < head_dim
    (dict(B=-1), pa.PA_ERR_INVALID),
    (dict(scale=float("nan")), pa.PA_ERR_INVALID),
])
def test_decode_rejects_bad_arguments(lib, kw, code):
    assert _decode(lib, **kw) == code
    assert lib.pa_last_error()


def test_split_rejects_small_workspace(lib):
    need = pa.decode_split_workspace_size(2, 8, 128, 1000)
    rc = lib.pa_decode_split(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 8, 2, 128, 16, 63, 100,
                             2 * 16 * 128, 16 * 128, 128, 0.1, 0, 0, 1.0, 1.0, 1000, ctypes.c_void_p(0x100000),
                             need - 1, None)
    assert rc == pa.PA_ERR_WORKSPACE
    rc = lib.pa_decode_split(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 8, 2, 128, 16, 63, 100,
                             2 * 16 * 128, 16 * 128, 128, 0.1, 0, 0, 1.0, 1.0, 1000, ctypes.c_void_p(0x100010),
                             need, None)
    assert rc == pa.PA_ERR_WORKSPACE                      # not 256-byte aligned
    rc = lib.pa_decode_split(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 8, 2, 128, 16, 10, 100,
                             2 * 16 * 128, 16 * 128, 128, 0.1, 0, 0, 1.0, 1.0, 1000, ctypes.c_void_p(0x100000),
                             need, None)
    assert rc == pa.PA_ERR_INVALID                        # max_seq_len > table capacity


def test_split_workspace_layout():
    B, nq, hd, L = 3, 8, 128, 1025                       # 3 partitions
    oo, om, ol = (ctypes.c_size_t() for _ in range(3))
    pa.load().pa_decode_split_workspace_offsets(B, nq, hd, L, ctypes.byref(oo), ctypes.byref(om),
                                                ctypes.byref(ol))
    rows = B * nq * 3
    assert oo.value == 0
    assert om.value >= rows * hd * 4 and om.value % 256 == 0
    assert ol.value >= om.value + rows * 4 and ol.value % 256 == 0
    assert pa.decode_split_workspace_size(B, nq, hd, L) >= ol.value + rows * 4


def test_write_cache_rejects_bad_arguments(lib):
    ok = dict(T=4, nkv=2, hd=128, bs=16, nb=10, sb=4096, sh=2048, st=128)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return lib.pa_write_cache(FAKE, FAKE, FAKE, FAKE, FAKE, a["T"], a["nkv"], a["hd"],
                                  a["bs"], a["nb"], a["sb"], a["sh"], a["st"], a.get("dt", 0),
                                  a.get("ks", 1.0), a.get("vs", 1.0), None)
    assert call(hd=80) == pa.PA_ERR_UNSUPPORTED
    assert call(T=-1) == pa.PA_ERR_INVALID
    assert call(bs=8) == pa.PA_ERR_UNSUPPORTED
    assert call(sh=0) == pa.PA_ERR_INVALID
    assert call(dt=2) == pa.PA_ERR_UNSUPPORTED                  # no such kv_dtype
    assert call(dt=1, ks=0.0) == pa.PA_ERR_INVALID              # fp8 scales must be > 0
    assert call(dt=1, vs=float("inf")) == pa.PA_ERR_INVALID
    assert call(dt=1, sb=4096 + 8) == pa.PA_ERR_INVALID         # 16-byte stride rule


def test_error_raises_with_message(lib):
    with pytest.raises(pa.PaError) as ei:
        pa._check(_decode(lib, hd=96))
    assert "head_dim" in str(ei.value)


def test_block_table_sync_uploads_nothing_when_unchanged():
    # host logic only: an unchanged table makes no CUDA call, so this runs without a GPU
    import ctypes
    import numpy as np
    import paged_kv_gqa_15_gb300 as pa
    lib = pa.load()
    host = np.arange(12, dtype=np.int32).reshape(3, 4)
    snap = host.copy()
    n = ctypes.c_int(-1)
    rc = lib.pa_block_table_sync(host.ctypes.data, snap.ctypes.data, ctypes.c_void_p(8),
                                 3, 4, ctypes.byref(n), None)
    assert rc == pa.PA_OK and n.value == 0
    assert lib.pa_block_table_sync(None, snap.ctypes.data, ctypes.c_void_p(8), 3, 4, None,
                                   None) == pa.PA_ERR_INVALID
    assert lib.pa_block_table_sync(host.ctypes.data, snap.ctypes.data, ctypes.c_void_p(8),
                                   -1, 4, None, None) == pa.PA_ERR_INVALID


def test_page_copies_reject_bad_arguments(lib):
    # validation happens before any CUDA call, so this runs without a GPU
    pools = (ctypes.c_void_p * 2)(0x10000, 0x20000)
    odd = (ctypes.c_void_p * 2)(0x10000, 0x20008)

    def copy(pl=pools, n=2, m=FAKE, pairs=3, nb=10, bb=32768):
        return lib.pa_copy_blocks(pl, n, m, pairs, nb, bb, None)
    assert copy(bb=100) == pa.PA_ERR_INVALID          # not a multiple of 16
    assert copy(bb=0) == pa.PA_ERR_INVALID
    assert copy(pairs=-1) == pa.PA_ERR_INVALID
    assert copy(n=-1) == pa.PA_ERR_INVALID
    assert copy(m=None) == pa.PA_ERR_INVALID
    assert copy(nb=0) == pa.PA_ERR_INVALID
    assert copy(pl=odd) == pa.PA_ERR_INVALID
    assert copy(pl=None) == pa.PA_ERR_INVALID
    assert copy(pairs=0) == pa.PA_OK                  # nothing to do, nothing enqueued
    assert copy(n=0) == pa.PA_OK

    def swap(src=pools, dst=pools, n=2, m=FAKE, pairs=3, snb=10, dnb=4, bb=32768):
        return lib.pa_swap_blocks(src, dst, n, m, pairs, snb, dnb, bb, None)
    assert swap(bb=24) == pa.PA_ERR_INVALID
    assert swap(dnb=0) == pa.PA_ERR_INVALID
    assert swap(m=None) == pa.PA_ERR_INVALID
    assert swap(src=None) == pa.PA_ERR_INVALID
    assert swap(n=5000) == pa.PA_ERR_UNSUPPORTED
    assert swap(pairs=0) == pa.PA_OK
