"""Page copies on the GPU (pa_copy_blocks / pa_swap_blocks) against the oracle's byte
copies on host copies of the same pools: bit-exact, for several page sizes (one
16 KB segment, several, and a ragged tail), more pools than one launch carries,
pinned host pools on either side, padding and out-of-range pairs, a CUDA-graph
replay, and a copy-on-write fork that the decode must read exactly like its parent."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_15_gb300 as pa
from paged_kv_gqa_15_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    yield
    assert pa.device_status() == 0


def _pools(n, num_blocks, page_shape, dtype, seed, device=DEV, pin=False):
    g = torch.Generator().manual_seed(seed)
    out = []
    for _ in range(n):
        bits = torch.randint(-32768, 32767, (num_blocks,) + page_shape, generator=g,
                             dtype=torch.int16)
        t = bits.view(dtype) if dtype != torch.int16 else bits
        t = t.pin_memory() if pin else t.to(device)
        out.append(t)
    return out


def _host_bytes(t):
    return t.detach().cpu().contiguous().view(torch.uint8).numpy().reshape(t.shape[0], -1).copy()


def _pairs(num_blocks, n, seed, pad=0):
    """n pairs: sources drawn with repeats, destinations distinct and never sources."""
    rng = np.random.default_rng(seed)
    perm = rng.permutation(num_blocks)
    dst = perm[:n]
    src = rng.choice(perm[n:], size=n, replace=True)
    pairs = np.stack([src, dst], 1).astype(np.int64)
    if pad:
        pads = np.full((pad, 2), -1, np.int64)
        pads[::2, 0] = 0        # (0, -1): a padding pair with a valid source
        pairs = np.concatenate([pairs, pads])
        pairs = pairs[rng.permutation(len(pairs))]
    return pairs


@pytest.mark.parametrize("page_shape,dtype", [
    ((8, 16, 128), torch.bfloat16),     # Llama-3-8B page: 32 KB, two 16 KB segments
    ((1, 16, 64), torch.bfloat16),      # 2 KB page: one partial segment
    ((8, 16, 256), torch.bfloat16),     # 64 KB page: four segments
    ((520,), torch.int16),              # 1040-byte page: a ragged 16-byte multiple
])
def test_copy_blocks_matches_oracle(page_shape, dtype):
    nb, layers = 96, 3
    k = _pools(layers, nb, page_shape, dtype, seed=1)
    v = _pools(layers, nb, page_shape, dtype, seed=2)
    host = [_host_bytes(t) for kv in zip(k, v) for t in kv]
    pairs = _pairs(nb, 40, seed=3, pad=6)
    pa.pa_copy_blocks(k, v, torch.from_numpy(pairs).to(DEV))
    torch.cuda.synchronize()
    assert oracle.copy_blocks(host, pairs) == 0
    got = [_host_bytes(t) for kv in zip(k, v) for t in kv]
    for i, (g, h) in enumerate(zip(got, host)):
        assert np.array_equal(g, h), f"pool {i}"


def test_copy_blocks_across_more_pools_than_one_launch_carries():
    nb, layers = 20, 70                 # 140 pools: two launches of at most 128
    k = _pools(layers, nb, (2, 16, 64), torch.bfloat16, seed=4)
    v = _pools(layers, nb, (2, 16, 64), torch.bfloat16, seed=5)
    host = [_host_bytes(t) for kv in zip(k, v) for t in kv]
    pairs = _pairs(nb, 7, seed=6)
    pa.pa_copy_blocks(k, v, torch.from_numpy(pairs).to(DEV))
    torch.cuda.synchronize()
    oracle.copy_blocks(host, pairs)
    for i, t in enumerate(t for kv in zip(k, v) for t in kv):
        assert np.array_equal(_host_bytes(t), host[i]), f"pool {i}"


@pytest.mark.parametrize("mapping_on", ["device", "pinned"])
def test_swap_out_to_pinned_host_and_back(mapping_on):
    nb_dev, nb_host, layers = 64, 24, 2
    dev = _pools(2 * layers, nb_dev, (8, 16, 128), torch.bfloat16, seed=7)
    hostp = _pools(2 * layers, nb_host, (8, 16, 128), torch.bfloat16, seed=8, pin=True)
    ref_dev = [_host_bytes(t) for t in dev]
    ref_host = [_host_bytes(t) for t in hostp]
    rng = np.random.default_rng(9)
    out_pairs = np.stack([rng.choice(nb_dev, 20, replace=False),
                          rng.choice(nb_host, 20, replace=False)], 1).astype(np.int64)

    def mapping(p):
        t = torch.from_numpy(p)
        return t.to(DEV) if mapping_on == "device" else t.pin_memory()

    m_out = mapping(out_pairs)
    pa.pa_swap_blocks(dev, hostp, m_out)              # swap out: device -> host
    torch.cuda.synchronize()
    for s, h in zip(ref_dev, ref_host):
        assert oracle.swap_blocks(s, h, out_pairs) == 0
    for i, t in enumerate(hostp):
        assert np.array_equal(_host_bytes(t), ref_host[i]), f"host pool {i}"
    # swap in to other device pages: host -> device
    in_pairs = np.stack([out_pairs[:, 1], rng.permutation(nb_dev)[:20]], 1).astype(np.int64)
    m_in = mapping(in_pairs)
    pa.pa_swap_blocks(hostp, dev, m_in)
    torch.cuda.synchronize()
    for h, d in zip(ref_host, ref_dev):
        oracle.swap_blocks(h, d, in_pairs)
    for i, t in enumerate(dev):
        assert np.array_equal(_host_bytes(t), ref_dev[i]), f"device pool {i}"


def test_out_of_range_pairs_are_skipped_and_flagged():
    nb = 16
    k = _pools(1, nb, (2, 16, 64), torch.bfloat16, seed=10)
    v = _pools(1, nb, (2, 16, 64), torch.bfloat16, seed=11)
    host = [_host_bytes(k[0]), _host_bytes(v[0])]
    pairs = np.array([[1, 2], [nb, 3], [4, nb + 5], [6, 7]], np.int64)
    assert pa.device_status() == 0
    pa.pa_copy_blocks(k, v, torch.from_numpy(pairs).to(DEV))
    assert pa.device_status() == 1 << pa.PA_ERR_DEVICE_BOUNDS
    assert oracle.copy_blocks(host, pairs) == 2 * 2
    assert np.array_equal(_host_bytes(k[0]), host[0])
    assert np.array_equal(_host_bytes(v[0]), host[1])


def test_copy_blocks_replayed_from_a_cuda_graph():
    nb = 48
    k = _pools(2, nb, (8, 16, 128), torch.bfloat16, seed=12)
    v = _pools(2, nb, (8, 16, 128), torch.bfloat16, seed=13)
    m_d = torch.full((8, 2), -1, dtype=torch.int64, device=DEV)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        pa.pa_copy_blocks(k, v, m_d, stream=stream)   # all padding: a no-op warm-up
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        pa.pa_copy_blocks(k, v, m_d, stream=stream)
    torch.cuda.synchronize()
    host = [_host_bytes(t) for kv in zip(k, v) for t in kv]
    for seed in (14, 15, 16):
        pairs = _pairs(nb, 8, seed=seed)
        m_d.copy_(torch.from_numpy(pairs))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        oracle.copy_blocks(host, pairs)
        for i, t in enumerate(t for kv in zip(k, v) for t in kv):
            assert np.array_equal(_host_bytes(t), host[i]), f"seed {seed}, pool {i}"


def test_forked_sequence_decodes_like_its_parent():
    w = W.make_decode("fork", [700, 129, 1024], 32, 8, 128, seed=17, num_blocks=256)
    t = w.tensors(DEV)
    bt = w.block_tables
    used = set(int(x) for x in bt[bt != W.PAD_ENTRY].ravel())
    free = [b for b in range(w.num_blocks) if b not in used]
    child = bt.copy()
    pairs = []
    for b in range(w.batch):
        for i in range((int(w.seq_lens[b]) + 15) // 16):
            new = free.pop()
            pairs.append((int(bt[b, i]), new))
            child[b, i] = new
    pa.pa_copy_blocks([t["k_cache"]], [t["v_cache"]],
                      torch.tensor(pairs, dtype=torch.int64, device=DEV))
    sl = torch.from_numpy(w.seq_lens).to(DEV)
    out_p = torch.empty_like(t["q"])
    out_c = torch.empty_like(t["q"])
    pa.pa_decode(out_p, t["q"], t["k_cache"], t["v_cache"], torch.from_numpy(bt).to(DEV), sl,
                 w.scale)
    pa.pa_decode(out_c, t["q"], t["k_cache"], t["v_cache"], torch.from_numpy(child).to(DEV), sl,
                 w.scale)
    torch.cuda.synchronize()
    assert torch.equal(out_p, out_c)
