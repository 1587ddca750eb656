"""Seeded synthetic inputs shared by the tests and the benchmark.

This module only draws inputs: lengths, shuffled block tables, slot mappings
and N(0, 1) bf16 values.  It holds none of the attention arithmetic, so both
the CUDA path and the CPU oracle can be fed from it without sharing any of
the computation.

Recipe (all five workloads):
  * metadata from ``numpy.random.default_rng(seed)``: lengths are inclusive
    uniform integers; physical pages are handed out by a random permutation
    of the pool (pool = ceil(1.1 * pages used), or a fixed pool), each
    sequence taking the next ceil(L / 16) ids; block-table padding is
    INT32_MAX, so any read past a sequence's pages would trip the guards;
  * values: N(0, 1) float32 from a seeded ``torch.Generator`` on the target
    device, rounded to bf16 (round-to-nearest-even) -- the whole pool is
    filled, so unused pages and stale rows hold finite garbage too.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

BLOCK_SIZE = 16
PAD_ENTRY = np.iinfo(np.int32).max


def bf16_normal(shape, seed: int, device="cpu") -> torch.Tensor:
    """N(0, 1) values rounded to bf16, reproducible for (shape, seed, device type)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    n = int(np.prod(shape)) if len(shape) else 1
    out = torch.empty(n, dtype=torch.bfloat16, device=device)
    chunk = 1 << 26  # bound the float32 staging buffer (256 MB)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = torch.randn(e - s, generator=gen, device=device,
                               dtype=torch.float32).to(torch.bfloat16)
    return out.view(*shape)


def to_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor (any device) -> numpy uint16 bit patterns on the host."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bits_to_float(bits: np.ndarray) -> np.ndarray:
    """numpy uint16 bf16 bit patterns -> float32 (exact)."""
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def float_to_bits(x) -> np.ndarray:
    """float32 -> bf16 bit patterns, round-to-nearest-even (finite inputs)."""
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def hash_uniform(counter: np.ndarray) -> np.ndarray:
    """Counter-based values in [-0.25, 0.25): the deterministic input recipe of
    the CPU-reference test on the "spark_runtime/flashinfer.rs" page
    (golden-ratio multiply, xor-shift 31, multiply by 0xBF58476D1CE4E5B9, top
    24 bits scaled to [0, 1), centred and halved)."""
    x = np.asarray(counter, np.uint64)
    with np.errstate(over="ignore"):
        x = x * np.uint64(0x9E3779B97F4A7C15) + np.uint64(1)
        x ^= x >> np.uint64(31)
        x = x * np.uint64(0xBF58476D1CE4E5B9)
    return (((x >> np.uint64(40)).astype(np.float64) / float(1 << 24)) - 0.5) * 0.5


def assign_pages(lens, block_size, rng, num_blocks=None, slack=0.10, max_blocks=None):
    """Shuffled block tables: returns (block_tables int32 [B, max_blocks], num_blocks)."""
    lens = np.asarray(lens, np.int64)
    need = [(int(L) + block_size - 1) // block_size for L in lens]
    used = int(sum(need))
    if num_blocks is None:
        num_blocks = max(1, int(math.ceil(used * (1.0 + slack))))
    assert num_blocks >= used, "pool too small"
    perm = rng.permutation(num_blocks).astype(np.int32)
    mb = max(1, max(need) if need else 1) if max_blocks is None else max_blocks
    bt = np.full((len(lens), mb), PAD_ENTRY, np.int32)
    pos = 0
    for b, n in enumerate(need):
        bt[b, :n] = perm[pos:pos + n]
        pos += n
    return bt, num_blocks


def slots_for_positions(block_tables, positions, block_size):
    """slot = page * block_size + row for token position pos of each row b."""
    pos = np.asarray(positions, np.int64)
    b = np.arange(len(pos))
    return block_tables[b, pos // block_size].astype(np.int64) * block_size + pos % block_size


@dataclass
class DecodeWorkload:
    name: str
    seq_lens: np.ndarray          # int32 [B]
    block_tables: np.ndarray      # int32 [B, max_blocks]
    num_blocks: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int = BLOCK_SIZE
    seed: int = 0
    new_token_write: bool = False  # write K/V of position L-1 via pa_write_cache first
    split: bool = False
    slot_mapping: Optional[np.ndarray] = None  # int64 [B] when new_token_write
    window: int = 0               # sliding window in keys (0: none)
    kv_fp8: bool = False          # the pools hold FP8 E4M3 codes (one byte per element)

    @property
    def batch(self):
        return int(self.seq_lens.size)

    @property
    def scale(self):
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def max_seq_len(self):
        return int(self.seq_lens.max()) if self.seq_lens.size else 0

    @property
    def pool_shape(self):  # HND pages
        return (self.num_blocks, self.num_kv_heads, self.block_size, self.head_dim)

    def visible_tokens(self):
        """Keys the queries attend to: all of each sequence, or its last `window`."""
        lens = self.seq_lens.astype(np.int64)
        if self.window > 0:
            lens = np.minimum(lens, self.window)
        return int(lens.sum())

    def kv_bytes(self):
        """Algorithmic decode bytes: K and V of every visible token."""
        elem = 1 if self.kv_fp8 else 2
        return self.visible_tokens() * self.num_kv_heads * self.head_dim * 2 * elem

    def tensors(self, device="cpu"):
        """q, k_cache, v_cache (and k_new, v_new if new_token_write) as bf16 tensors."""
        B, nq, nkv, hd = self.batch, self.num_q_heads, self.num_kv_heads, self.head_dim
        t = {
            "q": bf16_normal((B, nq, hd), self.seed * 10 + 1, device),
            "k_cache": bf16_normal(self.pool_shape, self.seed * 10 + 2, device),
            "v_cache": bf16_normal(self.pool_shape, self.seed * 10 + 3, device),
        }
        if self.new_token_write:
            t["k_new"] = bf16_normal((B, nkv, hd), self.seed * 10 + 4, device)
            t["v_new"] = bf16_normal((B, nkv, hd), self.seed * 10 + 5, device)
        return t


def make_decode(name, seq_lens, num_q_heads, num_kv_heads, head_dim, seed,
                block_size=BLOCK_SIZE, num_blocks=None, new_token_write=False, split=False,
                max_blocks=None, window=0, kv_fp8=False):
    rng = np.random.default_rng(seed)
    seq_lens = np.asarray(seq_lens, np.int32)
    bt, nb = assign_pages(seq_lens, block_size, rng, num_blocks=num_blocks,
                          max_blocks=max_blocks)
    w = DecodeWorkload(name, seq_lens, bt, nb, num_q_heads, num_kv_heads, head_dim,
                       block_size, seed, new_token_write, split, window=window, kv_fp8=kv_fp8)
    if new_token_write:
        w.slot_mapping = slots_for_positions(bt, np.maximum(seq_lens.astype(np.int64) - 1, 0),
                                             block_size)
        w.slot_mapping[seq_lens == 0] = -1
    return w


@dataclass
class PrefillWorkload:
    name: str
    qo_lens: np.ndarray
    kv_lens: np.ndarray
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    causal: bool = True
    seed: int = 0
    paged: bool = False
    block_size: int = BLOCK_SIZE
    block_tables: Optional[np.ndarray] = None
    num_blocks: int = 0
    chunk_write: bool = False           # paged: the new chunk's K/V go in via pa_write_cache
    chunk_slot_mapping: Optional[np.ndarray] = None  # int64 [sum qo]
    extra: dict = field(default_factory=dict)
    window: int = 0                     # sliding window in keys (0: none)

    @property
    def batch(self):
        return int(self.qo_lens.size)

    @property
    def scale(self):
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def qo_indptr(self):
        return np.concatenate([[0], np.cumsum(self.qo_lens)]).astype(np.int32)

    @property
    def kv_indptr(self):
        return np.concatenate([[0], np.cumsum(self.kv_lens)]).astype(np.int32)

    @property
    def total_qo(self):
        return int(self.qo_lens.sum())

    @property
    def total_kv(self):
        return int(self.kv_lens.sum())

    def visible_pairs(self):
        """Number of (query row, key) pairs left by the mask, per query head: row i sits
        at position i + kv - qo and sees keys j < kv, j <= position if causal, and
        j > position - window under a window."""
        tot = 0
        for qo, kv in zip(self.qo_lens.astype(np.int64), self.kv_lens.astype(np.int64)):
            pos = np.arange(qo, dtype=np.int64) + (kv - qo)
            hi = np.clip(pos + 1, 0, kv) if self.causal else np.full(qo, kv)
            lo = np.maximum(pos - self.window + 1, 0) if self.window > 0 else np.zeros(qo, np.int64)
            tot += int(np.clip(hi - lo, 0, None).sum())
        return int(tot)

    def flops(self):
        """Algorithmic FLOPs: 2 matmuls x 2 flop per MAC over the unmasked pairs."""
        return 4 * self.head_dim * self.num_q_heads * self.visible_pairs()

    def kv_bytes(self):
        return self.total_kv * self.num_kv_heads * self.head_dim * 2 * 2

    def tensors(self, device="cpu"):
        nq, nkv, hd = self.num_q_heads, self.num_kv_heads, self.head_dim
        t = {"q": bf16_normal((self.total_qo, nq, hd), self.seed * 10 + 1, device)}
        if not self.paged:
            t["k"] = bf16_normal((self.total_kv, nkv, hd), self.seed * 10 + 2, device)
            t["v"] = bf16_normal((self.total_kv, nkv, hd), self.seed * 10 + 3, device)
        else:
            shape = (self.num_blocks, nkv, self.block_size, hd)
            t["k_cache"] = bf16_normal(shape, self.seed * 10 + 2, device)
            t["v_cache"] = bf16_normal(shape, self.seed * 10 + 3, device)
            if self.chunk_write:
                t["k_new"] = bf16_normal((self.total_qo, nkv, hd), self.seed * 10 + 4, device)
                t["v_new"] = bf16_normal((self.total_qo, nkv, hd), self.seed * 10 + 5, device)
        return t


def make_prefill(name, qo_lens, kv_lens, num_q_heads, num_kv_heads, head_dim, seed,
                 causal=True, paged=False, chunk_write=False, block_size=BLOCK_SIZE,
                 num_blocks=None, window=0):
    qo = np.asarray(qo_lens, np.int32)
    kv = np.asarray(kv_lens, np.int32)
    w = PrefillWorkload(name, qo, kv, num_q_heads, num_kv_heads, head_dim, causal, seed,
                        paged, block_size, window=window)
    if paged:
        rng = np.random.default_rng(seed)
        w.block_tables, w.num_blocks = assign_pages(kv, block_size, rng, num_blocks=num_blocks)
        if chunk_write:
            # the new chunk occupies the last qo positions of each request
            slots = []
            for r in range(len(qo)):
                pos = np.arange(kv[r] - qo[r], kv[r], dtype=np.int64)
                pages = w.block_tables[r, pos // block_size].astype(np.int64)
                slots.append(pages * block_size + pos % block_size)
            w.chunk_slot_mapping = (np.concatenate(slots) if slots
                                    else np.zeros(0, np.int64)).astype(np.int64)
            w.chunk_write = True
    return w


# ---- the five named workloads -------------------------------------------------

def tiny_decode():
    """batch 4, 4 q / 2 kv heads, hd 64, bs 16, seq_lens {17,33,64,100}, pool of 64."""
    return make_decode("tiny_decode_b4_h4kv2_d64", [17, 33, 64, 100], 4, 2, 64, seed=1000,
                       num_blocks=64)


def llama8b_decode():
    """batch 64, 32 q / 8 kv heads, hd 128, seq_lens U[512, 4096], +10% pool."""
    rng = np.random.default_rng(1001)
    lens = rng.integers(512, 4096, size=64, endpoint=True)
    return make_decode("llama8b_decode_b64_h32kv8_d128", lens, 32, 8, 128, seed=1001,
                       new_token_write=True, split=True)


def long_context_decode():
    """batch 8, 32 q / 8 kv heads, hd 128, seq_lens U[32768, 131072], split-KV."""
    rng = np.random.default_rng(1002)
    lens = rng.integers(32768, 131072, size=8, endpoint=True)
    return make_decode("long_split_decode_b8_h32kv8_d128", lens, 32, 8, 128, seed=1002,
                       split=True)


def ragged_prefill():
    """16 requests, qo = kv ~ U[128, 2048], 32 q / 8 kv heads, hd 128, causal."""
    rng = np.random.default_rng(1003)
    lens = rng.integers(128, 2048, size=16, endpoint=True)
    return make_prefill("ragged_prefill_r16_h32kv8_d128", lens, lens, 32, 8, 128, seed=1003)


def chunked_paged_prefill():
    """8 requests, prefix U[1024, 8192] + 512-token chunk, 16 q / 8 kv, hd 256, paged."""
    rng = np.random.default_rng(1004)
    prefix = rng.integers(1024, 8192, size=8, endpoint=True)
    qo = np.full(8, 512, np.int64)
    return make_prefill("chunked_paged_prefill_r8_h16kv8_d256", qo, prefix + 512, 16, 8, 256,
                        seed=1004, paged=True, chunk_write=True)


def llama8b_decode_fp8():
    """llama8b_decode over an FP8 E4M3 cache (the same sequences and pages)."""
    rng = np.random.default_rng(1001)
    lens = rng.integers(512, 4096, size=64, endpoint=True)
    return make_decode("llama8b_decode_fp8_b64_h32kv8_d128", lens, 32, 8, 128, seed=1001,
                       new_token_write=True, split=True, kv_fp8=True)


def long_context_decode_fp8():
    """long_context_decode over an FP8 E4M3 cache (the same sequences and pages)."""
    rng = np.random.default_rng(1002)
    lens = rng.integers(32768, 131072, size=8, endpoint=True)
    return make_decode("long_split_decode_fp8_b8_h32kv8_d128", lens, 32, 8, 128, seed=1002,
                       split=True, kv_fp8=True)


def window_decode():
    """Sliding-window decode shaped like Mistral-7B (32 q / 8 kv heads, hd 128, a
    4096-key window): batch 32, seq_lens U[8192, 32768], split-KV."""
    rng = np.random.default_rng(1005)
    lens = rng.integers(8192, 32768, size=32, endpoint=True)
    return make_decode("window_decode_b32_h32kv8_d128_w4096", lens, 32, 8, 128, seed=1005,
                       split=True, window=4096)


def window_prefill():
    """Sliding-window ragged causal prefill: 8 requests, qo = kv ~ U[2048, 8192],
    32 q / 8 kv heads, hd 128, a 1024-key window."""
    rng = np.random.default_rng(1006)
    lens = rng.integers(2048, 8192, size=8, endpoint=True)
    return make_prefill("window_prefill_r8_h32kv8_d128_w1024", lens, lens, 32, 8, 128,
                        seed=1006, window=1024)


def llama8b_decode_single():
    """llama8b_decode (the same sequences, pages and new token) through the single-pass
    pa_decode: one pass over each whole sequence per (sequence, kv head), no split."""
    rng = np.random.default_rng(1001)
    lens = rng.integers(512, 4096, size=64, endpoint=True)
    return make_decode("llama8b_decode_single_b64_h32kv8_d128", lens, 32, 8, 128, seed=1001,
                       new_token_write=True, split=False)


def mha_decode():
    """Split-KV decode without grouping, shaped like Llama-2-7B (32 q / 32 kv heads,
    hd 128): batch 32, seq_lens U[512, 4096]."""
    rng = np.random.default_rng(1007)
    lens = rng.integers(512, 4096, size=32, endpoint=True)
    return make_decode("mha_decode_b32_h32kv32_d128", lens, 32, 32, 128, seed=1007,
                       split=True)


def gqa7_decode():
    """Split-KV decode with groups of 7 query heads, shaped like Qwen-2.5-7B (28 q / 4 kv
    heads, hd 128): batch 64, seq_lens U[512, 4096]."""
    rng = np.random.default_rng(1008)
    lens = rng.integers(512, 4096, size=64, endpoint=True)
    return make_decode("gqa7_decode_b64_h28kv4_d128", lens, 28, 4, 128, seed=1008, split=True)


WORKLOADS = {
    "tiny_decode": tiny_decode,
    "llama8b_decode": llama8b_decode,
    "long_context_decode": long_context_decode,
    "ragged_prefill": ragged_prefill,
    "chunked_paged_prefill": chunked_paged_prefill,
    "window_decode": window_decode,
    "llama8b_decode_fp8": llama8b_decode_fp8,
    "long_context_decode_fp8": long_context_decode_fp8,
    "window_prefill": window_prefill,
    "llama8b_decode_single": llama8b_decode_single,
    "mha_decode": mha_decode,
    "gqa7_decode": gqa7_decode,
}
