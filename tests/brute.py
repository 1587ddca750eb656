"""Brute-force dense attention, written independently of the oracle.

Used only to pin the oracle on tiny inputs: it materialises contiguous K / V
for each sequence by walking the block table token by token in Python, builds
the whole score matrix with a numpy matmul, masks it, and normalises it with
numpy's exp -- a different code path from the oracle's per-row C loops.
"""
import numpy as np

from paged_kv_gqa_15_gb300.workloads import bits_to_float


def widen(bits):
    return bits_to_float(bits).astype(np.float64)


def gather_paged(pool_bits, block_table_row, length, kv_head, block_size, strides):
    """Contiguous [length, hd] float64 rows of one kv head, read token by token.  A
    float64 pool holds values already; any other dtype holds bf16 bit patterns."""
    sb, sh, st = strides
    flat = pool_bits.reshape(-1)
    hd = None
    rows = []
    for j in range(length):
        page = int(block_table_row[j // block_size])
        base = page * sb + kv_head * sh + (j % block_size) * st
        if hd is None:
            hd = _hd_from(pool_bits)
        rows.append(flat[base:base + hd])
    if not rows:
        return np.zeros((0, _hd_from(pool_bits)))
    if pool_bits.dtype == np.float64:
        return np.stack(rows)
    return widen(np.stack(rows))


def _hd_from(pool_bits):
    return pool_bits.shape[-1]


def dense_softmax_attention(q, K, V, scale, visible=None):
    """q [n_q, hd], K/V [n_k, hd] (float64); visible bool [n_q, n_k] or None."""
    S = scale * (q @ K.T)
    if visible is not None:
        S = np.where(visible, S, -np.inf)
    out = np.zeros((q.shape[0], V.shape[1]))
    for i in range(q.shape[0]):
        row = S[i]
        if not np.isfinite(row).any():
            continue
        w = np.exp(row - row[np.isfinite(row)].max())
        out[i] = (w / w.sum()) @ V
    return out


def brute_decode(q_bits, kc_bits, vc_bits, bt, seq_lens, nkv, bs, scale, strides, window=0):
    """window > 0: the query (position L - 1) sees only keys j > L - 1 - window."""
    B, nq, hd = q_bits.shape
    g = nq // nkv
    q = widen(q_bits)
    out = np.zeros((B, nq, hd))
    for b in range(B):
        L = int(seq_lens[b])
        for kh in range(nkv):
            K = gather_paged(kc_bits, bt[b], L, kh, bs, strides)
            V = gather_paged(vc_bits, bt[b], L, kh, bs, strides)
            if L == 0:
                continue
            heads = list(range(kh * g, (kh + 1) * g))
            vis = None
            if window > 0:
                vis = np.repeat((np.arange(L) > L - 1 - window)[None, :], g, axis=0)
            out[b, heads] = dense_softmax_attention(q[b, heads], K, V, scale, vis)
    return out


def causal_visible(qo, kv, causal, window=0):
    """Query row i sits at position i + kv - qo; causal keeps keys j <= that position and a
    window W > 0 keeps keys j > position - W."""
    i = np.arange(qo)[:, None]
    j = np.arange(kv)[None, :]
    vis = np.ones((qo, kv), bool)
    if causal:
        vis &= j <= i + (kv - qo)
    if window > 0:
        vis &= j > i + (kv - qo) - window
    return vis


def brute_prefill_contiguous(q_bits, k_bits, v_bits, qo_indptr, kv_indptr, nkv, scale, causal,
                             window=0):
    T, nq, hd = q_bits.shape
    g = nq // nkv
    q, k, v = widen(q_bits), widen(k_bits), widen(v_bits)
    out = np.zeros((T, nq, hd))
    for r in range(len(qo_indptr) - 1):
        q0, q1 = qo_indptr[r], qo_indptr[r + 1]
        k0, k1 = kv_indptr[r], kv_indptr[r + 1]
        vis = causal_visible(q1 - q0, k1 - k0, causal, window)
        for h in range(nq):
            out[q0:q1, h] = dense_softmax_attention(q[q0:q1, h], k[k0:k1, h // g],
                                                    v[k0:k1, h // g], scale, vis)
    return out


def brute_decode_values(q_bits, kc_vals, vc_vals, bt, seq_lens, nkv, bs, scale, strides):
    """brute_decode over float64 pools of values (e.g. a dequantised fp8 cache)."""
    return brute_decode(q_bits, np.asarray(kc_vals, np.float64), np.asarray(vc_vals, np.float64),
                        bt, seq_lens, nkv, bs, scale, strides)
