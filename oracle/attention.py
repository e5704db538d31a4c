"""Oracle: decode attention in float64 (test infrastructure only, see package doc).

Definitions followed
--------------------
[KV Cache篇] §2.1 computes ``scores = Q K^T / 2`` (2 = sqrt(4) for head_dim 4),
adds a causal mask, applies softmax along the key axis and multiplies by V.
§3.1 (the LLaMA ``Attention.forward``) writes the new token's K/V into the cache
*before* reading ``cache[:start_pos + seqlen]``, scales by ``1/sqrt(head_dim)``
and takes the softmax in fp32; with ``seqlen == 1`` no mask is built.
[KV缓存机制解析] §5.1 states the decode step as
``out_n = softmax(Q_n [K_0..K_n]^T) [V_0..V_n]``: the current query against every
cached key *including its own*.

So for one (sequence, head) with ``n`` cached tokens (the one appended this
step included)::

    x_t   = scale * sum_j q[j] * K[t, j]          t = 0 .. n-1
    m     = max_t x_t
    p_t   = exp(x_t - m) / sum_u exp(x_u - m)
    out_j = sum_t p_t * V[t, j]

All arithmetic is float64 on values widened exactly from their storage type.
``n == 0`` is an empty sum: the output is zeros (a reading; the pages never
attend over an empty cache).
"""

from __future__ import annotations

import numpy as np


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def decode_attention_one(q, K, V, scale: float) -> np.ndarray:
    """One query row against ``n`` cached keys/values, as defined in the module doc.

    q: [d]; K, V: [n, d].  Returns out [d] (float64).
    """
    q, K, V = _f64(q), _f64(K), _f64(V)
    n, d = K.shape
    if n == 0:
        return np.zeros(q.shape[-1], dtype=np.float64)
    x = scale * (K @ q)                     # x_t = scale * q . K_t
    m = np.max(x)
    e = np.exp(x - m)
    p = e / np.sum(e)
    return p @ V                            # out_j = sum_t p_t V[t, j]


def decode_attention(q, k_seqs, v_seqs, scale: float) -> np.ndarray:
    """Decode attention for a batch over contiguous per-sequence caches.

    q:      [batch, H, d]
    k_seqs: list (len batch) of [n_s, H, d] arrays — the token-major per-sequence
            cache of [KV缓存机制解析] §2.2 / [KV Cache篇] §3.1 (``cache_k[b, :n]``).
    v_seqs: same shapes as ``k_seqs``.
    Returns [batch, H, d] float64.
    """
    q = _f64(q)
    b, H, d = q.shape
    out = np.zeros((b, H, d), dtype=np.float64)
    for s in range(b):
        Ks, Vs = _f64(k_seqs[s]), _f64(v_seqs[s])
        for h in range(H):
            out[s, h] = decode_attention_one(q[s, h], Ks[:, h, :], Vs[:, h, :], scale)
    return out


def causal_attention(Q, K, V, scale: float) -> np.ndarray:
    """Full recompute without a cache ([KV Cache篇] §2.1): every row i attends to
    keys 0..i; entries above the diagonal get -inf before the softmax.

    Q, K, V: [n, d].  Returns [n, d].
    """
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    n = Q.shape[0]
    scores = scale * (Q @ K.T)
    mask = np.triu(np.full((n, n), -np.inf), k=1)
    scores = scores + mask
    out = np.zeros_like(Q)
    for i in range(n):
        row = scores[i]
        e = np.exp(row - np.max(row))
        out[i] = (e / np.sum(e)) @ V
    return out


def paged_gather(pool, table_row, n: int, block_size: int) -> np.ndarray:
    """Rebuild a sequence's contiguous ``[n, H, d]`` cache from a paged pool.

    pool: [num_blocks, H, block_size, d] (one layer, head-major inside a block).
    Logical block ``j`` of the sequence lives in physical block ``table_row[j]``
    ([PagedAttention] §2.1: logical blocks map to non-contiguous physical
    blocks through the sequence's block table), so token ``t`` is at
    ``pool[table_row[t // B], :, t % B, :]``.
    """
    pool = np.asarray(pool)
    H, d = pool.shape[1], pool.shape[3]
    out = np.empty((n, H, d), dtype=pool.dtype)
    for t in range(n):
        phys = int(table_row[t // block_size])
        out[t] = pool[phys, :, t % block_size, :]
    return out


def paged_decode_attention(q, k_pool, v_pool, block_tables, context_lens, scale: float,
                           block_size: int, k_block_scale=None, v_block_scale=None,
                           dequant=None) -> np.ndarray:
    """Decode attention read through block tables: gather, then the contiguous form.

    q: [batch, H, d]; k_pool/v_pool: [num_blocks, H, B, d]; block_tables: [batch, >=
    ceil(n_s/B)] physical ids; context_lens: [batch].  For an FP8 pool pass the
    per-physical-block scales and ``dequant`` (code array -> float64 values); each
    gathered element is ``dequant(code) * scale[block]``, computed exactly in
    float64 ([KV缓存机制解析] §8: a low-precision cache stored with a scaling
    factor).
    """
    b = len(context_lens)
    k_seqs, v_seqs = [], []
    for s in range(b):
        n = int(context_lens[s])
        Ks = paged_gather(k_pool, block_tables[s], n, block_size)
        Vs = paged_gather(v_pool, block_tables[s], n, block_size)
        if dequant is not None:
            ks = np.array([k_block_scale[int(block_tables[s][t // block_size])] for t in range(n)],
                          dtype=np.float64).reshape(n, 1, 1)
            vs = np.array([v_block_scale[int(block_tables[s][t // block_size])] for t in range(n)],
                          dtype=np.float64).reshape(n, 1, 1)
            Ks = dequant(Ks) * ks
            Vs = dequant(Vs) * vs
        k_seqs.append(Ks)
        v_seqs.append(Vs)
    return decode_attention(q, k_seqs, v_seqs, scale)


def decode_attention_gqa(q, k_seqs, v_seqs, scale: float) -> np.ndarray:
    """Grouped-query decode attention ([KV Cache篇] §6.2: groups of query heads share one
    K/V head; MQA is a single shared head).

    q: [batch, Hq, d]; k_seqs/v_seqs: list of [n_s, Hkv, d] with Hq a multiple of Hkv.
    Query head j of a group of G = Hq / Hkv consecutive heads reads K/V head j // G.
    """
    q = _f64(q)
    b, Hq, d = q.shape
    out = np.zeros((b, Hq, d), dtype=np.float64)
    for s in range(b):
        Ks, Vs = _f64(k_seqs[s]), _f64(v_seqs[s])
        Hkv = Ks.shape[1]
        assert Hq % Hkv == 0
        G = Hq // Hkv
        for j in range(Hq):
            out[s, j] = decode_attention_one(q[s, j], Ks[:, j // G, :], Vs[:, j // G, :], scale)
    return out


def decode_attention_window(q, k_seqs, v_seqs, scale: float, window: int) -> np.ndarray:
    """Sliding-window decode ([KV缓存机制解析] §8, 滚动窗口缓存: keep only the most recent
    WINDOW_SIZE tokens): each query attends to the last ``window`` cached tokens of its
    sequence (all of them when the context is shorter).  ``window <= 0`` means no window.
    Query heads may be grouped over K/V heads as in ``decode_attention_gqa``."""
    ks, vs = [], []
    for K, V in zip(k_seqs, v_seqs):
        n = np.asarray(K).shape[0]
        lo = max(0, n - window) if window > 0 else 0
        ks.append(np.asarray(K)[lo:])
        vs.append(np.asarray(V)[lo:])
    return decode_attention_gqa(q, ks, vs, scale)
