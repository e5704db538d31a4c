"""Runs the float64 oracle over every (sequence, head) output of a full-size decode call.

Test infrastructure.  It calls only ``oracle.attention.decode_attention_window`` (and
``oracle.fp8.decode`` for FP8 pools) on host arrays that a test prepared from seeded
inputs; nothing here computes attention itself, and no value comes from the CUDA path.

The (sequence, head) problems are independent, so they are spread over a thread pool:
numpy releases the interpreter lock inside its casts, products and reductions, so the
threads run in parallel (about 5x on 8 host cores).  A process pool would need the
inputs copied or shared between processes; threads read them in place.
"""

from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from oracle import attention as OA
from oracle import fp8 as OF


def host_threads() -> int:
    n = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    return max(1, n)


def oracle_sequences(q, k_seqs, v_seqs, scale: float, *, group: int = 1, window: int = 0,
                     k_tok_scale=None, v_tok_scale=None, threads: int | None = None) -> np.ndarray:
    """Oracle decode attention of every (sequence, query head).

    q:       [S, Hq, d] (fp16 or fp32 values)
    k_seqs:  list of S arrays [Hkv, n_s, d], head-major: the n_s cached tokens of each K/V
             head of sequence s, in token order (fp16 / fp32 values, or E4M3 codes)
    v_seqs:  same
    group:   query heads per K/V head (Hq = group * Hkv); query head j reads K/V head j // group
    window:  0, or attend only to the last ``window`` tokens (as the oracle defines it)
    k_tok_scale, v_tok_scale: FP8 pools only: lists of S float arrays [n_s], the scale of
             the physical block holding each token; a token's value is decode(code) * scale
    Returns [S, Hq, d] float64.
    """
    q = np.asarray(q)
    S, Hq, d = q.shape
    out = np.zeros((S, Hq, d), dtype=np.float64)
    fp8 = k_tok_scale is not None

    def one(s: int) -> None:
        Ks, Vs = k_seqs[s], v_seqs[s]
        hkv = Ks.shape[0]
        for hk in range(hkv):
            Kh, Vh = Ks[hk], Vs[hk]                          # [n, d]
            if fp8:
                Kh = OF.decode(Kh) * np.asarray(k_tok_scale[s], dtype=np.float64)[:, None]
                Vh = OF.decode(Vh) * np.asarray(v_tok_scale[s], dtype=np.float64)[:, None]
            qs = q[s, hk * group:(hk + 1) * group][None]     # [1, G, d]
            out[s, hk * group:(hk + 1) * group] = OA.decode_attention_window(
                qs, [Kh[:, None, :]], [Vh[:, None, :]], scale, window)[0]

    # longest sequences first, so the pool ends evenly
    order = sorted(range(S), key=lambda s: -k_seqs[s].shape[1])
    with ThreadPoolExecutor(threads or host_threads()) as ex:
        list(ex.map(one, order))
    return out


def gather_seqs(pool, tables, lens, block_size: int, seqs=None, tok_scale=None):
    """Host copies of sequences' caches read from a (device) pool through their tables.

    pool: torch tensor [num_blocks, H, B, d] of one layer (the test's own snapshot of the
    inputs); tables: host int32 [S, max_blocks]; lens: context lengths.  Returns a list of
    [H, n_s, d] numpy arrays (and, with tok_scale = a host per-block scale array, a list of
    per-token scales [n_s]).  The gather runs on the device with torch (input preparation).
    """
    import torch

    seqs = range(len(lens)) if seqs is None else seqs
    ks, sc = [], []
    for s in seqs:
        n = int(lens[s])
        nb = -(-n // block_size)
        idx = torch.as_tensor(np.asarray(tables[s][:nb], dtype=np.int64), device=pool.device)
        t = pool.index_select(0, idx)                       # [nb, H, B, d]
        t = t.permute(1, 0, 2, 3).reshape(t.shape[1], nb * block_size, t.shape[3])[:, :n]
        ks.append(t.contiguous().cpu().numpy())
        if tok_scale is not None:
            phys = np.asarray(tables[s][:nb], dtype=np.int64)
            sc.append(np.repeat(np.asarray(tok_scale, dtype=np.float64)[phys], block_size)[:n])
    return (ks, sc) if tok_scale is not None else ks
