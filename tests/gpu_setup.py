"""Shared set-up for the GPU parity tests: build workloads on the device through the
product path (allocator + kv_append), and hand the oracle the same inputs as host
arrays.  Nothing here computes attention, paging or quantisation itself."""

from __future__ import annotations

import numpy as np
import torch

import workloads as W
from paged_kv_cache_169_gb300.cache import BlockAllocator, PagedKVCache

TORCH_DT = {"f32": torch.float32, "f16": torch.float16}
NP_DT = {"f32": np.float32, "f16": np.float16}


def tol_for(dtype: str) -> float:
    """Max-abs tolerance against the float64 oracle: 1e-5 for fp32 K/V, 2e-3 for fp16 and
    FP8 (dequantised) K/V with fp32 accumulation."""
    return 1e-5 if dtype == "f32" else 2e-3


def poison(cache: PagedKVCache) -> None:
    """Fill every pool with NaN (FP8: the NaN code 0x7F) so unread slots stay visible."""
    for t in cache.k + cache.v:
        if t.dtype == torch.uint8:
            t.fill_(0x7F)
        else:
            t.fill_(float("nan"))


def prefill(cache: PagedKVCache, alloc: BlockAllocator, seqs, tokens_k, tokens_v, layer: int = 0):
    """Append every sequence's tokens through the allocator's slots and kv_append.
    tokens_k[s]: host [n_s, H, d] array.  Returns the slots per sequence."""
    out = []
    for s, sid in enumerate(seqs):
        n = tokens_k[s].shape[0]
        if n == 0:
            out.append([])
            continue
        slots, cow = alloc.append_slots(sid, n)
        assert cow is None
        k = torch.from_numpy(np.ascontiguousarray(tokens_k[s])).cuda()
        v = torch.from_numpy(np.ascontiguousarray(tokens_v[s])).cuda()
        cache.append(layer, k, v, torch.tensor(slots, dtype=torch.int64, device="cuda"))
        out.append(slots)
    return out


def tables_for(alloc: BlockAllocator, seqs, max_blocks: int):
    tabs, lens = alloc.build_tables(seqs, max_blocks)
    return (torch.tensor(tabs, dtype=torch.int32, device="cuda"),
            torch.tensor(lens, dtype=torch.int32, device="cuda"), lens)


def max_abs(a, b) -> float:
    return float(np.max(np.abs(np.asarray(a, dtype=np.float64) - np.asarray(b, dtype=np.float64))))


def fp8_block_scales(tokens, B: int):
    """Per logical block: amax over the block's tokens (all heads, all dims) / 448, floored
    at 2^-20 (input preparation: the caller's choice of scale for a prefilled block)."""
    n = tokens.shape[0]
    nb = -(-n // B)
    sc = np.empty(nb, dtype=np.float32)
    for j in range(nb):
        amax = float(np.max(np.abs(tokens[j * B:(j + 1) * B].astype(np.float32))))
        sc[j] = np.float32(max(amax / 448.0, 2.0 ** -20))
    return sc


__all__ = ["W", "tol_for", "poison", "prefill", "tables_for", "max_abs", "fp8_block_scales",
           "TORCH_DT", "NP_DT"]
