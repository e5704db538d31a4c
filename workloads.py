"""Seeded synthetic inputs for the five decode-attention workloads.

This module only draws random numbers and fixes shapes; it holds none of the
method's arithmetic (no attention, no paging, no quantisation).  Both the CUDA
path's tests/bench and the oracle take their inputs from here.

Host-side randomness (lengths, permutations, small tensors) uses
``numpy.random.default_rng(seed)``; large device tensors use a
``torch.Generator`` seeded with the same seed (plus a per-layer / per-sequence
offset).  Values are N(0, 1) in the stated dtype.

Workloads (shapes of LLaMA-7B / LLaMA-13B attention layers as given on the
pages "KV缓存机制解析" §3.1 and "KV Cache与PagedAttention" §1.1):

  tiny      1 layer, batch 2, 2 heads, d 64, fp32, lengths 37 and 5 after the
            decode append, B 16, 16-block pool, free list = permutation(16).
  llama7b   1 layer, 32 heads, d 128, fp16, batch 8, initial lengths uniform in
            [512, 2048], B 16, 64 decode steps of one token each.
  llama13b  40 layers, 40 heads, d 128, fp16, batch 48, every length 2048 after
            the decode append, B 16, 6144 blocks per layer (~75 GiB pool).
  parallel  1 layer, 40 heads, d 128, fp16, B 16: 8 candidates share a 1030-token
            prompt, each decodes 128 tokens.
  ragged    256 sequences, lengths floor(exp(U(ln 16, ln 16384))), 32 heads,
            d 128, fp16 (and an FP8-E4M3 pool variant), B in {8, 16, 32}.
  gqa70b    80 layers, 64 query heads over 8 K/V heads (LLaMA-2-70B shape), d 128, fp16,
            B 16, batch 32, every length 4096.
  longctx13b  8 layers of the LLaMA-13B shape (40 heads, d 128, fp16, B 16) with only 2
            sequences of 32768 tokens: few (sequence, head) units, so one sequence's
            context is split into many partitions.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np


@dataclass
class Workload:
    name: str
    seed: int
    num_layers: int
    num_heads: int
    head_dim: int
    block_size: int
    dtype: str                      # "f32" | "f16"   (storage of q and of the K/V inputs)
    batch: int
    lens: list = field(default_factory=list)  # context length after this step's append
    num_blocks: int = 0
    scale: float = 0.0
    steps: int = 1
    num_q_heads: int = 0            # query heads (0: same as num_heads; more = grouped-query)

    @property
    def q_heads(self) -> int:
        return self.num_q_heads or self.num_heads

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2


def _np_dtype(dtype: str):
    return np.float32 if dtype == "f32" else np.float16


# ----------------------------------------------------------------------------
# workload descriptions
# ----------------------------------------------------------------------------

def tiny() -> Workload:
    return Workload("tiny", seed=1, num_layers=1, num_heads=2, head_dim=64, block_size=16,
                    dtype="f32", batch=2, lens=[37, 5], num_blocks=16, scale=1.0 / 8.0)


def llama7b() -> Workload:
    rng = np.random.default_rng(2)
    init = rng.integers(512, 2049, 8).tolist()          # lengths before the 64 decode steps
    steps = 64
    need = sum(-(-(n + steps) // 16) for n in init)
    return Workload("llama7b", seed=2, num_layers=1, num_heads=32, head_dim=128, block_size=16,
                    dtype="f16", batch=8, lens=[n + 1 for n in init],
                    num_blocks=int(math.ceil(need * 1.1)), scale=1.0 / math.sqrt(128), steps=steps)


def llama13b(num_layers: int = 40) -> Workload:
    return Workload("llama13b", seed=3, num_layers=num_layers, num_heads=40, head_dim=128,
                    block_size=16, dtype="f16", batch=48, lens=[2048] * 48,
                    num_blocks=48 * 128, scale=1.0 / math.sqrt(128))


def parallel_sampling() -> Workload:
    return Workload("parallel", seed=4, num_layers=1, num_heads=40, head_dim=128, block_size=16,
                    dtype="f16", batch=8, lens=[1031] * 8, num_blocks=160,
                    scale=1.0 / math.sqrt(128), steps=128)


def ragged(block_size: int = 16) -> Workload:
    rng = np.random.default_rng(5)
    u = rng.uniform(math.log(16), math.log(16384), 256)
    lens = np.clip(np.floor(np.exp(u)).astype(np.int64), 16, 16384).tolist()
    need = sum(-(-n // block_size) for n in lens)
    return Workload(f"ragged_b{block_size}", seed=5, num_layers=1, num_heads=32, head_dim=128,
                    block_size=block_size, dtype="f16", batch=256, lens=lens,
                    num_blocks=need + need // 10, scale=1.0 / math.sqrt(128))


def gqa70b(num_layers: int = 80) -> Workload:
    """LLaMA-2-70B-shaped grouped-query layer stack: 64 query heads share 8 K/V heads,
    d 128, fp16, B 16, batch 32, every context 4096 after the decode append."""
    return Workload("gqa70b", seed=6, num_layers=num_layers, num_heads=8, head_dim=128, block_size=16,
                    dtype="f16", batch=32, lens=[4096] * 32, num_blocks=32 * 256,
                    scale=1.0 / math.sqrt(128), num_q_heads=64)


def longctx13b(num_layers: int = 8) -> Workload:
    return Workload("longctx13b", seed=7, num_layers=num_layers, num_heads=40, head_dim=128, block_size=16,
                    dtype="f16", batch=2, lens=[32768] * 2, num_blocks=2 * 2048, scale=1.0 / math.sqrt(128))


PROMPT_LEN_PARALLEL = 1030
CANDIDATES_PARALLEL = 8


# ----------------------------------------------------------------------------
# random draws
# ----------------------------------------------------------------------------

def free_order(w: Workload, salt: int = 0) -> np.ndarray:
    """A seeded permutation of the physical block ids: the allocator's initial free list."""
    rng = np.random.default_rng(w.seed * 7919 + 17 + salt)
    return rng.permutation(w.num_blocks).astype(np.int32)


def tiny_free_order(w: Workload) -> np.ndarray:
    """The tiny workload's free list is exactly ``default_rng(1).permutation(16)``."""
    return np.random.default_rng(w.seed).permutation(w.num_blocks).astype(np.int32)


def host_tokens(w: Workload, seq: int, n_tokens: int, kind: str) -> np.ndarray:
    """N(0,1) values ``[n_tokens, H, d]`` of sequence ``seq`` for ``kind`` in {"k","v"}.

    Drawn from a generator keyed by (seed, seq, kind) so any sequence can be
    regenerated on its own.
    """
    salt = {"k": 1, "v": 2}[kind]
    rng = np.random.default_rng([w.seed, seq, salt])
    x = rng.standard_normal((n_tokens, w.num_heads, w.head_dim), dtype=np.float32)
    return x.astype(_np_dtype(w.dtype))


def host_queries(w: Workload, step: int = 0, layer: int = 0) -> np.ndarray:
    """N(0,1) queries ``[batch, Hq, d]`` for one decode step of one layer."""
    rng = np.random.default_rng([w.seed, 1_000_000 + step, layer])
    x = rng.standard_normal((w.batch, w.q_heads, w.head_dim), dtype=np.float32)
    return x.astype(_np_dtype(w.dtype))


def host_step_tokens(w: Workload, step: int, layer: int, kind: str) -> np.ndarray:
    """N(0,1) new-token K or V ``[batch, H, d]`` for one decode step of one layer."""
    salt = {"k": 1, "v": 2}[kind]
    rng = np.random.default_rng([w.seed, 2_000_000 + step, layer, salt])
    x = rng.standard_normal((w.batch, w.num_heads, w.head_dim), dtype=np.float32)
    return x.astype(_np_dtype(w.dtype))


def device_fill_normal(t, seed_key: int) -> None:
    """Fill a device tensor with N(0,1) in its own dtype from a seeded device generator.

    Filled in slices of at most 256 Mi elements so no large float32 temporary is needed.
    """
    import torch

    g = torch.Generator(device=t.device)
    g.manual_seed(int(seed_key))
    flat = t.view(-1)
    step = 1 << 28
    for i in range(0, flat.numel(), step):
        n = min(step, flat.numel() - i)
        flat[i:i + n].normal_(0.0, 1.0, generator=g)


def shuffled_tables(w: Workload, blocks_per_seq, salt: int = 0) -> np.ndarray:
    """Block tables drawn from one seeded permutation of the pool: seq s gets the next
    ``blocks_per_seq[s]`` ids of the permutation.  Padded with -1 to the longest row."""
    perm = free_order(w, salt)
    rows = max(blocks_per_seq) if len(blocks_per_seq) else 0
    tab = np.full((len(blocks_per_seq), max(rows, 1)), -1, dtype=np.int32)
    pos = 0
    for s, nb in enumerate(blocks_per_seq):
        tab[s, :nb] = perm[pos:pos + nb]
        pos += nb
    assert pos <= w.num_blocks
    return tab
