"""GPU: the allocation-free decode-attention entry point (paged_decode_attention_static).

Some callers cannot call cudaMalloc — a plugin whose host application owns all device
memory and gives it no allocator, or a serving loop that forbids device allocation once
it runs.  For them the library keeps its scratch (work counters, split-context
partials) in a fixed device array instead of a caller workspace.  This test calls that
entry point through the C ABI twice in a row, on two different batches, and checks each
result against the workspace entry point (paged_decode_attention) on the same inputs,
within the fp16 tolerance used throughout (2e-3 max abs); and checks that a request
needing more scratch than the array holds is refused.

This file is collected last on purpose, so that a run stopping at its first failure has
already run every other test.
"""

import math

import numpy as np
import pytest
import torch

import workloads as W
from paged_kv_cache_169_gb300 import abi, build
from paged_kv_cache_169_gb300.cache import BlockAllocator, PagedKVCache

pytestmark = pytest.mark.gpu


def _setup(seed, lens, H=8, d=128, B=16):
    nb = sum(-(-n // B) for n in lens) + 3
    w = W.Workload("noalloc", seed, 1, H, d, B, "f16", len(lens), lens, nb, 1 / math.sqrt(d))
    cache = PagedKVCache(1, nb, B, H, d, "f16")
    for t in cache.k + cache.v:
        t.fill_(float("nan"))
    alloc = BlockAllocator(nb, B, W.free_order(w))
    seqs = [alloc.new_seq() for _ in lens]
    for s, sid in enumerate(seqs):
        slots, _ = alloc.append_slots(sid, lens[s])
        cache.append(0, torch.from_numpy(W.host_tokens(w, s, lens[s], "k")).cuda(),
                     torch.from_numpy(W.host_tokens(w, s, lens[s], "v")).cuda(),
                     torch.tensor(slots, dtype=torch.int64, device="cuda"))
    max_blocks = max(-(-n // B) for n in lens)
    tabs, cl = alloc.build_tables(seqs, max_blocks)
    bt = torch.tensor(tabs, dtype=torch.int32, device="cuda")
    cl_t = torch.tensor(cl, dtype=torch.int32, device="cuda")
    q = torch.from_numpy(W.host_queries(w)).cuda()
    return w, cache, alloc, q, bt, cl_t, max_blocks


def _static_call(cache, w, q, bt, cl, max_blocks, out, partition=0):
    abi.paged_decode_attention_static(
        cache.handle, 0, q.data_ptr(), out.data_ptr(), bt.data_ptr(), max_blocks, cl.data_ptr(),
        w.batch, max(w.lens), w.scale, partition, torch.cuda.current_stream().cuda_stream)


def test_static_scratch_entry_point_matches_workspace_entry_point():
    build.build()
    batches = [
        (71, [1, 17, 600, 2048, 1500, 33, 900, 5]),                 # split partitions + short ones
        (72, [4000, 3, 257, 1024, 64, 2500]),                        # different shape, same scratch
    ]
    for seed, lens in batches:
        w, cache, alloc, q, bt, cl, max_blocks = _setup(seed, lens)
        assert cache.workspace_bytes(w.batch, max(lens)) > 256      # partials are in use
        want = cache.attention(0, q, bt, cl, max(lens), w.scale).cpu().numpy()
        out = torch.full((w.batch, w.num_heads, w.head_dim), float("nan"), device="cuda")
        _static_call(cache, w, q, bt, cl, max_blocks, out)
        got = out.cpu().numpy()
        assert np.all(np.isfinite(got))
        assert float(np.max(np.abs(got - want))) <= 2e-3
        assert cache.device_error() == 0
        cache.close()
        alloc.close()


def test_static_scratch_refuses_requests_that_do_not_fit():
    build.build()
    w, cache, alloc, q, bt, cl, max_blocks = _setup(73, [40, 70])
    # a huge max_context with small partitions needs far more than the fixed scratch
    need = cache.workspace_bytes(w.batch, 2_000_000, 32)
    assert need > abi.KV_STATIC_SCRATCH_BYTES
    out = torch.zeros((w.batch, w.num_heads, w.head_dim), device="cuda")
    with pytest.raises(abi.KvError) as e:
        abi.paged_decode_attention_static(
            cache.handle, 0, q.data_ptr(), out.data_ptr(), bt.data_ptr(), max_blocks, cl.data_ptr(),
            w.batch, 2_000_000, w.scale, 32, torch.cuda.current_stream().cuda_stream)
    assert e.value.status == abi.KV_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert float(out.abs().sum()) == 0.0                           # nothing was launched
    cache.close()
    alloc.close()
