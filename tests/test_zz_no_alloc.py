"""GPU: the allocation-free decode-attention entry point (paged_decode_attention_static).

Some callers cannot call cudaMalloc — a plugin whose host application owns all device
memory and gives it no allocator, or a serving loop that forbids device allocation once
it runs.  For them the library keeps its scratch (work counters, split-context
partials) in a fixed device array instead of a caller workspace.  This test calls that
entry point through the C ABI on two differently shaped batches in a row and then on the
first batch again, and checks:
  * each result is bit-identical to the workspace entry point's (paged_decode_attention)
    on the same inputs: the same kernel and plan run, and the split-context merge adds
    the partials in partition order, so nothing depends on which warp merges; the third
    call shows that the partials the second batch left in the shared array do not leak;
  * each result is within the fp16 tolerance used throughout (2e-3 max abs) of the
    float64 oracle on the tokens that were appended;
  * the device's free memory is the same before and after those calls (the first call's
    one-time set-up is done before the first reading);
and that a request needing more scratch than the array holds is refused.

This file is collected last on purpose, so that a run stopping at its first failure has
already run every other test.
"""

import math

import numpy as np
import pytest
import torch

import workloads as W
from gpu_setup import max_abs, tol_for
from oracle import attention as OA
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
    ks = [W.host_tokens(w, s, n, "k") for s, n in enumerate(lens)]
    vs = [W.host_tokens(w, s, n, "v") for s, n in enumerate(lens)]
    for s, sid in enumerate(seqs):
        slots, _ = alloc.append_slots(sid, lens[s])
        cache.append(0, torch.from_numpy(ks[s]).cuda(), torch.from_numpy(vs[s]).cuda(),
                     torch.tensor(slots, dtype=torch.int64, device="cuda"))
    max_blocks = max(-(-n // B) for n in lens)
    tabs, cl = alloc.build_tables(seqs, max_blocks)
    bt = torch.tensor(tabs, dtype=torch.int32, device="cuda")
    cl_t = torch.tensor(cl, dtype=torch.int32, device="cuda")
    qh = W.host_queries(w)
    return dict(w=w, cache=cache, alloc=alloc, q=torch.from_numpy(qh).cuda(), qh=qh, ks=ks, vs=vs,
                bt=bt, cl=cl_t, max_blocks=max_blocks)


def _static_call(c, out, partition=0):
    w = c["w"]
    abi.paged_decode_attention_static(
        c["cache"].handle, 0, c["q"].data_ptr(), out.data_ptr(), c["bt"].data_ptr(), c["max_blocks"],
        c["cl"].data_ptr(), w.batch, max(w.lens), w.scale, partition, torch.cuda.current_stream().cuda_stream)


def test_static_scratch_entry_point_matches_workspace_entry_point():
    build.build()
    cases = [
        _setup(71, [1, 17, 600, 2048, 1500, 33, 900, 5]),           # split partitions + short ones
        _setup(72, [4000, 3, 257, 1024, 64, 2500]),                 # another shape, same scratch
    ]
    wants, outs = [], []
    for c in cases:
        w = c["w"]
        assert c["cache"].workspace_bytes(w.batch, max(w.lens)) > 256   # partials are in use
        wants.append(c["cache"].attention(0, c["q"], c["bt"], c["cl"], max(w.lens), w.scale).cpu().numpy())
        outs.append([torch.full((w.batch, w.num_heads, w.head_dim), float("nan"), device="cuda")
                     for _ in range(2)])
    # one-time set-up (the scratch address lookup) before the memory reading
    _static_call(cases[0], outs[0][1])
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    _static_call(cases[0], outs[0][0])
    _static_call(cases[1], outs[1][0])
    _static_call(cases[0], outs[0][1])                              # the first batch again
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before              # nothing was allocated
    for i, c in enumerate(cases):
        w = c["w"]
        got = outs[i][0].cpu().numpy()
        assert np.array_equal(got, wants[i])                        # bit-identical
        if i == 0:
            assert np.array_equal(outs[0][1].cpu().numpy(), wants[0])
        want = OA.decode_attention(c["qh"], c["ks"], c["vs"], w.scale)
        assert max_abs(got, want) <= tol_for("f16")
        assert c["cache"].device_error() == 0
    for c in cases:
        c["cache"].close()
        c["alloc"].close()


def test_static_scratch_refuses_requests_that_do_not_fit():
    build.build()
    c = _setup(73, [40, 70])
    w, cache = c["w"], c["cache"]
    # a huge max_context with small partitions needs far more than the fixed scratch
    need = cache.workspace_bytes(w.batch, 2_000_000, 32)
    assert need > abi.KV_STATIC_SCRATCH_BYTES
    out = torch.zeros((w.batch, w.num_heads, w.head_dim), device="cuda")
    with pytest.raises(abi.KvError) as e:
        abi.paged_decode_attention_static(
            cache.handle, 0, c["q"].data_ptr(), out.data_ptr(), c["bt"].data_ptr(), c["max_blocks"],
            c["cl"].data_ptr(), w.batch, 2_000_000, w.scale, 32, torch.cuda.current_stream().cuda_stream)
    assert e.value.status == abi.KV_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert float(out.abs().sum()) == 0.0                           # nothing was launched
    cache.close()
    c["alloc"].close()
