"""GPU: the largest inputs one decode-attention call takes, against the float64 oracle.

* The largest batch (KV_MAX_DECODE_BATCH = 65536 sequences: 64 launches of 1024), short
  ragged contexts with a few long ones in several launches (two-level merges), and the
  first batch past the limit refused before anything runs.
* One sequence of 262144 tokens: 1024 to 8192 partitions per head, merged in two levels
  (64 to 512 groups of 16), on the CUDA-core consumer and the grouped-query tensor-core
  consumer.
"""

import math

import numpy as np
import pytest
import torch

import workloads as W
from gpu_setup import max_abs, poison, tables_for, tol_for
from oracle import attention as OA
from paged_kv_cache_169_gb300 import abi
from paged_kv_cache_169_gb300.cache import BlockAllocator, PagedKVCache

pytestmark = pytest.mark.gpu


def _fill(cache, alloc, seqs, ks, vs):
    """Every sequence's tokens in one kv_append call (slots from the allocator)."""
    slots = []
    for sid, k in zip(seqs, ks):
        if k.shape[0]:
            slots.extend(alloc.append_slots(sid, k.shape[0])[0])
    kk = torch.from_numpy(np.concatenate(ks)).cuda()
    vv = torch.from_numpy(np.concatenate(vs)).cuda()
    cache.append(0, kk, vv, torch.tensor(slots, dtype=torch.int64, device="cuda"))


def test_largest_batch_and_the_first_refused():
    n = abi.KV_MAX_DECODE_BATCH
    B, H, d = 8, 1, 64
    rng = np.random.default_rng(171)
    lens = rng.integers(0, 25, n)
    lens[::8191] = 700                     # long sequences in several launches: 22 partitions of 32
    lens[-1] = 33                          # the very last sequence of the last launch
    lens = lens.tolist()
    nb = sum(-(-x // B) for x in lens) + 8
    w = W.Workload("max_batch", 171, 1, H, d, B, "f16", n, lens, nb, 1 / math.sqrt(d))
    cache = PagedKVCache(1, nb, B, H, d, "f16")
    poison(cache)
    alloc = BlockAllocator(nb, B, W.free_order(w))
    seqs = [alloc.new_seq() for _ in lens]
    ks = [W.host_tokens(w, s, x, "k") for s, x in enumerate(lens)]
    vs = [W.host_tokens(w, s, x, "v") for s, x in enumerate(lens)]
    _fill(cache, alloc, seqs, ks, vs)
    bt, cl, _ = tables_for(alloc, seqs, max(-(-x // B) for x in lens))
    q = W.host_queries(w)
    want = OA.decode_attention(q, ks, vs, w.scale)
    qd = torch.from_numpy(q).cuda()
    for P in (0, 32):
        out = cache.attention(0, qd, bt, cl, max(lens), w.scale, partition_tokens=P).cpu().numpy()
        assert max_abs(out, want) <= tol_for("f16"), P
        assert np.all(out[np.asarray(lens) == 0] == 0)
    assert cache.device_error() == 0
    # one sequence more: refused before any launch (the output keeps its contents)
    q1 = torch.zeros((n + 1, H, d), dtype=torch.float16, device="cuda")
    bt1 = torch.zeros((n + 1, 1), dtype=torch.int32, device="cuda")
    cl1 = torch.ones(n + 1, dtype=torch.int32, device="cuda")
    out1 = torch.full((n + 1, H, d), 7.0, device="cuda")
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(abi.KvError) as e:
        cache.attention(0, q1, bt1, cl1, 1, w.scale, out=out1, workspace=ws)
    assert e.value.status == abi.KV_ERR_INVALID_ARG
    with pytest.raises(abi.KvError):                    # the size query answers 0
        abi.paged_decode_workspace_size(cache.handle, n + 1, 1, 0)
    # split counts whose item numbers or workspace bytes would overflow are refused too
    with pytest.raises(abi.KvError):
        abi.paged_decode_workspace_size(cache.handle, n, 2 ** 31 - 1, 32)
    with pytest.raises(abi.KvError) as e:
        cache.attention(0, q1[:n], bt1[:n], cl1[:n], 2 ** 31 - 1, w.scale, out=out1[:n], partition_tokens=32,
                        workspace=ws)
    assert e.value.status == abi.KV_ERR_INVALID_ARG
    assert abi.paged_decode_workspace_size(cache.handle, n, 2 ** 20, 32) > 0   # 2^25 items: fine
    torch.cuda.synchronize()
    assert bool(torch.all(out1 == 7.0))
    cache.close()
    alloc.close()


def test_one_sequence_of_262144_tokens():
    n, B, H, d = 262144, 32, 2, 128
    nb = n // B + 2
    w = W.Workload("max_context", 172, 1, H, d, B, "f16", 1, [n], nb, 1 / math.sqrt(d), num_q_heads=8 * H)
    cache = PagedKVCache(1, nb, B, H, d, "f16")
    alloc = BlockAllocator(nb, B, W.free_order(w))
    seqs = [alloc.new_seq()]
    k, v = W.host_tokens(w, 0, n, "k"), W.host_tokens(w, 0, n, "v")
    _fill(cache, alloc, seqs, [k], [v])
    bt, cl, _ = tables_for(alloc, seqs, n // B)
    q = W.host_queries(w)                                   # [1, 16, 128]: 8 query heads per K/V head
    want = OA.decode_attention_gqa(q, [k], [v], w.scale)
    qd = torch.from_numpy(q).cuda()
    for P in (0, 32):
        got = cache.attention_gqa(0, qd, bt, cl, n, w.scale, partition_tokens=P).cpu().numpy()
        assert max_abs(got, want) <= tol_for("f16"), ("gqa", P)
    q1 = np.ascontiguousarray(q[:, ::8])                     # one query per K/V head
    want1 = OA.decode_attention(q1, [k], [v], w.scale)
    for P in (0, 32):
        got = cache.attention(0, torch.from_numpy(q1).cuda(), bt, cl, n, w.scale, partition_tokens=P)
        assert max_abs(got.cpu().numpy(), want1) <= tol_for("f16"), ("mha", P)
    assert cache.device_error() == 0
    cache.close()
    alloc.close()
