"""GPU: failure detection without a GPU fault.  A kernel wait that runs out (an mbarrier
nothing arrives at, with a short limit) must set KV_DEVERR_TIMEOUT and return, leaving the
context usable: the next decode call on the same pool and stream is still exact."""

import math
import time

import numpy as np
import pytest
import torch

import workloads as W
from gpu_setup import max_abs, poison, prefill, tables_for, tol_for
from oracle import attention as OA
from paged_kv_cache_169_gb300 import abi
from paged_kv_cache_169_gb300.cache import BlockAllocator, PagedKVCache

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_stays_usable():
    lens = [5, 40, 300]
    B, H, d = 16, 2, 128
    nb = sum(-(-n // B) for n in lens) + 2
    w = W.Workload("failure", 170, 1, H, d, B, "f16", len(lens), lens, nb, 1 / math.sqrt(d))
    cache = PagedKVCache(1, nb, B, H, d, "f16")
    poison(cache)
    alloc = BlockAllocator(nb, B, W.free_order(w))
    seqs = [alloc.new_seq() for _ in lens]
    ks = [W.host_tokens(w, s, n, "k") for s, n in enumerate(lens)]
    vs = [W.host_tokens(w, s, n, "v") for s, n in enumerate(lens)]
    prefill(cache, alloc, seqs, ks, vs)
    assert cache.device_error() == 0
    stream = torch.cuda.current_stream().cuda_stream
    t0 = time.perf_counter()
    abi.kv_selftest_wait_timeout(cache.handle, 20_000_000, stream)       # 20 ms
    code = cache.device_error()
    elapsed = time.perf_counter() - t0
    assert code == abi.KV_DEVERR_TIMEOUT
    assert 0.015 < elapsed < 5.0
    assert cache.device_error() == 0                                      # read-and-clear
    bt, cl, _ = tables_for(alloc, seqs, max(-(-n // B) for n in lens))
    q = W.host_queries(w)
    out = cache.attention(0, torch.from_numpy(q).cuda(), bt, cl, max(lens), w.scale).cpu().numpy()
    assert max_abs(out, OA.decode_attention(q, ks, vs, w.scale)) <= tol_for("f16")
    assert cache.device_error() == 0
    with pytest.raises(abi.KvError) as e:
        abi.kv_selftest_wait_timeout(cache.handle, 0, stream)
    assert e.value.status == abi.KV_ERR_INVALID_ARG
    with pytest.raises(abi.KvError):
        abi.kv_selftest_wait_timeout(cache.handle, 2_000_000_000, stream)
    cache.close()
