"""GPU: block swap to / from pinned host memory (kv_swap_out, kv_swap_in) through the C ABI,
bit-exact against the oracle's host-image model, and a preempt / resume flow whose
attention output must not change."""

import math

import numpy as np
import pytest
import torch

import workloads as W
from gpu_setup import max_abs, poison, prefill, tables_for
from oracle import cache as OC
from paged_kv_cache_169_gb300 import abi
from paged_kv_cache_169_gb300.cache import BlockAllocator, PagedKVCache

pytestmark = pytest.mark.gpu


def _bytes(t):
    return t.cpu().contiguous().view(torch.uint8).numpy()


@pytest.mark.parametrize("dtype", ["f16", "fp8", "f32"])
def test_swap_image_and_round_trip_bit_exact(dtype):
    rng = np.random.default_rng(150)
    L, nb, B, H, d = 3, 12, 16, 4, 64
    cache = PagedKVCache(L, nb, B, H, d, dtype)
    hk, hv, hks, hvs = [], [], [], []
    for l in range(L):
        for pool, store in ((cache.k[l], hk), (cache.v[l], hv)):
            if pool.dtype == torch.uint8:
                a = rng.integers(0, 256, pool.shape, dtype=np.uint8)
            else:
                a = rng.standard_normal(pool.shape).astype(np.float16 if pool.dtype == torch.float16 else np.float32)
                a[:, :, 9:] = np.nan
            pool.copy_(torch.from_numpy(a))
            store.append(a)
        if dtype == "fp8":
            for sc, store in ((cache.k_scale[l], hks), (cache.v_scale[l], hvs)):
                a = rng.uniform(0.01, 1, sc.shape).astype(np.float32)
                sc.copy_(torch.from_numpy(a))
                store.append(a)
    blocks = [7, 2, 11, 0]
    bt = torch.tensor(blocks, dtype=torch.int32, device="cuda")
    img = cache.swap_out(bt, layer_begin=1, layer_end=3)
    torch.cuda.synchronize()
    want = OC.swap_out(hk[1:3], hv[1:3], blocks, hks[1:3], hvs[1:3])
    assert img.numel() == want.size == abi.kv_swap_bytes(cache.handle, 4, 1, 3)
    assert np.array_equal(img.numpy(), want)
    # bring the image back into other blocks of layers 1..2
    dst = [3, 5, 6, 8]
    cache.swap_in(img, torch.tensor(dst, dtype=torch.int32, device="cuda"), layer_begin=1, layer_end=3)
    torch.cuda.synchronize()
    OC.swap_in(hk[1:3], hv[1:3], dst, want, hks[1:3], hvs[1:3])
    for l in range(L):
        assert np.array_equal(_bytes(cache.k[l]), hk[l].view(np.uint8))
        assert np.array_equal(_bytes(cache.v[l]), hv[l].view(np.uint8))
        if dtype == "fp8":
            assert np.array_equal(cache.k_scale[l].cpu().numpy()[:nb], hks[l][:nb])
            assert np.array_equal(cache.v_scale[l].cpu().numpy()[:nb], hvs[l][:nb])
    assert cache.device_error() == 0
    # a bad id is flagged and skipped; unpinned host memory is refused
    cache.swap_out(torch.tensor([1, nb + 3], dtype=torch.int32, device="cuda"), layer_begin=0, layer_end=1)
    assert cache.device_error() == abi.KV_DEVERR_BLOCK_ID
    # ordinary (pageable) host memory: refused where the GPU cannot address it; on a
    # coherent system (pageable memory access) accepted, and then it must be exact too
    plain = torch.zeros(abi.kv_swap_bytes(cache.handle, 1, 1, 3), dtype=torch.uint8)
    try:
        abi.kv_swap_out(cache.handle, bt.data_ptr(), 1, 1, 3, plain.data_ptr(),
                        torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        assert np.array_equal(plain.numpy(), OC.swap_out(hk[1:3], hv[1:3], blocks[:1], hks[1:3], hvs[1:3]))
    except abi.KvError as e:
        assert e.status == abi.KV_ERR_INVALID_ARG
    cache.close()


def test_preempt_and_resume_keeps_attention_output():
    """Swap a sequence out, free its blocks, let another sequence reuse (and dirty) them,
    swap it back into newly allocated blocks: the decode output is bit-identical."""
    B, H, d, L = 16, 8, 128, 2
    lens = [600, 333, 1000]
    nb = sum(-(-n // B) for n in lens) + 40
    w = W.Workload("swap", 151, L, H, d, B, "f16", len(lens), lens, nb, 1 / math.sqrt(d))
    cache = PagedKVCache(L, nb, B, H, d, "f16")
    poison(cache)
    alloc = BlockAllocator(nb, B, W.free_order(w))
    seqs = [alloc.new_seq() for _ in lens]
    ks = [W.host_tokens(w, s, n, "k") for s, n in enumerate(lens)]
    vs = [W.host_tokens(w, s, n, "v") for s, n in enumerate(lens)]
    for l in range(L):
        if l == 0:
            prefill(cache, alloc, seqs, ks, vs, layer=0)
        else:
            for s, sid in enumerate(seqs):
                tab = alloc.table(sid)
                slots = [tab[t // B] * B + t % B for t in range(lens[s])]
                cache.append(l, torch.from_numpy(ks[s]).cuda(), torch.from_numpy(vs[s]).cuda(),
                             torch.tensor(slots, dtype=torch.int64, device="cuda"))
    max_blocks = max(-(-n // B) for n in lens)
    bt, cl, _ = tables_for(alloc, seqs, max_blocks)
    q = torch.from_numpy(W.host_queries(w)).cuda()
    before = [cache.attention(l, q, bt, cl, max(lens), w.scale).clone() for l in range(L)]
    # preempt sequence 1
    victim = seqs[1]
    old_table = alloc.table(victim)
    img = cache.swap_out(torch.tensor(old_table, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    alloc.free_seq(victim)
    intruder = alloc.new_seq()
    slots, _ = alloc.append_slots(intruder, len(old_table) * B)
    junk = torch.full((len(slots), H, d), float("nan"), dtype=torch.float16, device="cuda")
    for l in range(L):
        cache.append(l, junk, junk, torch.tensor(slots, dtype=torch.int64, device="cuda"))
    # resume while the intruder still holds the old blocks: fresh blocks, same content
    resumed = alloc.new_seq()
    alloc.append_slots(resumed, lens[1])
    new_table = alloc.table(resumed)
    assert new_table != old_table
    cache.swap_in(img, torch.tensor(new_table, dtype=torch.int32, device="cuda"))
    seqs[1] = resumed
    bt2, cl2, _ = tables_for(alloc, seqs, max_blocks)
    for l in range(L):
        after = cache.attention(l, q, bt2, cl2, max(lens), w.scale)
        assert torch.equal(after, before[l]), max_abs(after.cpu().numpy(), before[l].cpu().numpy())
    assert cache.device_error() == 0
