"""GPU: paged_decode_attention through the C ABI against the float64 oracle.

Tolerances (max abs error): 1e-5 for fp32 K/V; 2e-3 for fp16 K/V and for FP8 K/V
(compared with the oracle on the dequantised values) — fp32 accumulation throughout.
Unused slots of every pool hold NaN, so a read past context_len would show.
"""

import math

import numpy as np
import pytest
import torch

import workloads as W
from gpu_setup import fp8_block_scales, max_abs, poison, prefill, tables_for, tol_for
from oracle import attention as OA
from oracle import fp8 as OF
from paged_kv_cache_169_gb300 import abi
from paged_kv_cache_169_gb300.cache import BlockAllocator, PagedKVCache

pytestmark = pytest.mark.gpu


def _decode_step(cache, alloc, seqs, new_k, new_v, layer=0):
    """Reserve one slot per sequence and append the new token (product path)."""
    slots, cows = [], []
    for sid in seqs:
        sl, cow = alloc.append_slots(sid, 1)
        slots += sl
        if cow:
            cows.append(cow)
    if cows:
        cache.copy_blocks(torch.tensor(cows, dtype=torch.int32, device="cuda"))
    cache.append(layer, torch.from_numpy(new_k).cuda(), torch.from_numpy(new_v).cuda(),
                 torch.tensor(slots, dtype=torch.int64, device="cuda"))
    return cows


# ------------------------------------------------------------------ tiny (fp32)

@pytest.mark.parametrize("partition_tokens", [0, 32, 64, 512])
def test_tiny_decode_step(partition_tokens):
    w = W.tiny()
    cache = PagedKVCache(1, w.num_blocks, w.block_size, w.num_heads, w.head_dim, "f32")
    poison(cache)
    alloc = BlockAllocator(w.num_blocks, w.block_size, W.tiny_free_order(w))
    seqs = [alloc.new_seq() for _ in range(w.batch)]
    ks = [W.host_tokens(w, s, n, "k") for s, n in enumerate(w.lens)]
    vs = [W.host_tokens(w, s, n, "v") for s, n in enumerate(w.lens)]
    prefill(cache, alloc, seqs, [k[:-1] for k in ks], [v[:-1] for v in vs])
    _decode_step(cache, alloc, seqs, np.stack([k[-1] for k in ks]), np.stack([v[-1] for v in vs]))
    # the page-specified physical placement: blocks taken from permutation(16) in order
    perm = W.tiny_free_order(w).tolist()
    assert alloc.table(seqs[0]) == perm[:3] and alloc.table(seqs[1]) == perm[3:4]
    bt, cl, lens = tables_for(alloc, seqs, 4)
    assert lens == w.lens
    q = W.host_queries(w)
    out = cache.attention(0, torch.from_numpy(q).cuda(), bt, cl, max(lens), w.scale,
                          partition_tokens=partition_tokens)
    want = OA.decode_attention(q, ks, vs, w.scale)
    assert max_abs(out.cpu().numpy(), want) <= tol_for("f32")
    assert cache.device_error() == 0


# ------------------------------------------------------------------ LLaMA-7B layer, 64 steps

def test_llama7b_64_decode_steps():
    w = W.llama7b()
    init = [n - 1 for n in w.lens]
    total = [n + w.steps for n in init]
    cache = PagedKVCache(1, w.num_blocks, w.block_size, w.num_heads, w.head_dim, "f16")
    poison(cache)
    alloc = BlockAllocator(w.num_blocks, w.block_size, W.free_order(w))
    seqs = [alloc.new_seq() for _ in range(w.batch)]
    ks = [W.host_tokens(w, s, n, "k") for s, n in enumerate(total)]
    vs = [W.host_tokens(w, s, n, "v") for s, n in enumerate(total)]
    prefill(cache, alloc, seqs, [k[:n] for k, n in zip(ks, init)], [v[:n] for v, n in zip(vs, init)])
    max_blocks = -(-max(total) // w.block_size)
    worst = 0.0
    for step in range(w.steps):
        pos = [n + step for n in init]
        _decode_step(cache, alloc, seqs, np.stack([k[p] for k, p in zip(ks, pos)]),
                     np.stack([v[p] for v, p in zip(vs, pos)]))
        bt, cl, lens = tables_for(alloc, seqs, max_blocks)
        assert lens == [p + 1 for p in pos]
        q = W.host_queries(w, step)
        out = cache.attention(0, torch.from_numpy(q).cuda(), bt, cl, max(total), w.scale)
        want = OA.decode_attention(q, [k[:p + 1] for k, p in zip(ks, pos)],
                                   [v[:p + 1] for v, p in zip(vs, pos)], w.scale)
        worst = max(worst, max_abs(out.cpu().numpy(), want))
    assert worst <= tol_for("f16"), worst
    assert cache.device_error() == 0


# ------------------------------------------------------------------ parallel sampling + CoW

def test_parallel_sampling_cow_and_attention():
    w = W.parallel_sampling()
    P0, NCAND = W.PROMPT_LEN_PARALLEL, W.CANDIDATES_PARALLEL
    cache = PagedKVCache(1, w.num_blocks, w.block_size, w.num_heads, w.head_dim, "f16")
    poison(cache)
    alloc = BlockAllocator(w.num_blocks, w.block_size, W.free_order(w))
    root = alloc.new_seq()
    prompt_k = W.host_tokens(w, 0, P0, "k")
    prompt_v = W.host_tokens(w, 0, P0, "v")
    prefill(cache, alloc, [root], [prompt_k], [prompt_v])
    cands = [root] + [alloc.fork(root) for _ in range(NCAND - 1)]
    assert all(alloc.ref_count(b) == NCAND for b in alloc.table(root))
    gen_k = [W.host_tokens(w, 100 + c, w.steps, "k") for c in range(NCAND)]
    gen_v = [W.host_tokens(w, 100 + c, w.steps, "v") for c in range(NCAND)]
    shared_last = alloc.table(root)[-1]
    before_k = cache.k[0][shared_last].clone()
    before_v = cache.v[0][shared_last].clone()
    max_blocks = -(-(P0 + w.steps) // w.block_size)
    worst = 0.0
    for step in range(w.steps):
        cows = _decode_step(cache, alloc, cands, np.stack([g[step] for g in gen_k]),
                            np.stack([g[step] for g in gen_v]))
        if step == 0:
            assert len(cows) == NCAND - 1 and all(c[0] == shared_last for c in cows)
            for _, dst in cows:            # whole-block copies, bit-exact (NaN slots included)
                assert torch.equal(cache.k[0][dst][:, :P0 % 16].view(torch.int16),
                                   before_k[:, :P0 % 16].view(torch.int16))
                assert torch.equal(cache.v[0][dst][:, :P0 % 16].view(torch.int16),
                                   before_v[:, :P0 % 16].view(torch.int16))
                assert torch.isnan(cache.k[0][dst][:, P0 % 16 + 1:].float()).all()
        else:
            assert not cows
        if step in (0, 1, 9, 10, 63, 127):
            bt, cl, lens = tables_for(alloc, cands, max_blocks)
            assert lens == [P0 + step + 1] * NCAND
            q = W.host_queries(w, step)
            out = cache.attention(0, torch.from_numpy(q).cuda(), bt, cl, P0 + w.steps, w.scale)
            kk = [np.concatenate([prompt_k, g[:step + 1]]) for g in gen_k]
            vv = [np.concatenate([prompt_v, g[:step + 1]]) for g in gen_v]
            worst = max(worst, max_abs(out.cpu().numpy(), OA.decode_attention(q, kk, vv, w.scale)))
    assert worst <= tol_for("f16"), worst
    st = alloc.stats()
    assert st.num_blocks - st.free_blocks == 136            # 64 shared + 8 x 9 private
    assert all(alloc.seq_info(c) == (P0 + w.steps, 73) for c in cands)
    assert cache.device_error() == 0


# ------------------------------------------------------------------ ragged (fp16 / fp8), small

def _ragged_small(B, dtype, seed, H=4):
    rng = np.random.default_rng(seed)
    lens = np.floor(np.exp(rng.uniform(0, math.log(3000), 24))).astype(int).tolist()
    lens[:5] = [1, B, B + 1, 32, 33]
    d = 128
    nb = sum(-(-n // B) for n in lens) + 9
    w = W.Workload("ragged_small", seed, 1, H, d, B, "f16", len(lens), lens, nb, 1 / math.sqrt(d))
    cache = PagedKVCache(1, nb, B, H, d, dtype)
    poison(cache)
    alloc = BlockAllocator(nb, B, W.free_order(w))
    seqs = [alloc.new_seq() for _ in lens]
    ks = [W.host_tokens(w, s, n, "k") for s, n in enumerate(lens)]
    vs = [W.host_tokens(w, s, n, "v") for s, n in enumerate(lens)]
    if dtype == "fp8":
        # set each block's scale before appending into it (caller's prefill choice)
        for s, sid in enumerate(seqs):
            n = lens[s]
            slots, _ = alloc.append_slots(sid, n)
            phys = [slots[j * B] // B for j in range(-(-n // B))]
            ksc, vsc = fp8_block_scales(ks[s], B), fp8_block_scales(vs[s], B)
            idx = torch.tensor(phys, dtype=torch.int64, device="cuda")
            cache.k_scale[0][idx] = torch.from_numpy(ksc).cuda()
            cache.v_scale[0][idx] = torch.from_numpy(vsc).cuda()
            cache.append(0, torch.from_numpy(ks[s]).cuda(), torch.from_numpy(vs[s]).cuda(),
                         torch.tensor(slots, dtype=torch.int64, device="cuda"))
    else:
        prefill(cache, alloc, seqs, ks, vs)
    return w, cache, alloc, seqs, ks, vs


@pytest.mark.parametrize("B", [8, 16, 32])
@pytest.mark.parametrize("dtype", ["f16", "fp8"])
@pytest.mark.parametrize("H", [4, 3])
def test_ragged_small_against_full_oracle(B, dtype, H):
    """An even head count takes the head-pair launch shape for FP8 pools with B 8 or 16 and
    fp16 pools with B 8; an odd one keeps one head per work item."""
    w, cache, alloc, seqs, ks, vs = _ragged_small(B, dtype, 50 + B, H)
    max_blocks = max(-(-n // B) for n in w.lens)
    bt, cl, lens = tables_for(alloc, seqs, max_blocks)
    q = W.host_queries(w)
    if dtype == "fp8":
        # oracle on the dequantised cache it quantises itself from the same inputs
        ksd, vsd = [], []
        for s in range(len(lens)):
            ksc, vsc = fp8_block_scales(ks[s], B), fp8_block_scales(vs[s], B)
            rows = np.arange(lens[s]) // B
            ksd.append(OF.decode(OF.quantize(ks[s], ksc[rows].reshape(-1, 1, 1))) *
                       ksc[rows].astype(np.float64).reshape(-1, 1, 1))
            vsd.append(OF.decode(OF.quantize(vs[s], vsc[rows].reshape(-1, 1, 1))) *
                       vsc[rows].astype(np.float64).reshape(-1, 1, 1))
        want = OA.decode_attention(q, ksd, vsd, w.scale)
    else:
        want = OA.decode_attention(q, ks, vs, w.scale)
    for P in (0, 32, 32 * B):
        out = cache.attention(0, torch.from_numpy(q).cuda(), bt, cl, max(lens), w.scale,
                              partition_tokens=P).cpu().numpy()
        assert max_abs(out, want) <= tol_for("f16"), (P, max_abs(out, want))
    assert cache.device_error() == 0


# ------------------------------------------------------------------ edge cases

def test_edge_lengths_and_errors():
    B, H, d = 16, 2, 64
    lens = [0, 1, 15, 16, 17, 32, 33, 64, 65, 511, 512, 513]
    nb = sum(-(-n // B) for n in lens) + 4
    w = W.Workload("edges", 77, 1, H, d, B, "f32", len(lens), lens, nb, 0.125)
    cache = PagedKVCache(1, nb, B, H, d, "f32")
    poison(cache)
    alloc = BlockAllocator(nb, B, W.free_order(w))
    seqs = [alloc.new_seq() for _ in lens]
    ks = [W.host_tokens(w, s, n, "k") for s, n in enumerate(lens)]
    vs = [W.host_tokens(w, s, n, "v") for s, n in enumerate(lens)]
    prefill(cache, alloc, seqs, ks, vs)
    max_blocks = max(-(-n // B) for n in lens)
    bt, cl, _ = tables_for(alloc, seqs, max_blocks)
    q = W.host_queries(w)
    want = OA.decode_attention(q, ks, vs, w.scale)
    for P in (0, 32, 64, 256, 512):
        out = cache.attention(0, torch.from_numpy(q).cuda(), bt, cl, max(lens), w.scale,
                              partition_tokens=P).cpu().numpy()
        assert max_abs(out, want) <= tol_for("f32"), P
        assert np.all(out[0] == 0.0)                     # empty context -> zeros
        assert np.array_equal(out[1], vs[1][0])         # n = 1: exactly the one value row
    assert cache.device_error() == 0
    # context longer than the table allows: clamped and flagged
    cl_bad = cl.clone()
    cl_bad[3] = max_blocks * B + 5
    cache.attention(0, torch.from_numpy(q).cuda(), bt, cl_bad, max_blocks * B + 5, w.scale)
    assert cache.device_error() & abi.KV_DEVERR_CONTEXT
    # a block id outside the pool: flagged, no fault
    bt_bad = bt.clone()
    bt_bad[2, 0] = nb + 100
    cache.attention(0, torch.from_numpy(q).cuda(), bt_bad, cl, max(lens), w.scale)
    assert cache.device_error() & abi.KV_DEVERR_BLOCK_ID
    # invalid host arguments are refused before any launch
    with pytest.raises(abi.KvError):
        cache.attention(0, torch.from_numpy(q).cuda(), bt, cl, max(lens), w.scale, partition_tokens=48)
    with pytest.raises(abi.KvError):
        cache.attention(0, torch.from_numpy(q).cuda(), bt, cl, max(lens), -1.0)


def test_large_batch_uses_several_launches():
    """More than 1024 sequences: the batch is split across launches with separate counters.
    A few long sequences in every launch split into more than 16 partitions, so the
    two-level merge's group counters of each launch are exercised too."""
    B, H, d = 8, 1, 64
    rng = np.random.default_rng(9)
    lens = rng.integers(0, 70, 2100).tolist()
    lens[5], lens[1024 + 5], lens[2048 + 5] = 900, 1000, 700   # same slot in every launch
    nb = sum(-(-n // B) for n in lens) + 1
    w = W.Workload("bigbatch", 91, 1, H, d, B, "f16", len(lens), lens, nb, 0.125)
    cache = PagedKVCache(1, nb, B, H, d, "f16")
    poison(cache)
    alloc = BlockAllocator(nb, B, W.free_order(w))
    seqs = [alloc.new_seq() for _ in lens]
    ks = [W.host_tokens(w, s, n, "k") for s, n in enumerate(lens)]
    vs = [W.host_tokens(w, s, n, "v") for s, n in enumerate(lens)]
    prefill(cache, alloc, seqs, ks, vs)
    bt, cl, _ = tables_for(alloc, seqs, max(1, max(-(-n // B) for n in lens)))
    q = W.host_queries(w)
    out = cache.attention(0, torch.from_numpy(q).cuda(), bt, cl, max(lens), w.scale, partition_tokens=32)
    assert max_abs(out.cpu().numpy(), OA.decode_attention(q, ks, vs, w.scale)) <= tol_for("f16")
    # grouped queries (2 per K/V head) over the same cache and launches
    q2 = np.concatenate([q, q[:, :, ::-1]], axis=1).copy()
    out2 = cache.attention_gqa(0, torch.from_numpy(q2).cuda(), bt, cl, max(lens), w.scale, partition_tokens=32)
    assert max_abs(out2.cpu().numpy(), OA.decode_attention_gqa(q2, ks, vs, w.scale)) <= tol_for("f16")
    assert cache.device_error() == 0


@pytest.mark.parametrize("dtype,d", [("f32", 128), ("f16", 64), ("fp8", 64)])
def test_other_head_dims_and_dtypes(dtype, d):
    B, H = 16, 3
    lens = [1, 40, 100, 300]
    nb = sum(-(-n // B) for n in lens) + 2
    w = W.Workload("dims", 33, 1, H, d, B, "f32" if dtype == "f32" else "f16", 4, lens, nb, d ** -0.5)
    cache = PagedKVCache(1, nb, B, H, d, dtype)
    poison(cache)
    alloc = BlockAllocator(nb, B, W.free_order(w))
    seqs = [alloc.new_seq() for _ in lens]
    ks = [W.host_tokens(w, s, n, "k") for s, n in enumerate(lens)]
    vs = [W.host_tokens(w, s, n, "v") for s, n in enumerate(lens)]
    if dtype == "fp8":
        for t in cache.k_scale + cache.v_scale:
            t.fill_(0.01)
    prefill(cache, alloc, seqs, ks, vs)
    bt, cl, _ = tables_for(alloc, seqs, max(-(-n // B) for n in lens))
    q = W.host_queries(w)
    out = cache.attention(0, torch.from_numpy(q).cuda(), bt, cl, max(lens), w.scale).cpu().numpy()
    if dtype == "fp8":
        ks = [OF.decode(OF.quantize(k, np.float32(0.01))) * float(np.float32(0.01)) for k in ks]
        vs = [OF.decode(OF.quantize(v, np.float32(0.01))) * float(np.float32(0.01)) for v in vs]
    assert max_abs(out, OA.decode_attention(q, ks, vs, w.scale)) <= tol_for(w.dtype)
    assert cache.device_error() == 0


# ------------------------------------------------------------------ long splits

@pytest.mark.parametrize("G", [1, 8])
def test_two_level_merge_of_long_splits(G):
    """With 32-token partitions these contexts split into 15, 16, 17, 32, 33, 257 and 282
    partitions: one-step merges up to 16, two-level merges beyond (groups of 16, the
    last group ragged, and more than 16 groups at the top)."""
    B, Hkv, d = 16, 2, 128
    lens = [15 * 32, 16 * 32, 16 * 32 + 1, 32 * 32, 33 * 32 - 5, 257 * 32, 9000]
    nb = sum(-(-n // B) for n in lens) + 4
    w = W.Workload("long_splits", 160 + G, 1, Hkv, d, B, "f16", len(lens), lens, nb, 1 / math.sqrt(d),
                   num_q_heads=G * Hkv)
    cache = PagedKVCache(1, nb, B, Hkv, d, "f16")
    poison(cache)
    alloc = BlockAllocator(nb, B, W.free_order(w))
    seqs = [alloc.new_seq() for _ in lens]
    ks = [W.host_tokens(w, s, n, "k") for s, n in enumerate(lens)]
    vs = [W.host_tokens(w, s, n, "v") for s, n in enumerate(lens)]
    prefill(cache, alloc, seqs, ks, vs)
    bt, cl, _ = tables_for(alloc, seqs, max(-(-n // B) for n in lens))
    q = W.host_queries(w)
    want = OA.decode_attention_gqa(q, ks, vs, w.scale) if G > 1 else OA.decode_attention(q, ks, vs, w.scale)
    qt = torch.from_numpy(q).cuda()
    for P in (32, 64, 0):
        if G > 1:
            out = cache.attention_gqa(0, qt, bt, cl, max(lens), w.scale, partition_tokens=P)
        else:
            out = cache.attention(0, qt, bt, cl, max(lens), w.scale, partition_tokens=P)
        out = out.cpu().numpy()
        assert np.all(np.isfinite(out))
        assert max_abs(out, want) <= tol_for("f16"), (P, max_abs(out, want))
    assert cache.device_error() == 0
